"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad configurations, pointers and workspaces on the host."""

import os
import re

import pytest

import expert_ffn_decode_gb300 as ffn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def built():
    if not os.path.exists(ffn.LIB_PATH):
        from expert_ffn_decode_gb300 import build
        build.build()
    return ffn.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moeffn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(moe_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(ffn.EXPORTS)


def test_library_exports_every_declared_symbol(built):
    for name in declared_functions():
        assert hasattr(built, name), name
        assert getattr(built, name) is not None


def _cfg(**kw):
    base = dict(hidden=2048, n_experts=256, top_k=6, expert_ff=512, shared_ff=1024, n_tokens=1,
                qtype=ffn.MOE_Q4_1)
    base.update(kw)
    return ffn.make_cfg(**base)


BAD = [
    dict(hidden=100), dict(hidden=0), dict(hidden=4096), dict(expert_ff=48), dict(shared_ff=-32),
    dict(n_experts=0), dict(n_experts=2048), dict(top_k=0), dict(top_k=33), dict(n_experts=4, top_k=5),
    dict(n_groups=3), dict(n_groups=256), dict(n_groups=8, groups_used=0),
    dict(n_groups=8, groups_used=9), dict(n_groups=16, groups_used=1, top_k=17),
    dict(n_tokens=-1), dict(qtype=8), dict(weights_scale=float("inf")), dict(norm_min=-1.0),
    dict(flags=256), dict(swiglu_limit=-1.0), dict(swiglu_limit_shared=float("nan")),
    dict(swiglu_limit=float("inf")), dict(rms_eps=-1.0), dict(rms_eps=float("nan")),
    dict(qtype=14), dict(qtype_down=13), dict(qtype_down=-1),
    dict(qtype=12, hidden=96),                      # K-quant gate/up rows: hidden % 256
    dict(qtype_down=14, expert_ff=128),             # K-quant down rows: expert_ff % 256
    dict(qtype_down=12, expert_ff=256, shared_ff=96),
]


@pytest.mark.parametrize("kw", BAD, ids=[str(b) for b in BAD])
def test_invalid_cfg_rejected(built, kw):
    cfg = _cfg(**kw)
    assert ffn.moe_workspace_size(cfg) == 0
    rc = ffn.moe_ffn_forward_ex(16, 16, None, 16, 16, cfg, 4096, 256, 1 << 20, None)
    assert rc == ffn.MOE_ERR_INVALID_CFG, (rc, ffn.moe_last_error())
    assert ffn.moe_last_error()


@pytest.mark.parametrize("kw", [dict(qtype=12, hidden=256, expert_ff=256), dict(qtype=12, qtype_down=14,
                                hidden=512, expert_ff=768, shared_ff=256), dict(qtype_down=14, expert_ff=512),
                                dict(qtype=12, qtype_down=2, hidden=256, expert_ff=96)])
def test_kquant_cfg_accepted(built, kw):
    assert ffn.moe_workspace_size(_cfg(**kw)) > 0, ffn.moe_last_error()


def test_valid_cfg_workspace_size(built):
    cfg = _cfg()
    n = ffn.moe_workspace_size(cfg)
    # control block, f32 logits and the f32 SwiGLU activations
    assert n >= 512 + 256 * 4 + (6 * 512 + 1024) * 4
    assert n % 256 == 0
    # host staging adds room for x, out and the top-k outputs
    assert ffn.moe_workspace_size(_cfg(flags=ffn.MOE_HOST_IO, n_tokens=4)) > ffn.moe_workspace_size(_cfg(n_tokens=4))


def test_null_and_empty(built):
    assert ffn.moe_ffn_forward_ex(None, None, None, None, None, _cfg(n_tokens=0), None, None, 0, None) == ffn.MOE_OK
    rc = ffn.moe_ffn_forward_ex(None, 16, None, 16, 16, _cfg(), 4096, 256, 1 << 20, None)
    assert rc == ffn.MOE_ERR_NULL_PTR
    rc = ffn.moe_ffn_forward_ex(4096, 16, None, 16, None, _cfg(), 8192, 256, 1 << 20, None)
    assert rc == ffn.MOE_ERR_NULL_PTR  # shared_ff > 0 without shared blocks
    rc = ffn.moe_ffn_forward_ex(4096, 16, None, 16, 16, _cfg(), 1 << 16, None, 1 << 20, None)
    assert rc == ffn.MOE_ERR_NULL_PTR  # no workspace
    # the plain form checks the configuration before touching the device
    assert ffn.moe_ffn_forward(None, None, None, None, None, _cfg(hidden=100), None) == ffn.MOE_ERR_INVALID_CFG
    assert ffn.moe_ffn_forward(None, None, None, None, None, _cfg(n_tokens=0), None) == ffn.MOE_OK


def test_alignment_and_workspace_checks(built):
    cfg = _cfg()
    big = 1 << 20
    X, O, R, EX, SH, WS = 1 << 24, 1 << 26, 1 << 28, 1 << 30, 1 << 32, 1 << 34
    call = lambda x=X, r=R, ex=EX, sh=SH, o=O, ws=WS, n=big: ffn.moe_ffn_forward_ex(x, r, None, ex, sh, cfg, o, ws, n, None)
    assert call(r=R + 4) == ffn.MOE_ERR_ALIGNMENT
    assert call(ex=EX + 2) == ffn.MOE_ERR_ALIGNMENT
    assert call(sh=SH + 8) == ffn.MOE_ERR_ALIGNMENT
    assert call(x=X + 4) == ffn.MOE_ERR_ALIGNMENT
    assert call(o=O + 4) == ffn.MOE_ERR_ALIGNMENT
    assert call(ws=WS + 16) == ffn.MOE_ERR_ALIGNMENT
    assert call(n=64) == ffn.MOE_ERR_WORKSPACE
    # x and out overlapping
    assert call(o=X + 1024) == ffn.MOE_ERR_INVALID_CFG
    assert "overlap" in ffn.moe_last_error()
