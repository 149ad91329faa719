"""GPU parity of the batched (prefill) path against the float64 oracle.

Calls of at least 44 tokens take the batched path, and so does any call with
MOE_BATCHED, which these tests set so that small shapes exercise it too: a router GEMM, one warp
per token for the selection, a stable counting sort of the (token, pick) pairs
by expert, and grouped GEMMs on the tensor cores over 4-bit weights dequantised
to f16. Bars as for decode: identical ordered picks, weights within W_REL, each
token's output within relative L2 OUT_REL_L2.
"""

import os

import numpy as np
import pytest

from expert_ffn_decode_gb300 import synth
from oracle import moe_oracle as mo
from tests.helpers import GpuLayer, compare, margin_tokens, oracle_cfg, rel_l2

pytestmark = pytest.mark.gpu

BATCHED = 32  # MOE_BATCHED


@pytest.fixture(scope="module", autouse=True)
def built():
    import expert_ffn_decode_gb300 as ffn
    if not os.path.exists(ffn.LIB_PATH):
        from expert_ffn_decode_gb300 import build
        build.build()
    import torch
    assert torch.cuda.is_available()
    yield
    ffn.moe_shutdown()


def _small(seed, **kw):
    w = dict(hidden=256, n_experts=16, top_k=4, expert_ff=128, shared_ff=0, n_groups=1, groups_used=1,
             qtype=mo.Q4_1, weights_scale=1.0, n_tokens=24, router_std=0.1, bias_std=None, seed=seed)
    w.update(kw)
    return w


SHAPES = [
    _small(40, n_tokens=8),                                              # smallest batched call
    _small(41, qtype=mo.Q4_0, shared_ff=64, n_tokens=37),                # ragged token tail
    _small(42, hidden=96, expert_ff=96, qtype=mo.Q4_0),                  # K chunk of 3 blocks
    _small(43, hidden=96, expert_ff=160, shared_ff=96, qtype=mo.Q4_1, n_tokens=130),
    _small(44, n_experts=40, top_k=7, bias_std=0.1, n_tokens=50),
    _small(45, n_experts=4, top_k=2, n_tokens=300, shared_ff=32),        # > 128 pairs per expert
    _small(46, n_experts=32, n_groups=4, groups_used=2, top_k=5, bias_std=0.1, weights_scale=2.5),
    _small(47, n_experts=64, n_groups=8, groups_used=3, top_k=6, bias_std=0.1, qtype=mo.Q4_0),
    _small(48, hidden=3072, expert_ff=64, shared_ff=3072, n_experts=8, top_k=2, router_std=0.02, n_tokens=16),
    _small(49, hidden=512, expert_ff=3072, n_experts=6, top_k=3, router_std=0.05, qtype=mo.Q4_0, n_tokens=20),
    _small(50, hidden=1024, expert_ff=32, shared_ff=32, n_experts=1000, top_k=32, router_std=0.05, n_tokens=64),
    _small(51, n_experts=128, n_groups=64, groups_used=5, top_k=9, bias_std=0.1, n_tokens=33),
    _small(52, hidden=32, expert_ff=32, n_experts=2, top_k=1, n_tokens=9),
    _small(53, n_experts=12, top_k=12, n_tokens=12),                     # k = E: every expert every token
    # shapes of whole 128-value (Q4_1) or 256-value (Q4_0) chunks take the tile pipeline
    _small(54, n_experts=4, top_k=2, n_tokens=300, shared_ff=128),       # > 64 pairs per expert
    _small(55, hidden=512, expert_ff=256, shared_ff=256, qtype=mo.Q4_0, n_tokens=70),
    _small(56, hidden=1024, expert_ff=128, shared_ff=128, n_experts=1000, top_k=32, router_std=0.05,
           n_tokens=40),                                                 # ragged 64-expert router tile
    _small(57, n_experts=64, n_groups=8, groups_used=3, top_k=6, bias_std=0.1, n_tokens=130,
           shared_ff=128),
    # the tile router's K slices: 7 units of 128 values in slices of 2, the last holding one
    _small(65, hidden=896, expert_ff=128, shared_ff=128, n_tokens=50),
    # 3 units, one a slice; a ragged 64-expert tile; two passes (512 and 128 tokens)
    _small(66, hidden=384, expert_ff=256, n_experts=96, top_k=5, n_tokens=640),
]


@pytest.mark.parametrize("w", SHAPES, ids=[f"s{w['seed']}_t{w['n_tokens']}" for w in SHAPES])
def test_prefill_shapes(w):
    layer = synth.make_layer(w)
    x, _ = margin_tokens(layer, w, w["n_tokens"], seed=w["seed"])
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                               layer["shared_blocks"], oracle_cfg(w))
    out, ids, wts = GpuLayer(layer, w).run(x, flags=BATCHED)
    err = compare(out, ids, wts, ref, rid, rwt, f"seed {w['seed']}")
    print(f"seed {w['seed']} T={w['n_tokens']}: max rel-L2 {err:.3e}")


CLAMP = [
    _small(58, shared_ff=128, n_tokens=40, swiglu_limit=0.8, swiglu_limit_shared=0.5),   # tile path
    _small(59, hidden=96, expert_ff=96, shared_ff=96, qtype=mo.Q4_0, n_tokens=20, swiglu_limit=0.7,
           swiglu_limit_shared=0.3),                                                      # general path
]


@pytest.mark.parametrize("w", CLAMP, ids=["tile", "general"])
def test_prefill_swiglu_clamp(w):
    layer = synth.make_layer(w)
    x, _ = margin_tokens(layer, w, w["n_tokens"], seed=w["seed"])
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                               layer["shared_blocks"], oracle_cfg(w))
    out, ids, wts = GpuLayer(layer, w).run(x, flags=BATCHED)
    compare(out, ids, wts, ref, rid, rwt, f"clamp seed {w['seed']}")
    unclamped, _, _ = GpuLayer(layer, {**w, "swiglu_limit": 0.0, "swiglu_limit_shared": 0.0}).run(x, flags=BATCHED)
    assert min(rel_l2(out[t], unclamped[t]) for t in range(len(x))) > 1e-2


PROLOGUE = [
    _small(62, shared_ff=128, n_tokens=40, rms_eps=1e-5),                                 # tile path
    _small(63, hidden=96, expert_ff=96, shared_ff=96, qtype=mo.Q4_0, n_tokens=20, rms_eps=1e-6),
    _small(64, hidden=512, expert_ff=1024, n_experts=1, top_k=1, n_tokens=24, rms_eps=1e-5),  # dense layer
]


@pytest.mark.parametrize("w", PROLOGUE, ids=["tile", "general", "dense"])
def test_prefill_rms_norm_prologue(w):
    import expert_ffn_decode_gb300 as ffn
    import torch
    layer = synth.make_layer(w)
    norm = np.random.default_rng(w["seed"] + 100).uniform(0.5, 1.5, w["hidden"]).astype(np.float32)
    x, _ = margin_tokens(layer, w, w["n_tokens"], seed=w["seed"], norm=norm, scale=3.0)
    wn = {**w, "ffn_norm": torch.from_numpy(norm).cuda()}
    for flags, oflags in ((0, 0), (ffn.MOE_RESIDUAL, mo.RESIDUAL)):
        ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                                   layer["shared_blocks"], oracle_cfg(w, oflags), ffn_norm=norm)
        out, ids, wts = GpuLayer(layer, wn).run(x, flags=flags | BATCHED)
        compare(out, ids, wts, ref, rid, rwt, f"prologue seed {w['seed']} flags {flags}")


@pytest.mark.parametrize("shared_ff", [64, 128], ids=["general", "tile"])
def test_prefill_two_passes_and_decode_boundary(shared_ff):
    # without the flag 43 tokens decode (16 + 16 + 11 per launch), 44 take the batched path,
    # 600 run as passes of 512 + 88
    w = _small(60, n_experts=16, top_k=3, shared_ff=shared_ff)
    layer = synth.make_layer(w)
    x, _ = margin_tokens(layer, w, 600, seed=60)
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                               layer["shared_blocks"], oracle_cfg(w))
    g = GpuLayer(layer, w)
    for T in (43, 44, 513, 600):
        out, ids, wts = g.run(x[:T])
        compare(out, ids, wts, ref[:T], rid[:T], rwt[:T], f"T={T}")


def test_prefill_flags_and_determinism():
    import expert_ffn_decode_gb300 as ffn
    import torch
    w = _small(61, shared_ff=128, n_tokens=40)
    layer = synth.make_layer(w)
    x, _ = margin_tokens(layer, w, 40, seed=61)
    g = GpuLayer(layer, w)
    base, ids, wts = g.run(x, flags=BATCHED)
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                               layer["shared_blocks"], oracle_cfg(w))
    compare(base, ids, wts, ref, rid, rwt, "plain")
    init = np.random.default_rng(62).standard_normal(x.shape).astype(np.float32)
    acc, _, _ = g.run(x, flags=ffn.MOE_ACCUMULATE | BATCHED, out_init=init)
    assert rel_l2(acc - init, base) < 1e-6
    res, _, _ = g.run(x, flags=ffn.MOE_RESIDUAL | BATCHED)
    assert rel_l2(res - x, base) < 1e-6
    for _ in range(3):  # a fixed summation order: repeat calls agree bit for bit
        again, ia, wa = g.run(x, flags=BATCHED)
        assert np.array_equal(again, base) and np.array_equal(ia, ids) and np.array_equal(wa, wts)
    T, H = x.shape
    cfg = ffn.make_cfg(**{**w, "n_tokens": T, "flags": ffn.MOE_HOST_IO | BATCHED})
    ws = torch.zeros(ffn.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    xh = np.ascontiguousarray(x, np.float32)
    oh = np.full((T, H), np.nan, np.float32)
    ih = np.full((T, w["top_k"]), -1, np.int32)
    wh = np.full((T, w["top_k"]), np.nan, np.float32)
    st = torch.cuda.current_stream()
    ffn.check(ffn.moe_ffn_forward_ex(xh, g.router_w, g.bias, g.experts, g.shared, cfg, oh, ws, ws.numel(),
                                     st, ih, wh))
    ffn.check(ffn.moe_workspace_status(ws, st))
    assert np.array_equal(oh, base) and np.array_equal(ih, ids) and np.array_equal(wh, wts)
    # page-locked outputs are written in place by the kernels (no staging copy), also when
    # accumulating into them
    po = torch.full((T, H), float("nan")).pin_memory()
    pi = torch.full((T, w["top_k"]), -1, dtype=torch.int32).pin_memory()
    pw = torch.full((T, w["top_k"]), float("nan")).pin_memory()
    ffn.check(ffn.moe_ffn_forward_ex(xh, g.router_w, g.bias, g.experts, g.shared, cfg, po, ws, ws.numel(),
                                     st, pi, pw))
    st.synchronize()
    assert np.array_equal(po.numpy(), base) and np.array_equal(pi.numpy(), ids) and np.array_equal(pw.numpy(), wts)
    cfg_acc = ffn.make_cfg(**{**w, "n_tokens": T, "flags": ffn.MOE_HOST_IO | ffn.MOE_ACCUMULATE | BATCHED})
    po.copy_(torch.from_numpy(init))
    ffn.check(ffn.moe_ffn_forward_ex(xh, g.router_w, g.bias, g.experts, g.shared, cfg_acc, po, ws, ws.numel(),
                                     st, None, None))
    ffn.check(ffn.moe_workspace_status(ws, st))
    assert np.array_equal(po.numpy(), acc)


def test_flint_prefill_t512_all_tokens():
    # the full Flint-shaped batch, every token against the oracle: its picks and weights, and
    # its output element by element (relative L2 per token), as every parity test does
    w = synth.WORKLOADS["flint_prefill_t512"]
    layer = synth.make_layer(w)
    T = w["n_tokens"]
    x, _ = margin_tokens(layer, w, T, seed=w["seed"])
    out, ids, wts = GpuLayer(layer, w).run(x, flags=BATCHED)
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                               layer["shared_blocks"], oracle_cfg(w))
    err = compare(out, ids, wts, ref, rid, rwt, "flint T=512")
    print(f"flint_prefill_t512: all {T} tokens, max rel-L2 {err:.3e}")


def test_prefill_matches_decode_path():
    # the same tokens decoded one call at a time and as one batch: both near the oracle,
    # and near each other
    name = "flint_decode_t1"
    w = synth.WORKLOADS[name]
    layer = synth.make_layer(w)
    x, _ = margin_tokens(layer, w, 8, seed=70)
    g = GpuLayer(layer, w)
    batch, ib, wb = g.run(x, flags=BATCHED)
    one = [g.run(x[t:t + 1]) for t in range(8)]
    for t in range(8):
        assert np.array_equal(one[t][1][0], ib[t])
        assert rel_l2(one[t][0][0], batch[t]) < 2e-3
