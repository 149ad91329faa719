"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Bars: identical ordered picks, routing weights within W_REL, each token's
output within relative L2 OUT_REL_L2 (2e-3). Tokens are drawn with a selection
margin so fp32/fp64 rounding cannot reorder the picks.
"""

import os

import numpy as np
import pytest

from expert_ffn_decode_gb300 import synth
from oracle import moe_oracle as mo
from tests.helpers import GpuLayer, compare, margin_tokens, oracle_cfg, rel_l2

pytestmark = pytest.mark.gpu

_layers = {}


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


def layer_of(name):
    if name not in _layers:
        w = synth.WORKLOADS[name]
        _layers[name] = (w, synth.make_layer(w))
    return _layers[name]


DECODE = ["tiny_q4_0_t4", "flint_decode_t1", "lfm25_decode_t1", "ling_decode_t1"]


F32 = 64  # MOE_F32_ACT: the decode chain's f32 activations (the default is 16-bit block fixed point)


@pytest.mark.parametrize("flags", [0, F32], ids=["fixed", "f32"])
@pytest.mark.parametrize("name", DECODE)
def test_workload_parity(name, flags):
    w, layer = layer_of(name)
    T = w["n_tokens"]
    x, _ = margin_tokens(layer, w, T, seed=w["seed"])
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                               layer["shared_blocks"], oracle_cfg(w))
    g = GpuLayer(layer, w)
    out, ids, wts = g.run(x, flags=flags)
    err = compare(out, ids, wts, ref, rid, rwt, name)
    for t in range(T):  # and one token per call
        compare(*g.run(x[t:t + 1], flags=flags), ref[t:t + 1], rid[t:t + 1], rwt[t:t + 1], f"{name} token {t}")
    print(f"{name} ({'f32' if flags else 'fixed point'}): max rel-L2 {err:.3e}")


@pytest.mark.parametrize("name", DECODE[1:])
def test_workload_more_tokens(name):
    # eight more tokens of the decode layers, as one call of T = 8 (one launch of the decode chain)
    w, layer = layer_of(name)
    x, redraws = margin_tokens(layer, w, 8, seed=w["seed"], stream=2)
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                               layer["shared_blocks"], oracle_cfg(w))
    out, ids, wts = GpuLayer(layer, w).run(x)
    compare(out, ids, wts, ref, rid, rwt, name)


def _small(seed, **kw):
    w = dict(hidden=256, n_experts=16, top_k=4, expert_ff=128, shared_ff=0, n_groups=1, groups_used=1,
             qtype=mo.Q4_1, weights_scale=1.0, n_tokens=3, router_std=0.1, bias_std=None, seed=seed)
    w.update(kw)
    return w


RANDOM = [
    _small(10),
    _small(11, qtype=mo.Q4_0, shared_ff=64),
    _small(12, hidden=96, expert_ff=96, qtype=mo.Q4_0),                 # odd block count per row
    _small(13, hidden=96, expert_ff=160, shared_ff=96, qtype=mo.Q4_1),
    _small(14, n_experts=40, top_k=7, bias_std=0.1),                    # E not a multiple of 32
    _small(15, n_experts=12, top_k=12),                                 # k = E
    _small(16, n_experts=32, n_groups=4, groups_used=2, top_k=5, bias_std=0.1, weights_scale=2.5),
    _small(17, n_experts=64, n_groups=8, groups_used=3, top_k=6, bias_std=0.1, qtype=mo.Q4_0),
    _small(18, hidden=3072, expert_ff=64, shared_ff=3072, n_experts=8, top_k=2, router_std=0.02),
    _small(19, hidden=512, expert_ff=3072, n_experts=6, top_k=3, router_std=0.05, qtype=mo.Q4_0),
    _small(20, hidden=1024, expert_ff=32, shared_ff=32, n_experts=1000, top_k=32, router_std=0.05),
    _small(21, n_experts=128, n_groups=64, groups_used=5, top_k=9, bias_std=0.1),
    _small(22, hidden=32, expert_ff=32, n_experts=2, top_k=1),
]


@pytest.mark.parametrize("w", RANDOM, ids=[f"s{w['seed']}" for w in RANDOM])
def test_random_shapes(w):
    layer = synth.make_layer(w)
    x, _ = margin_tokens(layer, w, w["n_tokens"], seed=w["seed"])
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                               layer["shared_blocks"], oracle_cfg(w))
    g = GpuLayer(layer, w)
    for flags in (0, F32):
        out, ids, wts = g.run(x, flags=flags)
        compare(out, ids, wts, ref, rid, rwt, f"seed {w['seed']} flags {flags}")
        o1, i1, w1 = g.run(x[:1], flags=flags)
        compare(o1, i1, w1, ref[:1], rid[:1], rwt[:1], f"seed {w['seed']} flags {flags} one token")


CLAMP = [
    _small(30, shared_ff=64, swiglu_limit=0.8, swiglu_limit_shared=0.5),
    _small(31, qtype=mo.Q4_0, shared_ff=128, swiglu_limit=0.6, n_groups=4, groups_used=2, top_k=3,
           bias_std=0.1),
    _small(32, hidden=96, expert_ff=160, shared_ff=96, swiglu_limit=0.5, swiglu_limit_shared=0.9),
]


@pytest.mark.parametrize("w", CLAMP, ids=[f"s{w['seed']}" for w in CLAMP])
def test_swiglu_clamp(w):
    # the clamped SwiGLU (ling_moe_ssd.js swiglu), with limits that clamp a good share of
    # the gate and up values, against the oracle; the clamp must change the output
    layer = synth.make_layer(w)
    x, _ = margin_tokens(layer, w, w["n_tokens"], seed=w["seed"])
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                               layer["shared_blocks"], oracle_cfg(w))
    g = GpuLayer(layer, w)
    out, ids, wts = g.run(x)
    compare(out, ids, wts, ref, rid, rwt, f"clamp seed {w['seed']}")
    plain = {**w, "swiglu_limit": 0.0, "swiglu_limit_shared": 0.0}
    unclamped, _, _ = GpuLayer(layer, plain).run(x)
    assert min(rel_l2(out[t], unclamped[t]) for t in range(len(x))) > 1e-2


def test_ling_decode_with_clamp():
    # the Ling-shaped layer with both clamp limits set
    w0, layer = layer_of("ling_decode_t1")
    w = {**w0, "swiglu_limit": 1.0, "swiglu_limit_shared": 0.7}
    x, _ = margin_tokens(layer, w, 2, seed=9, stream=5)
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                               layer["shared_blocks"], oracle_cfg(w))
    out, ids, wts = GpuLayer(layer, w).run(x)
    compare(out, ids, wts, ref, rid, rwt, "ling clamp")


PROLOGUE = [
    _small(33, shared_ff=64, rms_eps=1e-5),
    _small(34, qtype=mo.Q4_0, n_experts=64, n_groups=8, groups_used=3, top_k=6, bias_std=0.1, rms_eps=1e-6),
    # a dense SwiGLU layer: one expert, always picked with weight 1 (the router is moot)
    _small(35, hidden=512, expert_ff=1024, n_experts=1, top_k=1, rms_eps=1e-5),
]


@pytest.mark.parametrize("w", PROLOGUE, ids=[f"s{w['seed']}" for w in PROLOGUE])
def test_rms_norm_prologue(w):
    # x += ffn(rms_norm(x) * ffn_norm): the prologue folded into the step, with the raw x
    # added back by the residual form; tokens scaled by 3 so the norm matters
    import expert_ffn_decode_gb300 as ffn
    import torch
    layer = synth.make_layer(w)
    norm = np.random.default_rng(w["seed"] + 100).uniform(0.5, 1.5, w["hidden"]).astype(np.float32)
    x, _ = margin_tokens(layer, w, w["n_tokens"], seed=w["seed"], norm=norm, scale=3.0)
    wn = {**w, "ffn_norm": torch.from_numpy(norm).cuda()}
    for flags, oflags in ((0, 0), (ffn.MOE_RESIDUAL, mo.RESIDUAL)):
        ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                                   layer["shared_blocks"], oracle_cfg(w, oflags), ffn_norm=norm)
        out, ids, wts = GpuLayer(layer, wn).run(x, flags=flags)
        compare(out, ids, wts, ref, rid, rwt, f"prologue seed {w['seed']} flags {flags}")


@pytest.mark.parametrize("name,T", [("flint_decode_t1", 16), ("flint_decode_t1", 21),
                                    ("ling_decode_t1", 7), ("lfm25_decode_t1", 39)])
def test_multi_token_decode(name, T):
    # calls of several tokens run the decode chain on up to 16 tokens per launch, with one
    # selection per token; each token's arithmetic is that of a single-token call, so the
    # outputs agree bit for bit with calls of one token, and with the oracle
    w, layer = layer_of(name)
    x, _ = margin_tokens(layer, w, T, seed=w["seed"], stream=6)
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                               layer["shared_blocks"], oracle_cfg(w))
    g = GpuLayer(layer, w)
    out, ids, wts = g.run(x)
    compare(out, ids, wts, ref, rid, rwt, f"{name} T={T}")
    for t in (0, T // 2, T - 1):
        o1, i1, w1 = g.run(x[t:t + 1])
        assert np.array_equal(o1[0], out[t]) and np.array_equal(i1[0], ids[t]) and np.array_equal(w1[0], wts[t])


def test_flags_accumulate_residual_hostio_nopdl():
    import expert_ffn_decode_gb300 as ffn
    w, layer = layer_of("flint_decode_t1")
    x, _ = margin_tokens(layer, w, 2, seed=5, stream=3)
    g = GpuLayer(layer, w)
    base, ids, wts = g.run(x)
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                               layer["shared_blocks"], oracle_cfg(w))
    compare(base, ids, wts, ref, rid, rwt, "plain")
    init = np.random.default_rng(6).standard_normal(x.shape).astype(np.float32)
    acc, _, _ = g.run(x, flags=ffn.MOE_ACCUMULATE, out_init=init)
    assert rel_l2(acc - init, base) < 1e-6
    res, _, _ = g.run(x, flags=ffn.MOE_RESIDUAL)
    assert rel_l2(res - x, base) < 1e-6
    nopdl, _, _ = g.run(x, flags=ffn.MOE_NO_PDL)
    assert np.array_equal(nopdl, base)
    # host buffers: the library stages x and out through its workspace
    import torch
    T, H = x.shape
    cfg = ffn.make_cfg(**{**w, "n_tokens": T, "flags": ffn.MOE_HOST_IO})
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
    cfg_acc = ffn.make_cfg(**{**w, "n_tokens": T, "flags": ffn.MOE_HOST_IO | ffn.MOE_ACCUMULATE})
    po.copy_(torch.from_numpy(init))
    ffn.check(ffn.moe_ffn_forward_ex(xh, g.router_w, g.bias, g.experts, g.shared, cfg_acc, po, ws, ws.numel(),
                                     st, None, None))
    ffn.check(ffn.moe_workspace_status(ws, st))
    assert np.array_equal(po.numpy(), acc)


def test_plain_entry_point_and_repeat_determinism():
    import expert_ffn_decode_gb300 as ffn
    import torch
    w, layer = layer_of("lfm25_decode_t1")
    x, _ = margin_tokens(layer, w, 1, seed=7, stream=4)
    g = GpuLayer(layer, w)
    first, ids, wts = g.run(x)
    cfg = ffn.make_cfg(**{**w, "n_tokens": 1})
    xd = torch.from_numpy(x).cuda()
    out = torch.empty_like(xd)
    ffn.check(ffn.moe_ffn_forward(xd, g.router_w, g.bias, g.experts, g.shared, cfg, out))
    assert np.array_equal(out.cpu().numpy(), first)
    # one workspace reused for many calls in a row: control words reset every call
    ws = torch.zeros(ffn.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    for _ in range(20):
        again, _, _ = g.run(x, workspace=ws)
        assert np.array_equal(again, first)


@pytest.mark.parametrize("name,T", [("flint_decode_t1", 1), ("lfm25_decode_t1", 3), ("tiny_q4_0_t4", 48)])
def test_graph_replay_matches_direct_calls(name, T):
    # MOE_GRAPH: the first call runs directly, the second captures, later ones replay the
    # graph; every call must equal the direct path bit for bit, with device and host buffers
    import expert_ffn_decode_gb300 as ffn
    import torch
    w, layer = layer_of(name)
    x, _ = margin_tokens(layer, w, T, seed=w["seed"], stream=15)
    g = GpuLayer(layer, w)
    want, wid, ww = g.run(x)
    st = torch.cuda.current_stream()
    for host in (False, True):
        flags = ffn.MOE_GRAPH | (ffn.MOE_HOST_IO if host else 0)
        cfg = ffn.make_cfg(**{**w, "n_tokens": T, "flags": flags})
        ws = torch.zeros(ffn.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
        if host:
            xd = torch.from_numpy(x).pin_memory()
            out = torch.full((T, w["hidden"]), float("nan")).pin_memory()
            ids = torch.full((T, w["top_k"]), -1, dtype=torch.int32).pin_memory()
            wts = torch.full((T, w["top_k"]), float("nan")).pin_memory()
        else:
            xd = torch.from_numpy(x).cuda()
            out = torch.full((T, w["hidden"]), float("nan"), device="cuda")
            ids = torch.full((T, w["top_k"]), -1, dtype=torch.int32, device="cuda")
            wts = torch.full((T, w["top_k"]), float("nan"), device="cuda")
        for call in range(4):
            out.fill_(float("nan"))
            ffn.check(ffn.moe_ffn_forward_ex(xd, g.router_w, g.bias, g.experts, g.shared, cfg, out, ws,
                                             ws.numel(), st, ids, wts))
            ffn.check(ffn.moe_workspace_status(ws, st))
            assert np.array_equal(out.cpu().numpy(), want), (host, call)
            assert np.array_equal(ids.cpu().numpy(), wid) and np.array_equal(wts.cpu().numpy(), ww), (host, call)
    ffn.moe_shutdown()  # drops the cached graphs


def test_bias_none_equals_zero_bias_and_empty_batch():
    import expert_ffn_decode_gb300 as ffn
    w = _small(30, bias_std=None)
    layer = synth.make_layer(w)
    x, _ = margin_tokens(layer, w, 2, seed=30)
    a, ia, wa = GpuLayer(layer, w).run(x)
    layer0 = dict(layer, bias=np.zeros(w["n_experts"], np.float32))
    b, ib, wb = GpuLayer(layer0, w).run(x)
    assert np.array_equal(a, b) and np.array_equal(ia, ib)
    cfg = ffn.make_cfg(**{**w, "n_tokens": 0})
    assert ffn.moe_ffn_forward_ex(None, None, None, None, None, cfg, None, None, 0, None) == ffn.MOE_OK


def test_weight_clamp_case():
    # every logit about -30: the picked sigmoids sum far below 2^-14, so w = p / 2^-14 * scale;
    # equal logits tie exactly and both sides pick the lowest indices
    w = _small(31, n_experts=8, top_k=3, weights_scale=2.5)
    layer = synth.make_layer(w)
    H = w["hidden"]
    layer["router_w"] = np.full((8, H), -30.0 / H, np.float32)
    x = np.ones((1, H), np.float32)
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], None, layer["expert_blocks"], None, oracle_cfg(w))
    assert list(rid[0]) == [0, 1, 2]
    out, ids, wts = GpuLayer(layer, w).run(x)
    compare(out, ids, wts, ref, rid, rwt, "clamp")


TIES = [
    # (experts, picks, groups, groups used, distinct router rows): the top class holds about
    # E / rows experts that tie exactly; up to 64 candidates take the pruned ranking, more
    # take the sorted-list rounds
    (256, 6, 1, 1, 5),
    (256, 8, 1, 1, 3),
    (512, 8, 8, 4, 6),
    (64, 6, 8, 3, 4),
    (1000, 7, 1, 1, 40),
]


@pytest.mark.parametrize("E,K,G,Gu,rows", TIES, ids=[f"E{t[0]}k{t[1]}g{t[2]}r{t[4]}" for t in TIES])
def test_selection_exact_ties(E, K, G, Gu, rows):
    # duplicated router rows give bit-identical logits on both sides: the picks are the
    # lowest experts of the best tie classes, in index order within a class
    w = _small(90 + rows, n_experts=E, top_k=K, n_groups=G, groups_used=Gu, hidden=128, expert_ff=64,
               router_std=0.1)
    layer = synth.make_layer(w)
    base = layer["router_w"][:rows].copy()
    layer["router_w"] = base[(np.arange(E) * 37) % rows]
    x = synth.make_tokens(5, w["hidden"], 2)
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], None, layer["expert_blocks"], None, oracle_cfg(w))
    out, ids, wts = GpuLayer(layer, w).run(x)
    compare(out, ids, wts, ref, rid, rwt, "ties")
    for t in range(2):  # and one token per call (the selection inside the gate/up and down CTAs)
        o1, i1, w1 = GpuLayer(layer, w).run(x[t:t + 1])
        compare(o1, i1, w1, ref[t:t + 1], rid[t:t + 1], rwt[t:t + 1], f"ties token {t}")


def test_device_wait_timeout_is_reported_and_cleared():
    # a bounded device wait that nothing completes gives up, the status word says so, reading
    # it clears it, and the context keeps working (no fault, trap or unbounded loop involved)
    import expert_ffn_decode_gb300 as ffn
    import torch
    w, layer = layer_of("tiny_q4_0_t4")
    cfg = ffn.make_cfg(**{**w, "n_tokens": 1})
    ws = torch.zeros(ffn.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    assert ffn.moe_selftest_timeout(ws, st) == ffn.MOE_OK
    assert ffn.moe_workspace_status(ws, st) == ffn.MOE_ERR_TIMEOUT
    assert "timed out" in ffn.moe_last_error()
    assert ffn.moe_workspace_status(ws, st) == ffn.MOE_OK
    x, _ = margin_tokens(layer, w, 1, seed=w["seed"], stream=7)
    ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                               layer["shared_blocks"], oracle_cfg(w))
    compare(*GpuLayer(layer, w).run(x, workspace=ws), ref, rid, rwt, "after the timeout")
