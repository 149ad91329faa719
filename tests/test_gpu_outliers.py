"""GPU parity on heavy-tailed activations, against the float64 oracle.

Trained models' FFN inputs carry a few outlier channels far larger than the rest. These
tests put one outlier channel in every 32-value block (the same channels for every
token), at 50, 300 and 1000 times the rest, and compare the CUDA path with the oracle
under the usual bars: identical ordered picks, weights within W_REL, each token within
relative L2 OUT_REL_L2 (2e-3).

The router matrix of these layers is divided by the tokens' typical RMS growth, so that
the logits keep the spread of the plain workloads: otherwise every sigmoid saturates to
1.0 and no token clears the tie margin. The experts see the outliers at full size.

Batched cases run near the f16 range the batched path states (every SwiGLU activation
below 65504): the outlier factor is the largest of a ladder whose activations, computed
with the oracle's own matrices, stay below that bound, and the test requires them to
reach at least a quarter of it.
"""

import os

import numpy as np
import pytest

from expert_ffn_decode_gb300 import synth
from oracle import moe_oracle as mo
from tests.helpers import GpuLayer, compare, margin_tokens, oracle_cfg

pytestmark = pytest.mark.gpu

BATCHED = 32  # MOE_BATCHED
F16_MAX = 65504.0

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


def rescaled(layer, factor):
    """The layer with its router divided by the RMS growth of a token whose 32-blocks each
    carry one channel `factor` times the rest."""
    s = np.float32(np.sqrt(1.0 + (factor * factor - 1.0) / 32.0))
    return dict(layer, router_w=(layer["router_w"] / s).astype(np.float32))


def oracle(layer, w, x, **kw):
    return mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"], layer["shared_blocks"],
                      oracle_cfg(w), **kw)


F32 = 64  # MOE_F32_ACT


@pytest.mark.parametrize("flags", [0, F32], ids=["fixed", "f32"])
@pytest.mark.parametrize("factor", [50.0, 300.0, 1000.0])
@pytest.mark.parametrize("name", ["flint_decode_t1", "lfm25_decode_t1", "ling_decode_t1"])
def test_outlier_channels_decode(name, factor, flags):
    # one call of three tokens and three single-token calls (the two decode forms), with f32
    # activations and with the 16-bit block fixed-point ones (the default)
    w, base = layer_of(name)
    layer = rescaled(base, factor)
    ch = synth.outlier_channels(w["hidden"], w["seed"])
    x, _ = margin_tokens(layer, w, 3, seed=w["seed"], stream=11,
                         transform=lambda v: synth.with_outliers(v, factor, ch))
    ref, rid, rwt = oracle(layer, w, x)
    g = GpuLayer(layer, w)
    err = compare(*g.run(x, flags=flags), ref, rid, rwt, f"{name} x{factor:g} T=3")
    for t in range(3):
        compare(*g.run(x[t:t + 1], flags=flags), ref[t:t + 1], rid[t:t + 1], rwt[t:t + 1],
                f"{name} x{factor:g} token {t}")
    print(f"{name} outliers x{factor:g} flags {flags}: max rel-L2 {err:.3e}")


@pytest.mark.parametrize("name", ["flint_decode_t1", "ling_decode_t1"])
def test_norm_prologue_with_large_norm_entries(name):
    # x += ffn(rms_norm(x) * ffn_norm) where eight ffn_norm entries are 100 times the rest:
    # the normalised input carries outlier channels of the norm's making
    import expert_ffn_decode_gb300 as ffn
    import torch
    w0, base = layer_of(name)
    w = {**w0, "rms_eps": 1e-6}
    H = w["hidden"]
    rng = np.random.default_rng(w["seed"] + 200)
    norm = rng.uniform(0.5, 1.5, H).astype(np.float32)
    big = rng.choice(H, 8, replace=False)
    norm[big] *= np.float32(100.0)
    # the normalised token's RMS grows by the norm vector's RMS: divide the router by it
    layer = dict(base, router_w=(base["router_w"] / np.float32(np.sqrt(np.mean(norm.astype(np.float64) ** 2))))
                 .astype(np.float32))
    x, _ = margin_tokens(layer, w, 3, seed=w["seed"], stream=12, norm=norm, scale=3.0)
    wn = {**w, "ffn_norm": torch.from_numpy(norm).cuda()}
    g = GpuLayer(layer, wn)
    for flags, oflags in ((0, 0), (ffn.MOE_RESIDUAL, mo.RESIDUAL)):
        ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                                   layer["shared_blocks"], oracle_cfg(w, oflags), ffn_norm=norm)
        compare(*g.run(x, flags=flags), ref, rid, rwt, f"{name} large norm entries flags {flags}")
        for t in range(2):
            compare(*g.run(x[t:t + 1], flags=flags), ref[t:t + 1], rid[t:t + 1], rwt[t:t + 1],
                    f"{name} large norm entries token {t}")


def max_activation(layer, w, x):
    """Largest |SwiGLU activation| over every token's picked experts and the shared
    expert, from the oracle's routing and dequantised matrices."""
    cfg = oracle_cfg(w)
    ids, _, _ = mo.route(x, layer["router_w"], layer["bias"], cfg)
    cache = mo.ExpertCache(layer["expert_blocks"], cfg)
    shared = (mo.expert_matrices(layer["shared_blocks"], w["hidden"], w["shared_ff"], w["qtype"],
                                 w.get("qtype_down", 0)) if w["shared_ff"] else None)
    top = 0.0
    for t in range(len(x)):
        mats = [cache(int(e)) for e in ids[t]] + ([shared] if shared is not None else [])
        for w_gu, _ in mats:
            gu = w_gu @ x[t].astype(np.float64)
            ff = len(gu) // 2
            g, u = gu[:ff], gu[ff:]
            top = max(top, float(np.max(np.abs(g / (1.0 + np.exp(-g)) * u))))
    return top


def _mid(seed, **kw):
    w = dict(hidden=1024, n_experts=16, top_k=4, expert_ff=256, shared_ff=256, n_groups=1, groups_used=1,
             qtype=mo.Q4_1, weights_scale=1.0, n_tokens=48, router_std=0.02, bias_std=None, seed=seed)
    w.update(kw)
    return w


NEAR_BOUND = [
    "flint",                                                    # the Flint-shaped layer, tile pipeline
    _mid(80),                                                   # tile pipeline (Q4_1, multiples of 128)
    _mid(81, qtype=mo.Q4_0, expert_ff=160, shared_ff=96),       # general contractions
]


@pytest.mark.parametrize("w", NEAR_BOUND, ids=["flint", "tile", "general"])
def test_outlier_channels_batched_near_f16_bound(w):
    if w == "flint":
        w0, base = layer_of("flint_decode_t1")
        w = {**w0, "n_tokens": 48}
    else:
        base = synth.make_layer(w)
    ch = synth.outlier_channels(w["hidden"], w["seed"])
    chosen = None
    for factor in (20.0, 30.0, 40.0, 60.0, 80.0, 120.0, 160.0, 240.0, 320.0, 480.0, 640.0):
        layer = rescaled(base, factor)
        x, _ = margin_tokens(layer, w, w["n_tokens"], seed=w["seed"], stream=13,
                             transform=lambda v, f=factor: synth.with_outliers(v, f, ch))
        top = max_activation(layer, w, x)
        if top >= 0.9 * F16_MAX:
            break
        chosen = (factor, layer, x, top)
    assert chosen is not None
    factor, layer, x, top = chosen
    assert top >= 0.25 * F16_MAX, f"largest activation {top:.0f} is not near the f16 bound"
    ref, rid, rwt = oracle(layer, w, x)
    out, ids, wts = GpuLayer(layer, w).run(x, flags=BATCHED)
    err = compare(out, ids, wts, ref, rid, rwt, f"batched outliers x{factor:g}")
    print(f"batched outliers x{factor:g}: largest activation {top:.0f}, max rel-L2 {err:.3e}")
