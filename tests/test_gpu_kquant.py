"""GPU parity of K-quant layers (Q4_K gate/up rows, Q6_K / Q4_K / Q4_0 / Q4_1 down rows).

The Ling store keeps Q4_K gate/up rows and Q6_K or Q4_K down rows (ling_moe_ssd.js, file
header and planLayoutLing). Both paths run them: the decode chain (block dots on 16-bit
fixed-point activations by default) and the batched path (the tile pipeline where the shapes fit
its copies, H, F, Fs multiples of 256 and Q6_K rows of at most 768 values; the general
contractions otherwise; super-blocks dequantised to f16 in both). Same bars as every parity test: identical ordered picks, weights
within W_REL, each token within relative L2 OUT_REL_L2.
"""

import os

import numpy as np
import pytest

from expert_ffn_decode_gb300 import synth
from oracle import moe_oracle as mo
from tests.helpers import GpuLayer, compare, margin_tokens, oracle_cfg

pytestmark = pytest.mark.gpu

BATCHED = 32  # MOE_BATCHED: the batched path whatever the token count

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


def _oracle(layer, w, x):
    return mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"], layer["shared_blocks"],
                      oracle_cfg(w))


@pytest.mark.parametrize("name", ["tiny_kq_t4", "tiny_k4_t4"])
def test_tiny_kquant_decode(name):
    w, layer = layer_of(name)
    x, _ = margin_tokens(layer, w, w["n_tokens"], seed=w["seed"])
    ref, rid, rwt = _oracle(layer, w, x)
    g = GpuLayer(layer, w)
    compare(*g.run(x), ref, rid, rwt, f"{name} T={len(x)}")   # one call of 4 tokens
    for t in range(len(x)):                                   # and single-token calls
        compare(*g.run(x[t:t + 1]), ref[t:t + 1], rid[t:t + 1], rwt[t:t + 1], f"{name} token {t}")


def _small(seed, **kw):
    w = dict(hidden=256, n_experts=16, top_k=4, expert_ff=256, shared_ff=0, n_groups=1, groups_used=1,
             qtype=mo.Q4_K, qtype_down=mo.Q6_K, weights_scale=1.0, n_tokens=3, router_std=0.1,
             bias_std=None, seed=seed)
    w.update(kw)
    return w


MIXED = [
    _small(70),
    _small(71, qtype_down=mo.Q4_K, shared_ff=256),
    _small(72, qtype_down=mo.Q4_0, expert_ff=96, shared_ff=160),       # K gate/up, 4-bit down
    _small(73, qtype=mo.Q4_1, qtype_down=mo.Q6_K, hidden=96),          # 4-bit gate/up, Q6_K down
    _small(74, hidden=512, expert_ff=768, shared_ff=512, n_experts=40, top_k=7, bias_std=0.1),
    _small(75, n_experts=64, n_groups=8, groups_used=3, top_k=6, bias_std=0.1, weights_scale=2.5),
    _small(76, hidden=3072, expert_ff=256, shared_ff=3072, n_experts=8, top_k=2, router_std=0.02),
    _small(77, hidden=256, expert_ff=3072, n_experts=6, top_k=3, router_std=0.05, qtype_down=mo.Q4_K),
    _small(78, shared_ff=256, swiglu_limit=0.6, swiglu_limit_shared=0.9),
]


@pytest.mark.parametrize("flags", [0, 64], ids=["fixed", "f32"])  # 64: MOE_F32_ACT
@pytest.mark.parametrize("w", MIXED, ids=[f"s{w['seed']}" for w in MIXED])
def test_mixed_types_decode(w, flags):
    layer = synth.make_layer(w)
    x, _ = margin_tokens(layer, w, w["n_tokens"], seed=w["seed"])
    ref, rid, rwt = _oracle(layer, w, x)
    g = GpuLayer(layer, w)
    compare(*g.run(x, flags=flags), ref, rid, rwt, f"seed {w['seed']}")
    compare(*g.run(x[:1], flags=flags), ref[:1], rid[:1], rwt[:1], f"seed {w['seed']} one token")


@pytest.mark.parametrize("w", MIXED, ids=[f"s{w['seed']}" for w in MIXED])
def test_mixed_types_batched(w):
    # the same layers through the batched path (tile pipeline: seeds 70, 71, 74, 75, 77, 78;
    # general contractions: 72, 73, 76)
    w = {**w, "n_tokens": 37}
    layer = synth.make_layer(w)
    x, _ = margin_tokens(layer, w, w["n_tokens"], seed=w["seed"], stream=3)
    ref, rid, rwt = _oracle(layer, w, x)
    compare(*GpuLayer(layer, w).run(x, flags=BATCHED), ref, rid, rwt, f"batched seed {w['seed']}")


def test_ling_kquant_decode():
    # the full Ling-shaped Q4_K / Q6_K layer: two single-token calls and one call of 8 tokens
    w, layer = layer_of("ling_kq_decode_t1")
    x, _ = margin_tokens(layer, w, 10, seed=w["seed"])
    ref, rid, rwt = _oracle(layer, w, x)
    g = GpuLayer(layer, w)
    for flags in (0, 64):  # 64: MOE_F32_ACT
        for t in range(2):
            compare(*g.run(x[t:t + 1], flags=flags), ref[t:t + 1], rid[t:t + 1], rwt[t:t + 1], f"ling kq token {t}")
        compare(*g.run(x[2:], flags=flags), ref[2:], rid[2:], rwt[2:], "ling kq T=8")


def test_ling_kquant_batched_all_tokens():
    # 96 tokens of the full Ling-shaped K-quant layer on the batched path (96 is above the
    # batched threshold), every token against the oracle
    w, layer = layer_of("ling_kq_decode_t1")
    x, _ = margin_tokens(layer, w, 96, seed=w["seed"], stream=4)
    out, ids, wts = GpuLayer(layer, w).run(x)
    ref, rid, rwt = _oracle(layer, w, x)
    err = compare(out, ids, wts, ref, rid, rwt, "ling kq batched")
    print(f"ling_kq batched: all 96 tokens, max rel-L2 {err:.3e}")
