"""Seeded synthetic inputs for the routed MoE-FFN step.

This module only draws random numbers and lays them out in the byte formats the
layer consumes. It holds none of the layer's arithmetic (no dequantisation, no
routing, no SwiGLU): both the CUDA path and the CPU oracle receive the same
bytes from here.

Byte formats (ggml block layout, little-endian):
  * Q4_0 block, 18 bytes: f16 scale ``d`` then 16 nibble bytes.
  * Q4_1 block, 20 bytes: f16 scale ``d``, f16 offset ``m``, then 16 nibble bytes.
  * An expert record is the gate matrix [F][H/32 blocks], then the up matrix
    [F][H/32 blocks], then the down matrix [H][F/32 blocks]; records are packed
    back to back, expert 0 first.

The workloads below are shaped like the three MoE models whose engines the
source pages describe ("Recursive Flint" Q4_1, LFM2.5-24B-A2B Q4_0, Ling 3.0
Flash), at the sizes their layer headers state; the distributions are the
synthetic ones stated per workload (no trained weights are used anywhere).
"""

from __future__ import annotations

import numpy as np

Q4_0 = 2  # ggml type id of Q4_0
Q4_1 = 3  # ggml type id of Q4_1
BLOCK_BYTES = {Q4_0: 18, Q4_1: 20}

# Shapes and distributions of the synthetic layers. ``router_std`` is the std of
# the f32 router matrix, ``bias_std`` the std of the selection-only bias (None:
# no bias), ``d`` and ``m`` the uniform ranges of the block scale and offset.
WORKLOADS = {
    # Tiny layer: H=256, 16 experts, top-2, F=128, no shared expert, Q4_0, T=4.
    "tiny_q4_0_t4": dict(hidden=256, n_experts=16, top_k=2, expert_ff=128, shared_ff=0,
                         n_groups=1, groups_used=1, qtype=Q4_0, weights_scale=1.0,
                         n_tokens=4, router_std=0.05, bias_std=None, seed=0),
    # Flint-shaped decode: H=2048, 256 experts, top-6, F=512, shared F=1024, Q4_1, T=1.
    "flint_decode_t1": dict(hidden=2048, n_experts=256, top_k=6, expert_ff=512, shared_ff=1024,
                            n_groups=1, groups_used=1, qtype=Q4_1, weights_scale=1.0,
                            n_tokens=1, router_std=0.02, bias_std=None, seed=1),
    # LFM2.5-shaped decode: H=2048, 64 experts, top-4 with selection bias, F=1536, Q4_0, T=1.
    "lfm25_decode_t1": dict(hidden=2048, n_experts=64, top_k=4, expert_ff=1536, shared_ff=0,
                            n_groups=1, groups_used=1, qtype=Q4_0, weights_scale=1.0,
                            n_tokens=1, router_std=0.02, bias_std=0.1, seed=2),
    # Ling-shaped decode: H=2560, 512 experts in 8 groups (keep 4), top-8, F=768,
    # shared F=768, scale 2.5, Q4_1, T=1.
    "ling_decode_t1": dict(hidden=2560, n_experts=512, top_k=8, expert_ff=768, shared_ff=768,
                           n_groups=8, groups_used=4, qtype=Q4_1, weights_scale=2.5,
                           n_tokens=1, router_std=0.02, bias_std=0.1, seed=3),
    # Flint-shaped batched prefill: the Flint decode layer over T=512 tokens.
    "flint_prefill_t512": dict(hidden=2048, n_experts=256, top_k=6, expert_ff=512, shared_ff=1024,
                               n_groups=1, groups_used=1, qtype=Q4_1, weights_scale=1.0,
                               n_tokens=512, router_std=0.02, bias_std=None, seed=4),
}

D_RANGE = (0.005, 0.02)   # block scale d ~ U(0.005, 0.02), stored as f16
M_RANGE = (-0.1, 0.0)     # Q4_1 block offset m ~ U(-0.1, 0), stored as f16


def record_bytes(hidden: int, expert_ff: int, qtype: int) -> int:
    """Bytes of one expert record (gate, up and down matrices)."""
    return 3 * expert_ff * (hidden // 32) * BLOCK_BYTES[qtype]


def q4_blocks(rng: np.random.Generator, qtype: int, n_blocks: int) -> np.ndarray:
    """``n_blocks`` random blocks as a flat uint8 array, drawn in block order.

    Per block: d (then m for Q4_1) from the uniform ranges above, rounded to
    f16; the 16 nibble bytes uniform over 0..255 (every nibble uniform 0..15).
    """
    bb = BLOCK_BYTES[qtype]
    out = np.empty((n_blocks, bb), np.uint8)
    d = rng.uniform(*D_RANGE, n_blocks).astype("<f2")
    out[:, 0:2] = d.view(np.uint8).reshape(n_blocks, 2)
    off = 2
    if qtype == Q4_1:
        m = rng.uniform(*M_RANGE, n_blocks).astype("<f2")
        out[:, 2:4] = m.view(np.uint8).reshape(n_blocks, 2)
        off = 4
    out[:, off:] = rng.integers(0, 256, (n_blocks, 16), dtype=np.uint8)
    return out.reshape(-1)


def make_layer(w: dict, seed: int | None = None) -> dict:
    """One synthetic MoE layer as numpy arrays (host memory).

    Draw order from ``default_rng(seed)``: router matrix [E][H] f32, bias [E]
    f32 (if the workload has one), every expert record in expert order, then
    the shared-expert record (if any).
    """
    seed = w["seed"] if seed is None else seed
    rng = np.random.default_rng(seed)
    H, E, F, Fs, qt = w["hidden"], w["n_experts"], w["expert_ff"], w["shared_ff"], w["qtype"]
    router_w = rng.normal(0.0, w["router_std"], (E, H)).astype(np.float32)
    bias = None
    if w.get("bias_std") is not None:
        bias = rng.normal(0.0, w["bias_std"], E).astype(np.float32)
    nb_rec = record_bytes(H, F, qt) // BLOCK_BYTES[qt]
    experts = q4_blocks(rng, qt, E * nb_rec)
    shared = None
    if Fs:
        shared = q4_blocks(rng, qt, record_bytes(H, Fs, qt) // BLOCK_BYTES[qt])
    return dict(router_w=router_w, bias=bias, expert_blocks=experts, shared_blocks=shared)


def token_stream(seed: int, hidden: int, stream: int = 1):
    """Endless stream of fp32 tokens x ~ N(0, 1), one [H] vector per draw.

    Seeded by ``(seed, stream)`` so tokens are independent of the weight draw.
    """
    rng = np.random.default_rng([seed, stream])
    while True:
        yield rng.standard_normal(hidden).astype(np.float32)


def make_tokens(seed: int, hidden: int, n_tokens: int, stream: int = 1) -> np.ndarray:
    """The first ``n_tokens`` draws of :func:`token_stream` as [T][H] f32."""
    it = token_stream(seed, hidden, stream)
    if n_tokens == 0:
        return np.zeros((0, hidden), np.float32)
    return np.stack([next(it) for _ in range(n_tokens)])


# ---------------------------------------------------------------------------
# Device-side generation for large benchmark layers (same distributions, drawn
# with torch's seeded generator on the device; not byte-identical to the numpy
# draw above).
# ---------------------------------------------------------------------------

def q4_blocks_torch(gen, qtype: int, n_blocks: int, device):
    import torch
    bb = BLOCK_BYTES[qtype]
    out = torch.empty((n_blocks, bb), dtype=torch.uint8, device=device)
    d = torch.empty(n_blocks, device=device).uniform_(*D_RANGE, generator=gen).half()
    out[:, 0:2] = d.view(torch.uint8).view(n_blocks, 2)
    off = 2
    if qtype == Q4_1:
        m = torch.empty(n_blocks, device=device).uniform_(*M_RANGE, generator=gen).half()
        out[:, 2:4] = m.view(torch.uint8).view(n_blocks, 2)
        off = 4
    out[:, off:] = torch.randint(0, 256, (n_blocks, 16), dtype=torch.uint8, device=device,
                                 generator=gen)
    return out.view(-1)


def make_layer_torch(w: dict, seed: int, device) -> dict:
    """One synthetic layer drawn directly into device memory (torch tensors)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    H, E, F, Fs, qt = w["hidden"], w["n_experts"], w["expert_ff"], w["shared_ff"], w["qtype"]
    router_w = torch.empty((E, H), device=device).normal_(0.0, w["router_std"], generator=gen)
    bias = None
    if w.get("bias_std") is not None:
        bias = torch.empty(E, device=device).normal_(0.0, w["bias_std"], generator=gen)
    experts = q4_blocks_torch(gen, qt, E * (record_bytes(H, F, qt) // BLOCK_BYTES[qt]), device)
    shared = None
    if Fs:
        shared = q4_blocks_torch(gen, qt, record_bytes(H, Fs, qt) // BLOCK_BYTES[qt], device)
    return dict(router_w=router_w, bias=bias, expert_blocks=experts, shared_blocks=shared)


def make_tokens_torch(seed: int, hidden: int, n_tokens: int, device):
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.empty((n_tokens, hidden), device=device).normal_(0.0, 1.0, generator=gen)
