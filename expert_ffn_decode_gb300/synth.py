"""Seeded synthetic inputs for the routed MoE-FFN step.

This module only draws random numbers and lays them out in the byte formats the
layer consumes. It holds none of the layer's arithmetic (no dequantisation, no
routing, no SwiGLU): both the CUDA path and the CPU oracle receive the same
bytes from here.

Byte formats (ggml block layout, little-endian):
  * Q4_0 block, 18 bytes: f16 scale ``d`` then 16 nibble bytes.
  * Q4_1 block, 20 bytes: f16 scale ``d``, f16 offset ``m``, then 16 nibble bytes.
  * Q4_K super-block (256 values), 144 bytes: f16 ``d``, f16 ``dmin``, 12 bytes of
    packed 6-bit sub-block scales and mins, 128 nibble bytes.
  * Q6_K super-block (256 values), 210 bytes: 128 bytes of low nibbles, 64 bytes of
    2-bit high parts, 16 int8 sub-block scales, f16 ``d``.
  * An expert record is the gate matrix [F rows], then the up matrix [F rows] (rows
    of H values in the gate/up type), then the down matrix [H rows of F values in
    the down type, which defaults to the gate/up type]; records are packed back to
    back, expert 0 first.

The workloads below are shaped like the three MoE models whose engines the
source pages describe ("Recursive Flint" Q4_1, LFM2.5-24B-A2B Q4_0, Ling 3.0
Flash), at the sizes their layer headers state; the distributions are the
synthetic ones stated per workload (no trained weights are used anywhere).
"""

from __future__ import annotations

import numpy as np

Q4_0 = 2   # ggml type id of Q4_0
Q4_1 = 3   # ggml type id of Q4_1
Q4_K = 12  # ggml type id of Q4_K
Q6_K = 14  # ggml type id of Q6_K
BLOCK_BYTES = {Q4_0: 18, Q4_1: 20, Q4_K: 144, Q6_K: 210}   # bytes per block
BLOCK_VALUES = {Q4_0: 32, Q4_1: 32, Q4_K: 256, Q6_K: 256}  # values per block

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
    # The Ling-shaped layer as the Ling store holds it: Q4_K gate/up rows, Q6_K down rows.
    "ling_kq_decode_t1": dict(hidden=2560, n_experts=512, top_k=8, expert_ff=768, shared_ff=768,
                              n_groups=8, groups_used=4, qtype=Q4_K, qtype_down=Q6_K, weights_scale=2.5,
                              n_tokens=1, router_std=0.02, bias_std=0.1, seed=5),
    # The same K-quant layer over T=512 tokens (the batched path's general contractions).
    "ling_kq_prefill_t512": dict(hidden=2560, n_experts=512, top_k=8, expert_ff=768, shared_ff=768,
                                 n_groups=8, groups_used=4, qtype=Q4_K, qtype_down=Q6_K, weights_scale=2.5,
                                 n_tokens=512, router_std=0.02, bias_std=0.1, seed=8),
    # Small K-quant layers for the parity tests: H=256, 16 experts, top-2, F=256,
    # shared F=256, Q4_K gate/up with Q6_K (or Q4_K) down, T=4.
    "tiny_kq_t4": dict(hidden=256, n_experts=16, top_k=2, expert_ff=256, shared_ff=256,
                       n_groups=1, groups_used=1, qtype=Q4_K, qtype_down=Q6_K, weights_scale=1.0,
                       n_tokens=4, router_std=0.05, bias_std=None, seed=6),
    "tiny_k4_t4": dict(hidden=256, n_experts=16, top_k=2, expert_ff=256, shared_ff=256,
                       n_groups=1, groups_used=1, qtype=Q4_K, qtype_down=Q4_K, weights_scale=1.0,
                       n_tokens=4, router_std=0.05, bias_std=None, seed=7),
}

D_RANGE = (0.005, 0.02)   # block scale d ~ U(0.005, 0.02), stored as f16
M_RANGE = (-0.1, 0.0)     # Q4_1 block offset m ~ U(-0.1, 0), stored as f16
# K-quant super-block scales, chosen so the values span about what the 4-bit blocks
# above span: Q4_K d * sc (sc uniform 0..63) and dmin * mn (mn uniform 0..63) cover
# about [0, 0.04] and [0, 0.16]; Q6_K d * sc * (q - 32) (sc uniform int8) stays
# within +-0.82. All stored as normal f16 numbers.
Q4K_D_RANGE = (1.5e-4, 6.5e-4)
Q4K_DMIN_RANGE = (5e-4, 2.5e-3)
Q6K_D_RANGE = (1e-4, 2e-4)


def down_type(w: dict) -> int:
    """Block type of a workload's down matrices (the gate/up type unless stated)."""
    return w.get("qtype_down") or w["qtype"]


def row_bytes(n_values: int, qtype: int) -> int:
    """Bytes of one weight row of ``n_values`` values."""
    return n_values // BLOCK_VALUES[qtype] * BLOCK_BYTES[qtype]


def record_bytes(hidden: int, expert_ff: int, qtype: int, qtype_down: int = 0) -> int:
    """Bytes of one expert record (gate, up and down matrices)."""
    qd = qtype_down or qtype
    return 2 * expert_ff * row_bytes(hidden, qtype) + hidden * row_bytes(expert_ff, qd)


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


def kq_blocks(rng: np.random.Generator, qtype: int, n_blocks: int) -> np.ndarray:
    """``n_blocks`` random K-quant super-blocks as a flat uint8 array.

    Q4_K, per super-block: d then dmin from the ranges above (f16), then the 12
    scale bytes and the 128 nibble bytes uniform over 0..255. Q6_K: the 128 low
    and 64 high bytes uniform, the 16 scale bytes uniform (int8 -128..127), then
    d (f16). Each field is drawn for all super-blocks at once, in that order.
    """
    bb = BLOCK_BYTES[qtype]
    out = np.empty((n_blocks, bb), np.uint8)
    if qtype == Q4_K:
        d = rng.uniform(*Q4K_D_RANGE, n_blocks).astype("<f2")
        dmin = rng.uniform(*Q4K_DMIN_RANGE, n_blocks).astype("<f2")
        out[:, 0:2] = d.view(np.uint8).reshape(n_blocks, 2)
        out[:, 2:4] = dmin.view(np.uint8).reshape(n_blocks, 2)
        out[:, 4:144] = rng.integers(0, 256, (n_blocks, 140), dtype=np.uint8)
    elif qtype == Q6_K:
        out[:, 0:208] = rng.integers(0, 256, (n_blocks, 208), dtype=np.uint8)
        d = rng.uniform(*Q6K_D_RANGE, n_blocks).astype("<f2")
        out[:, 208:210] = d.view(np.uint8).reshape(n_blocks, 2)
    else:
        raise ValueError(f"not a K-quant type: {qtype}")
    return out.reshape(-1)


def any_blocks(rng: np.random.Generator, qtype: int, n_blocks: int) -> np.ndarray:
    return kq_blocks(rng, qtype, n_blocks) if qtype in (Q4_K, Q6_K) else q4_blocks(rng, qtype, n_blocks)


def records(rng: np.random.Generator, n_records: int, hidden: int, ff: int, qtype: int, qtype_down: int):
    """``n_records`` expert records. One block type for all three matrices: every
    block in record order. Otherwise the gate/up blocks of every record first, then
    the down blocks of every record, interleaved into records afterwards."""
    if qtype_down == qtype:
        return any_blocks(rng, qtype, n_records * record_bytes(hidden, ff, qtype) // BLOCK_BYTES[qtype])
    n_gu = 2 * ff * row_bytes(hidden, qtype) // BLOCK_BYTES[qtype]
    n_dn = hidden * row_bytes(ff, qtype_down) // BLOCK_BYTES[qtype_down]
    gu = any_blocks(rng, qtype, n_records * n_gu).reshape(n_records, -1)
    dn = any_blocks(rng, qtype_down, n_records * n_dn).reshape(n_records, -1)
    return np.concatenate([gu, dn], axis=1).reshape(-1)


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
    qd = down_type(w)
    experts = records(rng, E, H, F, qt, qd)
    shared = records(rng, 1, H, Fs, qt, qd) if Fs else None
    return dict(router_w=router_w, bias=bias, expert_blocks=experts, shared_blocks=shared)


def token_stream(seed: int, hidden: int, stream: int = 1):
    """Endless stream of fp32 tokens x ~ N(0, 1), one [H] vector per draw.

    Seeded by ``(seed, stream)`` so tokens are independent of the weight draw.
    """
    rng = np.random.default_rng([seed, stream])
    while True:
        yield rng.standard_normal(hidden).astype(np.float32)


def outlier_channels(hidden: int, seed: int) -> np.ndarray:
    """One channel index per 32-value block: the channel a heavy-tailed token scales.

    Drawn once from ``default_rng([seed, 999])``, uniform over the block's 32 positions,
    so every token of a test shares the same outlier channels, as trained models'
    activations do.
    """
    rng = np.random.default_rng([seed, 999])
    return np.arange(0, hidden, 32) + rng.integers(0, 32, hidden // 32)


def with_outliers(x: np.ndarray, factor: float, channels: np.ndarray) -> np.ndarray:
    """``x`` (f32 [..., H]) with the given channels multiplied by ``factor`` (rounded to f32)."""
    y = np.array(x, np.float32, copy=True)
    y[..., channels] *= np.float32(factor)
    return y


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


def kq_blocks_torch(gen, qtype: int, n_blocks: int, device):
    import torch
    bb = BLOCK_BYTES[qtype]
    out = torch.empty((n_blocks, bb), dtype=torch.uint8, device=device)
    if qtype == Q4_K:
        d = torch.empty(n_blocks, device=device).uniform_(*Q4K_D_RANGE, generator=gen).half()
        dmin = torch.empty(n_blocks, device=device).uniform_(*Q4K_DMIN_RANGE, generator=gen).half()
        out[:, 0:2] = d.view(torch.uint8).view(n_blocks, 2)
        out[:, 2:4] = dmin.view(torch.uint8).view(n_blocks, 2)
        out[:, 4:] = torch.randint(0, 256, (n_blocks, 140), dtype=torch.uint8, device=device, generator=gen)
    else:
        out[:, 0:208] = torch.randint(0, 256, (n_blocks, 208), dtype=torch.uint8, device=device, generator=gen)
        d = torch.empty(n_blocks, device=device).uniform_(*Q6K_D_RANGE, generator=gen).half()
        out[:, 208:210] = d.view(torch.uint8).view(n_blocks, 2)
    return out.view(-1)


def records_torch(gen, n_records: int, hidden: int, ff: int, qtype: int, qtype_down: int, device):
    import torch

    def blocks(qt, n):
        return kq_blocks_torch(gen, qt, n, device) if qt in (Q4_K, Q6_K) else q4_blocks_torch(gen, qt, n, device)

    if qtype_down == qtype:
        return blocks(qtype, n_records * record_bytes(hidden, ff, qtype) // BLOCK_BYTES[qtype])
    n_gu = 2 * ff * row_bytes(hidden, qtype) // BLOCK_BYTES[qtype]
    n_dn = hidden * row_bytes(ff, qtype_down) // BLOCK_BYTES[qtype_down]
    gu = blocks(qtype, n_records * n_gu).view(n_records, -1)
    dn = blocks(qtype_down, n_records * n_dn).view(n_records, -1)
    return torch.cat([gu, dn], dim=1).reshape(-1)


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
    qd = down_type(w)
    experts = records_torch(gen, E, H, F, qt, qd, device)
    shared = records_torch(gen, 1, H, Fs, qt, qd, device) if Fs else None
    return dict(router_w=router_w, bias=bias, expert_blocks=experts, shared_blocks=shared)


def make_tokens_torch(seed: int, hidden: int, n_tokens: int, device):
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.empty((n_tokens, hidden), device=device).normal_(0.0, 1.0, generator=gen)
