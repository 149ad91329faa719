"""CPU oracle of the routed MoE-FFN step, in float64.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import or call this
module: only the tests, the smoke check and the benchmark's CPU-baseline leg do.
It shares no code with the CUDA library; it receives the same input bytes.

What it computes, step by step, each written from the passage named beside it
(sources: the engine modules ``flint_moe_ssd.js``, ``ling_moe_ssd.js`` and
``lfm2_moe_ssd.js`` of the npm package diskformer, as shown by diffend.io):

1. Dequantise blocks (flint_moe_ssd.js, WGSL section, the Q4_1 comment above
   ``Q41DOT``: word 0 = f16 d | f16 m << 16, nibble bytes in ggml's order, low
   nibbles = values 0..15, high nibbles = values 16..31, value = d*q + m). Q4_0:
   f16 d followed by 16 nibble bytes, value = d*(q - 8) (the pages name the
   format only; the value rule is the plain ggml reading, listed as a reading).
   K-quant super-blocks of 256 values (ling_moe_ssd.js header and
   ``planLayoutLing``: the Ling store keeps Q4_K gate/up rows and Q6_K or Q4_K
   down rows; the block layouts themselves are not on the pages, so they are
   the public ggml layouts, restated in ``dequant_q4k`` and ``dequant_q6k``).
2. Router logits = router matrix (F32 ``ffn_gate_inp``, row e = expert e) times
   x (lfm2_moe_ssd.js, ``matmulF32`` router binding in ``initBuffers``).
3. p = sigmoid(logit); selection score s = p + bias; the bias only selects
   (lfm2_moe_ssd.js, ``TOPK_SIG_BODY`` and the comment above it).
4. With groups (ling_moe_ssd.js, ``routeLing``): group score = sum of the two
   largest s in the group; keep the ``groups_used`` best groups, scanning with
   a strict ``>`` so the lowest group wins ties.
5. k rounds of argmax over the allowed s, ties to the lowest index, the pick
   masked out after each round; picks kept in selection order (``TOPK_SIG_BODY``).
6. Weights w_j = p_pick_j / max(sum_j p_pick_j, 2^-14) * scale (``TOPK_SIG_BODY``,
   ``routeLing``: the sum clamped at 6.103515625e-5, scale applied after the
   division).
7. Each picked expert: gu = W_gu x (gate rows then up rows), act = silu(g) * u,
   y = W_down act (ling_moe_ssd.js ``swiglu``; flint_moe_ssd.js header: "SwiGLU
   experts (512)"). With a clamp limit L > 0 (ling_moe_ssd.js, the ``swiglu``
   kernel and the comment above it; its header: some layers clamp the SwiGLU,
   with separate per-layer limits for the routed and the shared experts), act =
   min(silu(g), L) * clamp(u, -L, L); L = 0 means no clamp.
8. The shared expert: the same SwiGLU on its own record with weight 1, no gate
   (flint_moe_ssd.js header: "one always-on shared SwiGLU expert (1024, no
   gate)").
9. out = sum_j w_j y_j + shared (ling_moe_ssd.js ``moeAccum``: x[h] += sum_j
   w_j out[j*H + h] + shared[h]); the oracle returns the contribution, or adds
   it to ``out_in`` when accumulating, or to x for the residual form.
0. Optional layer prologue: the step's input is rms_norm(x) * ffn_norm, with
   rms_norm(x) = x / sqrt(mean(x^2) + eps) (flint_moe_ssd.js and
   lfm2_moe_ssd.js headers: "x += ffn(rms_norm(x) * ffn_norm)"; eps is the
   model's ``attention.layer_norm_rms_epsilon``). The residual form then adds
   the un-normalised x, which makes the whole FFN block x += ffn(...).

Parity status: every step above is pinned by the not-gpu tests (golden blocks,
closed forms, brute-force routing, invariants); none is "parity unpinned". The
K-quant layouts are pinned to hand-built super-blocks and to the Q4_1 rule,
not to the pages, which do not print them.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

Q4_0 = 2
Q4_1 = 3
Q4_K = 12
Q6_K = 14
BLOCK_BYTES = {Q4_0: 18, Q4_1: 20, Q4_K: 144, Q6_K: 210}
BLOCK_VALUES = {Q4_0: 32, Q4_1: 32, Q4_K: 256, Q6_K: 256}
NORM_MIN = 6.103515625e-05  # 2^-14, the clamp on the sum of the picked sigmoids

ACCUMULATE = 1  # out = out_in + contribution
RESIDUAL = 2    # out = x + contribution


@dataclass
class MoeConfig:
    hidden: int
    n_experts: int
    top_k: int
    expert_ff: int
    shared_ff: int = 0
    n_groups: int = 1
    groups_used: int = 1
    qtype: int = Q4_1
    qtype_down: int = 0               # block type of the down matrices (0: qtype)
    weights_scale: float = 1.0
    norm_min: float = NORM_MIN
    flags: int = 0
    swiglu_limit: float = 0.0         # routed experts' clamp limit L (0: none)
    swiglu_limit_shared: float = 0.0  # the shared expert's
    rms_eps: float = 0.0              # the prologue's epsilon (used with an ffn_norm vector)


# --------------------------------------------------------------------------
# 1. Blocks
# --------------------------------------------------------------------------

def half_to_float(bits) -> np.ndarray:
    """IEEE 754 binary16 bit patterns -> float64, decoded from the bit fields.

    sign (1 bit), exponent e (5 bits, bias 15), fraction f (10 bits):
    e = 0: (-1)^s * f * 2^-24 (zero and subnormals); 0 < e < 31:
    (-1)^s * (1024 + f) * 2^(e - 25); e = 31: inf (f = 0) or NaN.
    """
    h = np.asarray(bits, dtype=np.int64)
    sign = np.where((h >> 15) & 1, -1.0, 1.0)
    e = (h >> 10) & 0x1F
    f = (h & 0x3FF).astype(np.float64)
    mag = np.where(e == 0, f * 2.0 ** -24, (1024.0 + f) * np.exp2((e - 25).astype(np.float64)))
    mag = np.where(e == 31, np.where(f == 0, np.inf, np.nan), mag)
    return sign * mag


def dequant_rows(blocks: np.ndarray, n_rows: int, n_cols: int, qtype: int) -> np.ndarray:
    """Dequantise ``n_rows`` rows of ``n_cols`` values each from raw block bytes.

    Row r holds blocks r*nb .. r*nb + nb - 1 (nb = n_cols / 32). In a block the
    16 nibble bytes give value i (i < 16) from the low nibble of byte i and value
    16 + i from its high nibble.
    """
    if qtype == Q4_K:
        return dequant_q4k(blocks, n_rows, n_cols)
    if qtype == Q6_K:
        return dequant_q6k(blocks, n_rows, n_cols)
    bb = BLOCK_BYTES[qtype]
    nb = n_cols // 32
    b = np.asarray(blocks, dtype=np.uint8).reshape(n_rows, nb, bb).astype(np.int64)
    d = half_to_float(b[..., 0] | (b[..., 1] << 8))
    if qtype == Q4_1:
        m = half_to_float(b[..., 2] | (b[..., 3] << 8))
        qs = b[..., 4:20]
    elif qtype == Q4_0:
        qs = b[..., 2:18]
    else:
        raise ValueError(f"unknown block type {qtype}")
    q = np.concatenate([qs & 0x0F, qs >> 4], axis=-1).astype(np.float64)  # (rows, nb, 32)
    if qtype == Q4_1:
        v = d[..., None] * q + m[..., None]
    else:
        v = d[..., None] * (q - 8.0)
    return v.reshape(n_rows, nb * 32)


def dequant_q4k(blocks: np.ndarray, n_rows: int, n_cols: int) -> np.ndarray:
    """Q4_K rows: super-blocks of 256 values, 144 bytes each.

    Bytes 0-1 f16 d, 2-3 f16 dmin, 4-15 the packed 6-bit scale sc_j and min mn_j of
    the eight 32-value sub-blocks, 16-143 the nibbles. With S the 12 packed bytes:
    sub-block j < 4 takes sc_j = low 6 bits of S[j] and mn_j = low 6 bits of S[j+4];
    j >= 4 takes its low 4 bits from S[j+4] (sc: low nibble, mn: high nibble) and
    its top 2 bits from the top 2 bits of S[j-4] (sc) and S[j] (mn). Nibble bytes
    come in four runs of 32: run c holds values 64c .. 64c+31 in its low nibbles and
    64c+32 .. 64c+63 in its high nibbles. Value = d * sc_j * q - dmin * mn_j.
    """
    nsb = n_cols // 256
    b = np.asarray(blocks, dtype=np.uint8).reshape(n_rows, nsb, 144).astype(np.int64)
    d = half_to_float(b[..., 0] | (b[..., 1] << 8))
    dmin = half_to_float(b[..., 2] | (b[..., 3] << 8))
    S = b[..., 4:16]
    sc = np.zeros((n_rows, nsb, 8))
    mn = np.zeros((n_rows, nsb, 8))
    for j in range(8):
        if j < 4:
            sc[..., j] = S[..., j] & 63
            mn[..., j] = S[..., j + 4] & 63
        else:
            sc[..., j] = (S[..., j + 4] & 15) | ((S[..., j - 4] >> 6) << 4)
            mn[..., j] = (S[..., j + 4] >> 4) | ((S[..., j] >> 6) << 4)
    qs = b[..., 16:144]
    v = np.zeros((n_rows, nsb, 256))
    for c in range(4):
        run = qs[..., 32 * c:32 * c + 32]
        for half, q in ((0, run & 15), (1, run >> 4)):
            j = 2 * c + half
            v[..., 32 * j:32 * j + 32] = (d * sc[..., j])[..., None] * q - (dmin * mn[..., j])[..., None]
    return v.reshape(n_rows, n_cols)


def dequant_q6k(blocks: np.ndarray, n_rows: int, n_cols: int) -> np.ndarray:
    """Q6_K rows: super-blocks of 256 values, 210 bytes each.

    Bytes 0-127 ql (low 4 bits), 128-191 qh (high 2 bits), 192-207 sixteen int8
    scales (one per 16 values), 208-209 f16 d. Each half n (values 128n ..
    128n+127) reads ql[64n ..] and qh[32n ..]: its value 32r + i (r < 4, i < 32)
    takes its low 4 bits from ql[64n + 32 (r % 2) + i] (the low nibble for r < 2,
    the high nibble for r >= 2) and its high 2 bits from bits 2r, 2r+1 of
    qh[32n + i]; q = low + 16 high. Value = d * scale[8n + 2r + i // 16] * (q - 32).
    """
    nsb = n_cols // 256
    b = np.asarray(blocks, dtype=np.uint8).reshape(n_rows, nsb, 210).astype(np.int64)
    ql, qh = b[..., 0:128], b[..., 128:192]
    scale = b[..., 192:208]
    scale = np.where(scale >= 128, scale - 256, scale).astype(np.float64)
    d = half_to_float(b[..., 208] | (b[..., 209] << 8))
    v = np.zeros((n_rows, nsb, 256))
    for n in range(2):
        for r in range(4):
            i = np.arange(32)
            low = (ql[..., 64 * n + 32 * (r % 2) + i] >> (4 * (r // 2))) & 15
            high = (qh[..., 32 * n + i] >> (2 * r)) & 3
            q = low + 16 * high
            s = scale[..., 8 * n + 2 * r + i // 16]
            v[..., 128 * n + 32 * r + i] = d[..., None] * s * (q - 32)
    return v.reshape(n_rows, n_cols)


def row_bytes(n_values: int, qtype: int) -> int:
    return n_values // BLOCK_VALUES[qtype] * BLOCK_BYTES[qtype]


def record_bytes(hidden: int, ff: int, qtype: int, qtype_down: int = 0) -> int:
    return 2 * ff * row_bytes(hidden, qtype) + hidden * row_bytes(ff, qtype_down or qtype)


def expert_matrices(record: np.ndarray, hidden: int, ff: int, qtype: int, qtype_down: int = 0):
    """Split one expert record into dequantised W_gu [2F][H] and W_down [H][F].

    Record = gate rows [F], up rows [F] (rows of H values in ``qtype``), down rows
    [H] (rows of F values in ``qtype_down``, default ``qtype``). The Flint store
    keeps "gate rows then up rows (guQ), down rows (dQ)" (flint_moe_ssd.js
    ``planLayoutFlint``); the Ling store types its down rows separately from its
    gate/up rows (ling_moe_ssd.js ``planLayoutLing``).
    """
    qd = qtype_down or qtype
    gu_bytes = 2 * ff * row_bytes(hidden, qtype)
    rec = np.asarray(record, dtype=np.uint8)
    w_gu = dequant_rows(rec[:gu_bytes], 2 * ff, hidden, qtype)
    w_dn = dequant_rows(rec[gu_bytes:gu_bytes + hidden * row_bytes(ff, qd)], hidden, ff, qd)
    return w_gu, w_dn


# --------------------------------------------------------------------------
# 2-6. Router and selection
# --------------------------------------------------------------------------

def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-np.asarray(z, dtype=np.float64)))


def router_logits(x: np.ndarray, router_w: np.ndarray) -> np.ndarray:
    """logit[t][e] = sum_h W[e][h] x[t][h], in float64 from the f32 inputs."""
    return np.asarray(x, np.float64) @ np.asarray(router_w, np.float64).T


def group_scores(s: np.ndarray, n_groups: int) -> np.ndarray:
    """Per group: the largest plus the second largest s, by a running scan.

    Scan as ``routeLing`` does: a = best so far, b = second; v > a moves a to b,
    else v > b replaces b. Equal values count twice (a multiset top-2).
    """
    per = len(s) // n_groups
    out = np.empty(n_groups)
    for g in range(n_groups):
        a = -math.inf
        b = -math.inf
        for v in s[g * per:(g + 1) * per]:
            if v > a:
                b = a
                a = v
            elif v > b:
                b = v
        out[g] = a + b
    return out


def select_experts(s: np.ndarray, top_k: int, n_groups: int = 1, groups_used: int = 1) -> list:
    """Ordered expert picks for one token from selection scores ``s``.

    Groups (if n_groups > 1): ``groups_used`` rounds, each taking the not yet
    kept group with the largest score (strict >, lowest group on ties). Then
    ``top_k`` rounds of argmax over the experts of kept groups, lowest index on
    ties, each pick masked out.
    """
    s = np.asarray(s, np.float64)
    E = len(s)
    allowed = np.ones(E, dtype=bool)
    if n_groups > 1:
        per = E // n_groups
        gs = group_scores(s, n_groups)
        keep = np.zeros(n_groups, dtype=bool)
        for _ in range(groups_used):
            best, bv = 0, -math.inf
            for g in range(n_groups):
                if not keep[g] and gs[g] > bv:
                    bv, best = gs[g], g
            keep[best] = True
        allowed = np.repeat(keep, per)
    picks = []
    taken = np.zeros(E, dtype=bool)
    for _ in range(top_k):
        best, bv = -1, -math.inf
        for e in range(E):
            if allowed[e] and not taken[e] and (best < 0 or s[e] > bv):
                best, bv = e, s[e]
        picks.append(best)
        taken[best] = True
    return picks


def route_weights(p: np.ndarray, picks: list, scale: float, norm_min: float = NORM_MIN) -> np.ndarray:
    """w_j = p[pick_j] / max(sum_j p[pick_j], norm_min) * scale."""
    pp = np.array([p[e] for e in picks], np.float64)
    wsum = max(float(pp.sum()), norm_min)
    return pp / wsum * scale


def route(x: np.ndarray, router_w: np.ndarray, bias, cfg: MoeConfig):
    """Routing of T tokens: (ids [T][k] int, w [T][k] float64, s [T][E])."""
    logits = router_logits(np.atleast_2d(x), router_w)
    T = logits.shape[0]
    ids = np.zeros((T, cfg.top_k), np.int64)
    w = np.zeros((T, cfg.top_k), np.float64)
    s_all = np.zeros_like(logits)
    for t in range(T):
        p = sigmoid(logits[t])
        s = p + (np.asarray(bias, np.float64) if bias is not None else 0.0)
        picks = select_experts(s, cfg.top_k, cfg.n_groups, cfg.groups_used)
        ids[t] = picks
        w[t] = route_weights(p, picks, cfg.weights_scale, cfg.norm_min)
        s_all[t] = s
    return ids, w, s_all


# --------------------------------------------------------------------------
# 7-9. Experts and combine
# --------------------------------------------------------------------------

def swiglu(x: np.ndarray, w_gu: np.ndarray, w_dn: np.ndarray, limit: float = 0.0) -> np.ndarray:
    """y = W_down (silu(g) * u), with [g; u] = W_gu x and silu(g) = g / (1 + e^-g);
    with limit L > 0, act = min(silu(g), L) * clamp(u, -L, L) (ling_moe_ssd.js
    ``swiglu``)."""
    ff = w_gu.shape[0] // 2
    gu = w_gu @ np.asarray(x, np.float64)
    g, u = gu[:ff], gu[ff:]
    sg = g / (1.0 + np.exp(-g))
    if limit > 0.0:
        u = np.minimum(np.maximum(u, -limit), limit)
        sg = np.minimum(sg, limit)
    act = sg * u
    return w_dn @ act


class ExpertCache:
    """Dequantised expert matrices, built on first use (memoisation only)."""

    def __init__(self, expert_blocks, cfg: MoeConfig):
        self.blocks = np.asarray(expert_blocks, np.uint8)
        self.cfg = cfg
        self.rb = record_bytes(cfg.hidden, cfg.expert_ff, cfg.qtype, cfg.qtype_down)
        self.cache = {}

    def __call__(self, e: int):
        if e not in self.cache:
            rec = self.blocks[e * self.rb:(e + 1) * self.rb]
            self.cache[e] = expert_matrices(rec, self.cfg.hidden, self.cfg.expert_ff, self.cfg.qtype,
                                            self.cfg.qtype_down)
        return self.cache[e]


def rms_norm(x: np.ndarray, weight: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * weight, per row, in float64 (step 0)."""
    x = np.atleast_2d(np.asarray(x, np.float64))
    r = 1.0 / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + eps)
    return x * r * np.asarray(weight, np.float64)[None, :]


def moe_ffn(x, router_w, bias, expert_blocks, shared_blocks, cfg: MoeConfig, out_in=None, ffn_norm=None):
    """The whole step for T tokens. Returns (out [T][H] f64, ids [T][k], w [T][k]).

    out[t] = sum_j w[t][j] * E_{ids[t][j]}(xn[t]) + S(xn[t]) (+ out_in[t] when
    ``cfg.flags & ACCUMULATE``, + x[t] when ``cfg.flags & RESIDUAL``), where xn = x, or
    rms_norm(x) * ffn_norm when a norm vector is given.
    """
    x_in = np.atleast_2d(np.asarray(x, np.float32))
    x = x_in if ffn_norm is None else rms_norm(x_in, ffn_norm, cfg.rms_eps)
    T, H = x.shape
    ids, w, _ = route(x, router_w, bias, cfg)
    experts = ExpertCache(expert_blocks, cfg)
    shared = None
    if cfg.shared_ff:
        shared = expert_matrices(shared_blocks, H, cfg.shared_ff, cfg.qtype, cfg.qtype_down)
    out = np.zeros((T, H), np.float64)
    for t in range(T):
        acc = np.zeros(H, np.float64)
        for j in range(cfg.top_k):
            w_gu, w_dn = experts(int(ids[t, j]))
            acc += w[t, j] * swiglu(x[t], w_gu, w_dn, cfg.swiglu_limit)
        if shared is not None:
            acc += swiglu(x[t], shared[0], shared[1], cfg.swiglu_limit_shared)
        if cfg.flags & ACCUMULATE:
            acc += np.asarray(out_in[t], np.float64)
        if cfg.flags & RESIDUAL:
            acc += x_in[t].astype(np.float64)
        out[t] = acc
    return out, ids, w
