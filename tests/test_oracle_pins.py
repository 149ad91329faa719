"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each ``check_*`` function raises AssertionError when the oracle disagrees with
what the source pages or the mathematics fix; the ``test_*`` functions run them,
and ``test_planted_mistakes_are_caught`` plants plausible mistakes in the oracle
(on the CPU) and requires that some check fails for each.
"""

import itertools
import math
import os

import numpy as np
import pytest

from oracle import moe_oracle as mo

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [p.strip() for p in line.split("|")]


# ---------------------------------------------------------------- f16 decode

def check_half_decode():
    # every finite f16 pattern against numpy's own binary16 conversion
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = mo.half_to_float(bits)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.all(np.isinf(got[np.isinf(ref)]))
    assert np.all(np.isnan(got[np.isnan(ref)]))
    # hand values: 1, -2, smallest subnormal, largest finite, 1/3 rounded
    hand = {0x3C00: 1.0, 0xC000: -2.0, 0x0001: 2.0 ** -24, 0x7BFF: 65504.0,
            0x3555: 0.333251953125, 0x0400: 2.0 ** -14, 0x8000: -0.0}
    for b, v in hand.items():
        assert mo.half_to_float(b) == v, hex(b)


def test_half_decode():
    check_half_decode()


# ---------------------------------------------------------------- blocks

def check_golden_blocks():
    n = 0
    for name, qt, hexbytes, values in _golden_lines("q4_blocks.txt"):
        qt = int(qt)
        raw = np.array([int(h, 16) for h in hexbytes.split()], np.uint8)
        assert len(raw) == mo.BLOCK_BYTES[qt], name
        want = np.array([float(v) for v in values.split()])
        got = mo.dequant_rows(raw, 1, 32, qt)[0]
        assert np.array_equal(got, want), (name, got, want)
        n += 1
    assert n >= 6


def test_golden_blocks():
    check_golden_blocks()


def check_q4_0_is_q4_1_with_offset():
    # Q4_0 (d, q) equals Q4_1 (d, m = -8d, q): -8d is exact in f16 (a power-of-two
    # scaling that stays normal for these d), so the two decodes agree exactly.
    rng = np.random.default_rng(11)
    nb = 64
    d = rng.uniform(0.005, 0.02, nb).astype("<f2")
    qs = rng.integers(0, 256, (nb, 16), dtype=np.uint8)
    b0 = np.concatenate([d.view(np.uint8).reshape(nb, 2), qs], axis=1)
    m = (-8 * d.astype(np.float32)).astype("<f2")
    assert np.array_equal(m.astype(np.float64), -8.0 * d.astype(np.float64))
    b1 = np.concatenate([d.view(np.uint8).reshape(nb, 2), m.view(np.uint8).reshape(nb, 2), qs], axis=1)
    v0 = mo.dequant_rows(b0.reshape(-1), 2, 32 * nb // 2, mo.Q4_0)
    v1 = mo.dequant_rows(b1.reshape(-1), 2, 32 * nb // 2, mo.Q4_1)
    assert np.array_equal(v0, v1)


def test_q4_0_is_q4_1_with_offset():
    check_q4_0_is_q4_1_with_offset()


def check_block_dot_identity():
    # The pages' block dot: dot(block, x) = d * sum(q x) + m * sum(x) (flint_moe_ssd.js,
    # Q41DOT). q is read with plain integer shifts here, independently of the oracle.
    rng = np.random.default_rng(12)
    raw = np.concatenate([np.frombuffer(np.float16(0.0125).tobytes(), np.uint8),
                          np.frombuffer(np.float16(-0.0625).tobytes(), np.uint8),
                          rng.integers(0, 256, 16, dtype=np.uint8)])
    x = rng.standard_normal(32)
    q = [(raw[4 + i] & 15) if i < 16 else (raw[4 + i - 16] >> 4) for i in range(32)]
    d16 = float(np.float16(0.0125))  # 0.0125 rounded to f16; -0.0625 is exact
    want = d16 * sum(qi * xi for qi, xi in zip(q, x)) + (-0.0625) * sum(x)
    got = float(mo.dequant_rows(raw, 1, 32, mo.Q4_1)[0] @ x)
    assert math.isclose(got, want, rel_tol=1e-12, abs_tol=1e-12)


def test_block_dot_identity():
    check_block_dot_identity()


# ---------------------------------------------------------------- K-quant super-blocks

def check_kquant_golden():
    n = 0
    for name, qt, hexbytes, pairs in _golden_lines("kquant_blocks.txt"):
        qt = int(qt)
        raw = np.array([int(h, 16) for h in hexbytes.split()], np.uint8)
        assert len(raw) == mo.BLOCK_BYTES[qt], name
        got = mo.dequant_rows(raw, 1, 256, qt)[0]
        for pair in pairs.split():
            i, v = pair.split("=")
            assert got[int(i)] == float(v), (name, i, got[int(i)], v)
        n += 1
    assert n >= 5


def test_kquant_golden():
    check_kquant_golden()


def _q4_1_block(d, m, vals):
    """A Q4_1 block from f16 d, m and its 32 nibble values, in the pinned Q4_1 byte order."""
    qs = [int(vals[i]) | (int(vals[16 + i]) << 4) for i in range(16)]
    return (list(np.frombuffer(np.float16(d).tobytes(), np.uint8)) +
            list(np.frombuffer(np.float16(m).tobytes(), np.uint8)) + qs)


def check_q4k_is_eight_q4_1():
    # A Q4_K sub-block j is a Q4_1 block with d_j = d * sc_j and m_j = -dmin * mn_j. With d and
    # dmin powers of two both products are exact in f16, so the two decodes agree exactly. The
    # scales are random (every packed bit used) and the nibbles are read here with plain shifts.
    rng = np.random.default_rng(21)
    for _ in range(8):
        d, dmin = 2.0 ** rng.integers(-12, -6), 2.0 ** rng.integers(-12, -6)
        S = rng.integers(0, 256, 12)
        qs = rng.integers(0, 256, 128)
        raw = np.concatenate([np.frombuffer(np.float16(d).tobytes(), np.uint8),
                              np.frombuffer(np.float16(dmin).tobytes(), np.uint8),
                              S.astype(np.uint8), qs.astype(np.uint8)])
        sc = [S[0] & 63, S[1] & 63, S[2] & 63, S[3] & 63,
              (S[8] & 15) | ((S[0] >> 6) << 4), (S[9] & 15) | ((S[1] >> 6) << 4),
              (S[10] & 15) | ((S[2] >> 6) << 4), (S[11] & 15) | ((S[3] >> 6) << 4)]
        mn = [S[4] & 63, S[5] & 63, S[6] & 63, S[7] & 63,
              (S[8] >> 4) | ((S[4] >> 6) << 4), (S[9] >> 4) | ((S[5] >> 6) << 4),
              (S[10] >> 4) | ((S[6] >> 6) << 4), (S[11] >> 4) | ((S[7] >> 6) << 4)]
        blocks = []
        for j in range(8):
            run = qs[32 * (j // 2):32 * (j // 2) + 32]
            vals = (run >> 4) if j % 2 else (run & 15)
            blocks += _q4_1_block(d * sc[j], -dmin * mn[j], vals)
        want = mo.dequant_rows(np.array(blocks, np.uint8), 1, 256, mo.Q4_1)[0]
        got = mo.dequant_rows(raw, 1, 256, mo.Q4_K)[0]
        assert np.array_equal(got, want)


def test_q4k_is_eight_q4_1():
    check_q4k_is_eight_q4_1()


def check_q6k_is_eight_q4_1():
    # With the two scales of each 32-value quarter equal, a Q6_K quarter (n, r) is a Q4_1 block:
    # d_j = d * scale, nibbles from the quarter's ql run, and m_j = (16 * field - 32) * d * scale
    # where every 2-bit field of qh is the same number (a qh byte of four equal fields). Each
    # field value 0..3 is taken in turn; all products are exact in f16 (d a power of two).
    rng = np.random.default_rng(22)
    for field in range(4):
        d = 2.0 ** rng.integers(-10, -5)
        pair = rng.integers(-128, 128, 8)
        scales = np.repeat(pair, 2)
        ql = rng.integers(0, 256, 128)
        qh = np.full(64, field * 0x55)
        raw = np.concatenate([ql.astype(np.uint8), qh.astype(np.uint8), scales.astype(np.int8).view(np.uint8),
                              np.frombuffer(np.float16(d).tobytes(), np.uint8)])
        blocks = []
        for j in range(8):
            n, r = j // 4, j % 4
            run = ql[64 * n + 32 * (r % 2):64 * n + 32 * (r % 2) + 32]
            vals = (run >> 4) if r >= 2 else (run & 15)
            s = float(pair[j])
            blocks += _q4_1_block(d * s, (16 * field - 32) * d * s, vals)
        want = mo.dequant_rows(np.array(blocks, np.uint8), 1, 256, mo.Q4_1)[0]
        got = mo.dequant_rows(raw, 1, 256, mo.Q6_K)[0]
        assert np.array_equal(got, want), field


def test_q6k_is_eight_q4_1():
    check_q6k_is_eight_q4_1()


def check_kquant_record_split():
    # A mixed record (Q4_K gate/up, Q6_K down) splits at 2F rows of H/256 * 144 bytes; the
    # down part decodes as Q6_K rows of F/256 * 210 bytes.
    H, F = 256, 512
    assert mo.record_bytes(H, F, mo.Q4_K, mo.Q6_K) == 2 * F * 144 + H * 2 * 210
    rng = np.random.default_rng(23)
    rec = rng.integers(0, 256, mo.record_bytes(H, F, mo.Q4_K, mo.Q6_K)).astype(np.uint8)
    rec[2 * F * 144:][208::210] = 0x00   # keep every Q6_K d finite: f16 bits 0x3C00 (1.0)
    rec[2 * F * 144:][209::210] = 0x3C
    rec[:2 * F * 144][0::144] = 0x00     # and every Q4_K d, dmin: 1.0
    rec[:2 * F * 144][1::144] = 0x3C
    rec[:2 * F * 144][2::144] = 0x00
    rec[:2 * F * 144][3::144] = 0x3C
    w_gu, w_dn = mo.expert_matrices(rec, H, F, mo.Q4_K, mo.Q6_K)
    assert w_gu.shape == (2 * F, H) and w_dn.shape == (H, F)
    assert np.array_equal(w_gu[F + 3], mo.dequant_rows(rec[(F + 3) * 144:(F + 4) * 144], 1, H, mo.Q4_K)[0])
    dn = rec[2 * F * 144:]
    assert np.array_equal(w_dn[7], mo.dequant_rows(dn[7 * 420:8 * 420], 1, F, mo.Q6_K)[0])


def test_kquant_record_split():
    check_kquant_record_split()


# ---------------------------------------------------------------- routing

def check_golden_routing():
    n = 0
    for name, kgg, svals, picks in _golden_lines("routing_cases.txt"):
        k, g, gu = (int(v) for v in kgg.split())
        s = np.array([float(v) for v in svals.split()])
        want = [int(v) for v in picks.split()]
        got = mo.select_experts(s, k, g, gu)
        assert got == want, (name, got, want)
        n += 1
    assert n >= 6


def test_golden_routing():
    check_golden_routing()


def _brute_force_picks(s, k, n_groups, groups_used):
    """Selection by exhaustive search: the kept groups are the subset of size
    groups_used with the largest summed group score (group score from a full
    sort of the group), then a full sort of the allowed experts by (-s, index)."""
    E = len(s)
    per = E // n_groups
    if n_groups > 1:
        gsc = [sum(sorted(s[g * per:(g + 1) * per], reverse=True)[:2]) for g in range(n_groups)]
        best = max(itertools.combinations(range(n_groups), groups_used),
                   key=lambda c: (sum(gsc[g] for g in c), [-g for g in c]))
        allowed = [e for e in range(E) if e // per in best]
    else:
        allowed = list(range(E))
    return sorted(allowed, key=lambda e: (-s[e], e))[:k]


def check_routing_brute_force():
    rng = np.random.default_rng(13)
    for trial in range(300):
        n_groups = int(rng.choice([1, 2, 4, 8]))
        per = int(rng.integers(2, 9))
        E = n_groups * per
        groups_used = int(rng.integers(1, n_groups + 1))
        k = int(rng.integers(1, groups_used * per + 1))
        s = rng.standard_normal(E)  # continuous: no ties
        got = mo.select_experts(s, k, n_groups, groups_used)
        want = _brute_force_picks(s, k, n_groups, groups_used)
        assert got == want, (trial, got, want)


def test_routing_brute_force():
    check_routing_brute_force()


def check_routing_reductions():
    rng = np.random.default_rng(14)
    for _ in range(50):
        E, k = 32, int(rng.integers(1, 9))
        s = rng.standard_normal(E)
        plain = mo.select_experts(s, k)
        # one group, or every group kept, is plain top-k
        assert mo.select_experts(s, k, 4, 4) == plain
        assert mo.select_experts(s, k, 1, 1) == plain
        # zero bias: the picks follow the logits' order (sigmoid is increasing)
        logits = rng.standard_normal(E) * 3
        p = mo.sigmoid(logits)
        assert mo.select_experts(p, k) == list(np.argsort(-logits, kind="stable")[:k])
        # k = E: a permutation sorted by descending s
        allp = mo.select_experts(s, E)
        assert sorted(allp) == list(range(E))
        assert all(s[allp[i]] >= s[allp[i + 1]] for i in range(E - 1))


def test_routing_reductions():
    check_routing_reductions()


def check_route_weights_closed_form():
    # logits ln 3, 0, -ln 3, ln 9 give sigmoids 3/4, 1/2, 1/4, 9/10 exactly (up to rounding)
    logits = np.array([math.log(3), 0.0, -math.log(3), math.log(9)])
    router_w = np.diag([1.0, 1.0, 1.0, 1.0]).astype(np.float32)
    # x equal to the logits through an identity router; f32 rounding of x is the only error
    x = logits.astype(np.float32)
    cfg = mo.MoeConfig(hidden=4, n_experts=4, top_k=2, expert_ff=32)
    ids, w, _ = mo.route(x, router_w, None, cfg)
    assert list(ids[0]) == [3, 0]
    assert np.allclose(w[0], [0.9 / 1.65, 0.75 / 1.65], rtol=1e-7)  # = 6/11, 5/11
    # the bias changes the picks but never enters the weights; scale multiplies after
    cfg2 = mo.MoeConfig(hidden=4, n_experts=4, top_k=2, expert_ff=32, weights_scale=2.5)
    bias = np.array([0.0, 0.5, 0.0, -0.5], np.float32)
    ids, w, s = mo.route(x, router_w, bias, cfg2)
    assert list(ids[0]) == [1, 0]  # s = 0.75, 1.0, 0.25, 0.4
    assert np.allclose(w[0], [2.5 * 0.5 / 1.25, 2.5 * 0.75 / 1.25], rtol=1e-7)
    # the weights sum to the scale whenever the picked sigmoids sum past 2^-14
    rng = np.random.default_rng(15)
    for _ in range(20):
        E = 16
        rw = rng.standard_normal((E, 8)).astype(np.float32)
        xx = rng.standard_normal(8).astype(np.float32)
        c = mo.MoeConfig(hidden=8, n_experts=E, top_k=4, expert_ff=32, weights_scale=1.75)
        _, ww, _ = mo.route(xx, rw, None, c)
        assert math.isclose(ww.sum(), 1.75, rel_tol=1e-12)
    # clamp: logits of -30 give sigmoids far below 2^-14, so w = p * 2^14 * scale
    x = np.full(4, -30.0, np.float32)
    ids, w, _ = mo.route(x, router_w, None, cfg2)
    pz = 1.0 / (1.0 + math.exp(30.0))
    assert 2 * pz < 2.0 ** -14
    assert np.allclose(w[0], [pz * 2 ** 14 * 2.5] * 2, rtol=1e-12)


def test_route_weights_closed_form():
    check_route_weights_closed_form()


# ---------------------------------------------------------------- SwiGLU and combine

def _q4_1_block(d, m, q):
    """One Q4_1 block from d, m and 32 nibble values (value i -> low nibble of
    byte i for i < 16, high nibble of byte i - 16 otherwise)."""
    q = list(q)
    qs = bytes((q[i] & 15) | ((q[16 + i] & 15) << 4) for i in range(16))
    return (np.float16(d).tobytes() + np.float16(m).tobytes() + qs)


def check_swiglu_closed_form():
    # One expert, H = F = 32. Gate row f picks x_f (q = 1 at column f), up row f
    # picks 2 * x_{f+1}, down row h picks act_h / 2. So y_h = silu(x_h) * x_{h+1}
    # exactly, gate rows first then up rows (flint_moe_ssd.js planLayoutFlint).
    H = F = 32
    one_hot = lambda c, v: [v if i == c else 0 for i in range(32)]
    rec = b"".join(_q4_1_block(1.0, 0.0, one_hot(f, 1)) for f in range(F))
    rec += b"".join(_q4_1_block(1.0, 0.0, one_hot((f + 1) % 32, 2)) for f in range(F))
    rec += b"".join(_q4_1_block(0.5, 0.0, one_hot(h, 1)) for h in range(H))
    rec = np.frombuffer(rec, np.uint8)
    ln3 = math.log(3.0)
    x = np.zeros(H, np.float32)
    x[:4] = [ln3, 2.0, -ln3, 0.5]
    x = x.astype(np.float32)
    x64 = x.astype(np.float64)
    cfg = mo.MoeConfig(hidden=H, n_experts=1, top_k=1, expert_ff=F, weights_scale=1.0)
    out, ids, w = mo.moe_ffn(x, np.zeros((1, H), np.float32), None, rec, None, cfg)
    silu = lambda z: z / (1.0 + math.exp(-z))
    want = np.array([silu(x64[h]) * x64[(h + 1) % 32] for h in range(H)])
    assert list(ids[0]) == [0] and w[0, 0] == 1.0
    assert np.allclose(out[0], want, rtol=1e-12, atol=1e-15)
    # the closed form at the chosen points: silu(ln 3) = 0.75 ln 3, silu(-ln 3) = -0.25 ln 3
    assert math.isclose(out[0][0], 0.75 * ln3 * 2.0, rel_tol=1e-6)
    assert math.isclose(out[0][2], -0.25 * ln3 * 0.5, rel_tol=1e-6)


def test_swiglu_closed_form():
    check_swiglu_closed_form()


def check_swiglu_clamp_closed_form():
    # The same one-hot expert (y_h = act(g = x_h, u = 2 x_{h+1}) / 2) with a clamp limit
    # L = 1 (ling_moe_ssd.js swiglu: act = min(silu(g), L) * clamp(u, -L, L)):
    #   h = 0: g = ln 3 -> silu = 0.75 ln 3 < 1 kept; u = 4 -> 1;        y = 0.375 ln 3
    #   h = 1: g = 2 -> silu(2) = 1.76 -> 1;       u = -2 ln 3 -> -1;   y = -0.5
    #   h = 2: g = -ln 3 -> silu = -0.25 ln 3 kept; u = 1 -> 1 (edge);  y = -0.125 ln 3
    # The shared expert takes its own limit: 0 (no clamp) here, on the same record.
    H = F = 32
    one_hot = lambda c, v: [v if i == c else 0 for i in range(32)]
    rec = b"".join(_q4_1_block(1.0, 0.0, one_hot(f, 1)) for f in range(F))
    rec += b"".join(_q4_1_block(1.0, 0.0, one_hot((f + 1) % 32, 2)) for f in range(F))
    rec += b"".join(_q4_1_block(0.5, 0.0, one_hot(h, 1)) for h in range(H))
    rec = np.frombuffer(rec, np.uint8)
    ln3 = math.log(3.0)
    x = np.zeros(H, np.float32)
    x[:4] = [ln3, 2.0, -ln3, 0.5]
    cfg = mo.MoeConfig(hidden=H, n_experts=1, top_k=1, expert_ff=F, swiglu_limit=1.0)
    out, _, _ = mo.moe_ffn(x, np.zeros((1, H), np.float32), None, rec, None, cfg)
    x64 = x.astype(np.float64)
    assert math.isclose(out[0][0], 0.375 * math.log(3.0), rel_tol=1e-6)
    assert math.isclose(out[0][1], -0.5, rel_tol=1e-12)
    assert math.isclose(out[0][2], -0.125 * math.log(3.0), rel_tol=1e-6)
    # limit 0: exactly the unclamped step; the shared expert ignores the routed limit
    cfg0 = mo.MoeConfig(hidden=H, n_experts=1, top_k=1, expert_ff=F)
    plain, _, _ = mo.moe_ffn(x, np.zeros((1, H), np.float32), None, rec, None, cfg0)
    assert math.isclose(plain[0][1], 0.5 * (2.0 / (1.0 + math.exp(-2.0))) * (2.0 * float(x64[2])), rel_tol=1e-6)
    cfgs = mo.MoeConfig(hidden=H, n_experts=1, top_k=1, expert_ff=F, shared_ff=F, swiglu_limit=1.0,
                        swiglu_limit_shared=0.0)
    both, _, _ = mo.moe_ffn(x, np.zeros((1, H), np.float32), None, rec, rec, cfgs)
    assert np.allclose(both[0] - out[0], plain[0], rtol=1e-12, atol=1e-15)


def test_swiglu_clamp_closed_form():
    check_swiglu_clamp_closed_form()


def check_rms_norm_prologue():
    # rms_norm(x) * w = x / sqrt(mean(x^2) + eps) * w (flint_moe_ssd.js header:
    # x += ffn(rms_norm(x) * ffn_norm)), in closed form on small vectors
    H = 32
    x = np.zeros(H, np.float32)
    x[:2] = [3.0, 4.0]                      # mean(x^2) = 25 / 32
    w = np.full(H, 2.0)
    xn = mo.rms_norm(x, w, 0.0)[0]
    assert math.isclose(xn[0], 3.0 * 2.0 * math.sqrt(32.0) / 5.0, rel_tol=1e-12)
    assert math.isclose(xn[1], 4.0 * 2.0 * math.sqrt(32.0) / 5.0, rel_tol=1e-12)
    assert xn[2] == 0.0
    y = np.zeros(H, np.float32)
    y[0] = 4.0                              # mean(y^2) = 1/2; with eps = 1/2 the scale is 1
    assert math.isclose(mo.rms_norm(y, np.ones(H), 0.5)[0][0], 4.0, rel_tol=1e-12)
    # the step with the prologue is the step on the normalised input; the residual form
    # adds the raw x
    rng = np.random.default_rng(5)
    Hs, E, F = 64, 8, 32
    cfg = mo.MoeConfig(hidden=Hs, n_experts=E, top_k=3, expert_ff=F, rms_eps=1e-5)
    rec = mo.record_bytes(Hs, F, mo.Q4_1)
    blocks = rng.integers(0, 256, E * rec, dtype=np.uint8)
    for e in range(E):  # sane f16 scales in every block (d ~ 0.01, m ~ -0.05)
        b = blocks[e * rec:(e + 1) * rec].reshape(-1, 20)
        b[:, 0:2] = np.frombuffer(np.float16(0.01).tobytes(), np.uint8)
        b[:, 2:4] = np.frombuffer(np.float16(-0.05).tobytes(), np.uint8)
    router = rng.standard_normal((E, Hs)).astype(np.float32) * 0.2
    xt = (rng.standard_normal((2, Hs)) * 3.0).astype(np.float32)
    norm = rng.uniform(0.5, 1.5, Hs)
    a, ia, wa = mo.moe_ffn(xt, router, None, blocks, None, cfg, ffn_norm=norm)
    xn = mo.rms_norm(xt, norm, 1e-5)
    b_, ib, wb = mo.moe_ffn(xn, router, None, blocks, None, cfg)  # xn enters as f32, hence rtol 1e-5
    assert np.array_equal(ia, ib) and np.allclose(a, b_, rtol=1e-5, atol=1e-9)
    cfgr = mo.MoeConfig(**{**cfg.__dict__, "flags": mo.RESIDUAL})
    r, _, _ = mo.moe_ffn(xt, router, None, blocks, None, cfgr, ffn_norm=norm)
    assert np.allclose(r - xt.astype(np.float64), a, rtol=1e-12, atol=1e-12)


def test_rms_norm_prologue():
    check_rms_norm_prologue()


def _random_cfg_layer(seed, shared=True, groups=False):
    from expert_ffn_decode_gb300 import synth
    w = dict(hidden=64, n_experts=8, top_k=3, expert_ff=32, shared_ff=64 if shared else 0,
             n_groups=2 if groups else 1, groups_used=1 if groups else 1, qtype=mo.Q4_1,
             weights_scale=1.5, router_std=0.5, bias_std=0.1, seed=seed)
    layer = synth.make_layer(w)
    cfg = mo.MoeConfig(hidden=64, n_experts=8, top_k=3, expert_ff=32, shared_ff=w["shared_ff"],
                       n_groups=w["n_groups"], groups_used=w["groups_used"], qtype=mo.Q4_1,
                       weights_scale=1.5)
    return layer, cfg


def check_combine_invariants():
    layer, cfg = _random_cfg_layer(21)
    x = np.random.default_rng(22).standard_normal((3, 64)).astype(np.float32)
    rb = mo.record_bytes(64, 32, mo.Q4_1)
    # every expert identical: out = scale * E(x) + S(x), whatever the picks
    same = np.tile(layer["expert_blocks"][:rb], cfg.n_experts)
    out, _, _ = mo.moe_ffn(x, layer["router_w"], layer["bias"], same, layer["shared_blocks"], cfg)
    w_gu, w_dn = mo.expert_matrices(same[:rb], 64, 32, mo.Q4_1)
    s_gu, s_dn = mo.expert_matrices(layer["shared_blocks"], 64, 64, mo.Q4_1)
    for t in range(3):
        want = cfg.weights_scale * mo.swiglu(x[t], w_gu, w_dn) + mo.swiglu(x[t], s_gu, s_dn)
        assert np.allclose(out[t], want, rtol=1e-12, atol=1e-12)
    # the shared expert adds linearly with weight 1
    cfg0 = mo.MoeConfig(**{**cfg.__dict__, "shared_ff": 0})
    o1, _, _ = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"], layer["shared_blocks"], cfg)
    o0, _, _ = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"], None, cfg0)
    for t in range(3):
        assert np.allclose(o1[t] - o0[t], mo.swiglu(x[t], s_gu, s_dn), rtol=1e-10, atol=1e-12)
    # accumulate adds out_in; residual adds x
    base = np.random.default_rng(23).standard_normal((3, 64))
    cfga = mo.MoeConfig(**{**cfg.__dict__, "flags": mo.ACCUMULATE})
    oa, _, _ = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"], layer["shared_blocks"], cfga, out_in=base)
    assert np.allclose(oa - base, o1, rtol=1e-12, atol=1e-12)
    cfgr = mo.MoeConfig(**{**cfg.__dict__, "flags": mo.RESIDUAL})
    orr, _, _ = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"], layer["shared_blocks"], cfgr)
    assert np.allclose(orr - x.astype(np.float64), o1, rtol=1e-12, atol=1e-12)


def test_combine_invariants():
    check_combine_invariants()


def check_expert_matches_textbook_dense():
    # A dense SwiGLU written from the textbook definition with scipy's expit, on
    # matrices dequantised by plain per-element integer reads of the block bytes.
    from scipy.special import expit
    rng = np.random.default_rng(24)
    H, F = 64, 32
    from expert_ffn_decode_gb300 import synth
    rec = synth.q4_blocks(rng, mo.Q4_0, 3 * F * H // 32)

    def deq(raw, rows, cols):
        out = np.zeros((rows, cols))
        nb = cols // 32
        for r in range(rows):
            for b in range(nb):
                blk = raw[(r * nb + b) * 18:(r * nb + b + 1) * 18]
                d = float(np.frombuffer(bytes(blk[0:2]), "<f2")[0])
                for i in range(32):
                    byte = blk[2 + (i % 16)]
                    q = (byte & 15) if i < 16 else (byte >> 4)
                    out[r, b * 32 + i] = d * (int(q) - 8)
        return out

    gu_bytes = 2 * F * (H // 32) * 18
    w_gu = deq(rec[:gu_bytes], 2 * F, H)
    w_dn = deq(rec[gu_bytes:], H, F)
    x = rng.standard_normal(H)
    g, u = w_gu[:F] @ x, w_gu[F:] @ x
    want = w_dn @ (g * expit(g) * u)
    a, b = mo.expert_matrices(rec, H, F, mo.Q4_0)
    assert np.allclose(mo.swiglu(x, a, b), want, rtol=1e-12, atol=1e-12)


def test_expert_matches_textbook_dense():
    check_expert_matches_textbook_dense()


ALL_CHECKS = [check_half_decode, check_golden_blocks, check_q4_0_is_q4_1_with_offset,
              check_block_dot_identity, check_kquant_golden, check_q4k_is_eight_q4_1,
              check_q6k_is_eight_q4_1, check_kquant_record_split, check_golden_routing, check_routing_brute_force,
              check_routing_reductions, check_route_weights_closed_form,
              check_swiglu_closed_form, check_swiglu_clamp_closed_form, check_rms_norm_prologue,
              check_combine_invariants,
              check_expert_matches_textbook_dense]


def _some_check_fails():
    for chk in ALL_CHECKS:
        try:
            chk()
        except AssertionError:
            return True
    return False


# ---------------------------------------------------------------- planted mistakes

def _mut_nibble_order(blocks, n_rows, n_cols, qtype):
    # high nibble read as value i, low as 16 + i
    v = ORIG["dequant_rows"](blocks, n_rows, n_cols, qtype).reshape(n_rows, -1, 32)
    return np.concatenate([v[..., 16:], v[..., :16]], axis=-1).reshape(n_rows, n_cols)


def _mut_drop_m(blocks, n_rows, n_cols, qtype):
    if qtype == mo.Q4_1:
        b = np.array(blocks, np.uint8).reshape(n_rows, n_cols // 32, 20).copy()
        b[..., 2:4] = 0
        return ORIG["dequant_rows"](b.reshape(-1), n_rows, n_cols, qtype)
    return ORIG["dequant_rows"](blocks, n_rows, n_cols, qtype)


def _mut_q4_0_no_offset(blocks, n_rows, n_cols, qtype):
    v = ORIG["dequant_rows"](blocks, n_rows, n_cols, qtype)
    if qtype == mo.Q4_0:
        b = np.array(blocks, np.uint8).reshape(n_rows, n_cols // 32, 18).astype(np.int64)
        d = mo.half_to_float(b[..., 0] | (b[..., 1] << 8))
        v = v + 8.0 * np.repeat(d, 32, axis=-1).reshape(v.shape)
    return v


def _q4k_variant(blocks, n_rows, n_cols, hi_from=-4, min_sign=-1.0, runs_swapped=False):
    # a Q4_K decode with one knob turned away from the layout
    nsb = n_cols // 256
    b = np.asarray(blocks, np.uint8).reshape(n_rows, nsb, 144).astype(np.int64)
    d = mo.half_to_float(b[..., 0] | (b[..., 1] << 8))
    dmin = mo.half_to_float(b[..., 2] | (b[..., 3] << 8))
    S = b[..., 4:16]
    v = np.zeros((n_rows, nsb, 256))
    for j in range(8):
        if j < 4:
            sc, mn = S[..., j] & 63, S[..., j + 4] & 63
        else:
            sc = (S[..., j + 4] & 15) | ((S[..., j + hi_from] >> 6) << 4)
            mn = (S[..., j + 4] >> 4) | ((S[..., j] >> 6) << 4)
        run = b[..., 16 + 32 * (j // 2):16 + 32 * (j // 2) + 32]
        q = (run & 15) if (j % 2 == 0) != runs_swapped else (run >> 4)
        v[..., 32 * j:32 * j + 32] = (d * sc)[..., None] * q + min_sign * (dmin * mn)[..., None]
    return v.reshape(n_rows, n_cols)


def _mut_q4k_high_bits(blocks, n_rows, n_cols):
    return _q4k_variant(blocks, n_rows, n_cols, hi_from=0)


def _mut_q4k_min_added(blocks, n_rows, n_cols):
    return _q4k_variant(blocks, n_rows, n_cols, min_sign=1.0)


def _mut_q4k_runs_swapped(blocks, n_rows, n_cols):
    return _q4k_variant(blocks, n_rows, n_cols, runs_swapped=True)


def _q6k_variant(blocks, n_rows, n_cols, qh_step=2, scale_step=2, unsigned=False, ql_roles=False):
    nsb = n_cols // 256
    b = np.asarray(blocks, np.uint8).reshape(n_rows, nsb, 210).astype(np.int64)
    ql, qh, scale = b[..., 0:128], b[..., 128:192], b[..., 192:208]
    if not unsigned:
        scale = np.where(scale >= 128, scale - 256, scale)
    d = mo.half_to_float(b[..., 208] | (b[..., 209] << 8))
    v = np.zeros((n_rows, nsb, 256))
    i = np.arange(32)
    for n in range(2):
        for r in range(4):
            run, sh = (r // 2, 4 * (r % 2)) if ql_roles else (r % 2, 4 * (r // 2))
            q = ((ql[..., 64 * n + 32 * run + i] >> sh) & 15) + 16 * ((qh[..., 32 * n + i] >> (qh_step * r)) & 3)
            sidx = np.minimum(8 * n + scale_step * r + i // 16, 15)
            v[..., 128 * n + 32 * r + i] = d[..., None] * scale[..., sidx] * (q - 32)
    return v.reshape(n_rows, n_cols)


def _mut_q6k_qh_shift(blocks, n_rows, n_cols):
    return _q6k_variant(blocks, n_rows, n_cols, qh_step=1)


def _mut_q6k_scale_index(blocks, n_rows, n_cols):
    return _q6k_variant(blocks, n_rows, n_cols, scale_step=1)


def _mut_q6k_unsigned_scale(blocks, n_rows, n_cols):
    return _q6k_variant(blocks, n_rows, n_cols, unsigned=True)


def _mut_q6k_ql_roles(blocks, n_rows, n_cols):
    return _q6k_variant(blocks, n_rows, n_cols, ql_roles=True)


def _mut_ties_highest(s, top_k, n_groups=1, groups_used=1):
    # ties broken toward the highest index
    r = ORIG["select_experts"](np.asarray(s)[::-1], top_k, 1, 1) if n_groups == 1 else None
    if r is None:
        return ORIG["select_experts"](s, top_k, n_groups, groups_used)
    return [len(s) - 1 - e for e in r]


def _mut_group_top1(s, n_groups):
    per = len(s) // n_groups
    return np.array([max(s[g * per:(g + 1) * per]) for g in range(n_groups)])


def _mut_weights_bias(p, picks, scale, norm_min=mo.NORM_MIN):
    # normalising s instead of p is caught by the bias closed form; here: no clamp
    pp = np.array([p[e] for e in picks])
    return pp / pp.sum() * scale


def _mut_scale_inside(p, picks, scale, norm_min=mo.NORM_MIN):
    pp = np.array([p[e] for e in picks])
    return pp / max(pp.sum() * scale, norm_min)


def _mut_swiglu_swap(x, w_gu, w_dn, limit=0.0):
    ff = w_gu.shape[0] // 2
    gu = w_gu @ np.asarray(x, np.float64)
    u, g = gu[:ff], gu[ff:]
    return w_dn @ (g / (1.0 + np.exp(-g)) * u)


def _mut_silu_sign(x, w_gu, w_dn, limit=0.0):
    ff = w_gu.shape[0] // 2
    gu = w_gu @ np.asarray(x, np.float64)
    g, u = gu[:ff], gu[ff:]
    return w_dn @ (g / (1.0 + np.exp(g)) * u)


def _mut_clamp_gate_first(x, w_gu, w_dn, limit=0.0):
    # the limit applied to g before the silu instead of to silu(g)
    ff = w_gu.shape[0] // 2
    gu = w_gu @ np.asarray(x, np.float64)
    g, u = gu[:ff], gu[ff:]
    if limit > 0.0:
        g = np.minimum(g, limit)
        u = np.minimum(np.maximum(u, -limit), limit)
    return w_dn @ (g / (1.0 + np.exp(-g)) * u)


def _mut_clamp_up_one_sided(x, w_gu, w_dn, limit=0.0):
    # u clamped from above only
    ff = w_gu.shape[0] // 2
    gu = w_gu @ np.asarray(x, np.float64)
    g, u = gu[:ff], gu[ff:]
    sg = g / (1.0 + np.exp(-g))
    if limit > 0.0:
        u = np.minimum(u, limit)
        sg = np.minimum(sg, limit)
    return w_dn @ (sg * u)


def _mut_rms_eps_outside(x, weight, eps):
    x = np.atleast_2d(np.asarray(x, np.float64))
    return x / (np.sqrt(np.mean(x * x, axis=1, keepdims=True)) + eps) * np.asarray(weight, np.float64)[None, :]


def _mut_rms_sum_not_mean(x, weight, eps):
    x = np.atleast_2d(np.asarray(x, np.float64))
    return x / np.sqrt(np.sum(x * x, axis=1, keepdims=True) + eps) * np.asarray(weight, np.float64)[None, :]


def _mut_half_no_subnormal(bits):
    v = ORIG["half_to_float"](bits)
    h = np.asarray(bits, np.int64)
    return np.where(((h >> 10) & 0x1F) == 0, 0.0, v)


ORIG = {name: getattr(mo, name) for name in
        ["dequant_rows", "select_experts", "group_scores", "route_weights", "swiglu", "half_to_float",
         "rms_norm", "dequant_q4k", "dequant_q6k"]}

MUTANTS = [
    ("dequant_rows", _mut_nibble_order),
    ("dequant_rows", _mut_drop_m),
    ("dequant_rows", _mut_q4_0_no_offset),
    ("select_experts", _mut_ties_highest),
    ("group_scores", _mut_group_top1),
    ("route_weights", _mut_weights_bias),
    ("route_weights", _mut_scale_inside),
    ("swiglu", _mut_swiglu_swap),
    ("swiglu", _mut_silu_sign),
    ("swiglu", _mut_clamp_gate_first),
    ("swiglu", _mut_clamp_up_one_sided),
    ("half_to_float", _mut_half_no_subnormal),
    ("dequant_q4k", _mut_q4k_high_bits),
    ("dequant_q4k", _mut_q4k_min_added),
    ("dequant_q4k", _mut_q4k_runs_swapped),
    ("dequant_q6k", _mut_q6k_qh_shift),
    ("dequant_q6k", _mut_q6k_scale_index),
    ("dequant_q6k", _mut_q6k_unsigned_scale),
    ("dequant_q6k", _mut_q6k_ql_roles),
    ("rms_norm", _mut_rms_eps_outside),
    ("rms_norm", _mut_rms_sum_not_mean),
]


@pytest.mark.parametrize("target,mutant", MUTANTS, ids=[m.__name__ for _, m in MUTANTS])
def test_planted_mistakes_are_caught(monkeypatch, target, mutant):
    monkeypatch.setattr(mo, target, mutant)
    assert _some_check_fails(), f"planted mistake {mutant.__name__} passed every pin"
