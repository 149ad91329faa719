"""CPU check of the batched path's chunk plan against the operand-image sizes.

The expert sort (csrc/prefill.cu, prefill_sort) cuts each expert's sorted (token, pick) pairs
into chunks of at most `nmax` pairs (64 on both batched paths; 128 is checked as well) and
gives every chunk a first padded row: each chunk's rows are rounded up to 16 for the MMA's N
dimension, and the chunks follow each other in expert order. The workspace sizes the tile
pipeline's routed operand images for P + 15 * max_routed padded rows (csrc/prefill.cu,
prefill_ws_layout: P = T * k pairs, max_routed = ceil(P / nmax) + E chunks at most).

These tests restate the plan's arithmetic and check, for random, skewed and single-expert
routings over the batched path's token counts (T = 1 .. 512 per pass), that:
  - every chunk holds 1 .. nmax pairs (a chunk of 0 pairs would make an MMA of N = 0 and a
    bulk copy of 0 bytes, neither of which is allowed);
  - the chunks' padded rows never reach past the images' allocation;
  - the chunk count stays within the chunk table's capacity.
They guard the bounds that a fault of the tile pipeline would most plausibly have broken.
"""

import numpy as np
import pytest


def plan(counts, nmax):
    """(slot, row0, n, prow) for every routed chunk, in expert order, as prefill_sort makes them."""
    chunks = []
    off = 0
    pbase = 0
    for e, cnt in enumerate(counts):
        nck = (cnt + nmax - 1) // nmax
        prows = (nck - 1) * nmax + ((cnt - (nck - 1) * nmax + 15) & ~15) if nck else 0
        for r in range(nck):
            chunks.append((e, off + r * nmax, min(cnt - r * nmax, nmax), pbase + r * nmax))
        off += cnt
        pbase += prows
    return chunks, pbase


def image_rows(T, K, E, nmax):
    P = T * K
    max_routed = (P + nmax - 1) // nmax + E
    return P + 15 * max_routed, max_routed


def routings(T, K, E, rng):
    """Per-expert pair counts of a few routings of T tokens with k distinct picks each."""
    out = []
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)])
    out.append(np.bincount(ids.ravel(), minlength=E))                  # uniform
    p = rng.dirichlet(np.full(E, 0.05)) + 1e-6                           # skewed
    p /= p.sum()
    ids = np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(T)])
    out.append(np.bincount(ids.ravel(), minlength=E))
    c = np.zeros(E, int)                                                 # every token on experts 0..k-1
    c[:K] = T
    out.append(c)
    return out


@pytest.mark.parametrize("E,K", [(256, 6), (16, 4), (4, 2), (512, 8), (1000, 32), (12, 12), (2, 1)])
@pytest.mark.parametrize("nmax", [64, 128])
def test_chunks_fit_the_operand_images(E, K, nmax):
    rng = np.random.default_rng(E * 100 + K + nmax)
    for T in (1, 2, 7, 8, 9, 15, 16, 17, 43, 44, 63, 64, 65, 130, 300, 511, 512):
        for counts in routings(T, K, E, rng):
            assert counts.sum() == T * K
            chunks, rows = plan(counts, nmax)
            cap, max_routed = image_rows(T, K, E, nmax)
            assert len(chunks) <= max_routed
            assert rows <= cap, (T, rows, cap)
            for e, row0, n, prow in chunks:
                assert 1 <= n <= nmax
                assert prow + ((n + 15) & ~15) <= rows
            # the chunks of an expert cover its pairs exactly, in order
            seen = np.zeros(T * K, int)
            for e, row0, n, prow in chunks:
                seen[row0:row0 + n] += 1
            assert np.all(seen == 1)


def test_flint_eight_tokens():
    # the shape of the run whose fault is on record: the Flint layer (256 experts, top-6)
    # with 8 tokens on the tile pipeline: at most 48 chunks of 1 .. 8 pairs, 16 padded rows each
    rng = np.random.default_rng(8)
    ids = np.stack([rng.choice(256, 6, replace=False) for _ in range(8)])
    counts = np.bincount(ids.ravel(), minlength=256)
    chunks, rows = plan(counts, 64)
    cap, _ = image_rows(8, 6, 256, 64)
    assert all(1 <= n <= 8 for _, _, n, _ in chunks)
    assert rows == 16 * len(chunks) <= cap


# ---- K-quant layers on the tile pipeline: every copy's bounds ------------------------------
# Q4_K gate/up rows go through 3-D tensor maps (x = byte of the row, y = row, z = expert) in
# boxes of one 144-byte super-block x 64 rows; Q4_K down rows in boxes of 144 bytes x 128
# rows; Q6_K down rows by one bulk copy of 128 whole rows (prefill_tc.cu, tile_unit and the
# weight producer). A bulk copy and a map's base and strides need 16-byte multiples, and a
# box's x coordinate times the element size too.

def kq_tile_ok(H, F, Fs, qt, qd):
    """prefill.cu, prefill_tile_ok, for the K-quant types."""
    if qt != 12 or qd not in (12, 14):
        return False
    if H % 256 or F % 256 or Fs % 256:
        return False
    return qd == 12 or (F <= 768 and Fs <= 768)


ROW_BYTES = {12: lambda n: n // 256 * 144, 14: lambda n: n // 256 * 210}
STAGE_Q6 = 128 * 630          # a Q6_K raw stage: 128 rows of up to 768 values
SMEM_MAX = 227 * 1024 - 2048  # the tile kernels' dynamic shared memory bound


@pytest.mark.parametrize("H,F,Fs,qd", [(2560, 768, 768, 14), (256, 256, 256, 14), (256, 256, 256, 12),
                                      (512, 768, 512, 14), (256, 3072, 0, 12), (2048, 512, 1024, 12),
                                      (4096, 256, 0, 14), (256, 512, 768, 14)])
def test_kquant_tile_copies_aligned(H, F, Fs, qd):
    assert kq_tile_ok(H, F, Fs, 12, qd)
    rb_h = ROW_BYTES[12](H)
    rb_f, rb_fs = ROW_BYTES[qd](F), ROW_BYTES[qd](Fs)
    rec = 2 * F * rb_h + H * rb_f
    srec = 2 * Fs * rb_h + H * rb_fs
    for v in (rb_h, rec, srec, 2 * F * rb_h, 2 * Fs * rb_h):
        assert v % 16 == 0
    # gate/up boxes: x = 144 kc inside the row, y rows inside the 2F rows of a record
    for kc in range(H // 256):
        assert (144 * kc) % 16 == 0 and 144 * kc + 144 <= rb_h
    assert F % 64 == 0 and (Fs % 64 == 0)
    if qd == 12:
        assert rb_f % 16 == 0 and H % 128 == 0
        for kc in range(F // 256):
            assert 144 * kc + 144 <= rb_f
    else:
        # one bulk copy of 128 whole rows per down tile, from the record's down matrix
        for ff, rb in ((F, rb_f), (Fs, rb_fs)):
            if not ff:
                continue
            assert (128 * rb) % 16 == 0 and 128 * rb <= STAGE_Q6
            for mt in range(H // 128):
                off = 2 * ff * rb_h + 128 * mt * rb
                assert off % 16 == 0
                assert off + 128 * rb <= 2 * ff * rb_h + H * rb
            # the converter's last reads: the d word of the last super-block of row 127, read
            # as two aligned words, stay within 8 bytes past the stage
            last = 127 * rb + 210 * (ff // 256 - 1) + 208
            assert (last & ~3) + 8 <= STAGE_Q6 + 8
    # shared memory: two Q6_K stages (1024-aligned), two 32 KB token stages, alignment slack
    raw = ((2 * STAGE_Q6 + 1023) // 1024) * 1024
    assert raw + 2 * 32768 + 1024 <= SMEM_MAX


@pytest.mark.parametrize("H,F,Fs,qd", [(96, 256, 0, 14), (256, 96, 0, 12), (256, 1024, 0, 14),
                                      (256, 256, 1024, 14), (256, 256, 160, 12)])
def test_kquant_shapes_left_to_the_general_path(H, F, Fs, qd):
    assert not kq_tile_ok(H, F, Fs, 12, qd)
