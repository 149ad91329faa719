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
    # the shape of the run whose fault round 1 recorded: the Flint layer (256 experts, top-6)
    # with 8 tokens on the tile pipeline: at most 48 chunks of 1 .. 8 pairs, 16 padded rows each
    rng = np.random.default_rng(8)
    ids = np.stack([rng.choice(256, 6, replace=False) for _ in range(8)])
    counts = np.bincount(ids.ravel(), minlength=256)
    chunks, rows = plan(counts, 64)
    cap, _ = image_rows(8, 6, 256, 64)
    assert all(1 <= n <= 8 for _, _, n, _ in chunks)
    assert rows == 16 * len(chunks) <= cap
