"""Pins of the oracle's W12 format (pack / unpack / table / layout).

The lossless property comes from "SpecPilot: AI Agent Framework Boosts
Speculative Decoding 10.87x", section "(1) W12: Lossless 12-bit Weight
Format": the original bf16 weights are restored bit-exactly, out-of-range
exponents through a sparse side list.  The table rule (15 most frequent
exponents) and the byte layout are the spec's and ours.
"""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic import workloads


def _all_patterns():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)


def test_exhaustive_roundtrip_every_bf16_pattern():
    W = _all_patterns()
    p = oracle.w12_pack(W)
    # every exponent occurs 256 times: ties go to the smaller exponent
    assert list(p.table) == list(range(15))
    assert p.n_esc == 65536 - 15 * 256
    back = oracle.w12_unpack(p)
    assert np.array_equal(back, W)  # NaN payloads, +-Inf, +-0, subnormals included


def test_exhaustive_roundtrip_shuffled_rows():
    W = _all_patterns().reshape(-1)
    rng = np.random.default_rng(1)
    W = W[rng.permutation(W.size)].reshape(128, 512)
    p = oracle.w12_pack(W)
    assert np.array_equal(oracle.w12_unpack(p), W)


def _independent_top15(W):
    e = (W.astype(np.uint32) >> 7) & 0xFF
    vals, counts = np.unique(e, return_counts=True)
    order = np.lexsort((vals, -counts))  # count desc, exponent asc
    return np.sort(vals[order][:15]).astype(np.uint8)


@pytest.mark.parametrize("sigma", [0.02, 1.0, 1e-30])
def test_table_matches_independent_histogram(sigma):
    W = synthetic.normal_bf16(synthetic.key(7, 99), 64 * 256, sigma).reshape(64, 256)
    p = oracle.w12_pack(W)
    assert np.array_equal(p.table, _independent_top15(W))
    in_tab = np.isin((W.astype(np.uint32) >> 7) & 0xFF, p.table.astype(np.uint32))
    assert p.n_esc == int((~in_tab).sum())
    assert np.array_equal(oracle.w12_unpack(p), W)


def test_gaussian_table_is_contiguous_109_to_123():
    W = synthetic.normal_bf16(synthetic.key(0, 123), 1 << 20, 0.02).reshape(1024, 1024)
    p = oracle.w12_pack(W)
    assert list(p.table) == list(range(109, 124))
    assert p.n_esc / W.size < 5e-4


def test_fewer_than_15_exponents_and_noncontiguous_table():
    rng = np.random.default_rng(3)
    exps = np.array([90, 100, 101, 140], dtype=np.uint32)
    e = exps[rng.integers(0, 4, size=32 * 128)]
    W = ((rng.integers(0, 2, size=e.size).astype(np.uint32) << 15) | (e << 7)
         | rng.integers(0, 128, size=e.size).astype(np.uint32)).astype(np.uint16).reshape(32, 128)
    p = oracle.w12_pack(W)
    assert list(p.table) == [90, 100, 101, 140]
    assert p.n_esc == 0
    assert np.array_equal(oracle.w12_unpack(p), W)


def test_escape_list_sorted_and_row_ptr():
    wl = workloads.tiny()
    for W, forced in ((wl.W1, wl.forced_w1), (wl.Wlm, wl.forced_lm)):
        p = oracle.w12_pack(W)
        assert p.n_esc >= forced.size  # every forced exponent is off the table
        assert np.all(np.diff(p.esc_idx.astype(np.int64)) > 0)
        assert set(forced.tolist()) <= set(p.esc_idx.tolist())
        N, K = W.shape
        rows = p.esc_idx.astype(np.int64) // K
        counts = np.bincount(rows, minlength=N)
        assert np.array_equal(np.diff(p.row_ptr.astype(np.int64)), counts)
        assert np.array_equal(p.esc_val, W.reshape(-1)[p.esc_idx.astype(np.int64)])
        assert np.array_equal(oracle.w12_unpack(p), W)


# ---- the layout, checked from the tensor-core fragment definition ----------
# PTX ISA, mma.m16n8k16 with .bf16 A operand: lane = 4*g + q holds
#   a0 = A[g][2q..2q+1], a1 = A[g+8][2q..2q+1], a2 = A[g][2q+8..2q+9],
#   a3 = A[g+8][2q+8..2q+9]   (lower column in the lower 16 bits).
# The stored words of (strip, super-tile, sub-tile j, lane) must decode to
# exactly these fragments when the table is contiguous from `base`:
#   a_p = (W_p & 0x87FF87FF) + base*(2^7 + 2^23)        p = 0, 1, 2
#   X   = (W0>>11 & 0x000F000F) | (W1>>7 & 0x00F000F0) | (W2>>3 & 0x0F000F00)
#   a3  = ((X & 0x07FF07FF) + base*(2^7 + 2^23)) | (X<<4 & 0x80008000)

def _decode_fragments(words, N, K, base):
    w = words.reshape(N // 16, K // 64, 3, 32, 4).astype(np.uint64)
    B2 = np.uint64(base * (2 ** 7 + 2 ** 23))
    a = [((w[:, :, p] & 0x87FF87FF) + B2) & 0xFFFFFFFF for p in range(3)]
    X = ((w[:, :, 0] >> 11) & 0x000F000F) | ((w[:, :, 1] >> 7) & 0x00F000F0) | ((w[:, :, 2] >> 3) & 0x0F000F00)
    a.append((((X & 0x07FF07FF) + B2) | ((X << 4) & 0x80008000)) & 0xFFFFFFFF)
    return a  # each [strips][tiles][lane][j]


def test_layout_matches_mma_fragments():
    N, K = 48, 192
    W = synthetic.normal_bf16(synthetic.key(5, 5), N * K, 0.02).reshape(N, K)
    p = oracle.w12_pack(W, table=np.arange(109, 124, dtype=np.uint8))  # a contiguous table, given
    a = _decode_fragments(p.words, N, K, 109)
    esc = np.zeros(N * K, dtype=bool)
    esc[p.esc_idx.astype(np.int64)] = True
    esc = esc.reshape(N, K)
    checked = 0
    for s in range(N // 16):
        for t in range(K // 64):
            for j in range(4):
                A = W[16 * s:16 * s + 16, 64 * t + 16 * j:64 * t + 16 * j + 16]
                E = esc[16 * s:16 * s + 16, 64 * t + 16 * j:64 * t + 16 * j + 16]
                for lane in range(32):
                    g, q = lane // 4, lane % 4
                    want = [(g, 2 * q), (g + 8, 2 * q), (g, 2 * q + 8), (g + 8, 2 * q + 8)]
                    for reg, (r, c) in enumerate(want):
                        v = int(a[reg][s, t, lane, j])
                        for h in range(2):
                            if not E[r, c + h]:
                                assert (v >> (16 * h)) & 0xFFFF == int(A[r, c + h])
                                checked += 1
    assert checked == N * K - int(esc.sum())


def test_escape_slot_field():
    W = _all_patterns()[:16, :64].copy()
    W[3, 5] = 0x7F80  # +Inf, exponent 255: off a table of 0..14
    p = oracle.w12_pack(W)
    assert oracle.w12_field(p, 3, 5) == 15 << 7
