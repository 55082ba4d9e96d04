"""The nested 8-bit plane of W12 (w12_plane8_pack_host / _unpack_host):
unpacking gives exactly the oracle's 8-bit view of every weight (escaped
weights from the side list, through the same view), and every non-escaped
weight's byte is the high byte of its 12-bit field as the oracle packs it
(read through the oracle's layout accessor).  Host code: no GPU."""
import numpy as np
import pytest

import oracle
import synthetic
import speculative_decoding_tree_bit_gb300 as sdv
from speculative_decoding_tree_bit_gb300 import _build


@pytest.fixture(scope="module")
def L():
    _build.build()
    return sdv.lib()


def _lane_byte(plane, N, K, n, k):
    # the byte of weight (n, k) in the plane layout
    s, r, t, c = n // 16, n % 16, k // 64, k % 64
    j, cc = c // 16, c % 16
    g, hi_row = r % 8, r // 8
    p, q, odd = cc // 8, (cc % 8) // 2, cc % 2
    word = (s * (K // 64) + t) * 256 + p * 128 + (4 * g + q) * 4 + j
    return (int(plane[word]) >> (8 * (2 * hi_row + odd))) & 0xFF


@pytest.mark.parametrize("rare", [0, 25])
def test_plane_is_the_nested_view(L, rare):
    N, K = 48, 192
    W = synthetic.normal_bf16(synthetic.key(71, rare), N * K, 0.02).reshape(N, K)
    if rare:
        synthetic.force_rare_exponents(synthetic.key(72, 1), W, rare)
    p12 = oracle.w12_pack(W)
    table = np.zeros(16, np.uint8)
    table[:p12.n_table] = p12.table
    plane = np.zeros(N * K // 4, np.uint32)
    assert L.w12_plane8_pack_host(W.ctypes.data, N, K, table.ctypes.data, p12.n_table, plane.ctypes.data) == 0
    out = np.zeros((N, K), np.uint16)
    ei = np.ascontiguousarray(p12.esc_idx if p12.n_esc else np.zeros(1, np.uint32), np.uint32)
    ev = np.ascontiguousarray(p12.esc_val if p12.n_esc else np.zeros(1, np.uint16), np.uint16)
    assert L.w12_plane8_unpack_host(plane.ctypes.data, N, K, table.ctypes.data, p12.n_table, ei.ctypes.data,
                                    ev.ctypes.data, p12.n_esc, out.ctypes.data) == 0
    np.testing.assert_array_equal(out, oracle.w12_view8(W))
    esc = set(int(i) for i in p12.esc_idx)
    for n in range(N):
        for k in range(K):
            b = _lane_byte(plane, N, K, n, k)
            if n * K + k in esc:
                assert b == 15 << 3
            else:
                assert b == oracle.w12_field(p12, n, k) >> 4
    assert rare == 0 or len(esc) >= rare


def test_arguments(L):
    W = np.zeros((16, 64), np.uint16)
    t = np.zeros(16, np.uint8)
    plane = np.zeros(256, np.uint32)
    assert L.w12_plane8_pack_host(None, 16, 64, t.ctypes.data, 1, plane.ctypes.data) == 1
    assert L.w12_plane8_pack_host(W.ctypes.data, 16, 48, t.ctypes.data, 1, plane.ctypes.data) == 2
    assert L.w12_plane8_pack_host(W.ctypes.data, 16, 64, t.ctypes.data, 16, plane.ctypes.data) == 1
    out = np.zeros((16, 64), np.uint16)
    bad = np.array([16 * 64], np.uint32)
    assert L.w12_plane8_unpack_host(plane.ctypes.data, 16, 64, t.ctypes.data, 1, bad.ctypes.data,
                                    np.zeros(1, np.uint16).ctypes.data, 1, out.ctypes.data) == 11
