"""The library's per-channel W12 host packer and unpacker (w12c_pack_host,
w12c_unpack_host) against the oracle (w12c_pack): the same row bases, side
list and row pointers; every non-escaped weight's 12-bit field, read back
from the packed words through the oracle's own layout accessor, equals the
oracle's field (escaped weights hold code 15); unpacking restores every
weight bit for bit.  Host code: no GPU."""
import ctypes

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


def _pack(L, W):
    N, K = W.shape
    W = np.ascontiguousarray(W, dtype=np.uint16)
    base = np.zeros(N, np.uint8)
    words = np.zeros(int(L.w12_words_count(N, K)), np.uint32)
    row_ptr = np.zeros(N + 1, np.uint32)
    n = ctypes.c_int64()
    rc = L.w12c_pack_host(W.ctypes.data, N, K, base.ctypes.data, words.ctypes.data, None, None, 0,
                          row_ptr.ctypes.data, ctypes.byref(n))
    assert rc in (0, 9)
    ne = int(n.value)
    esc_idx = np.zeros(max(ne, 1), np.uint32)
    esc_val = np.zeros(max(ne, 1), np.uint16)
    assert L.w12c_pack_host(W.ctypes.data, N, K, base.ctypes.data, words.ctypes.data, esc_idx.ctypes.data,
                            esc_val.ctypes.data, ne, row_ptr.ctypes.data, ctypes.byref(n)) == 0
    return base, words, esc_idx[:ne], esc_val[:ne], row_ptr


def _unpack(L, N, K, base, words, esc_idx, esc_val):
    out = np.zeros((N, K), np.uint16)
    ei = np.ascontiguousarray(esc_idx if esc_idx.size else np.zeros(1, np.uint32), np.uint32)
    ev = np.ascontiguousarray(esc_val if esc_val.size else np.zeros(1, np.uint16), np.uint16)
    assert L.w12c_unpack_host(words.ctypes.data, base.ctypes.data, N, K, ei.ctypes.data, ev.ctypes.data,
                              esc_idx.size, out.ctypes.data) == 0
    return out


def _row_scaled(seed, N, K, spread):
    u = synthetic.uniform_int(synthetic.key(seed, 2), N, 0, 1 << 20) / float(1 << 20) * 2 * spread - spread
    W = np.empty((N, K), dtype=np.uint16)
    k = synthetic.key(seed, 3)
    for n in range(N):
        synthetic.normal_bf16(k, K, 0.02 * 2.0 ** u[n], offset=n * K, out=W[n])
    return W


def _cases():
    yield "normal", synthetic.normal_bf16(synthetic.key(61, 1), 64 * 256, 0.02).reshape(64, 256)
    yield "row_scaled", _row_scaled(62, 48, 192, 2.0)
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    perm = synthetic.permutation(synthetic.key(63, 1), 65536)
    yield "every_pattern", allbits[perm].reshape(256, 256)
    yield "exponent_major", allbits.reshape(512, 128)


@pytest.mark.parametrize("name,W", list(_cases()), ids=[c[0] for c in _cases()])
def test_host_packer_matches_the_oracle(L, name, W):
    N, K = W.shape
    base, words, esc_idx, esc_val, row_ptr = _pack(L, W)
    ref = oracle.w12c_pack(W)
    np.testing.assert_array_equal(base, ref.base)
    np.testing.assert_array_equal(esc_idx, ref.esc_idx)
    np.testing.assert_array_equal(esc_val, ref.esc_val)
    np.testing.assert_array_equal(row_ptr, np.searchsorted(ref.esc_idx, np.arange(N + 1) * K).astype(np.uint32))
    # the fields, read through the oracle's layout accessor (a W12 object over the library's words)
    view = oracle.W12(N, K, np.zeros(0, np.uint8), words, esc_idx, esc_val, row_ptr)
    esc = np.zeros(N * K, bool)
    esc[ref.esc_idx] = True
    d = synthetic.uniform_int(synthetic.key(64, len(name)), 2000, 0, N * K - 1)
    for flat in [int(x) for x in d] + [0, N * K - 1] + [int(x) for x in ref.esc_idx[:50]]:
        n, k = divmod(flat, K)
        f = oracle.w12_field(view, n, k)
        if esc[flat]:
            assert f == 15 << 7
        else:
            assert f == int(ref.fields[n, k])
    np.testing.assert_array_equal(_unpack(L, N, K, base, words, esc_idx, esc_val), W)


def test_arguments(L):
    W = np.zeros((16, 64), np.uint16)
    n = ctypes.c_int64()
    base = np.zeros(16, np.uint8)
    words = np.zeros(int(L.w12_words_count(16, 64)), np.uint32)
    rp = np.zeros(17, np.uint32)
    assert L.w12c_pack_host(None, 16, 64, base.ctypes.data, words.ctypes.data, None, None, 0, rp.ctypes.data,
                            ctypes.byref(n)) == 1
    assert L.w12c_pack_host(W.ctypes.data, 24, 64, base.ctypes.data, words.ctypes.data, None, None, 0,
                            rp.ctypes.data, ctypes.byref(n)) == 2
    # all zeros: exponent 0 everywhere, base 0, no escapes
    assert L.w12c_pack_host(W.ctypes.data, 16, 64, base.ctypes.data, words.ctypes.data, None, None, 0,
                            rp.ctypes.data, ctypes.byref(n)) == 0
    assert n.value == 0 and (base == 0).all()
    bad = np.array([16 * 64], np.uint32)
    out = np.zeros((16, 64), np.uint16)
    assert L.w12c_unpack_host(words.ctypes.data, base.ctypes.data, 16, 64, bad.ctypes.data,
                              np.zeros(1, np.uint16).ctypes.data, 1, out.ctypes.data) == 11
