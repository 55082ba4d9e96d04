"""Per-channel W12 on the GPU ("SpecPilot: AI Agent Framework Boosts
Speculative Decoding 10.87x", "(1) W12: Lossless 12-bit Weight Format", read
literally: a 4-bit exponent offset within each output channel).

* The device packer (w12c_pack_analyze / w12c_pack_encode) writes the host
  packer's format bit for bit - bases, words, side list, row pointers -
  which is pinned against the oracle (tests/test_w12_channel_host.py), for
  i.i.d. weights, rows of different norms, rare exponents, every bf16 bit
  pattern, and a row permutation.
* The device unpack restores every weight bit for bit.
* The fused GEMM with a per-row base in the decode (and a per-row slot
  value for the escapes) matches the oracle's fp64 linear over the exact
  weights; a tensor whose bases reach the top of the exponent range packs
  and unpacks but is refused by the GEMM."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import workloads as wl
from helpers import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from speculative_decoding_tree_bit_gb300 import model
    return model


def _host_pack(W):
    from speculative_decoding_tree_bit_gb300 import lib
    L = lib()
    N, K = W.shape
    W = np.ascontiguousarray(W, dtype=np.uint16)
    base = np.zeros(N, np.uint8)
    words = np.zeros(int(L.w12_words_count(N, K)), np.uint32)
    row_ptr = np.zeros(N + 1, np.uint32)
    n = ctypes.c_int64()
    L.w12c_pack_host(W.ctypes.data, N, K, base.ctypes.data, words.ctypes.data, None, None, 0, row_ptr.ctypes.data,
                     ctypes.byref(n))
    ne = int(n.value)
    esc_idx = np.zeros(max(ne, 1), np.uint32)
    esc_val = np.zeros(max(ne, 1), np.uint16)
    assert L.w12c_pack_host(W.ctypes.data, N, K, base.ctypes.data, words.ctypes.data, esc_idx.ctypes.data,
                            esc_val.ctypes.data, ne, row_ptr.ctypes.data, ctypes.byref(n)) == 0
    return base, words, esc_idx[:ne], esc_val[:ne], row_ptr


def _cases():
    yield "normal", synthetic.normal_bf16(synthetic.key(71, 1), 128 * 512, 0.02).reshape(128, 512)
    yield "row_scaled", wl.row_scaled(72, 256, 1024, 2.0)
    r = synthetic.normal_bf16(synthetic.key(73, 1), 64 * 256, 0.02).reshape(64, 256)
    synthetic.force_rare_exponents(synthetic.key(73, 2), r, 300)
    yield "rare", r
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    yield "every_pattern", allbits[synthetic.permutation(synthetic.key(74, 1), 65536)].reshape(256, 256)


def _np(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("name,W", list(_cases()), ids=[c[0] for c in _cases()])
@pytest.mark.parametrize("perm", [False, True])
def test_device_packer_equals_host_packer(M, name, W, perm):
    N = W.shape[0]
    row_src = np.random.default_rng(N).permutation(N).astype(np.int32) if perm else None
    p = M.pack_channel(M.to_device_u16(W), row_src)
    Wp = W[row_src] if perm else W
    base, words, esc_idx, esc_val, row_ptr = _host_pack(Wp)
    ne = p.n_escapes
    assert ne == esc_idx.size
    np.testing.assert_array_equal(_np(p.row_base), base)
    np.testing.assert_array_equal(_np(p.row_ptr).view(np.uint32), row_ptr)
    np.testing.assert_array_equal(_np(p.words).view(np.uint32), words)
    if ne:
        np.testing.assert_array_equal(_np(p.esc_idx).view(np.uint32)[:ne], esc_idx)
        np.testing.assert_array_equal(_np(p.esc_val).view(np.uint16)[:ne], esc_val)
    np.testing.assert_array_equal(base, oracle.w12c_bases(Wp))
    # the device unpack restores every weight
    np.testing.assert_array_equal(_np(M.unpack(p)).view(np.uint16), Wp)
    assert p.meta.affine == (1 if int(base.max()) <= 239 else 0)


@pytest.mark.parametrize("Mrows", [1, 5, 16, 40, 64])
def test_per_channel_gemm_matches_the_oracle(M, Mrows):
    W = wl.row_scaled(75, 512, 2048, 2.0)
    synthetic.force_rare_exponents(synthetic.key(75, 9), W, 400)
    p = M.pack_channel(M.to_device_u16(W))
    assert p.meta.affine == 1 and p.n_escapes > 0
    x = synthetic.normal_bf16(synthetic.key(76, Mrows), Mrows * 2048, 1.0).reshape(Mrows, 2048)
    y = M.linear(p, M.to_device_u16(x)).cpu().numpy().view(np.uint16)
    ref = oracle.linear(x, W)
    assert_close(y, ref)
    assert np.mean(oracle.round_bf16(ref) == y) >= 0.99


def test_per_channel_gemm_refuses_what_it_cannot_decode(M):
    from speculative_decoding_tree_bit_gb300 import SdvError
    W = wl.row_scaled(77, 128, 512, 2.0)
    p = M.pack_channel(M.to_device_u16(W))
    x = M.to_device_u16(synthetic.normal_bf16(synthetic.key(78, 0), 65 * 512, 1.0).reshape(65, 512))
    with pytest.raises(SdvError):
        M.linear(p, x)  # more than 64 rows: the tcgen05 kernel has no per-row decode
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    q = M.pack_channel(M.to_device_u16(allbits.reshape(512, 128)))
    assert q.meta.affine == 0  # rows of NaN and infinity patterns: bases up to 241
    with pytest.raises(SdvError):
        M.linear(q, M.to_device_u16(np.zeros((16, 128), np.uint16)))
