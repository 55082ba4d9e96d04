"""GPU W12 packer/unpacker vs the oracle: bit-exact words, escapes, row
pointers and round trip ("(1) W12: Lossless 12-bit Weight Format")."""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from speculative_decoding_tree_bit_gb300 import model
    return model


def _cmp(M, W, row_src=None):
    p = M.pack(M.to_device_u16(W), row_src)
    Wsrc = W if row_src is None else W[row_src]
    o = oracle.w12_pack(Wsrc)
    assert list(p.table) == list(o.table)
    assert p.n_escapes == o.n_esc
    assert np.array_equal(p.words.cpu().numpy().view(np.uint32), o.words)
    if o.n_esc:
        assert np.array_equal(p.esc_idx[: o.n_esc].cpu().numpy().view(np.uint32), o.esc_idx)
        assert np.array_equal(p.esc_val[: o.n_esc].cpu().numpy().view(np.uint16), o.esc_val)
    assert np.array_equal(p.row_ptr.cpu().numpy().view(np.uint32), o.row_ptr)
    assert np.array_equal(M.unpack(p).cpu().numpy().view(np.uint16), Wsrc)
    _cmp_tile_index(p, o)
    return p


def _cmp_tile_index(p, o):
    """The escape tile index regroups the oracle's side list by (128-row
    block, 64-column tile), row-major inside a group: bit-exact."""
    N, K = p.N, p.K
    NB, KT = (N + 127) // 128, K // 64
    idx = o.esc_idx.astype(np.int64)
    n, k = idx // K, idx % K
    key = (n // 128) * KT + k // 64
    order = np.argsort(key, kind="stable")  # side list is row-major: stable keeps it inside a group
    want_ptr = np.zeros(NB * KT + 1, np.int64)
    np.add.at(want_ptr, key + 1, 1)
    want_ptr = np.cumsum(want_ptr)
    want_esc = ((o.esc_val.astype(np.uint32) << 16) | ((n % 128).astype(np.uint32) << 6)
                | (k % 64).astype(np.uint32))[order]
    assert np.array_equal(p.tile_ptr.cpu().numpy().view(np.uint32).astype(np.int64), want_ptr)
    if o.n_esc:
        assert np.array_equal(p.tile_esc[: o.n_esc].cpu().numpy().view(np.uint32), want_esc)


def test_every_bf16_pattern(M):
    W = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)
    p = _cmp(M, W)
    assert p.meta.affine == 1 and list(p.table) == list(range(15))


def test_tiny_tensors_with_forced_escapes(M):
    t = wl.tiny()
    for W in (t.W1, t.Wlm):
        assert _cmp(M, W).n_escapes >= 1049


def test_noncontiguous_table_and_ragged(M):
    rng = np.random.default_rng(3)
    exps = np.array([60, 90, 100, 101, 140, 141, 142, 150, 200, 201, 202, 203, 204, 205, 206, 207, 3], np.uint32)
    e = exps[rng.integers(0, exps.size, size=48 * 192)]
    W = ((rng.integers(0, 2, size=e.size).astype(np.uint32) << 15) | (e << 7)
         | rng.integers(0, 128, size=e.size).astype(np.uint32)).astype(np.uint16).reshape(48, 192)
    assert _cmp(M, W).meta.affine == 0


def test_row_permutation(M):
    W = synthetic.normal_bf16(synthetic.key(1, 2), 64 * 128, 0.02).reshape(64, 128)
    _cmp(M, W, np.random.default_rng(0).permutation(64).astype(np.int32))


def test_full_size_gate_up_of_8b(M):
    sh = wl.SHAPES["8b"]
    w = wl.SyntheticWeights(sh, 0)
    W = np.concatenate([w.layer(0, "w_gate"), w.layer(0, "w_up")])
    p = _cmp(M, W, M.row_map(1, sh.Hq, sh.Hkv, sh.I, W.shape[0]))
    assert p.meta.affine == 1 and list(p.table) == list(range(109, 124))
