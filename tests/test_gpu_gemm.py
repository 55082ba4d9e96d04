"""Fused W12-decode GEMMs (sd_w12_linear: warp-level and tcgen05 kernels;
sd_w12_linear_stream: the weight-streaming kernel, 12-bit weights or the
nested 8-bit view) vs the oracle's fp64 linear.

Tolerance: |gpu - oracle| <= 2e-2 + 1e-2 |oracle| per element (the rule for
bf16 outputs with fp32 accumulation); in addition almost every element must
equal the oracle's correctly rounded bf16 value, since a single GEMM differs
from it only by the fp32 summation order."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import workloads as wl
from helpers import ATOL, RTOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from speculative_decoding_tree_bit_gb300 import model
    return model


def _x(Mrows, K, seed=0):
    return synthetic.normal_bf16(synthetic.key(seed, 77 + Mrows), Mrows * K, 1.0).reshape(Mrows, K)


def _check(M, W, x, rows=None, exact_frac=0.99, p=None, lin=None):
    p = p or M.pack(M.to_device_u16(W))
    y = (lin or M.linear)(p, M.to_device_u16(x)).cpu().numpy().view(np.uint16)
    if rows is not None:
        W, y = W[rows], y[:, rows]
    ref = oracle.linear(x, W)
    got = oracle.bf16_to_f64(y)
    err = np.abs(got - ref)
    assert np.all(err <= ATOL + RTOL * np.abs(ref)), float(err.max())
    same = np.mean(oracle.round_bf16(ref) == y)
    assert same >= exact_frac, same
    return p


@pytest.mark.parametrize("Mrows", [1, 5, 8, 13, 16, 17, 32, 48, 64, 100, 128, 129, 200, 256])
def test_tiny_shape_all_row_counts(M, Mrows):
    t = wl.tiny()
    _check(M, t.W1, _x(Mrows, 1024))


@pytest.mark.parametrize("N,K,Mrows", [(16, 64, 8), (48, 192, 16), (4000, 512, 8), (512, 512, 8), (1024, 4096, 16),
                                       (144, 1088, 3), (4000, 512, 64)])
def test_ragged_shapes(M, N, K, Mrows):
    W = synthetic.normal_bf16(synthetic.key(2, N * 7 + K), N * K, 0.02).reshape(N, K)
    _check(M, W, _x(Mrows, K, 1))


def test_escapes_affine_path(M):
    t = wl.tiny()
    p = _check(M, t.Wlm, _x(8, 1024, 2))
    assert p.meta.affine == 1 and p.n_escapes >= 4194


def test_general_table_path(M):
    rng = np.random.default_rng(5)
    exps = np.array([110, 112, 114, 116, 118, 120, 121, 122, 123, 124, 100, 102, 104, 106, 108, 90], np.uint32)
    e = exps[rng.integers(0, exps.size, size=256 * 512)]
    W = ((rng.integers(0, 2, size=e.size).astype(np.uint32) << 15) | (e << 7)
         | rng.integers(0, 128, size=e.size).astype(np.uint32)).astype(np.uint16).reshape(256, 512)
    p = _check(M, W, _x(16, 512, 3))
    assert p.meta.affine == 0 and p.n_escapes > 0


@pytest.mark.parametrize("name,Mrows", [("wq", 16), ("w_down", 16), ("lm", 16), ("lm", 64)])
def test_full_size_8b(M, name, Mrows):
    sh = wl.SHAPES["8b"]
    w = wl.SyntheticWeights(sh, 0)
    W = w.lm_head() if name == "lm" else w.layer(0, name)
    rows = np.sort(np.random.default_rng(0).choice(W.shape[0], 1024, replace=False))
    _check(M, W, _x(Mrows, W.shape[1], 4), rows=rows)


# ------------------------------------------- strip-parallel kernel (M <= 16) --

@pytest.mark.parametrize("N,K,Mrows", [(4096, 4096, 16), (4096, 12288, 16), (4096, 4096, 1), (4000, 4160, 8),
                                        (2000, 448, 13), (160, 64, 16), (4864, 1024, 9)])
def test_strip_kernel_matches_oracle(M, N, K, Mrows):
    """One CTA per 16-row strip over the whole k range: ragged last strips of
    a block (N = 4000, 2000, 160), k-tile counts not a multiple of the 8
    consumer warps (65, 7, 1), one wave at the limit (4864 rows = 304
    strips); the same rows against the split-K kernel within the tolerance."""
    assert M.set_strip(None)
    W = synthetic.normal_bf16(synthetic.key(6, N * 7 + K), N * K, 0.02).reshape(N, K)
    x = _x(Mrows, K, 8)
    p = _check(M, W, x)
    y_strip = oracle.bf16_to_f64(M.linear(p, M.to_device_u16(x)).cpu().numpy().view(np.uint16))
    M.set_strip(False)
    try:
        y_split = oracle.bf16_to_f64(M.linear(p, M.to_device_u16(x)).cpu().numpy().view(np.uint16))
    finally:
        M.set_strip(True)
    assert np.all(np.abs(y_strip - y_split) <= 2 * (ATOL + RTOL * np.abs(y_split)))


@pytest.mark.parametrize("rare", [0, 400, 5000])
def test_strip_kernel_escapes(M, rare):
    """Escapes by the strip's run of the side list: none, a few per strip,
    and more than 32 per strip (several index chunks)."""
    N, K = 1024, 2048
    W = synthetic.normal_bf16(synthetic.key(7, rare), N * K, 0.02).reshape(N, K)
    if rare:
        synthetic.force_rare_exponents(synthetic.key(7, rare + 1), W, rare)
    p = _check(M, W, _x(16, K, 9))
    if rare > 1000:
        assert p.n_escapes > 32 * (N // 16)


def test_strip_kernel_general_table(M):
    """A non-contiguous exponent table (the table decode; escaped weights
    decode to zero) on the strip kernel."""
    rng = np.random.default_rng(11)
    exps = np.array([110, 112, 114, 116, 118, 120, 121, 122, 123, 124, 100, 102, 104, 106, 108, 90], np.uint32)
    e = exps[rng.integers(0, exps.size, size=512 * 1024)]
    W = ((rng.integers(0, 2, size=e.size).astype(np.uint32) << 15) | (e << 7)
         | rng.integers(0, 128, size=e.size).astype(np.uint32)).astype(np.uint16).reshape(512, 1024)
    p = _check(M, W, _x(16, 1024, 4))
    assert p.meta.affine == 0 and p.n_escapes > 0


@pytest.fixture()
def deferred(M):
    """Split row blocks finished by the separate finish kernel (default: the
    in-kernel finisher), restored afterwards; the strip-parallel kernel off
    (it takes these launches otherwise)."""
    M.set_deferred_finish(True)
    M.set_strip(False)
    yield M
    M.set_deferred_finish(False)
    M.set_strip(True)


@pytest.mark.parametrize("name,Mrows", [("wq", 16), ("wo", 1), ("wo", 8), ("w_down", 16), ("w_down", 4),
                                        ("w_down", 32)])
def test_deferred_finish_8b(deferred, name, Mrows):
    """The deferred finish kernel sums the partials in the in-kernel
    finisher's order and grouping: bit-identical outputs, and within
    tolerance of the oracle on sampled rows."""
    M = deferred
    sh = wl.SHAPES["8b"]
    W = wl.SyntheticWeights(sh, 0).layer(0, name)
    x = _x(Mrows, W.shape[1], 7)
    p = M.pack(M.to_device_u16(W))
    xd = M.to_device_u16(x)
    assert M.set_deferred_finish(None)
    y_def = M.linear(p, xd).cpu()
    M.set_deferred_finish(False)
    try:
        y_in = M.linear(p, xd).cpu()
    finally:
        M.set_deferred_finish(True)
    assert torch.equal(y_def, y_in)
    rows = np.sort(np.random.default_rng(2).choice(W.shape[0], 512, replace=False))
    _check(M, W, x, rows=rows, p=p)


@pytest.mark.parametrize("N,K,Mrows", [(3008, 1024, 8), (4000, 512, 1), (2448, 4096, 16), (3008, 2048, 3),
                                        (4000, 512, 32)])
def test_deferred_finish_ragged(deferred, N, K, Mrows):
    """Ragged last row blocks (strips past N; 9 to 15 CTAs per block, the
    deferred layout)."""
    M = deferred
    W = synthetic.normal_bf16(synthetic.key(4, N * 3 + K), N * K, 0.02).reshape(N, K)
    x = _x(Mrows, K, 5)
    p = _check(M, W, x)
    y_def = M.linear(p, M.to_device_u16(x)).cpu()
    M.set_deferred_finish(False)
    try:
        y_in = M.linear(p, M.to_device_u16(x)).cpu()
    finally:
        M.set_deferred_finish(True)
    assert torch.equal(y_def, y_in)


@pytest.fixture()
def cluster_finish(M):
    """Split row blocks finished through thread-block clusters (default:
    workspace partials and a ticket), restored afterwards; the strip-parallel
    kernel off (it takes these launches otherwise)."""
    M.set_cluster_finish(True)
    M.set_strip(False)
    yield M
    M.set_cluster_finish(False)
    M.set_strip(True)


@pytest.mark.parametrize("name,Mrows", [("wq", 16), ("wo", 1), ("wo", 8), ("w_down", 16), ("w_down", 32)])
def test_cluster_finish_8b(cluster_finish, name, Mrows):
    """The cluster finish sums the same partials in the same order as the
    ticket path: bit-identical outputs, and within tolerance of the oracle on
    sampled rows.  down (224 k-tiles over 9 CTAs per block) wraps the weight
    ring, so a CTA's last stages sit in the slot the partials are staged in."""
    M = cluster_finish
    sh = wl.SHAPES["8b"]
    W = wl.SyntheticWeights(sh, 0).layer(0, name)
    x = _x(Mrows, W.shape[1], 6)
    p = M.pack(M.to_device_u16(W))
    xd = M.to_device_u16(x)
    y_cl = M.linear(p, xd).cpu()
    M.set_cluster_finish(False)
    y_ws = M.linear(p, xd).cpu()
    M.set_cluster_finish(True)
    assert torch.equal(y_cl, y_ws)
    rows = np.sort(np.random.default_rng(1).choice(W.shape[0], 512, replace=False))
    _check(M, W, x, rows=rows, p=p)


@pytest.mark.parametrize("N,K,Mrows", [(4000, 512, 64), (2048, 1024, 8), (1024, 4096, 3)])
def test_cluster_finish_ragged(cluster_finish, N, K, Mrows):
    W = synthetic.normal_bf16(synthetic.key(3, N * 5 + K), N * K, 0.02).reshape(N, K)
    _check(cluster_finish, W, _x(Mrows, K, 2))


def test_repeat_calls_are_deterministic_with_dirty_workspace(M):
    t = wl.tiny()
    p = M.pack(M.to_device_u16(t.W1))
    x = M.to_device_u16(_x(16, 1024, 9))
    ws = M.Workspace(int(M.lib().sd_w12_linear_workspace(1024, 1024, 16)))
    ws.buf.fill_(0x7F)  # garbage in the scratch must not leak into results
    a = M.linear(p, x, ws)
    ws.buf.fill_(0xFF)
    b = M.linear(p, x, ws)
    assert torch.equal(a, b)


# ------------------------------------------- tcgen05 kernel at any row count --

@pytest.fixture()
def tc_all(M):
    """Every launch on the tcgen05 kernel (default: only launches of more
    than 64 rows), restored afterwards."""
    M.set_tc_min_rows(1)
    yield M
    M.set_tc_min_rows(0)


@pytest.mark.parametrize("Mrows", [1, 5, 16, 17, 32, 48, 64, 100, 128])
def test_tc_tiny_shape_row_counts(tc_all, Mrows):
    t = wl.tiny()
    _check(tc_all, t.W1, _x(Mrows, 1024))


@pytest.mark.parametrize("N,K,Mrows", [(16, 64, 8), (48, 192, 16), (4000, 512, 40), (144, 1088, 3), (4000, 512, 64)])
def test_tc_ragged_shapes(tc_all, N, K, Mrows):
    W = synthetic.normal_bf16(synthetic.key(2, N * 7 + K), N * K, 0.02).reshape(N, K)
    _check(tc_all, W, _x(Mrows, K, 1))


def test_tc_escapes_and_general_table(tc_all):
    t = wl.tiny()
    p = _check(tc_all, t.Wlm, _x(24, 1024, 2))
    assert p.meta.affine == 1 and p.n_escapes >= 4194
    rng = np.random.default_rng(5)
    exps = np.array([110, 112, 114, 116, 118, 120, 121, 122, 123, 124, 100, 102, 104, 106, 108, 90], np.uint32)
    e = exps[rng.integers(0, exps.size, size=256 * 512)]
    W = ((rng.integers(0, 2, size=e.size).astype(np.uint32) << 15) | (e << 7)
         | rng.integers(0, 128, size=e.size).astype(np.uint32)).astype(np.uint16).reshape(256, 512)
    p = _check(tc_all, W, _x(40, 512, 3))
    assert p.meta.affine == 0 and p.n_escapes > 0


@pytest.mark.parametrize("name,Mrows", [("w_down", 256), ("lm", 256), ("wq", 64)])
def test_tc_full_size_8b(tc_all, name, Mrows):
    sh = wl.SHAPES["8b"]
    w = wl.SyntheticWeights(sh, 0)
    W = w.lm_head() if name == "lm" else w.layer(0, name)
    rows = np.sort(np.random.default_rng(0).choice(W.shape[0], 1024, replace=False))
    _check(tc_all, W, _x(Mrows, W.shape[1], 4), rows=rows)


def test_tc_repeat_calls_are_deterministic(tc_all):
    t = wl.tiny()
    p = tc_all.pack(tc_all.to_device_u16(t.W1))
    x = tc_all.to_device_u16(_x(200, 1024, 9))
    ws = tc_all.Workspace(int(tc_all.lib().sd_w12_linear_workspace(1024, 1024, 200)))
    ws.buf.fill_(0x7F)
    a = tc_all.linear(p, x, ws)
    ws.buf.fill_(0xFF)
    b = tc_all.linear(p, x, ws)
    assert torch.equal(a, b)


# ------------------------------------ weight-streaming kernel (M <= 64) --

@pytest.mark.parametrize("Mrows", [1, 5, 8, 13, 16, 17, 32, 48, 64])
def test_stream_tiny_shape_row_counts(M, Mrows):
    t = wl.tiny()
    _check(M, t.W1, _x(Mrows, 1024), lin=M.linear_stream)


@pytest.mark.parametrize("N,K,Mrows", [(16, 64, 8), (48, 192, 16), (4000, 512, 8), (512, 512, 8), (1024, 4096, 16),
                                       (144, 1088, 3), (4000, 512, 64)])
def test_stream_ragged_shapes(M, N, K, Mrows):
    W = synthetic.normal_bf16(synthetic.key(2, N * 7 + K), N * K, 0.02).reshape(N, K)
    _check(M, W, _x(Mrows, K, 1), lin=M.linear_stream)


def test_stream_escapes_and_general_table(M):
    t = wl.tiny()
    p = _check(M, t.Wlm, _x(8, 1024, 2), lin=M.linear_stream)
    assert p.meta.affine == 1 and p.n_escapes >= 4194
    rng = np.random.default_rng(5)
    exps = np.array([110, 112, 114, 116, 118, 120, 121, 122, 123, 124, 100, 102, 104, 106, 108, 90], np.uint32)
    e = exps[rng.integers(0, exps.size, size=256 * 512)]
    W = ((rng.integers(0, 2, size=e.size).astype(np.uint32) << 15) | (e << 7)
         | rng.integers(0, 128, size=e.size).astype(np.uint32)).astype(np.uint16).reshape(256, 512)
    p = _check(M, W, _x(16, 512, 3), lin=M.linear_stream)
    assert p.meta.affine == 0 and p.n_escapes > 0


@pytest.mark.parametrize("name,Mrows", [("wq", 16), ("w_down", 16), ("lm", 16), ("lm", 64)])
def test_stream_full_size_8b(M, name, Mrows):
    sh = wl.SHAPES["8b"]
    w = wl.SyntheticWeights(sh, 0)
    W = w.lm_head() if name == "lm" else w.layer(0, name)
    rows = np.sort(np.random.default_rng(0).choice(W.shape[0], 1024, replace=False))
    _check(M, W, _x(Mrows, W.shape[1], 4), rows=rows, lin=M.linear_stream)


@pytest.mark.parametrize("Mrows", [1, 16, 40, 64])
def test_stream_view8_matches_the_oracle_view(M, Mrows):
    """Streaming the nested 8-bit plane multiplies by the 8-bit view of W
    (oracle.w12_view8), escapes included."""
    t = wl.tiny()
    W = t.Wlm
    p = M.pack(M.to_device_u16(W), view8=True)
    x = _x(Mrows, W.shape[1], 6)
    y = M.linear_stream(p, M.to_device_u16(x), p.plane8).cpu().numpy().view(np.uint16)
    ref = oracle.linear(x, oracle.w12_view8(W))
    got = oracle.bf16_to_f64(y)
    assert np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))
    assert np.mean(oracle.round_bf16(ref) == y) >= 0.99


def test_stream_rejects_rows_beyond_64(M):
    t = wl.tiny()
    p = M.pack(M.to_device_u16(t.W1))
    from speculative_decoding_tree_bit_gb300 import SdvError
    with pytest.raises(SdvError):
        M.linear_stream(p, M.to_device_u16(_x(65, 1024)))


@pytest.mark.parametrize("Mrows", [1, 16, 40, 64])
def test_view8_linear_matches_the_oracle_view(M, Mrows):
    """sd_w12_linear_view8: the warp-level kernel in its 8-bit decode mode
    (contiguous table) and the streaming kernel (general table) multiply by
    oracle.w12_view8(W), escapes included."""
    rng = np.random.default_rng(9)
    exps = np.array([110, 112, 114, 116, 118, 120, 121, 122, 123, 124, 100, 102, 104, 106, 108, 90], np.uint32)
    e = exps[rng.integers(0, exps.size, size=256 * 512)]
    Wg = ((rng.integers(0, 2, size=e.size).astype(np.uint32) << 15) | (e << 7)
          | rng.integers(0, 128, size=e.size).astype(np.uint32)).astype(np.uint16).reshape(256, 512)
    for W in (wl.tiny().Wlm, Wg):
        p = M.pack(M.to_device_u16(W), view8=True)
        x = _x(Mrows, W.shape[1], 7)
        y = M.linear_view8(p, M.to_device_u16(x), p.plane8).cpu().numpy().view(np.uint16)
        ref = oracle.linear(x, oracle.w12_view8(W))
        got = oracle.bf16_to_f64(y)
        assert np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))
        assert np.mean(oracle.round_bf16(ref) == y) >= 0.99
