"""sd_w12_linear_static, the allocation-free variant of the fused W12 linear.

It serves callers that cannot allocate device memory themselves (a host
framework that owns all device memory, a real-time thread that must not
synchronise through cudaMalloc, a plug-in that may not grow the device
footprint).  Its output must match sd_w12_linear's within the tolerance the
GEMM tests use, call after call, with the shared static scratch reused.
This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import workloads as wl
from helpers import ATOL, RTOL, assert_close

pytestmark = pytest.mark.gpu


def test_static_linear_matches_workspace_linear_twice():
    from speculative_decoding_tree_bit_gb300 import check, lib, stream_ptr
    from speculative_decoding_tree_bit_gb300 import model as M
    t = wl.tiny()
    for W, Mrows in ((t.W1, 16), (t.Wlm, 64)):
        p = M.pack(M.to_device_u16(W))
        st = p.struct()
        for call in range(2):
            x = synthetic.normal_bf16(synthetic.key(call, 31 + Mrows), Mrows * W.shape[1], 1.0).reshape(Mrows, -1)
            xd = M.to_device_u16(x)
            ref = M.linear(p, xd).cpu().numpy().view(np.uint16)
            y = torch.empty((Mrows, p.N), dtype=torch.int16, device="cuda")
            check(lib().sd_w12_linear_static(ctypes.byref(st), xd.data_ptr(), Mrows, y.data_ptr(), stream_ptr()))
            got = y.cpu().numpy().view(np.uint16)
            a, b = oracle.bf16_to_f64(got), oracle.bf16_to_f64(ref)
            assert np.all(np.abs(a - b) <= ATOL + RTOL * np.abs(b))


@pytest.mark.parametrize("Mrows", [1, 5, 33, 64])
def test_static_linear_matches_the_oracle(Mrows):
    """Element by element against oracle.linear (fp64 sums of the decoded
    weights), for escapes included: rare exponents are forced into W."""
    from speculative_decoding_tree_bit_gb300 import check, lib, stream_ptr
    from speculative_decoding_tree_bit_gb300 import model as M
    N, K = 384, 1536
    W = synthetic.normal_bf16(synthetic.key(61, Mrows), N * K, 0.02).reshape(N, K)
    synthetic.force_rare_exponents(synthetic.key(62, Mrows), W, 30)
    p = M.pack(M.to_device_u16(W))
    assert p.meta.n_escapes > 0
    st = p.struct()
    x = synthetic.normal_bf16(synthetic.key(63, Mrows), Mrows * K, 1.0).reshape(Mrows, K)
    y = torch.empty((Mrows, N), dtype=torch.int16, device="cuda")
    check(lib().sd_w12_linear_static(ctypes.byref(st), M.to_device_u16(x).data_ptr(), Mrows, y.data_ptr(),
                                     stream_ptr()))
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy().view(np.uint16), oracle.linear(x, W))


def test_static_linear_at_the_lm_head_height():
    """N = 151936 output rows (the lm_head's vocabulary; 1187 row blocks,
    far more than CTAs): sampled rows against oracle.linear."""
    from speculative_decoding_tree_bit_gb300 import check, lib, stream_ptr
    from speculative_decoding_tree_bit_gb300 import model as M
    N, K, Mrows = 151936, 1024, 16
    W = synthetic.normal_bf16(synthetic.key(66, 0), N * K, 0.02).reshape(N, K)
    p = M.pack(M.to_device_u16(W))
    st = p.struct()
    x = synthetic.normal_bf16(synthetic.key(67, 0), Mrows * K, 1.0).reshape(Mrows, K)
    y = torch.empty((Mrows, N), dtype=torch.int16, device="cuda")
    check(lib().sd_w12_linear_static(ctypes.byref(st), M.to_device_u16(x).data_ptr(), Mrows, y.data_ptr(),
                                     stream_ptr()))
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(3).choice(N, 1024, replace=False))
    assert_close(y.cpu().numpy().view(np.uint16)[:, rows], oracle.linear(x, W[rows]))


def test_static_linear_ignores_the_tensor_core_threshold():
    """The static scratch is sized for the warp-level kernel, which the call
    runs whatever sd_gemm_set_tc_min_rows says."""
    from speculative_decoding_tree_bit_gb300 import check, lib, stream_ptr
    from speculative_decoding_tree_bit_gb300 import model as M
    N, K, Mrows = 256, 1024, 48
    W = synthetic.normal_bf16(synthetic.key(64, 0), N * K, 0.02).reshape(N, K)
    p = M.pack(M.to_device_u16(W))
    st = p.struct()
    x = synthetic.normal_bf16(synthetic.key(65, 0), Mrows * K, 1.0).reshape(Mrows, K)
    y = torch.empty((Mrows, N), dtype=torch.int16, device="cuda")
    assert M.set_tc_min_rows(16) == 16
    try:
        check(lib().sd_w12_linear_static(ctypes.byref(st), M.to_device_u16(x).data_ptr(), Mrows, y.data_ptr(),
                                         stream_ptr()))
        torch.cuda.synchronize()
    finally:
        M.set_tc_min_rows(0)
    assert_close(y.cpu().numpy().view(np.uint16), oracle.linear(x, W))


def test_static_linear_rejects_sizes_beyond_its_scratch():
    from speculative_decoding_tree_bit_gb300 import lib
    from speculative_decoding_tree_bit_gb300 import model as M
    t = wl.tiny()
    p = M.pack(M.to_device_u16(t.W1))
    st = p.struct()
    x = torch.zeros((65, 1024), dtype=torch.int16, device="cuda")
    y = torch.empty((65, 1024), dtype=torch.int16, device="cuda")
    assert lib().sd_w12_linear_static(ctypes.byref(st), x.data_ptr(), 65, y.data_ptr(), None) == 2
    assert b"M must be <= 64" in lib().sd_last_error()
