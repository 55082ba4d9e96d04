"""The bounded waits' give-up path on the GPU, made to happen on purpose.

Every wait of the library's kernels (on an mbarrier or a device flag) gives
up after a time limit, records SD_ERR_TIMEOUT in a status word and lets the
kernel return, so that a stuck pipeline never hangs the GPU.  Here a small
kernel waits, with the same helpers and a limit of a few milliseconds, on
something nothing completes; the test checks that the status comes back,
that the kernel ended after (not before) the limit, and that the context
is still usable for a real verify-step GEMM afterwards."""
import time

import numpy as np
import pytest
import torch

import oracle
import synthetic
from helpers import assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("which", [0, 1])
def test_a_wait_that_nothing_completes_gives_up_with_a_timeout_status(which):
    from speculative_decoding_tree_bit_gb300 import check, lib, stream_ptr
    limit_ns = 20_000_000
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    check(lib().sd_debug_bounded_wait(st.data_ptr(), limit_ns, which, stream_ptr()))
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st[0]) == 6  # SD_ERR_TIMEOUT
    assert dt >= limit_ns * 1e-9 * 0.9 and dt < 1.5


def test_the_context_stays_usable_after_a_timeout():
    from speculative_decoding_tree_bit_gb300 import check, lib, stream_ptr
    from speculative_decoding_tree_bit_gb300 import model as M
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    check(lib().sd_debug_bounded_wait(st.data_ptr(), 5_000_000, 0, stream_ptr()))
    torch.cuda.synchronize()
    assert int(st[0]) == 6
    N, K, Mr = 256, 512, 16
    W = synthetic.normal_bf16(synthetic.key(71, 0), N * K, 0.02).reshape(N, K)
    x = synthetic.normal_bf16(synthetic.key(72, 0), Mr * K, 1.0).reshape(Mr, K)
    y = M.linear(M.pack(M.to_device_u16(W)), M.to_device_u16(x))
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy().view(np.uint16), oracle.linear(x, W))


def test_bad_arguments_are_refused_on_the_host():
    from speculative_decoding_tree_bit_gb300 import lib
    assert lib().sd_debug_bounded_wait(None, 1000, 0, None) == 1
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib().sd_debug_bounded_wait(st.data_ptr(), 1000, 2, None) == 1
