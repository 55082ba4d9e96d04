"""Pins of the oracle's per-output-channel W12 ("SpecPilot: AI Agent Framework
Boosts Speculative Decoding 10.87x", "(1) W12: Lossless 12-bit Weight
Format", read literally: sign, a 4-bit exponent offset from a per-channel
base, 7-bit mantissa, out-of-range weights restored exactly from a sparse
list).  Pinned by a hand-worked row, bit-exact restoration of every bf16
pattern, a brute-force search of the base, and the comparison with the
per-tensor exponent table on two weight recipes."""
import numpy as np

import oracle
import synthetic


def test_hand_worked_row():
    # 1.0 (exponent 127), -0.5 (126), 2^-7 (120) and +0: the bases holding
    # the three non-zero exponents are 113 .. 120, the smallest is taken;
    # codes 14, 13, 7; the zero (exponent 0) escapes
    W = np.array([[0x3F80, 0xBF00, 0x3C00, 0x0000]], dtype=np.uint16)
    p = oracle.w12c_pack(W)
    assert list(p.base) == [113]
    assert [int(f) for f in p.fields[0]] == [14 << 7, (1 << 11) | (13 << 7), 7 << 7, 15 << 7]
    assert list(p.esc_idx) == [3] and list(p.esc_val) == [0]
    np.testing.assert_array_equal(oracle.w12c_unpack(p), W)


def test_every_bf16_pattern_round_trips():
    W = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)  # row n: exponent-major slice
    p = oracle.w12c_pack(W)
    np.testing.assert_array_equal(oracle.w12c_unpack(p), W)
    # the same patterns shuffled across rows (every row sees many exponents)
    perm = synthetic.permutation(synthetic.key(2, 5), 65536)
    W2 = W.ravel()[perm].reshape(256, 256)
    np.testing.assert_array_equal(oracle.w12c_unpack(oracle.w12c_pack(W2)), W2)


def test_base_maximises_the_window_brute_force():
    d = synthetic.uniform_int(synthetic.key(4, 6), 200 * 24, 0, 1 << 30)
    for n in range(200):
        K = 1 + int(d[n * 24]) % 20
        lo = int(d[n * 24 + 1]) % 230
        span = 1 + int(d[n * 24 + 2]) % 26
        e = np.array([lo + int(x) % span for x in d[n * 24 + 3:n * 24 + 3 + K]], dtype=np.uint16)
        w = (e << 7) | np.uint16(n & 0x7F)
        best, best_b = -1, None
        for b in range(242):
            c = sum(1 for x in e if b <= int(x) <= b + 14)
            if c > best:
                best, best_b = c, b
        p = oracle.w12c_pack(w[None, :])
        assert int(p.base[0]) == best_b
        assert p.n_esc == K - best
        np.testing.assert_array_equal(oracle.w12c_unpack(p), w[None, :])


def _row_scaled(seed, N, K, spread):
    # row n ~ N(0, (0.02 * 2^u_n)^2), u_n uniform in [-spread, spread]: channels of different norms
    u = synthetic.uniform_int(synthetic.key(seed, 2), N, 0, 1 << 20) / float(1 << 20) * 2 * spread - spread
    W = np.empty((N, K), dtype=np.uint16)
    k = synthetic.key(seed, 3)
    for n in range(N):
        synthetic.normal_bf16(k, K, 0.02 * 2.0 ** u[n], offset=n * K, out=W[n])
    return W


def test_comparison_with_the_per_tensor_table():
    N, K = 512, 4096
    # i.i.d. N(0, 0.02): one shared exponent range; both readings coincide
    W = synthetic.normal_bf16(synthetic.key(21, 1), N * K, 0.02).reshape(N, K)
    pt, pc = oracle.w12_pack(W), oracle.w12c_pack(W)
    assert list(pt.table) == list(range(109, 124))
    assert (pc.base == 109).all() and pc.n_esc == pt.n_esc
    assert 1e-4 < pc.n_esc / W.size < 2.5e-4
    # channels whose scales spread over 2^-2 .. 2^2: each row's window
    # follows its own range, the tensor's table cannot
    Wr = _row_scaled(21, N, K, 2.0)
    pt, pc = oracle.w12_pack(Wr), oracle.w12c_pack(Wr)
    np.testing.assert_array_equal(oracle.w12c_unpack(pc), Wr)
    np.testing.assert_array_equal(oracle.w12_unpack(pt), Wr)
    assert pc.n_esc * 3 < pt.n_esc
    assert pc.n_esc / Wr.size < 2.5e-4
