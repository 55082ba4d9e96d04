"""Pins of the oracle's arithmetic pieces against closed forms, library
routines and special cases (bf16 rounding, linear, RMSNorm, RoPE, SiLU,
tree attention, the linear recurrence)."""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic


def _bits(x):
    return oracle.round_bf16(np.asarray(x, dtype=np.float64))


# ------------------------------------------------------------------ bf16 --

def test_round_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    f = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-40, 38, 100000),
                        np.array([0.0, -0.0, 1e-45, -1e-45, 3.4e38, -3.4e38], dtype=np.float32)])
    f = f[np.isfinite(f)].astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16(f.astype(np.float64))
    assert np.array_equal(got, ref)


def test_round_bf16_is_a_single_rounding_from_double():
    # 1 + 2^-8 + 2^-30 lies just above the midpoint of 1 and 1+2^-7; going
    # through float32 would land on the midpoint and round to even (1.0)
    assert oracle.round_bf16(np.array([1 + 2 ** -8 + 2 ** -30]))[0] == 0x3F81
    assert oracle.round_bf16(np.array([1 + 2 ** -8]))[0] == 0x3F80          # tie -> even
    assert oracle.round_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 0x3F82      # tie -> even (up)
    assert oracle.round_bf16(np.array([2.0 ** -133]))[0] == 0x0001          # smallest subnormal
    assert oracle.round_bf16(np.array([2.0 ** -134]))[0] == 0x0000          # tie -> even (zero)
    assert oracle.round_bf16(np.array([3 * 2.0 ** -135]))[0] == 0x0001
    assert oracle.round_bf16(np.array([2.0 ** 128]))[0] == 0x7F80
    assert oracle.round_bf16(np.array([-(2.0 ** 127) * (2 - 2 ** -8)]))[0] == 0xFF80  # rounds up to -inf
    assert oracle.round_bf16(np.array([np.nan]))[0] & 0x7FC0 == 0x7FC0


def test_bf16_to_f64_exact():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = oracle.bf16_to_f64(b)
    ref = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(v[fin], ref[fin])
    assert np.array_equal(np.isnan(v), np.isnan(ref))


# ---------------------------------------------------------------- linear --

def test_linear_matches_numpy_matmul():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 320))
    W = synthetic.normal_bf16(synthetic.key(1, 1), 96 * 320, 0.02).reshape(96, 320)
    y = oracle.linear(x, W)
    ref = x @ oracle.bf16_to_f64(W).T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)


def test_linear_exact_on_integers():
    rng = np.random.default_rng(2)
    x = rng.integers(-8, 9, size=(5, 128)).astype(np.float64)
    Wf = rng.integers(-8, 9, size=(32, 128)).astype(np.float64)
    y = oracle.linear(x, _bits(Wf))
    assert np.array_equal(y, x @ Wf.T)


# ------------------------------------------------------------ rms / silu --

def test_rmsnorm_closed_forms():
    H = 256
    x = _bits(np.full((1, H), 3.0))
    g = _bits(np.ones(H))
    y = oracle.bf16_to_f64(oracle.rmsnorm(x, g, 0.0))
    assert np.all(y == 1.0)
    rng = np.random.default_rng(3)
    xr = _bits(rng.standard_normal((4, H)))
    gr = _bits(1 + 0.1 * rng.standard_normal(H))
    a = oracle.rmsnorm(xr, gr, 0.0)
    b = oracle.rmsnorm(_bits(oracle.bf16_to_f64(xr) * 8.0), gr, 0.0)  # power-of-two scale is exact
    assert np.array_equal(a, b)
    xv = oracle.bf16_to_f64(xr)
    want = xv / np.sqrt((xv ** 2).mean(1, keepdims=True) + 1e-6) * oracle.bf16_to_f64(gr)
    assert np.array_equal(oracle.rmsnorm(xr, gr, 1e-6), _bits(want))


def test_silu_mul_matches_torch():
    rng = np.random.default_rng(4)
    g = _bits(rng.standard_normal(1000) * 3)
    u = _bits(rng.standard_normal(1000))
    ref = torch.nn.functional.silu(torch.from_numpy(oracle.bf16_to_f64(g))) * torch.from_numpy(oracle.bf16_to_f64(u))
    assert np.array_equal(oracle.silu_mul(g, u), _bits(ref.numpy()))
    assert oracle.silu_mul(_bits([0.0]), _bits([5.0]))[0] == 0


# ------------------------------------------------------------------ rope --

def test_rope_position_zero_is_identity():
    rng = np.random.default_rng(5)
    x = _bits(rng.standard_normal((3, 2, 128)))
    assert np.array_equal(oracle.rope(x, np.zeros(3), 1e6), x)


def test_rope_first_pair_by_hand():
    x = np.zeros((1, 1, 128))
    x[0, 0, 0], x[0, 0, 64] = 1.0, 0.5
    pos = 7
    y = oracle.bf16_to_f64(oracle.rope(_bits(x), np.array([pos]), 1e6))
    assert y[0, 0, 0] == oracle.bf16_to_f64(_bits([math.cos(7) - 0.5 * math.sin(7)]))[0]
    assert y[0, 0, 64] == oracle.bf16_to_f64(_bits([0.5 * math.cos(7) + math.sin(7)]))[0]
    # last pair rotates by pos * base^(-126/128)
    x2 = np.zeros((1, 1, 128))
    x2[0, 0, 63] = 1.0
    y2 = oracle.bf16_to_f64(oracle.rope(_bits(x2), np.array([1000]), 1e6))
    th = 1000 * 1e6 ** (-126 / 128)
    assert y2[0, 0, 63] == oracle.bf16_to_f64(_bits([math.cos(th)]))[0]
    assert y2[0, 0, 127] == oracle.bf16_to_f64(_bits([math.sin(th)]))[0]


def test_rope_relative_position():
    # <R(p1) q, R(p2) k> depends on p1 - p2 only (checked before rounding)
    rng = np.random.default_rng(6)
    q, k = rng.standard_normal(128), rng.standard_normal(128)

    def rot(v, p):
        th = oracle.rope_angles(np.array([p]), 128, 1e6)[0]
        a, b = v[:64], v[64:]
        return np.concatenate([a * np.cos(th) - b * np.sin(th), b * np.cos(th) + a * np.sin(th)])

    d1 = rot(q, 100) @ rot(k, 90)
    d2 = rot(q, 2010) @ rot(k, 2000)
    assert abs(d1 - d2) < 1e-9


# ------------------------------------------------------------- attention --

def _rand_bits(rng, shape, s=1.0):
    return _bits(rng.standard_normal(shape) * s)


def test_attention_root_alone_returns_its_value():
    rng = np.random.default_rng(7)
    q = _rand_bits(rng, (1, 4, 128))
    kn = _rand_bits(rng, (1, 2, 128))
    vn = _rand_bits(rng, (1, 2, 128))
    kp = np.zeros((2, 8, 128), np.uint16)
    out = oracle.tree_attention(q, kp, kp, kn, vn, np.ones((1, 1), bool), 0)
    for h in range(4):
        assert np.array_equal(out[0, h], vn[0, h // 2])


def test_attention_equal_keys_average_values():
    rng = np.random.default_rng(8)
    M, ctx = 3, 5
    parents = np.array([-1, 0, 1])
    ti = oracle.tree_info(parents)
    q = _rand_bits(rng, (M, 2, 128))
    key = _rand_bits(rng, (128,))
    kp = np.broadcast_to(key, (1, ctx, 128)).copy()
    kn = np.broadcast_to(key, (M, 1, 128)).copy()
    vp = _rand_bits(rng, (1, ctx, 128))
    vn = _rand_bits(rng, (M, 1, 128))
    out = oracle.bf16_to_f64(oracle.tree_attention(q, kp, vp, kn, vn, ti.anc, ctx))
    allv = oracle.bf16_to_f64(np.concatenate([vp[0], vn[:, 0]], 0))
    for i in range(M):
        vis = list(range(ctx)) + [ctx + j for j in range(M) if ti.anc[i, j]]
        want = oracle.bf16_to_f64(_bits(allv[vis].mean(0)))
        assert np.allclose(out[i, 0], want, atol=0, rtol=2 ** -7)


def test_attention_brute_force_loop():
    rng = np.random.default_rng(9)
    M, ctx, Hq, Hkv = 5, 6, 4, 2
    parents = np.array([-1, 0, 0, 1, 3])
    ti = oracle.tree_info(parents)
    q = _rand_bits(rng, (M, Hq, 128))
    kp, vp = _rand_bits(rng, (Hkv, ctx + 3, 128)), _rand_bits(rng, (Hkv, ctx + 3, 128))
    kn, vn = _rand_bits(rng, (M, Hkv, 128)), _rand_bits(rng, (M, Hkv, 128))
    out = oracle.tree_attention(q, kp, vp, kn, vn, ti.anc, ctx)
    f = oracle.bf16_to_f64
    for i in range(M):
        anc = []
        j = i
        while j >= 0:
            anc.append(j)
            j = parents[j]
        for h in range(Hq):
            g = h // 2
            ks = [f(kp[g, t]) for t in range(ctx)] + [f(kn[j, g]) for j in anc]
            vs = [f(vp[g, t]) for t in range(ctx)] + [f(vn[j, g]) for j in anc]
            sc = [float(np.dot(f(q[i, h]), kk)) / math.sqrt(128) for kk in ks]
            mx = max(sc)
            w = [math.exp(s - mx) for s in sc]
            o = sum(wi * vi for wi, vi in zip(w, vs)) / sum(w)
            assert np.array_equal(out[i, h], _bits(o))


# ----------------------------------------------------------- recurrence --

def test_linrec_literal_equals_closed_form():
    rng = np.random.default_rng(10)
    M, nh, hd = 6, 2, 128
    parents = np.array([-1, 0, 1, 0, 3, 3])
    ti = oracle.tree_info(parents)
    q, k, v = (_rand_bits(rng, (M, nh, hd)) for _ in range(3))
    S0 = rng.standard_normal((nh, hd, hd)) * 0.01
    z0 = np.abs(rng.standard_normal((nh, hd))) * 0.1
    out, S, z = oracle.linrec_literal(q, k, v, S0, z0, parents, 1e-6)
    f = oracle.bf16_to_f64
    # closed form: o_i = (S0^T fq_i + sum_{j in path(i)} (fk_j . fq_i) v_j) / (z0.fq_i + sum (fk_j . fq_i) + eps)
    fq = np.where(f(q) > 0, f(q) + 1, np.exp(np.minimum(f(q), 0)))
    fk = np.where(f(k) > 0, f(k) + 1, np.exp(np.minimum(f(k), 0)))
    for i in range(M):
        for h in range(nh):
            w = np.array([fk[j, h] @ fq[i, h] if ti.anc[i, j] else 0.0 for j in range(M)])
            num = S0[h].T @ fq[i, h] + w @ f(v)[:, h, :]
            den = z0[h] @ fq[i, h] + w.sum() + 1e-6
            assert np.array_equal(out[i, h], _bits(num / den))


def test_phi_is_elu_plus_one():
    x = np.linspace(-5, 5, 101)
    ref = torch.nn.functional.elu(torch.from_numpy(x)).numpy() + 1.0
    assert np.allclose(oracle.phi(x), ref, rtol=1e-15, atol=1e-15)


def test_argmax_margin_by_hand():
    L = np.array([[1.0, 3.0, 2.0, 3.0],      # tie at the top: the smaller index, margin 0
                  [-5.0, -1.0, -2.0, -7.0],  # margin 1
                  [0.5, 0.25, 0.125, 0.0]])  # first column wins, margin 0.25
    idx, margin = oracle.argmax_margin(L)
    assert list(idx) == [1, 1, 0]
    assert list(margin) == [0.0, 1.0, 0.25]


def test_residual_is_one_rounding_of_the_exact_sum():
    # 1 + 2^-8 is not a bf16 (7 mantissa bits): ties to even gives 1; 1 + 3*2^-8 rounds up to 1 + 2^-6
    one, e8 = np.uint16(0x3F80), np.uint16(0x3B80)  # 1.0 and 2^-8
    three_e8 = np.uint16(0x3C40)                    # 3 * 2^-8 = 1.5 * 2^-7
    assert int(oracle.residual(np.array([one]), np.array([e8]))[0]) == 0x3F80
    assert int(oracle.residual(np.array([one]), np.array([three_e8]))[0]) == 0x3F82
    # exact sums stay exact
    assert int(oracle.residual(np.array([one]), np.array([one]))[0]) == 0x4000
