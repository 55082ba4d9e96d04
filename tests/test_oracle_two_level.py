"""Pins of the oracle's two-level verification ("SpecPilot: AI Agent Framework
Boosts Speculative Decoding 10.87x", "(3) Two-Level Verification": a round
over W12's nested 8-bit weight view proposes a chain without accepting, the
drafter extends it, one exact verification decides).  Pinned by the nested
relation between the 8-bit view and the packed 12-bit field, the view's
truncation bound, losslessness against exact greedy decoding token by token
(brute force), the case where the view is exact, and the untouched state."""
import copy

import numpy as np
import pytest

import oracle
import synthetic
from helpers import oracle_request
from synthetic import workloads as wl


def test_view_is_the_high_byte_of_the_packed_field():
    W = synthetic.normal_bf16(synthetic.key(31, 1), 64 * 128, 0.02).reshape(64, 128)
    W[3, 5] = 0x0001  # a subnormal: escapes
    p = oracle.w12_pack(W)
    v8 = oracle.w12_view8(W)
    esc = set(int(i) for i in p.esc_idx)
    table = [int(t) for t in p.table]
    checked = 0
    for n in range(64):
        for k in range(128):
            if n * 128 + k in esc:
                continue
            f = oracle.w12_field(p, n, k)  # sign << 11 | code << 7 | mantissa
            hi = f >> 4                    # sign << 7 | code << 3 | top 3 mantissa bits
            sign, code, m3 = hi >> 7, (hi >> 3) & 15, hi & 7
            assert int(v8[n, k]) == (sign << 15) | (table[code] << 7) | (m3 << 4)
            checked += 1
    assert checked == 64 * 128 - len(esc) and len(esc) >= 1


def test_view_truncates_toward_zero_within_its_bound():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    e = (bits >> 7) & 0xFF
    finite = (e > 0) & (e < 255)
    w = oracle.bf16_to_f64(bits[finite])
    v = oracle.bf16_to_f64(oracle.w12_view8(bits[finite]))
    assert (np.sign(v) == np.sign(w)).all() and (np.abs(v) <= np.abs(w)).all()
    # at most 15/128 of the leading power of two is dropped
    lead = 2.0 ** (e[finite].astype(np.float64) - 127)
    assert (np.abs(w - v) <= lead * 15 / 128).all()
    np.testing.assert_array_equal(oracle.w12_view8(oracle.w12_view8(bits)), oracle.w12_view8(bits))


@pytest.fixture(scope="module")
def mini():
    shape = wl.SHAPES["mini"]
    return shape, wl.SyntheticWeights(shape, seed=3, cache=True)


def _greedy(shape, W, root, ctx, n):
    """Exact greedy decoding, one token at a time: n tokens after the root."""
    seq = [int(root)]
    for _ in range(n):
        req = oracle_request(shape, 3, 0, ctx, seq, np.arange(-1, len(seq) - 1))
        seq.append(int(oracle.forward(shape, W, [req]).argmax[-1]))
    return seq[1:]


def _extend_with(shape, W, ctx, good: int, rng_key: int):
    """A drafter that continues the chain with `good` exact greedy tokens and
    then two random ones (as a chain)."""
    def extend(chain):
        seq = [int(t) for t in chain]
        out = []
        for _ in range(good):
            req = oracle_request(shape, 3, 0, ctx, seq, np.arange(-1, len(seq) - 1))
            t = int(oracle.forward(shape, W, [req]).argmax[-1])
            seq.append(t)
            out.append(t)
        out += [int(x) for x in synthetic.uniform_int(rng_key, 2, 0, shape.V - 1)]  # bounds inclusive
        return np.array(out, np.int32), np.arange(-1, len(out) - 1)
    return extend


@pytest.mark.parametrize("case", range(3))
def test_two_levels_accept_exactly_what_greedy_decoding_produces(mini, case):
    shape, W = mini
    ctx = 40 + 7 * case
    td = wl.draft(50 + case, 0, 9, 4, 0.8, shape.V)
    toks = wl.copy_rule_tokens(td, lambda tok, par: oracle.forward(
        shape, W, [oracle_request(shape, 3, 0, ctx, tok, par)]).argmax)
    req = oracle_request(shape, 3, 0, ctx, toks, td.parents)
    tl = oracle.two_level_verify(shape, W, req, _extend_with(shape, W, ctx, case, synthetic.key(60, case)))
    L = tl.exact.accepted_len
    got = [int(t) for t in tl.exact.accepted_tokens] + [int(tl.exact.bonus)]
    assert got == _greedy(shape, W, toks[0], ctx, L + 1)
    # the exact round's tree is the chain (a path from the root) with the drafts below its end
    n = len(tl.chain)
    assert list(tl.parents[:n]) == list(range(-1, n - 1))
    assert (tl.parents[n:] >= n - 1).all()


def test_exact_view_makes_both_levels_agree(mini):
    # weights whose 4 low mantissa bits are zero: the 8-bit view is exact, so
    # round one's chain is the exact walk of the draft tree plus its bonus
    shape, W = mini

    class Rounded:
        def __init__(self, base):
            self.base = base

        def layer(self, l, name):
            return oracle.w12_view8(self.base.layer(l, name))

        def lm_head(self):
            return oracle.w12_view8(self.base.lm_head())

        def __getattr__(self, name):
            return getattr(self.base, name)

    Wr = Rounded(W)
    ctx = 33
    td = wl.draft(70, 0, 8, 4, 0.9, shape.V)
    toks = wl.copy_rule_tokens(td, lambda tok, par: oracle.forward(
        shape, Wr, [oracle_request(shape, 3, 0, ctx, tok, par)]).argmax)
    req = oracle_request(shape, 3, 0, ctx, toks, td.parents)
    ex = oracle.accept(toks, td.parents, oracle.forward(shape, Wr, [req]).argmax)
    tl = oracle.two_level_verify(shape, Wr, req, lambda chain: (np.zeros(0, np.int32), np.zeros(0, np.int32)))
    assert tl.low.path == ex.path
    assert list(tl.chain) == [int(toks[0])] + [int(t) for t in ex.accepted_tokens] + [int(ex.bonus)]
    # with no new drafts the exact round accepts the whole chain
    assert tl.exact.accepted_len == len(tl.chain) - 1


def test_round_one_leaves_the_state_alone(mini):
    shape, W = mini
    td = wl.draft(80, 0, 6, 3, 0.7, shape.V)
    req = oracle_request(shape, 3, 0, 25, np.arange(6) + 11, td.parents)
    before = copy.deepcopy(req.layers)
    oracle.two_level_verify(shape, W, req, lambda chain: (np.array([5, 6], np.int32), np.array([-1, 0])))
    for a, b in zip(before, req.layers):
        for f in ("k", "v", "S", "z"):
            x, y = getattr(a, f), getattr(b, f)
            assert (x is None and y is None) or np.array_equal(x, y)
