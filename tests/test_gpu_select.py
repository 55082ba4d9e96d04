"""Best-first node selection under a shared node budget on the GPU
(sd_best_first_select) against the oracle, bit for bit: kept nodes, their
order, renumbered parents, gathered tokens, fp32 path scores and the status
word.  Inputs: the hand-worked example, synthetic candidate batches (with
and without exact ties), the per-call and per-request maxima, deep chains,
roots-only and take-everything budgets, binding and non-binding caps, and
invalid requests."""
import numpy as np
import pytest
import torch

import oracle
from synthetic import workloads as wl

pytestmark = pytest.mark.gpu

GOLDEN_PARENTS = [-1, 0, 0, 1, 1, -1, 0, 1, 0]
GOLDEN_LP = [0, -0.5, -1, -0.25, -2, 0, -0.25, -0.25, -0.75]


@pytest.fixture(scope="module")
def sel():
    from speculative_decoding_tree_bit_gb300 import model
    return model.Selector(16384, 4096)


def _dev(a, dt):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=dt))).cuda()


def _check(sel, parents, logprob, cu, budget, cap, tokens=None):
    ref = oracle.best_first_select(parents, logprob, cu, budget, cap)
    tok = _dev(tokens, np.int32) if tokens is not None else None
    o = sel(_dev(parents, np.int32), _dev(logprob, np.float32), _dev(cu, np.int32), budget, cap, tokens=tok)
    torch.cuda.synchronize()
    assert int(o["status"].item()) == ref.status
    out_cu = o["cu"].cpu().numpy()
    np.testing.assert_array_equal(out_cu, ref.cu)
    k = int(out_cu[-1])
    np.testing.assert_array_equal(o["src"][:k].cpu().numpy(), ref.src)
    np.testing.assert_array_equal(o["parents"][:k].cpu().numpy(), ref.parents)
    got_s = o["score"][:k].cpu().numpy()
    np.testing.assert_array_equal(got_s.view(np.uint32), ref.scores.view(np.uint32))
    if tokens is not None:
        np.testing.assert_array_equal(o["tokens"][:k].cpu().numpy(), np.asarray(tokens)[ref.src])
    return ref


@pytest.mark.parametrize("budget,cap", [(6, 3), (6, 2), (4, 8), (7, 8), (2, 8), (9, 9), (20, 1)])
def test_hand_worked_example(sel, budget, cap):
    _check(sel, GOLDEN_PARENTS, GOLDEN_LP, [0, 5, 9], budget, cap)


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("step", [0.0, 0.25])
def test_synthetic_batches(sel, seed, step):
    from synthetic import key, uniform_int
    R = [1, 4, 32, 64][seed]
    ns = 1 + uniform_int(key(seed, 11), R, 0, 300)
    c = wl.candidates(100 + seed, R, ns, 8, 32000, step=step)
    N = int(c.cu[-1])
    for budget, cap in ((R, 64), (R + 5, 2), (8 * R, 64), (8 * R, 1 << 20), (N, 16), (N + 3, 1 << 20)):
        _check(sel, c.parents, c.logprob, c.cu, budget, cap, tokens=c.tokens)


def test_batch_of_32_requests_256_candidates(sel):
    # the size the selection probe times: 32 x 256 candidates, 256 nodes, <= 64 per request
    c = wl.candidates(7, 32, 256, 8, 32000)
    ref = _check(sel, c.parents, c.logprob, c.cu, 256, 64, tokens=c.tokens)
    assert ref.cu[-1] == 256


def test_maximum_sizes(sel):
    # 16384 candidates (the per-call maximum) as 8 requests of 2048 (the
    # per-request maximum); the cap binds, so every request ranks its own
    c = wl.candidates(8, 8, 2048, 12, 32000, step=0.5)
    _check(sel, c.parents, c.logprob, c.cu, 1000, 200, tokens=c.tokens)
    # one request: a 2048-node chain (2048 scoring rounds) with many zero log-probabilities
    par = np.arange(-1, 2047, dtype=np.int32)
    lp = wl.candidates(9, 1, 2048, 1, 10, step=2.0).logprob
    _check(sel, par, lp, [0, 2048], 700, 2048)
    _check(sel, par, lp, [0, 2048], 2048, 300)


def test_single_nodes_and_infinite_log_probabilities(sel):
    _check(sel, [-1], [0], [0, 1], 1, 1)
    _check(sel, [-1, -1, -1], [0, 0, 0], [0, 1, 2, 3], 3, 5)
    par = [-1, 0, 0, 1, 2, -1, 0, 1]
    lp = [0, -np.inf, -1, -0.5, -np.inf, 0, -np.inf, 0]
    for budget in range(2, 9):
        _check(sel, par, lp, [0, 5, 8], budget, 8)


@pytest.mark.parametrize("bad", ["parent", "root", "positive", "nan", "too_many"])
def test_invalid_request_keeps_nothing(sel, bad):
    c = wl.candidates(12, 4, 40, 5, 1000, step=0.125)
    par, lp, cu = c.parents.copy(), c.logprob.copy(), c.cu.copy()
    a = int(cu[1])
    if bad == "parent":
        par[a + 7] = 9
    elif bad == "root":
        par[a] = 3
    elif bad == "positive":
        lp[a + 2] = 1.0
    elif bad == "nan":
        lp[a + 9] = np.nan
    if bad == "too_many":
        # request 1 grows to 2049 candidates: past the per-request maximum
        big = wl.candidates(13, 1, 2049, 6, 1000)
        par = np.concatenate([par[:a], big.parents, par[cu[2]:]])
        lp = np.concatenate([lp[:a], big.logprob, lp[cu[2]:]])
        cu = np.concatenate([cu[:2], cu[2:] - cu[2] + a + 2049])
        o = sel(_dev(par, np.int32), _dev(lp, np.float32), _dev(cu, np.int32), 30, 8)
        torch.cuda.synchronize()
        assert int(o["status"].item()) == oracle.SELECT_BAD_TREE
        out_cu = o["cu"].cpu().numpy()
        assert out_cu[2] == out_cu[1]
        # the others: as the oracle selects them with request 1 absent
        keep = np.r_[0:cu[1], cu[2]:cu[4]]
        cu3 = np.array([0, cu[1], cu[1] + cu[3] - cu[2], cu[1] + cu[4] - cu[2]])
        ref = oracle.best_first_select(par[keep], lp[keep], cu3, 30, 8)
        k = int(out_cu[-1])
        np.testing.assert_array_equal(o["src"][:k].cpu().numpy(), keep[ref.src])
        return
    ref = _check(sel, par, lp, cu, 30, 8)
    assert ref.status == oracle.SELECT_BAD_TREE and ref.cu[2] == ref.cu[1]


def test_bad_cu_sets_status_and_selects_nothing(sel):
    c = wl.candidates(14, 3, 10, 4, 1000)
    cu = np.array([0, 10, 4, 30], dtype=np.int32)  # decreasing: not a split of the candidates
    o = sel(_dev(c.parents, np.int32), _dev(c.logprob, np.float32), _dev(cu, np.int32), 5, 4)
    torch.cuda.synchronize()
    assert int(o["status"].item()) == oracle.SELECT_BAD_TREE
    assert (o["cu"].cpu().numpy() == 0).all()


def test_selection_feeds_the_batched_verify(sel):
    """Kept nodes, renumbered parents and gathered tokens are a valid
    sd_verify_batch input: every kept request is a tree with its root first."""
    c = wl.candidates(15, 16, 120, 7, 32000, step=0.25)
    o = sel(_dev(c.parents, np.int32), _dev(c.logprob, np.float32), _dev(c.cu, np.int32), 160, 64,
            tokens=_dev(c.tokens, np.int32))
    torch.cuda.synchronize()
    cu = o["cu"].cpu().numpy()
    par = o["parents"].cpu().numpy()
    for r in range(16):
        p = par[cu[r]:cu[r + 1]]
        assert 1 <= len(p) <= 64 and p[0] == -1
        assert all(0 <= p[i] < i for i in range(1, len(p)))
