"""Pins of the oracle's best-first selection under a shared node budget.

Selection follows "SpecPilot: AI Agent Framework Boosts Speculative Decoding
10.87x", "(2) Best-first Tree Verification for Hybrid Architectures"
(candidates ranked by parent-conditioned log-probability, highest
cumulative path scores kept) and "(4) Three Batch Optimization Mechanisms",
Shared Node Budget.  Pinned by a hand-worked example, closed forms (chain,
star), exhaustive search on small inputs in exact rational arithmetic, the
tie rule and invariants that hold at any size."""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synthetic
import synthetic.workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "select_shared_budget.txt")


def _ints(s):
    return np.array([int(x) for x in s.split()], dtype=np.int64)


def _floats(s):
    return np.array([float(x) for x in s.split()], dtype=np.float32)


def _golden():
    base, cases, cur = {}, [], None
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        if line.startswith("case "):
            cur = dict(kv.split("=") for kv in line[5:].split())
            cases.append(cur)
            continue
        k, v = (t.strip() for t in line.split("=", 1))
        (cur if cur is not None else base)[k] = v
    return base, cases


def test_golden_shared_budget():
    base, cases = _golden()
    assert len(cases) == 5
    for c in cases:
        s = oracle.best_first_select(_ints(base["parents"]), _floats(base["logprob"]), _ints(base["cu"]),
                                     int(c["budget"]), int(c["cap"]))
        assert s.status == 0
        np.testing.assert_array_equal(s.cu, _ints(c["out_cu"]))
        np.testing.assert_array_equal(s.src, _ints(c["src"]))
        np.testing.assert_array_equal(s.parents, _ints(c["out_parents"]))
        np.testing.assert_array_equal(s.scores, _floats(c["scores"]))


def test_chain_closed_form():
    # a chain with logprob[i] = -i/8 scores -i(i+1)/16 (exact in fp32) and
    # the budget takes its first nodes in order
    n = 12
    parents = synthetic.chain(n)
    lp = np.array([0.0] + [-i / 8 for i in range(1, n)], dtype=np.float32)
    np.testing.assert_array_equal(oracle.path_scores(parents, lp),
                                  np.array([-i * (i + 1) / 16 for i in range(n)], dtype=np.float32))
    for B in range(1, n + 3):
        for cap in (1, 5, n):
            s = oracle.best_first_select(parents, lp, [0, n], B, cap)
            k = min(B, cap, n)
            np.testing.assert_array_equal(s.src, np.arange(k))
            np.testing.assert_array_equal(s.parents, np.arange(-1, k - 1))
            assert list(s.cu) == [0, k]


def test_star_is_top_k():
    # all candidates children of the root: the kept children are the B-1
    # largest log-probabilities (a plain top-k), listed in index order
    n = 20
    perm = synthetic.permutation(synthetic.key(5, 77), n - 1)
    lp = np.concatenate([[0.0], -(perm + 1) / 16.0]).astype(np.float32)
    parents = np.array([-1] + [0] * (n - 1), dtype=np.int32)
    for B in (1, 2, 7, n - 1, n, n + 4):
        s = oracle.best_first_select(parents, lp, [0, n], B, n)
        k = min(B, n) - 1
        top = np.sort(1 + np.argsort(-lp[1:], kind="stable")[:k])
        np.testing.assert_array_equal(s.src, np.concatenate([[0], top]))
        assert (s.parents[1:] == 0).all()


def _exact_scores(parents, lp):
    # rational sum of the log-probabilities on each node's root path, walking
    # up from the node (a different order and exact arithmetic)
    out = []
    for i in range(len(parents)):
        tot, j = Fraction(0), i
        while j > 0:
            tot += Fraction(float(lp[j]))
            j = int(parents[j])
        out.append(tot)
    return out


def _brute(trees, budget, cap):
    # best-first = the feasible K-subset whose sorted keys are smallest in
    # lexicographic order (keys: roots first, score descending, global index)
    keys, req = [], []
    g = 0
    for r, (parents, lp) in enumerate(trees):
        ex = _exact_scores(parents, lp)
        for i in range(len(parents)):
            keys.append((0 if i == 0 else 1, -ex[i], g))
            req.append(r)
            g += 1
    n_r = [len(p) for p, _ in trees]
    K = min(budget, sum(min(n, cap) for n in n_r))
    best = None
    for sub in itertools.combinations(range(g), K):
        cnt = [0] * len(trees)
        for x in sub:
            cnt[req[x]] += 1
        if max(cnt) > cap:
            continue
        ks = sorted(keys[x] for x in sub)
        if best is None or ks < best[0]:
            best = (ks, sub)
    return sorted(best[1])


def _small_trees(n):
    for ps in itertools.product(*[range(i) for i in range(1, n)]):
        yield np.array((-1,) + ps, dtype=np.int32)


def test_exhaustive_small_batches():
    vals = [0.0, -0.25, -0.5, -1.0]  # ties and zero log-probabilities included
    rng_k = synthetic.key(9, 1)
    draws = synthetic.uniform_int(rng_k, 4000, 0, 1 << 30)
    t = 0
    shapes = [[3, 3], [4, 2], [1, 4], [3, 2, 2], [4, 4]]
    checked = 0
    for sh in shapes:
        for rep in range(12):
            trees = []
            for n in sh:
                opts = list(_small_trees(n))
                parents = opts[int(draws[t]) % len(opts)]
                t += 1
                lp = np.array([0.0] + [vals[int(draws[t + i]) % 4] for i in range(n - 1)], dtype=np.float32)
                t += n
                trees.append((parents, lp))
            parents = np.concatenate([p for p, _ in trees])
            lp = np.concatenate([l for _, l in trees])
            cu = np.concatenate([[0], np.cumsum(sh)])
            for budget in range(len(sh), sum(sh) + 2):
                for cap in (1, 2, 3, 8):
                    s = oracle.best_first_select(parents, lp, cu, budget, cap)
                    assert s.status == 0
                    assert list(s.src) == _brute(trees, budget, cap)
                    checked += 1
    assert checked > 1000


def test_equal_scores_lower_request_then_lower_index():
    # two identical stars: each score level goes to request 0 first
    parents = [-1, 0, 0, -1, 0, 0]
    lp = [0, -0.25, -0.5, 0, -0.25, -0.5]
    cu = [0, 3, 6]
    assert list(oracle.best_first_select(parents, lp, cu, 3, 8).src) == [0, 1, 3]
    assert list(oracle.best_first_select(parents, lp, cu, 4, 8).src) == [0, 1, 3, 4]
    assert list(oracle.best_first_select(parents, lp, cu, 5, 8).src) == [0, 1, 2, 3, 4]
    # zero log-probabilities: a node ties its parent and follows it (lower index)
    parents = [-1, 0, 1, 2, 0]
    lp = [0, 0, 0, -0.0, 0]
    assert list(oracle.best_first_select(parents, lp, [0, 5], 3, 8).src) == [0, 1, 2]
    # -inf log-probabilities rank last, by index
    lp = [0, -np.inf, -1, -np.inf, -2]
    s = oracle.best_first_select(parents, lp, [0, 5], 4, 8)
    assert list(s.src) == [0, 1, 2, 4] and s.status == 0


def test_invalid_requests_keep_nothing():
    c = wl.candidates(3, 4, 9, 4, 1000, step=0.125)
    ok = oracle.best_first_select(c.parents, c.logprob, c.cu, 20, 6)
    assert ok.status == 0
    for bad in ("parent", "root", "positive", "nan"):
        p, lp = c.parents.copy(), c.logprob.copy()
        a = int(c.cu[2])
        if bad == "parent":
            p[a + 4] = 4
        elif bad == "root":
            p[a] = 0
        elif bad == "positive":
            lp[a + 3] = 0.5
        else:
            lp[a + 5] = np.nan
        s = oracle.best_first_select(p, lp, c.cu, 20, 6)
        assert s.status == oracle.SELECT_BAD_TREE
        assert s.cu[3] == s.cu[2]  # request 2 keeps nothing
        # the others get what they get with request 2 absent
        keep = np.r_[0:c.cu[2], c.cu[3]:c.cu[4]]
        cu3 = np.array([0, c.cu[1], c.cu[2], c.cu[2] + c.cu[4] - c.cu[3]])
        ref = oracle.best_first_select(c.parents[keep], c.logprob[keep], cu3, 20, 6)
        np.testing.assert_array_equal(keep[ref.src], s.src)
        np.testing.assert_array_equal(ref.parents, s.parents)


@pytest.mark.parametrize("seed", range(6))
def test_invariants_on_synthetic_batches(seed):
    R = 5 + seed
    ns = 1 + synthetic.uniform_int(synthetic.key(seed, 3), R, 0, 40)
    c = wl.candidates(seed, R, ns, 6, 1000, step=0.25 if seed % 2 else 0.0)
    for budget, cap in ((R, 64), (R + 7, 3), (3 * R, 8), (int(ns.sum()) + 1, 64)):
        s = oracle.best_first_select(c.parents, c.logprob, c.cu, budget, cap)
        assert s.status == 0
        full = []
        worst = None  # the worst kept non-root key
        for r in range(R):
            a, b = int(c.cu[r]), int(c.cu[r + 1])
            sel = s.src[s.cu[r]:s.cu[r + 1]]
            assert len(sel) >= 1 and sel[0] == a  # root kept
            assert len(sel) <= cap
            full.append(len(sel) == min(cap, b - a))
            kept = set(int(x) for x in sel)
            sc = oracle.path_scores(c.parents[a:b], c.logprob[a:b])
            for j, g in enumerate(sel):  # prefix closed, parents renumbered
                if j:
                    pg = a + int(c.parents[g])
                    assert pg in kept and sel[s.parents[s.cu[r] + j]] == pg
                    assert s.scores[s.cu[r] + j] == sc[g - a]
                    k = (-float(sc[g - a]), int(g))
                    worst = k if worst is None or k > worst else worst
        total = int(s.cu[-1])
        assert total == min(budget, sum(min(cap, int(n)) for n in ns))
        # nothing left out that ranks above a kept node, unless its request is full
        for r in range(R):
            if full[r] or worst is None:
                continue
            a, b = int(c.cu[r]), int(c.cu[r + 1])
            sc = oracle.path_scores(c.parents[a:b], c.logprob[a:b])
            kept = set(int(x) for x in s.src[s.cu[r]:s.cu[r + 1]])
            for i in range(1, b - a):
                if a + i not in kept:
                    assert (-float(sc[i]), a + i) > worst
