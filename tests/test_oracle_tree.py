"""Pins of the oracle's tree bookkeeping and greedy acceptance.

Acceptance follows "SpecPilot: AI Agent Framework Boosts Speculative
Decoding 10.87x", "(3) Two-Level Verification" (only the exact target
verification accepts tokens) with greedy matching: checked against brute
force enumeration of root-to-node paths on every small tree."""
import itertools

import numpy as np

import oracle
import synthetic


def _all_trees(M):
    # every parent array with parent[i] < i
    for ps in itertools.product(*[range(i) for i in range(1, M)]):
        yield np.array((-1,) + ps, dtype=np.int32)


def _brute(tokens, parents, argmax):
    M = len(parents)
    best_depth, best_node = -1, None
    for node in range(M):
        path = []
        j = node
        while j >= 0:
            path.append(j)
            j = parents[j]
        path.reverse()
        if all(tokens[path[i]] == argmax[path[i - 1]] for i in range(1, len(path))):
            d = len(path) - 1
            if d > best_depth:  # ascending node scan: first deepest = smallest index
                best_depth, best_node, best_path = d, node, path
    return best_depth, best_node, best_path


def test_accept_matches_brute_force_all_small_trees():
    cases = 0
    for M in range(1, 7):
        for parents in _all_trees(M):
            for pattern in range(1 << (M - 1)):
                # argmax[i] = 100 + i; token[i] matches its parent iff bit set
                argmax = np.array([100 + i for i in range(M)])
                tokens = np.array([7] + [argmax[parents[i]] if (pattern >> (i - 1)) & 1 else 5 for i in range(1, M)])
                a = oracle.accept(tokens, parents, argmax)
                d, node, path = _brute(tokens, parents, argmax)
                assert (a.accepted_len, a.last, a.path) == (d, node, path)
                assert a.accepted_tokens == [int(tokens[j]) for j in path[1:]]
                assert a.bonus == argmax[node]
                cases += 1
    assert cases == sum(np.prod(range(1, M)) * (1 << (M - 1)) for M in range(1, 7))


def test_accept_duplicate_siblings_prefer_smallest_index():
    parents = np.array([-1, 0, 0, 1, 2])
    argmax = np.array([9, 4, 4, 1, 1])
    tokens = np.array([0, 9, 9, 4, 4])  # both branches fully match, equal depth
    a = oracle.accept(tokens, parents, argmax)
    assert a.path == [0, 1, 3] and a.accepted_len == 2 and a.bonus == 1


def test_tree_info_closed_form():
    parents = synthetic.tree(synthetic.key(0, 1), 40, 6)
    ti = oracle.tree_info(parents)
    assert ti.valid
    for i in range(40):
        assert ti.anc[i, i]
        if i:
            # anc(i) = {i} U anc(parent(i)); depth(i) = depth(parent(i)) + 1
            assert np.array_equal(ti.anc[i] & ~np.eye(40, dtype=bool)[i], ti.anc[parents[i]])
            assert ti.depth[i] == ti.depth[parents[i]] + 1
    assert ti.depth.max() <= 6


def test_tree_info_rejects_bad_parents():
    for bad in ([0, 0], [-1, 1], [-1, 0, 3], [-1, -1], []):
        assert not oracle.tree_info(np.array(bad, dtype=np.int64)).valid


def test_generated_tree_respects_depth():
    for seed in range(5):
        p = synthetic.tree(synthetic.key(seed, 1), 64, 10)
        assert p[0] == -1 and all(0 <= p[i] < i for i in range(1, 64))
        assert oracle.tree_info(p).depth.max() <= 10
