"""Model-level pins of the oracle on small decoders (dense and hybrid).

* a chain-shaped tree gives the same logits as M one-token decodes, each
  committing its token (this pins tree masks, positions and the recurrent
  state's root path against plain decoding);
* relabelling the nodes of a tree permutes its outputs;
* siblings with equal tokens get equal outputs;
* rows of different requests do not interact (batched == one by one);
* after committing an accepted path, a one-token decode of the bonus token
  equals the last node of a chain verify of the accepted tokens.
"""
import numpy as np
import pytest

import oracle
from synthetic import workloads as wl


def _request(shape, seed, r, ctx, tokens, parents, cap=None):
    cap = cap or ctx + 80
    layers = []
    for l, kind in enumerate(shape.layer_kinds):
        if kind == "attn":
            k, v = wl.kv_prefix(shape, seed, r, l, ctx, cap)
            layers.append(oracle.LayerState(k=k, v=v))
        else:
            S, z = wl.rec_state(shape, seed, r, l)
            layers.append(oracle.LayerState(S=S.astype(np.float64), z=z.astype(np.float64)))
    return oracle.Request(np.asarray(tokens, np.int32), np.asarray(parents, np.int32), ctx, layers)


@pytest.fixture(scope="module", params=["mini", "mini_hybrid"])
def model(request):
    shape = wl.SHAPES[request.param]
    return shape, wl.SyntheticWeights(shape, seed=3, cache=True)


def _close(a, b):
    return np.allclose(a, b, rtol=1e-9, atol=1e-9)


def test_chain_equals_sequential_decode(model):
    shape, W = model
    M, ctx = 6, 20
    rng = np.random.default_rng(0)
    toks = rng.integers(0, shape.V, M)
    req = _request(shape, 3, 0, ctx, toks, np.arange(-1, M - 1))
    out = oracle.forward(shape, W, [req])
    cur = _request(shape, 3, 0, ctx, toks[:1], [-1])
    for i in range(M):
        cur.tokens = np.array([toks[i]], np.int32)
        cur.parents = np.array([-1], np.int32)
        o1 = oracle.forward(shape, W, [cur])
        assert _close(o1.logits[0], out.logits[i])
        assert o1.argmax[0] == out.argmax[i]
        acc = oracle.Accept(0, [], int(o1.argmax[0]), [0], 0)
        cur = oracle.commit(shape, [cur], o1, [acc])[0]


def test_relabelled_tree_permutes_outputs(model):
    shape, W = model
    parents = np.array([-1, 0, 0, 1, 1, 2, 4, 3])
    rng = np.random.default_rng(1)
    toks = rng.integers(0, shape.V, parents.size)
    # new order: breadth-first (depth, then old index) keeps parent < child
    d = wl.depths(parents)
    order = sorted(range(parents.size), key=lambda i: (d[i], -i if i else 0))
    new_of = {o: n for n, o in enumerate(order)}
    p2 = np.array([-1 if parents[o] < 0 else new_of[parents[o]] for o in order])
    assert all(p2[i] < i for i in range(1, p2.size))
    a = oracle.forward(shape, W, [_request(shape, 3, 0, 12, toks, parents)])
    b = oracle.forward(shape, W, [_request(shape, 3, 0, 12, toks[order], p2)])
    assert _close(a.logits[order], b.logits)


def test_equal_siblings_equal_outputs(model):
    shape, W = model
    parents = np.array([-1, 0, 0, 1, 2])
    toks = np.array([11, 42, 42, 7, 7])
    o = oracle.forward(shape, W, [_request(shape, 3, 0, 9, toks, parents)])
    assert np.array_equal(o.logits[1], o.logits[2])
    assert np.array_equal(o.logits[3], o.logits[4])


def test_requests_do_not_interact(model):
    shape, W = model
    r0 = _request(shape, 3, 0, 15, [5, 6, 7], [-1, 0, 0])
    r1 = _request(shape, 3, 1, 33, [8, 9, 10, 11], [-1, 0, 1, 2])
    both = oracle.forward(shape, W, [r0, r1])
    a = oracle.forward(shape, W, [r0])
    b = oracle.forward(shape, W, [r1])
    assert np.array_equal(both.logits, np.concatenate([a.logits, b.logits]))


def test_commit_then_decode_equals_chain_verify(model):
    shape, W = model
    ctx = 17
    td = wl.draft(5, 0, 10, 4, 0.9, shape.V)

    def am(tok, par):
        return oracle.forward(shape, W, [_request(shape, 3, 0, ctx, tok, par)]).argmax

    toks = wl.copy_rule_tokens(td, am)
    req = _request(shape, 3, 0, ctx, toks, td.parents)
    out, (acc,), (st,) = oracle.verify(shape, W, [req])
    assert acc.accepted_len >= 1  # p = 0.9 copy rule on a 10-node tree
    assert st.ctx == ctx + acc.accepted_len + 1
    # one-token decode of the bonus over the committed state
    st.tokens, st.parents = np.array([acc.bonus], np.int32), np.array([-1], np.int32)
    dec = oracle.forward(shape, W, [st])
    chain_toks = [int(toks[0])] + acc.accepted_tokens + [acc.bonus]
    ch = oracle.forward(shape, W, [_request(shape, 3, 0, ctx, chain_toks, np.arange(-1, len(chain_toks) - 1))])
    assert _close(dec.logits[0], ch.logits[-1])
    # the accepted path's logits are the tree's logits at those nodes
    assert _close(ch.logits[:-1], out.logits[acc.path])
