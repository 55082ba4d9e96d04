"""The synthetic candidate-tree generator keeps the guarantees the selection
and the batched verify rely on: trees rooted at entry 0 with parent[i] < i
and depth within the bound, log-probabilities <= 0 (0 at the roots, exact
ties on a grid when asked), tokens inside the vocabulary, consistent
offsets, and the same draws for the same seed."""
import numpy as np

from synthetic import workloads as wl


def _depths(par):
    d = np.zeros(len(par), np.int64)
    for i in range(1, len(par)):
        d[i] = d[par[i]] + 1
    return d


def test_generator_guarantees():
    for seed, step in ((1, 0.0), (2, 0.25)):
        ns = [1, 7, 64, 300]
        c = wl.candidates(seed, len(ns), ns, 6, 1000, step=step)
        assert list(c.cu) == [0, 1, 8, 72, 372]
        assert c.parents.dtype == np.int32 and c.logprob.dtype == np.float32 and c.tokens.dtype == np.int32
        assert ((c.tokens >= 0) & (c.tokens < 1000)).all()
        for r in range(len(ns)):
            a, b = c.cu[r], c.cu[r + 1]
            p, lp = c.parents[a:b], c.logprob[a:b]
            assert p[0] == -1 and all(0 <= p[i] < i for i in range(1, len(p)))
            assert _depths(p).max() <= 6
            assert lp[0] == 0 and (lp <= 0).all() and np.isfinite(lp).all()
            if step:
                assert (np.abs(lp / step - np.round(lp / step)) == 0).all()
        if step:
            # exact ties occur on the grid
            assert len(np.unique(c.logprob)) < len(c.logprob) // 2
    x, y = wl.candidates(5, 3, 20, 4, 50), wl.candidates(5, 3, 20, 4, 50)
    assert all(np.array_equal(getattr(x, f), getattr(y, f)) for f in ("parents", "logprob", "tokens", "cu"))
