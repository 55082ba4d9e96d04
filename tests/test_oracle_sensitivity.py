"""How far an fp32-accumulating implementation of the model definition moves
from the fp64 oracle: the oracle's own fp32-accumulation twin (every GEMM
summed in fp32, everything else unchanged, no code shared with the CUDA
path) against the oracle.

The workloads' rule gives the tolerance for bf16 logits computed in fp32
accumulation and exempts argmax positions whose top-2 margin is under 1e-3.
Each bf16 rounding point downstream of a GEMM turns the tiny fp32-vs-fp64
difference of a sum into a whole-ulp difference for some elements, and the
residual stream carries these forward, so the twin itself:

* flips argmax positions whose oracle margin is above 1e-3 on the small
  dense decoder (its logits still meet the element-wise tolerance), and
* breaks the element-wise logit tolerance on some elements at the 8B-class
  widths after two layers (every row's relative 2-norm error stays below
  1e-2, the largest at about 0.7e-2, and no argmax changes).

These are properties of the definition, so the end-to-end GPU tests read the
rule as follows: element-wise tolerance on the small models, per-row relative
2-norm error <= 1e-2 at the full widths; an argmax may differ where the
oracle margin is under 1e-3, or where the two tokens' oracle logits are within
the logit tolerance of each other (both are correct answers under it), such
cases counted and bounded.  The strict margin rule is applied unrelaxed where
both sides take the decision from the same inputs (the lm_head and argmax
over the step's own final hidden state, the tiny model, single GEMMs)."""
import numpy as np
import pytest

import oracle
from synthetic import workloads as wl
from helpers import ATOL, MARGIN, RTOL, oracle_request


def _pair(shape, W, td, tokens, ctx, seed):
    req = oracle_request(shape, seed, 0, ctx, tokens, td.parents, cap=ctx + 80)
    return oracle.forward(shape, W, [req]), oracle.forward(shape, W, [req], gemm=oracle.linear_f32)


@pytest.mark.parametrize("s", [4, 21])
def test_fp32_accumulation_flips_argmax_above_the_margin_on_the_small_decoder(s):
    shape = wl.SHAPES["mini"]
    W = wl.SyntheticWeights(shape, seed=3, cache=True)
    td = wl.draft(100 + s, 0, 64, 10, 0.7, shape.V)
    tokens = np.concatenate([[td.root_token], td.rand_tok[1:]]).astype(np.int32)
    ref, alt = _pair(shape, W, td, tokens, 50 + 7 * s, 3)
    err = np.abs(alt.logits - ref.logits)
    assert np.all(err <= ATOL + RTOL * np.abs(ref.logits))
    flips = np.nonzero(alt.argmax != ref.argmax)[0]
    assert any(ref.margin[i] >= MARGIN for i in flips), [(int(i), float(ref.margin[i])) for i in flips]
    for i in flips:
        top, other = ref.logits[i, ref.argmax[i]], ref.logits[i, alt.argmax[i]]
        assert top - other <= ATOL + RTOL * abs(top)


def test_fp32_accumulation_breaks_the_elementwise_tolerance_at_8b_widths():
    shape = wl.SHAPES["8b_2l"]
    W = wl.SyntheticWeights(shape, seed=0, cache=True)
    td = wl.draft(0, 0, 16, 8, 0.7, shape.V)
    tokens = np.concatenate([[td.root_token], td.rand_tok[1:]]).astype(np.int32)
    ref, alt = _pair(shape, W, td, tokens, 2048, 0)
    err = np.abs(alt.logits - ref.logits)
    assert np.any(err > ATOL + RTOL * np.abs(ref.logits))
    rel = np.linalg.norm(alt.logits - ref.logits, axis=1) / np.linalg.norm(ref.logits, axis=1)
    assert rel.max() < RTOL, rel.max()
    assert np.array_equal(alt.argmax, ref.argmax)
