"""Two-level verification on the GPU ("SpecPilot: AI Agent Framework Boosts
Speculative Decoding 10.87x", "(3) Two-Level Verification") against the
oracle (oracle.w12_view8, View8Weights, two_level_verify).

* The device packer of the nested 8-bit plane writes the host packer's
  plane bit for bit (row orders of the fused tensors included).
* Round one (sd_forward_view8) streams the planes: its logits and argmax
  match the oracle's forward over the 8-bit view, and it commits nothing.
* The whole protocol - round one, its greedy walk (sd_accept) as the
  candidate chain, a drafter's extension, one exact sd_verify_step - gives
  the oracle's chain and the oracle's exact acceptance, which is what exact
  greedy decoding gives."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import workloads as wl
from helpers import (assert_accept, assert_argmax, assert_close, assert_final_hidden, oracle_copy_tokens,
                     oracle_request)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from speculative_decoding_tree_bit_gb300 import model
    return model


@pytest.fixture(scope="module")
def mdl(M):
    shape = wl.SHAPES["mini"]
    W = wl.SyntheticWeights(shape, seed=3, cache=True)
    model = M.Model(shape, W, max_rows=64, max_requests=1, max_positions=512, view8=True)
    yield shape, W, model
    model.close()


def _np(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("rare,perm", [(0, False), (40, True)])
def test_device_plane_equals_host_plane(M, rare, perm):
    from speculative_decoding_tree_bit_gb300 import check, lib
    N, K = 256, 512
    W = synthetic.normal_bf16(synthetic.key(81, rare), N * K, 0.02).reshape(N, K)
    if rare:
        synthetic.force_rare_exponents(synthetic.key(82, 1), W, rare)
    row_src = np.random.default_rng(rare).permutation(N).astype(np.int32) if perm else None
    p = M.pack(M.to_device_u16(W), row_src, view8=True)
    table = np.zeros(16, np.uint8)
    table[:p.meta.n_table] = p.table
    Wp = W[row_src] if perm else W
    host = np.zeros(N * K // 4, np.uint32)
    check(lib().w12_plane8_pack_host(np.ascontiguousarray(Wp).ctypes.data, N, K, table.ctypes.data, p.meta.n_table,
                                     host.ctypes.data))
    assert np.array_equal(_np(p.plane8).view(np.uint32), host)


def test_round_one_matches_the_oracle_view(M, mdl):
    shape, W, model = mdl
    ctx = 60
    td = wl.draft(91, 0, 16, 6, 0.8, shape.V)
    tokens = oracle_copy_tokens(shape, W, 3, 0, ctx, td)
    req = oracle_request(shape, 3, 0, ctx, tokens, td.parents, cap=ctx + 80)
    low = oracle.forward(shape, oracle.View8Weights(W), [req])
    exact = oracle.forward(shape, W, [req])
    kv = M.KVCache(shape, ctx + 80).fill(3, ctx)
    lg, am = model.forward_view8(tokens, td.parents, kv)
    torch.cuda.synchronize()
    assert model.status() == 0 and int(kv.ctx_len[0]) == ctx  # nothing committed
    assert_close(_np(lg), low.logits)
    # the lm_head over the step's own final hidden state, through the view
    am_h = _view8_tap(model, W, len(tokens), lg, am)
    assert_argmax(_np(am), low.argmax, low.margin, tap_am=am_h)
    # the view really differs from the exact weights (else the test shows nothing)
    assert np.abs(low.logits - exact.logits).max() > 1e-3


def _view8_tap(model, W, rows, lg, am):
    """The oracle's lm_head (through the 8-bit view) over the step's own
    final hidden state: element-wise logits and the strict argmax rule;
    returns that argmax."""
    xf = model.final_hidden(rows).cpu().numpy().view(np.uint16)
    lg_h = oracle.linear(xf, oracle.w12_view8(W.lm_head()))
    am_h, margin_h = oracle.argmax_margin(lg_h)
    if lg is not None:
        assert_close(_np(lg), lg_h)
    assert_argmax(_np(am), am_h, margin_h)
    return am_h


def _extension(chain):
    """A drafter continuing from the chain's end: a small seeded tree (its
    tokens depend on the chain, as a drafter's would)."""
    rng = np.random.default_rng(int(chain.sum()) % 1000)
    par = np.array([-1, 0, -1, 2, 1], dtype=np.int64)  # parents local to the extension, -1: the chain's end
    return rng.integers(0, 4000, size=5).astype(np.int32), par


def test_two_level_verification_matches_the_oracle(M, mdl):
    from speculative_decoding_tree_bit_gb300 import check, lib
    shape, W, model = mdl
    for seed, (m, depth, ctx) in enumerate([(16, 6, 40), (12, 8, 90), (9, 4, 130)]):
        td = wl.draft(100 + seed, 0, m, depth, 0.8, shape.V)
        tokens = oracle_copy_tokens(shape, W, 3, 0, ctx, td)
        req = oracle_request(shape, 3, 0, ctx, tokens, td.parents, cap=ctx + 80)
        ref = oracle.two_level_verify(shape, W, req, _extension)
        kv = M.KVCache(shape, ctx + 80).fill(3, ctx)
        # round one: the 8-bit view, then its greedy walk gives the chain
        _, am = model.forward_view8(tokens, td.parents, kv, logits=False)
        torch.cuda.synchronize()
        assert int(kv.ctx_len[0]) == ctx
        low = oracle.forward(shape, oracle.View8Weights(W), [req])
        assert_argmax(_np(am), low.argmax, low.margin, tap_am=_view8_tap(model, W, m, None, am))
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).cuda()
        tok_d, par_d = dev(tokens), dev(td.parents)
        L, acc, bonus, st = (torch.zeros(n, dtype=torch.int32, device="cuda") for n in (1, m, 1, 1))
        check(lib().sd_accept(tok_d.data_ptr(), par_d.data_ptr(), am.data_ptr(), m, L.data_ptr(), acc.data_ptr(),
                              bonus.data_ptr(), None, st.data_ptr(), None))
        torch.cuda.synchronize()
        chain = np.array([int(tokens[0])] + [int(t) for t in _np(acc)[:int(L[0])]] + [int(bonus[0])], np.int32)
        if np.array_equal(_np(am), low.argmax):
            assert np.array_equal(chain, ref.chain)
        # exact round on the chain plus the drafter's extension
        ext_tok, ext_par = _extension(chain)
        n = len(chain)
        tok2 = np.concatenate([chain, ext_tok]).astype(np.int32)
        par2 = np.concatenate([np.arange(-1, n - 1), np.where(ext_par < 0, n - 1, ext_par + n)]).astype(np.int32)
        o = model.verify(tok2, par2, kv, logits=True)
        torch.cuda.synchronize()
        assert model.status() == 0
        exact = oracle.forward(shape, W, [oracle_request(shape, 3, 0, ctx, tok2, par2, cap=ctx + 80)])
        assert_close(_np(o["logits"]), exact.logits)
        tap = assert_final_hidden(model, o, W.lm_head(), len(tok2))
        am2 = _np(o["argmax"])
        assert_argmax(am2, exact.argmax, exact.margin, tap_am=tap)
        assert_accept(tok2, par2, am2, int(o["accepted_len"][0]), _np(o["accepted_tokens"]), int(o["bonus"][0]),
                      exact.argmax)
        if np.array_equal(chain, ref.chain) and np.array_equal(am2, exact.argmax):
            assert int(o["accepted_len"][0]) == ref.exact.accepted_len and int(o["bonus"][0]) == ref.exact.bonus
        assert int(kv.ctx_len[0]) == ctx + int(o["accepted_len"][0]) + 1
