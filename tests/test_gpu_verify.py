"""End-to-end verify step on the GPU vs the oracle: the tiny model, small
dense and hybrid decoders (several GEMM tiles, ragged row blocks), batched
paged verify, and the device-side error paths."""
import numpy as np
import pytest
import torch

import oracle
from synthetic import workloads as wl
from helpers import (assert_accept, assert_argmax, assert_close, assert_committed, assert_final_hidden,
                     oracle_copy_tokens, oracle_request,
                     sub_out)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from speculative_decoding_tree_bit_gb300 import model
    return model


def _np(t):
    return t.cpu().numpy()


# ------------------------------------------------------------------ tiny --

def test_tiny_verify(M):
    t = wl.tiny()
    lo = oracle.tiny_forward(t.W1, t.Wlm, t.act)
    am_o, margin = oracle.argmax_margin(lo)
    tokens = wl.copy_rule_tokens_static(t.draft, am_o)
    p1, p2 = M.pack(M.to_device_u16(t.W1)), M.pack(M.to_device_u16(t.Wlm))
    o = M.tiny_verify(p1, p2, M.to_device_u16(t.act), tokens, t.draft.parents)
    torch.cuda.synchronize()
    assert int(o["status"][0]) == 0
    assert_close(_np(o["logits"]), lo)
    am = _np(o["argmax"])
    assert_argmax(am, am_o, margin)
    assert_accept(tokens, t.draft.parents, am, int(o["accepted_len"][0]), _np(o["accepted_tokens"]),
                  int(o["bonus"][0]), am_o)
    assert int(o["accepted_len"][0]) >= 1


def test_tiny_rejects_bad_tree(M):
    t = wl.tiny()
    p1, p2 = M.pack(M.to_device_u16(t.W1)), M.pack(M.to_device_u16(t.Wlm))
    parents = t.draft.parents.copy()
    parents[3] = 5  # parent after child
    o = M.tiny_verify(p1, p2, M.to_device_u16(t.act), np.zeros(8, np.int32), parents)
    torch.cuda.synchronize()
    assert int(o["status"][0]) == 5 and int(o["accepted_len"][0]) == 0


# ------------------------------------------------------------ decoders --

@pytest.fixture(scope="module", params=["mini", "mini_hybrid"])
def dec(request, M):
    shape = wl.SHAPES[request.param]
    W = wl.SyntheticWeights(shape, seed=3, cache=True)
    model = M.Model(shape, W, max_rows=64, max_requests=4, max_positions=512)
    yield shape, W, model
    model.close()


def _verify_case(M, shape, W, model, td, ctx, seed=3):
    tokens = oracle_copy_tokens(shape, W, seed, 0, ctx, td)
    req = oracle_request(shape, seed, 0, ctx, tokens, td.parents, cap=ctx + 80)
    out = oracle.forward(shape, W, [req])
    kv = M.KVCache(shape, ctx + 80).fill(seed, ctx)
    o = model.verify(tokens, td.parents, kv, logits=True)
    torch.cuda.synchronize()
    assert model.status() == 0
    assert_close(_np(o["logits"]), out.logits)
    tap = assert_final_hidden(model, o, W.lm_head(), len(tokens))
    am = _np(o["argmax"])
    assert_argmax(am, out.argmax, out.margin, tap_am=tap)
    path = assert_accept(tokens, td.parents, am, int(o["accepted_len"][0]), _np(o["accepted_tokens"]),
                         int(o["bonus"][0]), out.argmax)
    L = int(o["accepted_len"][0])
    assert int(kv.ctx_len[0]) == ctx + L + 1
    assert_committed(shape, req, out, path, ctx, kv, 0)
    return L


def test_tree_verify_matches_oracle(M, dec):
    shape, W, model = dec
    _verify_case(M, shape, W, model, wl.draft(11, 0, 16, 8, 0.8, shape.V), 37)


def test_tree_verify_on_tensor_core_gemms(M, dec):
    """Every GEMM of the step (fused QKV/RoPE/KV write, residual, SiLU-mul,
    logits + argmax epilogues) on the tcgen05 kernel."""
    shape, W, model = dec
    M.set_tc_min_rows(1)
    try:
        _verify_case(M, shape, W, model, wl.draft(11, 0, 16, 8, 0.8, shape.V), 37)
        _verify_case(M, shape, W, model, wl.draft(12, 0, 64, 10, 0.7, shape.V), 130)
    finally:
        M.set_tc_min_rows(0)


def test_tree_verify_on_the_fused_schedule(M, dec):
    """The linears between two attention (or recurrence) kernels as one
    launch of four dependent GEMMs with the RMSNorms folded in: trees of 1,
    16 and 64 nodes, and a batch of paged requests."""
    shape, W, model = dec
    model.set_fused(True)
    M.set_tc_min_rows(65)  # every step of at most 64 rows on the fused schedule
    try:
        _verify_case(M, shape, W, model, wl.draft(11, 0, 16, 8, 0.8, shape.V), 37)
        _verify_case(M, shape, W, model, wl.draft(12, 0, 64, 10, 0.7, shape.V), 130)
        assert _verify_case(M, shape, W, model, wl.draft(13, 0, 1, 1, 0.7, shape.V), 300) == 0
        test_batched_paged_equals_oracle(M, dec)
    finally:
        model.set_fused(False)
        M.set_tc_min_rows(0)


@pytest.mark.parametrize("splits", [1, 3, 64])
def test_tree_verify_with_fixed_attention_splits(M, dec, splits):
    """One prefix split (no merge across CTAs), an odd count whose last
    split is ragged, and the maximum (most splits empty at this context)."""
    shape, W, model = dec
    assert M.set_attn_splits(splits) == splits
    try:
        _verify_case(M, shape, W, model, wl.draft(14, 0, 16, 8, 0.8, shape.V), 200)
        _verify_case(M, shape, W, model, wl.draft(15, 0, 5, 3, 0.7, shape.V), 61)
        test_batched_paged_equals_oracle(M, dec)
    finally:
        assert M.set_attn_splits(0) == 0


def test_wide_tree_64_nodes(M, dec):
    shape, W, model = dec
    _verify_case(M, shape, W, model, wl.draft(12, 0, 64, 10, 0.7, shape.V), 130)


def test_single_node_and_long_context(M, dec):
    shape, W, model = dec
    assert _verify_case(M, shape, W, model, wl.draft(13, 0, 1, 1, 0.7, shape.V), 300) == 0


def test_chain_equals_sequential_on_gpu(M, dec):
    shape, W, model = dec
    ctx, n = 40, 6
    toks = np.random.default_rng(4).integers(0, shape.V, n).astype(np.int32)
    kv = M.KVCache(shape, ctx + 80).fill(3, ctx)
    lg_chain, _ = model.forward(toks, np.arange(-1, n - 1), kv)
    kv2 = M.KVCache(shape, ctx + 80).fill(3, ctx)
    for i in range(n):
        # a one-node verify accepts nothing and commits that node (ctx += 1)
        o = model.verify(toks[i:i + 1], [-1], kv2, logits=True)
        torch.cuda.synchronize()
        assert_close(_np(o["logits"][0]), oracle.bf16_to_f64(_np(lg_chain[i]).view(np.uint16)))
    assert int(kv2.ctx_len[0]) == ctx + n


def test_batched_paged_equals_oracle(M, dec):
    shape, W, model = dec
    ctxs = [23, 61, 40]
    drafts = [wl.draft(20 + r, r, m, 5, 0.8, shape.V) for r, m in enumerate([5, 9, 1])]
    toks = [oracle_copy_tokens(shape, W, 3, r, ctxs[r], td) for r, td in enumerate(drafts)]
    reqs = [oracle_request(shape, 3, r, ctxs[r], toks[r], drafts[r].parents, cap=ctxs[r] + 32) for r in range(3)]
    out = oracle.forward(shape, W, reqs)
    table, n_pages = wl.page_tables(7, ctxs, 16, 16)
    kv = M.PagedKVCache(shape, table, n_pages, 16).fill(3, ctxs)
    cu = np.cumsum([0] + [len(t) for t in toks])
    o = model.verify_batch(np.concatenate(toks), np.concatenate([d.parents for d in drafts]), cu, kv, logits=True)
    torch.cuda.synchronize()
    assert model.status() == 0
    assert_close(_np(o["logits"]), out.logits)
    tap = assert_final_hidden(model, o, W.lm_head(), int(cu[-1]))
    am = _np(o["argmax"])
    assert_argmax(am, out.argmax, out.margin, tap_am=tap)
    for r in range(3):
        a, b = cu[r], cu[r + 1]
        path = assert_accept(toks[r], drafts[r].parents, am[a:b], int(o["accepted_len"][r]),
                             _np(o["accepted_tokens"][a:b]), int(o["bonus"][r]), out.argmax[a:b])
        assert int(kv.ctx_len[r]) == ctxs[r] + int(o["accepted_len"][r]) + 1
        assert_committed(shape, reqs[r], sub_out(out, a, b), path, ctxs[r], kv, r)


def test_batched_paged_on_tensor_core_gemms(M, dec):
    M.set_tc_min_rows(1)
    try:
        test_batched_paged_equals_oracle(M, dec)
    finally:
        M.set_tc_min_rows(0)


def test_bad_inputs_set_status_and_commit_nothing(M, dec):
    shape, W, model = dec
    ctx = 30
    kv = M.KVCache(shape, ctx + 8).fill(3, ctx)
    model.verify([1, 2, 3], [-1, 0, 2], kv)  # parent[2] == 2
    assert model.status() == 5 and int(kv.ctx_len[0]) == ctx
    model.verify([1, shape.V, 3], [-1, 0, 0], kv)  # token out of range
    assert model.status() == 8 and int(kv.ctx_len[0]) == ctx
    model.verify(list(range(9)), list(range(-1, 8)), kv)  # ctx + 9 > cap
    assert model.status() == 7 and int(kv.ctx_len[0]) == ctx
    o = model.verify([1, 2], [-1, 0], kv)  # still usable afterwards
    assert model.status() == 0 and int(kv.ctx_len[0]) == ctx + int(o["accepted_len"][0]) + 1


def test_graph_capture_and_replay_match_direct_launches(M, dec):
    """A step captured into a CUDA graph (first call on a side stream) and its
    replays give the same bits as direct kernel launches."""
    shape, W, model = dec
    ctx = 50
    td = wl.draft(31, 0, 12, 5, 0.8, shape.V)
    tok = torch.from_numpy(np.random.default_rng(5).integers(0, shape.V, 12).astype(np.int32)).cuda()
    par = torch.from_numpy(td.parents.astype(np.int32)).cuda()
    kv = M.KVCache(shape, ctx + 80).fill(3, ctx)
    out = model.outputs(12, logits=True)
    s = torch.cuda.Stream()
    S0, z0 = kv.S.clone(), kv.z.clone()  # a step commits into the recurrent state
    results = []
    for graphs in (False, True, True, True):
        model.set_graphs(graphs)
        kv.ctx_len.fill_(ctx)
        kv.S.copy_(S0)
        kv.z.copy_(z0)
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            model.verify(tok, par, kv, out=out, stream=s)
        s.synchronize()
        assert model.status() == 0
        results.append({k: v.clone() for k, v in out.items()} | {"k": kv.k.clone(), "v": kv.v.clone(),
                                                                 "ctx": kv.ctx_len.clone()})
    model.set_graphs(True)
    for r in results[1:]:
        for k in r:
            assert torch.equal(r[k], results[0][k]), k


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("n", [5, 16, 64])
def test_repeated_steps_give_identical_bits(M, dec, n, fused):
    """The streamed GEMMs' split row blocks are finished by whichever
    contributor arrives last (it changes from run to run), which sums the
    partials in CTA order: every run gives the same bits, on both
    schedules."""
    shape, W, model = dec
    model.set_fused(fused)
    M.set_tc_min_rows(65)
    try:
        _repeat(M, shape, W, model, n)
    finally:
        model.set_fused(False)
        M.set_tc_min_rows(0)


def _repeat(M, shape, W, model, n):
    ctx = 45
    td = wl.draft(40 + n, 0, n, 6, 0.8, shape.V)
    tok = np.random.default_rng(n).integers(0, shape.V, n).astype(np.int32)
    results = []
    for _ in range(3):
        kv = M.KVCache(shape, ctx + 80).fill(3, ctx)
        o = model.verify(tok, td.parents, kv, logits=True)
        torch.cuda.synchronize()
        assert model.status() == 0
        results.append({k: v.clone() for k, v in o.items()} | {"k": kv.k.clone(), "v": kv.v.clone(),
                                                               "S": kv.S.clone(), "ctx": kv.ctx_len.clone()})
    for r in results[1:]:
        for k in r:
            assert torch.equal(r[k], results[0][k]), k
