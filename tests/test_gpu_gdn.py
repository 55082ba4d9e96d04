"""Gated delta rule over draft trees on the GPU (sd_gdn_tree_verify,
sd_gdn_commit) against the oracle's node-by-node recurrence
(oracle.gdn_tree, oracle.gdn_commit): the WY form of the whole tree in one
solve must give every node's output and the accepted node's state.

Tolerances: outputs are bf16 (a kernel boundary): |gpu - oracle| <= 2^-7
|oracle| + 1e-4 (at most a one-ulp difference at the rounding point, fp32
against fp64 inside); the committed state is fp32: |gpu - oracle| <= 1e-5
(|oracle| + 1e-2)."""
import numpy as np
import pytest
import torch

import oracle
from synthetic import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from speculative_decoding_tree_bit_gb300 import model
    return model


def _dev(M, g):
    return (M.to_device_u16(g.q), M.to_device_u16(g.k), M.to_device_u16(g.v), torch.from_numpy(g.alpha).cuda(),
            torch.from_numpy(g.beta).cuda(), torch.from_numpy(np.ascontiguousarray(g.S)).cuda())


def _check_outputs(o_gpu, g):
    got = oracle.bf16_to_f64(o_gpu.cpu().numpy().view(np.uint16))
    states = []
    for r in range(len(g.cu) - 1):
        a, b = int(g.cu[r]), int(g.cu[r + 1])
        o_ref, S_nodes = oracle.gdn_tree(g.q[a:b], g.k[a:b], g.v[a:b], g.alpha[a:b], g.beta[a:b],
                                         g.S[r].astype(np.float64), g.parents[a:b])
        ref = oracle.bf16_to_f64(o_ref)
        err = np.abs(got[a:b] - ref)
        assert np.all(err <= 2.0 ** -7 * np.abs(ref) + 1e-4), float(err.max())
        states.append(S_nodes)
    return states


@pytest.mark.parametrize("Ms,depth,nh", [([16], 8, 4), ([1, 5, 64, 23], 10, 2), ([64], 64, 2), ([64] * 3, 4, 3)])
def test_outputs_and_commit_match_the_recurrence(M, Ms, depth, nh):
    """Trees of 1..64 nodes: a single node, a chain of 64 (depth 64), wide
    shallow trees, several requests of different sizes."""
    g = wl.gdn_inputs(len(Ms) * 7 + depth, Ms, depth, nh)
    q, k, v, al, be, S = _dev(M, g)
    layer = M.GdnLayer(int(g.cu[-1]), nh)
    o = layer.verify(q, k, v, al, be, g.parents, g.cu, S)
    torch.cuda.synchronize()
    assert int(layer.status[0]) == 0
    states = _check_outputs(o, g)
    # commit the deepest node of each request (the accept walk's output)
    last = []
    for r in range(len(Ms)):
        d = wl.depths(g.parents[g.cu[r]:g.cu[r + 1]])
        last.append(int(np.argmax(d)))
    layer.commit(last, S)
    torch.cuda.synchronize()
    got = S.cpu().numpy()
    for r in range(len(Ms)):
        acc = oracle.Accept(0, [], -1, [], last[r])
        ref = oracle.gdn_commit(states[r], acc)
        assert np.all(np.abs(got[r] - ref) <= 1e-5 * (np.abs(ref) + 1e-2)), float(np.abs(got[r] - ref).max())


def test_commit_of_a_rejected_request_keeps_the_state_and_bad_trees_are_flagged(M):
    g = wl.gdn_inputs(3, [6, 9], 4, 2)
    q, k, v, al, be, S = _dev(M, g)
    S_before = S.clone()
    layer = M.GdnLayer(15, 2)
    layer.verify(q, k, v, al, be, g.parents, g.cu, S)
    layer.commit([-1, 99], S)  # out of range: nothing moves
    torch.cuda.synchronize()
    assert torch.equal(S, S_before)
    par = g.parents.copy()
    par[8] = 8  # request 1, node 2: parent not before it
    layer.verify(q, k, v, al, be, par, g.cu, S)
    torch.cuda.synchronize()
    assert int(layer.status[0]) == 5


def test_no_write_keeps_the_state_exactly(M):
    """beta = 0, alpha = 1: every node reads the committed state; its commit
    is the identity (no fp32 rounding anywhere on that path)."""
    g = wl.gdn_inputs(4, [12], 5, 2)
    g.alpha[:] = 1.0
    g.beta[:] = 0.0
    q, k, v, al, be, S = _dev(M, g)
    S_before = S.clone()
    layer = M.GdnLayer(12, 2)
    o = layer.verify(q, k, v, al, be, g.parents, g.cu, S)
    layer.commit([11], S)
    torch.cuda.synchronize()
    assert torch.equal(S, S_before)
    _check_outputs(o, g)
