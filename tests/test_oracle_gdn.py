"""Pins of the oracle's gated delta rule over a draft tree ("SpecPilot: AI
Agent Framework Boosts Speculative Decoding 10.87x", "(2) Best-first Tree
Verification for Hybrid Architectures": Gated DeltaNet layers recompute the
state along each root path, and a WY-form kernel processes many paths at
once).  Pinned by the rule's special cases (no write, gate only, an exact
delta write), by the WY closed form of each root path computed with a
triangular solve, and by the independence of sibling branches."""
import numpy as np

import oracle
import synthetic

NH, HD = 2, 16


def _inputs(seed, M, max_depth, alpha_lo=0.6):
    parents = synthetic.tree(synthetic.key(seed, 1), M, max_depth)
    q, k, v = (synthetic.normal_bf16(synthetic.key(seed, 2 + j), M * NH * HD, 1.0).reshape(M, NH, HD)
               for j in range(3))
    u = synthetic.uniform_int(synthetic.key(seed, 5), 2 * M * NH, 0, 1 << 20).reshape(2, M, NH) / float(1 << 20)
    alpha = alpha_lo + (1 - alpha_lo) * u[0]
    beta = u[1]
    S0 = synthetic.normal_f32(synthetic.key(seed, 6), NH * HD * HD, 0.1).reshape(NH, HD, HD).astype(np.float64)
    return parents, q, k, v, alpha, beta, S0


def _path(parents, i):
    p = []
    while i >= 0:
        p.append(i)
        i = int(parents[i])
    return p[::-1]


def _wy_state(k, v, alpha, beta, S0):
    """State after the chain (k_t, v_t, alpha_t, beta_t), t = 1..L, from S0,
    in WY form: with G_t the product of alpha_1..alpha_t and
    A = (I + strict_lower(diag(beta) K K^T))^-1 diag(beta),
    S_L = G_L [(I - K^T A K) S0 + K^T A (V / G)]."""
    L = k.shape[0]
    G = np.cumprod(alpha)
    T = np.eye(L) + np.tril(beta[:, None] * (k @ k.T), -1)
    A = np.linalg.solve(T, np.diag(beta))
    W = A @ k
    U = A @ (v / G[:, None])
    return G[-1] * ((np.eye(k.shape[1]) - k.T @ W) @ S0 + k.T @ U)


def test_no_write_and_no_decay_keeps_the_state():
    parents, q, k, v, _, _, S0 = _inputs(1, 9, 4)
    o, S = oracle.gdn_tree(q, k, v, np.ones((9, NH)), np.zeros((9, NH)), S0, parents)
    for i in range(9):
        np.testing.assert_array_equal(S[i], S0)
    qn = oracle.l2_normalise(oracle.bf16_to_f64(q))
    np.testing.assert_array_equal(o, oracle.round_bf16(np.einsum("hab,mha->mhb", S0, qn)))


def test_gate_only_scales_by_the_path_product():
    parents, q, k, v, alpha, _, S0 = _inputs(2, 11, 5)
    _, S = oracle.gdn_tree(q, k, v, alpha, np.zeros((11, NH)), S0, parents)
    for i in range(11):
        g = np.prod([alpha[j] for j in _path(parents, i)], axis=0)
        np.testing.assert_allclose(S[i], g[:, None, None] * S0, rtol=1e-13, atol=0)


def test_full_write_stores_v_at_k():
    # alpha = beta = 1: the new state maps the node's (unit) key to its value exactly
    parents, q, k, v, _, _, S0 = _inputs(3, 10, 4)
    _, S = oracle.gdn_tree(q, k, v, np.ones((10, NH)), np.ones((10, NH)), S0, parents)
    kn = oracle.l2_normalise(oracle.bf16_to_f64(k))
    vv = oracle.bf16_to_f64(v)
    for i in range(10):
        for h in range(NH):
            np.testing.assert_allclose(S[i, h].T @ kn[i, h], vv[i, h], rtol=0, atol=1e-12)


def test_every_node_matches_the_wy_form_of_its_root_path():
    for seed in range(4):
        M = 14
        parents, q, k, v, alpha, beta, S0 = _inputs(10 + seed, M, 6)
        o, S = oracle.gdn_tree(q, k, v, alpha, beta, S0, parents)
        kn = oracle.l2_normalise(oracle.bf16_to_f64(k))
        vv = oracle.bf16_to_f64(v)
        qn = oracle.l2_normalise(oracle.bf16_to_f64(q))
        for i in range(M):
            p = _path(parents, i)
            for h in range(NH):
                ref = _wy_state(kn[p, h], vv[p, h], alpha[p, h], beta[p, h], S0[h])
                np.testing.assert_allclose(S[i, h], ref, rtol=1e-9, atol=1e-11)
                # the output is the state read at the unit query, rounded to bf16
                np.testing.assert_allclose(oracle.bf16_to_f64(o[i, h]), ref.T @ qn[i, h], rtol=2.0 ** -8, atol=1e-6)


def test_siblings_do_not_see_each_other():
    # a node's state depends on its root path only: the tree computed alone
    # on that path gives the same bits
    parents, q, k, v, alpha, beta, S0 = _inputs(5, 13, 5)
    _, S = oracle.gdn_tree(q, k, v, alpha, beta, S0, parents)
    for i in range(13):
        p = _path(parents, i)
        chain = np.arange(-1, len(p) - 1, dtype=np.int32)
        _, Sc = oracle.gdn_tree(q[p], k[p], v[p], alpha[p], beta[p], S0, chain)
        np.testing.assert_array_equal(Sc[-1], S[i])


def _wy_tree(parents, k, v, q, alpha, beta, S0):
    """Every node of a tree at once, in WY form: with the strict-ancestor
    mask A_ij (j a proper ancestor of i) and G_i the product of alpha over
    i's root path, one unit-lower-triangular solve
    T = I + A * (diag(beta) K K^T), W = T^-1 diag(beta) K, U = T^-1 diag(beta) (V / G),
    then S_i = G_i [S0 - sum_{j in path(i)} k_j (w_j^T S0 - u_j^T)] and
    o_i = G_i [S0^T q_i + sum_{j in path(i)} (k_j . q_i) (u_j - S0^T w_j)]."""
    M = len(parents)
    anc = np.zeros((M, M))
    for i in range(M):
        j = int(parents[i])
        while j >= 0:
            anc[i, j] = 1.0
            j = int(parents[j])
    path = anc + np.eye(M)
    G = np.array([np.prod(alpha[np.nonzero(path[i])[0]]) for i in range(M)])
    T = np.eye(M) + anc * (beta[:, None] * (k @ k.T))
    W = np.linalg.solve(T, beta[:, None] * k)
    U = np.linalg.solve(T, beta[:, None] * (v / G[:, None]))
    D = U - W @ S0                                   # rows: u_j - S0^T w_j
    o = G[:, None] * (q @ S0 + (path * (q @ k.T)) @ D)
    S = np.stack([G[i] * (S0 + k.T @ (path[i][:, None] * D)) for i in range(M)])
    return o, S


def test_whole_tree_in_one_masked_wy_solve():
    for seed in range(3):
        M = 16
        parents, q, k, v, alpha, beta, S0 = _inputs(20 + seed, M, 6)
        o_bits, S = oracle.gdn_tree(q, k, v, alpha, beta, S0, parents)
        kn = oracle.l2_normalise(oracle.bf16_to_f64(k))
        qn = oracle.l2_normalise(oracle.bf16_to_f64(q))
        vv = oracle.bf16_to_f64(v)
        for h in range(NH):
            o, Sw = _wy_tree(parents, kn[:, h], vv[:, h], qn[:, h], alpha[:, h], beta[:, h], S0[h])
            np.testing.assert_allclose(Sw, S[:, h], rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(oracle.bf16_to_f64(o_bits[:, h]), o, rtol=2.0 ** -8, atol=1e-6)


def test_commit_is_the_accepted_path_run_as_a_chain():
    # after acceptance the state is that of the deepest accepted node, the
    # same as running the rule over the accepted path alone
    parents, q, k, v, alpha, beta, S0 = _inputs(30, 12, 5)
    _, S = oracle.gdn_tree(q, k, v, alpha, beta, S0, parents)
    toks = np.arange(12, dtype=np.int32) + 100
    am = np.zeros(12, dtype=np.int32)
    leaf = 11
    path = _path(parents, leaf)
    for a, b in zip(path[:-1], path[1:]):  # the target agrees with the tokens along this path only
        am[a] = toks[b]
    acc = oracle.accept(toks, parents, am)
    assert acc.last == leaf and acc.path == path
    chain = np.arange(-1, len(path) - 1, dtype=np.int32)
    _, Sc = oracle.gdn_tree(q[path], k[path], v[path], alpha[path], beta[path], S0, chain)
    np.testing.assert_array_equal(oracle.gdn_commit(S, acc), Sc[-1])
