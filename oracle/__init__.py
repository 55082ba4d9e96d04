"""ORACLE -- test infrastructure only.

A plain, slow CPU implementation of the tree-verification step, written from
the SpecPilot pages' description and the synthetic model definitions, in
fp64 with bf16 rounding at every kernel boundary of the model definition.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the CUDA library and the
product path never calls it.

Sources followed (page title, section):
  * "SpecPilot: AI Agent Framework Boosts Speculative Decoding 10.87x ...",
    "(1) W12: Lossless 12-bit Weight Format" -- 12-bit code, exponent table,
    sparse escape list, bit-exact restoration (``w12_*``; C in oracle.c).
  * same page, "(2) Best-first Tree Verification for Hybrid Architectures" --
    the target scores every node of a draft tree in one pass, each node seeing
    its root path (``tree_info``, ``tree_attention``), and a recurrent state
    that follows each root path (``linrec_literal``).
  * same page, "(3) Two-Level Verification" and "SpecPilot Uses Agentic
    Discovery ...", "Core Idea" (token forcing) -- only exact greedy target
    verification accepts tokens (``accept``).
  * "SpecPilot Uses Agentic Discovery ...", "Technical Mechanisms" -- a
    drafter proposes candidates, the target verifies them in parallel.
  * same page, "(3) Two-Level Verification": a first round over the nested
    8-bit weight view proposes a chain and accepts nothing, one exact round
    decides (``w12_view8``, ``View8Weights``, ``two_level_verify``).
  * same page, "(2) Best-first Tree Verification ...": Gated DeltaNet
    layers follow each root path of the tree (``gdn_tree``, the published
    gated delta rule).
  * same page, "(1) W12: Lossless 12-bit Weight Format", read literally: a
    4-bit exponent OFFSET from a base chosen per output channel (``w12c_*``;
    the per-tensor table above is the other reading).
  * "SpecPilot: AI Agent Framework ...", "(2) Best-first Tree Verification
    for Hybrid Architectures" (candidates ranked by parent-conditioned
    log-probability, highest cumulative path scores kept) and "(4) Three
    Batch Optimization Mechanisms", Shared Node Budget (requests share one
    node budget, given to the candidates of highest path probability) --
    ``path_scores``, ``best_first_select``.
The dense decoder itself (RMSNorm, RoPE, GQA, SwiGLU) is the synthetic
architecture the workloads name; the pages do not define it.

Where the pages are silent, each function's docstring states the reading it
takes (the arithmetic, the order of operations, the tie rules).

Parity pins for every function live in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + ".tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
            L.or_bf16_to_double.restype = ctypes.c_double
            L.or_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.or_double_to_bf16.restype = ctypes.c_uint16
            L.or_double_to_bf16.argtypes = [ctypes.c_double]
            L.or_round_bf16.restype = None
            L.or_round_bf16.argtypes = [vp, i64, vp]
            L.or_bf16_to_f64.restype = None
            L.or_bf16_to_f64.argtypes = [vp, i64, vp]
            L.or_w12_histogram.restype = None
            L.or_w12_histogram.argtypes = [vp, i64, vp]
            L.or_w12_table.restype = ctypes.c_int
            L.or_w12_table.argtypes = [vp, vp]
            L.or_w12_count_escapes.restype = i64
            L.or_w12_count_escapes.argtypes = [vp, i64, vp, ctypes.c_int]
            L.or_w12_pack.restype = i64
            L.or_w12_pack.argtypes = [vp, i64, i64, vp, ctypes.c_int, vp, vp, vp, i64, vp]
            L.or_w12_unpack.restype = ctypes.c_int
            L.or_w12_unpack.argtypes = [vp, i64, i64, vp, ctypes.c_int, vp, vp, i64, vp]
            L.or_w12_field.restype = ctypes.c_uint32
            L.or_w12_field.argtypes = [vp, i64, i64, i64]
            L.or_linear.restype = None
            L.or_linear.argtypes = [vp, i64, i64, vp, i64, vp]
            _lib = L
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ bf16 --

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns."""
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().or_bf16_to_f64(b.ctypes.data, b.size, out.ctypes.data)
    return out


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (nearest, ties to even); returns bit patterns."""
    a = _c(x, np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    lib().or_round_bf16(a.ctypes.data, a.size, out.ctypes.data)
    return out


# ------------------------------------------------------------------- W12 --

@dataclass
class W12:
    """A packed tensor in the W12 layout described in oracle.c."""
    N: int
    K: int
    table: np.ndarray      # uint8 [n_table] ascending exponents
    words: np.ndarray      # uint32 [N*K*3/8]
    esc_idx: np.ndarray    # uint32 [n_esc], increasing flat index
    esc_val: np.ndarray    # uint16 [n_esc], bf16 bits
    row_ptr: np.ndarray    # uint32 [N+1]

    @property
    def n_table(self) -> int:
        return int(self.table.size)

    @property
    def n_esc(self) -> int:
        return int(self.esc_idx.size)


def w12_histogram(w: np.ndarray) -> np.ndarray:
    a = _c(w, np.uint16)
    h = np.zeros(256, dtype=np.uint64)
    lib().or_w12_histogram(a.ctypes.data, a.size, h.ctypes.data)
    return h


def w12_table(hist: np.ndarray) -> np.ndarray:
    """The 15 most frequent exponents (ties -> smaller exponent), ascending."""
    h = _c(hist, np.uint64)
    t = np.zeros(16, dtype=np.uint8)
    n = lib().or_w12_table(h.ctypes.data, t.ctypes.data)
    return t[:n].copy()


def w12_pack(W: np.ndarray, table: np.ndarray | None = None) -> W12:
    W = _c(W, np.uint16)
    N, K = W.shape
    if table is None:
        table = w12_table(w12_histogram(W))
    t16 = np.zeros(16, dtype=np.uint8)
    t16[: table.size] = table
    n_esc = int(lib().or_w12_count_escapes(W.ctypes.data, W.size, t16.ctypes.data, int(table.size)))
    words = np.empty(N * K * 3 // 8, dtype=np.uint32)
    esc_idx = np.empty(max(n_esc, 1), dtype=np.uint32)
    esc_val = np.empty(max(n_esc, 1), dtype=np.uint16)
    row_ptr = np.empty(N + 1, dtype=np.uint32)
    got = lib().or_w12_pack(W.ctypes.data, N, K, t16.ctypes.data, int(table.size), words.ctypes.data,
                            esc_idx.ctypes.data, esc_val.ctypes.data, max(n_esc, 1), row_ptr.ctypes.data)
    if got < 0:
        raise ValueError(f"w12_pack failed ({got}) for shape {W.shape}")
    assert got == n_esc
    return W12(N, K, table.astype(np.uint8).copy(), words, esc_idx[:n_esc].copy(), esc_val[:n_esc].copy(), row_ptr)


def w12_unpack(p: W12) -> np.ndarray:
    W = np.empty((p.N, p.K), dtype=np.uint16)
    t16 = np.zeros(16, dtype=np.uint8)
    t16[: p.n_table] = p.table
    ei = _c(p.esc_idx if p.n_esc else np.zeros(1, np.uint32), np.uint32)
    ev = _c(p.esc_val if p.n_esc else np.zeros(1, np.uint16), np.uint16)
    rc = lib().or_w12_unpack(_c(p.words, np.uint32).ctypes.data, p.N, p.K, t16.ctypes.data, p.n_table,
                             ei.ctypes.data, ev.ctypes.data, p.n_esc, W.ctypes.data)
    if rc != 0:
        raise ValueError("w12_unpack: bad shape")
    return W


def w12_field(p: W12, n: int, k: int) -> int:
    """The stored 12-bit field (sign<<11 | code<<7 | mantissa) of weight (n, k)."""
    w = _c(p.words, np.uint32)
    return int(lib().or_w12_field(w.ctypes.data, n, k, p.K))


# ---------------------------------------------------------------- linear --

def linear(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """y = x W^T in fp64, each output summed in k order.  x: fp64 [M][K]
    (or bf16 bits, converted exactly), W: bf16 bits [N][K]."""
    if x.dtype == np.uint16:
        x = bf16_to_f64(x)
    x = _c(x, np.float64)
    W = _c(W, np.uint16)
    M, K = x.shape
    N, K2 = W.shape
    assert K == K2
    y = np.empty((M, N), dtype=np.float64)
    if M and N:
        lib().or_linear(x.ctypes.data, M, K, W.ctypes.data, N, y.ctypes.data)
    return y


def linear_bf16(x: np.ndarray, W: np.ndarray, gemm=None) -> np.ndarray:
    """A GEMM kernel boundary: bf16(x W^T)."""
    return round_bf16((gemm or linear)(x, W))


def linear_f32(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """y = x W^T with every product and sum in fp32 (the products of two bf16
    values are exact in fp32; the summation order is numpy's).  Not part of
    the definition: the fp32-accumulation twin of ``linear``, used to measure
    how far an implementation that sums in fp32 (as the workloads' rule
    allows) may move from the fp64 oracle through the bf16 rounding points
    downstream."""
    if x.dtype == np.uint16:
        x = bf16_to_f64(x)
    xf = np.asarray(x, dtype=np.float32)
    Wf = bf16_to_f64(W).astype(np.float32)
    return (xf @ Wf.T).astype(np.float64)


# -------------------------------------------------------------- layers ----

def rmsnorm(x_bits: np.ndarray, gamma_bits: np.ndarray, eps: float) -> np.ndarray:
    """bf16( (x / sqrt(mean(x^2) + eps)) * gamma ), row-wise."""
    x = bf16_to_f64(x_bits)
    g = bf16_to_f64(gamma_bits)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return round_bf16((x * r) * g)


def rope_angles(positions: np.ndarray, hd: int, base: float) -> np.ndarray:
    """theta[m][d] = pos[m] * base^(-2d/hd), d < hd/2 (rotate-half pairing d, d+hd/2)."""
    d = np.arange(hd // 2, dtype=np.float64)
    inv = base ** (-2.0 * d / hd)
    return np.asarray(positions, dtype=np.float64)[:, None] * inv[None, :]


def rope(x_bits: np.ndarray, positions: np.ndarray, base: float) -> np.ndarray:
    """Rotate-half RoPE of x [M][nh][hd] at per-row positions; bf16 out."""
    x = bf16_to_f64(x_bits)
    hd = x.shape[-1]
    th = rope_angles(positions, hd, base)[:, None, :]
    c, s = np.cos(th), np.sin(th)
    a, b = x[..., : hd // 2], x[..., hd // 2:]
    return round_bf16(np.concatenate([a * c - b * s, b * c + a * s], axis=-1))


def silu_mul(g_bits: np.ndarray, u_bits: np.ndarray) -> np.ndarray:
    g = bf16_to_f64(g_bits)
    u = bf16_to_f64(u_bits)
    return round_bf16(g / (1.0 + np.exp(-g)) * u)


def residual(x_bits: np.ndarray, y_bits: np.ndarray) -> np.ndarray:
    return round_bf16(bf16_to_f64(x_bits) + bf16_to_f64(y_bits))


# ------------------------------------------------------------------ tree --

@dataclass
class TreeInfo:
    valid: bool
    depth: np.ndarray   # int32 [M]
    anc: np.ndarray     # bool [M][M]; anc[i][j] = j is i or an ancestor of i


def tree_info(parents: np.ndarray) -> TreeInfo:
    """Validate a parent array (root at 0 with parent -1, parent[i] < i) and
    derive depths and ancestor sets."""
    p = np.asarray(parents, dtype=np.int64)
    M = p.size
    valid = M >= 1 and p[0] == -1 and all(0 <= p[i] < i for i in range(1, M))
    depth = np.zeros(M, dtype=np.int32)
    anc = np.zeros((M, M), dtype=bool)
    if valid:
        for i in range(M):
            j = i
            while j >= 0:
                anc[i, j] = True
                j = p[j]
            depth[i] = anc[i].sum() - 1
    return TreeInfo(bool(valid), depth, anc)


def tree_attention(q_bits, k_prefix_bits, v_prefix_bits, k_new_bits, v_new_bits, anc, ctx):
    """Tree-masked GQA attention, softmax in fp64, bf16 out.

    q: [M][Hq][hd]; k/v prefix: [Hkv][>=ctx][hd] (first ctx used);
    k/v new: [M][Hkv][hd] (node j's key/value); anc: [M][M] bool.
    Node i attends to every prefix position and to the nodes j with
    anc[i][j] (its root path, itself included).  q head h reads kv head
    h // (Hq/Hkv).  Scores are q.k / sqrt(hd)."""
    q = bf16_to_f64(q_bits)
    M, Hq, hd = q.shape
    Hkv = k_new_bits.shape[1]
    G = Hq // Hkv
    kp = bf16_to_f64(k_prefix_bits[:, :ctx])
    vp = bf16_to_f64(v_prefix_bits[:, :ctx])
    kn = bf16_to_f64(k_new_bits)
    vn = bf16_to_f64(v_new_bits)
    out = np.empty((M, Hq, hd), dtype=np.float64)
    scale = 1.0 / np.sqrt(hd)
    for h in range(Hq):
        g = h // G
        keys = np.concatenate([kp[g], kn[:, g, :]], axis=0)      # [ctx+M][hd]
        vals = np.concatenate([vp[g], vn[:, g, :]], axis=0)
        s = (q[:, h, :] @ keys.T) * scale                          # [M][ctx+M]
        mask = np.concatenate([np.ones((M, ctx), dtype=bool), anc], axis=1)
        s = np.where(mask, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        e = np.exp(s)
        pr = e / e.sum(axis=1, keepdims=True)
        out[:, h, :] = pr @ vals
    return round_bf16(out)


def phi(x: np.ndarray) -> np.ndarray:
    """Feature map of the linear-recurrent layer: elu(x) + 1."""
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def linrec_literal(q_bits, k_bits, v_bits, S0, z0, parents, eps):
    """Tree linear recurrence, literal per-node state.

    Per head: S_i = S_parent(i) + phi(k_i) v_i^T, z_i = z_parent(i) + phi(k_i),
    with (S0, z0) the state before the root; output
    o_i = S_i^T phi(q_i) / (z_i . phi(q_i) + eps), rounded to bf16.
    q/k/v: bf16 [M][nh][hd]; S0: [nh][hd][hd] (row = key dim, column = value
    dim); z0: [nh][hd].  Returns (o bits [M][nh][hd], S nodes [M][nh][hd][hd],
    z nodes [M][nh][hd])."""
    q = phi(bf16_to_f64(q_bits))
    k = phi(bf16_to_f64(k_bits))
    v = bf16_to_f64(v_bits)
    S0 = np.asarray(S0, dtype=np.float64)
    z0 = np.asarray(z0, dtype=np.float64)
    M, nh, hd = q.shape
    S = np.empty((M, nh, hd, hd))
    z = np.empty((M, nh, hd))
    o = np.empty((M, nh, hd))
    for i in range(M):
        Sp = S0 if parents[i] < 0 else S[parents[i]]
        zp = z0 if parents[i] < 0 else z[parents[i]]
        S[i] = Sp + k[i][:, :, None] * v[i][:, None, :]
        z[i] = zp + k[i]
        num = np.einsum("hab,ha->hb", S[i], q[i])
        den = np.einsum("ha,ha->h", z[i], q[i]) + eps
        o[i] = num / den[:, None]
    return round_bf16(o), S, z


def gdn_commit(S_nodes: np.ndarray, acc: "Accept") -> np.ndarray:
    """The committed state after a verify over a gated-delta-rule tree: the
    state of the deepest accepted node (the path root .. acc.last is what the
    sequence now holds), [nh][hd][hd]."""
    return S_nodes[acc.last].copy()


def l2_normalise(x: np.ndarray) -> np.ndarray:
    """x / ||x|| over the last axis (zero vectors stay zero)."""
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return np.where(n > 0, x / np.where(n > 0, n, 1.0), 0.0)


def gdn_tree(q_bits, k_bits, v_bits, alpha, beta, S0, parents):
    """Gated delta rule over a draft tree, literal per-node state ("(2)
    Best-first Tree Verification for Hybrid Architectures": in Gated
    DeltaNet layers the state is recomputed along each root path; the page
    names the layer without writing its recurrence, which is the published
    gated delta rule).

    Per head, with q and k L2-normalised:
      S_i = alpha_i (I - beta_i k_i k_i^T) S_parent(i) + beta_i k_i v_i^T
      o_i = S_i^T q_i, rounded to bf16,
    S0 the committed state before the root (row = key dim, column = value
    dim).  q/k/v: bf16 [M][nh][hd]; alpha (gate, in (0, 1]) and beta
    (write strength, in [0, 1]): [M][nh]; S0: [nh][hd][hd].  Returns
    (o bits [M][nh][hd], S nodes [M][nh][hd][hd])."""
    q = l2_normalise(bf16_to_f64(q_bits))
    k = l2_normalise(bf16_to_f64(k_bits))
    v = bf16_to_f64(v_bits)
    a = np.asarray(alpha, dtype=np.float64)
    b = np.asarray(beta, dtype=np.float64)
    S0 = np.asarray(S0, dtype=np.float64)
    M, nh, hd = q.shape
    S = np.empty((M, nh, hd, hd))
    o = np.empty((M, nh, hd))
    for i in range(M):
        Sp = S0 if parents[i] < 0 else S[parents[i]]
        for h in range(nh):
            kk = k[i, h]
            # (I - beta k k^T) Sp = Sp - beta k (k^T Sp)
            S[i, h] = a[i, h] * (Sp[h] - b[i, h] * np.outer(kk, kk @ Sp[h])) + b[i, h] * np.outer(kk, v[i, h])
            o[i, h] = S[i, h].T @ q[i, h]
    return round_bf16(o), S


# -------------------------------------------------------- argmax / accept --

def argmax_margin(logits: np.ndarray):
    """Per row: index of the largest logit (smallest index on ties) and the
    gap between the largest and the second largest value."""
    idx = np.argmax(logits, axis=1).astype(np.int32)
    part = np.partition(logits, -2, axis=1)
    margin = part[:, -1] - part[:, -2]
    return idx, margin


@dataclass
class Accept:
    accepted_len: int
    accepted_tokens: list
    bonus: int
    path: list          # node ids root .. deepest accepted node
    last: int           # deepest accepted node


def accept(tokens, parents, argmax) -> Accept:
    """Greedy longest accepted path.  Node i >= 1 matches when its token equals
    the target's argmax at its parent; a node is accepted when it and all its
    ancestors match (the root always is).  The deepest accepted node wins,
    the smallest index among equally deep ones.  The accepted tokens are the
    path's tokens below the root; the bonus is the target's argmax there."""
    M = len(parents)
    ti = tree_info(parents)
    ok = [False] * M
    ok[0] = True
    for i in range(1, M):
        ok[i] = ok[parents[i]] and int(tokens[i]) == int(argmax[parents[i]])
    best = 0
    for i in range(M):
        if ok[i] and ti.depth[i] > ti.depth[best]:
            best = i
    path = []
    j = best
    while j >= 0:
        path.append(j)
        j = parents[j]
    path.reverse()
    return Accept(int(ti.depth[best]), [int(tokens[j]) for j in path[1:]], int(argmax[best]), path, best)


# ----------------------------------------------------------------- model --

@dataclass
class LayerState:
    """Per-layer cache of one request: KV prefix (attention layers) or the
    recurrent state (linear-recurrent layers)."""
    k: np.ndarray | None = None    # bf16 bits [Hkv][cap][hd]
    v: np.ndarray | None = None
    S: np.ndarray | None = None    # fp64 [nh][hd][hd]
    z: np.ndarray | None = None    # fp64 [nh][hd]


@dataclass
class Request:
    tokens: np.ndarray             # int32 [M]
    parents: np.ndarray            # int32 [M]
    ctx: int
    layers: list = field(default_factory=list)   # list[LayerState]


@dataclass
class ForwardOut:
    logits: np.ndarray             # fp64 [sum M][V]
    argmax: np.ndarray
    margin: np.ndarray
    new_kv: list                   # per layer: (k bits [M][Hkv][hd], v bits) or (phi k, v) rows
    infos: list                    # TreeInfo per request


def forward(shape, weights, requests: list, n_layers: int | None = None, gemm=None) -> ForwardOut:
    """One verify forward over the draft trees of all requests.

    Every GEMM sees the rows of all requests together (rows never interact);
    attention and recurrence act per request.  Layer order (pre-norm):
      h = x + O(mix(RMSNorm(x)));  x' = h + down(silu(gate(n)) * up(n)), n = RMSNorm(h)
    with mix = tree attention (RoPE on q,k at position ctx + depth) or the
    tree linear recurrence.  Final RMSNorm then lm_head.  ``n_layers`` runs
    only the first layers (a bounded sample for timing); ``gemm`` replaces
    ``linear`` in every GEMM (``linear_f32``: the fp32-accumulation twin)."""
    gemm = gemm or linear
    hd, Hq, Hkv, eps = shape.hd, shape.Hq, shape.Hkv, shape.eps
    infos = [tree_info(r.parents) for r in requests]
    for inf in infos:
        if not inf.valid:
            raise ValueError("invalid parent array")
    seg = np.cumsum([0] + [len(r.tokens) for r in requests])
    tokens = np.concatenate([np.asarray(r.tokens, dtype=np.int64) for r in requests])
    Mt = tokens.size
    x = weights.embed_rows(tokens)                                      # bf16 [Mt][H]
    pos = np.concatenate([r.ctx + inf.depth for r, inf in zip(requests, infos)])
    new_kv = []
    kinds = shape.layer_kinds if n_layers is None else shape.layer_kinds[:n_layers]
    for l, kind in enumerate(kinds):
        xn = rmsnorm(x, weights.norm(l, "attn"), eps)
        if kind == "attn":
            q = linear_bf16(xn, weights.layer(l, "wq"), gemm).reshape(Mt, Hq, hd)
            k = linear_bf16(xn, weights.layer(l, "wk"), gemm).reshape(Mt, Hkv, hd)
            v = linear_bf16(xn, weights.layer(l, "wv"), gemm).reshape(Mt, Hkv, hd)
            q = rope(q, pos, shape.rope_base)
            k = rope(k, pos, shape.rope_base)
            att = np.empty((Mt, Hq, hd), dtype=np.uint16)
            for r, req in enumerate(requests):
                a, b = seg[r], seg[r + 1]
                st = req.layers[l]
                att[a:b] = tree_attention(q[a:b], st.k, st.v, k[a:b], v[a:b], infos[r].anc, req.ctx)
            new_kv.append((k, v))
        else:
            nh = shape.H // hd
            q = linear_bf16(xn, weights.layer(l, "wq"), gemm).reshape(Mt, nh, hd)
            k = linear_bf16(xn, weights.layer(l, "wk"), gemm).reshape(Mt, nh, hd)
            v = linear_bf16(xn, weights.layer(l, "wv"), gemm).reshape(Mt, nh, hd)
            att = np.empty((Mt, nh, hd), dtype=np.uint16)
            for r, req in enumerate(requests):
                a, b = seg[r], seg[r + 1]
                st = req.layers[l]
                att[a:b], _, _ = linrec_literal(q[a:b], k[a:b], v[a:b], st.S, st.z, req.parents, shape.rec_eps)
            new_kv.append((k, v))
        o = linear_bf16(att.reshape(Mt, -1), weights.layer(l, "wo"), gemm)
        h = residual(x, o)
        hn = rmsnorm(h, weights.norm(l, "mlp"), eps)
        g = linear_bf16(hn, weights.layer(l, "w_gate"), gemm)
        u = linear_bf16(hn, weights.layer(l, "w_up"), gemm)
        a_ = silu_mul(g, u)
        d = linear_bf16(a_, weights.layer(l, "w_down"), gemm)
        x = residual(h, d)
    xf = rmsnorm(x, weights.final_norm(), eps)
    logits = gemm(xf, weights.lm_head())
    idx, margin = argmax_margin(logits)
    return ForwardOut(logits, idx, margin, new_kv, infos)


def commit(shape, requests: list, out: ForwardOut, accepts: list) -> list:
    """State after acceptance, per request: for attention layers the K/V of
    the root and the accepted path nodes land at positions ctx + depth (the
    prefix grows by accepted_len + 1); for recurrent layers the state becomes
    the accepted node's state (root path included).  Returns new Requests
    with ctx advanced (tokens/parents left empty)."""
    seg = np.cumsum([0] + [len(r.tokens) for r in requests])
    res = []
    for r, (req, acc) in enumerate(zip(requests, accepts)):
        a = seg[r]
        layers = []
        for l, kind in enumerate(shape.layer_kinds):
            st = req.layers[l]
            kk, vv = out.new_kv[l]
            if kind == "attn":
                K = st.k.copy()
                V = st.v.copy()
                for d, node in enumerate(acc.path):
                    K[:, req.ctx + d, :] = kk[a + node]
                    V[:, req.ctx + d, :] = vv[a + node]
                layers.append(LayerState(k=K, v=V))
            else:
                S = np.asarray(st.S, dtype=np.float64).copy()
                z = np.asarray(st.z, dtype=np.float64).copy()
                kf = phi(bf16_to_f64(kk))
                vf = bf16_to_f64(vv)
                for node in acc.path:
                    S += kf[a + node][:, :, None] * vf[a + node][:, None, :]
                    z += kf[a + node]
                layers.append(LayerState(S=S, z=z))
        res.append(Request(np.zeros(0, np.int32), np.zeros(0, np.int32), req.ctx + acc.accepted_len + 1, layers))
    return res


def verify(shape, weights, requests: list):
    """forward + greedy acceptance per request + committed state."""
    out = forward(shape, weights, requests)
    seg = np.cumsum([0] + [len(r.tokens) for r in requests])
    accepts = [accept(req.tokens, req.parents, out.argmax[seg[i]:seg[i + 1]]) for i, req in enumerate(requests)]
    return out, accepts, commit(shape, requests, out, accepts)


def tiny_forward(W1, Wlm, act_bits):
    """Tiny verify model: y = bf16(a W1^T), logits = y Wlm^T (fp64)."""
    y = linear_bf16(act_bits, W1)
    return linear(y, Wlm)


# ------------------------------------------------- best-first selection --

SELECT_BAD_TREE = 5  # the library's SD_ERR_BAD_TREE


@dataclass
class Selection:
    cu: np.ndarray       # int32 [R+1]: request r's selected nodes are cu[r] .. cu[r+1]-1
    src: np.ndarray      # int32 [total]: global candidate index of each selected node
    parents: np.ndarray  # int32 [total]: parent among the request's selected nodes (-1 at the root)
    scores: np.ndarray   # float32 [total]: path score of each selected node
    status: int          # 0, or SELECT_BAD_TREE when some request's input was invalid


def path_scores(parents, logprob) -> np.ndarray:
    """Path score of every candidate of one request ("(2) Best-first Tree
    Verification ...": cumulative score of the parent-conditioned
    log-probabilities along the root path).  The root scores 0; node i
    scores its parent's score plus logprob[i], one fp32 addition per node
    taken from the root down (the rounding the selection decides on)."""
    parents = np.asarray(parents)
    lp = np.asarray(logprob, dtype=np.float32)
    s = np.zeros(len(parents), dtype=np.float32)
    for i in range(1, len(parents)):
        s[i] = np.float32(s[parents[i]]) + lp[i]
    return s


def select_request_valid(parents, logprob) -> bool:
    """A request's candidates form a tree rooted at node 0 (parent[0] = -1,
    0 <= parent[i] < i) and every non-root log-probability is <= 0 (NaN and
    positive values are rejected)."""
    n = len(parents)
    if n < 1 or int(parents[0]) != -1:
        return False
    for i in range(1, n):
        if not (0 <= int(parents[i]) < i):
            return False
        if not (float(logprob[i]) <= 0.0):
            return False
    return True


def best_first_select(parents, logprob, cu, budget: int, cap: int) -> Selection:
    """Best-first node selection under a shared node budget ("(4) Three
    Batch Optimization Mechanisms", Shared Node Budget, with the ranking of
    "(2) Best-first Tree Verification ...").  Every request keeps its root
    (the node verification starts from).  The other candidates of all
    requests are then taken one at a time in order of path score, highest
    first, equal scores by lower request and then lower node index, passing
    over a candidate whose request already holds `cap` nodes, until `budget`
    nodes are held in total.  With log-probabilities <= 0 a node never
    scores above its parent, so the kept nodes of a request form a tree.
    Output per request in node-index order with parents renumbered.  A
    request with invalid input keeps nothing and sets the status."""
    parents = np.asarray(parents, dtype=np.int32)
    logprob = np.asarray(logprob, dtype=np.float32)
    cu = np.asarray(cu, dtype=np.int64)
    R = len(cu) - 1
    status = 0
    scores = np.zeros(len(parents), dtype=np.float32)
    order = []
    for r in range(R):
        a, b = int(cu[r]), int(cu[r + 1])
        if not select_request_valid(parents[a:b], logprob[a:b]):
            status = SELECT_BAD_TREE
            continue
        scores[a:b] = path_scores(parents[a:b], logprob[a:b])
        for i in range(b - a):
            g = a + i
            # roots first; then score, highest first; then global index
            order.append(((0 if i == 0 else 1), -float(scores[g]), g, r))
    order.sort(key=lambda t: (t[0], t[1], t[2]))
    taken = [[] for _ in range(R)]
    total = 0
    for _, _, g, r in order:
        if total >= budget:
            break
        if len(taken[r]) >= cap:
            continue
        taken[r].append(g)
        total += 1
    out_cu = np.zeros(R + 1, dtype=np.int32)
    src, par, sc = [], [], []
    for r in range(R):
        sel = sorted(taken[r])
        local = {g: j for j, g in enumerate(sel)}
        a = int(cu[r])
        for g in sel:
            src.append(g)
            p = int(parents[g])
            par.append(-1 if g == a else local[a + p])
            sc.append(scores[g])
        out_cu[r + 1] = out_cu[r] + len(sel)
    return Selection(out_cu, np.array(src, dtype=np.int32), np.array(par, dtype=np.int32),
                     np.array(sc, dtype=np.float32), status)


# -------------------------------------------- W12, per-channel exponent base --

@dataclass
class W12C:
    """Per-output-channel W12: row n stores each weight as sign, a 4-bit
    offset of its exponent from the row's base, and the 7-bit mantissa;
    offset 15 marks an escape whose original bf16 is in the side list."""
    N: int
    K: int
    base: np.ndarray     # uint8 [N]: the row's base exponent
    fields: np.ndarray   # uint16 [N][K]: sign << 11 | code << 7 | mantissa
    esc_idx: np.ndarray  # uint32: n * K + k of every escape, ascending
    esc_val: np.ndarray  # uint16: the escaped weights' bf16 bits

    @property
    def n_esc(self) -> int:
        return int(self.esc_idx.size)


def w12c_bases(W: np.ndarray) -> np.ndarray:
    """Per output row, the base exponent b (0..241) whose window b .. b+14
    holds the most of the row's exponents; ties go to the smaller b ("(1)
    W12 ...": exponents concentrate within each output channel, so one
    4-bit offset range per channel covers most of them)."""
    W = np.asarray(W, dtype=np.uint16)
    e = (W >> 7) & 0xFF
    out = np.zeros(W.shape[0], dtype=np.uint8)
    for n in range(W.shape[0]):
        h = np.bincount(e[n], minlength=256).astype(np.int64)
        c = np.concatenate([[0], np.cumsum(h)])
        cover = c[15:257] - c[0:242]  # cover[b] = weights with exponent in b .. b+14
        out[n] = int(np.argmax(cover))  # first maximum: the smaller base
    return out


def w12c_pack(W: np.ndarray, base: np.ndarray | None = None) -> W12C:
    """Fields and escapes of W (bf16 bits [N][K]) under the per-row bases."""
    W = np.asarray(W, dtype=np.uint16)
    N, K = W.shape
    if base is None:
        base = w12c_bases(W)
    base = np.asarray(base, dtype=np.uint8)
    e = ((W >> 7) & 0xFF).astype(np.int32)
    off = e - base.astype(np.int32)[:, None]
    inside = (off >= 0) & (off <= 14)
    code = np.where(inside, off, 15).astype(np.uint16)
    fields = ((W >> 15) << 11) | (code << 7) | (W & 0x7F)
    flat = np.flatnonzero(~inside.ravel()).astype(np.uint32)
    return W12C(N, K, base.copy(), fields.astype(np.uint16), flat, W.ravel()[flat].copy())


def w12c_unpack(p: W12C) -> np.ndarray:
    """The bf16 bits back: exponent = base + code for codes 0..14, the side
    list for code 15 (bit-exact restoration)."""
    f = p.fields.astype(np.uint32)
    code = (f >> 7) & 15
    e = (p.base.astype(np.uint32)[:, None] + code) & 0xFF
    W = (((f >> 11) & 1) << 15) | (e << 7) | (f & 0x7F)
    W = W.astype(np.uint16).ravel()
    W[p.esc_idx] = p.esc_val
    return W.reshape(p.N, p.K)


# ------------------------------------------------- two-level verification --

def w12_view8(W_bits) -> np.ndarray:
    """The nested 8-bit view of W12 weights ("(3) Two-Level Verification":
    the first round runs on W12's nested 8-bit weight view).  A weight's
    12-bit field is sign, 4-bit exponent code and 7-bit mantissa; its high
    byte keeps the sign, the code and the top 3 mantissa bits, so the view
    is the weight with its 4 low mantissa bits cleared (an escaped weight
    likewise, from the side list).  Truncates toward zero."""
    return np.asarray(W_bits, dtype=np.uint16) & np.uint16(0xFFF0)


class View8Weights:
    """A model's W12-stored linear weights (q/k/v, O, gate/up, down,
    lm_head) seen through the 8-bit view; the embedding and the norm
    weights are not W12 tensors and stay as they are."""

    def __init__(self, base):
        self.base = base

    def layer(self, l: int, name: str) -> np.ndarray:
        return w12_view8(self.base.layer(l, name))

    def lm_head(self) -> np.ndarray:
        return w12_view8(self.base.lm_head())

    def __getattr__(self, name):
        return getattr(self.base, name)


@dataclass
class TwoLevel:
    chain: np.ndarray    # int32: root token, the low-precision accepted path, its bonus token
    low: Accept          # the low-precision walk over the draft tree (accepts nothing)
    tokens: np.ndarray   # int32: the exact round's tree, the chain then the extension
    parents: np.ndarray  # int32
    exact: Accept        # the exact round's result: the only acceptance


def two_level_verify(shape, weights, request: Request, extend) -> TwoLevel:
    """Two-level verification ("(3) Two-Level Verification").  Round one
    runs the request's draft tree with the 8-bit weight view and walks it
    greedily: the path it would accept plus the token it would add form a
    candidate chain; nothing is accepted and no state changes.  The drafter
    then continues from the chain's end: ``extend(chain)`` returns (tokens,
    parents) of new drafts, parents local to them with -1 meaning the
    chain's last node.  One exact verification of the chain and the new
    drafts decides what is accepted, so the result is what exact greedy
    decoding would produce."""
    low_out = forward(shape, View8Weights(weights), [request])
    low = accept(request.tokens, request.parents, low_out.argmax)
    chain = np.array([int(request.tokens[0])] + [int(t) for t in low.accepted_tokens] + [int(low.bonus)],
                     dtype=np.int32)
    ext_tok, ext_par = extend(chain)
    ext_tok = np.asarray(ext_tok, dtype=np.int32)
    ext_par = np.asarray(ext_par, dtype=np.int64)
    n = len(chain)
    tokens = np.concatenate([chain, ext_tok]).astype(np.int32)
    parents = np.concatenate([np.arange(-1, n - 1), np.where(ext_par < 0, n - 1, ext_par + n)]).astype(np.int32)
    out = forward(shape, weights, [Request(tokens, parents, request.ctx, request.layers)])
    return TwoLevel(chain, low, tokens, parents, accept(tokens, parents, out.argmax))

