"""Workload recipes: model shapes, seeded weights, trees, caches, tokens.

Shared by the CUDA path's harness and by the tests that drive the oracle.
Everything is drawn from the counter-based streams of ``synthetic`` so any
tensor (or any row of one) can be regenerated on demand.  Nothing here
computes the verify method; the copy-rule token driver takes the target's
argmax from a caller-supplied function.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import (SID_ACT, SID_CAND_LP, SID_CAND_TOKEN, SID_CAND_TREE, SID_COINS, SID_CTX, SID_EMBED, SID_ESC,
               SID_GAMMA, SID_KV, SID_LM_HEAD, SID_PAGES, SID_ROOT_TOKEN, SID_STATE, SID_TINY_W1, SID_TREE, chain, copy_coins, force_rare_exponents, key,
               layer_key, normal_bf16, normal_f32, ones_bf16, permutation, tree, uniform_int)

WEIGHT_SLOTS = {"wq": 0, "wk": 1, "wv": 2, "wo": 3, "w_gate": 4, "w_up": 5, "w_down": 6, "attn": 7, "mlp": 8}
FINAL_NORM_LAYER = 4095


@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    H: int
    I: int
    Hq: int
    Hkv: int
    hd: int
    V: int
    layer_kinds: tuple          # "attn" | "rec" per layer
    eps: float = 1e-6
    rope_base: float = 1e6
    rec_eps: float = 1e-6
    sigma: float = 0.02
    gamma_sigma: float = 0.0    # 0 -> all norm weights are 1

    def weight_shape(self, l: int, name: str):
        H, I, hd = self.H, self.I, self.hd
        if self.layer_kinds[l] == "attn":
            qd, kvd = self.Hq * hd, self.Hkv * hd
        else:
            qd = kvd = H
        return {"wq": (qd, H), "wk": (kvd, H), "wv": (kvd, H), "wo": (H, qd),
                "w_gate": (I, H), "w_up": (I, H), "w_down": (H, I)}[name]

    @property
    def n_attn(self) -> int:
        return sum(k == "attn" for k in self.layer_kinds)

    @property
    def n_rec(self) -> int:
        return sum(k == "rec" for k in self.layer_kinds)

    def n_weights(self) -> int:
        tot = 0
        for l in range(self.n_layers):
            for nm in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"):
                a, b = self.weight_shape(l, nm)
                tot += a * b
        return tot + self.V * self.H


def _dense(name, L, H, I, Hq, Hkv, V, **kw):
    return ModelShape(name, L, H, I, Hq, Hkv, 128, V, tuple(["attn"] * L), **kw)


def _hybrid(name, L, H, I, Hq, Hkv, V, **kw):
    return ModelShape(name, L, H, I, Hq, Hkv, 128, V, tuple("attn" if l % 4 == 3 else "rec" for l in range(L)), **kw)


SHAPES = {
    "8b": _dense("8b", 36, 4096, 12288, 32, 8, 151936),
    "27b": _dense("27b", 64, 5120, 21504, 40, 8, 151936),
    "hybrid": _hybrid("hybrid", 32, 4096, 12288, 32, 8, 151936),
    # small models for parity at sizes the oracle finishes in seconds; still
    # several GEMM tiles with ragged row blocks (V = 4000 = 31.25 * 128).
    "mini": _dense("mini", 2, 512, 1024, 4, 2, 4000, gamma_sigma=0.1),
    # the 8B dimensions with 2 layers: profiling captures of one layer's
    # kernels with a few GB on the device
    "8b_2l": _dense("8b_2l", 2, 4096, 12288, 32, 8, 151936),
    "mini_hybrid": _hybrid("mini_hybrid", 4, 512, 1024, 4, 2, 4000, gamma_sigma=0.1),
    # full layer dimensions with few layers: end-to-end parity against the
    # oracle at the named models' widths, head groups and vocabulary
    "27b_2l": _dense("27b_2l", 2, 5120, 21504, 40, 8, 151936),
    "hybrid_4l": _hybrid("hybrid_4l", 4, 4096, 12288, 32, 8, 151936),
}


class SyntheticWeights:
    """bf16 ~ N(0, sigma) weights of a ModelShape, natural layout
    (PyTorch Linear: W[out][in]).  Tensors are regenerated on each request
    unless ``cache`` is set."""

    def __init__(self, shape: ModelShape, seed: int = 0, cache: bool = False):
        self.shape, self.seed, self.cache = shape, seed, cache
        self._c = {}

    def _get(self, k, fn):
        if not self.cache:
            return fn()
        if k not in self._c:
            self._c[k] = fn()
        return self._c[k]

    def layer(self, l: int, name: str) -> np.ndarray:
        def mk():
            N, K = self.shape.weight_shape(l, name)
            return normal_bf16(layer_key(self.seed, l, WEIGHT_SLOTS[name]), N * K, self.shape.sigma).reshape(N, K)
        return self._get((l, name), mk)

    def norm(self, l: int, which: str) -> np.ndarray:
        return self._gamma(layer_key(self.seed, l, WEIGHT_SLOTS[which]))

    def final_norm(self) -> np.ndarray:
        return self._gamma(layer_key(self.seed, FINAL_NORM_LAYER, WEIGHT_SLOTS["attn"]))

    def _gamma(self, k) -> np.ndarray:
        H = self.shape.H
        if self.shape.gamma_sigma == 0.0:
            return ones_bf16(H)
        from . import bf16_bits_to_f32
        g = normal_f32(k ^ SID_GAMMA, H, self.shape.gamma_sigma) + 1.0
        b = g.view(np.uint32)
        return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)

    def embed_rows(self, tokens) -> np.ndarray:
        H = self.shape.H
        k = key(self.seed, SID_EMBED)
        t = np.asarray(tokens, dtype=np.int64)
        out = np.empty((t.size, H), dtype=np.uint16)
        for i, tok in enumerate(t):
            normal_bf16(k, H, self.shape.sigma, offset=int(tok) * H, out=out[i])
        return out

    def embedding(self) -> np.ndarray:
        H, V = self.shape.H, self.shape.V
        return self._get("embed", lambda: normal_bf16(key(self.seed, SID_EMBED), V * H, self.shape.sigma).reshape(V, H))

    def lm_head(self) -> np.ndarray:
        H, V = self.shape.H, self.shape.V
        return self._get("lm", lambda: normal_bf16(key(self.seed, SID_LM_HEAD), V * H, self.shape.sigma).reshape(V, H))


# ----------------------------------------------------------- caches/state --

def _rkey(seed: int, sid: int, r: int) -> int:
    return key(seed, sid + (r << 20))


def kv_prefix(shape: ModelShape, seed: int, r: int, l: int, ctx: int, cap: int):
    """K, V prefix of request r, layer l: bf16 ~ N(0,1) [Hkv][cap][hd], slots
    >= ctx zero.  Treated as keys that already carry their rotation."""
    Hkv, hd = shape.Hkv, shape.hd
    k = np.zeros((Hkv, cap, hd), dtype=np.uint16)
    v = np.zeros((Hkv, cap, hd), dtype=np.uint16)
    base = key(seed, SID_KV)
    for which, arr in ((0, k), (1, v)):
        off = (((r * shape.n_layers + l) * 2 + which) << 32)
        vals = normal_bf16(base, Hkv * ctx * hd, 1.0, offset=off).reshape(Hkv, ctx, hd)
        arr[:, :ctx, :] = vals
    return k, v


def rec_state(shape: ModelShape, seed: int, r: int, l: int):
    """Initial recurrent state of request r, layer l: S0 ~ N(0, 0.01) fp32
    [nh][hd][hd] (row = key dim), z0 = 0."""
    nh, hd = shape.H // shape.hd, shape.hd
    S = normal_f32(key(seed, SID_STATE), nh * hd * hd, 0.01, offset=(r * shape.n_layers + l) << 32)
    return S.reshape(nh, hd, hd), np.zeros((nh, hd), dtype=np.float32)


# ------------------------------------------------------------ trees/tokens --

@dataclass
class TreeDraft:
    parents: np.ndarray
    copy: np.ndarray
    rand_tok: np.ndarray
    root_token: int


def draft(seed: int, r: int, M: int, max_depth: int, p: float, V: int, shape_kind: str = "tree") -> TreeDraft:
    parents = tree(_rkey(seed, SID_TREE, r), M, max_depth) if shape_kind == "tree" else chain(M)
    cp, rt = copy_coins(_rkey(seed, SID_COINS, r), M, p, V)
    from . import lib
    root = int(lib().sg_u64(_rkey(seed, SID_ROOT_TOKEN, r), 0) % V)
    return TreeDraft(parents, cp, rt, root)


@dataclass
class Candidates:
    """Draft candidate trees of R requests, concatenated: request r owns
    entries cu[r] .. cu[r+1]-1; parents are local to the request (root first,
    parent[i] < i); logprob[i] <= 0 is the draft log-probability of node i's
    token given its parent (0 at the roots); tokens are the draft tokens."""
    parents: np.ndarray
    logprob: np.ndarray
    tokens: np.ndarray
    cu: np.ndarray


def candidates(seed: int, R: int, n, max_depth: int, V: int, step: float = 0.0) -> Candidates:
    """Synthetic candidate trees: n (an int, or one per request) nodes per
    request in a random tree of depth <= max_depth; log-probabilities log(u)
    with u uniform in (0, 1] (a drafter's softmax tail), rounded down to a
    multiple of `step` when step > 0 (exact ties, zeros included); tokens
    uniform in [0, V)."""
    ns = [int(n)] * R if np.isscalar(n) else [int(x) for x in n]
    par, lp, tok = [], [], []
    for r in range(R):
        m = ns[r]
        par.append(tree(_rkey(seed, SID_CAND_TREE, r), m, max_depth))
        u = (uniform_int(_rkey(seed, SID_CAND_LP, r), m, 1, 1 << 24).astype(np.float64)) / float(1 << 24)
        l = np.log(u)
        if step > 0:
            l = -np.floor(-l / step) * step
            l = np.minimum(l, 0.0)
        l = l.astype(np.float32)
        if m:
            l[0] = 0.0
        lp.append(l)
        tok.append(uniform_int(_rkey(seed, SID_CAND_TOKEN, r), m, 0, V - 1).astype(np.int32))  # bounds inclusive
    cu = np.zeros(R + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ns)
    cat = lambda xs, dt: np.concatenate(xs).astype(dt) if xs else np.zeros(0, dt)
    return Candidates(cat(par, np.int32), cat(lp, np.float32), cat(tok, np.int32), cu)


def depths(parents) -> np.ndarray:
    d = np.zeros(len(parents), dtype=np.int32)
    for i in range(1, len(parents)):
        d[i] = d[parents[i]] + 1
    return d


def copy_rule_tokens(td: TreeDraft, argmax_fn, max_waves: int | None = None, full_tree: bool = False) -> np.ndarray:
    """Draft tokens by depth waves: node i at depth d copies the target's
    argmax at its parent when its coin says so, else takes its random token.
    ``argmax_fn(tokens_sub, parents_sub)`` must return the target argmax of
    every node of the prefix-closed sub-tree it is given.  With
    ``max_waves`` only nodes down to that depth follow the rule (one target
    pass per wave); deeper nodes take their random tokens.  full_tree: every
    wave passes the whole tree (nodes not yet decided hold their random
    tokens; a node's argmax depends on its root path only), so each node
    keeps the row it has in the final tree - for a target whose fp32
    rounding, and so an argmax at a near tie, may depend on the row."""
    return copy_rule_tokens_batch([td], lambda subs: [argmax_fn(*subs[0])], max_waves, full_tree)[0]


def copy_rule_tokens_batch(tds, argmax_fn, max_waves: int | None = None, full_tree: bool = False) -> list:
    """The copy rule for several requests at once: each wave makes one call
    ``argmax_fn([(tokens_sub, parents_sub) per request])`` returning the
    target argmax of every node of each sub-tree (of each whole tree with
    full_tree)."""
    parents = [np.asarray(td.parents) for td in tds]
    d = [depths(p) for p in parents]
    tok = []
    for td, p, dd in zip(tds, parents, d):
        t = np.zeros(p.size, dtype=np.int32)
        t[0] = td.root_token
        deep = np.nonzero(dd > (max_waves if max_waves is not None else p.size))[0]
        t[deep] = td.rand_tok[deep]
        if full_tree:
            later = np.nonzero(dd >= 1)[0]
            t[later] = td.rand_tok[later]
        tok.append(t)
    last = max((int(dd.max()) for dd in d if dd.size), default=0)
    if max_waves is not None:
        last = min(last, max_waves)
    for wave in range(1, last + 1):
        subs, maps = [], []
        for p, dd, t in zip(parents, d, tok):
            sub = np.arange(p.size) if full_tree else np.nonzero(dd < wave)[0]
            pos = {int(n): i for i, n in enumerate(sub)}
            psub = np.array([-1 if p[n] < 0 else pos[int(p[n])] for n in sub], dtype=np.int32)
            subs.append((t[sub].copy(), psub))
            maps.append(pos)
        ams = argmax_fn(subs)
        for td, p, dd, t, pos, am in zip(tds, parents, d, tok, maps, ams):
            am = np.asarray(am)
            for i in np.nonzero(dd == wave)[0]:
                t[i] = am[pos[int(p[i])]] if td.copy[i] else td.rand_tok[i]
    return tok


def copy_rule_tokens_static(td: TreeDraft, argmax_all) -> np.ndarray:
    """Copy rule when the target's argmax does not depend on the tokens
    (the tiny model): one pass over the nodes."""
    parents = np.asarray(td.parents)
    tok = np.zeros(parents.size, dtype=np.int32)
    tok[0] = td.root_token
    for i in range(1, parents.size):
        tok[i] = argmax_all[parents[i]] if td.copy[i] else td.rand_tok[i]
    return tok


# ------------------------------------------------------------------- tiny --

@dataclass
class TinyWorkload:
    W1: np.ndarray        # bf16 [1024][1024]
    Wlm: np.ndarray       # bf16 [4096][1024]
    act: np.ndarray       # bf16 [M][1024]
    draft: TreeDraft
    forced_w1: np.ndarray
    forced_lm: np.ndarray


def tiny(seed: int = 0, M: int = 8, max_depth: int = 4, p: float = 0.6, K: int = 1024, V: int = 4096,
         escape_frac: float = 0.001) -> TinyWorkload:
    """One linear layer K=N=1024 and an lm_head 1024 -> 4096, bf16 ~ N(0,0.02),
    with 0.1% of each weight tensor forced to exponents outside the table."""
    W1 = normal_bf16(key(seed, SID_TINY_W1), K * K, 0.02)
    Wlm = normal_bf16(key(seed, SID_LM_HEAD), V * K, 0.02)
    f1 = force_rare_exponents(key(seed, SID_ESC), W1, int(round(escape_frac * W1.size)))
    f2 = force_rare_exponents(key(seed, SID_ESC + 1), Wlm, int(round(escape_frac * Wlm.size)))
    act = normal_bf16(key(seed, SID_ACT), M * K, 1.0).reshape(M, K)
    return TinyWorkload(W1.reshape(K, K), Wlm.reshape(V, K), act, draft(seed, 0, M, max_depth, p, V), f1, f2)


# -------------------------------------------------------------- decoders --

@dataclass
class DecoderWorkload:
    shape: ModelShape
    seed: int
    M: int                   # nodes per request
    max_depth: int
    ctx: list                # per request
    p: float
    drafts: list             # TreeDraft per request
    page_size: int = 0       # 0: contiguous cache

    @property
    def R(self) -> int:
        return len(self.ctx)


def decoder(shape_name: str, seed: int = 0, M: int = 16, max_depth: int = 8, ctx: int = 2048, p: float = 0.7,
            R: int = 1, chain_draft: bool = False, ctx_range=None, page_size: int = 0) -> DecoderWorkload:
    shape = SHAPES[shape_name]
    if ctx_range is not None:
        ctxs = [int(c) for c in uniform_int(key(seed, SID_CTX), R, ctx_range[0], ctx_range[1])]
    else:
        ctxs = [ctx] * R
    drafts = [draft(seed, r, M, max_depth, p, shape.V, "chain" if chain_draft else "tree") for r in range(R)]
    return DecoderWorkload(shape, seed, M, max_depth, ctxs, p, drafts, page_size)


WORKLOADS = {
    "tiny": dict(kind="tiny"),
    "8b_m16": dict(kind="decoder", shape="8b", M=16, max_depth=8, ctx=2048, p=0.7),
    "8b_2l_m16": dict(kind="decoder", shape="8b_2l", M=16, max_depth=8, ctx=2048, p=0.7),
    "27b_m8": dict(kind="decoder", shape="27b", M=8, max_depth=10, ctx=4096, p=0.7),
    "27b_m16": dict(kind="decoder", shape="27b", M=16, max_depth=10, ctx=4096, p=0.7),
    "27b_m32": dict(kind="decoder", shape="27b", M=32, max_depth=10, ctx=4096, p=0.7),
    "27b_m64": dict(kind="decoder", shape="27b", M=64, max_depth=10, ctx=4096, p=0.7),
    "hybrid_m16": dict(kind="decoder", shape="hybrid", M=16, max_depth=8, ctx=2048, p=0.7),
    # four-layer profiling case of the hybrid step (3 recurrent + 1 attention)
    "hybrid_4l_m16": dict(kind="decoder", shape="hybrid_4l", M=16, max_depth=8, ctx=2048, p=0.7),
    "batched_r32": dict(kind="decoder", shape="8b", M=8, max_depth=7, R=32, chain_draft=True, p=0.6,
                        ctx_range=(1024, 4096), page_size=16),
    # two-layer profiling case of the batched step
    "8b_2l_r32": dict(kind="decoder", shape="8b_2l", M=8, max_depth=7, R=32, chain_draft=True, p=0.6,
                      ctx_range=(1024, 4096), page_size=16),
}
# the batched step at fewer requests (M = 8R rows): the sweep over the
# bandwidth-bound to tensor-bound crossover
for _r in (1, 2, 4, 8, 16):
    WORKLOADS[f"batched_r{_r}"] = dict(WORKLOADS["batched_r32"], R=_r)


def make(name: str, seed: int = 0, **over):
    spec = dict(WORKLOADS[name])
    spec.update(over)
    kind = spec.pop("kind")
    if kind == "tiny":
        return tiny(seed, **spec)
    sh = spec.pop("shape")
    return decoder(sh, seed, **spec)


def page_tables(seed: int, ctxs, M: int, page_size: int, slack_pages: int = 1):
    """Random physical page assignment: request r gets ceil((ctx_r + M)/ps) +
    slack pages, all requests' pages drawn from one random permutation."""
    need = [-(-(c + M) // page_size) + slack_pages for c in ctxs]
    total = int(sum(need))
    perm = permutation(key(seed, SID_PAGES), total)
    maxp = max(need)
    table = np.full((len(ctxs), maxp), -1, dtype=np.int32)
    o = 0
    for r, n in enumerate(need):
        table[r, :n] = perm[o:o + n]
        o += n
    return table, total


# ------------------------------------------------------- gated delta rule --

@dataclass
class GdnInputs:
    """Inputs of one gated-delta-rule layer over the draft trees of R
    requests: q, k, v bf16 [rows][nh][128], gates alpha in [alpha_lo, 1] and
    write strengths beta in [0, 1] fp32 [rows][nh], parents local to each
    request, cu [R+1], committed states S fp32 [R][nh][128][128]."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    alpha: np.ndarray
    beta: np.ndarray
    parents: np.ndarray
    cu: np.ndarray
    S: np.ndarray


def row_scaled(seed: int, N: int, K: int, spread: float = 2.0) -> np.ndarray:
    """bf16 bits [N][K]: row n ~ N(0, (0.02 * 2^u_n)^2), u_n uniform in
    [-spread, spread] (output channels of different norms, the case a
    per-channel exponent base is for)."""
    u = uniform_int(key(seed, 2), N, 0, 1 << 20) / float(1 << 20) * 2 * spread - spread
    W = np.empty((N, K), dtype=np.uint16)
    k = key(seed, 3)
    for n in range(N):
        normal_bf16(k, K, 0.02 * 2.0 ** u[n], offset=n * K, out=W[n])
    return W


def gdn_inputs(seed: int, Ms, max_depth: int, nh: int, alpha_lo: float = 0.8, s_sigma: float = 0.01) -> GdnInputs:
    R = len(Ms)
    cu = np.zeros(R + 1, dtype=np.int32)
    cu[1:] = np.cumsum(Ms)
    rows = int(cu[-1])
    par = np.concatenate([tree(_rkey(seed, SID_TREE, r), int(m), max_depth) for r, m in enumerate(Ms)]).astype(np.int32)
    q, k, v = (normal_bf16(key(seed, SID_ACT + j), rows * nh * 128, 1.0).reshape(rows, nh, 128) for j in range(3))
    u = uniform_int(key(seed, SID_COINS), 2 * rows * nh, 0, (1 << 24) - 1).reshape(2, rows, nh) / float(1 << 24)
    alpha = (alpha_lo + (1.0 - alpha_lo) * u[0]).astype(np.float32)
    beta = u[1].astype(np.float32)
    S = normal_f32(key(seed, SID_STATE), R * nh * 128 * 128, s_sigma).reshape(R, nh, 128, 128)
    return GdnInputs(q, k, v, alpha, beta, par, cu, S)
