"""Device-side objects around libsdv: packed tensors, the model, the caches.

Marshalling and memory only (PyTorch allocates, the library computes).
Weights come from any provider with the methods of
``synthetic.workloads.SyntheticWeights`` (natural PyTorch-Linear layout,
bf16 bit patterns as uint16 numpy arrays).
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import KV, LayerWeights, ModelConfig, ModelWeights, PagedKV, W12Meta, W12Tensor, check, lib, stream_ptr


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def to_device_u16(a: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bit patterns -> int16 device tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device)


def _i32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).to(device)


class Packed:
    """A W12-packed tensor on the device (owns its buffers)."""

    def __init__(self, meta: W12Meta, words, esc_idx, esc_val, row_ptr, tile_ptr=None, tile_esc=None):
        self.meta, self.words, self.esc_idx, self.esc_val, self.row_ptr = meta, words, esc_idx, esc_val, row_ptr
        self.tile_ptr, self.tile_esc = tile_ptr, tile_esc

    N = property(lambda self: int(self.meta.N))
    K = property(lambda self: int(self.meta.K))
    n_escapes = property(lambda self: int(self.meta.n_escapes))

    @property
    def table(self):
        return np.array(self.meta.table[: self.meta.n_table], dtype=np.uint8)

    def struct(self) -> W12Tensor:
        t = W12Tensor()
        t.N, t.K = self.meta.N, self.meta.K
        t.words, t.esc_idx, t.esc_val, t.row_ptr = (_ptr(self.words), _ptr(self.esc_idx), _ptr(self.esc_val),
                                                    _ptr(self.row_ptr))
        t.tile_ptr, t.tile_esc = _ptr(self.tile_ptr), _ptr(self.tile_esc)
        t.n_escapes = self.meta.n_escapes
        t.table = self.meta.table
        t.n_table = self.meta.n_table
        t.affine = self.meta.affine
        t.row_base = _ptr(getattr(self, "row_base", None))
        return t

    def copy(self) -> "Packed":
        """A copy in new device buffers (same meta); the 8-bit plane too."""
        cl = lambda t: None if t is None else t.clone()
        q = Packed(self.meta, cl(self.words), cl(self.esc_idx), cl(self.esc_val), cl(self.row_ptr), cl(self.tile_ptr),
                   cl(self.tile_esc))
        if getattr(self, "row_base", None) is not None:
            q.row_base = self.row_base.clone()
        if getattr(self, "plane8", None) is not None:
            q.plane8 = self.plane8.clone()
        return q

    def nbytes(self) -> int:
        """Bytes a GEMM streams: the packed words plus the escape tile index."""
        return self.words.numel() * 4 + self.n_escapes * 4 + int(lib().w12_tile_ptr_count(self.N, self.K)) * 4


def pack(w: torch.Tensor, row_src: np.ndarray | None = None, stream=None, view8: bool = False) -> Packed:
    """Pack a bf16 device tensor [N][K] (int16/uint16/bfloat16 storage); with
    view8 also its nested 8-bit plane (p.plane8, w12_plane8_pack)."""
    assert w.is_cuda and w.dim() == 2 and w.element_size() == 2 and w.is_contiguous()
    N, K = w.shape
    s = stream_ptr(stream)
    meta = W12Meta()
    check(lib().w12_pack_analyze(w.data_ptr(), N, K, ctypes.byref(meta), s))
    dev = w.device
    words = torch.empty(int(lib().w12_words_count(N, K)), dtype=torch.int32, device=dev)
    ne = max(int(meta.n_escapes), 1)
    esc_idx = torch.empty(ne, dtype=torch.int32, device=dev)
    esc_val = torch.empty(ne, dtype=torch.int16, device=dev)
    row_ptr = torch.empty(N + 1, dtype=torch.int32, device=dev)
    rs = None if row_src is None else _i32(row_src, dev)
    check(lib().w12_pack_encode(w.data_ptr(), _ptr(rs), ctypes.byref(meta), words.data_ptr(), esc_idx.data_ptr(),
                                esc_val.data_ptr(), row_ptr.data_ptr(), s))
    p = Packed(meta, words, esc_idx, esc_val, row_ptr)
    p.tile_ptr = torch.empty(int(lib().w12_tile_ptr_count(N, K)), dtype=torch.int32, device=dev)
    p.tile_esc = torch.empty(ne, dtype=torch.int32, device=dev)
    t = p.struct()
    check(lib().w12_pack_tile_index(ctypes.byref(t), p.tile_ptr.data_ptr(), p.tile_esc.data_ptr(), s))
    p.plane8 = None
    if view8:
        p.plane8 = torch.empty(int(lib().w12_plane8_words_count(N, K)), dtype=torch.int32, device=dev)
        check(lib().w12_plane8_pack(w.data_ptr(), _ptr(rs), ctypes.byref(meta), p.plane8.data_ptr(), s))
    torch.cuda.synchronize()
    return p


def pack_channel(w: torch.Tensor, row_src: np.ndarray | None = None, stream=None) -> Packed:
    """Pack a bf16 device tensor [N][K] in the per-channel format
    (w12c_pack_analyze / w12c_pack_encode): a base exponent per output row
    (p.row_base), the per-tensor word layout, the same side list."""
    assert w.is_cuda and w.dim() == 2 and w.element_size() == 2 and w.is_contiguous()
    N, K = w.shape
    s = stream_ptr(stream)
    dev = w.device
    rs = None if row_src is None else _i32(row_src, dev)
    base = torch.empty(N, dtype=torch.uint8, device=dev)
    row_ptr = torch.empty(N + 1, dtype=torch.int32, device=dev)
    meta = W12Meta()
    check(lib().w12c_pack_analyze(w.data_ptr(), _ptr(rs), N, K, base.data_ptr(), row_ptr.data_ptr(),
                                  ctypes.byref(meta), s))
    words = torch.empty(int(lib().w12_words_count(N, K)), dtype=torch.int32, device=dev)
    ne = max(int(meta.n_escapes), 1)
    esc_idx = torch.empty(ne, dtype=torch.int32, device=dev)
    esc_val = torch.empty(ne, dtype=torch.int16, device=dev)
    check(lib().w12c_pack_encode(w.data_ptr(), _ptr(rs), N, K, base.data_ptr(), row_ptr.data_ptr(), words.data_ptr(),
                                 esc_idx.data_ptr(), esc_val.data_ptr(), s))
    p = Packed(meta, words, esc_idx, esc_val, row_ptr)
    p.row_base = base
    p.tile_ptr = torch.empty(int(lib().w12_tile_ptr_count(N, K)), dtype=torch.int32, device=dev)
    p.tile_esc = torch.empty(ne, dtype=torch.int32, device=dev)
    t = p.struct()
    check(lib().w12_pack_tile_index(ctypes.byref(t), p.tile_ptr.data_ptr(), p.tile_esc.data_ptr(), s))
    p.plane8 = None
    torch.cuda.synchronize()
    return p


def unpack(p: Packed, stream=None) -> torch.Tensor:
    out = torch.empty((p.N, p.K), dtype=torch.int16, device=p.words.device)
    t = p.struct()
    check(lib().w12_unpack(ctypes.byref(t), out.data_ptr(), stream_ptr(stream)))
    return out


def save(p: Packed, path: str) -> None:
    """Write a packed tensor to a W12 file (w12_save): the arrays are copied
    to host memory first."""
    host = {k: getattr(p, k).cpu().numpy() for k in ("words", "esc_idx", "esc_val", "row_ptr", "tile_ptr", "tile_esc")}
    t = p.struct()
    t.words, t.esc_idx, t.esc_val = (host[k].ctypes.data for k in ("words", "esc_idx", "esc_val"))
    t.row_ptr, t.tile_ptr, t.tile_esc = (host[k].ctypes.data for k in ("row_ptr", "tile_ptr", "tile_esc"))
    check(lib().w12_save(str(path).encode(), ctypes.byref(t)))


def load_host(path: str):
    """Read a W12 file into host arrays (w12_load_info, w12_load): returns
    (meta, dict of numpy arrays words, esc_idx, esc_val, row_ptr, tile_ptr,
    tile_esc; the escape arrays have at least one element)."""
    meta = W12Meta()
    ntp = ctypes.c_int64()
    check(lib().w12_load_info(str(path).encode(), ctypes.byref(meta), ctypes.byref(ntp)))
    ne = max(int(meta.n_escapes), 1)
    a = {"words": np.empty(int(lib().w12_words_count(meta.N, meta.K)), dtype=np.int32),
         "esc_idx": np.empty(ne, dtype=np.int32), "esc_val": np.empty(ne, dtype=np.int16),
         "row_ptr": np.empty(int(meta.N) + 1, dtype=np.int32), "tile_ptr": np.empty(int(ntp.value), dtype=np.int32),
         "tile_esc": np.empty(ne, dtype=np.int32)}
    check(lib().w12_load(str(path).encode(), *(a[k].ctypes.data for k in ("words", "esc_idx", "esc_val", "row_ptr",
                                                                           "tile_ptr", "tile_esc")),
                         ctypes.byref(meta)))
    return meta, a


def load(path: str, device="cuda") -> Packed:
    """A packed tensor from a W12 file, its arrays copied to `device`."""
    meta, a = load_host(path)
    t = {k: torch.from_numpy(v).to(device) for k, v in a.items()}
    return Packed(meta, t["words"], t["esc_idx"], t["esc_val"], t["row_ptr"], t["tile_ptr"], t["tile_esc"])


class Workspace:
    """Caller-owned device scratch for the stand-alone entry points."""

    def __init__(self, nbytes: int, device="cuda"):
        self.buf = torch.empty(max(int(nbytes), 256) + 256, dtype=torch.uint8, device=device)
        self.ptr = (self.buf.data_ptr() + 255) & ~255
        self.nbytes = int(nbytes)


def linear(p: Packed, x: torch.Tensor, ws: Workspace | None = None, stream=None) -> torch.Tensor:
    """y = bf16(x W^T) through the fused W12 GEMM; x int16 bits [M][K]."""
    M = x.shape[0]
    need = int(lib().sd_w12_linear_workspace(p.N, p.K, M))
    if ws is None or ws.nbytes < need:
        ws = Workspace(need, x.device)
    y = torch.empty((M, p.N), dtype=torch.int16, device=x.device)
    t = p.struct()
    check(lib().sd_w12_linear(ctypes.byref(t), x.data_ptr(), M, y.data_ptr(), ws.ptr, ws.nbytes, stream_ptr(stream)))
    return y


def linear_stream(p: Packed, x: torch.Tensor, plane8: torch.Tensor | None = None, ws: Workspace | None = None,
                  stream=None) -> torch.Tensor:
    """y = bf16(x W^T) on the weight-streaming kernel (M <= 64); with plane8
    (the tensor's nested 8-bit plane) the product with the 8-bit view."""
    M = x.shape[0]
    need = int(lib().sd_w12_linear_stream_workspace(p.N, p.K, M))
    if ws is None or ws.nbytes < need:
        ws = Workspace(need, x.device)
    y = torch.empty((M, p.N), dtype=torch.int16, device=x.device)
    t = p.struct()
    check(lib().sd_w12_linear_stream(ctypes.byref(t), None if plane8 is None else plane8.data_ptr(), x.data_ptr(), M,
                                     y.data_ptr(), ws.ptr, ws.nbytes, stream_ptr(stream)))
    return y


def linear_view8(p: Packed, x: torch.Tensor, plane8: torch.Tensor, ws: Workspace | None = None,
                 stream=None) -> torch.Tensor:
    """y = bf16(x V^T), V the nested 8-bit view of W (sd_w12_linear_view8,
    M <= 64), streaming the plane at 1 byte per weight."""
    M = x.shape[0]
    need = int(lib().sd_w12_linear_view8_workspace(p.N, p.K, M))
    if ws is None or ws.nbytes < need:
        ws = Workspace(need, x.device)
    y = torch.empty((M, p.N), dtype=torch.int16, device=x.device)
    t = p.struct()
    check(lib().sd_w12_linear_view8(ctypes.byref(t), plane8.data_ptr(), x.data_ptr(), M, y.data_ptr(), ws.ptr,
                                    ws.nbytes, stream_ptr(stream)))
    return y


def set_strip(on: bool | None) -> bool:
    """Skinny launches whose 16-row strips fit one wave on the strip-parallel
    kernel (True, the default: no split-K across CTAs) or on the warp-level
    kernel (False); None only queries.  Returns the setting in force."""
    return bool(lib().sd_gemm_set_strip(-1 if on is None else (1 if on else 0)))


def set_deferred_finish(on: bool | None) -> bool:
    """Split row blocks of the warp-level GEMM finished by a separate kernel
    after the GEMM (True) or by their last contributor inside it (False, the
    default); None only queries.  Returns the setting in force."""
    return bool(lib().sd_gemm_set_deferred_finish(-1 if on is None else (1 if on else 0)))


def set_cluster_finish(on: bool | None) -> bool:
    """Split row blocks of the warp-level GEMM finished through thread-block
    clusters (True) or partials in the workspace (False, the default);
    None only queries.  Returns the setting in force."""
    return bool(lib().sd_gemm_set_cluster_finish(-1 if on is None else (1 if on else 0)))


def set_tc_min_rows(rows: int) -> int:
    """Rows per launch from which the W12 GEMMs run on the tcgen05 kernel
    (process-wide; <= 0 restores the default).  Returns the value in force."""
    return int(lib().sd_gemm_set_tc_min_rows(int(rows)))


def set_attn_splits(splits: int) -> int:
    """Prefix key splits of the step's attention per (request, kv head, row
    chunk); <= 0 restores the automatic choice.  Returns the value in force
    (0: automatic)."""
    return int(lib().sd_attn_set_splits(int(splits)))


def row_map(kind: int, Hq: int, Hkv: int, inter: int, N: int) -> np.ndarray:
    out = np.empty(N, dtype=np.int32)
    check(lib().sd_model_row_map(kind, Hq, Hkv, 128, inter, out.ctypes.data, N))
    return out


class Model:
    """A decoder whose linear weights are W12-packed on the device."""

    def __init__(self, shape, weights, max_rows: int = 64, max_requests: int = 1, max_positions: int = 4352,
                 device: str = "cuda", progress=None, view8: bool = False):
        self.shape = shape
        self.device = device
        keep = []
        L = shape.n_layers
        layers = (LayerWeights * L)()
        H, I, Hq, Hkv = shape.H, shape.I, shape.Hq, shape.Hkv
        self.packed_bytes = 0
        self.layer_bytes = []
        for l, kind in enumerate(shape.layer_kinds):
            qkv = to_device_u16(np.concatenate([weights.layer(l, n) for n in ("wq", "wk", "wv")]), device)
            p_qkv = pack(qkv, row_map(0, Hq, Hkv, I, qkv.shape[0]) if kind == "attn" else None, view8=view8)
            del qkv
            p_o = pack(to_device_u16(weights.layer(l, "wo"), device), view8=view8)
            gu = to_device_u16(np.concatenate([weights.layer(l, "w_gate"), weights.layer(l, "w_up")]), device)
            p_gu = pack(gu, row_map(1, Hq, Hkv, I, gu.shape[0]), view8=view8)
            del gu
            p_d = pack(to_device_u16(weights.layer(l, "w_down"), device), view8=view8)
            an = to_device_u16(weights.norm(l, "attn"), device)
            mn = to_device_u16(weights.norm(l, "mlp"), device)
            keep += [p_qkv, p_o, p_gu, p_d, an, mn]
            layers[l].qkv, layers[l].o, layers[l].gate_up, layers[l].down = (p.struct() for p in (p_qkv, p_o, p_gu, p_d))
            layers[l].attn_norm, layers[l].mlp_norm = an.data_ptr(), mn.data_ptr()
            self.layer_bytes.append({k: p.nbytes() for k, p in (("qkv", p_qkv), ("o", p_o), ("gate_up", p_gu),
                                                                ("down", p_d))})
            self.packed_bytes += sum(self.layer_bytes[-1].values())
            if progress:
                progress(l)
        self.embed = to_device_u16(weights.embedding(), device)
        self.final_norm = to_device_u16(weights.final_norm(), device)
        self.lm_head = pack(to_device_u16(weights.lm_head(), device), view8=view8)
        self.packed_bytes += self.lm_head.nbytes()
        keep += [self.embed, self.final_norm, self.lm_head]
        self._keep, self._layers = keep, layers
        self._kinds = (ctypes.c_int8 * L)(*[0 if k == "attn" else 1 for k in shape.layer_kinds])
        cfg = ModelConfig()
        cfg.n_layers, cfg.hidden, cfg.inter, cfg.n_q_heads, cfg.n_kv_heads = L, H, I, Hq, Hkv
        cfg.head_dim, cfg.vocab = 128, shape.V
        cfg.rms_eps, cfg.rope_base, cfg.rec_eps = shape.eps, shape.rope_base, shape.rec_eps
        cfg.layer_kind_host = ctypes.addressof(self._kinds)
        cfg.max_rows, cfg.max_requests, cfg.max_positions = max_rows, max_requests, max_positions
        mw = ModelWeights()
        mw.layers_host = ctypes.addressof(layers)
        mw.embed, mw.final_norm = self.embed.data_ptr(), self.final_norm.data_ptr()
        mw.lm_head = self.lm_head.struct()
        self._cfg, self._mw = cfg, mw
        h = ctypes.c_void_p()
        torch.cuda.synchronize()
        check(lib().sd_model_create(ctypes.byref(cfg), ctypes.byref(mw), ctypes.byref(h)))
        self.handle = h
        if view8:
            packed = [p for p in keep if isinstance(p, Packed)]  # per layer qkv, o, gate_up, down; then lm_head
            planes = (ctypes.c_void_p * len(packed))(*[p.plane8.data_ptr() for p in packed])
            self._planes = planes
            check(lib().sd_model_set_view8(self.handle, planes, len(packed)))

    def close(self):
        if getattr(self, "handle", None):
            lib().sd_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def status(self) -> int:
        st = ctypes.c_int32()
        check(lib().sd_status(self.handle, ctypes.byref(st)))
        return int(st.value)

    def last_launches(self) -> int:
        return int(lib().sd_model_last_launches(self.handle))

    def final_hidden(self, rows: int, stream=None) -> torch.Tensor:
        """The last call's final RMSNorm output (the lm_head input), int16
        bits [rows][hidden] (sd_model_final_hidden)."""
        out = torch.empty((rows, self.shape.H), dtype=torch.int16, device=self.device)
        check(lib().sd_model_final_hidden(self.handle, out.data_ptr(), rows, stream_ptr(stream)))
        return out

    def set_graphs(self, on: bool):
        check(lib().sd_model_set_graphs(self.handle, 1 if on else 0))

    def set_fused(self, on: bool):
        """Skinny steps: the linears between two attention kernels as one
        launch with the RMSNorms folded in (on) or one launch per linear."""
        check(lib().sd_model_set_fused(self.handle, 1 if on else 0))

    def set_timing(self, on: bool):
        """Event timing of every kernel launch of the following calls."""
        check(lib().sd_model_set_timing(self.handle, 1 if on else 0))

    def timeline(self, max_entries: int = 4096):
        """[(kind name, ms, algorithmic bytes)] of the last timed call."""
        from . import KERNEL_KINDS
        k = np.zeros(max_entries, np.int32)
        ms = np.zeros(max_entries, np.float32)
        b = np.zeros(max_entries, np.float64)
        n = lib().sd_model_timeline(self.handle, max_entries, k.ctypes.data, ms.ctypes.data, b.ctypes.data)
        if n < 0:
            check(3)
        return [(KERNEL_KINDS[int(k[i])], float(ms[i]), float(b[i])) for i in range(n)]

    def outputs(self, M: int, logits: bool = False, R: int = 1):
        d = self.device
        o = {"accepted_len": torch.zeros(R, dtype=torch.int32, device=d),
             "accepted_tokens": torch.zeros(M, dtype=torch.int32, device=d),
             "bonus": torch.zeros(R, dtype=torch.int32, device=d),
             "argmax": torch.zeros(M, dtype=torch.int32, device=d)}
        if logits:
            o["logits"] = torch.empty((M, self.shape.V), dtype=torch.int16, device=d)
        return o

    def forward(self, tokens, parents, kv: "KVCache", logits: bool = True, stream=None):
        tok, par = _i32(tokens, self.device), _i32(parents, self.device)
        M = tok.numel()
        lg = torch.empty((M, self.shape.V), dtype=torch.int16, device=self.device) if logits else None
        am = torch.empty(M, dtype=torch.int32, device=self.device)
        kvs = kv.struct()
        check(lib().sd_forward(self.handle, tok.data_ptr(), par.data_ptr(), M, ctypes.byref(kvs), _ptr(lg),
                               am.data_ptr(), stream_ptr(stream)))
        return lg, am

    def forward_view8(self, tokens, parents, kv: "KVCache", logits: bool = True, stream=None):
        """Round one of two-level verification (sd_forward_view8): the
        forward over the weights' 8-bit view; (logits or None, argmax)."""
        tok, par = _i32(tokens, self.device), _i32(parents, self.device)
        M = tok.numel()
        lg = torch.empty((M, self.shape.V), dtype=torch.int16, device=self.device) if logits else None
        am = torch.empty(M, dtype=torch.int32, device=self.device)
        kvs = kv.struct()
        check(lib().sd_forward_view8(self.handle, tok.data_ptr(), par.data_ptr(), M, ctypes.byref(kvs), _ptr(lg),
                                     am.data_ptr(), stream_ptr(stream)))
        return lg, am

    def verify(self, tokens, parents, kv: "KVCache", logits: bool = False, out=None, stream=None):
        tok = tokens if isinstance(tokens, torch.Tensor) else _i32(tokens, self.device)
        par = parents if isinstance(parents, torch.Tensor) else _i32(parents, self.device)
        M = tok.numel()
        o = out or self.outputs(M, logits)
        kvs = kv.struct()
        check(lib().sd_verify_step(self.handle, tok.data_ptr(), par.data_ptr(), M, ctypes.byref(kvs),
                                   o["accepted_len"].data_ptr(), o["accepted_tokens"].data_ptr(),
                                   o["bonus"].data_ptr(), _ptr(o.get("logits")), o["argmax"].data_ptr(),
                                   stream_ptr(stream)))
        return o

    def verify_batch(self, tokens, parents, cu_nodes, kv: "PagedKVCache", logits: bool = False, out=None,
                     stream=None):
        tok = tokens if isinstance(tokens, torch.Tensor) else _i32(tokens, self.device)
        par = parents if isinstance(parents, torch.Tensor) else _i32(parents, self.device)
        cu = np.ascontiguousarray(np.asarray(cu_nodes, dtype=np.int32))
        R = cu.size - 1
        o = out or self.outputs(tok.numel(), logits, R)
        kvs = kv.struct()
        check(lib().sd_verify_batch(self.handle, tok.data_ptr(), par.data_ptr(), cu.ctypes.data, R,
                                    ctypes.byref(kvs), o["accepted_len"].data_ptr(), o["accepted_tokens"].data_ptr(),
                                    o["bonus"].data_ptr(), _ptr(o.get("logits")), o["argmax"].data_ptr(),
                                    stream_ptr(stream)))
        return o


class KVCache:
    """Contiguous cache of one request: K/V [n_attn][Hkv][cap][128] bf16,
    recurrent state S [n_rec][nh][128][128] fp32, z [n_rec][nh][128]."""

    def __init__(self, shape, cap: int, device="cuda"):
        self.shape, self.cap, self.device = shape, cap, device
        na, nr, nh = max(shape.n_attn, 1), max(shape.n_rec, 1), shape.H // 128
        self.k = torch.zeros((na, shape.Hkv, cap, 128), dtype=torch.int16, device=device)
        self.v = torch.zeros_like(self.k)
        self.S = torch.zeros((nr, nh, 128, 128), dtype=torch.float32, device=device)
        self.z = torch.zeros((nr, nh, 128), dtype=torch.float32, device=device)
        self.ctx_len = torch.zeros(1, dtype=torch.int32, device=device)

    def fill(self, seed: int, ctx: int, r: int = 0):
        from synthetic import workloads as wl
        la = lr = 0
        for l, kind in enumerate(self.shape.layer_kinds):
            if kind == "attn":
                k, v = wl.kv_prefix(self.shape, seed, r, l, ctx, ctx)
                self.k[la, :, :ctx] = to_device_u16(k, self.device)
                self.v[la, :, :ctx] = to_device_u16(v, self.device)
                la += 1
            else:
                S, z = wl.rec_state(self.shape, seed, r, l)
                self.S[lr] = torch.from_numpy(S).to(self.device)
                self.z[lr] = torch.from_numpy(z).to(self.device)
                lr += 1
        self.ctx_len.fill_(ctx)
        return self

    def struct(self) -> KV:
        s = KV()
        s.k, s.v, s.cap = self.k.data_ptr(), self.v.data_ptr(), self.cap
        s.S, s.z = self.S.data_ptr(), self.z.data_ptr()
        s.ctx_len = self.ctx_len.data_ptr()
        return s


class PagedKVCache:
    """Paged cache of R requests: pools [n_attn][n_pages][Hkv][page][128]."""

    def __init__(self, shape, page_table: np.ndarray, n_pages: int, page_size: int = 16, device="cuda"):
        self.shape, self.device, self.page_size, self.n_pages = shape, device, page_size, n_pages
        self.page_table_host = np.ascontiguousarray(page_table, dtype=np.int32)
        self.R, self.max_pages = self.page_table_host.shape
        na, nr, nh = max(shape.n_attn, 1), max(shape.n_rec, 1), shape.H // 128
        self.k = torch.zeros((na, n_pages, shape.Hkv, page_size, 128), dtype=torch.int16, device=device)
        self.v = torch.zeros_like(self.k)
        self.S = torch.zeros((self.R, nr, nh, 128, 128), dtype=torch.float32, device=device)
        self.z = torch.zeros((self.R, nr, nh, 128), dtype=torch.float32, device=device)
        self.page_table = _i32(self.page_table_host, device)
        self.ctx_len = torch.zeros(self.R, dtype=torch.int32, device=device)

    def fill(self, seed: int, ctxs):
        from synthetic import workloads as wl
        ps = self.page_size
        la = lr = 0
        for l, kind in enumerate(self.shape.layer_kinds):
            if kind == "attn":
                kp = np.zeros((self.n_pages, self.shape.Hkv, ps, 128), dtype=np.uint16)
                vp = np.zeros_like(kp)
                for r, ctx in enumerate(ctxs):
                    k, v = wl.kv_prefix(self.shape, seed, r, l, ctx, ctx)
                    t = np.arange(ctx)
                    pages = self.page_table_host[r, t // ps]
                    kp[pages, :, t % ps, :] = k.transpose(1, 0, 2)
                    vp[pages, :, t % ps, :] = v.transpose(1, 0, 2)
                self.k[la] = to_device_u16(kp, self.device)
                self.v[la] = to_device_u16(vp, self.device)
                la += 1
            else:
                for r in range(len(ctxs)):
                    S, z = wl.rec_state(self.shape, seed, r, l)
                    self.S[r, lr] = torch.from_numpy(S).to(self.device)
                    self.z[r, lr] = torch.from_numpy(z).to(self.device)
                lr += 1
        self.ctx_len.copy_(_i32(ctxs, self.device))
        return self

    def struct(self) -> PagedKV:
        s = PagedKV()
        s.k_pool, s.v_pool = self.k.data_ptr(), self.v.data_ptr()
        s.n_pages, s.page_size = self.n_pages, self.page_size
        s.page_table, s.max_pages = self.page_table.data_ptr(), self.max_pages
        s.S, s.z, s.ctx_len = self.S.data_ptr(), self.z.data_ptr(), self.ctx_len.data_ptr()
        return s


class Selector:
    """Best-first node selection under a shared node budget through the C
    ABI (sd_best_first_select): owns the workspace and output buffers for up
    to `max_total` candidates, so repeated calls allocate nothing."""

    def __init__(self, max_total: int, max_requests: int, device="cuda"):
        self.max_total, self.max_requests, self.device = int(max_total), int(max_requests), device
        self.ws = Workspace(int(lib().sd_select_workspace(self.max_total)), device)
        n, R = self.max_total, self.max_requests
        self.out_cu = torch.zeros(R + 1, dtype=torch.int32, device=device)
        self.out_src = torch.zeros(n, dtype=torch.int32, device=device)
        self.out_parents = torch.zeros(n, dtype=torch.int32, device=device)
        self.out_tokens = torch.zeros(n, dtype=torch.int32, device=device)
        self.out_score = torch.zeros(n, dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def __call__(self, parents: torch.Tensor, logprob: torch.Tensor, cu: torch.Tensor, budget: int, cap: int,
                 tokens: torch.Tensor | None = None, stream=None, clear_status: bool = True):
        """parents / cu int32, logprob float32, tokens int32 (optional), all on
        the device.  Returns views of the output buffers (valid until the next
        call): cu [R+1], src, parents, tokens, score (each min(budget, n)
        long; entries past cu[R] are unused) and status [1]."""
        R, n = cu.numel() - 1, parents.numel()
        if n > self.max_total or R > self.max_requests:
            raise ValueError("more candidates or requests than the selector was made for")
        if clear_status:
            self.status.zero_()
        k = min(int(budget), n)
        check(lib().sd_best_first_select(parents.data_ptr(), logprob.data_ptr(), cu.data_ptr(), R, n, int(budget),
                                         int(cap), _ptr(tokens), self.out_cu.data_ptr(), self.out_src.data_ptr(),
                                         self.out_parents.data_ptr(),
                                         self.out_tokens.data_ptr() if tokens is not None else 0,
                                         self.out_score.data_ptr(), self.status.data_ptr(), self.ws.ptr,
                                         self.ws.nbytes, stream_ptr(stream)))
        return {"cu": self.out_cu[:R + 1], "src": self.out_src[:k], "parents": self.out_parents[:k],
                "tokens": self.out_tokens[:k] if tokens is not None else None, "score": self.out_score[:k],
                "status": self.status}


def tiny_verify(W1: Packed, Wlm: Packed, act: torch.Tensor, tokens, parents, logits: bool = True, stream=None):
    """The tiny verify model through the C ABI; returns a dict of device tensors."""
    dev = act.device
    tok, par = _i32(tokens, dev), _i32(parents, dev)
    M = tok.numel()
    ws = Workspace(int(lib().sd_tiny_workspace(W1.N, W1.K, Wlm.N, M)), dev)
    o = {"accepted_len": torch.zeros(1, dtype=torch.int32, device=dev),
         "accepted_tokens": torch.zeros(M, dtype=torch.int32, device=dev),
         "bonus": torch.zeros(1, dtype=torch.int32, device=dev),
         "argmax": torch.zeros(M, dtype=torch.int32, device=dev),
         "status": torch.zeros(1, dtype=torch.int32, device=dev)}
    if logits:
        o["logits"] = torch.empty((M, Wlm.N), dtype=torch.int16, device=dev)
    t1, t2 = W1.struct(), Wlm.struct()
    check(lib().sd_tiny_verify(ctypes.byref(t1), ctypes.byref(t2), act.data_ptr(), tok.data_ptr(), par.data_ptr(), M,
                               o["accepted_len"].data_ptr(), o["accepted_tokens"].data_ptr(), o["bonus"].data_ptr(),
                               _ptr(o.get("logits")), o["argmax"].data_ptr(), o["status"].data_ptr(), ws.ptr,
                               ws.nbytes, stream_ptr(stream)))
    o["_ws"] = ws
    return o


class GdnLayer:
    """Gated delta rule over draft trees through the C ABI (sd_gdn_tree_verify,
    sd_gdn_commit); owns the workspace for up to `max_rows` rows."""

    def __init__(self, max_rows: int, nh: int, device="cuda"):
        self.nh, self.device = int(nh), device
        self.ws = Workspace(int(lib().sd_gdn_workspace(int(max_rows), self.nh)), device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def verify(self, q, k, v, alpha, beta, parents, cu, S, stream=None, cu_dev=None) -> torch.Tensor:
        """q, k, v int16 bits [rows][nh][128]; alpha, beta float32 [rows][nh];
        parents int32 [rows]; cu host array [R+1] (cu_dev: the same on the
        device, e.g. for a call inside a stream capture); S float32
        [R][nh][128][128].  Returns o (int16 bf16 bits [rows][nh][128])."""
        cu_h = np.ascontiguousarray(np.asarray(cu, dtype=np.int32))
        cu_d = cu_dev if cu_dev is not None else _i32(cu_h, self.device)
        par = parents if isinstance(parents, torch.Tensor) else _i32(parents, self.device)
        out = torch.empty_like(q)
        self._cu = (cu_h, cu_d, par)
        check(lib().sd_gdn_tree_verify(q.data_ptr(), k.data_ptr(), v.data_ptr(), alpha.data_ptr(), beta.data_ptr(),
                                       par.data_ptr(), cu_d.data_ptr(), cu_h.ctypes.data, cu_h.size - 1, self.nh,
                                       S.data_ptr(), out.data_ptr(), self.ws.ptr, self.ws.nbytes, self.status.data_ptr(),
                                       stream_ptr(stream)))
        return out

    def commit(self, last, S, stream=None):
        """S of each request becomes the state of its node last[r] (the
        requests and parents of the preceding verify call)."""
        cu_h, cu_d, par = self._cu
        la = last if isinstance(last, torch.Tensor) else _i32(last, self.device)
        check(lib().sd_gdn_commit(par.data_ptr(), cu_d.data_ptr(), cu_h.ctypes.data, cu_h.size - 1, self.nh,
                                  la.data_ptr(), S.data_ptr(), self.ws.ptr, self.ws.nbytes, stream_ptr(stream)))
