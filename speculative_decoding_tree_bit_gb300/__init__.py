"""Python binding of libsdv, the GB300 tree-verify library (ctypes).

Argument marshalling only: every step of the verify path runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.  The
library must be built (``__graft_entry__.build()`` or ``_build.build()``);
loading the binding without it raises, there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from ._build import INCLUDE, LIB

SD_OK = 0
STATUS_NAMES = {0: "SD_OK", 1: "SD_ERR_INVALID_ARG", 2: "SD_ERR_UNSUPPORTED", 3: "SD_ERR_CUDA", 4: "SD_ERR_OOM",
                5: "SD_ERR_BAD_TREE", 6: "SD_ERR_TIMEOUT", 7: "SD_ERR_CAPACITY", 8: "SD_ERR_BAD_TOKEN",
                9: "SD_ERR_WORKSPACE", 10: "SD_ERR_IO", 11: "SD_ERR_CORRUPT"}


class SdvError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


vp, i32, i64, u8 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint8


class W12Meta(ctypes.Structure):
    _fields_ = [("N", i64), ("K", i64), ("table", u8 * 16), ("n_table", i32), ("affine", i32), ("n_escapes", i64)]


class W12Tensor(ctypes.Structure):
    _fields_ = [("N", i64), ("K", i64), ("words", vp), ("esc_idx", vp), ("esc_val", vp), ("row_ptr", vp),
                ("tile_ptr", vp), ("tile_esc", vp), ("n_escapes", i64), ("table", u8 * 16), ("n_table", i32),
                ("affine", i32), ("row_base", vp)]


class ModelConfig(ctypes.Structure):
    _fields_ = [("n_layers", i32), ("hidden", i32), ("inter", i32), ("n_q_heads", i32), ("n_kv_heads", i32),
                ("head_dim", i32), ("vocab", i32), ("rms_eps", ctypes.c_float), ("rope_base", ctypes.c_float),
                ("rec_eps", ctypes.c_float), ("layer_kind_host", vp), ("max_rows", i32), ("max_requests", i32),
                ("max_positions", i32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [("qkv", W12Tensor), ("o", W12Tensor), ("gate_up", W12Tensor), ("down", W12Tensor),
                ("attn_norm", vp), ("mlp_norm", vp)]


class ModelWeights(ctypes.Structure):
    _fields_ = [("layers_host", vp), ("embed", vp), ("final_norm", vp), ("lm_head", W12Tensor)]


class KV(ctypes.Structure):
    _fields_ = [("k", vp), ("v", vp), ("cap", i64), ("S", vp), ("z", vp), ("ctx_len", vp)]


class PagedKV(ctypes.Structure):
    _fields_ = [("k_pool", vp), ("v_pool", vp), ("n_pages", i32), ("page_size", i32), ("page_table", vp),
                ("max_pages", i32), ("S", vp), ("z", vp), ("ctx_len", vp)]


P = ctypes.POINTER
_SIGS = {
    "sd_last_error": (ctypes.c_char_p, []),
    "sd_version": (ctypes.c_char_p, []),
    "sd_debug_bounded_wait": (ctypes.c_int, [vp, i64, i32, vp]),
    "sd_stream_set_trace": (ctypes.c_int, [vp, i64]),
    "sd_attn_set_trace": (ctypes.c_int, [vp, i64]),
    "sd_stream_trace_launches": (i32, []),
    "sd_stream_grid": (i32, [i32]),
    "w12_words_count": (i64, [i64, i64]),
    "w12_pack_analyze": (ctypes.c_int, [vp, i64, i64, P(W12Meta), vp]),
    "w12_pack_encode": (ctypes.c_int, [vp, vp, P(W12Meta), vp, vp, vp, vp, vp]),
    "w12_unpack": (ctypes.c_int, [P(W12Tensor), vp, vp]),
    "w12_tile_ptr_count": (i64, [i64, i64]),
    "w12_pack_tile_index": (ctypes.c_int, [P(W12Tensor), vp, vp, vp]),
    "sd_w12_linear_workspace": (ctypes.c_size_t, [i64, i64, i32]),
    "sd_w12_linear": (ctypes.c_int, [P(W12Tensor), vp, i32, vp, vp, ctypes.c_size_t, vp]),
    "sd_w12_linear_static": (ctypes.c_int, [P(W12Tensor), vp, i32, vp, vp]),
    "sd_w12_linear_stream_workspace": (ctypes.c_size_t, [i64, i64, i32]),
    "sd_w12_linear_view8_workspace": (ctypes.c_size_t, [i64, i64, i32]),
    "sd_w12_linear_view8": (ctypes.c_int, [P(W12Tensor), vp, vp, i32, vp, vp, ctypes.c_size_t, vp]),
    "sd_w12_linear_stream": (ctypes.c_int, [P(W12Tensor), vp, vp, i32, vp, vp, ctypes.c_size_t, vp]),
    "sd_gemm_set_tc_min_rows": (i32, [i32]),
    "sd_gemm_set_cluster_finish": (i32, [i32]),
    "sd_gemm_set_deferred_finish": (i32, [i32]),
    "sd_gemm_set_strip": (i32, [i32]),
    "sd_attn_set_splits": (i32, [i32]),
    "sd_tree_info": (ctypes.c_int, [vp, i32, i32, vp, vp, vp, vp, vp]),
    "sd_accept": (ctypes.c_int, [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp]),
    "w12_plane8_pack_host": (ctypes.c_int, [vp, i64, i64, vp, i32, vp]),
    "w12_plane8_unpack_host": (ctypes.c_int, [vp, i64, i64, vp, i32, vp, vp, i64, vp]),
    "w12c_pack_host": (ctypes.c_int, [vp, i64, i64, vp, vp, vp, vp, i64, vp, P(i64)]),
    "w12c_pack_analyze": (ctypes.c_int, [vp, vp, i64, i64, vp, vp, P(W12Meta), vp]),
    "w12c_pack_encode": (ctypes.c_int, [vp, vp, i64, i64, vp, vp, vp, vp, vp, vp]),
    "w12c_unpack_host": (ctypes.c_int, [vp, vp, i64, i64, vp, vp, i64, vp]),
    "w12_crc32": (ctypes.c_uint32, [vp, ctypes.c_size_t]),
    "w12_save": (ctypes.c_int, [ctypes.c_char_p, P(W12Tensor)]),
    "w12_load_info": (ctypes.c_int, [ctypes.c_char_p, P(W12Meta), P(i64)]),
    "w12_load": (ctypes.c_int, [ctypes.c_char_p, vp, vp, vp, vp, vp, vp, P(W12Meta)]),
    "sd_select_workspace": (ctypes.c_size_t, [i32]),
    "sd_best_first_select": (ctypes.c_int, [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                            ctypes.c_size_t, vp]),
    "sd_tiny_workspace": (ctypes.c_size_t, [i64, i64, i64, i32]),
    "sd_tiny_verify": (ctypes.c_int, [P(W12Tensor), P(W12Tensor), vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp,
                                      ctypes.c_size_t, vp]),
    "sd_model_row_map": (ctypes.c_int, [i32, i32, i32, i32, i32, vp, i64]),
    "sd_model_create": (ctypes.c_int, [P(ModelConfig), P(ModelWeights), P(vp)]),
    "sd_model_destroy": (ctypes.c_int, [vp]),
    "sd_verify_step": (ctypes.c_int, [vp, vp, vp, i32, P(KV), vp, vp, vp, vp, vp, vp]),
    "sd_forward": (ctypes.c_int, [vp, vp, vp, i32, P(KV), vp, vp, vp]),
    "sd_verify_batch": (ctypes.c_int, [vp, vp, vp, vp, i32, P(PagedKV), vp, vp, vp, vp, vp, vp]),
    "sd_status": (ctypes.c_int, [vp, vp]),
    "sd_model_last_launches": (ctypes.c_int, [vp]),
    "sd_model_final_hidden": (ctypes.c_int, [vp, vp, i32, vp]),
    "sd_model_set_view8": (ctypes.c_int, [vp, vp, i32]),
    "sd_model_set_fused": (ctypes.c_int, [vp, i32]),
    "sd_forward_view8": (ctypes.c_int, [vp, vp, vp, i32, P(KV), vp, vp, vp]),
    "w12_plane8_words_count": (i64, [i64, i64]),
    "w12_plane8_pack": (ctypes.c_int, [vp, vp, P(W12Meta), vp, vp]),
    "sd_gdn_workspace": (ctypes.c_size_t, [i32, i32]),
    "sd_gdn_tree_verify": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, vp, ctypes.c_size_t, vp,
                                          vp]),
    "sd_gdn_commit": (ctypes.c_int, [vp, vp, vp, i32, i32, vp, vp, vp, ctypes.c_size_t, vp]),
    "sd_model_set_timing": (ctypes.c_int, [vp, i32]),
    "sd_model_set_graphs": (ctypes.c_int, [vp, i32]),
    "sd_model_timeline": (ctypes.c_int, [vp, i32, vp, vp, vp]),
}

KERNEL_KINDS = ["tree", "rmsnorm", "gemm_qkv", "attention", "linrec", "gemm_o", "gemm_gate_up", "gemm_down",
                "gemm_lm_head", "accept", "commit", "gemm_stream"]

_lib = None
_lock = threading.Lock()


def lib():
    """The loaded libsdv.so with its signatures declared (raises if unbuilt)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(f"{LIB} is not built: run __graft_entry__.build() first "
                                   "(there is no fallback path)")
            L = ctypes.CDLL(LIB)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def check(rc: int):
    if rc != SD_OK:
        raise SdvError(rc, lib().sd_last_error().decode())


def header_functions() -> list:
    """Names of every function declared in include/*.h."""
    names = set()
    for f in os.listdir(INCLUDE):
        if not f.endswith(".h"):
            continue
        src = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, f)).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**([a-z][a-z0-9_]*)\s*\(",
                                src, flags=re.M))
    return sorted(names)


def stream_ptr(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)
