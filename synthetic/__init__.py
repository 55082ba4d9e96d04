"""Seeded synthetic inputs shared by the CUDA path's harness and by the tests.

Counter-based splitmix64 streams, Box-Muller normals stored as bf16 bits,
random draft trees, copy-rule coins and page permutations.  Nothing here
computes any part of the verify method.  The C source (gen.c) is compiled on
first use into this directory.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_libsynthetic.so")
_lock = threading.Lock()
_lib = None

# Stream ids (tensor_id in the key derivation); one per kind of input.
SID_TREE = 1
SID_COINS = 2
SID_ACT = 3
SID_KV = 4
SID_STATE = 5
SID_ESC = 6
SID_CTX = 7
SID_PAGES = 8
SID_GAMMA = 9
SID_EMBED = 10
SID_LM_HEAD = 11
SID_TINY_W1 = 12
SID_ROOT_TOKEN = 13
SID_CAND_TREE = 14
SID_CAND_LP = 15
SID_CAND_TOKEN = 16
SID_LAYER_BASE = 1000  # + 16 * layer + weight slot


def build(force: bool = False) -> str:
    """Compile gen.c into a shared library next to it (idempotent)."""
    src = os.path.join(_HERE, "gen.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + ".tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            u64, i64, i32, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
            vp = ctypes.c_void_p
            L.sg_mix64.restype = u64
            L.sg_mix64.argtypes = [u64]
            L.sg_key.restype = u64
            L.sg_key.argtypes = [u64, u64]
            L.sg_u64.restype = u64
            L.sg_u64.argtypes = [u64, u64]
            L.sg_uniform.restype = dbl
            L.sg_uniform.argtypes = [u64, u64]
            L.sg_normal.restype = dbl
            L.sg_normal.argtypes = [u64, u64]
            L.sg_normal_bf16.restype = None
            L.sg_normal_bf16.argtypes = [u64, dbl, i64, i64, vp]
            L.sg_normal_f32.restype = None
            L.sg_normal_f32.argtypes = [u64, dbl, i64, i64, vp]
            L.sg_fill_bf16.restype = None
            L.sg_fill_bf16.argtypes = [ctypes.c_uint16, i64, vp]
            L.sg_tree.restype = None
            L.sg_tree.argtypes = [u64, i32, i32, vp]
            L.sg_copy_coins.restype = None
            L.sg_copy_coins.argtypes = [u64, i32, dbl, i32, vp, vp]
            L.sg_uniform_int.restype = None
            L.sg_uniform_int.argtypes = [u64, i64, i64, i64, vp]
            L.sg_permutation.restype = None
            L.sg_permutation.argtypes = [u64, i64, vp]
            L.sg_force_rare_exponents.restype = i64
            L.sg_force_rare_exponents.argtypes = [u64, vp, i64, i64, vp]
            _lib = L
    return _lib


def key(seed: int, stream_id: int) -> int:
    return int(lib().sg_key(seed & (2**64 - 1), stream_id & (2**64 - 1)))


def layer_key(seed: int, layer: int, slot: int) -> int:
    return key(seed, SID_LAYER_BASE + 16 * layer + slot)


def normal_bf16(k: int, n: int, sigma: float, offset: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16) of sigma * N(0,1), elements offset..offset+n-1."""
    if out is None:
        out = np.empty(n, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.size == n and out.flags.c_contiguous
    lib().sg_normal_bf16(k, sigma, offset, n, out.ctypes.data)
    return out


def normal_f32(k: int, n: int, sigma: float, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().sg_normal_f32(k, sigma, offset, n, out.ctypes.data)
    return out


def ones_bf16(n: int) -> np.ndarray:
    return np.full(n, 0x3F80, dtype=np.uint16)


def tree(k: int, M: int, max_depth: int) -> np.ndarray:
    p = np.empty(max(M, 1), dtype=np.int32)
    lib().sg_tree(k, M, max_depth, p.ctypes.data)
    return p[:M].copy()


def chain(M: int) -> np.ndarray:
    return np.arange(-1, M - 1, dtype=np.int32)


def copy_coins(k: int, M: int, p: float, V: int):
    c = np.empty(max(M, 1), dtype=np.uint8)
    t = np.empty(max(M, 1), dtype=np.int32)
    lib().sg_copy_coins(k, M, p, V, c.ctypes.data, t.ctypes.data)
    return c[:M].astype(bool), t[:M].copy()


def uniform_int(k: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in lo .. hi, both ends included."""
    out = np.empty(max(n, 1), dtype=np.int64)
    lib().sg_uniform_int(k, n, lo, hi, out.ctypes.data)
    return out[:n].copy()


def permutation(k: int, n: int) -> np.ndarray:
    out = np.empty(max(n, 1), dtype=np.int32)
    lib().sg_permutation(k, n, out.ctypes.data)
    return out[:n].copy()


def force_rare_exponents(k: int, w: np.ndarray, count: int) -> np.ndarray:
    """In-place on a contiguous uint16 array; returns the chosen flat positions."""
    assert w.dtype == np.uint16 and w.flags.c_contiguous
    pos = np.empty(max(count, 1), dtype=np.int64)
    got = lib().sg_force_rare_exponents(k, w.ctypes.data, w.size, count, pos.ctypes.data)
    return pos[:got].copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Storage conversion (exact): bf16 bits -> float32 values."""
    return (b.astype(np.uint32) << 16).view(np.float32)
