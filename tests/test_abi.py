"""The C ABI without a GPU: the library builds and loads, exports every
function include/*.h declares, and its host-side logic (row maps, argument
checks) behaves."""
import ctypes

import numpy as np
import pytest

import speculative_decoding_tree_bit_gb300 as sdv
from speculative_decoding_tree_bit_gb300 import _build


@pytest.fixture(scope="module")
def L():
    _build.build()
    return sdv.lib()


def test_every_declared_function_is_exported(L):
    names = sdv.header_functions()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert set(names) == set(sdv._SIGS), "binding signatures and header differ"


def test_words_count(L):
    assert L.w12_words_count(16, 64) == 384
    assert L.w12_words_count(151936, 4096) == 151936 * 4096 * 3 // 8


def test_qkv_row_map_pairs_rope_halves(L):
    Hq, Hkv = 4, 2
    N = (Hq + 2 * Hkv) * 128
    m = np.empty(N, np.int32)
    assert L.sd_model_row_map(0, Hq, Hkv, 128, 0, m.ctypes.data, N) == 0
    assert sorted(m.tolist()) == list(range(N))
    for head in range(Hq + Hkv):
        for strip in range(8):
            rows = m[head * 128 + strip * 16: head * 128 + strip * 16 + 16] - head * 128
            assert list(rows[:8]) == list(range(8 * strip, 8 * strip + 8))
            assert list(rows[8:]) == [64 + d for d in range(8 * strip, 8 * strip + 8)]
    assert list(m[(Hq + Hkv) * 128:]) == list(range((Hq + Hkv) * 128, N))


def test_gate_up_row_map_interleaves(L):
    I = 64
    m = np.empty(2 * I, np.int32)
    assert L.sd_model_row_map(1, 4, 2, 128, I, m.ctypes.data, 2 * I) == 0
    assert sorted(m.tolist()) == list(range(2 * I))
    for j in range(I // 8):
        assert list(m[16 * j:16 * j + 8]) == list(range(8 * j, 8 * j + 8))
        assert list(m[16 * j + 8:16 * j + 16]) == list(range(I + 8 * j, I + 8 * j + 8))


def test_host_argument_checks(L):
    meta = sdv.W12Meta()
    # N % 16 != 0 is refused before any device call
    assert L.w12_pack_analyze(ctypes.c_void_p(16), 10, 64, ctypes.byref(meta), None) == 2
    assert b"N % 16" in L.sd_last_error()
    assert L.w12_pack_analyze(None, 16, 64, ctypes.byref(meta), None) == 1
    bad = np.empty(4, np.int32)
    assert L.sd_model_row_map(7, 4, 2, 128, 64, bad.ctypes.data, 4) == 1
    cfg = sdv.ModelConfig()
    cfg.n_layers, cfg.head_dim = 1, 64
    kinds = (ctypes.c_int8 * 1)(0)
    cfg.layer_kind_host = ctypes.addressof(kinds)
    w = sdv.ModelWeights()
    lw = (sdv.LayerWeights * 1)()
    w.layers_host, w.embed, w.final_norm = ctypes.addressof(lw), 16, 16
    h = ctypes.c_void_p()
    assert L.sd_model_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == 2
    assert L.sd_accept(None, None, None, 4, None, None, None, None, None, None) == 1
    # process-wide tuning knobs: host state only, clamped, <= 0 restores the default
    assert L.sd_attn_set_splits(7) == 7
    assert L.sd_attn_set_splits(1000) == 64
    assert L.sd_attn_set_splits(-3) == 0
    assert L.sd_attn_set_splits(0) == 0
    assert L.sd_gemm_set_tc_min_rows(129) == 129
    assert L.sd_gemm_set_tc_min_rows(0) == 65
    assert L.sd_gemm_set_tc_min_rows(-1) == 65
    # the skinny GEMM's paths: strip-parallel on, deferred and cluster
    # finishes off by default; < 0 only queries
    assert L.sd_gemm_set_strip(-1) == 1
    assert L.sd_gemm_set_deferred_finish(-1) == 0
    assert L.sd_gemm_set_cluster_finish(-1) == 0
    for setter, default in ((L.sd_gemm_set_strip, 1), (L.sd_gemm_set_deferred_finish, 0),
                            (L.sd_gemm_set_cluster_finish, 0)):
        assert setter(1 - default) == 1 - default
        assert setter(-1) == 1 - default
        assert setter(default) == default
    # best-first selection: argument checks run before any device work
    assert L.sd_select_workspace(0) == 0
    assert L.sd_select_workspace(1000) == 20 * 1000 + 16
    d = ctypes.c_void_p(16)
    sel = lambda R, n, budget, cap, ws=1 << 20, tokens=d, out_tokens=d: L.sd_best_first_select(
        d, d, d, R, n, budget, cap, tokens, d, d, d, out_tokens, None, d, d, ws, None)
    assert sel(0, 4, 4, 1) == 1          # no request
    assert sel(3, 2, 4, 1) == 1          # fewer candidates than requests
    assert sel(3, 9, 2, 1) == 1          # budget below the number of roots
    assert sel(3, 9, 4, 0) == 1          # cap below one
    assert sel(3, 9, 4, 1, tokens=None) == 1  # gathered tokens without input tokens
    assert sel(3, 16385, 4, 1) == 2      # more candidates than one call takes
    assert sel(3, 9, 4, 1, ws=100) == 9  # workspace too small
    assert L.sd_best_first_select(None, d, d, 1, 1, 1, 1, None, d, d, d, None, None, d, d, 1 << 20, None) == 1
    assert L.sd_tree_info(ctypes.c_void_p(16), 65, 0, ctypes.c_void_p(16), ctypes.c_void_p(16),
                          ctypes.c_void_p(16), None, None) == 2


def test_header_is_plain_c_and_links_from_c(L, tmp_path):
    """include/sdv.h is a C header (C99, pedantic) and a C program linked
    against the library calls it (host-only entry points: no GPU)."""
    import os
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    inc = os.path.join(root, "include")
    libdir = os.path.dirname(_build.build())
    src = tmp_path / "use_sdv.c"
    src.write_text(
        '#include <stdio.h>\n#include "sdv.h"\n'
        'int main(void) {\n'
        '  const char msg[] = "123456789";\n'
        '  if (w12_crc32(msg, 9) != 0xCBF43926u) return 1;\n'
        '  if (w12_words_count(16, 64) != 384) return 2;\n'
        '  if (sd_select_workspace(10) != 216) return 3;\n'
        '  if (sd_best_first_select(0, 0, 0, 1, 1, 1, 1, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0) != SD_ERR_INVALID_ARG) return 4;\n'
        '  printf("ok\\n");\n  return 0;\n}\n')
    exe = tmp_path / "use_sdv"
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc, str(src), "-L", libdir,
                        "-lsdv", "-Wl,-rpath," + libdir, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
