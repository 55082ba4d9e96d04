"""W12 tensors on disk (w12_save, w12_load_info, w12_load), host memory only,
so no GPU: a packed tensor written and read back restores every weight bit
for bit; each section's and the header's CRC-32 catch a changed byte; a
short or foreign file is rejected; bad arguments return their codes."""
import ctypes
import struct
import zlib

import numpy as np
import pytest

import oracle
import synthetic
import speculative_decoding_tree_bit_gb300 as sdv
from speculative_decoding_tree_bit_gb300 import _build

SECTIONS = ("words", "esc_idx", "esc_val", "row_ptr", "tile_ptr", "tile_esc")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return sdv.lib()


def _packed(N, K, seed, rare=0, no_escapes=False):
    if no_escapes:
        # every exponent in 110 .. 124: one 15-exponent table covers all
        e = synthetic.uniform_int(synthetic.key(seed, 1), N * K, 110, 124).astype(np.uint16)  # bounds inclusive
        m = synthetic.uniform_int(synthetic.key(seed, 2), N * K, 0, 255).astype(np.uint16)
        W = ((m & 0x80) << 8 | (e << 7) | (m & 0x7F)).astype(np.uint16).reshape(N, K)
    else:
        W = synthetic.normal_bf16(synthetic.key(seed, 1), N * K, 0.02).reshape(N, K)
    if rare:
        synthetic.force_rare_exponents(synthetic.key(seed, 2), W, rare)
    p = oracle.w12_pack(W)
    return W, p


def _tile_index(N, K, esc_idx, esc_val):
    """The escape tile index as the header defines it: per 128-row block and
    64-column tile, the block's escapes in side-list order, each entry
    (bf16 << 16) | (row - 128 b) << 6 | (column - 64 t)."""
    KT, NB = K // 64, (N + 127) // 128
    ptr, ent = [], []
    for b in range(NB):
        mine = [(int(i), int(v)) for i, v in zip(esc_idx, esc_val) if b * 128 <= int(i) // K < (b + 1) * 128]
        for t in range(KT):
            ptr.append(len(ent))
            for i, v in mine:
                n, k = divmod(i, K)
                if k // 64 == t:
                    ent.append((v << 16) | ((n - 128 * b) << 6) | (k & 63))
    ptr.append(len(ent))
    return np.array(ptr, np.uint32), np.array(ent, np.uint32)


def _tensor(L, p, seed):
    """W12Tensor over host arrays: the oracle's words / escapes / row
    pointers and the escape tile index they define."""
    tp, te = _tile_index(p.N, p.K, p.esc_idx, p.esc_val)
    assert tp.size == int(L.w12_tile_ptr_count(p.N, p.K))
    a = {"words": np.ascontiguousarray(p.words, dtype=np.uint32),
         "esc_idx": np.ascontiguousarray(p.esc_idx, dtype=np.uint32),
         "esc_val": np.ascontiguousarray(p.esc_val, dtype=np.uint16),
         "row_ptr": np.ascontiguousarray(p.row_ptr, dtype=np.uint32),
         "tile_ptr": tp, "tile_esc": te}
    t = sdv.W12Tensor()
    t.N, t.K, t.n_escapes = p.N, p.K, p.n_esc
    for k in SECTIONS:
        setattr(t, k, a[k].ctypes.data if a[k].size else None)
    tab = list(p.table)
    for i, e in enumerate(tab):
        t.table[i] = int(e)
    t.n_table = len(tab)
    # the packer's reading: an empty table, or a contiguous one whose last code
    # stays below the escape exponent
    t.affine = int(len(tab) == 0 or (all(tab[c] == tab[0] + c for c in range(len(tab))) and tab[0] + 15 <= 254))
    return t, a


def _read(L, path):
    meta = sdv.W12Meta()
    ntp = ctypes.c_int64()
    rc = L.w12_load_info(str(path).encode(), ctypes.byref(meta), ctypes.byref(ntp))
    if rc:
        return rc, None, None
    ne = max(int(meta.n_escapes), 1)
    b = {"words": np.zeros(int(L.w12_words_count(meta.N, meta.K)), np.uint32), "esc_idx": np.zeros(ne, np.uint32),
         "esc_val": np.zeros(ne, np.uint16), "row_ptr": np.zeros(int(meta.N) + 1, np.uint32),
         "tile_ptr": np.zeros(int(ntp.value), np.uint32), "tile_esc": np.zeros(ne, np.uint32)}
    rc = L.w12_load(str(path).encode(), *(b[k].ctypes.data for k in SECTIONS), ctypes.byref(meta))
    return rc, meta, b


def test_crc32_is_the_ieee_checksum(L):
    msg = b"123456789"
    assert L.w12_crc32(msg, len(msg)) == 0xCBF43926  # the standard check value
    data = synthetic.uniform_int(synthetic.key(7, 7), 10000, 0, 255).astype(np.uint8)
    assert L.w12_crc32(data.ctypes.data, data.size) == zlib.crc32(data.tobytes())
    assert L.w12_crc32(b"", 0) == 0


@pytest.mark.parametrize("rare,no_escapes", [(0, True), (0, False), (40, False)])
def test_round_trip_restores_every_weight(L, tmp_path, rare, no_escapes):
    W, p = _packed(64, 192, 11 + rare, rare, no_escapes)
    assert (p.n_esc == 0) if no_escapes else p.n_esc >= rare
    t, a = _tensor(L, p, 5)
    path = tmp_path / "w.w12"
    assert L.w12_save(str(path).encode(), ctypes.byref(t)) == 0
    rc, meta, b = _read(L, path)
    assert rc == 0
    assert (meta.N, meta.K, meta.n_escapes, meta.n_table, meta.affine) == (p.N, p.K, p.n_esc, t.n_table, t.affine)
    assert list(meta.table[:meta.n_table]) == list(p.table)
    for k in SECTIONS:
        n = a[k].size
        np.testing.assert_array_equal(b[k][:n], a[k])
    back = oracle.W12(p.N, p.K, np.array(meta.table[:meta.n_table], np.uint8), b["words"],
                      b["esc_idx"][:p.n_esc].copy(), b["esc_val"][:p.n_esc].copy(), b["row_ptr"])
    np.testing.assert_array_equal(oracle.w12_unpack(back), W)


def test_every_changed_byte_is_caught(L, tmp_path):
    W, p = _packed(32, 128, 21, 12)
    t, a = _tensor(L, p, 6)
    path = tmp_path / "w.w12"
    assert L.w12_save(str(path).encode(), ctypes.byref(t)) == 0
    raw = bytearray(path.read_bytes())
    # one byte inside each section, and bytes of the header
    offs = [struct.unpack_from("<Q", raw, 72 + 24 * s)[0] for s in range(6)]
    sizes = [struct.unpack_from("<Q", raw, 80 + 24 * s)[0] for s in range(6)]
    for s in range(6):
        assert sizes[s] > 0
        bad = bytearray(raw)
        bad[offs[s] + sizes[s] // 2] ^= 0x10
        path.write_bytes(bad)
        assert _read(L, path)[0] == 11
    for pos in (0, 9, 20, 50, 100, 216):
        bad = bytearray(raw)
        bad[pos] ^= 0x01
        path.write_bytes(bad)
        assert _read(L, path)[0] == 11
    path.write_bytes(raw[: len(raw) - 7])       # short file
    assert _read(L, path)[0] == 11
    path.write_bytes(raw[:100])                 # short header
    assert _read(L, path)[0] == 11
    path.write_bytes(raw)
    assert _read(L, path)[0] == 0


def test_bad_arguments_and_paths(L, tmp_path):
    W, p = _packed(16, 64, 31)
    t, a = _tensor(L, p, 8)
    assert L.w12_save(None, ctypes.byref(t)) == 1
    t.N = 24                                      # not a multiple of 16
    assert L.w12_save(str(tmp_path / "x").encode(), ctypes.byref(t)) == 1
    t.N = 16
    assert L.w12_save(str(tmp_path).encode(), ctypes.byref(t)) == 10   # a directory
    meta = sdv.W12Meta()
    assert L.w12_load_info(str(tmp_path / "missing").encode(), ctypes.byref(meta), None) == 10
    assert L.w12_load_info(str(tmp_path / "missing").encode(), None, None) == 1


def test_python_save_and_load_round_trip(L, tmp_path):
    # the binding's save / load on CPU tensors (the device copies are the only
    # step the GPU path adds)
    import torch
    from speculative_decoding_tree_bit_gb300 import model as M
    W, p = _packed(48, 128, 41, 9)
    t, a = _tensor(L, p, 9)
    meta = sdv.W12Meta()
    meta.N, meta.K, meta.n_escapes, meta.n_table, meta.affine = p.N, p.K, p.n_esc, t.n_table, t.affine
    for i in range(16):
        meta.table[i] = t.table[i]
    as_t = {k: torch.from_numpy(a[k].view(np.int32 if a[k].dtype == np.uint32 else np.int16).copy()) for k in SECTIONS}
    packed = M.Packed(meta, as_t["words"], as_t["esc_idx"], as_t["esc_val"], as_t["row_ptr"], as_t["tile_ptr"],
                      as_t["tile_esc"])
    path = tmp_path / "p.w12"
    M.save(packed, path)
    m2, arrays = M.load_host(path)
    assert (m2.N, m2.K, m2.n_escapes) == (p.N, p.K, p.n_esc)
    for k in SECTIONS:
        np.testing.assert_array_equal(arrays[k][:a[k].size].view(a[k].dtype), a[k])
    back = M.load(path, device="cpu")
    assert (back.N, back.K, back.n_escapes) == (p.N, p.K, p.n_esc)
    np.testing.assert_array_equal(back.words.numpy().view(np.uint32), a["words"])
    with pytest.raises(sdv.SdvError):
        M.load_host(tmp_path / "missing.w12")


@pytest.mark.parametrize("fault", ["esc_order", "esc_range", "row_ptr", "tile_ptr", "tile_entry", "tile_total"])
def test_checksummed_but_inconsistent_arrays_are_rejected(L, tmp_path, fault):
    # w12_save writes whatever it is given (with valid checksums); w12_load
    # must still refuse arrays that are not a packed tensor
    W, p = _packed(160, 128, 51, 30)  # two row blocks, the second ragged
    t, a = _tensor(L, p, 10)
    b = {k: v.copy() for k, v in a.items()}
    if fault == "esc_order":
        b["esc_idx"][[3, 4]] = b["esc_idx"][[4, 3]]
    elif fault == "esc_range":
        b["esc_idx"][-1] = p.N * p.K
    elif fault == "row_ptr":
        b["row_ptr"][5] += 1
    elif fault == "tile_ptr":
        b["tile_ptr"][1] += 1
    elif fault == "tile_entry":
        b["tile_esc"][2] ^= 1 << 13  # a row field past the block
    else:
        b["tile_ptr"][-1] -= 1
    for k in SECTIONS:
        setattr(t, k, b[k].ctypes.data if b[k].size else None)
    path = tmp_path / "bad.w12"
    assert L.w12_save(str(path).encode(), ctypes.byref(t)) == 0
    assert _read(L, path)[0] == 11
    assert b"packed tensor" in L.sd_last_error()



@pytest.mark.parametrize("affine", ["flipped", 7])
def test_affine_flag_must_match_the_table(L, tmp_path, affine):
    # the kernels pick their decode from this flag: a checksummed header whose
    # flag is not the packer's reading of its own table is refused
    W, p = _packed(160, 128, 52, 30)
    t, a = _tensor(L, p, 11)
    good = int(t.affine)
    t.affine = (1 - good) if affine == "flipped" else affine
    path = tmp_path / "aff.w12"
    assert L.w12_save(str(path).encode(), ctypes.byref(t)) == 0
    assert _read(L, path)[0] == 11
    assert b"affine" in L.sd_last_error()
    t.affine = good
    assert L.w12_save(str(path).encode(), ctypes.byref(t)) == 0
    assert _read(L, path)[0] == 0
