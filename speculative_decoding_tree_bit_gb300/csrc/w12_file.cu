// Packed W12 tensors on disk, so that weights are packed once ("SpecPilot:
// AI Agent Framework Boosts Speculative Decoding 10.87x", "(1) W12:
// Lossless 12-bit Weight Format": the 12-bit codes and the sparse list of
// out-of-range weights restore every weight exactly at load time).  Host
// code only: the caller copies the arrays between device and host memory.
//
// File (little-endian): a fixed header, then six sections at 16-byte
// aligned offsets: words, escape indices, escape values, row pointers, the
// escape tile index (tile_ptr, tile_esc).  The header holds the shape, the
// code table, the escape count, each section's offset, size and CRC-32,
// and a CRC-32 of the header itself.  CRC-32 is the IEEE 802.3 checksum
// (reflected polynomial 0xEDB88320, initial value and final xor 0xFFFFFFFF).

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "common.cuh"
#include "sdv.h"

namespace sdv {
namespace {

constexpr char kMagic[8] = {'S', 'D', 'V', 'W', '1', '2', 'F', '\n'};
constexpr uint32_t kVersion = 1;
constexpr int kSections = 6;  // words, esc_idx, esc_val, row_ptr, tile_ptr, tile_esc

struct Section {
  uint64_t offset, bytes;
  uint32_t crc, pad;
};

struct Header {
  char magic[8];
  uint32_t version, header_bytes;
  int64_t N, K, n_escapes, n_tile_ptr;
  uint8_t table[16];
  int32_t n_table, affine;
  Section sec[kSections];
  uint32_t header_crc;  // over every byte before this field
  uint32_t pad;
};
static_assert(sizeof(Header) == 8 + 8 + 32 + 16 + 8 + kSections * 24 + 8, "packed header layout");

struct CrcTable {
  uint32_t t[256];
  CrcTable() {
    for (uint32_t i = 0; i < 256; i++) {
      uint32_t c = i;
      for (int k = 0; k < 8; k++) c = (c & 1u) ? (0xEDB88320u ^ (c >> 1)) : (c >> 1);
      t[i] = c;
    }
  }
};

uint32_t crc32_update(uint32_t crc, const void* data, size_t n) {
  static const CrcTable tab;
  const uint8_t* p = static_cast<const uint8_t*>(data);
  uint32_t c = crc ^ 0xFFFFFFFFu;
  for (size_t i = 0; i < n; i++) c = tab.t[(c ^ p[i]) & 0xFFu] ^ (c >> 8);
  return c ^ 0xFFFFFFFFu;
}

bool shape_ok(int64_t N, int64_t K) {
  return N > 0 && K > 0 && N % 16 == 0 && K % 64 == 0 && N * K < (int64_t(1) << 32);
}

// expected byte size of each section for a tensor of this shape
void section_bytes(int64_t N, int64_t K, int64_t n_esc, int64_t n_tile_ptr, uint64_t out[kSections]) {
  out[0] = (uint64_t)w12_words_count(N, K) * 4;
  out[1] = (uint64_t)n_esc * 4;
  out[2] = (uint64_t)n_esc * 2;
  out[3] = (uint64_t)(N + 1) * 4;
  out[4] = (uint64_t)n_tile_ptr * 4;
  out[5] = (uint64_t)n_esc * 4;
}

struct File {
  FILE* f = nullptr;
  File(const char* path, const char* mode) : f(std::fopen(path, mode)) {}
  ~File() {
    if (f) std::fclose(f);
  }
};

int read_header(FILE* f, Header& h, const char* who) {
  if (std::fread(&h, sizeof h, 1, f) != 1) {
    set_error(std::string(who) + ": short header");
    return SD_ERR_CORRUPT;
  }
  if (std::memcmp(h.magic, kMagic, sizeof kMagic) != 0 || h.version != kVersion || h.header_bytes != sizeof h) {
    set_error(std::string(who) + ": not a W12 file of this version");
    return SD_ERR_CORRUPT;
  }
  if (crc32_update(0, &h, offsetof(Header, header_crc)) != h.header_crc) {
    set_error(std::string(who) + ": header checksum mismatch");
    return SD_ERR_CORRUPT;
  }
  uint64_t want[kSections];
  if (!shape_ok(h.N, h.K) || h.n_escapes < 0 || h.n_escapes > h.N * h.K || h.n_table < 0 || h.n_table > 15 ||
      h.n_tile_ptr != w12_tile_ptr_count(h.N, h.K)) {
    set_error(std::string(who) + ": header fields out of range");
    return SD_ERR_CORRUPT;
  }
  // the decode the kernels take follows this flag: it must be the packer's
  // reading of the stored table (1: empty, or contiguous with its last code
  // below the escape exponent; else 0)
  int aff = 1;
  for (int c = 0; c < h.n_table; c++)
    if (h.table[c] != h.table[0] + c) aff = 0;
  if (h.n_table > 0 && h.table[0] + 15 > 254) aff = 0;
  if (h.affine != aff) {
    set_error(std::string(who) + ": header fields out of range (affine flag does not match the table)");
    return SD_ERR_CORRUPT;
  }
  section_bytes(h.N, h.K, h.n_escapes, h.n_tile_ptr, want);
  for (int s = 0; s < kSections; s++)
    if (h.sec[s].bytes != want[s] || h.sec[s].offset % 16 != 0 || h.sec[s].offset < sizeof h) {
      set_error(std::string(who) + ": section table inconsistent with the shape");
      return SD_ERR_CORRUPT;
    }
  return SD_OK;
}

// A file whose checksums pass may still hold arrays that do not form a
// packed tensor (written from inconsistent buffers): the kernels index
// memory with these values, so a loaded tensor must be one.  Checks, all
// from the layout's definition: escape indices strictly increasing and
// below N*K; row_ptr[n] = the number of escapes before row n; the escape
// tile index exactly the one the side list defines (per 128-row block, the
// block's escapes grouped by 64-column tile in side-list order, each entry
// (bf16 << 16) | (row - 128 b) << 6 | (column - 64 t)).
bool consistent(int64_t N, int64_t K, int64_t n_esc, const uint32_t* esc_idx, const uint16_t* esc_val,
                const uint32_t* row_ptr, const uint32_t* tile_ptr, const uint32_t* tile_esc) {
  const uint64_t NK = (uint64_t)N * (uint64_t)K;
  for (int64_t e = 0; e < n_esc; e++)
    if (esc_idx[e] >= NK || (e > 0 && esc_idx[e] <= esc_idx[e - 1])) return false;
  int64_t e = 0;
  for (int64_t n = 0; n <= N; n++) {
    while (e < n_esc && (uint64_t)esc_idx[e] < (uint64_t)n * (uint64_t)K) e++;
    if ((int64_t)row_ptr[n] != e) return false;
  }
  const int64_t KT = K / 64, NB = (N + 127) / 128;
  std::vector<uint32_t> cursor((size_t)KT);
  for (int64_t b = 0; b < NB; b++) {
    const int64_t n0 = b * 128, n1 = n0 + 128 < N ? n0 + 128 : N;
    const uint32_t e0 = row_ptr[n0], e1 = row_ptr[n1];
    std::fill(cursor.begin(), cursor.end(), 0u);
    for (uint32_t i = e0; i < e1; i++) cursor[(size_t)((esc_idx[i] % (uint64_t)K) / 64)]++;
    uint32_t run = e0;
    for (int64_t t = 0; t < KT; t++) {
      if (tile_ptr[b * KT + t] != run) return false;
      const uint32_t c = cursor[(size_t)t];
      cursor[(size_t)t] = run;
      run += c;
    }
    for (uint32_t i = e0; i < e1; i++) {
      const uint64_t idx = esc_idx[i];
      const uint32_t n = (uint32_t)(idx / (uint64_t)K), k = (uint32_t)(idx % (uint64_t)K);
      const uint32_t want = ((uint32_t)esc_val[i] << 16) | ((n - (uint32_t)n0) << 6) | (k & 63u);
      if (tile_esc[cursor[k / 64]++] != want) return false;
    }
  }
  return (int64_t)tile_ptr[NB * KT] == n_esc;
}

}  // namespace
}  // namespace sdv

using namespace sdv;

extern "C" uint32_t w12_crc32(const void* data, size_t n) { return crc32_update(0, data, n); }

extern "C" int w12_save(const char* path, const w12_tensor* t) {
  if (!path || !t || !shape_ok(t->N, t->K) || t->n_escapes < 0 || t->n_table < 0 || t->n_table > 15 || !t->words ||
      !t->row_ptr || !t->tile_ptr || (t->n_escapes > 0 && (!t->esc_idx || !t->esc_val || !t->tile_esc))) {
    set_error("w12_save: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (t->row_base) {
    set_error("w12_save: the file format holds per-tensor tables only (not a per-channel tensor)");
    return SD_ERR_UNSUPPORTED;
  }
  Header h{};
  std::memcpy(h.magic, kMagic, sizeof kMagic);
  h.version = kVersion;
  h.header_bytes = sizeof h;
  h.N = t->N;
  h.K = t->K;
  h.n_escapes = t->n_escapes;
  h.n_tile_ptr = w12_tile_ptr_count(t->N, t->K);
  std::memcpy(h.table, t->table, 16);
  h.n_table = t->n_table;
  h.affine = t->affine;
  const void* src[kSections] = {t->words, t->esc_idx, t->esc_val, t->row_ptr, t->tile_ptr, t->tile_esc};
  uint64_t bytes[kSections];
  section_bytes(h.N, h.K, h.n_escapes, h.n_tile_ptr, bytes);
  uint64_t off = (sizeof h + 15) & ~uint64_t(15);
  for (int s = 0; s < kSections; s++) {
    h.sec[s].offset = off;
    h.sec[s].bytes = bytes[s];
    h.sec[s].crc = crc32_update(0, bytes[s] ? src[s] : "", bytes[s]);
    off = (off + bytes[s] + 15) & ~uint64_t(15);
  }
  h.header_crc = crc32_update(0, &h, offsetof(Header, header_crc));
  File f(path, "wb");
  if (!f.f) {
    set_error(std::string("w12_save: cannot open ") + path);
    return SD_ERR_IO;
  }
  static const char zeros[16] = {};
  bool ok = std::fwrite(&h, sizeof h, 1, f.f) == 1;
  uint64_t at = sizeof h;
  for (int s = 0; s < kSections && ok; s++) {
    ok = std::fwrite(zeros, 1, h.sec[s].offset - at, f.f) == h.sec[s].offset - at;
    if (ok && bytes[s]) ok = std::fwrite(src[s], 1, bytes[s], f.f) == bytes[s];
    at = h.sec[s].offset + bytes[s];
  }
  ok = ok && std::fflush(f.f) == 0;
  if (!ok) {
    set_error(std::string("w12_save: write failed for ") + path);
    return SD_ERR_IO;
  }
  return SD_OK;
}

extern "C" int w12_load_info(const char* path, w12_meta* meta, int64_t* n_tile_ptr) {
  if (!path || !meta) {
    set_error("w12_load_info: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  File f(path, "rb");
  if (!f.f) {
    set_error(std::string("w12_load_info: cannot open ") + path);
    return SD_ERR_IO;
  }
  Header h;
  const int rc = read_header(f.f, h, "w12_load_info");
  if (rc) return rc;
  meta->N = h.N;
  meta->K = h.K;
  std::memcpy(meta->table, h.table, 16);
  meta->n_table = h.n_table;
  meta->affine = h.affine;
  meta->n_escapes = h.n_escapes;
  if (n_tile_ptr) *n_tile_ptr = h.n_tile_ptr;
  return SD_OK;
}

extern "C" int w12_load(const char* path, uint32_t* words, uint32_t* esc_idx, uint16_t* esc_val, uint32_t* row_ptr,
                        uint32_t* tile_ptr, uint32_t* tile_esc, w12_meta* meta) {
  if (!path || !words || !row_ptr || !tile_ptr || !meta) {
    set_error("w12_load: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  File f(path, "rb");
  if (!f.f) {
    set_error(std::string("w12_load: cannot open ") + path);
    return SD_ERR_IO;
  }
  Header h;
  int rc = read_header(f.f, h, "w12_load");
  if (rc) return rc;
  if (h.n_escapes > 0 && (!esc_idx || !esc_val || !tile_esc)) {
    set_error("w12_load: the file has escapes but no escape buffers were given");
    return SD_ERR_INVALID_ARG;
  }
  void* dst[kSections] = {words, esc_idx, esc_val, row_ptr, tile_ptr, tile_esc};
  for (int s = 0; s < kSections; s++) {
    const uint64_t n = h.sec[s].bytes;
    if (!n) continue;
    if (std::fseek(f.f, (long)h.sec[s].offset, SEEK_SET) != 0 || std::fread(dst[s], 1, n, f.f) != n) {
      set_error("w12_load: file shorter than its section table");
      return SD_ERR_CORRUPT;
    }
    if (crc32_update(0, dst[s], n) != h.sec[s].crc) {
      set_error("w12_load: section checksum mismatch");
      return SD_ERR_CORRUPT;
    }
  }
  if (!consistent(h.N, h.K, h.n_escapes, esc_idx, esc_val, row_ptr, tile_ptr, tile_esc)) {
    set_error("w12_load: the arrays do not form a packed tensor (escape list, row pointers or tile index)");
    return SD_ERR_CORRUPT;
  }
  meta->N = h.N;
  meta->K = h.K;
  std::memcpy(meta->table, h.table, 16);
  meta->n_table = h.n_table;
  meta->affine = h.affine;
  meta->n_escapes = h.n_escapes;
  return SD_OK;
}
