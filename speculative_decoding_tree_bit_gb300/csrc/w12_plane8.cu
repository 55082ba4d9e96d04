// The nested 8-bit plane of W12 ("SpecPilot: AI Agent Framework Boosts
// Speculative Decoding 10.87x", "(3) Two-Level Verification": the first
// round verifies with W12's nested 8-bit weight view).  A weight's 12-bit
// field is sign, 4-bit exponent code, 7-bit mantissa; its high byte (sign,
// code, top 3 mantissa bits) is the 8-bit view, stored here as its own plane
// (1 byte per weight) so that a low-precision pass streams two thirds of the
// 12-bit bytes.  Offline (host) code: packer and unpacker of the plane.
//
// Layout: per 16-row strip and 64-column super-tile, 2 planes x 32 lanes x
// 4 sub-tiles of u32 (1024 bytes), the lane mapping of the 12-bit layout
// (lane = 4 g + q, sub-tile j: rows g and g + 8, columns 16 j + 2 q + {0, 1}
// and + 8): plane 0 holds the bytes of (row g, c), (row g, c + 1),
// (row g + 8, c), (row g + 8, c + 1); plane 1 the same at column c + 8.  On
// the contiguous-table path a byte b decodes to the bf16
// ((b & 0x80) << 8) | (((b & 0x7F) << 4) + (table[0] << 7)).  The device
// packer writes the same layout from the bf16 weights on the device.

#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "sdv.h"

namespace sdv {

struct Plane8Lut {
  uint8_t code_of[256];  // exponent -> code (15: not in the table, escaped)
};

// One thread per (strip, super-tile, lane, sub-tile): the two words of that
// lane's fragment bytes.
__global__ void k_plane8_encode(const uint16_t* __restrict__ w, const int32_t* __restrict__ row_src, int64_t N,
                                int64_t K, Plane8Lut lut, uint32_t* __restrict__ plane) {
  const int64_t KT = K / 64;
  const int64_t total = (N / 16) * KT * 128;
  for (int64_t id = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; id < total; id += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(id & 3), lane = (int)((id >> 2) & 31);
    const int64_t st = id >> 7;  // strip * KT + tile
    const int64_t s = st / KT, t = st % KT;
    const int g = lane >> 2, q = lane & 3;
    const int64_t r0 = row_src ? row_src[s * 16 + g] : s * 16 + g;
    const int64_t r1 = row_src ? row_src[s * 16 + g + 8] : s * 16 + g + 8;
    const int64_t c = t * 64 + j * 16 + 2 * q;
    auto byte_of = [&](uint32_t b) -> uint32_t {
      const uint32_t code = lut.code_of[(b >> 7) & 0xFF];
      if (code == 15) return 15u << 3;
      return ((b >> 15) << 7) | (code << 3) | ((b >> 4) & 7u);
    };
#pragma unroll
    for (int p = 0; p < 2; p++) {
      const uint32_t a = *reinterpret_cast<const uint32_t*>(w + r0 * K + c + 8 * p);
      const uint32_t b = *reinterpret_cast<const uint32_t*>(w + r1 * K + c + 8 * p);
      plane[st * 256 + p * 128 + lane * 4 + j] =
          byte_of(a & 0xFFFF) | (byte_of(a >> 16) << 8) | (byte_of(b & 0xFFFF) << 16) | (byte_of(b >> 16) << 24);
    }
  }
}

namespace {

inline int64_t plane8_word(int64_t s, int64_t t, int64_t KT, int p, int lane, int j) {
  return (s * KT + t) * 256 + p * 128 + lane * 4 + j;
}

bool plane8_shape_ok(int64_t N, int64_t K) {
  return N > 0 && K > 0 && N % 16 == 0 && K % 64 == 0 && N * K < (int64_t(1) << 32);
}

}  // namespace
}  // namespace sdv

using namespace sdv;

extern "C" int w12_plane8_pack_host(const uint16_t* w, int64_t N, int64_t K, const uint8_t* table, int32_t n_table,
                                    uint32_t* plane) {
  if (!w || !table || !plane || n_table < 0 || n_table > 15) {
    set_error("w12_plane8_pack_host: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (!plane8_shape_ok(N, K)) {
    set_error("w12_plane8_pack_host: N % 16, K % 64 and N*K < 2^32 required");
    return SD_ERR_UNSUPPORTED;
  }
  uint8_t code_of[256];
  for (int e = 0; e < 256; e++) code_of[e] = 15;
  for (int c = 0; c < n_table; c++) code_of[table[c]] = (uint8_t)c;
  auto byte_of = [&](uint16_t b) -> uint32_t {
    const uint32_t code = code_of[(b >> 7) & 0xFF];
    if (code == 15) return 15u << 3;  // escaped: code 15, sign and mantissa zero
    return ((uint32_t)(b >> 15) << 7) | (code << 3) | ((b >> 4) & 7u);
  };
  const int64_t KT = K / 64;
  for (int64_t s = 0; s < N / 16; s++)
    for (int64_t t = 0; t < KT; t++)
      for (int lane = 0; lane < 32; lane++)
        for (int j = 0; j < 4; j++) {
          const int g = lane >> 2, q = lane & 3;
          const int64_t r0 = s * 16 + g, r1 = r0 + 8;
          const int64_t c = t * 64 + j * 16 + 2 * q;
          for (int p = 0; p < 2; p++) {
            const int64_t cc = c + 8 * p;
            const uint32_t v = byte_of(w[r0 * K + cc]) | (byte_of(w[r0 * K + cc + 1]) << 8) |
                               (byte_of(w[r1 * K + cc]) << 16) | (byte_of(w[r1 * K + cc + 1]) << 24);
            plane[plane8_word(s, t, KT, p, lane, j)] = v;
          }
        }
  return SD_OK;
}

extern "C" int64_t w12_plane8_words_count(int64_t N, int64_t K) { return N * K / 4; }

extern "C" int w12_plane8_pack(const uint16_t* w, const int32_t* row_src, const w12_meta* meta, uint32_t* plane,
                               void* stream) {
  if (!w || !meta || !plane || meta->n_table < 0 || meta->n_table > 15) {
    set_error("w12_plane8_pack: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (!plane8_shape_ok(meta->N, meta->K)) {
    set_error("w12_plane8_pack: N % 16, K % 64 and N*K < 2^32 required");
    return SD_ERR_UNSUPPORTED;
  }
  Plane8Lut lut;
  for (int e = 0; e < 256; e++) lut.code_of[e] = 15;
  for (int c = 0; c < meta->n_table; c++) lut.code_of[meta->table[c]] = (uint8_t)c;
  const int64_t total = (meta->N / 16) * (meta->K / 64) * 128;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, 65536);
  k_plane8_encode<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(w, row_src, meta->N, meta->K, lut, plane);
  SD_CK(cudaGetLastError());
  return SD_OK;
}

extern "C" int w12_plane8_unpack_host(const uint32_t* plane, int64_t N, int64_t K, const uint8_t* table,
                                      int32_t n_table, const uint32_t* esc_idx, const uint16_t* esc_val,
                                      int64_t n_escapes, uint16_t* w) {
  if (!plane || !table || !w || n_table < 0 || n_table > 15 || n_escapes < 0 ||
      (n_escapes > 0 && (!esc_idx || !esc_val))) {
    set_error("w12_plane8_unpack_host: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (!plane8_shape_ok(N, K)) {
    set_error("w12_plane8_unpack_host: N % 16, K % 64 and N*K < 2^32 required");
    return SD_ERR_UNSUPPORTED;
  }
  uint32_t exp_of[16];
  for (int c = 0; c < 16; c++) exp_of[c] = c < n_table ? table[c] : 0u;
  auto bf16_of = [&](uint32_t b) -> uint16_t {
    return (uint16_t)(((b & 0x80u) << 8) | (exp_of[(b >> 3) & 15u] << 7) | ((b & 7u) << 4));
  };
  const int64_t KT = K / 64;
  for (int64_t s = 0; s < N / 16; s++)
    for (int64_t t = 0; t < KT; t++)
      for (int lane = 0; lane < 32; lane++)
        for (int j = 0; j < 4; j++) {
          const int g = lane >> 2, q = lane & 3;
          const int64_t r0 = s * 16 + g, r1 = r0 + 8;
          const int64_t c = t * 64 + j * 16 + 2 * q;
          for (int p = 0; p < 2; p++) {
            const int64_t cc = c + 8 * p;
            const uint32_t v = plane[plane8_word(s, t, KT, p, lane, j)];
            w[r0 * K + cc] = bf16_of(v & 0xFFu);
            w[r0 * K + cc + 1] = bf16_of((v >> 8) & 0xFFu);
            w[r1 * K + cc] = bf16_of((v >> 16) & 0xFFu);
            w[r1 * K + cc + 1] = bf16_of(v >> 24);
          }
        }
  // escaped weights: their exact value from the side list, seen through the same view
  for (int64_t e = 0; e < n_escapes; e++) {
    if ((uint64_t)esc_idx[e] >= (uint64_t)N * (uint64_t)K) {
      set_error("w12_plane8_unpack_host: escape index out of range");
      return SD_ERR_CORRUPT;
    }
    w[esc_idx[e]] = (uint16_t)(esc_val[e] & 0xFFF0u);
  }
  return SD_OK;
}
