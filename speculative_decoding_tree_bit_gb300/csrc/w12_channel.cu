// Per-output-channel W12, host packer and unpacker ("SpecPilot: AI Agent
// Framework Boosts Speculative Decoding 10.87x", "(1) W12: Lossless 12-bit
// Weight Format", read literally: a 4-bit exponent offset within each output
// channel).  Row n keeps base[n], the exponent that starts the 15-exponent
// window holding most of the row's weights (the smaller base on ties); a
// weight stores its sign, e - base[n] (15: escaped, its bf16 in the side
// list) and its 7-bit mantissa.  The words use the per-tensor format's
// layout unchanged (the register decode then adds the row's base where the
// contiguous-table path adds the tensor's), escaped weights store code 15
// with sign and mantissa zero, and the side list and row pointers are the
// same as the per-tensor format's.  Offline (host) code.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>

#include "common.cuh"
#include "sdv.h"

namespace sdv {
namespace {

// u32 index of the word holding the fields of (strip s, super-tile t, lane,
// sub-tile j) in plane p: [strip][super-tile][plane][lane][sub-tile]
inline int64_t word_index(int64_t s, int64_t t, int64_t KT, int p, int lane, int j) {
  return (s * KT + t) * 384 + p * 128 + lane * 4 + j;
}

inline uint32_t field_of(uint16_t b, uint32_t base) {
  const uint32_t e = (b >> 7) & 0xFFu;
  if (e < base || e > base + 14) return 15u << 7;
  return ((uint32_t)(b >> 15) << 11) | ((e - base) << 7) | (b & 0x7Fu);
}

bool shape_ok(int64_t N, int64_t K) {
  return N > 0 && K > 0 && N % 16 == 0 && K % 64 == 0 && N * K < (int64_t(1) << 32);
}

}  // namespace
}  // namespace sdv

using namespace sdv;

extern "C" int w12c_pack_host(const uint16_t* w, int64_t N, int64_t K, uint8_t* base, uint32_t* words,
                              uint32_t* esc_idx, uint16_t* esc_val, int64_t esc_cap, uint32_t* row_ptr,
                              int64_t* n_escapes) {
  if (!w || !base || !words || !row_ptr || !n_escapes || esc_cap < 0 || (esc_cap > 0 && (!esc_idx || !esc_val))) {
    set_error("w12c_pack_host: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (!shape_ok(N, K)) {
    set_error("w12c_pack_host: N % 16, K % 64 and N*K < 2^32 required");
    return SD_ERR_UNSUPPORTED;
  }
  // bases: per row, the window b .. b+14 (b <= 241) covering the most exponents
  std::vector<uint32_t> hist(256);
  int64_t n_esc = 0;
  for (int64_t n = 0; n < N; n++) {
    std::fill(hist.begin(), hist.end(), 0u);
    for (int64_t k = 0; k < K; k++) hist[(w[n * K + k] >> 7) & 0xFF]++;
    uint32_t cover = 0;
    for (int e = 0; e < 15; e++) cover += hist[e];
    uint32_t best = cover, best_b = 0;
    for (uint32_t b = 1; b <= 241; b++) {
      cover += hist[b + 14] - hist[b - 1];
      if (cover > best) {
        best = cover;
        best_b = b;
      }
    }
    base[n] = (uint8_t)best_b;
    n_esc += K - best;
  }
  *n_escapes = n_esc;
  if (n_esc > esc_cap) {
    set_error("w12c_pack_host: escape buffers too small (*n_escapes holds the count)");
    return SD_ERR_WORKSPACE;
  }
  // words: the per-tensor layout, fields coded against the row's base
  const int64_t KT = K / 64;
  for (int64_t s = 0; s < N / 16; s++)
    for (int64_t t = 0; t < KT; t++)
      for (int lane = 0; lane < 32; lane++)
        for (int j = 0; j < 4; j++) {
          const int g = lane >> 2, q = lane & 3;
          const int64_t r_lo = s * 16 + g, r_hi = r_lo + 8;
          const int64_t c0 = t * 64 + j * 16 + 2 * q;
          const int64_t rows[4] = {r_lo, r_hi, r_lo, r_hi};
          const int64_t cols[4] = {c0, c0, c0 + 8, c0 + 8};
          uint32_t f[4][2];
          for (int p = 0; p < 4; p++)
            for (int h = 0; h < 2; h++) f[p][h] = field_of(w[rows[p] * K + cols[p] + h], base[rows[p]]);
          // planes 0..2 hold fields 0..2 directly (sign in bit 15, the rest in
          // bits 0..10) and the fourth field's nibbles in bits 11..14
          for (int p = 0; p < 3; p++) {
            uint32_t v = 0;
            for (int h = 0; h < 2; h++) {
              const uint32_t half = (f[p][h] & 0x7FFu) | ((f[p][h] >> 11) << 15) | (((f[3][h] >> (4 * p)) & 0xFu) << 11);
              v |= half << (16 * h);
            }
            words[word_index(s, t, KT, p, lane, j)] = v;
          }
        }
  // side list in flat order, row pointers
  int64_t e = 0;
  for (int64_t n = 0; n < N; n++) {
    row_ptr[n] = (uint32_t)e;
    const uint32_t b = base[n];
    for (int64_t k = 0; k < K; k++) {
      const uint16_t x = w[n * K + k];
      const uint32_t ex = (x >> 7) & 0xFF;
      if (ex < b || ex > b + 14) {
        esc_idx[e] = (uint32_t)(n * K + k);
        esc_val[e] = x;
        e++;
      }
    }
  }
  row_ptr[N] = (uint32_t)e;
  return SD_OK;
}

extern "C" int w12c_unpack_host(const uint32_t* words, const uint8_t* base, int64_t N, int64_t K,
                                const uint32_t* esc_idx, const uint16_t* esc_val, int64_t n_escapes, uint16_t* w) {
  if (!words || !base || !w || n_escapes < 0 || (n_escapes > 0 && (!esc_idx || !esc_val))) {
    set_error("w12c_unpack_host: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (!shape_ok(N, K)) {
    set_error("w12c_unpack_host: N % 16, K % 64 and N*K < 2^32 required");
    return SD_ERR_UNSUPPORTED;
  }
  const int64_t KT = K / 64;
  for (int64_t s = 0; s < N / 16; s++)
    for (int64_t t = 0; t < KT; t++)
      for (int lane = 0; lane < 32; lane++)
        for (int j = 0; j < 4; j++) {
          const int g = lane >> 2, q = lane & 3;
          const int64_t r_lo = s * 16 + g, r_hi = r_lo + 8;
          const int64_t c0 = t * 64 + j * 16 + 2 * q;
          const int64_t rows[4] = {r_lo, r_hi, r_lo, r_hi};
          const int64_t cols[4] = {c0, c0, c0 + 8, c0 + 8};
          uint32_t v[3];
          for (int p = 0; p < 3; p++) v[p] = words[word_index(s, t, KT, p, lane, j)];
          for (int h = 0; h < 2; h++) {
            uint32_t f[4];
            for (int p = 0; p < 3; p++) {
              const uint32_t half = (v[p] >> (16 * h)) & 0xFFFFu;
              f[p] = (half & 0x7FFu) | ((half >> 15) << 11);
            }
            f[3] = 0;
            for (int p = 0; p < 3; p++) f[3] |= (((v[p] >> (16 * h)) >> 11) & 0xFu) << (4 * p);
            for (int p = 0; p < 4; p++) {
              const uint32_t code = (f[p] >> 7) & 15u;
              const uint32_t e = code == 15 ? 0u : (uint32_t)base[rows[p]] + code;
              w[rows[p] * K + cols[p] + h] = (uint16_t)(((f[p] >> 11) << 15) | ((e & 0xFFu) << 7) | (f[p] & 0x7Fu));
            }
          }
        }
  for (int64_t e = 0; e < n_escapes; e++) {
    if ((uint64_t)esc_idx[e] >= (uint64_t)N * (uint64_t)K) {
      set_error("w12c_unpack_host: escape index out of range");
      return SD_ERR_CORRUPT;
    }
    w[esc_idx[e]] = esc_val[e];
  }
  return SD_OK;
}
