// Device building blocks of the fused W12 GEMM shared by the per-GEMM kernel
// (gemm.cu) and the persistent GEMM-chain kernel (chain.cu).
#pragma once

#include "gemm.cuh"

namespace sdv {

constexpr int kNCW = 8;            // consumer warps
constexpr int kRB = kNCW;          // strips per row block
constexpr int kThreads = (kNCW + 1) * 32;
constexpr int kStripBytes = 1536;  // one strip x one super-tile (16 x 64 x 12 bit)

template <int NT>
struct Cfg {
  static constexpr int MP = NT * 8;    // padded rows (tokens) per launch
  static constexpr int XB = MP * 128;  // x tile bytes per stage (64 columns of bf16)
  static constexpr int WB = kRB * kStripBytes;
  static constexpr int S = NT <= 1 ? 8 : NT <= 2 ? 7 : NT <= 4 ? 6 : NT <= 8 ? 5 : 4;
  static constexpr int SMEM = 1024 + S * (XB + WB) + 2 * S * 8 + kNCW * MP * 8 + 16;
};

struct GemmParams {
  const uint32_t* words;
  int64_t N, K;
  int KT, NS, NB;
  int64_t U;
  uint32_t base2;
  uint32_t tab[4];
  float esc_slot;
  const uint32_t* row_ptr;
  const uint32_t* esc_idx;
  const uint16_t* esc_val;
  const uint16_t* x;
  int M, m0;
  float* partial;
  int32_t* counters;
  GemmEpilogue e;
  int32_t* status;
};

__device__ __forceinline__ uint32_t lut_exp(uint32_t c, const uint32_t* tab) {
  const uint32_t lo = __byte_perm(tab[0], tab[1], c & 7);
  const uint32_t hi = __byte_perm(tab[2], tab[3], c & 7);
  return ((c & 8) ? hi : lo) & 0xFF;
}

// Stored half (sign in bit 15, code in bits 7..10, mantissa 0..6) -> bf16.
__device__ __forceinline__ uint32_t general_pair(uint32_t v, const uint32_t* tab) {
  const uint32_t e0 = lut_exp((v >> 7) & 15, tab), e1 = lut_exp((v >> 23) & 15, tab);
  return (v & 0x807F807Fu) | (e0 << 7) | (e1 << 23);
}

template <bool AFFINE>
__device__ __forceinline__ void decode(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t base2, const uint32_t* tab,
                                       uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
  const uint32_t X = ((w0 >> 11) & 0x000F000Fu) | ((w1 >> 7) & 0x00F000F0u) | ((w2 >> 3) & 0x0F000F00u);
  if (AFFINE) {
    a0 = (w0 & 0x87FF87FFu) + base2;
    a1 = (w1 & 0x87FF87FFu) + base2;
    a2 = (w2 & 0x87FF87FFu) + base2;
    a3 = ((X & 0x07FF07FFu) + base2) | ((X << 4) & 0x80008000u);
  } else {
    a0 = general_pair(w0 & 0x87FF87FFu, tab);
    a1 = general_pair(w1 & 0x87FF87FFu, tab);
    a2 = general_pair(w2 & 0x87FF87FFu, tab);
    a3 = general_pair((X & 0x07FF07FFu) | ((X << 4) & 0x80008000u), tab);
  }
}

__device__ __forceinline__ uint32_t comp(const uint4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

template <int NT>
__device__ __forceinline__ void epilogue(const GemmParams& p, int strip, int lane, float (&acc)[NT][4],
                                         float (&bestv)[NT][2], int (&besti)[NT][2]) {
  const int g = lane >> 2, q = lane & 3;
  const int64_t n_lo = (int64_t)strip * 16 + g;
  const int64_t K = p.K;
  // escapes of rows n_lo and n_lo + 8
#pragma unroll
  for (int h = 0; h < 2; h++) {
    const int64_t n = n_lo + 8 * h;
    const uint32_t e0 = p.row_ptr[n], e1 = p.row_ptr[n + 1];
    for (uint32_t e = e0; e < e1; e++) {
      const int64_t k = (int64_t)p.esc_idx[e] - n * K;
      const float w = bf2f(p.esc_val[e]);
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int cc = 0; cc < 2; cc++) {
          const int m = p.m0 + nt * 8 + 2 * q + cc;
          if (m < p.M) {
            const float xv = bf2f(p.x[(int64_t)m * K + k]);
            const float a = fmaf(w, xv, acc[nt][2 * h + cc]);
            acc[nt][2 * h + cc] = fmaf(-p.esc_slot, xv, a);
          }
        }
    }
  }
  const GemmEpilogue& E = p.e;
#pragma unroll
  for (int nt = 0; nt < NT; nt++)
#pragma unroll
    for (int cc = 0; cc < 2; cc++) {
      const int m = p.m0 + nt * 8 + 2 * q + cc;
      if (m >= p.M) continue;
      const float v_lo = acc[nt][cc], v_hi = acc[nt][2 + cc];
      switch (E.epi) {
        case EPI_STORE:
          E.out[(int64_t)m * E.ldo + n_lo] = f2bf(v_lo);
          E.out[(int64_t)m * E.ldo + n_lo + 8] = f2bf(v_hi);
          break;
        case EPI_RESID: {
          const int64_t i0 = (int64_t)m * E.ldo + n_lo, i1 = i0 + 8;
          const float r0 = bf2f(E.resid[i0]), r1 = bf2f(E.resid[i1]);
          E.out[i0] = f2bf(r0 + rbf(v_lo));
          E.out[i1] = f2bf(r1 + rbf(v_hi));
          break;
        }
        case EPI_SILU: {
          const float gt = rbf(v_lo), up = rbf(v_hi);
          const float s = gt / (1.0f + expf(-gt));
          E.out[(int64_t)m * E.ldo + (int64_t)strip * 8 + g] = f2bf(s * up);
          break;
        }
        case EPI_QKV: {
          const int64_t qrows = (int64_t)E.hq * 128, krows = (int64_t)E.hkv * 128;
          const int64_t row0 = (int64_t)strip * 16;
          if (row0 < qrows + krows) {
            const bool is_q = row0 < qrows;
            const int64_t rr = is_q ? row0 : row0 - qrows;
            const int head = (int)(rr / 128);
            const int d = (int)((rr % 128) / 16) * 8 + g;
            const float x1 = rbf(v_lo), x2 = rbf(v_hi);
            const int pos = E.rows.pos[m];
            const float c = E.rope_cos[(int64_t)pos * 64 + d], sn = E.rope_sin[(int64_t)pos * 64 + d];
            const uint16_t o1 = f2bf(x1 * c - x2 * sn), o2 = f2bf(x2 * c + x1 * sn);
            if (is_q) {
              uint16_t* dst = E.q_out + ((int64_t)m * E.hq + head) * 128;
              dst[d] = o1;
              dst[d + 64] = o2;
            } else {
              const int r = E.rows.req[m];
              if (E.rows.req_ok[r]) {
                const int slot = E.rows.slot[m];
                const int page = E.cache.page_table[(int64_t)r * E.cache.max_pages + slot / E.cache.page_size];
                uint16_t* dst = E.cache.k + (((int64_t)page * E.cache.hkv + head) * E.cache.page_size +
                                             slot % E.cache.page_size) * 128;
                dst[d] = o1;
                dst[d + 64] = o2;
              }
            }
          } else {
            const int64_t vr = row0 - qrows - krows;
            const int head = (int)(vr / 128);
            const int d = (int)(vr % 128) + g;
            const int r = E.rows.req[m];
            if (E.rows.req_ok[r]) {
              const int slot = E.rows.slot[m];
              const int page = E.cache.page_table[(int64_t)r * E.cache.max_pages + slot / E.cache.page_size];
              uint16_t* dst = E.cache.v + (((int64_t)page * E.cache.hkv + head) * E.cache.page_size +
                                           slot % E.cache.page_size) * 128;
              dst[d] = f2bf(v_lo);
              dst[d + 8] = f2bf(v_hi);
            }
          }
          break;
        }
        case EPI_LOGITS: {
          if (E.out) {
            E.out[(int64_t)m * E.ldo + n_lo] = f2bf(v_lo);
            E.out[(int64_t)m * E.ldo + n_lo + 8] = f2bf(v_hi);
          }
          if (v_lo > bestv[nt][cc] || (v_lo == bestv[nt][cc] && (int)n_lo < besti[nt][cc])) {
            bestv[nt][cc] = v_lo;
            besti[nt][cc] = (int)n_lo;
          }
          if (v_hi > bestv[nt][cc] || (v_hi == bestv[nt][cc] && (int)n_lo + 8 < besti[nt][cc])) {
            bestv[nt][cc] = v_hi;
            besti[nt][cc] = (int)n_lo + 8;
          }
          break;
        }
      }
    }
}

}  // namespace sdv
