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

// ------------------------------------------------------------- device --
// The same format packed on the GPU: one CTA per packed row chooses its base
// (the exponent histogram of the row in shared memory, then the window scan
// in the host packer's order: the first window of largest cover) and counts
// its escapes; one scan gives the side list's row pointers; the words are
// coded by one thread per (strip, super-tile, lane, sub-tile) as in the
// per-tensor packer; one CTA per row writes the row's escapes in column
// order.

namespace sdv {
namespace {

constexpr int kChThreads = 256;

__global__ void k_c_bases(const uint16_t* __restrict__ w, const int32_t* __restrict__ row_src, int64_t K,
                          uint8_t* __restrict__ base, uint32_t* __restrict__ esc_count) {
  __shared__ uint32_t hist[256];
  const int64_t n = blockIdx.x;
  const int64_t src = row_src ? row_src[n] : n;
  for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const uint16_t* row = w + src * K;
  for (int64_t k = threadIdx.x; k < K; k += blockDim.x) atomicAdd(&hist[(row[k] >> 7) & 0xFF], 1u);
  __syncthreads();
  if (threadIdx.x == 0) {
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
    esc_count[n] = (uint32_t)(K - best);
  }
}

// Single-CTA exclusive scan of counts[0..n) into ptr[0..n], and the largest
// base (for the decodable flag) into aux[0].
__global__ void k_c_scan(const uint32_t* __restrict__ counts, const uint8_t* __restrict__ base, int64_t n,
                         uint32_t* __restrict__ ptr, uint32_t* __restrict__ aux) {
  __shared__ uint32_t part[kChThreads];
  __shared__ uint32_t bmax[kChThreads];
  const int64_t per = (n + blockDim.x - 1) / blockDim.x;
  const int64_t b0 = threadIdx.x * per, b1 = min(n, b0 + per);
  uint32_t s = 0, m = 0;
  for (int64_t i = b0; i < b1; i++) {
    s += counts[i];
    m = max(m, (uint32_t)base[i]);
  }
  part[threadIdx.x] = s;
  bmax[threadIdx.x] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t run = 0, mm = 0;
    for (int i = 0; i < (int)blockDim.x; i++) {
      const uint32_t v = part[i];
      part[i] = run;
      run += v;
      mm = max(mm, bmax[i]);
    }
    ptr[n] = run;
    aux[0] = mm;
  }
  __syncthreads();
  uint32_t run = part[threadIdx.x];
  for (int64_t i = b0; i < b1; i++) {
    ptr[i] = run;
    run += counts[i];
  }
}

__device__ __forceinline__ uint32_t c_field(uint32_t b, uint32_t base) {
  const uint32_t e = (b >> 7) & 0xFFu;
  if (e < base || e > base + 14) return 15u << 7;
  return ((b >> 15) << 11) | ((e - base) << 7) | (b & 0x7Fu);
}

__global__ void k_c_encode(const uint16_t* __restrict__ w, const int32_t* __restrict__ row_src, int64_t N, int64_t K,
                           const uint8_t* __restrict__ base, uint32_t* __restrict__ words) {
  const int64_t KT = K / 64;
  const int64_t total = (N / 16) * KT * 128;
  for (int64_t id = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; id < total; id += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(id & 3);
    const int lane = (int)((id >> 2) & 31);
    const int64_t st = id >> 7;  // strip * KT + super-tile
    const int64_t s = st / KT, t = st % KT;
    const int g = lane >> 2, q = lane & 3;
    const int64_t r_lo = s * 16 + g, r_hi = r_lo + 8;
    const int64_t src_lo = row_src ? row_src[r_lo] : r_lo;
    const int64_t src_hi = row_src ? row_src[r_hi] : r_hi;
    const uint32_t b_lo = base[r_lo], b_hi = base[r_hi];
    const int64_t c0 = t * 64 + j * 16 + 2 * q;
    const int64_t srcs[4] = {src_lo, src_hi, src_lo, src_hi};
    const uint32_t bases[4] = {b_lo, b_hi, b_lo, b_hi};
    const int64_t cols[4] = {c0, c0, c0 + 8, c0 + 8};
    uint32_t f[4][2];
#pragma unroll
    for (int p = 0; p < 4; p++) {
      const uint32_t two = *reinterpret_cast<const uint32_t*>(w + srcs[p] * K + cols[p]);
#pragma unroll
      for (int h = 0; h < 2; h++) f[p][h] = c_field((two >> (16 * h)) & 0xFFFF, bases[p]);
    }
    uint32_t* dst = words + st * 384 + lane * 4 + j;
#pragma unroll
    for (int p = 0; p < 3; p++) {
      uint32_t v = 0;
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const uint32_t half = (f[p][h] & 0x7FF) | ((f[p][h] >> 11) << 15) | (((f[3][h] >> (4 * p)) & 0xF) << 11);
        v |= half << (16 * h);
      }
      dst[128 * p] = v;
    }
  }
}

// One CTA per packed row: its escapes in column order at row_ptr[n].
__global__ void k_c_escapes(const uint16_t* __restrict__ w, const int32_t* __restrict__ row_src, int64_t K,
                            const uint8_t* __restrict__ base, const uint32_t* __restrict__ row_ptr,
                            uint32_t* __restrict__ esc_idx, uint16_t* __restrict__ esc_val) {
  __shared__ uint32_t warp_tot[kChThreads / 32];
  __shared__ uint32_t run_base;
  const int64_t n = blockIdx.x;
  const int64_t src = row_src ? row_src[n] : n;
  const uint32_t b = base[n];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) run_base = row_ptr[n];
  __syncthreads();
  for (int64_t k0 = 0; k0 < K; k0 += blockDim.x) {
    const int64_t k = k0 + threadIdx.x;
    uint16_t v = 0;
    bool e = false;
    if (k < K) {
      v = w[src * K + k];
      const uint32_t ex = (v >> 7) & 0xFF;
      e = ex < b || ex > b + 14;
    }
    const uint32_t m = __ballot_sync(0xffffffffu, e);
    if (lane == 0) warp_tot[warp] = __popc(m);
    __syncthreads();
    uint32_t before = run_base;
    for (int i = 0; i < warp; i++) before += warp_tot[i];
    if (e) {
      const uint32_t pos = before + __popc(m & ((1u << lane) - 1));
      esc_idx[pos] = (uint32_t)(n * K + k);
      esc_val[pos] = v;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t t = 0;
      for (int i = 0; i < kChThreads / 32; i++) t += warp_tot[i];
      run_base += t;
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace sdv

extern "C" int w12c_pack_analyze(const uint16_t* w, const int32_t* row_src, int64_t N, int64_t K, uint8_t* base,
                                 uint32_t* row_ptr, w12_meta* meta, void* stream) {
  if (!w || !base || !row_ptr || !meta) {
    set_error("w12c_pack_analyze: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (!shape_ok(N, K)) {
    set_error("w12c_pack_analyze: N % 16, K % 64 and N*K < 2^32 required");
    return SD_ERR_UNSUPPORTED;
  }
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* scratch = nullptr;  // per-row escape counts, then the largest base
  SD_CK(cudaMallocAsync(reinterpret_cast<void**>(&scratch), (size_t)(N + 1) * sizeof(uint32_t), s));
  k_c_bases<<<(unsigned)N, kChThreads, 0, s>>>(w, row_src, K, base, scratch);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) {
    k_c_scan<<<1, kChThreads, 0, s>>>(scratch, base, N, row_ptr, scratch + N);
    e = cudaGetLastError();
  }
  uint32_t host[2] = {0, 0};
  if (e == cudaSuccess) e = cudaMemcpyAsync(&host[0], row_ptr + N, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&host[1], scratch + N, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  cudaFreeAsync(scratch, s);
  if (e != cudaSuccess) return cuda_fail(e, "w12c_pack_analyze");
  memset(meta, 0, sizeof(*meta));
  meta->N = N;
  meta->K = K;
  meta->n_table = 0;
  meta->affine = host[1] <= 239 ? 1 : 0;
  meta->n_escapes = host[0];
  return SD_OK;
}

extern "C" int w12c_pack_encode(const uint16_t* w, const int32_t* row_src, int64_t N, int64_t K, const uint8_t* base,
                                const uint32_t* row_ptr, uint32_t* words, uint32_t* esc_idx, uint16_t* esc_val,
                                void* stream) {
  if (!w || !base || !row_ptr || !words) {
    set_error("w12c_pack_encode: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (!shape_ok(N, K)) {
    set_error("w12c_pack_encode: N % 16, K % 64 and N*K < 2^32 required");
    return SD_ERR_UNSUPPORTED;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t total = (N / 16) * (K / 64) * 128;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, 65535LL * 32);
  k_c_encode<<<(unsigned)blocks, 256, 0, s>>>(w, row_src, N, K, base, words);
  SD_CK(cudaGetLastError());
  if (esc_idx && esc_val) {
    k_c_escapes<<<(unsigned)N, kChThreads, 0, s>>>(w, row_src, K, base, row_ptr, esc_idx, esc_val);
    SD_CK(cudaGetLastError());
  }
  return SD_OK;
}
