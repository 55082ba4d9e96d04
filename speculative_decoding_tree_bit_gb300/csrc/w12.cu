// W12 lossless 12-bit weight format: packer and unpacker kernels.
//
// "SpecPilot: AI Agent Framework Boosts Speculative Decoding 10.87x for
// Qwen3.8-27B", section "(1) W12: Lossless 12-bit Weight Format": every bf16
// weight keeps sign and 7-bit mantissa; its exponent becomes a 4-bit code
// into a table of the tensor's 15 most frequent exponents; weights whose
// exponent is not in the table are restored exactly from a sparse list.  The
// conversion runs once, ahead of time ("SpecPilot Uses Agentic Discovery
// ...", "Engineering Trade-offs"), so these kernels are offline tools: the
// verify step only ever decodes, inside the GEMM.
//
// Layout: see include/sdv.h (strip-major, fragment-ordered words).
#include <algorithm>
#include <vector>

#include "common.cuh"

namespace sdv {

// ----------------------------------------------------------- histogram --

__global__ void k_exp_histogram(const uint16_t* __restrict__ w, int64_t n, unsigned long long* __restrict__ hist) {
  __shared__ unsigned int h[256];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int64_t n8 = n / 8;
  const uint4* w8 = reinterpret_cast<const uint4*>(w);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = w8[i];
    const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; j++) {
      atomicAdd(&h[(a[j] >> 7) & 0xFF], 1u);
      atomicAdd(&h[(a[j] >> 23) & 0xFF], 1u);
    }
  }
  for (int64_t i = n8 * 8 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    atomicAdd(&h[(w[i] >> 7) & 0xFF], 1u);
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += blockDim.x)
    if (h[i]) atomicAdd(&hist[i], (unsigned long long)h[i]);
}

// Table rule: largest counts first, the smaller exponent first on equal
// counts, only exponents present, at most 15; codes in ascending exponent
// order.
static int choose_table(const unsigned long long* hist, uint8_t* table) {
  std::vector<int> e;
  for (int i = 0; i < 256; i++)
    if (hist[i]) e.push_back(i);
  std::stable_sort(e.begin(), e.end(), [&](int a, int b) { return hist[a] > hist[b]; });
  if (e.size() > 15) e.resize(15);
  std::sort(e.begin(), e.end());
  for (int i = 0; i < 16; i++) table[i] = 0;
  for (size_t i = 0; i < e.size(); i++) table[i] = (uint8_t)e[i];
  return (int)e.size();
}

static int is_affine(const uint8_t* table, int n) {
  if (n == 0) return 1;
  for (int c = 0; c < n; c++)
    if (table[c] != table[0] + c) return 0;
  return table[0] + 15 <= 254 ? 1 : 0;
}

// ---------------------------------------------------------------- encode --

struct CodeLut {
  uint8_t code_of[256];  // exponent -> code (15 = escape)
};

// One thread per (strip, super-tile, lane, sub-tile): gathers the 8 weights
// of that lane's A fragment and writes its three words.
__global__ void k_encode(const uint16_t* __restrict__ w, const int32_t* __restrict__ row_src, int64_t N, int64_t K,
                         CodeLut lut, uint32_t* __restrict__ words) {
  const int64_t KT = K / 64;
  const int64_t total = (N / 16) * KT * 128;
  for (int64_t id = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; id < total; id += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(id & 3);
    const int lane = (int)((id >> 2) & 31);
    const int64_t st = id >> 7;  // strip * KT + t
    const int64_t s = st / KT, t = st % KT;
    const int g = lane >> 2, q = lane & 3;
    const int64_t r_lo = s * 16 + g, r_hi = r_lo + 8;
    const int64_t src_lo = row_src ? row_src[r_lo] : r_lo;
    const int64_t src_hi = row_src ? row_src[r_hi] : r_hi;
    const int64_t c0 = t * 64 + j * 16 + 2 * q;
    uint32_t f[4][2];
    const int64_t rows[4] = {src_lo, src_hi, src_lo, src_hi};
    const int64_t cols[4] = {c0, c0, c0 + 8, c0 + 8};
#pragma unroll
    for (int p = 0; p < 4; p++) {
      const uint32_t two = *reinterpret_cast<const uint32_t*>(w + rows[p] * K + cols[p]);
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const uint32_t b = (two >> (16 * h)) & 0xFFFF;
        const uint32_t code = lut.code_of[(b >> 7) & 0xFF];
        f[p][h] = code == 15 ? (15u << 7) : (((b >> 15) << 11) | (code << 7) | (b & 0x7F));
      }
    }
    uint32_t out[3];
#pragma unroll
    for (int p = 0; p < 3; p++) {
      uint32_t v = 0;
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const uint32_t half = (f[p][h] & 0x7FF) | ((f[p][h] >> 11) << 15) | (((f[3][h] >> (4 * p)) & 0xF) << 11);
        v |= half << (16 * h);
      }
      out[p] = v;
    }
    uint32_t* base = words + st * 384 + lane * 4 + j;
    base[0] = out[0];
    base[128] = out[1];
    base[256] = out[2];
  }
}

// --------------------------------------------------------------- escapes --
// Escapes in packed-row flat order, order-preserving compaction in three
// passes: count per block, exclusive scan of the counts, write.

constexpr int kEscBlock = 256;
constexpr int kEscPerThread = 16;
constexpr int64_t kEscTile = (int64_t)kEscBlock * kEscPerThread;

__device__ __forceinline__ bool is_escape(const uint16_t* w, const int32_t* row_src, int64_t K, const CodeLut& lut,
                                          int64_t idx, uint16_t* val) {
  const int64_t n = idx / K, k = idx - n * K;
  const int64_t src = row_src ? row_src[n] : n;
  const uint16_t b = w[src * K + k];
  *val = b;
  return lut.code_of[(b >> 7) & 0xFF] == 15;
}

__global__ void k_esc_count(const uint16_t* __restrict__ w, const int32_t* __restrict__ row_src, int64_t N, int64_t K,
                            CodeLut lut, uint32_t* __restrict__ counts) {
  const int64_t n = N * K;
  const int64_t base = blockIdx.x * kEscTile;
  uint32_t c = 0;
  for (int i = 0; i < kEscPerThread; i++) {
    const int64_t idx = base + (int64_t)i * kEscBlock + threadIdx.x;
    uint16_t v;
    if (idx < n && is_escape(w, row_src, K, lut, idx, &v)) c++;
  }
  __shared__ uint32_t red[kEscBlock / 32];
  for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
    for (int i = 0; i < kEscBlock / 32; i++) t += red[i];
    counts[blockIdx.x] = t;
  }
}

// Single-block exclusive scan of counts[0..nb) -> offsets, total at offsets[nb].
__global__ void k_scan(const uint32_t* __restrict__ counts, int64_t nb, uint32_t* __restrict__ offsets) {
  __shared__ uint32_t part[1024];
  const int64_t per = (nb + blockDim.x - 1) / blockDim.x;
  const int64_t b0 = threadIdx.x * per, b1 = min(nb, b0 + per);
  uint32_t s = 0;
  for (int64_t i = b0; i < b1; i++) s += counts[i];
  part[threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t run = 0;
    for (int i = 0; i < (int)blockDim.x; i++) {
      const uint32_t v = part[i];
      part[i] = run;
      run += v;
    }
    offsets[nb] = run;
  }
  __syncthreads();
  uint32_t run = part[threadIdx.x];
  for (int64_t i = b0; i < b1; i++) {
    offsets[i] = run;
    run += counts[i];
  }
}

__global__ void k_esc_write(const uint16_t* __restrict__ w, const int32_t* __restrict__ row_src, int64_t N, int64_t K,
                            CodeLut lut, const uint32_t* __restrict__ offsets, uint32_t* __restrict__ esc_idx,
                            uint16_t* __restrict__ esc_val) {
  __shared__ uint32_t warp_tot[kEscBlock / 32];
  __shared__ uint32_t run_base;
  const int64_t n = N * K;
  const int64_t base = blockIdx.x * kEscTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) run_base = offsets[blockIdx.x];
  __syncthreads();
  for (int i = 0; i < kEscPerThread; i++) {
    const int64_t idx = base + (int64_t)i * kEscBlock + threadIdx.x;
    uint16_t v = 0;
    const bool e = idx < n && is_escape(w, row_src, K, lut, idx, &v);
    const uint32_t m = __ballot_sync(0xffffffffu, e);
    if (lane == 0) warp_tot[warp] = __popc(m);
    __syncthreads();
    uint32_t before = run_base;
    for (int k = 0; k < warp; k++) before += warp_tot[k];
    if (e) {
      const uint32_t pos = before + __popc(m & ((1u << lane) - 1));
      esc_idx[pos] = (uint32_t)idx;
      esc_val[pos] = v;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t t = 0;
      for (int k = 0; k < kEscBlock / 32; k++) t += warp_tot[k];
      run_base += t;
    }
    __syncthreads();
  }
}

// row_ptr[n] = number of escapes with flat index < n*K (binary search).
__global__ void k_row_ptr(const uint32_t* __restrict__ esc_idx, int64_t n_esc, int64_t N, int64_t K,
                          uint32_t* __restrict__ row_ptr) {
  for (int64_t n = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; n <= N; n += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t key = (uint64_t)n * (uint64_t)K;
    int64_t lo = 0, hi = n_esc;
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if ((uint64_t)esc_idx[mid] < key) lo = mid + 1;
      else hi = mid;
    }
    row_ptr[n] = (uint32_t)lo;
  }
}

// Escape tile index of one 128-row block (one CTA): count the block's
// escapes per 64-column tile, prefix-sum from the block's first side-list
// index, then place them tile by tile keeping the side list's (row-major)
// order within each tile.
__global__ void k_tile_index(const uint32_t* __restrict__ esc_idx, const uint16_t* __restrict__ esc_val,
                             const uint32_t* __restrict__ row_ptr, int64_t N, int64_t K,
                             uint32_t* __restrict__ tile_ptr, uint32_t* __restrict__ tile_esc) {
  extern __shared__ uint32_t cursor[];  // [KT]
  const int KT = (int)(K / 64);
  const int64_t b = blockIdx.x;
  const int64_t n0 = b * 128, n1 = n0 + 128 < N ? n0 + 128 : N;
  const uint32_t e0 = row_ptr[n0], e1 = row_ptr[n1];
  for (int t = threadIdx.x; t < KT; t += blockDim.x) cursor[t] = 0;
  __syncthreads();
  for (uint32_t e = e0 + threadIdx.x; e < e1; e += blockDim.x)
    atomicAdd(&cursor[(int)((esc_idx[e] % (uint64_t)K) / 64)], 1u);
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t run = e0;
    for (int t = 0; t < KT; t++) {
      const uint32_t c = cursor[t];
      tile_ptr[b * KT + t] = run;
      cursor[t] = run;
      run += c;
    }
    if (b == gridDim.x - 1) tile_ptr[(b + 1) * KT] = e1;
    for (uint32_t e = e0; e < e1; e++) {
      const uint64_t idx = esc_idx[e];
      const uint32_t n = (uint32_t)(idx / (uint64_t)K), k = (uint32_t)(idx % (uint64_t)K);
      tile_esc[cursor[k / 64]++] = ((uint32_t)esc_val[e] << 16) | ((n - (uint32_t)n0) << 6) | (k & 63u);
    }
  }
}

// ---------------------------------------------------------------- unpack --

struct TableArg {
  uint8_t t[16];
};

__global__ void k_unpack(const uint32_t* __restrict__ words, int64_t N, int64_t K, TableArg tab,
                         const uint8_t* __restrict__ row_base, uint16_t* __restrict__ out) {
  const int64_t KT = K / 64;
  const int64_t total = (N / 16) * KT * 128;
  for (int64_t id = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; id < total; id += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(id & 3);
    const int lane = (int)((id >> 2) & 31);
    const int64_t st = id >> 7;
    const int64_t s = st / KT, t = st % KT;
    const uint32_t* base = words + st * 384 + lane * 4 + j;
    const uint32_t W[3] = {base[0], base[128], base[256]};
    const int g = lane >> 2, q = lane & 3;
    const int64_t r_lo = s * 16 + g, c0 = t * 64 + j * 16 + 2 * q;
    const int64_t rows[4] = {r_lo, r_lo + 8, r_lo, r_lo + 8};
    const int64_t cols[4] = {c0, c0, c0 + 8, c0 + 8};
#pragma unroll
    for (int p = 0; p < 4; p++) {
      uint32_t pairbits = 0;
#pragma unroll
      for (int h = 0; h < 2; h++) {
        uint32_t f;
        if (p < 3) {
          const uint32_t v = (W[p] >> (16 * h)) & 0xFFFF;
          f = (v & 0x7FF) | (((v >> 15) & 1) << 11);
        } else {
          f = ((W[0] >> (11 + 16 * h)) & 0xF) | (((W[1] >> (11 + 16 * h)) & 0xF) << 4) |
              (((W[2] >> (11 + 16 * h)) & 0xF) << 8);
        }
        const uint32_t code = (f >> 7) & 15;
        const uint32_t e = code == 15 ? 0u : row_base ? (row_base[rows[p]] + code) & 0xFF : tab.t[code];
        const uint32_t b = ((f >> 11) << 15) | (e << 7) | (f & 0x7F);
        pairbits |= b << (16 * h);
      }
      *reinterpret_cast<uint32_t*>(out + rows[p] * K + cols[p]) = pairbits;
    }
  }
}

__global__ void k_scatter_escapes(const uint32_t* __restrict__ esc_idx, const uint16_t* __restrict__ esc_val,
                                  int64_t n_esc, uint16_t* __restrict__ out) {
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n_esc; e += (int64_t)gridDim.x * blockDim.x)
    out[esc_idx[e]] = esc_val[e];
}

static int grid_for(int64_t work, int block) {
  const int64_t g = (work + block - 1) / block;
  const int64_t cap = (int64_t)num_sms() * 16;
  return (int)std::max<int64_t>(1, std::min<int64_t>(g, cap));
}

static CodeLut make_lut(const w12_meta* meta) {
  CodeLut lut;
  for (int e = 0; e < 256; e++) lut.code_of[e] = 15;
  for (int c = 0; c < meta->n_table; c++) lut.code_of[meta->table[c]] = (uint8_t)c;
  return lut;
}

}  // namespace sdv

using namespace sdv;

extern "C" int64_t w12_words_count(int64_t N, int64_t K) { return N * K / 8 * 3; }

extern "C" int w12_pack_analyze(const uint16_t* w, int64_t N, int64_t K, w12_meta* meta, void* stream) {
  if (!w || !meta || N <= 0 || K <= 0) {
    set_error("w12_pack_analyze: null pointer or empty shape");
    return SD_ERR_INVALID_ARG;
  }
  if (N % 16 || K % 64 || N * K >= (int64_t)1 << 32) {
    set_error("w12_pack_analyze: need N % 16 == 0, K % 64 == 0, N*K < 2^32");
    return SD_ERR_UNSUPPORTED;
  }
  cudaStream_t s = (cudaStream_t)stream;
  unsigned long long* d_hist = nullptr;
  SD_CK(cudaMallocAsync(&d_hist, 256 * sizeof(unsigned long long), s));
  SD_CK(cudaMemsetAsync(d_hist, 0, 256 * sizeof(unsigned long long), s));
  k_exp_histogram<<<grid_for(N * K / 8, 256), 256, 0, s>>>(w, N * K, d_hist);
  SD_CK(cudaGetLastError());
  unsigned long long hist[256];
  SD_CK(cudaMemcpyAsync(hist, d_hist, sizeof(hist), cudaMemcpyDeviceToHost, s));
  SD_CK(cudaFreeAsync(d_hist, s));
  SD_CK(cudaStreamSynchronize(s));
  meta->N = N;
  meta->K = K;
  meta->n_table = choose_table(hist, meta->table);
  meta->affine = is_affine(meta->table, meta->n_table);
  unsigned long long in_tab = 0, tot = 0;
  for (int e = 0; e < 256; e++) tot += hist[e];
  for (int c = 0; c < meta->n_table; c++) in_tab += hist[meta->table[c]];
  meta->n_escapes = (int64_t)(tot - in_tab);
  return SD_OK;
}

extern "C" int w12_pack_encode(const uint16_t* w, const int32_t* row_src, const w12_meta* meta, uint32_t* words,
                               uint32_t* esc_idx, uint16_t* esc_val, uint32_t* row_ptr, void* stream) {
  if (!w || !meta || !words || !row_ptr || (meta->n_escapes > 0 && (!esc_idx || !esc_val))) {
    set_error("w12_pack_encode: null pointer");
    return SD_ERR_INVALID_ARG;
  }
  const int64_t N = meta->N, K = meta->K;
  if (N <= 0 || K <= 0 || N % 16 || K % 64 || N * K >= (int64_t)1 << 32 || meta->n_table > 15) {
    set_error("w12_pack_encode: bad meta");
    return SD_ERR_UNSUPPORTED;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const CodeLut lut = make_lut(meta);
  k_encode<<<grid_for((N / 16) * (K / 64) * 128, 256), 256, 0, s>>>(w, row_src, N, K, lut, words);
  SD_CK(cudaGetLastError());
  const int64_t nb = (N * K + kEscTile - 1) / kEscTile;
  uint32_t* scratch = nullptr;
  SD_CK(cudaMallocAsync(&scratch, (2 * nb + 1) * sizeof(uint32_t), s));
  k_esc_count<<<(unsigned)nb, kEscBlock, 0, s>>>(w, row_src, N, K, lut, scratch);
  SD_CK(cudaGetLastError());
  k_scan<<<1, 1024, 0, s>>>(scratch, nb, scratch + nb);
  SD_CK(cudaGetLastError());
  if (meta->n_escapes > 0) {
    k_esc_write<<<(unsigned)nb, kEscBlock, 0, s>>>(w, row_src, N, K, lut, scratch + nb, esc_idx, esc_val);
    SD_CK(cudaGetLastError());
  }
  k_row_ptr<<<grid_for(N + 1, 256), 256, 0, s>>>(esc_idx, meta->n_escapes, N, K, row_ptr);
  SD_CK(cudaGetLastError());
  SD_CK(cudaFreeAsync(scratch, s));
  return SD_OK;
}

extern "C" int64_t w12_tile_ptr_count(int64_t N, int64_t K) { return ((N + 127) / 128) * (K / 64) + 1; }

extern "C" int w12_pack_tile_index(const w12_tensor* t, uint32_t* tile_ptr, uint32_t* tile_esc, void* stream) {
  if (!t || !tile_ptr || !t->row_ptr || (t->n_escapes > 0 && (!t->esc_idx || !t->esc_val || !tile_esc))) {
    set_error("w12_pack_tile_index: null pointer");
    return SD_ERR_INVALID_ARG;
  }
  if (t->N <= 0 || t->K <= 0 || t->N % 16 || t->K % 64 || t->N * t->K >= (int64_t)1 << 32) {
    set_error("w12_pack_tile_index: bad shape");
    return SD_ERR_UNSUPPORTED;
  }
  const int64_t NB = (t->N + 127) / 128, KT = t->K / 64;
  const size_t smem = (size_t)KT * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    set_error("w12_pack_tile_index: K too large (K/64 tiles must fit 48 KB of shared memory)");
    return SD_ERR_UNSUPPORTED;
  }
  k_tile_index<<<(unsigned)NB, 256, smem, (cudaStream_t)stream>>>(t->esc_idx, t->esc_val, t->row_ptr, t->N, t->K,
                                                                  tile_ptr, tile_esc);
  SD_CK(cudaGetLastError());
  return SD_OK;
}

extern "C" int w12_unpack(const w12_tensor* t, uint16_t* w_out, void* stream) {
  if (!t || !w_out || !t->words || (t->n_escapes > 0 && (!t->esc_idx || !t->esc_val))) {
    set_error("w12_unpack: null pointer");
    return SD_ERR_INVALID_ARG;
  }
  if (t->N <= 0 || t->K <= 0 || t->N % 16 || t->K % 64 || t->n_table > 15) {
    set_error("w12_unpack: bad shape");
    return SD_ERR_UNSUPPORTED;
  }
  cudaStream_t s = (cudaStream_t)stream;
  TableArg tab;
  for (int i = 0; i < 16; i++) tab.t[i] = i < t->n_table ? t->table[i] : 0;
  k_unpack<<<grid_for((t->N / 16) * (t->K / 64) * 128, 256), 256, 0, s>>>(t->words, t->N, t->K, tab, t->row_base,
                                                                           w_out);
  SD_CK(cudaGetLastError());
  if (t->n_escapes > 0) {
    k_scatter_escapes<<<grid_for(t->n_escapes, 256), 256, 0, s>>>(t->esc_idx, t->esc_val, t->n_escapes, w_out);
    SD_CK(cudaGetLastError());
  }
  return SD_OK;
}
