// Fused W12-decode skinny GEMM for sm_103a.
//
// "SpecPilot: AI Agent Framework Boosts Speculative Decoding 10.87x for
// Qwen3.8-27B", "(1) W12": a dedicated GEMM decodes the 12-bit weights
// directly in registers, so the weights cross HBM once at 1.5 bytes each and
// no bf16 copy is ever materialised.  "SpecPilot Uses Agentic Discovery ...",
// "Technical Mechanisms": decode-time verification is bound by the bytes of
// the target weights, so this kernel is built as a weight streamer:
//
//  * y[m][n] = sum_k x[m][k] W[n][k] with weights as the 16-row A operand of
//    mma.m16n8k16 (tokens are the 8-wide N side, "swap-AB"): up to 128 tree
//    rows per launch ride along while the step is bandwidth-bound.
//  * One persistent CTA per SM: warp 8 is a producer that streams the packed
//    words with cp.async.bulk and the activation slice with a 2-D TMA box
//    (128-byte swizzle) into a multi-stage mbarrier ring; warps 0..7 each own
//    one 16-row strip of the current 128-row block, decode their words
//    (3 words -> 4 bf16x2 fragment registers, about two integer operations
//    per weight when the exponent table is contiguous) and issue the MMAs.
//  * Work = (row block, 64-column super-tile) units, split evenly over the
//    CTAs in row-block-major order (stream-K), so every SM streams the same
//    number of bytes.  A row block split between CTAs is finished by the last
//    contributor (atomic ticket, no spinning), which sums the partials in CTA
//    order (deterministic) and runs the epilogue.
//  * Escaped weights decode to a fixed slot value; the epilogue adds
//    (w - slot) * x for the few escapes of its rows from the CSR side list.
//  * Fused epilogues: store, residual add, SiLU(gate)*up, RoPE + KV-cache
//    write for q/k/v, bf16 logits + running argmax.
//  * Programmatic dependent launch: the producer streams weights into the
//    ring before waiting for the previous kernel's activations.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "gemm_impl.cuh"
#include "stream.cuh"

namespace sdv {

// Two CTAs per SM for small tiles (more warps to hide decode and MMA latency).
template <int NT>
constexpr int ctas_per_sm() { return NT <= 4 ? 2 : 1; }

template <int NT, bool AFFINE, bool V8 = false, bool CH = false>
__global__ void __launch_bounds__(kThreads, ctas_per_sm<NT>())
    k_w12_gemm(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap xmap,
               const __grid_constant__ CUtensorMap wmap) {
  using C = Cfg<NT, V8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sx = smem;
  uint8_t* sw = smem + C::OFF_W;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_FULL);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + C::OFF_EMPTY);
  float* red_v = reinterpret_cast<float*>(smem + C::OFF_RED_V);
  int* red_i = reinterpret_cast<int*>(smem + C::OFF_RED_I);
  int* flag = reinterpret_cast<int*>(smem + C::OFF_FLAG);
  volatile int* abort = flag + 1;
  uint64_t* corr_full = reinterpret_cast<uint64_t*>(smem + C::OFF_CBAR);
  uint64_t* corr_empty = corr_full + 1;
  float* corr = reinterpret_cast<float*>(smem + C::OFF_CORR);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;  // trace layout [4][grid]
  int64_t u0, u1;
  unit_range(p, u0, u1);
  const int KT = p.KT;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::S; i++) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kNCW + 1);  // consumer warps + escape warp
    }
    mbar_init(corr_full, 1);
    mbar_init(corr_empty, kNCW);
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------- producer --
    if (lane == 0) {
      const int64_t n = u1 - u0;
      int64_t issued = 0;
      if (n > 0) {
        const int pre = (int)(n < C::S ? n : C::S);
        int b = (int)udiv(u0, KT), t = (int)(u0 - (int64_t)b * KT);
        const int t_first = t;
        // one 2-D box per stage: 8 strips x 1536 bytes (ragged row blocks are
        // zero-filled by the copy engine and never read)
        auto issue_weights = [&](int slot, int bb, int tt) {
          // 8 strips x 1536 bytes, or 8 strips x 1024 bytes of the 8-bit plane
          mbar_arrive_expect_tx(&full[slot], C::WB + C::XB);
          tma2d_g2s(sw + slot * C::WB, &wmap, tt * (V8 ? 128 : 192), bb * kRB, &full[slot]);
        };
        for (int i = 0; i < pre; i++) {
          issue_weights(i, b, t);
          if (++t == KT) {
            t = 0;
            b++;
          }
        }
        pdl_wait();  // activations come from the previous kernel
        {
          int tt = t_first;
          for (int i = 0; i < pre; i++) {
            tma2d_g2s(sx + i * C::XB, &xmap, tt * 64, p.m0, &full[i]);
            if (++tt == KT) tt = 0;
          }
        }
        issued = pre;
        // the loop below runs only when pre == S: stage S reuses slot 0,
        // whose first use completed phase 0 of its empty barrier
        int slot = 0;
        uint32_t par = 0;
        for (int64_t i = pre; i < n; i++) {
          if (!mbar_wait_or_abort(&empty[slot], par, abort)) {
            set_status(p.status, SD_TIMEOUT_AT(1));
            break;
          }
          issue_weights(slot, b, t);
          tma2d_g2s(sx + slot * C::XB, &xmap, t * 64, p.m0, &full[slot]);
          issued++;
          if (++t == KT) {
            t = 0;
            b++;
          }
          if (++slot == C::S) {
            slot = 0;
            par ^= 1u;
          }
        }
      } else {
        pdl_wait();
      }
      // every copy this CTA started has landed before it exits
      for (int s = 0; s < C::S && s < issued; s++) {
        const int64_t n_s = issued / C::S + (s < issued % C::S ? 1 : 0);
        if (!mbar_wait(&full[s], (uint32_t)((n_s - 1) & 1))) set_status(p.status, SD_TIMEOUT_AT(2));
      }
    }
    if (p.cluster_k > 1) {
      // the consumers' two cluster barriers (partials staged, partials read)
      __syncwarp();
      cluster_sync_all();
      cluster_sync_all();
    }
    return;
  }

  if (warp == kEscapeWarp) {
    // -------------------------------------------------- escape warp --
    int eseg = 0, eslot = 0;
    uint32_t ephase = 0;
    escape_segments<NT, V8>(p, sx, full, empty, eslot, ephase, corr, corr_full, corr_empty, eseg, abort);
    if (p.cluster_k > 1) {
      __syncwarp();
      cluster_sync_all();
      cluster_sync_all();
    }
    return;
  }

  // --------------------------------------------------------- consumers --
  pdl_wait();
  if (p.trace && threadIdx.x == 0) p.trace[blockIdx.x] = globaltimer();
  int slot = 0, cseg = 0;
  uint32_t phase = 0;
  consume_gemm<NT, AFFINE, V8, CH>(p, sx, sw, full, empty, red_v, red_i, flag, slot, phase, corr, corr_full, corr_empty,
                           cseg, abort, p.trace ? p.trace + G + blockIdx.x : nullptr, G);
  if (p.trace) {
    bar_sync(1, kNCW * 32);
    if (threadIdx.x == 0) p.trace[3 * G + blockIdx.x] = globaltimer();
  }
}

// ------------------------------------------------------------------ host --

int pad_rows(int M) { return M <= 8 ? 8 : M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

static int nt_of(int M) { return M > 128 ? 16 : pad_rows(M) / 8; }

// Default crossover of the two kernels (rows per launch), measured on whole
// verify steps on GB300 (graph replay, programmatic dependent launch): at
// 64 rows the warp-level kernel takes the 27B-class step in 23.7 ms
// (tcgen05: 26.8) and the 8B-class batched step of 8 requests in 8.2 ms
// (tcgen05: 9.2); at 128 rows the tcgen05 kernel wins (12.5 vs 16.0 ms).
// A lone gate/up launch (no neighbours to overlap) favours tcgen05 from 48
// rows, by 2-6%.
constexpr int kTcMinRowsDefault = 65;
static int g_tc_min_rows = kTcMinRowsDefault;

int gemm_tc_min_rows() { return g_tc_min_rows; }
void gemm_set_tc_min_rows(int rows) { g_tc_min_rows = rows > 0 ? rows : kTcMinRowsDefault; }

static int warp_grid(int M) { return (nt_of(M) <= 4 ? 2 : 1) * num_sms(); }

// Row blocks split over a whole number of CTAs may finish in a separate
// kernel (sd_gemm_set_deferred_finish); off by default: the extra kernel
// boundary measured slower than the in-kernel finisher (8B-class step 4.75
// vs 4.29 ms at 16 rows).
static bool g_defer_finish = false;

// Row blocks split over a whole number of CTAs may finish through a
// thread-block cluster (sd_gemm_set_cluster_finish); off by default: the
// cluster launch measured slower than the workspace ticket at every shape
// (O 24.0 vs 20.7 us, down 41.9 vs 32.8 us at 16 rows).
static bool g_cluster_finish = false;
int gemm_warp_grid(int M) { return warp_grid(M); }
int gemm_finish_mode() {
  return (g_cluster_finish ? 2 : 0) | (g_defer_finish ? 1 : 0) | (gemm_strip_eligible_setting() ? 4 : 0);
}

int gemm_grid(int M) { return gemm_use_tc(M) ? num_sms() : warp_grid(M); }

int gemm_warp_launch_grid(const w12_tensor& W, int M, int epi) {
  int grid = warp_grid(M);
  // few row blocks (q/k/v, O, down): a whole number of CTAs per row block,
  // so that no CTA's range straddles two row blocks (a straddling CTA
  // finishes two segments and trails the others); the argmax partials of
  // the logits GEMM keep one slot per CTA of gemm_grid
  const int nb = gemm_counters(W.N);
  if (epi != EPI_LOGITS && nb * 4 <= grid) grid = nb * (grid / nb);
  return grid;
}

int gemm_launch_grid(const w12_tensor& W, int M, int epi) {
  if (gemm_use_tc(M)) {
    // few row blocks: a whole number of CTAs per block (no CTA's range
    // straddles two blocks, every block has the same contributors)
    const int nb = gemm_counters(W.N), sms = num_sms();
    return (epi != EPI_LOGITS && nb * 2 <= sms) ? nb * (sms / nb) : sms;
  }
  return gemm_warp_launch_grid(W, M, epi);
}

size_t gemm_partial_floats(int M) {
  const size_t mma = (size_t)(nt_of(M) <= 4 ? 2 : 1) * num_sms() * 2 * kRB * nt_of(M) * 128;
  return std::max(mma, gemm_tc_partial_floats(M));
}

int gemm_counters(int64_t N) { return (int)((N / 16 + kRB - 1) / kRB); }

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

int make_x_map(XMap* xm, const uint16_t* x, int rows_total, int64_t K, int box_rows) {
  auto fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled unavailable");
    return SD_ERR_CUDA;
  }
  if ((reinterpret_cast<uintptr_t>(x) & 15) || K % 64 || box_rows < 8 || box_rows > 256 || rows_total < 1) {
    set_error("make_x_map: x must be 16-byte aligned, K % 64 == 0");
    return SD_ERR_INVALID_ARG;
  }
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows_total};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(&xm->map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed: " + std::to_string((int)r));
    return SD_ERR_CUDA;
  }
  xm->rows_total = rows_total;
  xm->box_rows = box_rows;
  return SD_OK;
}

// The packed words as a 2-D tensor of u64: [strips][K/64 * 192]; one box is
// 192 u64 (one strip's 1536-byte super-tile) x 8 strips.
int make_w_map(CUtensorMap* map, const w12_tensor& W) {
  auto fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled unavailable");
    return SD_ERR_CUDA;
  }
  if (reinterpret_cast<uintptr_t>(W.words) & 15) {
    set_error("gemm: packed words must be 16-byte aligned");
    return SD_ERR_INVALID_ARG;
  }
  const int64_t KT = W.K / 64;
  cuuint64_t dims[2] = {(cuuint64_t)KT * 192, (cuuint64_t)(W.N / 16)};
  cuuint64_t strides[1] = {(cuuint64_t)KT * kStripBytes};
  cuuint32_t box[2] = {192, (cuuint32_t)kRB};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint32_t*>(W.words), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (weights) failed: " + std::to_string((int)r));
    return SD_ERR_CUDA;
  }
  return SD_OK;
}

// The 8-bit plane as a 2-D tensor of u64: [strips][K/64 * 128]; one box is
// 128 u64 (one strip's 1024-byte super-tile) x 8 strips.
int make_w8_map(CUtensorMap* map, const uint32_t* plane, int64_t N, int64_t K) {
  auto fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled unavailable");
    return SD_ERR_CUDA;
  }
  if (reinterpret_cast<uintptr_t>(plane) & 15) {
    set_error("gemm: the 8-bit plane must be 16-byte aligned");
    return SD_ERR_INVALID_ARG;
  }
  const int64_t KT = K / 64;
  cuuint64_t dims[2] = {(cuuint64_t)KT * 128, (cuuint64_t)(N / 16)};
  cuuint64_t strides[1] = {(cuuint64_t)KT * 1024};
  cuuint32_t box[2] = {128, (cuuint32_t)kRB};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint32_t*>(plane), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (8-bit plane) failed: " + std::to_string((int)r));
    return SD_ERR_CUDA;
  }
  return SD_OK;
}

// Whether clusters of k CTAs of this kernel can be scheduled (checked once
// per kernel instance and k, with `known` the instance's own cache; sizes
// above 8 are allowed on the kernel first; a cluster that cannot be
// co-scheduled falls back to the global finish).
template <typename K>
static bool cluster_ok(K kern, int k, int smem, int* known) {
  if (k < 2 || k > 16) return false;
  if (known[k]) return known[k] == 1;
  bool ok = true;
  if (k > 8) ok = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  if (ok) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(k * 16);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)k;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    ok = cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0;
  }
  cudaGetLastError();  // a refused query leaves no error behind
  known[k] = ok ? 1 : 2;
  return ok;
}

// The cluster finish for this launch: k CTAs per row block, every CTA one
// non-empty k-range of exactly one block, and clusters of k schedulable.
template <int NT, bool AFF, bool V8, bool CH>
static int cluster_for(const GemmParams& p, int grid) {
  if (!g_cluster_finish || p.e.epi == EPI_LOGITS || p.M > 128 || grid % p.NB) return 0;
  const int k = grid / p.NB;
  if (k < 2 || k > 16 || p.KT < k) return 0;
  // the staged partial lives in the weight ring
  if ((size_t)Cfg<NT, V8>::S * Cfg<NT, V8>::WB < (size_t)128 * Cfg<NT, V8>::MP * 4) return 0;
  static int known[17] = {0};  // per kernel instance and k: 0 unknown, 1 schedulable, 2 not
  if (!cluster_ok(k_w12_gemm<NT, AFF, V8, CH>, k, Cfg<NT, V8>::SMEM, known)) return 0;
  return k;
}

// Split-K finish of a deferred launch (GemmParams::defer): one warp per
// 16-row strip sums the fragments the row block's contributors left in their
// partial slots, in CTA order and in the in-kernel finisher's grouping (the
// same sums, up to nothing), and runs the epilogue.  Every contributor's
// loads are in flight at once (one round trip where the in-kernel finisher
// takes one per batch, after its release / acquire ticket).  It follows the
// GEMM on the stream; under programmatic dependent launch it starts early
// and waits for the GEMM's completion.
template <int NT>
__global__ void __launch_bounds__(128) k_gemm_finish(const __grid_constant__ GemmParams p) {
  pdl_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x >> 1;
  const int w = (blockIdx.x & 1) * 4 + warp;  // strip within the block
  const int strip = b * kRB + w;
  pdl_wait();
  if (strip >= p.NS) return;
  const int64_t G = unit_ctas(p);
  const int KT = p.KT;
  const int64_t c_first = udiv(((int64_t)b * KT + 1) * G - 1, p.U);
  const int64_t c_last = udiv(((int64_t)(b + 1) * KT) * G - 1, p.U);
  constexpr int kLoad = NT <= 2 ? 16 : NT <= 4 ? 8 : 4;  // contributors in flight (a launch has at most 16)
  constexpr int kB = finish_batch(NT);
  static_assert(kLoad % kB == 0, "loads cover whole batches");
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; nt++)
#pragma unroll
    for (int c = 0; c < 4; c++) acc[nt][c] = 0.f;
  for (int64_t c0 = c_first; c0 <= c_last; c0 += kLoad) {
    float4 v[kLoad][NT];
#pragma unroll
    for (int u = 0; u < kLoad; u++) {
      const int64_t c = c0 + u;
      const int64_t cs = udiv(c * p.U, G), ce = udiv((c + 1) * p.U, G);
      const bool use = c <= c_last && cs != ce;
      const int64_t sid = use && cs < (int64_t)b * KT ? 1 : 0;  // the range began in an earlier block
      const float* src = p.partial + (((use ? c : 0) * 2 + sid) * kRB + w) * NT * 128 + lane * 4;
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
        v[u][nt] = use ? __ldcg(reinterpret_cast<const float4*>(src + nt * 128)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // the in-kernel finisher's batches start at c_first in steps of kB and
    // add every slot of a batch (+0 past the last contributor)
#pragma unroll
    for (int u = 0; u < kLoad; u++) {
      if (c0 + (u / kB) * kB > c_last) break;  // a batch the finisher never starts
#pragma unroll
      for (int nt = 0; nt < NT; nt++) {
        acc[nt][0] += v[u][nt].x;
        acc[nt][1] += v[u][nt].y;
        acc[nt][2] += v[u][nt].z;
        acc[nt][3] += v[u][nt].w;
      }
    }
  }
  float bestv[NT][2];
  int besti[NT][2];
  epilogue<NT>(p, strip, lane, acc, bestv, besti);
}

// A deferred finish for this launch: split row blocks with a whole number
// (2..16) of CTAs each (no CTA's range meets two blocks), the argmax
// epilogue excepted (its partials are per CTA), one row tile.
static bool defer_for(int NB, int M, int epi, int grid) {
  if (!g_defer_finish || g_cluster_finish || epi == EPI_LOGITS || M > 128 || grid % NB) return false;
  const int k = grid / NB;
  return k >= 2 && k <= 16;
}

template <int NT, bool AFF, bool V8 = false, bool CH = false>
static cudaError_t launch_nt(const GemmParams& p, const CUtensorMap& map, const CUtensorMap& wmap, cudaStream_t s,
                             bool pdl, int grid) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(k_w12_gemm<NT, AFF, V8, CH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               Cfg<NT, V8>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  GemmParams q = p;
  q.cluster_k = cluster_for<NT, AFF, V8, CH>(q, grid);
  if (q.cluster_k > 1)
    return launch_cluster(k_w12_gemm<NT, AFF, V8, CH>, dim3(grid), dim3(kThreads), Cfg<NT, V8>::SMEM, s, pdl,
                          q.cluster_k, q, map, wmap);
  q.defer = defer_for(q.NB, q.M, q.e.epi, grid) ? 1 : 0;
  const cudaError_t e =
      launch(k_w12_gemm<NT, AFF, V8, CH>, dim3(grid), dim3(kThreads), Cfg<NT, V8>::SMEM, s, pdl, q, map, wmap);
  if (e != cudaSuccess || !q.defer) return e;
  return launch(k_gemm_finish<NT>, dim3(2 * q.NB), dim3(128), 0, s, pdl, q);
}

int gemm_kernel_count(const w12_tensor& W, int M, int epi, int grid) {
  if (gemm_use_tc(M) && !W.row_base) return 1;
  if (grid <= 0 && gemm_strip_eligible(W, M, epi)) return 1;
  if (grid <= 0) grid = gemm_warp_launch_grid(W, M, epi);
  return (M + 127) / 128 + (defer_for(gemm_counters(W.N), M, epi, grid) ? 1 : 0);
}



int make_gemm_params(GemmParams* out, const w12_tensor& W, const uint16_t* x, int M, const GemmEpilogue& epi,
                     const GemmWorkspace& ws, int32_t* status) {
  if (W.N % 16 || W.K % 64 || M < 1 || M > 256) {
    set_error("gemm: unsupported shape");
    return SD_ERR_UNSUPPORTED;
  }
  GemmParams& p = *out;
  p = GemmParams{};
  p.words = W.words;
  p.N = W.N;
  p.K = W.K;
  p.KT = (int)(W.K / 64);
  p.NS = (int)(W.N / 16);
  p.NB = gemm_counters(W.N);
  p.U = (int64_t)p.NB * p.KT;
  const uint32_t base = W.n_table > 0 ? W.table[0] : 0;
  p.base2 = (base << 7) | (base << 23);
  uint8_t t16[16] = {0};
  for (int i = 0; i < W.n_table && i < 15; i++) t16[i] = W.table[i];
  for (int i = 0; i < 4; i++)
    p.tab[i] = t16[4 * i] | (t16[4 * i + 1] << 8) | (t16[4 * i + 2] << 16) | ((uint32_t)t16[4 * i + 3] << 24);
  p.esc_slot = W.affine ? ldexpf(1.0f, (int)base + 15 - 127) : 0.0f;
  p.view8 = 0;
  p.esc_mask = 0xFFFFu;
  p.row_base = W.row_base;
  p.cluster_k = 0;
  p.defer = 0;
  if (W.n_escapes > 0 && (!W.tile_ptr || !W.tile_esc)) {
    set_error("gemm: the tensor has escapes but no escape tile index (w12_pack_tile_index)");
    return SD_ERR_INVALID_ARG;
  }
  p.tile_ptr = W.n_escapes > 0 ? W.tile_ptr : nullptr;
  p.tile_esc = W.tile_esc;
  p.x = x;
  p.M = M;
  p.m0 = 0;
  p.partial = ws.partial;
  p.counters = ws.counters;
  p.e = epi;
  p.status = status;
  return SD_OK;
}

int gemm_launch(const w12_tensor& W, const uint16_t* x, const XMap& xm, int M, const GemmEpilogue& epi,
                const GemmWorkspace& ws, int32_t* status, cudaStream_t s, bool pdl, int grid, uint64_t* trace) {
  // a per-channel tensor has the warp-level kernel's decode only
  if (gemm_use_tc(M) && !W.row_base) return gemm_tc_launch(W, x, xm.rows_total, M, epi, ws, status, s, pdl);
  if (grid <= 0 && !trace && gemm_strip_eligible(W, M, epi.epi))
    return gemm_strip_launch(W, x, xm, M, epi, status, s, pdl);
  return gemm_warp_launch(W, x, xm, M, epi, ws, status, s, pdl, grid, trace);
}

int gemm_warp_launch(const w12_tensor& W, const uint16_t* x, const XMap& xm, int M, const GemmEpilogue& epi,
                     const GemmWorkspace& ws, int32_t* status, cudaStream_t s, bool pdl, int grid, uint64_t* trace,
                     const uint32_t* plane8) {
  if (grid <= 0) grid = gemm_warp_launch_grid(W, M, epi.epi);
  GemmParams p;
  const int prc = make_gemm_params(&p, W, x, M, epi, ws, status);
  if (prc) return prc;
  if (plane8 && (!W.affine || M > 64)) {
    set_error("gemm: the 8-bit view runs on the warp-level kernel for a contiguous exponent table and M <= 64");
    return SD_ERR_UNSUPPORTED;
  }
  if (plane8) {
    p.view8 = 1;
    p.esc_mask = 0xFFF0u;
  }
  p.trace = M <= 128 ? trace : nullptr;
  p.G = grid;
  if (ws.counters_len < p.NB) {
    set_error("gemm: workspace counters too small");
    return SD_ERR_WORKSPACE;
  }
  const int NT = nt_of(M);
  if (xm.box_rows != NT * 8) {
    set_error("gemm: tensor map box does not match the row count");
    return SD_ERR_INVALID_ARG;
  }
  if (ws.partial_floats < (size_t)grid * 2 * kRB * NT * 128) {
    set_error("gemm: workspace too small");
    return SD_ERR_WORKSPACE;
  }
  const bool aff = W.affine != 0;
  CUtensorMap wmap;
  const int wrc = plane8 ? make_w8_map(&wmap, plane8, W.N, W.K) : make_w_map(&wmap, W);
  if (wrc) return wrc;
  if (W.row_base) {
    // a per-channel tensor: the warp-level kernel's per-row decode (M <= 64,
    // every base at most 239)
    if (!W.affine || M > 64 || plane8) {
      set_error("gemm: a per-channel tensor multiplies on the warp-level kernel (M <= 64, bases <= 239, no 8-bit view)");
      return SD_ERR_UNSUPPORTED;
    }
    cudaError_t e;
    switch (NT) {
      case 1: e = launch_nt<1, true, false, true>(p, xm.map, wmap, s, pdl, grid); break;
      case 2: e = launch_nt<2, true, false, true>(p, xm.map, wmap, s, pdl, grid); break;
      case 4: e = launch_nt<4, true, false, true>(p, xm.map, wmap, s, pdl, grid); break;
      default: e = launch_nt<8, true, false, true>(p, xm.map, wmap, s, pdl, grid); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "k_w12_gemm (per-channel) launch");
    return SD_OK;
  }
  if (plane8) {
    cudaError_t e;
    switch (NT) {
      case 1: e = launch_nt<1, true, true>(p, xm.map, wmap, s, pdl, grid); break;
      case 2: e = launch_nt<2, true, true>(p, xm.map, wmap, s, pdl, grid); break;
      case 4: e = launch_nt<4, true, true>(p, xm.map, wmap, s, pdl, grid); break;
      default: e = launch_nt<8, true, true>(p, xm.map, wmap, s, pdl, grid); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "k_w12_gemm (8-bit view) launch");
    return SD_OK;
  }
  for (int m0 = 0; m0 < M; m0 += 128) {
    p.m0 = m0;
    cudaError_t e;
    switch (NT) {
      case 1: e = aff ? launch_nt<1, true>(p, xm.map, wmap, s, pdl, grid) : launch_nt<1, false>(p, xm.map, wmap, s, pdl, grid); break;
      case 2: e = aff ? launch_nt<2, true>(p, xm.map, wmap, s, pdl, grid) : launch_nt<2, false>(p, xm.map, wmap, s, pdl, grid); break;
      case 4: e = aff ? launch_nt<4, true>(p, xm.map, wmap, s, pdl, grid) : launch_nt<4, false>(p, xm.map, wmap, s, pdl, grid); break;
      case 8: e = aff ? launch_nt<8, true>(p, xm.map, wmap, s, pdl, grid) : launch_nt<8, false>(p, xm.map, wmap, s, pdl, grid); break;
      default: e = aff ? launch_nt<16, true>(p, xm.map, wmap, s, pdl, grid) : launch_nt<16, false>(p, xm.map, wmap, s, pdl, grid); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "k_w12_gemm launch");
  }
  return SD_OK;
}

}  // namespace sdv

using namespace sdv;

extern "C" int32_t sd_gemm_set_deferred_finish(int32_t enable) {
  if (enable >= 0) g_defer_finish = enable != 0;
  return g_defer_finish ? 1 : 0;
}

extern "C" int32_t sd_gemm_set_cluster_finish(int32_t enable) {
  if (enable >= 0) g_cluster_finish = enable != 0;
  return g_cluster_finish ? 1 : 0;
}

extern "C" int32_t sd_gemm_set_tc_min_rows(int32_t rows) {
  gemm_set_tc_min_rows(rows);
  return gemm_tc_min_rows();
}

static size_t al256b(size_t x) { return (x + 255) & ~size_t(255); }

extern "C" size_t sd_w12_linear_workspace(int64_t N, int64_t K, int32_t M) {
  (void)K;
  const int m = std::max(1, std::min<int>(M, 256));
  const size_t pf = gemm_partial_floats(m);
  return al256b(pf * sizeof(float)) + (size_t)gemm_counters(N) * sizeof(int32_t) + 256;
}

extern "C" int sd_w12_linear(const w12_tensor* W, const uint16_t* x, int32_t M, uint16_t* y, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (!W || !x || !y || !workspace || M < 1 || M > 256) {
    set_error("sd_w12_linear: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (W->N % 16 || W->K % 64) {
    set_error("sd_w12_linear: need N % 16 == 0 and K % 64 == 0");
    return SD_ERR_UNSUPPORTED;
  }
  if (workspace_bytes < sd_w12_linear_workspace(W->N, W->K, M) || (reinterpret_cast<uintptr_t>(workspace) & 255)) {
    set_error("sd_w12_linear: workspace too small or not 256-byte aligned");
    return SD_ERR_WORKSPACE;
  }
  cudaStream_t s = (cudaStream_t)stream;
  GemmEpilogue e;
  e.epi = EPI_STORE;
  e.out = y;
  e.ldo = (int)W->N;
  GemmWorkspace ws;
  ws.partial = reinterpret_cast<float*>(workspace);
  ws.partial_floats = gemm_partial_floats(M);
  const size_t pbytes = (ws.partial_floats * sizeof(float) + 255) & ~size_t(255);
  ws.counters = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(workspace) + pbytes);
  ws.counters_len = gemm_counters(W->N);
  SD_CK(cudaMemsetAsync(ws.counters, 0, (size_t)ws.counters_len * sizeof(int32_t), s));
  XMap xm;
  const int rc = make_x_map(&xm, x, M, W->K, M > 128 ? 128 : pad_rows(M));
  if (rc) return rc;
  return gemm_launch(*W, x, xm, M, e, ws, nullptr, s, false);
}

extern "C" size_t sd_w12_linear_view8_workspace(int64_t N, int64_t K, int32_t M) {
  return std::max(sd_w12_linear_workspace(N, K, M), sd_w12_linear_stream_workspace(N, K, M));
}

extern "C" int sd_w12_linear_view8(const w12_tensor* W, const uint32_t* plane8, const uint16_t* x, int32_t M,
                                   uint16_t* y, void* workspace, size_t workspace_bytes, void* stream) {
  if (!W || !plane8 || !x || !y || !workspace || M < 1) {
    set_error("sd_w12_linear_view8: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (M > 64 || W->N % 16 || W->K % 64) {
    set_error("sd_w12_linear_view8: need 1 <= M <= 64, N % 16 == 0 and K % 64 == 0");
    return SD_ERR_UNSUPPORTED;
  }
  if (workspace_bytes < sd_w12_linear_view8_workspace(W->N, W->K, M) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) || (reinterpret_cast<uintptr_t>(plane8) & 15)) {
    set_error("sd_w12_linear_view8: workspace too small or misaligned (256 bytes), or plane8 not 16-byte aligned");
    return SD_ERR_WORKSPACE;
  }
  if (!W->affine)  // a general exponent table: the streaming kernel decodes it
    return sd_w12_linear_stream(W, plane8, x, M, y, workspace, workspace_bytes, stream);
  cudaStream_t s = (cudaStream_t)stream;
  GemmEpilogue e;
  e.epi = EPI_STORE;
  e.out = y;
  e.ldo = (int)W->N;
  GemmWorkspace ws;
  ws.partial = reinterpret_cast<float*>(workspace);
  ws.partial_floats = gemm_partial_floats(M);
  const size_t pbytes = (ws.partial_floats * sizeof(float) + 255) & ~size_t(255);
  ws.counters = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(workspace) + pbytes);
  ws.counters_len = gemm_counters(W->N);
  SD_CK(cudaMemsetAsync(ws.counters, 0, (size_t)ws.counters_len * sizeof(int32_t), s));
  XMap xm;
  const int rc = make_x_map(&xm, x, M, W->K, pad_rows(M));
  if (rc) return rc;
  return gemm_warp_launch(*W, x, xm, M, e, ws, nullptr, s, false, 0, nullptr, plane8);
}
