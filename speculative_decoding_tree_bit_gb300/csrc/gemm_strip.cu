// Strip-parallel W12 GEMM for skinny launches with a short k range and few
// row blocks (the O and q/k/v projections: N = 4096 is 256 strips of 16
// rows, 6144 is 384).
//
// "SpecPilot: AI Agent Framework Boosts Speculative Decoding 10.87x for
// Qwen3.8-27B", "(1) W12" (decode fused into the GEMM) and "Phase 0:
// Bottleneck Analysis" (the step is a stream of weight bytes): the
// warp-level kernel splits such GEMMs over the k dimension across 6-9 CTAs
// per 128-row block, and the last CTA of a block sums the others' fp32 partials
// from global memory before the epilogue - a chain of an acq_rel ticket and
// dependent round trips that ends the launch 8-10 us after the other CTAs.
// Here a CTA owns SPC (1 or 2) 16-row strips and the whole k range, so
// nothing is summed across CTAs:
//
//  * Stage = KG = 8 / SPC consecutive 64-column tiles of each strip: each
//    strip's packed words are one contiguous run (a bulk copy), 12 KB per
//    stage in all, and the KG activation tiles, shared by the strips, come
//    by the 2-D TMA map of the warp-level kernel (64 columns x padded rows,
//    128-byte swizzle).
//  * Consumer warp w takes strip w / KG and tile w % KG of every stage - the
//    warp-level kernel's decode and mma.sync code unchanged - so the KG
//    warps of a strip hold fp32 partials over disjoint k ranges; at the end
//    the first of them sums them in shared memory in warp order
//    (deterministic) and runs the epilogue.
//  * Escapes: the CTA's strips' escapes are one contiguous run of the
//    row-major side list.  The escape warp forms their correction sum
//    (w - slot) x[m][k] per (row, m) from the activations in global memory
//    (L2) while the consumers stream, in side-list order, and hands it once
//    to the first warp of each strip.
// Results equal the warp-level kernel's up to the order of fp32 sums.
#include <cudaTypedefs.h>

#include "gemm_impl.cuh"

namespace sdv {

struct StripEsc {
  const uint32_t* row_ptr;  // side list: escapes of row n are [row_ptr[n], row_ptr[n + 1])
  const uint32_t* esc_idx;  // n * K + k
  const uint16_t* esc_val;  // bf16 bits
};

template <int NT, int SPC>
struct SCfgStrip {
  static constexpr int MP = NT * 8;
  static constexpr int KG = kNCW / SPC;          // tiles per strip per stage (k-groups)
  static constexpr int XB = MP * 128;            // one activation tile (64 columns)
  static constexpr int XS = KG * XB;             // a stage's activation tiles
  static constexpr int WB = kNCW * kStripBytes;  // a stage's weight tiles (SPC strips x KG tiles)
  // stages: as many as two CTAs per SM allow
  static constexpr int S = SPC == 1 ? (NT <= 1 ? 4 : 3) : (NT <= 1 ? 6 : 5);
  static constexpr int OFF_W = S * XS;
  static constexpr int OFF_FULL = OFF_W + S * WB;
  static constexpr int OFF_EMPTY = OFF_FULL + S * 8;
  static constexpr int OFF_CBAR = OFF_EMPTY + S * 8;   // corrections ready
  static constexpr int OFF_FLAG = OFF_CBAR + 8;        // abort flag
  static constexpr int OFF_CORR = (OFF_FLAG + 8 + 15) & ~15;  // [16 SPC rows][MP] fp32
  static constexpr int END = OFF_CORR + 16 * SPC * MP * 4;
  static constexpr int SMEM = 1024 + END;
  static_assert(kNCW * NT * 128 * 4 <= S * WB, "the reduction buffer fits the weight ring");
  static_assert(2 * (SMEM + 1024) <= 228 * 1024, "two CTAs per SM");
};

// Escapes per batch whose activation loads are in flight together.
constexpr int kStripEscBatch = 8;

template <int NT, int SPC, bool AFFINE>
__global__ void __launch_bounds__(kThreads, 2)
    k_w12_gemm_strip(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap xmap,
                     const __grid_constant__ StripEsc es) {
  using C = SCfgStrip<NT, SPC>;
  constexpr int KG = C::KG;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sx = smem;
  uint8_t* sw = smem + C::OFF_W;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_FULL);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + C::OFF_EMPTY);
  uint64_t* corr_full = reinterpret_cast<uint64_t*>(smem + C::OFF_CBAR);
  volatile int* abort = reinterpret_cast<int*>(smem + C::OFF_FLAG);
  float* corr = reinterpret_cast<float*>(smem + C::OFF_CORR);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s0 = blockIdx.x * SPC;                       // the CTA's first strip
  const int nsp = min(SPC, (int)p.NS - s0);              // its strips (the last CTA may have fewer)
  const int KT = p.KT;
  const int NJ = (KT + KG - 1) / KG;  // stages
  auto tiles_of = [&](int j) { return min(KG, KT - j * KG); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::S; i++) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kNCW);
    }
    mbar_init(corr_full, 1);
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // The grid (one CTA per strip) leaves SM slots free; a dependent launched
  // at once would take them and start its own weight stream against this
  // one's, so each warp triggers the dependents when its streaming is done.

  if (warp == kProducerWarp) {
    // ------------------------------------------------------- producer --
    if (lane == 0 && nsp > 0) {
      auto issue_w = [&](int slot, int j) {
        const int nk = tiles_of(j);
        mbar_arrive_expect_tx(&full[slot], (uint32_t)(nk * (nsp * kStripBytes + C::XB)));
        for (int si = 0; si < nsp; si++)
          bulk_g2s(sw + slot * C::WB + si * KG * kStripBytes,
                   p.words + ((int64_t)(s0 + si) * KT + (int64_t)j * KG) * (kStripBytes / 4),
                   (uint32_t)(nk * kStripBytes), &full[slot]);
      };
      auto issue_x = [&](int slot, int j) {
        const int nk = tiles_of(j);
        for (int t = 0; t < nk; t++) tma2d_g2s(sx + slot * C::XS + t * C::XB, &xmap, (j * KG + t) * 64, p.m0, &full[slot]);
      };
      const int pre = NJ < C::S ? NJ : C::S;
      for (int j = 0; j < pre; j++) issue_w(j, j);
      pdl_wait();  // activations come from the previous kernel
      for (int j = 0; j < pre; j++) issue_x(j, j);
      int slot = 0;
      uint32_t par = 0;
      for (int j = pre; j < NJ; j++) {  // runs only when pre == S
        if (!mbar_wait_or_abort(&empty[slot], par, abort)) {
          set_status(p.status, SD_TIMEOUT_AT(40));
          break;
        }
        issue_w(slot, j);
        issue_x(slot, j);
        if (++slot == C::S) {
          slot = 0;
          par ^= 1u;
        }
      }
      pdl_launch();
      // every copy this CTA started has landed before it exits
      const int issued = NJ;
      for (int s = 0; s < C::S && s < issued; s++) {
        const int n_s = issued / C::S + (s < issued % C::S ? 1 : 0);
        if (!mbar_wait(&full[s], (uint32_t)((n_s - 1) & 1))) set_status(p.status, SD_TIMEOUT_AT(41));
      }
    } else if (lane == 0) {
      pdl_wait();
    }
    pdl_launch();
    return;
  }

  if (warp == kEscapeWarp) {
    // ------------------------------------------------- escape warp --
    // corr[r][m] = sum over the strips' escapes (row 16 s0 + r, column k,
    // weight w) of (w - slot) x[m][k], in side-list order; lanes over m
    const int mrows = min(C::MP, p.M - p.m0);
    for (int i = lane; i < 16 * SPC * C::MP; i += 32) corr[i] = 0.f;
    if (p.tile_ptr != nullptr && nsp > 0) {  // the tensor has escapes
      const int64_t n0 = (int64_t)s0 * 16;
      const int64_t n1 = n0 + 16 * nsp < p.N ? n0 + 16 * nsp : p.N;
      const uint32_t e0 = __ldg(es.row_ptr + n0), e1 = __ldg(es.row_ptr + n1);
      pdl_wait();  // the activations come from the previous kernel
      const float slot_v = p.esc_slot;
      const uint16_t* xg = p.x + (int64_t)p.m0 * p.K;
      for (uint32_t c0 = e0; c0 < e1; c0 += 32) {
        // 32 escapes' (index, value) at a time, one per lane
        const uint32_t ce = c0 + lane;
        const uint32_t idx = ce < e1 ? __ldg(es.esc_idx + ce) : 0u;
        const uint32_t val = ce < e1 ? (uint32_t)__ldg(es.esc_val + ce) : 0u;
        const int cnt = (int)min(32u, e1 - c0);
        for (int b0 = 0; b0 < cnt; b0 += kStripEscBatch) {
          float xv[kStripEscBatch];
          int rr[kStripEscBatch];
          float wv[kStripEscBatch];
#pragma unroll
          for (int u = 0; u < kStripEscBatch; u++) {
            const int i = b0 + u;
            const uint32_t id = __shfl_sync(0xffffffffu, idx, i & 31);
            const uint32_t vv = __shfl_sync(0xffffffffu, val, i & 31);
            const int64_t n = (int64_t)(id / (uint64_t)p.K), k = (int64_t)(id % (uint64_t)p.K);
            rr[u] = (int)(n - n0);
            wv[u] = bf2f((uint16_t)vv);
            xv[u] = (i < cnt && lane < mrows) ? bf2f(__ldg(xg + (int64_t)lane * p.K + k)) : 0.f;
          }
#pragma unroll
          for (int u = 0; u < kStripEscBatch; u++) {
            if (b0 + u >= cnt || lane >= mrows) continue;
            float* cr = corr + rr[u] * C::MP + lane;
            const float a = fmaf(wv[u], xv[u], *cr);
            *cr = fmaf(-slot_v, xv[u], a);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(corr_full);
    pdl_launch();
    return;
  }

  // --------------------------------------------------------- consumers --
  pdl_wait();
  constexpr bool kDual = NT <= 4;
  float acc[NT][4], acc2[kDual ? NT : 1][4];
#pragma unroll
  for (int nt = 0; nt < NT; nt++)
#pragma unroll
    for (int c = 0; c < 4; c++) {
      acc[nt][c] = 0.f;
      if constexpr (kDual) acc2[nt][c] = 0.f;
    }
  int slot = 0;
  uint32_t phase = 0;
  for (int j = 0; j < NJ; j++) {
    if (!mbar_wait_or_abort(&full[slot], phase, abort)) set_status(p.status, SD_TIMEOUT_AT(42));
    if (warp / KG < nsp && j * KG + warp % KG < KT) {
      const uint8_t* wsm = sw + slot * C::WB + warp * kStripBytes;
      const uint4 W0 = *reinterpret_cast<const uint4*>(wsm + lane * 16);
      const uint4 W1 = *reinterpret_cast<const uint4*>(wsm + 512 + lane * 16);
      const uint4 W2 = *reinterpret_cast<const uint4*>(wsm + 1024 + lane * 16);
      const uint32_t xb = smem_u32(sx + slot * C::XS + (warp % KG) * C::XB);
#pragma unroll
      for (int jj = 0; jj < 4; jj++) {
        uint32_t a0, a1, a2, a3;
        decode<AFFINE>(comp(W0, jj), comp(W1, jj), comp(W2, jj), p.base2, p.tab, a0, a1, a2, a3);
        const int kchunk = 2 * jj + ((lane >> 3) & 1);
        float(*A)[4] = (kDual && (jj & 1)) ? acc2 : acc;
        if (NT == 1) {
          const int mrow = lane & 7;
          uint32_t b0, b1;
          ldsm_x2(xb + mrow * 128 + ((kchunk ^ mrow) << 4), b0, b1);
          mma_bf16(A[0], a0, a1, a2, a3, b0, b1);
        } else {
#pragma unroll
          for (int np = 0; np < NT; np += 2) {
            const int mrow = (np + (lane >> 4)) * 8 + (lane & 7);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(xb + mrow * 128 + ((kchunk ^ (lane & 7)) << 4), b0, b1, b2, b3);
            mma_bf16(A[np], a0, a1, a2, a3, b0, b1);
            mma_bf16(A[np + 1], a0, a1, a2, a3, b2, b3);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (++slot == C::S) {
      slot = 0;
      phase ^= 1u;
    }
  }
  pdl_launch();
  if constexpr (kDual) {
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int c = 0; c < 4; c++) acc[nt][c] += acc2[nt][c];
  }
  // the KG warps' partials of a strip meet in the weight ring, idle once
  // every consumer warp is past its last stage
  bar_sync(1, kNCW * 32);
  float* red = reinterpret_cast<float*>(sw);
#pragma unroll
  for (int nt = 0; nt < NT; nt++)
    *reinterpret_cast<float4*>(red + ((warp * NT + nt) * 32 + lane) * 4) =
        make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
  bar_sync(1, kNCW * 32);
  const int sidx = warp / KG;  // the warp's strip in the CTA
  if (warp % KG != 0 || sidx >= nsp) return;
  const int strip = s0 + sidx;
  float sum[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; nt++)
#pragma unroll
    for (int c = 0; c < 4; c++) sum[nt][c] = 0.f;
#pragma unroll
  for (int w = warp; w < warp + KG; w++)
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
      const float4 v = *reinterpret_cast<const float4*>(red + ((w * NT + nt) * 32 + lane) * 4);
      sum[nt][0] += v.x;
      sum[nt][1] += v.y;
      sum[nt][2] += v.z;
      sum[nt][3] += v.w;
    }
  if (!mbar_wait_or_abort(corr_full, 0u, abort)) set_status(p.status, SD_TIMEOUT_AT(43));
  {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int cc = 0; cc < 2; cc++) {
        sum[nt][cc] += corr[(sidx * 16 + g) * C::MP + nt * 8 + 2 * q + cc];
        sum[nt][2 + cc] += corr[(sidx * 16 + g + 8) * C::MP + nt * 8 + 2 * q + cc];
      }
  }
  float bestv[NT][2];
  int besti[NT][2];
  epilogue<NT>(p, strip, lane, sum, bestv, besti);
}

template <int NT, int SPC, bool AFF>
static cudaError_t launch_strip(const GemmParams& p, const CUtensorMap& xmap, const StripEsc& es, cudaStream_t s,
                                bool pdl) {
  using C = SCfgStrip<NT, SPC>;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(k_w12_gemm_strip<NT, SPC, AFF>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch(k_w12_gemm_strip<NT, SPC, AFF>, dim3((unsigned)((p.NS + SPC - 1) / SPC)), dim3(kThreads), C::SMEM, s,
                pdl, p, xmap, es);
}

static bool g_strip_gemm = true;
// Longest k range taken: a strip's CTA keeps 3 stages (36 KB of weights) in
// flight, so a long k range streams slower than the split-K kernel's deeper
// rings (the 8B-class down projection, K = 12288: 26.2 vs 22.0 us in the
// step), while for K = 4096 the removed finisher wins (O: 12.6 vs 18.0 us).
static int64_t g_strip_max_k = 4096;
bool gemm_strip_eligible_setting() { return g_strip_gemm; }

bool gemm_strip_eligible(const w12_tensor& W, int M, int epi) {
  // skinny launches (at most 16 rows, k range at most g_strip_max_k) of the
  // 12-bit words whose strips fit one wave of two CTAs per SM at one or two
  // strips per CTA; the argmax epilogue keeps its per-CTA partials on the
  // warp-level kernel
  return g_strip_gemm && M >= 1 && M <= 16 && epi != EPI_LOGITS && !W.row_base && W.N % 16 == 0 && W.K % 64 == 0 &&
         W.K <= g_strip_max_k && W.N / 16 <= 4 * (int64_t)num_sms() &&
         (W.n_escapes == 0 || (W.row_ptr && W.esc_idx && W.esc_val));
}

int gemm_strip_launch(const w12_tensor& W, const uint16_t* x, const XMap& xm, int M, const GemmEpilogue& epi,
                      int32_t* status, cudaStream_t s, bool pdl) {
  GemmParams p;
  GemmWorkspace ws;  // no partials: nothing is summed across CTAs
  const int rc = make_gemm_params(&p, W, x, M, epi, ws, status);
  if (rc) return rc;
  const int NT = M <= 8 ? 1 : 2;
  if (xm.box_rows != NT * 8) {
    set_error("gemm: tensor map box does not match the row count");
    return SD_ERR_INVALID_ARG;
  }
  StripEsc es{W.row_ptr, W.esc_idx, W.esc_val};
  // one strip per CTA while the strips fit one wave of two CTAs per SM, else
  // two (the 8B-class q/k/v: 384 strips on 192 CTAs)
  const bool two = p.NS > 2 * (int64_t)num_sms();
  cudaError_t e;
  if (NT == 1)
    e = two ? (W.affine ? launch_strip<1, 2, true>(p, xm.map, es, s, pdl) : launch_strip<1, 2, false>(p, xm.map, es, s, pdl))
            : (W.affine ? launch_strip<1, 1, true>(p, xm.map, es, s, pdl) : launch_strip<1, 1, false>(p, xm.map, es, s, pdl));
  else
    e = two ? (W.affine ? launch_strip<2, 2, true>(p, xm.map, es, s, pdl) : launch_strip<2, 2, false>(p, xm.map, es, s, pdl))
            : (W.affine ? launch_strip<2, 1, true>(p, xm.map, es, s, pdl) : launch_strip<2, 1, false>(p, xm.map, es, s, pdl));
  if (e != cudaSuccess) return cuda_fail(e, "k_w12_gemm_strip launch");
  return SD_OK;
}

}  // namespace sdv

using namespace sdv;

extern "C" int32_t sd_gemm_set_strip(int32_t enable) {
  if (enable >= 0) g_strip_gemm = enable != 0;
  return g_strip_gemm ? 1 : 0;
}
