// Persistent chain of fused W12 GEMMs and RMSNorms for sm_103a.
//
// "SpecPilot Uses Agentic Discovery ...", "Technical Mechanisms": the verify
// step is bound by the bytes of the target weights, so every microsecond in
// which HBM is not streaming weights is lost.  Launched one by one, each GEMM
// pays a ramp (ring fill), a tail (split row blocks finished after the last
// weight byte arrived) and a launch gap, and the RMSNorm between two GEMMs is
// a whole kernel of latency.  This kernel runs a run of consecutive steps of
// one layer - O (+residual) -> RMSNorm -> gate/up (+SiLU*up) -> down
// (+residual) -> RMSNorm -> next layer's q/k/v (or the lm_head) - in a single
// persistent launch:
//
//  * Phases are separated by a grid barrier: a 64-bit arrival counter in
//    global memory that only grows (one release-add per CTA and barrier,
//    nothing for the last arrival to do); barrier k of a launch is complete
//    when the counter has reached base + grid x (k + 1), base being the
//    counter's final value of the previous launch, which every CTA stores in
//    a second word before it exits (after the launch's last barrier, so no
//    CTA of the same launch can still be reading the old base).  Waits are
//    bounded.
//  * The producer warp streams the weights of the following phases into the
//    ring as soon as slots free up, without waiting for the barrier: weights
//    never depend on the previous phase.  Only the activation tile of a stage
//    waits; stages whose activations are not ready yet are queued and issued
//    the moment the producer sees the barrier generation advance.  The tail
//    of one phase and the barrier are thus hidden behind weight streaming of
//    the next.
//  * Consumer and escape warps run exactly the per-GEMM code (decode, MMA,
//    stream-K finisher, fused epilogue; escape corrections computed ahead);
//    RMSNorm phases spread the rows over the CTAs.
//  * Data produced in one phase and read in a later one is read either by the
//    copy engine after an acquire of the barrier generation and a proxy fence,
//    or with L1-bypassing loads.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "chain.cuh"
#include "gemm_impl.cuh"

namespace sdv {

struct Phase {
  int type;
  int affine;
  GemmParams g;
  ChainNorm nrm;
};

struct ChainArgs {
  CUtensorMap xmap[kChainMaxPhases];
  CUtensorMap wmap[kChainMaxPhases];
  Phase ph[kChainMaxPhases];
  int n, M;
  unsigned long long* bar;  // [0] grid-barrier arrival counter (only grows), [1] its value after the last launch
  int32_t* status;
  uint64_t* trace;  // optional: [1 + 3n][grid] globaltimer stamps (start; per phase: first stage ready,
                    // last stage consumed, phase finished)
};
static_assert(sizeof(Phase) % 4 == 0, "phase copied as words");
static_assert(sizeof(ChainArgs) <= 8192, "chain parameters too large");

template <int NT>
constexpr int chain_ctas_per_sm() { return NT <= 4 ? 2 : 1; }

template <int NT>
struct ChainCfg {
  using C = Cfg<NT>;
  // the per-GEMM layout, then the start handshake (mbarrier + the counter
  // value at launch), the RMSNorm reduction scratch and the current phase's
  // descriptor (read from shared memory in the hot loops)
  static constexpr int BASE = C::END;
  static constexpr int PHASE = BASE + 64;
  static constexpr int SMEM = C::SMEM + 64 + (int)((sizeof(Phase) + 15) & ~size_t(15));
};

__device__ __forceinline__ uint64_t ld_acquire_u64(const unsigned long long* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// One arrival per CTA, after the CTA's writes of the phase are ordered before
// this thread (named barrier): a release add, nothing to wait for.
__device__ __forceinline__ void grid_arrive(unsigned long long* bar) {
  __threadfence();
  fence_proxy_async_global();
  asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(bar) : "memory");
}

// Wait until the arrival counter reaches target; false on timeout or when
// the CTA already gave up (abort).
__device__ __forceinline__ bool grid_wait(const unsigned long long* bar, uint64_t target, volatile int* abort) {
  if ((int64_t)(ld_acquire_u64(bar) - target) >= 0) return true;
  const uint64_t t0 = globaltimer();
  while ((int64_t)(ld_acquire_u64(bar) - target) < 0) {
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *abort = 1;
      return false;
    }
  }
  return true;
}

// RMSNorm of rows blockIdx.x, blockIdx.x + G, ... by the 256 consumer threads.
__device__ __forceinline__ void norm_rows(const ChainNorm& nr, int M, float* s_red) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n8 = nr.H / 8;
  for (int m = blockIdx.x; m < M; m += gridDim.x) {
    const uint4* row = reinterpret_cast<const uint4*>(nr.src + (int64_t)m * nr.H);
    float ss = 0.f;
    for (int i = tid; i < n8; i += kNCW * 32) {
      const uint4 v = __ldcg(row + i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const float lo = bf2f(w[j] & 0xFFFF), hi = bf2f(w[j] >> 16);
        ss = fmaf(lo, lo, ss);
        ss = fmaf(hi, hi, ss);
      }
    }
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) s_red[warp] = ss;
    bar_sync(1, kNCW * 32);
    float tot = 0.f;
    for (int i = 0; i < kNCW; i++) tot += s_red[i];
    const float rinv = 1.0f / sqrtf(tot / (float)nr.H + nr.eps);
    for (int i = tid; i < n8; i += kNCW * 32) {
      const uint4 v = __ldcg(row + i);
      const uint4 gm = reinterpret_cast<const uint4*>(nr.gamma)[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      const uint32_t gg[4] = {gm.x, gm.y, gm.z, gm.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const float lo = (bf2f(w[j] & 0xFFFF) * rinv) * bf2f(gg[j] & 0xFFFF);
        const float hi = (bf2f(w[j] >> 16) * rinv) * bf2f(gg[j] >> 16);
        o[j] = pack_bf16x2(lo, hi);
      }
      reinterpret_cast<uint4*>(nr.dst + (int64_t)m * nr.H)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    bar_sync(1, kNCW * 32);  // s_red is reused by the next row
  }
}

// Producer (one thread): weights of every GEMM phase in order, activation
// tiles once their phase's input is complete.
template <int NT>
__device__ __forceinline__ void chain_produce(const ChainArgs& a, uint8_t* sx, uint8_t* sw, uint64_t* full,
                                              uint64_t* empty, uint64_t* start_ready, uint64_t* s_cnt0,
                                              volatile int* abort) {
  using C = Cfg<NT>;
  const int64_t G = gridDim.x;
  int slot = 0;
  uint32_t pph = 0;
  int64_t issued = 0;
  bool pdl_done = false;
  uint64_t cnt0 = 0;
  int seen = 0;  // barriers of this launch known to be complete
  // queued activation loads (slot, phase, column tile), oldest first
  int q_slot[C::S] = {}, q_ph[C::S] = {}, q_t[C::S] = {};
  int qh = 0, qn = 0;

  auto ensure_pdl = [&]() {
    if (pdl_done) return;
    pdl_wait();  // the previous kernel (first phase's input) is complete
    cnt0 = ld_acquire_u64(a.bar + 1);
    fence_proxy_async_global();
    *s_cnt0 = cnt0;
    mbar_arrive(start_ready);
    pdl_done = true;
  };
  auto ready = [&](int p) -> bool {
    if (!pdl_done) return false;
    if (p <= seen) return true;
    const int now = (int)((ld_acquire_u64(a.bar) - cnt0) / (uint64_t)G);
    if (now > seen) {
      seen = now;
      fence_proxy_async_global();
    }
    return p <= seen;
  };
  auto issue_x = [&]() {
    const int p = q_ph[qh];
    tma2d_g2s(sx + q_slot[qh] * C::XB, &a.xmap[p], q_t[qh] * 64, a.ph[p].g.m0, &full[q_slot[qh]]);
    qh = qh + 1 == C::S ? 0 : qh + 1;
    qn--;
  };
  auto flush = [&]() {
    while (qn > 0 && ready(q_ph[qh])) issue_x();
  };
  bool ok = true;
  for (int p = 0; p < a.n && ok; p++) {
    const Phase& P = a.ph[p];
    if (P.type != PH_GEMM) continue;
    const GemmParams& g = P.g;
    int64_t u0, u1;
    unit_range(g, u0, u1);
    if (u1 <= u0) continue;
    int b = (int)(u0 / g.KT), t = (int)(u0 % g.KT);
    for (int64_t i = u0; i < u1; i++) {
      // a free slot; queued activation loads are issued while waiting
      const uint32_t ea = smem_u32(&empty[slot]);
      if (!mbar_try_wait(ea, pph ^ 1u)) {
        ensure_pdl();
        const uint64_t t0 = globaltimer();
        bool got = false;
        for (;;) {
          flush();
          if (mbar_try_wait(ea, pph ^ 1u)) {
            got = true;
            break;
          }
          if (*abort || globaltimer() - t0 > kWaitLimitNs) break;
        }
        if (!got) {
          *abort = 1;
          set_status(a.status, SD_TIMEOUT_AT(6));
          ok = false;
          break;
        }
      }
      mbar_arrive_expect_tx(&full[slot], C::WB + C::XB);
      tma2d_g2s(sw + slot * C::WB, &a.wmap[p], t * 192, b * kRB, &full[slot]);
      const int qi = (qh + qn) % C::S;
      q_slot[qi] = slot;
      q_ph[qi] = p;
      q_t[qi] = t;
      qn++;
      flush();
      issued++;
      if (++slot == C::S) {
        slot = 0;
        pph ^= 1u;
      }
      if (++t == g.KT) {
        t = 0;
        b++;
      }
    }
  }
  ensure_pdl();
  {
    const uint64_t t0 = globaltimer();
    while (qn > 0) {
      flush();
      if (qn > 0 && (*abort || globaltimer() - t0 > kWaitLimitNs)) {
        // give up waiting for the barrier but still complete every stage
        // this CTA started (stale, in-bounds activations)
        *abort = 1;
        set_status(a.status, SD_TIMEOUT_AT(7));
        while (qn > 0) issue_x();
      }
    }
  }
  // every copy this CTA issued has landed before it exits
  for (int s = 0; s < C::S && s < issued; s++) {
    const int64_t n_s = issued / C::S + (s < issued % C::S ? 1 : 0);
    if (!mbar_wait(&full[s], (uint32_t)((n_s - 1) & 1))) set_status(a.status, SD_TIMEOUT_AT(8));
  }
}

template <int NT>
__global__ void __launch_bounds__(kThreads, chain_ctas_per_sm<NT>()) k_w12_chain(const __grid_constant__ ChainArgs a) {
  using C = Cfg<NT>;
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
  uint64_t* start_ready = reinterpret_cast<uint64_t*>(smem + ChainCfg<NT>::BASE);
  uint64_t* s_cnt0 = start_ready + 1;
  float* s_red = reinterpret_cast<float*>(s_cnt0 + 1);
  Phase* s_ph = reinterpret_cast<Phase*>(smem + ChainCfg<NT>::PHASE);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::S; i++) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kNCW + 1);  // consumer warps + escape warp
    }
    mbar_init(corr_full, 1);
    mbar_init(corr_empty, kNCW);
    mbar_init(start_ready, 1);
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch();
  const uint64_t G = gridDim.x;

  if (warp == kProducerWarp) {
    if (lane == 0) chain_produce<NT>(a, sx, sw, full, empty, start_ready, s_cnt0, abort);
    return;
  }

  // the counter's base for this launch, read by the producer after the
  // previous kernel completed
  pdl_wait();
  if (!mbar_wait_or_abort(start_ready, 0, abort)) set_status(a.status, SD_TIMEOUT_AT(9));
  const uint64_t cnt0 = *s_cnt0;

  if (warp == kEscapeWarp) {
    // ---------------------------------------------------- escape warp --
    int eseg = 0, eslot = 0;
    uint32_t ephase = 0;
    for (int p = 0; p < a.n; p++) {
      const Phase& P = a.ph[p];
      if (P.type != PH_GEMM) continue;
      // activations come staged through the ring: no wait for the phase's input
      escape_segments<NT>(P.g, sx, full, empty, eslot, ephase, corr, corr_full, corr_empty, eseg, abort);
    }
    return;
  }

  // --------------------------------------------------------- consumers --
  // After a failed wait every later wait of this CTA returns at once: the
  // consumers still run every phase (stale data, status set) and arrive at
  // every barrier, so neither this CTA's warps nor the other CTAs hang.
  if (a.trace && threadIdx.x == 0) a.trace[blockIdx.x] = globaltimer();
  int slot = 0, cseg = 0;
  uint32_t cph = 0;
  for (int p = 0; p < a.n; p++) {
    // the phase descriptor in shared memory: uniform loads with constant
    // offsets in the hot loops instead of indexed parameter reads
    {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(&a.ph[p]);
      uint32_t* dst = reinterpret_cast<uint32_t*>(s_ph);
      for (int i = threadIdx.x; i < (int)(sizeof(Phase) / 4); i += kNCW * 32) dst[i] = src[i];
      bar_sync(1, kNCW * 32);
    }
    const Phase& P = *s_ph;
    if (P.type == PH_GEMM) {
      uint64_t* st = a.trace ? a.trace + (int64_t)(1 + 3 * p) * G + blockIdx.x : nullptr;
      if (P.affine)
        consume_gemm<NT, true>(P.g, sx, sw, full, empty, red_v, red_i, flag, slot, cph, corr, corr_full, corr_empty,
                               cseg, abort, st, (int64_t)G);
      else
        consume_gemm<NT, false>(P.g, sx, sw, full, empty, red_v, red_i, flag, slot, cph, corr, corr_full, corr_empty,
                                cseg, abort, st, (int64_t)G);
    } else {
      if (p > 0) {
        // the rows were written by phase p - 1 of every CTA
        if (threadIdx.x == 0 && !grid_wait(a.bar, cnt0 + G * (uint64_t)p, abort)) set_status(a.status, SD_TIMEOUT_AT(11));
        bar_sync(1, kNCW * 32);
      }
      if (a.trace && threadIdx.x == 0) a.trace[(int64_t)(1 + 3 * p) * G + blockIdx.x] = globaltimer();
      norm_rows(P.nrm, a.M, s_red);
      if (a.trace && threadIdx.x == 0) a.trace[(int64_t)(2 + 3 * p) * G + blockIdx.x] = globaltimer();
    }
    bar_sync(1, kNCW * 32);
    if (a.trace && threadIdx.x == 0) a.trace[(int64_t)(3 + 3 * p) * G + blockIdx.x] = globaltimer();
    if (p + 1 < a.n && threadIdx.x == 0) {
      // barriers are passed in order: a CTA without work in this phase must
      // not be counted towards barrier p before barrier p - 1 has completed
      if (p > 0 && !grid_wait(a.bar, cnt0 + G * (uint64_t)p, abort)) set_status(a.status, SD_TIMEOUT_AT(12));
      grid_arrive(a.bar);
    }
  }
  if (threadIdx.x == 0) {
    // the next launch's base: the final count, stored once every CTA has
    // passed the last barrier (and so has read this launch's base)
    const uint64_t fin = cnt0 + G * (uint64_t)(a.n - 1);
    if (a.n > 1 && !grid_wait(a.bar, fin, abort)) set_status(a.status, SD_TIMEOUT_AT(13));
    *reinterpret_cast<volatile unsigned long long*>(a.bar + 1) = fin;
  }
}

// ------------------------------------------------------------------ host --

template <int NT>
static int chain_blocks_per_sm() {
  static int nb = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    carveout_once(reinterpret_cast<const void*>(k_w12_chain<NT>));
    if (cudaFuncSetAttribute(k_w12_chain<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, ChainCfg<NT>::SMEM) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k_w12_chain<NT>, kThreads, ChainCfg<NT>::SMEM) !=
            cudaSuccess)
      nb = 0;
  });
  return nb;
}

int chain_grid(int M) {
  if (M < 1 || M > 128 || gemm_use_tc(M)) return 0;
  int nb = 0, want = 0;
  switch (pad_rows(M) / 8) {
    case 1: nb = chain_blocks_per_sm<1>(); want = chain_ctas_per_sm<1>(); break;
    case 2: nb = chain_blocks_per_sm<2>(); want = chain_ctas_per_sm<2>(); break;
    case 4: nb = chain_blocks_per_sm<4>(); want = chain_ctas_per_sm<4>(); break;
    case 8: nb = chain_blocks_per_sm<8>(); want = chain_ctas_per_sm<8>(); break;
    default: nb = chain_blocks_per_sm<16>(); want = chain_ctas_per_sm<16>(); break;
  }
  // all CTAs must be resident at once (grid barriers), with the same grid as
  // the per-GEMM kernel (argmax partials per CTA)
  if (nb < want || want * num_sms() != gemm_grid(M)) return 0;
  return gemm_grid(M);
}

int chain_launch(const ChainPhaseDesc* ph, int n, int M, const GemmWorkspace& ws, unsigned long long* bar,
                 int32_t* status, cudaStream_t s, bool pdl, uint64_t* trace) {
  if (!ph || n < 1 || n > kChainMaxPhases || M < 1 || M > 128 || !bar) {
    set_error("chain: bad argument (1..6 phases, M <= 128)");
    return SD_ERR_INVALID_ARG;
  }
  const int grid = chain_grid(M);
  if (grid == 0) {
    set_error("chain: the chain kernel cannot keep its grid resident");
    return SD_ERR_UNSUPPORTED;
  }
  const int NT = pad_rows(M) / 8;
  ChainArgs a;
  memset(&a, 0, sizeof(a));
  for (int i = 0; i < n; i++) {
    Phase& P = a.ph[i];
    P.type = ph[i].type;
    if (ph[i].type == PH_GEMM) {
      if (!ph[i].W || !ph[i].x || !ph[i].xm) {
        set_error("chain: GEMM phase without weights or input");
        return SD_ERR_INVALID_ARG;
      }
      int rc = make_gemm_params(&P.g, *ph[i].W, ph[i].x, M, ph[i].epi, ws, status);
      if (rc) return rc;
      // the same partition of the units as the phase's own launch would use
      // (same contributors per row block: the same bits)
      P.g.G = gemm_launch_grid(*ph[i].W, M, ph[i].epi.epi);
      if (ws.counters_len < P.g.NB) {
        set_error("chain: workspace counters too small");
        return SD_ERR_WORKSPACE;
      }
      if (ph[i].xm->box_rows != NT * 8) {
        set_error("chain: tensor map box does not match the row count");
        return SD_ERR_INVALID_ARG;
      }
      rc = make_w_map(&a.wmap[i], *ph[i].W);
      if (rc) return rc;
      a.xmap[i] = ph[i].xm->map;
      P.affine = ph[i].W->affine != 0;
    } else if (ph[i].type == PH_NORM) {
      const ChainNorm& nr = ph[i].norm;
      if (!nr.src || !nr.gamma || !nr.dst || nr.H < 8 || nr.H % 8) {
        set_error("chain: bad RMSNorm phase");
        return SD_ERR_INVALID_ARG;
      }
      P.nrm = nr;
    } else {
      set_error("chain: unknown phase type");
      return SD_ERR_INVALID_ARG;
    }
  }
  if (ws.partial_floats < (size_t)grid * 2 * kRB * NT * 128) {
    set_error("chain: workspace too small");
    return SD_ERR_WORKSPACE;
  }
  a.n = n;
  a.M = M;
  a.bar = bar;
  a.status = status;
  a.trace = trace;
  cudaError_t e;
  switch (NT) {
    case 1: e = launch(k_w12_chain<1>, dim3(grid), dim3(kThreads), ChainCfg<1>::SMEM, s, pdl, a); break;
    case 2: e = launch(k_w12_chain<2>, dim3(grid), dim3(kThreads), ChainCfg<2>::SMEM, s, pdl, a); break;
    case 4: e = launch(k_w12_chain<4>, dim3(grid), dim3(kThreads), ChainCfg<4>::SMEM, s, pdl, a); break;
    case 8: e = launch(k_w12_chain<8>, dim3(grid), dim3(kThreads), ChainCfg<8>::SMEM, s, pdl, a); break;
    default: e = launch(k_w12_chain<16>, dim3(grid), dim3(kThreads), ChainCfg<16>::SMEM, s, pdl, a); break;
  }
  if (e != cudaSuccess) return cuda_fail(e, "k_w12_chain launch");
  return SD_OK;
}

}  // namespace sdv
