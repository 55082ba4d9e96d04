// Fused W12-decode GEMM on the fifth-generation tensor cores (tcgen05 + TMEM)
// for launches with many rows.
//
// "SpecPilot: AI Agent Framework Boosts Speculative Decoding 10.87x for
// Qwen3.8-27B", "(1) W12" and the batched results: once a verify call
// carries a few hundred rows (many requests' trees at once), the GEMM's
// FLOPs per weight byte reach the tensor cores' balance point and the
// warp-level MMA path of the skinny kernel becomes the bound.  This kernel
// keeps the weights crossing HBM once at 1.5 bytes each and moves the math to
// tcgen05:
//
//  * D[n][m] = sum_k W[n][k] x[m][k] per 128-row weight block: weights are the
//    M = 128 side of tcgen05.mma.cta_group::1.kind::f16, the launch's rows
//    (padded to a multiple of 16, at most 256) the N side; fp32 accumulators
//    live in tensor memory, two buffers so that one block's epilogue overlaps
//    the next block's main loop.
//  * Warp 0 streams, per 64-column k-tile, the packed words of the block
//    (one 2-D TMA box: 8 strips x 1536 bytes) and the activation tile
//    (2-D TMA box, 128-byte swizzle) into separate mbarrier rings.
//  * Warps 6..13 decode one 16-row strip each into a bf16 tile laid out as
//    the MMA's K-major 128-byte-swizzled operand, then write the strip's
//    escaped weights (from the escape tile index) over their slots: the
//    operand is the exact bf16 weight block.
//  * Warp 1 (one thread) issues four K = 16 MMAs per k-tile and releases
//    the stage with one tcgen05.commit.  An mbarrier wait costs its warp a
//    round trip of over a hundred cycles even on a completed phase, so the
//    MMA thread and the decoders probe the next k-tile's barriers with
//    test_wait before the current k-tile's work and block only when a probe
//    found a phase incomplete.
//  * Warps 2..5 (one TMEM lane quarter each) read the accumulators
//    (tcgen05.ld) and run the same fused epilogues as the skinny kernel.
//  * Work = (row block, k-tile) units split evenly over one CTA per SM
//    (stream-K); a block split between CTAs is finished by the last
//    contributor, which sums the fp32 partials in CTA order (deterministic).
#include <cudaTypedefs.h>

#include <algorithm>

#include "gemm_impl.cuh"

namespace sdv {

namespace tc {
constexpr int kProducer = 0;
constexpr int kMma = 1;
constexpr int kEpi0 = 2;  // warps 2..5: epilogue
constexpr int kDec0 = 6;  // warps 6..13: decoders (strip = warp - kDec0)
constexpr int kThreads = (kDec0 + kRB) * 32;
constexpr int kATile = 128 * 128;             // decoded block: 128 rows x 64 bf16
constexpr int kWTile = kRB * kStripBytes;     // packed block: 8 strips x 1536 bytes
constexpr int kSmemMax = 227 * 1024;
constexpr int kMaxCon = 512;  // CTAs of a launch (bounds a finisher's list of contributors)
}  // namespace tc

struct TcParams {
  GemmParams g;
  int MP;          // rows of the MMA's N side (multiple of 16, 32..256)
  int acc_cols;    // TMEM columns between the two accumulator buffers
  int tmem_cols;   // TMEM columns allocated (power of two)
  uint32_t idesc;  // instruction descriptor
  int S, SW;       // ring stages: (activation + decoded weight) tiles, packed weights
  int off_a, off_w, off_bar, off_red, off_rows, off_con, smem;
};

// ------------------------------------------------------- tcgen05 helpers --

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (tmem) (+)= A (smem) * B (smem)^T, both K-major.
__device__ __forceinline__ void umma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier receives one arrival once every MMA this thread issued so far
// has completed (and its shared-memory reads with it).
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  // the registers are tied to the wait so that no use moves above it
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// Shared-memory operand descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (the leading offset is unused for this layout).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Byte offset of (row, column k) in a K-major 128-byte-swizzled tile of
// 64-column rows (the layout the copy engine writes for SWIZZLE_128B).
__device__ __forceinline__ uint32_t sw128_off(int row, int k) {
  return (uint32_t)(row * 128 + ((((k >> 3) ^ (row & 7))) << 4) + (k & 7) * 2);
}

// ---------------------------------------------------------- epilogue --

// Running argmax candidate: larger value, then smaller index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

// Per-row (token) data of the QKV epilogue, staged in shared memory once per
// launch: RoPE position and the offset of the row's KV-cache slot (-1 when
// the row's request is not written).
struct TcRows {
  int* pos;
  long long* kv_off;
};

// Epilogue of 16 accumulator columns (rows m = c0 .. c0 + 15 of the launch)
// of weight row n (this thread's TMEM lane).  Rows of a 16-row strip pair
// up (g, g + 8) for SiLU(gate) * up and the RoPE halves: the partner value
// comes from lane + 8.  Every global load of a chunk is issued before its
// stores (no load waits behind a store that might alias it).
template <int EPI>
__device__ __forceinline__ void tc_emit(const TcParams& P, int64_t n, int c0, const float (&v)[16], float* red_v,
                                        int* red_i, int quarter, const TcRows& rows) {
  const GemmParams& p = P.g;
  const GemmEpilogue& E = p.e;
  const int lane = threadIdx.x & 31;
  const bool valid_n = n < p.N;
  const int g = (int)(n & 15);
  const int mlim = p.M - c0;  // rows j < mlim are real
  switch (EPI) {
    case EPI_LOGITS: {
#pragma unroll
      for (int j = 0; j < 16; j++) {
        const int m = c0 + j;
        float bv = valid_n ? v[j] : -INFINITY;
        int bi = valid_n ? (int)n : 0x7FFFFFFF;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
          if (better(ov, oi, bv, bi)) {
            bv = ov;
            bi = oi;
          }
        }
        if (j < mlim) {
          if (lane == 0 && better(bv, bi, red_v[quarter * P.MP + m], red_i[quarter * P.MP + m])) {
            red_v[quarter * P.MP + m] = bv;
            red_i[quarter * P.MP + m] = bi;
          }
          if (E.out && valid_n) E.out[(int64_t)m * E.ldo + n] = f2bf(v[j]);
        }
      }
      break;
    }
    case EPI_STORE:
      if (valid_n)
#pragma unroll
        for (int j = 0; j < 16; j++)
          if (j < mlim) E.out[(int64_t)(c0 + j) * E.ldo + n] = f2bf(v[j]);
      break;
    case EPI_RESID: {
      if (!valid_n) break;
      float r[16];
#pragma unroll
      for (int j = 0; j < 16; j++) r[j] = j < mlim ? bf2f(__ldcg(E.resid + (int64_t)(c0 + j) * E.ldo + n)) : 0.f;
#pragma unroll
      for (int j = 0; j < 16; j++)
        if (j < mlim) E.out[(int64_t)(c0 + j) * E.ldo + n] = f2bf(r[j] + rbf(v[j]));
      break;
    }
    case EPI_SILU: {
      float hi[16];
#pragma unroll
      for (int j = 0; j < 16; j++) hi[j] = __shfl_down_sync(0xffffffffu, v[j], 8);
      if (valid_n && g < 8)
#pragma unroll
        for (int j = 0; j < 16; j++)
          if (j < mlim) {
            const float gt = rbf(v[j]), up = rbf(hi[j]);
            const float sv = gt / (1.0f + expf(-gt));
            E.out[(int64_t)(c0 + j) * E.ldo + (n >> 4) * 8 + g] = f2bf(sv * up);
          }
      break;
    }
    case EPI_QKV: {
      float hi[16];
#pragma unroll
      for (int j = 0; j < 16; j++) hi[j] = __shfl_down_sync(0xffffffffu, v[j], 8);
      if (!valid_n) break;
      const int64_t qrows = (int64_t)E.hq * 128, krows = (int64_t)E.hkv * 128;
      const int64_t row0 = n - g;
      const int64_t head_stride = (int64_t)E.cache.page_size * 128;
      if (row0 < qrows + krows) {
        if (g >= 8) break;
        const bool is_q = row0 < qrows;
        const int64_t rr = is_q ? row0 : row0 - qrows;
        const int head = (int)(rr / 128);
        const int d = (int)((rr % 128) / 16) * 8 + g;
        float cs[16], sn[16];
#pragma unroll
        for (int j = 0; j < 16; j++) {
          const int pos = j < mlim ? rows.pos[c0 + j] : 0;
          cs[j] = E.rope_cos[(int64_t)pos * 64 + d];
          sn[j] = E.rope_sin[(int64_t)pos * 64 + d];
        }
#pragma unroll
        for (int j = 0; j < 16; j++) {
          if (j >= mlim) continue;
          const int m = c0 + j;
          const float x1 = rbf(v[j]), x2 = rbf(hi[j]);
          const uint16_t o1 = f2bf(x1 * cs[j] - x2 * sn[j]), o2 = f2bf(x2 * cs[j] + x1 * sn[j]);
          if (is_q) {
            uint16_t* dst = E.q_out + ((int64_t)m * E.hq + head) * 128;
            dst[d] = o1;
            dst[d + 64] = o2;
          } else {
            const long long off = rows.kv_off[m];
            if (off >= 0) {
              uint16_t* dst = E.cache.k + off + head * head_stride;
              dst[d] = o1;
              dst[d + 64] = o2;
            }
          }
        }
      } else {
        const int64_t vr = n - qrows - krows;
        const int head = (int)(vr / 128);
        const int d = (int)(vr % 128);
#pragma unroll
        for (int j = 0; j < 16; j++) {
          if (j >= mlim) continue;
          const long long off = rows.kv_off[c0 + j];
          if (off >= 0) E.cache.v[off + head * head_stride + d] = f2bf(v[j]);
        }
      }
      break;
    }
  }
}

// ------------------------------------------------------------ kernel --

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

template <bool AFFINE, int EPI>
__global__ void __launch_bounds__(tc::kThreads, 1)
    k_w12_gemm_tc(const __grid_constant__ TcParams P, const __grid_constant__ CUtensorMap xmap,
                  const __grid_constant__ CUtensorMap wmap) {
  const GemmParams& p = P.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sx = smem;
  uint8_t* sa = smem + P.off_a;
  uint8_t* sw = smem + P.off_w;
  uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + P.off_bar);
  uint64_t* wempty = wfull + P.SW;
  uint64_t* xfull = wempty + P.SW;   // activation tile landed (copy engine)
  uint64_t* afull = xfull + P.S;     // decoded tile written and activation tile seen (8 decoder warps)
  uint64_t* sempty = afull + P.S;    // the stage's MMAs are done (commit)
  uint64_t* accfull = sempty + P.S;
  uint64_t* accempty = accfull + 2;
  uint64_t* mma_done = accempty + 2;
  uint64_t* gbar = mma_done + 1;  // [2] finisher staging (bulk copies of partial slices)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbar + 2);
  int* flag = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* abort = flag + 1;
  float* red_v = reinterpret_cast<float*>(smem + P.off_red);
  int* red_i = reinterpret_cast<int*>(red_v + 4 * P.MP);
  TcRows rows;
  rows.kv_off = reinterpret_cast<long long*>(smem + P.off_rows);
  rows.pos = reinterpret_cast<int*>(rows.kv_off + P.MP);
  int* con = reinterpret_cast<int*>(smem + P.off_con);  // finisher: the others' partial slices
  int* con_cnt = con + tc::kMaxCon;                      // [0..3] per-warp counts, [4] this CTA's place

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  const int64_t u0 = udiv((int64_t)blockIdx.x * p.U, G), u1 = udiv((int64_t)(blockIdx.x + 1) * p.U, G);
  const int64_t n_units = u1 - u0;
  const int KT = p.KT;
  const int XB = P.MP * 128;

  if (threadIdx.x == 0) {
    for (int i = 0; i < P.SW; i++) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], kRB);
    }
    for (int i = 0; i < P.S; i++) {
      mbar_init(&xfull[i], 1);
      mbar_init(&afull[i], kRB);
      mbar_init(&sempty[i], 1);
    }
    for (int i = 0; i < 2; i++) {
      mbar_init(&accfull[i], 1);
      mbar_init(&accempty[i], 4);
    }
    mbar_init(mma_done, 1);
    mbar_init(&gbar[0], 1);
    mbar_init(&gbar[1], 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == tc::kMma) {
    tmem_alloc(tmem_slot, (uint32_t)P.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch();

  if (warp == tc::kProducer) {
    // ------------------------------------------------------- producer --
    if (lane == 0) {
      int64_t nw = 0, nx = 0;  // copies issued
      if (n_units > 0) {
        const int pre = (int)min64(n_units, P.SW);
        for (int i = 0; i < pre; i++) {
          const int64_t u = u0 + i, ub = udiv(u, KT);
          mbar_arrive_expect_tx(&wfull[i], tc::kWTile);
          tma2d_g2s(sw + i * tc::kWTile, &wmap, (int)(u - ub * KT) * 192, (int)ub * kRB, &wfull[i]);
        }
        nw = pre;
        pdl_wait();  // activations come from the previous kernel
        int xs = 0, ws = 0;
        uint32_t xph = 0, wph = 0;
        for (int64_t i = 0; i < n_units; i++) {
          const int64_t u = u0 + i;
          if (i >= P.S && !mbar_wait_or_abort(&sempty[xs], xph ^ 1u, abort)) {
            set_status(p.status, SD_TIMEOUT_AT(21));
            break;
          }
          mbar_arrive_expect_tx(&xfull[xs], (uint32_t)XB);
          tma2d_g2s(sx + xs * XB, &xmap, (int)(u - udiv(u, KT) * KT) * 64, 0, &xfull[xs]);
          nx++;
          if (++xs == P.S) {
            xs = 0;
            xph ^= 1u;
          }
          const int64_t j = i + P.SW;  // weights run SW k-tiles ahead
          if (j < n_units) {
            if (!mbar_wait_or_abort(&wempty[ws], wph, abort)) {
              set_status(p.status, SD_TIMEOUT_AT(22));
              break;
            }
            const int64_t uj = u0 + j, ujb = udiv(uj, KT);
            mbar_arrive_expect_tx(&wfull[ws], tc::kWTile);
            tma2d_g2s(sw + ws * tc::kWTile, &wmap, (int)(uj - ujb * KT) * 192, (int)ujb * kRB, &wfull[ws]);
            nw++;
          }
          if (++ws == P.SW) {
            ws = 0;
            wph ^= 1u;
          }
        }
      } else {
        pdl_wait();
      }
      // every copy this CTA started has landed before it exits
      for (int s = 0; s < P.SW && s < nw; s++) {
        const int64_t k = nw / P.SW + (s < nw % P.SW ? 1 : 0);
        if (!mbar_wait(&wfull[s], (uint32_t)((k - 1) & 1))) set_status(p.status, SD_TIMEOUT_AT(23));
      }
      for (int s = 0; s < P.S && s < nx; s++) {
        const int64_t k = nx / P.S + (s < nx % P.S ? 1 : 0);
        if (!mbar_wait(&xfull[s], (uint32_t)((k - 1) & 1))) set_status(p.status, SD_TIMEOUT_AT(24));
      }
    }
    __syncwarp();  // the teardown barrier below wants every warp converged
  } else if (warp == tc::kMma) {
    // ---------------------------------------------------- MMA issuer --
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      bool ready = false;  // the current stage's probes found it complete
      int64_t i = 0;
      int seg = 0;
      const uint32_t a0 = smem_u32(sa), x0 = smem_u32(sx);
      while (i < n_units) {
        const int64_t u = u0 + i;
        const int t0 = (int)(u - udiv(u, KT) * KT);
        const int len = (int)min64(KT - t0, n_units - i);
        const int buf = seg & 1;
        if (seg >= 2 && !mbar_wait_or_abort(&accempty[buf], (uint32_t)(((seg >> 1) - 1) & 1), abort))
          set_status(p.status, SD_TIMEOUT_AT(25));
        tc_fence_after();  // the epilogue's reads of this buffer come first
        const uint32_t d = tmem + (uint32_t)(buf * P.acc_cols);
        for (int k = 0; k < len; k++) {
          // the probes of this stage were issued a k-tile ago; block only if
          // they found it incomplete
          if (!ready) {
            bool ok = mbar_wait_or_abort(&afull[st], ph, abort);
            ok = mbar_wait_or_abort(&xfull[st], ph, abort) && ok;
            if (!ok) set_status(p.status, SD_TIMEOUT_AT(26));
          }
          const int cur = st;
          if (++st == P.S) {
            st = 0;
            ph ^= 1u;
          }
          // both probes go out before the MMAs (no branch on their results here)
          bool pa = false, px = false;
          if (i + k + 1 < n_units) {
            pa = mbar_test_wait(&afull[st], ph);
            px = mbar_test_wait(&xfull[st], ph);
          }
          if (!*abort) {
            const uint64_t da = sdesc_sw128(a0 + (uint32_t)(cur * tc::kATile));
            const uint64_t db = sdesc_sw128(x0 + (uint32_t)(cur * XB));
#pragma unroll
            for (int kk = 0; kk < 4; kk++)  // K = 16 per MMA: +32 bytes inside the swizzle atom
              umma_bf16(d, da + 2 * kk, db + 2 * kk, P.idesc, (k | kk) != 0 ? 1u : 0u);
          }
          umma_commit(&sempty[cur]);
          ready = pa && px;
        }
        umma_commit(&accfull[buf]);
        seg++;
        i += len;
      }
      // nothing may still write tensor memory when it is freed
      umma_commit(mma_done);
      if (!mbar_wait(mma_done, 0)) set_status(p.status, SD_TIMEOUT_AT(27));
    }
    __syncwarp();
  } else if (warp < tc::kDec0) {
    // ------------------------------------------------------- epilogue --
    const int quarter = warp & 3;  // TMEM lanes 32 * quarter .. + 31
    const int r = quarter * 32 + lane;
    pdl_wait();
    if (EPI == EPI_LOGITS)
      for (int m = lane; m < P.MP; m += 32) {
        red_v[quarter * P.MP + m] = -INFINITY;
        red_i[quarter * P.MP + m] = 0x7FFFFFFF;
      }
    if (EPI == EPI_QKV) {
      const GemmEpilogue& E = p.e;
      for (int m = threadIdx.x - tc::kEpi0 * 32; m < p.M && m < P.MP; m += 128) {
        rows.pos[m] = E.rows.pos[m];
        const int rq = E.rows.req[m];
        long long off = -1;
        if (E.rows.req_ok[rq]) {
          const int slot = E.rows.slot[m];
          const int page = E.cache.page_table[(int64_t)rq * E.cache.max_pages + slot / E.cache.page_size];
          off = ((long long)page * E.cache.hkv * E.cache.page_size + slot % E.cache.page_size) * 128;
        }
        rows.kv_off[m] = off;
      }
    }
    bar_sync(2, 128);
    const int mrows = P.MP < p.M ? P.MP : p.M;
    const int nch = (mrows + 15) / 16;
    const int first_b = n_units > 0 ? (int)udiv(u0, KT) : -1;
    uint32_t stg_par = 0;  // bit b: parity of the next phase of staging barrier b
    int64_t i = 0;
    int seg = 0;
    while (i < n_units) {
      const int64_t u = u0 + i;
      const int b = (int)udiv(u, KT), t0 = (int)(u - (int64_t)b * KT);
      const int len = (int)min64(KT - t0, n_units - i);
      const int buf = seg & 1;
      if (!mbar_wait_or_abort(&accfull[buf], (uint32_t)((seg >> 1) & 1), abort))
        set_status(p.status, SD_TIMEOUT_AT(28));
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * P.acc_cols);
      const int64_t n = (int64_t)b * 128 + r;
      if (t0 == 0 && len == KT) {
        for (int c = 0; c < nch; c++) {
          float v[16];
          tmem_ld16(taddr + 16 * c, v);
          tc_emit<EPI>(P, n, 16 * c, v, red_v, red_i, quarter, rows);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&accempty[buf]);
      } else {
        const int sid = (b == first_b) ? 0 : 1;
        float* dst = p.partial + ((int64_t)(blockIdx.x * 2 + sid) * P.MP) * 128 + r;
        for (int c = 0; c < nch; c++) {
          float v[16];
          tmem_ld16(taddr + 16 * c, v);
#pragma unroll
          for (int j = 0; j < 16; j++) __stcg(dst + (16 * c + j) * 128, v[j]);
        }
        // the named barrier orders every thread's partial before the ticket
        bar_sync(2, 128);
        if (threadIdx.x == tc::kEpi0 * 32) {
          const int old = atomic_add_acq_rel(&p.counters[b], len);
          *flag = (old + len == KT) ? 1 : 0;
        }
        bar_sync(2, 128);
        if (*flag) {
          // contributors: the CTAs whose (non-empty) unit range meets block b,
          // summed in CTA order; this CTA's own share comes from TMEM (still
          // held)
          const int64_t c_first = udiv(((int64_t)b * KT + 1) * G - 1, p.U);
          const int64_t c_last = udiv(((int64_t)(b + 1) * KT) * G - 1, p.U);
          // the others' partial slices in CTA order, con[0 .. n_oth), and
          // k_self, how many of them precede this CTA: listed once by the 128
          // epilogue threads (a contributor each), so that the loops below
          // divide nothing
          const int et = threadIdx.x - tc::kEpi0 * 32, ew = et >> 5;
          int n_oth = 0;
          for (int64_t w = c_first; w <= c_last; w += 128) {
            const int64_t cc = w + et;
            bool o = false;
            int64_t cs = 0;
            if (cc <= c_last) {
              cs = udiv(cc * p.U, G);
              o = cs != udiv((cc + 1) * p.U, G) && cc != (int64_t)blockIdx.x;  // empty ranges wrote no partial
            }
            const uint32_t om = __ballot_sync(0xffffffffu, o);
            if (lane == 0) con_cnt[ew] = __popc(om);
            bar_sync(2, 128);
            int at = n_oth + __popc(om & ((1u << lane) - 1u));
            for (int q = 0; q < ew; q++) at += con_cnt[q];
            // a range that began in an earlier block left this block's share
            // in its second slice
            if (o) con[at] = (int)(cc * 2 + (cs < (int64_t)b * KT ? 1 : 0));
            if (cc == (int64_t)blockIdx.x) con_cnt[4] = at;
            n_oth += con_cnt[0] + con_cnt[1] + con_cnt[2] + con_cnt[3];
            bar_sync(2, 128);
          }
          const int k_self = con_cnt[4];
          // the CTA's last segment: the rings are idle (every copy consumed,
          // every MMA complete), so one thread stages the others' partial
          // slices there with bulk copies, two column groups in flight
          int GC = 64;
          while (GC > 16 && 2 * n_oth * GC * 512 > P.off_bar) GC >>= 1;
          const bool staged = i + len == n_units && n_oth > 0 && 2 * n_oth * GC * 512 <= P.off_bar;
          if (staged) {
            float* stage = reinterpret_cast<float*>(smem);
            const int ngroups = (nch * 16 + GC - 1) / GC;
            auto issue = [&](int gi) {
              if (threadIdx.x != tc::kEpi0 * 32) return;
              const int cols = min(GC, P.MP - gi * GC);
              fence_async_smem();  // earlier generic reads of the buffer come first
              mbar_arrive_expect_tx(&gbar[gi & 1], (uint32_t)(n_oth * cols * 512));
              for (int k = 0; k < n_oth; k++)
                bulk_g2s(stage + (int64_t)((gi & 1) * n_oth + k) * GC * 128,
                         p.partial + ((int64_t)con[k] * P.MP + gi * GC) * 128, (uint32_t)(cols * 512), &gbar[gi & 1]);
            };
            issue(0);
            for (int gi = 0; gi < ngroups; gi++) {
              if (gi + 1 < ngroups) {
                bar_sync(2, 128);  // every thread is done with the buffer group gi + 1 reuses
                issue(gi + 1);
              }
              if (!mbar_wait_or_abort(&gbar[gi & 1], (stg_par >> (gi & 1)) & 1u, abort))
                set_status(p.status, SD_TIMEOUT_AT(31));
              stg_par ^= 1u << (gi & 1);
              const float* sb = stage + (int64_t)((gi & 1) * n_oth) * GC * 128 + r;
              for (int cl = 0; cl < GC / 16; cl++) {
                const int c = gi * (GC / 16) + cl;
                if (c >= nch) break;
                float own[16], v[16];
                tmem_ld16(taddr + 16 * c, own);
#pragma unroll
                for (int j = 0; j < 16; j++) v[j] = 0.f;
                for (int k = 0; k < n_oth; k++) {
                  if (k == k_self)
#pragma unroll
                    for (int j = 0; j < 16; j++) v[j] += own[j];
                  const float* src = sb + (int64_t)k * GC * 128 + cl * 16 * 128;
#pragma unroll
                  for (int j = 0; j < 16; j++) v[j] += src[j * 128];
                }
                if (k_self == n_oth)
#pragma unroll
                  for (int j = 0; j < 16; j++) v[j] += own[j];
                tc_emit<EPI>(P, n, 16 * c, v, red_v, red_i, quarter, rows);
              }
            }
          } else {
            // two contributors' loads in flight at a time
            for (int c = 0; c < nch; c++) {
              float own[16], v[16];
              tmem_ld16(taddr + 16 * c, own);
#pragma unroll
              for (int j = 0; j < 16; j++) v[j] = 0.f;
              for (int k0 = 0; k0 < n_oth; k0 += 2) {
                float w[2][16];
#pragma unroll
                for (int u = 0; u < 2; u++) {
                  const bool use = k0 + u < n_oth;
                  const float* src = p.partial + ((int64_t)(use ? con[k0 + u] : 0) * P.MP + 16 * c) * 128 + r;
#pragma unroll
                  for (int j = 0; j < 16; j++) w[u][j] = use ? __ldcg(src + j * 128) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 2; u++) {
                  if (k0 + u >= n_oth) break;
                  if (k0 + u == k_self)
#pragma unroll
                    for (int j = 0; j < 16; j++) v[j] += own[j];
#pragma unroll
                  for (int j = 0; j < 16; j++) v[j] += w[u][j];
                }
              }
              if (k_self == n_oth)
#pragma unroll
                for (int j = 0; j < 16; j++) v[j] += own[j];
              tc_emit<EPI>(P, n, 16 * c, v, red_v, red_i, quarter, rows);
            }
          }
          if (threadIdx.x == tc::kEpi0 * 32) p.counters[b] = 0;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&accempty[buf]);
      }
      seg++;
      i += len;
    }
    if (EPI == EPI_LOGITS) {
      bar_sync(2, 128);
      const int et = threadIdx.x - tc::kEpi0 * 32;
      for (int m = et; m < mrows; m += 128) {
        float v = red_v[m];
        int ix = red_i[m];
        for (int q = 1; q < 4; q++)
          if (better(red_v[q * P.MP + m], red_i[q * P.MP + m], v, ix)) {
            v = red_v[q * P.MP + m];
            ix = red_i[q * P.MP + m];
          }
        p.e.amax_val[(int64_t)blockIdx.x * p.e.ld_amax + m] = v;
        p.e.amax_idx[(int64_t)blockIdx.x * p.e.ld_amax + m] = ix;
      }
    }
  } else {
    // ------------------------------------------------------- decoders --
    const int d = warp - tc::kDec0;  // strip of the block
    const int g = lane >> 2, q = lane & 3;
    const bool any = p.tile_ptr != nullptr;
    // escape tile index of the unit range: entries of unit u are
    // tile_esc[tile_ptr[u] .. tile_ptr[u + 1]); lane l holds the pointers of
    // unit (chunk base + l), chunks of 32 units, the next chunk loaded 32
    // units ahead.  Lane l's entry l of the next kEscAhead units is in flight
    // (shift registers: slot 0 is the current unit).
    constexpr int kEscAhead = 8;
    uint32_t pa = 0, pb = 0, pan = 0, pbn = 0;
    auto load_ptrs = [&](int64_t base, uint32_t& a, uint32_t& bb) {
      a = __ldg(p.tile_ptr + min64(base + lane, u1));
      bb = __ldg(p.tile_ptr + min64(base + lane + 1, u1));
    };
    uint32_t q_ent[kEscAhead], q_base[kEscAhead], q_cnt[kEscAhead];
#pragma unroll
    for (int k = 0; k < kEscAhead; k++) q_ent[k] = q_base[k] = q_cnt[k] = 0;
    // unit k's entries (k in the current pointer chunk)
    auto fetch = [&](int64_t k, uint32_t& ent, uint32_t& base, uint32_t& cnt) {
      const int pos = (int)(k & 31);
      base = __shfl_sync(0xffffffffu, pa, pos);
      cnt = __shfl_sync(0xffffffffu, pb, pos) - base;
      ent = lane < (int)cnt ? __ldg(p.tile_esc + base + lane) : 0u;
    };
    if (any && n_units > 0) {
      load_ptrs(u0, pa, pb);
      if (n_units > 32) load_ptrs(u0 + 32, pan, pbn);
#pragma unroll
      for (int k = 0; k < kEscAhead; k++)
        if (k < n_units) fetch(k, q_ent[k], q_base[k], q_cnt[k]);
    }
    int ws = 0, as = 0;
    uint32_t wph = 0, aph = 0;
    bool w_ok = false, s_ok = false;  // probes of the current k-tile's barriers found them complete
    const uint32_t off_lo = (uint32_t)((16 * d + g) * 128) + 4 * q, off_hi = off_lo + 8 * 128;
    for (int64_t i = 0; i < n_units; i++) {
      // entries of unit i + kEscAhead go in flight now
      uint32_t ent_n = 0, base_n = 0, cnt_n = 0;
      const int64_t kn = i + kEscAhead;
      if (any && kn < n_units) {
        if ((kn & 31) == 0) {
          pa = pan;
          pb = pbn;
          if (kn + 32 < n_units) load_ptrs(u0 + kn + 32, pan, pbn);
        }
        fetch(kn, ent_n, base_n, cnt_n);
      }
      const uint32_t ent = q_ent[0], e_base = q_base[0], e_cnt = q_cnt[0];
      if (!w_ok && !mbar_wait_or_abort(&wfull[ws], wph, abort)) set_status(p.status, SD_TIMEOUT_AT(29));
      const uint8_t* src = sw + ws * tc::kWTile + d * kStripBytes + lane * 16;
      const uint4 W0 = *reinterpret_cast<const uint4*>(src);
      const uint4 W1 = *reinterpret_cast<const uint4*>(src + 512);
      const uint4 W2 = *reinterpret_cast<const uint4*>(src + 1024);
      __syncwarp();
      if (lane == 0) mbar_arrive(&wempty[ws]);
      if (++ws == P.SW) {
        ws = 0;
        wph ^= 1u;
      }
      if (i >= P.S && !s_ok && !mbar_wait_or_abort(&sempty[as], aph ^ 1u, abort))
        set_status(p.status, SD_TIMEOUT_AT(30));
      // probe the next k-tile's barriers now; the decode below hides the round trip
      {
        const int nas = as + 1 == P.S ? 0 : as + 1;
        const uint32_t naph = as + 1 == P.S ? aph ^ 1u : aph;
        w_ok = i + 1 < n_units && mbar_test_wait(&wfull[ws], wph);
        s_ok = i + 1 < P.S || (i + 1 < n_units && mbar_test_wait(&sempty[nas], naph ^ 1u));
      }
      uint8_t* dst = sa + as * tc::kATile;
#pragma unroll
      for (int j = 0; j < 4; j++) {
        uint32_t a0, a1, a2, a3;
        decode<AFFINE>(comp(W0, j), comp(W1, j), comp(W2, j), p.base2, p.tab, a0, a1, a2, a3);
        const uint32_t c_lo = (uint32_t)(((2 * j) ^ g) << 4), c_hi = (uint32_t)(((2 * j + 1) ^ g) << 4);
        *reinterpret_cast<uint32_t*>(dst + off_lo + c_lo) = a0;
        *reinterpret_cast<uint32_t*>(dst + off_hi + c_lo) = a1;
        *reinterpret_cast<uint32_t*>(dst + off_lo + c_hi) = a2;
        *reinterpret_cast<uint32_t*>(dst + off_hi + c_hi) = a3;
      }
      if (any && e_cnt > 0) {
        // escaped weights of this strip overwrite their slots
        __syncwarp();
        for (uint32_t e = lane; e < e_cnt; e += 32) {
          const uint32_t v = e < 32 ? ent : __ldg(p.tile_esc + e_base + e);
          const int row = (int)((v >> 6) & 127);
          if ((row >> 4) == d) *reinterpret_cast<uint16_t*>(dst + sw128_off(row, (int)(v & 63))) = (uint16_t)(v >> 16);
        }
      }
      // the tile is read by the tensor cores (async proxy)
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull[as]);
      if (++as == P.S) {
        as = 0;
        aph ^= 1u;
      }
#pragma unroll
      for (int k = 0; k + 1 < kEscAhead; k++) {
        q_ent[k] = q_ent[k + 1];
        q_base[k] = q_base[k + 1];
        q_cnt[k] = q_cnt[k + 1];
      }
      q_ent[kEscAhead - 1] = ent_n;
      q_base[kEscAhead - 1] = base_n;
      q_cnt[kEscAhead - 1] = cnt_n;
    }
  }

  tc_fence_before();
  __syncwarp();
  __syncthreads();
  if (warp == tc::kMma) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)P.tmem_cols);
  }
}

// ------------------------------------------------------------------ host --

int gemm_tc_rows(int M) {
  const int mp = (M + 15) / 16 * 16;
  return mp < 32 ? 32 : mp;
}

static int tc_setup(TcParams* P, int M) {
  const int MP = gemm_tc_rows(M);
  if (MP > 256) return SD_ERR_UNSUPPORTED;
  P->MP = MP;
  int ac = 32;
  while (ac < MP) ac *= 2;
  P->acc_cols = ac;
  P->tmem_cols = 2 * ac;
  P->idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(MP >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  const int XB = MP * 128;
  // stages of (activation tile, decoded tile): 3 of up to 48 KB, 4 for up to
  // 128 rows; as many 12 KB packed-weight stages as fit
  P->S = MP > 128 ? 3 : 4;
  const int bar_bytes = 512;
  const int red_bytes = 8 * MP * 4;
  const int rows_bytes = 12 * MP;
  const int con_bytes = 4 * (tc::kMaxCon + 8);
  const int budget =
      tc::kSmemMax - 1024 - bar_bytes - red_bytes - rows_bytes - con_bytes - P->S * (XB + tc::kATile);
  P->SW = std::min(8, budget / tc::kWTile);
  if (P->SW < 2) return SD_ERR_UNSUPPORTED;
  P->off_a = P->S * XB;
  P->off_w = P->off_a + P->S * tc::kATile;
  P->off_bar = P->off_w + P->SW * tc::kWTile;
  P->off_red = P->off_bar + bar_bytes;
  P->off_rows = P->off_red + red_bytes;
  P->off_con = P->off_rows + rows_bytes;
  P->smem = 1024 + P->off_con + con_bytes;
  return SD_OK;
}

size_t gemm_tc_partial_floats(int M) { return (size_t)num_sms() * 2 * gemm_tc_rows(std::min(M, 256)) * 128; }

template <bool AFF, int EPI>
static cudaError_t launch_tc(const TcParams& P, const CUtensorMap& xmap, const CUtensorMap& wmap, cudaStream_t s,
                             bool pdl, int grid) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(k_w12_gemm_tc<AFF, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemMax);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch(k_w12_gemm_tc<AFF, EPI>, dim3(grid), dim3(tc::kThreads), (size_t)P.smem, s, pdl, P, xmap, wmap);
}

// One kernel per (table kind, epilogue): no per-element dispatch, and each
// keeps only its own epilogue's registers.
template <bool AFF>
static cudaError_t launch_tc_epi(const TcParams& P, const CUtensorMap& xmap, const CUtensorMap& wmap,
                                 cudaStream_t s, bool pdl, int grid) {
  switch (P.g.e.epi) {
    case EPI_STORE: return launch_tc<AFF, EPI_STORE>(P, xmap, wmap, s, pdl, grid);
    case EPI_RESID: return launch_tc<AFF, EPI_RESID>(P, xmap, wmap, s, pdl, grid);
    case EPI_SILU: return launch_tc<AFF, EPI_SILU>(P, xmap, wmap, s, pdl, grid);
    case EPI_QKV: return launch_tc<AFF, EPI_QKV>(P, xmap, wmap, s, pdl, grid);
    default: return launch_tc<AFF, EPI_LOGITS>(P, xmap, wmap, s, pdl, grid);
  }
}

int gemm_tc_launch(const w12_tensor& W, const uint16_t* x, int rows_total, int M, const GemmEpilogue& epi,
                   const GemmWorkspace& ws, int32_t* status, cudaStream_t s, bool pdl) {
  TcParams P{};
  int rc = make_gemm_params(&P.g, W, x, M, epi, ws, status);
  if (rc) return rc;
  if ((rc = tc_setup(&P, M))) {
    set_error("gemm: no tensor-core configuration for this row count");
    return rc;
  }
  if (ws.counters_len < P.g.NB) {
    set_error("gemm: workspace counters too small");
    return SD_ERR_WORKSPACE;
  }
  const int grid = gemm_launch_grid(W, M, epi.epi);
  if (grid > tc::kMaxCon) {
    set_error("gemm: more CTAs than the tensor-core finisher lists");
    return SD_ERR_UNSUPPORTED;
  }
  if (ws.partial_floats < (size_t)grid * 2 * P.MP * 128) {
    set_error("gemm: workspace too small");
    return SD_ERR_WORKSPACE;
  }
  XMap xm;
  if ((rc = make_x_map(&xm, x, std::max(rows_total, M), W.K, P.MP))) return rc;
  CUtensorMap wmap;
  if ((rc = make_w_map(&wmap, W))) return rc;
  const cudaError_t e = W.affine ? launch_tc_epi<true>(P, xm.map, wmap, s, pdl, grid)
                                 : launch_tc_epi<false>(P, xm.map, wmap, s, pdl, grid);
  if (e != cudaSuccess) return cuda_fail(e, "k_w12_gemm_tc launch");
  return SD_OK;
}

}  // namespace sdv
