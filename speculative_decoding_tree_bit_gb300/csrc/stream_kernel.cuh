// W12 weight-streaming GEMMs for sm_103a: several GEMMs in one persistent
// launch.
//
// "SpecPilot Uses Agentic Discovery ...", "Technical Mechanisms": a verify
// step of a few tree nodes is bound by the bytes of the target weights, so
// HBM must stream weights without pause.  "SpecPilot: AI Agent Framework
// Boosts Speculative Decoding 10.87x for Qwen3.8-27B", "(1) W12": the 12-bit
// weights are decoded in registers on their way into the tensor cores, so
// they cross HBM once at 1.5 bytes each.  Launched one by one, every GEMM
// pays a ramp, a tail and a launch gap, and an RMSNorm between two GEMMs is
// a kernel of its own.  Here:
//
//  * A launch runs up to four GEMMs (phases), e.g. O (+residual), gate/up
//    (+SiLU*up), down (+residual), the next layer's q/k/v (+RoPE, KV
//    write).  Each phase's tiles (128-row block x 64-column k-tile, row-
//    block major) are split stream-K style: CTA c of the phase's G takes
//    the contiguous range [c U / G, (c + 1) U / G).  A CTA's producer walks
//    its ranges phase after phase and streams the weights into an mbarrier
//    ring ahead of the consumers, across phase boundaries: weights never
//    depend on activations.  A phase with few row blocks gets a whole
//    number of CTAs per block (G = NB floor(grid / NB)); the CTAs left over
//    go straight on to the next phase.
//  * An activation tile waits only for what it reads: the whole previous
//    phase when it feeds an RMSNorm, one row block of it when the tile is
//    that block's output (gate/up -> down).  Completion is published per
//    row block (release flag) by the CTA that finishes the block.
//  * RMSNorm is folded in: a residual epilogue writes per row block the
//    sums of squares of its bf16 outputs; the stage warp of the consuming
//    phase turns them into 1/rms per token and rewrites each staged
//    activation tile as bf16((x / rms) * gamma) before the MMAs read it.
//  * Split blocks: each contributor leaves its fp32 partial in its own
//    slot and adds its tile count to the block's ticket (acq_rel); the one
//    that completes the count sums the partials in CTA order
//    (deterministic) and runs the fused epilogue.
//  * Escaped weights decode to a fixed slot value; the stage warp adds
//    (w - slot) x from the staged tiles into a per-segment correction tile.
//  * The launch's last CTA to exit clears the counters and flags for the
//    next launch at the same site.
#pragma once

#include <cudaTypedefs.h>

#include "gemm_impl.cuh"
#include "stream.cuh"

namespace sdv {

constexpr int kSCons = 8;       // consumer warps 0..7: one 16-row strip each
constexpr int kSProd = 8;       // producer warp (lane 0)
constexpr int kSStage = 9;      // stage warp: RMSNorm of activation tiles, escape corrections
constexpr int kSThreads = 10 * 32;
constexpr int kUq = 8;           // entries of the segment queue (producer -> stage warp)

template <int NT>
constexpr int s_ctas_per_sm() { return NT <= 4 ? 2 : 1; }

// Weight decode of a launch: every phase 12-bit on the contiguous-table
// path, every phase the 8-bit view on that path, or any mix (a runtime
// choice per phase, for general tables): the common cases keep the hot
// loop small.
enum StreamDecode : int { DM_A12 = 0, DM_A8 = 1, DM_ANY = 2 };

struct StreamPhase {
  const uint32_t* words;
  const uint32_t* tile_ptr;  // escape tile index (null: no escapes)
  const uint32_t* tile_esc;
  int64_t N, K;
  int KT, NS, NB;
  int G;       // CTAs sharing the phase's tiles (the others have none)
  int64_t U;   // tiles: NB * KT, in row-block-major order
  int affine;
  int view8;  // words is the 8-bit plane
  uint32_t base2;
  uint32_t tab[4];
  float esc_slot;
  GemmEpilogue e;
  const uint16_t* gamma;  // input RMSNorm (null: none)
  float eps;
  const float* in_ss;  // sums of squares of phase dep, [nss][128]
  int nss;
  uint16_t* norm_out;
  int dep, dep_fine;
  float* out_ss;  // [NB][128] block sums, then [NB][8][128] strip sums
  float* part;    // partials of blocks split between CTAs: [G][2 (first / later segment)][128 * MP]
  int32_t* st;    // [1] blocks done, [2, 2 + NB) tickets (tiles summed), [2 + NB, 2 + 2 NB) done flags
};

struct StreamArgs {
  CUtensorMap xmap[kStreamMaxPhases];
  CUtensorMap wmap[kStreamMaxPhases];
  StreamPhase ph[kStreamMaxPhases];
  int n, M;
  int any_norm;    // some phase has an input RMSNorm (tiles go through the stage warp)
  int32_t* state;  // [0]: CTAs that exited (the site's state follows)
  int state_ints;  // ints the last CTA clears
  int32_t* status;
  uint64_t* trace;  // optional event log, [grid][kTraceEv][2] (time, tag); null: off
};

// Event log of a launch (diagnostics): per CTA kTraceEv / 2 events of the
// producer lane, then as many of consumer thread 0; each is the device
// clock and a tag = kind | phase << 8 | row block << 16 | k-tile << 40.
constexpr int kTraceEv = 64;
enum StreamTraceKind : int { TR_PROD_START = 1, TR_W_ISSUE = 2, TR_X_ISSUE = 3, TR_SEG_READY = 4, TR_SEG_DONE = 5,
                             TR_CONS_END = 6, TR_SEG_LAST = 7, TR_TICKET = 8, TR_SUMMED = 9, TR_EPI = 10 };
__device__ __forceinline__ void trace_ev(uint64_t* tr, int half, int& n, int kind, int p, int b, int t) {
  if (!tr || n >= kTraceEv / 2) return;
  uint64_t* e = tr + ((int64_t)blockIdx.x * kTraceEv + half * (kTraceEv / 2) + n) * 2;
  e[0] = globaltimer();
  e[1] = (uint64_t)kind | ((uint64_t)p << 8) | ((uint64_t)(uint32_t)b << 16) | ((uint64_t)(t & 0xFFFF) << 40);
  n++;
}

template <int NT>
struct SCfg {
  static constexpr int MP = NT * 8;
  static constexpr int XB = MP * 128;
  static constexpr int WB = kRB * kStripBytes;
  static constexpr int WB8 = kRB * 1024;  // the 8-bit plane: 16 x 64 bytes per strip
  static constexpr int RING = NT == 1 ? 8 : NT == 2 ? 7 : NT == 8 ? 9 : 5;
  static constexpr int OFF_W = RING * XB;
  static constexpr int OFF_INFO = OFF_W + RING * WB;
  static constexpr int OFF_FULL = OFF_INFO + RING * 16;
  static constexpr int OFF_XRDY = OFF_FULL + RING * 8;
  static constexpr int OFF_EMPTY = OFF_XRDY + RING * 8;
  static constexpr int OFF_CBAR = OFF_EMPTY + RING * 8;
  static constexpr int OFF_FLAG = OFF_CBAR + 24;  // [0] finisher, [1] abort, [2] last CTA
  static constexpr int OFF_RINV = OFF_FLAG + 16;
  static constexpr int OFF_RED_V = OFF_RINV + MP * 4;
  static constexpr int OFF_RED_I = OFF_RED_V + kSCons * MP * 4;
  static constexpr int OFF_SSB = OFF_RED_I + kSCons * MP * 4;  // [2][8 warps][MP] strip sums of squares
  static constexpr int OFF_PH = (OFF_SSB + 2 * kSCons * MP * 4 + 15) & ~15;
  static constexpr int OFF_UQ = (OFF_PH + kStreamMaxPhases * (int)sizeof(StreamPhase) + 15) & ~15;
  static constexpr int OFF_CORR = (OFF_UQ + kUq * 20 + 15) & ~15;
  static constexpr int END = OFF_CORR + 128 * MP * 4;
  static constexpr int SMEM = 1024 + END;
  // two CTAs per SM share 228 KB (1 KB of it reserved per CTA); one CTA
  // may take 227 KB
  static_assert(s_ctas_per_sm<NT>() == 1 ? SMEM <= 232448 : 2 * (SMEM + 1024) <= 233472, "ring too deep");
};

// Barrier of the 8 consumer warps (one arrival per warp), bounded: a warp
// whose wait gives up (abort) returns false and leaves the loop, and every
// other consumer warp's next wait then gives up at once, so no warp is left
// waiting for one that left (a named bar.sync would be).
__device__ __forceinline__ bool cons_sync(uint64_t* bar, uint32_t& ph, volatile int* abort) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  const bool ok = mbar_wait_or_abort(bar, ph, abort);
  ph ^= 1u;
  __syncwarp();
  return ok;
}

// slot info: x = phase (-1: end), y = row block, z = k-tile, w = segment
// start (bit 0) | segment end (bit 1) | whole block (bit 2) | partial slot
// (bit 3: 0 for the CTA's first block, 1 for a later one) | segment end
// tile << 16
__device__ __forceinline__ int info_tend(int w) { return (w >> 16) & 0xFFFF; }

// n / d for 0 <= n, 0 < d: one 32-bit division when both fit
__device__ __forceinline__ int64_t sdiv(int64_t n, int64_t d) {
  if ((((uint64_t)n | (uint64_t)d) >> 32) == 0) return (int64_t)((uint32_t)n / (uint32_t)d);
  return (int64_t)((uint64_t)n / (uint64_t)d);
}

// CTA c's tiles of a phase: [u0, u1) of the row-block-major tile order
// (stream-K: an even share, contiguous)
__device__ __forceinline__ void cta_range(const StreamPhase& P, int64_t c, int64_t& u0, int64_t& u1) {
  u0 = c < P.G ? sdiv(c * P.U, P.G) : P.U;
  u1 = c < P.G ? sdiv((c + 1) * P.U, P.G) : P.U;
}

__device__ __forceinline__ int ld_acquire_s32(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global_s() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// ------------------------------------------------------------ producer --
// Lane 0 of the producer warp walks the CTA's segments (its range of each
// phase cut at row-block boundaries), announces each segment in a small
// queue (so the stage warp can prefetch its escape index entries a segment
// ahead) and streams the segments' weight tiles; activation tiles are queued
// until what they read is complete.

struct UnitQ {
  int4 d[kUq];        // phase, row block, first tile, end tile
  volatile int seq[kUq];  // the CTA's segment number held in the entry
};

template <int NT>
__device__ __forceinline__ void s_produce(const StreamArgs& a, const StreamPhase* sp, uint8_t* sx, uint8_t* sw,
                                          int4* info, uint64_t* full, uint64_t* empty, UnitQ* uq,
                                          volatile int* abort) {
  using C = SCfg<NT>;
  int slot = 0, round = 0;
  int64_t uses = 0;  // slot uses, the end marker included
  bool pdl_done = false;
  bool all_ready[kStreamMaxPhases] = {};
  int q_slot[C::RING] = {}, q_p[C::RING] = {}, q_t[C::RING] = {};
  int qh = 0, qn = 0;
  bool ok = true;
  int n_tr = 0;
  trace_ev(a.trace, 0, n_tr, TR_PROD_START, 0, 0, 0);

  auto ready = [&](int p, int t) -> bool {
    const StreamPhase& P = sp[p];
    if (P.dep < 0) {
      if (!pdl_done) {
        pdl_wait();  // activations come from the previous kernel
        fence_proxy_async_global_s();
        pdl_done = true;
      }
      return true;
    }
    if (all_ready[p]) return true;
    const StreamPhase& Q = sp[P.dep];
    if (ld_acquire_s32(Q.st + 1) >= Q.NB) {
      all_ready[p] = true;
    } else if (!P.dep_fine || ld_acquire_s32(Q.st + 2 + Q.NB + t) == 0) {
      return false;
    }
    fence_proxy_async_global_s();
    return true;
  };
  auto issue_x = [&]() {
    if (a.trace && info[q_slot[qh]].w & 1) trace_ev(a.trace, 0, n_tr, TR_X_ISSUE, q_p[qh], info[q_slot[qh]].y, q_t[qh]);
    tma2d_g2s(sx + q_slot[qh] * C::XB, &a.xmap[q_p[qh]], q_t[qh] * 64, 0, &full[q_slot[qh]]);
    qh = qh + 1 == C::RING ? 0 : qh + 1;
    qn--;
  };
  auto flush = [&]() {
    while (qn > 0 && ready(q_p[qh], q_t[qh])) issue_x();
  };
  // the current slot is free for this round (its previous use consumed)
  auto wait_slot = [&]() -> bool {
    if (round == 0) return true;
    const uint32_t ea = smem_u32(&empty[slot]);
    const uint32_t par = (uint32_t)(round - 1) & 1u;
    if (mbar_try_wait(ea, par)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
      flush();
      if (mbar_try_wait(ea, par)) return true;
      if (*abort || globaltimer() - t0 > kWaitLimitNs) {
        *abort = 1;
        set_status(a.status, SD_TIMEOUT_AT(31));
        return false;
      }
    }
  };
  auto advance = [&]() {
    uses++;
    if (++slot == C::RING) {
      slot = 0;
      round++;
    }
  };
  // segments of this CTA (its range cut at block boundaries), phase after
  // phase; each is announced in the unit queue a segment ahead
  struct Seg {
    int p, b, t0, t1, slot;
  };
  int sp_p = 0;
  int64_t su = 0, su1 = 0, sfirst = -1;
  bool s_started = false;
  auto next_seg = [&](Seg& g) -> bool {
    for (;;) {
      if (sp_p >= a.n) return false;
      const StreamPhase& P = sp[sp_p];
      if (!s_started) {
        cta_range(P, blockIdx.x, su, su1);
        sfirst = su < su1 ? sdiv(su, P.KT) : -1;
        s_started = true;
      }
      if (su < su1) {
        const int b = (int)sdiv(su, P.KT);
        const int t0 = (int)(su - (int64_t)b * P.KT);
        const int64_t bend = (int64_t)(b + 1) * P.KT;
        const int64_t e = su1 < bend ? su1 : bend;
        g = Seg{sp_p, b, t0, (int)(e - (int64_t)b * P.KT), b == sfirst ? 0 : 1};
        su = e;
        return true;
      }
      sp_p++;
      s_started = false;
    }
  };
  auto publish = [&](int k, bool have, const Seg& g) {
    uq->d[k % kUq] = have ? make_int4(g.p, g.b, g.t0, g.t1) : make_int4(-1, 0, 0, 0);
    __threadfence_block();
    uq->seq[k % kUq] = k;
  };

  int k = 0;
  Seg g{}, gn{};
  bool have = next_seg(g);
  publish(0, have, g);
  while (have && ok) {
    const StreamPhase& P = sp[g.p];
    const bool v8 = P.view8 != 0;
    const bool whole = g.t0 == 0 && g.t1 == P.KT;
    bool have_n = false;
    for (int t = g.t0; t < g.t1; t++) {
      if (!wait_slot()) {
        ok = false;
        break;
      }
      info[slot] = make_int4(g.p, g.b, t, (t == g.t0 ? 1 : 0) | (t == g.t1 - 1 ? 2 : 0) | (whole ? 4 : 0) |
                                              (g.slot << 3) | (g.t1 << 16));
      if (t == g.t0) trace_ev(a.trace, 0, n_tr, TR_W_ISSUE, g.p, g.b, t);
      mbar_arrive_expect_tx(&full[slot], (v8 ? C::WB8 : C::WB) + C::XB);
      tma2d_g2s(sw + slot * C::WB, &a.wmap[g.p], t * (v8 ? 128 : 192), g.b * kRB, &full[slot]);
      const int qi = (qh + qn) % C::RING;
      q_slot[qi] = slot;
      q_p[qi] = g.p;
      q_t[qi] = t;
      qn++;
      flush();
      advance();
      if (t == g.t0) {
        have_n = next_seg(gn);
        publish(k + 1, have_n, gn);
      }
    }
    g = gn;
    have = have_n;
    k++;
  }
  // end marker (plain arrival: no bytes)
  if (ok && wait_slot()) {
    info[slot] = make_int4(-1, 0, 0, 0);
    mbar_arrive(&full[slot]);
    advance();
  }
  {
    const uint64_t t0 = globaltimer();
    while (qn > 0) {
      flush();
      if (qn > 0 && (*abort || globaltimer() - t0 > kWaitLimitNs)) {
        // give up on the dependency but complete every stage this CTA
        // started (stale, in-bounds activations), so that no copy is left
        // in flight when the CTA exits
        *abort = 1;
        set_status(a.status, SD_TIMEOUT_AT(32));
        if (!pdl_done) {
          pdl_wait();
          pdl_done = true;
        }
        while (qn > 0) issue_x();
      }
    }
  }
  if (!pdl_done) pdl_wait();
  for (int s = 0; s < C::RING && s < uses; s++) {
    const int64_t n_s = uses / C::RING + (s < uses % C::RING ? 1 : 0);
    if (!mbar_wait(&full[s], (uint32_t)((n_s - 1) & 1))) set_status(a.status, SD_TIMEOUT_AT(33));
  }
}

// ------------------------------------------------------------ RMSNorm --
// Rewrites a staged activation tile of a phase with an input RMSNorm as
// bf16((x * rinv[m]) * gamma[k]) in place (the stage warp, below, calls it
// before it releases the tile to the consumers).  cur: the phase rinv holds.

// The gamma chunks a lane applies to a tile: lane handles the 16-byte
// chunks lane + 32 i of the tile (token row m = lane / 8 + 4 i, stored
// chunk lane % 8), whose logical column chunk (the 128-byte swizzle: stored
// chunk ^ (m % 8)) is lcA for even i and lcA ^ 4 for odd i.
struct GammaPair {
  uint4 g0, g1;
};

__device__ __forceinline__ GammaPair gamma_load(const uint16_t* gamma, int t) {
  const int lane = threadIdx.x & 31;
  const int lcA = (lane & 7) ^ (lane >> 3);
  GammaPair r;
  r.g0 = __ldg(reinterpret_cast<const uint4*>(gamma + t * 64 + lcA * 8));
  r.g1 = __ldg(reinterpret_cast<const uint4*>(gamma + t * 64 + (lcA ^ 4) * 8));
  return r;
}

template <int NT>
__device__ __forceinline__ void s_norm_tile(const StreamArgs& a, const StreamPhase* sp, const int4& in, uint8_t* xs,
                                            float* rinv, int& cur, const GammaPair& gm2) {
  constexpr int MP = NT * 8;
  const int lane = threadIdx.x & 31;
  const StreamPhase& P = sp[in.x];
  if (in.x != cur) {
    // 1/rms per token row from the producing phase's per-block sums of
    // squares: lanes over the blocks, all loads in flight, then a fixed
    // butterfly (the acquire orders them after the blocks' flags)
    const StreamPhase& Q = sp[P.dep];
    if (lane == 0) (void)ld_acquire_s32(Q.st + 1);
    __syncwarp();
#pragma unroll 1
    for (int m0 = 0; m0 < MP; m0 += 16) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; j++) v[j] = 0.f;
      for (int bq = lane; bq < P.nss; bq += 32) {
#pragma unroll
        for (int j = 0; j < 16; j++) v[j] += __ldcg(P.in_ss + bq * 128 + m0 + j);
      }
#pragma unroll
      for (int j = 0; j < 16; j++) {
#pragma unroll
        for (int o = 16; o; o >>= 1) v[j] += __shfl_xor_sync(0xffffffffu, v[j], o);
      }
      if (lane < 16) {
        float mine = v[0];
#pragma unroll
        for (int j = 1; j < 16; j++) mine = lane == j ? v[j] : mine;
        rinv[m0 + lane] = 1.0f / sqrtf(mine / (float)P.K + P.eps);
      }
    }
    __syncwarp();
    cur = in.x;
  }
  const int k0 = in.z * 64;
  const bool tap = P.norm_out != nullptr && in.y == 0;
  const int pc = lane & 7, lcA = pc ^ (lane >> 3);
#pragma unroll
  for (int i = 0; i < MP / 4; i++) {
    const int m = (lane >> 3) + 4 * i, lc = (i & 1) ? lcA ^ 4 : lcA;
    uint4* p4 = reinterpret_cast<uint4*>(xs + m * 128 + pc * 16);
    const uint4 v = *p4;
    const uint4 gm = (i & 1) ? gm2.g1 : gm2.g0;
    const float r = rinv[m];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w}, gg[4] = {gm.x, gm.y, gm.z, gm.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const float lo = (bf2f(w[j] & 0xFFFF) * r) * bf2f(gg[j] & 0xFFFF);
      const float hi = (bf2f(w[j] >> 16) * r) * bf2f(gg[j] >> 16);
      o[j] = pack_bf16x2(lo, hi);
    }
    const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
    *p4 = ov;
    if (tap && m < a.M) *reinterpret_cast<uint4*>(P.norm_out + (int64_t)m * P.K + k0 + lc * 8) = ov;
  }
  fence_async_smem();  // the slot's next fill is an async-proxy copy
  __syncwarp();
}

// ---------------------------------------------------------- stage warp --
// Takes each stage first: a tile of a phase with an input RMSNorm is
// normalised in place, then the stage goes to the consumers (xrdy; when no
// phase of the launch has a norm they take the stages as they land).
// Per segment, the corrections (w - slot) x[m][k] of the escapes of its rows
// and k-tiles into corr[128 rows][MP], from the staged (normalised) tiles,
// one escape at a time with the lanes over the token rows (fixed order).
// The index entries of a segment (tile pointers of up to 32 tiles, the first
// 128 entries) are loaded when the previous segment starts, from the
// queue, so that they are in registers when the segment's tiles arrive.

struct EscMeta {
  int p = -1, b = 0, tc = 0, tend = 0;
  uint32_t tpa = 0, tpb = 0, e_lo = 0;
  uint32_t ent[4] = {0, 0, 0, 0};
};

__device__ __forceinline__ void esc_meta_load(const StreamPhase& P, int p, int b, int tc, int tend, EscMeta& m) {
  const int lane = threadIdx.x & 31;
  m.p = p;
  m.b = b;
  m.tc = tc;
  m.tend = tend;
  if (!P.tile_ptr) return;
  const uint32_t* tp = P.tile_ptr + (int64_t)b * P.KT;
  m.tpa = __ldg(tp + min(tc + lane, tend));
  m.tpb = __ldg(tp + min(tc + lane + 1, tend));
  m.e_lo = __shfl_sync(0xffffffffu, m.tpa, 0);
  const uint32_t e_hi = __shfl_sync(0xffffffffu, m.tpb, min(31, tend - 1 - tc));
#pragma unroll
  for (int j = 0; j < 4; j++) {
    const uint32_t e = m.e_lo + lane + 32 * j;
    m.ent[j] = e < e_hi ? __ldg(P.tile_esc + e) : 0u;
  }
}

template <int NT>
__device__ __forceinline__ void s_stage(const StreamArgs& a, const StreamPhase* sp, uint8_t* sx, const int4* info,
                                        uint64_t* full, uint64_t* xrdy, uint64_t* empty, float* corr,
                                        uint64_t* corr_full, uint64_t* corr_empty, const UnitQ* uq, float* rinv,
                                        volatile int* abort) {
  using C = SCfg<NT>;
  constexpr int MP = C::MP;
  const int lane = threadIdx.x & 31;
  const int mrows = min(MP, a.M);
  int slot = 0, round = 0, eseg = 0, k = -1, ncur = -1, g_p = -1, g_t = 0;
  GammaPair gpre;
  EscMeta cur, nxt;
  if (a.any_norm) pdl_wait();  // the norm's tap rewrites a buffer earlier kernels may read
  for (;;) {
    if (!mbar_wait_or_abort(&full[slot], (uint32_t)round & 1u, abort)) {
      set_status(a.status, SD_TIMEOUT_AT(35));
      break;
    }
    const int4 in = info[slot];
    if (in.x < 0) {
      if (a.any_norm && lane == 0) mbar_arrive(&xrdy[slot]);
      break;
    }
    const StreamPhase& P = sp[in.x];
    if (a.any_norm) {
      if (P.gamma) {
        // this tile's gamma (prefetched with the previous tile when that
        // was its predecessor), then the next tile's, in flight meanwhile
        const GammaPair gm = (in.x == g_p && in.z == g_t) ? gpre : gamma_load(P.gamma, in.z);
        g_p = -1;
        if (in.z + 1 < P.KT) {
          gpre = gamma_load(P.gamma, in.z + 1);
          g_p = in.x;
          g_t = in.z + 1;
        }
        s_norm_tile<NT>(a, sp, in, sx + slot * C::XB, rinv, ncur, gm);
      }
      if (lane == 0) mbar_arrive(&xrdy[slot]);
    }
    const int b = in.y, t = in.z, tend = info_tend(in.w);
    if (in.w & 1) {
      k++;
      if (!mbar_wait_or_abort(corr_empty, (uint32_t)(eseg & 1) ^ 1u, abort)) set_status(a.status, SD_TIMEOUT_AT(36));
#pragma unroll
      for (int i = 0; i < 4; i++) {
        float* row = corr + (lane + 32 * i) * MP;
#pragma unroll
        for (int m = 0; m < MP; m += 4) *reinterpret_cast<float4*>(row + m) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (nxt.p == in.x && nxt.b == b && nxt.tc == t && nxt.tend == tend) {
        cur = nxt;
      } else {
        esc_meta_load(P, in.x, b, t, tend, cur);
      }
      nxt.p = -1;
      // the next segment's entries, if it is announced already
      const int j = (k + 1) % kUq;
      if (uq->seq[j] == k + 1) {
        __threadfence_block();
        const int4 d = uq->d[j];
        if (d.x >= 0) esc_meta_load(sp[d.x], d.x, d.y, d.z, d.w, nxt);
      }
    }
    if (P.tile_ptr) {
      if (t - cur.tc >= 32) esc_meta_load(P, in.x, b, t, tend, cur);  // a segment of more than 32 tiles
      const uint32_t lo = __shfl_sync(0xffffffffu, cur.tpa, t - cur.tc);
      const uint32_t hi = __shfl_sync(0xffffffffu, cur.tpb, t - cur.tc);
      const uint8_t* xs = sx + slot * C::XB;
      for (uint32_t e = lo; e < hi; e++) {
        const uint32_t idx = e - cur.e_lo;
        uint32_t v;
        if (idx < 128) {
          const uint32_t r = idx < 32 ? cur.ent[0] : idx < 64 ? cur.ent[1] : idx < 96 ? cur.ent[2] : cur.ent[3];
          v = __shfl_sync(0xffffffffu, r, idx & 31);
        } else {
          v = __ldg(P.tile_esc + e);
        }
        const int row = (v >> 6) & 127, kk = v & 63;
        const float w = bf2f((v >> 16) & (P.view8 ? 0xFFF0u : 0xFFFFu));
        float* cr = corr + row * MP;
        for (int m = lane; m < mrows; m += 32) {
          const float xv =
              bf2f(*reinterpret_cast<const uint16_t*>(xs + m * 128 + (((kk >> 3) ^ (m & 7)) << 4) + (kk & 7) * 2));
          const float acc = fmaf(w, xv, cr[m]);
          cr[m] = fmaf(-P.esc_slot, xv, acc);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (in.w & 2) {
      __syncwarp();
      if (lane == 0) mbar_arrive(corr_full);
      eseg++;
    }
    if (++slot == C::RING) {
      slot = 0;
      round++;
    }
  }
}

// ----------------------------------------------------------- epilogue --
// Fused epilogue of one finished row block (strip = this warp's 16 rows).
// EPI_RESID also leaves in rs[nt][cc] the thread's share of the sum of
// squares of its bf16 outputs (rows g and g + 8, token column nt*8+2q+cc).

template <int NT>
__device__ __forceinline__ void s_epilogue(const StreamPhase& P, int M, int strip, int lane, float (&acc)[NT][4],
                                           float (&bestv)[NT][2], int (&besti)[NT][2], float (&rs)[NT][2]) {
  const int g = lane >> 2, q = lane & 3;
  const int64_t n_lo = (int64_t)strip * 16 + g;
  const GemmEpilogue& E = P.e;
#pragma unroll
  for (int nt = 0; nt < NT; nt++) rs[nt][0] = rs[nt][1] = 0.f;
  if (E.epi == EPI_RESID) {
    float r[NT][2][2];
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int cc = 0; cc < 2; cc++) {
        const int m = nt * 8 + 2 * q + cc;
        const int64_t i0 = (int64_t)m * E.ldo + n_lo;
        const bool ok = m < M;
        r[nt][cc][0] = ok ? bf2f(__ldcg(E.resid + i0)) : 0.f;
        r[nt][cc][1] = ok ? bf2f(__ldcg(E.resid + i0 + 8)) : 0.f;
      }
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int cc = 0; cc < 2; cc++) {
        const int m = nt * 8 + 2 * q + cc;
        if (m >= M) continue;
        const int64_t i0 = (int64_t)m * E.ldo + n_lo;
        const uint16_t o1 = f2bf(r[nt][cc][0] + rbf(acc[nt][cc]));
        const uint16_t o2 = f2bf(r[nt][cc][1] + rbf(acc[nt][2 + cc]));
        E.out[i0] = o1;
        E.out[i0 + 8] = o2;
        const float f1 = bf2f(o1), f2 = bf2f(o2);
        rs[nt][cc] = fmaf(f2, f2, f1 * f1);
      }
    return;
  }
  if (E.epi == EPI_QKV) {
    const int64_t qrows = (int64_t)E.hq * 128, krows = (int64_t)E.hkv * 128;
    const int64_t row0 = (int64_t)strip * 16;
    const bool rope = row0 < qrows + krows;
    const bool is_q = row0 < qrows;
    const int64_t rr = rope ? (is_q ? row0 : row0 - qrows) : row0 - qrows - krows;
    const int head = (int)(rr / 128);
    const int d = rope ? (int)((rr % 128) / 16) * 8 + g : (int)(rr % 128) + g;
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
      int pos[2], rq[2], slot[2];
#pragma unroll
      for (int cc = 0; cc < 2; cc++) {
        const int m = nt * 8 + 2 * q + cc;
        const bool ok = m < M;
        pos[cc] = ok && rope ? E.rows.pos[m] : 0;
        rq[cc] = ok && !is_q ? E.rows.req[m] : 0;
        slot[cc] = ok && !is_q ? E.rows.slot[m] : 0;
      }
      float cs[2], sn[2];
      int okr[2], page[2];
#pragma unroll
      for (int cc = 0; cc < 2; cc++) {
        cs[cc] = rope ? E.rope_cos[(int64_t)pos[cc] * 64 + d] : 1.f;
        sn[cc] = rope ? E.rope_sin[(int64_t)pos[cc] * 64 + d] : 0.f;
        okr[cc] = is_q ? 1 : E.rows.req_ok[rq[cc]];
        page[cc] = is_q ? 0 : E.cache.page_table[(int64_t)rq[cc] * E.cache.max_pages + slot[cc] / E.cache.page_size];
      }
#pragma unroll
      for (int cc = 0; cc < 2; cc++) {
        const int m = nt * 8 + 2 * q + cc;
        if (m >= M || !okr[cc]) continue;
        const float v_lo = acc[nt][cc], v_hi = acc[nt][2 + cc];
        if (rope) {
          const float x1 = rbf(v_lo), x2 = rbf(v_hi);
          const uint16_t o1 = f2bf(x1 * cs[cc] - x2 * sn[cc]), o2 = f2bf(x2 * cs[cc] + x1 * sn[cc]);
          uint16_t* dst = is_q ? E.q_out + ((int64_t)m * E.hq + head) * 128
                               : E.cache.k + (((int64_t)page[cc] * E.cache.hkv + head) * E.cache.page_size +
                                              slot[cc] % E.cache.page_size) * 128;
          dst[d] = o1;
          dst[d + 64] = o2;
        } else {
          uint16_t* dst = E.cache.v + (((int64_t)page[cc] * E.cache.hkv + head) * E.cache.page_size +
                                       slot[cc] % E.cache.page_size) * 128;
          dst[d] = f2bf(v_lo);
          dst[d + 8] = f2bf(v_hi);
        }
      }
    }
    return;
  }
#pragma unroll
  for (int nt = 0; nt < NT; nt++)
#pragma unroll
    for (int cc = 0; cc < 2; cc++) {
      const int m = nt * 8 + 2 * q + cc;
      if (m >= M) continue;
      const float v_lo = acc[nt][cc], v_hi = acc[nt][2 + cc];
      switch (E.epi) {
        case EPI_STORE:
          E.out[(int64_t)m * E.ldo + n_lo] = f2bf(v_lo);
          E.out[(int64_t)m * E.ldo + n_lo + 8] = f2bf(v_hi);
          break;
        case EPI_SILU: {
          const float gt = rbf(v_lo), up = rbf(v_hi);
          const float s = gt / (1.0f + expf(-gt));
          E.out[(int64_t)m * E.ldo + (int64_t)strip * 8 + g] = f2bf(s * up);
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

// ---------------------------------------------------------- consumers --
// The consumer warps of a CTA work on one segment at a time, each on one
// 16-row strip.  A segment that is a whole row block runs its epilogue at
// once; one that is part of a split block stores its fp32 partial in the
// CTA's slot and thread 0 adds the segment's tile count to the block's
// ticket (acq_rel, after a consumer barrier): the CTA that completes the
// count sums the contributors' partials in CTA order (deterministic) and
// runs the epilogue.  A finished block's per-token sums of squares (residual
// epilogues, strips added in order) and its done flag are published by one
// thread after a consumer barrier.

// the block's sums of squares from the warps' strip sums (ssb), then its
// flag and the phase's done count (release)
template <int NT>
__device__ __forceinline__ bool s_block_done(const StreamPhase& P, int b, int warp, int lane, float (&rs)[NT][2],
                                             float* ssb, uint64_t* cbar, uint32_t& cph, volatile int* abort) {
  constexpr int MP = NT * 8;
  if (P.out_ss) {
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int cc = 0; cc < 2; cc++) {
        float v = rs[nt][cc];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        if (lane < 4) ssb[warp * MP + nt * 8 + 2 * lane + cc] = v;
      }
  }
  if (!cons_sync(cbar, cph, abort)) return false;
  if (warp == 0) {
    if (P.out_ss) {
      for (int m = lane; m < MP; m += 32) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kSCons; w++) v += ssb[w * MP + m];
        __stcg(P.out_ss + (int64_t)b * 128 + m, v);
      }
    }
    __syncwarp();
    if (lane == 0) {
      asm volatile("st.release.gpu.global.s32 [%0], 1;" ::"l"(P.st + 2 + P.NB + b) : "memory");
      asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(P.st + 1) : "memory");
    }
  }
  return true;
}

template <int NT, int DM>
__device__ __forceinline__ void s_consume(const StreamArgs& a, const uint8_t* sx, const uint8_t* sw, const int4* info,
                                          uint64_t* full, uint64_t* xrdy, uint64_t* empty, const float* corr,
                                          uint64_t* corr_full, uint64_t* corr_empty, const StreamPhase* sp,
                                          float* red_v, int* red_i, float* ssb, int* fin_flag, uint64_t* cbar,
                                          volatile int* abort) {
  using C = SCfg<NT>;
  constexpr int MP = C::MP;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
  uint32_t cph = 0;  // phase of the consumer-group barrier
  constexpr bool kDual = NT <= 4;
  float acc[NT][4], acc2[kDual ? NT : 1][4];
  float bestv[NT][2];
  int besti[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; nt++)
#pragma unroll
    for (int c = 0; c < 2; c++) {
      bestv[nt][c] = -INFINITY;
      besti[nt][c] = 0x7FFFFFFF;
    }
  auto zero = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int c = 0; c < 4; c++) {
        acc[nt][c] = 0.f;
        if constexpr (kDual) acc2[nt][c] = 0.f;
      }
  };
  // this warp's share of a CTA's partial slot: [CTA][slot][warp][NT][lane][4]
  auto part_ptr = [&](const StreamPhase& P, int64_t cta, int sl) {
    return P.part + (((cta * 2 + sl) * kSCons + warp) * NT) * 128 + lane * 4;
  };
  int nfin = 0;  // blocks this CTA finished (double-buffers ssb)
  pdl_wait();  // residuals and cache positions come from earlier kernels
  uint64_t* rdy = a.any_norm ? xrdy : full;  // tiles pass the stage warp first only when some phase needs it
  int slot = 0, round = 0, cseg = 0, seg_t0 = 0, n_tr = 0;
  bool fresh = true;  // acc holds nothing of the current segment yet
  zero();
  for (;;) {
    if (!mbar_wait_or_abort(&rdy[slot], (uint32_t)round & 1u, abort)) {
      set_status(a.status, SD_TIMEOUT_AT(37));
      break;
    }
    const int4 in = info[slot];
    if (in.x < 0) break;
    const StreamPhase& P = sp[in.x];
    const int b = in.y;
    if (in.w & 1) {
      if (!fresh) zero();
      seg_t0 = in.z;
      if (tid == 0) trace_ev(a.trace, 1, n_tr, TR_SEG_READY, in.x, b, in.z);
    }
    fresh = false;
    const int strip = b * kRB + warp;
    if (strip < P.NS) {
      const bool v8 = DM == DM_A8 || (DM == DM_ANY && P.view8 != 0);
      const uint8_t* wsm = sw + slot * C::WB + warp * (v8 ? 1024 : kStripBytes);
      const uint4 W0 = *reinterpret_cast<const uint4*>(wsm + lane * 16);
      const uint4 W1 = *reinterpret_cast<const uint4*>(wsm + 512 + lane * 16);
      uint4 W2 = W1;
      if (!v8) W2 = *reinterpret_cast<const uint4*>(wsm + 1024 + lane * 16);
      const uint32_t xb = smem_u32(sx + slot * C::XB);
      const uint32_t base2 = P.base2;
#pragma unroll
      for (int j = 0; j < 4; j++) {
        uint32_t a0, a1, a2, a3;
        if constexpr (DM == DM_A12) {
          decode<true>(comp(W0, j), comp(W1, j), comp(W2, j), base2, P.tab, a0, a1, a2, a3);
        } else if constexpr (DM == DM_A8) {
          decode_view8(comp(W0, j), comp(W1, j), true, base2, P.tab, a0, a1, a2, a3);
        } else {
          const bool aff = P.affine != 0;
          if (v8)
            decode_view8(comp(W0, j), comp(W1, j), aff, base2, P.tab, a0, a1, a2, a3);
          else if (aff)
            decode<true>(comp(W0, j), comp(W1, j), comp(W2, j), base2, P.tab, a0, a1, a2, a3);
          else
            decode<false>(comp(W0, j), comp(W1, j), comp(W2, j), base2, P.tab, a0, a1, a2, a3);
        }
        const int kchunk = 2 * j + ((lane >> 3) & 1);
        float(*A)[4] = (kDual && (j & 1)) ? acc2 : acc;
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
    if (++slot == C::RING) {
      slot = 0;
      round++;
    }
    if (!(in.w & 2)) continue;

    // --------------------------------------------- segment finished --
    if (tid == 0) trace_ev(a.trace, 1, n_tr, TR_SEG_LAST, in.x, b, 0);
    if constexpr (kDual) {
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int c = 0; c < 4; c++) acc[nt][c] += acc2[nt][c];
    }
    if (!mbar_wait_or_abort(corr_full, (uint32_t)(cseg & 1), abort)) set_status(a.status, SD_TIMEOUT_AT(38));
    {
      const float* c0 = corr + (warp * 16 + g) * MP;
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int cc = 0; cc < 2; cc++) {
          acc[nt][cc] += c0[nt * 8 + 2 * q + cc];
          acc[nt][2 + cc] += c0[8 * MP + nt * 8 + 2 * q + cc];
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(corr_empty);
    cseg++;
    if (!(in.w & 4)) {
      // part of a split block: the partial, then the block's ticket
      float* mine = part_ptr(P, blockIdx.x, (in.w >> 3) & 1);
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
        __stcg(reinterpret_cast<float4*>(mine + nt * 128),
               make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]));
      // the barrier orders every warp's partial before thread 0's acq_rel
      // ticket, and the ticket before the others read the verdict
      if (!cons_sync(cbar, cph, abort)) break;
      if (tid == 0) {
        const int add = info_tend(in.w) - seg_t0;
        const int old = atomic_add_acq_rel(P.st + 2 + b, add);
        fin_flag[0] = old + add == P.KT ? 1 : 0;
      }
      if (!cons_sync(cbar, cph, abort)) break;
      if (tid == 0) trace_ev(a.trace, 1, n_tr, TR_TICKET, in.x, b, 0);
      if (!fin_flag[0]) {
        if (tid == 0) trace_ev(a.trace, 1, n_tr, TR_SEG_DONE, in.x, b, 0);
        zero();
        fresh = true;
        continue;
      }
      // the last contributor: the contributors' partials in CTA order
      zero();
      const int64_t c_first = sdiv(((int64_t)b * P.KT + 1) * P.G - 1, P.U);
      const int64_t c_last = sdiv((int64_t)(b + 1) * P.KT * P.G - 1, P.U);
      constexpr int kBatch = NT <= 1 ? 8 : NT <= 2 ? 4 : 2;
      for (int64_t c0 = c_first; c0 <= c_last; c0 += kBatch) {
        float4 v[kBatch][NT];
        bool use[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; u++) {
          const int64_t c = c0 + u;
          int64_t cs = 0, ce = 0;
          if (c <= c_last) cta_range(P, c, cs, ce);
          use[u] = c <= c_last && cs != ce;  // an empty range wrote no partial
          // slot 1 when the contributor's range began in an earlier block
          const float* src = part_ptr(P, use[u] ? c : blockIdx.x, (use[u] && cs < (int64_t)b * P.KT) ? 1 : 0);
#pragma unroll
          for (int nt = 0; nt < NT; nt++)
            v[u][nt] = use[u] ? __ldcg(reinterpret_cast<const float4*>(src + nt * 128)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kBatch; u++)
#pragma unroll
          for (int nt = 0; nt < NT; nt++) {
            acc[nt][0] += v[u][nt].x;
            acc[nt][1] += v[u][nt].y;
            acc[nt][2] += v[u][nt].z;
            acc[nt][3] += v[u][nt].w;
          }
      }
    }
    {
      if (tid == 0) trace_ev(a.trace, 1, n_tr, TR_SUMMED, in.x, b, 0);
      float rs[NT][2];
      const int strip = b * kRB + warp;
      if (strip < P.NS) {
        s_epilogue<NT>(P, a.M, strip, lane, acc, bestv, besti, rs);
      } else {
#pragma unroll
        for (int nt = 0; nt < NT; nt++) rs[nt][0] = rs[nt][1] = 0.f;
      }
      if (tid == 0) trace_ev(a.trace, 1, n_tr, TR_EPI, in.x, b, 0);
      if (!s_block_done<NT>(P, b, warp, lane, rs, ssb + (nfin & 1) * kSCons * MP, cbar, cph, abort)) break;
      nfin++;
      if (tid == 0) trace_ev(a.trace, 1, n_tr, TR_SEG_DONE, in.x, b, 1);
    }
    zero();
    fresh = true;
  }

  if (tid == 0) trace_ev(a.trace, 1, n_tr, TR_CONS_END, 0, 0, 0);
  // per-CTA argmax partial of a logits phase (every CTA writes one)
  bool logits = false;
  const GemmEpilogue* le = nullptr;
  for (int p = 0; p < a.n; p++)
    if (sp[p].e.epi == EPI_LOGITS) {
      logits = true;
      le = &sp[p].e;
    }
  if (logits) {
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int c = 0; c < 2; c++) {
        float v = bestv[nt][c];
        int i = besti[nt][c];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, v, off);
          const int oi = __shfl_xor_sync(0xffffffffu, i, off);
          if (ov > v || (ov == v && oi < i)) {
            v = ov;
            i = oi;
          }
        }
        if (lane < 4) {
          red_v[warp * MP + nt * 8 + 2 * lane + c] = v;
          red_i[warp * MP + nt * 8 + 2 * lane + c] = i;
        }
      }
    if (!cons_sync(cbar, cph, abort)) return;
    if (tid < MP) {
      float v = -INFINITY;
      int i = 0x7FFFFFFF;
      for (int w = 0; w < kSCons; w++) {
        const float ov = red_v[w * MP + tid];
        const int oi = red_i[w * MP + tid];
        if (ov > v || (ov == v && oi < i)) {
          v = ov;
          i = oi;
        }
      }
      if (tid < a.M) {
        le->amax_val[(int64_t)blockIdx.x * le->ld_amax + tid] = v;
        le->amax_idx[(int64_t)blockIdx.x * le->ld_amax + tid] = i;
      }
    }
  }
}

// --------------------------------------------------------------- kernel --

template <int NT, int DM>
__global__ void __launch_bounds__(kSThreads, s_ctas_per_sm<NT>()) k_w12_stream(const __grid_constant__ StreamArgs a) {
  using C = SCfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sx = smem;
  uint8_t* sw = smem + C::OFF_W;
  int4* info = reinterpret_cast<int4*>(smem + C::OFF_INFO);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_FULL);
  uint64_t* xrdy = reinterpret_cast<uint64_t*>(smem + C::OFF_XRDY);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + C::OFF_EMPTY);
  uint64_t* corr_full = reinterpret_cast<uint64_t*>(smem + C::OFF_CBAR);
  uint64_t* corr_empty = corr_full + 1;
  uint64_t* cbar = corr_full + 2;
  int* flag = reinterpret_cast<int*>(smem + C::OFF_FLAG);
  volatile int* abort = flag + 1;
  float* rinv = reinterpret_cast<float*>(smem + C::OFF_RINV);
  float* red_v = reinterpret_cast<float*>(smem + C::OFF_RED_V);
  int* red_i = reinterpret_cast<int*>(smem + C::OFF_RED_I);
  float* ssb = reinterpret_cast<float*>(smem + C::OFF_SSB);
  StreamPhase* sp = reinterpret_cast<StreamPhase*>(smem + C::OFF_PH);
  UnitQ* uq = reinterpret_cast<UnitQ*>(smem + C::OFF_UQ);
  float* corr = reinterpret_cast<float*>(smem + C::OFF_CORR);

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::RING; i++) {
      mbar_init(&full[i], 1);
      mbar_init(&xrdy[i], 1);
      mbar_init(&empty[i], kSCons + 1);  // consumer warps + stage warp
    }
    mbar_init(corr_full, 1);
    mbar_init(corr_empty, kSCons);
    mbar_init(cbar, kSCons);
    flag[0] = 0;
    flag[1] = 0;
    flag[2] = 0;
    for (int i = 0; i < kUq; i++) uq->seq[i] = -1;
    fence_mbar_init();
  }
  // the phases' descriptors in shared memory: every role reads them with
  // plain shared loads (runtime-indexed parameter reads are slow loads)
  {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(a.ph);
    uint32_t* dst = reinterpret_cast<uint32_t*>(sp);
    for (int i = threadIdx.x; i < a.n * (int)(sizeof(StreamPhase) / 4); i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  pdl_launch();

  if (warp == kSProd) {
    if ((threadIdx.x & 31) == 0) s_produce<NT>(a, sp, sx, sw, info, full, empty, uq, abort);
  } else if (warp == kSStage) {
    s_stage<NT>(a, sp, sx, info, full, xrdy, empty, corr, corr_full, corr_empty, uq, rinv, abort);
  } else {
    s_consume<NT, DM>(a, sx, sw, info, full, xrdy, empty, corr, corr_full, corr_empty, sp, red_v, red_i, ssb, flag, cbar,
                      abort);
  }
  __syncthreads();
  // the last CTA to get here clears the site's counters, tickets and flags
  if (threadIdx.x == 0) {
    __threadfence();
    flag[2] = atomicAdd(a.state, 1) == (int)gridDim.x - 1 ? 1 : 0;
  }
  __syncthreads();
  if (flag[2]) {
    __threadfence();
    for (int i = 1 + threadIdx.x; i < a.state_ints; i += blockDim.x) a.state[i] = 0;
    __syncthreads();
    if (threadIdx.x == 0) a.state[0] = 0;
  }
}

// cudaSuccess when the kernel fits the CTAs per SM its grid assumes
// (cudaErrorInvalidConfiguration otherwise); sets the shared-memory carveout.
cudaError_t stream_check_residency(const void* kern, int NT);

// Launch of the streamed kernel for one decode mode (a translation unit per
// mode, compiled in parallel).
template <int DM>
cudaError_t stream_launch_dm(const StreamArgs& a, int NT, int grid, cudaStream_t s, bool pdl);

}  // namespace sdv
