// W12 weight-streaming GEMMs for sm_103a: several GEMMs in one persistent
// launch, scheduled unit by unit.
//
// "SpecPilot Uses Agentic Discovery ...", "Technical Mechanisms": a verify
// step of a few tree nodes is bound by the bytes of the target weights, so
// HBM must stream weights without pause.  "SpecPilot: AI Agent Framework
// Boosts Speculative Decoding 10.87x for Qwen3.8-27B", "(1) W12": the 12-bit
// weights are decoded in registers on their way into the tensor cores, so
// they cross HBM once at 1.5 bytes each.  Launched one by one, every GEMM
// pays a ramp, a tail of straggling CTAs and split-K finishers, and a launch
// gap, and an RMSNorm between two GEMMs is a kernel of its own.  Here:
//
//  * A launch runs up to four GEMMs (phases), e.g. O (+residual), gate/up
//    (+SiLU*up), down (+residual), the next layer's q/k/v (+RoPE, KV
//    write).  Work of a phase = units of one 128-row block x a range of
//    64-column k-tiles; most blocks are one unit, the last split_blocks
//    blocks are split into k-chunks so that the end of a phase is made of
//    small units.  Each CTA's producer takes the next unit from the phase's
//    counter (dynamic: no CTA waits for a slow one) and streams its weights
//    into an mbarrier ring ahead of the consumers, across phase boundaries:
//    weights never depend on activations.
//  * An activation tile waits only for what it reads: the whole previous
//    phase when it feeds an RMSNorm, one row block of it when the tile is
//    that block's output (gate/up -> down).  Completion is published per
//    row block (release flags) by the CTA that finishes the block.
//  * RMSNorm is folded in: a residual epilogue writes per row block the
//    sums of squares of its bf16 outputs; a norm warp of the consuming
//    phase turns them into 1/rms per token and rewrites each staged
//    activation tile as bf16((x / rms) * gamma) before the MMAs read it.
//  * Split blocks: each k-chunk's fp32 partial goes to its own slot; the
//    last chunk to finish (acq_rel ticket) sums the slots in chunk order
//    (deterministic) and runs the fused epilogue.
//  * Escaped weights decode to a fixed slot value; an escape warp adds
//    (w - slot) x from the staged tiles into a per-unit correction tile.
//  * The launch's last CTA to exit clears the counters and flags for the
//    next launch at the same site.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "gemm_impl.cuh"
#include "stream.cuh"

namespace sdv {

constexpr int kSCons = 8;       // consumer warps 0..7: one 16-row strip each
constexpr int kSProd = 8;       // producer warp (lane 0)
constexpr int kSEsc = 9;        // escape-correction warp
constexpr int kSNorm = 10;      // activation-tile warp (RMSNorm rewrite)
constexpr int kSThreads = 11 * 32;
constexpr int kSChunkTiles = 8;  // k-tiles per chunk of a split block (target)
constexpr int kUq = 8;           // entries of the unit queue (producer -> escape warp)

template <int NT>
constexpr int s_ctas_per_sm() { return NT <= 4 ? 2 : 1; }

struct StreamPhase {
  const uint32_t* words;
  const uint32_t* tile_ptr;  // escape tile index (null: no escapes)
  const uint32_t* tile_esc;
  int64_t N, K;
  int KT, NS, NB;
  int S, KC;     // chunks of a split block, k-tiles per chunk
  int nb_whole;  // blocks [0, nb_whole) are one unit each
  int U;         // units
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
  float* part;    // split partials [(NB - nb_whole) * S][128 * MP]
  int32_t* st;    // [0] next unit, [1] blocks done, [2, 2 + 8 NB) strip tickets, then NB block counters, NB done flags
};

struct StreamArgs {
  CUtensorMap xmap[kStreamMaxPhases];
  CUtensorMap wmap[kStreamMaxPhases];
  StreamPhase ph[kStreamMaxPhases];
  int n, M;
  int32_t* state;  // [0]: CTAs that exited (the site's state follows)
  int state_ints;  // ints the last CTA clears
  int32_t* status;
};

template <int NT>
struct SCfg {
  static constexpr int MP = NT * 8;
  static constexpr int XB = MP * 128;
  static constexpr int WB = kRB * kStripBytes;
  static constexpr int WB8 = kRB * 1024;  // the 8-bit plane: 16 x 64 bytes per strip
  static constexpr int RING = NT == 1 ? 7 : NT == 2 ? 6 : NT == 4 ? 5 : NT == 8 ? 8 : 5;
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
  static constexpr int OFF_PH = (OFF_RED_I + kSCons * MP * 4 + 15) & ~15;
  static constexpr int OFF_UQ = (OFF_PH + (int)sizeof(StreamPhase) + 15) & ~15;
  static constexpr int OFF_CORR = (OFF_UQ + kUq * 20 + 15) & ~15;
  static constexpr int END = OFF_CORR + 128 * MP * 4;
  static constexpr int SMEM = 1024 + END;
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

// slot info: x = phase (-1: end), y = row block, z = k-tile,
// w = first (bit 0) | last (bit 1) | (chunk + 1) << 8 (0: whole block) | unit end tile << 16
__device__ __forceinline__ int info_chunk(int w) { return ((w >> 8) & 0xFF) - 1; }
__device__ __forceinline__ int info_tend(int w) { return (w >> 16) & 0xFFFF; }

__device__ __forceinline__ void unit_of(const StreamPhase& P, int u, int& b, int& c, int& t0, int& t1) {
  if (u < P.nb_whole) {
    b = u;
    c = -1;
    t0 = 0;
    t1 = P.KT;
  } else {
    const int v = u - P.nb_whole;
    b = P.nb_whole + v / P.S;
    c = v % P.S;
    t0 = c * P.KC;
    t1 = min(P.KT, t0 + P.KC);
  }
}

// Two bytes of the 8-bit plane (bits 0..7 and 16..23: sign << 7 | code << 3
// | top mantissa bits) -> their bf16 view, as a bf16x2 fragment register.
__device__ __forceinline__ uint32_t view8_pair(uint32_t v, bool aff, uint32_t base2, const uint32_t* tab) {
  if (aff) return (((v & 0x007F007Fu) << 4) + base2) | ((v & 0x00800080u) << 8);
  const uint32_t e0 = lut_exp((v >> 3) & 15, tab), e1 = lut_exp((v >> 19) & 15, tab);
  return ((v & 0x00070007u) << 4) | (e0 << 7) | (e1 << 23) | ((v & 0x00800080u) << 8);
}

// A fragment of one sub-tile from its two plane words: p0 holds (row g,
// k), (g, k + 1), (g + 8, k), (g + 8, k + 1), p1 the same at k + 8.
__device__ __forceinline__ void decode_view8(uint32_t p0, uint32_t p1, bool aff, uint32_t base2, const uint32_t* tab,
                                             uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
  a0 = view8_pair(__byte_perm(p0, 0, 0x4140), aff, base2, tab);
  a1 = view8_pair(__byte_perm(p0, 0, 0x4342), aff, base2, tab);
  a2 = view8_pair(__byte_perm(p1, 0, 0x4140), aff, base2, tab);
  a3 = view8_pair(__byte_perm(p1, 0, 0x4342), aff, base2, tab);
}

__device__ __forceinline__ int ld_acquire_s32(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global_s() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// ------------------------------------------------------------ producer --
// Lane 0 of the producer warp takes units (moving on through the phases),
// announces each unit in a small queue (so the escape warp can prefetch its
// escape index entries a unit ahead) and streams the units' weight tiles;
// activation tiles are queued until what they read is complete.

struct UnitQ {
  int4 d[kUq];        // phase, row block, first tile, end tile
  volatile int seq[kUq];  // the CTA's unit number held in the entry
};

template <int NT>
__device__ __forceinline__ void s_produce(const StreamArgs& a, uint8_t* sx, uint8_t* sw, int4* info, uint64_t* full,
                                          uint64_t* empty, UnitQ* uq, volatile int* abort) {
  using C = SCfg<NT>;
  int slot = 0, round = 0;
  int64_t uses = 0;  // slot uses, the end marker included
  bool pdl_done = false;
  bool all_ready[kStreamMaxPhases] = {};
  int q_slot[C::RING] = {}, q_p[C::RING] = {}, q_t[C::RING] = {};
  int qh = 0, qn = 0;
  bool ok = true;

  auto ready = [&](int p, int t) -> bool {
    const StreamPhase& P = a.ph[p];
    if (P.dep < 0) {
      if (!pdl_done) {
        pdl_wait();  // activations come from the previous kernel
        fence_proxy_async_global_s();
        pdl_done = true;
      }
      return true;
    }
    if (all_ready[p]) return true;
    const StreamPhase& Q = a.ph[P.dep];
    if (ld_acquire_s32(Q.st + 1) >= Q.NB) {
      all_ready[p] = true;
    } else if (!P.dep_fine || ld_acquire_s32(Q.st + 2 + 9 * Q.NB + t) == 0) {
      return false;
    }
    fence_proxy_async_global_s();
    return true;
  };
  auto issue_x = [&]() {
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
  // the next unit, moving on to the next phase when one runs out
  auto grab = [&](int& p, int& u) -> bool {
    while (p < a.n) {
      u = atomicAdd(a.ph[p].st, 1);
      if (u < a.ph[p].U) return true;
      p++;
    }
    return false;
  };
  auto publish = [&](int k, bool have, int p, int u) {
    int4 d = make_int4(-1, 0, 0, 0);
    if (have) {
      int b, c, t0, t1;
      unit_of(a.ph[p], u, b, c, t0, t1);
      d = make_int4(p, b, t0, t1);
    }
    uq->d[k % kUq] = d;
    __threadfence_block();
    uq->seq[k % kUq] = k;
  };

  int p = 0, u = 0, k = 0;
  bool have = grab(p, u);
  publish(0, have, p, u);
  while (have && ok) {
    const StreamPhase& P = a.ph[p];
    int b, c, t0, t1;
    unit_of(P, u, b, c, t0, t1);
    int pn = p, un = 0;
    bool have_n = false;
    for (int t = t0; t < t1; t++) {
      if (!wait_slot()) {
        ok = false;
        break;
      }
      info[slot] = make_int4(p, b, t, (t == t0 ? 1 : 0) | (t == t1 - 1 ? 2 : 0) | ((c + 1) << 8) | (t1 << 16));
      mbar_arrive_expect_tx(&full[slot], (P.view8 ? C::WB8 : C::WB) + C::XB);
      tma2d_g2s(sw + slot * C::WB, &a.wmap[p], t * (P.view8 ? 128 : 192), b * kRB, &full[slot]);
      const int qi = (qh + qn) % C::RING;
      q_slot[qi] = slot;
      q_p[qi] = p;
      q_t[qi] = t;
      qn++;
      flush();
      advance();
      if (t == t0) {
        // the next unit, announced while this one streams
        have_n = grab(pn, un);
        publish(k + 1, have_n, pn, un);
      }
    }
    p = pn;
    u = un;
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

// ---------------------------------------------------------- norm warp --
// Turns each staged activation tile of a phase with an input RMSNorm into
// bf16((x * rinv[m]) * gamma[k]) in place; forwards every stage (xready).

template <int NT>
__device__ __forceinline__ void s_norm(const StreamArgs& a, uint8_t* sx, const int4* info, uint64_t* full,
                                       uint64_t* xrdy, float* rinv, volatile int* abort) {
  using C = SCfg<NT>;
  constexpr int MP = C::MP;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  int slot = 0, round = 0, cur = -1;
  for (;;) {
    if (!mbar_wait_or_abort(&full[slot], (uint32_t)round & 1u, abort)) {
      set_status(a.status, SD_TIMEOUT_AT(34));
      break;
    }
    const int4 in = info[slot];
    if (in.x < 0) {
      if (lane == 0) mbar_arrive(&xrdy[slot]);
      break;
    }
    const StreamPhase& P = a.ph[in.x];
    if (P.gamma) {
      if (in.x != cur) {
        // 1/rms per token row from the producing phase's per-block sums of
        // squares: lanes over the blocks, all loads in flight, then a fixed
        // butterfly (the acquire orders them after the blocks' flags)
        const StreamPhase& Q = a.ph[P.dep];
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
      }
      uint8_t* xs = sx + slot * C::XB;
      const int k0 = in.z * 64;
      const bool tap = P.norm_out != nullptr && in.y == 0;
      for (int ch = lane; ch < MP * 8; ch += 32) {
        const int m = ch >> 3, pc = ch & 7, lc = pc ^ (m & 7);
        uint4* p4 = reinterpret_cast<uint4*>(xs + m * 128 + pc * 16);
        const uint4 v = *p4;
        const uint4 gm = __ldg(reinterpret_cast<const uint4*>(P.gamma + k0 + lc * 8));
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
    }
    cur = in.x;
    __syncwarp();
    if (lane == 0) mbar_arrive(&xrdy[slot]);
    if (++slot == C::RING) {
      slot = 0;
      round++;
    }
  }
}

// -------------------------------------------------------- escape warp --
// Per unit, the corrections (w - slot) x[m][k] of the escapes of its rows
// and k-tiles into corr[128 rows][MP], from the staged (normalised) tiles,
// one escape at a time with the lanes over the token rows (fixed order).
// The index entries of a unit (tile pointers of up to 32 tiles, the first
// 128 entries) are loaded when the previous unit starts, from the unit
// queue, so that they are in registers when the unit's tiles arrive.

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
__device__ __forceinline__ void s_escape(const StreamArgs& a, const uint8_t* sx, const int4* info, uint64_t* xrdy,
                                         uint64_t* empty, float* corr, uint64_t* corr_full, uint64_t* corr_empty,
                                         const UnitQ* uq, volatile int* abort) {
  using C = SCfg<NT>;
  constexpr int MP = C::MP;
  const int lane = threadIdx.x & 31;
  const int mrows = min(MP, a.M);
  int slot = 0, round = 0, eseg = 0, k = -1;
  EscMeta cur, nxt;
  for (;;) {
    if (!mbar_wait_or_abort(&xrdy[slot], (uint32_t)round & 1u, abort)) {
      set_status(a.status, SD_TIMEOUT_AT(35));
      break;
    }
    const int4 in = info[slot];
    if (in.x < 0) break;
    const StreamPhase& P = a.ph[in.x];
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
      // the next unit's entries, if it is announced already
      const int j = (k + 1) % kUq;
      if (uq->seq[j] == k + 1) {
        __threadfence_block();
        const int4 d = uq->d[j];
        if (d.x >= 0) esc_meta_load(a.ph[d.x], d.x, d.y, d.z, d.w, nxt);
      }
    }
    if (P.tile_ptr) {
      if (t - cur.tc >= 32) esc_meta_load(P, in.x, b, t, tend, cur);  // a unit of more than 32 tiles
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
// Each consumer warp owns one 16-row strip of the current row block and
// finishes its strip on its own: a k-chunk of a split block leaves its fp32
// partial in the chunk's slot and takes a per-strip ticket (its result is
// looked at one stage later, so the warp does not wait for the atomic); the
// warp whose ticket completes the strip sums the strip's slots in chunk
// order (deterministic) and runs the strip's epilogue.  The strip
// finishers of a block count in a per-block counter; the last one adds the
// strips' sums of squares (residual epilogues) and publishes the block.

template <int NT>
__device__ __forceinline__ void s_strip_done(const StreamPhase& P, int b, int warp, int lane, float (&rs)[NT][2]) {
  constexpr int MP = NT * 8;
  if (P.out_ss) {
    // the strip's sum of squares per token row (its 16 rows by shuffles)
    float* dst = P.out_ss + (int64_t)P.NB * 128 + ((int64_t)b * 8 + warp) * 128;
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int cc = 0; cc < 2; cc++) {
        float v = rs[nt][cc];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        if (lane < 4) __stcg(dst + nt * 8 + 2 * lane + cc, v);
      }
  }
  __syncwarp();
  int old = 0;
  if (lane == 0) {
    __threadfence();
    old = atomicAdd(P.st + 2 + 8 * P.NB + b, 1);
  }
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old + 1 != kRB) return;
  // the block's last strip: the block sums (strips in order), then its flag
  if (P.out_ss) {
    __threadfence();
    const float* src = P.out_ss + (int64_t)P.NB * 128 + (int64_t)b * 8 * 128;
    for (int m = lane; m < MP; m += 32) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kRB; w++) v += __ldcg(src + w * 128 + m);
      P.out_ss[(int64_t)b * 128 + m] = v;
    }
  }
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    asm volatile("st.release.gpu.global.s32 [%0], 1;" ::"l"(P.st + 2 + 9 * P.NB + b) : "memory");
    asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(P.st + 1) : "memory");
  }
}

template <int NT>
__device__ __forceinline__ void s_consume(const StreamArgs& a, const uint8_t* sx, const uint8_t* sw, const int4* info,
                                          uint64_t* xrdy, uint64_t* empty, const float* corr, uint64_t* corr_full,
                                          uint64_t* corr_empty, StreamPhase* sph, float* red_v, int* red_i,
                                          uint64_t* cbar, volatile int* abort) {
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
  // the strip region of a split block's chunk slot
  auto slot_ptr = [&](const StreamPhase& P, int b, int c) {
    return P.part + ((int64_t)(b - P.nb_whole) * P.S + c) * (128 * MP) + ((warp * NT) * 32 + lane) * 4;
  };
  // epilogue of this warp's strip of block b from its sums, then the
  // block's bookkeeping
  auto finish_strip = [&](const StreamPhase& P, int b, float (&sum)[NT][4]) {
    float rs[NT][2];
    const int strip = b * kRB + warp;
    if (strip < P.NS) {
      s_epilogue<NT>(P, a.M, strip, lane, sum, bestv, besti, rs);
    } else {
#pragma unroll
      for (int nt = 0; nt < NT; nt++) rs[nt][0] = rs[nt][1] = 0.f;
    }
    s_strip_done<NT>(P, b, warp, lane, rs);
  };
  // a pending ticket (split chunk): if it completed the strip, sum the
  // strip's chunk slots in order and finish it
  int pend_b = -1, pend_old = 0;
  auto resolve = [&](const StreamPhase& P) {
    if (pend_b < 0) return;
    const int old = __shfl_sync(0xffffffffu, pend_old, 0);
    const int b = pend_b;
    pend_b = -1;
    if (old + 1 != P.S) return;
    float tot[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; nt++) tot[nt][0] = tot[nt][1] = tot[nt][2] = tot[nt][3] = 0.f;
    constexpr int kB = NT <= 1 ? 8 : NT <= 2 ? 4 : 2;
    for (int c0 = 0; c0 < P.S; c0 += kB) {
      float4 v[kB][NT];
#pragma unroll
      for (int u = 0; u < kB; u++) {
        const bool ld = c0 + u < P.S;
        const float* src = slot_ptr(P, b, ld ? c0 + u : 0);
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
          v[u][nt] = ld ? __ldcg(reinterpret_cast<const float4*>(src + nt * 128)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kB; u++) {
        if (c0 + u >= P.S) continue;
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
          tot[nt][0] += v[u][nt].x;
          tot[nt][1] += v[u][nt].y;
          tot[nt][2] += v[u][nt].z;
          tot[nt][3] += v[u][nt].w;
        }
      }
    }
    finish_strip(P, b, tot);  // acc may already hold the next unit's sums
  };

  pdl_wait();  // residuals and cache positions come from earlier kernels
  int slot = 0, round = 0, cseg = 0, cur = -1;
  bool fresh = true;  // acc holds nothing of the current unit yet
  zero();
  for (;;) {
    // a pending ticket is settled before any wait that is not already over:
    // the next tile may read the very block that ticket completes
    if (pend_b >= 0 && !mbar_test_wait(&xrdy[slot], (uint32_t)round & 1u)) resolve(*sph);
    if (!mbar_wait_or_abort(&xrdy[slot], (uint32_t)round & 1u, abort)) {
      set_status(a.status, SD_TIMEOUT_AT(37));
      break;
    }
    const int4 in = info[slot];
    if (in.x < 0) break;
    if (in.x != cur) {
      // a pending ticket belongs to the old phase: settle it first; then the
      // phase's descriptor in shared memory (uniform loads in the hot loop)
      if (cur >= 0) resolve(*sph);
      if (!cons_sync(cbar, cph, abort)) break;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(&a.ph[in.x]);
      uint32_t* dst = reinterpret_cast<uint32_t*>(sph);
      for (int i = tid; i < (int)(sizeof(StreamPhase) / 4); i += kSCons * 32) dst[i] = src[i];
      if (!cons_sync(cbar, cph, abort)) break;
      cur = in.x;
    }
    const StreamPhase& P = *sph;
    const int b = in.y;
    if ((in.w & 1) && !fresh) zero();
    fresh = false;
    const int strip = b * kRB + warp;
    if (strip < P.NS) {
      const bool v8 = P.view8 != 0;
      const uint8_t* wsm = sw + slot * C::WB + warp * (v8 ? 1024 : kStripBytes);
      const uint4 W0 = *reinterpret_cast<const uint4*>(wsm + lane * 16);
      const uint4 W1 = *reinterpret_cast<const uint4*>(wsm + 512 + lane * 16);
      const uint4 W2 = v8 ? W1 : *reinterpret_cast<const uint4*>(wsm + 1024 + lane * 16);
      const uint32_t xb = smem_u32(sx + slot * C::XB);
      const bool aff = P.affine != 0;
#pragma unroll
      for (int j = 0; j < 4; j++) {
        uint32_t a0, a1, a2, a3;
        if (v8)
          decode_view8(comp(W0, j), comp(W1, j), aff, P.base2, P.tab, a0, a1, a2, a3);
        else if (aff)
          decode<true>(comp(W0, j), comp(W1, j), comp(W2, j), P.base2, P.tab, a0, a1, a2, a3);
        else
          decode<false>(comp(W0, j), comp(W1, j), comp(W2, j), P.base2, P.tab, a0, a1, a2, a3);
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
    // the ticket of the previous unit has had a stage's time to come back
    resolve(P);
    if (!(in.w & 2)) continue;

    // ------------------------------------------------ unit finished --
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
    const int chunk = info_chunk(in.w);
    if (chunk < 0) {
      finish_strip(P, b, acc);  // a whole block: no partial, no ticket
    } else {
      float* mine = slot_ptr(P, b, chunk);
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
        __stcg(reinterpret_cast<float4*>(mine + nt * 128),
               make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]));
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        pend_old = atomicAdd(P.st + 2 + b * kRB + warp, 1);
      }
      pend_b = b;
    }
    zero();
    fresh = true;
  }
  if (cur >= 0) resolve(*sph);

  // per-CTA argmax partial of a logits phase (every CTA writes one)
  bool logits = false;
  const GemmEpilogue* le = nullptr;
  for (int p = 0; p < a.n; p++)
    if (a.ph[p].e.epi == EPI_LOGITS) {
      logits = true;
      le = &a.ph[p].e;
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

template <int NT>
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
  StreamPhase* sph = reinterpret_cast<StreamPhase*>(smem + C::OFF_PH);
  UnitQ* uq = reinterpret_cast<UnitQ*>(smem + C::OFF_UQ);
  float* corr = reinterpret_cast<float*>(smem + C::OFF_CORR);

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::RING; i++) {
      mbar_init(&full[i], 1);
      mbar_init(&xrdy[i], 1);
      mbar_init(&empty[i], kSCons + 1);  // consumer warps + escape warp
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
  __syncthreads();
  pdl_launch();

  if (warp == kSProd) {
    if ((threadIdx.x & 31) == 0) s_produce<NT>(a, sx, sw, info, full, empty, uq, abort);
  } else if (warp == kSNorm) {
    s_norm<NT>(a, sx, info, full, xrdy, rinv, abort);
  } else if (warp == kSEsc) {
    s_escape<NT>(a, sx, info, xrdy, empty, corr, corr_full, corr_empty, uq, abort);
  } else {
    s_consume<NT>(a, sx, sw, info, xrdy, empty, corr, corr_full, corr_empty, sph, red_v, red_i, cbar, abort);
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

// ------------------------------------------------------------------ host --

static int nt_of_rows(int M) { return pad_rows(M) / 8; }

int stream_grid(int M) { return (nt_of_rows(M) <= 4 ? 2 : 1) * num_sms(); }

static int blocks_of(const w12_tensor& W) { return (int)((W.N / 16 + kRB - 1) / kRB); }

size_t stream_state_ints(const StreamPhaseDesc* ph, int n) {
  size_t s = 1;
  for (int i = 0; i < n; i++) s += 2 + 10 * (size_t)blocks_of(*ph[i].W);
  return s;
}

size_t stream_state_ints_bound(int64_t n_max) {
  return 1 + (size_t)kStreamMaxPhases * (2 + 10 * (size_t)((n_max / 16 + kRB - 1) / kRB));
}

struct SplitPlan {
  int KT, NB, S, KC, nb_split;
};

static SplitPlan split_plan(const w12_tensor& W, int grid, int split_blocks) {
  SplitPlan sp;
  sp.KT = (int)(W.K / 64);
  sp.NB = blocks_of(W);
  sp.S = (sp.KT + kSChunkTiles - 1) / kSChunkTiles;
  if (sp.S < 1) sp.S = 1;
  sp.KC = (sp.KT + sp.S - 1) / sp.S;
  sp.S = (sp.KT + sp.KC - 1) / sp.KC;
  const int cap = split_blocks > 0 ? split_blocks : grid;
  sp.nb_split = sp.S > 1 ? std::min(sp.NB, cap) : 0;
  return sp;
}

size_t stream_partial_floats(const StreamPhaseDesc* ph, int n, int M) {
  size_t f = 0;
  const int grid = stream_grid(M);
  for (int i = 0; i < n; i++) {
    const SplitPlan sp = split_plan(*ph[i].W, grid, 0);
    f += (size_t)sp.nb_split * sp.S * 128 * pad_rows(M);
  }
  return f;
}

size_t stream_partial_floats_bound(int64_t n_max, int64_t k_max, int M) {
  const int64_t nb = (n_max / 16 + kRB - 1) / kRB;
  const int64_t kt = k_max / 64;
  const int64_t S = std::max<int64_t>(1, (kt + kSChunkTiles - 1) / kSChunkTiles);
  const int64_t split = std::min<int64_t>(nb, stream_grid(M));
  return (size_t)kStreamMaxPhases * split * S * 128 * pad_rows(M);
}

template <int NT>
static cudaError_t stream_launch_nt(const StreamArgs& a, int grid, cudaStream_t s, bool pdl) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(k_w12_stream<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, SCfg<NT>::SMEM);
  });
  if (attr != cudaSuccess) return attr;
  return launch(k_w12_stream<NT>, dim3(grid), dim3(kSThreads), SCfg<NT>::SMEM, s, pdl, a);
}

int stream_launch(const StreamPhaseDesc* ph, int n, int M, const StreamWorkspace& ws, int32_t* status, cudaStream_t s,
                  bool pdl, int split_blocks) {
  if (!ph || n < 1 || n > kStreamMaxPhases || M < 1 || M > 128) {
    set_error("stream: bad argument (1..4 phases, 1..128 rows)");
    return SD_ERR_INVALID_ARG;
  }
  if (!ws.state) {
    set_error("stream: no state scratch");
    return SD_ERR_WORKSPACE;
  }
  const int grid = stream_grid(M);
  const int MP = pad_rows(M);
  StreamArgs a;
  memset(&a, 0, sizeof(a));
  size_t st_off = 1, part_off = 0;
  for (int i = 0; i < n; i++) {
    const StreamPhaseDesc& d = ph[i];
    if (!d.W || !d.x || d.x_rows < M) {
      set_error("stream: phase without weights or input rows");
      return SD_ERR_INVALID_ARG;
    }
    const w12_tensor& W = *d.W;
    if (W.N % 16 || W.K % 64 || W.N < 16 || W.K < 64 || W.K / 64 > 0xFFFF) {
      set_error("stream: unsupported shape (N % 16, K % 64)");
      return SD_ERR_UNSUPPORTED;
    }
    if (W.n_escapes > 0 && (!W.tile_ptr || !W.tile_esc)) {
      set_error("stream: the tensor has escapes but no escape tile index (w12_pack_tile_index)");
      return SD_ERR_INVALID_ARG;
    }
    if (d.dep >= i || d.dep < -1 || (d.dep_fine && d.dep < 0)) {
      set_error("stream: a phase may depend on an earlier phase only");
      return SD_ERR_INVALID_ARG;
    }
    if (d.norm_gamma && (d.dep < 0 || !ph[d.dep].out_ss || ph[d.dep].W->N != W.K)) {
      set_error("stream: an input RMSNorm needs an earlier residual phase with out_ss of width K");
      return SD_ERR_INVALID_ARG;
    }
    if (d.out_ss && d.epi.epi != EPI_RESID) {
      set_error("stream: out_ss needs a residual epilogue");
      return SD_ERR_INVALID_ARG;
    }
    StreamPhase& P = a.ph[i];
    const SplitPlan sp = split_plan(W, grid, split_blocks);
    P.words = d.view8 ? d.view8 : W.words;
    P.view8 = d.view8 ? 1 : 0;
    P.tile_ptr = W.n_escapes > 0 ? W.tile_ptr : nullptr;
    P.tile_esc = W.tile_esc;
    P.N = W.N;
    P.K = W.K;
    P.KT = sp.KT;
    P.NS = (int)(W.N / 16);
    P.NB = sp.NB;
    P.S = sp.S;
    P.KC = sp.KC;
    P.nb_whole = sp.NB - sp.nb_split;
    P.U = P.nb_whole + sp.nb_split * sp.S;
    P.affine = W.affine != 0;
    const uint32_t base = W.n_table > 0 ? W.table[0] : 0;
    P.base2 = (base << 7) | (base << 23);
    uint8_t t16[16] = {0};
    for (int j = 0; j < W.n_table && j < 15; j++) t16[j] = W.table[j];
    for (int j = 0; j < 4; j++)
      P.tab[j] = t16[4 * j] | (t16[4 * j + 1] << 8) | (t16[4 * j + 2] << 16) | ((uint32_t)t16[4 * j + 3] << 24);
    P.esc_slot = W.affine ? ldexpf(1.0f, (int)base + 15 - 127) : 0.0f;
    P.e = d.epi;
    P.gamma = d.norm_gamma;
    P.eps = d.norm_eps;
    P.in_ss = d.norm_gamma ? ph[d.dep].out_ss : nullptr;
    P.nss = d.norm_gamma ? blocks_of(*ph[d.dep].W) : 0;
    P.norm_out = d.norm_gamma ? d.norm_out : nullptr;
    P.dep = d.dep;
    P.dep_fine = d.dep_fine;
    P.out_ss = d.out_ss;
    P.st = ws.state + st_off;
    st_off += 2 + 10 * (size_t)P.NB;
    P.part = ws.partial + part_off;
    part_off += (size_t)sp.nb_split * sp.S * 128 * MP;
    XMap xm;
    int rc = make_x_map(&xm, d.x, d.x_rows, W.K, MP);
    if (rc) return rc;
    a.xmap[i] = xm.map;
    rc = d.view8 ? make_w8_map(&a.wmap[i], d.view8, W.N, W.K) : make_w_map(&a.wmap[i], W);
    if (rc) return rc;
  }
  if (st_off > ws.state_ints || part_off > ws.partial_floats) {
    set_error("stream: workspace too small");
    return SD_ERR_WORKSPACE;
  }
  for (int i = 0; i < n; i++)
    if (ph[i].epi.epi == EPI_LOGITS && (!ph[i].epi.amax_val || !ph[i].epi.amax_idx || ph[i].epi.ld_amax < M)) {
      set_error("stream: logits phase without argmax partials");
      return SD_ERR_INVALID_ARG;
    }
  a.n = n;
  a.M = M;
  a.state = ws.state;
  a.state_ints = (int)st_off;
  a.status = status;
  cudaError_t e;
  switch (MP / 8) {
    case 1: e = stream_launch_nt<1>(a, grid, s, pdl); break;
    case 2: e = stream_launch_nt<2>(a, grid, s, pdl); break;
    case 4: e = stream_launch_nt<4>(a, grid, s, pdl); break;
    case 8: e = stream_launch_nt<8>(a, grid, s, pdl); break;
    default: e = stream_launch_nt<16>(a, grid, s, pdl); break;
  }
  if (e != cudaSuccess) return cuda_fail(e, "k_w12_stream launch");
  return SD_OK;
}

}  // namespace sdv
