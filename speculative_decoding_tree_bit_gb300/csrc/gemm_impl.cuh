// Device building blocks of the warp-level fused W12 GEMM (gemm.cu): the
// shared-memory layout, the decodes, the epilogues, the escape warp and the
// consumers' main loop and split-K finish.
#pragma once

#include "gemm.cuh"

namespace sdv {

constexpr int kNCW = 8;            // consumer warps 0..7
constexpr int kRB = kNCW;          // strips per row block
constexpr int kProducerWarp = kNCW;     // streams weights and activations into the ring
constexpr int kEscapeWarp = kNCW + 1;   // computes escape corrections ahead of the consumers
constexpr int kThreads = (kNCW + 2) * 32;
constexpr int kStripBytes = 1536;  // one strip x one super-tile (16 x 64 x 12 bit)

// Shared-memory layout of the GEMM kernels (after 1024-byte alignment).
// V8: the weights are the nested 8-bit plane (1024 bytes per strip and
// super-tile instead of 1536), the freed shared memory goes to more stages.
template <int NT, bool V8 = false>
struct Cfg {
  static constexpr int MP = NT * 8;    // padded rows (tokens) per launch
  static constexpr int XB = MP * 128;  // x tile bytes per stage (64 columns of bf16)
  static constexpr int WB = kRB * (V8 ? 1024 : kStripBytes);
  static constexpr int S = V8 ? (NT <= 1 ? 11 : NT <= 2 ? 10 : NT <= 4 ? 7 : NT <= 8 ? 6 : 4)
                              : (NT <= 1 ? 8 : NT <= 2 ? 7 : NT <= 8 ? 5 : 4);  // ring stages
  static constexpr int OFF_W = S * XB;
  static constexpr int OFF_FULL = OFF_W + S * WB;
  static constexpr int OFF_EMPTY = OFF_FULL + S * 8;
  static constexpr int OFF_RED_V = OFF_EMPTY + S * 8;          // argmax scratch [8][MP]
  static constexpr int OFF_RED_I = OFF_RED_V + kNCW * MP * 4;
  static constexpr int OFF_FLAG = OFF_RED_I + kNCW * MP * 4;    // finisher flag, abort flag
  static constexpr int OFF_CBAR = OFF_FLAG + 16;                // escape tile full / empty barriers
  static constexpr int OFF_CORR = (OFF_CBAR + 16 + 15) & ~15;   // escape corrections [128 rows][MP] fp32
  static constexpr int END = OFF_CORR + 128 * MP * 4;
  static constexpr int SMEM = 1024 + END;
};

struct GemmParams {
  const uint32_t* words;
  int64_t N, K;
  int KT, NS, NB;
  int64_t U;
  uint32_t base2;
  uint32_t tab[4];
  float esc_slot;
  const uint32_t* tile_ptr;  // escape tile index (null when there are no escapes)
  const uint32_t* tile_esc;
  const uint16_t* x;
  int M, m0;
  float* partial;
  int32_t* counters;
  GemmEpilogue e;
  int32_t* status;
  uint64_t* trace;  // optional: [4][grid] device-clock stamps (start, first stage ready, last consumed, finished)
  int64_t G;        // CTAs sharing the units (<= the grid; 0: the grid); CTAs beyond it have no work
  int view8;         // the weights are the nested 8-bit plane (1 KB per strip and super-tile)
  uint32_t esc_mask;  // applied to an escape's bf16 bits: 0xFFFF, or 0xFFF0 for the 8-bit view
  const uint8_t* row_base;  // per-channel bases [N] (null: the tensor's table)
  // > 1: the launch is in clusters of cluster_k CTAs, one cluster per row
  // block, each CTA one k-range of it; the block is finished through
  // distributed shared memory instead of partials in global memory
  int cluster_k;
  // 1: split row blocks leave their partials and return; k_gemm_finish,
  // launched after the GEMM, sums them and runs the epilogue
  int defer;
};

// Contributors whose partials the in-kernel finisher loads at a time (empty
// slots of a batch add +0); the deferred finish adds in the same grouping.
__host__ __device__ constexpr int finish_batch(int NT) { return NT <= 2 ? 4 : 2; }

// n / d for 0 <= n and 0 < d: one 32-bit division when both fit (a 64-bit
// division is a long software sequence, and the unit bookkeeping of every
// realistic shape fits in 32 bits).
__device__ __forceinline__ int64_t udiv(int64_t n, int64_t d) {
  if ((((uint64_t)n | (uint64_t)d) >> 32) == 0) return (int64_t)((uint32_t)n / (uint32_t)d);
  return (int64_t)((uint64_t)n / (uint64_t)d);
}

// This CTA's stream-K unit range [u0, u1) and the number of CTAs sharing
// the units.
__device__ __forceinline__ int64_t unit_ctas(const GemmParams& p) { return p.G > 0 ? p.G : (int64_t)gridDim.x; }
__device__ __forceinline__ void unit_range(const GemmParams& p, int64_t& u0, int64_t& u1) {
  const int64_t G = unit_ctas(p), c = blockIdx.x;
  u0 = c < G ? udiv(c * p.U, G) : p.U;
  u1 = c < G ? udiv((c + 1) * p.U, G) : p.U;
}

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

// Two bytes of the nested 8-bit plane (bits 0..7 and 16..23: sign << 7 |
// code << 3 | top mantissa bits) -> their bf16 view, as a bf16x2 fragment
// register.
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

// Per-channel decode (contiguous window per row): a0 and a2 hold row g of
// the strip, a1 and a3 row g + 8, so each takes its own row's base.
__device__ __forceinline__ void decode_rows(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t b2lo, uint32_t b2hi,
                                            uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
  const uint32_t X = ((w0 >> 11) & 0x000F000Fu) | ((w1 >> 7) & 0x00F000F0u) | ((w2 >> 3) & 0x0F000F00u);
  a0 = (w0 & 0x87FF87FFu) + b2lo;
  a1 = (w1 & 0x87FF87FFu) + b2hi;
  a2 = (w2 & 0x87FF87FFu) + b2lo;
  a3 = ((X & 0x07FF07FFu) + b2hi) | ((X << 4) & 0x80008000u);
}

__device__ __forceinline__ uint32_t comp(const uint4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// Residuals may have been written earlier in the same launch by other CTAs
// (chained phases): they are read with L1-bypassing loads.  The residual and
// QKV epilogues issue every load of the thread's rows before any store (the
// output may alias the residual, so a load placed after a store would wait
// for it: one memory round trip per element).
template <int NT>
__device__ __forceinline__ void epilogue(const GemmParams& p, int strip, int lane, float (&acc)[NT][4],
                                         float (&bestv)[NT][2], int (&besti)[NT][2]) {
  const int g = lane >> 2, q = lane & 3;
  const int64_t n_lo = (int64_t)strip * 16 + g;
  const GemmEpilogue& E = p.e;
  if (E.epi == EPI_RESID) {
    float r[NT][2][2];
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int cc = 0; cc < 2; cc++) {
        const int m = p.m0 + nt * 8 + 2 * q + cc;
        const int64_t i0 = (int64_t)m * E.ldo + n_lo;
        const bool ok = m < p.M;
        r[nt][cc][0] = ok ? bf2f(__ldcg(E.resid + i0)) : 0.f;
        r[nt][cc][1] = ok ? bf2f(__ldcg(E.resid + i0 + 8)) : 0.f;
      }
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int cc = 0; cc < 2; cc++) {
        const int m = p.m0 + nt * 8 + 2 * q + cc;
        if (m >= p.M) continue;
        const int64_t i0 = (int64_t)m * E.ldo + n_lo;
        E.out[i0] = f2bf(r[nt][cc][0] + rbf(acc[nt][cc]));
        E.out[i0 + 8] = f2bf(r[nt][cc][1] + rbf(acc[nt][2 + cc]));
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
      // the thread's two rows of this token tile: loads first, then stores
      int pos[2], rq[2], slot[2];
#pragma unroll
      for (int cc = 0; cc < 2; cc++) {
        const int m = p.m0 + nt * 8 + 2 * q + cc;
        const bool ok = m < p.M;
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
        const int m = p.m0 + nt * 8 + 2 * q + cc;
        if (m >= p.M || !okr[cc]) continue;
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
      const int m = p.m0 + nt * 8 + 2 * q + cc;
      if (m >= p.M) continue;
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

// ----------------------------------------------------------- escapes --
// Escaped weights decode to the slot value in the main loop; the escape warp
// supplies, for each row-block segment [t0, t1) of a CTA's unit range (in the
// consumers' order), the correction sum (w - slot) x[m][k] over the escapes of
// the segment's rows and columns in a shared tile corr[128 rows][MP].  It is
// a ninth reader of the ring: each stage's escapes - one contiguous run of
// the escape tile index - are applied from the activation tile already
// staged in shared memory, one escape at a time with the lanes parallel over
// the token rows m, in the index's fixed order (deterministic).  The index is
// read in chunks of 32 tiles: lane i holds the tile pointers of tile tc + i
// and tc + i + 1 and entries e_lo + i + 32 j; the next chunk's pointers and
// entries are loaded while the current chunk's stages are processed.

struct EscChunk {
  uint32_t tpa, tpb;  // tile_ptr of tiles tc + lane, tc + lane + 1 (clamped to the segment end)
  uint32_t ent[4];    // entries e_lo + lane + 32 j
  uint32_t e_lo, e_hi;
};

__device__ __forceinline__ void esc_chunk_ptrs(const GemmParams& p, int b, int tc, int tend, EscChunk& c) {
  const int lane = threadIdx.x & 31;
  const uint32_t* tp = p.tile_ptr + (int64_t)b * p.KT;
  c.tpa = __ldg(tp + min(tc + lane, tend));
  c.tpb = __ldg(tp + min(tc + lane + 1, tend));
}

__device__ __forceinline__ void esc_chunk_entries(const GemmParams& p, int tc, int tend, EscChunk& c) {
  const int lane = threadIdx.x & 31;
  c.e_lo = __shfl_sync(0xffffffffu, c.tpa, 0);
  c.e_hi = __shfl_sync(0xffffffffu, c.tpb, min(31, tend - 1 - tc));
#pragma unroll
  for (int j = 0; j < 4; j++) {
    const uint32_t e = c.e_lo + lane + 32 * j;
    c.ent[j] = e < c.e_hi ? __ldg(p.tile_esc + e) : 0u;
  }
}

// The escape warp's work for one GEMM; slot / phase follow the ring exactly
// as the consumers do (it arrives on every stage's empty barrier).  eseg
// counts the tiles produced.  Returns false on a failed wait (status set).
template <int NT, bool V8 = false>
__device__ __forceinline__ bool escape_segments(const GemmParams& p, const uint8_t* sx, uint64_t* full,
                                                uint64_t* empty, int& slot, uint32_t& phase, float* corr,
                                                uint64_t* corr_full, uint64_t* corr_empty, int& eseg,
                                                volatile int* abort) {
  using C = Cfg<NT, V8>;
  constexpr int MP = C::MP;
  const int lane = threadIdx.x & 31;
  int64_t u0, u1;
  unit_range(p, u0, u1);
  if (u1 <= u0) return true;
  const int KT = p.KT;
  const int b_first = (int)udiv(u0, KT), b_last = (int)udiv(u1 - 1, KT);
  const bool any = p.tile_ptr != nullptr;
  const int mrows = min(MP, p.M - p.m0);
  auto tbeg = [&](int b) { return b == b_first ? (int)(u0 - (int64_t)b_first * KT) : 0; };
  auto tend = [&](int b) { return b == b_last ? (int)(u1 - 1 - (int64_t)b_last * KT) + 1 : KT; };
  bool ok = true;
  EscChunk cur{}, nxt{};
  int cb = b_first, ctc = tbeg(b_first), seg_b = -1;
  if (any) {
    esc_chunk_ptrs(p, cb, ctc, tend(cb), cur);
    esc_chunk_entries(p, ctc, tend(cb), cur);
  }
  for (;;) {
    if (cb != seg_b) {
      if (seg_b >= 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(corr_full);
        eseg++;
      }
      if (!mbar_wait_or_abort(corr_empty, (uint32_t)(eseg & 1) ^ 1u, abort)) {
        set_status(p.status, SD_TIMEOUT_AT(3));
        ok = false;
      }
#pragma unroll
      for (int i = 0; i < 4; i++) {
        float* row = corr + (lane + 32 * i) * MP;
#pragma unroll
        for (int m = 0; m < MP; m += 4) *reinterpret_cast<float4*>(row + m) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      seg_b = cb;
    }
    const int ce = min(ctc + 32, tend(cb));
    int nb = cb, ntc = ce;
    if (ntc >= tend(cb)) {
      nb = cb + 1;
      ntc = nb <= b_last ? tbeg(nb) : 0;
    }
    const bool has_next = nb <= b_last;
    if (any && has_next) esc_chunk_ptrs(p, nb, ntc, tend(nb), nxt);
    for (int t = ctc; t < ce; t++) {
      if (!mbar_wait_or_abort(&full[slot], phase, abort)) {
        set_status(p.status, SD_TIMEOUT_AT(14));
        ok = false;
      }
      if (any) {
        const uint8_t* xs = sx + slot * C::XB;
        const uint32_t lo = __shfl_sync(0xffffffffu, cur.tpa, t - ctc);
        const uint32_t hi = __shfl_sync(0xffffffffu, cur.tpb, t - ctc);
        for (uint32_t e = lo; e < hi; e++) {
          const uint32_t idx = e - cur.e_lo;
          uint32_t v;
          if (idx < 128) {
            const uint32_t r = idx < 32 ? cur.ent[0] : idx < 64 ? cur.ent[1] : idx < 96 ? cur.ent[2] : cur.ent[3];
            v = __shfl_sync(0xffffffffu, r, idx & 31);
          } else {
            v = __ldg(p.tile_esc + e);  // a chunk with more than 128 escapes
          }
          const int row = (v >> 6) & 127, kk = v & 63;
          const float w = bf2f((v >> 16) & p.esc_mask);
          // the value the slot decodes to: 2^(base + 15 - 127), per row for
          // a per-channel tensor
          const float slot_v = p.row_base ? __uint_as_float((uint32_t)(p.row_base[(int64_t)cb * 128 + row] + 15) << 23)
                                          : p.esc_slot;
          float* cr = corr + row * MP;
          for (int m = lane; m < mrows; m += 32) {
            const float xv = bf2f(
                *reinterpret_cast<const uint16_t*>(xs + m * 128 + (((kk >> 3) ^ (m & 7)) << 4) + (kk & 7) * 2));
            const float a = fmaf(w, xv, cr[m]);
            cr[m] = fmaf(-slot_v, xv, a);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (++slot == C::S) {
        slot = 0;
        phase ^= 1u;
      }
      if (any && has_next && t == ctc) esc_chunk_entries(p, ntc, tend(nb), nxt);
    }
    if (!has_next) break;
    cb = nb;
    ctc = ntc;
    cur = nxt;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(corr_full);
  eseg++;
  return ok;
}

// Consumer warps (0..7) of one GEMM over this CTA's stream-K unit range:
// wait for each ring stage, decode + MMA, finish row blocks (split ones by
// the last contributor) and run the epilogue; for EPI_LOGITS also write this
// CTA's per-row argmax partial.  slot / phase continue the ring position
// across calls.  Returns false after a timed-out wait (status set).
// stamps (optional): thread 0 records the device clock when its first stage
// is ready (stamps[0]) and when its last stage is consumed (stamps[stride]).
// Escape corrections of each segment come from the escape warp's tile (cseg
// counts the tiles taken).  After a failed wait (status set) the warps run
// on with stale data, so all of them keep meeting at the named barriers.
template <int NT, bool AFFINE, bool V8 = false, bool CH = false>
__device__ __forceinline__ bool consume_gemm(const GemmParams& p, uint8_t* sx, uint8_t* sw, uint64_t* full,
                                             uint64_t* empty, float* red_v, int* red_i, int* flag, int& slot,
                                             uint32_t& phase, const float* corr, uint64_t* corr_full,
                                             uint64_t* corr_empty, int& cseg, volatile int* abort,
                                             uint64_t* stamps = nullptr, int64_t stride = 0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = unit_ctas(p);
  int64_t u0, u1;
  unit_range(p, u0, u1);
  const int KT = p.KT;
  // small tiles: even and odd sub-tiles feed separate accumulators so that
  // consecutive MMAs do not wait on each other; larger tiles have NT
  // independent MMAs per sub-tile already
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
  const int first_b = u1 > u0 ? (int)udiv(u0, KT) : -1;

  auto zero = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int c = 0; c < 4; c++) {
        acc[nt][c] = 0.f;
        if constexpr (kDual) acc2[nt][c] = 0.f;
      }
  };
  auto partial_ptr = [&](int64_t cta, int slot_id) {
    return p.partial + (((cta * 2 + slot_id) * kRB + warp) * NT) * 128 + lane * 4;
  };
  // finish the segment [t0, t1) of row block b
  auto finish = [&](int b, int t0, int t1) {
    const int strip = b * kRB + warp;
    if constexpr (kDual) {
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int c = 0; c < 4; c++) acc[nt][c] += acc2[nt][c];
    }
    // this segment's escape corrections
    if (!mbar_wait_or_abort(corr_full, (uint32_t)(cseg & 1), abort)) set_status(p.status, SD_TIMEOUT_AT(4));
    {
      constexpr int MP = Cfg<NT, V8>::MP;
      const int g = lane >> 2, q = lane & 3;
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
    if (!(t0 == 0 && t1 == KT) && p.cluster_k > 1) {
      // the cluster's CTAs are the block's contributors, in CTA order: each
      // stages its partial in its own shared memory (the weight ring is idle
      // once the segment's last stage is consumed), the leader (rank 0, the
      // first contributor) adds the others' through distributed shared
      // memory in rank order - the sum the global path forms - and runs the
      // epilogue; the second barrier keeps every CTA's shared memory alive
      // until the leader has read it.  The staging area overlaps the first
      // ring slot, which another consumer warp may still be reading for its
      // last stage: every consumer warp is past its last stage first.
      bar_sync(1, kNCW * 32);
      float* stage = reinterpret_cast<float*>(sw) + ((warp * NT) * 32 + lane) * 4;
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
        *reinterpret_cast<float4*>(stage + nt * 128) = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
      cluster_sync_all();
      const bool leader = cluster_rank() == 0;
      if (leader) {
        const uint32_t mine = smem_u32(stage);
        for (int r = 1; r < p.cluster_k; r++) {
          const uint32_t remote = cluster_map(mine, (uint32_t)r);
          float4 v[NT];
#pragma unroll
          for (int nt = 0; nt < NT; nt++) v[nt] = ld_cluster_f4(remote + nt * 128 * 4);
#pragma unroll
          for (int nt = 0; nt < NT; nt++) {
            acc[nt][0] += v[nt].x;
            acc[nt][1] += v[nt].y;
            acc[nt][2] += v[nt].z;
            acc[nt][3] += v[nt].w;
          }
        }
      }
      cluster_sync_all();
      if (!leader) return;
    } else if (!(t0 == 0 && t1 == KT)) {
      const int slot_id = (b == first_b) ? 0 : 1;
      float* dst = partial_ptr(blockIdx.x, slot_id);
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
        __stcg(reinterpret_cast<float4*>(dst + nt * 128), make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]));
      if (p.defer) return;  // the finish kernel sums the block's partials
      // the named barrier orders every thread's partial before thread 0's
      // device-scope fence and ticket (and the ticket before the others'
      // reads of the contributors' partials)
      bar_sync(1, kNCW * 32);
      if (threadIdx.x == 0) {
        const int add = t1 - t0;
        const int old = atomic_add_acq_rel(&p.counters[b], add);
        *flag = (old + add == KT) ? 1 : 0;
      }
      bar_sync(1, kNCW * 32);
      if (!*flag) return;
      zero();
      // contributors: the CTAs whose (non-empty) unit range meets row block b
      const int64_t c_first = udiv(((int64_t)b * KT + 1) * G - 1, p.U);
      const int64_t c_last = udiv(((int64_t)(b + 1) * KT) * G - 1, p.U);
      // partial slots of the contributors, read kBatch at a time with all
      // loads in flight before any is used (CTA order kept: deterministic)
      constexpr int kBatch = finish_batch(NT);
      for (int64_t c0 = c_first; c0 <= c_last; c0 += kBatch) {
        float4 v[kBatch][NT];
        bool use[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; u++) {
          const int64_t c = c0 + u;
          const int64_t cs = udiv(c * p.U, G), ce = udiv((c + 1) * p.U, G);
          use[u] = c <= c_last && cs != ce;  // empty ranges never wrote a partial
          // slot 1 when the contributor's range began in an earlier block
          const float* src = partial_ptr(use[u] ? c : blockIdx.x, (use[u] && cs < (int64_t)b * KT) ? 1 : 0);
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
      if (threadIdx.x == 0) p.counters[b] = 0;
    }
    if (strip < p.NS) epilogue<NT>(p, strip, lane, acc, bestv, besti);
  };

  zero();
  int cur_b = -1, seg_t0 = 0;
  uint32_t b2lo = 0, b2hi = 0;  // per-channel bases of the lane's rows (CH)
  bool ok = true;
  int b = u1 > u0 ? (int)udiv(u0, KT) : 0, t = u1 > u0 ? (int)(u0 - (int64_t)b * KT) : 0;
  for (int64_t n = u1 - u0; n > 0; --n) {
    if (b != cur_b) {
      if (cur_b >= 0) finish(cur_b, seg_t0, KT);
      cur_b = b;
      seg_t0 = t;
      zero();
      if constexpr (CH) {
        // the bases of this lane's two rows of its strip, shifted into both
        // halves' exponent fields
        const int64_t r0 = (int64_t)(b * kRB + warp) * 16 + (lane >> 2);
        const uint32_t blo = r0 < p.N ? p.row_base[r0] : 0u, bhi = r0 + 8 < p.N ? p.row_base[r0 + 8] : 0u;
        b2lo = (blo << 7) | (blo << 23);
        b2hi = (bhi << 7) | (bhi << 23);
      }
    }
    if (!mbar_wait_or_abort(&full[slot], phase, abort)) {
      set_status(p.status, SD_TIMEOUT_AT(5));
      ok = false;
    }
    if (stamps && threadIdx.x == 0 && n == u1 - u0) stamps[0] = globaltimer();
    const int strip = b * kRB + warp;
    if (strip < p.NS) {
      const uint8_t* wsm = sw + slot * Cfg<NT, V8>::WB + warp * (V8 ? 1024 : kStripBytes);
      const uint4 W0 = *reinterpret_cast<const uint4*>(wsm + lane * 16);
      const uint4 W1 = *reinterpret_cast<const uint4*>(wsm + 512 + lane * 16);
      uint4 W2 = W1;
      if (!V8) W2 = *reinterpret_cast<const uint4*>(wsm + 1024 + lane * 16);
      const uint32_t xb = smem_u32(sx + slot * Cfg<NT, V8>::XB);
#pragma unroll
      for (int j = 0; j < 4; j++) {
        uint32_t a0, a1, a2, a3;
        if constexpr (V8)
          decode_view8(comp(W0, j), comp(W1, j), AFFINE, p.base2, p.tab, a0, a1, a2, a3);
        else if constexpr (CH)
          decode_rows(comp(W0, j), comp(W1, j), comp(W2, j), b2lo, b2hi, a0, a1, a2, a3);
        else
          decode<AFFINE>(comp(W0, j), comp(W1, j), comp(W2, j), p.base2, p.tab, a0, a1, a2, a3);
        const int kchunk = 2 * j + ((lane >> 3) & 1);
        // even and odd sub-tiles accumulate into separate sets (shorter MMA chains)
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
    if (++slot == Cfg<NT, V8>::S) {
      slot = 0;
      phase ^= 1u;
    }
    if (++t == KT) {
      t = 0;
      b++;
    }
  }
  if (stamps && threadIdx.x == 0) stamps[stride] = globaltimer();
  if (cur_b >= 0) finish(cur_b, seg_t0, (int)(u1 - 1 - udiv(u1 - 1, KT) * KT) + 1);

  if (p.e.epi == EPI_LOGITS) {
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
          red_v[warp * Cfg<NT, V8>::MP + nt * 8 + 2 * lane + c] = v;
          red_i[warp * Cfg<NT, V8>::MP + nt * 8 + 2 * lane + c] = i;
        }
      }
    bar_sync(1, kNCW * 32);
    if (threadIdx.x < Cfg<NT, V8>::MP) {
      const int ml = threadIdx.x;
      float v = -INFINITY;
      int i = 0x7FFFFFFF;
      for (int w = 0; w < kNCW; w++) {
        const float ov = red_v[w * Cfg<NT, V8>::MP + ml];
        const int oi = red_i[w * Cfg<NT, V8>::MP + ml];
        if (ov > v || (ov == v && oi < i)) {
          v = ov;
          i = oi;
        }
      }
      const int m = p.m0 + ml;
      if (m < p.M) {
        p.e.amax_val[(int64_t)blockIdx.x * p.e.ld_amax + m] = v;
        p.e.amax_idx[(int64_t)blockIdx.x * p.e.ld_amax + m] = i;
      }
    }
  }
  return ok;
}

}  // namespace sdv
