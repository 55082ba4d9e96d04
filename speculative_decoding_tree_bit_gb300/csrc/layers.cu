// Tree-verify kernels other than the W12 GEMM.
//
// Tree bookkeeping, RMSNorm (+ embedding gather), tree-masked GQA attention
// (split over the cached prefix, one more split for the tree's own keys, then
// a combine), the tree linear recurrence, argmax reduction + greedy
// acceptance, and the commit (K/V compaction, recurrent state update).
//
// "SpecPilot: AI Agent Framework Boosts Speculative Decoding 10.87x for
// Qwen3.8-27B", "(2) Best-first Tree Verification for Hybrid Architectures":
// the target scores all tree nodes in one pass; each node must see exactly
// its root path, and a recurrent state has to follow each root path.
// "(3) Two-Level Verification": only the exact verification accepts tokens.
#include <mutex>

#include "layers.cuh"

namespace sdv {

// ------------------------------------------------------------------ tree --

__global__ void k_tree(const int32_t* __restrict__ tokens, const int32_t* __restrict__ parents,
                       const int32_t* __restrict__ cu, CacheView cv, int vocab, int max_positions, StepRows rows,
                       int32_t* status) {
  pdl_launch();  // the next kernel may start streaming its (independent) weights now
  pdl_wait();
  __shared__ uint64_t anc[64];
  __shared__ int dep[64];
  __shared__ int okflag, ctx_s;
  const int r = blockIdx.x;
  const int a = cu[r], M = cu[r + 1] - a;
  if (threadIdx.x == 0) {
    int code = 0;
    const int ctx = cv.ctx_len[r];
    if (M < 1 || M > 64) code = SD_ERR_BAD_TREE;
    for (int i = 0; i < M && i < 64 && !code; i++) {
      const int p = parents[a + i];
      if (i == 0 ? p != -1 : (p < 0 || p >= i)) {
        code = SD_ERR_BAD_TREE;
        break;
      }
      anc[i] = (i ? anc[p] : 0ull) | (1ull << i);
      dep[i] = i ? dep[p] + 1 : 0;
    }
    for (int i = 0; i < M && i < 64 && !code; i++) {
      const int t = tokens[a + i];
      if (t < 0 || t >= vocab) code = SD_ERR_BAD_TOKEN;
    }
    if (!code) {
      const int64_t need = (int64_t)ctx + M;
      if (ctx < 0 || need > (int64_t)cv.max_pages * cv.page_size || need > max_positions) code = SD_ERR_CAPACITY;
      const int np = code ? 0 : (int)((need + cv.page_size - 1) / cv.page_size);
      for (int pg = 0; pg < np && !code; pg++) {
        const int id = cv.page_table[(int64_t)r * cv.max_pages + pg];
        if (id < 0 || id >= cv.n_pages) code = SD_ERR_CAPACITY;
      }
    }
    if (code) {
      set_status(status, code);
      for (int i = 0; i < 64; i++) {
        anc[i] = 1ull << i;
        dep[i] = 0;
      }
    }
    okflag = code ? 0 : 1;
    ctx_s = code ? 0 : ctx;
  }
  __syncthreads();
  const int n = M < 64 ? M : 64;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    rows.pos[a + i] = ctx_s + dep[i];
    rows.slot[a + i] = ctx_s + i;
    rows.req[a + i] = r;
    rows.depth[a + i] = dep[i];
    rows.anc[a + i] = anc[i];
  }
  if (threadIdx.x == 0) {
    rows.ctx_snap[r] = ctx_s;
    rows.req_ok[r] = okflag;
  }
}

cudaError_t launch_tree(const int32_t* tokens, const int32_t* parents, const int32_t* cu, int R, const CacheView& cv,
                        int vocab, int max_positions, const StepRows& rows, int32_t* status, cudaStream_t s, bool pdl) {
  return launch(k_tree, dim3(R), dim3(64), 0, s, pdl, tokens, parents, cu, cv, vocab, max_positions, rows, status);
}

// ------------------------------------------------------------- RMSNorm --
// y = bf16((x * (1 / sqrt(mean(x^2) + eps))) * gamma), fp32 inside.

__global__ void __launch_bounds__(256) k_rmsnorm(const uint16_t* __restrict__ src, const uint16_t* __restrict__ gamma,
                                                 int H, float eps, uint16_t* __restrict__ xn,
                                                 const int32_t* __restrict__ tokens,
                                                 const uint16_t* __restrict__ embed, uint16_t* __restrict__ x_out,
                                                 const int32_t* __restrict__ row_req,
                                                 const int32_t* __restrict__ req_ok) {
  pdl_launch();  // the next kernel may start streaming its (independent) weights now
  // up to kKeep 8-element chunks per thread stay in registers between the
  // two passes (H <= 8192 at 256 threads); gamma is a weight, so it is read
  // before the wait for the previous kernel
  constexpr int kKeep = 4;
  const int n8 = H / 8;
  uint4 gk[kKeep], vk[kKeep];
#pragma unroll
  for (int it = 0; it < kKeep; it++) {
    const int i = threadIdx.x + it * blockDim.x;
    if (i < n8) gk[it] = reinterpret_cast<const uint4*>(gamma)[i];
  }
  pdl_wait();
  const int m = blockIdx.x;
  const uint16_t* row;
  if (embed) {
    int t = tokens[m];
    if (!req_ok[row_req[m]]) t = 0;
    row = embed + (int64_t)t * H;
  } else {
    row = src + (int64_t)m * H;
  }
  float ss = 0.f;
  auto square_add = [&](const uint4& v, int i) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const float lo = bf2f(w[j] & 0xFFFF), hi = bf2f(w[j] >> 16);
      ss = fmaf(lo, lo, ss);
      ss = fmaf(hi, hi, ss);
    }
    if (x_out) reinterpret_cast<uint4*>(x_out + (int64_t)m * H)[i] = v;
  };
#pragma unroll
  for (int it = 0; it < kKeep; it++) {
    const int i = threadIdx.x + it * blockDim.x;
    if (i < n8) vk[it] = reinterpret_cast<const uint4*>(row)[i];
  }
#pragma unroll
  for (int it = 0; it < kKeep; it++) {
    const int i = threadIdx.x + it * blockDim.x;
    if (i < n8) square_add(vk[it], i);
  }
  for (int i = threadIdx.x + kKeep * blockDim.x; i < n8; i += blockDim.x)
    square_add(reinterpret_cast<const uint4*>(row)[i], i);
  __shared__ float red[8];
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); i++) tot += red[i];
  const float rinv = 1.0f / sqrtf(tot / (float)H + eps);
  auto scale_store = [&](const uint4& v, const uint4& gm, int i) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const uint32_t gg[4] = {gm.x, gm.y, gm.z, gm.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const float lo = (bf2f(w[j] & 0xFFFF) * rinv) * bf2f(gg[j] & 0xFFFF);
      const float hi = (bf2f(w[j] >> 16) * rinv) * bf2f(gg[j] >> 16);
      o[j] = pack_bf16x2(lo, hi);
    }
    reinterpret_cast<uint4*>(xn + (int64_t)m * H)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  };
#pragma unroll
  for (int it = 0; it < kKeep; it++) {
    const int i = threadIdx.x + it * blockDim.x;
    if (i < n8) scale_store(vk[it], gk[it], i);
  }
  for (int i = threadIdx.x + kKeep * blockDim.x; i < n8; i += blockDim.x)
    scale_store(reinterpret_cast<const uint4*>(row)[i], reinterpret_cast<const uint4*>(gamma)[i], i);
}

cudaError_t launch_rmsnorm(const uint16_t* src, const uint16_t* gamma, int rows, int H, float eps, uint16_t* xn,
                           const int32_t* tokens, const uint16_t* embed, uint16_t* x_out, const int32_t* row_req,
                           const int32_t* req_ok, cudaStream_t s, bool pdl) {
  return launch(k_rmsnorm, dim3(rows), dim3(256), 0, s, pdl, src, gamma, H, eps, xn, tokens, embed, x_out, row_req,
                req_ok);
}

// ------------------------------------------------------------ attention --
// CTA = (split, kv head x row chunk, request).  Query rows of a (request,
// kv head) are its G = Hq/Hkv heads x M nodes (head-major); a row chunk is 64
// rows (4 warps x 16).  Keys of a prefix split are a contiguous range of the
// committed prefix; the last split holds the tree's own keys (slots ctx ..
// ctx+M-1) masked by the row's ancestor bits.  Keys stream through a
// 2-stage ring of 64-key K and V tiles (cp.async, 16-byte XOR swizzle); S =
// Q K^T and O += P V run on mma.m16n8k16 with an online (base-2) softmax in
// fp32.  Many short splits keep the tensor-core latency chains of one warp
// short.  Each split writes its (max, sum, unnormalised O) partial, then the
// splits of a (request, kv head, row chunk) merge them in split order
// (deterministic) into the bf16 output: when the whole grid fits on the GPU
// at once, every split waits (bounded) for its group's partials and merges a
// 1/P share of the rows; otherwise the last split to finish merges them all.
// The group counters return to zero for the next call.

// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32: a few ulp,
// subnormal results flushed to zero); softmax weights of the main loop only
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr int kAttnTile = 64;
constexpr int kAttnStages = 2;
constexpr int kAttnSmem = kAttnStages * 2 * kAttnTile * 128 * 2;  // K and V tiles

int attn_rows_per_group(int hq, int hkv, int max_m) { return (hq / hkv) * max_m; }
int attn_key_split(int rows_per_group) { return rows_per_group <= 32 ? 2 : 1; }
int attn_chunks(int rows_per_group) {
  const int cr = 16 * (4 / attn_key_split(rows_per_group));
  return (rows_per_group + cr - 1) / cr;
}

struct AttnKernelArgs {
  AttnArgs a;
  int rpg;     // row stride of one (request, kv head, split) group in the partial arrays
  int chunks;  // row chunks of 64 per (request, kv head)
  int coop;    // 1: the whole grid is resident, splits merge together
};

// KS = 2 (groups of at most 32 rows, e.g. many requests with short trees):
// the warps pair up on the same 16-row tile and each takes half of every
// 64-key tile, so that all four warps work; a pair merges its two
// online-softmax states in shared memory before the split's partial.
// MINB: CTAs per SM the registers are budgeted for.  KS = 1 needs its 255
// registers (two); KS = 2 holds half the scores per warp and also compiles
// for three without spills, which pays for grids beyond one wave of three
// per SM (16 and 32 requests of 8-row chains: 13.2 -> 12.8 and 19.55 ->
// 19.0 ms per step) but not below (8 requests: 8.80 -> 8.98 ms)
template <int KS, int MINB = 2>
__global__ void __launch_bounds__(128, MINB) k_attn(AttnKernelArgs ka) {
  constexpr int kRowTiles = 4 / KS;       // 16-row tiles per chunk
  constexpr int kChunkRows = 16 * kRowTiles;
  constexpr int kNT = 8 / KS;             // 8-key n-tiles of a warp per 64-key tile
  pdl_launch();  // the next kernel may start streaming its (independent) weights now
  const AttnArgs& a = ka.a;
  const int64_t cta = blockIdx.x + (int64_t)gridDim.x * (blockIdx.y + (int64_t)gridDim.y * blockIdx.z);
  const int64_t ncta = (int64_t)gridDim.x * gridDim.y * gridDim.z;
  auto stamp = [&](int row) {
    if (a.trace && threadIdx.x == 0) a.trace[row * ncta + cta] = globaltimer();
  };
  extern __shared__ __align__(128) uint8_t smem_attn[];
  uint16_t* sK = reinterpret_cast<uint16_t*>(smem_attn);
  uint16_t* sV = sK + kAttnStages * kAttnTile * 128;
  __shared__ int s_last;
  __shared__ int s_pg[64];  // page ids of the split's key range (pages pg0 .. pg0 + npg - 1), read before the wait
  const int sp = blockIdx.x;
  const int h = blockIdx.y % a.hkv, rc = blockIdx.y / a.hkv;
  const int r = blockIdx.z;
  const int G = a.hq / a.hkv;
  // request offsets are host inputs: readable before the wait
  const int node0 = a.cu[r], Mr = a.cu[r + 1] - node0;
  const int rows = G * Mr;
  if (rc * kChunkRows >= rows) {  // no rows: no split of this chunk writes or merges anything
    stamp(0);
    stamp(1);
    stamp(2);
    stamp(3);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int rt = rc * kRowTiles + warp % kRowTiles;
  const int kh = warp / kRowTiles;  // key half of every tile (KS = 2)
  const bool tree = sp == a.splits;
  const int cap = a.max_pages * a.page_size;
  // a prefix split's keys: the committed prefix, which no kernel of the step
  // writes before its commit, located through the host's page table and the
  // context length as passed in; the first key tile is requested before the
  // wait for the previous kernel
  auto prefix_range = [&](int c, int& lo, int& hi) {
    c = c < 0 ? 0 : (c > cap ? cap : c);
    lo = (int)((int64_t)sp * c / a.splits);
    hi = (int)((int64_t)(sp + 1) * c / a.splits);
  };
  int k0 = 0, k1 = 0;
  const int ctx_pre = a.ctx_in[r];
  if (!tree) prefix_range(ctx_pre, k0, k1);
  // the page ids of the split's keys are staged once, before the wait (the
  // tree's own keys, slots ctx .. ctx + M - 1, are written by the q/k/v GEMM,
  // but their page ids are known); a range of more than 64 pages looks its
  // ids up per key
  int pg0 = 0, npg = 0;
  {
    int lo = k0, hi = k1;
    if (tree) {
      lo = ctx_pre < 0 ? 0 : (ctx_pre > cap ? cap : ctx_pre);
      hi = lo + Mr > cap ? cap : lo + Mr;
    }
    if (hi > lo) {
      pg0 = lo / a.page_size;
      npg = (hi - 1) / a.page_size - pg0 + 1;
      if (npg > 64) npg = 0;
    }
    if (threadIdx.x < npg) s_pg[threadIdx.x] = a.page_table[(int64_t)r * a.max_pages + pg0 + threadIdx.x];
    __syncthreads();
  }
  bool has_rows = rt * 16 < rows;
  // this lane's two query rows
  const int rho0 = rt * 16 + g, rho1 = rho0 + 8;
  const bool v0 = rho0 < rows, v1 = rho1 < rows;
  const int n0 = v0 ? rho0 % Mr : 0, n1 = v1 ? rho1 % Mr : 0;
  const int qh0 = h * G + (v0 ? rho0 / Mr : 0), qh1 = h * G + (v1 ? rho1 / Mr : 0);

  const int64_t head_stride = (int64_t)a.page_size * 128;
  auto load_tile = [&](int tile, int buf) {
    const int kb = k0 + tile * kAttnTile;
    for (int c = threadIdx.x; c < kAttnTile * 16; c += 128) {
      const int kr = c >> 4, ch = c & 15;
      const int t = kb + kr;
      bool valid = t < k1;
      int64_t off = 0;
      if (valid) {
        // page ids may be read before the tree kernel validated them
        const int pi = t / a.page_size - pg0;
        const int page = (pi >= 0 && pi < npg) ? s_pg[pi] : a.page_table[(int64_t)r * a.max_pages + t / a.page_size];
        valid = page >= 0 && page < a.n_pages;
        if (valid) off = ((int64_t)page * a.hkv + h) * head_stride + (int64_t)(t % a.page_size) * 128 + ch * 8;
      }
      const int so = (buf * kAttnTile + kr) * 128 + ((ch ^ (kr & 7)) * 8);
      cp_async16_zfill(sK + so, a.k_pool + off, valid);
      cp_async16_zfill(sV + so, a.v_pool + off, valid);
    }
  };
  static_assert(kAttnStages == 2, "one tile is requested ahead of the loop");
  // exactly kAttnStages - 1 groups before the loop and one per iteration, so
  // that waiting for all but the newest kAttnStages - 1 completes the tile
  if (!tree && k1 > k0) load_tile(0, 0);
  cp_async_commit();
  pdl_wait();
  stamp(0);
  // everything the split reads from earlier kernels, requested at once: the
  // context and the request flag (tree kernel), the rows' ancestor masks,
  // the query fragments (q/k/v GEMM)
  const int ctx_now = a.ctx[r], ok_now = a.req_ok[r];
  const uint64_t anc0 = v0 ? a.anc[node0 + n0] : 0ull, anc1 = v1 ? a.anc[node0 + n1] : 0ull;
  uint32_t qa[8][4];
  {
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(a.q + ((int64_t)(node0 + n0) * a.hq + qh0) * 128);
    const uint32_t* q1 = reinterpret_cast<const uint32_t*>(a.q + ((int64_t)(node0 + n1) * a.hq + qh1) * 128);
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
      qa[kk][0] = v0 ? q0[(16 * kk + 2 * q) / 2] : 0u;
      qa[kk][1] = v1 ? q1[(16 * kk + 2 * q) / 2] : 0u;
      qa[kk][2] = v0 ? q0[(16 * kk + 8 + 2 * q) / 2] : 0u;
      qa[kk][3] = v1 ? q1[(16 * kk + 8 + 2 * q) / 2] : 0u;
    }
  }
  {
    const int ctx = ctx_now;
    int lo = 0, hi = 0;
    if (!ok_now) {
      lo = hi = 0;
    } else if (tree) {
      lo = ctx;
      hi = ctx + Mr;
    } else {
      prefix_range(ctx, lo, hi);
    }
    if (lo != k0 || hi != k1 || tree) {
      // the tree split (its keys were just written), or a request whose range
      // differs from the one requested early: start over
      cp_async_wait<0>();
      if (!(tree && ctx == ctx_pre)) npg = 0;  // staged page ids belong to another range
      k0 = lo;
      k1 = hi;
      if (k1 > k0) load_tile(0, 0);
      cp_async_commit();
    }
  }
  const int ntiles = (k1 - k0 + kAttnTile - 1) / kAttnTile;

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const float sl2 = 0.08838834764831845f * 1.4426950408889634f;  // log2(e) / sqrt(128)

  for (int tile = 0; tile < ntiles; tile++) {
    const int buf = tile % kAttnStages;
    if (tile + kAttnStages - 1 < ntiles) load_tile(tile + kAttnStages - 1, (tile + kAttnStages - 1) % kAttnStages);
    cp_async_commit();
    cp_async_wait<kAttnStages - 1>();
    __syncthreads();
    if (has_rows) {
      float s[kNT][4];
#pragma unroll
      for (int i = 0; i < kNT; i++) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
      const uint32_t kb = smem_u32(sK + buf * kAttnTile * 128);
      const int key0 = kh * (kAttnTile / KS);  // this warp's first key of the tile
#pragma unroll
      for (int kk = 0; kk < 8; kk++) {
#pragma unroll
        for (int np = 0; np < kNT / 2; np++) {
          const int key = key0 + np * 16 + (lane >> 4) * 8 + (lane & 7);
          const int ch = 2 * kk + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + key * 256 + ((ch ^ (key & 7)) << 4), b0, b1, b2, b3);
          mma_bf16(s[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
          mma_bf16(s[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
        }
      }
      const int tb = k0 + tile * kAttnTile + key0;
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < kNT; nt++)
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int rr = e >> 1;
          const int t = tb + nt * 8 + 2 * q + (e & 1);
          bool ok = t < k1 && (rr ? v1 : v0);
          if (tree && ok) ok = ((rr ? anc1 : anc0) >> (t - k0)) & 1ull;  // the tree split starts at ctx
          s[nt][e] = ok ? s[nt][e] * sl2 : -INFINITY;
          mx[rr] = fmaxf(mx[rr], s[nt][e]);
        }
      float alpha[2], ms[2], sum[2] = {0.f, 0.f};
#pragma unroll
      for (int rr = 0; rr < 2; rr++) {
        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
        const float mn = fmaxf(mrow[rr], mx[rr]);
        ms[rr] = mn == -INFINITY ? 0.f : mn;
        alpha[rr] = ex2_fast(mrow[rr] - ms[rr]);
        mrow[rr] = mn;
      }
#pragma unroll
      for (int nt = 0; nt < kNT; nt++)
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int rr = e >> 1;
          s[nt][e] = ex2_fast(s[nt][e] - ms[rr]);
          sum[rr] += s[nt][e];
        }
#pragma unroll
      for (int rr = 0; rr < 2; rr++) {
        sum[rr] += __shfl_xor_sync(0xffffffffu, sum[rr], 1);
        sum[rr] += __shfl_xor_sync(0xffffffffu, sum[rr], 2);
        lrow[rr] = lrow[rr] * alpha[rr] + sum[rr];
      }
#pragma unroll
      for (int dn = 0; dn < 16; dn++) {
        o[dn][0] *= alpha[0];
        o[dn][1] *= alpha[0];
        o[dn][2] *= alpha[1];
        o[dn][3] *= alpha[1];
      }
      // P enters the bf16 MMA as two terms, P = hi + lo (hi = bf16(P), lo =
      // bf16(P - hi)): about 16 significant bits, so the product carries the
      // fp32 softmax weights rather than their bf16 rounding (which would
      // move the output by up to half a bf16 unit before its own rounding)
      const uint32_t vb = smem_u32(sV + buf * kAttnTile * 128);
#pragma unroll
      for (int k2 = 0; k2 < kNT / 2; k2++) {
        uint32_t ph[4], pl[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
          const float* sj = s[2 * k2 + (j >> 1)] + 2 * (j & 1);
          ph[j] = pack_bf16x2(sj[0], sj[1]);
          pl[j] = pack_bf16x2(sj[0] - bf2f(ph[j] & 0xFFFFu), sj[1] - bf2f(ph[j] >> 16));
        }
#pragma unroll
        for (int dp = 0; dp < 8; dp++) {
          const int key = key0 + k2 * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
          const int ch = 2 * dp + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + key * 256 + ((ch ^ (key & 7)) << 4), b0, b1, b2, b3);
          mma_bf16(o[2 * dp], ph[0], ph[1], ph[2], ph[3], b0, b1);
          mma_bf16(o[2 * dp + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
          mma_bf16(o[2 * dp], pl[0], pl[1], pl[2], pl[3], b0, b1);
          mma_bf16(o[2 * dp + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  if constexpr (KS == 2) {
    // the second warp of each pair hands its (max, sum, O) to the first
    float* xs = reinterpret_cast<float*>(smem_attn);  // [2 row tiles][32 lanes][68]
    float* mine = xs + ((warp & 1) * 32 + lane) * 68;
    __syncthreads();  // every warp is done with the key tiles
    if (kh == 1 && has_rows) {
#pragma unroll
      for (int dn = 0; dn < 16; dn++)
        *reinterpret_cast<float4*>(mine + 4 * dn) = make_float4(o[dn][0], o[dn][1], o[dn][2], o[dn][3]);
      *reinterpret_cast<float4*>(mine + 64) = make_float4(mrow[0], mrow[1], lrow[0], lrow[1]);
    }
    __syncthreads();
    if (kh == 0 && has_rows) {
      const float4 ml = *reinterpret_cast<const float4*>(mine + 64);
      const float m1[2] = {ml.x, ml.y}, l1[2] = {ml.z, ml.w};
      float a0[2], a1[2];
#pragma unroll
      for (int rr = 0; rr < 2; rr++) {
        const float mn = fmaxf(mrow[rr], m1[rr]);
        a0[rr] = mrow[rr] == -INFINITY ? 0.f : exp2f(mrow[rr] - mn);
        a1[rr] = m1[rr] == -INFINITY ? 0.f : exp2f(m1[rr] - mn);
        lrow[rr] = lrow[rr] * a0[rr] + l1[rr] * a1[rr];
        mrow[rr] = mn;
      }
#pragma unroll
      for (int dn = 0; dn < 16; dn++) {
        const float4 v = *reinterpret_cast<const float4*>(mine + 4 * dn);
        o[dn][0] = o[dn][0] * a0[0] + v.x * a1[0];
        o[dn][1] = o[dn][1] * a0[0] + v.y * a1[0];
        o[dn][2] = o[dn][2] * a0[1] + v.z * a1[1];
        o[dn][3] = o[dn][3] * a0[1] + v.w * a1[1];
      }
    }
    if (kh == 1) has_rows = false;  // the first warp of the pair writes the partial
  }
  stamp(1);

  // this split's partial
  const int64_t gbase = (int64_t)(r * a.hkv + h) * (a.splits + 1);
  if (has_rows) {
#pragma unroll
    for (int rr = 0; rr < 2; rr++) {
      const int rho = rr ? rho1 : rho0;
      if (rho >= rows) continue;
      const int64_t b = (gbase + sp) * ka.rpg + rho;
      if (q == 0) {
        __stcg(a.part_ml + b * 2, mrow[rr]);
        __stcg(a.part_ml + b * 2 + 1, lrow[rr]);
      }
      float* dst = a.part_o + b * 128;
#pragma unroll
      for (int dn = 0; dn < 16; dn++)
        __stcg(reinterpret_cast<float2*>(dst + dn * 8 + 2 * q), make_float2(o[dn][2 * rr], o[dn][2 * rr + 1]));
    }
  }
  // group counters: [0] splits that wrote their partial, [1] splits done merging
  const int P = a.splits + 1;
  int32_t* gc = a.tickets + (((int64_t)r * a.hkv + h) * ka.chunks + rc) * 2;
  __syncthreads();
  if (threadIdx.x == 0) {
    if (ka.coop) {
      // a release add (this CTA's partial, ordered before it by the
      // barrier, becomes visible with it; no value comes back), then wait
      // (bounded) for the group's other splits
      asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(gc) : "memory");
      int v = 0;
      const uint64_t t0 = globaltimer();
      while (v < P) {
        if (globaltimer() - t0 > kWaitLimitNs) {
          set_status(a.status, SD_TIMEOUT_AT(20));
          break;
        }
        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(gc) : "memory");
      }
      s_last = 1;
    } else {
      __threadfence();
      const int old = atomicAdd(gc, 1);
      s_last = old == P - 1;
      if (s_last) *gc = 0;
      __threadfence();
    }
  }
  __syncthreads();
  stamp(2);
  if (!s_last) {
    stamp(3);
    return;
  }
  // rows merged by this CTA
  const int rbeg0 = rc * kChunkRows, nrow0 = min(rows, rbeg0 + kChunkRows) - rbeg0;
  const int rbeg = ka.coop ? rbeg0 + sp * nrow0 / P : rbeg0;
  const int nrow = ka.coop ? rbeg0 + (sp + 1) * nrow0 / P - rbeg : nrow0;
  // merge: every (row, split) (max, sum) pair into shared memory with all
  // loads in flight, then per row the split weights 2^(m_p - max) / L; then
  // each thread forms 4-wide slices of the output with its partial loads
  // batched
  constexpr int kMaxParts = 65;
  float* wsm = reinterpret_cast<float*>(smem_attn);                // [64 rows][kMaxParts] weights
  float2* mlsm = reinterpret_cast<float2*>(wsm + 64 * kMaxParts);  // [64 rows][kMaxParts] (max, sum)
  for (int e = threadIdx.x; e < nrow * P; e += 128) {
    const int i = e / P, p = e - i * P;
    mlsm[i * kMaxParts + p] = __ldcg(reinterpret_cast<const float2*>(a.part_ml + ((gbase + p) * ka.rpg + rbeg + i) * 2));
  }
  __syncthreads();
  if (P <= 16) {
    // few splits (many requests): one thread per row
    for (int i = threadIdx.x; i < nrow; i += 128) {
      const float2* ml = mlsm + i * kMaxParts;
      float mx = -INFINITY;
      for (int p = 0; p < P; p++) mx = fmaxf(mx, ml[p].x);
      float L = 0.f;
      for (int p = 0; p < P; p++) {
        const float w = ml[p].x == -INFINITY ? 0.f : exp2f(ml[p].x - mx);
        wsm[i * kMaxParts + p] = w;
        L += w * ml[p].y;
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      for (int p = 0; p < P; p++) wsm[i * kMaxParts + p] *= inv;
    }
  } else {
    // many splits: one warp per row, lanes over the splits (butterfly
    // reductions: a fixed order, deterministic)
    const int wp = threadIdx.x >> 5, ln = threadIdx.x & 31;
    for (int i = wp; i < nrow; i += 4) {
      const float2* ml = mlsm + i * kMaxParts;
      float mx = -INFINITY;
      for (int p = ln; p < P; p += 32) mx = fmaxf(mx, ml[p].x);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      float L = 0.f;
      for (int p = ln; p < P; p += 32) {
        const float w = ml[p].x == -INFINITY ? 0.f : exp2f(ml[p].x - mx);
        wsm[i * kMaxParts + p] = w;
        L += w * ml[p].y;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
      const float inv = L > 0.f ? 1.f / L : 0.f;
      for (int p = ln; p < P; p += 32) wsm[i * kMaxParts + p] *= inv;
    }
  }
  __syncthreads();
  // slice = (row, 4 dims): 32 slices per row.  With few rows per CTA (the
  // cooperative merge) the splits of a slice are dealt to nsub adjacent
  // threads (split p to thread p % nsub), so that every thread's loads are in
  // flight at once; the nsub partial sums are added with shuffles in a fixed
  // order (deterministic).  Loads go 16 splits at a time.
  const int nsub = nrow * 32 * 4 <= 128 ? 4 : nrow * 32 * 2 <= 128 ? 2 : 1;
  const int nslices = nrow * 32;
  for (int t0 = 0; t0 < nslices * nsub; t0 += 128) {
    const int t = t0 + threadIdx.x;
    const int sl = t / nsub, sub = t % nsub;
    const bool live = sl < nslices;
    const int i = live ? sl >> 5 : 0, d4 = sl & 31;
    const float4* src = reinterpret_cast<const float4*>(a.part_o + (gbase * ka.rpg + rbeg + i) * 128) + d4;
    const int64_t pstride = (int64_t)ka.rpg * 32;  // float4 per split
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = sub; p0 < P; p0 += 16 * nsub) {
      float4 v[16];
#pragma unroll
      for (int u = 0; u < 16; u++) {
        const int pp = p0 + u * nsub;
        v[u] = live && pp < P ? __ldcg(src + pp * pstride) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 16; u++) {
        const int pp = p0 + u * nsub;
        const float w = live && pp < P ? wsm[i * kMaxParts + pp] : 0.f;
        acc.x = fmaf(w, v[u].x, acc.x);
        acc.y = fmaf(w, v[u].y, acc.y);
        acc.z = fmaf(w, v[u].z, acc.z);
        acc.w = fmaf(w, v[u].w, acc.w);
      }
    }
    // adjacent lanes hold the nsub shares of one slice (nsub divides 32)
    for (int off = 1; off < nsub; off <<= 1) {
      acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
      acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
      acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
      acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
    }
    if (live && sub == 0) {
      const int rho = rbeg + i;
      const int node = rho % Mr, qh = h * G + rho / Mr;
      uint2 o2;
      o2.x = pack_bf16x2(acc.x, acc.y);
      o2.y = pack_bf16x2(acc.z, acc.w);
      *reinterpret_cast<uint2*>(a.out + (int64_t)(node0 + node) * a.hq * 128 + qh * 128 + d4 * 4) = o2;
    }
  }
  if (ka.coop) {
    // the last split to finish merging resets the group's counters (every
    // split has passed its wait by then)
    __syncthreads();
    if (threadIdx.x == 0 && atomicAdd(gc + 1, 1) == P - 1) {
      gc[0] = 0;
      gc[1] = 0;
    }
  }
  __syncthreads();
  stamp(3);
}

// Device-clock stamps of attention launches (diagnostics; sd_attn_set_trace):
// each launch while a buffer is set takes the next 4 x grid stamps.
static std::mutex g_attn_trace_mu;
static uint64_t* g_attn_trace = nullptr;
static size_t g_attn_trace_cap = 0, g_attn_trace_used = 0;

int attn_set_trace(uint64_t* buf, size_t n) {
  std::lock_guard<std::mutex> lock(g_attn_trace_mu);
  g_attn_trace = buf;
  g_attn_trace_cap = buf ? n : 0;
  g_attn_trace_used = 0;
  return SD_OK;
}

cudaError_t launch_attention(const AttnArgs& a_in, int rows_total, cudaStream_t s, bool pdl) {
  (void)rows_total;
  AttnArgs a = a_in;
  static bool attr = false;
  static int per_sm[3] = {-1, -1, -1};  // k_attn<1>, k_attn<2>, k_attn<2, 3>
  if (!attr) {
    for (auto kern : {k_attn<1>, k_attn<2>, k_attn<2, 3>}) {
      const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
      if (e != cudaSuccess) return e;
      carveout_once(reinterpret_cast<const void*>(kern));
    }
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm[0], k_attn<1>, 128, kAttnSmem) != cudaSuccess) per_sm[0] = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm[1], k_attn<2>, 128, kAttnSmem) != cudaSuccess) per_sm[1] = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm[2], k_attn<2, 3>, 128, kAttnSmem) != cudaSuccess)
      per_sm[2] = 0;
    attr = true;
  }
  const int rpg = attn_rows_per_group(a.hq, a.hkv, a.max_m);
  const int cm = attn_rows_per_group(a.hq, a.hkv, a.chunk_m > 0 ? a.chunk_m : a.max_m);
  const int ks = attn_key_split(cm);
  const int chunks = attn_chunks(cm);
  const int64_t grid = (int64_t)(a.splits + 1) * a.hkv * chunks * a.R;
  {
    std::lock_guard<std::mutex> lock(g_attn_trace_mu);
    if (g_attn_trace && g_attn_trace_used + 4 * (size_t)grid <= g_attn_trace_cap) {
      a.trace = g_attn_trace + g_attn_trace_used;
      g_attn_trace_used += 4 * (size_t)grid;
    }
  }
  // the key-split kernel budgeted for three CTAs per SM once the grid is
  // more than one wave of three
  const int var = ks == 1 ? 0 : (per_sm[2] >= 3 && grid > (int64_t)per_sm[2] * num_sms()) ? 2 : 1;
  const AttnKernelArgs ka{a, rpg, chunks, grid <= (int64_t)per_sm[var] * num_sms() ? 1 : 0};
  const dim3 g3(a.splits + 1, a.hkv * chunks, a.R);
  if (var == 0) return launch(k_attn<1>, g3, dim3(128), kAttnSmem, s, pdl, ka);
  if (var == 1) return launch(k_attn<2>, g3, dim3(128), kAttnSmem, s, pdl, ka);
  return launch(k_attn<2, 3>, g3, dim3(128), kAttnSmem, s, pdl, ka);
}

// ------------------------------------------------- linear recurrence -----
// CTA = (value-dim chunk of 32, head, request).  Closed form of the tree
// recurrence: S_i = S0 + sum_{j in path(i)} phi(k_j) v_j^T gives
//   o_i = (S0^T phi(q_i) + sum_j (phi(k_j).phi(q_i)) v_j) / (z0.phi(q_i) + sum_j phi(k_j).phi(q_i) + eps)
// so the per-node states are never materialised.

__device__ __forceinline__ float phi(float x) { return x > 0.f ? x + 1.0f : expf(x); }

// phi(q), phi(k) rows padded to 129 floats: the tree dot products read
// element d of many rows at once, which a 128-float stride puts in one bank
constexpr int kRecFS = 129;
// 16 warps: the output phase's per-thread chains (128 + tree terms each) are
// its critical path at one CTA per (32 value columns, head, request); at 16
// nodes every thread then owns one output (hybrid step, 24 recurrent layers:
// 0.432 / 0.343 / 0.328 ms of recurrence at 4 / 8 / 16 warps)
constexpr int kRecThreads = 512;
constexpr int kSIt = 128 * 32 / kRecThreads;  // state-tile elements per thread
constexpr int kRecSmem = (64 * kRecFS * 2 + 128 * 32 + 64 * 32 + 128 + 64 * 64 + 64) * 4 + 64 * 8;

__global__ void __launch_bounds__(kRecThreads) k_linrec(LinrecArgs a) {
  pdl_launch();  // the next kernel may start streaming its (independent) weights now
  pdl_wait();
  extern __shared__ __align__(16) float smem_rec[];
  float* fq = smem_rec;          // [64][kRecFS]
  float* fk = fq + 64 * kRecFS;  // [64][kRecFS]
  float* sS = fk + 64 * kRecFS;  // [128][32]
  float* sv = sS + 128 * 32;  // [64][32]
  float* sz = sv + 64 * 32;   // [128]
  float* dots = sz + 128;     // [64][64]
  float* zq = dots + 64 * 64; // [64]
  const int cc = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
  uint64_t* sanc = reinterpret_cast<uint64_t*>(zq + 64);  // [64] ancestor masks
  const int node0 = a.cu[r], Mr = min(a.cu[r + 1] - node0, 64);
  const int64_t H3 = (int64_t)a.H * 3;
  // staging: every thread's global loads of a batch are in flight before
  // any is stored (a load-store loop waits one L2 round trip per element)
  constexpr int kB = 8;
  for (int base = 0; base < Mr * 128; base += kB * kRecThreads) {
    uint16_t lq[kB], lk[kB];
#pragma unroll
    for (int u = 0; u < kB; u++) {
      const int idx = base + u * kRecThreads + threadIdx.x;
      const int i = idx >> 7, d = idx & 127;
      const uint16_t* row = a.qkv + (int64_t)(node0 + i) * H3;
      lq[u] = idx < Mr * 128 ? row[h * 128 + d] : (uint16_t)0;
      lk[u] = idx < Mr * 128 ? row[a.H + h * 128 + d] : (uint16_t)0;
    }
#pragma unroll
    for (int u = 0; u < kB; u++) {
      const int idx = base + u * kRecThreads + threadIdx.x;
      if (idx >= Mr * 128) break;
      const int i = idx >> 7, d = idx & 127;
      fq[i * kRecFS + d] = phi(bf2f(lq[u]));
      fk[i * kRecFS + d] = phi(bf2f(lk[u]));
    }
  }
  for (int base = 0; base < Mr * 32; base += kB * kRecThreads) {
    uint16_t lv[kB];
#pragma unroll
    for (int u = 0; u < kB; u++) {
      const int idx = base + u * kRecThreads + threadIdx.x;
      const int i = idx >> 5, c = idx & 31;
      lv[u] = idx < Mr * 32 ? a.qkv[(int64_t)(node0 + i) * H3 + 2 * a.H + h * 128 + cc * 32 + c] : (uint16_t)0;
    }
#pragma unroll
    for (int u = 0; u < kB; u++) {
      const int idx = base + u * kRecThreads + threadIdx.x;
      if (idx >= Mr * 32) break;
      sv[(idx >> 5) * 32 + (idx & 31)] = bf2f(lv[u]);
    }
  }
  const float* Sg = a.S + r * a.req_stride_S + (int64_t)h * 128 * 128;
  const float* zg = a.z + r * a.req_stride_z + (int64_t)h * 128;
  for (int base = 0; base < 128 * 32; base += kSIt * kRecThreads) {
    float ls[kSIt];
#pragma unroll
    for (int u = 0; u < kSIt; u++) {
      const int idx = base + u * kRecThreads + threadIdx.x;
      ls[u] = Sg[(idx >> 5) * 128 + cc * 32 + (idx & 31)];
    }
#pragma unroll
    for (int u = 0; u < kSIt; u++) sS[base + u * kRecThreads + threadIdx.x] = ls[u];
  }
  for (int k = threadIdx.x; k < 128; k += blockDim.x) sz[k] = zg[k];
  for (int i = threadIdx.x; i < Mr; i += blockDim.x) sanc[i] = a.anc[node0 + i];
  __syncthreads();
  for (int idx = threadIdx.x; idx < Mr * Mr; idx += blockDim.x) {
    const int i = idx / Mr, j = idx % Mr;
    float dt = 0.f;
    if ((sanc[i] >> j) & 1ull) {
      for (int d = 0; d < 128; d++) dt = fmaf(fk[j * kRecFS + d], fq[i * kRecFS + d], dt);
    }
    dots[i * 64 + j] = dt;
  }
  for (int i = threadIdx.x; i < Mr; i += blockDim.x) {
    float t = 0.f;
    for (int d = 0; d < 128; d++) t = fmaf(sz[d], fq[i * kRecFS + d], t);
    zq[i] = t;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < Mr * 32; idx += blockDim.x) {
    const int i = idx >> 5, c = idx & 31;
    float num = 0.f;
    for (int k = 0; k < 128; k++) num = fmaf(fq[i * kRecFS + k], sS[k * 32 + c], num);
    float den = zq[i];
    for (int j = 0; j < Mr; j++) {
      const float w = dots[i * 64 + j];
      num = fmaf(w, sv[j * 32 + c], num);
      den += w;
    }
    a.out[(int64_t)(node0 + i) * a.H + h * 128 + cc * 32 + c] = f2bf(num / (den + a.eps));
  }
}

cudaError_t launch_linrec(const LinrecArgs& a, cudaStream_t s, bool pdl) {
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(k_linrec, cudaFuncAttributeMaxDynamicSharedMemorySize, kRecSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch(k_linrec, dim3(4, a.nh, a.R), dim3(kRecThreads), kRecSmem, s, pdl, a);
}

// --------------------------------------------------- argmax + accept -----

__global__ void __launch_bounds__(512) k_accept(AcceptArgs a) {
  pdl_launch();  // the next kernel may start streaming its (independent) weights now
  pdl_wait();
  __shared__ int am[64], par[64], dep[64], okn[64], pth[65];
  const int r = blockIdx.x;
  const int node0 = a.cu ? a.cu[r] : 0, Mr = a.cu ? a.cu[r + 1] - node0 : a.single_M;
  const int i = threadIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // per node: the argmax over the GEMM's per-CTA partials, one warp per node
  // with the lanes over the partials (larger value, then smaller index: a
  // total order, so the reduction order does not matter)
  for (int n = warp; n < Mr && n < 64; n += 16) {
    int best;
    if (a.amax_val) {
      float v = -INFINITY;
      best = 0x7FFFFFFF;
      for (int c = lane; c < a.n_part; c += 32) {
        const float ov = a.amax_val[(int64_t)c * a.ld + node0 + n];
        const int oi = a.amax_idx[(int64_t)c * a.ld + node0 + n];
        if (ov > v || (ov == v && oi < best)) {
          v = ov;
          best = oi;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, off);
        const int oi = __shfl_xor_sync(0xffffffffu, best, off);
        if (ov > v || (ov == v && oi < best)) {
          v = ov;
          best = oi;
        }
      }
    } else {
      best = a.argmax_in[node0 + n];
    }
    if (lane == 0) {
      am[n] = best;
      if (a.argmax_out) a.argmax_out[node0 + n] = best;
    }
  }
  if (i < Mr && i < 64) par[i] = a.parents[node0 + i];
  __syncthreads();
  if (i != 0) return;
  bool valid = Mr >= 1 && Mr <= 64 && (a.req_ok ? a.req_ok[r] != 0 : true);
  for (int j = 0; j < Mr && j < 64 && valid; j++)
    if (j == 0 ? par[0] != -1 : (par[j] < 0 || par[j] >= j)) valid = false;
  if (!valid) {
    if (!a.req_ok) set_status(a.status, SD_ERR_BAD_TREE);
    a.accepted_len[r] = 0;
    a.bonus[r] = -1;
    if (a.path_len) a.path_len[r] = 0;
    return;
  }
  dep[0] = 0;
  okn[0] = 1;
  int best = 0;
  for (int j = 1; j < Mr; j++) {
    dep[j] = dep[par[j]] + 1;
    okn[j] = okn[par[j]] && a.tokens[node0 + j] == am[par[j]];
    if (okn[j] && dep[j] > dep[best]) best = j;
  }
  const int L = dep[best];
  for (int d = L, j = best; d >= 0; d--, j = par[j]) pth[d] = j;
  a.accepted_len[r] = L;
  a.bonus[r] = am[best];
  for (int d = 1; d <= L; d++) a.accepted_tokens[node0 + d - 1] = a.tokens[node0 + pth[d]];
  if (a.path)
    for (int d = 0; d <= L; d++) a.path[r * 65 + d] = pth[d];
  if (a.path_len) a.path_len[r] = L + 1;
  if (a.ctx_len) a.ctx_len[r] = a.ctx_snap[r] + L + 1;
}

cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s, bool pdl) {
  return launch(k_accept, dim3(a.R), dim3(512), 0, s, pdl, a);
}

// ------------------------------------------------------------- commit ----
// K/V of the root and the accepted nodes move from slot ctx + node to slot
// ctx + depth.  A destination can be another path node's source, so every
// row is read into shared memory before any is written.

__global__ void __launch_bounds__(128) k_compact(CacheView cv, int hkv, const int32_t* __restrict__ ctx_snap,
                                                 const int32_t* __restrict__ path,
                                                 const int32_t* __restrict__ path_len) {
  pdl_launch();  // the next kernel may start streaming its (independent) weights now
  pdl_wait();
  __shared__ uint4 bk[65][16], bv[65][16];
  const int r = blockIdx.x, la = blockIdx.y, h = blockIdx.z;
  const int P = path_len[r];
  if (P <= 0) return;
  const int ctx = ctx_snap[r];
  const int64_t layer = (int64_t)la * cv.n_pages * hkv * cv.page_size * 128;
  auto at = [&](int t) -> int64_t {
    const int page = cv.page_table[(int64_t)r * cv.max_pages + t / cv.page_size];
    return layer + ((int64_t)page * hkv + h) * cv.page_size * 128 + (int64_t)(t % cv.page_size) * 128;
  };
  for (int idx = threadIdx.x; idx < P * 16; idx += blockDim.x) {
    const int d = idx >> 4, ch = idx & 15;
    const int64_t src = at(ctx + path[r * 65 + d]);
    bk[d][ch] = reinterpret_cast<const uint4*>(cv.k_pool + src)[ch];
    bv[d][ch] = reinterpret_cast<const uint4*>(cv.v_pool + src)[ch];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < P * 16; idx += blockDim.x) {
    const int d = idx >> 4, ch = idx & 15;
    const int64_t dst = at(ctx + d);
    reinterpret_cast<uint4*>(cv.k_pool + dst)[ch] = bk[d][ch];
    reinterpret_cast<uint4*>(cv.v_pool + dst)[ch] = bv[d][ch];
  }
}

cudaError_t launch_compact(const CacheView& cv, int n_attn_layers, int hkv, int R, const int32_t* ctx_snap,
                           const int32_t* path, const int32_t* path_len, cudaStream_t s, bool pdl) {
  return launch(k_compact, dim3(R, n_attn_layers, hkv), dim3(128), 0, s, pdl, cv, hkv, ctx_snap, path, path_len);
}

// Recurrent state after acceptance: S0 += sum_{path} phi(k) v^T, z0 += sum phi(k).
__global__ void __launch_bounds__(128) k_rec_commit(CacheView cv, int n_rec, int nh, int H, int max_rows,
                                                    const uint16_t* __restrict__ qkv_rec,
                                                    const int32_t* __restrict__ cu, const int32_t* __restrict__ path,
                                                    const int32_t* __restrict__ path_len) {
  pdl_launch();  // the next kernel may start streaming its (independent) weights now
  pdl_wait();
  __shared__ float fk[65][128];
  __shared__ float vv[65][32];
  const int r = blockIdx.x / n_rec, lr = blockIdx.x % n_rec, h = blockIdx.y, cc = blockIdx.z;
  const int P = path_len[r];
  if (P <= 0) return;
  const int64_t H3 = (int64_t)H * 3;
  const uint16_t* base = qkv_rec + (int64_t)lr * max_rows * H3;
  for (int idx = threadIdx.x; idx < P * 128; idx += blockDim.x) {
    const int p = idx >> 7, d = idx & 127;
    const int row = cu[r] + path[r * 65 + p];
    fk[p][d] = phi(bf2f(base[(int64_t)row * H3 + H + h * 128 + d]));
  }
  for (int idx = threadIdx.x; idx < P * 32; idx += blockDim.x) {
    const int p = idx >> 5, c = idx & 31;
    const int row = cu[r] + path[r * 65 + p];
    vv[p][c] = bf2f(base[(int64_t)row * H3 + 2 * H + h * 128 + cc * 32 + c]);
  }
  __syncthreads();
  float* S = cv.S + (((int64_t)r * n_rec + lr) * nh + h) * 128 * 128;
  float* z = cv.z + (((int64_t)r * n_rec + lr) * nh + h) * 128;
  // lanes over the chunk's 32 columns (one 128-byte row segment per warp
  // access), warps over the rows, 8 rows' loads in flight at a time
  const int warp = threadIdx.x >> 5, c = threadIdx.x & 31;
  constexpr int kRows = 8;
  for (int k0 = warp * kRows; k0 < 128; k0 += 4 * kRows) {
    float cur[kRows];
#pragma unroll
    for (int u = 0; u < kRows; u++) cur[u] = S[(k0 + u) * 128 + cc * 32 + c];
#pragma unroll
    for (int u = 0; u < kRows; u++) {
      float add = 0.f;
      for (int p = 0; p < P; p++) add = fmaf(fk[p][k0 + u], vv[p][c], add);
      S[(k0 + u) * 128 + cc * 32 + c] = cur[u] + add;
    }
  }
  if (cc == 0) {
    const int k = threadIdx.x;
    float add = 0.f;
    for (int p = 0; p < P; p++) add += fk[p][k];
    z[k] += add;
  }
}

cudaError_t launch_rec_commit(const CacheView& cv, int n_rec, int nh, int H, int R, int max_rows,
                              const uint16_t* qkv_rec, const int32_t* cu, const int32_t* path,
                              const int32_t* path_len, cudaStream_t s, bool pdl) {
  return launch(k_rec_commit, dim3(R * n_rec, nh, 4), dim3(128), 0, s, pdl, cv, n_rec, nh, H, max_rows, qkv_rec, cu,
                path, path_len);
}

// Busy-waits for `ns` nanoseconds of %globaltimer (bounded by construction).
// The per-kernel timing mode puts it in front of a step so that the host can
// enqueue the whole step while the GPU is still busy: the step's kernels then
// run back to back and the events around them measure GPU time only.
__global__ void k_delay(uint64_t ns) {
  const uint64_t t0 = globaltimer();
  while (globaltimer() - t0 < ns) {
  }
}

cudaError_t launch_delay(uint64_t ns, cudaStream_t s) { return launch(k_delay, dim3(1), dim3(1), 0, s, false, ns); }

}  // namespace sdv

extern "C" int sd_attn_set_trace(uint64_t* buf, int64_t bytes) {
  if (bytes < 0) {
    sdv::set_error("sd_attn_set_trace: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  return sdv::attn_set_trace(bytes > 0 ? buf : nullptr, (size_t)bytes / 8);
}
