// Best-first node selection under a shared node budget: turns the drafted
// candidate trees of a batch into the node lists one batched verify checks
// ("SpecPilot: AI Agent Framework Boosts Speculative Decoding 10.87x",
// "(2) Best-first Tree Verification for Hybrid Architectures": candidates
// ranked by parent-conditioned log-probability, the highest cumulative path
// scores kept; "(4) Three Batch Optimization Mechanisms", Shared Node Budget:
// the requests share one node budget, given to the candidates of highest
// path probability).
//
// The selection: every request keeps its root; the other candidates are
// taken in order of path score, highest first (equal scores: lower request,
// then lower node index), passing over a candidate whose request holds
// `cap` nodes, until `budget` nodes are held.  Taken in that order with a
// per-request cap, the kept set is exactly the first `budget` candidates
// (in the same order) among those ranked below `cap` within their request.
// Two launches compute that:
//  k_sel_keys (one CTA per request): validates the request, computes the
//   path scores level by level (each node adds its log-probability to its
//   parent's score: the fp32 additions of the recursive definition, in its
//   order), forms each candidate's 64-bit order key (roots first, then
//   score descending, then global index; unique, integer order = taking
//   order) and drops the candidates ranked cap or worse in their request.
//  k_sel_pick (one CTA): the budget-th smallest remaining key by an 8-pass
//   radix select, then an exclusive scan that places the kept candidates per
//   request in index order, parents renumbered, tokens and scores gathered.

#include <cstdint>

#include "common.cuh"
#include "sdv.h"

namespace sdv {
namespace {

constexpr int kSelMaxNodes = 2048;   // candidates per request
constexpr int kSelMaxTotal = 16384;  // candidates per call
constexpr int kKeyThreads = 256;
constexpr int kPickThreads = 1024;
constexpr int kPerThread = kSelMaxTotal / kPickThreads;  // keys a k_sel_pick thread holds
constexpr uint64_t kNoKey = ~0ull;                       // dropped / invalid candidate

// Order key of candidate i (global index g) with path score s: smaller key =
// taken earlier.  Roots: g (bit 63 clear).  Others: bit 63 set, then the
// score mapped to an unsigned integer that falls as the score rises, then g.
__device__ __forceinline__ uint64_t order_key(int i, float s, int g) {
  if (i == 0) return (uint64_t)g;
  const float z = (s == 0.f) ? 0.f : s;  // -0 ranks as +0
  const uint32_t u = __float_as_uint(z);
  const uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // unsigned order = float order
  return (1ull << 63) | ((uint64_t)(~asc) << 31) | (uint64_t)g;
}

__global__ void __launch_bounds__(kKeyThreads) k_sel_keys(const int32_t* __restrict__ parents,
                                                          const float* __restrict__ logprob,
                                                          const int32_t* __restrict__ cu, int n_total, int cap,
                                                          uint64_t* __restrict__ ekey, float* __restrict__ score,
                                                          int32_t* __restrict__ req, int32_t* status) {
  pdl_launch();  // the pick kernel waits for this grid to finish before it reads
  __shared__ float s[kSelMaxNodes];
  __shared__ float lp[kSelMaxNodes];
  __shared__ int par[kSelMaxNodes];
  __shared__ int16_t lvl[kSelMaxNodes];
  __shared__ uint64_t key[kSelMaxNodes];
  const int r = blockIdx.x;
  const int c0 = cu[r], c1 = cu[r + 1];
  const int n = c1 - c0;
  if (c0 < 0 || c1 > n_total || n < 1 || n > kSelMaxNodes) {
    if (threadIdx.x == 0) set_status(status, SD_ERR_BAD_TREE);
    return;  // the request's slots keep the no-key fill
  }
  int bad = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int p = parents[c0 + i];
    const float l = logprob[c0 + i];
    par[i] = p;
    lp[i] = l;
    lvl[i] = (int16_t)(i == 0 ? 0 : -1);
    if (i == 0) {
      s[0] = 0.f;
      bad |= p != -1;
    } else {
      bad |= !(p >= 0 && p < i && l <= 0.f);  // NaN fails the comparison
    }
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) set_status(status, SD_ERR_BAD_TREE);
    return;
  }
  // round t scores the nodes whose parent was scored in an earlier round
  // (lvl < t); a valid tree needs depth + 1 <= n rounds
  for (int t = 1; t <= n; t++) {
    int changed = 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      if (lvl[i] < 0) {
        const int p = par[i];
        const int lp_lvl = lvl[p];
        if (lp_lvl >= 0 && lp_lvl < t) {
          s[i] = __fadd_rn(s[p], lp[i]);
          lvl[i] = (int16_t)t;
          changed = 1;
        }
      }
    }
    if (!__syncthreads_or(changed)) break;
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x) key[i] = order_key(i, s[i], c0 + i);
  __syncthreads();
  const bool capped = cap < n;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint64_t k = key[i];
    bool keep = true;
    if (capped) {
      int rank = 0;
      for (int j = 0; j < n; j++) rank += key[j] < k;
      keep = rank < cap;
    }
    ekey[c0 + i] = keep ? k : kNoKey;
    score[c0 + i] = s[i];
    req[c0 + i] = r;
  }
}

__device__ __forceinline__ int block_excl_scan(int v, int* wsum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = (int)(blockDim.x >> 5);
    int w = lane < nw ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    if (lane < nw) wsum[lane] = w;  // inclusive per warp
  }
  __syncthreads();
  total = wsum[(blockDim.x >> 5) - 1];
  const int before = warp ? wsum[warp - 1] : 0;
  __syncthreads();  // wsum is reused by the caller's next scan
  return before + inc - v;
}

__global__ void __launch_bounds__(kPickThreads) k_sel_pick(
    const uint64_t* __restrict__ ekey, const float* __restrict__ score, const int32_t* __restrict__ req,
    const int32_t* __restrict__ cu, const int32_t* __restrict__ parents, const int32_t* __restrict__ tokens,
    int R, int n_total, int budget, int32_t* __restrict__ pos, int32_t* __restrict__ out_cu,
    int32_t* __restrict__ out_src, int32_t* __restrict__ out_parents, int32_t* __restrict__ out_tokens,
    float* __restrict__ out_score, int32_t* status) {
  pdl_wait();
  __shared__ int hist[256];
  __shared__ int wsum[32];
  __shared__ uint64_t s_prefix;
  __shared__ int s_k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // cu must split [0, n_total) into consecutive requests
  int badl = (tid == 0) ? (cu[0] != 0 || cu[R] != n_total) : 0;
  for (int r = tid; r < R; r += blockDim.x) badl |= cu[r + 1] < cu[r];
  if (__syncthreads_or(badl)) {
    if (tid == 0) set_status(status, SD_ERR_BAD_TREE);
    for (int r = tid; r <= R; r += blockDim.x) out_cu[r] = 0;
    return;
  }
  // this thread's candidates: [lo, lo + per)
  const int per = (n_total + kPickThreads - 1) / kPickThreads;
  const int lo = tid * per;
  uint64_t k[kPerThread];
  int n_keep = 0;
#pragma unroll
  for (int it = 0; it < kPerThread; it++) {
    const int g = lo + it;
    k[it] = (it < per && g < n_total) ? ekey[g] : kNoKey;
    n_keep += k[it] != kNoKey;
  }
  int E;
  block_excl_scan(n_keep, wsum, E);
  uint64_t T = kNoKey;  // keep the keys <= T
  if (E > budget) {
    // the budget-th smallest key (keys are unique), 8 bits per pass from the top
    uint64_t prefix = 0, mask = 0;
    int kk = budget;
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int b = tid; b < 256; b += blockDim.x) hist[b] = 0;
      __syncthreads();
#pragma unroll
      for (int it = 0; it < kPerThread; it++) {
        const bool m = k[it] != kNoKey && (k[it] & mask) == prefix;
        const int bin = m ? (int)((k[it] >> shift) & 255) : 256;
        const unsigned grp = __match_any_sync(0xffffffffu, bin);
        if (bin < 256 && lane == __ffs(grp) - 1) atomicAdd(&hist[bin], __popc(grp));
      }
      __syncthreads();
      if (warp == 0) {
        int c[8], tot = 0;
#pragma unroll
        for (int j = 0; j < 8; j++) {
          c[j] = hist[8 * lane + j];
          tot += c[j];
        }
        int inc = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += u;
        }
        const int before = inc - tot;
        if (before < kk && kk <= inc) {
          int acc = before, d = 7;
#pragma unroll
          for (int j = 0; j < 8; j++) {
            if (acc + c[j] >= kk) {
              d = j;
              break;
            }
            acc += c[j];
          }
          s_prefix = prefix | ((uint64_t)(8 * lane + d) << shift);
          s_k = kk - acc;
        }
      }
      __syncthreads();
      prefix = s_prefix;
      kk = s_k;
      mask |= 0xFFull << shift;
    }
    T = prefix;
  }
  // positions: exclusive count of kept candidates before each one; pos[g]
  // holds it for kept candidates and its complement for the others
  unsigned keep = 0;
  int cnt = 0;
#pragma unroll
  for (int it = 0; it < kPerThread; it++)
    if (k[it] != kNoKey && k[it] <= T) {
      keep |= 1u << it;
      cnt++;
    }
  int total;
  const int excl = block_excl_scan(cnt, wsum, total);
  {
    int run = excl;
#pragma unroll
    for (int it = 0; it < kPerThread; it++) {
      const int g = lo + it;
      if (it < per && g < n_total) pos[g] = ((keep >> it) & 1) ? run++ : ~run;
    }
  }
  __syncthreads();  // pos of every candidate visible to the block
  for (int r = tid; r <= R; r += blockDim.x) {
    const int c = cu[r];
    int v = total;
    if (c < n_total) {
      const int pc = pos[c];
      v = pc >= 0 ? pc : ~pc;
    }
    out_cu[r] = v;
  }
  int run = excl;
#pragma unroll
  for (int it = 0; it < kPerThread; it++) {
    if (!((keep >> it) & 1)) continue;
    const int g = lo + it;
    const int p = run++;
    out_src[p] = g;
    const int r = req[g];
    int op = -1;
    if (r >= 0 && r < R) {
      const int a = cu[r];
      if (g != a) {
        const int pg = a + parents[g];  // 0 <= parent < g - a: checked by k_sel_keys
        const int pp = (pg >= a && pg < g) ? pos[pg] : -1;
        const int base = pos[a];
        if (pp >= 0 && base >= 0) {
          op = pp - base;
        } else {
          set_status(status, SD_ERR_BAD_TREE);  // unreachable for valid input: a kept node's parent is kept
        }
      }
    } else {
      set_status(status, SD_ERR_BAD_TREE);
    }
    out_parents[p] = op;
    if (out_tokens) out_tokens[p] = tokens[g];
    if (out_score) out_score[p] = score[g];
  }
}

}  // namespace
}  // namespace sdv

using namespace sdv;

extern "C" size_t sd_select_workspace(int32_t n_total) {
  if (n_total < 1) return 0;
  return (size_t)n_total * (8 + 4 + 4 + 4) + 16;
}

extern "C" int sd_best_first_select(const int32_t* parents, const float* logprob, const int32_t* cu, int32_t R,
                                    int32_t n_total, int32_t budget, int32_t cap, const int32_t* tokens,
                                    int32_t* out_cu, int32_t* out_src, int32_t* out_parents, int32_t* out_tokens,
                                    float* out_score, int32_t* status, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  if (!parents || !logprob || !cu || !out_cu || !out_src || !out_parents || !status || !workspace ||
      (out_tokens && !tokens) || R < 1 || n_total < R || budget < R || cap < 1) {
    set_error("sd_best_first_select: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (n_total > kSelMaxTotal) {
    set_error("sd_best_first_select: at most 16384 candidates per call");
    return SD_ERR_UNSUPPORTED;
  }
  if (workspace_bytes < sd_select_workspace(n_total)) {
    set_error("sd_best_first_select: workspace too small");
    return SD_ERR_WORKSPACE;
  }
  const uintptr_t base = ((uintptr_t)workspace + 15) & ~(uintptr_t)15;
  uint64_t* ekey = reinterpret_cast<uint64_t*>(base);
  float* score = reinterpret_cast<float*>(ekey + n_total);
  int32_t* req = reinterpret_cast<int32_t*>(score + n_total);
  int32_t* pos = req + n_total;
  cudaStream_t s = (cudaStream_t)stream;
  SD_CK(cudaMemsetAsync(ekey, 0xFF, (size_t)n_total * sizeof(uint64_t), s));
  SD_CK(launch(k_sel_keys, dim3(R), dim3(kKeyThreads), 0, s, false, parents, logprob, cu, (int)n_total, (int)cap,
               ekey, score, req, status));
  SD_CK(launch(k_sel_pick, dim3(1), dim3(kPickThreads), 0, s, true, (const uint64_t*)ekey, (const float*)score,
               (const int32_t*)req, cu, parents, tokens, (int)R, (int)n_total, (int)budget, pos, out_cu, out_src,
               out_parents, out_tokens, out_score, status));
  return SD_OK;
}
