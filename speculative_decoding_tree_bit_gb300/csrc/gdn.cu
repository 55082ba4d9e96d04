// Gated delta rule over a draft tree, in WY form, for sm_103a.
//
// "SpecPilot: AI Agent Framework Boosts Speculative Decoding 10.87x for
// Qwen3.8-27B", "(2) Best-first Tree Verification for Hybrid Architectures":
// in Gated DeltaNet layers the recurrent state has to follow each root path
// of the draft tree, and a WY-form kernel evaluates many paths at once.  The
// rule (per head, q and k L2-normalised, row of S = key dimension):
//   S_i = alpha_i (I - beta_i k_i k_i^T) S_parent(i) + beta_i k_i v_i^T,
//   o_i = S_i^T q_i.
// The whole tree takes one unit-lower-triangular solve.  With Anc the
// strict-ancestor mask (parents precede children), G_i the product of alpha
// over i's root path,
//   T = I + Anc .* (diag(beta) K K^T),  W = T^-1 diag(beta) K,
//   U = T^-1 diag(beta) (V / G),         D = U - W S0,
//   o_i = G_i [S0^T q_i + sum_{j on path(i)} (k_j . q_i) d_j],
//   S_i = G_i [S0 + sum_{j on path(i)} k_j d_j^T],
// so S0 is read once per (request, head) whatever the tree's shape, and no
// per-node state is ever formed.  One CTA per (32 value columns, head,
// request) holds the whole tree of its request (at most 64 nodes) on chip:
// normalised q and k, the path dot products, W and its slice of U, D and S0.
// The solve walks the nodes in order; each step touches only the node's
// ancestors.  The commit after acceptance forms S of the deepest accepted
// node from the D rows and normalised keys this kernel leaves in the
// workspace.  fp32 throughout (the state is fp32); bf16 outputs.
#include "common.cuh"

namespace sdv {

constexpr int kGdnMaxM = 64;
constexpr int kGdnCols = 32;       // value columns per CTA
// 16 warps in the verify kernel: its output phases give each thread one
// (node, column) chain at 16 nodes (1 x 16: 16.8 -> 15.2 us, 8 x 16: 108.5
// -> 98.4 us against 8 warps); 8 warps in the commit (at 32 x 8 its 16-warp
// form measured slower)
constexpr int kGdnThreads = 512;
constexpr int kGdnCommitThreads = 256;
constexpr int kGdnHd = 128;

struct GdnArgs {
  const uint16_t* q;  // bf16 [rows][nh][128]
  const uint16_t* k;
  const uint16_t* v;
  const float* alpha;  // [rows][nh]
  const float* beta;
  const int32_t* parents;  // [rows], local to each request
  const int32_t* cu;       // [R + 1] device
  int R, nh;
  const float* S;  // [R][nh][128][128]
  uint16_t* out;   // bf16 [rows][nh][128]
  float* ws_d;     // [rows][nh][128]  rows of D
  float* ws_k;     // [rows][nh][128]  normalised keys
  float* ws_g;     // [rows][nh]       path gate products
  int32_t* status;
};

struct GdnSmem {
  float kn[kGdnMaxM][kGdnHd];
  float qn[kGdnMaxM][kGdnHd];
  float w[kGdnMaxM][kGdnHd];
  float s0[kGdnHd][kGdnCols];
  float u[kGdnMaxM][kGdnCols];
  float d[kGdnMaxM][kGdnCols];
  float t[kGdnMaxM][kGdnMaxM];  // beta_i (k_i . k_j), j a strict ancestor of i
  float p[kGdnMaxM][kGdnMaxM];  // q_i . k_j, j on i's root path
  float g[kGdnMaxM];
  float b[kGdnMaxM];
  uint64_t anc[kGdnMaxM];  // bit j: j on i's root path (i included)
  int par[kGdnMaxM];
  int ok;
};

// Validates one request's parent array (staged in s.par) into s.anc
// (thread 0; no global loads on its serial chain).
__device__ __forceinline__ bool gdn_tree_ok(int M, GdnSmem& s) {
  if (M < 1 || M > kGdnMaxM) return false;
  for (int i = 0; i < M; i++) {
    const int p = s.par[i];
    if (i == 0 ? p != -1 : (p < 0 || p >= i)) return false;
    s.anc[i] = (i ? s.anc[p] : 0ull) | (1ull << i);
  }
  return true;
}

__global__ void __launch_bounds__(kGdnThreads, 1) k_gdn_tree(GdnArgs a) {
  pdl_launch();
  extern __shared__ __align__(16) uint8_t smem_gdn[];
  GdnSmem& s = *reinterpret_cast<GdnSmem*>(smem_gdn);
  const int cc = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int kWarps = kGdnThreads / 32;
  const int nh = a.nh;
  pdl_wait();  // q, k, v, the gates and the state may come from the previous kernel
  const float* S0 = a.S + ((int64_t)r * nh + h) * kGdnHd * kGdnHd;
  {
    // the state tile: every thread's loads in flight before its stores
    constexpr int kIt = kGdnHd * kGdnCols / 4 / kGdnThreads;
    static_assert(kIt * kGdnThreads * 4 == kGdnHd * kGdnCols, "whole float4 per thread");
    float4 v[kIt];
#pragma unroll
    for (int u = 0; u < kIt; u++) {
      const int e = tid + u * kGdnThreads, row = e / (kGdnCols / 4), c4 = e % (kGdnCols / 4);
      v[u] = __ldcg(reinterpret_cast<const float4*>(S0 + (int64_t)row * kGdnHd + cc * kGdnCols) + c4);
    }
#pragma unroll
    for (int u = 0; u < kIt; u++) {
      const int e = tid + u * kGdnThreads, row = e / (kGdnCols / 4), c4 = e % (kGdnCols / 4);
      *reinterpret_cast<float4*>(&s.s0[row][4 * c4]) = v[u];
    }
  }
  const int node0 = a.cu[r], M = a.cu[r + 1] - node0;
  // the parents and gates of the request, all loads at once (the serial
  // chains below then run on shared memory)
  for (int i = tid; i < M && i < kGdnMaxM; i += kGdnThreads) {
    s.par[i] = a.parents[node0 + i];
    s.g[i] = a.alpha[(int64_t)(node0 + i) * nh + h];
  }
  __syncthreads();
  if (tid == 0) {
    s.ok = gdn_tree_ok(M, s) ? 1 : 0;
    if (!s.ok) set_status(a.status, SD_ERR_BAD_TREE);
  }
  __syncthreads();
  if (!s.ok) return;

  // this CTA's value columns of every node, staged in u (the solve below
  // overwrites each row with its result); loads before stores
  {
    constexpr int kIt = kGdnMaxM * kGdnCols / kGdnThreads;
    uint16_t vv[kIt];
#pragma unroll
    for (int u = 0; u < kIt; u++) {
      const int e = tid + u * kGdnThreads, i = e / kGdnCols, c = e % kGdnCols;
      vv[u] = i < M ? a.v[((int64_t)(node0 + i) * nh + h) * kGdnHd + cc * kGdnCols + c] : (uint16_t)0;
    }
#pragma unroll
    for (int u = 0; u < kIt; u++) {
      const int e = tid + u * kGdnThreads, i = e / kGdnCols, c = e % kGdnCols;
      if (i < M) s.u[i][c] = bf2f(vv[u]);
    }
  }
  // normalised q and k (x / ||x||, zero stays zero), one warp per node, a
  // warp's two nodes' loads in flight together
  for (int i0 = warp; i0 < M; i0 += 2 * kWarps) {
    float qv[2][4], kv[2][4];
#pragma unroll
    for (int t = 0; t < 2; t++) {
      const int i = i0 + t * kWarps;
      const int64_t row = ((int64_t)(node0 + (i < M ? i : i0)) * nh + h) * kGdnHd;
#pragma unroll
      for (int j = 0; j < 4; j++) {
        qv[t][j] = bf2f(a.q[row + lane + 32 * j]);
        kv[t][j] = bf2f(a.k[row + lane + 32 * j]);
      }
    }
#pragma unroll
    for (int t = 0; t < 2; t++) {
      const int i = i0 + t * kWarps;
      if (i >= M) break;
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int j = 0; j < 4; j++) {
        sq = fmaf(qv[t][j], qv[t][j], sq);
        sk = fmaf(kv[t][j], kv[t][j], sk);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
      }
      const float nq = sqrtf(sq), nk = sqrtf(sk);
#pragma unroll
      for (int j = 0; j < 4; j++) {
        s.qn[i][lane + 32 * j] = nq > 0.f ? qv[t][j] / nq : 0.f;
        s.kn[i][lane + 32 * j] = nk > 0.f ? kv[t][j] / nk : 0.f;
      }
      if (lane == 0) s.b[i] = a.beta[(int64_t)(node0 + i) * nh + h];
    }
  }
  if (tid == 0) {
    // path products of the gates, root first (G_i = alpha_i G_parent), in
    // place over the staged gates (parents precede children)
    for (int i = 1; i < M; i++) s.g[i] = s.g[i] * s.g[s.par[i]];
  }
  __syncthreads();
  // dot products along root paths: t (strict ancestors, scaled by beta_i)
  // and p (ancestors and the node itself); one warp per (i, j) pair
  for (int i = warp; i < M; i += kWarps) {
    uint64_t m = s.anc[i];
    while (m) {
      const int j = __ffsll((long long)m) - 1;
      m &= m - 1;
      float kk = 0.f, qk = 0.f;
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const float kj = s.kn[j][lane + 32 * e];
        kk = fmaf(s.kn[i][lane + 32 * e], kj, kk);
        qk = fmaf(s.qn[i][lane + 32 * e], kj, qk);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        kk += __shfl_xor_sync(0xffffffffu, kk, o);
        qk += __shfl_xor_sync(0xffffffffu, qk, o);
      }
      if (lane == 0) {
        s.t[i][j] = j == i ? 0.f : s.b[i] * kk;
        s.p[i][j] = qk;
      }
    }
  }
  __syncthreads();
  // forward substitution, nodes in order: w_i = beta_i k_i - sum_j t_ij w_j
  // over all 128 key dims, u_i = beta_i v_i / G_i - sum_j t_ij u_j over this
  // CTA's value columns
  for (int i = 0; i < M; i++) {
    const uint64_t strict = s.anc[i] & ~(1ull << i);
    if (tid < kGdnHd) {
      float acc = s.b[i] * s.kn[i][tid];
      uint64_t m = strict;
      while (m) {
        const int j = __ffsll((long long)m) - 1;
        m &= m - 1;
        acc = fmaf(-s.t[i][j], s.w[j][tid], acc);
      }
      s.w[i][tid] = acc;
    } else if (tid < kGdnHd + kGdnCols) {
      const int c = tid - kGdnHd;
      float acc = s.b[i] * (s.u[i][c] / s.g[i]);
      uint64_t m = strict;
      while (m) {
        const int j = __ffsll((long long)m) - 1;
        m &= m - 1;
        acc = fmaf(-s.t[i][j], s.u[j][c], acc);
      }
      s.u[i][c] = acc;
    }
    __syncthreads();
  }
  // D = U - W S0 and Q S0 (this CTA's columns): thread = (node, column)
  for (int e = tid; e < M * kGdnCols; e += kGdnThreads) {
    const int i = e / kGdnCols, c = e % kGdnCols;
    float ws = 0.f;
#pragma unroll 8
    for (int x = 0; x < kGdnHd; x++) ws = fmaf(s.w[i][x], s.s0[x][c], ws);
    s.d[i][c] = s.u[i][c] - ws;
  }
  __syncthreads();
  for (int e = tid; e < M * kGdnCols; e += kGdnThreads) {
    const int i = e / kGdnCols, c = e % kGdnCols;
    float qs = 0.f;
#pragma unroll 8
    for (int x = 0; x < kGdnHd; x++) qs = fmaf(s.qn[i][x], s.s0[x][c], qs);
    uint64_t m = s.anc[i];
    while (m) {
      const int j = __ffsll((long long)m) - 1;
      m &= m - 1;
      qs = fmaf(s.p[i][j], s.d[j][c], qs);
    }
    const int64_t row = (int64_t)(node0 + i) * nh + h;
    a.out[row * kGdnHd + cc * kGdnCols + c] = f2bf(s.g[i] * qs);
    a.ws_d[row * kGdnHd + cc * kGdnCols + c] = s.d[i][c];
  }
  if (cc == 0) {
    for (int e = tid; e < M * kGdnHd; e += kGdnThreads) {
      const int i = e / kGdnHd, x = e % kGdnHd;
      a.ws_k[((int64_t)(node0 + i) * nh + h) * kGdnHd + x] = s.kn[i][x];
    }
    for (int i = tid; i < M; i += kGdnThreads) a.ws_g[(int64_t)(node0 + i) * nh + h] = s.g[i];
  }
}

// Commit: S0 <- S of node last[r] = G [S0 + sum_{j on its path} k_j d_j^T].
// CTA = (16 key rows, head, request); a request whose last[r] is out of range
// (a rejected tree) keeps its state.
constexpr int kGdnCommitRows = 16;

__global__ void __launch_bounds__(kGdnCommitThreads) k_gdn_commit(const int32_t* __restrict__ parents,
                                                            const int32_t* __restrict__ cu, int nh,
                                                            const int32_t* __restrict__ last, float* S,
                                                            const float* __restrict__ ws_d,
                                                            const float* __restrict__ ws_k,
                                                            const float* __restrict__ ws_g) {
  pdl_launch();
  pdl_wait();
  __shared__ int path[kGdnMaxM];
  __shared__ int par_s[kGdnMaxM];
  __shared__ int n_path;
  __shared__ float kp[kGdnMaxM][kGdnCommitRows];
  const int rb = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
  const int node0 = cu[r], M = cu[r + 1] - node0;
  // the request's parents, all loads at once; the walk then runs on shared
  // memory
  for (int i = threadIdx.x; i < M && i < kGdnMaxM; i += blockDim.x) par_s[i] = parents[node0 + i];
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = 0;
    int j = last[r];
    if (j >= 0 && j < M && M <= kGdnMaxM) {
      int tmp[kGdnMaxM];
      while (j >= 0 && n < kGdnMaxM) {
        tmp[n++] = j;
        const int p = par_s[j];
        j = (p < j) ? p : -1;  // parents precede children (validated by the verify kernel)
      }
      for (int i = 0; i < n; i++) path[i] = tmp[n - 1 - i];
    }
    n_path = n;
  }
  __syncthreads();
  const int P = n_path;
  if (P == 0) return;
  for (int e = threadIdx.x; e < P * kGdnCommitRows; e += blockDim.x) {
    const int pi = e / kGdnCommitRows, x = e % kGdnCommitRows;
    kp[pi][x] = ws_k[((int64_t)(node0 + path[pi]) * nh + h) * kGdnHd + rb * kGdnCommitRows + x];
  }
  __syncthreads();
  const float G = ws_g[(int64_t)(node0 + path[P - 1]) * nh + h];
  float* Sh = S + ((int64_t)r * nh + h) * kGdnHd * kGdnHd;
  // the thread's state elements: all loads before the first store (a store
  // to S could alias a later load of it, so one element at a time would wait
  // one round trip each)
  constexpr int kIt = kGdnCommitRows * kGdnHd / kGdnCommitThreads;
  static_assert(kIt * kGdnCommitThreads == kGdnCommitRows * kGdnHd, "whole elements per thread");
  float acc[kIt];
#pragma unroll
  for (int u = 0; u < kIt; u++) {
    const int e = threadIdx.x + u * kGdnCommitThreads, x = e / kGdnHd, c = e % kGdnHd;
    acc[u] = Sh[(int64_t)(rb * kGdnCommitRows + x) * kGdnHd + c];
  }
  for (int pi = 0; pi < P; pi++) {
    const float* dp = ws_d + ((int64_t)(node0 + path[pi]) * nh + h) * kGdnHd;
#pragma unroll
    for (int u = 0; u < kIt; u++) {
      const int e = threadIdx.x + u * kGdnCommitThreads, x = e / kGdnHd, c = e % kGdnHd;
      acc[u] = fmaf(kp[pi][x], dp[c], acc[u]);
    }
  }
#pragma unroll
  for (int u = 0; u < kIt; u++) {
    const int e = threadIdx.x + u * kGdnCommitThreads, x = e / kGdnHd, c = e % kGdnHd;
    Sh[(int64_t)(rb * kGdnCommitRows + x) * kGdnHd + c] = G * acc[u];
  }
}

}  // namespace sdv

using namespace sdv;

extern "C" size_t sd_gdn_workspace(int32_t rows, int32_t nh) {
  if (rows < 1 || nh < 1) return 0;
  return (size_t)rows * nh * (2 * kGdnHd + 1) * sizeof(float) + 256;
}

static int gdn_check(const int32_t* cu_host, int32_t R, int32_t nh, int32_t* rows) {
  if (!cu_host || R < 1 || nh < 1 || cu_host[0] != 0) {
    set_error("sd_gdn: bad R, nh or cu_nodes");
    return SD_ERR_INVALID_ARG;
  }
  for (int r = 0; r < R; r++)
    if (cu_host[r + 1] - cu_host[r] < 1 || cu_host[r + 1] - cu_host[r] > kGdnMaxM) {
      set_error("sd_gdn: each request needs 1..64 nodes");
      return SD_ERR_UNSUPPORTED;
    }
  *rows = cu_host[R];
  return SD_OK;
}

extern "C" int sd_gdn_tree_verify(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* alpha,
                                  const float* beta, const int32_t* parents, const int32_t* cu, const int32_t* cu_host,
                                  int32_t R, int32_t nh, const float* S, uint16_t* out, void* workspace,
                                  size_t workspace_bytes, int32_t* status, void* stream) {
  if (!q || !k || !v || !alpha || !beta || !parents || !cu || !S || !out || !workspace) {
    set_error("sd_gdn_tree_verify: null argument");
    return SD_ERR_INVALID_ARG;
  }
  int32_t rows = 0;
  int rc = gdn_check(cu_host, R, nh, &rows);
  if (rc) return rc;
  if (workspace_bytes < sd_gdn_workspace(rows, nh) || (reinterpret_cast<uintptr_t>(workspace) & 255)) {
    set_error("sd_gdn_tree_verify: workspace too small or not 256-byte aligned");
    return SD_ERR_WORKSPACE;
  }
  static bool attr = false;
  if (!attr) {
    SD_CK(cudaFuncSetAttribute(k_gdn_tree, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(GdnSmem)));
    attr = true;
  }
  GdnArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.alpha = alpha;
  a.beta = beta;
  a.parents = parents;
  a.cu = cu;
  a.R = R;
  a.nh = nh;
  a.S = S;
  a.out = out;
  float* ws = reinterpret_cast<float*>(workspace);
  a.ws_d = ws;
  a.ws_k = ws + (size_t)rows * nh * kGdnHd;
  a.ws_g = ws + (size_t)rows * nh * kGdnHd * 2;
  a.status = status;
  SD_CK(launch(k_gdn_tree, dim3(kGdnHd / kGdnCols, nh, R), dim3(kGdnThreads), sizeof(GdnSmem), (cudaStream_t)stream,
               true, a));
  return SD_OK;
}

extern "C" int sd_gdn_commit(const int32_t* parents, const int32_t* cu, const int32_t* cu_host, int32_t R,
                             int32_t nh, const int32_t* last, float* S, const void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (!parents || !cu || !last || !S || !workspace) {
    set_error("sd_gdn_commit: null argument");
    return SD_ERR_INVALID_ARG;
  }
  int32_t rows = 0;
  int rc = gdn_check(cu_host, R, nh, &rows);
  if (rc) return rc;
  if (workspace_bytes < sd_gdn_workspace(rows, nh)) {
    set_error("sd_gdn_commit: workspace too small");
    return SD_ERR_WORKSPACE;
  }
  const float* ws = reinterpret_cast<const float*>(workspace);
  SD_CK(launch(k_gdn_commit, dim3(kGdnHd / kGdnCommitRows, nh, R), dim3(kGdnCommitThreads), 0, (cudaStream_t)stream, true,
               parents, cu, nh, last, S, ws, ws + (size_t)rows * nh * kGdnHd, ws + (size_t)rows * nh * kGdnHd * 2));
  return SD_OK;
}
