// C ABI: errors, stand-alone tree helpers and the tiny verify model.
#include <algorithm>
#include <mutex>
#include <vector>

#include "gemm.cuh"
#include "layers.cuh"

namespace sdv {

static thread_local std::string g_last_error;

void set_error(const std::string& s) { g_last_error = s; }

int cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return e == cudaErrorMemoryAllocation ? SD_ERR_OOM : SD_ERR_CUDA;
}

void carveout_once(const void* kern) {
  static std::mutex mu;
  static std::vector<const void*> done;
  std::lock_guard<std::mutex> lock(mu);
  for (const void* k : done)
    if (k == kern) return;
  cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  done.push_back(kern);
}

int num_sms() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  });
  return n;
}

// [TREE] one tree: validation, ancestor masks, depth, position.
__global__ void k_tree_single(const int32_t* __restrict__ parents, int M, int ctx, uint64_t* __restrict__ anc,
                              int32_t* __restrict__ depth, int32_t* __restrict__ pos, int32_t* status) {
  if (threadIdx.x != 0) return;
  uint64_t a[64];
  int d[64];
  bool ok = M >= 1 && M <= 64;
  for (int i = 0; i < M && ok; i++) {
    const int p = parents[i];
    if (i == 0 ? p != -1 : (p < 0 || p >= i)) {
      ok = false;
      break;
    }
    a[i] = (i ? a[p] : 0ull) | (1ull << i);
    d[i] = i ? d[p] + 1 : 0;
  }
  if (!ok) set_status(status, SD_ERR_BAD_TREE);
  for (int i = 0; i < M && i < 64; i++) {
    anc[i] = ok ? a[i] : (1ull << i);
    depth[i] = ok ? d[i] : 0;
    pos[i] = ctx + (ok ? d[i] : 0);
  }
}

// The bounded waits' give-up path, exercised on purpose: one CTA waits with
// the library's own helpers on something nothing completes - an mbarrier
// nobody arrives at (which = 0: two warps, the first to give up aborts the
// other, as in the GEMM pipelines) or a device flag nobody sets (which = 1:
// the acquire poll of the streamed GEMM's dependency waits) - and reports
// SD_ERR_TIMEOUT in *status once limit_ns has passed.
static __device__ int g_never_set;

__global__ void k_debug_wait(int32_t* status, uint64_t limit_ns, int which) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  if (which == 0) {
    bool ok = true;
    if (lane == 0) ok = mbar_wait_or_abort(&bar, 0, &abort, limit_ns);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok && lane == 0) set_status(status, SD_ERR_TIMEOUT);
  } else if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer();
    for (;;) {
      int v;
      asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(&g_never_set) : "memory");
      if (v != 0) break;
      if (globaltimer() - t0 > limit_ns) {
        set_status(status, SD_ERR_TIMEOUT);
        break;
      }
    }
  }
}

}  // namespace sdv

using namespace sdv;

extern "C" int sd_debug_bounded_wait(int32_t* status, int64_t limit_ns, int32_t which, void* stream) {
  if (!status || (which != 0 && which != 1)) {
    set_error("sd_debug_bounded_wait: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  const uint64_t lim = (uint64_t)std::min<int64_t>(std::max<int64_t>(limit_ns, 1000), (int64_t)kWaitLimitNs);
  k_debug_wait<<<1, 64, 0, (cudaStream_t)stream>>>(status, lim, which);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SD_OK : cuda_fail(e, "k_debug_wait launch");
}

extern "C" const char* sd_last_error(void) { return g_last_error.c_str(); }
extern "C" const char* sd_version(void) { return "sdv 0.1 (sm_103a)"; }

extern "C" int sd_tree_info(const int32_t* parents, int32_t M, int32_t ctx, uint64_t* anc, int32_t* depth,
                            int32_t* pos, int32_t* status, void* stream) {
  if (!parents || !anc || !depth || !pos || M < 1) {
    set_error("sd_tree_info: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (M > 64) {
    set_error("sd_tree_info: at most 64 nodes");
    return SD_ERR_UNSUPPORTED;
  }
  k_tree_single<<<1, 32, 0, (cudaStream_t)stream>>>(parents, M, ctx, anc, depth, pos, status);
  SD_CK(cudaGetLastError());
  return SD_OK;
}

extern "C" int sd_accept(const int32_t* tokens, const int32_t* parents, const int32_t* argmax, int32_t M,
                         int32_t* accepted_len, int32_t* accepted_tokens, int32_t* bonus, int32_t* path,
                         int32_t* status, void* stream) {
  if (!tokens || !parents || !argmax || !accepted_len || !accepted_tokens || !bonus || M < 1) {
    set_error("sd_accept: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (M > 64) {
    set_error("sd_accept: at most 64 nodes");
    return SD_ERR_UNSUPPORTED;
  }
  AcceptArgs a{};
  a.tokens = tokens;
  a.parents = parents;
  a.cu = nullptr;
  a.R = 1;
  a.single_M = M;
  a.argmax_in = argmax;
  a.accepted_len = accepted_len;
  a.accepted_tokens = accepted_tokens;
  a.bonus = bonus;
  a.status = status;
  a.path = path;
  SD_CK(launch_accept(a, (cudaStream_t)stream, false));
  return SD_OK;
}

// ---------------------------------------------------------------- tiny --

struct TinyLayout {
  size_t y, partial, counters, amax_val, amax_idx, total;
  size_t partial_floats;
  int counters_len;
};

static size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

static TinyLayout tiny_layout(int64_t N1, int64_t V, int M) {
  TinyLayout L;
  size_t o = 0;
  L.y = o;
  o = al256(o + (size_t)M * N1 * 2);
  L.partial_floats = gemm_partial_floats(M);
  L.partial = o;
  o = al256(o + L.partial_floats * 4);
  L.counters_len = std::max(gemm_counters(N1), gemm_counters(V));
  L.counters = o;
  o = al256(o + (size_t)L.counters_len * 4);
  L.amax_val = o;
  o = al256(o + (size_t)gemm_grid(M) * M * 4);
  L.amax_idx = o;
  o = al256(o + (size_t)gemm_grid(M) * M * 4);
  L.total = o;
  return L;
}

extern "C" size_t sd_tiny_workspace(int64_t N1, int64_t K, int64_t V, int32_t M) {
  (void)K;
  return tiny_layout(N1, V, std::max(1, M)).total;
}

extern "C" int sd_tiny_verify(const w12_tensor* W1, const w12_tensor* Wlm, const uint16_t* act, const int32_t* tokens,
                              const int32_t* parents, int32_t M, int32_t* accepted_len, int32_t* accepted_tokens,
                              int32_t* bonus, uint16_t* logits, int32_t* argmax, int32_t* status, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (!W1 || !Wlm || !act || !tokens || !parents || !accepted_len || !accepted_tokens || !bonus || !workspace ||
      M < 1) {
    set_error("sd_tiny_verify: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (M > 64 || W1->K % 64 || W1->N % 16 || Wlm->K != W1->N || Wlm->N % 16 || W1->N % 64) {
    set_error("sd_tiny_verify: unsupported shape (M <= 64, W1 [N1][K], Wlm [V][N1])");
    return SD_ERR_UNSUPPORTED;
  }
  const TinyLayout L = tiny_layout(W1->N, Wlm->N, M);
  if (workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255)) {
    set_error("sd_tiny_verify: workspace too small or not 256-byte aligned");
    return SD_ERR_WORKSPACE;
  }
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  uint16_t* y = reinterpret_cast<uint16_t*>(ws + L.y);
  GemmWorkspace gw;
  gw.partial = reinterpret_cast<float*>(ws + L.partial);
  gw.partial_floats = L.partial_floats;
  gw.counters = reinterpret_cast<int32_t*>(ws + L.counters);
  gw.counters_len = L.counters_len;
  float* av = reinterpret_cast<float*>(ws + L.amax_val);
  int32_t* ai = reinterpret_cast<int32_t*>(ws + L.amax_idx);
  SD_CK(cudaMemsetAsync(gw.counters, 0, (size_t)gw.counters_len * 4, s));
  XMap m1, m2;
  int rc = make_x_map(&m1, act, M, W1->K, pad_rows(M));
  if (!rc) rc = make_x_map(&m2, y, M, W1->N, pad_rows(M));
  if (rc) return rc;
  GemmEpilogue e1;
  e1.epi = EPI_STORE;
  e1.out = y;
  e1.ldo = (int)W1->N;
  rc = gemm_launch(*W1, act, m1, M, e1, gw, status, s, false);
  if (rc) return rc;
  GemmEpilogue e2;
  e2.epi = EPI_LOGITS;
  e2.out = logits;
  e2.ldo = (int)Wlm->N;
  e2.amax_val = av;
  e2.amax_idx = ai;
  e2.ld_amax = M;
  rc = gemm_launch(*Wlm, y, m2, M, e2, gw, status, s, true);
  if (rc) return rc;
  AcceptArgs a{};
  a.tokens = tokens;
  a.parents = parents;
  a.cu = nullptr;
  a.R = 1;
  a.single_M = M;
  a.amax_val = av;
  a.amax_idx = ai;
  a.n_part = gemm_grid(M);
  a.ld = M;
  a.argmax_out = argmax;
  a.accepted_len = accepted_len;
  a.accepted_tokens = accepted_tokens;
  a.bonus = bonus;
  a.status = status;
  SD_CK(launch_accept(a, s, true));
  return SD_OK;
}
