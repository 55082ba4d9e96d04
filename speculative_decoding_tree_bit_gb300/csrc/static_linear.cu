// sd_w12_linear_static: the fused W12 linear without any allocation.
//
// sd_w12_linear needs a caller-provided device workspace for the split-K
// partial sums and the finishing tickets.  Some callers cannot obtain one:
// code that runs where cudaMalloc is off limits (a host framework that owns
// every device byte through its own pool, a real-time thread that must not
// take cudaMalloc's implicit device synchronisation, a plug-in loaded into a
// process that forbids growing its device footprint after start-up).  This
// variant keeps that scratch in a file-scope device array instead, so a call
// needs nothing but the inputs and the output.
#include <mutex>

#include "gemm.cuh"

namespace sdv {

// Limits of the static scratch (every GPU that loads the library holds it
// until the process exits: 1216 CTA-tiles x 2 partial slots x 8 warps x 8
// rows x 128 floats = 9.5 MiB, plus one ticket per 128 output rows).  A
// launch of G CTAs over NT token tiles of 8 needs G * NT <= 1216: 152 CTAs
// at 64 rows, 304 at 32 rows or fewer, as sd_w12_linear uses on 152 SMs.
constexpr int kStaticMaxRows = 64;           // M <= 64 (8 token tiles of 8)
constexpr int kStaticCtaTiles = 1216;        // CTAs x token tiles per launch
constexpr int64_t kStaticMaxN = 1 << 18;     // output rows
constexpr size_t kStaticPartialFloats = (size_t)kStaticCtaTiles * 2 * 8 * 128;
constexpr int kStaticCounters = (int)(kStaticMaxN / 128);

static __device__ __align__(256) float g_static_partial[kStaticPartialFloats];
static __device__ __align__(256) int32_t g_static_counters[kStaticCounters];

// Device addresses of the arrays in the current context (the names are
// host-side stand-ins in host code, never valid device pointers).  Looked
// up on every call, so that a new context (after cudaDeviceReset, or on
// another device) gets its own addresses.
struct StaticScratch {
  float* partial = nullptr;
  int32_t* counters = nullptr;
};

static int static_scratch(StaticScratch* out) {
  void* p = nullptr;
  void* c = nullptr;
  SD_CK(cudaGetSymbolAddress(&p, g_static_partial));
  SD_CK(cudaGetSymbolAddress(&c, g_static_counters));
  out->partial = static_cast<float*>(p);
  out->counters = static_cast<int32_t*>(c);
  return SD_OK;
}

}  // namespace sdv

using namespace sdv;

extern "C" int sd_w12_linear_static(const w12_tensor* W, const uint16_t* x, int32_t M, uint16_t* y, void* stream) {
  if (!W || !x || !y || M < 1) {
    set_error("sd_w12_linear_static: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (W->N % 16 || W->K % 64) {
    set_error("sd_w12_linear_static: need N % 16 == 0 and K % 64 == 0");
    return SD_ERR_UNSUPPORTED;
  }
  if (M > kStaticMaxRows || W->N > kStaticMaxN) {
    set_error("sd_w12_linear_static: M must be <= 64 and N <= 262144 (size of the static scratch); "
              "use sd_w12_linear with a workspace for larger calls");
    return SD_ERR_UNSUPPORTED;
  }
  StaticScratch sc;
  int rc = static_scratch(&sc);
  if (rc) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  GemmWorkspace ws;
  ws.partial = sc.partial;
  ws.partial_floats = kStaticPartialFloats;
  ws.counters = sc.counters;
  ws.counters_len = gemm_counters(W->N);
  // the finishing tickets must start at zero; the partial slots are always
  // written before they are read
  SD_CK(cudaMemsetAsync(ws.counters, 0, (size_t)ws.counters_len * sizeof(int32_t), s));
  XMap xm;
  rc = make_x_map(&xm, x, M, W->K, pad_rows(M));
  if (rc) return rc;
  GemmEpilogue e;
  e.epi = EPI_STORE;
  e.out = y;
  e.ldo = (int)W->N;
  // the warp-level kernel whatever the tensor-core threshold (the static
  // scratch is sized for it), with the grid sd_w12_linear gives it
  const int nt = pad_rows(M) / 8;
  int grid = gemm_warp_launch_grid(*W, M, EPI_STORE);
  if (grid * nt > kStaticCtaTiles) grid = kStaticCtaTiles / nt;
  return gemm_warp_launch(*W, x, xm, M, e, ws, nullptr, s, false, grid);
}
