// W12 weight-streaming GEMMs: host side (per-phase CTA counts, scratch
// layout, launch).  The kernel and its design are in stream_kernel.cuh; one
// translation unit per weight-decode mode instantiates it.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "stream_kernel.cuh"

namespace sdv {

// ------------------------------------------------------------------ host --

// Padded rows of a streamed launch: 8, 16 or 64 (17..64 rows run the
// 64-row variant: the 32-row variant is not used, see the design notes).
static int stream_pad_rows(int M) { return M <= 8 ? 8 : M <= 16 ? 16 : 64; }
static int nt_of_rows(int M) { return stream_pad_rows(M) / 8; }

int stream_grid(int M) { return (nt_of_rows(M) <= 4 ? 2 : 1) * num_sms(); }

static int blocks_of(const w12_tensor& W) { return (int)((W.N / 16 + kRB - 1) / kRB); }

size_t stream_state_ints(const StreamPhaseDesc* ph, int n) {
  size_t s = 1;
  for (int i = 0; i < n; i++) s += 2 + 2 * (size_t)blocks_of(*ph[i].W);
  return s;
}

size_t stream_state_ints_bound(int64_t n_max) {
  return 1 + (size_t)kStreamMaxPhases * (2 + 2 * (size_t)((n_max / 16 + kRB - 1) / kRB));
}

// CTAs that share a phase's tiles: with few row blocks a whole number of
// CTAs per block (no CTA straddles two blocks, every block has the same
// number of contributors); a logits phase keeps every CTA (one argmax
// partial per CTA of the launch).
static int phase_ctas(const w12_tensor& W, int epi, int grid) {
  const int nb = blocks_of(W);
  return (epi != EPI_LOGITS && nb * 4 <= grid) ? nb * (grid / nb) : grid;
}

static size_t phase_partial_floats(int M) { return (size_t)stream_grid(M) * 2 * 128 * stream_pad_rows(M); }

size_t stream_partial_floats(const StreamPhaseDesc*, int n, int M) { return (size_t)n * phase_partial_floats(M); }

size_t stream_partial_floats_bound(int64_t, int64_t, int M) { return kStreamMaxPhases * phase_partial_floats(M); }

// Every CTA of a launch must be resident at once (a phase's activation
// tiles wait for blocks other CTAs finish): the kernel takes the whole
// shared-memory carveout and must fit s_ctas_per_sm CTAs per SM.
cudaError_t stream_check_residency(const void* kern, int NT) {
  carveout_once(kern);
  const int want = NT <= 4 ? 2 : 1;
  const int smem = NT == 1 ? SCfg<1>::SMEM : NT == 2 ? SCfg<2>::SMEM : SCfg<8>::SMEM;
  int n = 0;
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kSThreads, smem);
  if (e != cudaSuccess) return e;
  return n >= want ? cudaSuccess : cudaErrorInvalidConfiguration;
}

// Event log of streamed launches (diagnostics): each launch while a buffer
// is set takes the next stream_grid(M) * kTraceEv records of it.
static std::mutex g_trace_mu;
static uint64_t* g_trace = nullptr;
static size_t g_trace_records = 0, g_trace_used = 0;
static int g_trace_launches = 0;

int stream_set_trace(uint64_t* buf, size_t bytes) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  g_trace = buf;
  g_trace_records = buf ? bytes / 16 : 0;
  g_trace_used = 0;
  g_trace_launches = 0;
  return SD_OK;
}

int stream_trace_launches() {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  return g_trace_launches;
}

static uint64_t* trace_take(int grid) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  const size_t need = (size_t)grid * kTraceEv;
  if (!g_trace || g_trace_used + need > g_trace_records) return nullptr;
  uint64_t* p = g_trace + 2 * g_trace_used;
  g_trace_used += need;
  g_trace_launches++;
  return p;
}

int stream_launch(const StreamPhaseDesc* ph, int n, int M, const StreamWorkspace& ws, int32_t* status, cudaStream_t s,
                  bool pdl) {
  if (!ph || n < 1 || n > kStreamMaxPhases || M < 1 || M > kStreamMaxRows) {
    set_error("stream: bad argument (1..4 phases, 1..64 rows)");
    return SD_ERR_INVALID_ARG;
  }
  if (!ws.state) {
    set_error("stream: no state scratch");
    return SD_ERR_WORKSPACE;
  }
  const int grid = stream_grid(M);
  const int MP = stream_pad_rows(M);
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
    if (W.row_base) {
      set_error("stream: per-channel tensors multiply on the warp-level kernel (sd_w12_linear)");
      return SD_ERR_UNSUPPORTED;
    }
    if (d.dep >= i || d.dep < -1 || (d.dep_fine && d.dep < 0)) {
      set_error("stream: a phase may depend on an earlier phase only");
      return SD_ERR_INVALID_ARG;
    }
    if (d.dep_fine && (int64_t)blocks_of(*ph[d.dep].W) * 64 != W.K) {
      set_error("stream: a fine dependency needs one k-tile of x per row block of the phase it reads");
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
    P.words = d.view8 ? d.view8 : W.words;
    P.view8 = d.view8 ? 1 : 0;
    P.tile_ptr = W.n_escapes > 0 ? W.tile_ptr : nullptr;
    P.tile_esc = W.tile_esc;
    P.N = W.N;
    P.K = W.K;
    P.KT = (int)(W.K / 64);
    P.NS = (int)(W.N / 16);
    P.NB = blocks_of(W);
    P.G = phase_ctas(W, d.epi.epi, grid);
    P.U = (int64_t)P.NB * P.KT;
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
    st_off += 2 + 2 * (size_t)P.NB;
    P.part = ws.partial + part_off;
    part_off += phase_partial_floats(M);
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
  int dm_a12 = 1, dm_a8 = 1;
  for (int i = 0; i < n; i++) {
    a.any_norm |= a.ph[i].gamma != nullptr;
    dm_a12 &= a.ph[i].affine && !a.ph[i].view8;
    dm_a8 &= a.ph[i].affine && a.ph[i].view8;
  }
  const int dm = dm_a12 ? DM_A12 : dm_a8 ? DM_A8 : DM_ANY;
  a.state = ws.state;
  a.state_ints = (int)st_off;
  a.status = status;
  a.trace = trace_take(grid);
  cudaError_t e;
  switch (dm) {
    case DM_A12: e = stream_launch_dm<DM_A12>(a, MP / 8, grid, s, pdl); break;
    case DM_A8: e = stream_launch_dm<DM_A8>(a, MP / 8, grid, s, pdl); break;
    default: e = stream_launch_dm<DM_ANY>(a, MP / 8, grid, s, pdl); break;
  }
  if (e != cudaSuccess) return cuda_fail(e, "k_w12_stream launch");
  return SD_OK;
}

}  // namespace sdv

extern "C" int sd_stream_set_trace(uint64_t* buf, int64_t bytes) {
  if (bytes < 0 || (buf && bytes > 0 && (reinterpret_cast<uintptr_t>(buf) & 15))) {
    sdv::set_error("sd_stream_set_trace: bad argument (16-byte aligned buffer, bytes >= 0)");
    return SD_ERR_INVALID_ARG;
  }
  return sdv::stream_set_trace(bytes > 0 ? buf : nullptr, (size_t)bytes);
}

extern "C" int32_t sd_stream_trace_launches(void) { return sdv::stream_trace_launches(); }

extern "C" int32_t sd_stream_grid(int32_t M) { return M >= 1 && M <= sdv::kStreamMaxRows ? sdv::stream_grid(M) : 0; }

static size_t al256s(size_t x) { return (x + 255) & ~size_t(255); }

// One streamed phase: scratch = the state ints, then the split partials.
static void linear_stream_sizes(int64_t N, int64_t K, int M, size_t* state_ints, size_t* part_floats) {
  w12_tensor t{};
  t.N = N;
  t.K = K;
  sdv::StreamPhaseDesc d;
  d.W = &t;
  *state_ints = sdv::stream_state_ints(&d, 1);
  *part_floats = sdv::stream_partial_floats(&d, 1, M);
}

extern "C" size_t sd_w12_linear_stream_workspace(int64_t N, int64_t K, int32_t M) {
  if (N < 16 || K < 64 || M < 1 || M > sdv::kStreamMaxRows) return 256;
  size_t si = 0, sp = 0;
  linear_stream_sizes(N, K, M, &si, &sp);
  return al256s(si * sizeof(int32_t)) + al256s(sp * sizeof(float)) + 256;
}

extern "C" int sd_w12_linear_stream(const w12_tensor* W, const uint32_t* plane8, const uint16_t* x, int32_t M,
                                    uint16_t* y, void* workspace, size_t workspace_bytes, void* stream) {
  if (!W || !x || !y || !workspace || M < 1) {
    sdv::set_error("sd_w12_linear_stream: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (M > sdv::kStreamMaxRows || W->N % 16 || W->K % 64 || W->N < 16 || W->K < 64) {
    sdv::set_error("sd_w12_linear_stream: need 1 <= M <= 64, N % 16 == 0 and K % 64 == 0");
    return SD_ERR_UNSUPPORTED;
  }
  if (plane8 && (reinterpret_cast<uintptr_t>(plane8) & 15)) {
    sdv::set_error("sd_w12_linear_stream: plane8 must be 16-byte aligned");
    return SD_ERR_INVALID_ARG;
  }
  if (workspace_bytes < sd_w12_linear_stream_workspace(W->N, W->K, M) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255)) {
    sdv::set_error("sd_w12_linear_stream: workspace too small or not 256-byte aligned");
    return SD_ERR_WORKSPACE;
  }
  cudaStream_t s = (cudaStream_t)stream;
  size_t si = 0, sp = 0;
  linear_stream_sizes(W->N, W->K, M, &si, &sp);
  sdv::StreamWorkspace ws;
  ws.state = reinterpret_cast<int32_t*>(workspace);
  ws.state_ints = si;
  ws.partial = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(workspace) + al256s(si * sizeof(int32_t)));
  ws.partial_floats = sp;
  const cudaError_t e = cudaMemsetAsync(ws.state, 0, si * sizeof(int32_t), s);
  if (e != cudaSuccess) return sdv::cuda_fail(e, "sd_w12_linear_stream: state clear");
  sdv::StreamPhaseDesc d;
  d.W = W;
  d.view8 = plane8;
  d.x = x;
  d.x_rows = M;
  d.epi.epi = sdv::EPI_STORE;
  d.epi.out = y;
  d.epi.ldo = (int)W->N;
  return sdv::stream_launch(&d, 1, M, ws, nullptr, s, false);
}
