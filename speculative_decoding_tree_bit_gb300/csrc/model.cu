// Verify-step orchestration: model object, workspace, kernel sequence.
//
// One step = tree bookkeeping -> embedding + RMSNorm -> per layer
// [QKV GEMM (+RoPE, K/V write) -> tree attention (or linear recurrence)
//  -> O GEMM (+residual) -> RMSNorm -> gate/up GEMM (+SiLU*up)
//  -> down GEMM (+residual) -> RMSNorm] -> lm_head GEMM (+argmax)
// -> greedy acceptance -> K/V compaction / state commit.
// Every kernel is launched with programmatic dependent launch, so a GEMM's
// producer streams its weights while the previous kernel is still finishing.
// Each linear is one GEMM launch with RMSNorm kernels between them: the
// warp-level kernel (gemm.cu) up to 64 rows below the tensor-core
// threshold, the tcgen05 kernel (gemm_tc.cu) above.  The 8-bit view of
// two-level verification streams its planes through the weight-streaming
// kernel (stream.cu); with the fused schedule (sd_model_set_fused) the GEMMs
// between two attention (or recurrence) kernels - O, gate/up, down and the
// next layer's q/k/v (or the lm_head) - run as one launch of that kernel
// with the RMSNorms folded into it.
#include <algorithm>
#include <cmath>
#include <map>
#include <vector>

#include "gemm.cuh"
#include "layers.cuh"
#include "stream.cuh"

struct sd_model {
  sd_model_config cfg;
  std::vector<int8_t> kind;
  std::vector<int> slot;  // index among attention or among recurrent layers
  std::vector<sd_layer_weights> layers;
  sd_model_weights w;
  int n_attn = 0, n_rec = 0;
  int H, I, Hq, Hkv, hd, V, max_rows, max_req, max_m, nh_rec;
  void* arena = nullptr;
  uint16_t *x, *h, *xn, *q, *attn, *act, *qkv_rec;
  float *rope_cos, *rope_sin;
  int32_t *ctx_snap, *req_ok, *pos, *slotv, *req, *depth, *path, *path_len, *status, *cu, *page0, *acc_scratch;
  uint64_t* anc;
  float *attn_o, *attn_ml;
  int32_t* attn_tickets;
  size_t attn_units;  // capacity in (request x (splits+1)) units
  float* amax_val;
  int32_t* amax_idx;
  sdv::GemmWorkspace gws;
  std::map<int, sdv::XMap> map_xn, map_attn, map_act;
  std::vector<int32_t> cu_host;  // last uploaded cu
  int last_launches = 0;
  // captured steps: one executable graph per distinct argument set
  struct Graph {
    std::vector<uintptr_t> key;
    cudaGraphExec_t exec;
    int launches;
    std::vector<int32_t> t_kind;  // timeline entries captured with it
    std::vector<double> t_bytes;
  };
  std::vector<Graph> graphs;
  bool use_graphs = true;
  // the tensors' nested 8-bit planes (borrowed): [layer][qkv, o, gate_up,
  // down], then the lm_head; empty until sd_model_set_view8
  std::vector<const uint32_t*> view8;
  // streamed GEMM launches: per-site state (one site per launch of a step),
  // shared partials, per-row-block sums of squares of the residual stream
  int32_t* stream_state = nullptr;
  size_t site_ints = 0;
  int n_sites = 0;
  float* stream_part = nullptr;
  size_t stream_part_floats = 0;
  float* ss_h = nullptr;  // [H/128][128]: of h (O's output)
  float* ss_x = nullptr;  // [H/128][128]: of x (down's output)
  // optional per-kernel timing
  bool timing = false;  // events around every kernel launch
  bool fused = false;   // skinny steps: O..next q/k/v as one streamed launch
  std::vector<cudaEvent_t> events;  // 2 per entry
  std::vector<int32_t> t_kind;
  std::vector<double> t_bytes;
};

namespace sdv {

static size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// Prefix splits per (request, kv head, row chunk): about two CTAs per SM
// (the tensor-core latency chains of one warp bound the kernel, so more
// warps per SM and shorter key ranges per split pay for the larger merge),
// and at least one split per 1024 keys of the longest possible context (many
// requests: otherwise each CTA walks a whole context; 32 requests at ctx up
// to 4096 measured 19.65 / 19.69 / 20.09 ms per step at 4 / 5 / 9 splits).
// Prefix key splits per (request, kv head, row chunk): set by
// sd_attn_set_splits (<= 0: chosen from the grid and the context bound).
static int g_attn_splits = 0;

static int attn_splits(int R, int hkv, int chunks, int max_keys) {
  if (g_attn_splits > 0) return g_attn_splits;
  const int ctas = R * hkv * chunks;
  const int by_sms = (2 * num_sms() + ctas - 1) / ctas - 1;
  const int by_keys = (max_keys + 1023) / 1024;
  return std::max(1, std::min(64, std::max(by_sms, by_keys)));
}

static int get_map(std::map<int, XMap>& cache, const uint16_t* buf, int rows_total, int64_t K, int M, XMap** out) {
  const int box = M > 128 ? 128 : pad_rows(M);
  auto it = cache.find(box);
  if (it == cache.end()) {
    XMap xm;
    const int rc = make_x_map(&xm, buf, rows_total, K, box);
    if (rc) return rc;
    it = cache.emplace(box, xm).first;
  }
  *out = &it->second;
  return SD_OK;
}

struct StepIO {
  const int32_t* tokens;
  const int32_t* parents;
  int R, rows;
  CacheView cv;
  int32_t* accepted_len;
  int32_t* accepted_tokens;
  int32_t* bonus;
  uint16_t* logits;
  int32_t* argmax;
  bool commit;
  bool view8;  // round one of two-level verification: the weights' 8-bit view
};

static double gemm_bytes(const w12_tensor& W, int rows, int epi) {
  // packed words, escape tile index (entries and pointers), activations in,
  // outputs (+ residual) out
  double b = (double)W.N * W.K * 1.5 + (double)W.n_escapes * 4.0 + (double)w12_tile_ptr_count(W.N, W.K) * 4.0;
  b += (double)rows * W.K * 2.0;
  b += (double)rows * W.N * (epi == EPI_SILU ? 1.0 : 2.0);
  if (epi == EPI_RESID) b += (double)rows * W.N * 2.0;
  return b;
}

static int run_step(sd_model* m, const StepIO& io, cudaStream_t s) {
  // programmatic dependent launch between the step's kernels, except in the
  // per-kernel timing pass: there each kernel runs alone between its events
  // (with the attribute a kernel could start inside its predecessor's
  // bracket, and its own time would depend on its neighbours)
  const bool pdl = !m->timing;
  int launches = 0;
  const int rows = io.rows;
  int rc;
  m->t_kind.clear();
  m->t_bytes.clear();
  // bracket one launch with events when timing is on
  auto tbegin = [&](int kind, double bytes) -> int {
    if (!m->timing) return SD_OK;
    const size_t i = m->t_kind.size();
    while (m->events.size() < 2 * (i + 1)) {
      cudaEvent_t e;
      SD_CK(cudaEventCreate(&e));
      m->events.push_back(e);
    }
    m->t_kind.push_back(kind);
    m->t_bytes.push_back(bytes);
    SD_CK(cudaEventRecord(m->events[2 * i], s));
    return SD_OK;
  };
  auto tend = [&]() -> int {
    if (!m->timing) return SD_OK;
    SD_CK(cudaEventRecord(m->events[2 * (m->t_kind.size() - 1) + 1], s));
    return SD_OK;
  };
#define LK(kind, bytes, expr)                           \
  do {                                                  \
    if ((rc = tbegin(kind, bytes))) return rc;          \
    cudaError_t _e = (expr);                            \
    if (_e != cudaSuccess) return cuda_fail(_e, #expr); \
    if ((rc = tend())) return rc;                       \
    launches++;                                         \
  } while (0)

  // one launch per linear with RMSNorm kernels between them: the warp-level
  // kernel for skinny steps (rows <= 64 below the tensor-core threshold), the
  // tcgen05 kernel above; the 8-bit view streams its planes through the
  // weight-streaming kernel; fused (skinny steps): the GEMMs between two
  // attention / recurrence kernels as one launch of that kernel with the
  // RMSNorms folded in
  const bool skinny = rows <= kStreamMaxRows && !gemm_use_tc(rows);
  const bool fused = skinny && m->fused;
  if (io.view8 && (rows > kStreamMaxRows || m->view8.size() != (size_t)4 * m->cfg.n_layers + 1)) {
    set_error("model: the 8-bit view needs sd_model_set_view8 and at most 64 rows");
    return SD_ERR_UNSUPPORTED;
  }
  auto v8 = [&](int l, int k) -> const uint32_t* {
    return io.view8 ? m->view8[l < 0 ? 4 * m->cfg.n_layers : 4 * l + k] : nullptr;
  };
  int site = 0;
  std::vector<StreamPhaseDesc> ph;
  auto flush_stream = [&](int kind) -> int {
    if (ph.empty()) return SD_OK;
    if (site >= m->n_sites) {
      set_error("model: more streamed launches than sites");
      return SD_ERR_INVALID_ARG;
    }
    double bytes = 0.0;
    for (auto& d : ph) bytes += gemm_bytes(*d.W, rows, d.epi.epi);
    StreamWorkspace ws;
    ws.state = m->stream_state + (size_t)site * m->site_ints;
    ws.state_ints = m->site_ints;
    ws.partial = m->stream_part;
    ws.partial_floats = m->stream_part_floats;
    if ((rc = tbegin(kind, bytes))) return rc;
    if ((rc = stream_launch(ph.data(), (int)ph.size(), rows, ws, m->status, s, pdl))) return rc;
    if ((rc = tend())) return rc;
    launches++;
    site++;
    ph.clear();
    return SD_OK;
  };
  // one linear: the 8-bit view (plane) on the warp-level kernel in its
  // 8-bit mode (a contiguous exponent table; else the streaming kernel), the
  // fused schedule's first q/k/v on the streaming kernel; else the
  // warp-level kernel (skinny steps) or the tcgen05 kernel.  lm_part: the
  // argmax partials the lm_head launch leaves (one per CTA of its grid)
  int lm_part = gemm_grid(rows);
  auto gemm_one = [&](int kind, const w12_tensor& W, const uint16_t* x, const XMap* xm, const GemmEpilogue& e,
                      const uint32_t* plane) -> int {
    if (plane && !fused && W.affine && xm) {
      if ((rc = tbegin(kind, gemm_bytes(W, rows, e.epi) * (1.0 / 1.5)))) return rc;
      if ((rc = gemm_warp_launch(W, x, *xm, rows, e, m->gws, m->status, s, pdl, 0, nullptr, plane))) return rc;
      if ((rc = tend())) return rc;
      launches += gemm_kernel_count(W, rows, e.epi, gemm_warp_launch_grid(W, rows, e.epi));
      if (kind == SD_K_GEMM_LM_HEAD) lm_part = gemm_warp_grid(rows);
      return SD_OK;
    }
    if (plane || fused) {
      if (kind == SD_K_GEMM_LM_HEAD) lm_part = stream_grid(rows);
      StreamPhaseDesc d;
      d.W = &W;
      d.view8 = plane;
      d.x = x;
      d.x_rows = m->max_rows;
      d.epi = e;
      ph = {d};
      return flush_stream(kind);
    }
    if (!xm) {
      set_error("model: no activation tensor map for a GEMM launch");
      return SD_ERR_INVALID_ARG;
    }
    if ((rc = tbegin(kind, gemm_bytes(W, rows, e.epi)))) return rc;
    if ((rc = gemm_launch(W, x, *xm, rows, e, m->gws, m->status, s, pdl))) return rc;
    if ((rc = tend())) return rc;
    launches += gemm_kernel_count(W, rows, e.epi);
    return SD_OK;
  };
  auto norm = [&](const uint16_t* src, const uint16_t* gamma, uint16_t* dst) -> int {
    LK(SD_K_NORM, (double)rows * m->H * 4.0,
       launch_rmsnorm(src, gamma, rows, m->H, m->cfg.rms_eps, dst, nullptr, nullptr, nullptr, nullptr, nullptr, s, pdl));
    return SD_OK;
  };

  if (m->timing) {
    // let the host enqueue the whole step before the GPU starts on it
    const cudaError_t e = launch_delay(30000000ull, s);
    if (e != cudaSuccess) return cuda_fail(e, "delay");
  }
  XMap *mx = nullptr, *ma = nullptr, *mc = nullptr;
  if (!fused) {
    if ((rc = get_map(m->map_xn, m->xn, m->max_rows, m->H, rows, &mx))) return rc;
    if ((rc = get_map(m->map_attn, m->attn, m->max_rows, (int64_t)m->Hq * m->hd, rows, &ma))) return rc;
    if ((rc = get_map(m->map_act, m->act, m->max_rows, m->I, rows, &mc))) return rc;
  }

  const StepRows sr{m->ctx_snap, m->req_ok, m->pos, m->slotv, m->req, m->depth, m->anc};
  // the step's first kernel starts only after the previous step (its KV
  // commit) is complete: later kernels of the step may read the committed
  // prefix before their programmatic-launch wait
  LK(SD_K_TREE, 0.0,
     launch_tree(io.tokens, io.parents, m->cu, io.R, io.cv, m->V, m->cfg.max_positions, sr, m->status, s, false));
  LK(SD_K_NORM, (double)rows * m->H * 4.0,
     launch_rmsnorm(nullptr, m->layers[0].attn_norm, rows, m->H, m->cfg.rms_eps, m->xn, io.tokens, m->w.embed, m->x,
                    m->req, m->req_ok, s, pdl));

  // row chunks of the attention grid: the largest request of this call
  int max_mr = 1;
  for (int r = 0; r < io.R && r + 1 < (int)m->cu_host.size(); r++)
    max_mr = std::max(max_mr, m->cu_host[r + 1] - m->cu_host[r]);
  max_mr = std::min(max_mr, m->max_m);
  const int chunks = attn_chunks(attn_rows_per_group(m->Hq, m->Hkv, max_mr));
  int splits = attn_splits(io.R, m->Hkv, chunks, m->cfg.max_positions);
  while (splits > 1 && (size_t)io.R * (splits + 1) > m->attn_units) splits--;
  const int64_t layer_elems = (int64_t)io.cv.n_pages * m->Hkv * io.cv.page_size * m->hd;

  // epilogue of layer l's q/k/v GEMM
  auto qkv_epi = [&](int l) {
    GemmEpilogue eq;
    const int ls = m->slot[l];
    if (m->kind[l] == 0) {
      eq.epi = EPI_QKV;
      eq.q_out = m->q;
      eq.hq = m->Hq;
      eq.hkv = m->Hkv;
      eq.cache.k = io.cv.k_pool + ls * layer_elems;
      eq.cache.v = io.cv.v_pool + ls * layer_elems;
      eq.cache.page_table = io.cv.page_table;
      eq.cache.max_pages = io.cv.max_pages;
      eq.cache.page_size = io.cv.page_size;
      eq.cache.hkv = m->Hkv;
      eq.rows = RowInfo{m->pos, m->slotv, m->req, m->req_ok};
      eq.rope_cos = m->rope_cos;
      eq.rope_sin = m->rope_sin;
    } else {
      eq.epi = EPI_STORE;
      eq.out = m->qkv_rec + (int64_t)ls * m->max_rows * 3 * m->H;
      eq.ldo = 3 * m->H;
    }
    return eq;
  };
  GemmEpilogue el;  // lm_head: logits + argmax partials
  el.epi = EPI_LOGITS;
  el.out = io.logits;
  el.ldo = m->V;
  el.amax_val = m->amax_val;
  el.amax_idx = m->amax_idx;
  el.ld_amax = m->max_rows;

  if ((rc = gemm_one(SD_K_GEMM_QKV, m->layers[0].qkv, m->xn, mx, qkv_epi(0), v8(0, 0)))) return rc;

  for (int l = 0; l < m->cfg.n_layers; l++) {
    const sd_layer_weights& Lw = m->layers[l];
    const bool is_attn = m->kind[l] == 0;
    const int ls = m->slot[l];
    if (is_attn) {
      AttnArgs aa{};
      aa.q = m->q;
      aa.k_pool = io.cv.k_pool + ls * layer_elems;
      aa.v_pool = io.cv.v_pool + ls * layer_elems;
      aa.page_table = io.cv.page_table;
      aa.max_pages = io.cv.max_pages;
      aa.page_size = io.cv.page_size;
      aa.hq = m->Hq;
      aa.hkv = m->Hkv;
      aa.cu = m->cu;
      aa.ctx = m->ctx_snap;
      aa.ctx_in = io.cv.ctx_len;
      aa.n_pages = io.cv.n_pages;
      aa.anc = m->anc;
      aa.row_req = m->req;
      aa.req_ok = m->req_ok;
      aa.R = io.R;
      aa.max_m = m->max_m;
      aa.chunk_m = max_mr;
      aa.splits = splits;
      aa.part_o = m->attn_o;
      aa.part_ml = m->attn_ml;
      aa.tickets = m->attn_tickets;
      aa.status = m->status;
      aa.out = m->attn;
      LK(SD_K_ATTN, 0.0, launch_attention(aa, rows, s, pdl));
    } else {
      LinrecArgs la{};
      la.qkv = m->qkv_rec + (int64_t)ls * m->max_rows * 3 * m->H;
      const int64_t per_layer_S = (int64_t)m->nh_rec * m->hd * m->hd, per_layer_z = (int64_t)m->nh_rec * m->hd;
      la.S = io.cv.S + ls * per_layer_S;
      la.z = io.cv.z + ls * per_layer_z;
      la.req_stride_S = per_layer_S * m->n_rec;
      la.req_stride_z = per_layer_z * m->n_rec;
      la.cu = m->cu;
      la.anc = m->anc;
      la.R = io.R;
      la.nh = m->nh_rec;
      la.H = m->H;
      la.eps = m->cfg.rec_eps;
      la.out = m->attn;
      LK(SD_K_LINREC, 0.0, launch_linrec(la, s, pdl));
    }
    GemmEpilogue eo;  // h = x + O(attn)
    eo.epi = EPI_RESID;
    eo.out = m->h;
    eo.resid = m->x;
    eo.ldo = m->H;
    GemmEpilogue eg;  // act = silu(gate) * up
    eg.epi = EPI_SILU;
    eg.out = m->act;
    eg.ldo = m->I;
    GemmEpilogue ed;  // x = h + down(act)
    ed.epi = EPI_RESID;
    ed.out = m->x;
    ed.resid = m->h;
    ed.ldo = m->H;
    const bool last = l + 1 == m->cfg.n_layers;
    const uint16_t* gnext = last ? m->w.final_norm : m->layers[l + 1].attn_norm;
    if (fused) {
      StreamPhaseDesc o, g, d, n;
      o.W = &Lw.o;
      o.view8 = v8(l, 1);
      o.x = m->attn;
      o.x_rows = m->max_rows;
      o.epi = eo;
      o.out_ss = m->ss_h;
      g.W = &Lw.gate_up;
      g.view8 = v8(l, 2);
      g.x = m->h;
      g.x_rows = m->max_rows;
      g.epi = eg;
      g.dep = 0;
      g.norm_gamma = Lw.mlp_norm;
      g.norm_eps = m->cfg.rms_eps;
      d.W = &Lw.down;
      d.view8 = v8(l, 3);
      d.x = m->act;
      d.x_rows = m->max_rows;
      d.epi = ed;
      d.dep = 1;
      d.dep_fine = 1;
      d.out_ss = m->ss_x;
      n.W = last ? &m->w.lm_head : &m->layers[l + 1].qkv;
      n.view8 = last ? v8(-1, 0) : v8(l + 1, 0);
      n.x = m->x;
      n.x_rows = m->max_rows;
      n.epi = last ? el : qkv_epi(l + 1);
      n.dep = 2;
      n.norm_gamma = gnext;
      n.norm_eps = m->cfg.rms_eps;
      n.norm_out = last ? m->xn : nullptr;  // the final hidden state (the lm_head's input), kept for the tap
      ph = {o, g, d, n};
      if ((rc = flush_stream(SD_K_GEMM_STREAM))) return rc;
    } else {
      if ((rc = gemm_one(SD_K_GEMM_O, Lw.o, m->attn, ma, eo, v8(l, 1)))) return rc;
      if ((rc = norm(m->h, Lw.mlp_norm, m->xn))) return rc;
      if ((rc = gemm_one(SD_K_GEMM_GATE_UP, Lw.gate_up, m->xn, mx, eg, v8(l, 2)))) return rc;
      if ((rc = gemm_one(SD_K_GEMM_DOWN, Lw.down, m->act, mc, ed, v8(l, 3)))) return rc;
      if ((rc = norm(m->x, gnext, m->xn))) return rc;
      if (last) {
        if ((rc = gemm_one(SD_K_GEMM_LM_HEAD, m->w.lm_head, m->xn, mx, el, v8(-1, 0)))) return rc;
      } else {
        if ((rc = gemm_one(SD_K_GEMM_QKV, m->layers[l + 1].qkv, m->xn, mx, qkv_epi(l + 1), v8(l + 1, 0)))) return rc;
      }
    }
  }

  AcceptArgs ac{};
  ac.tokens = io.tokens;
  ac.parents = io.parents;
  ac.cu = m->cu;
  ac.R = io.R;
  ac.amax_val = m->amax_val;
  ac.amax_idx = m->amax_idx;
  ac.n_part = fused ? stream_grid(rows) : lm_part;  // the lm_head's argmax partials
  ac.ld = m->max_rows;
  ac.req_ok = m->req_ok;
  ac.ctx_snap = m->ctx_snap;
  ac.ctx_len = io.commit ? io.cv.ctx_len : nullptr;
  ac.argmax_out = io.argmax;
  ac.accepted_len = io.accepted_len;
  ac.accepted_tokens = io.accepted_tokens;
  ac.bonus = io.bonus;
  ac.path = m->path;
  ac.path_len = m->path_len;
  ac.status = m->status;
  LK(SD_K_ACCEPT, 0.0, launch_accept(ac, s, pdl));
  if (io.commit) {
    if (m->n_attn)
      LK(SD_K_COMMIT, 0.0, launch_compact(io.cv, m->n_attn, m->Hkv, io.R, m->ctx_snap, m->path, m->path_len, s, pdl));
    if (m->n_rec)
      LK(SD_K_COMMIT, 0.0,
         launch_rec_commit(io.cv, m->n_rec, m->nh_rec, m->H, io.R, m->max_rows, m->qkv_rec, m->cu, m->path,
                           m->path_len, s, pdl));
  }
#undef LK
  m->last_launches = launches;
  return SD_OK;
}

// Enqueue one step.  On a non-default stream that is not already capturing,
// the step is captured once per distinct argument set into a CUDA graph and
// replayed from then on (no per-kernel host launch cost); the captured
// kernels keep their programmatic-dependent-launch edges.  The key holds
// every pointer and size the kernels see, so a replay is the same launch
// sequence; values behind the pointers are read at run time.
static int launch_step(sd_model* m, const StepIO& io, cudaStream_t s, std::vector<uintptr_t> key) {
  if (!m->use_graphs || m->timing || s == nullptr) return run_step(m, io, s);
  key.push_back((uintptr_t)gemm_tc_min_rows());
  key.push_back((uintptr_t)g_attn_splits);
  key.push_back((uintptr_t)gemm_finish_mode());
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  SD_CK(cudaStreamIsCapturing(s, &cs));
  if (cs != cudaStreamCaptureStatusNone) return run_step(m, io, s);
  for (auto& g : m->graphs)
    if (g.key == key) {
      SD_CK(cudaGraphLaunch(g.exec, s));
      m->last_launches = g.launches;
      m->t_kind = g.t_kind;
      m->t_bytes = g.t_bytes;
      return SD_OK;
    }
  SD_CK(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
  const int rc = run_step(m, io, s);
  cudaGraph_t graph = nullptr;
  const cudaError_t e = cudaStreamEndCapture(s, &graph);
  if (rc) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  SD_CK(e);
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  SD_CK(ei);
  if (m->graphs.size() >= 16) {
    cudaGraphExecDestroy(m->graphs.front().exec);
    m->graphs.erase(m->graphs.begin());
  }
  m->graphs.push_back({key, exec, m->last_launches, m->t_kind, m->t_bytes});
  SD_CK(cudaGraphLaunch(exec, s));
  return SD_OK;
}

static std::vector<uintptr_t> step_key(const StepIO& io, int M) {
  auto u = [](const void* p) { return reinterpret_cast<uintptr_t>(p); };
  return {(uintptr_t)M, (uintptr_t)io.R, (uintptr_t)io.rows, u(io.tokens), u(io.parents), u(io.cv.k_pool),
          u(io.cv.v_pool), (uintptr_t)io.cv.n_pages, (uintptr_t)io.cv.page_size, u(io.cv.page_table),
          (uintptr_t)io.cv.max_pages, u(io.cv.S), u(io.cv.z), u(io.cv.ctx_len), u(io.accepted_len),
          u(io.accepted_tokens), u(io.bonus), u(io.logits), u(io.argmax), (uintptr_t)io.commit,
          (uintptr_t)io.view8};
}

static int upload_cu(sd_model* m, const std::vector<int32_t>& cu, cudaStream_t s) {
  if (cu != m->cu_host) {
    SD_CK(cudaMemcpyAsync(m->cu, cu.data(), cu.size() * sizeof(int32_t), cudaMemcpyHostToDevice, s));
    SD_CK(cudaStreamSynchronize(s));
    m->cu_host = cu;
  }
  return SD_OK;
}

}  // namespace sdv

using namespace sdv;

extern "C" int sd_model_row_map(int32_t kind, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t inter,
                                int32_t* out_host, int64_t N) {
  if (!out_host || N <= 0) {
    set_error("sd_model_row_map: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (kind == 0) {
    if (head_dim != 128 || N != (int64_t)(n_q_heads + 2 * n_kv_heads) * head_dim) {
      set_error("sd_model_row_map: qkv rows must be (Hq + 2 Hkv) * 128");
      return SD_ERR_INVALID_ARG;
    }
    const int64_t rope_rows = (int64_t)(n_q_heads + n_kv_heads) * head_dim;
    for (int64_t n = 0; n < N; n++) {
      if (n >= rope_rows) {
        out_host[n] = (int32_t)n;
        continue;
      }
      const int64_t head = n / 128, r = n % 128, strip = r / 16, w = r % 16;
      const int64_t dim = w < 8 ? strip * 8 + w : 64 + strip * 8 + (w - 8);
      out_host[n] = (int32_t)(head * 128 + dim);
    }
  } else if (kind == 1) {
    if (N != 2 * (int64_t)inter || inter % 8) {
      set_error("sd_model_row_map: gate_up rows must be 2 * inter, inter % 8 == 0");
      return SD_ERR_INVALID_ARG;
    }
    for (int64_t n = 0; n < N; n++) {
      const int64_t j = n / 16, w = n % 16;
      out_host[n] = (int32_t)(w < 8 ? j * 8 + w : inter + j * 8 + (w - 8));
    }
  } else if (kind == 2) {
    for (int64_t n = 0; n < N; n++) out_host[n] = (int32_t)n;
  } else {
    set_error("sd_model_row_map: unknown kind");
    return SD_ERR_INVALID_ARG;
  }
  return SD_OK;
}

static bool tensor_ok(const w12_tensor& t, int64_t N, int64_t K) {
  return t.words && t.N == N && t.K == K && (t.n_escapes == 0 || (t.tile_ptr && t.tile_esc));
}

extern "C" int sd_model_create(const sd_model_config* cfg, const sd_model_weights* w, sd_model** out) {
  if (!cfg || !w || !out || !cfg->layer_kind_host || !w->layers_host || !w->embed || !w->final_norm) {
    set_error("sd_model_create: null argument");
    return SD_ERR_INVALID_ARG;
  }
  const sd_model_config& c = *cfg;
  if (c.n_layers < 1 || c.head_dim != 128 || c.hidden % 64 || c.inter % 64 || c.n_q_heads < 1 || c.n_kv_heads < 1 ||
      c.n_q_heads % c.n_kv_heads || c.n_q_heads * 128 != c.hidden || c.vocab % 16 || c.max_rows < 1 ||
      c.max_rows > 256 || c.max_requests < 1 || c.max_positions < 2) {
    set_error("sd_model_create: unsupported config (head_dim 128, n_q_heads*128 == hidden, hidden/inter % 64, "
              "vocab % 16, max_rows <= 256)");
    return SD_ERR_UNSUPPORTED;
  }
  for (int l = 0; l < c.n_layers; l++)
    if (c.layer_kind_host[l] != 0 && c.layer_kind_host[l] != 1) {
      set_error("sd_model_create: layer_kind must be 0 or 1");
      return SD_ERR_INVALID_ARG;
    }
  sd_model* m = new sd_model();
  m->cfg = c;
  m->H = c.hidden;
  m->I = c.inter;
  m->Hq = c.n_q_heads;
  m->Hkv = c.n_kv_heads;
  m->hd = c.head_dim;
  m->V = c.vocab;
  m->max_rows = c.max_rows;
  m->max_req = c.max_requests;
  m->max_m = std::min(64, c.max_rows);
  m->nh_rec = c.hidden / 128;
  m->kind.assign(c.layer_kind_host, c.layer_kind_host + c.n_layers);
  m->layers.assign(w->layers_host, w->layers_host + c.n_layers);
  m->w = *w;
  int64_t max_n = m->V;
  for (int l = 0; l < c.n_layers; l++) {
    m->slot.push_back(m->kind[l] == 0 ? m->n_attn++ : m->n_rec++);
    const sd_layer_weights& L = m->layers[l];
    const int64_t qkv_rows = m->kind[l] == 0 ? (int64_t)(m->Hq + 2 * m->Hkv) * 128 : 3 * (int64_t)m->H;
    if (!tensor_ok(L.qkv, qkv_rows, m->H) || !tensor_ok(L.o, m->H, m->H) ||
        !tensor_ok(L.gate_up, 2 * (int64_t)m->I, m->H) || !tensor_ok(L.down, m->H, m->I) || !L.attn_norm ||
        !L.mlp_norm) {
      delete m;
      set_error("sd_model_create: layer " + std::to_string(l) + " weights missing or of the wrong shape");
      return SD_ERR_INVALID_ARG;
    }
    max_n = std::max(max_n, std::max<int64_t>(L.qkv.N, L.gate_up.N));
  }
  if (!tensor_ok(w->lm_head, m->V, m->H)) {
    delete m;
    set_error("sd_model_create: lm_head missing or of the wrong shape");
    return SD_ERR_INVALID_ARG;
  }
  // ---- workspace (one allocation)
  const int MR = m->max_rows, R = m->max_req;
  const int rpg = attn_rows_per_group(m->Hq, m->Hkv, m->max_m);
  // tickets are indexed by the grid's row chunk: size them for the most
  // chunks any call can use (32-row chunks when groups are small)
  const int chunks = std::max(attn_chunks(rpg), (rpg + 31) / 32);
  size_t units = 0;
  for (int ch = 1; ch <= chunks; ch++)
    for (int r = 1; r <= R; r++)
      units = std::max(units, (size_t)r * (attn_splits(r, m->Hkv, ch, c.max_positions) + 1));
  m->attn_units = units;
  // streamed launches of a step: one per linear, or (fused) [q/k/v of
  // layer 0], then per layer [O, gate/up, down, next q/k/v or lm_head];
  // scratch for the largest of them at any row count the model accepts
  {
    size_t ints = 0, floats = 0;
    for (int l = -1; l < c.n_layers; l++) {
      StreamPhaseDesc d[4];
      int n = 0;
      if (l < 0) {
        d[n++].W = &m->layers[0].qkv;
      } else {
        d[n++].W = &m->layers[l].o;
        d[n++].W = &m->layers[l].gate_up;
        d[n++].W = &m->layers[l].down;
        d[n++].W = l + 1 < c.n_layers ? &m->layers[l + 1].qkv : &m->w.lm_head;
      }
      ints = std::max(ints, stream_state_ints(d, n));
      for (int rows = 1; rows <= std::min(MR, kStreamMaxRows); rows *= 2)
        floats = std::max(floats, stream_partial_floats(d, n, rows));
      floats = std::max(floats, stream_partial_floats(d, n, std::min(MR, kStreamMaxRows)));
    }
    m->site_ints = (ints + 63) & ~size_t(63);
    m->n_sites = 4 * c.n_layers + 1;  // one per linear (the fused schedule uses n_layers + 1)
    m->stream_part_floats = std::max<size_t>(floats, 4);
  }
  struct Item {
    void** p;
    size_t bytes;
  };
  const std::vector<Item> items = {
      {(void**)&m->x, (size_t)MR * m->H * 2},
      {(void**)&m->h, (size_t)MR * m->H * 2},
      {(void**)&m->xn, (size_t)MR * m->H * 2},
      {(void**)&m->q, (size_t)MR * m->Hq * 128 * 2},
      {(void**)&m->attn, (size_t)MR * m->H * 2},
      {(void**)&m->act, (size_t)MR * m->I * 2},
      {(void**)&m->qkv_rec, (size_t)std::max(1, m->n_rec) * MR * 3 * m->H * 2},
      {(void**)&m->rope_cos, (size_t)c.max_positions * 64 * 4},
      {(void**)&m->rope_sin, (size_t)c.max_positions * 64 * 4},
      {(void**)&m->ctx_snap, (size_t)R * 4},
      {(void**)&m->req_ok, (size_t)R * 4},
      {(void**)&m->pos, (size_t)MR * 4},
      {(void**)&m->slotv, (size_t)MR * 4},
      {(void**)&m->req, (size_t)MR * 4},
      {(void**)&m->depth, (size_t)MR * 4},
      {(void**)&m->path, (size_t)R * 65 * 4},
      {(void**)&m->path_len, (size_t)R * 4},
      {(void**)&m->status, 4},
      {(void**)&m->cu, (size_t)(R + 1) * 4},
      {(void**)&m->page0, 4},
      {(void**)&m->acc_scratch, (size_t)(2 * R + MR) * 4},
      {(void**)&m->anc, (size_t)MR * 8},
      {(void**)&m->attn_o, units * m->Hkv * rpg * 128 * 4},
      {(void**)&m->attn_ml, units * m->Hkv * rpg * 2 * 4},
      {(void**)&m->attn_tickets, (size_t)R * m->Hkv * chunks * 2 * 4},
      // one argmax partial per CTA of the widest GEMM grid (two per SM)
      {(void**)&m->amax_val, (size_t)2 * num_sms() * MR * 4},
      {(void**)&m->amax_idx, (size_t)2 * num_sms() * MR * 4},
      {(void**)&m->gws.partial, gemm_partial_floats(MR) * 4},
      {(void**)&m->gws.counters, (size_t)gemm_counters(max_n) * 4},
      {(void**)&m->stream_state, (size_t)m->n_sites * m->site_ints * 4},
      {(void**)&m->stream_part, m->stream_part_floats * 4},
      {(void**)&m->ss_h, (size_t)((m->H + 127) / 128) * 128 * 4},
      {(void**)&m->ss_x, (size_t)((m->H + 127) / 128) * 128 * 4},
  };
  size_t total = 0;
  for (auto& it : items) total = al256(total + it.bytes);
  cudaError_t e = cudaMalloc(&m->arena, total);
  if (e != cudaSuccess) {
    delete m;
    return cuda_fail(e, "sd_model_create: cudaMalloc");
  }
  size_t off = 0;
  for (auto& it : items) {
    *it.p = static_cast<uint8_t*>(m->arena) + off;
    off = al256(off + it.bytes);
  }
  m->gws.partial_floats = gemm_partial_floats(MR);
  m->gws.counters_len = gemm_counters(max_n);
  e = cudaMemset(m->arena, 0, total);
  // RoPE table: theta = pos * base^(-2d/128), d < 64
  std::vector<float> cs((size_t)c.max_positions * 64), sn((size_t)c.max_positions * 64);
  for (int d = 0; d < 64; d++) {
    const double inv = std::pow((double)c.rope_base, -2.0 * d / 128.0);
    for (int p = 0; p < c.max_positions; p++) {
      const double th = (double)p * inv;
      cs[(size_t)p * 64 + d] = (float)std::cos(th);
      sn[(size_t)p * 64 + d] = (float)std::sin(th);
    }
  }
  if (e == cudaSuccess) e = cudaMemcpy(m->rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(m->rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(m->arena);
    delete m;
    return cuda_fail(e, "sd_model_create: init");
  }
  *out = m;
  return SD_OK;
}

extern "C" int32_t sd_attn_set_splits(int32_t splits) {
  g_attn_splits = splits > 0 ? std::min(splits, 64) : 0;
  return g_attn_splits;
}

extern "C" int sd_model_destroy(sd_model* m) {
  if (!m) return SD_OK;
  for (auto& g : m->graphs) cudaGraphExecDestroy(g.exec);
  for (cudaEvent_t e : m->events) cudaEventDestroy(e);
  cudaFree(m->arena);
  delete m;
  return SD_OK;
}

static int single_step(sd_model* m, const int32_t* tokens, const int32_t* parents, int32_t M, const sd_kv* kv,
                       int32_t* accepted_len, int32_t* accepted_tokens, int32_t* bonus, uint16_t* logits,
                       int32_t* argmax, bool commit, void* stream, bool view8 = false) {
  if (!m || !tokens || !parents || !kv || !kv->k || !kv->v || !kv->ctx_len || M < 1) {
    set_error("sd_verify_step: null argument");
    return SD_ERR_INVALID_ARG;
  }
  if (M > 64 || M > m->max_rows || kv->cap < 1 || kv->cap > (1 << 30)) {
    set_error("sd_verify_step: M must be <= 64 and <= max_rows");
    return SD_ERR_UNSUPPORTED;
  }
  if (m->n_rec && (!kv->S || !kv->z)) {
    set_error("sd_verify_step: hybrid model needs kv->S and kv->z");
    return SD_ERR_INVALID_ARG;
  }
  if (commit && (!accepted_len || !accepted_tokens || !bonus)) {
    set_error("sd_verify_step: outputs missing");
    return SD_ERR_INVALID_ARG;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int rc = upload_cu(m, {0, M}, s);
  if (rc) return rc;
  StepIO io{};
  io.tokens = tokens;
  io.parents = parents;
  io.R = 1;
  io.rows = M;
  io.cv = CacheView{kv->k, kv->v, 1, (int32_t)kv->cap, m->page0, 1, kv->S, kv->z, kv->ctx_len};
  io.accepted_len = accepted_len;
  io.accepted_tokens = accepted_tokens;
  io.bonus = bonus;
  if (!commit) {
    // forward-only: acceptance results go to private scratch
    io.accepted_len = m->acc_scratch;
    io.bonus = m->acc_scratch + m->max_req;
    io.accepted_tokens = m->acc_scratch + 2 * m->max_req;
  }
  io.logits = logits;
  io.argmax = argmax;
  io.commit = commit;
  io.view8 = view8;
  return launch_step(m, io, s, step_key(io, M));
}

extern "C" int sd_verify_step(sd_model* m, const int32_t* tree_tokens, const int32_t* parents, int32_t M,
                              const sd_kv* kv, int32_t* accepted_len, int32_t* accepted_tokens, int32_t* bonus_token,
                              uint16_t* logits, int32_t* argmax, void* stream) {
  return single_step(m, tree_tokens, parents, M, kv, accepted_len, accepted_tokens, bonus_token, logits, argmax, true,
                     stream);
}

extern "C" int sd_forward(sd_model* m, const int32_t* tree_tokens, const int32_t* parents, int32_t M, const sd_kv* kv,
                          uint16_t* logits, int32_t* argmax, void* stream) {
  return single_step(m, tree_tokens, parents, M, kv, nullptr, nullptr, nullptr, logits, argmax, false, stream);
}

extern "C" int sd_forward_view8(sd_model* m, const int32_t* tree_tokens, const int32_t* parents, int32_t M,
                                const sd_kv* kv, uint16_t* logits, int32_t* argmax, void* stream) {
  return single_step(m, tree_tokens, parents, M, kv, nullptr, nullptr, nullptr, logits, argmax, false, stream, true);
}

extern "C" int sd_model_set_view8(sd_model* m, const uint32_t* const* planes_host, int32_t n) {
  if (!m || !planes_host || n != 4 * m->cfg.n_layers + 1) {
    set_error("sd_model_set_view8: need 4 planes per layer (qkv, o, gate_up, down) and the lm_head's");
    return SD_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n; i++)
    if (!planes_host[i] || (reinterpret_cast<uintptr_t>(planes_host[i]) & 15)) {
      set_error("sd_model_set_view8: null or unaligned plane");
      return SD_ERR_INVALID_ARG;
    }
  m->view8.assign(planes_host, planes_host + n);
  for (auto& g : m->graphs) cudaGraphExecDestroy(g.exec);  // captured steps may hold the old planes
  m->graphs.clear();
  return SD_OK;
}

extern "C" int sd_verify_batch(sd_model* m, const int32_t* tokens, const int32_t* parents, const int32_t* cu_nodes_host,
                               int32_t R, const sd_paged_kv* kv, int32_t* accepted_len, int32_t* accepted_tokens,
                               int32_t* bonus, uint16_t* logits, int32_t* argmax, void* stream) {
  if (!m || !tokens || !parents || !cu_nodes_host || !kv || !kv->k_pool || !kv->v_pool || !kv->page_table ||
      !kv->ctx_len || !accepted_len || !accepted_tokens || !bonus || R < 1) {
    set_error("sd_verify_batch: null argument");
    return SD_ERR_INVALID_ARG;
  }
  if (R > m->max_req || cu_nodes_host[0] != 0 || kv->page_size < 1 || kv->max_pages < 1 || kv->n_pages < 1) {
    set_error("sd_verify_batch: R > max_requests or bad cu_nodes / pages");
    return SD_ERR_INVALID_ARG;
  }
  const std::vector<int32_t> cu(cu_nodes_host, cu_nodes_host + R + 1);
  for (int r = 0; r < R; r++)
    if (cu[r + 1] - cu[r] < 1 || cu[r + 1] - cu[r] > m->max_m) {
      set_error("sd_verify_batch: each request needs 1..64 nodes");
      return SD_ERR_UNSUPPORTED;
    }
  if (cu[R] > m->max_rows) {
    set_error("sd_verify_batch: total nodes exceed max_rows");
    return SD_ERR_UNSUPPORTED;
  }
  if (m->n_rec && (!kv->S || !kv->z)) {
    set_error("sd_verify_batch: hybrid model needs S and z");
    return SD_ERR_INVALID_ARG;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int rc = upload_cu(m, cu, s);
  if (rc) return rc;
  StepIO io{};
  io.tokens = tokens;
  io.parents = parents;
  io.R = R;
  io.rows = cu[R];
  io.cv = CacheView{kv->k_pool, kv->v_pool, kv->n_pages, kv->page_size, kv->page_table, kv->max_pages,
                    kv->S, kv->z, kv->ctx_len};
  io.accepted_len = accepted_len;
  io.accepted_tokens = accepted_tokens;
  io.bonus = bonus;
  io.logits = logits;
  io.argmax = argmax;
  io.commit = true;
  std::vector<uintptr_t> key = step_key(io, io.rows);
  for (int32_t c : cu) key.push_back((uintptr_t)(uint32_t)c);
  return launch_step(m, io, s, key);
}

extern "C" int sd_status(sd_model* m, int32_t* status_host) {
  if (!m || !status_host) {
    set_error("sd_status: null argument");
    return SD_ERR_INVALID_ARG;
  }
  SD_CK(cudaDeviceSynchronize());
  SD_CK(cudaMemcpy(status_host, m->status, 4, cudaMemcpyDeviceToHost));
  SD_CK(cudaMemset(m->status, 0, 4));
  // a streamed launch that gave up on a wait may have left its unit
  // counters, tickets or flags set: start the next step from zero
  if (*status_host != SD_OK) SD_CK(cudaMemset(m->stream_state, 0, (size_t)m->n_sites * m->site_ints * 4));
  return SD_OK;
}

extern "C" int sd_model_last_launches(sd_model* m) { return m ? m->last_launches : 0; }

extern "C" int sd_model_final_hidden(sd_model* m, uint16_t* out, int32_t rows, void* stream) {
  if (!m || !out || rows < 1 || rows > m->max_rows) {
    set_error("sd_model_final_hidden: bad argument (rows must be 1..max_rows)");
    return SD_ERR_INVALID_ARG;
  }
  SD_CK(cudaMemcpyAsync(out, m->xn, (size_t)rows * m->H * sizeof(uint16_t), cudaMemcpyDeviceToDevice,
                        (cudaStream_t)stream));
  return SD_OK;
}

extern "C" int sd_model_set_fused(sd_model* m, int32_t enable) {
  if (!m) {
    set_error("sd_model_set_fused: null model");
    return SD_ERR_INVALID_ARG;
  }
  if ((enable != 0) != m->fused) {
    for (auto& g : m->graphs) cudaGraphExecDestroy(g.exec);  // captured steps follow the old schedule
    m->graphs.clear();
  }
  m->fused = enable != 0;
  return SD_OK;
}

extern "C" int sd_model_set_timing(sd_model* m, int32_t enable) {
  if (!m) {
    set_error("sd_model_set_timing: null model");
    return SD_ERR_INVALID_ARG;
  }
  m->timing = enable != 0;
  return SD_OK;
}

extern "C" int sd_model_timeline(sd_model* m, int32_t max, int32_t* kind_host, float* ms_host, double* bytes_host) {
  if (!m || max < 0 || (max > 0 && (!kind_host || !ms_host || !bytes_host))) {
    set_error("sd_model_timeline: bad argument");
    return -1;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) {
    set_error("sd_model_timeline: device error");
    return -1;
  }
  int n = 0;
  for (size_t i = 0; i < m->t_kind.size() && n < max; i++) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, m->events[2 * i], m->events[2 * i + 1]) != cudaSuccess) ms = -1.f;
    kind_host[n] = m->t_kind[i];
    ms_host[n] = ms;
    bytes_host[n] = m->t_bytes[i];
    n++;
  }
  return n;
}

extern "C" int sd_model_set_graphs(sd_model* m, int32_t enable) {
  if (!m) {
    set_error("sd_model_set_graphs: null model");
    return SD_ERR_INVALID_ARG;
  }
  m->use_graphs = enable != 0;
  return SD_OK;
}
