// Verify-step orchestration: model object, workspace, kernel sequence.
//
// One step = tree bookkeeping -> embedding + RMSNorm -> per layer
// [QKV GEMM (+RoPE, K/V write) -> tree attention (or linear recurrence)
//  -> O GEMM (+residual) -> RMSNorm -> gate/up GEMM (+SiLU*up)
//  -> down GEMM (+residual) -> RMSNorm] -> lm_head GEMM (+argmax)
// -> greedy acceptance -> K/V compaction / state commit.
// Every kernel is launched with programmatic dependent launch, so a GEMM's
// producer streams its weights while the previous kernel is still finishing.
// With the chain enabled (up to 128 rows; off by default), each run of GEMMs
// and RMSNorms between two attention (or recurrence) kernels - O, RMSNorm,
// gate/up, down, RMSNorm, next q/k/v or lm_head - is one persistent launch.
#include <algorithm>
#include <cmath>
#include <map>
#include <vector>

#include "chain.cuh"
#include "gemm.cuh"
#include "layers.cuh"

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
  bool use_chain = false;
  unsigned long long* chain_bar;  // grid-barrier words of the chain kernel (counter, base)
  // optional per-kernel timing
  bool timing = false;   // events around every kernel group (+ device-clock traces)
  bool tracing = false;  // device-clock traces only: launches as in untimed steps (no graph)
  std::vector<cudaEvent_t> events;  // 2 per entry
  std::vector<int32_t> t_kind;
  std::vector<double> t_bytes;
  // per-phase stamps of the chain launches of a timed step
  uint64_t* trace = nullptr;
  size_t trace_cap = 0;  // u64 entries
  struct ChainRec {
    size_t entry, off;
    int n, G;
    std::vector<int32_t> kinds;
    std::vector<double> bytes;
  };
  std::vector<ChainRec> t_chain;
};

namespace sdv {

static size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// Prefix splits per (request, kv head, row chunk): about two CTAs per SM
// (the tensor-core latency chains of one warp bound the kernel, so more
// warps per SM and shorter key ranges per split pay for the larger merge),
// and at least one split per 512 keys of the longest possible context (many
// requests: otherwise each CTA walks a whole context).
// Prefix key splits per (request, kv head, row chunk): set by
// sd_attn_set_splits (<= 0: chosen from the grid and the context bound).
static int g_attn_splits = 0;

static int attn_splits(int R, int hkv, int chunks, int max_keys) {
  if (g_attn_splits > 0) return g_attn_splits;
  const int ctas = R * hkv * chunks;
  const int by_sms = (2 * num_sms() + ctas - 1) / ctas - 1;
  const int by_keys = (max_keys + 511) / 512;
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
};

static int run_step(sd_model* m, const StepIO& io, cudaStream_t s) {
  const bool pdl = true;
  int launches = 0;
  const int rows = io.rows;
  int rc;
  m->t_kind.clear();
  m->t_bytes.clear();
  m->t_chain.clear();
  size_t trace_off = 0;
  // bracket one kernel group with events when timing is on
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
  auto gbytes = [&](const w12_tensor& W, int epi) -> double {
    // packed words, escape tile index (entries and pointers)
    double b = (double)W.N * W.K * 1.5 + (double)W.n_escapes * 4.0 + (double)w12_tile_ptr_count(W.N, W.K) * 4.0;
    b += (double)rows * W.K * 2.0;                                        // activations read
    b += (double)rows * W.N * (epi == EPI_SILU ? 1.0 : 2.0);              // outputs written
    if (epi == EPI_RESID) b += (double)rows * W.N * 2.0;                  // residual read
    return b;
  };
#define LK(kind, expr)                                  \
  do {                                                  \
    if ((rc = tbegin(kind, 0.0))) return rc;            \
    cudaError_t _e = (expr);                            \
    if (_e != cudaSuccess) return cuda_fail(_e, #expr); \
    if ((rc = tend())) return rc;                       \
    launches++;                                         \
  } while (0)

  // GEMMs and RMSNorms are queued and launched at the next attention /
  // recurrence / acceptance kernel: as chain launches, or one by one
  struct PendingOp {
    int kind;
    ChainPhaseDesc d;
  };
  std::vector<PendingOp> pend;
  const bool chain = m->use_chain && rows <= 128 && chain_grid(rows) > 0;
  auto add_gemm = [&](int kind, const w12_tensor& W, const uint16_t* x, const XMap* xm, const GemmEpilogue& e) {
    PendingOp op{};
    op.kind = kind;
    op.d.type = PH_GEMM;
    op.d.W = &W;
    op.d.x = x;
    op.d.xm = xm;
    op.d.epi = e;
    pend.push_back(op);
  };
  auto add_norm = [&](const uint16_t* src, const uint16_t* gamma, uint16_t* dst) {
    PendingOp op{};
    op.kind = SD_K_NORM;
    op.d.type = PH_NORM;
    op.d.norm.src = src;
    op.d.norm.gamma = gamma;
    op.d.norm.dst = dst;
    op.d.norm.H = m->H;
    op.d.norm.eps = m->cfg.rms_eps;
    pend.push_back(op);
  };
  auto flush = [&]() -> int {
    size_t i = 0;
    while (i < pend.size()) {
      size_t n = 1;
      if (chain)
        while (i + n < pend.size() && n < (size_t)kChainMaxPhases) n++;
      if (n >= 2) {
        std::vector<ChainPhaseDesc> d;
        double bytes = 0.0;
        for (size_t j = i; j < i + n; j++) {
          d.push_back(pend[j].d);
          if (pend[j].d.type == PH_GEMM) bytes += gbytes(*pend[j].d.W, pend[j].d.epi.epi);
        }
        if ((rc = tbegin(SD_K_GEMM_CHAIN, bytes))) return rc;
        uint64_t* trace = nullptr;
        const int G = chain_grid(rows);
        const size_t rows_tr = 1 + 3 * n;
        if ((m->timing || m->tracing) && m->trace && trace_off + rows_tr * (size_t)G <= m->trace_cap) {
          trace = m->trace + trace_off;
          sd_model::ChainRec cr;
          cr.entry = m->t_kind.size() - 1;
          cr.off = trace_off;
          cr.n = (int)n;
          cr.G = G;
          for (size_t j = i; j < i + n; j++) {
            cr.kinds.push_back(pend[j].kind);
            cr.bytes.push_back(pend[j].d.type == PH_GEMM ? gbytes(*pend[j].d.W, pend[j].d.epi.epi) : 0.0);
          }
          m->t_chain.push_back(cr);
          trace_off += rows_tr * (size_t)G;
        }
        if ((rc = chain_launch(d.data(), (int)n, rows, m->gws, m->chain_bar, m->status, s, pdl, trace))) return rc;
        if ((rc = tend())) return rc;
        launches++;
      } else {
        const PendingOp& op = pend[i];
        if (op.d.type == PH_GEMM) {
          if ((rc = tbegin(op.kind, gbytes(*op.d.W, op.d.epi.epi)))) return rc;
          // timed steps record the launch's per-CTA stamps as a one-phase trace
          uint64_t* trace = nullptr;
          const int G = gemm_launch_grid(*op.d.W, rows, op.d.epi.epi);
          if ((m->timing || m->tracing) && m->trace && rows <= 128 && !gemm_use_tc(rows) &&
              trace_off + 4 * (size_t)G <= m->trace_cap) {
            trace = m->trace + trace_off;
            sd_model::ChainRec cr;
            cr.entry = m->t_kind.size() - 1;
            cr.off = trace_off;
            cr.n = 1;
            cr.G = G;
            cr.kinds.push_back(op.kind);
            cr.bytes.push_back(gbytes(*op.d.W, op.d.epi.epi));
            m->t_chain.push_back(cr);
            trace_off += 4 * (size_t)G;
          }
          if ((rc = gemm_launch(*op.d.W, op.d.x, *op.d.xm, rows, op.d.epi, m->gws, m->status, s, pdl, 0, trace)))
            return rc;
          if ((rc = tend())) return rc;
          launches += (rows > 128 && !gemm_use_tc(rows)) ? 2 : 1;
        } else {
          if ((rc = tbegin(SD_K_NORM, 0.0))) return rc;
          const cudaError_t e = launch_rmsnorm(op.d.norm.src, op.d.norm.gamma, rows, op.d.norm.H, op.d.norm.eps,
                                               op.d.norm.dst, nullptr, nullptr, nullptr, nullptr, nullptr, s, pdl);
          if (e != cudaSuccess) return cuda_fail(e, "rmsnorm");
          if ((rc = tend())) return rc;
          launches++;
        }
      }
      i += n;
    }
    pend.clear();
    return SD_OK;
  };

  if (m->timing) {
    // let the host enqueue the whole step before the GPU starts on it
    const cudaError_t e = launch_delay(30000000ull, s);
    if (e != cudaSuccess) return cuda_fail(e, "delay");
  }
  XMap *mx, *ma, *mc;
  if ((rc = get_map(m->map_xn, m->xn, m->max_rows, m->H, rows, &mx))) return rc;
  if ((rc = get_map(m->map_attn, m->attn, m->max_rows, (int64_t)m->Hq * m->hd, rows, &ma))) return rc;
  if ((rc = get_map(m->map_act, m->act, m->max_rows, m->I, rows, &mc))) return rc;

  const StepRows sr{m->ctx_snap, m->req_ok, m->pos, m->slotv, m->req, m->depth, m->anc};
  // the step's first kernel starts only after the previous step (its KV
  // commit) is complete: later kernels of the step may read the committed
  // prefix before their programmatic-launch wait
  LK(SD_K_TREE, launch_tree(io.tokens, io.parents, m->cu, io.R, io.cv, m->V, m->cfg.max_positions, sr, m->status, s, false));
  LK(SD_K_NORM, launch_rmsnorm(nullptr, m->layers[0].attn_norm, rows, m->H, m->cfg.rms_eps, m->xn, io.tokens, m->w.embed, m->x,
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

  for (int l = 0; l < m->cfg.n_layers; l++) {
    const sd_layer_weights& Lw = m->layers[l];
    const bool is_attn = m->kind[l] == 0;
    const int ls = m->slot[l];
    GemmEpilogue eq;
    if (is_attn) {
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
    add_gemm(SD_K_GEMM_QKV, Lw.qkv, m->xn, mx, eq);
    if ((rc = flush())) return rc;
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
      if ((rc = tbegin(SD_K_ATTN, 0.0))) return rc;
      {
        // traced steps record the attention's per-CTA stamps as a one-phase trace
        const int G = (splits + 1) * m->Hkv * chunks * io.R;
        if ((m->timing || m->tracing) && m->trace && trace_off + 4 * (size_t)G <= m->trace_cap) {
          aa.trace = m->trace + trace_off;
          sd_model::ChainRec cr;
          cr.entry = m->t_kind.size() - 1;
          cr.off = trace_off;
          cr.n = 1;
          cr.G = G;
          cr.kinds.push_back(SD_K_ATTN);
          cr.bytes.push_back(0.0);
          m->t_chain.push_back(cr);
          trace_off += 4 * (size_t)G;
        }
      }
      const cudaError_t e = launch_attention(aa, rows, s, pdl);
      if (e != cudaSuccess) return cuda_fail(e, "attention");
      if ((rc = tend())) return rc;
      launches += 1;
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
      LK(SD_K_LINREC, launch_linrec(la, s, pdl));
    }
    GemmEpilogue eo;  // h = x + O(attn)
    eo.epi = EPI_RESID;
    eo.out = m->h;
    eo.resid = m->x;
    eo.ldo = m->H;
    add_gemm(SD_K_GEMM_O, Lw.o, m->attn, ma, eo);
    add_norm(m->h, Lw.mlp_norm, m->xn);
    GemmEpilogue eg;
    eg.epi = EPI_SILU;
    eg.out = m->act;
    eg.ldo = m->I;
    add_gemm(SD_K_GEMM_GATE_UP, Lw.gate_up, m->xn, mx, eg);
    GemmEpilogue ed;  // x = h + down(act)
    ed.epi = EPI_RESID;
    ed.out = m->x;
    ed.resid = m->h;
    ed.ldo = m->H;
    add_gemm(SD_K_GEMM_DOWN, Lw.down, m->act, mc, ed);
    const uint16_t* gnext = l + 1 < m->cfg.n_layers ? m->layers[l + 1].attn_norm : m->w.final_norm;
    add_norm(m->x, gnext, m->xn);
  }
  GemmEpilogue el;
  el.epi = EPI_LOGITS;
  el.out = io.logits;
  el.ldo = m->V;
  el.amax_val = m->amax_val;
  el.amax_idx = m->amax_idx;
  el.ld_amax = m->max_rows;
  add_gemm(SD_K_GEMM_LM_HEAD, m->w.lm_head, m->xn, mx, el);
  if ((rc = flush())) return rc;

  AcceptArgs ac{};
  ac.tokens = io.tokens;
  ac.parents = io.parents;
  ac.cu = m->cu;
  ac.R = io.R;
  ac.amax_val = m->amax_val;
  ac.amax_idx = m->amax_idx;
  ac.n_part = gemm_grid(rows);
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
  LK(SD_K_ACCEPT, launch_accept(ac, s, pdl));
  if (io.commit) {
    if (m->n_attn) LK(SD_K_COMMIT, launch_compact(io.cv, m->n_attn, m->Hkv, io.R, m->ctx_snap, m->path, m->path_len, s, pdl));
    if (m->n_rec)
      LK(SD_K_COMMIT, launch_rec_commit(io.cv, m->n_rec, m->nh_rec, m->H, io.R, m->max_rows, m->qkv_rec, m->cu, m->path,
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
  if (!m->use_graphs || m->timing || m->tracing || s == nullptr) return run_step(m, io, s);
  key.push_back((uintptr_t)m->use_chain);
  key.push_back((uintptr_t)gemm_tc_min_rows());
  key.push_back((uintptr_t)g_attn_splits);
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
          u(io.accepted_tokens), u(io.bonus), u(io.logits), u(io.argmax), (uintptr_t)io.commit};
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
      {(void**)&m->chain_bar, 16},
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
  if (m->trace) cudaFree(m->trace);
  cudaFree(m->arena);
  delete m;
  return SD_OK;
}

static int single_step(sd_model* m, const int32_t* tokens, const int32_t* parents, int32_t M, const sd_kv* kv,
                       int32_t* accepted_len, int32_t* accepted_tokens, int32_t* bonus, uint16_t* logits,
                       int32_t* argmax, bool commit, void* stream) {
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
  // a chain that gave up on a barrier may have left its arrival counter
  // short of a multiple of the grid: start the next one from zero
  if (*status_host != SD_OK) SD_CK(cudaMemset(m->chain_bar, 0, 16));
  return SD_OK;
}

extern "C" int sd_model_last_launches(sd_model* m) { return m ? m->last_launches : 0; }

extern "C" int sd_model_set_timing(sd_model* m, int32_t enable) {
  if (!m) {
    set_error("sd_model_set_timing: null model");
    return SD_ERR_INVALID_ARG;
  }
  m->timing = enable == 1;
  m->tracing = enable == 2;
  if ((m->timing || m->tracing) && !m->trace) {
    // stamps of every traced launch of one step: at most (layers + 2) chains
    // of 1 + 3 x 6 rows, or per layer 4 GEMMs and the attention of 4 rows,
    // x the largest grid (zero-filled: a CTA without work in a phase leaves
    // two of its stamps unwritten)
    const size_t cap = (size_t)(m->cfg.n_layers + 2) * (1 + 3 * kChainMaxPhases) * gemm_grid(1) * 2;
    SD_CK(cudaMalloc(&m->trace, cap * sizeof(uint64_t)));
    SD_CK(cudaMemset(m->trace, 0, cap * sizeof(uint64_t)));
    m->trace_cap = cap;
  }
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
  size_t ci = 0;
  for (size_t i = 0; i < m->t_kind.size() && n < max; i++) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, m->events[2 * i], m->events[2 * i + 1]) != cudaSuccess) ms = -1.f;
    kind_host[n] = m->t_kind[i];
    ms_host[n] = ms;
    bytes_host[n] = m->t_bytes[i];
    n++;
    if (ci < m->t_chain.size() && m->t_chain[ci].entry == i) {
      // the chain's phases from the device stamps: phase p lasts from the
      // last CTA finishing phase p - 1 (the first CTA starting, for p = 0)
      // to the last CTA finishing phase p
      const sd_model::ChainRec& cr = m->t_chain[ci++];
      std::vector<uint64_t> st((size_t)(1 + 3 * cr.n) * cr.G);
      if (cudaMemcpy(st.data(), m->trace + cr.off, st.size() * sizeof(uint64_t), cudaMemcpyDeviceToHost) !=
          cudaSuccess) {
        set_error("sd_model_timeline: trace copy failed");
        return -1;
      }
      uint64_t prev = ~0ull;
      for (int c = 0; c < cr.G; c++) prev = std::min(prev, st[c]);
      for (int p = 0; p < cr.n && n < max; p++) {
        uint64_t end = 0;
        for (int c = 0; c < cr.G; c++) end = std::max(end, st[(size_t)(3 + 3 * p) * cr.G + c]);
        kind_host[n] = 100 + cr.kinds[p];
        ms_host[n] = (float)((double)(end - prev) * 1e-6);
        bytes_host[n] = cr.bytes[p];
        n++;
        prev = end;
      }
    }
  }
  return n;
}

extern "C" int sd_model_chain_trace(sd_model* m, int32_t launch, int32_t* n_phases, int32_t* n_ctas,
                                    uint64_t* stamps_host, int64_t max_stamps) {
  if (!m || !n_phases || !n_ctas || launch < 0) {
    set_error("sd_model_chain_trace: bad argument");
    return SD_ERR_INVALID_ARG;
  }
  if (launch >= (int)m->t_chain.size()) {
    set_error("sd_model_chain_trace: no such chain launch in the last timed step");
    return SD_ERR_INVALID_ARG;
  }
  const sd_model::ChainRec& cr = m->t_chain[launch];
  *n_phases = cr.n;
  *n_ctas = cr.G;
  const size_t cnt = (size_t)(1 + 3 * cr.n) * cr.G;
  if (stamps_host) {
    if (max_stamps < (int64_t)cnt) {
      set_error("sd_model_chain_trace: buffer too small");
      return SD_ERR_INVALID_ARG;
    }
    SD_CK(cudaDeviceSynchronize());
    SD_CK(cudaMemcpy(stamps_host, m->trace + cr.off, cnt * sizeof(uint64_t), cudaMemcpyDeviceToHost));
  }
  return SD_OK;
}

extern "C" int sd_model_set_chain(sd_model* m, int32_t enable) {
  if (!m) {
    set_error("sd_model_set_chain: null model");
    return SD_ERR_INVALID_ARG;
  }
  m->use_chain = enable != 0;
  return SD_OK;
}

extern "C" int sd_model_set_graphs(sd_model* m, int32_t enable) {
  if (!m) {
    set_error("sd_model_set_graphs: null model");
    return SD_ERR_INVALID_ARG;
  }
  m->use_graphs = enable != 0;
  return SD_OK;
}
