// Fused W12-decode skinny GEMM: launch interface.
#pragma once

#include "common.cuh"

namespace sdv {

enum Epi : int {
  EPI_STORE = 0,   // out[m][n] = bf16(acc)
  EPI_RESID = 1,   // out[m][n] = bf16(resid[m][n] + bf16(acc))       (out may alias resid)
  EPI_SILU = 2,    // gate/up strips: out[m][8s+g] = bf16(silu(bf16(gate)) * bf16(up))
  EPI_QKV = 3,     // rope-paired q/k strips + v: q -> q_out, k/v -> paged cache
  EPI_LOGITS = 4,  // optional bf16 logits + per-CTA running fp32 argmax per row
};

// Per-row (token) bookkeeping written by the tree kernel each step.
struct RowInfo {
  const int32_t* pos;     // [rows] position ctx + depth (RoPE)
  const int32_t* slot;    // [rows] cache slot ctx + local node index
  const int32_t* req;     // [rows] request index
  const int32_t* req_ok;  // [R] 1 if the request's tree is valid and fits
};

struct PagedCache {
  uint16_t* k;  // this layer's pool: [n_pages][Hkv][page][hd]
  uint16_t* v;
  const int32_t* page_table;  // [R][max_pages]
  int32_t max_pages, page_size, hkv;
};

struct GemmEpilogue {
  int epi = EPI_STORE;
  uint16_t* out = nullptr;
  int ldo = 0;
  const uint16_t* resid = nullptr;
  // QKV
  uint16_t* q_out = nullptr;  // [rows][Hq][hd]
  int hq = 0, hkv = 0;
  PagedCache cache{};
  RowInfo rows{};
  const float* rope_cos = nullptr;  // [positions][hd/2]
  const float* rope_sin = nullptr;
  // LOGITS
  float* amax_val = nullptr;  // [grid][ld_amax]
  int32_t* amax_idx = nullptr;
  int ld_amax = 0;
};

struct GemmWorkspace {
  float* partial = nullptr;  // partial sums of row blocks split between CTAs
  int32_t* counters = nullptr;
  size_t partial_floats = 0;
  int counters_len = 0;
};

// Launches of at least gemm_tc_min_rows() rows run on the tcgen05 kernel
// (gemm_tc.cu, one CTA per SM, up to 256 rows in one launch); fewer rows run
// on the warp-level MMA kernel (gemm.cu).
int gemm_tc_min_rows();
void gemm_set_tc_min_rows(int rows);  // <= 0: the default
inline bool gemm_use_tc(int M) { return M >= gemm_tc_min_rows(); }
int gemm_tc_rows(int M);               // MMA N side for M rows (multiple of 16, >= 32)
size_t gemm_tc_partial_floats(int M);  // workspace floats of the tcgen05 kernel
int gemm_tc_launch(const w12_tensor& W, const uint16_t* x, int rows_total, int M, const GemmEpilogue& epi,
                   const GemmWorkspace& ws, int32_t* status, cudaStream_t s, bool pdl);

int gemm_grid(int M);               // CTAs per launch for M rows (persistent: 1 or 2 per SM)
int gemm_launch_grid(const w12_tensor& W, int M, int epi);  // the grid gemm_launch uses by default
size_t gemm_partial_floats(int M);  // workspace floats for M rows (either kernel)
int gemm_counters(int64_t N);       // counters for N rows
int pad_rows(int M);                // rows of one launch's TMA box: 8, 16, 32, 64 or 128

// TMA descriptor of an activation buffer bf16 [rows_total][K].
struct XMap {
  CUtensorMap map;
  int rows_total;
  int box_rows;
};
int make_x_map(XMap* xm, const uint16_t* x, int rows_total, int64_t K, int box_rows);

// y = epilogue(x W^T) for rows [0, M).  With gemm_use_tc(M) one tcgen05
// launch covers all rows (grid and trace are ignored, the x map is rebuilt
// with a box of gemm_tc_rows(M) rows); otherwise M > 128 runs in launches of
// 128 rows.  grid: CTAs per launch, 0 = gemm_grid(M); the partial-sum
// workspace must hold grid * 2 * 8 * (padded rows / 8) * 128 floats.  trace
// (optional, M <= 128): [4][grid] device-clock stamps per CTA - start, first
// stage ready, last stage consumed, finished.
// Strip-parallel kernel (gemm_strip.cu): one CTA per 16-row strip over the
// whole k range, no split-K across CTAs; for skinny launches (M <= 16) whose
// strips fit one wave (the O and down projections).  gemm_launch takes it at
// its default grid when eligible (sd_gemm_set_strip).
bool gemm_strip_eligible(const w12_tensor& W, int M, int epi);
bool gemm_strip_eligible_setting();  // sd_gemm_set_strip
int gemm_strip_launch(const w12_tensor& W, const uint16_t* x, const XMap& xm, int M, const GemmEpilogue& epi,
                      int32_t* status, cudaStream_t s, bool pdl);

// The process-wide split-K finish settings (cluster << 1 | deferred): part of
// a captured step's identity.
int gemm_finish_mode();
// Kernels gemm_launch (grid <= 0: its default grid) issues for one call: the
// GEMM's row tiles and, for a deferred split-K finish, the finish kernel.
int gemm_kernel_count(const w12_tensor& W, int M, int epi, int grid = 0);
int gemm_launch(const w12_tensor& W, const uint16_t* x, const XMap& xm, int M, const GemmEpilogue& epi,
                const GemmWorkspace& ws, int32_t* status, cudaStream_t s, bool pdl, int grid = 0,
                uint64_t* trace = nullptr);
// The same on the warp-level kernel whatever the row count (M <= 64 in one
// launch), with its own default grid.  plane8 (W's nested 8-bit plane, W
// with a contiguous exponent table, M <= 64): the product with the 8-bit
// view, streaming the plane at 1 byte per weight.
int gemm_warp_launch(const w12_tensor& W, const uint16_t* x, const XMap& xm, int M, const GemmEpilogue& epi,
                     const GemmWorkspace& ws, int32_t* status, cudaStream_t s, bool pdl, int grid = 0,
                     uint64_t* trace = nullptr, const uint32_t* plane8 = nullptr);
int gemm_warp_launch_grid(const w12_tensor& W, int M, int epi);
int gemm_warp_grid(int M);  // CTAs of a warp-level launch of M rows

// Descriptor of the packed words for the 2-D weight loads (one box = 8
// strips x 1536 bytes).
int make_w_map(CUtensorMap* map, const w12_tensor& W);
// Descriptor of a tensor's 8-bit plane (one box = 8 strips x 1024 bytes).
int make_w8_map(CUtensorMap* map, const uint32_t* plane, int64_t N, int64_t K);

struct GemmParams;
int make_gemm_params(GemmParams* out, const w12_tensor& W, const uint16_t* x, int M, const GemmEpilogue& epi,
                     const GemmWorkspace& ws, int32_t* status);

}  // namespace sdv
