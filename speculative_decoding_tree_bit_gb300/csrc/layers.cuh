// Tree-verify kernels other than the GEMM: launch interface.
#pragma once

#include "common.cuh"

namespace sdv {

// Per-step view of the (paged) cache of all requests.  A contiguous
// single-request cache is the special case n_pages = max_pages = 1,
// page_size = cap, page_table = {0}.
struct CacheView {
  uint16_t* k_pool;  // [n_attn_layers][n_pages][Hkv][page][hd]
  uint16_t* v_pool;
  int32_t n_pages, page_size;
  const int32_t* page_table;  // [R][max_pages]
  int32_t max_pages;
  float* S;          // [R][n_rec][nh][hd][hd]
  float* z;          // [R][n_rec][nh][hd]
  int32_t* ctx_len;  // [R]
};

struct StepRows {
  int32_t* ctx_snap;  // [R]
  int32_t* req_ok;    // [R]
  int32_t* pos;       // [rows]
  int32_t* slot;      // [rows]
  int32_t* req;       // [rows]
  int32_t* depth;     // [rows]
  uint64_t* anc;      // [rows]
};

cudaError_t launch_tree(const int32_t* tokens, const int32_t* parents, const int32_t* cu, int R, const CacheView& cv,
                        int vocab, int max_positions, const StepRows& rows, int32_t* status, cudaStream_t s, bool pdl);

// xn = RMSNorm(src) (bf16); with embed != nullptr, src row m is
// embed[token[m]] and is also written to x_out (the residual stream).
cudaError_t launch_rmsnorm(const uint16_t* src, const uint16_t* gamma, int rows, int H, float eps, uint16_t* xn,
                           const int32_t* tokens, const uint16_t* embed, uint16_t* x_out, const int32_t* row_req,
                           const int32_t* req_ok, cudaStream_t s, bool pdl);

struct AttnArgs {
  const uint16_t* q;       // [rows][Hq][hd]
  const uint16_t* k_pool;  // this layer
  const uint16_t* v_pool;
  const int32_t* page_table;
  int32_t max_pages, page_size, hq, hkv;
  int32_t n_pages;          // physical pages in the pool (page ids read before validation are checked)
  const int32_t* cu;       // [R+1]
  const int32_t* ctx;      // ctx_snap [R]
  const int32_t* ctx_in;   // [R] the context lengths as passed in (not written before the step's commit)
  const uint64_t* anc;     // [rows]
  const int32_t* row_req;  // [rows]
  const int32_t* req_ok;   // [R]: requests whose tree failed validation read no keys
  int R, max_m, splits;    // splits = prefix splits (the tree segment is one more)
  int chunk_m;             // rows of the call's largest request (<= max_m; 0: max_m): sets the grid's row chunks
  float* part_o;           // [R][Hkv][splits+1][rows_per_group][hd]
  float* part_ml;          // [R][Hkv][splits+1][rows_per_group][2]
  int32_t* tickets;        // [R][Hkv][row chunks][2]: zero between calls (each call resets its own)
  int32_t* status;         // a bounded wait that gave up records SD_ERR_TIMEOUT
  uint16_t* out;           // [rows][Hq*hd]
  uint64_t* trace;         // optional [4][grid] device-clock stamps: start, keys done, group ready, end
};
int attn_rows_per_group(int hq, int hkv, int max_m);
// Key split of the attention kernel for groups of this many rows (2: pairs of
// warps share a 16-row tile, each taking half of every key tile) and the
// grid's row chunks per (request, kv head).
int attn_key_split(int rows_per_group);
int attn_chunks(int rows_per_group);
cudaError_t launch_attention(const AttnArgs& a, int rows_total, cudaStream_t s, bool pdl);

struct LinrecArgs {
  const uint16_t* qkv;  // [rows][3H]: q | k | v
  const float* S;       // this layer's state of request 0; request r at + r*req_stride_S
  const float* z;
  int64_t req_stride_S, req_stride_z;
  const int32_t* cu;
  const uint64_t* anc;
  int R, nh, H;
  float eps;
  uint16_t* out;        // [rows][H]
};
cudaError_t launch_linrec(const LinrecArgs& a, cudaStream_t s, bool pdl);

struct AcceptArgs {
  const int32_t* tokens;
  const int32_t* parents;
  const int32_t* cu;         // [R+1] (device), or nullptr for one request of single_M nodes
  int R, single_M;
  const float* amax_val;     // [n_part][ld] partial argmax (or nullptr: use argmax_in)
  const int32_t* amax_idx;
  int n_part, ld;
  const int32_t* argmax_in;  // [rows]
  const int32_t* req_ok;     // [R] or nullptr
  const int32_t* ctx_snap;   // [R] or nullptr
  int32_t* ctx_len;          // [R] advanced when committing (or nullptr)
  int32_t* argmax_out;       // [rows] optional
  int32_t* accepted_len;     // [R]
  int32_t* accepted_tokens;  // [rows]: request r's at cu[r]
  int32_t* bonus;            // [R]
  int32_t* path;             // [R][65] or nullptr
  int32_t* path_len;         // [R] or nullptr (path nodes incl. root; 0 = nothing to commit)
  int32_t* status;
};
cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s, bool pdl);

cudaError_t launch_compact(const CacheView& cv, int n_attn_layers, int hkv, int R, const int32_t* ctx_snap,
                           const int32_t* path, const int32_t* path_len, cudaStream_t s, bool pdl);

cudaError_t launch_rec_commit(const CacheView& cv, int n_rec, int nh, int H, int R, int max_rows,
                              const uint16_t* qkv_rec, const int32_t* cu, const int32_t* path,
                              const int32_t* path_len, cudaStream_t s, bool pdl);

cudaError_t launch_delay(uint64_t ns, cudaStream_t s);

}  // namespace sdv
