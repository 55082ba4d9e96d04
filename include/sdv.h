/*
 * sdv -- tree verification with lossless 12-bit weights on one GB300.
 *
 * C ABI of the library libsdv.so.  Every pointer is a DEVICE pointer unless
 * its name ends in _host, or the function works in host memory only (the
 * functions whose names end in _host, and the W12 file functions w12_save,
 * w12_load_info and w12_load), as its comment states.  Streams are passed as `void*` holding a
 * cudaStream_t (NULL = legacy default stream).  Every function returns an
 * `int` status (SD_OK = 0); host-checkable argument errors are reported
 * synchronously, data errors found on the device (a bad parent array, a token
 * outside the vocabulary, a full cache, a wait that timed out) are recorded in
 * a device status word and never trap.  The caller owns every buffer it
 * passes; the library never frees caller memory.  sd_last_error() returns a
 * text for the last failing call on this thread.
 *
 * The pages this library follows:
 *   [W12]  "SpecPilot: AI Agent Framework Boosts Speculative Decoding 10.87x
 *          for Qwen3.8-27B", section "(1) W12: Lossless 12-bit Weight Format".
 *   [TREE] same page, "(2) Best-first Tree Verification for Hybrid
 *          Architectures"; "SpecPilot Uses Agentic Discovery to Push
 *          Speculative Decoding to 10.87x", "Core Idea" (the drafter proposes a
 *          block, the target verifies it in one parallel pass).
 *   [EXACT] first page, "(3) Two-Level Verification": only the exact target
 *          verification accepts tokens; second page "Core Idea", item 4
 *          (token forcing: outputs equal the stock greedy outputs).
 *   [BATCH] first page, "(4) Three Batch Optimization Mechanisms", Shared
 *          Node Budget (best-first node selection across a batch).
 */
#ifndef SDV_H
#define SDV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status -- */
enum {
  SD_OK = 0,
  SD_ERR_INVALID_ARG = 1,  /* a host-side argument is wrong */
  SD_ERR_UNSUPPORTED = 2,  /* shape outside what the kernels handle (N%16, K%64, M>64 per request ...) */
  SD_ERR_CUDA = 3,         /* a CUDA runtime call failed (text in sd_last_error) */
  SD_ERR_OOM = 4,          /* device allocation failed */
  SD_ERR_BAD_TREE = 5,     /* device: parent array not a tree rooted at node 0 with parent[i] < i */
  SD_ERR_TIMEOUT = 6,      /* device: a bounded wait gave up */
  SD_ERR_CAPACITY = 7,     /* device: ctx + nodes exceeds the cache capacity / page table / RoPE table */
  SD_ERR_BAD_TOKEN = 8,    /* device: a token outside [0, vocab) */
  SD_ERR_WORKSPACE = 9,    /* caller workspace smaller than the size query returned */
  SD_ERR_IO = 10,          /* a file could not be opened or written */
  SD_ERR_CORRUPT = 11      /* a file is not a W12 file of this version, or fails its checksums */
};

const char* sd_last_error(void);
const char* sd_version(void);

/* Test hook for the device-side bounded waits: every wait of the library's
 * kernels on an mbarrier or a device flag gives up after 2 s, records
 * SD_ERR_TIMEOUT in the caller's status word and lets the kernel return, so
 * that a stuck pipeline never hangs the GPU.  This launches one small kernel
 * that waits, with those same helpers, on something nothing completes
 * (which = 0: an mbarrier nobody arrives at, waited by two warps sharing an
 * abort flag; which = 1: a device flag nobody sets, polled with acquire
 * loads) for limit_ns nanoseconds (clamped to [1 us, 2 s]), then sets
 * *status (device int32, caller-owned, not cleared here) to SD_ERR_TIMEOUT.
 * Errors: SD_ERR_INVALID_ARG, SD_ERR_CUDA (launch). */
int sd_debug_bounded_wait(int32_t* status, int64_t limit_ns, int32_t which, void* stream);

/* Event log of the streamed W12 GEMM launches (diagnostics: where a launch
 * of several GEMMs spends its time).  While a buffer is set (device memory,
 * 16-byte aligned, zeroed by the caller), each streamed launch takes the
 * next sd_stream_grid(M) * 64 records of 16 bytes, in launch order, until
 * the buffer is full (later launches log nothing).  Records of CTA c:
 * [c * 64, c * 64 + 32) from its producer, [c * 64 + 32, c * 64 + 64) from
 * its consumers, unused ones left zero; each is {device clock in ns, tag},
 * tag = kind | phase << 8 | row block << 16 | k-tile << 40 with kind 1
 * producer start, 2 first weight tile of a segment issued, 3 its first
 * activation tile issued (what it reads is complete), 4 the segment's first
 * stage ready at the consumers, 5 the segment finished (k-tile field 1: the
 * block's epilogue ran here, 0: a partial was left for another CTA), 6 the
 * consumers done.  buf null or bytes 0 turns the log off.  Process-wide; not
 * thread-safe against concurrent launches.  sd_stream_trace_launches: the
 * launches logged since the buffer was set; sd_stream_grid: CTAs of a
 * streamed launch of M rows (0 outside 1..64). */
int sd_stream_set_trace(uint64_t* buf, int64_t bytes);

/* Device-clock stamps of the verify step's attention launches (diagnostics):
 * while a buffer is set (device memory, zeroed by the caller), each launch
 * takes the next 4 x grid u64 of it in launch order until it is full: for
 * CTA c (x fastest, then y, z of the launch grid) at [i * grid + c] the time
 * in ns after its wait for the previous kernel (i = 0), after its keys
 * (1), once its split group is ready to merge (2), at its end (3).  buf
 * null or bytes 0 turns the log off; process-wide. */
int sd_attn_set_trace(uint64_t* buf, int64_t bytes);
int32_t sd_stream_trace_launches(void);
int32_t sd_stream_grid(int32_t M);

/* ---------------------------------------------------------------- W12 -- */
/* [W12] Each bf16 weight is stored in 12 bits: sign, 7-bit mantissa and a
 * 4-bit code into a per-tensor table of the 15 most frequent exponents
 * (count descending, ties to the smaller exponent, stored in ascending
 * exponent order).  Code 15 marks an escape; the escaped weight's exact bf16
 * bits are kept in a side list sorted by flat index n*K+k, with a CSR row
 * pointer.  Unpacking restores every bf16 bit pattern exactly (NaN payloads,
 * infinities, zeros and subnormals included).
 *
 * Layout (requires N % 16 == 0 and K % 64 == 0): rows form strips of 16,
 * columns super-tiles of 64 split into four 16-wide sub-tiles.  The words of
 * strip s, super-tile t are the 384 u32 at offset (s*(K/64)+t)*384, ordered
 * [plane p = 0..2][lane 0..31][sub-tile j = 0..3].  Lane 4g+q holds the
 * tensor-core A fragment of its sub-tile: pair 0 = W[g][2q..2q+1], pair 1 =
 * W[g+8][2q..2q+1], pair 2 = W[g][2q+8..2q+9], pair 3 = W[g+8][2q+8..2q+9]
 * (rows and columns relative to the sub-tile).  With f = sign<<11 | code<<7 |
 * mantissa, plane p (p < 3) stores pair p as f&0x7FF with the sign in bit 15
 * of each 16-bit half; pair 3's three nibbles fill bits 11..14 / 27..30 of
 * planes 0, 1, 2.  An escaped weight stores code 15, sign 0, mantissa 0. */

typedef struct {
  int64_t N, K;             /* rows (outputs), columns (inputs) */
  uint8_t table[16];        /* exponents of codes 0..n_table-1, ascending; rest 0 */
  int32_t n_table;          /* <= 15 */
  int32_t affine;           /* 1 if table[c] == table[0] + c for all c < n_table
                               and table[0] + 15 <= 254 (fast decode path) */
  int64_t n_escapes;
} w12_meta;

typedef struct {
  int64_t N, K;
  const uint32_t* words;    /* device, w12_words_count(N,K) u32 */
  const uint32_t* esc_idx;  /* device [n_escapes], increasing */
  const uint16_t* esc_val;  /* device [n_escapes], bf16 bits */
  const uint32_t* row_ptr;  /* device [N+1] */
  const uint32_t* tile_ptr; /* device [w12_tile_ptr_count(N,K)]: escape tile index (w12_pack_tile_index) */
  const uint32_t* tile_esc; /* device [n_escapes] */
  int64_t n_escapes;
  uint8_t table[16];
  int32_t n_table;
  int32_t affine;
  /* device [N] or null.  Non-null: a per-channel tensor (w12c_pack_*): row n
   * decodes code c < 15 as exponent row_base[n] + c and table / n_table are
   * unused; affine = 1 when every base is at most 239 (the GEMM decodes
   * such tensors; others pack, unpack and round-trip but do not multiply). */
  const uint8_t* row_base;
} w12_tensor;

/* Number of u32 words of a packed N x K tensor (N*K*3/8). */
int64_t w12_words_count(int64_t N, int64_t K);

/* Histogram of the exponents of w[N][K] (bf16 bits, row-major, device) and
 * the code table.  Fills meta (including n_escapes); synchronises `stream`.
 * Errors: SD_ERR_UNSUPPORTED if N%16 or K%64 or N*K >= 2^32, SD_ERR_CUDA. */
int w12_pack_analyze(const uint16_t* w, int64_t N, int64_t K, w12_meta* meta, void* stream);

/* Encode w into the W12 layout using meta from w12_pack_analyze.
 * row_src (optional, device int32[N]): packed row n is taken from row
 * row_src[n] of w; it must be a permutation of 0..N-1 (the histogram is
 * permutation-invariant).  Escape indices refer to packed rows.  Outputs are
 * caller-allocated: words[w12_words_count], esc_idx/esc_val[meta->n_escapes],
 * row_ptr[N+1].  Allocates and frees its own scratch (stream-ordered);
 * asynchronous on `stream`. */
int w12_pack_encode(const uint16_t* w, const int32_t* row_src, const w12_meta* meta, uint32_t* words,
                    uint32_t* esc_idx, uint16_t* esc_val, uint32_t* row_ptr, void* stream);

/* Restore the bf16 tensor [N][K] (bit-exact).  Asynchronous.  Uses words,
 * esc_idx, esc_val only. */
int w12_unpack(const w12_tensor* t, uint16_t* w_out, void* stream);

/* Escape tile index (no counterpart in the pages: an access structure of
 * this library over the side list, which stays the format's record of the
 * escapes).  The fused kernels stream a tensor by blocks of 128 rows and
 * tiles of 64 columns and need each (block, tile)'s escapes as one
 * contiguous run: with NB = ceil(N/128) and KT = K/64, the escapes of row
 * block b and column tile t are tile_esc[tile_ptr[b*KT+t] ..
 * tile_ptr[b*KT+t+1]), each encoded as (bf16 bits << 16) | (row - 128b) << 6
 * | (column - 64t), in row-major order within the (block, tile);
 * tile_ptr[NB*KT] = n_escapes.  The escapes of block b occupy the same index
 * range as in the side list.  w12_tile_ptr_count(N, K) = NB*KT + 1. */
int64_t w12_tile_ptr_count(int64_t N, int64_t K);

/* Build the escape tile index of t from its side list (esc_idx, esc_val,
 * row_ptr).  Outputs are caller-allocated device arrays:
 * tile_ptr[w12_tile_ptr_count], tile_esc[n_escapes] (may be NULL when
 * n_escapes == 0).  Asynchronous on `stream`.  Every fused kernel requires
 * t->tile_ptr and, with escapes, t->tile_esc (SD_ERR_INVALID_ARG if missing). */
int w12_pack_tile_index(const w12_tensor* t, uint32_t* tile_ptr, uint32_t* tile_esc, void* stream);

/* ------------------------------------------------ fused W12 linear -- */
/* [W12] y[m][n] = bf16( sum_k x[m][k] * W[n][k] ), fp32 accumulation, with
 * the weights decoded in registers straight from the packed words (they
 * cross HBM once, 1.5 bytes each) and the escapes added from the escape tile
 * index (W->tile_ptr / tile_esc must be set).  A per-channel tensor
 * (W->row_base set, affine) runs on the warp-level kernel, M <= 64.
 * x: bf16 [M][K] row-major, 16-byte aligned; y: bf16 [M][N] row-major.
 * 1 <= M <= 256.  workspace: caller-owned device scratch of
 * sd_w12_linear_workspace(N, K, M) bytes, 256-byte aligned; it needs no
 * initialisation (the call clears what it must).  Errors: SD_ERR_UNSUPPORTED
 * (shape), SD_ERR_WORKSPACE, SD_ERR_CUDA. */
size_t sd_w12_linear_workspace(int64_t N, int64_t K, int32_t M);
int sd_w12_linear(const w12_tensor* W, const uint16_t* x, int32_t M, uint16_t* y, void* workspace,
                  size_t workspace_bytes, void* stream);

/* The same linear on the weight-streaming kernel (the kernel of the fused
 * schedule and of the 8-bit view of two-level verification), 1 <= M <= 64.
 * plane8: null for the exact 12-bit weights, or W's nested 8-bit plane
 * (w12_plane8_pack; N*K/4 u32, 16-byte aligned), in which case the call
 * multiplies by the 8-bit view of W (each weight with its 4 low mantissa
 * bits cleared, escapes likewise) while streaming 1 byte per weight.
 * workspace: sd_w12_linear_stream_workspace(N, K, M) bytes, 256-byte
 * aligned, no initialisation needed.  Errors: SD_ERR_INVALID_ARG,
 * SD_ERR_UNSUPPORTED (shape, M), SD_ERR_WORKSPACE, SD_ERR_CUDA. */
size_t sd_w12_linear_stream_workspace(int64_t N, int64_t K, int32_t M);
int sd_w12_linear_stream(const w12_tensor* W, const uint32_t* plane8, const uint16_t* x, int32_t M, uint16_t* y,
                         void* workspace, size_t workspace_bytes, void* stream);

/* The product with the nested 8-bit view of W ("SpecPilot ...", "(3)
 * Two-Level Verification": round one of two-level verification), streaming
 * W's 8-bit plane at 1 byte per weight (plane8: w12_plane8_pack, 16-byte
 * aligned), 1 <= M <= 64: the warp-level kernel in its 8-bit decode mode
 * for a contiguous exponent table, the weight-streaming kernel otherwise.
 * workspace: sd_w12_linear_view8_workspace(N, K, M) bytes, 256-byte
 * aligned.  Errors: SD_ERR_INVALID_ARG, SD_ERR_UNSUPPORTED,
 * SD_ERR_WORKSPACE, SD_ERR_CUDA. */
size_t sd_w12_linear_view8_workspace(int64_t N, int64_t K, int32_t M);
int sd_w12_linear_view8(const w12_tensor* W, const uint32_t* plane8, const uint16_t* x, int32_t M, uint16_t* y,
                        void* workspace, size_t workspace_bytes, void* stream);

/* The same linear for callers that cannot allocate device memory: a host
 * framework that owns all device memory through its own pool, a real-time
 * thread that must not take cudaMalloc's implicit synchronisation, a plug-in
 * that may not grow the process's device footprint.  No counterpart in the
 * SpecPilot pages; it is a packaging variant of sd_w12_linear.  The split-K
 * scratch lives in a static device array inside the library (about 9.5 MiB
 * that every GPU loading the library holds until the process exits), so the
 * call allocates nothing; the caller passes only W, x and y.
 * Limits: 1 <= M <= 64 and N <= 262144, else SD_ERR_UNSUPPORTED.  The
 * call always runs the warp-level kernel (the static scratch is sized for
 * it), whatever sd_gemm_set_tc_min_rows says, with the grid sd_w12_linear
 * gives that kernel (up to 1216 CTAs x 8-row tiles).
 * Each call looks up the array's address in the current context (a context
 * made after cudaDeviceReset gets its own); inside a stream capture use
 * cudaStreamCaptureModeRelaxed, which allows that lookup.
 * Every call on a device shares the one array: calls that can overlap on the
 * GPU (different streams without ordering between them) race and give wrong
 * results; serialise them. */
int sd_w12_linear_static(const w12_tensor* W, const uint16_t* x, int32_t M, uint16_t* y, void* stream);

/* Rows per launch from which the fused W12 GEMMs (sd_w12_linear and every
 * GEMM of the verify step) run on the tcgen05 tensor-core kernel: weights
 * decoded into a shared-memory operand tile, escapes written over their
 * slots, fp32 accumulators in tensor memory, up to 256 rows in one launch.
 * Fewer rows run on the warp-level MMA kernel, which streams weights with
 * less on-chip traffic while a launch is bandwidth-bound ("SpecPilot ...",
 * batched results: the batched step crosses from the weight-bandwidth bound
 * to the tensor-core bound).  Process-wide; applies to calls issued
 * afterwards (a model re-captures its step graphs).  rows <= 0 restores the
 * default, 65 (the measured crossover in whole verify steps: the warp-level
 * kernel is faster up to 64 rows).  Returns the value now in force.  Not thread-safe against
 * concurrent GEMM calls. */
int32_t sd_gemm_set_tc_min_rows(int32_t rows);

/* Finish of row blocks split over a whole number k (2..16) of CTAs in the
 * warp-level GEMM (q/k/v, O, down and other GEMMs with few row blocks): with
 * enable = 1 the k CTAs of a block run as one thread-block
 * cluster, stage their fp32 partials in shared memory and the first of them
 * sums the others' through distributed shared memory in CTA order before
 * the epilogue; with 0 (the default) they leave the partials in the
 * workspace and the last to finish sums them (an acq_rel ticket, measured
 * faster on GB300 at every shape tried).  The sums are the same up
 * to the sign of an all-zero sum.  A cluster size the GPU cannot schedule
 * falls back to the workspace path.  enable < 0 only queries.  Returns the
 * setting in force.  Process-wide; not thread-safe against concurrent GEMM
 * calls; a model re-captures its step graphs. */
int32_t sd_gemm_set_cluster_finish(int32_t enable);

/* Finish of row blocks split over a whole number k (2..16) of CTAs in the
 * warp-level GEMM (q/k/v, O, down: the launches with few row blocks), when
 * the cluster finish is off: with enable = 1 the GEMM's CTAs
 * leave their fp32 partials in the workspace and return, and a second
 * kernel on the same stream (one warp per 16-row strip) sums them in CTA
 * order and runs the epilogue - every contributor's partial in flight at
 * once, no ticket; with 0 (the default: the extra kernel boundary measured
 * slower on GB300) the last CTA of a block to finish sums them inside the
 * GEMM (an acq_rel ticket).  The sums are identical.  enable < 0 only
 * queries.  Returns the setting in force.  Process-wide; not thread-safe
 * against concurrent GEMM calls; a model re-captures its step graphs. */
int32_t sd_gemm_set_deferred_finish(int32_t enable);

/* Strip-parallel W12 GEMM for skinny launches ("SpecPilot ...", "(1) W12";
 * the O and down projections of the 8B-class decoder): with enable = 1 (the
 * default) a launch of at most 16 rows whose 16-row strips fit one wave of
 * two CTAs per SM (N / 16 <= 2 x SMs), without the argmax epilogue, runs one
 * CTA per strip over the whole k range - the 8 consumer warps take
 * alternate 64-column tiles and sum their fp32 partials in shared memory in
 * warp order, the strip's escape corrections come from the side list - so
 * no partial crosses CTAs (no split-K finisher); 0 sends such launches to
 * the warp-level kernel's split-K path.  Results equal up to the order of
 * fp32 sums.  enable < 0 only queries.  Returns the setting in force.
 * Process-wide; not thread-safe against concurrent GEMM calls; a model
 * re-captures its step graphs. */
int32_t sd_gemm_set_strip(int32_t enable);

/* Prefix key splits per (request, kv head, 64-row chunk) of the verify
 * step's attention ("SpecPilot ...", tree attention: the committed prefix
 * is split over CTAs and the splits' softmax states are merged; the tree's
 * own keys are one more split).  splits in 1..64 fixes the count (values
 * above 64 are clamped; a smaller count may still be taken when the model's
 * attention workspace holds fewer); splits <= 0 restores the automatic
 * choice (about two CTAs per SM, at least one split per 512 keys of the
 * context bound).  Process-wide; applies to steps issued afterwards (a
 * model re-captures its step graphs).  Returns the value now in force (0:
 * automatic).  Not thread-safe against concurrent steps. */
int32_t sd_attn_set_splits(int32_t splits);

/* ------------------------------------------------------ tree helpers -- */
/* [TREE] Validate one draft tree (parents[0] == -1, 0 <= parents[i] < i,
 * M <= 64) and derive per node the ancestor bitmask anc[i] = anc[parent[i]]
 * | 1<<i, the depth and the position ctx + depth.  On a bad tree, *status is
 * set to SD_ERR_BAD_TREE and anc[i] = 1<<i, depth = 0.  All device. */
int sd_tree_info(const int32_t* parents, int32_t M, int32_t ctx, uint64_t* anc, int32_t* depth, int32_t* pos,
                 int32_t* status, void* stream);

/* [EXACT] Greedy acceptance.  Node i >= 1 matches when tokens[i] ==
 * argmax[parents[i]]; a node is accepted when it and all its ancestors match
 * (the root always is).  The deepest accepted node d* wins (smallest index on
 * ties); accepted_len = depth(d*), accepted_tokens[0..len) = tokens on the
 * path below the root, bonus = argmax[d*], path[0..len] = node ids root..d*.
 * All device; path may be NULL.  A bad tree sets *status = SD_ERR_BAD_TREE,
 * accepted_len = 0 and bonus = -1. */
int sd_accept(const int32_t* tokens, const int32_t* parents, const int32_t* argmax, int32_t M,
              int32_t* accepted_len, int32_t* accepted_tokens, int32_t* bonus, int32_t* path, int32_t* status,
              void* stream);

/* ------------------------------------------ W12 with per-channel bases -- */
/* Device packer of the per-channel format (the format of w12c_pack_host,
 * bit for bit; words in the per-tensor layout).  w: bf16 [N][K] device;
 * row_src (device [N] or null): packed row n takes source row row_src[n]
 * (the fused tensors' row orders).  w12c_pack_analyze writes each packed
 * row's base (device uint8 [N]) and the side list's CSR row pointers
 * (device u32 [N+1]), fills meta (n_escapes; affine = 1 when every base is
 * at most 239; n_table 0) and synchronises `stream`.  w12c_pack_encode then
 * writes the words (w12_words_count) and the side list (esc_idx / esc_val
 * [meta->n_escapes], flat index order).  Errors: SD_ERR_INVALID_ARG,
 * SD_ERR_UNSUPPORTED (N % 16, K % 64, N*K < 2^32), SD_ERR_CUDA. */
int w12c_pack_analyze(const uint16_t* w, const int32_t* row_src, int64_t N, int64_t K, uint8_t* base,
                      uint32_t* row_ptr, w12_meta* meta, void* stream);
int w12c_pack_encode(const uint16_t* w, const int32_t* row_src, int64_t N, int64_t K, const uint8_t* base,
                     const uint32_t* row_ptr, uint32_t* words, uint32_t* esc_idx, uint16_t* esc_val, void* stream);

/* Per-output-channel W12 ("SpecPilot: AI Agent Framework Boosts Speculative
 * Decoding 10.87x", "(1) W12: Lossless 12-bit Weight Format", read
 * literally: a 4-bit exponent offset within each output channel), offline
 * host code.  Row n keeps base[n], the exponent starting the 15-exponent
 * window that holds most of the row's weights (the smaller base on ties);
 * a weight stores sign, e - base[n] (15: escaped, its bf16 in the side
 * list) and the 7-bit mantissa, in the per-tensor format's word layout
 * (escaped weights: code 15, sign and mantissa zero).  Host buffers: w
 * bf16 [N][K]; base u8 [N]; words u32 [w12_words_count(N,K)]; esc_idx u32
 * and esc_val u16 [esc_cap]; row_ptr u32 [N+1].  *n_escapes gets the
 * number of escapes; SD_ERR_WORKSPACE (nothing written past the bases)
 * when it exceeds esc_cap, so a call with esc_cap = 0 counts them.  Other
 * errors: SD_ERR_INVALID_ARG, SD_ERR_UNSUPPORTED (N%16, K%64, N*K < 2^32). */
int w12c_pack_host(const uint16_t* w, int64_t N, int64_t K, uint8_t* base, uint32_t* words, uint32_t* esc_idx,
                   uint16_t* esc_val, int64_t esc_cap, uint32_t* row_ptr, int64_t* n_escapes);

/* The bf16 weights back from a per-channel packed tensor (host buffers, as
 * w12c_pack_host writes them).  Errors: SD_ERR_INVALID_ARG,
 * SD_ERR_UNSUPPORTED, SD_ERR_CORRUPT (an escape index >= N*K). */
int w12c_unpack_host(const uint32_t* words, const uint8_t* base, int64_t N, int64_t K, const uint32_t* esc_idx,
                     const uint16_t* esc_val, int64_t n_escapes, uint16_t* w);

/* ------------------------------------------------ nested 8-bit plane -- */
/* [2-LEVEL] The nested 8-bit view of W12 as its own plane ("SpecPilot: AI
 * Agent Framework Boosts Speculative Decoding 10.87x", "(3) Two-Level
 * Verification": the first round verifies with W12's nested 8-bit weight
 * view): each weight's high byte of its 12-bit field, sign << 7 | code << 3
 * | top 3 mantissa bits (escaped weights: code 15, sign and mantissa zero),
 * 1 byte per weight, offline host code.  Layout: per 16-row strip and
 * 64-column super-tile, u32 [2 planes][32 lanes][4 sub-tiles]; lane 4g + q,
 * sub-tile j: plane 0 holds (row g, col c), (row g, c + 1), (row g + 8, c),
 * (row g + 8, c + 1) in bytes 0..3, c = 16 j + 2 q; plane 1 the same at
 * c + 8.  plane: u32 [N*K/4].  Pack from the bf16 weights w [N][K] and the
 * tensor's code table (w12_pack_analyze's).  Unpack gives the view: each
 * weight with its 4 low mantissa bits cleared (escaped weights from the
 * side list, cleared the same way).  Errors: SD_ERR_INVALID_ARG,
 * SD_ERR_UNSUPPORTED (N%16, K%64, N*K < 2^32), SD_ERR_CORRUPT (unpack: an
 * escape index >= N*K). */
int w12_plane8_pack_host(const uint16_t* w, int64_t N, int64_t K, const uint8_t* table, int32_t n_table,
                         uint32_t* plane);
/* The same plane on the device: from the bf16 weights w [N][K] (device),
 * with the code table of meta (w12_pack_analyze) and the optional row order
 * row_src of w12_pack_encode, into plane (device,
 * w12_plane8_words_count(N, K) u32, caller-allocated).  Asynchronous on
 * `stream`.  Errors: SD_ERR_INVALID_ARG, SD_ERR_UNSUPPORTED (shape). */
int64_t w12_plane8_words_count(int64_t N, int64_t K);
int w12_plane8_pack(const uint16_t* w, const int32_t* row_src, const w12_meta* meta, uint32_t* plane, void* stream);
int w12_plane8_unpack_host(const uint32_t* plane, int64_t N, int64_t K, const uint8_t* table, int32_t n_table,
                           const uint32_t* esc_idx, const uint16_t* esc_val, int64_t n_escapes, uint16_t* w);

/* ------------------------------------------------------- W12 on disk -- */
/* A packed tensor in a file, so that weights are packed once ("SpecPilot:
 * AI Agent Framework Boosts Speculative Decoding 10.87x", "(1) W12:
 * Lossless 12-bit Weight Format").  Host memory only: the caller copies the
 * arrays between the device and host buffers.  File (little-endian): a
 * 224-byte header (magic "SDVW12F\n", version 1, N, K, n_escapes, the
 * length of the escape tile index, the code table, n_table, affine, then
 * offset / size / CRC-32 of each section, then the CRC-32 of the header's
 * preceding bytes), followed by the sections at 16-byte aligned offsets:
 * words (u32 [w12_words_count(N,K)]), esc_idx (u32 [n_escapes]), esc_val
 * (u16 [n_escapes]), row_ptr (u32 [N+1]), tile_ptr (u32
 * [w12_tile_ptr_count(N,K)]), tile_esc (u32 [n_escapes]).  CRC-32: IEEE
 * 802.3 (reflected polynomial 0xEDB88320), as w12_crc32 computes it. */
uint32_t w12_crc32(const void* data, size_t n);

/* Write *t to path; t's array pointers are HOST pointers here (sizes as
 * above; the escape arrays may be NULL when n_escapes == 0).  Errors:
 * SD_ERR_INVALID_ARG (null pointer, shape outside N%16, K%64, N*K < 2^32),
 * SD_ERR_UNSUPPORTED (a per-channel tensor: the file holds per-tensor
 * tables only), SD_ERR_IO (open or write failed; the file may be partial). */
int w12_save(const char* path, const w12_tensor* t);

/* Read and check path's header (magic, version, header CRC, section sizes
 * against the shape): *meta gets N, K, the table, n_table, affine and
 * n_escapes, *n_tile_ptr (optional) the tile index length, so the caller
 * can size its buffers.  Errors: SD_ERR_INVALID_ARG, SD_ERR_IO (cannot
 * open), SD_ERR_CORRUPT. */
int w12_load_info(const char* path, w12_meta* meta, int64_t* n_tile_ptr);

/* Read every section into caller-allocated HOST buffers (sizes from
 * w12_load_info; the escape buffers may be NULL when there are no escapes),
 * checking each section's CRC and that the arrays form a packed tensor
 * (escape indices strictly increasing and below N*K, row_ptr counting the
 * escapes before each row, the escape tile index the one the side list
 * defines); fills *meta.  w12_save writes what it is given; this is where a
 * file is checked.  Errors: SD_ERR_INVALID_ARG, SD_ERR_IO, SD_ERR_CORRUPT
 * (bad header, short file, checksum mismatch or inconsistent arrays: the
 * buffers' contents are then unspecified). */
int w12_load(const char* path, uint32_t* words, uint32_t* esc_idx, uint16_t* esc_val, uint32_t* row_ptr,
             uint32_t* tile_ptr, uint32_t* tile_esc, w12_meta* meta);

/* ------------------------------------------ best-first node selection -- */
/* Gated delta rule over draft trees, in WY form ("SpecPilot: AI Agent
 * Framework Boosts Speculative Decoding 10.87x", "(2) Best-first Tree
 * Verification for Hybrid Architectures": Gated DeltaNet layers recompute
 * the state along each root path; a WY-form kernel evaluates many paths at
 * once).  Per request and head, q and k L2-normalised (zero stays zero):
 *   S_i = alpha_i (I - beta_i k_i k_i^T) S_parent(i) + beta_i k_i v_i^T,
 *   o_i = S_i^T q_i   (bf16),
 * S_root's parent state being the committed state S.  Evaluated for every
 * node at once (one unit-lower-triangular solve over the tree's ancestor
 * mask; S read once per request and head; no per-node state formed).
 *
 * Input (device): R requests, request r owning rows cu[r] .. cu[r+1]-1 (cu
 * int32 [R+1] on the device, the same values in cu_host; 1..64 rows per
 * request); q, k, v bf16 [rows][nh][128]; alpha (gate, in (0, 1]) and beta
 * (write strength, in [0, 1]) fp32 [rows][nh]; parents int32 [rows], local
 * to the request (root first with parent -1, 0 <= parent[i] < i); S fp32
 * [R][nh][128][128] (row = key dimension), not modified.  The path products
 * of alpha must stay in fp32's normal range.
 * Output: out bf16 [rows][nh][128]; workspace (sd_gdn_workspace(rows, nh)
 * bytes, 256-byte aligned, any content) receives what sd_gdn_commit needs.
 * A request whose parent array is invalid sets *status (device int32) to
 * SD_ERR_BAD_TREE and leaves its outputs unwritten.  Asynchronous on
 * `stream`.  Errors: SD_ERR_INVALID_ARG (null pointer, bad cu_host),
 * SD_ERR_UNSUPPORTED (a request outside 1..64 rows), SD_ERR_WORKSPACE. */
size_t sd_gdn_workspace(int32_t rows, int32_t nh);
int sd_gdn_tree_verify(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* alpha, const float* beta,
                       const int32_t* parents, const int32_t* cu, const int32_t* cu_host, int32_t R, int32_t nh,
                       const float* S, uint16_t* out, void* workspace, size_t workspace_bytes, int32_t* status,
                       void* stream);

/* After acceptance: S of request r becomes the state of its node last[r]
 * (device int32 [R], local index; the deepest accepted node), i.e. the rule
 * run over that node's root path ("(3) Two-Level Verification": only the
 * exact verification commits state).  Uses the workspace of the
 * sd_gdn_tree_verify call on the same inputs, which must precede it on
 * `stream`.  A request with last[r] outside its rows keeps its state.  S is
 * updated in place. */
int sd_gdn_commit(const int32_t* parents, const int32_t* cu, const int32_t* cu_host, int32_t R, int32_t nh,
                  const int32_t* last, float* S, const void* workspace, size_t workspace_bytes, void* stream);

/* [SELECT] Best-first selection of the nodes one batched verify checks,
 * under a node budget the requests share ("SpecPilot: AI Agent Framework
 * Boosts Speculative Decoding 10.87x", "(2) Best-first Tree Verification
 * for Hybrid Architectures": candidates ranked by parent-conditioned
 * log-probability, highest cumulative path scores kept; "(4) Three Batch
 * Optimization Mechanisms", Shared Node Budget).
 *
 * Input (device): R requests of drafted candidates, request r owning
 * entries cu[r] .. cu[r+1]-1 (cu: int32 [R+1], cu[0] = 0, cu[R] = n_total,
 * non-decreasing, 1..2048 candidates per request); parents: int32, local
 * to the request (entry 0 is the root with parent -1, 0 <= parent[i] < i);
 * logprob: fp32, the draft log-probability of node i given its parent
 * (<= 0, -inf allowed; ignored at the root); tokens (optional): int32.
 * Path score: 0 at the root, parent's score + logprob[i] (fp32, from the
 * root down).  Every request keeps its root; the other candidates are taken
 * in order of path score, highest first (equal scores: lower request, then
 * lower node index), passing over a candidate whose request holds `cap`
 * nodes (root included), until `budget` nodes are held in total.  Since a
 * node never scores above its parent, each request keeps a tree.
 *
 * Output (device, caller-allocated): out_cu int32 [R+1] (request r's kept
 * nodes are out_cu[r] .. out_cu[r+1]-1, in their original index order);
 * out_src int32, out_parents int32 (renumbered within the request, -1 at the
 * root), out_tokens int32 (optional, needs tokens), out_score fp32
 * (optional), each with room for min(budget, n_total) entries.  out_cu,
 * out_parents and the gathered tokens are the tokens / parents / cu of
 * sd_verify_batch (its cu is read on the host: copy out_cu back).
 *
 * Limits: 1 <= R <= n_total <= 16384 (else SD_ERR_INVALID_ARG /
 * SD_ERR_UNSUPPORTED), budget >= R and cap >= 1 (SD_ERR_INVALID_ARG).
 * workspace: sd_select_workspace(n_total) bytes of device memory, any
 * content.  *status (device int32, zeroed by the caller) becomes
 * SD_ERR_BAD_TREE when a request's parents or log-probabilities are invalid
 * (NaN, > 0): that request keeps nothing, the others are selected as if it
 * were absent; an invalid cu array sets it and zeroes out_cu.  Asynchronous
 * on `stream` (two kernels and a memset). */
size_t sd_select_workspace(int32_t n_total);
int sd_best_first_select(const int32_t* parents, const float* logprob, const int32_t* cu, int32_t R,
                         int32_t n_total, int32_t budget, int32_t cap, const int32_t* tokens, int32_t* out_cu,
                         int32_t* out_src, int32_t* out_parents, int32_t* out_tokens, float* out_score,
                         int32_t* status, void* workspace, size_t workspace_bytes, void* stream);

/* -------------------------------------------------------- tiny verify -- */
/* One linear layer and an lm_head: logits = (bf16(act W1^T)) Wlm^T, argmax
 * per node in fp32, then greedy acceptance over the tree.  act: bf16 [M][K];
 * logits (optional): bf16 [M][V]; argmax (optional) int32 [M].  M <= 64.
 * workspace: sd_tiny_workspace(W1->N, W1->K, Wlm->N, M) bytes. */
size_t sd_tiny_workspace(int64_t N1, int64_t K, int64_t V, int32_t M);
int sd_tiny_verify(const w12_tensor* W1, const w12_tensor* Wlm, const uint16_t* act, const int32_t* tokens,
                   const int32_t* parents, int32_t M, int32_t* accepted_len, int32_t* accepted_tokens,
                   int32_t* bonus, uint16_t* logits, int32_t* argmax, int32_t* status, void* workspace,
                   size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------- model -- */
/* Decoder whose every linear weight is W12.  Per layer (pre-norm):
 *   h = x + O(mix(RMSNorm(x))),  x' = h + down(silu(gate(n)) * up(n)), n = RMSNorm(h)
 * mix = tree-masked GQA attention with rotate-half RoPE at position
 * ctx + depth (layer_kind 0) or the tree linear recurrence (layer_kind 1):
 *   S_i = S_parent + phi(k_i) v_i^T, z_i = z_parent + phi(k_i),
 *   o_i = S_i^T phi(q_i) / (z_i . phi(q_i) + rec_eps), phi = elu + 1.
 * Then a final RMSNorm and the lm_head.  bf16 activations between kernels,
 * fp32 inside them. */

typedef struct {
  int32_t n_layers, hidden, inter, n_q_heads, n_kv_heads, head_dim, vocab;
  float rms_eps, rope_base, rec_eps;
  const int8_t* layer_kind_host; /* [n_layers]: 0 attention, 1 linear recurrent (copied) */
  int32_t max_rows;              /* max tree nodes per call summed over requests (<= 256) */
  int32_t max_requests;          /* max requests per sd_verify_batch call */
  int32_t max_positions;         /* RoPE table length: > largest ctx + depth used */
} sd_model_config;

/* Weight row orders the kernels expect (build them with w12_pack_encode's
 * row_src, see sd_model_row_map):
 *   qkv     = [q heads; k heads; v heads] rows, hidden columns.  Within each
 *             q or k head of 128 rows, strip i (16 rows) holds dims 8i..8i+7
 *             then 64+8i..64+8i+7 (the two halves of each RoPE pair);
 *             v heads in natural order.  Recurrent layers: [q; k; v], all
 *             natural, no RoPE.
 *   gate_up = 16-row strips j holding gate rows 8j..8j+7 then up rows
 *             8j..8j+7.
 *   o, down = natural. */
typedef struct {
  w12_tensor qkv, o, gate_up, down;
  const uint16_t* attn_norm;  /* bf16 [hidden] */
  const uint16_t* mlp_norm;   /* bf16 [hidden] */
} sd_layer_weights;

typedef struct {
  const sd_layer_weights* layers_host; /* [n_layers], copied */
  const uint16_t* embed;               /* bf16 [vocab][hidden], unpacked */
  const uint16_t* final_norm;          /* bf16 [hidden] */
  w12_tensor lm_head;                  /* [vocab][hidden] */
} sd_model_weights;

typedef struct sd_model sd_model;

/* Source row of packed row n for the fused tensors above.  kind 0: qkv of an
 * attention layer (rows = (Hq + 2 Hkv) * head_dim), kind 1: gate_up (rows =
 * 2 * inter; source = [gate; up]), kind 2: identity.  out_host[N]. */
int sd_model_row_map(int32_t kind, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t inter,
                     int32_t* out_host, int64_t N);

/* The model keeps the weight pointers (borrowed; they must outlive it) and
 * owns its workspace, activations, RoPE table and status word. */
int sd_model_create(const sd_model_config* cfg, const sd_model_weights* w, sd_model** out);
int sd_model_destroy(sd_model* m);

/* Contiguous per-request cache.  K/V: bf16 [n_attn_layers][n_kv_heads][cap][head_dim];
 * the committed prefix occupies slots [0, *ctx_len).  S, z (hybrid only):
 * fp32 [n_rec_layers][n_heads][head_dim][head_dim] (row = key dim) and
 * [n_rec_layers][n_heads][head_dim]. */
typedef struct {
  uint16_t* k;
  uint16_t* v;
  int64_t cap;
  float* S;
  float* z;
  int32_t* ctx_len;   /* device [1] */
} sd_kv;

/* Paged cache for batched verify.  K/V pools: bf16
 * [n_attn_layers][n_pages][n_kv_heads][page_size][head_dim]; request r's
 * logical slot t lives in page page_table[r*max_pages + t/page_size].
 * S, z (hybrid): [R][n_rec_layers][...] as in sd_kv.  ctx_len: device [R]. */
typedef struct {
  uint16_t* k_pool;
  uint16_t* v_pool;
  int32_t n_pages, page_size;
  const int32_t* page_table;  /* device [R][max_pages] */
  int32_t max_pages;
  float* S;
  float* z;
  int32_t* ctx_len;
} sd_paged_kv;

/* [TREE][EXACT] One verification step of a draft tree of M <= 64 nodes:
 * node 0 is the last committed token (its K/V is not in the cache yet), the
 * others are draft tokens with parents[i] < i.  Runs the target forward over
 * all nodes at once (node i at position ctx + depth(i), seeing the prefix and
 * its root path), takes the fp32 argmax per node, walks the greedy longest
 * accepted path (see sd_accept), moves the K/V of the root and the accepted
 * nodes to slots ctx + depth (recurrent layers: state += the path's updates)
 * and advances *ctx_len by accepted_len + 1.  Outputs (device):
 * accepted_len[1], accepted_tokens[M], bonus_token[1], logits (optional, bf16
 * [M][vocab]), argmax (optional, int32 [M]).  Asynchronous on `stream`; the
 * caller synchronises.  Requires ctx + M <= cap (else SD_ERR_CAPACITY on the
 * device and nothing is committed). */
int sd_verify_step(sd_model* m, const int32_t* tree_tokens, const int32_t* parents, int32_t M, const sd_kv* kv,
                   int32_t* accepted_len, int32_t* accepted_tokens, int32_t* bonus_token, uint16_t* logits,
                   int32_t* argmax, void* stream);

/* The forward part of sd_verify_step only: argmax (and logits) per node; the
 * new K/V are written to slots ctx + node but nothing is committed. */
int sd_forward(sd_model* m, const int32_t* tree_tokens, const int32_t* parents, int32_t M, const sd_kv* kv,
               uint16_t* logits, int32_t* argmax, void* stream);

/* Two-level verification ("SpecPilot: AI Agent Framework Boosts Speculative
 * Decoding 10.87x", "(3) Two-Level Verification"): round one runs the draft
 * tree on W12's nested 8-bit weight view, each weight with its 4 low
 * mantissa bits cleared, streaming 1 byte per weight; it produces argmax
 * (and logits) per node and accepts and commits nothing - its greedy walk
 * (sd_accept) gives the candidate chain the drafter continues from, and
 * one exact sd_verify_step of the chain and the new drafts decides.
 * sd_model_set_view8 registers the planes (w12_plane8_pack of each W12
 * tensor with the row order it was packed with; device, borrowed, 16-byte
 * aligned): planes_host[4 l + 0..3] = layer l's qkv, o, gate_up, down, then
 * planes_host[4 n_layers] = the lm_head's; n = 4 n_layers + 1.
 * sd_forward_view8 is sd_forward over the view (every linear on the
 * weight-streaming kernel); it needs M <= 64 and the registered planes,
 * else SD_ERR_UNSUPPORTED.  The new K/V it writes to
 * slots ctx + node are the view's (an exact step rewrites them). */
int sd_model_set_view8(sd_model* m, const uint32_t* const* planes_host, int32_t n);
int sd_forward_view8(sd_model* m, const int32_t* tree_tokens, const int32_t* parents, int32_t M, const sd_kv* kv,
                     uint16_t* logits, int32_t* argmax, void* stream);

/* Batched verify of R requests over a paged cache: request r owns nodes
 * [cu_nodes_host[r], cu_nodes_host[r+1]) of tokens/parents (parents local to
 * the request, <= 64 nodes each).  Every GEMM processes all rows at once;
 * attention, acceptance and compaction act per request.  Outputs per request
 * r: accepted_len[r], bonus[r], accepted_tokens[cu_nodes_host[r] ...]. */
int sd_verify_batch(sd_model* m, const int32_t* tokens, const int32_t* parents, const int32_t* cu_nodes_host,
                    int32_t R, const sd_paged_kv* kv, int32_t* accepted_len, int32_t* accepted_tokens,
                    int32_t* bonus, uint16_t* logits, int32_t* argmax, void* stream);

/* Copy the device status word of the model's last calls (synchronises the
 * device) and clear it; after a non-zero status the counters of the
 * streamed GEMM launches are also cleared (a launch that gave up on a wait
 * may have left them set). */
int sd_status(sd_model* m, int32_t* status_host);

/* Number of kernels the last sd_verify_step / sd_forward / sd_verify_batch
 * call launched. */
int sd_model_last_launches(sd_model* m);

/* The final RMSNorm's output of the last sd_verify_step / sd_forward /
 * sd_verify_batch call: the lm_head's input, bf16 [rows][hidden], rows in
 * the call's row order ("(2) Best-first Tree Verification ...": every node
 * is scored by the target's lm_head over this state).  Copied device to
 * device into the caller's `out` on `stream`, ordered after the step when
 * issued on the step's stream; valid until the next call on the model.
 * rows must be 1..max_rows (SD_ERR_INVALID_ARG otherwise).  A test tap:
 * with it, the argmax decision of a step can be checked against the lm_head
 * applied to the very state the step scored. */
int sd_model_final_hidden(sd_model* m, uint16_t* out, int32_t rows, void* stream);

/* Step execution mode.  With enable = 1 (the default), a call on a
 * non-default stream that is not itself being captured is recorded once per
 * distinct argument set (every pointer and size) into a CUDA graph, which is
 * replayed by later calls with the same arguments: no per-kernel launch cost
 * on the host.  Up to 16 graphs are kept per model.  enable = 0 launches the
 * kernels directly every call (also the behaviour on the legacy default
 * stream and inside a caller's own stream capture). */
int sd_model_set_graphs(sd_model* m, int32_t enable);

/* Schedule of skinny steps (rows <= 64, below the tensor-core threshold):
 * enable = 0 (the default) launches the warp-level W12 GEMM once per linear
 * with an RMSNorm kernel before gate/up and before the next q/k/v;
 * enable = 1 runs, on the weight-streaming kernel (sd_w12_linear_stream),
 * the linears between two attention (or recurrence)
 * kernels - O, gate/up, down and the next layer's q/k/v or the lm_head - as
 * one launch of four dependent GEMMs with the RMSNorms folded in (each
 * activation tile waits only for the blocks it reads).  Both give the same
 * results up to the order of fp32 split-K sums; drops captured graphs. */
int sd_model_set_fused(sd_model* m, int32_t enable);

/* Kernel kinds reported by sd_model_timeline (SD_K_GEMM_STREAM: one
 * streamed launch of several GEMMs; its bytes are those of the GEMMs it
 * runs). */
enum {
  SD_K_TREE = 0, SD_K_NORM = 1, SD_K_GEMM_QKV = 2, SD_K_ATTN = 3, SD_K_LINREC = 4, SD_K_GEMM_O = 5,
  SD_K_GEMM_GATE_UP = 6, SD_K_GEMM_DOWN = 7, SD_K_GEMM_LM_HEAD = 8, SD_K_ACCEPT = 9, SD_K_COMMIT = 10,
  SD_K_GEMM_STREAM = 11
};

/* Per-kernel timing of the following model calls: with enable = 1 every
 * kernel group of a step is bracketed by CUDA events on the call's stream and
 * the step is launched directly (no graph) behind a 30 ms busy-wait kernel,
 * so that the host has queued the whole step before the GPU reaches it and
 * host launch gaps do not enter the times.  The kernels launch without
 * programmatic dependent launch in this mode, each alone between its events,
 * so timed steps are slower than untimed ones; use the numbers for the
 * breakdown, not the step time. */
int sd_model_set_timing(sd_model* m, int32_t enable);

/* Timeline of the last timed call: for entry i, kind_host[i] (SD_K_*),
 * ms_host[i] (event-measured duration) and bytes_host[i] (algorithmic bytes
 * of the GEMMs of the launch: packed words, escape tile index, activations
 * read and written; an RMSNorm's rows read and written; 0 for other
 * kinds).  Synchronises the device.  Returns the number of entries written
 * (<= max), or -1 with sd_last_error set. */
int sd_model_timeline(sd_model* m, int32_t max, int32_t* kind_host, float* ms_host, double* bytes_host);

#ifdef __cplusplus
}
#endif
#endif /* SDV_H */
