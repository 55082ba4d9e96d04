// W12 weight-streaming GEMM launches: interface.
#pragma once

#include "gemm.cuh"

namespace sdv {

constexpr int kStreamMaxPhases = 4;
constexpr int kStreamMaxRows = 64;  // rows of one streamed launch (up to 8 token tiles)

// One GEMM of a streamed launch, as the host describes it.
struct StreamPhaseDesc {
  const w12_tensor* W = nullptr;
  // the tensor's nested 8-bit plane (w12_plane8_pack): when set, the phase
  // streams it (1 byte per weight) and multiplies by the 8-bit view of W,
  // each weight with its 4 low mantissa bits cleared (escapes likewise)
  const uint32_t* view8 = nullptr;
  const uint16_t* x = nullptr;  // activations bf16 [x_rows][K]
  int x_rows = 0;               // rows of the x buffer (the tensor map's extent)
  GemmEpilogue epi{};
  // Activations from an earlier phase of the same launch: dep is its index
  // (-1: x was written before the launch).  dep_fine = 1: k-tile t of x is
  // row block t of phase dep (the SiLU-mul output of a gate/up phase feeding
  // a down phase), so each tile waits for that block only; otherwise every
  // block of phase dep.
  int dep = -1;
  int dep_fine = 0;
  // RMSNorm of x folded into the activation load: xn = bf16((x / rms) *
  // gamma), rms from the per-row-block sums of squares that phase `dep`
  // (EPI_RESID with out_ss) writes; gamma null: x is used as it is.
  const uint16_t* norm_gamma = nullptr;
  float norm_eps = 0.f;
  uint16_t* norm_out = nullptr;  // optional: the normalised activations, bf16 [M][K]
  // EPI_RESID: per row block b and token row m, the sum of squares of the
  // block's bf16 outputs, out_ss[b * 128 + m] (feeds a later phase's norm);
  // room for NB * 128 floats
  float* out_ss = nullptr;
};

// Scratch of streamed launches.  state: per launch site, ints that are zero
// between launches (each launch's last CTA clears what it used); partial:
// split-K partial sums, shared by all sites (a launch writes them only
// after the previous kernel completed).
struct StreamWorkspace {
  int32_t* state = nullptr;
  size_t state_ints = 0;
  float* partial = nullptr;
  size_t partial_floats = 0;
};

// CTAs of a streamed launch for M rows.
int stream_grid(int M);
// State ints and partial floats one launch of these phases needs.
size_t stream_state_ints(const StreamPhaseDesc* ph, int n);
size_t stream_partial_floats(const StreamPhaseDesc* ph, int n, int M);
// Upper bounds for any launch of at most kStreamMaxPhases GEMMs with at most
// n_max output rows and k_max inputs each (workspace sizing).
size_t stream_state_ints_bound(int64_t n_max);
size_t stream_partial_floats_bound(int64_t n_max, int64_t k_max, int M);

// y = epilogue(x W^T) for every phase, rows [0, M) (M <= 64), in one
// persistent launch: each CTA takes a contiguous share of each phase's
// (row block, k-tile) tiles in turn (stream-K) while its producer streams
// their weights; activation tiles wait only for the blocks of earlier
// phases they read.
int stream_launch(const StreamPhaseDesc* ph, int n, int M, const StreamWorkspace& ws, int32_t* status,
                  cudaStream_t s, bool pdl);

// Event log of streamed launches (diagnostics; see sd_stream_set_trace).
int stream_set_trace(uint64_t* buf, size_t bytes);
int stream_trace_launches();

}  // namespace sdv
