// Persistent GEMM chain: launch interface.
#pragma once

#include "gemm.cuh"

namespace sdv {

enum ChainPhaseType : int { PH_GEMM = 0, PH_NORM = 1 };

constexpr int kChainMaxPhases = 6;

// dst[m] = bf16((src[m] * (1 / sqrt(mean(src[m]^2) + eps))) * gamma), fp32 inside.
struct ChainNorm {
  const uint16_t* src = nullptr;
  const uint16_t* gamma = nullptr;
  uint16_t* dst = nullptr;
  int H = 0;
  float eps = 0.f;
};

// One phase as the host describes it.
struct ChainPhaseDesc {
  int type = PH_GEMM;
  const w12_tensor* W = nullptr;  // PH_GEMM: weights, input x [rows][K] and its map, epilogue
  const uint16_t* x = nullptr;
  const XMap* xm = nullptr;
  GemmEpilogue epi{};
  ChainNorm norm{};  // PH_NORM
};

// Grid of the chain kernel for M rows (equal to gemm_grid(M)); 0 when the
// chain cannot keep all its CTAs resident (then GEMMs are launched one by one).
int chain_grid(int M);

// Run phases ph[0..n) (n <= kChainMaxPhases, M <= 128 rows) in one persistent
// launch; phase i + 1 starts on a CTA once every CTA has finished phase i.
// bar: two zero-initialised 64-bit words (arrival counter, its value after the
// last launch) owned by the caller and used by one chain at a time (the
// counter only grows; 2^64 arrivals never wrap).  trace (optional, [1 + 3n][grid] u64): globaltimer when each
// CTA starts (row 0) and, for phase i, when its first stage is ready (row
// 1 + 3i; for an RMSNorm phase: its input is complete), when its last stage
// is consumed (row 2 + 3i; RMSNorm: rows written) and when it finished the
// phase (row 3 + 3i).  A CTA without work in a GEMM phase leaves rows 1 + 3i
// and 2 + 3i unwritten.
int chain_launch(const ChainPhaseDesc* ph, int n, int M, const GemmWorkspace& ws, unsigned long long* bar,
                 int32_t* status, cudaStream_t s, bool pdl, uint64_t* trace = nullptr);

}  // namespace sdv
