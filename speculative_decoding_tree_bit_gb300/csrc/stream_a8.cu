// The streamed W12 kernel instantiated for one weight-decode mode.
#include <mutex>

#include "stream_kernel.cuh"

namespace sdv {

template <int NT>
static cudaError_t launch_nt(const StreamArgs& a, int grid, cudaStream_t s, bool pdl) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(k_w12_stream<NT, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, SCfg<NT>::SMEM);
    if (attr == cudaSuccess) attr = stream_check_residency(reinterpret_cast<const void*>(k_w12_stream<NT, 1>), NT);
  });
  if (attr != cudaSuccess) return attr;
  return launch(k_w12_stream<NT, 1>, dim3(grid), dim3(kSThreads), SCfg<NT>::SMEM, s, pdl, a);
}

template <>
cudaError_t stream_launch_dm<1>(const StreamArgs& a, int NT, int grid, cudaStream_t s, bool pdl) {
  switch (NT) {
    case 1: return launch_nt<1>(a, grid, s, pdl);
    case 2: return launch_nt<2>(a, grid, s, pdl);
    default: return launch_nt<8>(a, grid, s, pdl);
  }
}

}  // namespace sdv
