// Backward-side GEMM launchers: the G tile (recomputed logits -> bf16
// softmax-Jacobian rows) and the dH accumulation.
#include "launch.h"

namespace grpo {

cudaError_t prepare_bwd_gemms() {
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<MODE_BWDG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       GEMM_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tc_gemm_kernel<MODE_DH>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM_BYTES);
}

cudaError_t launch_bwdg_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b,
                             const TileArgs& args, int grid, cudaStream_t stream) {
  tc_gemm_kernel<MODE_BWDG><<<grid, GEMM_THREADS, GEMM_SMEM_BYTES, stream>>>(map_a, map_b,
                                                                             args);
  return cudaGetLastError();
}

cudaError_t launch_dh_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b,
                           const TileArgs& args, int grid, cudaStream_t stream) {
  tc_gemm_kernel<MODE_DH><<<grid, GEMM_THREADS, GEMM_SMEM_BYTES, stream>>>(map_a, map_b, args);
  return cudaGetLastError();
}

}  // namespace grpo
