// Launchers of the backward GEMM variants, and the translation unit that
// instantiates them (the kernel template itself is tc_gemm_kernel in
// gemm_tc.cuh): the G tile (recomputed logits -> bf16 softmax-Jacobian rows),
// the dH accumulation from a G block or straight from a stored fp16 logit
// block, the single pass's U accumulation, and the lm_head gradient, each in
// the single-CTA and the CTA-pair variant, and the fixup pass of the
// tail-split dH launches. No kernel is defined here; the file exists so that these
// instantiations compile in parallel with the others.
#include "launch.h"

namespace grpo {

cudaError_t prepare_bwd_gemms() {
  cudaError_t e = prepare_gemm_variant<MODE_BWDG, 1>();
  if (e == cudaSuccess) e = prepare_gemm_variant<MODE_BWDG, 2>();
  if (e == cudaSuccess) e = prepare_gemm_variant<MODE_DH, 1>();
  if (e == cudaSuccess) e = prepare_gemm_variant<MODE_DH, 2>();
  if (e == cudaSuccess) e = prepare_gemm_variant<MODE_DW, 1>();
  if (e == cudaSuccess) e = prepare_gemm_variant<MODE_DW, 2>();
  if (e == cudaSuccess) e = prepare_gemm_variant<MODE_DHS, 1>();
  if (e == cudaSuccess) e = prepare_gemm_variant<MODE_DHS, 2>();
  if (e == cudaSuccess) e = prepare_gemm_variant<MODE_UAC, 1>();
  if (e == cudaSuccess) e = prepare_gemm_variant<MODE_UAC, 2>();
  if (e == cudaSuccess) e = prepare_gemm_variant<MODE_UAP, 1>();
  if (e == cudaSuccess) e = prepare_gemm_variant<MODE_UAP, 2>();
  return e;
}

cudaError_t launch_dw_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const CUtensorMap& map_h16,
                           const CUtensorMap& map_dw, const TileArgs& args, int grid,
                           cudaStream_t stream) {
  return ctas == 2 ? launch_gemm_variant<MODE_DW, 2>(map_a, map_b, args, grid, stream, &map_dw, &map_h16)
                   : launch_gemm_variant<MODE_DW, 1>(map_a, map_b, args, grid, stream, nullptr, &map_h16);
}

cudaError_t launch_bwdg_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const CUtensorMap& map_h16,
                             const CUtensorMap& map_g, const TileArgs& args, int grid,
                             cudaStream_t stream,
                             const CUtensorMap* map_hc) {
  return ctas == 2 ? launch_gemm_variant<MODE_BWDG, 2>(map_a, map_b, args, grid, stream, &map_g, &map_h16, map_hc)
                   : launch_gemm_variant<MODE_BWDG, 1>(map_a, map_b, args, grid, stream, nullptr, &map_h16, map_hc);
}

cudaError_t launch_dh_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                           const TileArgs& args, int grid, cudaStream_t stream) {
  return ctas == 2 ? launch_gemm_variant<MODE_DH, 2>(map_a, map_b, args, grid, stream)
                   : launch_gemm_variant<MODE_DH, 1>(map_a, map_b, args, grid, stream);
}

cudaError_t launch_dhs_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const TileArgs& args, int grid, cudaStream_t stream) {
  return ctas == 2 ? launch_gemm_variant<MODE_DHS, 2>(map_a, map_b, args, grid, stream)
                   : launch_gemm_variant<MODE_DHS, 1>(map_a, map_b, args, grid, stream);
}

cudaError_t launch_tail_fixup(int ctas, const TileArgs& args, int units, bool uacc,
                            cudaStream_t stream) {
  if (units <= 0) return cudaSuccess;
  LaunchTimer timer("tail_fixup_kernel", stream);
  const dim3 grid2(units, PairCfg<MODE_DH, 2>::kTileN / 32), grid1(units, PairCfg<MODE_DH, 1>::kTileN / 32);
  if (ctas == 2) {
    if (uacc) tail_fixup_kernel<2, true><<<grid2, BM * 2, 0, stream>>>(args);
    else tail_fixup_kernel<2, false><<<grid2, BM * 2, 0, stream>>>(args);
  } else {
    if (uacc) tail_fixup_kernel<1, true><<<grid1, BM, 0, stream>>>(args);
    else tail_fixup_kernel<1, false><<<grid1, BM, 0, stream>>>(args);
  }
  return cudaGetLastError();
}

cudaError_t launch_uac_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const TileArgs& args, int grid, cudaStream_t stream) {
  return ctas == 2 ? launch_gemm_variant<MODE_UAC, 2>(map_a, map_b, args, grid, stream)
                   : launch_gemm_variant<MODE_UAC, 1>(map_a, map_b, args, grid, stream);
}

cudaError_t launch_uap_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const TileArgs& args, int grid, cudaStream_t stream) {
  return ctas == 2 ? launch_gemm_variant<MODE_UAP, 2>(map_a, map_b, args, grid, stream)
                   : launch_gemm_variant<MODE_UAP, 1>(map_a, map_b, args, grid, stream);
}

}  // namespace grpo
