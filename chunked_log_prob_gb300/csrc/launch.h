// Internal launch interface between the host ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_tc.cuh"

namespace grpo {

struct FinalizeArgs {
  long long n;           // rows
  int splits;            // vocab splits of the forward pass
  long long part_ld;     // leading dimension of the split partials
  int vocab;
  int seq_len;
  int loss_mode;         // 0: logp only; 1: logp + GRPO loss + g
  const float* part_m;
  const float* part_s;
  const float* zy;
  const int32_t* ids;
  const uint8_t* mask;   // may be null (every row counts)
  const float* old_logp;
  const float* ref_logp;
  const float* adv;
  float eps_low, eps_high, beta, loss_den;
  const double* msum;    // device sum of the mask
  int seq_mode;          // 1: per-completion mean (weights 1 / (len_b B'))
  const int* seq_lens;   // [n / seq_len] unmasked tokens per completion
  const int* n_nonempty; // completions with len_b > 0
  float* lse_ws;         // [n]
  float* lse_out;        // optional
  float* logp_out;       // optional
  float* g_ws;           // [n] (loss mode)
  double* block_partials;
  unsigned* counter;
  float* loss_out;
  int* status;
};

// Stored-logit backward: per-row finish (lse, logp, token loss, g), and
// either in-place G formation (finalize_gform) or the row values alone for
// the dH GEMM that converts the logits itself (finalize_rows).
struct GformArgs {
  long long n_total;
  int n_rb, rb_offset;   // as TileArgs: row blocks of kSegs entries of seg_list
  const int* seg_list;
  const int* n_seg;
  int splits;
  long long part_ld;
  int vocab, seq_len;
  const float* part_m;
  const float* part_s;
  const float* zy;
  const int32_t* ids;
  const uint8_t* mask;
  const float* old_logp;
  const float* ref_logp;
  const float* adv;
  float eps_low, eps_high, beta, loss_den;
  const double* msum;
  int seq_mode;
  const int* seq_lens;
  const int* n_nonempty;
  float* logp_out;       // optional
  double* lt;            // [N] weighted token loss w_t l_t of unmasked rows
  float* lse_out;        // finalize_rows: [rows] lse (natural log), by global row
  float* g_out;          // finalize_rows: [rows] dL/dlogp (0 for rows that do not count)
  uint16_t* S;           // [chunk rows][ldS]: fp16 logits in (each 64-column box
                         // relative to its maximum, in log2 units), bf16 G out
  long long ldS;
  const float* box_max;  // [ceil(V / 64)][ldM] the boxes' maxima times log2 e
  long long ldM;
  int v0, width;         // single_pass_p: the vocabulary block of S (splits = slots so far)
  int xmode;
  float k0, k2;
  int* status;
};

struct FinishArgs {
  long long n;
  const int* status;     // the call's status word (a timed-out wait -> NaN outputs)
  const uint8_t* mask;
  const double* lt;
  float* logp_out;
  double* block_partials;
  unsigned* counter;
  float* loss_out;
};

constexpr int kGformThreads = 256;
constexpr int kFinalizeThreads = 256;
constexpr int kMaxFinalizeBlocks = 1024;

// Opt-in per-launch timing (grpo_launch_timing_enable). While it is on for the
// calling host thread, each launcher brackets its launch with two CUDA events
// recorded on the launch's own stream; grpo_launch_timing_read sums them per
// kernel. Off (the default), a LaunchTimer costs one thread-local load. Launches
// into a stream that is being captured are not timed. Defined in api.cu.
bool launch_timing_on();
class LaunchTimer {
 public:
  LaunchTimer(const char* name, cudaStream_t stream);
  LaunchTimer(int mode, int ctas, cudaStream_t stream);  // "tc_gemm_kernel<mode, ctas>"
  ~LaunchTimer();
  LaunchTimer(const LaunchTimer&) = delete;
  LaunchTimer& operator=(const LaunchTimer&) = delete;

 private:
  void begin(const char* name, cudaStream_t stream);
  int slot_ = -1;
  cudaStream_t stream_ = nullptr;
};

// Launch of one GEMM variant; a CTA pair (CTAS = 2) runs as a 2-CTA cluster.
// `grid` counts CTAs (a multiple of CTAS). map_c: the store map of the
// variants that write through TMA (PairCfg::kTmaStore), unused otherwise.
// map_h16: the hidden states in boxes of SEG rows (64 x 16, 128-byte swizzle),
// for the variants that read h by segments of the active-row list (the logit,
// G-tile and dW GEMMs), unused otherwise. map_hc: the chunk's copy of the rows
// of its non-consecutive row blocks (64 x 128 boxes; with args.hc set).
template <int MODE, int CTAS>
cudaError_t launch_gemm_variant(const CUtensorMap& map_a, const CUtensorMap& map_b,
                                const TileArgs& args, int grid, cudaStream_t stream,
                                const CUtensorMap* map_c = nullptr,
                                const CUtensorMap* map_h16 = nullptr,
                                const CUtensorMap* map_hc = nullptr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(PairCfg<MODE, CTAS>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = PairCfg<MODE, CTAS>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (CTAS == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  LaunchTimer timer(MODE, CTAS, stream);
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<MODE, CTAS>, map_a, map_b,
                            map_c != nullptr ? *map_c : map_a,
                            map_h16 != nullptr ? *map_h16 : map_a,
                            map_hc != nullptr ? *map_hc : map_a, args);
}

template <int MODE, int CTAS>
cudaError_t prepare_gemm_variant() {
  return cudaFuncSetAttribute(tc_gemm_kernel<MODE, CTAS>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              PairCfg<MODE, CTAS>::kSmemBytes);
}

// Each launcher lives in the translation unit that instantiates its kernels;
// ctas selects the single-CTA (1) or CTA-pair (2) variant.
cudaError_t prepare_fwd_gemm();   // opt-in to the large dynamic smem
cudaError_t prepare_bwd_gemms();
cudaError_t launch_fwd_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const CUtensorMap& map_h16,
                            const TileArgs& args, int grid, cudaStream_t stream,
                            const CUtensorMap* map_hc = nullptr);
// map_g: the chunk's bf16 G block [rows][ldG] as a store map, 64 x 32 boxes with
// the 128-byte swizzle (used by the CTA-pair variant).
cudaError_t launch_bwdg_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const CUtensorMap& map_h16,
                             const CUtensorMap& map_g, const TileArgs& args, int grid,
                             cudaStream_t stream,
                            const CUtensorMap* map_hc = nullptr);
cudaError_t launch_dh_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                           const TileArgs& args, int grid, cudaStream_t stream);
cudaError_t launch_dhs_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const TileArgs& args, int grid, cudaStream_t stream);
// After a tail-split dH-type launch (args.ts_part set): adds the pieces of its
// cut units and writes their dH rows (uacc: a U GEMM's units, whose sum goes
// through the single pass's U update). `units`: the launch's host-side bound.
cudaError_t launch_tail_fixup(int ctas, const TileArgs& args, int units, bool uacc,
                            cudaStream_t stream);
// map_a: one vocabulary block of stored fp16 logits [rows][width] (64 x 128
// boxes, 128-byte swizzle); map_b: W MN-major (64 x 64 boxes).
cudaError_t launch_uac_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const TileArgs& args, int grid, cudaStream_t stream);
// map_a: one vocabulary block of bf16 P [rows][width] (64 x 128 boxes), as
// single_pass_p_kernel leaves it; map_b: W MN-major.
cudaError_t launch_uap_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const TileArgs& args, int grid, cudaStream_t stream);
// map_dw: dW[v0 : v0 + dw_rows) as fp32 [rows][hidden], 32 x 32 boxes with the
// 128-byte swizzle (used by the CTA-pair variant).
cudaError_t launch_dw_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const CUtensorMap& map_h16,
                           const CUtensorMap& map_dw, const TileArgs& args, int grid,
                           cudaStream_t stream);
// Before a chunk's logit, G-tile or dW GEMM: the rows of its row blocks whose
// segments are not consecutive rows, copied into `out` (chunk rows x hidden).
// `args`: the chunk's TileArgs (rb_offset, n_rb, seg_list, n_seg, hidden, n_total).
cudaError_t launch_gather_blocks(const void* h, void* out, const TileArgs& args,
                                 cudaStream_t stream);
cudaError_t launch_row_plan(const uint8_t* mask, long long n, int n_segs, int* seg_list,
                            int* n_seg, double* msum, cudaStream_t stream);
cudaError_t launch_seq_lens(const uint8_t* mask, long long n, int seq_len, int* lens,
                            int* n_nonempty, cudaStream_t stream);
cudaError_t launch_zero_padding_blocks(const uint8_t* mask, long long n, int n_rb, int hidden,
                                       void* dH, int sms, cudaStream_t stream);
cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t stream);
cudaError_t prepare_fwds_gemm();
// map_s: the chunk's fp16 logit block [rows][ldS] as a store map, 64 x 32 boxes
// with the 128-byte swizzle (used by the CTA-pair variant).
cudaError_t launch_fwds_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const CUtensorMap& map_h16,
                             const CUtensorMap& map_s, const TileArgs& args, int grid,
                             cudaStream_t stream,
                            const CUtensorMap* map_hc = nullptr);
cudaError_t launch_finalize_gform(const GformArgs& a, int rows, cudaStream_t stream);
cudaError_t launch_finalize_rows(const GformArgs& a, int rows, cudaStream_t stream);
cudaError_t launch_single_pass_p(const GformArgs& a, int rows, cudaStream_t stream);
cudaError_t launch_finish_loss(const FinishArgs& a, cudaStream_t stream);
cudaError_t launch_bounded_wait_selftest(int* status, int* waited_out, cudaStream_t stream);

}  // namespace grpo
