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
  float* lse_ws;         // [n]
  float* lse_out;        // optional
  float* logp_out;       // optional
  float* g_ws;           // [n] (loss mode)
  double* block_partials;
  unsigned* counter;
  float* loss_out;
  int* status;
};

// Stored-logit backward: per-row finish + in-place G formation.
struct GformArgs {
  long long n_total;
  int n_rb, rb_offset;
  const int* rb_list;
  const int* n_active;
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
  float* logp_out;       // optional
  double* lt;            // [N] token loss of unmasked rows
  uint16_t* S;           // [chunk rows][ldS]: fp16 logits in, bf16 G out
  long long ldS;
  int xmode;
  float k0, k2;
  int* status;
};

struct FinishArgs {
  long long n;
  const uint8_t* mask;
  const double* lt;
  float* logp_out;
  float loss_den;
  const double* msum;
  double* block_partials;
  unsigned* counter;
  float* loss_out;
};

constexpr int kGformThreads = 256;
constexpr int kFinalizeThreads = 256;
constexpr int kMaxFinalizeBlocks = 1024;

// Each launcher lives in the translation unit that instantiates its kernel.
cudaError_t prepare_fwd_gemm();   // opt-in to the large dynamic smem
cudaError_t prepare_bwd_gemms();
cudaError_t launch_fwd_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const TileArgs& args, int grid, cudaStream_t stream);
cudaError_t launch_bwdg_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b,
                             const TileArgs& args, int grid, cudaStream_t stream);
cudaError_t launch_dh_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b,
                           const TileArgs& args, int grid, cudaStream_t stream);
cudaError_t launch_row_plan(const uint8_t* mask, long long n, int n_rb, int* rb_list,
                            int* n_active, double* msum, cudaStream_t stream);
cudaError_t launch_zero_padding_blocks(const uint8_t* mask, long long n, int n_rb, int hidden,
                                       void* dH, int sms, cudaStream_t stream);
cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t stream);
cudaError_t prepare_fwds_gemm();
cudaError_t launch_fwds_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b,
                             const TileArgs& args, int grid, cudaStream_t stream);
cudaError_t launch_finalize_gform(const GformArgs& a, int rows, cudaStream_t stream);
cudaError_t launch_finish_loss(const FinishArgs& a, cudaStream_t stream);

}  // namespace grpo
