// Forward-side kernels: the logit GEMM with online log-sum-exp (MODE_FWD),
// the mask count, and the per-row finalisation (log-sum-exp combine,
// selective log-prob, GRPO token loss and its derivative, deterministic
// fp64 loss reduction).
#include "launch.h"

namespace grpo {

cudaError_t prepare_fwd_gemm() {
  return cudaFuncSetAttribute(tc_gemm_kernel<MODE_FWD>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM_BYTES);
}

cudaError_t launch_fwd_gemm(const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const TileArgs& args, int grid, cudaStream_t stream) {
  tc_gemm_kernel<MODE_FWD><<<grid, GEMM_THREADS, GEMM_SMEM_BYTES, stream>>>(map_a, map_b, args);
  return cudaGetLastError();
}

__global__ void __launch_bounds__(1024) count_mask_kernel(const uint8_t* __restrict__ mask,
                                                          long long n, double* out) {
  __shared__ unsigned long long warp_sums[32];
  unsigned long long s = 0;
  if (mask == nullptr) {
    s = threadIdx.x == 0 ? static_cast<unsigned long long>(n) : 0ull;
  } else {
    for (long long i = threadIdx.x; i < n; i += blockDim.x) s += mask[i] != 0;
  }
  for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    s = threadIdx.x < (blockDim.x >> 5) ? warp_sums[threadIdx.x] : 0ull;
    for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
    if (threadIdx.x == 0) *out = static_cast<double>(s);
  }
}

// Fixed-shape block sum of a double (deterministic for a given blockDim).
__device__ double block_sum(double v, double* sh) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) sh[w] = v;
  __syncthreads();
  double r = 0.0;
  if (threadIdx.x < 32) {
    r = threadIdx.x < (blockDim.x >> 5) ? sh[threadIdx.x] : 0.0;
    for (int o = 16; o > 0; o >>= 1) r += __shfl_down_sync(0xffffffffu, r, o);
  }
  __syncthreads();
  return r;  // valid in thread 0
}

__global__ void __launch_bounds__(kFinalizeThreads) finalize_kernel(const FinalizeArgs a) {
  __shared__ double sh[32];
  __shared__ bool is_last;
  const double mden = a.loss_mode ? (a.loss_den > 0.f ? static_cast<double>(a.loss_den) : *a.msum)
                                  : 0.0;
  double local = 0.0;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < a.n;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    // log-sum-exp from the per-split (max, sum) pairs, base-2 domain.
    float m2 = -INFINITY;
    for (int s = 0; s < a.splits; ++s) m2 = fmaxf(m2, a.part_m[s * a.part_ld + t]);
    float ssum = 0.f;
    for (int s = 0; s < a.splits; ++s)
      ssum += a.part_s[s * a.part_ld + t] * exp2f(a.part_m[s * a.part_ld + t] - m2);
    const float lse = (m2 + log2f(ssum)) * 0.69314718055994531f;
    a.lse_ws[t] = lse;
    if (a.lse_out) a.lse_out[t] = lse;

    const bool counted = !a.loss_mode || a.mask == nullptr || a.mask[t] != 0;
    float logp = 0.f;
    float gval = 0.f;
    if (counted) {
      const int y = a.ids[t];
      if (y < 0 || y >= a.vocab) {
        atomicCAS(a.status, 0, GRPO_ERR_BAD_TOKEN_ID);
        logp = __int_as_float(0x7fc00000);  // NaN
      } else {
        logp = a.zy[t] - lse;
      }
      if (a.loss_mode) {
        const double lp = logp;
        const double A = a.adv[t / a.seq_len];
        const double r = exp(lp - static_cast<double>(a.old_logp[t]));
        const double lo = 1.0 - static_cast<double>(a.eps_low);
        const double hi = 1.0 + static_cast<double>(a.eps_high);
        const double c = fmin(fmax(r, lo), hi);
        const double surr = fmin(r * A, c * A);
        const double d = static_cast<double>(a.ref_logp[t]) - lp;
        const double ed = exp(d);
        const double kl = ed - d - 1.0;
        local += -surr + static_cast<double>(a.beta) * kl;
        const bool clipped = (A > 0.0 && r > hi) || (A < 0.0 && r < lo);
        const double dl = -(clipped ? 0.0 : A * r) + static_cast<double>(a.beta) * (1.0 - ed);
        gval = mden != 0.0 ? static_cast<float>(dl / mden) : 0.f;
      }
    }
    if (a.logp_out) a.logp_out[t] = logp;
    if (a.loss_mode) a.g_ws[t] = gval;
  }
  if (!a.loss_mode) return;

  // Deterministic two-level reduction: fixed block partials, summed in order
  // by the last block to finish.
  const double bsum = block_sum(local, sh);
  if (threadIdx.x == 0) {
    a.block_partials[blockIdx.x] = bsum;
    __threadfence();
    const unsigned done = atomicAdd(a.counter, 1u);
    is_last = (done == gridDim.x - 1);
  }
  __syncthreads();
  if (is_last) {
    __threadfence();
    double v = 0.0;
    for (unsigned i = threadIdx.x; i < gridDim.x; i += blockDim.x)
      v += reinterpret_cast<volatile double*>(a.block_partials)[i];
    const double tot = block_sum(v, sh);
    if (threadIdx.x == 0) {
      *a.loss_out = mden != 0.0 ? static_cast<float>(tot / mden) : 0.f;
      *a.counter = 0;
    }
  }
}

cudaError_t launch_count_mask(const uint8_t* mask, long long n, double* out,
                              cudaStream_t stream) {
  count_mask_kernel<<<1, 1024, 0, stream>>>(mask, n, out);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t stream) {
  long long blocks = (a.n + kFinalizeThreads - 1) / kFinalizeThreads;
  if (blocks < 1) blocks = 1;
  if (blocks > kMaxFinalizeBlocks) blocks = kMaxFinalizeBlocks;
  finalize_kernel<<<static_cast<int>(blocks), kFinalizeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace grpo
