// Forward-side kernels: the logit GEMM with online log-sum-exp (MODE_FWD),
// the mask count, and the per-row finalisation (log-sum-exp combine,
// selective log-prob, GRPO token loss and its derivative, deterministic
// fp64 loss reduction).
#include <cuda_fp16.h>

#include <algorithm>

#include "launch.h"

namespace grpo {

cudaError_t prepare_fwd_gemm() {
  cudaError_t e = prepare_gemm_variant<MODE_FWD, 1>();
  return e == cudaSuccess ? prepare_gemm_variant<MODE_FWD, 2>() : e;
}

cudaError_t launch_fwd_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const CUtensorMap& map_h16,
                            const TileArgs& args, int grid, cudaStream_t stream,
                            const CUtensorMap* map_hc) {
  return ctas == 2 ? launch_gemm_variant<MODE_FWD, 2>(map_a, map_b, args, grid, stream, nullptr, &map_h16, map_hc)
                   : launch_gemm_variant<MODE_FWD, 1>(map_a, map_b, args, grid, stream, nullptr, &map_h16, map_hc);
}

// The active-row list of a loss call: the 16-row segments that hold any
// unmasked row, in order (seg_list, n_seg), and the mask's sum.
__global__ void __launch_bounds__(1024) row_plan_kernel(const uint8_t* __restrict__ mask,
                                                        long long n, int n_segs,
                                                        int* __restrict__ seg_list,
                                                        int* __restrict__ n_seg,
                                                        double* __restrict__ msum) {
  __shared__ int warp_off[32];
  __shared__ int chunk_total;
  __shared__ unsigned long long warp_tok[32];
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const int n_warps = blockDim.x >> 5;
  int base = 0;
  unsigned long long tokens = 0;
  for (int b0 = 0; b0 < n_segs; b0 += blockDim.x) {
    const int sg = b0 + threadIdx.x;
    int cnt = 0;
    if (sg < n_segs) {
      const long long r0 = static_cast<long long>(sg) * SEG;
      const long long r1 = min(r0 + SEG, n);
      if (mask == nullptr) {
        cnt = static_cast<int>(r1 - r0);
      } else {
        for (long long r = r0; r < r1; ++r) cnt += mask[r] != 0;
      }
    }
    tokens += static_cast<unsigned long long>(cnt);
    const bool active = cnt > 0;
    const unsigned bal = __ballot_sync(0xffffffffu, active);
    const int pre = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) warp_off[w] = __popc(bal);
    __syncthreads();
    if (w == 0) {
      const int v = lane < n_warps ? warp_off[lane] : 0;
      int incl = v;
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
      }
      if (lane < n_warps) warp_off[lane] = incl - v;
      if (lane == 31) chunk_total = incl;
    }
    __syncthreads();
    if (active) seg_list[base + warp_off[w] + pre] = sg;
    base += chunk_total;
    __syncthreads();
  }
  for (int o = 16; o > 0; o >>= 1) tokens += __shfl_down_sync(0xffffffffu, tokens, o);
  if (lane == 0) warp_tok[w] = tokens;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long t = 0;
    for (int i = 0; i < n_warps; ++i) t += warp_tok[i];
    *msum = static_cast<double>(t);
    *n_seg = base;
  }
}

// dH rows of row blocks without any unmasked token are never touched by the
// backward GEMMs; they are written as exact zeros here.
// dH rows of the 16-row segments without an unmasked row (no GEMM computes
// them): zeros. Per 128-row block, the inactive segments' rows.
__global__ void __launch_bounds__(256) zero_padding_blocks_kernel(
    const uint8_t* __restrict__ mask, long long n, int n_rb, int hidden,
    __nv_bfloat16* __restrict__ dH) {
  __shared__ int any[kSegs];
  for (int rb = blockIdx.x; rb < n_rb; rb += gridDim.x) {
    if (threadIdx.x < kSegs) any[threadIdx.x] = 0;
    __syncthreads();
    const long long r0 = static_cast<long long>(rb) * BM;
    const long long r1 = min(r0 + BM, n);
    if (r0 + threadIdx.x < r1 && mask[r0 + threadIdx.x] != 0) any[threadIdx.x / SEG] = 1;
    __syncthreads();
    // hidden % 8 == 0: 16-byte stores of 8 bf16.
    const int vecs_row = hidden / 8;
    const long long vecs = (r1 - r0) * vecs_row;
    uint4* dst = reinterpret_cast<uint4*>(dH + r0 * hidden);
    for (long long i = threadIdx.x; i < vecs; i += blockDim.x)
      if (!any[static_cast<int>(i / vecs_row) / SEG]) dst[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
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

// Unmasked tokens per completion (b = t / seq_len) and the number of
// completions that have any; one block per completion (grid-stride).
__global__ void __launch_bounds__(256) seq_lens_kernel(const uint8_t* __restrict__ mask,
                                                       long long n, int seq_len,
                                                       int* __restrict__ lens,
                                                       int* __restrict__ n_nonempty) {
  __shared__ int warp_cnt[8];
  const long long n_seq = n / seq_len;
  for (long long b = blockIdx.x; b < n_seq; b += gridDim.x) {
    int c = 0;
    const long long r0 = b * seq_len;
    if (mask == nullptr) {
      c = threadIdx.x == 0 ? seq_len : 0;
    } else {
      for (long long r = r0 + threadIdx.x; r < r0 + seq_len; r += blockDim.x) c += mask[r] != 0;
    }
    for (int o = 16; o > 0; o >>= 1) c += __shfl_down_sync(0xffffffffu, c, o);
    if ((threadIdx.x & 31) == 0) warp_cnt[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) tot += warp_cnt[w];
      lens[b] = tot;
      if (tot > 0) atomicAdd(n_nonempty, 1);
    }
    __syncthreads();
  }
}

// Weight of an unmasked token in the loss: 1 / M for the token mean, or
// 1 / (len_b B') for the mean over completions of their token means.
__device__ __forceinline__ double token_weight(int seq_mode, float loss_den, const double* msum,
                                               const int* seq_lens, const int* n_nonempty,
                                               long long t, int seq_len) {
  double den;
  if (seq_mode) {
    const double bcount = loss_den > 0.f ? static_cast<double>(loss_den) : *n_nonempty;
    den = static_cast<double>(seq_lens[t / seq_len]) * bcount;
  } else {
    den = loss_den > 0.f ? static_cast<double>(loss_den) : *msum;
  }
  return den != 0.0 ? 1.0 / den : 0.0;
}

__global__ void __launch_bounds__(kFinalizeThreads) finalize_kernel(const FinalizeArgs a) {
  __shared__ double sh[32];
  __shared__ bool is_last;
  double local = 0.0;
  // A wait of the logit GEMM that ran out leaves its partials incomplete:
  // every output of the call is then NaN (the status word says why).
  const bool aborted = *reinterpret_cast<const volatile int*>(a.status) == GRPO_ERR_DEVICE_TIMEOUT;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < a.n;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const bool counted = !a.loss_mode || a.mask == nullptr || a.mask[t] != 0;
    // log-sum-exp from the per-split (max, sum) pairs, base-2 domain. Masked
    // rows of a loss call may sit in skipped row blocks with no partials.
    float lse = 0.f;
    if (counted) {
      float m2 = -INFINITY;
      for (int s = 0; s < a.splits; ++s) m2 = fmaxf(m2, a.part_m[s * a.part_ld + t]);
      float ssum = 0.f;
      for (int s = 0; s < a.splits; ++s)
        ssum += a.part_s[s * a.part_ld + t] * exp2f(a.part_m[s * a.part_ld + t] - m2);
      lse = (m2 + log2f(ssum)) * 0.69314718055994531f;
      if (aborted) lse = __int_as_float(0x7fc00000);
      else if (!isfinite(lse)) atomicCAS(a.status, 0, GRPO_ERR_NONFINITE);
    }
    a.lse_ws[t] = lse;
    if (a.lse_out) a.lse_out[t] = lse;

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
        const double wt = token_weight(a.seq_mode, a.loss_den, a.msum, a.seq_lens,
                                       a.n_nonempty, t, a.seq_len);
        local += (-surr + static_cast<double>(a.beta) * kl) * wt;
        const bool clipped = (A > 0.0 && r > hi) || (A < 0.0 && r < lo);
        const double dl = -(clipped ? 0.0 : A * r) + static_cast<double>(a.beta) * (1.0 - ed);
        gval = static_cast<float>(dl * wt);
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
      *a.loss_out = aborted ? __int_as_float(0x7fc00000) : static_cast<float>(tot);
      *a.counter = 0;
    }
  }
}

cudaError_t launch_seq_lens(const uint8_t* mask, long long n, int seq_len, int* lens,
                            int* n_nonempty, cudaStream_t stream) {
  const long long n_seq = n / seq_len;
  if (n_seq <= 0) return cudaSuccess;
  LaunchTimer timer("seq_lens_kernel", stream);
  seq_lens_kernel<<<static_cast<int>(std::min<long long>(n_seq, 4096)), 256, 0, stream>>>(
      mask, n, seq_len, lens, n_nonempty);
  return cudaGetLastError();
}

// Copies the rows of h of every row block of one chunk whose segments are not
// consecutive rows (a block that spans the end of a completion) into the
// chunk's copy of h, at the block's local rows li * BM, with zeros for rows
// past the active list or past N; the GEMMs then read every block in one TMA
// box (a block of consecutive rows from h itself). One CTA per segment (16
// rows) of each row block of the chunk's host-side bound; those of blocks of
// consecutive rows return at once.
__global__ void __launch_bounds__(256) gather_blocks_kernel(const __nv_bfloat16* __restrict__ h,
                                                            __nv_bfloat16* __restrict__ out,
                                                            const TileArgs a) {
  const int li = static_cast<int>(blockIdx.x);
  const int j = static_cast<int>(blockIdx.y);  // segment of the block
  if (li >= launch_row_blocks(a)) return;
  int rows[kSegs];
  if (h_rows(a, li, rows)) return;
  const int vecs = a.hidden / 8;  // 16-byte vectors per row (hidden % 8 == 0)
  uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<long long>(li) * BM + j * SEG) *
                                                  a.hidden);
  for (int r = 0; r < SEG; ++r) {
    const long long src = static_cast<long long>(rows[j]) + r;
    const uint4* s = reinterpret_cast<const uint4*>(h + src * a.hidden);
    for (int v = threadIdx.x; v < vecs; v += blockDim.x)
      dst[r * vecs + v] = src < a.n_total ? s[v] : make_uint4(0u, 0u, 0u, 0u);
  }
}

cudaError_t launch_gather_blocks(const void* h, void* out, const TileArgs& args,
                                 cudaStream_t stream) {
  if (args.n_rb <= 0 || args.seg_list == nullptr) return cudaSuccess;
  LaunchTimer timer("gather_blocks_kernel", stream);
  gather_blocks_kernel<<<dim3(args.n_rb, kSegs), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(h), static_cast<__nv_bfloat16*>(out), args);
  return cudaGetLastError();
}

cudaError_t launch_row_plan(const uint8_t* mask, long long n, int n_segs, int* seg_list,
                            int* n_seg, double* msum, cudaStream_t stream) {
  LaunchTimer timer("row_plan_kernel", stream);
  row_plan_kernel<<<1, 1024, 0, stream>>>(mask, n, n_segs, seg_list, n_seg, msum);
  return cudaGetLastError();
}

cudaError_t launch_zero_padding_blocks(const uint8_t* mask, long long n, int n_rb, int hidden,
                                       void* dH, int sms, cudaStream_t stream) {
  if (mask == nullptr || n_rb <= 0) return cudaSuccess;
  const int grid = std::min(n_rb, 4 * std::max(sms, 1));
  LaunchTimer timer("zero_padding_blocks_kernel", stream);
  zero_padding_blocks_kernel<<<grid, 256, 0, stream>>>(mask, n, n_rb, hidden,
                                                       static_cast<__nv_bfloat16*>(dH));
  return cudaGetLastError();
}

cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t stream) {
  long long blocks = (a.n + kFinalizeThreads - 1) / kFinalizeThreads;
  if (blocks < 1) blocks = 1;
  if (blocks > kMaxFinalizeBlocks) blocks = kMaxFinalizeBlocks;
  LaunchTimer timer("finalize_kernel", stream);
  finalize_kernel<<<static_cast<int>(blocks), kFinalizeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace grpo

// ---------------------------------------------------------------------------
// Stored-logit backward: per chunk, the forward GEMM also keeps the chunk's
// logits in fp16; this kernel finishes each row (log-sum-exp, logp, token
// loss, g) and rewrites the row in place as the bf16 G row that the dH GEMM
// consumes: G_v = g (onehot_v(y) - exp(z'_v - lse)) f'(z_v). One CTA per row.
namespace grpo {

cudaError_t launch_fwds_gemm(int ctas, const CUtensorMap& map_a, const CUtensorMap& map_b,
                            const CUtensorMap& map_h16,
                             const CUtensorMap& map_s, const TileArgs& args, int grid,
                             cudaStream_t stream,
                             const CUtensorMap* map_hc) {
  return ctas == 2 ? launch_gemm_variant<MODE_FWDS, 2>(map_a, map_b, args, grid, stream, &map_s, &map_h16, map_hc)
                   : launch_gemm_variant<MODE_FWDS, 1>(map_a, map_b, args, grid, stream, nullptr, &map_h16, map_hc);
}

cudaError_t prepare_fwds_gemm() {
  cudaError_t e = prepare_gemm_variant<MODE_FWDS, 1>();
  return e == cudaSuccess ? prepare_gemm_variant<MODE_FWDS, 2>() : e;
}

__device__ __forceinline__ float half_bits_to_float(uint32_t h16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h16)));
}

// Per-row finish of a stored-logit chunk: combines the forward's split
// partials into lse, writes logp and the weighted token loss, and returns
// g = dL/dlogp (0 for rows that do not count), lse and the target id (-1 when
// the row does not count or its id is out of range).
__device__ __forceinline__ void finish_row(const GformArgs& a, long long grow, float& lse,
                                           float& g, int& y) {
  g = 0.f;
  lse = 0.f;
  y = -1;
  const bool counted = grow < a.n_total && (a.mask == nullptr || a.mask[grow] != 0);
  if (!counted) return;
  float m2 = -INFINITY;
  for (int s = 0; s < a.splits; ++s) m2 = fmaxf(m2, a.part_m[s * a.part_ld + grow]);
  float ssum = 0.f;
  for (int s = 0; s < a.splits; ++s)
    ssum += a.part_s[s * a.part_ld + grow] * exp2f(a.part_m[s * a.part_ld + grow] - m2);
  lse = (m2 + log2f(ssum)) * 0.69314718055994531f;
  if (!isfinite(lse)) atomicCAS(a.status, 0, GRPO_ERR_NONFINITE);
  y = a.ids[grow];
  float logp;
  if (y < 0 || y >= a.vocab) {
    atomicCAS(a.status, 0, GRPO_ERR_BAD_TOKEN_ID);
    logp = __int_as_float(0x7fc00000);
    y = -1;
  } else {
    logp = a.zy[grow] - lse;
  }
  const double wt = token_weight(a.seq_mode, a.loss_den, a.msum, a.seq_lens, a.n_nonempty,
                                 grow, a.seq_len);
  const double lp = logp;
  const double A = a.adv[grow / a.seq_len];
  const double r = exp(lp - static_cast<double>(a.old_logp[grow]));
  const double lo = 1.0 - static_cast<double>(a.eps_low);
  const double hi = 1.0 + static_cast<double>(a.eps_high);
  const double c = fmin(fmax(r, lo), hi);
  const double surr = fmin(r * A, c * A);
  const double d = static_cast<double>(a.ref_logp[grow]) - lp;
  const double ed = exp(d);
  a.lt[grow] = (-surr + static_cast<double>(a.beta) * (ed - d - 1.0)) * wt;
  const bool clipped = (A > 0.0 && r > hi) || (A < 0.0 && r < lo);
  const double dl = -(clipped ? 0.0 : A * r) + static_cast<double>(a.beta) * (1.0 - ed);
  g = static_cast<float>(dl * wt);
  if (a.logp_out) a.logp_out[grow] = logp;
}

// Row blocks of the chunk that the GEMMs compute (the active list may be
// shorter than the host-side bound).
__device__ __forceinline__ int chunk_blocks(const GformArgs& a) {
  if (a.n_seg == nullptr) return a.n_rb;
  const int segs = *a.n_seg - a.rb_offset * kSegs;
  return max(0, min(a.n_rb, (segs + kSegs - 1) / kSegs));
}

// Global row of local row `lrow` of the chunk, or -1 past the active list
// (inside the chunk's last computed block, or past it).
__device__ __forceinline__ long long chunk_row(const GformArgs& a, int lrow) {
  if (lrow / BM >= chunk_blocks(a)) return -1;
  if (a.seg_list == nullptr) return static_cast<long long>(a.rb_offset) * BM + lrow;
  const int s = a.rb_offset * kSegs + lrow / SEG;
  if (a.n_seg != nullptr && s >= *a.n_seg) return -1;
  return static_cast<long long>(a.seg_list[s]) * SEG + lrow % SEG;
}

__global__ void __launch_bounds__(kGformThreads) finalize_gform_kernel(const GformArgs a) {
  __shared__ float sh_lse2, sh_g;
  __shared__ int sh_y;
  const int lrow = blockIdx.x;
  const long long grow = chunk_row(a, lrow);
  uint4* row = reinterpret_cast<uint4*>(a.S + static_cast<long long>(lrow) * a.ldS);
  const int n_vec = static_cast<int>(a.ldS / 8);
  if (grow < 0) {
    // Past the active list. In the chunk's last computed block the row is
    // zeroed, so that the dW GEMM, which sums over the block's rows, reads no
    // stale bytes; past it no GEMM reads the row.
    if (lrow / BM < chunk_blocks(a))
      for (int i = threadIdx.x; i < n_vec; i += blockDim.x) row[i] = make_uint4(0, 0, 0, 0);
    return;  // whole block: uniform
  }

  if (threadIdx.x == 0) {
    float lse, g;
    int y;
    finish_row(a, grow, lse, g, y);
    sh_lse2 = lse * kLog2e;
    sh_g = g;
    sh_y = y;
  }
  __syncthreads();
  const float lse2 = sh_lse2, g = sh_g;
  const int y = sh_y;
  if (g == 0.f) {
    for (int i = threadIdx.x; i < n_vec; i += blockDim.x) row[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  // Stored value of column v: z'_v log2e - m_b, m_b the maximum of its
  // 64-column box b = v / 64 times log2 e (vector i of 8 columns lies in box
  // i / 8), as kept beside the block.
  const float* bm = a.box_max + lrow;
  auto box_max = [&](int i) { return __ldg(bm + static_cast<long long>(i >> 3) * a.ldM); };
  if (a.xmode == 0) {
    // Without a transform: -g 2^(z log2e - lse2) = -sign(g) 2^(z log2e + log2|g| - lse2),
    // one add and one exponential per logit and the sign set on each packed
    // pair; the target column and the padding past the vocabulary are fixed
    // up afterwards.
    const float c = log2f(fabsf(g)) - lse2;
    const uint32_t sgn = g > 0.f ? 0x80008000u : 0u;
    auto fast = [&](const uint4 in, float mb) {
      const float cb = mb + c;
      const uint32_t w[4] = {in.x, in.y, in.z, in.w};
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float t0, t1;
        add_f16x2_f32(w[k], cb, t0, t1);
        o[k] = pack_bf16x2(ex2(t0), ex2(t1)) ^ sgn;
      }
      return make_uint4(o[0], o[1], o[2], o[3]);
    };
    const int step = 2 * blockDim.x;
    int i = threadIdx.x;
    for (; i + blockDim.x < n_vec; i += step) {
      const uint4 in0 = row[i];
      const uint4 in1 = row[i + blockDim.x];
      const float m0 = box_max(i), m1 = box_max(i + blockDim.x);
      row[i] = fast(in0, m0);
      row[i + blockDim.x] = fast(in1, m1);
    }
    if (i < n_vec) row[i] = fast(row[i], box_max(i));
    __syncthreads();  // the whole row is written before the fix-ups
    uint16_t* row16 = a.S + static_cast<long long>(lrow) * a.ldS;
    if (threadIdx.x == 0 && y >= 0) {
      // Target column: g (1 - p_y), from the forward's fp32 target logit.
      const float val = g - g * ex2(fmaf(a.zy[grow], kLog2e, -lse2));
      row16[y] = static_cast<uint16_t>(pack_bf16x2(val, 0.f) & 0xffffu);
    }
    if (threadIdx.x < a.ldS - a.vocab) row16[a.vocab + threadIdx.x] = 0;
    return;
  }
  const float ng = -g;
  // G_v from the stored z'_v: g (onehot_v(y) - exp(z'_v - lse)) f'(z_v).
  auto convert = [&](const uint4 in, int i) {
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    const float mb = i * 8 < a.vocab ? box_max(i) : 0.f;
    const float cb = mb - lse2;
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float gv[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int v = i * 8 + k * 2 + h;
        const float sv = half_bits_to_float(h == 0 ? (w[k] & 0xffffu) : (w[k] >> 16));
        const float z = (sv + mb) * kLn2;
        float d = 1.f;  // dz'/dz recovered from the stored z'
        if (a.xmode == 1) {
          d = a.k0;
        } else if (a.xmode == 2) {
          const float u = z / a.k2;
          d = a.k0 * fmaf(-u, u, 1.f);
        }
        float val = ng * ex2(sv + cb);
        if (v == y) val += g;
        gv[h] = v < a.vocab ? val * d : 0.f;
      }
      o[k] = pack_bf16x2(gv[0], gv[1]);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  };
  // Two 16-byte vectors per thread per step keep more loads in flight.
  const int step = 2 * blockDim.x;
  int i = threadIdx.x;
  for (; i + blockDim.x < n_vec; i += step) {
    const uint4 in0 = row[i];
    const uint4 in1 = row[i + blockDim.x];
    row[i] = convert(in0, i);
    row[i + blockDim.x] = convert(in1, i + blockDim.x);
  }
  if (i < n_vec) row[i] = convert(row[i], i);
}

// Closing reduction of a stored-logit call: masked rows get logp = 0, and the
// token losses of unmasked rows are summed in a fixed order (fp64).
__global__ void __launch_bounds__(kFinalizeThreads) finish_loss_kernel(const FinishArgs a) {
  __shared__ double sh[32];
  __shared__ bool is_last;
  double local = 0.0;
  // After a wait that ran out anywhere in the call, logp and the loss are NaN.
  const bool aborted = *reinterpret_cast<const volatile int*>(a.status) == GRPO_ERR_DEVICE_TIMEOUT;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < a.n;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const bool counted = a.mask == nullptr || a.mask[t] != 0;
    if (aborted) {
      if (a.logp_out) a.logp_out[t] = __int_as_float(0x7fc00000);
    } else if (counted) {
      local += a.lt[t];
    } else if (a.logp_out) {
      a.logp_out[t] = 0.f;
    }
  }
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
      *a.loss_out = aborted ? __int_as_float(0x7fc00000) : static_cast<float>(tot);
      *a.counter = 0;
    }
  }
}

cudaError_t launch_finalize_gform(const GformArgs& a, int rows, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  LaunchTimer timer("finalize_gform_kernel", stream);
  finalize_gform_kernel<<<rows, kGformThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

// The row values alone (one thread per row of the chunk), for the dH GEMM
// that turns the stored logits into G itself.
__global__ void __launch_bounds__(kFinalizeThreads) finalize_rows_kernel(const GformArgs a,
                                                                         int rows) {
  const int lrow = blockIdx.x * blockDim.x + threadIdx.x;
  if (lrow >= rows) return;
  const long long grow = chunk_row(a, lrow);
  if (grow < 0) return;
  float lse, g;
  int y;
  finish_row(a, grow, lse, g, y);
  a.lse_out[grow] = lse;
  a.g_out[grow] = g;
}

// Single pass at hidden sizes above 2048: one vocabulary block of a chunk's
// stored logits rewritten in place as the bf16
//   P_v = 2^(z'_v log2e - M) f'(S_v),
// M the row's running maximum (log2 units) over the forward's split partials
// of the blocks so far (slots [0, splits)); the target column and rows that do
// not count become zeros. The U GEMM then reads P through TMA, so each logit
// is converted once rather than once per hidden tile. Columns past the
// block's width are never read (the U GEMM's tensor map ends there). One CTA
// per row.
__global__ void __launch_bounds__(kGformThreads) single_pass_p_kernel(const GformArgs a) {
  __shared__ float sh_m2;
  __shared__ int sh_y, sh_on;
  const int lrow = blockIdx.x;
  const long long grow = chunk_row(a, lrow);
  if (grow < 0) return;  // whole block: uniform
  if (threadIdx.x == 0) {
    const bool on = grow < a.n_total && (a.mask == nullptr || a.mask[grow] != 0);
    float m2 = -INFINITY;
    int y = -1;
    if (on) {
      for (int s = 0; s < a.splits; ++s) m2 = fmaxf(m2, a.part_m[s * a.part_ld + grow]);
      const int yy = a.ids[grow];
      if (yy >= a.v0 && yy < a.v0 + a.width) y = yy - a.v0;
    }
    sh_m2 = m2;
    sh_y = y;
    sh_on = on ? 1 : 0;
  }
  __syncthreads();
  uint4* row = reinterpret_cast<uint4*>(a.S + static_cast<long long>(lrow) * a.ldS);
  const int n_vec = static_cast<int>(a.ldS / 8);
  if (!sh_on) {
    for (int i = threadIdx.x; i < n_vec; i += blockDim.x) row[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  const float m2 = sh_m2;
  const float* bm = a.box_max + lrow;
  auto box_max = [&](int i) { return __ldg(bm + static_cast<long long>(i >> 3) * a.ldM); };
  auto convert = [&](const uint4 in, int i) {
    const float mb = box_max(i);
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t o[4];
    const float c = mb - m2;
    if (a.xmode == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float t0, t1;
        add_f16x2_f32(w[k], c, t0, t1);
        o[k] = pack_bf16x2(ex2(t0), ex2(t1));
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float s0, s1;
        unpack_f16x2(w[k], s0, s1);
        const float z0 = (s0 + mb) * kLn2, z1 = (s1 + mb) * kLn2;
        float d0 = 1.f, d1 = 1.f;  // dz'/dz recovered from the stored z'
        if (a.xmode == 1) {
          d0 = d1 = a.k0;
        } else {
          const float u0 = z0 / a.k2, u1 = z1 / a.k2;
          d0 = a.k0 * fmaf(-u0, u0, 1.f);
          d1 = a.k0 * fmaf(-u1, u1, 1.f);
        }
        o[k] = pack_bf16x2(ex2(s0 + c) * d0, ex2(s1 + c) * d1);
      }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  };
  // Two 16-byte vectors per thread per step keep more loads in flight.
  const int step = 2 * blockDim.x;
  int i = threadIdx.x;
  for (; i + blockDim.x < n_vec; i += step) {
    const uint4 in0 = row[i];
    const uint4 in1 = row[i + blockDim.x];
    row[i] = convert(in0, i);
    row[i + blockDim.x] = convert(in1, i + blockDim.x);
  }
  if (i < n_vec) row[i] = convert(row[i], i);
  __syncthreads();  // the whole row is written before the target column is cleared
  if (threadIdx.x == 0 && sh_y >= 0) a.S[static_cast<long long>(lrow) * a.ldS + sh_y] = 0;
}

cudaError_t launch_single_pass_p(const GformArgs& a, int rows, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  LaunchTimer timer("single_pass_p_kernel", stream);
  single_pass_p_kernel<<<rows, kGformThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_finalize_rows(const GformArgs& a, int rows, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  LaunchTimer timer("finalize_rows_kernel", stream);
  finalize_rows_kernel<<<(rows + kFinalizeThreads - 1) / kFinalizeThreads, kFinalizeThreads, 0,
                         stream>>>(a, rows);
  return cudaGetLastError();
}

cudaError_t launch_finish_loss(const FinishArgs& a, cudaStream_t stream) {
  long long blocks = (a.n + kFinalizeThreads - 1) / kFinalizeThreads;
  blocks = std::max(1LL, std::min<long long>(blocks, kMaxFinalizeBlocks));
  LaunchTimer timer("finish_loss_kernel", stream);
  finish_loss_kernel<<<static_cast<int>(blocks), kFinalizeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace grpo

// ---------------------------------------------------------------------------
// Self-test of the bounded waits: one thread waits, with the same routine the
// GEMM roles use, on an mbarrier that nothing ever arrives on. The wait must
// run out, record GRPO_ERR_DEVICE_TIMEOUT in the status word and return; the
// kernel then exits normally and the context stays usable.
namespace grpo {

__global__ void bounded_wait_selftest_kernel(int* status, int* waited_out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_sh;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait(&bar, 0, &abort_sh, status);  // phase 0 never completes
    *waited_out = ok ? 0 : 1;
  }
}

cudaError_t launch_bounded_wait_selftest(int* status, int* waited_out, cudaStream_t stream) {
  LaunchTimer timer("bounded_wait_selftest_kernel", stream);
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(status, waited_out);
  return cudaGetLastError();
}

}  // namespace grpo
