/*
 * grpo_gb300.h - C ABI of the GB300 (sm_103a) selective log-prob / GRPO loss
 * library.
 *
 * What it computes (the web pages this library restates are cited by title
 * and section):
 *
 *   logp_t = h_t . W[y_t] - logsumexp_v(h_t . W_v)
 *
 * straight from the final hidden states h [N, D] and the lm_head weight
 * W [V, D], without ever holding the N x V logits ("GRPO with 7x longer
 * context", Unsloth docs, section "Flattened sequence length chunking" and
 * its chunked_hidden_states_selective_log_softmax call). On top of it, the
 * masked token-mean GRPO loss with a clipped importance ratio against the
 * old policy and a beta-weighted k3 reverse-KL term against the reference
 * policy ("Unsloth internals", section "The relationship to TRL"; "Train
 * reasoning models with 5GB VRAM", section "Under the Hood"), and its
 * gradient to the hidden states, obtained either by recomputing the logit
 * tiles as the pages' backward does (same Unsloth docs page, section
 * "Offloading activations for log-softmax") or from each chunk's logits kept
 * in fp16, which saves that second logit GEMM.
 *
 * Conventions shared by every entry point:
 *   - All tensor arguments are DEVICE pointers on the current CUDA device,
 *     row-major and densely packed, 16-byte aligned:
 *       hidden  bf16  [N, D]       W     bf16 [V, D]
 *       ids     int32 [N]          mask  uint8 [N] (nonzero = token counts)
 *       old_logp, ref_logp fp32 [N]
 *       adv     fp32  [N / T]      (advantage of completion b = t / T)
 *   - The caller owns every buffer, including the workspace; the library
 *     allocates no device memory. Calls are asynchronous on `stream`
 *     (a cudaStream_t; NULL = the legacy default stream).
 *   - Return value: GRPO_OK (0) or a negative grpo_status. Argument checks
 *     happen on the host before anything is launched; problems found on the
 *     device (out-of-range token ids, a non-finite log-sum-exp, a timed-out
 *     wait) are recorded in the workspace's status word, read back with
 *     grpo_read_device_status. After a timed-out wait the call's logp, lse
 *     and loss are NaN, and its dH (and dW) are undefined.
 *   - Two calls that share a workspace must not overlap on the GPU. Calls
 *     with separate workspaces may run concurrently from several host
 *     threads; the stored-logit path's side stream (one per device, created
 *     on first use together with a few events; no device memory) is then
 *     shared, which orders their row-wise G passes one after another.
 *   - Requires an sm_103 device (GB300).
 */
#ifndef GRPO_GB300_H_
#define GRPO_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum grpo_status {
  GRPO_OK = 0,
  GRPO_ERR_INVALID_ARG = -1,       /* null pointer, negative size, bad param  */
  GRPO_ERR_MISALIGNED = -2,        /* a pointer is not 16-byte aligned        */
  GRPO_ERR_UNSUPPORTED_SHAPE = -3, /* D % 8 != 0, N % T != 0, size too large  */
  GRPO_ERR_WORKSPACE_TOO_SMALL = -4,
  GRPO_ERR_UNSUPPORTED_DEVICE = -5, /* not an sm_103 GPU                      */
  GRPO_ERR_CUDA = -6,               /* a CUDA runtime/driver call failed      */
  GRPO_ERR_DEVICE_TIMEOUT = -7,     /* (device) a bounded wait ran out        */
  GRPO_ERR_BAD_TOKEN_ID = -8,       /* (device) unmasked id outside [0, V)   */
  GRPO_ERR_NONFINITE = -9           /* (device) a row's log-sum-exp is inf or
                                       NaN: the inputs hold inf/NaN or logits
                                       beyond the fp32 range                 */
} grpo_status;

typedef struct grpo_shape {
  int64_t n_tokens; /* N = B * T flattened tokens (rows of hidden)           */
  int32_t seq_len;  /* T: tokens per completion; row t is completion t / T    */
  int32_t hidden;   /* D: hidden size, a multiple of 8                        */
  int32_t vocab;    /* V: vocabulary size (rows of W)                         */
  int32_t reserved; /* must be 0                                              */
} grpo_shape;

/* The backward form. Three exist; without any of the three flags below the
 * call chooses (the default):
 *   - stored logits (GRPO_FLAG_STORED_LOGITS): 4 N D V flops, a workspace
 *     of chunk x V x 2 bytes (and twice that at D > 2048, see below);
 *   - single pass (GRPO_FLAG_SINGLE_PASS): 4 N D V flops, a workspace of
 *     one or two blocks of chunk x vocab_block x 2 bytes plus a chunk x D
 *     fp32 accumulator;
 *   - recomputed logit tiles (GRPO_FLAG_RECOMPUTE_LOGITS): 6 N D V flops
 *     (the pages' backward, which re-runs the forward), a workspace of
 *     chunk x vocab_block x 2 bytes plus a chunk x D fp32 accumulator.
 * The automatic choice is, among the forms that fit the workspace budget
 * (workspace_limit_bytes, or half the free device memory with
 * GRPO_FLAG_FIT_FREE_MEMORY; none by default), the one whose modelled GEMM
 * time is shortest (whole SM waves of each launch, the part of a separate G or
 * P pass the neighbouring GEMMs cannot hide, the cost of forming P on chip,
 * with factors measured on GB300). It is made
 * at GB300's SM count, so that grpo_workspace_size and the call agree;
 * grpo_get_plan reports it. Setting more than one of the three flags is
 * GRPO_ERR_INVALID_ARG.
 *
 * Tail split (stored form; single pass with P formed on chip): when the last
 * round of a dH-type GEMM launch has fewer units (256 rows x 512 hidden
 * columns) than the device has SM pairs, and no G or P pass runs beside it,
 * idle pairs take over the tails of that round's vocabulary loops, and a fixup
 * pass adds each cut unit's pieces in a fixed order (results do not depend on
 * timing). Its fp32 partial tiles take a fixed 76 MiB of the workspace (38 MiB
 * with GRPO_FLAG_SINGLE_CTA) when the K loop has at least 8129 columns (the
 * vocabulary, or the single pass's block), and none under a workspace budget
 * below 8 times that.
 *
 * grpo_params.flags bit: backward without a second logit GEMM. Per chunk of
 * rows, the forward GEMM also keeps the chunk's (transformed) logits in fp16
 * in the workspace, and the dH GEMM runs over the whole vocabulary once lse
 * and g are known. Each 64-column box of a row is stored relative to its own
 * maximum, in log2 units (z log2 e - m, with m = max log2 e kept beside it in
 * fp32), so any finite logit is stored without overflow, the box's largest
 * terms keep fp16's finest spacing, and every exponential of G takes the
 * stored value plus fp32 constants. The logits
 * are turned into G in one of two ways:
 *   - D <= 2048 without dW: the dH GEMM converts each landed tile on chip.
 *     One block of chunk x V x 2 bytes (capped at 4 GiB) serves every chunk.
 *   - otherwise: a row-wise pass rewrites the block in place, beside the next
 *     chunk's GEMMs. Two blocks when there is more than one chunk (each capped
 *     at 2 GiB).
 * Executes 4 N D V instead of 6 N D V flops; vocab_block is ignored. */
#define GRPO_FLAG_STORED_LOGITS 1u

/* grpo_params.flags bit: run every GEMM as one CTA per 128-row tile instead
 * of the default CTA pair per 256-row tile (tcgen05 cta_group::2). Same
 * results up to fp32 summation order; kept for comparison and debugging. */
#define GRPO_FLAG_SINGLE_CTA 2u

/* grpo_params.flags bit: loss = mean over completions of each completion's
 * masked token mean, L = (1/B') sum_b (1/len_b) sum_{t in b} m_t l_t, with
 * len_b the unmasked tokens of completion b (b = t / seq_len) and B' the
 * completions with len_b > 0 (loss_denominator > 0 replaces B'). Without the
 * flag: token mean over the batch. */
#define GRPO_FLAG_SEQUENCE_MEAN 4u

/* grpo_params.flags bit: size the chunk from the current device's free memory
 * (budget = half of what cudaMemGetInfo reports, or workspace_limit_bytes if
 * smaller) - the pages' "adjust to the available VRAM". With this flag
 * grpo_workspace_size queries the current device (no allocation, no launch). */
#define GRPO_FLAG_FIT_FREE_MEMORY 8u

/* grpo_params.flags bit: the backward recomputes the logit tiles chunk by
 * chunk and vocab block by vocab block (G = g (onehot - softmax) formed in
 * the GEMM's epilogue, then dH += G W[block]): the smallest workspace. */
#define GRPO_FLAG_RECOMPUTE_LOGITS 16u

/* grpo_params.flags bit: the single-pass backward. Per chunk of rows and per
 * vocabulary block of vocab_block columns (automatic: blocks of about 32768,
 * at most 32 of them), one logit GEMM keeps the block's logits in fp16
 * (box-shifted as above); they become P_v = exp(z'_v - M) f'(S_v), M the
 * row's running maximum, the target column left out (on chip in the next
 * GEMM; or, at D > 2048 when the planner models it faster within the budget,
 * by a row-wise pass beside the next block's logit GEMM, on a second block),
 * and one GEMM adds P W[block] into an fp32
 * accumulator U, rescaled whenever the maximum grows. After the last block,
 * dH = g (1 - p_y) f'_y W[y] - g exp(M - lse) U. Each logit is computed once
 * (4 N D V flops, like the stored form), while the workspace holds one or two
 * blocks of chunk x vocab_block x 2 bytes plus the chunk x D fp32
 * accumulator. With dW requested the call recomputes the logit tiles instead
 * (same chunk and vocab block). */
#define GRPO_FLAG_SINGLE_PASS 32u

typedef struct grpo_params {
  float eps_low;          /* ratio clip: lower bound 1 - eps_low (0.2)         */
  float eps_high;         /* ratio clip: upper bound 1 + eps_high (0.2)        */
  float beta;             /* weight of the k3 KL term (0.001)                  */
  float loss_denominator; /* <= 0: divide by sum(mask); > 0: divide by this    */
  int32_t chunk_tokens;   /* rows per backward chunk; 0 = automatic            */
  int32_t vocab_block;    /* vocab columns per backward block; 0 = automatic   */
  uint32_t flags;         /* GRPO_FLAG_* bits, or 0                           */
  int32_t raster_rows;    /* row units per raster group of the persistent GEMM
                             grids (a tuning knob; 0 = automatic)             */
  /* Logit transforms ("GRPO with 7x longer context", the options of the
   * selective log-softmax call: logit scale multiply/divide, softcapping,
   * temperature), applied to the raw logit z in that order:
   *   z' = s(z * logit_scale_multiply / logit_scale_divide) / temperature,
   *   s(x) = logit_softcapping * tanh(x / logit_softcapping)  (x when 0).
   * logp and the loss use z'; dH carries dz'/dz. 0 in any field = unused. */
  float logit_scale_multiply;
  float logit_scale_divide;
  float logit_softcapping;
  float temperature;
  /* Upper bound on the workspace in bytes (0 = none). The automatic chunk is
   * the largest that keeps the whole workspace within it; an explicit
   * chunk_tokens over the budget, or a budget below the chunk-independent
   * part, gives GRPO_ERR_WORKSPACE_TOO_SMALL. */
  uint64_t workspace_limit_bytes;
} grpo_params;

/* Defaults: eps 0.2/0.2, beta 0.001 (the pages' corrected GRPO default,
 * "How does Unsloth implement GRPO", section "Corrected hyperparameters"),
 * token-mean denominator, automatic chunking and backward form, no workspace
 * budget, no logit transform. Host only. */
void grpo_default_params(grpo_params* params);

/* Bytes of device workspace that grpo_loss_fwd_bwd needs for this shape and
 * these params (enough for grpo_logp_fwd too, which needs only the part that
 * does not depend on the chunking). Host only, touches no GPU (except with
 * GRPO_FLAG_FIT_FREE_MEMORY, which reads the free memory). The size grows
 * with N (a few fp32 per token) and with the chunk (chunk x V for the stored
 * form, chunk x vocab_block otherwise, and chunk x D for a copy of the rows
 * of h whose 16-row segments of active rows do not form consecutive rows),
 * never with N x V: the point of
 * "GRPO with 7x longer context", section "Flattened sequence length
 * chunking", Eq. 1-3, where the logit memory follows the chunk, not the
 * batch. Returns GRPO_OK or GRPO_ERR_INVALID_ARG / _UNSUPPORTED_SHAPE /
 * _WORKSPACE_TOO_SMALL (a budget below what any plan needs). */
int grpo_workspace_size(const grpo_shape* shape, const grpo_params* params, size_t* bytes);

/* Selective log-softmax ("GRPO with 7x longer context", section "Flattened
 * sequence length chunking"):
 *   logp[t] = h_t . W[ids[t]] - lse[t],  lse[t] = logsumexp_v h_t . W_v,
 * for every t in [0, N). logits are accumulated and reduced in fp32.
 *   logp:        fp32 [N] output (required)
 *   lse_or_null: fp32 [N] output, or NULL
 * params: the chunk/vocab and logit-transform fields are read (NULL = defaults).
 * ids outside [0, V) give logp = NaN and GRPO_ERR_BAD_TOKEN_ID in the device
 * status word. */
int grpo_logp_fwd(const void* hidden, const void* W, const int32_t* ids, float* logp,
                  float* lse_or_null, const grpo_shape* shape, const grpo_params* params,
                  void* workspace, size_t workspace_bytes, void* stream);

/* Fused GRPO loss forward + backward to the hidden states.
 *   r_t   = exp(logp_t - old_logp_t)
 *   surr  = min(r_t A_b, clamp(r_t, 1 - eps_low, 1 + eps_high) A_b)
 *   kl_t  = exp(ref_t - logp_t) - (ref_t - logp_t) - 1
 *   l_t   = -surr + beta kl_t
 *   loss  = sum_t mask_t l_t / M,  M = sum_t mask_t (or loss_denominator > 0);
 *           per-completion mean with GRPO_FLAG_SEQUENCE_MEAN
 *   dH_t  = dloss/dh_t = g_t (W[y_t] - sum_v softmax(h_t W^T)_v W_v),
 *           g_t = dloss/dlogp_t
 * ("Unsloth internals", section "The relationship to TRL"; "Train reasoning
 * models with 5GB VRAM", section "Under the Hood"; "GRPO with 7x longer
 * context", section "Offloading activations for log-softmax").
 *   loss:         fp32 [1] device scalar output (sum accumulated in fp64)
 *   logp_or_null: fp32 [N] output (0 on masked rows), or NULL
 *   dH:           bf16 [N, D] output; masked rows are exactly 0
 *   dW_or_null:   fp32 [V, D] output, the lm_head gradient
 *                 dW_v = sum_t g_t (onehot_v(y_t) - softmax_v) f'(z_tv) h_t
 *                 (overwritten, 16-byte aligned), or NULL when the head is
 *                 frozen (the LoRA case); costs one more GEMM of 2 N D V flops
 * M = 0 gives loss = 0 and dH = 0. Ids of masked rows are never read. */
int grpo_loss_fwd_bwd(const void* hidden, const void* W, const int32_t* ids,
                      const uint8_t* mask, const float* old_logp, const float* ref_logp,
                      const float* adv, float* loss, float* logp_or_null, void* dH,
                      float* dW_or_null, const grpo_shape* shape, const grpo_params* params,
                      void* workspace, size_t workspace_bytes, void* stream);

/* How a call with this shape and these params is carried out on the current
 * device (host only; reads the device's SM count, launches nothing): the
 * chunking whose memory the pages size by the chunk rather than the batch
 * ("GRPO with 7x longer context", section "Flattened sequence length
 * chunking", Eq. 1-3), and the backward form chosen for the budget. */
typedef struct grpo_plan_info {
  int32_t chunk_rows;        /* rows per backward chunk                      */
  int32_t vocab_block;       /* vocab columns per backward block             */
  int32_t n_chunks;          /* backward chunks                              */
  int32_t n_vocab_blocks;    /* backward vocab blocks per chunk              */
  int32_t fwd_splits;        /* forward vocab splits (partials per row) when
                                every row is active: of the loss call's
                                logit GEMMs in the stored and recomputed
                                forms, else of grpo_logp_fwd's one logit
                                GEMM (with masked rows the kernels set them
                                from the active rows, at most 32)          */
  int32_t launches_logp;     /* kernel launches of one grpo_logp_fwd call    */
  int32_t launches_loss;     /* kernel launches of one grpo_loss_fwd_bwd
                                with a mask (without one: one fewer, and
                                no fixup pass after a dH launch whose
                                units fill whole rounds of the SM pairs)  */
  int32_t g_in_dh_gemm;      /* 1: the stored-logit backward forms G (the
                                single pass P) inside the dH-type GEMM
                                (hidden <= 2048; not with dW); 0: in a
                                row-wise pass of its own beside the GEMMs  */
  int32_t stored_logits;     /* 1: the stored-logit backward              */
  int32_t single_pass;       /* 1: the single-pass backward (neither: the
                                recomputed logit tiles); the flags' or the
                                automatic choice                          */
  uint64_t workspace_bytes;  /* same as grpo_workspace_size                  */
} grpo_plan_info;

int grpo_get_plan(const grpo_shape* shape, const grpo_params* params, grpo_plan_info* info);

/* Synchronises `stream`, then copies the device status word of the last call
 * that used `workspace` into *device_status (GRPO_OK or a negative code). */
int grpo_read_device_status(const void* workspace, int* device_status, void* stream);

/* Workspace-free selective log-softmax. The pages have no counterpart to this
 * call: it exists for callers that cannot allocate device memory themselves,
 * for instance a plugin running inside a host framework that owns every byte
 * of device memory through its own pool and forbids side allocations, or a
 * latency-critical caller that cannot accept cudaMalloc's implicit device
 * synchronisation or its failure under memory pressure.
 *
 * Computes exactly what grpo_logp_fwd computes (same kernels, same results),
 * but its scratch lives in a file-scope device array of
 * GRPO_NOALLOC_SCRATCH_BYTES (2.25 MiB) inside the library instead of a
 * caller workspace. Every GPU on which the library's device code is loaded
 * holds that array until the process exits. The caller still passes the
 * inputs and the outputs (logp, optional lse) as device pointers.
 *   - n_tokens is limited to GRPO_NOALLOC_MAX_TOKENS (8192); larger sizes
 *     return GRPO_ERR_UNSUPPORTED_SHAPE before anything is launched.
 *   - Allocates nothing: no cudaMalloc/cudaFree, no allocating library call.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins.
 *   - If a wait inside the call runs out (GRPO_ERR_DEVICE_TIMEOUT, which the
 *     workspace calls report in their status word), every logp and lse of
 *     the call is NaN: this call has no status word the caller can read.
 *   - All calls share the one array, which keeps the previous call's
 *     contents; each call clears the parts that must start at zero. Two calls
 *     that overlap on the GPU (different streams, no ordering between them)
 *     race on the array and give wrong results: order them, e.g. on one stream.
 *   - Out-of-range ids give logp = NaN; there is no caller-visible status word. */
#define GRPO_NOALLOC_MAX_TOKENS 8192
#define GRPO_NOALLOC_SCRATCH_BYTES 2359296
int grpo_logp_fwd_noalloc(const void* hidden, const void* W, const int32_t* ids, float* logp,
                          float* lse_or_null, const grpo_shape* shape, void* stream);

/* Self-test of the device-side failure detection. Launches one tiny kernel
 * that waits, with the same bounded wait every GEMM role uses, on an mbarrier
 * that nothing ever arrives on: after about one second the wait gives up,
 * records GRPO_ERR_DEVICE_TIMEOUT in the status word of `workspace` (>= 64
 * bytes, 256-byte aligned) and the kernel returns normally - no trap, no
 * hang, the context stays usable. Read the outcome with
 * grpo_read_device_status. Returns GRPO_OK if the launch went through. */
int grpo_selftest_bounded_wait(void* workspace, size_t workspace_bytes, void* stream);

/* Opt-in per-launch timing, for profiling without an external profiler.
 *
 * grpo_launch_timing_enable(1) turns it on for the calling host thread. While it
 * is on, every kernel launch that thread makes through this library is
 * bracketed by two CUDA events recorded on the launch's own stream. That stream
 * is the caller's stream or the library's side stream. An event pair measures
 * the kernel's device time, plus any idle gap on that stream between the two
 * records. Timing adds about two event records of host time per launch, and
 * nothing on the device.
 *   - Off is the default. grpo_launch_timing_enable(0) stops recording; launches
 *     already recorded stay readable.
 *   - Launches into a stream that is being captured into a CUDA graph are not
 *     timed.
 *   - At most 65536 launches are kept between reads; later ones are not timed.
 *
 * grpo_launch_timing_read first waits for the recorded launches to finish. It
 * then sums them per kernel, empties the record, and writes up to `capacity`
 * entries to `out` in order of first launch. `*count` is set to the number of
 * distinct kernels seen, which may exceed `capacity`; entries past `capacity`
 * are lost. Kernel names are the device functions', e.g. "finalize_gform_kernel".
 * GEMM variants are named "tc_gemm_kernel<mode, ctas>": mode 0 is the logit GEMM
 * of the forward pass, 1 forms G from recomputed logits, 2 is G W -> dH, 3 is
 * the logit GEMM that also stores fp16 logits, 4 is the lm_head gradient,
 * 5 is the dH GEMM that forms G from the stored logits, 6 is the single
 * pass's GEMM that forms P from one block's stored logits and accumulates U,
 * and 7 the same GEMM reading P formed by single_pass_p_kernel; ctas is 2
 * for a CTA pair. Returns GRPO_OK, GRPO_ERR_INVALID_ARG (count null, capacity < 0, or out
 * null with capacity > 0) or GRPO_ERR_CUDA (an event could not be read; the
 * other launches are still summed). */
typedef struct grpo_kernel_time {
  char name[40];      /* NUL-terminated kernel name                         */
  int32_t launches;   /* launches summed                                    */
  int32_t reserved;
  double total_ms;    /* summed device time between each launch's events    */
} grpo_kernel_time;

int grpo_launch_timing_enable(int on);
int grpo_launch_timing_read(grpo_kernel_time* out, int capacity, int* count);

/* Static text for a status code. */
const char* grpo_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GRPO_GB300_H_ */
