// Host side of the C ABI: argument checks, work planning, TMA descriptor
// encoding and the launch sequence of the forward and backward passes.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "grpo_gb300.h"
#include "launch.h"

namespace grpo {
namespace {

constexpr int kMaxSplits = 32;          // forward vocab splits (per-row partials)
constexpr int kMaxAutoChunkBlocks = 32;  // automatic backward chunk <= 4096 rows
constexpr int kAutoVocabBlock = 32768;   // automatic backward vocab block
constexpr int kMaxStoredChunkBlocks = 64;                   // stored-logit chunk bound
constexpr int kMaxSinglePassChunkBlocks = 64;               // single-pass chunk <= 8192 rows
constexpr size_t kMaxStoredChunkBytes = size_t(2) << 30;    // 2 GiB of fp16 logits
// Hidden sizes up to which the stored-logit backward forms G inside the dH
// GEMM (MODE_DHS) rather than in a pass of its own over the logit block.
// Measured on GB300: the separate pass costs about 1/D of the dH GEMM and
// mostly hides behind the next chunk's GEMMs; the in-GEMM conversion costs a
// roughly constant share of the dH GEMM (the exponential and conversions per
// logit on its converter warps, measured: not its shared-memory traffic). At
// D = 1536 fusing is 7-12 % faster per call, at D = 2880 and 4096 the
// overlapped separate pass is faster.
constexpr int kFusedMaxHidden = 2048;
constexpr int kSplitsTarget = 8;        // forward vocab splits per raster group
// SM count at which the automatic choice between the stored and the
// recomputed backward is modelled (GB300's): the same choice then holds for
// the sizing without a device and for the call's own plan.
constexpr int kRefSms = 152;
constexpr size_t kHeaderBytes = 16384;   // status, counters, loss partials
constexpr int kMaxDevices = 64;

// Workspace header layout.
constexpr size_t kOffStatus = 0;       // int
constexpr size_t kOffCounter = 4;      // unsigned
constexpr size_t kOffMsum = 8;         // double
constexpr size_t kOffActive = 16;      // int: length of the active row-block list
constexpr size_t kOffNonempty = 20;    // int: completions with any unmasked token
constexpr size_t kOffPartials = 64;    // double[kMaxFinalizeBlocks]
static_assert(kOffPartials + kMaxFinalizeBlocks * sizeof(double) <= kHeaderBytes, "header");

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// An NVTX range around one ABI call (host side: it brackets the enqueueing of
// the call's launches), so that profilers can attribute the kernels to it.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

// D columns per dH unit, in units of 256: the pair kernel covers 512 (two
// 256-column accumulators, TMEM's 512 columns).
int dh_accumulators(int ctas) { return ctas == 2 ? 2 : 1; }

// Hidden-dimension units of a dH-type launch.
int dh_tiles(int hidden, int ctas) {
  return static_cast<int>(cdiv(hidden, BN * dh_accumulators(ctas)));
}

// Backward forms (grpo_params.flags, or the automatic choice). The single pass
// comes in two placements of its P conversion: on chip in the U GEMM (one
// logit block), or a row-wise pass beside the next block's logit GEMM (two
// blocks; hidden sizes above kFusedMaxHidden only).
enum Form { kFormRecompute = 0, kFormStored = 1, kFormSinglePass = 2, kFormSinglePassPass = 3 };

struct Layout {
  int ctas;         // 2: CTA-pair GEMMs (default); 1: single-CTA GEMMs
  bool stored;      // stored-logit backward (GRPO_FLAG_STORED_LOGITS)
  bool single_pass; // single-pass backward (GRPO_FLAG_SINGLE_PASS)
  int nvb;          // single pass: vocab blocks (each one logit GEMM + one U GEMM)
  long long ldS;    // stored mode: elements per row of the chunk logit block
  long long n, nr;  // rows, rows rounded up to BM
  int T, D, V;
  int nvt;          // vocab tiles (256 columns)
  int chunk_rows;   // backward chunk (multiple of BM)
  int n_sbuf;       // stored path: logit blocks (2 = double-buffered chunks)
  bool fused;       // stored path, D <= kFusedMaxHidden: G formed inside the dH
                    // GEMM, one logit block (the dW variant then runs unoverlapped)
  int vblock;       // backward vocab block (multiple of BN)
  bool need_acc;    // more than one vocab block -> fp32 dH accumulator
  double model_cost;  // modelled GEMM time of the plan in forward-tile times (0: no device)
  int nbox;         // stored path: 64-column boxes per row (their maxima are kept)
  int ts_slots;     // stored path: pairs of the tail-split dH launches (0: no split)
  int n_hc;         // chunk copies of h (the rows of non-consecutive row blocks): 1
  size_t off_pm, off_ps, off_zy, off_lse, off_g, off_rbl, off_lt, off_seq, off_sk, off_G,
      off_bmax, off_acc, off_hc, total;
};

// Tail split (see TailSplit in gemm_tc.cuh): a dH-type launch whose last round
// has fewer units than SM pairs splits that round's units between their own
// pairs and idle ones, when its K loop (the vocabulary, or the single pass's
// vocabulary block) is long enough to cut and nothing runs beside it. The
// stored form and the single pass with P formed on chip reserve its slots. The
// pairs are the device's, at most kRefSms / ctas, so that the slot region of
// the sizing without a device holds. The chunk planner models whole rounds all
// the same: the split only makes a launch's last round shorter.
int tail_split_slots(int k_cols, int ctas, int sms) {
  if (cdiv(k_cols, BK) < 2 * kTailMinStages) return 0;
  return std::min(sms > 0 ? sms : kRefSms, kRefSms) / ctas;
}

// Bytes of the tail split's partial slots: two fp32 tiles of a unit per pair.
size_t tail_split_bytes(int ts_slots, int ctas) {
  return static_cast<size_t>(2) * ts_slots * ctas * BM * (BN * dh_accumulators(ctas)) *
         sizeof(float);
}

// Stored-logit backward: largest chunk (row blocks) whose fp16 logit block
// stays within kMaxStoredChunkBytes (twice that when there is only one block).
int stored_max_blocks(long long ldS, int n_sbuf) {
  // One block may take the room (and the row bound) of two.
  const int f = n_sbuf == 1 ? 2 : 1;
  const long long by_mem = static_cast<long long>(f * kMaxStoredChunkBytes / (BM * ldS * 2));
  return static_cast<int>(
      std::max(1LL, std::min<long long>(f * kMaxStoredChunkBlocks, by_mem)));
}

// Fraction of SM time a launch of `units` equal units keeps busy.
double wave_eff(long long units, int sms) {
  const long long waves = cdiv(units, sms);
  return static_cast<double>(units) / static_cast<double>(waves * sms);
}

// Forward vocab splits for a chunk of nrb row blocks: whole waves of
// (row block x split) units, and splits of even length in vocab tiles.
int stored_fwd_splits(int nrb, int nvt, int sms, double* eff_out) {
  int best = 1;
  double best_eff = -1.0;
  for (int sp = 1; sp <= std::min(nvt, kMaxSplits); ++sp) {
    const double even = (static_cast<double>(nvt) / sp) / static_cast<double>(cdiv(nvt, sp));
    const double eff = wave_eff(static_cast<long long>(nrb) * sp, sms) * even;
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = sp;
    }
  }
  if (eff_out) *eff_out = best_eff;
  return best;
}

// Row units per raster group of a logit GEMM launch: all of its row units, as
// long as their hidden rows (re-read for every vocab tile) stay within a
// third of L2; past that the slots in flight would evict each other's rows.
int fwd_group_rows(int n_ru, int D, int ctas) {
  constexpr long long kHBudget = 40LL << 20;
  const long long per_ru = static_cast<long long>(BM) * ctas * D * 2;
  return static_cast<int>(std::max<long long>(1, std::min<long long>(n_ru, kHBudget / per_ru)));
}

// Row units per raster group: the slots in flight (one per SM pair) cover
// group_rows row units x (slots / group_rows) vocab tiles or splits, so each
// W tile fetched from HBM is shared through L2 by group_rows slots and each
// row unit's hidden states by the others.
int group_rows_for(int n_rb, int sms) {
  return std::max(1, std::min(n_rb, std::max(1, sms) / kSplitsTarget));
}

// Same, with group_rows a divisor of the slot count (at least 4 columns per
// group): a group is then exactly one round of the persistent grid, and the
// slots that share a W range all run in the same round.
int group_rows_exact(int n_ru, int slots) {
  slots = std::max(1, slots);
  const int cap = std::max(1, std::min(n_ru, slots / 4));
  for (int r = cap; r > 1; --r)
    if (slots % r == 0) return r;
  return 1;
}

// Raster and vocab splits of a logit GEMM over n_ru row units in one launch:
// one round of the slots per raster group (group_rows_exact, slots / group
// splits, long units) when that fills its rounds to 90 %; otherwise the splits
// that fill whole waves, over L2-sized groups (measured: at 512 row units the
// first is 10-20 % faster, at 32 the second 12 %).
void whole_batch_raster(int n_ru, int nvt, int D, int ctas, int slots, int* group, int* splits) {
  const int r = group_rows_exact(n_ru, slots);
  const int sp = std::min(std::max(1, slots / r), std::min(nvt, kMaxSplits));
  if (wave_eff(static_cast<long long>(n_ru) * sp, slots) >= 0.9) {
    *group = r;
    *splits = sp;
  } else {
    *group = fwd_group_rows(n_ru, D, ctas);
    *splits = stored_fwd_splits(n_ru, nvt, slots, nullptr);
  }
}

// Rounds of a dH-type launch of `units` units on `slots` SM pairs: whole
// rounds, or with the tail split the last round's U units spread over the U
// pairs and min(slots - U, slots / 3) tail pairs.
double dh_rounds(long long units, int slots, bool split) {
  const long long full = units / slots, u = units % slots;
  if (u == 0) return static_cast<double>(full);
  if (!split) return static_cast<double>(full + 1);
  return static_cast<double>(full) +
         static_cast<double>(u) / static_cast<double>(u + std::min<long long>(slots - u, slots / 3));
}

// Modelled GEMM time of the stored-logit schedule with chunks of nrb row
// units, in forward-tile times (one 256-row x 256-column x D tile on one SM
// pair). Each chunk runs a forward launch of (row units x splits) units and a
// dH launch of (row units x D tiles) units, both rounded up to whole waves,
// plus whatever of each chunk's separate G pass the GEMMs around it cannot
// hide. exposed_g is that pass's time relative to the forward GEMM of the same
// rows (0 when dH forms G itself). In the overlapped schedule pass c runs
// beside dH(c-1) and the forward of chunk c+1; with a single chunk it is fully
// exposed. split: every dH launch has the tail split (dh_rounds).
double stored_cost(long long n_rb_total, int nrb, int n_dt, int nvt, int sms, double exposed_g,
                   bool split = false) {
  std::vector<double> fwd, dh;
  double actual = 0.0;
  for (long long r0 = 0; r0 < n_rb_total; r0 += nrb) {
    const int n = static_cast<int>(std::min<long long>(nrb, n_rb_total - r0));
    const int sp = stored_fwd_splits(n, nvt, sms, nullptr);
    // forward: waves x tiles per unit (the longest unit sets the pace)
    fwd.push_back(static_cast<double>(cdiv(static_cast<long long>(n) * sp, sms)) *
                  cdiv(nvt, sp));
    // dH: units of equal K; scaled to the forward's per-row work
    dh.push_back(dh_rounds(static_cast<long long>(n) * n_dt, sms, split) * nvt / n_dt);
    actual += fwd.back() + dh.back();
  }
  const size_t nc = fwd.size();
  for (size_t c = 0; c < nc; ++c) {
    const double window = (c > 0 ? dh[c - 1] : 0.0) + (c + 1 < nc ? fwd[c + 1] : 0.0);
    actual += std::max(0.0, exposed_g * fwd[c] - window);
  }
  return actual;
}

// Row units per chunk for the stored-logit backward: the best ratio of the
// ideal SM time of the whole schedule (every chunk, including a shorter last
// one) to its modelled time. Plans of more than one chunk take at most
// max_multi row units per chunk (they may need two chunk blocks). Near-ties go
// to the larger chunk.
int auto_stored_chunk_blocks(long long n_rb_total, int n_dt, int nvt, int sms, int max_units,
                             int max_multi, double exposed_g) {
  const int hi = static_cast<int>(std::min<long long>(n_rb_total, max_units));
  int best = std::min(hi, std::max(1, max_multi));
  if (hi >= n_rb_total) best = hi;
  double best_score = -1.0;
  const double ideal = 2.0 * static_cast<double>(n_rb_total) * nvt / sms;
  for (int nrb = hi; nrb >= 1; --nrb) {
    if (nrb < n_rb_total && nrb > max_multi) continue;
    const double score = ideal / stored_cost(n_rb_total, nrb, n_dt, nvt, sms, exposed_g);
    if (score > best_score + 0.005) {
      best_score = score;
      best = nrb;
    }
  }
  return best;
}

// Modelled GEMM time of the recomputed-logit schedule (same unit as
// stored_cost): per chunk of nrb row units a forward of (row units x splits)
// units, the splits those of a full chunk's whole waves, then per vocab block
// of vb_tiles tiles a G-tile launch of (row units x tiles) units and a dH
// launch of (row units x D tiles) units of K = the block.
double recompute_cost(long long n_rb_total, int nrb, int n_dt, int nvt, int vb_tiles, int sms) {
  const int splits =
      stored_fwd_splits(static_cast<int>(std::min<long long>(nrb, n_rb_total)), nvt, sms, nullptr);
  double actual = 0.0;
  for (long long r0 = 0; r0 < n_rb_total; r0 += nrb) {
    const long long n = std::min<long long>(nrb, n_rb_total - r0);
    actual += static_cast<double>(cdiv(n * splits, sms)) * cdiv(nvt, splits);
    for (int t0 = 0; t0 < nvt; t0 += vb_tiles) {
      const int w = std::min(vb_tiles, nvt - t0);
      actual += static_cast<double>(cdiv(n * w, sms));
      actual += static_cast<double>(cdiv(n * n_dt, sms)) * w / n_dt;
    }
  }
  return actual;
}

// Forward vocab splits of one block of the single-pass backward: whole waves
// of (row unit x split) units, at most `cap` splits (every block's splits
// share the kMaxSplits partial slots of a row).
int single_pass_fwd_splits(int nrb, int tiles, int cap, int sms) {
  int best = 1;
  double best_eff = -1.0;
  for (int sp = 1; sp <= std::min(tiles, cap); ++sp) {
    const double even = (static_cast<double>(tiles) / sp) / static_cast<double>(cdiv(tiles, sp));
    const double eff = wave_eff(static_cast<long long>(nrb) * sp, sms) * even;
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = sp;
    }
  }
  return best;
}

// Modelled GEMM time of the single-pass schedule (same unit as stored_cost):
// per chunk of nrb row units and per vocab block of `tiles` tiles, a logit
// GEMM of (row units x splits) units and a U GEMM of (row units x D tiles)
// units of K = the block. The U GEMM converts every landed logit stage on chip
// (measured: about a fifth of its time on GB300) and, with several blocks,
// reads and rewrites its fp32 accumulator once per block.
double single_pass_cost(long long n_rb_total, int nrb, int n_dt, int nvt, int vb_tiles, int nvb,
                        int sms, double exposed_p, bool split = false) {
  // exposed_p = 0: P formed on chip; otherwise the P pass's time relative to
  // the block's forward GEMM, of which the neighbouring GEMMs hide what they
  // can (as in stored_cost). Measured on GB300 against the stored form's GEMMs
  // over the same rows: the U GEMM takes 1.07-1.12x the dH GEMM reading P
  // (Llama-3.1-8B, gpt-oss-20b heads), 1.24x forming P on chip (Llama); the
  // per-block logit GEMMs 0.99-1.05x the whole-vocabulary one.
  const double uac_factor = exposed_p > 0.0 ? 1.10 : 1.22;
  const double fwd_factor = 1.03;
  std::vector<double> fwd, uac;
  double actual = 0.0;
  for (long long r0 = 0; r0 < n_rb_total; r0 += nrb) {
    const int n = static_cast<int>(std::min<long long>(nrb, n_rb_total - r0));
    for (int t0 = 0; t0 < nvt; t0 += vb_tiles) {
      const int w = std::min(vb_tiles, nvt - t0);
      const int sp = single_pass_fwd_splits(n, w, kMaxSplits / nvb, sms);
      fwd.push_back(static_cast<double>(cdiv(static_cast<long long>(n) * sp, sms)) * cdiv(w, sp) *
                    fwd_factor);
      uac.push_back(dh_rounds(static_cast<long long>(n) * n_dt, sms, split) * w / n_dt *
                    uac_factor);
      actual += fwd.back() + uac.back();
    }
  }
  if (exposed_p > 0.0) {
    const size_t nb = fwd.size();
    for (size_t b = 0; b < nb; ++b) {
      const double window = (b > 0 ? uac[b - 1] : 0.0) + (b + 1 < nb ? fwd[b + 1] : 0.0);
      actual += std::max(0.0, exposed_p * fwd[b] - window);
    }
  }
  return actual;
}

// Workspace budget of a call in bytes (0 = none): the caller's limit, or half
// of the device's free memory with GRPO_FLAG_FIT_FREE_MEMORY.
size_t workspace_budget(const grpo_params* p) {
  if (p == nullptr) return 0;
  size_t budget = static_cast<size_t>(p->workspace_limit_bytes);
  if ((p->flags & GRPO_FLAG_FIT_FREE_MEMORY) != 0) {
    size_t free_b = 0, total_b = 0;
    if (cudaMemGetInfo(&free_b, &total_b) == cudaSuccess) {
      const size_t half = free_b / 2;
      budget = budget == 0 ? half : std::min(budget, half);
    }
  }
  return budget;
}

// Layout of a call with the backward form fixed (stored: fp16 logits of the
// whole vocabulary kept per chunk; single pass: one vocabulary block's logits
// at a time and an fp32 U accumulator; recompute: recomputed logit tiles).
// sms = 0: the sizing without a device (the largest automatic chunk).
int make_layout_mode(const grpo_shape* s, const grpo_params* p, int sms, Form form,
                     Layout* L) {
  L->ctas = (p != nullptr && (p->flags & GRPO_FLAG_SINGLE_CTA) != 0) ? 1 : 2;
  L->stored = form == kFormStored;
  L->single_pass = form == kFormSinglePass || form == kFormSinglePassPass;
  L->model_cost = 0.0;
  L->ldS = cdiv(std::max(s->vocab, 1), 8) * 8;
  L->n = s->n_tokens;
  L->nr = cdiv(std::max<long long>(s->n_tokens, 1), BM) * BM;
  L->T = s->seq_len;
  L->D = s->hidden;
  L->V = s->vocab;
  L->nvt = static_cast<int>(cdiv(s->vocab, BN));
  L->ctas = (p != nullptr && (p->flags & GRPO_FLAG_SINGLE_CTA) != 0) ? 1 : 2;
  const int n_dt = dh_tiles(s->hidden, L->ctas);
  long long vb = (p && p->vocab_block > 0) ? p->vocab_block : kAutoVocabBlock;
  if (L->single_pass) {
    // Equal blocks (the automatic size split evenly), at most kMaxSplits of
    // them: every block's forward splits need partial slots of their own.
    long long nb = cdiv(s->vocab, cdiv(vb, BN) * BN);
    if (p == nullptr || p->vocab_block <= 0) vb = cdiv(s->vocab, nb);
    nb = cdiv(s->vocab, cdiv(vb, BN) * BN);
    if (nb > kMaxSplits) vb = cdiv(s->vocab, kMaxSplits);
  }
  vb = cdiv(vb, BN) * BN;
  vb = std::min<long long>(vb, static_cast<long long>(L->nvt) * BN);
  L->nvb = static_cast<int>(cdiv(s->vocab, vb));
  if (L->stored) {
    L->vblock = static_cast<int>(L->ldS);
  } else {
    L->vblock = static_cast<int>(vb);
  }
  if (L->single_pass) L->ldS = L->vblock;
  L->need_acc = !L->stored && L->vblock < L->V;
  // Stored form and single pass at D <= kFusedMaxHidden: the dH-type GEMM forms
  // G (or P) from the stored logits itself; above it a row-wise pass does,
  // beside the next GEMMs, on a second block.
  L->fused = (L->stored && L->D <= kFusedMaxHidden) || form == kFormSinglePass;
  // 64-column boxes of a stored row (the whole vocabulary, or one block).
  L->nbox = static_cast<int>(cdiv(L->single_pass ? L->vblock : std::max(s->vocab, 1), 64));

  // Everything before the backward chunk block depends on N only.
  size_t off = kHeaderBytes;
  const size_t part = static_cast<size_t>(kMaxSplits) * L->nr * sizeof(float);
  L->off_pm = off; off = align_up(off + part, 256);
  L->off_ps = off; off = align_up(off + part, 256);
  L->off_zy = off; off = align_up(off + L->nr * sizeof(float), 256);
  L->off_lse = off; off = align_up(off + L->nr * sizeof(float), 256);
  L->off_g = off; off = align_up(off + L->nr * sizeof(float), 256);
  L->off_rbl = off; off = align_up(off + (L->nr / SEG) * sizeof(int), 256);
  L->off_lt = off; off = align_up(off + L->nr * sizeof(double), 256);
  L->off_seq = off; off = align_up(off + L->nr * sizeof(int), 256);  // >= N / T lengths
  // Tail-split slots: stored form, single pass with P on chip; not under a
  // budget they would take more than an eighth of.
  const size_t budget = workspace_budget(p);
  L->ts_slots = L->stored ? tail_split_slots(s->vocab, L->ctas, sms)
                : form == kFormSinglePass ? tail_split_slots(static_cast<int>(L->vblock), L->ctas, sms)
                                          : 0;
  if (L->ts_slots > 0 && budget > 0 && tail_split_bytes(L->ts_slots, L->ctas) * 8 > budget)
    L->ts_slots = 0;
  L->off_sk = off;
  if (L->ts_slots > 0) off = align_up(off + tail_split_bytes(L->ts_slots, L->ctas), 256);
  L->off_G = off;

  // Chunks are whole row units (BM * ctas rows: what one CTA pair covers).
  const long long ru_rows = static_cast<long long>(BM) * L->ctas;
  const long long n_ru_total = cdiv(L->nr, ru_rows);
  const int slots = sms / L->ctas;
  // Bytes of the chunk block per row unit: bf16 G (+ fp32 dH accumulator) or
  // fp16 logits.
  // The stored path keeps two chunk blocks when there is more than one chunk
  // (one being turned into G while the next chunk's logits are computed),
  // one when the dH GEMM forms G itself.
  const int sbufs = (L->stored || L->single_pass) && !L->fused ? 2 : 1;
  const bool boxes = L->stored || L->single_pass;  // fp16 logits with box maxima
  // A chunk's copy of h for the row blocks whose active segments are not
  // consecutive rows (read by its logit or G-tile GEMMs, which run one chunk
  // after another on the caller's stream; the dW GEMM reads h itself).
  const int hc_bufs = 1;
  const size_t unit_bytes = static_cast<size_t>(ru_rows) *
                            (static_cast<size_t>(L->vblock) * 2 * sbufs +
                             (boxes ? static_cast<size_t>(L->nbox) * 4 * sbufs : 0) +
                             (L->need_acc ? L->D * 4 : 0) + static_cast<size_t>(L->D) * 2 * hc_bufs);
  long long max_units = L->stored        ? std::max(1, stored_max_blocks(L->ldS, sbufs) / L->ctas)
                        : L->single_pass ? kMaxSinglePassChunkBlocks / L->ctas
                                         : kMaxAutoChunkBlocks / L->ctas;
  if (budget > 0) {
    const long long fit =
        budget > off + 512 ? static_cast<long long>((budget - off - 512) / unit_bytes) : 0;
    if (fit < 1) return GRPO_ERR_WORKSPACE_TOO_SMALL;
    max_units = std::min(max_units, fit);
  }
  long long crows;
  if (p && p->chunk_tokens > 0) {
    crows = cdiv(p->chunk_tokens, ru_rows) * ru_rows;
  } else if (L->stored) {
    // The G pass moves 4 bytes per logit against the forward's 2 D flops:
    // about 550 / D of the forward GEMM's time on GB300 (measured at D = 4096).
    const double exposed_g = L->fused ? 0.0 : 550.0 / L->D;
    // A device plan never needs more than the sizing without a device (the
    // largest chunk): when that is one block for the whole batch, a plan of
    // several double-buffered chunks gets half of it per chunk.
    const long long big = std::min<long long>(n_ru_total, max_units);
    const long long room = big * (sbufs == 2 && big < n_ru_total ? 2 : 1);
    const int max_multi = static_cast<int>(std::max<long long>(1, room / sbufs));
    crows = (sms > 0 ? auto_stored_chunk_blocks(n_ru_total, n_dt, L->nvt, slots,
                                                static_cast<int>(max_units), max_multi,
                                                exposed_g)
                     : std::min<long long>(n_ru_total, max_units)) *
            ru_rows;
  } else if (sms > 0 && L->single_pass) {
    // The best modelled schedule (near-ties to the larger chunk). With a
    // separate P pass and one vocabulary block, a plan of several chunks
    // needs two blocks: like the stored form, it then gets half of what the
    // sizing without a device (one chunk of the largest size) holds.
    const int hi = static_cast<int>(std::min<long long>(n_ru_total, max_units));
    const int vbt = static_cast<int>(cdiv(L->vblock, BN));
    const long long room = static_cast<long long>(hi) * (hi < n_ru_total ? 2 : 1);
    const int max_multi =
        (sbufs == 2 && L->nvb == 1) ? static_cast<int>(std::max<long long>(1, room / 2)) : hi;
    int best = (hi < n_ru_total) ? std::min(hi, max_multi) : hi;
    double best_cost = 0.0;
    bool have = false;
    for (int nrb = hi; nrb >= 1; --nrb) {
      if (nrb < n_ru_total && nrb > max_multi) continue;
      const double cost = single_pass_cost(n_ru_total, nrb, n_dt, L->nvt, vbt, L->nvb, slots,
                                           L->fused ? 0.0 : 550.0 / L->D);
      if (!have || cost < best_cost * 0.995) {
        best_cost = cost;
        best = nrb;
        have = true;
      }
    }
    crows = static_cast<long long>(best) * ru_rows;
  } else if (sms > 0) {
    // Recomputed logits: the best modelled schedule (per-chunk forward, G-tile
    // and dH launches), near-ties to the larger chunk.
    const int hi = static_cast<int>(std::min<long long>(n_ru_total, max_units));
    const int vbt = static_cast<int>(cdiv(L->vblock, BN));
    int best = hi;
    double best_cost = 0.0;
    for (int nrb = hi; nrb >= 1; --nrb) {
      const double cost = recompute_cost(n_ru_total, nrb, n_dt, L->nvt, vbt, slots);
      if (nrb == hi || cost < best_cost * 0.995) {
        best_cost = cost;
        best = nrb;
      }
    }
    crows = static_cast<long long>(best) * ru_rows;
  } else {  // sizing without a device: the largest automatic chunk
    crows = std::min<long long>(n_ru_total, max_units) * ru_rows;
  }
  crows = std::min(crows, n_ru_total * ru_rows);
  if (crows > INT_MAX / 2) return GRPO_ERR_UNSUPPORTED_SHAPE;
  L->chunk_rows = static_cast<int>(crows);
  // Two blocks when one can be converted while the next is written: more than
  // one chunk (stored form), more than one chunk x vocab block (single pass).
  L->n_sbuf = (sbufs == 2 && cdiv(L->nr, L->chunk_rows) * (L->single_pass ? L->nvb : 1) > 1)
                  ? 2 : 1;

  // Backward chunk block: bf16 G [C x V_b] (recompute path) or the chunk's
  // fp16 logits, rewritten in place as bf16 G [C x ldS] (stored path; two of
  // them when double-buffered).
  off = align_up(off + static_cast<size_t>(L->n_sbuf) * L->chunk_rows * L->vblock * 2, 256);
  // Stored and single-pass paths: the maxima of each block's 64-column boxes,
  // fp32 [nbox][chunk rows].
  L->off_bmax = off;
  if (boxes)
    off = align_up(off + static_cast<size_t>(L->n_sbuf) * L->nbox * L->chunk_rows * 4, 256);
  L->off_acc = off;
  if (L->need_acc) off = align_up(off + static_cast<size_t>(L->chunk_rows) * L->D * 4, 256);
  L->n_hc = hc_bufs;
  L->off_hc = off;
  off = align_up(off + static_cast<size_t>(L->n_hc) * L->chunk_rows * L->D * 2, 256);
  L->total = off;
  if (budget > 0 && L->total > budget) return GRPO_ERR_WORKSPACE_TOO_SMALL;
  if (sms > 0) {
    const int rb = static_cast<int>(L->chunk_rows / ru_rows);
    const int vbt = static_cast<int>(cdiv(L->vblock, BN));
    // The forms compared at D <= kFusedMaxHidden (the stored form's fused dH
    // GEMM, the single pass with P on chip) split every dH-type launch when the
    // slots are reserved: counted here, when forms are compared. Chunk sizes
    // are still chosen counting whole rounds: with padding the device runs
    // fewer row units than planned, and the larger chunks that this favours
    // measured faster. Above kFusedMaxHidden the split covers at most a last
    // launch and is not counted.
    const bool split = L->ts_slots > 0 && L->fused && L->D <= kFusedMaxHidden;
    L->model_cost = L->stored        ? stored_cost(n_ru_total, rb, n_dt, L->nvt, slots,
                                                   L->fused ? 0.0 : 550.0 / L->D, split)
                    : L->single_pass ? single_pass_cost(n_ru_total, rb, n_dt, L->nvt, vbt,
                                                        L->nvb, slots,
                                                        L->fused ? 0.0 : 550.0 / L->D, split)
                                     : recompute_cost(n_ru_total, rb, n_dt, L->nvt, vbt, slots);
  }
  return GRPO_OK;
}

// The form with the shortest modelled GEMM time among `forms` that fit the
// workspace budget, modelled at the reference SM count (so that sizing and
// call agree); ties go to the earlier one. Returns its layout at `sms`.
int best_layout(const grpo_shape* s, const grpo_params* p, int sms, const Form* forms, int n,
                Layout* L) {
  int rc = GRPO_OK;
  int best = -1;
  double best_cost = 0.0;
  for (int i = 0; i < n; ++i) {
    Layout t;
    const int r = make_layout_mode(s, p, kRefSms, forms[i], &t);
    if (r != GRPO_OK) {
      rc = r;
      continue;
    }
    if (best < 0 || t.model_cost < best_cost) {
      best = i;
      best_cost = t.model_cost;
    }
  }
  if (best < 0) return rc;
  return make_layout_mode(s, p, sms, forms[best], L);
}

// Layout of a call. GRPO_FLAG_STORED_LOGITS, GRPO_FLAG_SINGLE_PASS or
// GRPO_FLAG_RECOMPUTE_LOGITS fix the backward form; without any of them the
// planner takes, among the forms that fit the workspace budget, the one with
// the shortest modelled GEMM time; ties go to the form listed first: stored,
// single pass, recompute. Above kFusedMaxHidden the single pass's P
// placement (on chip, one block; or a pass of its own, two blocks) is chosen
// the same way.
int make_layout(const grpo_shape* s, const grpo_params* p, int sms, Layout* L) {
  const uint32_t f = p != nullptr ? p->flags : 0u;
  const bool p_pass = s->hidden > kFusedMaxHidden;
  if ((f & GRPO_FLAG_STORED_LOGITS) != 0) return make_layout_mode(s, p, sms, kFormStored, L);
  if ((f & GRPO_FLAG_RECOMPUTE_LOGITS) != 0)
    return make_layout_mode(s, p, sms, kFormRecompute, L);
  if ((f & GRPO_FLAG_SINGLE_PASS) != 0) {
    const Form sp[2] = {kFormSinglePassPass, kFormSinglePass};
    return p_pass ? best_layout(s, p, sms, sp, 2, L)
                  : make_layout_mode(s, p, sms, kFormSinglePass, L);
  }
  const Form all[4] = {kFormStored, kFormSinglePassPass, kFormSinglePass, kFormRecompute};
  const Form fused[3] = {kFormStored, kFormSinglePass, kFormRecompute};
  return p_pass ? best_layout(s, p, sms, all, 4, L) : best_layout(s, p, sms, fused, 3, L);
}

int check_shape(const grpo_shape* s, bool need_seq) {
  if (!s) return GRPO_ERR_INVALID_ARG;
  if (s->n_tokens < 0 || s->hidden <= 0 || s->vocab <= 0 || s->reserved != 0)
    return GRPO_ERR_INVALID_ARG;
  if (s->hidden % 8 != 0) return GRPO_ERR_UNSUPPORTED_SHAPE;
  if (s->n_tokens > (1LL << 30)) return GRPO_ERR_UNSUPPORTED_SHAPE;
  if (need_seq) {
    if (s->seq_len <= 0) return GRPO_ERR_INVALID_ARG;
    if (s->n_tokens % s->seq_len != 0) return GRPO_ERR_UNSUPPORTED_SHAPE;
  }
  return GRPO_OK;
}

int check_params(const grpo_params* p) {
  if (!p) return GRPO_OK;
  if ((p->flags & ~(GRPO_FLAG_STORED_LOGITS | GRPO_FLAG_SINGLE_CTA | GRPO_FLAG_SEQUENCE_MEAN |
                    GRPO_FLAG_FIT_FREE_MEMORY | GRPO_FLAG_RECOMPUTE_LOGITS |
                    GRPO_FLAG_SINGLE_PASS)) != 0 ||
      p->raster_rows < 0 || p->chunk_tokens < 0 || p->vocab_block < 0)
    return GRPO_ERR_INVALID_ARG;
  const uint32_t forms =
      p->flags & (GRPO_FLAG_STORED_LOGITS | GRPO_FLAG_RECOMPUTE_LOGITS | GRPO_FLAG_SINGLE_PASS);
  if ((forms & (forms - 1)) != 0) return GRPO_ERR_INVALID_ARG;  // at most one form
  if (!(p->eps_low >= 0.f) || !(p->eps_high >= 0.f) || !(p->beta >= 0.f))
    return GRPO_ERR_INVALID_ARG;
  if (!(p->logit_scale_multiply >= 0.f) || !(p->logit_scale_divide >= 0.f) ||
      !(p->logit_softcapping >= 0.f) || !(p->temperature >= 0.f))
    return GRPO_ERR_INVALID_ARG;
  return GRPO_OK;
}

// Logit transform constants for the epilogues (see TileArgs::xmode).
void set_transform(TileArgs* a, const grpo_params* p) {
  a->xmode = 0;
  a->k0 = a->k1 = a->k2 = 1.f;
  if (!p) return;
  const double mul = p->logit_scale_multiply > 0.f ? p->logit_scale_multiply : 1.0;
  const double div = p->logit_scale_divide > 0.f ? p->logit_scale_divide : 1.0;
  const double temp = p->temperature > 0.f ? p->temperature : 1.0;
  const double cap = p->logit_softcapping;
  const double scale = mul / div;
  a->k0 = static_cast<float>(scale / temp);
  if (cap > 0.0) {
    a->xmode = 2;
    a->k1 = static_cast<float>(scale / cap);
    a->k2 = static_cast<float>(cap / temp);
  } else if (scale / temp != 1.0) {
    a->xmode = 1;
  }
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ------------------------------------------------------------ device ----

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceInfo {
  bool ready = false;
  int status = GRPO_OK;
  int sms = 0;
  // Side stream for the stored path's row-wise G formation, which overlaps
  // the next chunk's logit GEMM; events order it against the caller's stream.
  cudaStream_t side = nullptr;
  cudaEvent_t ev_main = nullptr;
  cudaEvent_t ev_fwd[2] = {nullptr, nullptr};
  cudaEvent_t ev_g[2] = {nullptr, nullptr};
  // Held while one call enqueues its work on the side stream: the events are
  // shared, and each record must be followed by its own waits before another
  // call records again (cudaStreamWaitEvent takes the record current at the
  // time it is enqueued).
  std::mutex side_mu;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

int device_setup(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GRPO_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GRPO_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    d.ready = true;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      d.status = GRPO_ERR_CUDA;
    } else if (major != 10 || minor != 3) {
      d.status = GRPO_ERR_UNSUPPORTED_DEVICE;
    } else if (prepare_fwd_gemm() != cudaSuccess || prepare_bwd_gemms() != cudaSuccess ||
               prepare_fwds_gemm() != cudaSuccess) {
      d.status = GRPO_ERR_CUDA;
    }
    if (d.status == GRPO_OK) {
      bool okc = cudaStreamCreateWithFlags(&d.side, cudaStreamNonBlocking) == cudaSuccess &&
                 cudaEventCreateWithFlags(&d.ev_main, cudaEventDisableTiming) == cudaSuccess;
      for (int i = 0; i < 2 && okc; ++i)
        okc = cudaEventCreateWithFlags(&d.ev_fwd[i], cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&d.ev_g[i], cudaEventDisableTiming) == cudaSuccess;
      if (!okc) d.status = GRPO_ERR_CUDA;
    }
    if (d.status == GRPO_OK && g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr) {
        d.status = GRPO_ERR_CUDA;
      } else {
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
      }
    }
  }
  *sms = d.sms;
  return d.status;
}

DeviceInfo* current_device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return &g_dev[dev];
}

// 2-D bf16 tensor map: `inner` contiguous elements per row, `outer` rows,
// `pitch_elems` elements between rows; box {box_inner, box_outer}; 128B swizzle.
bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
               uint64_t pitch_elems, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
               uint64_t elem_bytes = 2) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_elems * elem_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct Ws {
  uint8_t* base;
  int* status;
  unsigned* counter;
  double* msum;
  double* partials;
  double* lt;
  int* n_seg;     // length of the active-segment list
  int* n_nonempty;
  int* seq_lens;
  int* seg_list;  // the active 16-row segments (row plan)
  float *pm, *ps, *zy, *lse, *g, *acc, *sk;
  __nv_bfloat16* hc;  // chunk copies of h's rows (Layout::n_hc of chunk_rows x D)
  __nv_bfloat16* G;
};

Ws carve(void* ws, const Layout& L) {
  Ws w;
  w.base = static_cast<uint8_t*>(ws);
  w.status = reinterpret_cast<int*>(w.base + kOffStatus);
  w.counter = reinterpret_cast<unsigned*>(w.base + kOffCounter);
  w.msum = reinterpret_cast<double*>(w.base + kOffMsum);
  w.partials = reinterpret_cast<double*>(w.base + kOffPartials);
  w.n_seg = reinterpret_cast<int*>(w.base + kOffActive);
  w.n_nonempty = reinterpret_cast<int*>(w.base + kOffNonempty);
  w.seq_lens = reinterpret_cast<int*>(w.base + L.off_seq);
  w.seg_list = reinterpret_cast<int*>(w.base + L.off_rbl);
  w.lt = reinterpret_cast<double*>(w.base + L.off_lt);
  w.pm = reinterpret_cast<float*>(w.base + L.off_pm);
  w.ps = reinterpret_cast<float*>(w.base + L.off_ps);
  w.zy = reinterpret_cast<float*>(w.base + L.off_zy);
  w.lse = reinterpret_cast<float*>(w.base + L.off_lse);
  w.g = reinterpret_cast<float*>(w.base + L.off_g);
  w.G = reinterpret_cast<__nv_bfloat16*>(w.base + L.off_G);
  w.acc = reinterpret_cast<float*>(w.base + L.off_acc);
  w.sk = L.ts_slots > 0 ? reinterpret_cast<float*>(w.base + L.off_sk) : nullptr;
  w.hc = reinterpret_cast<__nv_bfloat16*>(w.base + L.off_hc);
  return w;
}

TileArgs base_args(const Layout& L, const Ws& w) {
  TileArgs a;
  std::memset(&a, 0, sizeof(a));
  a.vocab = L.V;
  a.hidden = L.D;
  a.status = w.status;
  return a;
}

// Forward logit GEMM: per-split (max, sum-exp) and z_y for every row of the
// active segments in `seg_list` (every row when it is null), in the raster of
// whole_batch_raster; with a segment list the kernel sets the splits from the
// active row units (whole waves), and the row finish reads every partial slot.
int run_forward(const void* hidden, const void* W, const int32_t* ids, const uint8_t* mask,
                const int* seg_list, const int* n_seg, const grpo_params* prm,
                const Layout& L, const Ws& w, int sms, int* splits_out, cudaStream_t st) {
  CUtensorMap map_h, map_h16, map_w;
  const int slots = std::max(1, sms / L.ctas);
  if (!encode_2d(&map_h, hidden, L.D, L.n, L.D, BK, BM) ||
      !encode_2d(&map_h16, hidden, L.D, L.n, L.D, BK, SEG) ||
      !encode_2d(&map_w, W, L.D, L.V, L.D, BK, BN / L.ctas))
    return GRPO_ERR_CUDA;
  TileArgs a = base_args(L, w);
  set_transform(&a, prm);
  a.n_total = L.n;
  a.n_rb = static_cast<int>(L.nr / BM);
  a.rb_offset = 0;
  a.seg_list = seg_list;
  a.n_seg = n_seg;
  a.k_iters = static_cast<int>(cdiv(L.D, BK));
  const int n_ru = static_cast<int>(cdiv(a.n_rb, L.ctas));
  int group = 1, splits = 1;
  whole_batch_raster(n_ru, L.nvt, L.D, L.ctas, slots, &group, &splits);
  a.group_rows = (prm != nullptr && prm->raster_rows > 0) ? std::min(prm->raster_rows, n_ru)
                                                         : group;
  a.n_cols = splits;
  if (seg_list != nullptr) a.max_cols = std::min(L.nvt, kMaxSplits);
  a.n_vtiles = L.nvt;
  a.v0 = 0;
  a.ids = ids;
  a.mask = mask;
  a.part_m = w.pm;
  a.part_s = w.ps;
  a.zy = w.zy;
  a.part_ld = L.nr;
  const long long units = static_cast<long long>(n_ru) * a.n_cols;
  const int grid =
      L.ctas * (a.max_cols > 0 ? slots : static_cast<int>(std::min<long long>(units, slots)));
  if (launch_fwd_gemm(L.ctas, map_h, map_w, map_h16, a, grid, st) != cudaSuccess)
    return GRPO_ERR_CUDA;
  *splits_out = a.max_cols > 0 ? a.max_cols : splits;
  return GRPO_OK;
}

// The recomputed form's forward of a loss call, one logit GEMM per chunk of
// the backward's chunking, after the chunk's non-consecutive row blocks of h
// are gathered (so that every row block loads in one box). Each launch splits
// the vocabulary into the count that makes its active row units whole waves
// of the SM pairs (set by the kernel; a count set by the whole batch leaves
// most pairs idle on a chunk of a few row units), and the row finish reads
// every partial slot. A row's partial sums, and so its last bits, depend on
// the chunk size.
int run_forward_chunks(const void* hidden, const void* W, const int32_t* ids,
                       const uint8_t* mask, const grpo_params* prm, const Layout& L,
                       const Ws& w, int sms, int* splits_out, cudaStream_t st) {
  CUtensorMap map_h, map_h16, map_w;
  const int slots = std::max(1, sms / L.ctas);
  if (!encode_2d(&map_h, hidden, L.D, L.n, L.D, BK, BM) ||
      !encode_2d(&map_h16, hidden, L.D, L.n, L.D, BK, SEG) ||
      !encode_2d(&map_w, W, L.D, L.V, L.D, BK, BN / L.ctas))
    return GRPO_ERR_CUDA;
  const int n_rb_total = static_cast<int>(L.nr / BM);
  const int rb_per_chunk = L.chunk_rows / BM;
  const int n_ru_full = static_cast<int>(cdiv(std::min(rb_per_chunk, n_rb_total), L.ctas));
  const int splits = stored_fwd_splits(n_ru_full, L.nvt, slots, nullptr);
  for (int rb0 = 0; rb0 < n_rb_total; rb0 += rb_per_chunk) {
    const int n_rb = std::min(rb_per_chunk, n_rb_total - rb0);
    const int n_ru = static_cast<int>(cdiv(n_rb, L.ctas));
    TileArgs a = base_args(L, w);
    set_transform(&a, prm);
    a.n_total = L.n;
    a.n_rb = n_rb;
    a.rb_offset = rb0;
    a.seg_list = w.seg_list;
    a.n_seg = w.n_seg;
    a.hc = 1;
    a.k_iters = static_cast<int>(cdiv(L.D, BK));
    a.group_rows = (prm != nullptr && prm->raster_rows > 0) ? std::min(prm->raster_rows, n_ru)
                                                            : fwd_group_rows(n_ru, L.D, L.ctas);
    a.n_cols = splits;
    a.max_cols = std::min(L.nvt, kMaxSplits);
    a.n_vtiles = L.nvt;
    a.v0 = 0;
    a.ids = ids;
    a.mask = mask;
    a.part_m = w.pm;
    a.part_s = w.ps;
    a.zy = w.zy;
    a.part_ld = L.nr;
    CUtensorMap map_hc;
    if (!encode_2d(&map_hc, w.hc, L.D, static_cast<uint64_t>(n_rb) * BM, L.D, BK, BM))
      return GRPO_ERR_CUDA;
    if (launch_gather_blocks(hidden, w.hc, a, st) != cudaSuccess) return GRPO_ERR_CUDA;
    if (launch_fwd_gemm(L.ctas, map_h, map_w, map_h16, a, L.ctas * slots, st, &map_hc) !=
        cudaSuccess)
      return GRPO_ERR_CUDA;
  }
  *splits_out = std::min(L.nvt, kMaxSplits);
  return GRPO_OK;
}

// dW[v0 : v0 + width) (+)= G^T H over the chunk's active row blocks; G is the
// chunk block (pitch ldG elements). first: this chunk starts the sum.
int launch_dw(const void* hidden, const __nv_bfloat16* G, long long ldG, int v0, int width,
              int rb0, int n_rb, float* dW, bool first, const Layout& L, const Ws& w, int sms,
              cudaStream_t st) {
  const int slots = std::max(1, sms / L.ctas);
  CUtensorMap map_gt, map_h_mn, map_h16, map_dw;
  if (!encode_2d(&map_gt, G, width, static_cast<uint64_t>(n_rb) * BM, ldG, 64, BK) ||
      !encode_2d(&map_h_mn, hidden, L.D, L.n, L.D, 64, BK) ||
      !encode_2d(&map_h16, hidden, L.D, L.n, L.D, 64, SEG) ||
      !encode_2d(&map_dw, dW + static_cast<size_t>(v0) * L.D, L.D, width, L.D, 32, 32,
                 CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4))
    return GRPO_ERR_CUDA;
  TileArgs a = base_args(L, w);
  a.n_total = L.n;
  a.n_rb = n_rb;
  a.rb_offset = rb0;
  a.seg_list = w.seg_list;
  a.n_seg = w.n_seg;
  const int n_vu = static_cast<int>(cdiv(width, static_cast<long long>(BM) * L.ctas));
  const int n_dt = static_cast<int>(cdiv(L.D, BN));
  a.group_rows = group_rows_for(n_vu, slots);
  a.n_cols = n_dt;
  a.v0 = v0;
  a.dw_rows = width;
  a.dW = dW;
  a.first = first ? 1 : 0;
  const long long units = static_cast<long long>(n_vu) * n_dt;
  if (launch_dw_gemm(L.ctas, map_gt, map_h_mn, map_h16, map_dw, a,
                     L.ctas * static_cast<int>(std::min<long long>(units, slots)),
                     st) != cudaSuccess)
    return GRPO_ERR_CUDA;
  return GRPO_OK;
}

// Backward over the active row blocks, in chunks of chunk_rows / BM list
// entries: G block, then dH accumulation, per vocab block. Chunks past the
// device-side list length find no work and return at once.
int run_backward(const void* hidden, const void* W, const int32_t* ids, void* dH, float* dW,
                 const grpo_params* prm, const Layout& L, const Ws& w, int sms,
                 cudaStream_t st) {
  CUtensorMap map_h, map_h16, map_w_k, map_w_mn;
  const int slots = std::max(1, sms / L.ctas);
  if (!encode_2d(&map_h, hidden, L.D, L.n, L.D, BK, BM) ||
      !encode_2d(&map_h16, hidden, L.D, L.n, L.D, BK, SEG) ||
      !encode_2d(&map_w_k, W, L.D, L.V, L.D, BK, BN / L.ctas) ||
      !encode_2d(&map_w_mn, W, L.D, L.V, L.D, 64, BK))
    return GRPO_ERR_CUDA;
  const int n_dt_dh = dh_tiles(L.D, L.ctas);
  const int n_rb_total = static_cast<int>(L.nr / BM);
  const int rb_per_chunk = L.chunk_rows / BM;
  for (int rb0 = 0; rb0 < n_rb_total; rb0 += rb_per_chunk) {
    const int n_rb = std::min(rb_per_chunk, n_rb_total - rb0);
    const int n_ru = static_cast<int>(cdiv(n_rb, L.ctas));
    // The chunk's non-consecutive row blocks of h, copied once for every
    // vocab block's G-tile GEMM.
    CUtensorMap map_hc;
    if (!encode_2d(&map_hc, w.hc, L.D, static_cast<uint64_t>(n_rb) * BM, L.D, BK, BM))
      return GRPO_ERR_CUDA;
    {
      TileArgs gh = base_args(L, w);
      gh.n_total = L.n;
      gh.n_rb = n_rb;
      gh.rb_offset = rb0;
      gh.seg_list = w.seg_list;
      gh.n_seg = w.n_seg;
      if (launch_gather_blocks(hidden, w.hc, gh, st) != cudaSuccess) return GRPO_ERR_CUDA;
    }
    for (long long v0 = 0; v0 < L.V; v0 += L.vblock) {
      const int width = static_cast<int>(std::min<long long>(L.vblock, L.V - v0));
      const int ntile = static_cast<int>(cdiv(width, BN));
      // (1) G = g (onehot - softmax) for this chunk x vocab block, bf16.
      TileArgs a = base_args(L, w);
      set_transform(&a, prm);
      a.n_total = L.n;
      a.n_rb = n_rb;
      a.rb_offset = rb0;
      a.seg_list = w.seg_list;
      a.n_seg = w.n_seg;
      a.k_iters = static_cast<int>(cdiv(L.D, BK));
      a.group_rows = (prm != nullptr && prm->raster_rows > 0) ? std::min(prm->raster_rows, n_ru)
                                                             : group_rows_exact(n_ru, slots);
      a.n_cols = ntile;
      a.v0 = static_cast<int>(v0);
      a.ids = ids;
      a.lse = w.lse;
      a.g = w.g;
      a.G = w.G;
      a.ldG = L.vblock;
      a.hc = 1;
      long long units = static_cast<long long>(n_ru) * ntile;
      CUtensorMap map_gst;  // the pair variant stores G through TMA
      if (!encode_2d(&map_gst, w.G, L.vblock, static_cast<uint64_t>(n_rb) * BM, L.vblock, 64,
                     32))
        return GRPO_ERR_CUDA;
      if (launch_bwdg_gemm(L.ctas, map_h, map_w_k, map_h16, map_gst, a,
                           L.ctas * static_cast<int>(std::min<long long>(units, slots)), st,
                           &map_hc) != cudaSuccess)
        return GRPO_ERR_CUDA;
      // (2) dH_chunk (+)= G W[v0 : v0 + width].
      CUtensorMap map_g;
      if (!encode_2d(&map_g, w.G, width, static_cast<uint64_t>(n_rb) * BM, L.vblock, BK, BM))
        return GRPO_ERR_CUDA;
      TileArgs b = base_args(L, w);
      b.n_total = L.n;
      b.n_rb = n_rb;
      b.rb_offset = rb0;
      b.seg_list = w.seg_list;
      b.n_seg = w.n_seg;
      b.k_iters = static_cast<int>(cdiv(width, BK));
      b.group_rows = group_rows_for(n_ru, slots);
      b.n_cols = n_dt_dh;
      b.v0 = static_cast<int>(v0);
      b.acc = w.acc;
      b.dH = static_cast<__nv_bfloat16*>(dH);
      b.first = v0 == 0;
      b.last = v0 + L.vblock >= L.V;
      units = static_cast<long long>(n_ru) * n_dt_dh;
      if (launch_dh_gemm(L.ctas, map_g, map_w_mn, b,
                         L.ctas * static_cast<int>(std::min<long long>(units, slots)),
                         st) != cudaSuccess)
        return GRPO_ERR_CUDA;
      // (3) optional lm_head gradient rows [v0, v0 + width) from the same G block.
      if (dW != nullptr) {
        const int r = launch_dw(hidden, w.G, L.vblock, static_cast<int>(v0), width, rb0, n_rb,
                                dW, rb0 == 0, L, w, sms, st);
        if (r != GRPO_OK) return r;
      }
    }
  }
  return GRPO_OK;
}

// Stored-logit path of a loss call, chunk by chunk over the active row
// blocks: forward GEMM that also stores the chunk's fp16 logits; per-row
// finish (lse, logp, token loss, g) rewriting the logits in place as bf16 G;
// dH GEMM over the whole vocabulary (and dW, when asked). With two chunk
// blocks the per-row finish of chunk c runs on a side stream while chunk c+1's
// logits are computed; the caller's stream sees one ordered sequence:
//   FWDS(0) FWDS(1) DH(0) FWDS(2) DH(1) ... DH(n-1), then the loss reduction.
int run_stored(const void* hidden, const void* W, const int32_t* ids, const uint8_t* mask,
               const float* old_logp, const float* ref_logp, const float* adv, float* loss,
               float* logp_out, void* dH, float* dW, const grpo_params* prm, const Layout& L,
               const Ws& w, int sms, cudaStream_t st) {
  CUtensorMap map_h, map_h16, map_w_k, map_w_mn;
  const int slots = std::max(1, sms / L.ctas);
  if (!encode_2d(&map_h, hidden, L.D, L.n, L.D, BK, BM) ||
      !encode_2d(&map_h16, hidden, L.D, L.n, L.D, BK, SEG) ||
      !encode_2d(&map_w_k, W, L.D, L.V, L.D, BK, BN / L.ctas) ||
      !encode_2d(&map_w_mn, W, L.D, L.V, L.D, 64, BK))
    return GRPO_ERR_CUDA;
  DeviceInfo* di = current_device_info();
  if (di == nullptr) return GRPO_ERR_CUDA;
  const bool overlap = L.n_sbuf == 2;
  const int n_dt_dh = dh_tiles(L.D, L.ctas);
  const int n_rb_total = static_cast<int>(L.nr / BM);
  const int rb_per_chunk = L.chunk_rows / BM;
  const int n_chunks = static_cast<int>(cdiv(n_rb_total, rb_per_chunk));
  auto sbuf = [&](int c) {
    return reinterpret_cast<uint16_t*>(w.G) +
           (overlap ? static_cast<size_t>(c & 1) * L.chunk_rows * L.ldS : 0);
  };
  auto bmax = [&](int c) {
    return reinterpret_cast<float*>(w.base + L.off_bmax) +
           (overlap ? static_cast<size_t>(c & 1) * L.nbox * L.chunk_rows : 0);
  };
  auto chunk_rbs = [&](int c) { return std::min(rb_per_chunk, n_rb_total - c * rb_per_chunk); };
  // dH launches: with the tail split every pair of the launch takes part (the
  // device decides from the active row blocks which units are cut), and a
  // fixup pass adds the cut units' pieces. Without a mask every row block is
  // active, so a unit count of whole rounds is known here to cut nothing. The
  // overlapped schedule splits only its last chunk's launch: before that the
  // next chunk's G pass runs on the pairs that a dH launch's last round leaves
  // idle (measured at the gpt-oss-20b head: splitting every launch made that
  // pass 19 % slower and the call 0.5 %).
  auto dh_grid = [&](long long units, bool split) {
    return L.ctas * (split ? L.ts_slots : static_cast<int>(std::min<long long>(units, slots)));
  };
  auto ts_fixup = [&](const TileArgs& b, long long units) -> int {
    if (b.ts_part == nullptr || (mask == nullptr && units % L.ts_slots == 0)) return GRPO_OK;
    return launch_tail_fixup(L.ctas, b, static_cast<int>(units), false, st) == cudaSuccess
               ? GRPO_OK
               : GRPO_ERR_CUDA;
  };

  // (1) logits of chunk c: online LSE partials, z_y, fp16 copy. The kernel
  // splits the vocabulary for the chunk's active row units (whole waves of
  // the SM pairs); the row finish reads every partial slot.
  auto fwds = [&](int c, int* splits_out) -> int {
    const int n_rb = chunk_rbs(c);
    const int n_ru = static_cast<int>(cdiv(n_rb, L.ctas));
    const int splits = stored_fwd_splits(n_ru, L.nvt, slots, nullptr);
    TileArgs a = base_args(L, w);
    set_transform(&a, prm);
    a.n_total = L.n;
    a.n_rb = n_rb;
    a.rb_offset = c * rb_per_chunk;
    a.seg_list = w.seg_list;
    a.n_seg = w.n_seg;
    a.k_iters = static_cast<int>(cdiv(L.D, BK));
    a.group_rows = fwd_group_rows(n_ru, L.D, L.ctas);
    a.n_cols = splits;
    a.max_cols = std::min(L.nvt, kMaxSplits);
    a.n_vtiles = L.nvt;
    a.v0 = 0;
    a.ids = ids;
    a.mask = mask;
    a.part_m = w.pm;
    a.part_s = w.ps;
    a.zy = w.zy;
    a.part_ld = L.nr;
    a.S = sbuf(c);
    a.ldS = L.ldS;
    a.box_max = bmax(c);
    a.ldM = L.chunk_rows;
    // The pair variant stores each warp's 32 rows x 64 logits through TMA.
    CUtensorMap map_st, map_hc;
    if (!encode_2d(&map_st, a.S, L.V, static_cast<uint64_t>(n_rb) * BM, L.ldS, 64, 32) ||
        !encode_2d(&map_hc, w.hc, L.D, static_cast<uint64_t>(n_rb) * BM, L.D, BK, BM))
      return GRPO_ERR_CUDA;
    // The chunk's non-consecutive row blocks of h, copied for the GEMM.
    a.hc = 1;
    if (launch_gather_blocks(hidden, w.hc, a, st) != cudaSuccess) return GRPO_ERR_CUDA;
    *splits_out = a.max_cols;
    return launch_fwds_gemm(L.ctas, map_h, map_w_k, map_h16, map_st, a, L.ctas * slots, st,
                            &map_hc) == cudaSuccess
               ? GRPO_OK
               : GRPO_ERR_CUDA;
  };
  // (2) per-row finish of chunk c: lse, logp, token loss and g.
  auto row_args = [&](int c, int splits) -> GformArgs {
    const int n_rb = chunk_rbs(c);
    GformArgs f;
    std::memset(&f, 0, sizeof(f));
    f.n_total = L.n;
    f.n_rb = n_rb;
    f.rb_offset = c * rb_per_chunk;
    f.seg_list = w.seg_list;
    f.n_seg = w.n_seg;
    f.splits = splits;
    f.part_ld = L.nr;
    f.vocab = L.V;
    f.seq_len = L.T;
    f.part_m = w.pm;
    f.part_s = w.ps;
    f.zy = w.zy;
    f.ids = ids;
    f.mask = mask;
    f.old_logp = old_logp;
    f.ref_logp = ref_logp;
    f.adv = adv;
    f.eps_low = prm->eps_low;
    f.eps_high = prm->eps_high;
    f.beta = prm->beta;
    f.loss_den = prm->loss_denominator;
    f.msum = w.msum;
    f.seq_mode = (prm->flags & GRPO_FLAG_SEQUENCE_MEAN) != 0;
    f.seq_lens = w.seq_lens;
    f.n_nonempty = w.n_nonempty;
    f.logp_out = logp_out;
    f.lt = w.lt;
    f.S = sbuf(c);
    f.ldS = L.ldS;
    f.box_max = bmax(c);
    f.ldM = L.chunk_rows;
    TileArgs t = base_args(L, w);
    set_transform(&t, prm);
    f.xmode = t.xmode;
    f.k0 = t.k0;
    f.k2 = t.k2;
    f.status = w.status;
    f.lse_out = w.lse;
    f.g_out = w.g;
    return f;
  };
  // (2a) ... and its logit block rewritten in place as G (hidden sizes above
  // kFusedMaxHidden, and dW, which reads G too).
  auto gform = [&](int c, int splits, cudaStream_t s2) -> int {
    return launch_finalize_gform(row_args(c, splits), chunk_rbs(c) * BM, s2) == cudaSuccess
               ? GRPO_OK
               : GRPO_ERR_CUDA;
  };
  // (2b) ... or the row values alone, for the dH GEMM that forms G itself.
  auto rowfin = [&](int c, int splits) -> int {
    return launch_finalize_rows(row_args(c, splits), chunk_rbs(c) * BM, st) == cudaSuccess
               ? GRPO_OK
               : GRPO_ERR_CUDA;
  };
  // (3) dH rows of chunk c = G W over the whole vocabulary; (4) dW.
  auto dh = [&](int c, bool split) -> int {
    const int n_rb = chunk_rbs(c);
    const int n_ru = static_cast<int>(cdiv(n_rb, L.ctas));
    CUtensorMap map_g;
    if (!encode_2d(&map_g, sbuf(c), L.V, static_cast<uint64_t>(n_rb) * BM, L.ldS, BK, BM))
      return GRPO_ERR_CUDA;
    TileArgs b = base_args(L, w);
    b.n_total = L.n;
    b.n_rb = n_rb;
    b.rb_offset = c * rb_per_chunk;
    b.seg_list = w.seg_list;
    b.n_seg = w.n_seg;
    b.k_iters = static_cast<int>(cdiv(L.V, BK));
    b.group_rows = group_rows_for(n_ru, slots);
    b.n_cols = n_dt_dh;
    b.v0 = 0;
    b.dH = static_cast<__nv_bfloat16*>(dH);
    b.first = 1;
    b.last = 1;
    split = split && L.ts_slots > 0;
    b.ts_part = split ? w.sk : nullptr;
    b.ts_slots = split ? L.ts_slots : 0;
    const long long units = static_cast<long long>(n_ru) * n_dt_dh;
    if (launch_dh_gemm(L.ctas, map_g, map_w_mn, b, dh_grid(units, split), st) != cudaSuccess)
      return GRPO_ERR_CUDA;
    if (const int rr = ts_fixup(b, units); rr != GRPO_OK) return rr;
    if (dW != nullptr)
      return launch_dw(hidden, reinterpret_cast<const __nv_bfloat16*>(sbuf(c)), L.ldS, 0, L.V,
                       c * rb_per_chunk, n_rb, dW, c == 0, L, w, sms, st);
    return GRPO_OK;
  };

  // (3') dH rows of chunk c straight from its stored logits: the GEMM's
  // epilogue warps turn each landed A stage into G in shared memory.
  auto dhs = [&](int c) -> int {
    const int n_rb = chunk_rbs(c);
    const int n_ru = static_cast<int>(cdiv(n_rb, L.ctas));
    CUtensorMap map_s;
    if (!encode_2d(&map_s, sbuf(c), L.V, static_cast<uint64_t>(n_rb) * BM, L.ldS, BK, BM))
      return GRPO_ERR_CUDA;
    TileArgs b = base_args(L, w);
    set_transform(&b, prm);
    b.n_total = L.n;
    b.n_rb = n_rb;
    b.rb_offset = c * rb_per_chunk;
    b.seg_list = w.seg_list;
    b.n_seg = w.n_seg;
    b.k_iters = static_cast<int>(cdiv(L.V, BK));
    b.group_rows = group_rows_for(n_ru, slots);
    b.n_cols = n_dt_dh;
    b.v0 = 0;
    b.ids = ids;
    b.lse = w.lse;
    b.g = w.g;
    b.zy = w.zy;
    b.box_max = bmax(c);
    b.ldM = L.chunk_rows;
    b.dH = static_cast<__nv_bfloat16*>(dH);
    b.first = 1;
    b.last = 1;
    const bool split = L.ts_slots > 0;
    b.ts_part = split ? w.sk : nullptr;
    b.ts_slots = split ? L.ts_slots : 0;
    const long long units = static_cast<long long>(n_ru) * n_dt_dh;
    if (launch_dhs_gemm(L.ctas, map_s, map_w_mn, b, dh_grid(units, split), st) != cudaSuccess)
      return GRPO_ERR_CUDA;
    return ts_fixup(b, units);
  };

  int r = GRPO_OK;
  if (dW == nullptr && L.fused) {
    // G never materialises: logits, row values, dH, chunk after chunk on the
    // caller's stream.
    for (int c = 0; c < n_chunks && r == GRPO_OK; ++c) {
      int splits = 1;
      r = fwds(c, &splits);
      if (r == GRPO_OK) r = rowfin(c, splits);
      if (r == GRPO_OK) r = dhs(c);
    }
  } else if (!overlap) {
    for (int c = 0; c < n_chunks && r == GRPO_OK; ++c) {
      int splits = 1;
      r = fwds(c, &splits);
      if (r == GRPO_OK) r = gform(c, splits, st);
      if (r == GRPO_OK) r = dh(c, true);
    }
  } else {
    std::lock_guard<std::mutex> side_lock(di->side_mu);
    // The side stream starts after everything already on the caller's stream.
    if (cudaEventRecord(di->ev_main, st) != cudaSuccess ||
        cudaStreamWaitEvent(di->side, di->ev_main, 0) != cudaSuccess)
      return GRPO_ERR_CUDA;
    auto fwd_then_gform = [&](int c) -> int {
      int splits = 1;
      int rr = fwds(c, &splits);
      if (rr != GRPO_OK) return rr;
      if (cudaEventRecord(di->ev_fwd[c & 1], st) != cudaSuccess ||
          cudaStreamWaitEvent(di->side, di->ev_fwd[c & 1], 0) != cudaSuccess)
        return GRPO_ERR_CUDA;
      rr = gform(c, splits, di->side);
      if (rr != GRPO_OK) return rr;
      return cudaEventRecord(di->ev_g[c & 1], di->side) == cudaSuccess ? GRPO_OK
                                                                        : GRPO_ERR_CUDA;
    };
    r = fwd_then_gform(0);
    for (int c = 0; c < n_chunks && r == GRPO_OK; ++c) {
      if (c + 1 < n_chunks) r = fwd_then_gform(c + 1);  // buffer (c+1)&1: free after dh(c-1)
      if (r != GRPO_OK) break;
      if (cudaStreamWaitEvent(st, di->ev_g[c & 1], 0) != cudaSuccess) return GRPO_ERR_CUDA;
      // Only the last chunk's dH launch has no G pass beside it.
      r = dh(c, c + 1 == n_chunks);
    }
  }  // side_lock released: this call's records and waits are all enqueued
  if (r != GRPO_OK) return r;
  FinishArgs fin;
  std::memset(&fin, 0, sizeof(fin));
  fin.n = L.n;
  fin.mask = mask;
  fin.lt = w.lt;
  fin.logp_out = logp_out;
  fin.block_partials = w.partials;
  fin.counter = w.counter;
  fin.loss_out = loss;
  fin.status = w.status;
  if (launch_finish_loss(fin, st) != cudaSuccess) return GRPO_ERR_CUDA;
  return GRPO_OK;
}

// Single-pass backward of a loss call, chunk by chunk over the active row
// blocks and, within a chunk, vocabulary block by vocabulary block. Per block
// b of chunk c:
//   FWDS(c, b)  the block's logits, once: online LSE partials in slots of
//               their own, z_y, and the block's box-shifted fp16 logits;
//   P(c, b)     (D > kFusedMaxHidden) a row-wise pass rewriting them in place
//               as bf16 P on the side stream, beside the next block's FWDS;
//   U(c, b)     U (+)= P W[block], rescaled to the running maximum: MODE_UAC
//               forms P from the logits on chip, MODE_UAP reads P.
// ROWS(c) finishes each row (lse, logp, token loss, g) once every block's
// partials are in, and the chunk's last U launch turns U into dH. Each logit
// is computed once: 4 N D V flops in all. On the caller's stream:
//   on chip:  FWDS(c,0) U(c,0) ... FWDS(c,nb-1) ROWS(c) U(c,nb-1) ...
//   P pass:   FWDS(0) FWDS(1) U(0) FWDS(2) U(1) ... over the (chunk, block)
//             sequence, with P(i) on the side stream between FWDS(i) and U(i).
int run_single_pass(const void* hidden, const void* W, const int32_t* ids, const uint8_t* mask,
                    const float* old_logp, const float* ref_logp, const float* adv, float* loss,
                    float* logp_out, void* dH, const grpo_params* prm, const Layout& L,
                    const Ws& w, int sms, cudaStream_t st) {
  CUtensorMap map_h, map_h16, map_w_k, map_w_mn;
  const int slots = std::max(1, sms / L.ctas);
  if (!encode_2d(&map_h, hidden, L.D, L.n, L.D, BK, BM) ||
      !encode_2d(&map_h16, hidden, L.D, L.n, L.D, BK, SEG) ||
      !encode_2d(&map_w_k, W, L.D, L.V, L.D, BK, BN / L.ctas) ||
      !encode_2d(&map_w_mn, W, L.D, L.V, L.D, 64, BK))
    return GRPO_ERR_CUDA;
  DeviceInfo* di = current_device_info();
  if (di == nullptr) return GRPO_ERR_CUDA;
  const int n_dt_dh = dh_tiles(L.D, L.ctas);
  const int n_rb_total = static_cast<int>(L.nr / BM);
  const int rb_per_chunk = L.chunk_rows / BM;
  const int n_chunks = static_cast<int>(cdiv(n_rb_total, rb_per_chunk));
  const int n_steps = n_chunks * L.nvb;  // (chunk, block) pairs
  const bool overlap = L.n_sbuf == 2;
  auto chunk_rbs = [&](int c) { return std::min(rb_per_chunk, n_rb_total - c * rb_per_chunk); };
  auto buf = [&](int i) {
    return reinterpret_cast<uint16_t*>(w.G) +
           (overlap ? static_cast<size_t>(i & 1) * L.chunk_rows * L.ldS : 0);
  };
  auto bmax = [&](int i) {
    return reinterpret_cast<float*>(w.base + L.off_bmax) +
           (overlap ? static_cast<size_t>(i & 1) * L.nbox * L.chunk_rows : 0);
  };
  auto width_of = [&](int b) { return std::min(L.vblock, L.V - b * L.vblock); };
  // Forward splits of block b of chunk c, and the partial slots before it.
  auto splits_of = [&](int c, int b) {
    const int n_ru = static_cast<int>(cdiv(chunk_rbs(c), L.ctas));
    return single_pass_fwd_splits(n_ru, static_cast<int>(cdiv(width_of(b), BN)),
                                  kMaxSplits / L.nvb, slots);
  };
  auto slot0_of = [&](int c, int b) {
    int s0 = 0;
    for (int j = 0; j < b; ++j) s0 += splits_of(c, j);
    return s0;
  };
  auto row_args = [&](int c) {
    GformArgs f;
    std::memset(&f, 0, sizeof(f));
    f.n_total = L.n;
    f.n_rb = chunk_rbs(c);
    f.rb_offset = c * rb_per_chunk;
    f.seg_list = w.seg_list;
    f.n_seg = w.n_seg;
    f.part_ld = L.nr;
    f.vocab = L.V;
    f.seq_len = L.T;
    f.part_m = w.pm;
    f.part_s = w.ps;
    f.zy = w.zy;
    f.ids = ids;
    f.mask = mask;
    f.old_logp = old_logp;
    f.ref_logp = ref_logp;
    f.adv = adv;
    f.eps_low = prm->eps_low;
    f.eps_high = prm->eps_high;
    f.beta = prm->beta;
    f.loss_den = prm->loss_denominator;
    f.msum = w.msum;
    f.seq_mode = (prm->flags & GRPO_FLAG_SEQUENCE_MEAN) != 0;
    f.seq_lens = w.seq_lens;
    f.n_nonempty = w.n_nonempty;
    f.logp_out = logp_out;
    f.lt = w.lt;
    f.status = w.status;
    f.lse_out = w.lse;
    f.g_out = w.g;
    f.ldS = L.ldS;
    f.ldM = L.chunk_rows;
    TileArgs t = base_args(L, w);
    set_transform(&t, prm);
    f.xmode = t.xmode;
    f.k0 = t.k0;
    f.k2 = t.k2;
    return f;
  };
  // (1) the logits of step i = (chunk c, block b).
  auto fwds = [&](int i) -> int {
    const int c = i / L.nvb, b = i % L.nvb;
    const int n_rb = chunk_rbs(c);
    const int n_ru = static_cast<int>(cdiv(n_rb, L.ctas));
    const int width = width_of(b);
    const int splits = splits_of(c, b);
    TileArgs a = base_args(L, w);
    set_transform(&a, prm);
    a.n_total = L.n;
    a.n_rb = n_rb;
    a.rb_offset = c * rb_per_chunk;
    a.seg_list = w.seg_list;
    a.n_seg = w.n_seg;
    a.k_iters = static_cast<int>(cdiv(L.D, BK));
    a.group_rows = n_ru;
    a.n_cols = splits;
    a.n_vtiles = static_cast<int>(cdiv(width, BN));
    a.v0 = b * L.vblock;
    a.ids = ids;
    a.mask = mask;
    a.part_m = w.pm;
    a.part_s = w.ps;
    a.zy = w.zy;
    a.part_ld = L.nr;
    a.part_slot0 = slot0_of(c, b);
    a.S = buf(i);
    a.ldS = L.ldS;
    a.box_max = bmax(i);
    a.ldM = L.chunk_rows;
    CUtensorMap map_st, map_hc;
    if (!encode_2d(&map_st, a.S, width, static_cast<uint64_t>(n_rb) * BM, L.ldS, 64, 32) ||
        !encode_2d(&map_hc, w.hc, L.D, static_cast<uint64_t>(n_rb) * BM, L.D, BK, BM))
      return GRPO_ERR_CUDA;
    // The chunk's non-consecutive row blocks of h, copied once before its
    // first block's logit GEMM (the blocks of a chunk run in a row).
    a.hc = 1;
    if (b == 0 && launch_gather_blocks(hidden, w.hc, a, st) != cudaSuccess) return GRPO_ERR_CUDA;
    return launch_fwds_gemm(L.ctas, map_h, map_w_k, map_h16, map_st, a,
                            L.ctas * static_cast<int>(std::min<long long>(
                                         static_cast<long long>(n_ru) * splits, slots)),
                            st, &map_hc) == cudaSuccess
               ? GRPO_OK
               : GRPO_ERR_CUDA;
  };
  // (2) the block's logits rewritten in place as bf16 P (not on chip).
  auto ppass = [&](int i, cudaStream_t s2) -> int {
    const int c = i / L.nvb, b = i % L.nvb;
    GformArgs f = row_args(c);
    f.splits = slot0_of(c, b) + splits_of(c, b);
    f.S = buf(i);
    f.box_max = bmax(i);
    f.v0 = b * L.vblock;
    f.width = width_of(b);
    return launch_single_pass_p(f, chunk_rbs(c) * BM, s2) == cudaSuccess ? GRPO_OK
                                                                          : GRPO_ERR_CUDA;
  };
  // (3) lse, logp, token loss and g of chunk c's rows, after its last block.
  auto rowfin = [&](int c) -> int {
    GformArgs f = row_args(c);
    f.splits = slot0_of(c, L.nvb - 1) + splits_of(c, L.nvb - 1);
    return launch_finalize_rows(f, chunk_rbs(c) * BM, st) == cudaSuccess ? GRPO_OK
                                                                          : GRPO_ERR_CUDA;
  };
  // (4) U (+)= P W[block]; dH on the chunk's last block. With the tail split
  // (split: nothing runs beside the launch) a fixup pass applies the U update
  // to the units it cut.
  auto uacc = [&](int i, bool split) -> int {
    const int c = i / L.nvb, b = i % L.nvb;
    const int n_rb = chunk_rbs(c);
    const int n_ru = static_cast<int>(cdiv(n_rb, L.ctas));
    const int width = width_of(b);
    CUtensorMap map_s;
    if (!encode_2d(&map_s, buf(i), width, static_cast<uint64_t>(n_rb) * BM, L.ldS, BK, BM))
      return GRPO_ERR_CUDA;
    TileArgs u = base_args(L, w);
    set_transform(&u, prm);
    u.n_total = L.n;
    u.n_rb = n_rb;
    u.rb_offset = c * rb_per_chunk;
    u.seg_list = w.seg_list;
    u.n_seg = w.n_seg;
    u.k_iters = static_cast<int>(cdiv(width, BK));
    u.group_rows = group_rows_for(n_ru, slots);
    u.n_cols = n_dt_dh;
    u.v0 = b * L.vblock;
    u.ids = ids;
    u.mask = mask;
    u.lse = w.lse;
    u.g = w.g;
    u.zy = w.zy;
    u.part_m = w.pm;
    u.part_ld = L.nr;
    u.slots_prev = slot0_of(c, b);
    u.slots_cur = u.slots_prev + splits_of(c, b);
    u.W = static_cast<const __nv_bfloat16*>(W);
    u.box_max = bmax(i);
    u.ldM = L.chunk_rows;
    u.acc = w.acc;
    u.dH = static_cast<__nv_bfloat16*>(dH);
    u.first = b == 0;
    u.last = b + 1 == L.nvb;
    split = split && L.ts_slots > 0;
    u.ts_part = split ? w.sk : nullptr;
    u.ts_slots = split ? L.ts_slots : 0;
    const long long units = static_cast<long long>(n_ru) * n_dt_dh;
    const int grid =
        L.ctas * (split ? L.ts_slots : static_cast<int>(std::min<long long>(units, slots)));
    const cudaError_t e = L.fused ? launch_uac_gemm(L.ctas, map_s, map_w_mn, u, grid, st)
                                  : launch_uap_gemm(L.ctas, map_s, map_w_mn, u, grid, st);
    if (e != cudaSuccess) return GRPO_ERR_CUDA;
    if (!split || (mask == nullptr && units % L.ts_slots == 0)) return GRPO_OK;
    return launch_tail_fixup(L.ctas, u, static_cast<int>(units), true, st) == cudaSuccess
               ? GRPO_OK
               : GRPO_ERR_CUDA;
  };

  int r = GRPO_OK;
  if (L.fused || !overlap) {
    for (int i = 0; i < n_steps && r == GRPO_OK; ++i) {
      const int c = i / L.nvb, b = i % L.nvb;
      r = fwds(i);
      if (r == GRPO_OK && !L.fused) r = ppass(i, st);
      if (r == GRPO_OK && b + 1 == L.nvb) r = rowfin(c);
      if (r == GRPO_OK) r = uacc(i, true);
    }
  } else {
    std::lock_guard<std::mutex> side_lock(di->side_mu);
    // The side stream starts after everything already on the caller's stream.
    if (cudaEventRecord(di->ev_main, st) != cudaSuccess ||
        cudaStreamWaitEvent(di->side, di->ev_main, 0) != cudaSuccess)
      return GRPO_ERR_CUDA;
    auto fwd_then_p = [&](int i) -> int {
      int rr = fwds(i);
      if (rr != GRPO_OK) return rr;
      if (cudaEventRecord(di->ev_fwd[i & 1], st) != cudaSuccess ||
          cudaStreamWaitEvent(di->side, di->ev_fwd[i & 1], 0) != cudaSuccess)
        return GRPO_ERR_CUDA;
      rr = ppass(i, di->side);
      if (rr != GRPO_OK) return rr;
      return cudaEventRecord(di->ev_g[i & 1], di->side) == cudaSuccess ? GRPO_OK
                                                                        : GRPO_ERR_CUDA;
    };
    r = fwd_then_p(0);
    for (int i = 0; i < n_steps && r == GRPO_OK; ++i) {
      // Block (i+1) & 1 was last read by U(i-1), enqueued before this FWDS.
      if (i + 1 < n_steps) r = fwd_then_p(i + 1);
      if (r != GRPO_OK) break;
      if (cudaStreamWaitEvent(st, di->ev_g[i & 1], 0) != cudaSuccess) return GRPO_ERR_CUDA;
      if (i % L.nvb + 1 == L.nvb) r = rowfin(i / L.nvb);
      if (r == GRPO_OK) r = uacc(i, false);
    }
  }  // side_lock released: this call's records and waits are all enqueued
  if (r != GRPO_OK) return r;
  FinishArgs fin;
  std::memset(&fin, 0, sizeof(fin));
  fin.n = L.n;
  fin.mask = mask;
  fin.lt = w.lt;
  fin.logp_out = logp_out;
  fin.block_partials = w.partials;
  fin.counter = w.counter;
  fin.loss_out = loss;
  fin.status = w.status;
  if (launch_finish_loss(fin, st) != cudaSuccess) return GRPO_ERR_CUDA;
  return GRPO_OK;
}

}  // namespace

// ---- Opt-in per-launch timing ------------------------------------------------
namespace {

constexpr size_t kMaxTimedLaunches = size_t(1) << 16;  // records kept between reads

struct TimedLaunch {
  char name[sizeof(grpo_kernel_time::name)];
  int device;
  cudaEvent_t start, stop;
  bool complete;  // both events recorded
};

// Per host thread: the switch, the launches recorded since the last read and
// a per-device pool of events for reuse (an event records only on streams of
// the device it was created on).
struct TimingState {
  bool on = false;
  std::vector<TimedLaunch> pending;
  std::vector<cudaEvent_t> pool[kMaxDevices];

  cudaEvent_t take(int dev) {
    if (!pool[dev].empty()) {
      cudaEvent_t e = pool[dev].back();
      pool[dev].pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    return e;
  }
  void give(int dev, cudaEvent_t e) {
    if (e != nullptr) pool[dev].push_back(e);
  }
  void release_pool() {
    for (auto& p : pool) {
      for (cudaEvent_t e : p) (void)cudaEventDestroy(e);
      p.clear();
    }
  }
  ~TimingState() {
    for (TimedLaunch& r : pending) {
      (void)cudaEventDestroy(r.start);
      (void)cudaEventDestroy(r.stop);
    }
    release_pool();
  }
};

thread_local TimingState t_timing;

}  // namespace

bool launch_timing_on() { return t_timing.on; }

void LaunchTimer::begin(const char* name, cudaStream_t stream) {
  TimingState& st = t_timing;
  if (st.pending.size() >= kMaxTimedLaunches) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    return;
  }
  if (cs != cudaStreamCaptureStatusNone) return;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return;
  }
  TimedLaunch r = {};
  std::snprintf(r.name, sizeof(r.name), "%s", name);
  r.device = dev;
  r.start = st.take(dev);
  r.stop = st.take(dev);
  if (r.start == nullptr || r.stop == nullptr || cudaEventRecord(r.start, stream) != cudaSuccess) {
    (void)cudaGetLastError();  // keep the launcher's own error check clean
    st.give(dev, r.start);
    st.give(dev, r.stop);
    return;
  }
  st.pending.push_back(r);
  slot_ = static_cast<int>(st.pending.size() - 1);
  stream_ = stream;
}

LaunchTimer::LaunchTimer(const char* name, cudaStream_t stream) {
  if (t_timing.on) begin(name, stream);
}

LaunchTimer::LaunchTimer(int mode, int ctas, cudaStream_t stream) {
  if (!t_timing.on) return;
  char name[sizeof(grpo_kernel_time::name)];
  std::snprintf(name, sizeof(name), "tc_gemm_kernel<%d, %d>", mode, ctas);
  begin(name, stream);
}

LaunchTimer::~LaunchTimer() {
  if (slot_ < 0) return;
  TimedLaunch& r = t_timing.pending[static_cast<size_t>(slot_)];
  if (cudaEventRecord(r.stop, stream_) == cudaSuccess) {
    r.complete = true;
  } else {
    (void)cudaGetLastError();
  }
}

}  // namespace grpo

using namespace grpo;

extern "C" {

void grpo_default_params(grpo_params* p) {
  if (!p) return;
  std::memset(p, 0, sizeof(*p));
  p->eps_low = 0.2f;
  p->eps_high = 0.2f;
  p->beta = 0.001f;
  p->loss_denominator = 0.f;
}

int grpo_workspace_size(const grpo_shape* shape, const grpo_params* params, size_t* bytes) {
  if (!bytes) return GRPO_ERR_INVALID_ARG;
  int r = check_shape(shape, false);
  if (r != GRPO_OK) return r;
  if ((r = check_params(params)) != GRPO_OK) return r;
  Layout L;
  if ((r = make_layout(shape, params, 0, &L)) != GRPO_OK) return r;
  *bytes = L.total;
  return GRPO_OK;
}

int grpo_logp_fwd(const void* hidden, const void* W, const int32_t* ids, float* logp,
                  float* lse_or_null, const grpo_shape* shape, const grpo_params* params,
                  void* workspace, size_t workspace_bytes, void* stream) {
  const NvtxRange range("grpo_logp_fwd");
  int r = check_shape(shape, false);
  if (r != GRPO_OK) return r;
  if ((r = check_params(params)) != GRPO_OK) return r;
  if (shape->n_tokens > 0 && (!hidden || !W || !ids || !logp || !workspace))
    return GRPO_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(W, 16) || !aligned(workspace, 256) || !aligned(ids, 4) ||
      !aligned(logp, 4) || !aligned(lse_or_null, 4))
    return GRPO_ERR_MISALIGNED;
  int sms = 0;
  if ((r = device_setup(&sms)) != GRPO_OK) return r;
  Layout L;
  if ((r = make_layout(shape, params, sms, &L)) != GRPO_OK) return r;
  // The forward uses the workspace only up to the backward's G block.
  if (workspace_bytes < L.off_G) return GRPO_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, 64, st) != cudaSuccess) return GRPO_ERR_CUDA;
  if (L.n == 0) return GRPO_OK;
  Ws w = carve(workspace, L);
  int splits = 1;
  if ((r = run_forward(hidden, W, ids, nullptr, nullptr, nullptr, params, L, w, sms, &splits, st)) != GRPO_OK) return r;
  FinalizeArgs f;
  std::memset(&f, 0, sizeof(f));
  f.n = L.n;
  f.splits = splits;
  f.part_ld = L.nr;
  f.vocab = L.V;
  f.seq_len = 1;
  f.loss_mode = 0;
  f.part_m = w.pm;
  f.part_s = w.ps;
  f.zy = w.zy;
  f.ids = ids;
  f.lse_ws = w.lse;
  f.lse_out = lse_or_null;
  f.logp_out = logp;
  f.status = w.status;
  if (launch_finalize(f, st) != cudaSuccess) return GRPO_ERR_CUDA;
  return GRPO_OK;
}

int grpo_loss_fwd_bwd(const void* hidden, const void* W, const int32_t* ids,
                      const uint8_t* mask, const float* old_logp, const float* ref_logp,
                      const float* adv, float* loss, float* logp_or_null, void* dH,
                      float* dW_or_null, const grpo_shape* shape, const grpo_params* params,
                      void* workspace, size_t workspace_bytes, void* stream) {
  const NvtxRange range("grpo_loss_fwd_bwd");
  int r = check_shape(shape, true);
  if (r != GRPO_OK) return r;
  if ((r = check_params(params)) != GRPO_OK) return r;
  if (!loss || !workspace) return GRPO_ERR_INVALID_ARG;
  if (shape->n_tokens > 0 &&
      (!hidden || !W || !ids || !old_logp || !ref_logp || !adv || !dH))
    return GRPO_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(W, 16) || !aligned(dH, 16) || !aligned(workspace, 256) ||
      !aligned(ids, 4) || !aligned(old_logp, 4) || !aligned(ref_logp, 4) || !aligned(adv, 4) ||
      !aligned(loss, 4) || !aligned(logp_or_null, 4) || !aligned(dW_or_null, 16))
    return GRPO_ERR_MISALIGNED;
  grpo_params prm;
  if (params) prm = *params; else grpo_default_params(&prm);
  int sms = 0;
  if ((r = device_setup(&sms)) != GRPO_OK) return r;
  Layout L;
  if ((r = make_layout(shape, &prm, sms, &L)) != GRPO_OK) return r;
  Layout Lmax;
  make_layout(shape, &prm, 0, &Lmax);
  if (workspace_bytes < std::max(L.total, Lmax.total)) return GRPO_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, 64, st) != cudaSuccess) return GRPO_ERR_CUDA;
  if (L.n == 0) {
    if (cudaMemsetAsync(loss, 0, sizeof(float), st) != cudaSuccess) return GRPO_ERR_CUDA;
    if (dW_or_null != nullptr &&
        cudaMemsetAsync(dW_or_null, 0, static_cast<size_t>(L.V) * L.D * sizeof(float), st) !=
            cudaSuccess)
      return GRPO_ERR_CUDA;
    return GRPO_OK;
  }
  Ws w = carve(workspace, L);
  const int n_rb_total = static_cast<int>(L.nr / BM);
  if (launch_row_plan(mask, L.n, static_cast<int>(L.nr / SEG), w.seg_list, w.n_seg, w.msum, st) !=
          cudaSuccess ||
      launch_zero_padding_blocks(mask, L.n, n_rb_total, L.D, dH, sms, st) != cudaSuccess)
    return GRPO_ERR_CUDA;
  if ((prm.flags & GRPO_FLAG_SEQUENCE_MEAN) != 0 &&
      launch_seq_lens(mask, L.n, L.T, w.seq_lens, w.n_nonempty, st) != cudaSuccess)
    return GRPO_ERR_CUDA;
  if (L.stored)
    return run_stored(hidden, W, ids, mask, old_logp, ref_logp, adv, loss, logp_or_null, dH,
                      dW_or_null, &prm, L, w, sms, st);
  if (L.single_pass && dW_or_null == nullptr)
    return run_single_pass(hidden, W, ids, mask, old_logp, ref_logp, adv, loss, logp_or_null, dH,
                           &prm, L, w, sms, st);
  if (L.single_pass) {
    // The lm_head gradient needs G explicitly, which the single pass never
    // forms: recompute the logit tiles instead, with the same chunk and vocab
    // block, whose workspace lies within the single pass's.
    grpo_params p2 = prm;
    p2.flags = (p2.flags & ~GRPO_FLAG_SINGLE_PASS) | GRPO_FLAG_RECOMPUTE_LOGITS;
    p2.chunk_tokens = L.chunk_rows;
    p2.vocab_block = L.vblock;
    p2.workspace_limit_bytes = 0;
    Layout L2;
    if ((r = make_layout_mode(shape, &p2, sms, kFormRecompute, &L2)) != GRPO_OK) return r;
    if (L2.total > workspace_bytes) return GRPO_ERR_WORKSPACE_TOO_SMALL;
    L = L2;
    w = carve(workspace, L);
  }
  int splits = 1;
  if ((r = run_forward_chunks(hidden, W, ids, mask, &prm, L, w, sms, &splits,
                       st)) != GRPO_OK)
    return r;
  FinalizeArgs f;
  std::memset(&f, 0, sizeof(f));
  f.n = L.n;
  f.splits = splits;
  f.part_ld = L.nr;
  f.vocab = L.V;
  f.seq_len = L.T;
  f.loss_mode = 1;
  f.part_m = w.pm;
  f.part_s = w.ps;
  f.zy = w.zy;
  f.ids = ids;
  f.mask = mask;
  f.old_logp = old_logp;
  f.ref_logp = ref_logp;
  f.adv = adv;
  f.eps_low = prm.eps_low;
  f.eps_high = prm.eps_high;
  f.beta = prm.beta;
  f.loss_den = prm.loss_denominator;
  f.msum = w.msum;
  f.seq_mode = (prm.flags & GRPO_FLAG_SEQUENCE_MEAN) != 0;
  f.seq_lens = w.seq_lens;
  f.n_nonempty = w.n_nonempty;
  f.lse_ws = w.lse;
  f.logp_out = logp_or_null;
  f.g_ws = w.g;
  f.block_partials = w.partials;
  f.counter = w.counter;
  f.loss_out = loss;
  f.status = w.status;
  if (launch_finalize(f, st) != cudaSuccess) return GRPO_ERR_CUDA;
  return run_backward(hidden, W, ids, dH, dW_or_null, &prm, L, w, sms, st);
}

int grpo_get_plan(const grpo_shape* shape, const grpo_params* params, grpo_plan_info* info) {
  if (!info) return GRPO_ERR_INVALID_ARG;
  int r = check_shape(shape, false);
  if (r != GRPO_OK) return r;
  if ((r = check_params(params)) != GRPO_OK) return r;
  int sms = 0;
  if ((r = device_setup(&sms)) != GRPO_OK) return r;
  Layout L, Lmax;
  if ((r = make_layout(shape, params, sms, &L)) != GRPO_OK) return r;
  make_layout(shape, params, 0, &Lmax);
  std::memset(info, 0, sizeof(*info));
  info->chunk_rows = L.chunk_rows;
  info->vocab_block = L.vblock;
  info->n_chunks = static_cast<int32_t>(cdiv(L.n, L.chunk_rows));
  info->n_vocab_blocks = static_cast<int32_t>(cdiv(L.V, L.vblock));
  const int n_rb = static_cast<int>(L.nr / BM);
  const int slots = std::max(1, sms / L.ctas);
  int group = 1;
  whole_batch_raster(static_cast<int>(cdiv(n_rb, L.ctas)), L.nvt, L.D, L.ctas, slots, &group,
                     &info->fwd_splits);
  info->launches_logp = L.n > 0 ? 2 : 0;
  // Tail-split dH-type launches (the stored form's fused dH GEMM, chunks that
  // run one after another, or the overlapped schedule's last chunk; the single
  // pass's U GEMMs that nothing runs beside) are each followed by a fixup pass.
  const bool tail_split = L.ts_slots > 0 && (L.fused || L.n_sbuf == 1);
  const int stored_fixups = L.ts_slots == 0 ? 0 : tail_split ? info->n_chunks : 1;
  // Every form gathers each chunk's non-consecutive row blocks of h once.
  info->launches_loss = L.n <= 0        ? 0
                        : L.stored      ? 3 + 4 * info->n_chunks + stored_fixups
                        : L.single_pass ? 3 + info->n_chunks *
                                                  (((L.fused ? 2 : 3) + (tail_split ? 1 : 0)) *
                                                       L.nvb +
                                                   2)
                                        : 3 + (2 * info->n_vocab_blocks + 3) * info->n_chunks;
  if (L.n > 0 && params != nullptr && (params->flags & GRPO_FLAG_SEQUENCE_MEAN) != 0)
    info->launches_loss += 1;
  if (L.stored) info->n_vocab_blocks = 1;
  // The loss call's forward of the stored and recomputed forms runs per chunk
  // (with padding, the kernels set the splits from the active rows).
  if (!L.single_pass)
    info->fwd_splits =
        stored_fwd_splits(L.chunk_rows / (BM * L.ctas), L.nvt, slots, nullptr);
  info->g_in_dh_gemm = L.fused ? 1 : 0;
  info->stored_logits = L.stored ? 1 : 0;
  info->single_pass = L.single_pass ? 1 : 0;
  info->workspace_bytes = std::max(L.total, Lmax.total);
  return GRPO_OK;
}

int grpo_read_device_status(const void* workspace, int* device_status, void* stream) {
  if (!workspace || !device_status) return GRPO_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return GRPO_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, static_cast<const uint8_t*>(workspace) + kOffStatus, sizeof(int),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return GRPO_ERR_CUDA;
  *device_status = v;
  return GRPO_OK;
}

int grpo_selftest_bounded_wait(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < 64) return GRPO_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return GRPO_ERR_MISALIGNED;
  int sms = 0;
  int r = device_setup(&sms);
  if (r != GRPO_OK) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  if (cudaMemsetAsync(workspace, 0, 64, st) != cudaSuccess) return GRPO_ERR_CUDA;
  if (launch_bounded_wait_selftest(reinterpret_cast<int*>(base + kOffStatus),
                                   reinterpret_cast<int*>(base + kOffCounter), st) !=
      cudaSuccess)
    return GRPO_ERR_CUDA;
  return GRPO_OK;
}

int grpo_launch_timing_enable(int on) {
  t_timing.on = on != 0;
  if (!t_timing.on && t_timing.pending.empty()) t_timing.release_pool();
  return GRPO_OK;
}

int grpo_launch_timing_read(grpo_kernel_time* out, int capacity, int* count) {
  if (count == nullptr || capacity < 0 || (capacity > 0 && out == nullptr)) {
    return GRPO_ERR_INVALID_ARG;
  }
  TimingState& st = t_timing;
  std::vector<grpo_kernel_time> agg;
  int rc = GRPO_OK;
  int prev_dev = -1;
  if (!st.pending.empty() && cudaGetDevice(&prev_dev) != cudaSuccess) {
    (void)cudaGetLastError();
    prev_dev = -1;
  }
  for (TimedLaunch& r : st.pending) {
    float ms = 0.0f;
    cudaError_t e = r.complete ? cudaSuccess : cudaErrorNotReady;
    if (e == cudaSuccess) e = cudaSetDevice(r.device);
    if (e == cudaSuccess) e = cudaEventSynchronize(r.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
    if (e == cudaSuccess) {
      auto it = std::find_if(agg.begin(), agg.end(), [&](const grpo_kernel_time& k) {
        return std::strncmp(k.name, r.name, sizeof(k.name)) == 0;
      });
      if (it == agg.end()) {
        grpo_kernel_time k = {};
        std::memcpy(k.name, r.name, sizeof(k.name));
        agg.push_back(k);
        it = agg.end() - 1;
      }
      it->launches += 1;
      it->total_ms += ms;
    } else if (r.complete) {
      (void)cudaGetLastError();
      rc = GRPO_ERR_CUDA;
    }
    st.give(r.device, r.start);
    st.give(r.device, r.stop);
  }
  st.pending.clear();
  if (prev_dev >= 0) (void)cudaSetDevice(prev_dev);
  if (!st.on) st.release_pool();
  *count = static_cast<int>(agg.size());
  const int n = std::min(capacity, static_cast<int>(agg.size()));
  for (int i = 0; i < n; ++i) out[i] = agg[static_cast<size_t>(i)];
  return rc;
}

const char* grpo_status_string(int s) {
  switch (s) {
    case GRPO_OK: return "ok";
    case GRPO_ERR_INVALID_ARG: return "invalid argument";
    case GRPO_ERR_MISALIGNED: return "pointer not aligned (hidden/W/dH need 16 bytes, workspace 256)";
    case GRPO_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (hidden % 8, N % seq_len, or too large)";
    case GRPO_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case GRPO_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103 / GB300)";
    case GRPO_ERR_CUDA: return "CUDA runtime or driver error";
    case GRPO_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case GRPO_ERR_BAD_TOKEN_ID: return "token id outside [0, vocab) on an unmasked row";
    case GRPO_ERR_NONFINITE: return "log-sum-exp of a row is not finite (inf/NaN inputs)";
    default: return "unknown status";
  }
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Workspace-free forward for callers that cannot allocate device memory (see
// grpo_logp_fwd_noalloc in the header). Its scratch is this file-scope device
// array; host code reaches it only through the address that
// cudaGetSymbolAddress returns for the current device (the array's name on the
// host is a stand-in, not a device address).
static __device__ __align__(256) unsigned char g_grpo_noalloc_scratch[GRPO_NOALLOC_SCRATCH_BYTES];

namespace grpo {
namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the static scratch on the current device; looked up once
// per device, with that device current.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GRPO_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GRPO_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_grpo_noalloc_scratch) != cudaSuccess || p == nullptr)
      return GRPO_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return GRPO_OK;
}

}  // namespace
}  // namespace grpo

extern "C" int grpo_logp_fwd_noalloc(const void* hidden, const void* W, const int32_t* ids,
                                     float* logp, float* lse_or_null, const grpo_shape* shape,
                                     void* stream) {
  const NvtxRange range("grpo_logp_fwd_noalloc");
  int r = check_shape(shape, false);
  if (r != GRPO_OK) return r;
  if (shape->n_tokens > GRPO_NOALLOC_MAX_TOKENS) return GRPO_ERR_UNSUPPORTED_SHAPE;
  if (shape->n_tokens > 0 && (!hidden || !W || !ids || !logp)) return GRPO_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(W, 16) || !aligned(ids, 4) || !aligned(logp, 4) ||
      !aligned(lse_or_null, 4))
    return GRPO_ERR_MISALIGNED;
  int sms = 0;
  if ((r = device_setup(&sms)) != GRPO_OK) return r;
  Layout L;
  if ((r = make_layout(shape, nullptr, sms, &L)) != GRPO_OK) return r;
  // The forward uses the workspace only up to the backward's part (the tail
  // split's slots, then the chunk block), which depends on the vocabulary.
  if (L.off_sk > GRPO_NOALLOC_SCRATCH_BYTES) return GRPO_ERR_UNSUPPORTED_SHAPE;
  void* scratch = nullptr;
  if ((r = noalloc_scratch(&scratch)) != GRPO_OK) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Status word and reduction counter must start at zero; the rest is fully
  // overwritten before it is read.
  if (cudaMemsetAsync(scratch, 0, 64, st) != cudaSuccess) return GRPO_ERR_CUDA;
  if (L.n == 0) return GRPO_OK;
  Ws w = carve(scratch, L);
  w.G = nullptr;  // beyond the forward's part of the scratch; never used here
  w.acc = nullptr;
  w.sk = nullptr;
  w.hc = nullptr;
  int splits = 1;
  if ((r = run_forward(hidden, W, ids, nullptr, nullptr, nullptr, nullptr, L, w, sms, &splits, st)) != GRPO_OK) return r;
  FinalizeArgs f;
  std::memset(&f, 0, sizeof(f));
  f.n = L.n;
  f.splits = splits;
  f.part_ld = L.nr;
  f.vocab = L.V;
  f.seq_len = 1;
  f.loss_mode = 0;
  f.part_m = w.pm;
  f.part_s = w.ps;
  f.zy = w.zy;
  f.ids = ids;
  f.lse_ws = w.lse;
  f.lse_out = lse_or_null;
  f.logp_out = logp;
  f.status = w.status;
  if (launch_finalize(f, st) != cudaSuccess) return GRPO_ERR_CUDA;
  return GRPO_OK;
}
