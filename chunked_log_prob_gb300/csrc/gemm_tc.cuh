// Persistent, warp-specialised tcgen05 GEMM for sm_103a with fused
// epilogues. One CTA per SM, 192 threads (320 for MODE_DHS and MODE_UAC):
//   warp 0      TMA producer (one elected thread) filling the smem stage ring
//   warp 1      TMEM allocator + MMA issuer (one elected thread)
//   warps 2..5  epilogue: 128 threads <-> the 128 TMEM lanes (= tile rows)
//   warps 6..9  MODE_DHS, MODE_UAC: converter warps (the second half of each row)
// The fp32 accumulator lives in TMEM, double buffered (2 x 256 columns), so
// the epilogue of tile j overlaps the MMAs of tile j+1.
//
// Tile: 128 rows x 256 columns, K step 64 (one 128-byte swizzle atom of
// bf16). Modes:
//   MODE_FWD   S = H W^T over a run of vocab tiles; epilogue keeps an online
//              max / sum-exp per row (base-2 domain) and picks the target logit.
//   MODE_BWDG  S = H W^T for one vocab tile; epilogue writes
//              G = g (onehot(y) - exp(S - lse)) in bf16 to the chunk workspace.
//   MODE_DH    dH_tile (+)= G W over one vocab block (B operand MN-major);
//              epilogue accumulates in fp32 and writes bf16 on the last block.
//   MODE_DW    dW[v0 + m, n] (+)= sum over the chunk's rows of G[row, m] H[row, n]:
//              the lm_head gradient; A (G^T) and B (H) are both MN-major, K runs
//              over the chunk's active row blocks; fp32 accumulation on the
//              output across chunks.
//   MODE_FWDS  MODE_FWD over the rows of one backward chunk that also stores
//              the (transformed) logits in fp16 to the chunk workspace, for a
//              backward that needs no second logit GEMM.
// On CTA pairs, MODE_FWDS, MODE_BWDG and MODE_DW write their outputs through
// shared memory and TMA stores (MODE_DW: TMA reduce-adds after the first
// chunk), in whole 128-byte lines.
//   MODE_DHS   MODE_DH whose A operand is that stored fp16 logit block: the
//              epilogue warps, idle during the long vocabulary K loop, and four
//              converter-only warps rewrite each landed A stage in place as
//              bf16 G (the softmax-Jacobian row, scaled by dL/dlogp) before the
//              MMA reads it, so G never goes through HBM.
//   MODE_UAC   the single-pass backward's second GEMM over one vocabulary block:
//              like MODE_DHS, but the landed logits become P_v = 2^(z'_v log2e
//              - M) f'(S_v) (M the row's running maximum after this block, the
//              target column excluded), and the epilogue keeps the fp32
//              accumulator U = sum_v P_v W_v across blocks, rescaled by
//              2^(M_prev - M) whenever the maximum grows; the last block turns
//              it into dH = g (1 - p_y) f'_y W_y - g 2^(M - lse2) U.
//   MODE_UAP   MODE_UAC for hidden sizes above 2048: the block's P was formed
//              by a row-wise pass of its own, so A arrives through TMA as bf16
//              like MODE_DH's G, and no converter warps run.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace grpo {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
// Rows of a segment of the active-row list: a loss call computes the 16-row
// segments that hold any unmasked row, packed into row blocks of kSegs
// segments, so that trailing padding costs at most 15 rows per completion
// rather than a part-filled 128-row block.
constexpr int SEG = 16;
constexpr int kSegs = BM / SEG;
constexpr int STAGES = 4;                 // pipeline depth of the single-CTA kernels
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int GEMM_THREADS = 192;
constexpr int TMEM_COLS = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum GemmMode { MODE_FWD = 0, MODE_BWDG = 1, MODE_DH = 2, MODE_FWDS = 3, MODE_DW = 4,
                MODE_DHS = 5, MODE_UAC = 6, MODE_UAP = 7 };

__host__ __device__ constexpr bool is_fwd(int mode) { return mode == MODE_FWD || mode == MODE_FWDS; }
__host__ __device__ constexpr bool is_dh(int mode) {
  return mode == MODE_DH || mode == MODE_DHS || mode == MODE_UAC || mode == MODE_UAP;
}
// dH-type modes whose A operand arrives ready for the MMA (bf16 G or P via TMA).
__host__ __device__ constexpr bool is_dh_plain(int mode) {
  return mode == MODE_DH || mode == MODE_UAP;
}
// Modes whose epilogue keeps the single pass's U accumulator.
__host__ __device__ constexpr bool is_uacc(int mode) { return mode == MODE_UAC || mode == MODE_UAP; }
// Modes whose A operand is stored fp16 logits, converted on chip before the MMA.
__host__ __device__ constexpr bool has_cvt(int mode) { return mode == MODE_DHS || mode == MODE_UAC; }

struct TileArgs {
  long long n_total;     // N: rows of hidden / dH; global rows >= N are padding
  int n_rb;              // row blocks this launch may cover (host-side bound)
  int rb_offset;         // the launch's first row block (of kSegs list entries each)
  const int* seg_list;   // global indices of the active 16-row segments, in order,
                         // or null (then local row r is global row rb_offset*BM + r)
  const int* n_seg;      // device-side length of seg_list, or null (= all)
  // The launch's row blocks whose segments are not consecutive rows were
  // copied into a chunk-sized copy of h (gather_blocks_kernel; map_hc, rows
  // li * BM..): read them from there in one box. 0: read those blocks from h
  // in boxes of SEG rows (map_h16).
  int hc;
  int k_iters;     // ceil(K / BK)
  int group_rows;  // row blocks per raster group
  int n_cols;      // FWD: vocab splits; BWDG: vocab tiles in block; DH: D tiles
  int max_cols;    // FWD, FWDS: > 0: the kernel sets the vocab splits (at most this
                   // many) from its active row units, and each row's split 0
                   // fills the row's unused partial slots below it with (-inf, 0)
  int n_vtiles;    // FWD: vocab tiles in total
  int v0;          // BWDG/DH: first vocab column of the block (0 for FWD)
  int vocab;
  int hidden;
  // Logit transform z' = f(S) applied before the log-softmax (FWD, BWDG):
  //   xmode 0: z' = S;  1: z' = k0 S;  2: z' = k2 tanh(k1 S), f'(S) = k0 (1 - tanh^2)
  int xmode;
  float k0, k1, k2;
  const int32_t* ids;    // indexed by global row
  const uint8_t* mask;   // FWD: optional; masked rows' ids are never read
  // MODE_FWD (written; MODE_UAC reads part_m)
  float* part_m;         // [slots][part_ld] running max (log2 units)
  float* part_s;         // [slots][part_ld] running sum of 2^(x - max)
  float* zy;             // [N] target logit, indexed by global row
  long long part_ld;
  int part_slot0;        // slot of this launch's first vocab split
  // MODE_UAC: the split partials of the blocks so far (slots_cur) and before
  // this block (slots_prev) give the row's running maximum now and before;
  // W (bf16 [V][hidden]) gives W_y on the last block.
  int slots_cur, slots_prev;
  const __nv_bfloat16* W;
  // MODE_BWDG, MODE_DHS
  const float* lse;      // indexed by global row
  const float* g;        // indexed by global row
  __nv_bfloat16* G;      // [local rows][ldG] chunk workspace
  long long ldG;
  // MODE_FWDS (written), MODE_DHS (read)
  uint16_t* S;           // [local rows][ldS] fp16 logits of the chunk, each 64-column
                         // box stored relative to its own maximum, in log2 units
  long long ldS;
  float* box_max;        // [ceil(V / 64)][ldM] those maxima times log2 e (fp32), box-major
  long long ldM;         // rows of the chunk block (stride between boxes)
  // MODE_DW
  float* dW;             // [V][hidden] fp32 output / accumulator
  int dw_rows;           // vocab rows of dW this launch covers (from v0)
  // MODE_DH, MODE_DHS, MODE_UAC
  float* acc;            // [local rows][hidden] fp32 accumulator
  __nv_bfloat16* dH;     // [N][hidden] output, indexed by global row
  int first;
  int last;
  // MODE_DH, MODE_DHS over the whole vocabulary (first and last): the tail
  // split of the last round (see TailSplit). ts_part: 2 slots per SM pair of
  // fp32 partial tiles, or null (units run whole, one per pair and round);
  // ts_slots: the pairs of the launch (its grid / CTAS), which the fixup
  // kernel must be given too.
  float* ts_part;
  int ts_slots;
  int* status;
};

__device__ __forceinline__ void decode_unit(int u, int n_rb, int n_cols, int R, int& rb,
                                            int& col) {
  const int per_group = R * n_cols;
  const int grp = u / per_group;
  const int rem = u - grp * per_group;
  const int rows_in_g = min(R, n_rb - grp * R);
  col = rem / rows_in_g;
  rb = grp * R + (rem - col * rows_in_g);
}

// True when every segment of the batch is active: the list (ascending) is
// then the identity, and a row's place needs no lookup.
__device__ __forceinline__ bool all_segs_active(const TileArgs& a, int n) {
  return static_cast<long long>(n) * SEG >= a.n_total;
}

// Global row of the launch's local row `lr` (row lr % BM of its local row
// block lr / BM), or -1 past the active list.
__device__ __forceinline__ long long row_of(const TileArgs& a, int lr) {
  if (a.seg_list == nullptr) return static_cast<long long>(a.rb_offset) * BM + lr;
  const int s = a.rb_offset * kSegs + lr / SEG;
  if (a.n_seg != nullptr) {
    const int n = *a.n_seg;
    if (s >= n) return -1;
    if (all_segs_active(a, n)) return static_cast<long long>(a.rb_offset) * BM + lr;
  }
  return static_cast<long long>(a.seg_list[s]) * SEG + lr % SEG;
}

// Row blocks this launch actually covers (the active list may be shorter
// than the host-side bound).
__device__ __forceinline__ int launch_row_blocks(const TileArgs& a) {
  if (a.n_seg == nullptr) return a.n_rb;
  const int segs = *a.n_seg - a.rb_offset * kSegs;
  return max(0, min(a.n_rb, (segs + kSegs - 1) / kSegs));
}

// Rows of the hidden states that local row block `li` reads, for the TMA
// loads of h: rows[j] is the first row of its j-th segment (past the list:
// n_total, a coordinate the load fills with zeros). Returns true when the
// segments are consecutive rows, so that one box of BM rows at rows[0] loads
// the block; otherwise each segment is a box of SEG rows of its own.
__device__ __forceinline__ bool h_rows(const TileArgs& a, int li, int (&rows)[kSegs]) {
  if (a.seg_list == nullptr) {
#pragma unroll
    for (int j = 0; j < kSegs; ++j) rows[j] = (a.rb_offset + li) * BM + j * SEG;
    return true;
  }
  const int s0 = (a.rb_offset + li) * kSegs;
  const int n = a.n_seg != nullptr ? *a.n_seg : s0 + kSegs;
  if (a.n_seg != nullptr && all_segs_active(a, n)) {
    // Rows past the batch read as zeros (the load's fill), as past the list.
#pragma unroll
    for (int j = 0; j < kSegs; ++j) rows[j] = s0 * SEG + j * SEG;
    return true;
  }
  bool consecutive = true;
#pragma unroll
  for (int j = 0; j < kSegs; ++j) {
    rows[j] = s0 + j < n ? a.seg_list[s0 + j] * SEG : static_cast<int>(a.n_total);
    consecutive = consecutive && rows[j] == rows[0] + j * SEG;
  }
  return consecutive;
}

// Vocab splits of a logit GEMM launch over n_ru row units: the count (at most
// cap) whose units fill the slots' rounds best, the longest split setting the
// pace; ties go to fewer splits. Exact integer comparison of
// units / (rounds * slots) * (nvt / sp) / ceil(nvt / sp).
__device__ __forceinline__ int fwd_splits_for(int n_ru, int nvt, int slots, int cap) {
  int best = 1;
  long long bn = 0, bd = 1;  // best efficiency as bn / bd
  const int hi = min(nvt, cap);
  for (int sp = 1; sp <= hi; ++sp) {
    const long long units = static_cast<long long>(n_ru) * sp;
    const long long rounds = (units + slots - 1) / slots;
    const long long per = (nvt + sp - 1) / sp;
    const long long num = units * nvt, den = rounds * slots * sp * per;
    if (sp == 1 || static_cast<__int128>(num) * bd > static_cast<__int128>(bn) * den) {
      best = sp;
      bn = num;
      bd = den;
    }
  }
  return best;
}

template <int MODE>
__device__ __forceinline__ void unit_tiles(const TileArgs& a, int n_cols, int col, int& t0,
                                           int& t1) {
  if (is_fwd(MODE)) {
    t0 = static_cast<int>((static_cast<long long>(col) * a.n_vtiles) / n_cols);
    t1 = static_cast<int>((static_cast<long long>(col + 1) * a.n_vtiles) / n_cols);
  } else {
    t0 = col;
    t1 = col + 1;
  }
}

// Blocking wait that ignores the abort flag (used only to drain in-flight
// async work on the abort path); bounded like every other wait.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return;
  }
}

// tanh(x) = 1 - 2 / (1 + e^{2x}), with the SFU exponential; absolute error a
// few 1e-7 over the whole range, saturating cleanly to +-1.
__device__ __forceinline__ float tanh_sfu(float x) {
  const float e = ex2(x * 2.8853900817779268f);  // e^{2x} = 2^{2x log2 e}
  return 1.f - __fdividef(2.f, 1.f + e);
}

// Applies the logit transform to 32 raw logits in place; returns nothing when
// the transform is the identity (xmode 0).
__device__ __forceinline__ void logit_transform(const TileArgs& a, float (&v)[32]) {
  if (a.xmode == 1) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= a.k0;
  } else if (a.xmode == 2) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = a.k2 * tanh_sfu(v[j] * a.k1);
  }
}

// f'(S) recovered from the transformed logit z' (1 without a transform).
__device__ __forceinline__ float dz_of_logit(const TileArgs& a, float z) {
  if (a.xmode == 1) return a.k0;
  if (a.xmode == 2) {
    const float u = z / a.k2;
    return a.k0 * fmaf(-u, u, 1.f);
  }
  return 1.f;
}

// Byte offset of stage column c (0..63) of row r in a 128B-swizzled A stage:
// 16-byte chunk j of row r sits at chunk j ^ (r & 7).
__device__ __forceinline__ int swz_offset(int r, int c) {
  return r * 128 + ((((c >> 3) ^ r) & 7) << 4) + (c & 7) * 2;
}

// Per-row constants of the in-GEMM conversion of stored logits (MODE_DHS,
// MODE_UAC). A stored value s of column v is z'_v log2e - zoff, zoff the
// maximum of the column's 64-column box (one pipeline stage) times log2 e, as
// kept in fp32 beside the box (the value subtracted, so that adding it back
// restores z'_v log2e exactly up to the fp16 rounding of s), and becomes the
// bf16
//   without a transform:  2^(s + zoff + c)
//   with one:             scale * 2^(s + zoff + shift2) f'(S_v)
// (f' recovered from z'_v = (s + zoff) ln2, as in dz_of_logit); the target
// column gets ytarget.
//   MODE_DHS (G / sigma, sigma = -sign(g) the same for the whole row, so that
//             the epilogue applies it to the row of dH once instead of to
//             every element): c = log2|g| - lse2, scale = |g|, shift2 = -lse2,
//             ytarget = sigma g (1 - p_y) f'_y
//   MODE_UAC (P):  c = -M, scale = 1, shift2 = -M, ytarget = 0
// with M the row's running maximum (log2 units).
struct RowCvt {
  bool zero;        // the row contributes nothing: zeros whatever the buffer held
  int y;            // target column (vocabulary index), or -1
  float c;          // see above (without the box maximum)
  bool neg;         // MODE_DHS: sigma = -1 (g > 0), the row of dH is negated
  float scale, shift2;
  float ytarget;
};

// Per-row constants of the single pass's U accumulator (MODE_UAC, MODE_UAP):
// the row's running maximum M after this block (log2 units, from the split
// partials of the blocks so far), the rescale of U from the blocks before,
// alpha = 2^(M_prev - M), and on the last block the factors of
// dH = cw W_y - cu U: cu = g 2^(M - lse2), cw = g (1 - p_y) f'_y.
struct UaccRow {
  bool zero;        // masked or outside the batch: U and dH get zeros
  int y;            // target column, or -1 (bad ids: the row finish sets the status)
  float mcur, alpha, cu, cw;
};

__device__ __forceinline__ UaccRow uacc_row(const TileArgs& a, long long grow, bool valid) {
  UaccRow r;
  r.zero = true;
  r.y = -1;
  r.mcur = 0.f;
  r.alpha = 0.f;
  r.cu = 0.f;
  r.cw = 0.f;
  if (!valid || (a.mask != nullptr && a.mask[grow] == 0)) return r;
  float mcur = -INFINITY;
  for (int sl = 0; sl < a.slots_cur; ++sl) mcur = fmaxf(mcur, a.part_m[sl * a.part_ld + grow]);
  const int yy = a.ids[grow];
  r.zero = false;
  r.y = (yy >= 0 && yy < a.vocab) ? yy : -1;
  r.mcur = mcur;
  if (!a.first) {
    float mprev = -INFINITY;
    for (int sl = 0; sl < a.slots_prev; ++sl) mprev = fmaxf(mprev, a.part_m[sl * a.part_ld + grow]);
    r.alpha = ex2(mprev - mcur);
  }
  if (a.last) {
    const float g = a.g[grow];
    const float l2 = a.lse[grow] * kLog2e;
    r.cu = g * ex2(mcur - l2);
    if (r.y >= 0) {
      const float zy = a.zy[grow];
      r.cw = (g - g * ex2(fmaf(zy, kLog2e, -l2))) * dz_of_logit(a, zy);
    }
  }
  return r;
}

// U update of 8 hidden columns of one row, x = this block's P W for them:
// U = alpha U_prev + x (U_prev read from accp unless this is the first block),
// then stored back to accp, or on the last block turned into dH (bf16, outp).
__device__ __forceinline__ void uacc_update8(const TileArgs& a, const UaccRow& r, float (&x)[8],
                                             float* accp, __nv_bfloat16* outp,
                                             const __nv_bfloat16* wy) {
  if (r.zero) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = 0.f;
  } else if (!a.first) {
    const float4 a0 = *reinterpret_cast<const float4*>(accp);
    const float4 a1 = *reinterpret_cast<const float4*>(accp + 4);
    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = fmaf(r.alpha, av[e], x[e]);
  }
  if (a.last) {
    if (!r.zero) {
      float wv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (r.y >= 0) {
        const uint4 wb = *reinterpret_cast<const uint4*>(wy);
        const uint32_t ww[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          wv[2 * e] = __uint_as_float(ww[e] << 16);
          wv[2 * e + 1] = __uint_as_float(ww[e] & 0xffff0000u);
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = fmaf(r.cw, wv[e], -r.cu * x[e]);
    }
    st_global_v4(outp, pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                 pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
  } else {
    *reinterpret_cast<float4*>(accp) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(accp + 4) = make_float4(x[4], x[5], x[6], x[7]);
  }
}

// Rewrites chunks jb..jb+NCH-1 (8 columns each) of row r of a landed A stage
// (64 stored values of vocab columns vbase.., box maximum zoff in log2 units) in place as
// bf16. Columns at or past the vocabulary size become zeros. The main loop
// runs over logical chunks, so the 8 lanes of a shared-memory phase (8
// consecutive rows, same chunk) touch 8 different physical chunks: no bank
// conflicts. The target column (at most once per row and unit) and the
// vocabulary edge (the last stage) are fixed up afterwards, off the hot path.
template <int NCH>
__device__ __forceinline__ void stage_row_to_bf16(const TileArgs& a, uint8_t* tile, int r, int jb,
                                                  int vbase, const RowCvt& rc, float zoff) {
  uint4* row = reinterpret_cast<uint4*>(tile + r * 128);
  const int sw = r & 7;
  if (rc.zero) {
#pragma unroll
    for (int j = 0; j < NCH; ++j) row[(jb + j) ^ sw] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  if (a.xmode == 0) {
    const float c = zoff + rc.c;
    uint4 in[NCH];
#pragma unroll
    for (int j = 0; j < NCH; ++j) in[j] = row[(jb + j) ^ sw];
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const uint32_t w[4] = {in[j].x, in[j].y, in[j].z, in[j].w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float t0, t1;
        add_f16x2_f32(w[e], c, t0, t1);
        o[e] = pack_bf16x2(ex2(t0), ex2(t1));
      }
      row[(jb + j) ^ sw] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  } else {
    const float c2 = zoff + rc.shift2;
#pragma unroll 1
    for (int j = jb; j < jb + NCH; ++j) {
      const uint4 x = row[j ^ sw];
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float s0, s1;
        unpack_f16x2(w[e], s0, s1);
        const float z0 = (s0 + zoff) * kLn2, z1 = (s1 + zoff) * kLn2;
        o[e] = pack_bf16x2(rc.scale * ex2(s0 + c2) * dz_of_logit(a, z0),
                           rc.scale * ex2(s1 + c2) * dz_of_logit(a, z1));
      }
      row[j ^ sw] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  const unsigned yoff = static_cast<unsigned>(rc.y - vbase - jb * 8);
  if (yoff < static_cast<unsigned>(NCH * 8) && rc.y < a.vocab) {
    *reinterpret_cast<uint16_t*>(tile + swz_offset(r, jb * 8 + static_cast<int>(yoff))) =
        static_cast<uint16_t>(pack_bf16x2(rc.ytarget, 0.f) & 0xffffu);
  }
  if (vbase + (jb + NCH) * 8 > a.vocab) {
#pragma unroll 1
    for (int c = max(jb * 8, a.vocab - vbase); c < (jb + NCH) * 8; ++c)
      *reinterpret_cast<uint16_t*>(tile + swz_offset(r, c)) = 0;
  }
}

// Per-variant geometry. CTAS = 1: one CTA computes a 128 x 256 tile. CTAS = 2:
// a CTA pair computes a 256 x 256 tile with tcgen05 cta_group::2; each CTA
// loads its own 128 A rows and half of the B tile (128 of its 256 rows/cols),
// the leader issues the MMAs, and each CTA's TMEM holds its 128 rows.
// The pair's dH GEMM runs units of 512 D columns: two 256-column accumulators
// fill TMEM (no double buffering; its units are whole-vocabulary K loops, so
// the single epilogue per unit costs ~1 %), and every A tile of G feeds twice
// the MMA work.
template <int MODE, int CTAS>
struct PairCfg {
  static constexpr int kNAcc = (is_dh(MODE) && CTAS == 2) ? 2 : 1;  // accumulators
  static constexpr int kNBuf = kNAcc == 2 ? 1 : 2;     // TMEM buffers (of kNAcc x 256)
  static constexpr int kTileN = BN * kNAcc;            // N columns per unit
  static constexpr int kBRows = BN / CTAS;             // B rows (cols) per CTA and MMA
  static constexpr int kBBytes = kNAcc * kBRows * BK * 2;
  // 64-wide K slices per stage: the pair's 256-column logit and dW GEMMs (a
  // lone accumulator) take two, so that each stage carries 8 MMAs like the dH
  // GEMM's 512-wide units. With 4 per stage the tensor pipe idled ~18 % of the
  // time whatever the ring depth, the operand traffic or the epilogue: a fixed
  // cost per stage (measured 81 % -> 91 % tensor-pipe activity).
  static constexpr int kKSub =
      (CTAS == 2 && kNAcc == 1 && (is_fwd(MODE) || MODE == MODE_BWDG || MODE == MODE_DW)) ? 2 : 1;
  static constexpr int kStageBytes = kKSub * (A_BYTES + kBBytes);
  // The pair's logit-storing, G-tile and dW GEMMs write their outputs through
  // shared memory: each epilogue warp stages a 32-row box of 128-byte rows (64
  // fp16 logits, 64 bf16 G values or 32 fp32 dW values; 4 KB, 128-byte
  // swizzle) in one of two buffers
  // and writes it with a TMA tensor store (dW after its first chunk: a TMA
  // reduce-add), in whole 128-byte lines. Written straight from registers,
  // each warp store touched 32 rows in 16-byte pieces: that cost the logit
  // GEMM 15 % of its time at D = 1536 (1.73 ms with the stores, 1.47 ms
  // without) and the dW GEMM 25 % at the Llama shape (3.22 against 2.43 ms).
  static constexpr bool kTmaStore =
      (MODE == MODE_FWDS || MODE == MODE_BWDG || MODE == MODE_DW) && CTAS == 2;
  static constexpr int kStoreBufBytes = 32 * 128;
  static constexpr int kStoreBytes = kTmaStore ? 4 * 2 * kStoreBufBytes : 0;
  static constexpr int kMaxDynSmem = 232448 - 1024 - 1024;  // 227 KB less slack and statics
  static constexpr int kStageRoom = (kMaxDynSmem - kStoreBytes) / kStageBytes;
  static constexpr int kStages = CTAS == 2 ? (kStageRoom < 7 ? kStageRoom : 7) : STAGES;
  static constexpr int kSmemBytes = kStages * kStageBytes + kStoreBytes + 1024;
  // Warp groups that convert A stages (MODE_DHS): the epilogue warps and a
  // second group of converter-only warps, each group half of every row.
  static constexpr int kCvtGroups = has_cvt(MODE) ? 2 : 1;
  static constexpr int kThreads = 64 + 128 * kCvtGroups;
};

// MODE_DH/DHS/UAC/DW (output columns = hidden): the MMA width of the
// accumulator starting at hidden column col0, i.e. its columns inside the
// hidden size in whole 64-column MN blocks of every CTA's share; 0 when the
// accumulator lies wholly past it. A ragged last tile thus runs narrower MMAs
// and loads fewer B boxes.
template <int CTAS>
__device__ __forceinline__ int mn_out_cols(const TileArgs& a, int col0) {
  const int w = a.hidden - col0;
  constexpr int q = 64 * CTAS;
  return w <= 0 ? 0 : min(BN, (w + q - 1) / q * q);
}

// ---------------------------------------------------------------------------
// Tail split of a dH-type launch (MODE_DH, MODE_DHS over the whole vocabulary;
// MODE_UAC, MODE_UAP over one vocabulary block, whose cut units the fixup
// passes through the U update). Its units (row unit x hidden tile) each run a
// K loop over the vocabulary, and the pairs run them whole, one per pair and
// round. When the last round
// has fewer units (U) than pairs, the pairs without one would idle (66 units
// on 76 pairs: 13 % of the launch). Instead, each of those U units runs on its
// own pair only up to a balance point m of its K loop (its main piece), and Q
// of the idle pairs share the units' tails [m, K) among them, laid end to end
// in unit order and cut at K-stage boundaries, so that every pair of the round
// does about the same work. The U main pieces all start at K = 0 together and
// the tails all lie in the last part of the vocabulary: at any moment the
// pairs read W and the logit rows from two narrow K windows, which stay in L2
// (cuts at arbitrary K offsets, one contiguous share of all units per pair,
// left every pair at its own place in the vocabulary and made the launch
// DRAM-bound). Q is at most a third of the pairs, whose tail reads may come
// from DRAM. Each cut piece leaves its fp32 partial tile in a slot of its own;
// tail_fixup_kernel adds a unit's pieces in a fixed order (the main piece, then
// the tails in pair order), so the result does not depend on timing.
constexpr int kTailMinStages = 64;  // least K stages of full width per tail pair
// What a cut piece costs beyond its stages (its partial tile leaves TMEM
// before the next piece's MMAs can start, and the pipeline refills), in cost
// units: about 8 full-width stages (6 us per piece measured on GB300 against
// 0.7 us per stage).
constexpr int kTailPieceCost = 8 * 4;

struct TailSplit {
  int w_dp;          // units [0, w_dp) run whole, round-robin (the whole rounds)
  int n_main;        // U: units of the last round; pair p < U runs unit w_dp + p
  int n_tail;        // Q: pairs U .. U+Q-1 share the tails; 0: no split
  int k;             // K stages of a unit
  int cs_f, cs_l;    // cost per stage: units of the other tiles, of the last tile
  int m_f, m_l;      // main stages of each
  long long t_f, t_l;   // tail cost of each
  long long tail_total;
};

// MMA column blocks (of 64 columns per CTA) per K stage of a dH unit of
// hidden tile `col`: its cost per stage.
template <int CTAS>
__device__ __forceinline__ int ts_blocks(const TileArgs& a, int col) {
  constexpr int kNAcc = CTAS == 2 ? 2 : 1;
  int b = 0;
#pragma unroll
  for (int na = 0; na < kNAcc; ++na)
    b += mn_out_cols<CTAS>(a, col * (BN * kNAcc) + na * BN) / (64 * CTAS);
  return b;
}

// Units in [u0, u1) of the last hidden tile, in the raster order of
// decode_unit (groups of group_rows row units, tile-major within a group).
__device__ __forceinline__ int ts_count_last(const TileArgs& a, int n_ru, int u0, int u1) {
  if (u1 <= u0) return 0;
  const int per_group = a.group_rows * a.n_cols;
  int n = 0;
  for (int g = u0 / per_group; g * per_group < u1; ++g) {
    const int rig = min(a.group_rows, n_ru - g * a.group_rows);
    const int lo = g * per_group + (a.n_cols - 1) * rig, hi = lo + rig;
    n += max(0, min(hi, u1) - max(lo, u0));
  }
  return n;
}

template <int CTAS>
__device__ __forceinline__ TailSplit tail_split(const TileArgs& a, int n_ru, int n_units, int slots) {
  TailSplit s;
  s.w_dp = n_units;
  s.n_main = 0;
  s.n_tail = 0;
  s.k = a.k_iters;
  s.cs_f = s.cs_l = 1;
  s.m_f = s.m_l = a.k_iters;
  s.t_f = s.t_l = 0;
  s.tail_total = 0;
  const int rem = slots > 0 ? n_units % slots : 0;
  if (a.ts_part == nullptr || rem == 0 || a.k_iters < 2 * kTailMinStages) return s;
  const int U = rem;
  const int w_dp = n_units - rem;
  const int k = a.k_iters;
  s.cs_f = ts_blocks<CTAS>(a, 0);
  s.cs_l = ts_blocks<CTAS>(a, a.n_cols - 1);
  const int n_l = a.n_cols == 1 ? U : ts_count_last(a, n_ru, w_dp, n_units);
  const int n_f = U - n_l;
  if (a.n_cols == 1) s.cs_f = s.cs_l;
  const long long c_f = static_cast<long long>(k) * s.cs_f, c_l = static_cast<long long>(k) * s.cs_l;
  const long long total = n_f * c_f + n_l * c_l;
  const long long min_cost = static_cast<long long>(kTailMinStages) * 4;
  const int Q = static_cast<int>(min(static_cast<long long>(min(slots - U, slots / 3)),
                                     total / min_cost - U));
  if (Q <= 0) return s;
  // Balance: every pair of the round takes about T of cost, the tail pairs'
  // pieces (about (U + Q) / Q each) counted with their overhead. A unit
  // cheaper than T (a narrow last tile) keeps no tail.
  const long long ovh = kTailPieceCost;
  long long T = (total + (U + Q) * ovh + U + Q - 1) / (U + Q);
  if (T > c_l && n_f > 0)
    T = max(c_l, (n_f * c_f + (n_f + Q) * ovh + n_f + Q - 1) / (n_f + Q));
  // No gain unless the round gets shorter by more than the pieces cost.
  if (T + 2 * ovh >= c_f) return s;
  s.m_f = static_cast<int>(min(static_cast<long long>(k), T / s.cs_f));
  s.m_l = static_cast<int>(min(static_cast<long long>(k), T / s.cs_l));
  s.t_f = static_cast<long long>(k - s.m_f) * s.cs_f;
  s.t_l = static_cast<long long>(k - s.m_l) * s.cs_l;
  s.tail_total = n_f * s.t_f + n_l * s.t_l;
  if (s.tail_total == 0) return s;
  s.w_dp = w_dp;
  s.n_main = U;
  s.n_tail = Q;
  return s;
}

__device__ __forceinline__ bool ts_is_last(const TileArgs& a, int n_ru, int u) {
  int ru, col;
  decode_unit(u, n_ru, a.n_cols, a.group_rows, ru, col);
  return col == a.n_cols - 1;
}

// Tail cost of the last round's units before u.
__device__ __forceinline__ long long ts_tail_prefix(const TileArgs& a, int n_ru, const TailSplit& s,
                                                    int u) {
  const int nl = ts_count_last(a, n_ru, s.w_dp, u);
  return static_cast<long long>(u - s.w_dp - nl) * s.t_f + static_cast<long long>(nl) * s.t_l;
}

// First tail cost of tail pair q (q = n_tail: the end).
__device__ __forceinline__ long long ts_tail_start(const TailSplit& s, int q) {
  return s.tail_total * q / s.n_tail;
}

// The tail pair whose share holds tail cost x (0 <= x < tail_total).
__device__ __forceinline__ int ts_tail_pair_of(const TailSplit& s, long long x) {
  int q = static_cast<int>(x * s.n_tail / s.tail_total);
  q = min(max(q, 0), s.n_tail - 1);
  while (q + 1 < s.n_tail && ts_tail_start(s, q + 1) <= x) ++q;
  while (q > 0 && ts_tail_start(s, q) > x) --q;
  return q;
}

// The last unit u of the last round with tail prefix <= x.
__device__ __forceinline__ int ts_tail_unit_at(const TileArgs& a, int n_ru, const TailSplit& s,
                                               int lo, long long x) {
  int hi = s.w_dp + s.n_main - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ts_tail_prefix(a, n_ru, s, mid) <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Stages [kb, ke) of unit u's tail that tail pair q runs (kb >= ke: none).
__device__ __forceinline__ void ts_tail_piece(const TileArgs& a, int n_ru, const TailSplit& s, int q,
                                              int u, int& kb, int& ke) {
  const bool last = ts_is_last(a, n_ru, u);
  const int cs = last ? s.cs_l : s.cs_f;
  const int m = last ? s.m_l : s.m_f;
  const long long t = last ? s.t_l : s.t_f;
  const long long p0 = ts_tail_prefix(a, n_ru, s, u);
  const long long q0 = ts_tail_start(s, q), q1 = ts_tail_start(s, q + 1);
  kb = m + static_cast<int>((max(q0, p0) - p0) / cs);
  ke = m + static_cast<int>((min(q1, p0 + t) - p0) / cs);
}

// Slot of a cut piece: main pieces 0 .. U-1, tail pieces U + (u - w_dp) + q
// (unique: along the units in order and the tail pairs in order, u + q grows).
__device__ __forceinline__ int ts_main_slot(const TailSplit& s, int u) { return u - s.w_dp; }
__device__ __forceinline__ int ts_tail_slot(const TailSplit& s, int u, int q) {
  return s.n_main + (u - s.w_dp) + q;
}

// One work item of a pair: unit u over K stages [kb, ke). A cut piece (not the
// whole K range) writes its fp32 partial tile to slot `slot` instead of dH.
struct WorkItem {
  int u, kb, ke, slot;
  bool cut;
  // A piece of the split that rounding left without stages: no role touches it.
  __device__ __forceinline__ bool empty() const { return slot >= 0 && ke <= kb; }
};

// The work items of one pair, in order: its round-robin units, then its main
// piece or its tail pieces of the last round.
template <int CTAS>
struct WorkList {
  TailSplit s;
  int slot, n_slots, n_dp;
  int n_extra;       // items after the round-robin ones
  int u_first;       // tail pair: first unit whose tail it meets
  int q;             // tail pair index, or -1 (main pair or none)

  __device__ __forceinline__ void init(const TileArgs& a, int n_ru, int n_units, int slot_,
                                       int n_slots_, bool dh_mode) {
    slot = slot_;
    n_slots = n_slots_;
    n_extra = 0;
    u_first = 0;
    q = -1;
    s = tail_split<CTAS>(a, n_ru, dh_mode ? n_units : 0, n_slots);
    if (!dh_mode) s.w_dp = n_units;
    if (s.n_tail > 0) {
      if (slot < s.n_main) {
        n_extra = 1;
      } else if (slot < s.n_main + s.n_tail) {
        q = slot - s.n_main;
        const long long x0 = ts_tail_start(s, q), x1 = ts_tail_start(s, q + 1);
        u_first = ts_tail_unit_at(a, n_ru, s, s.w_dp, x0);
        const int u_last = ts_tail_unit_at(a, n_ru, s, u_first, x1 - 1);
        n_extra = u_last - u_first + 1;
      }
    }
    n_dp = slot < s.w_dp ? (s.w_dp - slot + n_slots - 1) / n_slots : 0;
  }

  // Item i (false past the end).
  __device__ __forceinline__ bool get(const TileArgs& a, int n_ru, int k_iters, int i,
                                      WorkItem& w) const {
    if (i < n_dp) {
      w.u = slot + i * n_slots;
      w.kb = 0;
      w.ke = k_iters;
      w.slot = -1;
      w.cut = false;
      return true;
    }
    const int j = i - n_dp;
    if (j >= n_extra) return false;
    if (q < 0) {  // main piece
      w.u = s.w_dp + slot;
      w.kb = 0;
      w.ke = ts_is_last(a, n_ru, w.u) ? s.m_l : s.m_f;
      w.slot = ts_main_slot(s, w.u);
    } else {
      w.u = u_first + j;
      ts_tail_piece(a, n_ru, s, q, w.u, w.kb, w.ke);
      w.slot = ts_tail_slot(s, w.u, q);
    }
    w.cut = w.kb != 0 || w.ke != k_iters;
    return true;
  }
};

// fp32 partial tile of slot `slot`, CTA `rank`: [32-column chunk][8][BM rows][4],
// so that a warp's 32 rows write (and the fixup reads) 512 contiguous bytes.
__device__ __forceinline__ float* ts_slot_ptr(const TileArgs& a, int slot, int rank, int ctas,
                                              int tile_n) {
  return a.ts_part + (static_cast<long long>(slot) * ctas + rank) * (static_cast<long long>(BM) * tile_n);
}

// One TMA box into this CTA's stage; its bytes are counted on the leader's
// barrier (pair) or this CTA's own.
template <int CTAS>
__device__ __forceinline__ void load_box(void* dst, const CUtensorMap* map, uint64_t* bar,
                                         uint32_t lead, int c0, int c1, bool hint,
                                         uint64_t pol) {
  if (CTAS == 2) {
    if (hint) tma_load_2d_pair(dst, map, lead, c0, c1, pol);
    else tma_load_2d_pair_nohint(dst, map, lead, c0, c1);
  } else {
    if (hint) tma_load_2d_hint(dst, map, bar, c0, c1, pol);
    else tma_load_2d(dst, map, bar, c0, c1);
  }
}

template <int MODE, int CTAS>
__global__ void __launch_bounds__(PairCfg<MODE, CTAS>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_c,
                   const __grid_constant__ CUtensorMap map_h16,
                   const __grid_constant__ CUtensorMap map_hc, const TileArgs args) {
  using C = PairCfg<MODE, CTAS>;
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  // MODE_DHS, MODE_UAC: this CTA's A stage has landed (its own barrier); the
  // stage has been converted by the pair's converter warps (the leader's barrier).
  __shared__ __align__(8) uint64_t afull_bar[has_cvt(MODE) ? kStages : 1];
  __shared__ __align__(8) uint64_t cvt_bar[has_cvt(MODE) ? kStages : 1];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  // The 128-byte swizzle pattern is a function of address bits [4:9], so each
  // stage starts on a 1024-byte boundary.
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &abort_sh;
  const uint32_t rank = CTAS == 2 ? cluster_ctarank() : 0u;
  const int cta_slot = static_cast<int>(blockIdx.x) / CTAS;  // pair index
  const int n_slots = static_cast<int>(gridDim.x) / CTAS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], CTAS);  // pair: both CTAs' producers arrive (leader's)
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 4 * CTAS);  // every epilogue warp of the pair
    }
    mbar_init(&drain_bar, 1);
    if constexpr (has_cvt(MODE)) {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(&afull_bar[s], 1);
        mbar_init(&cvt_bar[s], 4 * C::kCvtGroups * CTAS);  // every converter warp of the pair
      }
    }
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b);
  }
  if (warp == 1) {
    if (CTAS == 2) {
      tmem_alloc_pair(&tmem_base_sh, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&tmem_base_sh, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (CTAS == 2) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;

  // Row blocks of the active list this launch covers. For MODE_DW they are the
  // K dimension; its units are vocab rows instead.
  const int n_rb = launch_row_blocks(args);
  const int n_ru = MODE == MODE_DW ? (args.dw_rows + BM * CTAS - 1) / (BM * CTAS)
                                   : (n_rb + CTAS - 1) / CTAS;  // units of 128*CTAS rows
  // Units per row unit: FWD vocab splits (set here from the active row units
  // when max_cols > 0), BWDG vocab tiles, dH-type D tiles.
  int n_cols = args.n_cols;
  if constexpr (is_fwd(MODE)) {
    if (args.max_cols > 0) n_cols = fwd_splits_for(n_ru, args.n_vtiles, n_slots, args.max_cols);
  }
  const int n_units = n_ru * n_cols;
  // Stages per tile (k_iters counts 64-wide K slices; a stage holds kKSub).
  const int k_iters = ((MODE == MODE_DW ? n_rb * (BM / BK) : args.k_iters) + C::kKSub - 1) / C::kKSub;
  // This pair's units, and with a tail split its part of the last round.
  WorkList<CTAS> wl;
  wl.init(args, n_ru, n_units, cta_slot, n_slots,
          MODE == MODE_DH || MODE == MODE_DHS || is_uacc(MODE));

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      const uint64_t pol_a = policy_evict_last();
      // MODE_DW: every segment active, so that h's rows are in order.
      const bool h_dense =
          args.seg_list == nullptr || (args.n_seg != nullptr && all_segs_active(args, *args.n_seg));
      for (int i = 0; ok; ++i) {
        WorkItem wk;
        if (!wl.get(args, n_ru, k_iters, i, wk)) break;
        if (wk.empty()) continue;
        int ru, col, t0, t1;
        decode_unit(wk.u, n_ru, n_cols, args.group_rows, ru, col);
        unit_tiles<MODE>(args, n_cols, col, t0, t1);
        // A CTA whose row block lies past the list computes its partner's rows
        // again and stores nothing.
        int li = ru * CTAS + static_cast<int>(rank);
        if (li >= n_rb) li = ru * CTAS;
        // The logit and G-tile GEMMs read rows of h: one box of BM rows when
        // the block's segments are consecutive rows, else one of SEG rows per
        // segment (map_h16); the dH-type GEMMs read chunk-local rows.
        int hr[kSegs];
        bool h_one = true;
        const CUtensorMap* map_h1 = &map_a;  // where a block of h is one box
        if constexpr (!is_dh(MODE) && MODE != MODE_DW) {
          h_one = h_rows(args, li, hr);
          if (!h_one && args.hc) {
            h_one = true;
            hr[0] = li * BM;  // the block's rows, copied in order
            map_h1 = &map_hc;
          }
        }
        int a_row = 0;  // MODE_DW: unused (its A rows are vocab rows)
        if constexpr (is_dh(MODE)) a_row = li * BM;
        else if constexpr (MODE != MODE_DW) a_row = hr[0];
        const int a_m0 = (ru * CTAS + static_cast<int>(rank)) * BM;  // MODE_DW: vocab row
        for (int t = t0; t < t1 && ok; ++t) {
          // MN-major B (DH, DHS, UAC, DW): 64-column boxes per accumulator in
          // this CTA, and their bytes.
          int nbox[C::kNAcc];
          uint32_t b_bytes = 0;
#pragma unroll
          for (int na = 0; na < C::kNAcc; ++na) {
            nbox[na] = mn_out_cols<CTAS>(args, t * C::kTileN + na * BN) / (64 * CTAS);
            b_bytes += static_cast<uint32_t>(nbox[na]) * (BK * 64 * 2);
          }
          int hk_next[kSegs];  // MODE_DW: rows of h of the next stage's row block
          if constexpr (MODE == MODE_DW) {
            if (!h_dense) h_rows(args, (wk.kb * C::kKSub * BK) / BM, hk_next);
          }
          for (int k = wk.kb; k < wk.ke; ++k, ++it) {
            const int s = it % kStages;
            const uint32_t round = it / kStages;
            if (!mbar_wait(&empty_bar[s], (round & 1u) ^ 1u, abort_flag, args.status)) {
              ok = false;
              break;
            }
            uint8_t* a_dst = smem + s * C::kStageBytes;
            uint8_t* b_dst = a_dst + C::kKSub * A_BYTES;
            if constexpr (has_cvt(MODE)) {
              // A (the stored fp16 logits) into this CTA's stage, counted on
              // its own barrier: the epilogue warps turn it into G in place.
              mbar_arrive_expect_tx(&afull_bar[s], A_BYTES);
              tma_load_2d_hint(a_dst, &map_a, &afull_bar[s], k * BK, a_row, pol_a);
              // B (W, MN-major): per accumulator, this CTA's share of its D
              // columns, counted on the leader's barrier (pair) or its own.
              const uint32_t lead = CTAS == 2 ? mapa_shared(smem_u32(&full_bar[s]), 0) : 0u;
              if (CTAS == 2) mbar_arrive_expect_tx_cluster(lead, b_bytes);
              else mbar_arrive_expect_tx(&full_bar[s], b_bytes);
#pragma unroll
              for (int na = 0; na < C::kNAcc; ++na)
                for (int jb = 0; jb < nbox[na]; ++jb)
                  load_box<CTAS>(b_dst + na * (C::kBRows * BK * 2) + jb * (BK * 64 * 2), &map_b,
                                 &full_bar[s], lead,
                                 t * C::kTileN + na * BN + static_cast<int>(rank) * nbox[na] * 64 +
                                     jb * 64,
                                 args.v0 + k * BK, false, 0);
            } else if (MODE == MODE_DW) {
              const uint32_t lead = CTAS == 2 ? mapa_shared(smem_u32(&full_bar[s]), 0) : 0u;
              if (CTAS == 2) mbar_arrive_expect_tx_cluster(lead, C::kKSub * (A_BYTES + b_bytes));
              else mbar_arrive_expect_tx(&full_bar[s], C::kKSub * (A_BYTES + b_bytes));
              // The rows of h of this stage's row block: in order when every
              // segment is active, else looked up a stage ahead, so that the
              // lookup's loads do not hold up the ring.
              int hk[kSegs];
              if (h_dense) {
                const int r0 = (args.rb_offset + (k * C::kKSub * BK) / BM) * BM;
#pragma unroll
                for (int j = 0; j < kSegs; ++j) hk[j] = r0 + j * SEG;
              } else {
#pragma unroll
                for (int j = 0; j < kSegs; ++j) hk[j] = hk_next[j];
                if (k + 1 < wk.ke) h_rows(args, ((k + 1) * C::kKSub * BK) / BM, hk_next);
              }
#pragma unroll
              for (int ks = 0; ks < C::kKSub; ++ks) {
                const int kr = (k * C::kKSub + ks) * BK;  // chunk-local row of this K slice
                const bool second = (kr % BM) >= BK;       // its half of the block's segments
                int h4[BK / SEG];
#pragma unroll
                for (int j = 0; j < BK / SEG; ++j) h4[j] = second ? hk[BK / SEG + j] : hk[j];
                bool one = true;
#pragma unroll
                for (int j = 1; j < BK / SEG; ++j) one = one && h4[j] == h4[0] + j * SEG;
                // A = G^T: 128 vocab rows (two 64-wide MN blocks) x 64 chunk rows.
#pragma unroll
                for (int j = 0; j < 2; ++j)
                  load_box<CTAS>(a_dst + ks * A_BYTES + j * (BK * 64 * 2), &map_a, &full_bar[s],
                                 lead, a_m0 + j * 64, kr, true, pol_a);
                // B = H: this CTA's D columns x the same 64 rows, in 64-wide
                // blocks (each a box of 64 rows, or one of SEG rows per segment).
                for (int jb = 0; jb < nbox[0]; ++jb) {
                  uint8_t* dst = b_dst + ks * C::kBBytes + jb * (BK * 64 * 2);
                  const int col = t * BN + static_cast<int>(rank) * nbox[0] * 64 + jb * 64;
                  if (one) {
                    load_box<CTAS>(dst, &map_b, &full_bar[s], lead, col, h4[0], false, 0);
                  } else {
#pragma unroll
                    for (int j = 0; j < BK / SEG; ++j)
                      load_box<CTAS>(dst + j * (SEG * 64 * 2), &map_h16, &full_bar[s], lead, col,
                                     h4[j], false, 0);
                  }
                }
              }
            } else if (CTAS == 2) {
              // Both CTAs count their bytes on the leader's barrier.
              const uint32_t lead = mapa_shared(smem_u32(&full_bar[s]), 0);
              mbar_arrive_expect_tx_cluster(lead, is_dh_plain(MODE) ? A_BYTES + b_bytes
                                                                  : C::kStageBytes);
#pragma unroll
              for (int ks = 0; ks < C::kKSub; ++ks) {
                const int kc = (k * C::kKSub + ks) * BK;
                if (h_one) {
                  tma_load_2d_pair(a_dst + ks * A_BYTES, map_h1, lead, kc, a_row, pol_a);
                } else {
#pragma unroll
                  for (int j = 0; j < kSegs; ++j)
                    tma_load_2d_pair(a_dst + ks * A_BYTES + j * (SEG * BK * 2), &map_h16, lead, kc,
                                     hr[j], pol_a);
                }
              }
              if (is_dh_plain(MODE)) {
                // Per accumulator, this CTA's share of its D columns.
#pragma unroll
                for (int na = 0; na < C::kNAcc; ++na)
                  for (int jb = 0; jb < nbox[na]; ++jb)
                    tma_load_2d_pair_nohint(
                        b_dst + na * (C::kBRows * BK * 2) + jb * (BK * 64 * 2), &map_b, lead,
                        t * C::kTileN + na * BN + static_cast<int>(rank) * nbox[na] * 64 +
                            jb * 64,
                        args.v0 + k * BK);
              } else {
                // Per K slice and accumulator, this CTA's 128 of its 256 vocab rows.
#pragma unroll
                for (int ks = 0; ks < C::kKSub; ++ks)
#pragma unroll
                  for (int na = 0; na < C::kNAcc; ++na)
                    tma_load_2d_pair_nohint(b_dst + ks * C::kBBytes + na * (C::kBRows * BK * 2),
                                            &map_b, lead, (k * C::kKSub + ks) * BK,
                                            args.v0 + t * C::kTileN + na * BN +
                                                static_cast<int>(rank) * C::kBRows);
              }
            } else {
              mbar_arrive_expect_tx(&full_bar[s],
                                    is_dh_plain(MODE) ? A_BYTES + b_bytes : C::kStageBytes);
              if (h_one) {
                tma_load_2d_hint(a_dst, map_h1, &full_bar[s], k * BK, a_row, pol_a);
              } else {
#pragma unroll
                for (int j = 0; j < kSegs; ++j)
                  tma_load_2d_hint(a_dst + j * (SEG * BK * 2), &map_h16, &full_bar[s], k * BK,
                                   hr[j], pol_a);
              }
              if (is_dh_plain(MODE)) {
                // W[v0 + k*64 .. +64, d0 .. d0+256) as up to four 64x64 MN-major boxes.
                for (int jb = 0; jb < nbox[0]; ++jb)
                  tma_load_2d(b_dst + jb * (BK * 64 * 2), &map_b, &full_bar[s],
                              t * BN + jb * 64, args.v0 + k * BK);
              } else {
                tma_load_2d(b_dst, &map_b, &full_bar[s], k * BK, args.v0 + t * BN);
              }
            }
          }
        }
      }
      if (!ok) {
        // Abort path: let the copies already issued land before the CTA exits
        // (the leader's barriers count the pair's copies; the peer passes the
        // closing cluster barrier only after this). MODE_DHS counts each
        // CTA's A copies on its own barriers.
        for (uint32_t j = (it >= kStages ? it - kStages : 0); j < it; ++j) {
          if (rank == 0) drain_wait(&full_bar[j % kStages], (j / kStages) & 1u);
          if constexpr (has_cvt(MODE))
            drain_wait(&afull_bar[j % kStages], (j / kStages) & 1u);
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0 && rank == 0) {
      constexpr bool kMnOut = is_dh(MODE) || MODE == MODE_DW;  // B MN-major, N = hidden
      uint32_t it = 0, tile_it = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        WorkItem wk;
        if (!wl.get(args, n_ru, k_iters, i, wk)) break;
        if (wk.empty()) continue;
        int ru, col, t0, t1;
        decode_unit(wk.u, n_ru, n_cols, args.group_rows, ru, col);
        unit_tiles<MODE>(args, n_cols, col, t0, t1);
        for (int t = t0; t < t1 && ok; ++t, ++tile_it) {
          const uint32_t buf = tile_it % C::kNBuf;
          const uint32_t use = tile_it / C::kNBuf;
          if (!mbar_wait(&tempty_bar[buf], (use & 1u) ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * BN;
          // Instruction descriptor per accumulator (0: skipped, past the hidden size).
          uint32_t idesc[C::kNAcc];
#pragma unroll
          for (int na = 0; na < C::kNAcc; ++na) {
            const int n = kMnOut ? mn_out_cols<CTAS>(args, t * C::kTileN + na * BN) : BN;
            idesc[na] = n == 0 ? 0u : idesc_bf16(BM * CTAS, n, MODE == MODE_DW, kMnOut);
          }
          for (int k = wk.kb; k < wk.ke; ++k, ++it) {
            const int s = it % kStages;
            const uint32_t round = it / kStages;
            if (!mbar_wait(&full_bar[s], round & 1u, abort_flag, args.status)) {
              ok = false;
              break;
            }
            if constexpr (has_cvt(MODE)) {
              if (!mbar_wait(&cvt_bar[s], round & 1u, abort_flag, args.status)) {
                ok = false;
                break;
              }
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + s * C::kStageBytes);
            const uint32_t b_addr = a_addr + C::kKSub * A_BYTES;
#pragma unroll
            for (int kq = 0; kq < C::kKSub * (BK / 16); ++kq) {
              const int kk = kq % (BK / 16);                      // K step in its slice
              const uint32_t a_sl = a_addr + (kq / (BK / 16)) * A_BYTES;  // slice base
              const uint32_t b_sl = b_addr + (kq / (BK / 16)) * C::kBBytes;
              // K-major, 128B swizzle: K advances by 32 bytes inside the atom;
              // 8-row groups are 1024 bytes apart.
              const uint64_t adesc = MODE == MODE_DW
                                         ? sdesc_sw128(a_sl + kk * 2048, BK * 64 * 2, 1024)
                                         : sdesc_sw128(a_sl + kk * 32, 16, 1024);
              uint64_t bdesc;
              if (is_dh(MODE) || MODE == MODE_DW) {
                // MN-major, 128B swizzle: 64-wide N blocks 8 KB apart (LBO),
                // 8-deep K groups 1 KB apart (SBO); K advances 16 rows.
                bdesc = sdesc_sw128(b_sl + kk * 2048, BK * 64 * 2, 1024);
              } else {
                bdesc = sdesc_sw128(b_sl + kk * 32, 16, 1024);
              }
              // The first MMA of the tile (or piece) overwrites the accumulator.
              const uint32_t acc = (k != wk.kb || kq != 0) ? 1u : 0u;
#pragma unroll
              for (int na = 0; na < C::kNAcc; ++na) {
                // Accumulator na: B columns na*256.. (its own B boxes), TMEM columns na*256..
                if (idesc[na] == 0u) continue;
                const uint64_t bd = bdesc + ((static_cast<uint64_t>(na) * C::kBRows * BK * 2) >> 4);
                if (CTAS == 2) tc_mma_bf16_pair(d_tmem + na * BN, adesc, bd, idesc[na], acc);
                else tc_mma_bf16(d_tmem + na * BN, adesc, bd, idesc[na], acc);
              }
            }
            if (CTAS == 2) tc_commit_pair_multicast(&empty_bar[s], 0x3);
            else tc_commit(&empty_bar[s]);
          }
          if (!ok) break;
          if (CTAS == 2) tc_commit_pair_multicast(&tfull_bar[buf], 0x3);
          else tc_commit(&tfull_bar[buf]);
        }
      }
      // Make sure every MMA issued by this thread has finished before TMEM is
      // released (matters only on the abort path).
      if (CTAS == 2) tc_commit_pair(&drain_bar); else tc_commit(&drain_bar);
      drain_wait(&drain_bar, 0);
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int lrow_in_tile = q * 32 + lane;
    const int part = (warp - 2) >> 2;  // 0: epilogue warps; 1: converter-only (has_cvt)
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    uint32_t tile_it = 0;
    bool ok = true;
    // Where this CTA's epilogue warps report a drained accumulator: the
    // leader's barrier (pair) or the CTA's own.
    const uint32_t tempty_addr0 =
        CTAS == 2 ? mapa_shared(smem_u32(&tempty_bar[0]), 0) : smem_u32(&tempty_bar[0]);
    const uint32_t cvt_addr0 =
        CTAS == 2 ? mapa_shared(smem_u32(&cvt_bar[0]), 0) : smem_u32(&cvt_bar[0]);
    uint32_t cit = 0;  // has_cvt: A stages converted so far
    // kTmaStore: this warp's two staging buffers and the boxes it has stored.
    uint8_t* const stage_out = smem + C::kStages * C::kStageBytes + q * 2 * C::kStoreBufBytes;
    uint32_t n_stores = 0;
    for (int i = 0; ok; ++i) {
      WorkItem wk;
      if (!wl.get(args, n_ru, k_iters, i, wk)) break;
      if (wk.empty()) continue;
      int ru, col, t0, t1;
      decode_unit(wk.u, n_ru, n_cols, args.group_rows, ru, col);
      unit_tiles<MODE>(args, n_cols, col, t0, t1);
      const int li = ru * CTAS + static_cast<int>(rank);
      const bool block_ok = li < n_rb;
      const int lrow = li * BM + lrow_in_tile;  // row of the chunk workspace
      const long long grow_l = block_ok ? row_of(args, li * BM + lrow_in_tile) : -1;
      const bool valid = grow_l >= 0 && grow_l < args.n_total;
      const long long grow = valid ? grow_l : 0;

      // Per-row state.
      float m2 = -INFINITY, ssum = 0.f;  // FWD
      int y = -1;
      float lse2 = 0.f, gval = 0.f;      // BWDG
      RowCvt rc;                         // DHS, UAC: conversion constants
      rc.zero = true;
      rc.y = -1;
      rc.c = 0.f;
      rc.neg = false;
      rc.scale = 1.f;
      rc.shift2 = 0.f;
      rc.ytarget = 0.f;
      UaccRow ur;                        // UAC, UAP: the U update's row constants
      ur.zero = true;
      if (is_fwd(MODE)) {
        if (valid && (args.mask == nullptr || args.mask[grow] != 0)) y = args.ids[grow];
      } else if (MODE == MODE_BWDG) {
        if (valid) {
          gval = args.g[grow];
          lse2 = args.lse[grow] * kLog2e;
          if (gval != 0.f) y = args.ids[grow];
        }
      } else if (MODE == MODE_DHS) {
        if (valid) {
          gval = args.g[grow];
          if (gval != 0.f) {
            lse2 = args.lse[grow] * kLog2e;
            const float zy = args.zy[grow];  // fp32 target logit
            rc.zero = false;
            rc.y = args.ids[grow];
            rc.c = log2f(fabsf(gval)) - lse2;
            rc.neg = gval > 0.f;
            rc.scale = fabsf(gval);
            rc.shift2 = -lse2;
            const float yt = (gval - gval * ex2(fmaf(zy, kLog2e, -lse2))) * dz_of_logit(args, zy);
            rc.ytarget = rc.neg ? -yt : yt;
          }
        }
      } else if (is_uacc(MODE)) {
        ur = uacc_row(args, grow, valid);
        if (!ur.zero) {
          rc.zero = false;
          rc.y = ur.y;
          rc.c = -ur.mcur;
          rc.shift2 = -ur.mcur;
        }
      }

      if constexpr (has_cvt(MODE)) {
        // Every A stage of this unit, as it lands: fp16 logits -> bf16 in
        // place (this thread's part of its row), then tell the MMA issuer.
        // Stage k is box k of the stored block. The box maxima of the next
        // kPre stages are loaded at the start of each group of kPre stages,
        // into registers that no instruction touches until the group after
        // (a register move of a load in flight would wait for it); rows that
        // contribute nothing need none.
        constexpr int kPre = 4;
        const float* bm = args.box_max + lrow;
        auto box_max_of = [&](int k) {
          return (!rc.zero && k < wk.ke) ? __ldg(bm + static_cast<long long>(k) * args.ldM)
                                         : 0.f;
        };
        float zc[kPre], zn[kPre];
#pragma unroll
        for (int j = 0; j < kPre; ++j) zc[j] = box_max_of(wk.kb + j);
        for (int k0 = wk.kb; k0 < wk.ke && ok; k0 += kPre) {
#pragma unroll
          for (int j = 0; j < kPre; ++j) zn[j] = box_max_of(k0 + kPre + j);
#pragma unroll
          for (int j = 0; j < kPre; ++j) {
            const int k = k0 + j;
            if (k >= wk.ke || !ok) break;
            const int s = static_cast<int>(cit % kStages);
            if (!mbar_wait(&afull_bar[s], (cit / kStages) & 1u, abort_flag, args.status)) {
              ok = false;
              break;
            }
            constexpr int kNch = 8 / C::kCvtGroups;
            stage_row_to_bf16<kNch>(args, smem + s * C::kStageBytes, lrow_in_tile, part * kNch,
                                    args.v0 + k * BK, rc, zc[j]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (CTAS == 2) mbar_arrive_cluster(cvt_addr0 + static_cast<uint32_t>(s) * 8u);
              else mbar_arrive(&cvt_bar[s]);
            }
            ++cit;
          }
#pragma unroll
          for (int j = 0; j < kPre; ++j) zc[j] = zn[j];
        }
        if (!ok) break;
        if (part != 0) continue;  // converter-only warps: no epilogue
      }

      for (int t = t0; t < t1; ++t, ++tile_it) {
        const uint32_t buf = tile_it % C::kNBuf;
        const uint32_t use = tile_it / C::kNBuf;
        if (!mbar_wait(&tfull_bar[buf], use & 1u, abort_flag, args.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tbase = tmem_base + lane_addr + buf * BN;

        if (MODE == MODE_FWD) {
#pragma unroll 1
          for (int c = 0; c < C::kTileN / 32; ++c) {
            const int col0 = args.v0 + t * C::kTileN + c * 32;
            if (col0 >= args.vocab) break;  // warp-uniform
            float v[32];
            tmem_ld32(tbase + c * 32, v);
            logit_transform(args, v);
            if (col0 + 32 > args.vocab) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (col0 + j >= args.vocab) v[j] = -INFINITY;
            }
            const unsigned off = static_cast<unsigned>(y - col0);
            if (off < 32u) {
              float z = 0.f;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (static_cast<unsigned>(j) == off) z = v[j];
              args.zy[grow] = z;
            }
            float mx0 = fmaxf(v[0], v[1]), mx1 = fmaxf(v[2], v[3]);
#pragma unroll
            for (int j = 4; j < 32; j += 4) {
              mx0 = fmaxf(mx0, fmaxf(v[j], v[j + 1]));
              mx1 = fmaxf(mx1, fmaxf(v[j + 2], v[j + 3]));
            }
            const float mn = fmaxf(m2, fmaxf(mx0, mx1) * kLog2e);
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              s0 += ex2(fmaf(v[j], kLog2e, -mn));
              s1 += ex2(fmaf(v[j + 1], kLog2e, -mn));
              s2 += ex2(fmaf(v[j + 2], kLog2e, -mn));
              s3 += ex2(fmaf(v[j + 3], kLog2e, -mn));
            }
            ssum = fmaf(ssum, ex2(m2 - mn), (s0 + s1) + (s2 + s3));
            m2 = mn;
          }
        } else if (MODE == MODE_FWDS) {
          // One 64-column box at a time. The box is stored in fp16 relative to
          // its own maximum, which goes beside it in fp32 (box-major, so a warp
          // writes 32 consecutive rows). Stored values then lie in [-inf, 0]:
          // no logit overflows fp16, and the columns near the box maximum (the
          // ones that carry probability) keep fp16's finest spacing whatever
          // the logits' magnitude. Unshifted, a logit near 40 kept only
          // 2^-6 of absolute precision, i.e. 1.6 % of its softmax term.
#pragma unroll 1
          for (int c = 0; c < C::kTileN / 64; ++c) {
            const int lcol = t * C::kTileN + c * 64;  // column of the stored block
            const int col0 = args.v0 + lcol;           // vocabulary column
            if (col0 >= args.vocab) break;  // warp-uniform
            float lo[32], hi[32];
            tmem_ld32(tbase + c * 64, lo);
            tmem_ld32(tbase + c * 64 + 32, hi);
            logit_transform(args, lo);
            logit_transform(args, hi);
            if (col0 + 64 > args.vocab) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                if (col0 + j >= args.vocab) lo[j] = -INFINITY;
                if (col0 + 32 + j >= args.vocab) hi[j] = -INFINITY;
              }
            }
            float mx0 = fmaxf(lo[0], hi[0]), mx1 = fmaxf(lo[1], hi[1]);
#pragma unroll
            for (int j = 2; j < 32; j += 2) {
              mx0 = fmaxf(mx0, fmaxf(lo[j], hi[j]));
              mx1 = fmaxf(mx1, fmaxf(lo[j + 1], hi[j + 1]));
            }
            const float mb = fmaxf(mx0, mx1);  // finite: col0 < V
            // Stored: z log2e - mb2 in fp16 with mb2 = mb log2e beside it in
            // fp32, so that every reader's exponent is the stored value plus
            // fp32 constants, and adding mb2 back cancels its rounding.
            const float nmb2 = -mb * kLog2e;
            const unsigned off = static_cast<unsigned>(y - col0);
            if (off < 64u) {
              float z = 0.f;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                if (static_cast<unsigned>(j) == off) z = lo[j];
                if (static_cast<unsigned>(j + 32) == off) z = hi[j];
              }
              args.zy[grow] = z;
            }
            if constexpr (C::kTmaStore) {
              if (block_ok) {
                // The box fills one 32-row x 128-byte staging buffer; the
                // store clips the columns past V.
                uint8_t* buf = stage_out + (n_stores & 1u) * C::kStoreBufBytes;
                if (lane == 0) bulk_wait_group_read<1>();  // this buffer's last store read it
                __syncwarp();
                uint4* srow = reinterpret_cast<uint4*>(buf + lane * 128);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  srow[j ^ (lane & 7)] =
                      make_uint4(pack_f16x2(fmaf(lo[8 * j], kLog2e, nmb2), fmaf(lo[8 * j + 1], kLog2e, nmb2)),
                                 pack_f16x2(fmaf(lo[8 * j + 2], kLog2e, nmb2), fmaf(lo[8 * j + 3], kLog2e, nmb2)),
                                 pack_f16x2(fmaf(lo[8 * j + 4], kLog2e, nmb2), fmaf(lo[8 * j + 5], kLog2e, nmb2)),
                                 pack_f16x2(fmaf(lo[8 * j + 6], kLog2e, nmb2), fmaf(lo[8 * j + 7], kLog2e, nmb2)));
                  srow[(4 + j) ^ (lane & 7)] =
                      make_uint4(pack_f16x2(fmaf(hi[8 * j], kLog2e, nmb2), fmaf(hi[8 * j + 1], kLog2e, nmb2)),
                                 pack_f16x2(fmaf(hi[8 * j + 2], kLog2e, nmb2), fmaf(hi[8 * j + 3], kLog2e, nmb2)),
                                 pack_f16x2(fmaf(hi[8 * j + 4], kLog2e, nmb2), fmaf(hi[8 * j + 5], kLog2e, nmb2)),
                                 pack_f16x2(fmaf(hi[8 * j + 6], kLog2e, nmb2), fmaf(hi[8 * j + 7], kLog2e, nmb2)));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                  tma_store_2d(&map_c, buf, lcol, li * BM + q * 32);
                  bulk_commit_group();
                }
                ++n_stores;
                args.box_max[static_cast<long long>(lcol >> 6) * args.ldM + lrow] = -nmb2;
              }
            } else if (valid) {
              uint16_t* dst = args.S + static_cast<long long>(lrow) * args.ldS + lcol;
              if (col0 + 64 <= args.vocab) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  st_global_v4(dst + j * 8, pack_f16x2(fmaf(lo[8 * j], kLog2e, nmb2), fmaf(lo[8 * j + 1], kLog2e, nmb2)),
                               pack_f16x2(fmaf(lo[8 * j + 2], kLog2e, nmb2), fmaf(lo[8 * j + 3], kLog2e, nmb2)),
                               pack_f16x2(fmaf(lo[8 * j + 4], kLog2e, nmb2), fmaf(lo[8 * j + 5], kLog2e, nmb2)),
                               pack_f16x2(fmaf(lo[8 * j + 6], kLog2e, nmb2), fmaf(lo[8 * j + 7], kLog2e, nmb2)));
                  st_global_v4(dst + 32 + j * 8, pack_f16x2(fmaf(hi[8 * j], kLog2e, nmb2), fmaf(hi[8 * j + 1], kLog2e, nmb2)),
                               pack_f16x2(fmaf(hi[8 * j + 2], kLog2e, nmb2), fmaf(hi[8 * j + 3], kLog2e, nmb2)),
                               pack_f16x2(fmaf(hi[8 * j + 4], kLog2e, nmb2), fmaf(hi[8 * j + 5], kLog2e, nmb2)),
                               pack_f16x2(fmaf(hi[8 * j + 6], kLog2e, nmb2), fmaf(hi[8 * j + 7], kLog2e, nmb2)));
                }
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  if (col0 + j < args.vocab)
                    dst[j] = static_cast<uint16_t>(pack_f16x2(fmaf(lo[j], kLog2e, nmb2), 0.f) & 0xffffu);
                  if (col0 + 32 + j < args.vocab)
                    dst[32 + j] = static_cast<uint16_t>(pack_f16x2(fmaf(hi[j], kLog2e, nmb2), 0.f) & 0xffffu);
                }
              }
              args.box_max[static_cast<long long>(lcol >> 6) * args.ldM + lrow] = -nmb2;
            }
            const float mn = fmaxf(m2, -nmb2);
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              s0 += ex2(fmaf(lo[j], kLog2e, -mn));
              s1 += ex2(fmaf(lo[j + 1], kLog2e, -mn));
              s2 += ex2(fmaf(hi[j], kLog2e, -mn));
              s3 += ex2(fmaf(hi[j + 1], kLog2e, -mn));
            }
            ssum = fmaf(ssum, ex2(m2 - mn), (s0 + s1) + (s2 + s3));
            m2 = mn;
          }
        } else if (MODE == MODE_BWDG) {
          __nv_bfloat16* grow_ptr = args.G + static_cast<long long>(lrow) * args.ldG + t * BN;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            const int col0 = args.v0 + t * BN + c * 32;  // global vocab index
            float v[32];
            tmem_ld32(tbase + c * 32, v);
            const float ng = -gval;
            const unsigned off = static_cast<unsigned>(y - col0);
            if (gval == 0.f) {
              // Rows that do not count (masked, padding, past N): exact zeros.
              // Their lse is 0, so the exponential below could overflow and
              // 0 * inf would leave NaN in G.
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0.f;
            } else if (args.xmode != 2) {
              // z' = k S (k = 1 without a transform): G = k g (onehot - p).
              const float k = args.xmode == 1 ? args.k0 : 1.f;
              const float kl = k * kLog2e;
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = ng * ex2(fmaf(v[j], kl, -lse2));
              if (off < 32u) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (static_cast<unsigned>(j) == off) v[j] += gval;
              }
              if (args.xmode == 1) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] *= k;
              }
            } else {
              // Softcap: z' = k2 u, u = tanh(k1 S), dz'/dS = k0 (1 - u^2).
              const float k2l = args.k2 * kLog2e;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float u = tanh_sfu(v[j] * args.k1);
                const float d = args.k0 * fmaf(-u, u, 1.f);
                const float pg = ng * ex2(fmaf(u, k2l, -lse2));
                v[j] = (static_cast<unsigned>(j) == off ? pg + gval : pg) * d;
              }
            }
            if (col0 + 32 > args.vocab) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (col0 + j >= args.vocab) v[j] = 0.f;
            }
            // Rows past N in an active block come out exactly 0 (zero-filled
            // hidden rows, g = 0); they are written too, so that the G block
            // holds no stale bytes for the dW GEMM.
            if constexpr (C::kTmaStore) {
              // map_c: the chunk's G block [rows][ldG], 64 x 32 boxes; chunk c
              // fills 16-byte pieces 4 (c & 1) .. +3 of this row of the box.
              if (block_ok) {
                uint8_t* buf = stage_out + (n_stores & 1u) * C::kStoreBufBytes;
                if ((c & 1) == 0) {
                  if (lane == 0) bulk_wait_group_read<1>();  // this buffer's last store read it
                  __syncwarp();
                }
                uint4* srow = reinterpret_cast<uint4*>(buf + lane * 128);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  srow[((c & 1) * 4 + j) ^ (lane & 7)] =
                      make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]),
                                 pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                 pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                                 pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
                if ((c & 1) == 1) {
                  fence_proxy_async_smem();
                  __syncwarp();
                  if (lane == 0) {
                    tma_store_2d(&map_c, buf, t * BN + (c >> 1) * 64, li * BM + q * 32);
                    bulk_commit_group();
                  }
                  ++n_stores;
                }
              }
            } else if (block_ok) {
              uint32_t p[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) p[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
              __nv_bfloat16* dst = grow_ptr + c * 32;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                st_global_v4(dst + j * 8, p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
            }
          }
        } else if (MODE == MODE_DW && C::kTmaStore) {
          // map_c: dW[v0 : v0 + dw_rows) as fp32 [rows][hidden], 32 x 32 boxes;
          // rows past the block and columns past D are clipped by the store.
          const int vrow0 = ru * CTAS * BM + static_cast<int>(rank) * BM + q * 32;
          if (vrow0 < args.dw_rows) {  // warp-uniform
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
              const int d0 = t * BN + c * 32;
              if (d0 >= args.hidden) break;  // warp-uniform
              float v[32];
              tmem_ld32(tbase + c * 32, v);
              if (k_iters == 0) {  // no row of the chunk is active: nothing accumulated
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
              }
              uint8_t* buf = stage_out + (n_stores & 1u) * C::kStoreBufBytes;
              if (lane == 0) bulk_wait_group_read<1>();  // this buffer's last store read it
              __syncwarp();
              uint4* srow = reinterpret_cast<uint4*>(buf + lane * 128);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                srow[j ^ (lane & 7)] =
                    make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                               __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                if (args.first) tma_store_2d(&map_c, buf, d0, vrow0);
                else tma_reduce_add_2d(&map_c, buf, d0, vrow0);
                bulk_commit_group();
              }
              ++n_stores;
            }
          }
        } else if (MODE == MODE_DW) {
          const int vrow = ru * CTAS * BM + static_cast<int>(rank) * BM + lrow_in_tile;
          const bool vvalid = vrow < args.dw_rows;
          float* out = args.dW + (static_cast<long long>(args.v0) + vrow) * args.hidden;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            const int d0 = t * BN + c * 32;
            if (d0 >= args.hidden) break;  // warp-uniform
            float v[32];
            tmem_ld32(tbase + c * 32, v);
            if (k_iters == 0) {  // no row of the chunk is active: nothing accumulated
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
            if (vvalid) {
#pragma unroll
              for (int j8 = 0; j8 < 4; ++j8) {
                if (d0 + j8 * 8 >= args.hidden) break;
                float* o8 = out + d0 + j8 * 8;
                if (!args.first) {
                  const float4 x0 = *reinterpret_cast<const float4*>(o8);
                  const float4 x1 = *reinterpret_cast<const float4*>(o8 + 4);
                  v[j8 * 8 + 0] += x0.x;
                  v[j8 * 8 + 1] += x0.y;
                  v[j8 * 8 + 2] += x0.z;
                  v[j8 * 8 + 3] += x0.w;
                  v[j8 * 8 + 4] += x1.x;
                  v[j8 * 8 + 5] += x1.y;
                  v[j8 * 8 + 6] += x1.z;
                  v[j8 * 8 + 7] += x1.w;
                }
                *reinterpret_cast<float4*>(o8) =
                    make_float4(v[j8 * 8 + 0], v[j8 * 8 + 1], v[j8 * 8 + 2], v[j8 * 8 + 3]);
                *reinterpret_cast<float4*>(o8 + 4) =
                    make_float4(v[j8 * 8 + 4], v[j8 * 8 + 5], v[j8 * 8 + 6], v[j8 * 8 + 7]);
              }
            }
          }
        } else if (is_uacc(MODE)) {
          // U (+)= this block's P W, rescaled to the running maximum; on the
          // last block dH = g (1 - p_y) f'_y W_y - g 2^(M - lse2) U. A cut piece
          // of the tail split leaves its partial tile for the fixup instead.
#pragma unroll 1
          for (int c = 0; c < C::kTileN / 32; ++c) {
            const int d0 = t * C::kTileN + c * 32;
            if (d0 >= args.hidden) break;  // warp-uniform
            float v[32];
            tmem_ld32(tbase + c * 32, v);
            if (wk.cut) {
              if (valid) {
                float* sp = ts_slot_ptr(args, wk.slot, static_cast<int>(rank), CTAS, C::kTileN) +
                            (c * 8 * BM + lrow_in_tile) * 4;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                  st_global_v4(sp + jj * BM * 4, __float_as_uint(v[4 * jj]),
                               __float_as_uint(v[4 * jj + 1]), __float_as_uint(v[4 * jj + 2]),
                               __float_as_uint(v[4 * jj + 3]));
              }
              continue;
            }
            if (valid) {
              float* accp = args.acc + static_cast<long long>(lrow) * args.hidden + d0;
              __nv_bfloat16* outp = args.dH + static_cast<long long>(grow) * args.hidden + d0;
              const __nv_bfloat16* wy =
                  args.W + static_cast<long long>(ur.y < 0 ? 0 : ur.y) * args.hidden + d0;
#pragma unroll
              for (int j8 = 0; j8 < 4; ++j8) {
                if (d0 + j8 * 8 >= args.hidden) break;
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = v[j8 * 8 + e];
                uacc_update8(args, ur, x, accp + j8 * 8, outp + j8 * 8, wy + j8 * 8);
              }
            }
          }
        } else {  // MODE_DH
#pragma unroll 1
          for (int c = 0; c < C::kTileN / 32; ++c) {
            const int d0 = t * C::kTileN + c * 32;
            if (d0 >= args.hidden) break;  // warp-uniform
            float v[32];
            tmem_ld32(tbase + c * 32, v);
            if constexpr (MODE == MODE_DHS) {
              if (rc.neg) {  // the converter wrote G / sigma
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = -v[e];
              }
            }
            if (wk.cut) {
              // A piece of a split unit: its fp32 partial tile goes to its slot.
              if (valid) {
                float* sp = ts_slot_ptr(args, wk.slot, static_cast<int>(rank), CTAS, C::kTileN) +
                            (c * 8 * BM + lrow_in_tile) * 4;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                  st_global_v4(sp + jj * BM * 4, __float_as_uint(v[4 * jj]),
                               __float_as_uint(v[4 * jj + 1]), __float_as_uint(v[4 * jj + 2]),
                               __float_as_uint(v[4 * jj + 3]));
              }
              continue;
            }
            if (valid) {
              float* accp = args.acc + static_cast<long long>(lrow) * args.hidden + d0;
              __nv_bfloat16* outp =
                  args.dH + static_cast<long long>(grow) * args.hidden + d0;
#pragma unroll
              for (int j8 = 0; j8 < 4; ++j8) {
                if (d0 + j8 * 8 >= args.hidden) break;
                float* a8 = accp + j8 * 8;
                if (!args.first) {
                  const float4 x0 = *reinterpret_cast<const float4*>(a8);
                  const float4 x1 = *reinterpret_cast<const float4*>(a8 + 4);
                  v[j8 * 8 + 0] += x0.x;
                  v[j8 * 8 + 1] += x0.y;
                  v[j8 * 8 + 2] += x0.z;
                  v[j8 * 8 + 3] += x0.w;
                  v[j8 * 8 + 4] += x1.x;
                  v[j8 * 8 + 5] += x1.y;
                  v[j8 * 8 + 6] += x1.z;
                  v[j8 * 8 + 7] += x1.w;
                }
                if (args.last) {
                  st_global_v4(outp + j8 * 8, pack_bf16x2(v[j8 * 8 + 0], v[j8 * 8 + 1]),
                               pack_bf16x2(v[j8 * 8 + 2], v[j8 * 8 + 3]),
                               pack_bf16x2(v[j8 * 8 + 4], v[j8 * 8 + 5]),
                               pack_bf16x2(v[j8 * 8 + 6], v[j8 * 8 + 7]));
                } else {
                  *reinterpret_cast<float4*>(a8) =
                      make_float4(v[j8 * 8 + 0], v[j8 * 8 + 1], v[j8 * 8 + 2], v[j8 * 8 + 3]);
                  *reinterpret_cast<float4*>(a8 + 4) =
                      make_float4(v[j8 * 8 + 4], v[j8 * 8 + 5], v[j8 * 8 + 6], v[j8 * 8 + 7]);
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (CTAS == 2) mbar_arrive_cluster(tempty_addr0 + buf * 8u);
          else mbar_arrive(&tempty_bar[buf]);
        }
      }
      if (is_fwd(MODE) && ok && valid) {
        args.part_m[static_cast<long long>(args.part_slot0 + col) * args.part_ld + grow] = m2;
        args.part_s[static_cast<long long>(args.part_slot0 + col) * args.part_ld + grow] = ssum;
        if (col == 0) {  // slots no split of this launch writes: merge as nothing
          for (int sl = n_cols; sl < args.max_cols; ++sl) {
            args.part_m[static_cast<long long>(args.part_slot0 + sl) * args.part_ld + grow] = -INFINITY;
            args.part_s[static_cast<long long>(args.part_slot0 + sl) * args.part_ld + grow] = 0.f;
          }
        }
      }
    }
    if constexpr (C::kTmaStore) {
      if (lane == 0) bulk_wait_group<0>();  // every staged box written before the exit
    }
  }

  tc_fence_before();
  if (CTAS == 2) cluster_sync(); else __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    if (CTAS == 2) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Adds the pieces of every dH-type unit that the tail split cut (see TailSplit)
// in a fixed order, its main piece and then its tails in pair order, and
// writes the unit's bf16 dH rows (kUacc: applies the single pass's U update to
// the sum instead, as the U GEMM's epilogue does). Grid: (the launch's host-side bound on units) x (32-
// column chunks of a unit); one thread per row of the unit. Units that ran
// whole return at once. `a` is the dH launch's own TileArgs.
template <int CTAS, bool kUacc>
__global__ void __launch_bounds__(BM * CTAS) tail_fixup_kernel(const TileArgs a) {
  constexpr int kTileN = PairCfg<MODE_DH, CTAS>::kTileN;
  __shared__ TailSplit sp_sh;
  __shared__ long long p0_sh;
  const int n_rb = launch_row_blocks(a);
  const int n_ru = (n_rb + CTAS - 1) / CTAS;
  const int n_units = n_ru * a.n_cols;
  const int u = static_cast<int>(blockIdx.x);
  // Only units of a last round with fewer units than pairs can be cut.
  if (a.ts_slots <= 0 || u >= n_units || u < n_units - n_units % a.ts_slots) return;
  int ru, col;
  decode_unit(u, n_ru, a.n_cols, a.group_rows, ru, col);
  const int c = static_cast<int>(blockIdx.y);
  const int d0 = col * kTileN + c * 32;
  if (d0 >= a.hidden) return;
  if (threadIdx.x == 0) {
    sp_sh = tail_split<CTAS>(a, n_ru, n_units, a.ts_slots);
    p0_sh = sp_sh.n_tail > 0 ? ts_tail_prefix(a, n_ru, sp_sh, u) : 0;
  }
  __syncthreads();
  const TailSplit& sp = sp_sh;
  if (sp.n_tail == 0) return;
  const bool last = col == a.n_cols - 1;
  const int m = last ? sp.m_l : sp.m_f;
  const int cs = last ? sp.cs_l : sp.cs_f;
  const long long t = last ? sp.t_l : sp.t_f;
  if (t == 0) return;  // the main piece was the whole unit
  const long long p0 = p0_sh;
  const int qa = ts_tail_pair_of(sp, p0);
  const int qb = ts_tail_pair_of(sp, p0 + t - 1);
  // Stages of tail pair q's piece of this unit (as ts_tail_piece).
  auto piece = [&](int q, int& kb, int& ke) {
    const long long q0 = ts_tail_start(sp, q), q1 = ts_tail_start(sp, q + 1);
    kb = m + static_cast<int>((max(q0, p0) - p0) / cs);
    ke = m + static_cast<int>((min(q1, p0 + t) - p0) / cs);
  };
  if (m == 0) {
    // No main piece: a single tail piece then covered the whole unit.
    int n = 0;
    for (int q = qa; q <= qb; ++q) {
      int kb, ke;
      piece(q, kb, ke);
      n += ke > kb;
    }
    if (n <= 1) return;
  }

  const int rank = static_cast<int>(threadIdx.x) / BM;
  const int lrow = static_cast<int>(threadIdx.x) % BM;
  const int li = ru * CTAS + rank;
  if (li >= n_rb) return;
  const long long grow = row_of(a, li * BM + lrow);
  if (grow < 0 || grow >= a.n_total) return;
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = 0.f;
  auto add_slot = [&](int slot) {
    const float* src = ts_slot_ptr(a, slot, rank, CTAS, kTileN) + (c * 8 * BM + lrow) * 4;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const float4 x = *reinterpret_cast<const float4*>(src + jj * BM * 4);
      v[4 * jj] += x.x;
      v[4 * jj + 1] += x.y;
      v[4 * jj + 2] += x.z;
      v[4 * jj + 3] += x.w;
    }
  };
  if (m > 0) add_slot(ts_main_slot(sp, u));
  for (int q = qa; q <= qb; ++q) {
    int kb, ke;
    piece(q, kb, ke);
    if (ke > kb) add_slot(ts_tail_slot(sp, u, q));
  }
  __nv_bfloat16* out = a.dH + grow * a.hidden + d0;
  if constexpr (kUacc) {
    // The single pass's U update, as the U GEMM's epilogue does it.
    const UaccRow ur = uacc_row(a, grow, true);
    float* accp = a.acc + (static_cast<long long>(li) * BM + lrow) * a.hidden + d0;
    const __nv_bfloat16* wy = a.W + static_cast<long long>(ur.y < 0 ? 0 : ur.y) * a.hidden + d0;
#pragma unroll
    for (int j8 = 0; j8 < 4; ++j8) {
      if (d0 + j8 * 8 >= a.hidden) break;
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = v[j8 * 8 + e];
      uacc_update8(a, ur, x, accp + j8 * 8, out + j8 * 8, wy + j8 * 8);
    }
  } else {
#pragma unroll
    for (int j8 = 0; j8 < 4; ++j8) {
      if (d0 + j8 * 8 >= a.hidden) break;
      st_global_v4(out + j8 * 8, pack_bf16x2(v[j8 * 8], v[j8 * 8 + 1]),
                   pack_bf16x2(v[j8 * 8 + 2], v[j8 * 8 + 3]),
                   pack_bf16x2(v[j8 * 8 + 4], v[j8 * 8 + 5]),
                   pack_bf16x2(v[j8 * 8 + 6], v[j8 * 8 + 7]));
    }
  }
}

}  // namespace grpo
