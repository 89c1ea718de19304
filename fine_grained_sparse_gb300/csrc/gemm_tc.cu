// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA.  bf16 operands, fp32 accumulation.
//
// What they compute ("Kimi K2 MoE", section 2: SwiGLU experts; section 3:
// shared expert always on):
//   gate/up pass:  H[r, f] = SiLU(sum_k X[r,k] W_gate[e,f,k]) * sum_k X[r,k] W_up[e,f,k]
//   down pass:     Y[r, o] = w_r * sum_f H[r,f] W_down[e,o,f]
// for every row r of every routed expert e (rows come in tiles from the
// dispatch) and, as a second segment of the same launch, for every token of
// every shared expert.  The K3 latent projections and the router logits use
// the down-pass form (store mode) with one group.
//
// (The layer forward applies the routing weight w_r in its combine; the
// down pass stores the unscaled product there.)
//
// Swap-AB tiling.  The MMA's M side is a block of WEIGHT rows and its N side
// (16..256, a multiple of 16) a block of token rows of one expert, so an
// expert with few tokens still streams its weights through full-height MMAs.
// A unit is 256 weight rows -- two 128-row A tiles, two TMEM accumulators --
// against one token tile, so each token tile in shared memory feeds twice
// the MMA work.  Weights and tokens flow through separate rings with their
// own producer warps (the weight ring takes what shared memory the token
// ring leaves: 4 stages of 32 KB beside 3 token stages of 256 rows), but
// share one full and one empty barrier per k step, so the MMA issuer waits
// once and commits once per k step.
//   A tiles: 2 x (128 rows x 64 k) bf16, K-major, 128-byte swizzle (32 KB)
//   B tile:  up to nt rows x 64 k, same layout (one bulk copy of packed
//            activation rows, or 32-row TMA boxes)
//   D:       2 accumulators x N fp32 columns in TMEM (regions below).
// For the gate/up pass each A tile interleaves the two halves of W_gate_up
// [E, 2F, d] in 16-row slices: rows 32q..32q+15 are gate features
// 16q + (0..15) of the tile's 64 and rows 32q+16..32q+31 the up features with
// the same indices.  TMEM lane quadrant q (the one warp q%4 may read) thus
// holds both halves of 16 features, and the SwiGLU is one shuffle away.
// The epilogue turns each lane's column of 16 tokens into 16-byte rows of
// the output with 8 x 8 transposes inside lane octets.
//
// Units are ordered (segment, expert, output block, token tile) with the
// token tile fastest, so the CTAs that share an expert's weight block run
// side by side and the second reader finds the block in L2; the second
// segment (the shared experts) comes first.
//
// Warp roles (one CTA per SM, persistent over the units):
//   warp 0 lane 0: weight producer (bulk copies of packed weights, or TMA);
//   warp 1 lane 0: MMA issuer; warp 2 lane 0: token producer;
//   warps 3..10: epilogue, warp w reads lane quadrant w%4 of accumulator
//   (w-3)/4, or of the single accumulator's column chunks (w-3)/4, 2 + ...
//   (TMEM -> registers -> global stores);
//   bf16 single-CTA form, warp 11 lane 0: with token tiles of 128 rows or
//   more, the MMA issuer of the second accumulator (warp 1 then issues the
//   first's only; see the MMA issuers);
//   FP8 weights only, warps 11..18: converters (FP8 stage -> bf16 stage, in
//   shared memory or, with token tiles of at most 64 rows, in TMEM), and
//   warp 19 lane 0: the MMA issuer of the second accumulator.
// A segment with implicit token tiles whose weights fit in L2 may instead
// take its units token-tile-major (GemmSegment::b_major).
// Split weights (GemmParams::pieces = R > 1; the router, whose fp32 weight is
// held as three bf16 pieces side by side along K): units of one weight tile,
// and each k step is R weight steps -- the unit's tile of piece 0, 1, ... at
// that k step, each a 16 KB stage -- against one token stage, all
// accumulated into the unit's one accumulator.  The token tile is thus read
// into shared memory once for the R pieces; the weight producer arrives for
// the token producer on the full barriers of pieces 1 .. R-1.
// Every wait is bounded (%globaltimer); on expiry the CTA records
// MOE_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
#include <cudaTypedefs.h>

#include <stdlib.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fgs {

namespace {

constexpr int kBK = 64;                      // k per stage: one 128-byte swizzle row
constexpr uint32_t kATileBytes = 128 * 128;  // one A tile: 128 rows x 128 B
constexpr int kBBoxRows = 32;
constexpr uint32_t kBBoxBytes = kBBoxRows * 128;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (3 + kEpiWarps);
// bf16 single-CTA form: a twelfth warp issues the MMAs of the second
// accumulator (see the kernel's MMA issuers)
constexpr int kThreadsTwo = kThreads + 32;
// FP8 weights: eight more warps convert each landed FP8 stage into the bf16
// weight ring (two per SM sub-partition; the kernel then has 96 registers a
// thread)
constexpr int kConvWarps = 8;
// and a twentieth warp issues the MMAs of the second accumulator (see the
// MMA issuers; weights in TMEM)
constexpr int kThreadsFp8 = kThreads + 32 * kConvWarps + 32;
constexpr uint32_t kF8TileBytes = 128 * 64;  // one 128-row x 64-k FP8 tile
constexpr int kMaxStages = 12;
constexpr size_t kSmemBudget = 229376;  // pipeline bytes per CTA (224 KB)
constexpr int kSmemMax = 232448;        // the per-block limit (227 KB)

// Token-ring stage: nt rows; for a CTA pair, this CTA's half rounded up to
// whole 32-row boxes.
__host__ __device__ constexpr uint32_t b_stage_bytes_of(int nt, bool pair) {
  return pair ? static_cast<uint32_t>((nt / 2 + kBBoxRows - 1) / kBBoxRows) * kBBoxRows * 128u
              : static_cast<uint32_t>(nt) * 128u;
}

struct Unit {
  int seg, group, b_row, out_row, n_rows, ob, n_a, ntiles;
  int scale_row;  // row of the tile's first token in row_scale (the unpadded row space)
  int blk0;    // first 128-row A tile of the unit along O
  int k0, k1;  // k steps [k0, k1) of this unit (all of K unless split)
  int split;
};

__device__ __forceinline__ int ksplit_of(const GemmSegment* s) { return s->ksplit > 1 ? s->ksplit : 1; }

// output blocks of a segment: pairs of A tiles (one unit, or one unit of a
// CTA pair), or single tiles
__device__ __forceinline__ int out_blocks(const GemmParams& p, const GemmSegment* s) {
  if (p.pair && p.a_per_unit == 2) return (s->a128 + 3) / 4;  // four tiles over a CTA pair
  return (p.a_per_unit == 2 || p.pair) ? (s->a128 + 1) / 2 : s->a128;
}

__device__ __forceinline__ int segment_units(const GemmParams& p, const GemmSegment* s) {
  const int nt = s->nt;
  const int ob = out_blocks(p, s);
  if (s->tiles) return *s->ntiles * ob;
  return s->groups * ((s->rows + nt - 1) / nt) * ob * ksplit_of(s);
}

// The second segment's units (the shared experts: compute-heavy, their
// weights shared by all token tiles) come first, the first segment's
// weight-streaming units after them.
__device__ __forceinline__ Unit decode_unit_body(const GemmParams& p, int u, int units0,
                                                 int units1, int rank) {
  Unit x;
  x.seg = u < units1 ? 1 : 0;
  int local = x.seg ? u : u - units1;
  const GemmSegment* s = x.seg ? &p.seg[1] : &p.seg[0];
  const int nt = s->nt;
  const int OB = out_blocks(p, s);
  const int ns = ksplit_of(s);
  x.split = 0;
  if (ns > 1 && !s->b_major) {  // the K part is the outermost index of a split segment
    const int per = s->groups * ((s->rows + nt - 1) / nt) * OB;
    x.split = local / per;
    local -= x.split * per;
  }
  if (s->b_major && !s->tiles) {
    // (group, token tile) outermost, then the K part, the output block fastest
    const int tpg = (s->rows + nt - 1) / nt;
    const int inner = ns * OB;
    const int gt = local / inner;
    const int r = local - gt * inner;
    x.split = r / OB;
    x.ob = r - x.split * OB;
    const int g = gt / tpg;
    const int t0 = (gt - g * tpg) * nt;
    x.group = g;
    x.n_rows = min(nt, s->rows - t0);
    x.b_row = static_cast<int>(g * s->b_group_stride + t0);
    x.out_row = static_cast<int>(g * s->out_group_stride + t0);
    x.scale_row = x.out_row;
    x.ntiles = tpg;
  } else if (s->tiles) {
    // the units of one expert are [first_tile * OB, (first_tile + ntiles) * OB)
    const RowTile& any = s->tiles[local / OB];
    const int r = local - any.first_tile * OB;
    x.ob = r / any.ntiles;
    const RowTile& t = s->tiles[any.first_tile + (r - x.ob * any.ntiles)];
    x.group = t.expert;
    // packed activations live in the padded row space
    x.b_row = s->b_packed ? t.prow : t.row_start;
    x.out_row = s->out_packed ? t.prow : t.row_start;
    x.scale_row = t.row_start;
    x.n_rows = t.n_rows;
    x.ntiles = any.ntiles;
  } else {
    const int tpg = (s->rows + nt - 1) / nt;
    const int g = local / (tpg * OB);
    const int r = local - g * tpg * OB;
    x.ob = r / tpg;
    const int t0 = (r - x.ob * tpg) * nt;
    x.group = g;
    x.n_rows = min(nt, s->rows - t0);
    x.b_row = static_cast<int>(g * s->b_group_stride + t0);
    x.out_row = static_cast<int>(g * s->out_group_stride + t0);
    x.scale_row = x.out_row;
    x.ntiles = tpg;
  }
  // part j of a split K: k steps [j K / ns, (j + 1) K / ns)
  if (ns > 1) {  // (split + 1) k_steps < 2^31: ns <= 48 parts of at most 2^20 k steps
    x.k0 = x.split * s->k_steps / ns;
    x.k1 = (x.split + 1) * s->k_steps / ns;
  } else {
    x.k0 = 0;
    x.k1 = s->k_steps;
  }
  if (p.pair && p.a_per_unit == 2) {  // CTA `rank` of the pair takes tiles 4 ob + 2 rank, + 1
    x.blk0 = 4 * x.ob + 2 * rank;
    x.n_a = max(0, min(2, s->a128 - x.blk0));
  } else if (p.a_per_unit == 2) {
    x.blk0 = 2 * x.ob;
    x.n_a = min(2, s->a128 - 2 * x.ob);
  } else if (p.pair) {  // CTA `rank` of the pair takes tile 2 ob + rank
    x.blk0 = 2 * x.ob + rank;
    x.n_a = 1;
  } else {
    x.blk0 = x.ob;
    x.n_a = 1;
  }
  return x;
}

// Out of line in the bf16 kernels: inlined at each role's two call sites it
// was a tenth of the kernel's machine code.  The FP8 kernel keeps it inline
// (measured faster there: K2 decode 5.81 vs 6.22 ms per step).
__device__ __noinline__ Unit decode_unit_call(const GemmParams& p, int u, int units0, int units1,
                                              int rank) {
  return decode_unit_body(p, u, units0, units1, rank);
}

template <bool kInline>
__device__ __forceinline__ Unit decode_unit(const GemmParams& p, int u, int units0, int units1,
                                            int rank) {
  if constexpr (kInline)
    return decode_unit_body(p, u, units0, units1, rank);
  else
    return decode_unit_call(p, u, units0, units1, rank);
}

// Epilogue helpers over one 16-column TMEM load (16 tokens from tok0).  The
// epilogue walks a unit's tokens in such blocks in a loop that is not
// unrolled: the kernel's instruction footprint stays small (unrolled 64-token
// chunks of every output form made it hundreds of KB, and the epilogue warps
// then waited on instruction fetch).  Tokens past n_rows are computed on the
// accumulator's padding columns and not stored.

// SwiGLU: lane l < 16 holds the gate and lane l + 16 the up value of feature
// blk*64 + 16q + (l & 15); the gate lane forms h for tokens 0..7 of the block
// and the up lane for 8..15, each receiving the other half's values for its
// tokens, and after the transpose within each lane octet lane i holds one
// token's 8 features: one 16-byte store.  Packed output: plane blk, 8-feature
// chunk fc swizzled by row % 8.
__device__ __forceinline__ void swiglu_block(const uint32_t (&v)[16], int tok0, int n_rows,
                                             int lane, int q, int blk, __nv_bfloat16* out,
                                             bool out_packed, int64_t plane_rows, int64_t out_row,
                                             int64_t ld) {
  const bool is_gate = lane < 16;
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    float hh[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int a = j + e, b = 8 + j + e;
      const float own = __uint_as_float(is_gate ? v[a] : v[b]);
      const float send = __uint_as_float(is_gate ? v[b] : v[a]);
      const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
      const float g = is_gate ? own : recv;
      const float u = is_gate ? recv : own;
      hh[e] = silu_f(g) * u;
    }
    w[j >> 1] = pack_bf16x2(hh[0], hh[1]);
  }
  transpose8x8_b16(w, lane);
  const int oct = lane >> 3;
  const int fc = 2 * q + (oct & 1);
  const int tok = tok0 + (oct >> 1) * 8 + (lane & 7);
  if (tok < n_rows) {
    const int64_t row = out_row + tok;
    const int64_t off = out_packed ? (((static_cast<int64_t>(blk) * plane_rows + row) << 6) +
                                      ((fc ^ static_cast<int>(row & 7)) << 3))
                                   : row * ld + blk * 64 + fc * 8;
    *reinterpret_cast<uint4*>(out + off) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Store mode, bf16 rows of whole 16-byte chunks: v holds this lane's output
// column for the 16 tokens (scaled by scale[t] when kScale); after the
// transposes lane i of each octet writes tokens i and 8 + i of its octet's 8
// columns, dst being the octet's first column in the tile's first row.
template <bool kScale>
__device__ __forceinline__ void store_rows8_block(const uint32_t (&v)[16], const float* scale,
                                                  int tok0, int n_rows, __nv_bfloat16* dst,
                                                  int64_t ld, bool col_ok, int lane) {
  uint32_t w[2][4];
#pragma unroll
  for (int m = 0; m < 2; ++m) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float a = __uint_as_float(v[8 * m + 2 * k]), b = __uint_as_float(v[8 * m + 2 * k + 1]);
      if (kScale) {  // padding tokens read the tile's last row's scale
        a *= __ldg(scale + min(tok0 + 8 * m + 2 * k, n_rows - 1));
        b *= __ldg(scale + min(tok0 + 8 * m + 2 * k + 1, n_rows - 1));
      }
      w[m][k] = pack_bf16x2(a, b);
    }
  }
#pragma unroll
  for (int m = 0; m < 2; ++m) transpose8x8_b16(w[m], lane);
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const int tok = tok0 + 8 * m + (lane & 7);
    if (tok < n_rows && col_ok)
      *reinterpret_cast<uint4*>(dst + tok * ld) = make_uint4(w[m][0], w[m][1], w[m][2], w[m][3]);
  }
}

// Wait on a barrier for a whole warp: lane 0 polls (bounded) and the outcome
// is broadcast, so the warp stays converged for the .sync.aligned tcgen05 ops.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
  bool ok = false;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, abort_flag, status);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok;
}

// Two barriers for a whole warp: lane 0 tests both at once (their latencies
// overlap when both phases have completed, the common case), then waits
// (bounded) for any that had not.
__device__ __forceinline__ bool warp_wait2(uint32_t bar1, uint32_t parity1, uint32_t bar2,
                                           uint32_t parity2, volatile int* abort_flag,
                                           int* status) {
  bool ok = false;
  if ((threadIdx.x & 31) == 0) {
    const bool d1 = mbar_try_wait(bar1, parity1);
    const bool d2 = mbar_try_wait(bar2, parity2);
    ok = (d1 || mbar_wait_bounded(bar1, parity1, abort_flag, status)) &&
         (d2 || mbar_wait_bounded(bar2, parity2, abort_flag, status));
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok;
}

// Drain wait: bounded by time only (ignores the abort flag).
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, int* status) {
  int local_abort = 0;
  return mbar_wait_bounded<true>(bar, parity, &local_abort, status);
}

// TMEM: two regions of 256 columns.  A unit whose token tile fits in 128
// columns keeps both accumulators in one region (columns 0 and 128 of it),
// and a single-tile unit keeps its one accumulator (up to 256 columns) in one
// region, so consecutive such units alternate regions and the epilogue
// overlaps the next main loop; a two-tile unit with a larger token tile takes
// one region per accumulator.  Every unit advances a region counter c by the
// regions it uses; region use c is region c % 2 in its (c / 2)-th phase --
// the same sequence in every role.
// With the weights in TMEM (GemmParams::tmem_a: token tiles of at most 64
// rows) the regions are columns [0, 128) and [128, 256), each accumulator 64
// columns, and columns [256, 512) hold the weight stages.
struct Regions {
  bool big;     // two accumulators of more than 128 columns: one region each
  bool narrow;  // 128-column regions (weights in TMEM)
  int c;        // first region use of the unit
};

__device__ __forceinline__ Regions regions_of(const GemmParams& p, uint32_t n, int c) {
  return Regions{p.a_per_unit == 2 && n > 128 && !p.tmem_a, p.tmem_a != 0, c};
}
__device__ __forceinline__ int region_of(const Regions& r, int acc) {
  return r.big ? ((r.c + acc) & 1) : (r.c & 1);
}
__device__ __forceinline__ uint32_t region_phase(int use) { return static_cast<uint32_t>(use >> 1) & 1u; }
__device__ __forceinline__ uint32_t acc_column(const Regions& r, int acc) {
  if (r.narrow) return 128u * static_cast<uint32_t>(r.c & 1) + 64u * static_cast<uint32_t>(acc);
  return r.big ? 256u * static_cast<uint32_t>((r.c + acc) & 1)
               : 256u * static_cast<uint32_t>(r.c & 1) + 128u * static_cast<uint32_t>(acc);
}
// TMEM column of weight stage s, tile a (weights in TMEM: 64 columns a
// stage, the two 128-row tiles side by side, two bf16 of k per column)
constexpr uint32_t kTmemAStage0 = 256;
__device__ __forceinline__ uint32_t tmem_a_column(int s, int a) {
  return kTmemAStage0 + 64u * static_cast<uint32_t>(s) + 32u * static_cast<uint32_t>(a);
}

// One kernel body, two tensor-core modes:
//   kPair = false: one CTA per unit; units of two 128-row weight tiles (or
//     one); MMAs of M = 128 issued by the CTA itself.
//   kPair = true: clusters of two CTAs share each unit of two weight tiles:
//     CTA r holds weight tile 2 ob + r and half of the token tile (rows
//     [r N/2, (r+1) N/2)), and CTA 0 issues MMAs of M = 256 over the pair
//     (tcgen05 cta_group::2): each CTA's TMEM receives its 128 weight rows x
//     all N tokens.  Each CTA keeps one accumulator per unit, so the two TMEM
//     regions alternate and the epilogue of a unit overlaps the next main
//     loop whatever the token tile; the token tile is split, not repeated,
//     across the pair.  Both CTAs' copies complete on CTA 0's full barriers;
//     CTA 0's commits release both CTAs' stages and signal both epilogues;
//     both epilogues release TMEM on CTA 0's barrier.
//
// kFp8 (never with kPair): the weight producer's bulk copies bring FP8 tiles
// and their 16-byte block-scale record into a ring of f8_stages stages; the
// converter warps wait for a stage and for a free bf16 weight stage, write
// code x scale as bf16 in the same swizzled layout (FP8 byte offset o of a
// tile becomes bf16 byte offset 2 o), fence for the tensor cores' proxy and
// arrive on the k step's full barrier in place of the weight producer.
template <bool kPair, bool kFp8>
__global__ void __launch_bounds__(kFp8 ? kThreadsFp8 : kThreadsTwo, 1)
    tc_gemm_kernel(const __grid_constant__ GemmParams p) {
  // two MMA issuers, one per accumulator (bf16 forms, large token tiles:
  // GemmParams::two)
  const bool two_issuers = p.two != 0;
  // the second issuer: the warp after the epilogue's (bf16), after the
  // converters' (FP8)
  const int issuer2_warp = kFp8 ? 3 + kEpiWarps + kConvWarps : 3 + kEpiWarps;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int sa_n = p.a_stages;
  const int sb_n = p.b_stages;
  const int nt = p.nt;
  const int R = p.pieces > 1 ? p.pieces : 1;  // weight steps per k step
  const uint32_t b_stage_bytes = b_stage_bytes_of(nt, kPair);
  // FP8 weights at small token tiles: the converters write the bf16 weights
  // into TMEM (no bf16 weight stages in shared memory)
  const bool tmem_a = kFp8 && p.tmem_a;
  const uint32_t a_stage_bytes = tmem_a ? 0u : kATileBytes * static_cast<uint32_t>(p.a_per_unit);
  const int s8_n = kFp8 ? p.f8_stages : 0;
  uint8_t* smem_b = smem + sa_n * a_stage_bytes;
  uint8_t* smem_f8 = smem_b + sb_n * b_stage_bytes;          // FP8 ring: s8 x 2 tiles
  uint8_t* smem_rec = smem_f8 + s8_n * (2 * kF8TileBytes);  // s8 x 16-byte records
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_rec + 16 * s8_n);
  // bars: full[Sa] | empty[Sa] | tfull[2] | tempty[2] | drain | f8full[S8] | f8empty[S8]
  // k step i of the CTA's sequence uses weight stage i % Sa and token stage
  // i % Sb.  full[i % Sa] counts the bytes of both (one wait per k step for
  // the MMA issuer) and empty[i % Sa] frees both (one commit per k step):
  // token stage i % Sb is reused by k step i + Sb once empty[i % Sa]
  // completes k step i's phase.  With Sb <= Sa that phase is never
  // ambiguous, and no token copy reaches a full barrier before the
  // barrier's previous phase completed.
  const int nbars = 2 * sa_n + 5 + 2 * s8_n;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + nbars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // a CTA pair walks the units together: unit u belongs to cluster u % count
  const int rank = kPair ? static_cast<int>(cluster_ctarank()) : 0;
  const int u_first = kPair ? static_cast<int>(cluster_index_x()) : static_cast<int>(blockIdx.x);
  const int u_step = kPair ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
  constexpr uint16_t kPairMask = 3;
  const uint32_t bar_base = smem_u32(bars);
  const uint32_t a_base = smem_u32(smem);
  const uint32_t b_base = smem_u32(smem_b);
  auto a_full = [&](int s) { return bar_base + 8u * s; };
  auto a_empty = [&](int s) { return bar_base + 8u * (sa_n + s); };
  auto tfull_bar = [&](int r) { return bar_base + 8u * (2 * sa_n + r); };
  auto tempty_bar = [&](int r) { return bar_base + 8u * (2 * sa_n + 2 + r); };
  const uint32_t drain_bar = bar_base + 8u * (2 * sa_n + 4);
  auto f8full = [&](int s) { return bar_base + 8u * (2 * sa_n + 5 + s); };
  auto f8empty = [&](int s) { return bar_base + 8u * (2 * sa_n + 5 + s8_n + s); };
  // the same barrier in CTA 0 of the pair (the MMA issuer's)
  auto lead = [&](uint32_t bar) { return kPair ? cluster_map(bar, 0) : bar; };
  constexpr uint32_t kTmemCols = 512;

  if (warp == 0) {
    tmem_alloc<kPair>(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish<kPair>();
  }
  if (warp == 1 && lane == 0) {
    for (int s = 0; s < sa_n; ++s) {
      // the two producers' arrivals (CTA 0's in a pair), or the token
      // producer's and the converter warps'
      mbar_init(a_full(s), kFp8 ? 1 + kConvWarps : 2);
      mbar_init(a_empty(s), two_issuers ? 2 : 1);  // each MMA issuer's commit
    }
    for (int s = 0; s < s8_n; ++s) {
      mbar_init(f8full(s), 1);
      mbar_init(f8empty(s), kConvWarps);
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(tfull_bar(r), two_issuers ? 2 : 1);
      // paired: both CTAs' epilogue warps release CTA 0's regions
      mbar_init(tempty_bar(r), kPair ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(drain_bar, two_issuers ? 2 : 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  tc_fence_before();
  __syncthreads();
  // the peer's barriers and TMEM must exist before any copy, commit or
  // arrival reaches them
  if (kPair) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the set-up above overlaps the previous kernel; global memory only after it
  pdl_wait();

  const int units0 = segment_units(p, &p.seg[0]);
  const int units1 = p.nseg > 1 ? segment_units(p, &p.seg[1]) : 0;
  const int total = units0 + units1;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ weight (A) producer
    for (int s = 0; s < p.nseg; ++s) prefetch_tensormap(&p.seg[s].tmA);
    const uint64_t pol_stream = l2_policy_evict_first();
    const uint64_t pol_normal = l2_policy_evict_normal();
    const uint64_t pol_keep = l2_policy_evict_last();
    // the producer's ring: the bf16 weight stages, or the FP8 stages
    const int ring = kFp8 ? s8_n : sa_n;
    auto slot_free = [&](int st) { return kFp8 ? f8empty(st) : a_empty(st); };
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    Unit nx = u_first < total ? decode_unit<kFp8>(p, u_first, units0, units1, rank) : Unit{};
    for (int u = u_first; u < total; u += u_step) {
      // the next unit's tile-table loads overlap this unit's work
      const Unit x = nx;
      if (u + u_step < total) nx = decode_unit<kFp8>(p, u + u_step, units0, units1, rank);
      const GemmSegment* s = x.seg ? &p.seg[1] : &p.seg[0];
      const uint32_t tx = (kFp8 ? kF8TileBytes : kATileBytes) * x.n_a;
      // a weight block read by one token tile is streamed; one shared by
      // several token tiles (running side by side) is kept for the others;
      // a token-tile-major segment's weights serve every token tile
      const uint64_t pol_w = s->b_major ? pol_keep : x.ntiles > 1 ? pol_normal : pol_stream;
      bool ok = true;
      // weight steps: k step ks, piece pc (pc fastest)
      for (int ks = x.k0, pc = 0; ks < x.k1; pc + 1 < R ? ++pc : (pc = 0, ++ks)) {
        if (!mbar_wait_bounded(slot_free(stage), phase ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint32_t fb = kFp8 ? f8full(stage) : a_full(stage);
        const uint32_t a_dst = a_base + stage * a_stage_bytes;
        const int kc = ks * kBK;
        // packed weights: the unit's tiles at k step ks (a pair, or the
        // pair member of this CTA) are contiguous
        const int pair_idx = x.blk0 >> 1;
        const int in_pair = min(2, s->a128 - 2 * pair_idx);
        const int64_t tile = 2ll * pair_idx * s->k_steps + static_cast<int64_t>(ks) * in_pair +
                             (x.blk0 & 1);
        if (kFp8) {
          // the FP8 tiles and the pair's block-scale record for this k step
          mbar_arrive_expect_tx(fb, tx + 16);
          bulk_load(smem_u32(smem_f8) + stage * (2 * kF8TileBytes),
                    s->a_packed + x.group * s->a_group_bytes + tile * kF8TileBytes, tx, fb, pol_w);
          bulk_load(smem_u32(smem_rec) + stage * 16,
                    s->a_rec + ((x.group * s->a_rec_group) + pair_idx * s->k_steps + ks) * 16, 16,
                    fb, pol_w);
        } else if (kPair) {
          // CTA 0 expects both CTAs' tiles on its barrier (one box: this
          // CTA's one tile, or its pair of tiles, contiguous at k step ks)
          if (rank == 0) mbar_arrive_expect_tx(fb, 2 * a_stage_bytes);
          tma_load_2d_pair(a_dst, &s->tmA, lead(fb), 0,
                           static_cast<int>(x.group * (s->a_group_bytes >> 7) + tile * 128), pol_w);
        } else if (s->a_packed) {
          mbar_arrive_expect_tx(fb, tx);
          bulk_load(a_dst, s->a_packed + x.group * s->a_group_bytes + tile * kATileBytes, tx, fb,
                    pol_w);
        } else if (R > 1) {
          // the unit's tile of weight piece pc at k step ks; the token
          // producer arrives only on a k step's first weight step, so this
          // thread arrives in its place on the others
          mbar_arrive_expect_tx(fb, kATileBytes);
          tma_load_3d(a_dst, &s->tmA, fb, kc + pc * s->a_piece_cols, x.blk0 * 128, x.group,
                      pol_w);
          if (pc) mbar_arrive(fb);
        } else {
          mbar_arrive_expect_tx(fb, tx);
          for (int a = 0; a < x.n_a; ++a) {
            const int blk = x.blk0 + a;  // 128-row A tile index along O
            const uint32_t dst = a_dst + a * kATileBytes;
            if (s->mode == kModeSwiGLU) {
              if (s->a_boxes == 1) {
                tma_load_5d(dst, &s->tmA, fb, kc, 0, 0, blk * 4, x.group, pol_w);
              } else {
                for (int j = 0; j < 8; ++j)
                  tma_load_3d(dst + j * 2048u, &s->tmA, fb, kc,
                              (j & 1) * s->a_rows + blk * 64 + (j >> 1) * 16, x.group, pol_w);
              }
            } else {
              tma_load_3d(dst, &s->tmA, fb, kc, blk * 128, x.group, pol_w);
            }
          }
        }
        ++issued;
        if (++stage == ring) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
    // drain: wait until the last stages issued were consumed (so every copy
    // into them, of either producer and either CTA, has landed)
    const int64_t first = issued > ring ? issued - ring : 0;
    for (int64_t q = first; q < issued; ++q) {
      const int st = static_cast<int>(q % ring);
      const uint32_t par = static_cast<uint32_t>((q / ring) & 1);
      if (!drain_wait(slot_free(st), par, p.status)) break;
    }
  } else if (warp == 2 && lane == 0) {
    // ------------------------------------------------- token (B) producer
    for (int s = 0; s < p.nseg; ++s)
      if (kPair || !p.seg[s].b_packed) prefetch_tensormap(&p.seg[s].tmB);
    const uint64_t pol_keep = l2_policy_evict_last();
    const uint64_t pol_normal = l2_policy_evict_normal();
    int stage = 0;       // token stage
    int64_t issued = 0;  // token stages issued: stage i goes with weight steps R i .. R i + R - 1
    int fstage = 0;      // weight stage of weight step R * issued (its full barrier)
    // weight stage and phase of weight step R (issued - Sb) + R - 1, the last
    // reader of the token stage about to be refilled
    int estage = R - 1;
    uint32_t ephase = 0;
    Unit nx = u_first < total ? decode_unit<kFp8>(p, u_first, units0, units1, rank) : Unit{};
    for (int u = u_first; u < total; u += u_step) {
      // the next unit's tile-table loads overlap this unit's work
      const Unit x = nx;
      if (u + u_step < total) nx = decode_unit<kFp8>(p, u + u_step, units0, units1, rank);
      const GemmSegment* s = x.seg ? &p.seg[1] : &p.seg[0];
      // token rows are kept for the units that re-read them, except in a
      // token-tile-major segment, whose readers of a tile run side by side
      const uint64_t pol_b = s->b_major ? pol_normal : pol_keep;
      // paired: this CTA's half of the tile's rows (rounded up to 16), as
      // 32-row boxes; the rows past the half that a box brings in are not
      // read by the MMA
      const int half = ((x.n_rows + 15) & ~15) >> 1;
      const int b_row = kPair ? x.b_row + rank * half : x.b_row;
      // tensor-map tiles: boxes of the segment's box height (its whole token
      // tile: one copy per k step), 32 rows for pairs
      const int br = (!kPair && s->b_box_rows) ? s->b_box_rows : kBBoxRows;
      const int nbox = kPair ? (half + kBBoxRows - 1) / kBBoxRows : (x.n_rows + br - 1) / br;
      // packed: the tile's rows (rounded up to 16) are one contiguous run
      const uint32_t tx = kPair ? 2u * static_cast<uint32_t>(nbox) * kBBoxBytes
                          : s->b_packed ? static_cast<uint32_t>((x.n_rows + 15) & ~15) * 128u
                                        : static_cast<uint32_t>(nbox * br) * 128u;
      bool ok = true;
      for (int ks = x.k0; ks < x.k1; ++ks) {
        if (issued >= sb_n) {
          // the token stage is free once the last weight step that read it
          // (that of token stage issued - Sb) was consumed
          if (!mbar_wait_bounded(a_empty(estage), ephase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if ((estage += R) >= sa_n) {
            estage -= sa_n;
            ephase ^= 1u;
          }
        }
        const uint32_t fb = a_full(fstage);
        if (!kPair || rank == 0) mbar_arrive_expect_tx(fb, tx);
        const uint32_t b_dst = b_base + stage * b_stage_bytes;
        if (kPair) {
          for (int bx = 0; bx < nbox; ++bx) {
            if (s->b_packed)
              tma_load_3d_pair(b_dst + bx * kBBoxBytes, &s->tmB, lead(fb), 0,
                               b_row + bx * kBBoxRows, ks, pol_b);
            else
              tma_load_2d_pair(b_dst + bx * kBBoxBytes, &s->tmB, lead(fb), ks * kBK,
                               b_row + bx * kBBoxRows, pol_b);
          }
        } else if (s->b_packed) {
          const uint8_t* src =
              s->b_packed + (static_cast<int64_t>(ks) * s->b_plane_rows + b_row) * 128;
          bulk_load(b_dst, src, tx, fb, pol_b);
        } else {
          for (int bx = 0; bx < nbox; ++bx)
            tma_load_2d(b_dst + bx * br * 128u, &s->tmB, fb, ks * kBK, b_row + bx * br, pol_b);
        }
        ++issued;
        if ((fstage += R) >= sa_n) fstage -= sa_n;
        if (++stage == sb_n) stage = 0;
      }
      if (!ok) break;
    }
    const int64_t first = issued > sb_n ? issued - sb_n : 0;
    for (int64_t q = first; q < issued; ++q) {
      const int64_t last = R * q + R - 1;
      const int st = static_cast<int>(last % sa_n);
      const uint32_t par = static_cast<uint32_t>((last / sa_n) & 1);
      if (!drain_wait(a_empty(st), par, p.status)) break;
    }
  } else if ((warp == 1 || (two_issuers && warp == issuer2_warp)) && lane == 0 && rank == 0) {
    // ------------------------------------------------------- MMA issuers
    // With two_issuers warp 1 issues the MMAs of accumulator 0 and the last
    // warp those of accumulator 1, each followed by its own commit: one
    // thread issuing a k step's 8 MMAs and its commit takes about twice the
    // tensor time of an N <= 176 k step, two threads issuing 4 each keep up
    // with it.  Both wait for every stage and both commits free it (a_empty
    // counts 2); the accumulation order of each accumulator is unchanged.
    // Each issuer also commits to every TMEM region the unit fills, so those
    // count 2 as well.
    const int my_acc = warp == 1 ? 0 : 1;
    int sa = 0, sb = 0;
    uint32_t pa = 0;
    int c = 0;
    Unit nx = u_first < total ? decode_unit<kFp8>(p, u_first, units0, units1, rank) : Unit{};
    for (int u = u_first; u < total; u += u_step) {
      // the next unit's tile-table loads overlap this unit's work
      const Unit x = nx;
      if (u + u_step < total) nx = decode_unit<kFp8>(p, u + u_step, units0, units1, rank);
      const uint32_t n = static_cast<uint32_t>((x.n_rows + 15) & ~15);
      const Regions rg = regions_of(p, n, c);
      bool ok;
      if (two_issuers) {  // the region this issuer's accumulator lives in
        const int use = rg.big ? c + my_acc : c;
        ok = mbar_wait_bounded<kPair>(tempty_bar(use & 1), region_phase(use) ^ 1u, abort_flag,
                                      p.status);
      } else {
        ok = mbar_wait_bounded<kPair>(tempty_bar(c & 1), region_phase(c) ^ 1u, abort_flag,
                                      p.status);
        if (ok && rg.big)
          ok = mbar_wait_bounded(tempty_bar((c + 1) & 1), region_phase(c + 1) ^ 1u, abort_flag,
                                 p.status);
      }
      if (!ok) break;
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(kPair ? 256 : 128, n);
      for (int t = x.k0 * R, pc = 0; t < x.k1 * R; ++t) {
        if (!mbar_wait_bounded<kPair>(a_full(sa), pa, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t bdesc = smem_desc_sw128(b_base + sb * b_stage_bytes);
        if (R > 1) {
          // weight piece pc against the k step's token stage, into the
          // unit's one accumulator
          const uint64_t adesc = smem_desc_sw128(a_base + sa * a_stage_bytes);
          const uint32_t d = tmem_base + acc_column(rg, 0);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc_mma_bf16<kPair>(d, adesc + 2u * kk, bdesc + 2u * kk, idesc,
                               ((t - x.k0 * R) | kk) != 0);
        } else {
          // accumulators of this CTA (of each CTA of a pair): its weight tiles
          const int n_acc = (kPair && p.a_per_unit == 1) ? 1 : x.n_a;
          const int a_lo = two_issuers ? my_acc : 0;
          const int a_hi = two_issuers ? min(my_acc + 1, n_acc) : n_acc;
          for (int a = a_lo; a < a_hi; ++a) {
            const uint32_t d = tmem_base + acc_column(rg, a);
            if (tmem_a) {  // the converters' bf16 tile in TMEM, 8 columns per 16 k
              const uint32_t at = tmem_base + tmem_a_column(sa, a);
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk)
                tc_mma_bf16_ta(d, at + 8u * kk, bdesc + 2u * kk, idesc, ((t - x.k0) | kk) != 0);
              continue;
            }
            const uint64_t adesc =
                smem_desc_sw128(a_base + sa * a_stage_bytes + a * kATileBytes);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              tc_mma_bf16<kPair>(d, adesc + 2u * kk, bdesc + 2u * kk, idesc,
                                 ((t - x.k0) | kk) != 0);
          }
        }
        if (kPair)  // release the stages of both CTAs
          tc_commit_pair(a_empty(sa), kPairMask);
        else
          tc_commit(a_empty(sa));
        if (++sa == sa_n) {
          sa = 0;
          pa ^= 1u;
        }
        if (++pc == R) {  // the k step's last weight step: next token stage
          pc = 0;
          if (++sb == sb_n) sb = 0;
        }
      }
      if (!ok) break;
      if (kPair) {  // both CTAs' accumulators are ready
        tc_commit_pair(tfull_bar(c & 1), kPairMask);
        if (rg.big) tc_commit_pair(tfull_bar((c + 1) & 1), kPairMask);
      } else {
        tc_commit(tfull_bar(c & 1));
        if (rg.big) tc_commit(tfull_bar((c + 1) & 1));
      }
      c += rg.big ? 2 : 1;
    }
    if (kPair)
      tc_commit_pair(drain_bar, 1);
    else
      tc_commit(drain_bar);
    drain_wait(drain_bar, 0, p.status);
  } else if (kFp8 && tmem_a && warp >= 3 + kEpiWarps && warp < 3 + kEpiWarps + kConvWarps) {
    // ------------------------------------- FP8 -> bf16 converters, into TMEM
    // Warp w converts row 32 (w % 4) + lane -- the TMEM lanes it may access
    // -- of tile (w - 3 - kEpiWarps) / 4 of each stage: the row's 64 codes
    // (8-byte pieces, logical piece c at (c ^ row % 8) * 8 of its 64 bytes)
    // into 32 columns, two bf16 of k per column, scaled by the scale of the
    // row's half (gate or up: row bit 4).  Software-pipelined by one k step:
    // a step's codes are converted before the previous step's TMEM store is
    // waited for and that step released (full and FP8-empty barriers), so
    // the store's latency overlaps the conversion.
    const int ct = threadIdx.x - 32 * (3 + kEpiWarps);
    const int tile = (ct >> 5) >> 2;
    const int row = 32 * (warp & 3) + lane;
    const int x7 = row & 7;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    int sa = 0, s8 = 0, pend_sa = -1, pend_s8 = 0;
    uint32_t pa = 0, p8 = 0;
    bool ok = true;
    auto release_pending = [&]() {
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(f8empty(pend_s8));
        mbar_arrive(a_full(pend_sa));
      }
    };
    Unit nx = u_first < total ? decode_unit<kFp8>(p, u_first, units0, units1, rank) : Unit{};
    for (int u = u_first; u < total && ok; u += u_step) {
      const Unit x = nx;
      if (u + u_step < total) nx = decode_unit<kFp8>(p, u + u_step, units0, units1, rank);
      const bool mine = tile < x.n_a;
      for (int ks = x.k0; ks < x.k1; ++ks) {
        if (!warp_wait2(f8full(s8), p8, a_empty(sa), pa ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        // the MMAs that read this TMEM stage have completed
        tc_fence_after();
        uint32_t w[32];
        if (mine) {
          const float scale =
              reinterpret_cast<const float*>(smem_rec + 16 * s8)[2 * tile + ((row >> 4) & 1)];
          const uint8_t* src = smem_f8 + s8 * (2 * kF8TileBytes) + tile * kF8TileBytes + row * 64;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // logical pieces 2j and 2j + 1 share a 16-byte pair, swapped
            // when the row's swizzle is odd
            const uint4 v = *reinterpret_cast<const uint4*>(src + ((j ^ (x7 >> 1)) << 4));
            const uint2 lo = (x7 & 1) ? make_uint2(v.z, v.w) : make_uint2(v.x, v.y);
            const uint2 hi = (x7 & 1) ? make_uint2(v.x, v.y) : make_uint2(v.z, v.w);
            e4m3x4_scaled_bf16x2x2(lo.x, scale, w[8 * j + 0], w[8 * j + 1]);
            e4m3x4_scaled_bf16x2x2(lo.y, scale, w[8 * j + 2], w[8 * j + 3]);
            e4m3x4_scaled_bf16x2x2(hi.x, scale, w[8 * j + 4], w[8 * j + 5]);
            e4m3x4_scaled_bf16x2x2(hi.y, scale, w[8 * j + 6], w[8 * j + 7]);
          }
        }
        if (pend_sa >= 0) release_pending();
        if (mine) tmem_st_x32(lane_base + tmem_a_column(sa, tile), w);
        pend_sa = sa;
        pend_s8 = s8;
        if (++s8 == s8_n) {
          s8 = 0;
          p8 ^= 1u;
        }
        if (++sa == sa_n) {
          sa = 0;
          pa ^= 1u;
        }
      }
    }
    if (ok && pend_sa >= 0) release_pending();
    tmem_st_wait();  // no store of this warp outlives it (TMEM is freed at the end)
  } else if (kFp8 && warp >= 3 + kEpiWarps && warp < 3 + kEpiWarps + kConvWarps) {
    // ---------------------------------------------- FP8 -> bf16 converters
    // Thread ct of the kCT converter threads handles the 8-byte FP8 pieces
    // pc = ct + kCT i of a stage: piece pc is row pc / 8 of the stage's 256
    // rows, in tile pc / 1024 (the same for every thread at a given i) and
    // in that tile's gate half (rows with bit 4 clear) or up half -- the
    // record's scale 2 (pc / 1024) + (pc / 128) % 2.  A plain store-mode tile
    // has one scale, written twice in its record.
    const int ct = threadIdx.x - 32 * (3 + kEpiWarps);
    int sa = 0, s8 = 0;
    uint32_t pa = 0, p8 = 0;
    Unit nx = u_first < total ? decode_unit<kFp8>(p, u_first, units0, units1, rank) : Unit{};
    for (int u = u_first; u < total; u += u_step) {
      const Unit x = nx;
      if (u + u_step < total) nx = decode_unit<kFp8>(p, u + u_step, units0, units1, rank);
      bool ok = true;
      for (int ks = x.k0; ks < x.k1; ++ks) {
        if (!warp_wait2(f8full(s8), p8, a_empty(sa), pa ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const float* rec = reinterpret_cast<const float*>(smem_rec + 16 * s8);
        float sc[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) sc[j] = rec[j];
        const uint8_t* src = smem_f8 + s8 * (2 * kF8TileBytes);
        uint8_t* dst = smem + sa * a_stage_bytes;
        constexpr int kCT = 32 * kConvWarps;
        const int n_i = (1024 / kCT) * x.n_a;
#pragma unroll
        for (int i = 0; i < 2048 / kCT; ++i) {
          if (i < n_i) {
            const int pc = ct + kCT * i;
            const int tile = i / (1024 / kCT);
            const float scale = ((pc >> 7) & 1) ? sc[2 * tile + 1] : sc[2 * tile];
            const uint2 v = *reinterpret_cast<const uint2*>(src + 8 * pc);
            uint4 o;
            e4m3x4_scaled_bf16x2x2(v.x, scale, o.x, o.y);
            e4m3x4_scaled_bf16x2x2(v.y, scale, o.z, o.w);
            *reinterpret_cast<uint4*>(dst + 16 * pc) = o;
          }
        }
        // the stage is read next by the tensor cores (async proxy)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(f8empty(s8));
          mbar_arrive(a_full(sa));
        }
        if (++s8 == s8_n) {
          s8 = 0;
          p8 ^= 1u;
        }
        if (++sa == sa_n) {
          sa = 0;
          pa ^= 1u;
        }
      }
      if (!ok) break;
    }
  } else if (warp >= 3 && warp < 3 + kEpiWarps) {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;           // TMEM lane quadrant this warp may access
    const int grp = (warp - 3) >> 2;  // warp group: accumulator (two-tile units)
                                      // or column half (single-tile units)

    const bool single = p.a_per_unit == 1;
    int c = 0;
    Unit nx = u_first < total ? decode_unit<kFp8>(p, u_first, units0, units1, rank) : Unit{};
    for (int u = u_first; u < total; u += u_step) {
      // the next unit's tile-table loads overlap this unit's work
      const Unit x = nx;
      if (u + u_step < total) nx = decode_unit<kFp8>(p, u + u_step, units0, units1, rank);
      const GemmSegment* s = x.seg ? &p.seg[1] : &p.seg[0];
      const bool swiglu = s->mode == kModeSwiGLU;
      // the segment's output description, once per unit, in registers
      __nv_bfloat16* const out = s->out;
      float* const out_f32 = s->out_f32 ? s->out_f32 + x.split * s->out_split_stride : nullptr;
      const int64_t ld = s->out_ld;
      const float* const row_scale = s->row_scale;
      const __nv_bfloat16* const add = s->add;
      const int64_t add_ld = s->add_ld;
      const bool out_packed = s->out_packed != 0;
      const int64_t plane_rows = s->out_plane_rows;
      const int o_limit = s->o_limit;
      // store mode, bf16 output without an addend, rows of whole 16-byte
      // chunks: written by 16-byte stores
      const bool rows8 = !add && !out_f32 && o_limit % 8 == 0 && ld % 8 == 0;
      const uint32_t n = static_cast<uint32_t>((x.n_rows + 15) & ~15);
      const Regions rg = regions_of(p, n, c);
      // A two-tile unit with both accumulators in one region: warp group g
      // drains accumulator g.  A two-tile unit with one region per
      // accumulator: all warps drain accumulator 0, release its region, then
      // accumulator 1, so a following unit that needs one region starts
      // half an epilogue earlier.  A single-tile unit: all warps, one pass.
      // In the all-warps passes the warp groups split the 16-token blocks.
      const bool all_warps = single || rg.big;
      const int npass = rg.big ? 2 : 1;
      bool aborted = false;
      for (int pass = 0; pass < npass; ++pass) {
      const int acc = rg.big ? pass : (single ? 0 : grp);
      const int use = rg.big ? c + acc : c;
      const int region = region_of(rg, acc);
      if (!warp_wait(tfull_bar(region), region_phase(use), abort_flag, p.status)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      if (acc < x.n_a) {
        const uint32_t taddr0 =
            tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc_column(rg, acc);
        const int blk = x.blk0 + acc;
        // 16 columns (tokens) per TMEM load, one wait each
        const int nblk = (x.n_rows + 15) / 16;
        const int step = all_warps ? 2 : 1;
#pragma unroll 1
        for (int bk = all_warps ? grp : 0; bk < nblk; bk += step) {
          const int tok0 = bk * 16;
          uint32_t v[16];
          tmem_ld_x16(taddr0 + static_cast<uint32_t>(tok0), v);
          tmem_ld_wait(v);
          if (swiglu) {
            swiglu_block(v, tok0, x.n_rows, lane, q, blk, out, out_packed, plane_rows,
                         x.out_row, ld);
          } else if (rows8) {
            const int o0 = blk * 128 + q * 32 + (lane & ~7);
            __nv_bfloat16* const dst = out + static_cast<int64_t>(x.out_row) * ld + o0;
            const bool col_ok = o0 < o_limit;
            if (row_scale)
              store_rows8_block<true>(v, row_scale + x.scale_row, tok0, x.n_rows, dst, ld,
                                      col_ok, lane);
            else
              store_rows8_block<false>(v, nullptr, tok0, x.n_rows, dst, ld, col_ok, lane);
          } else {
            const int o = blk * 128 + q * 32 + lane;
            if (o < o_limit) {
              if (out_f32 && !row_scale && !add && tok0 + 16 <= x.n_rows) {
                // fp32 partial sums (the router): one column of 16 rows
                float* const dst = out_f32 + (x.out_row + tok0) * ld + o;
#pragma unroll
                for (int j = 0; j < 16; ++j) dst[j * ld] = __uint_as_float(v[j]);
              } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  const int tok = tok0 + j;
                  if (tok < x.n_rows) {
                    const int64_t row = x.out_row + tok;
                    float val = __uint_as_float(v[j]);
                    if (row_scale) val *= __ldg(row_scale + x.scale_row + tok);
                    if (add) val += __bfloat162float(add[row * add_ld + o]);
                    if (out_f32)
                      out_f32[row * ld + o] = val;
                    else
                      out[row * ld + o] = __float2bfloat16_rn(val);
                  }
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // every epilogue warp arrives once per region it drained; paired
        // CTAs release CTA 0's region
        if (kPair)
          mbar_arrive_cluster(lead(tempty_bar(region)));
        else
          mbar_arrive(tempty_bar(region));
      }
      }
      if (aborted) break;
      c += rg.big ? 2 : 1;
    }
  }

  __syncthreads();
  // this CTA's work is done: the next kernel of the stream may start
  // launching (it still waits for this grid's completion before it reads)
  pdl_release();
  // neither CTA of a pair leaves (or frees TMEM) while the other may still
  // reach its shared memory, barriers or accumulators
  if (kPair) cluster_sync_all();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<kPair>(tmem_base, kTmemCols);
  }
}

// W_split[e, 0:d] = hi, [d:2d] = mid, [2d:3d] = lo: successive bf16 roundings
// of what is left of W_r[e, :], so hi + mid + lo keeps ~24 significant bits.
__global__ void __launch_bounds__(256) split_router_weight_kernel(const float* __restrict__ W,
                                                                  int E, int d,
                                                                  __nv_bfloat16* __restrict__ out) {
  pdl_wait();
  // eight consecutive weights per thread step (d % 8 == 0): two 16-byte
  // loads, one 16-byte store into each of the three pieces
  const int64_t n8 = static_cast<int64_t>(E) * d / 8;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = (8 * i) / d, k = 8 * i - e * d;
    const float4 a = __ldg(reinterpret_cast<const float4*>(W) + 2 * i);
    const float4 b = __ldg(reinterpret_cast<const float4*>(W) + 2 * i + 1);
    const float w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t hi[4], mid[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float h[2], m[2], l[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float v = w[2 * j + q];
        h[q] = __bfloat162float(__float2bfloat16_rn(v));
        const float r1 = v - h[q];
        m[q] = __bfloat162float(__float2bfloat16_rn(r1));
        l[q] = r1 - m[q];
      }
      hi[j] = pack_bf16x2(h[0], h[1]);
      mid[j] = pack_bf16x2(m[0], m[1]);
      lo[j] = pack_bf16x2(l[0], l[1]);
    }
    __nv_bfloat16* row = out + e * 3 * d + k;
    *reinterpret_cast<uint4*>(row) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(row + d) = make_uint4(mid[0], mid[1], mid[2], mid[3]);
    *reinterpret_cast<uint4*>(row + 2 * d) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// One 16-byte chunk of the packed bank per thread step: dst is written in
// order, src gathered (a one-time load step).
// V carries 8 consecutive elements: uint4 for bf16, uint2 for FP8 (whose
// tiles are 8 KB and whose rows are 64 bytes; the same chunk swizzle).
template <typename V>
__global__ void __launch_bounds__(256) pack_weights_kernel(int kind, int64_t groups, int64_t rows,
                                                           int64_t cols,
                                                           const V* __restrict__ src,
                                                           V* __restrict__ dst) {
  const int64_t ksteps = cols / kBK;
  const int64_t a128 = rows / 128;
  const int64_t per_group = a128 * ksteps;  // 16 KB tiles per group
  const int64_t full_pairs = a128 / 2;
  const int64_t n = groups * per_group * 1024;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i >> 10;
    const int r = static_cast<int>((i >> 3) & 127);
    const int pos = static_cast<int>(i & 7);
    const int64_t g = t / per_group;
    const int64_t tg = t - g * per_group;
    int64_t pair, ks, a;
    if (tg < full_pairs * 2 * ksteps) {
      pair = tg / (2 * ksteps);
      const int64_t rem = tg - pair * 2 * ksteps;
      ks = rem >> 1;
      a = rem & 1;
    } else {
      pair = full_pairs;
      ks = tg - full_pairs * 2 * ksteps;
      a = 0;
    }
    const int64_t blk = 2 * pair + a;
    const int chunk = pos ^ (r & 7);
    int64_t row;
    if (kind == 0) {
      const int64_t F = rows / 2;
      row = ((r >> 4) & 1) * F + 64 * blk + 16 * (r >> 5) + (r & 15);
    } else {
      row = blk * 128 + r;
    }
    dst[i] = src[((g * rows + row) * cols + ks * kBK + chunk * 8) >> 3];
  }
}

// One 16-byte record per (group, tile pair, k step): the block scales of
// the pair's two tiles at that k step, (tile 0 gate or plain, tile 0 up or
// plain, tile 1 ..., tile 1 ...); 0 for a missing second tile.
__global__ void __launch_bounds__(256) pack_scale_records_kernel(int kind, int64_t groups,
                                                                 int64_t rows, int64_t cols,
                                                                 const float* __restrict__ scales,
                                                                 float4* __restrict__ rec) {
  const int64_t ksteps = cols / kBK;
  const int64_t a128 = rows / 128;
  const int64_t npairs = (a128 + 1) / 2;
  const int64_t nbr = (rows + 127) / 128, nbc = (cols + 127) / 128;
  const int64_t n = groups * npairs * ksteps;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t g = i / (npairs * ksteps);
    const int64_t rem = i - g * npairs * ksteps;
    const int64_t pair = rem / ksteps;
    const int64_t cb = ((rem - pair * ksteps) * kBK) / 128;  // column block of the k step
    float v[4];
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int64_t blk = 2 * pair + a;
      if (blk >= a128) {
        v[2 * a] = v[2 * a + 1] = 0.0f;
        continue;
      }
      // row blocks of the tile's rows: gate/up tile blk holds rows
      // 64 blk.. of the gate half and F + 64 blk.. of the up half
      const int64_t rb0 = kind == 0 ? (64 * blk) / 128 : blk;
      const int64_t rb1 = kind == 0 ? (rows / 2 + 64 * blk) / 128 : blk;
      v[2 * a] = scales[(g * nbr + rb0) * nbc + cb];
      v[2 * a + 1] = scales[(g * nbr + rb1) * nbc + cb];
    }
    rec[i] = make_float4(v[0], v[1], v[2], v[3]);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

CUresult encode(CUtensorMap* map, const void* base, cuuint32_t rank, const cuuint64_t* dims,
                const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_INITIALIZED;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

CUresult encode_tmap_2d_rows(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                             int box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {kBK, static_cast<cuuint32_t>(box_rows)};
  return encode(map, base, 2, dims, strides, box);
}

CUresult encode_tmap_weights_3d(CUtensorMap* map, const void* base, int64_t groups, int64_t rows,
                                int64_t cols, int box_rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(groups)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2,
                                 static_cast<cuuint64_t>(rows * cols) * 2};
  const cuuint32_t box[3] = {kBK, static_cast<cuuint32_t>(box_rows), 1};
  return encode(map, base, 3, dims, strides, box);
}

CUresult encode_tmap_gate_up_5d(CUtensorMap* map, const void* base, int64_t groups, int64_t F,
                                int64_t cols) {
  // view W_gate_up [E, 2F, d] as (k, f_lo, half, f_hi, e) so one box yields
  // the interleaved 128-row A tile described at the top of this file
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(cols), 16, 2, static_cast<cuuint64_t>(F / 16),
                              static_cast<cuuint64_t>(groups)};
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(cols) * 2,
                                 static_cast<cuuint64_t>(F * cols) * 2,
                                 static_cast<cuuint64_t>(16 * cols) * 2,
                                 static_cast<cuuint64_t>(2 * F * cols) * 2};
  const cuuint32_t box[5] = {kBK, 16, 2, 4, 1};
  return encode(map, base, 5, dims, strides, box);
}

GemmPlan plan_gemm(int nt, int a_per_unit, bool pair, int pieces) {
  // token ring: 3 stages; weight ring: the rest of the budget
  static const int forced_b = [] {  // tuning override of the token ring depth
    const char* v = getenv("FGS_B_STAGES");
    return (v && *v) ? atoi(v) : 0;
  }();
  GemmPlan g;
  g.nt = nt;
  const size_t b_stage = b_stage_bytes_of(nt, pair);
  const size_t a_stage = static_cast<size_t>(kATileBytes) * a_per_unit;
  g.b_stages = 3;
  if (forced_b >= 2 && forced_b <= 8) g.b_stages = forced_b;
  const size_t b_bytes = g.b_stages * b_stage;
  int sa = b_bytes < kSmemBudget ? static_cast<int>((kSmemBudget - b_bytes) / a_stage) : 0;
  static const int forced_a = [] {  // tuning override: cap on the weight ring depth
    const char* v = getenv("FGS_A_STAGES");
    return (v && *v) ? atoi(v) : 0;
  }();
  if (sa > kMaxStages) sa = kMaxStages;
  if (forced_a >= 2 && sa > forced_a) sa = forced_a;
  if (sa < 2) {  // keep at least two weight stages
    sa = 2;
    g.b_stages = static_cast<int>((kSmemBudget - 2 * a_stage) / b_stage);
  }
  if (g.b_stages > sa) g.b_stages = sa;  // see the barrier layout in the kernel
  // R = pieces weight steps per token stage: a token copy reaches the full
  // barrier of weight step R i while the last weight step of token stage
  // i - Sb has been consumed, so weight step R i - Sa must precede it:
  // Sa >= R (Sb - 1) + 1 (R = 1: Sa >= Sb)
  while (pieces > 1 && g.b_stages > 1 && sa < pieces * (g.b_stages - 1) + 1) {
    --g.b_stages;
    const size_t left = kSmemBudget - g.b_stages * b_stage;
    sa = static_cast<int>(left / a_stage);
    if (sa > kMaxStages) sa = kMaxStages;
  }
  g.a_stages = sa;
  g.f8_stages = 0;
  g.smem_bytes = 1024 + a_stage * sa + b_stage * g.b_stages + 8 * (2 * sa + 5) + 16;
  return g;
}

// FP8 weights: two bf16 weight stages (the converters stay one stage ahead
// of the MMAs), two token stages, and every remaining byte as FP8 stages
// (the copies in flight from HBM), at most kMaxStages.
GemmPlan plan_gemm_fp8(int nt, bool tmem_a) {
  static const int forced_a = [] {  // tuning override: bf16 weight stages
    const char* v = getenv("FGS_FP8_A_STAGES");
    return (v && *v) ? atoi(v) : 0;
  }();
  static const int forced_8 = [] {  // tuning override: cap on the FP8 stages
    const char* v = getenv("FGS_F8_STAGES");
    return (v && *v) ? atoi(v) : 0;
  }();
  GemmPlan g;
  g.nt = nt;
  const size_t b_stage = b_stage_bytes_of(nt, false);
  // weights in TMEM: four stages there (columns 256..511), none in shared memory
  const size_t a_stage = tmem_a ? 0 : 2ull * kATileBytes;
  g.a_stages = tmem_a ? 4 : (forced_a >= 2 && forced_a <= 4) ? forced_a : 2;
  // weights in TMEM: the bf16 stages' shared memory goes to the token ring
  // (at most as deep as the weight ring)
  static const int forced_b = [] {  // tuning override: token stages with weights in TMEM
    const char* v = getenv("FGS_FP8_B_STAGES");
    return (v && *v) ? atoi(v) : 0;
  }();
  g.b_stages = tmem_a ? ((forced_b >= 2 && forced_b <= 4) ? forced_b : 4) : 2;
  const size_t f8_stage = 2ull * kF8TileBytes + 16 + 16;  // tiles, record, two barriers
  const size_t fixed = 1024 + a_stage * g.a_stages + b_stage * g.b_stages +
                       8 * (2 * g.a_stages + 5) + 16;
  int s8 = fixed < static_cast<size_t>(kSmemMax)
               ? static_cast<int>((static_cast<size_t>(kSmemMax) - fixed) / f8_stage)
               : 0;
  if (s8 > kMaxStages) s8 = kMaxStages;
  if (forced_8 >= 2 && s8 > forced_8) s8 = forced_8;
  g.f8_stages = s8;
  g.smem_bytes = fixed + f8_stage * s8;
  return g;
}

namespace {

// Paired launches read packed weights and packed activations through tensor
// maps (the pair's copies complete on one CTA's barriers, which only tensor
// copies can do): weights as rows of 128 bytes, one 128-row tile per box;
// activation planes as (64 columns, plane rows, planes), 32-row boxes.  The
// data are stored pre-swizzled, so the maps do not swizzle again.
CUresult encode_pair_maps(GemmSegment& s, int a_per_unit) {
  auto fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_INITIALIZED;
  cuuint32_t estr[3] = {1, 1, 1};
  // one box per k step: the CTA's weight tile, or its pair of tiles (the
  // packed bank keeps a pair's tiles of one k step together)
  const cuuint64_t a_dims[2] = {kBK, static_cast<cuuint64_t>(s.a_groups) *
                                         static_cast<cuuint64_t>(s.a_group_bytes / 128)};
  const cuuint64_t a_strides[1] = {128};
  const cuuint32_t a_box[2] = {kBK, static_cast<cuuint32_t>(128 * a_per_unit)};
  CUresult r = fn(&s.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint8_t*>(s.a_packed),
                  a_dims, a_strides, a_box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return r;
  if (!s.b_packed) {
    // activation rows of a plain tensor map: 32-row boxes for the pair's
    // halves of a token tile (128-byte swizzle, as the MMA reads them)
    if (!s.b_src) return CUDA_ERROR_INVALID_VALUE;
    return encode_tmap_2d_rows(&s.tmB, s.b_src, s.b_src_rows, 64ll * s.k_steps, kBBoxRows) ==
                   CUDA_SUCCESS
               ? CUDA_SUCCESS
               : CUDA_ERROR_INVALID_VALUE;
  }
  const cuuint64_t b_dims[3] = {kBK, static_cast<cuuint64_t>(s.b_plane_rows),
                                static_cast<cuuint64_t>(s.k_steps)};
  const cuuint64_t b_strides[2] = {128, static_cast<cuuint64_t>(s.b_plane_rows) * 128};
  const cuuint32_t b_box[3] = {kBK, kBBoxRows, 1};
  return fn(&s.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint8_t*>(s.b_packed), b_dims,
            b_strides, b_box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

bool pair_capable(const GemmParams& p) {
  for (int i = 0; i < p.nseg; ++i) {
    const GemmSegment& s = p.seg[i];
    if (!s.a_packed || s.a_fp8 || s.a_groups < 1 || s.a128 % 2 || s.ksplit > 1)
      return false;
  }
  return p.nseg > 0;
}

bool fp8_tmem_enabled() {
  static const int on = [] {  // tuning override: 0 = bf16 weight stages in shared memory
    const char* v = getenv("FGS_FP8_TMEM");
    return (v && *v) ? atoi(v) : 1;
  }();
  return on != 0;
}

cudaError_t launch_tc_gemm(const GemmParams& params, int num_sms, cudaStream_t stream) {
  GemmParams p = params;
  for (int i = 0; i < p.nseg; ++i) {
    GemmSegment& g = p.seg[i];
    if (!g.own_mode) {
      g.mode = params.mode;
      g.nt = params.nt;
    }
    if (g.nt > p.nt) p.nt = g.nt;  // the token ring holds the largest tile
  }
  // FP8 weights: every segment packed FP8, two weight tiles per unit, no pairs
  p.fp8 = p.seg[0].a_fp8 ? 1 : 0;
  for (int i = 0; i < p.nseg; ++i)
    if ((p.seg[i].a_fp8 != 0) != (p.fp8 != 0) || (p.seg[i].a_fp8 && !p.seg[i].a_packed))
      return cudaErrorInvalidValue;
  p.pair = (!p.fp8 && params.pair && pair_capable(params) && num_sms >= 2) ? 1 : 0;
  // pairs take two weight tiles per CTA (four per unit) when every segment
  // has a multiple of four 128-row tiles, else one
  bool pair_two = p.pair != 0;
  for (int i = 0; i < p.nseg; ++i)
    if (p.seg[i].a128 % 4) pair_two = false;
  p.a_per_unit = p.fp8 ? 2 : p.pair ? (pair_two ? 2 : 1) : (params.a_per_unit == 1 ? 1 : 2);
  if (p.pieces > 1) {  // single-CTA bf16 store mode, one weight tile per unit
    if (p.fp8 || p.pair || p.pieces > 4) return cudaErrorInvalidValue;
    for (int i = 0; i < p.nseg; ++i)
      if ((p.seg[i].own_mode ? p.seg[i].mode : p.mode) != kModeStore || p.seg[i].a_packed)
        return cudaErrorInvalidValue;
    p.a_per_unit = 1;
  }
  // FP8 weights with token tiles of at most 64 rows: the converters write the
  // weights into TMEM, beside two 128-column accumulator regions
  p.tmem_a = (p.fp8 && p.nt <= 64 && p.a_per_unit == 2 && fp8_tmem_enabled()) ? 1 : 0;
  const GemmPlan plan = p.fp8 ? plan_gemm_fp8(p.nt, p.tmem_a != 0)
                              : plan_gemm(p.nt, p.a_per_unit, p.pair != 0, p.pieces);
  if (p.fp8 && plan.f8_stages < 2) return cudaErrorInvalidValue;
  p.a_stages = plan.a_stages;
  p.b_stages = plan.b_stages;
  // two MMA issuers where token tiles are large enough for the single
  // issuer's per-k-step cost to show (with 32-token tiles the bf16 weight
  // stream sets the pace and the second commit per stage only delays its
  // release), and with the FP8 weights in TMEM, whose k steps come at half
  // the bytes (one issuer takes about 1000 cycles a k step, two about 500)
  p.two = (p.pieces <= 1 && (p.nt >= 128 || p.tmem_a)) ? 1 : 0;
  p.f8_stages = plan.f8_stages;
  if (p.pair)
    for (int i = 0; i < p.nseg; ++i)
      if (encode_pair_maps(p.seg[i], p.a_per_unit) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64 || !configured[dev]) {
    err = cudaFuncSetAttribute(tc_gemm_kernel<false, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(tc_gemm_kernel<true, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(tc_gemm_kernel<false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (err != cudaSuccess) return err;
    if (dev < 64) configured[dev] = 1;
  }
  if (p.pair) {  // clusters of two CTAs, one CTA per SM
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms / 2 * 2));
    cfg.blockDim = dim3(kThreadsTwo);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // as many pairs as can be resident at once (a pair's SMs share a GPC):
    // the units are dealt to the launched pairs in turn, so every pair of the
    // grid must run from the start
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, tc_gemm_kernel<true, false>, &cfg) !=
            cudaSuccess ||
        clusters < 1) {
      cudaGetLastError();
      clusters = num_sms / 2;
    }
    if (clusters > num_sms / 2) clusters = num_sms / 2;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    note_launch();
    return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<true, false>, p);
  }
  if (p.fp8)
    return launch_pdl(tc_gemm_kernel<false, true>, dim3(num_sms), dim3(kThreadsFp8),
                      plan.smem_bytes, stream, p);
  return launch_pdl(tc_gemm_kernel<false, false>, dim3(num_sms), dim3(kThreadsTwo), plan.smem_bytes,
                    stream, p);
}

cudaError_t launch_pack_weights(int kind, int64_t groups, int64_t rows, int64_t cols,
                                const void* src, void* dst, cudaStream_t stream) {
  const int64_t n = groups * rows * cols / 8;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  if (blocks < 1) return cudaSuccess;
  note_launch();
  pack_weights_kernel<uint4><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      kind, groups, rows, cols, static_cast<const uint4*>(src), static_cast<uint4*>(dst));
  return cudaGetLastError();
}

int64_t packed_fp8_bytes(int64_t groups, int64_t rows, int64_t cols) {
  const int64_t npairs = (rows / 128 + 1) / 2;
  return groups * rows * cols + groups * npairs * (cols / kBK) * 16;
}

cudaError_t launch_pack_weights_fp8(int kind, int64_t groups, int64_t rows, int64_t cols,
                                    const void* codes, const float* scales, void* dst,
                                    cudaStream_t stream) {
  const int64_t n = groups * rows * cols / 8;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  if (blocks < 1) return cudaSuccess;
  note_launch();
  pack_weights_kernel<uint2><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      kind, groups, rows, cols, static_cast<const uint2*>(codes), static_cast<uint2*>(dst));
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int64_t nrec = groups * ((rows / 128 + 1) / 2) * (cols / kBK);
  int64_t rblocks = (nrec + 255) / 256;
  if (rblocks > 65536) rblocks = 65536;
  note_launch();
  pack_scale_records_kernel<<<static_cast<unsigned>(rblocks), 256, 0, stream>>>(
      kind, groups, rows, cols, scales,
      reinterpret_cast<float4*>(static_cast<uint8_t*>(dst) + groups * rows * cols));
  return cudaGetLastError();
}

cudaError_t launch_split_router_weight(const float* W_r, int E, int d, __nv_bfloat16* W_split,
                                       cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(E) * d / 8;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  return launch_pdl(split_router_weight_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                    stream, W_r, E, d, W_split);
}

}  // namespace fgs
