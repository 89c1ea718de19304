// Launch interfaces between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace fgs {

// Every kernel launch of the library is counted once, on the host, when it is
// enqueued (read through moe_launch_count).
void note_launch();

// Launch a hot-path kernel with programmatic stream serialization (the
// kernel calls pdl_release / pdl_wait, see common.cuh), so that it starts
// while the previous kernel of the stream drains; FGS_PDL=0 launches plainly.
bool pdl_enabled();
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  note_launch();
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}


// ----------------------------------------------------------------- router
struct RouterArgs {
  const void* x = nullptr;        // [T, d] (bf16 when x_bf16, else fp32)
  const float* logits = nullptr;  // [T, E]; when set the GEMM is skipped
  int logit_parts = 1;            // logits = sum of this many [T, E] arrays
  int64_t logit_part_stride = 0;  // elements between the parts
  const float* W_r = nullptr;     // [E, d]
  const float* bias = nullptr;    // [E]
  int64_t T = 0;
  int d = 0, E = 0, K = 0, G = 1, Gk = 1;
  float scale = 2.827f;
  int norm = 1;
  bool x_bf16 = true;
  int32_t* topk_idx = nullptr;
  float* topk_w = nullptr;
};
cudaError_t launch_router(const RouterArgs& a, cudaStream_t stream);
// G [T, E] from the routing (0 off the selected experts); K <= 32.
cudaError_t launch_dense_gates(const int32_t* topk_idx, const float* topk_w, int64_t T, int K,
                               int E, float* G, cudaStream_t stream);
// bias[e] += gamma * sign(T K / E - counts[e]).
cudaError_t launch_bias_update(const int32_t* counts, int64_t T, int K, int E, float gamma,
                               float* bias, cudaStream_t stream);
// Quantile Balancing: theta[e] = the ceil(T K / E)-th largest fp32 score of
// expert e in logits [T, E]; bias[e] += rate (mean(theta) - theta[e] - bias[e]).
cudaError_t launch_quantile_bias(const float* logits, int64_t T, int K, int E, float rate,
                                 float* theta, float* bias, cudaStream_t stream);

// --------------------------------------------------------------- dispatch
// One row tile of a routed expert: rows [row_start, row_start + n_rows) of
// the gathered activations, all belonging to `expert`, whose tiles are
// [first_tile, first_tile + ntiles) of the table.
struct __align__(16) RowTile {
  int expert, row_start, n_rows, first_tile;
  int ntiles;
  int prow;  // first row in the padded (8-row aligned per expert) row space
  int pad0, pad1;
};

// Chunks of the pair sequence the permute counts separately (scratch:
// permute_chunks(T*K) * E int32 in ccount).
int64_t permute_chunks(int64_t n);
cudaError_t launch_permute(const int32_t* topk_idx, int64_t T, int K, int E, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* ccount,
                           int* status, cudaStream_t stream);

// Row tiles of the routed experts: for expert e with m_e rows starting at
// offsets[e], tiles of near-equal height (multiples of 8 but the last) and at
// most nt rows; *ntiles receives the count.  poffsets (E+1 entries, may be
// null) receives the padded offsets: expert e's rows start at poffsets[e] in
// a row space where every expert begins on a multiple of 8.
cudaError_t launch_build_tiles(const int32_t* offsets, int E, int nt, RowTile* tiles, int* ntiles,
                               int32_t* poffsets, cudaStream_t stream);

// Padded rows of the packed activation planes: T*K rows, up to 7 padding
// rows per expert, 32 rows of slack for whole-16-row reads.
inline int64_t packed_plane_rows(int64_t rows, int groups) { return rows + 8ll * groups + 32; }

// Xp in the packed activation layout: plane p (columns 64p..64p+63) holds
// one 128-byte row per padded row, its 16-byte chunks swizzled by (row % 8).
cudaError_t launch_gather_packed(const void* x, int K, int width, const int32_t* perm,
                                 const int32_t* offsets, const int32_t* poffsets, int E,
                                 const float* topk_w, void* Xp, int64_t plane_rows,
                                 float* w_perm, cudaStream_t stream);
int64_t max_tiles(int64_t rows, int E, int nt);
// The same packed rows written in token order: each x row is read once and
// stored to the padded rows of its K pairs (from topk_idx and inv).
cudaError_t launch_gather_tokens_packed(const void* x, int64_t T, int K, int width,
                                        const int32_t* topk_idx, const int32_t* inv,
                                        const int32_t* offsets, const int32_t* poffsets, int E,
                                        const float* topk_w, void* Xp, int64_t plane_rows,
                                        float* w_perm, cudaStream_t stream);

// Xp[r] = x[perm[r] / K] and w_perm[r] = topk_w[perm[r]] (1 if topk_w null)
// for r < rows (rows = offsets[E] read on the device).
cudaError_t launch_gather(const void* x, int64_t T, int K, int width, int elem_bytes,
                          const int32_t* perm, const int32_t* offsets, int E,
                          const float* topk_w, void* Xp, float* w_perm, cudaStream_t stream);

// y[t] = sum_k Y[inv[t*K+k]] (K may be 0) + sum_{a < n_add} add_a[t] where
// add_a = adds + a * add_stride rows of width D.  fp32 sums, fixed order.
// w: routing weights [T, K] in token order applied to the routed rows, or
// null (weights already in Y).
cudaError_t launch_combine(const void* Y, const int32_t* inv, const float* w, int64_t T, int K,
                           int D, const void* adds, int n_add, int64_t add_stride_rows, void* y,
                           bool bf16, cudaStream_t stream);

// ------------------------------------------------- tensor-core grouped GEMM
enum GemmMode : int { kModeSwiGLU = 0, kModeStore = 1 };

// One launch runs up to two segments (routed experts, then shared experts or
// a dense projection).  A unit is 256 weight rows (two 128-row A tiles; one
// at the tail of O) times one row tile of at most nt activation rows.
struct GemmSegment {
  CUtensorMap tmA;  // weights (see gemm_tc.cu for the layouts)
  CUtensorMap tmB;  // activation rows [rows, K] bf16, box 64 x b_box_rows
  int b_box_rows;   // rows of one tmB box: a whole token tile in one copy
  const void* b_src;   // the rows tmB maps (re-encoded with 32-row boxes for
  int64_t b_src_rows;  // CTA pairs, which load half tiles)
  int k_steps;      // A's K / 64
  int a128;         // 128-row A tiles along O (SwiGLU: F/64, store: O/128)
  int a_boxes;      // SwiGLU A tile: 1 = one 5-D box, 8 = eight 16-row boxes
  int a_rows;       // SwiGLU: F (row offset of the up half)
  int o_limit;      // store mode: columns o >= o_limit are not written
  int ksplit;       // K split into ksplit parts (0 or 1: none) of k_steps
                    // j / ksplit .. (j + 1) k_steps / ksplit; part j writes
                    // out_f32 + j * out_split_stride (fp32 store only)
  int a_piece_cols;  // GemmParams::pieces > 1: A column offset of piece p is
                     // p * a_piece_cols
  int64_t out_split_stride;
  // packed weights (one contiguous bulk copy per stage) instead of tmA
  const uint8_t* a_packed;
  int64_t a_group_bytes;
  int a_groups;  // groups in the packed bank
  // FP8 E4M3 packed weights (see moe_pack_weights_fp8): a_packed holds 8 KB
  // tiles, a_rec the 16-byte block-scale record of each (tile pair, k step),
  // a_rec_group records per group
  int a_fp8;
  const uint8_t* a_rec;
  int64_t a_rec_group;
  // explicit tiles (routed experts) or implicit ones (groups x rows)
  const RowTile* tiles;
  const int* ntiles;
  int groups;
  int rows;
  int64_t b_group_stride;
  int64_t out_group_stride;
  __nv_bfloat16* out;  // bf16 output, or
  float* out_f32;      // fp32 output (store mode)
  int64_t out_ld;
  const float* row_scale;    // store mode: per token row (the unpadded row space),
                             // scales the output row; may be null
  const __nv_bfloat16* add;  // store mode: added to the output, may be null
  int64_t add_ld;
  // packed activations (see launch_gather_packed): B read by one bulk copy
  // per stage from b_packed, and/or the SwiGLU output written to `out` in
  // that layout (plane rows out_plane_rows)
  const uint8_t* b_packed;
  int64_t b_plane_rows;
  int out_packed;
  int64_t out_plane_rows;
  // the segment's own pass (kModeSwiGLU / kModeStore) and token tile, when
  // own_mode is set; otherwise the launch's GemmParams::mode and ::nt
  int own_mode;
  int mode;
  int nt;
  // implicit tiles only: 1 = a token tile's units (all K parts and output
  // blocks) run side by side, so the tile is fetched from HBM once while the
  // weights, small enough to stay in L2, are re-read from there; 0 = the
  // output blocks outermost (weights fetched once, token tiles re-read)
  int b_major;
};

struct GemmParams {
  GemmSegment seg[2];
  int nseg;
  int mode;      // pass of the segments without their own (GemmSegment::own_mode)
  int nt;        // token tile (MMA N upper bound): 32, 64, 128 or 256; the
                 // launch takes the largest of its segments
  int a_per_unit;  // 128-row weight tiles per unit: 2 (default) or 1
  // 1: run on CTA pairs (clusters of two) with MMAs of M = 256 over the pair;
  // each CTA takes one of a unit's two 128-row weight tiles and half of its
  // token tile.  Applied only when pair_capable(); implies one weight tile
  // per CTA.
  int pair;
  int a_stages;  // weight ring depth (bf16 weight tiles the MMAs read)
  int b_stages;  // token ring depth
  // 1: the segments' weights are FP8 (a_fp8): their tiles land in a ring of
  // f8_stages FP8 stages and converter warps write the bf16 weight ring
  int fp8;
  int f8_stages;
  // 1: the MMAs of the two accumulators are issued by two threads, each
  // committing its own (set by launch_tc_gemm for large token tiles)
  int two;
  // > 1 (single-CTA bf16 store mode, one weight tile per unit): the weights
  // are the sum of `pieces` matrices side by side along A's columns (the
  // split router weight); each k step of B is matched by `pieces` weight
  // stages, one per piece, all accumulated into the unit's accumulator, so
  // a token stage is read by pieces x 4 MMAs
  int pieces;
  // FP8 weights, token tiles of at most 64 rows (set by launch_tc_gemm): the
  // converter warps write the bf16 weight tiles into TMEM, where the MMAs
  // read them, instead of into shared-memory stages
  int tmem_a;
  int* status;
};

struct GemmPlan {
  int nt, a_stages, b_stages, f8_stages;
  size_t smem_bytes;
};
GemmPlan plan_gemm(int nt, int a_per_unit, bool pair, int pieces = 1);
GemmPlan plan_gemm_fp8(int nt, bool tmem_a = false);
// Whether a launch can run on CTA pairs (packed weights with an even number
// of 128-row tiles in every segment, no K split).
bool pair_capable(const GemmParams& p);

cudaError_t launch_tc_gemm(const GemmParams& p, int num_sms, cudaStream_t stream);

// Rearrange an FP8 bank and its block scales into the packed FP8 order (see
// moe_pack_weights_fp8); packed_fp8_bytes is its size.
int64_t packed_fp8_bytes(int64_t groups, int64_t rows, int64_t cols);
cudaError_t launch_pack_weights_fp8(int kind, int64_t groups, int64_t rows, int64_t cols,
                                    const void* codes, const float* scales, void* dst,
                                    cudaStream_t stream);

// Rearrange a bf16 weight bank into the packed order (see moe_pack_weights).
cudaError_t launch_pack_weights(int kind, int64_t groups, int64_t rows, int64_t cols,
                                const void* src, void* dst, cudaStream_t stream);

// W_split[e] = [hi | mid | lo] (bf16, 3 d wide) with hi + mid + lo = W_r[e]
// to about 2^-24 relative: the router GEMM on bf16 tensor cores.
cudaError_t launch_split_router_weight(const float* W_r, int E, int d, __nv_bfloat16* W_split,
                                       cudaStream_t stream);

// Encode tensor maps (driver entry point fetched through the runtime).
CUresult encode_tmap_2d_rows(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                             int box_rows);
CUresult encode_tmap_weights_3d(CUtensorMap* map, const void* base, int64_t groups,
                                int64_t rows, int64_t cols, int box_rows);
CUresult encode_tmap_gate_up_5d(CUtensorMap* map, const void* base, int64_t groups, int64_t F,
                                int64_t cols);

// ------------------------------------------------------- fp32 CUDA-core path
// Same row tiles, 16 rows each; out[r, o] for o < O:
//   SwiGLU: SiLU(B[r] . W[g, o]) * (B[r] . W[g, O + o])
//   plain:  row_scale[r] * (B[r] . W[g, o])
struct SimtGemm {
  const float* B = nullptr;      // activation rows, row stride Kdim
  const float* W = nullptr;      // group g at W + g * w_group_stride, row stride Kdim
  int64_t w_group_stride = 0;
  int Kdim = 0;
  int O = 0;
  bool swiglu = false;
  const RowTile* tiles = nullptr;  // explicit tiles, or null for implicit ones
  const int* ntiles = nullptr;
  int groups = 0, rows = 0;      // implicit tiles over [0, rows) per group
  int64_t b_group_stride = 0, out_group_stride = 0;
  float* out = nullptr;          // row stride O
  const float* row_scale = nullptr;
};
constexpr int kSimtTile = 16;
cudaError_t launch_simt_gemm(const SimtGemm& g, int64_t tiles_bound, cudaStream_t stream);

}  // namespace fgs
