// Launch interfaces between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace fgs {

// ----------------------------------------------------------------- router
struct RouterArgs {
  const void* x = nullptr;        // [T, d] (bf16 when x_bf16, else fp32)
  const float* logits = nullptr;  // [T, E]; when set the GEMM is skipped
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

// --------------------------------------------------------------- dispatch
cudaError_t launch_permute(const int32_t* topk_idx, int64_t T, int K, int E, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, int* status,
                           cudaStream_t stream);

// Row tiles of the routed experts: for expert e with m_e rows starting at
// offsets[e], ceil(m_e / nt) tiles of near-equal height.  Entry
// {expert, first row, rows, 0}; *ntiles receives the count.
cudaError_t launch_build_tiles(const int32_t* offsets, int E, int nt, int4* tiles, int* ntiles,
                               cudaStream_t stream);
int64_t max_tiles(int64_t rows, int E, int nt);

// Xp[r] = x[perm[r] / K] and w_perm[r] = topk_w[perm[r]] (1 if topk_w null)
// for r < rows (rows = offsets[E] read on the device).
cudaError_t launch_gather(const void* x, int64_t T, int K, int width, int elem_bytes,
                          const int32_t* perm, const int32_t* offsets, int E,
                          const float* topk_w, void* Xp, float* w_perm, cudaStream_t stream);

// y[t] = sum_k Y[inv[t*K+k]] (K may be 0) + sum_{a < n_add} add_a[t] where
// add_a = adds + a * add_stride rows of width D.  fp32 sums, fixed order.
cudaError_t launch_combine(const void* Y, const int32_t* inv, int64_t T, int K, int D,
                           const void* adds, int n_add, int64_t add_stride_rows, void* y,
                           bool bf16, cudaStream_t stream);

// ------------------------------------------------- tensor-core grouped GEMM
enum GemmMode : int { kModeSwiGLU = 0, kModeStore = 1 };

struct GemmSegment {
  CUtensorMap tmA;  // weights (see gemm_tc.cu for the layouts)
  CUtensorMap tmB;  // activation rows [rows, K] bf16, box 64 x 32
  int k_steps;      // K / 64
  int o_blocks;     // output blocks per row tile (F/64 SwiGLU, O/128 store)
  int a_boxes;      // 1: one A box per stage; 8: eight 16-row boxes (SwiGLU only)
  int a_rows;       // SwiGLU: F (row offset of the up half); store: unused
  // explicit tiles (routed experts)
  const int4* tiles;
  const int* ntiles;
  // implicit tiles: groups x ceil(rows / nt) over rows [0, rows)
  int groups;
  int rows;
  int64_t b_group_stride;
  int64_t out_group_stride;
  __nv_bfloat16* out;
  int64_t out_ld;
  const float* row_scale;  // per output row, may be null
  const __nv_bfloat16* add;  // store mode: added to the output (same shape), may be null
  int64_t add_ld;
};

struct GemmParams {
  GemmSegment seg[2];
  int nseg;
  int mode;
  int nt;      // token tile (MMA N upper bound): 32, 64, 128 or 256
  int stages;  // pipeline depth
  int* status;
};

struct GemmPlan {
  int nt, stages;
  size_t smem_bytes;
};
GemmPlan plan_gemm(int nt);

cudaError_t launch_tc_gemm(const GemmParams& p, int num_sms, cudaStream_t stream);

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
  const int4* tiles = nullptr;   // explicit tiles, or null for implicit ones
  const int* ntiles = nullptr;
  int groups = 0, rows = 0;      // implicit tiles over [0, rows) per group
  int64_t b_group_stride = 0, out_group_stride = 0;
  float* out = nullptr;          // row stride O
  const float* row_scale = nullptr;
};
constexpr int kSimtTile = 16;
cudaError_t launch_simt_gemm(const SimtGemm& g, int64_t tiles_bound, cudaStream_t stream);

}  // namespace fgs
