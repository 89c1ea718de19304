// fp32 expert GEMMs on the CUDA cores, for layers whose activations and
// expert weights are fp32 (the tensor cores' fp32-class input, tf32, keeps
// only 10 mantissa bits and would not meet an fp32 tolerance).
//
// Same computation as the tensor-core path ("Kimi K2 MoE", section 2,
// SwiGLU experts): per row tile of one expert (16 rows), each CTA produces a
// 16 x 16 block of outputs with shared-memory tiles of the rows and weights,
// fp32 fused multiply-adds in ascending k order.
#include "common.cuh"
#include "internal.h"

namespace fgs {

namespace {

__global__ void __launch_bounds__(256) simt_gemm_kernel(const SimtGemm g) {
  constexpr int TS = kSimtTile;
  __shared__ float Bs[TS][TS + 1];
  __shared__ float Ws[TS][TS + 1];
  __shared__ float Us[TS][TS + 1];
  const int tile = blockIdx.x;
  int group, b_row, out_row, n_rows;
  if (g.tiles) {
    if (tile >= *g.ntiles) return;
    const RowTile t = g.tiles[tile];
    group = t.expert;
    b_row = t.row_start;
    out_row = t.row_start;
    n_rows = t.n_rows;
  } else {
    const int tpg = (g.rows + TS - 1) / TS;
    if (tile >= g.groups * tpg) return;
    group = tile / tpg;
    const int t0 = (tile - group * tpg) * TS;
    n_rows = min(TS, g.rows - t0);
    b_row = static_cast<int>(group * g.b_group_stride + t0);
    out_row = static_cast<int>(group * g.out_group_stride + t0);
  }
  const int tx = threadIdx.x % TS, ty = threadIdx.x / TS;
  const int o0 = blockIdx.y * TS;
  const float* W = g.W + group * g.w_group_stride;
  float acc = 0.f, acc_u = 0.f;
  for (int k0 = 0; k0 < g.Kdim; k0 += TS) {
    const int k = k0 + tx;
    Bs[ty][tx] = (ty < n_rows && k < g.Kdim) ? g.B[static_cast<int64_t>(b_row + ty) * g.Kdim + k] : 0.f;
    const int o = o0 + ty;
    Ws[ty][tx] = (o < g.O && k < g.Kdim) ? W[static_cast<int64_t>(o) * g.Kdim + k] : 0.f;
    if (g.swiglu)
      Us[ty][tx] = (o < g.O && k < g.Kdim) ? W[static_cast<int64_t>(g.O + o) * g.Kdim + k] : 0.f;
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TS; ++kk) {
      acc = fmaf(Bs[ty][kk], Ws[tx][kk], acc);
      if (g.swiglu) acc_u = fmaf(Bs[ty][kk], Us[tx][kk], acc_u);
    }
    __syncthreads();
  }
  const int o = o0 + tx;
  if (ty < n_rows && o < g.O) {
    float val;
    if (g.swiglu) {
      val = acc / (1.0f + expf(-acc)) * acc_u;
    } else {
      val = g.row_scale ? acc * g.row_scale[out_row + ty] : acc;
    }
    g.out[static_cast<int64_t>(out_row + ty) * g.O + o] = val;
  }
}

}  // namespace

cudaError_t launch_simt_gemm(const SimtGemm& g, int64_t tiles_bound, cudaStream_t stream) {
  if (tiles_bound <= 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(tiles_bound), static_cast<unsigned>((g.O + kSimtTile - 1) / kSimtTile));
  note_launch();
  simt_gemm_kernel<<<grid, kSimtTile * kSimtTile, 0, stream>>>(g);
  return cudaGetLastError();
}

}  // namespace fgs
