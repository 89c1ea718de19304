// Dispatch and combine of the fine-grained MoE layer.
//
// "Kimi K2 MoE", section 3: the routed output is produced by a dispatch of
// each token to its K experts and a weighted combine (dispatch_and_combine,
// whose body the page does not give), added to the shared expert's output.
// The order of the dispatched rows is this library's choice: expert-major,
// ascending token index within an expert, which makes every run bit-for-bit
// reproducible.
//
// Kernels
//   histogram_kernel  per-expert counts (shared-memory atomics; counts are
//                     integers, so the result does not depend on their order)
//   scatter_kernel    one CTA per expert: its offset from a block reduction
//                     over the counts, then a stable ballot/prefix scan over
//                     the T*K pairs -> perm / inv
//   build_tiles_kernel  row tiles for the grouped GEMMs (one CTA, E <= 1024)
//   gather_kernel     Xp[r] = x[perm[r] / K], w_perm[r] = topk_w[perm[r]]
//   combine_kernel    y[t] = sum_k w[t, k] Y[inv[t K + k]] + dense addends, fp32
//                     sums in that order (w = 1 when absent)
#include "common.cuh"
#include "internal.h"

namespace fgs {

namespace {

__global__ void histogram_kernel(const int32_t* __restrict__ idx, int64_t n, int E,
                                 int32_t* __restrict__ counts, int* status) {
  extern __shared__ int hist[];
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < n; j += stride) {
    const int e = __ldg(idx + j);
    if (e >= 0 && e < E) {
      atomicAdd(&hist[e], 1);
    } else {
      record_status(status, MOE_ERR_DEVICE_INDEX);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    if (hist[i]) atomicAdd(counts + i, hist[i]);
}

__device__ __forceinline__ int block_sum(int v, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int tot = 0;
  for (int w = 0; w < nw; ++w) tot += red[w];
  __syncthreads();
  return tot;
}

constexpr int kScatterThreads = 512;

__global__ void __launch_bounds__(kScatterThreads) scatter_kernel(
    const int32_t* __restrict__ idx, int64_t n, int E, const int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  __shared__ int red[kScatterThreads / 32];
  __shared__ int wcnt[kScatterThreads / 32];
  const int e = blockIdx.x;
  int part = 0;
  for (int i = threadIdx.x; i < e; i += blockDim.x) part += counts[i];
  const int base = block_sum(part, red);
  const int mine = counts[e];
  if (threadIdx.x == 0) {
    offsets[e] = base;
    if (e == E - 1) offsets[E] = base + mine;
  }
  if (mine == 0) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  int running = 0;
  for (int64_t j0 = 0; j0 < n && running < mine; j0 += blockDim.x) {
    const int64_t j = j0 + threadIdx.x;
    const bool hit = j < n && __ldg(idx + j) == e;
    const unsigned ballot = __ballot_sync(0xffffffffu, hit);
    if (lane == 0) wcnt[warp] = __popc(ballot);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < nw; ++w) {
      const int c = wcnt[w];
      before += (w < warp) ? c : 0;
      total += c;
    }
    if (hit) {
      const int slot = base + running + before + __popc(ballot & lt_mask);
      perm[slot] = static_cast<int32_t>(j);
      inv[j] = slot;
    }
    running += total;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(1024) build_tiles_kernel(const int32_t* __restrict__ offsets,
                                                           int E, int nt,
                                                           RowTile* __restrict__ tiles,
                                                           int* __restrict__ ntiles,
                                                           int32_t* __restrict__ poffsets) {
  __shared__ int scan[1024];
  __shared__ int pscan[1024];
  const int e = threadIdx.x;
  const int m = e < E ? offsets[e + 1] - offsets[e] : 0;
  // tile height: a multiple of 8, at most nt, tiles as even as that allows
  int per = 0, nti = 0;
  if (m > 0) {
    const int n0 = (m + nt - 1) / nt;
    per = (((m + n0 - 1) / n0) + 7) & ~7;
    if (per > nt) per = nt;
    nti = (m + per - 1) / per;
  }
  scan[e] = nti;
  pscan[e] = (m + 7) & ~7;
  __syncthreads();
  // inclusive Hillis-Steele scans over 1024 entries
  for (int off = 1; off < 1024; off <<= 1) {
    const int v = e >= off ? scan[e - off] : 0;
    const int pv = e >= off ? pscan[e - off] : 0;
    __syncthreads();
    scan[e] += v;
    pscan[e] += pv;
    __syncthreads();
  }
  const int first = scan[e] - nti;
  const int pfirst = pscan[e] - ((m + 7) & ~7);
  if (e == 1023) *ntiles = scan[1023];
  if (poffsets && e < E) {
    poffsets[e] = pfirst;
    if (e == E - 1) poffsets[E] = pscan[e];
  }
  if (nti == 0) return;
  const int row0 = offsets[e];
  for (int i = 0; i < nti; ++i) {
    const int start = i * per;
    RowTile t;
    t.expert = e;
    t.row_start = row0 + start;
    t.n_rows = min(per, m - start);
    t.first_tile = first;
    t.ntiles = nti;
    t.prow = pfirst + start;
    t.pad0 = t.pad1 = 0;
    tiles[first + i] = t;
  }
}

// Packed gather: one warp per slot row.  Row r of expert e (found by binary
// search in offsets) goes to padded row R = poffsets[e] + (r - offsets[e]);
// its 16-byte chunk v (columns 8v..8v+7) to plane v / 8 at chunk position
// (v % 8) XOR (R % 8) -- the 128-byte swizzle the tensor cores read.
__global__ void __launch_bounds__(256) gather_packed_kernel(
    const uint4* __restrict__ x, int K, int vec_per_row, const int32_t* __restrict__ perm,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ poffsets, int E,
    const float* __restrict__ topk_w, uint4* __restrict__ Xp, int64_t plane_rows,
    float* __restrict__ w_perm) {
  const int rows = offsets[E];
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = warp_global; r < rows; r += nwarps) {
    int lo = 0, hi = E;  // offsets[lo] <= r < offsets[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(offsets + mid) <= r) lo = mid; else hi = mid;
    }
    const int64_t R = __ldg(poffsets + lo) + (r - __ldg(offsets + lo));
    const int j = __ldg(perm + r);
    const uint4* src = x + static_cast<int64_t>(j / K) * vec_per_row;
    const int sw = static_cast<int>(R & 7);
    for (int v = lane; v < vec_per_row; v += 32) {
      const int64_t plane = v >> 3;
      Xp[(plane * plane_rows + R) * 8 + ((v & 7) ^ sw)] = __ldg(src + v);
    }
    if (lane == 0 && w_perm) w_perm[r] = topk_w ? __ldg(topk_w + j) : 1.0f;
  }
}

// One warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ x, int K,
                                                     int vec_per_row,
                                                     const int32_t* __restrict__ perm,
                                                     const int32_t* __restrict__ offsets, int E,
                                                     const float* __restrict__ topk_w,
                                                     uint4* __restrict__ Xp,
                                                     float* __restrict__ w_perm) {
  const int rows = offsets[E];
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = warp_global; r < rows; r += nwarps) {
    const int j = __ldg(perm + r);
    const int t = j / K;
    const uint4* src = x + static_cast<int64_t>(t) * vec_per_row;
    uint4* dst = Xp + r * vec_per_row;
    for (int v = lane; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
    if (lane == 0 && w_perm) w_perm[r] = topk_w ? __ldg(topk_w + j) : 1.0f;
  }
}

template <bool BF16>
struct Vec8;

template <>
struct Vec8<true> {
  static __device__ __forceinline__ void load(const void* p, int64_t i, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p) + i);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(h[q]);
      v[2 * q] = f.x;
      v[2 * q + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store(void* p, int64_t i, const float (&v)[8]) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) h[q] = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
    reinterpret_cast<uint4*>(p)[i] = u;
  }
};

template <>
struct Vec8<false> {
  static __device__ __forceinline__ void load(const void* p, int64_t i, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p) + 2 * i);
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 2 * i + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  static __device__ __forceinline__ void store(void* p, int64_t i, const float (&v)[8]) {
    reinterpret_cast<float4*>(p)[2 * i] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[2 * i + 1] = make_float4(v[4], v[5], v[6], v[7]);
  }
};

// One CTA per token row; D must be a multiple of 8.
template <bool BF16>
__global__ void __launch_bounds__(128) combine_kernel(const void* __restrict__ Y,
                                                      const int32_t* __restrict__ inv,
                                                      const float* __restrict__ w, int K,
                                                      int D, const void* __restrict__ adds,
                                                      int n_add, int64_t add_stride_rows,
                                                      void* __restrict__ y) {
  using V = Vec8<BF16>;
  const int64_t t = blockIdx.x;
  const int nvec = D / 8;
  __shared__ int slots[64];
  __shared__ float wts[64];
  if (threadIdx.x < K) {
    slots[threadIdx.x] = __ldg(inv + t * K + threadIdx.x);
    wts[threadIdx.x] = w ? __ldg(w + t * K + threadIdx.x) : 1.0f;
  }
  __syncthreads();
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float tmp[8];
    for (int k = 0; k < K; ++k) {
      V::load(Y, static_cast<int64_t>(slots[k]) * nvec + v, tmp);
      const float wk = wts[k];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = fmaf(wk, tmp[q], acc[q]);
    }
    for (int a = 0; a < n_add; ++a) {
      V::load(adds, (a * add_stride_rows + t) * nvec + v, tmp);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += tmp[q];
    }
    V::store(y, t * nvec + v, acc);
  }
}

}  // namespace

cudaError_t launch_permute(const int32_t* topk_idx, int64_t T, int K, int E, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, int* status,
                           cudaStream_t stream) {
  const int64_t n = T * K;
  cudaError_t err = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, stream);
  if (err != cudaSuccess) return err;
  const int threads = 256;
  int64_t blocks = (n + threads * 4 - 1) / (threads * 4);
  if (blocks > 1024) blocks = 1024;
  if (blocks < 1) blocks = 1;
  note_launch();
  histogram_kernel<<<static_cast<unsigned>(blocks), threads, sizeof(int) * E, stream>>>(
      topk_idx, n, E, counts, status);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  note_launch();
  scatter_kernel<<<E, kScatterThreads, 0, stream>>>(topk_idx, n, E, counts, offsets, perm, inv);
  return cudaGetLastError();
}

int64_t max_tiles(int64_t rows, int E, int nt) { return rows / nt + E; }

cudaError_t launch_build_tiles(const int32_t* offsets, int E, int nt, RowTile* tiles, int* ntiles,
                               int32_t* poffsets, cudaStream_t stream) {
  note_launch();
  build_tiles_kernel<<<1, 1024, 0, stream>>>(offsets, E, nt, tiles, ntiles, poffsets);
  return cudaGetLastError();
}

cudaError_t launch_gather_packed(const void* x, int K, int width, const int32_t* perm,
                                 const int32_t* offsets, const int32_t* poffsets, int E,
                                 const float* topk_w, void* Xp, int64_t plane_rows,
                                 float* w_perm, cudaStream_t stream) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  note_launch();
  gather_packed_kernel<<<sms * 8, 256, 0, stream>>>(
      static_cast<const uint4*>(x), K, width / 8, perm, offsets, poffsets, E, topk_w,
      static_cast<uint4*>(Xp), plane_rows, w_perm);
  return cudaGetLastError();
}

cudaError_t launch_gather(const void* x, int64_t T, int K, int width, int elem_bytes,
                          const int32_t* perm, const int32_t* offsets, int E,
                          const float* topk_w, void* Xp, float* w_perm, cudaStream_t stream) {
  (void)T;
  const int vec_per_row = width * elem_bytes / 16;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  note_launch();
  gather_kernel<<<sms * 8, 256, 0, stream>>>(static_cast<const uint4*>(x), K, vec_per_row, perm,
                                             offsets, E, topk_w, static_cast<uint4*>(Xp), w_perm);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* Y, const int32_t* inv, const float* w, int64_t T, int K,
                           int D, const void* adds, int n_add, int64_t add_stride_rows, void* y,
                           bool bf16, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  if (bf16) {
    note_launch();
    combine_kernel<true><<<static_cast<unsigned>(T), 128, 0, stream>>>(Y, inv, w, K, D, adds,
                                                                       n_add, add_stride_rows, y);
  } else {
    note_launch();
    combine_kernel<false><<<static_cast<unsigned>(T), 128, 0, stream>>>(Y, inv, w, K, D, adds,
                                                                        n_add, add_stride_rows, y);
  }
  return cudaGetLastError();
}

}  // namespace fgs
