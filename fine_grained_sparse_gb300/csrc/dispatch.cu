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
// A stable counting sort of the T*K (token, expert) pairs in chunks of
// consecutive pairs (a power of two from 32 to 1024, about 256 chunks):
//   chunk_count_kernel  per-chunk, per-expert counts (shared-memory atomics;
//                       integer counts do not depend on their order)
//   chunk_scan_kernel   a CTA per 32 experts: counts[e], and each chunk's
//                       start within each expert (exclusive scan over chunks)
//   chunk_scatter_kernel offsets (exclusive scan of counts over the experts,
//                       in every CTA; CTA 0 stores them), then one warp per
//                       chunk, its pairs in order, 32 at a
//                       time: a pair's slot is its expert's running position
//                       in the chunk plus its rank among the lanes of the
//                       same expert (match_any) -> perm / inv
//   build_tiles_kernel  row tiles for the grouped GEMMs (one CTA, E <= 1024)
//   gather_packed_kernel  Xp[r] = x[perm[r] / K] in the packed plane layout
//                     the tensor cores read (x read with an L2 evict-last
//                     hint, Xp written evict-first), w_perm[r] = topk_w[perm[r]]
//   gather_tokens_packed_kernel  the same rows written in token order: x[t]
//                     read once, stored to the padded rows of its K pairs
//                     (the layer forward, which has topk_idx and inv)
//   gather_kernel     the same in plain rows (fp32 layers)
//   combine_kernel    y[t] = sum_k w[t, k] Y[inv[t K + k]] + dense addends, fp32
//                     sums in that order (w = 1 when absent); a slot outside
//                     [0, T K) (inv = -1: a pair the permute rejected) adds
//                     nothing
// All are launched with programmatic stream serialization and wait for the
// previous kernel (pdl_wait) before touching global memory.
#include "common.cuh"
#include "internal.h"

namespace fgs {

namespace {

// 16-byte global load / store with an L2 eviction-priority hint.
__device__ __forceinline__ uint4 ld_global_hint(const uint4* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}
__device__ __forceinline__ void st_global_hint(uint4* p, uint4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
               : "memory");
}


constexpr int kChunkThreads = 256;
constexpr int kScatterWarps = 8;       // chunks per CTA of the scatter

__global__ void __launch_bounds__(kChunkThreads) chunk_count_kernel(
    const int32_t* __restrict__ idx, int64_t n, int chunk, int E, int32_t* __restrict__ ccount,
    int* status) {
  pdl_wait();
  extern __shared__ int hist[];
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * chunk;
  for (int i = threadIdx.x; i < chunk; i += blockDim.x) {
    const int64_t j = j0 + i;
    if (j >= n) break;
    const int e = __ldg(idx + j);
    if (e >= 0 && e < E)
      atomicAdd(&hist[e], 1);
    else
      record_status(status, MOE_ERR_DEVICE_INDEX);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    ccount[static_cast<int64_t>(blockIdx.x) * E + i] = hist[i];
}

// A CTA per 32 experts, 1024 threads: lane l serves expert 32 b + l and
// warp w a contiguous run of the chunks, so every load and store of a warp
// covers 32 consecutive experts.  Each warp sums its run, the warps' sums
// are scanned across the CTA, and each warp then rewrites ccount[c][e] as
// the count of e in the chunks before c; the last warp's total is counts[e].
// (The exclusive scan of counts over the experts -- the offsets -- is taken
// by the scatter kernel.)
__global__ void __launch_bounds__(1024) chunk_scan_kernel(int32_t* __restrict__ ccount,
                                                          int nchunks, int E,
                                                          int32_t* __restrict__ counts) {
  pdl_wait();
  __shared__ int part[32][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  const int per = (nchunks + 31) / 32;
  const int c0 = min(nchunks, w * per), c1 = min(nchunks, c0 + per);
  int sum = 0;
  if (e < E) {
    int c = c0;
    for (; c + 8 <= c1; c += 8) {  // eight loads in flight
      int v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = ccount[static_cast<int64_t>(c + i) * E + e];
#pragma unroll
      for (int i = 0; i < 8; ++i) sum += v[i];
    }
    for (; c < c1; ++c) sum += ccount[static_cast<int64_t>(c) * E + e];
  }
  part[w][lane] = sum;
  __syncthreads();
  int run = 0;  // this expert's count in the chunks before c0
  for (int i = 0; i < w; ++i) run += part[i][lane];
  if (e < E) {
    for (int c = c0; c < c1; ++c) {
      const int64_t at = static_cast<int64_t>(c) * E + e;
      const int v = ccount[at];
      ccount[at] = run;
      run += v;
    }
    if (w == 31) counts[e] = run;
  }
}

// offsets = the exclusive scan of counts over the experts (E <= 1024), in
// shared memory, by the 32 * kScatterWarps threads of a CTA: each thread a
// run of up to four experts, then a scan of the runs across the warps.
__device__ __forceinline__ void scan_counts(const int32_t* __restrict__ counts, int E,
                                            int* off_s, int* warp_s) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int per = (E + 32 * kScatterWarps - 1) / (32 * kScatterWarps);  // <= 4
  const int e0 = t * per;
  int v[4], run = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[i] = (i < per && e0 + i < E) ? counts[e0 + i] : 0;
    run += v[i];
  }
  int incl = run;  // inclusive scan of the runs within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) warp_s[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int i = 0; i < warp; ++i) base += warp_s[i];
  int acc = base + incl - run;  // exclusive start of this thread's run
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (i < per && e0 + i < E) off_s[e0 + i] = acc;
    acc += v[i];
  }
  if (t == 32 * kScatterWarps - 1) off_s[E] = acc;  // the last run ends the scan
  __syncthreads();
}

__global__ void __launch_bounds__(32 * kScatterWarps) chunk_scatter_kernel(
    const int32_t* __restrict__ idx, int64_t n, int chunk, int E,
    const int32_t* __restrict__ ccount, const int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int nchunks, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv) {
  pdl_wait();
  extern __shared__ int cnt_all[];
  int* off_s = cnt_all + kScatterWarps * E;  // E + 1 offsets
  __shared__ int warp_s[kScatterWarps];
  scan_counts(counts, E, off_s, warp_s);
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = off_s[e];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x * kScatterWarps + warp;
  if (c >= nchunks) return;
  int* cnt = cnt_all + warp * E;  // this chunk's next slot per expert
  for (int e = lane; e < E; e += 32)
    cnt[e] = off_s[e] + __ldg(ccount + static_cast<int64_t>(c) * E + e);
  __syncwarp();
  const unsigned lt_mask = (1u << lane) - 1u;
  const int64_t j0 = static_cast<int64_t>(c) * chunk;
  for (int s = 0; s < chunk; s += 32) {
    const int64_t j = j0 + s + lane;
    if (j0 + s >= n) break;
    const int e = j < n ? __ldg(idx + j) : -1;
    const bool ok = e >= 0 && e < E;
    // lanes of one expert share a key; every other lane has a key of its own
    const unsigned mask = __match_any_sync(0xffffffffu, ok ? e : E + lane);
    const int base = ok ? cnt[e] : 0;
    __syncwarp();
    if (ok) {
      const int slot = base + __popc(mask & lt_mask);
      perm[slot] = static_cast<int32_t>(j);
      inv[j] = slot;
      if ((mask & lt_mask) == 0) cnt[e] = base + __popc(mask);  // the group's first lane
    } else if (j < n) {
      inv[j] = -1;  // a pair whose expert index was rejected holds no slot
    }
    __syncwarp();
  }
}

__global__ void __launch_bounds__(1024) build_tiles_kernel(const int32_t* __restrict__ offsets,
                                                           int E, int nt,
                                                           RowTile* __restrict__ tiles,
                                                           int* __restrict__ ntiles,
                                                           int32_t* __restrict__ poffsets) {
  pdl_wait();
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
  pdl_wait();
  const int rows = offsets[E];
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  // each token row is read K times: keep x in L2, and let the gathered copy
  // (K times larger, read again only by the next GEMM) leave it first
  const uint64_t keep = l2_policy_evict_last();
  const uint64_t pass = l2_policy_evict_first();
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
    // eight 16-byte loads in flight per lane before their stores
    for (int v0 = lane; v0 < vec_per_row; v0 += 256) {
      uint4 t[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (v0 + 32 * u < vec_per_row) t[u] = ld_global_hint(src + v0 + 32 * u, keep);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = v0 + 32 * u;
        if (v < vec_per_row)
          st_global_hint(Xp + ((v >> 3) * plane_rows + R) * 8 + ((v & 7) ^ sw), t[u], pass);
      }
    }
    if (lane == 0 && w_perm) w_perm[r] = topk_w ? __ldg(topk_w + j) : 1.0f;
  }
}

// Packed gather in token order: one warp per token t reads x[t] once and
// writes it to the padded rows of its K pairs (the pair of slot
// s = inv[t K + k] and expert e = topk_idx[t K + k] sits in padded row
// poffsets[e] + s - offsets[e]), seven 16-byte vectors per lane at a time.
// Pairs whose expert index was rejected (inv = -1) are skipped.  Same layout
// as gather_packed_kernel; each x row is read from memory once instead of
// once per pair.
__global__ void __launch_bounds__(256) gather_tokens_packed_kernel(
    const uint4* __restrict__ x, int64_t T, int K, int vec_per_row,
    const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ inv,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ poffsets, int E,
    const float* __restrict__ topk_w, uint4* __restrict__ Xp, int64_t plane_rows,
    float* __restrict__ w_perm) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t rows = static_cast<int64_t>(T) * K;
  constexpr int kV = 7;  // vectors per lane per round (16 B each)
  const uint64_t pass = l2_policy_evict_first();
  for (int64_t t = warp_global; t < T; t += nwarps) {
    // lane k (< K) finds its pair's padded row; the warp shares them
    int64_t myR = -1;
    if (lane < K) {
      const int64_t j = t * K + lane;
      const int s = __ldg(inv + j);
      const int e = __ldg(topk_idx + j);
      if (s >= 0 && s < rows && e >= 0 && e < E) {
        myR = __ldg(poffsets + e) + (s - __ldg(offsets + e));
        if (w_perm) w_perm[s] = topk_w ? __ldg(topk_w + j) : 1.0f;
      }
    }
    const uint4* src = x + t * vec_per_row;
    for (int v0 = lane; v0 < vec_per_row; v0 += 32 * kV) {
      uint4 d[kV];
#pragma unroll
      for (int u = 0; u < kV; ++u)
        if (v0 + 32 * u < vec_per_row) d[u] = __ldg(src + v0 + 32 * u);
      for (int k = 0; k < K; ++k) {
        const int64_t R = __shfl_sync(0xffffffffu, myR, k);
        if (R < 0) continue;
        const int sw = static_cast<int>(R & 7);
#pragma unroll
        for (int u = 0; u < kV; ++u) {
          const int v = v0 + 32 * u;
          if (v < vec_per_row)
            st_global_hint(Xp + ((v >> 3) * plane_rows + R) * 8 + ((v & 7) ^ sw), d[u], pass);
        }
      }
    }
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
  pdl_wait();
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
  struct Raw {
    uint4 u;
  };
  static __device__ __forceinline__ Raw load_raw(const void* p, int64_t i) {
    return Raw{__ldg(reinterpret_cast<const uint4*>(p) + i)};
  }
  static __device__ __forceinline__ void unpack(const Raw& r, float (&v)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r.u);
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
  struct Raw {
    float4 a, b;
  };
  static __device__ __forceinline__ Raw load_raw(const void* p, int64_t i) {
    return Raw{__ldg(reinterpret_cast<const float4*>(p) + 2 * i),
               __ldg(reinterpret_cast<const float4*>(p) + 2 * i + 1)};
  }
  static __device__ __forceinline__ void unpack(const Raw& r, float (&v)[8]) {
    v[0] = r.a.x; v[1] = r.a.y; v[2] = r.a.z; v[3] = r.a.w;
    v[4] = r.b.x; v[5] = r.b.y; v[6] = r.b.z; v[7] = r.b.w;
  }
  static __device__ __forceinline__ void store(void* p, int64_t i, const float (&v)[8]) {
    reinterpret_cast<float4*>(p)[2 * i] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[2 * i + 1] = make_float4(v[4], v[5], v[6], v[7]);
  }
};

// One CTA per token row, or per (row, slice of 128 vectors) for small
// batches (gridDim.y slices); D must be a multiple of 8.  The rows of a
// batch of eight k are loaded before any is added, so their loads are in
// flight together; the sum still runs over k in order, then the addends.
template <bool BF16>
__global__ void __launch_bounds__(128) combine_kernel(const void* __restrict__ Y,
                                                      const int32_t* __restrict__ inv,
                                                      const float* __restrict__ w, int K,
                                                      int D, const void* __restrict__ adds,
                                                      int n_add, int64_t add_stride_rows,
                                                      void* __restrict__ y) {
  pdl_wait();
  using V = Vec8<BF16>;
  const int64_t t = blockIdx.x;
  const int nvec = D / 8;
  __shared__ int slots[64];
  __shared__ float wts[64];
  if (threadIdx.x < K) {
    // a slot outside the T K rows of Y (a rejected pair) is read as row 0
    // with weight 0, so that every load stays inside Y
    const int64_t rows = static_cast<int64_t>(gridDim.x) * K;
    const int sl = __ldg(inv + t * K + threadIdx.x);
    const bool in = sl >= 0 && sl < rows;
    slots[threadIdx.x] = in ? sl : 0;
    wts[threadIdx.x] = !in ? 0.0f : w ? __ldg(w + t * K + threadIdx.x) : 1.0f;
  }
  __syncthreads();
  constexpr int kB = 8;
  for (int v = blockIdx.y * blockDim.x + threadIdx.x; v < nvec; v += gridDim.y * blockDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float tmp[8];
    for (int k0 = 0; k0 < K; k0 += kB) {
      typename V::Raw raw[kB];
#pragma unroll
      for (int i = 0; i < kB; ++i)
        if (k0 + i < K) raw[i] = V::load_raw(Y, static_cast<int64_t>(slots[k0 + i]) * nvec + v);
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        if (k0 + i < K) {
          V::unpack(raw[i], tmp);
          const float wk = wts[k0 + i];
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] = fmaf(wk, tmp[q], acc[q]);
        }
      }
    }
    constexpr int kA = 2;  // addends per batch (the shared experts: one or two)
    for (int a0 = 0; a0 < n_add; a0 += kA) {
      typename V::Raw raw[kA];
#pragma unroll
      for (int i = 0; i < kA; ++i)
        if (a0 + i < n_add) raw[i] = V::load_raw(adds, ((a0 + i) * add_stride_rows + t) * nvec + v);
#pragma unroll
      for (int i = 0; i < kA; ++i) {
        if (a0 + i < n_add) {
          V::unpack(raw[i], tmp);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] += tmp[q];
        }
      }
    }
    V::store(y, t * nvec + v, acc);
  }
}

}  // namespace

int permute_chunk(int64_t n) {
  int c = 32;
  while (c < 1024 && static_cast<int64_t>(c) * 256 < n) c <<= 1;
  return c;
}

int64_t permute_chunks(int64_t n) {
  const int c = permute_chunk(n);
  return (n + c - 1) / c;
}

cudaError_t launch_permute(const int32_t* topk_idx, int64_t T, int K, int E, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* ccount,
                           int* status, cudaStream_t stream) {
  const int64_t n = T * K;
  const int chunk = permute_chunk(n);
  const int64_t nchunks = permute_chunks(n);
  if (nchunks < 1) return cudaSuccess;
  cudaError_t err = launch_pdl(chunk_count_kernel, dim3(static_cast<unsigned>(nchunks)),
                               dim3(kChunkThreads), sizeof(int) * E, stream, topk_idx, n, chunk, E,
                               ccount, status);
  if (err != cudaSuccess) return err;
  err = launch_pdl(chunk_scan_kernel, dim3(static_cast<unsigned>((E + 31) / 32)), dim3(1024), 0,
                   stream, ccount, static_cast<int>(nchunks), E, counts);
  if (err != cudaSuccess) return err;
  const unsigned blocks = static_cast<unsigned>((nchunks + kScatterWarps - 1) / kScatterWarps);
  return launch_pdl(chunk_scatter_kernel, dim3(blocks), dim3(32 * kScatterWarps),
                    sizeof(int) * (E * kScatterWarps + E + 1), stream, topk_idx, n, chunk, E,
                    static_cast<const int32_t*>(ccount), static_cast<const int32_t*>(counts),
                    offsets, static_cast<int>(nchunks), perm, inv);
}

int64_t max_tiles(int64_t rows, int E, int nt) { return rows / nt + E; }

cudaError_t launch_build_tiles(const int32_t* offsets, int E, int nt, RowTile* tiles, int* ntiles,
                               int32_t* poffsets, cudaStream_t stream) {
  return launch_pdl(build_tiles_kernel, dim3(1), dim3(1024), 0, stream, offsets, E, nt, tiles,
                    ntiles, poffsets);
}

cudaError_t launch_gather_packed(const void* x, int K, int width, const int32_t* perm,
                                 const int32_t* offsets, const int32_t* poffsets, int E,
                                 const float* topk_w, void* Xp, int64_t plane_rows,
                                 float* w_perm, cudaStream_t stream) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return launch_pdl(gather_packed_kernel, dim3(sms * 8), dim3(256), 0, stream,
                    static_cast<const uint4*>(x), K, width / 8, perm, offsets, poffsets, E, topk_w,
                    static_cast<uint4*>(Xp), plane_rows, w_perm);
}

cudaError_t launch_gather_tokens_packed(const void* x, int64_t T, int K, int width,
                                        const int32_t* topk_idx, const int32_t* inv,
                                        const int32_t* offsets, const int32_t* poffsets, int E,
                                        const float* topk_w, void* Xp, int64_t plane_rows,
                                        float* w_perm, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const int64_t blocks = (T + 7) / 8;  // a warp per token
  return launch_pdl(gather_tokens_packed_kernel,
                    dim3(static_cast<unsigned>(blocks < 65535 * 16 ? blocks : 65535 * 16)),
                    dim3(256), 0, stream, static_cast<const uint4*>(x), T, K, width / 8, topk_idx,
                    inv, offsets, poffsets, E, topk_w, static_cast<uint4*>(Xp), plane_rows,
                    w_perm);
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
  // small batches: several CTAs per row, one 8-element vector per thread
  const unsigned slices = T < 1024 ? static_cast<unsigned>((D / 8 + 127) / 128) : 1u;
  const dim3 grid(static_cast<unsigned>(T), slices);
  if (bf16)
    return launch_pdl(combine_kernel<true>, grid, dim3(128), 0, stream, Y, inv, w, K, D, adds,
                      n_add, add_stride_rows, y);
  return launch_pdl(combine_kernel<false>, grid, dim3(128), 0, stream, Y, inv, w, K, D, adds,
                    n_add, add_stride_rows, y);
}

}  // namespace fgs
