// Router of the fine-grained MoE layer.
//
// "Kimi K2 · Router · OpenModelAtlas", "All 4 steps":
//   z = x_ffn W_r, s = sigmoid(z), E_sel = [i in top_K(s + b)],
//   G_i = 2.827 s_i E_sel_i / sum_j s_j E_sel_j;
// the page's MoEGate listing adds the fp32 cast of x and W_r, the group
// limiting of noaux_tc (keep the topk_group groups whose two best biased
// scores sum highest, fill the other experts' scores with 0.0), the
// renormalisation with + 1e-20 (only when K > 1 and norm_topk_prob) and the
// final routed_scaling_factor.
//
// Two ways to the logits:
//  * bf16 x with a workspace: a tensor-core GEMM (gemm_tc.cu) against a
//    three-way bf16 split of W_r, written as K-split partial sums that
//    router_logits_kernel adds in a fixed order before it selects;
//  * otherwise router_fused_kernel: one thread-block cluster per 64 tokens,
//    one CTA per 128 experts (K2: 3 CTAs, K3: 7).  Each CTA runs the fp32 FFMA
//    GEMM for its 64 x 128 logit tile, keeps the tile in shared memory, and
//    after a cluster barrier every CTA selects for a share of the 64 tokens by
//    reading the whole 64 x E logit row set through distributed shared memory.
// Selection is one warp per token: sigmoid + bias per lane, group top-2 sums
// by warp shuffles, then the K (+1) best in one pass (a warp sort of the
// lanes' bests, then of the candidates they bound) or K rounds of a warp
// arg-max.  router_logits_kernel holds each lane's experts as one run of
// consecutive indices (a K2 group of 48 is 4 lanes of 12); the other kernels
// stride them across the warp.
#include <cooperative_groups.h>
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace fgs {

namespace {

constexpr int kTM = 64;   // tokens per cluster
constexpr int kEC = 128;  // experts per CTA
constexpr int kBK = 32;   // reduction chunk
constexpr int kThreads = 256;

// s rounded once from the fp64 sigmoid of the fp32 logit: the correctly
// rounded fp32 sigmoid except when the fp64 value lies within one fp64 ulp
// of an fp32 rounding boundary.
__device__ __noinline__ double sigmoid_f64(float z) {
  return 1.0 / (1.0 + exp(-static_cast<double>(z)));
}

// Order used for every discrete choice: larger value first, then the
// smaller index.
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// The selection decides on c = fp32(s + b) with s the correctly rounded fp32
// sigmoid (computed in fp64 and rounded once).  Each value is first taken
// from an fp32 sigmoid, rcp_rn(1 + expf(-z)) with expf within 2 ulp, whose
// distance to the exact c is below kFastErr.  A discrete decision taken on
// these values is the exact decision whenever the two values it separates
// are more than twice that apart; only when some decision is closer (a
// near-tie) are the values around it recomputed exactly and the decision
// taken again.  Either way the result equals the one taken on exact values.
// kFastErr = 5e-7 bounds |fast c - exact c| for |z| <= kFastRange.
constexpr float kMargin = 1.0f / 262144.0f;  // 3.8e-6 > 2 kFastErr
constexpr float kGroupMargin = 1.0f / 131072.0f;  // group sums: 7.6e-6 > 2 (2 kFastErr + rounding)
constexpr float kFastRange = 80.0f;           // beyond |z| > 80 the value is always exact

// Out of line: the exact path is rare, and inlining its fp64 exponential at
// every call site would cost registers on the common path.
__device__ __noinline__ float exact_c(float z, float b) {
  return __fadd_rn(static_cast<float>(sigmoid_f64(z)), b);
}

// Top-2 values over the warp of the lane-local pair (m1 >= m2).
__device__ __forceinline__ void warp_top2(float& m1, float& m2) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float o1 = __shfl_xor_sync(0xffffffffu, m1, off);
    const float o2 = __shfl_xor_sync(0xffffffffu, m2, off);
    if (m1 >= o1) {
      m2 = fmaxf(m2, o1);
    } else {
      m2 = fmaxf(m1, o2);
      m1 = o1;
    }
  }
}

// The expert a lane holds in its slot j: strided (lane + 32 j: a warp's
// loads of one slot are 128 consecutive bytes) or blocked (PM consecutive
// experts per lane: a group of E / G experts spans few lanes).
template <int PM, bool kBlocked>
__device__ __forceinline__ int expert_of(int lane, int j) {
  return kBlocked ? lane * PM + j : lane + 32 * j;
}

template <int PM, bool kBlocked>
__device__ __forceinline__ void group_top2(const float (&c)[PM], int lane, int E, int gsize, int g,
                                          float& m1, float& m2) {
  m1 = -CUDART_INF_F;
  m2 = -CUDART_INF_F;
  const int lo = g * gsize, hi = lo + gsize;
#pragma unroll
  for (int j = 0; j < PM; ++j) {
    const int e = expert_of<PM, kBlocked>(lane, j);
    if (e >= lo && e < hi && e < E) {
      const float v = c[j];
      if (v > m1) {
        m2 = m1;
        m1 = v;
      } else if (v > m2) {
        m2 = v;
      }
    }
  }
  warp_top2(m1, m2);
}

// Warp arg-max of (value, index) in the selection order.
__device__ __forceinline__ void warp_best(float& bv, int& bi) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
    if (before(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
}

// A 64-bit key whose unsigned order is the selection order: the value's
// bits mapped to an order-preserving unsigned integer (with -0 read as +0,
// which compares equal to it), then the complement of the index, so that
// equal values put the smaller index first.
__device__ __forceinline__ uint64_t order_key(float v, int idx) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(~idx);
}

__device__ __forceinline__ float key_value(uint64_t k) {
  const uint32_t o = static_cast<uint32_t>(k >> 32);
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

__device__ __forceinline__ int key_index(uint64_t k) {
  return static_cast<int>(~static_cast<uint32_t>(k));
}

// Bitonic sort of one key per lane into descending order across the warp
// (lane 0 the largest), moving `z` with its key when kCarry.
template <bool kCarry>
__device__ __forceinline__ void warp_sort_desc(uint64_t& key, float& z, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint32_t ohi = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(key >> 32), stride);
      const uint32_t olo = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(key), stride);
      const float oz = kCarry ? __shfl_xor_sync(0xffffffffu, z, stride) : 0.0f;
      const uint64_t other = (static_cast<uint64_t>(ohi) << 32) | olo;
      // a descending block keeps the larger key in its lower lane
      const bool desc = (lane & size) == 0;
      const bool lower = (lane & stride) == 0;
      const bool take = (lower == desc) ? other > key : other < key;
      if (take) {
        key = other;
        if (kCarry) z = oz;
      }
    }
  }
}

// Selection for one token by one warp.  Lane `lane` holds the logits of
// experts expert_of(lane, j), j < PM.  Writes topk_idx[0..K) and
// topk_w[0..K).  Every decision uses the (value, index) order alone, so the
// result does not depend on the layout.
template <int PM, bool kBlocked = false>
__device__ __forceinline__ void select_token(const float (&z)[PM], int lane, int E,
                                             const float* __restrict__ bias, int K, int G,
                                             int Gk, float scale, int norm,
                                             int32_t* __restrict__ out_idx,
                                             float* __restrict__ out_w,
                                             uint64_t* cand_key = nullptr,
                                             float* cand_z = nullptr) {
  const unsigned full = 0xffffffffu;
  float c[PM];
  unsigned exact = 0u;  // bit j: c[j] holds the exact value
#pragma unroll
  for (int j = 0; j < PM; ++j) {
    const int e = expert_of<PM, kBlocked>(lane, j);
    if (e < E) {
      const float b = __ldg(bias + e);
      if (fabsf(z[j]) <= kFastRange) {
        c[j] = __fadd_rn(__frcp_rn(1.0f + expf(-z[j])), b);
      } else {
        c[j] = exact_c(z[j], b);
        exact |= 1u << j;
      }
    } else {
      c[j] = -CUDART_INF_F;  // no such expert
      exact |= 1u << j;
    }
  }
  // recompute exactly every value >= threshold (optionally of one group)
  auto refine_above = [&](float threshold, int lo, int hi) {
#pragma unroll
    for (int j = 0; j < PM; ++j) {
      const int e = expert_of<PM, kBlocked>(lane, j);
      if (!((exact >> j) & 1u) && c[j] >= threshold && e >= lo && e < hi) {
        c[j] = exact_c(z[j], __ldg(bias + e));
        exact |= 1u << j;
      }
    }
  };

  if (G > 1) {
    // group score = sum of the two largest biased scores in the group
    const int gsize = E / G;
    // blocked layout with whole groups of a power-of-two count of lanes
    // each (K2: 48 experts = 4 lanes of 12): every lane's experts lie in one
    // group, so the top-2 is lane-local and then merged over the group's lanes
    const int lpg = kBlocked ? gsize / PM : 0;
    const bool lane_groups = kBlocked && gsize % PM == 0 && lpg > 0 && lpg <= 32 &&
                             (lpg & (lpg - 1)) == 0 && G * gsize == E;
    auto group_scores = [&]() {
      float mine = -CUDART_INF_F;
      if (lane_groups) {
        float m1 = -CUDART_INF_F, m2 = -CUDART_INF_F;
#pragma unroll
        for (int j = 0; j < PM; ++j) {
          if (expert_of<PM, kBlocked>(lane, j) < E) {
            const float v = c[j];
            if (v > m1) {
              m2 = m1;
              m1 = v;
            } else if (v > m2) {
              m2 = v;
            }
          }
        }
        for (int off = 1; off < lpg; off <<= 1) {
          const float o1 = __shfl_xor_sync(full, m1, off);
          const float o2 = __shfl_xor_sync(full, m2, off);
          if (m1 >= o1) {
            m2 = fmaxf(m2, o1);
          } else {
            m2 = fmaxf(m1, o2);
            m1 = o1;
          }
        }
        // group g's score sits in its lanes g lpg .. (g + 1) lpg - 1
        const float sum = __fadd_rn(m1, m2);
        const float got = __shfl_sync(full, sum, lane < G ? lane * lpg : 0);
        if (lane < G) mine = got;
        return mine;
      }
      for (int g = 0; g < G; ++g) {
        float m1, m2;
        group_top2<PM, kBlocked>(c, lane, E, gsize, g, m1, m2);
        if (lane == g) mine = __fadd_rn(m1, m2);
      }
      return mine;
    };
    // keep the Gk best groups (ties: smaller group index); returns the
    // margin between the last kept and the best dropped group
    auto choose = [&](float score, unsigned& kept_mask) {
      bool kept = false;
      float last = 0.0f, next = -CUDART_INF_F;
      for (int r = 0; r <= Gk && r < G; ++r) {
        float bv = (lane < G && !kept) ? score : -CUDART_INF_F;
        int bi = (lane < G && !kept) ? lane : 0x7fffffff;
        warp_best(bv, bi);
        if (r < Gk) {
          if (lane == bi) kept = true;
          last = bv;
        } else {
          next = bv;
        }
      }
      kept_mask = __ballot_sync(full, kept);
      return last - next;
    };
    unsigned kept_mask;
    float gscore = group_scores();
    if (choose(gscore, kept_mask) <= kGroupMargin) {
      // near-tie between groups: make every possible top-2 member exact
      for (int g = 0; g < G; ++g) {
        float m1, m2;
        group_top2<PM, kBlocked>(c, lane, E, gsize, g, m1, m2);
        refine_above(m2 - kMargin, g * gsize, (g + 1) * gsize);
      }
      gscore = group_scores();
      choose(gscore, kept_mask);
    }
#pragma unroll
    for (int j = 0; j < PM; ++j) {
      const int e = expert_of<PM, kBlocked>(lane, j);
      if (e < E && !((kept_mask >> (e / gsize)) & 1u)) {
        c[j] = 0.0f;  // literal 0.0 fill
        exact |= 1u << j;
      }
    }
  }

  // K (+1 for the boundary) rounds of warp arg-max; lane k keeps the k-th
  // winner's index, logit and value
  int sel_idx = 0;
  float sel_z = 0.0f, sel_v = -CUDART_INF_F;
  auto rounds = [&]() {
    unsigned taken = 0u;
    const int R = K < E ? K + 1 : K;
    for (int k = 0; k < R; ++k) {
      float bv = -CUDART_INF_F;
      int bi = 0x7fffffff;
      float bz = 0.0f;
#pragma unroll
      for (int j = 0; j < PM; ++j) {
        const int e = expert_of<PM, kBlocked>(lane, j);
        if (e < E && !((taken >> j) & 1u) && before(c[j], e, bv, bi)) {
          bv = c[j];
          bi = e;
          bz = z[j];
        }
      }
      const int mine = bi;
      warp_best(bv, bi);
      const int owner = kBlocked ? bi / PM : bi & 31;
      if (lane == owner && mine == bi) taken |= 1u << (kBlocked ? bi - owner * PM : bi >> 5);
      bz = __shfl_sync(full, bz, owner);
      if (lane == k) {
        sel_idx = bi;
        sel_z = bz;
        sel_v = bv;
      }
    }
  };
  // The same K (+1) winners in one pass when the warp has 32 words of
  // shared scratch: the R-th best of the lanes' own bests is at or after
  // the R-th best overall in the selection order, so the R best are among
  // the experts at or before it; when those candidates fit in the 32 lanes,
  // one sort across the warp orders them.  Otherwise the rounds run.
  auto one_pass = [&]() -> bool {
    const int R = K < E ? K + 1 : K;
    if (cand_key == nullptr || R > 32) return false;
    float lv = -CUDART_INF_F;
    int li = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < PM; ++j) {
      const int e = expert_of<PM, kBlocked>(lane, j);
      if (e < E && before(c[j], e, lv, li)) {
        lv = c[j];
        li = e;
      }
    }
    uint64_t key = order_key(lv, li);
    float unused = 0.0f;
    warp_sort_desc<false>(key, unused, lane);
    const uint64_t floor_key =
        (static_cast<uint64_t>(__shfl_sync(full, static_cast<uint32_t>(key >> 32), R - 1)) << 32) |
        __shfl_sync(full, static_cast<uint32_t>(key), R - 1);
    unsigned mine = 0u;
#pragma unroll
    for (int j = 0; j < PM; ++j) {
      const int e = expert_of<PM, kBlocked>(lane, j);
      if (e < E && order_key(c[j], e) >= floor_key) mine |= 1u << j;
    }
    const int n = __popc(mine);
    int incl = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(full, incl, off);
      if (lane >= off) incl += o;
    }
    const int total = __shfl_sync(full, incl, 31);
    if (total > 32) return false;
    int pos = incl - n;
#pragma unroll
    for (int j = 0; j < PM; ++j) {
      if ((mine >> j) & 1u) {
        cand_key[pos] = order_key(c[j], expert_of<PM, kBlocked>(lane, j));
        cand_z[pos] = z[j];
        ++pos;
      }
    }
    __syncwarp();
    uint64_t ck = lane < total ? cand_key[lane] : 0ull;
    float cz = lane < total ? cand_z[lane] : 0.0f;
    __syncwarp();
    warp_sort_desc<true>(ck, cz, lane);
    if (lane < R) {
      sel_idx = key_index(ck);
      sel_v = key_value(ck);
      sel_z = cz;
    }
    return true;
  };
  if (!one_pass()) rounds();
  // a near-tie among the K+1 best (order or boundary) -> exact values there
  const float next_v = __shfl_down_sync(full, sel_v, 1);
  const bool near = lane + 1 < (K < E ? K + 1 : K) && sel_v - next_v <= kMargin;
  if (__any_sync(full, near)) {
    const float floor_v = __shfl_sync(full, sel_v, K < E ? K : K - 1);
    refine_above(floor_v - kMargin, 0, E);
    rounds();
  }
  // weights from the unbiased scores, one lane per selected expert, in
  // fp32: the fast sigmoid's error (below 1e-6 relative) is far inside the
  // weights' tolerance, and fp64 throughput is scarce on this part
  const float sk = lane < K ? __frcp_rn(1.0f + expf(-sel_z)) : 0.0f;
  float sum = sk;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(full, sum, off);
  if (lane < K) {
    const float w = (K > 1 && norm) ? __fdiv_rn(sk, sum + 1e-20f) : sk;
    out_idx[lane] = sel_idx;
    out_w[lane] = w * scale;
  }
}

template <typename XT>
struct XLoad;

template <>
struct XLoad<__nv_bfloat16> {
  // 8 consecutive bf16 as fp32
  static __device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};

template <>
struct XLoad<float> {
  static __device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

struct RouterSmem {
  union {
    struct {
      float xs[2][kBK][kTM];  // x chunk, transposed: [k][token]
      float ws[2][kBK][kEC];  // W_r chunk, transposed: [k][expert]
    } pipe;
    float zs[kTM][kEC];  // the CTA's logit tile
  };
};

template <typename XT, int PM>
__global__ void __launch_bounds__(kThreads) router_fused_kernel(
    const XT* __restrict__ x, const float* __restrict__ W_r, const float* __restrict__ bias,
    int T, int d, int E, int K, int G, int Gk, float scale, int norm,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  __shared__ __align__(16) RouterSmem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int CS = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x;
  const int tok0 = blockIdx.y * kTM;
  const int e0 = rank * kEC;

  // loader roles
  const int lx_tok = tid % kTM, lx_k = (tid / kTM) * 8;     // 8 x values
  const int lw_e = tid % kEC, lw_k = (tid / kEC) * 16;      // 16 W values
  const bool x_ok = tok0 + lx_tok < T;
  const bool w_ok = e0 + lw_e < E;
  const XT* xrow = x + static_cast<int64_t>(x_ok ? tok0 + lx_tok : 0) * d + lx_k;
  const float* wrow = W_r + static_cast<int64_t>(w_ok ? e0 + lw_e : 0) * d + lw_k;

  // compute roles: 4 tokens x (4 + 4) experts per thread
  const int tx = tid % 16, ty = tid / 16;

  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

  float xv[8];
  float4 wv[4];
  auto load_chunk = [&](int k0) {
    if (x_ok) {
      XLoad<XT>::load8(xrow + k0, xv);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) xv[i] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      wv[i] = w_ok ? __ldg(reinterpret_cast<const float4*>(wrow + k0) + i)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  auto store_chunk = [&](int buf) {
#pragma unroll
    for (int i = 0; i < 8; ++i) sm.pipe.xs[buf][lx_k + i][lx_tok] = xv[i];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      sm.pipe.ws[buf][lw_k + 4 * i + 0][lw_e] = wv[i].x;
      sm.pipe.ws[buf][lw_k + 4 * i + 1][lw_e] = wv[i].y;
      sm.pipe.ws[buf][lw_k + 4 * i + 2][lw_e] = wv[i].z;
      sm.pipe.ws[buf][lw_k + 4 * i + 3][lw_e] = wv[i].w;
    }
  };

  const int nchunks = d / kBK;
  load_chunk(0);
  store_chunk(0);
  __syncthreads();
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    if (c + 1 < nchunks) load_chunk((c + 1) * kBK);
#pragma unroll 8
    for (int k = 0; k < kBK; ++k) {
      const float4 a = *reinterpret_cast<const float4*>(&sm.pipe.xs[buf][k][ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&sm.pipe.ws[buf][k][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&sm.pipe.ws[buf][k][64 + tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (c + 1 < nchunks) store_chunk(buf ^ 1);
    __syncthreads();
  }

  // logit tile to shared memory (the pipeline buffers are dead now)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sm.zs[ty * 4 + i][tx * 4 + j] = acc[i][j];
      sm.zs[ty * 4 + i][64 + tx * 4 + j] = acc[i][4 + j];
    }
  }
  cluster.sync();

  // selection: this CTA takes tokens tt = rank, rank + CS, ...; one warp each
  const int warp = tid / 32, lane = tid % 32;
  for (int tt = rank + CS * warp; tt < kTM; tt += CS * (kThreads / 32)) {
    const int t = tok0 + tt;
    if (t >= T) break;
    float z[PM];
#pragma unroll
    for (int j = 0; j < PM; ++j) {
      const int e = lane + 32 * j;
      if (e < E) {
        const float* peer = cluster.map_shared_rank(&sm.zs[0][0], e / kEC);
        z[j] = peer[tt * kEC + (e % kEC)];
      } else {
        z[j] = 0.0f;
      }
    }
    select_token<PM>(z, lane, E, bias, K, G, Gk, scale, norm,
                     topk_idx + static_cast<int64_t>(t) * K, topk_w + static_cast<int64_t>(t) * K);
  }
  cluster.sync();  // peers may still read this CTA's tile
}

// Logits given as `parts` partial arrays (a split reduction) are summed in
// ascending part order, so the result does not depend on scheduling.
constexpr int kSelWarps = 8;  // tokens (warps) per block of router_logits_kernel

// A lane's PM logits of one part in the blocked layout (experts lane PM ..
// lane PM + PM - 1): 16-byte loads when the lane's run is whole and aligned.
template <int PM>
__device__ __forceinline__ void load_blocked(const float* __restrict__ row, int lane, int E,
                                             float (&v)[PM]) {
  const int e0 = lane * PM;
  if (PM % 4 == 0 && E % 4 == 0 && e0 + PM <= E) {
    const float4* p4 = reinterpret_cast<const float4*>(row + e0);
#pragma unroll
    for (int i = 0; i < PM / 4; ++i) {
      const float4 f = __ldg(p4 + i);
      v[4 * i] = f.x;
      v[4 * i + 1] = f.y;
      v[4 * i + 2] = f.z;
      v[4 * i + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < PM; ++j) v[j] = e0 + j < E ? __ldg(row + e0 + j) : 0.0f;
  }
}

// One warp per token, in the blocked layout (each lane PM consecutive
// experts: whole-lane group scores, 16-byte loads).
template <int PM>
__global__ void __launch_bounds__(kSelWarps * 32, PM <= 12 ? 4 : 2) router_logits_kernel(
    const float* __restrict__ logits, int parts, int64_t part_stride,
    const float* __restrict__ bias, int T, int E, int K, int G, int Gk, float scale, int norm,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  pdl_wait();
  const int lane = threadIdx.x % 32;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= T) return;
  // z = the parts summed in order 0, 1, ..., parts - 1 for every expert;
  // the loads of a batch of parts of all the lane's experts are in flight
  // at once (small batches split the GEMM's K into dozens of parts)
  float z[PM];
  const float* row = logits + t * E;
  load_blocked<PM>(row, lane, E, z);
  // (two parts at a time for the widest rows, whose registers would
  // otherwise cap the kernel at one block per SM)
  constexpr int kBatch = PM > 16 ? 2 : 4;
  int q = 1;
  for (; q + kBatch <= parts; q += kBatch) {
    float b[kBatch][PM];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) load_blocked<PM>(row + (q + i) * part_stride, lane, E, b[i]);
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
#pragma unroll
      for (int j = 0; j < PM; ++j) z[j] += b[i][j];
  }
  for (; q < parts; ++q) {
    float b[PM];
    load_blocked<PM>(row + q * part_stride, lane, E, b);
#pragma unroll
    for (int j = 0; j < PM; ++j) z[j] += b[j];
  }
  __shared__ uint64_t cand_key[kSelWarps][32];
  __shared__ float cand_z[kSelWarps][32];
  const int w = threadIdx.x / 32;
  select_token<PM, true>(z, lane, E, bias, K, G, Gk, scale, norm, topk_idx + t * K,
                         topk_w + t * K, cand_key[w], cand_z[w]);
}

// Small batches whose GEMM split K into many parts: one block per token,
// so that the loads of all parts are in flight across eight warps instead of
// queued behind one.  Warp w sums its contiguous share of the parts in
// order, warp 0 adds the eight shares in warp order and selects.
constexpr int kSplitWarps = 8;

template <int PM>
__global__ void __launch_bounds__(kSplitWarps * 32) router_logits_split_kernel(
    const float* __restrict__ logits, int parts, int64_t part_stride,
    const float* __restrict__ bias, int T, int E, int K, int G, int Gk, float scale, int norm,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  pdl_wait();
  __shared__ float share[kSplitWarps][32 * PM];
  __shared__ uint64_t cand_key[32];
  __shared__ float cand_z[32];
  const int lane = threadIdx.x % 32;
  const int w = threadIdx.x / 32;
  const int64_t t = blockIdx.x;
  const int per = (parts + kSplitWarps - 1) / kSplitWarps;
  const int p0 = min(parts, w * per), p1 = min(parts, p0 + per);
  const float* pz = logits + t * E + lane;
  constexpr int kBatch = PM > 16 ? 2 : 4;
  float acc[PM];
  if (p0 < p1) {
#pragma unroll
    for (int j = 0; j < PM; ++j) acc[j] = lane + 32 * j < E ? __ldg(pz + p0 * part_stride + 32 * j) : 0.0f;
    int q = p0 + 1;
    for (; q + kBatch <= p1; q += kBatch) {
      float b[kBatch][PM];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
#pragma unroll
        for (int j = 0; j < PM; ++j)
          b[i][j] = lane + 32 * j < E ? __ldg(pz + (q + i) * part_stride + 32 * j) : 0.0f;
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
#pragma unroll
        for (int j = 0; j < PM; ++j) acc[j] += b[i][j];
    }
    for (; q < p1; ++q)
#pragma unroll
      for (int j = 0; j < PM; ++j)
        if (lane + 32 * j < E) acc[j] += __ldg(pz + q * part_stride + 32 * j);
#pragma unroll
    for (int j = 0; j < PM; ++j) share[w][lane + 32 * j] = acc[j];
  }
  __syncthreads();
  if (w != 0) return;
  const int nw = (parts + per - 1) / per;  // warps that had parts
  float z[PM];
#pragma unroll
  for (int j = 0; j < PM; ++j) z[j] = share[0][lane + 32 * j];
  for (int v = 1; v < nw; ++v)
#pragma unroll
    for (int j = 0; j < PM; ++j) z[j] += share[v][lane + 32 * j];
  select_token<PM>(z, lane, E, bias, K, G, Gk, scale, norm, topk_idx + t * K, topk_w + t * K,
                   cand_key, cand_z);
}

template <typename XT, int PM>
cudaError_t launch_fused(const RouterArgs& a, cudaStream_t stream) {
  const int CS = (a.E + kEC - 1) / kEC;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS, static_cast<unsigned>((a.T + kTM - 1) / kTM), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launch();
  return cudaLaunchKernelEx(&cfg, router_fused_kernel<XT, PM>, static_cast<const XT*>(a.x), a.W_r,
                            a.bias, static_cast<int>(a.T), a.d, a.E, a.K, a.G, a.Gk, a.scale,
                            a.norm, a.topk_idx, a.topk_w);
}

template <int PM>
cudaError_t launch_logits(const RouterArgs& a, cudaStream_t stream) {
  // a token per block when the token-per-warp grid would leave most SMs
  // idle while each warp walks many parts
  if (a.logit_parts >= kSplitWarps && a.T <= 1024)
    return launch_pdl(router_logits_split_kernel<PM>, dim3(static_cast<unsigned>(a.T)),
                      dim3(kSplitWarps * 32), 0, stream, a.logits, a.logit_parts,
                      a.logit_part_stride, a.bias, static_cast<int>(a.T), a.E, a.K, a.G, a.Gk,
                      a.scale, a.norm, a.topk_idx, a.topk_w);
  const int warps = kSelWarps;
  const unsigned blocks = static_cast<unsigned>((a.T + warps - 1) / warps);
  return launch_pdl(router_logits_kernel<PM>, dim3(blocks), dim3(warps * 32), 0, stream, a.logits,
                    a.logit_parts, a.logit_part_stride, a.bias, static_cast<int>(a.T), a.E, a.K,
                    a.G, a.Gk, a.scale, a.norm, a.topk_idx, a.topk_w);
}

// G [T, E]: each token's selected weights at their experts, 0 elsewhere.
// One CTA per row (grid-stride); every entry is written once, by the thread
// that owns it, after looking the expert up among the row's K indices.
__global__ void __launch_bounds__(128) dense_gates_kernel(const int32_t* __restrict__ idx,
                                                          const float* __restrict__ w, int64_t T,
                                                          int K, int E, float* __restrict__ G) {
  __shared__ int sidx[32];
  __shared__ float sw[32];
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    if (threadIdx.x < K) {
      sidx[threadIdx.x] = __ldg(idx + t * K + threadIdx.x);
      sw[threadIdx.x] = __ldg(w + t * K + threadIdx.x);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      float v = 0.0f;
      for (int k = 0; k < K; ++k)
        if (sidx[k] == e) v = sw[k];
      G[t * E + e] = v;
    }
    __syncthreads();
  }
}

// bias[e] += gamma * sign(T K / E - counts[e]): the comparison with the mean
// load in integers, then one fp32 addition.
__global__ void bias_update_kernel(const int32_t* __restrict__ counts, int64_t pairs, int E,
                                   float gamma, float* __restrict__ bias) {
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x) {
    const int64_t diff = pairs - static_cast<int64_t>(E) * __ldg(counts + e);
    const float step = diff > 0 ? gamma : (diff < 0 ? -gamma : 0.0f);
    bias[e] = bias[e] + step;
  }
}

// ------------------------------------------------------ Quantile Balancing
// ("Kimi K3's router picks 16 of 896 experts", "The router trains inside the
// main run": per expert, the score threshold at which it receives its target
// number of tokens, from a quantile of the router scores, updates the
// selection bias.)  theta_e is the r-th largest fp32 score s = sigmoid(z) of
// expert e over the batch, r = ceil(T K / E).  The sigmoid rounded to fp32
// is non-decreasing in z, so theta_e is the score of the r-th largest logit:
// the kernel selects that logit exactly (radix select on an order-preserving
// integer key of the fp32 bits, four 8-bit digits from the top) and takes
// one fp64 sigmoid of it.

// Unsigned key whose order is the order of the fp32 values (-0 below +0).
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// One CTA per expert: theta[e] from column e of z [T, E].
__global__ void __launch_bounds__(256) quantile_threshold_kernel(const float* __restrict__ z,
                                                                 int64_t T, int E, int64_t r,
                                                                 float* __restrict__ theta) {
  pdl_wait();
  __shared__ unsigned hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int64_t s_rank;
  const int e = blockIdx.x;
  uint32_t prefix = 0, mask = 0;
  int64_t rank = r;  // rank still to find among the keys matching prefix, from the top
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int64_t t = threadIdx.x; t < T; t += blockDim.x) {
      const uint32_t k = order_key(__ldg(z + t * E + e));
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      // the digit whose bin holds the rank-th largest key, counting from 255
      int64_t above = 0;
      int d = 255;
      for (; d > 0; --d) {
        if (above + hist[d] >= rank) break;
        above += hist[d];
      }
      s_prefix = prefix | (static_cast<uint32_t>(d) << shift);
      s_rank = rank - above;
    }
    __syncthreads();
    prefix = s_prefix;
    rank = s_rank;
    mask |= 255u << shift;
    __syncthreads();
  }
  if (threadIdx.x == 0) theta[e] = static_cast<float>(sigmoid_f64(key_value(prefix)));
}

// tau = (sum_e theta_e) / E, summed in fp64 in expert order by one thread;
// bias[e] = fp32(b + rate (tau - theta_e - b)) with every operation an fp64
// operation rounded on its own (no fused multiply-add), in the order written.
__global__ void __launch_bounds__(256) quantile_bias_kernel(const float* __restrict__ theta, int E,
                                                            float rate, float* __restrict__ bias) {
  pdl_wait();
  __shared__ double s_tau;
  if (threadIdx.x == 0) {
    double total = 0.0;
    for (int e = 0; e < E; ++e) total = __dadd_rn(total, static_cast<double>(theta[e]));
    s_tau = __ddiv_rn(total, static_cast<double>(E));
  }
  __syncthreads();
  const double tau = s_tau;
  const double rd = static_cast<double>(rate);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const double b = static_cast<double>(bias[e]);
    const double target = __dsub_rn(tau, static_cast<double>(theta[e]));
    const double step = __dmul_rn(rd, __dsub_rn(target, b));
    bias[e] = __double2float_rn(__dadd_rn(b, step));
  }
}

}  // namespace

cudaError_t launch_quantile_bias(const float* logits, int64_t T, int K, int E, float rate,
                                 float* theta, float* bias, cudaStream_t stream) {
  const int64_t r = (T * K + E - 1) / E;
  cudaError_t err = launch_pdl(quantile_threshold_kernel, dim3(static_cast<unsigned>(E)),
                               dim3(256), 0, stream, logits, T, E, r, theta);
  if (err != cudaSuccess) return err;
  return launch_pdl(quantile_bias_kernel, dim3(1), dim3(256), 0, stream,
                    static_cast<const float*>(theta), E, rate, bias);
}

cudaError_t launch_dense_gates(const int32_t* topk_idx, const float* topk_w, int64_t T, int K,
                               int E, float* G, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>(T < 8192 ? T : 8192);
  note_launch();
  dense_gates_kernel<<<blocks, 128, 0, stream>>>(topk_idx, topk_w, T, K, E, G);
  return cudaGetLastError();
}

cudaError_t launch_bias_update(const int32_t* counts, int64_t T, int K, int E, float gamma,
                               float* bias, cudaStream_t stream) {
  note_launch();
  bias_update_kernel<<<(E + 255) / 256, 256, 0, stream>>>(counts, T * K, E, gamma, bias);
  return cudaGetLastError();
}

cudaError_t launch_router(const RouterArgs& a, cudaStream_t stream) {
  if (a.logits) {
    if (a.E <= 128) return launch_logits<4>(a, stream);
    if (a.E <= 384) return launch_logits<12>(a, stream);
    if (a.E <= 896) return launch_logits<28>(a, stream);  // K3: every lane holds experts
    return launch_logits<32>(a, stream);
  }
  if (a.x_bf16) {
    if (a.E <= 128) return launch_fused<__nv_bfloat16, 4>(a, stream);
    if (a.E <= 384) return launch_fused<__nv_bfloat16, 12>(a, stream);
    return launch_fused<__nv_bfloat16, 32>(a, stream);
  }
  if (a.E <= 128) return launch_fused<float, 4>(a, stream);
  if (a.E <= 384) return launch_fused<float, 12>(a, stream);
  return launch_fused<float, 32>(a, stream);
}

}  // namespace fgs
