// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA.  bf16 operands, fp32 accumulation.
//
// What they compute ("Kimi K2 MoE", section 2: SwiGLU experts; section 3:
// shared expert always on):
//   gate/up pass:  H[r, f] = SiLU(sum_k X[r,k] W_gate[e,f,k]) * sum_k X[r,k] W_up[e,f,k]
//   down pass:     Y[r, o] = w_r * sum_f H[r,f] W_down[e,o,f]
// for every row r of every routed expert e (rows come in tiles from the
// dispatch) and, as a second segment of the same launch, for every token of
// every shared expert.  The K3 latent projections use the down-pass form with
// one group and no scale.
//
// Swap-AB tiling.  The MMA's M side (128 rows) is a block of WEIGHT rows and
// its N side (16..256, a multiple of 16) is the block of token rows of one
// expert, so an expert with few tokens still streams its weights through
// full-height MMAs and each weight byte is read from HBM once per token tile.
//   A tile: 128 weight rows x 64 k, bf16, K-major, 128-byte swizzle (16 KB)
//   B tile: up to nt token rows x 64 k, same layout, loaded as 32-row boxes
//   D:      128 lanes x N fp32 columns of TMEM, two accumulators so the
//           epilogue of one tile overlaps the main loop of the next.
// For the gate/up pass the A tile interleaves the two halves of W_gate_up
// [E, 2F, d] in 16-row slices: rows 32q..32q+15 are gate features
// 64 ob + 16q + (0..15) and rows 32q+16..32q+31 the up features with the same
// indices.  TMEM lane quadrant q (the one warp q%4 may read) therefore holds
// both halves of 16 features, and the SwiGLU is one shuffle away.
//
// Warp roles (one CTA per SM, persistent over the tile list):
//   warp 0 lane 0: TMA producer; warp 1 lane 0: MMA issuer;
//   warps 2..5: epilogue (TMEM -> registers -> bf16 global stores).
// Every wait is bounded (%globaltimer); on expiry the CTA records
// MOE_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fgs {

namespace {

constexpr int kBK = 64;                    // k per stage: one 128-byte swizzle row
constexpr uint32_t kABytes = 128 * 128;    // A stage: 128 rows x 128 B
constexpr int kBBoxRows = 32;
constexpr uint32_t kBBoxBytes = kBBoxRows * 128;
constexpr int kThreads = 192;
constexpr int kMaxStages = 8;
constexpr size_t kSmemBudget = 196608;     // pipeline bytes per CTA

struct Unit {
  int seg, group, b_row, out_row, n_rows, ob;
};

__device__ __forceinline__ int segment_tiles(const GemmSegment* s, int nt) {
  if (s->tiles) return *s->ntiles;
  return s->groups * ((s->rows + nt - 1) / nt);
}

__device__ __forceinline__ Unit decode_unit(const GemmParams& p, int u, int units0, int nt) {
  Unit x;
  x.seg = u >= units0 ? 1 : 0;
  const int local = u - (x.seg ? units0 : 0);
  const GemmSegment* s = x.seg ? &p.seg[1] : &p.seg[0];
  const int tile = local / s->o_blocks;
  x.ob = local - tile * s->o_blocks;
  if (s->tiles) {
    const int4 t = s->tiles[tile];
    x.group = t.x;
    x.b_row = t.y;
    x.out_row = t.y;
    x.n_rows = t.z;
  } else {
    const int tpg = (s->rows + nt - 1) / nt;
    const int g = tile / tpg;
    const int t0 = (tile - g * tpg) * nt;
    x.group = g;
    x.n_rows = min(nt, s->rows - t0);
    x.b_row = static_cast<int>(g * s->b_group_stride + t0);
    x.out_row = static_cast<int>(g * s->out_group_stride + t0);
  }
  return x;
}

// Wait on a barrier for the whole warp: lane 0 polls (bounded), the verdict
// is broadcast so the warp stays converged for the .sync.aligned tcgen05 ops.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
  bool ok = false;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, abort_flag, status);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok;
}

// Drain wait: bounded by time only (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int* status) {
  int local_abort = 0;
  mbar_wait_bounded(bar, parity, &local_abort, status);
}

__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int stages = p.stages;
  const int nt = p.nt;
  const uint32_t b_stage_bytes = static_cast<uint32_t>(nt) * 128u;
  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem_a + stages * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_b + stages * b_stage_bytes);
  // bars: full[stages] | empty[stages] | tmem_full[2] | tmem_empty[2] | drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * stages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t a_base = smem_u32(smem_a);
  const uint32_t b_base = smem_u32(smem_b);
  const uint32_t bar_base = smem_u32(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (stages + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * stages + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * stages + 2 + a); };
  const uint32_t drain_bar = bar_base + 8u * (2 * stages + 4);
  const uint32_t tmem_cols = 2u * static_cast<uint32_t>(nt);

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  if (warp == 1 && lane == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int units0 = segment_tiles(&p.seg[0], nt) * p.seg[0].o_blocks;
  const int units1 = p.nseg > 1 ? segment_tiles(&p.seg[1], nt) * p.seg[1].o_blocks : 0;
  const int total = units0 + units1;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------ TMA producer
    for (int s = 0; s < p.nseg; ++s) {
      prefetch_tensormap(&p.seg[s].tmA);
      prefetch_tensormap(&p.seg[s].tmB);
    }
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const Unit x = decode_unit(p, u, units0, nt);
      const GemmSegment* s = x.seg ? &p.seg[1] : &p.seg[0];
      const int nbox = (x.n_rows + kBBoxRows - 1) / kBBoxRows;
      const uint32_t tx = kABytes + static_cast<uint32_t>(nbox) * kBBoxBytes;
      bool ok = true;
      for (int ks = 0; ks < s->k_steps; ++ks) {
        if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint32_t fb = full_bar(stage);
        mbar_arrive_expect_tx(fb, tx);
        const uint32_t a_dst = a_base + stage * kABytes;
        const uint32_t b_dst = b_base + stage * b_stage_bytes;
        const int kc = ks * kBK;
        if (p.mode == kModeSwiGLU) {
          if (s->a_boxes == 1) {
            tma_load_5d(a_dst, &s->tmA, fb, kc, 0, 0, x.ob * 4, x.group, pol_w);
          } else {
            for (int j = 0; j < 8; ++j)
              tma_load_3d(a_dst + j * 2048u, &s->tmA, fb, kc,
                          (j & 1) * s->a_rows + x.ob * 64 + (j >> 1) * 16, x.group, pol_w);
          }
        } else {
          tma_load_3d(a_dst, &s->tmA, fb, kc, x.ob * 128, x.group, pol_w);
        }
        for (int bx = 0; bx < nbox; ++bx)
          tma_load_2d(b_dst + bx * kBBoxBytes, &s->tmB, fb, kc, x.b_row + bx * kBBoxRows, pol_x);
        ++issued;
        if (++stage == stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
    // wait for the copies still in flight (normally long complete)
    const int64_t first = issued > stages ? issued - stages : 0;
    for (int64_t q = first; q < issued; ++q)
      drain_wait(full_bar(static_cast<int>(q % stages)), static_cast<uint32_t>((q / stages) & 1),
                 p.status);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------- MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int i = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++i) {
      const Unit x = decode_unit(p, u, units0, nt);
      const GemmSegment* s = x.seg ? &p.seg[1] : &p.seg[0];
      const int acc = i & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(i >> 1) & 1u;
      if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * nt);
      const uint32_t n = static_cast<uint32_t>((x.n_rows + 15) & ~15);
      const uint32_t idesc = idesc_bf16_f32(128, n);
      bool ok = true;
      for (int ks = 0; ks < s->k_steps; ++ks) {
        if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t adesc = smem_desc_sw128(a_base + stage * kABytes);
        const uint64_t bdesc = smem_desc_sw128(b_base + stage * b_stage_bytes);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          tc_mma_bf16(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc, (ks | kk) != 0);
        tc_commit(empty_bar(stage));
        if (++stage == stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit(tfull_bar(acc));
    }
    tc_commit(drain_bar);
    drain_wait(drain_bar, 0, p.status);
  } else if (warp >= 2) {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    int i = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++i) {
      const Unit x = decode_unit(p, u, units0, nt);
      const GemmSegment* s = x.seg ? &p.seg[1] : &p.seg[0];
      const int acc = i & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(i >> 1) & 1u;
      if (!warp_wait(tfull_bar(acc), acc_phase, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t taddr0 =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * nt);
      const int nchunks = (x.n_rows + 15) / 16;
      __nv_bfloat16* out = s->out;
      const int64_t ld = s->out_ld;
      for (int c = 0; c < nchunks; ++c) {
        uint32_t v[16];
        tmem_ld_x16(taddr0 + static_cast<uint32_t>(c * 16), v);
        tmem_ld_wait();
        const int tok0 = c * 16;
        if (p.mode == kModeSwiGLU) {
          const bool is_gate = lane < 16;
          const int f = x.ob * 64 + q * 16 + (lane & 15);
          float h[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float mine = __uint_as_float(v[j]);
            const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
            const float g = is_gate ? mine : other;
            const float up = is_gate ? other : mine;
            h[j] = silu_f(g) * up;
          }
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int tok = tok0 + (is_gate ? jj : 8 + jj);
            const float val = is_gate ? h[jj] : h[8 + jj];
            if (tok < x.n_rows)
              out[static_cast<int64_t>(x.out_row + tok) * ld + f] = __float2bfloat16_rn(val);
          }
        } else {
          const int o = x.ob * 128 + q * 32 + lane;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = tok0 + j;
            if (tok < x.n_rows) {
              float val = __uint_as_float(v[j]);
              if (s->row_scale) val *= __ldg(s->row_scale + x.out_row + tok);
              if (s->add)
                val += __bfloat162float(s->add[static_cast<int64_t>(x.out_row + tok) * s->add_ld + o]);
              out[static_cast<int64_t>(x.out_row + tok) * ld + o] = __float2bfloat16_rn(val);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
    }
  }

  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
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

GemmPlan plan_gemm(int nt) {
  GemmPlan g;
  g.nt = nt;
  const size_t per_stage = kABytes + static_cast<size_t>(nt) * 128;
  int st = static_cast<int>(kSmemBudget / per_stage);
  if (st > kMaxStages) st = kMaxStages;
  g.stages = st;
  g.smem_bytes = 1024 + per_stage * st + 8 * (2 * st + 5) + 16;
  return g;
}

cudaError_t launch_tc_gemm(const GemmParams& params, int num_sms, cudaStream_t stream) {
  const GemmPlan plan = plan_gemm(params.nt);
  GemmParams p = params;
  p.stages = plan.stages;
  static int configured_bytes[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && configured_bytes[dev] < static_cast<int>(plan.smem_bytes)) {
    err = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmemBudget + 4096));
    if (err != cudaSuccess) return err;
    configured_bytes[dev] = static_cast<int>(kSmemBudget + 4096);
  }
  tc_gemm_kernel<<<num_sms, kThreads, plan.smem_bytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fgs
