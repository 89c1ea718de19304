// C ABI of the fine-grained MoE layer: argument checks, workspace layout and
// the order of kernel launches.  No call allocates; no exception escapes.
//
// The layer ("Kimi K2 MoE", sections 2-3; "Kimi K2 · Router", "All 4 steps";
// "Kimi K3's router picks 16 of 896 experts", Stable LatentMoE):
//   router -> dispatch -> grouped SwiGLU experts (+ shared experts)
//          -> weighted combine (+ K3 latent projections)
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cmath>
#include <atomic>
#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "internal.h"

using namespace fgs;

namespace fgs {
namespace {
std::atomic<uint64_t> g_launches{0};
}  // namespace
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("FGS_PDL");  // tuning override: 0 = plain launches
    return !(v && *v == '0');
  }();
  return on;
}
}  // namespace fgs

namespace {

thread_local char g_detail[256] = "";

int32_t fail(int32_t code, const char* what) {
  snprintf(g_detail, sizeof(g_detail), "%s", what);
  return code;
}

int32_t cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_detail, sizeof(g_detail), "%s: %s", where, cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

#define MOE_CUDA(call)                                      \
  do {                                                      \
    cudaError_t e_ = (call);                                \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);     \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

int elem_bytes(const moe_config* c) { return c->dtype == MOE_BF16 ? 2 : 4; }

int d_expert(const moe_config* c) { return c->d_latent ? c->d_latent : c->d_model; }

// Parts of the router's K (= 3 d: the hi, mid and lo weight pieces) summed
// separately: one per piece, and each piece cut further when T is small so
// that the GEMM has enough independent units.
int env_int(const char* name, int fallback) {
  const char* v = getenv(name);
  return (v && *v) ? atoi(v) : fallback;
}

int router_tile(int64_t T);

// K parts of the router GEMM: the count (at most 48, at most d / 64) that
// minimises an estimate of its time on a 152-SM GB300 (a fixed count, so
// that a workspace sized on one device fits the call on another): the waves
// of units times the k steps of the longest part at 12 MMAs of N = tile per
// k step (one per weight piece and 16-wide k slice; about max(N/2, 59)
// cycles each), plus the partial logits written and read back at the HBM
// rate (about 3.6 KB per cycle).  One wave with all SMs busy and few parts
// wins; each extra part costs T E 8 bytes of traffic.
int router_ksplit(int64_t T, int d, int E) {
  static const int forced = env_int("FGS_ROUTER_KSPLIT", 0);  // tuning override
  const int kd = d / 64;
  const int pmax = kd < 48 ? kd : 48;
  if (forced >= 1 && forced <= pmax) return forced;
  const int64_t nt = router_tile(T);
  const int64_t per_part = ((T + nt - 1) / nt) * ((E + 127) / 128);
  const double kstep_clk = 12.0 * (nt / 2 > 59 ? nt / 2 : 59);
  int best = 1;
  double best_cost = 0.0;
  for (int P = 1; P <= pmax; ++P) {
    const int64_t rounds = (per_part * P + 151) / 152;
    const int64_t steps = (kd + P - 1) / P;
    const double cost = static_cast<double>(rounds * steps) * kstep_clk +
                        8.0 * P * static_cast<double>(T) * E / 3571.0;
    if (P == 1 || cost < best_cost) {
      best = P;
      best_cost = cost;
    }
  }
  return best;
}

int router_tile(int64_t T) {
  static const int forced = env_int("FGS_ROUTER_TILE", 0);  // tuning override
  if (forced == 32 || forced == 64 || forced == 128 || forced == 256) return forced;
  return T <= 256 ? 32 : 256;
}

// Unit order of a segment with implicit token tiles: token-tile-major when
// the weights are small enough to stay in L2 (64 MB, half of it) and the
// activation rows are the larger operand, so neither is fetched from HBM
// twice.  FGS_B_MAJOR=0 keeps the output-block-major order everywhere.
int prefer_b_major(int64_t a_bytes, int64_t b_bytes) {
  static const int forced = env_int("FGS_B_MAJOR", 1);  // tuning override
  return forced && a_bytes <= (64ll << 20) && b_bytes > a_bytes ? 1 : 0;
}

// Token tiles: 32 rows for small batches; otherwise 256, so most experts are
// one tile and their weights stream once per pass.  A unit of two 128-row
// weight tiles against a tile of more than 128 tokens fills both TMEM
// regions; its epilogue is short next to its main loop.
int token_tile(int64_t T, bool down_pass = false) {
  static const int forced = env_int("FGS_TOKEN_TILE", 0);  // tuning override
  static const int forced_down = env_int("FGS_DOWN_TILE", 0);
  const int f = down_pass ? forced_down : forced;
  if (f >= 32 && f <= 256 && f % 32 == 0) return f;
  return T <= 256 ? 32 : 256;
}

// Weight tiles per unit of the down pass: two, so each token tile read into
// shared memory feeds two 128-row weight tiles.
int down_a_per_unit() {
  static const int forced = env_int("FGS_DOWN_A", 0);  // tuning override
  return forced == 1 ? 1 : 2;
}

// Weight tiles per unit of the gate/up pass (two: the token tile's B stages
// are shared by two 128-row tiles).
int gate_up_a_per_unit() {
  static const int forced = env_int("FGS_GATE_UP_A", 0);  // tuning override
  return forced == 1 ? 1 : 2;
}

// CTA pairs (see GemmParams::pair) for the expert passes; launch_tc_gemm
// applies them where the segments allow.
bool use_pairs(bool down_pass) {
  static const int gate_up = env_int("FGS_PAIR_GATE_UP", 0);  // tuning override
  static const int down = env_int("FGS_PAIR_DOWN", 0);
  return (down_pass ? down : gate_up) == 1;
}

int32_t check_router_cfg(const moe_config* c, int64_t T) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cfg is null");
  if (T < 1 || T > (1ll << 30)) return fail(MOE_ERR_INVALID_ARG, "T out of range");
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return fail(MOE_ERR_INVALID_ARG, "dtype");
  if (c->E_routed < 1 || c->E_routed > 1024) return fail(MOE_ERR_INVALID_ARG, "E_routed not in [1, 1024]");
  if (c->K < 1 || c->K > c->E_routed) return fail(MOE_ERR_INVALID_ARG, "K not in [1, E]");
  if (c->K > 32) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "K > 32");
  if (T * c->K >= (1ll << 31)) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "T*K too large");
  if (c->n_group < 1 || c->n_group > 32) return fail(MOE_ERR_INVALID_ARG, "n_group not in [1, 32]");
  if (c->E_routed % c->n_group) return fail(MOE_ERR_INVALID_ARG, "E % n_group != 0");
  if (c->n_group > 1 && c->E_routed / c->n_group < 2)
    return fail(MOE_ERR_INVALID_ARG, "group-limited selection needs >= 2 experts per group");
  if (c->topk_group < 1 || c->topk_group > c->n_group)
    return fail(MOE_ERR_INVALID_ARG, "topk_group not in [1, n_group]");
  if (static_cast<int64_t>(c->K) > static_cast<int64_t>(c->topk_group) * (c->E_routed / c->n_group) &&
      c->n_group > 1)
    return fail(MOE_ERR_INVALID_ARG, "K > topk_group * E / n_group");
  if (!std::isfinite(c->routed_scaling_factor)) return fail(MOE_ERR_INVALID_ARG, "scale not finite");
  if (c->d_model < 32 || c->d_model % 32) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "d_model % 32 != 0");
  if (c->router_weight != MOE_ROUTER_WEIGHT_F32 && c->router_weight != MOE_ROUTER_WEIGHT_SPLIT)
    return fail(MOE_ERR_INVALID_ARG, "router_weight not a moe_router_weight_form");
  return MOE_OK;
}

int32_t check_layer_cfg(const moe_config* c, int64_t T) {
  int32_t st = check_router_cfg(c, T);
  if (st != MOE_OK) return st;
  if (c->d_ff < 1) return fail(MOE_ERR_INVALID_ARG, "d_ff < 1");
  if (c->E_shared < 0 || c->E_shared > 8) return fail(MOE_ERR_INVALID_ARG, "E_shared not in [0, 8]");
  if (c->E_shared > 0 && c->d_ff_shared < 1) return fail(MOE_ERR_INVALID_ARG, "d_ff_shared < 1");
  if (c->d_latent < 0) return fail(MOE_ERR_INVALID_ARG, "d_latent < 0");
  if (c->weight_layout != MOE_WEIGHTS_NATURAL && c->weight_layout != MOE_WEIGHTS_PACKED &&
      c->weight_layout != MOE_WEIGHTS_PACKED_FP8)
    return fail(MOE_ERR_INVALID_ARG, "weight_layout");
  if (c->weight_layout != MOE_WEIGHTS_NATURAL && c->dtype != MOE_BF16)
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "packed weights need bf16 activations");
  if (c->weight_layout == MOE_WEIGHTS_PACKED_FP8 &&
      (c->d_model % 128 || c->d_ff % 128 || (c->E_shared > 0 && c->d_ff_shared % 128) ||
       c->d_latent % 128))
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "FP8 weights: d_model, d_ff, d_ff_shared, d_latent % 128");
  if (c->dtype == MOE_BF16) {
    if (c->d_model % 128) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "bf16 path: d_model % 128 != 0");
    if (c->d_ff % 64) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "bf16 path: d_ff % 64 != 0");
    if (c->E_shared > 0 && c->d_ff_shared % 64)
      return fail(MOE_ERR_UNSUPPORTED_SHAPE, "bf16 path: d_ff_shared % 64 != 0");
    if (c->d_latent % 128) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "bf16 path: d_latent % 128 != 0");
  } else {
    if (c->d_latent) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "fp32 path has no latent projection");
  }
  return MOE_OK;
}

// Workspace regions, each 256-byte aligned, in this order.
struct Layout {
  size_t status, topk_idx, topk_w, counts, offsets, poffsets, perm, inv, ccount, tiles, ntiles,
      tiles_down,
      w_perm, w_split, logits, Xp, H, Hs, Y, U, Ysh, x_lat, r_lat, x_stage, y_stage, total;
  int64_t plane_rows;    // packed activation planes of the routed rows
  int64_t plane_rows_s;  // and of the shared experts' rows
  int64_t Ts;            // shared-expert rows per group in the packed planes
};

Layout layout(const moe_config* c, int64_t T) {
  Layout L;
  const int64_t TK = T * c->K;
  const int eb = elem_bytes(c);
  const int de = d_expert(c);
  const int S = c->d_ff > 0 ? c->E_shared : 0;
  const int64_t tiles = TK / kSimtTile + c->E_routed + 1;  // bound for every tile height used
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o += round256(bytes);
    return at;
  };
  L.status = take(kWsHeader);
  L.topk_idx = take(4 * TK);
  L.topk_w = take(4 * TK);
  L.counts = take(4 * static_cast<size_t>(c->E_routed));
  L.offsets = take(4 * static_cast<size_t>(c->E_routed + 1));
  L.poffsets = take(4 * static_cast<size_t>(c->E_routed + 1));
  L.perm = take(4 * TK);
  L.inv = take(4 * TK);
  L.ccount = take(4 * static_cast<size_t>(permute_chunks(TK)) * c->E_routed);
  L.tiles = take(sizeof(RowTile) * tiles);
  L.ntiles = take(16);
  L.tiles_down = take(sizeof(RowTile) * tiles);
  L.w_perm = take(4 * TK);
  L.w_split = take(c->dtype == MOE_BF16 ? 3ull * c->E_routed * c->d_model * 2 : 0);
  L.logits = take(c->dtype == MOE_BF16 && c->d_model % 64 == 0
                      ? 4ull * router_ksplit(T, c->d_model, c->E_routed) * T * c->E_routed
                      : 0);
  // bf16: gathered rows and SwiGLU outputs in the packed activation layout
  // (64-column planes of 128-byte rows, experts 8-row aligned); fp32: plain
  L.Ts = (T + 7) & ~7ll;
  L.plane_rows = packed_plane_rows(TK, c->E_routed);
  L.plane_rows_s = packed_plane_rows(S * L.Ts, 0);
  const bool pk = c->dtype == MOE_BF16;
  L.Xp = take(pk ? static_cast<size_t>(de / 64) * L.plane_rows * 128
                 : static_cast<size_t>(TK) * de * eb);
  L.H = take(pk ? static_cast<size_t>(c->d_ff / 64) * L.plane_rows * 128
                : static_cast<size_t>(TK) * c->d_ff * eb);
  L.Hs = take(pk ? static_cast<size_t>(c->d_ff_shared / 64) * L.plane_rows_s * 128
                 : static_cast<size_t>(S) * T * c->d_ff_shared * eb);
  L.Y = take(static_cast<size_t>(TK) * de * eb);
  // U and Ysh are adjacent (no padding: both are whole rows of d) so that
  // the final combine reads them as one strided list of addends
  const size_t U_bytes = c->d_latent ? static_cast<size_t>(T) * c->d_model * eb : 0;
  L.U = o;
  L.Ysh = o + U_bytes;
  o = round256(o + U_bytes + static_cast<size_t>(S) * T * c->d_model * eb);
  L.x_lat = take(c->d_latent ? static_cast<size_t>(T) * c->d_latent * eb : 0);
  L.r_lat = take(c->d_latent ? static_cast<size_t>(T) * c->d_latent * eb : 0);
  L.x_stage = take(2 * round256(static_cast<size_t>(T) * c->d_model * eb));  // two, alternating
  L.y_stage = take(2 * round256(static_cast<size_t>(T) * c->d_model * eb));  // two, alternating
  L.total = o;
  return L;
}

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

// Weights in MOE_WEIGHTS_PACKED order stream as one bulk copy per stage;
// natural ones through tensor maps: for gate/up a 5-D map when the driver
// accepts it, else eight 16-row boxes.
// Records of a packed FP8 bank: one per (group, pair of 128-row tiles,
// 64-column k step), after the tiles.
void set_fp8_records(GemmSegment& s, const void* W, int groups, int64_t rows, int Kd) {
  s.a_fp8 = 1;
  s.a_rec = static_cast<const uint8_t*>(W) + static_cast<int64_t>(groups) * rows * Kd;
  s.a_rec_group = ((rows / 128 + 1) / 2) * (Kd / 64);
}

int32_t set_gate_up_A(GemmSegment& s, const void* W, int groups, int F, int Kd, int layout) {
  s.a_rows = F;
  if (layout == MOE_WEIGHTS_PACKED_FP8) {
    s.a_packed = static_cast<const uint8_t*>(W);
    s.a_group_bytes = 2ll * F * Kd;
    s.a_groups = groups;
    s.a_boxes = 1;
    set_fp8_records(s, W, groups, 2ll * F, Kd);
    return MOE_OK;
  }
  if (layout == MOE_WEIGHTS_PACKED) {
    s.a_packed = static_cast<const uint8_t*>(W);
    s.a_group_bytes = 2ll * F * Kd * 2;
    s.a_groups = groups;
    s.a_boxes = 1;
    return MOE_OK;
  }
  if (encode_tmap_gate_up_5d(&s.tmA, W, groups, F, Kd) == CUDA_SUCCESS) {
    s.a_boxes = 1;
  } else if (encode_tmap_weights_3d(&s.tmA, W, groups, 2 * static_cast<int64_t>(F), Kd, 16) ==
             CUDA_SUCCESS) {
    s.a_boxes = 8;
  } else {
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed for W_gate_up");
  }
  s.a_rows = F;
  return MOE_OK;
}

// Activation rows through a tensor map whose box is a whole token tile of
// `tile` rows, so that each k step of a unit is one copy.
int32_t set_B(GemmSegment& s, const void* B, int64_t rows, int Kd, int tile) {
  if (encode_tmap_2d_rows(&s.tmB, B, rows, Kd, tile) != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed for activations");
  s.b_box_rows = tile;
  s.b_src = B;
  s.b_src_rows = rows;
  s.k_steps = Kd / 64;
  return MOE_OK;
}

// Activations in the packed layout: one bulk copy per stage.
void set_B_packed(GemmSegment& s, const void* B, int64_t plane_rows, int Kd) {
  s.b_packed = static_cast<const uint8_t*>(B);
  s.b_plane_rows = plane_rows;
  s.k_steps = Kd / 64;
}

int32_t set_store_A(GemmSegment& s, const void* W, int groups, int O, int Kd, int layout) {
  if (layout == MOE_WEIGHTS_PACKED_FP8) {
    s.a_packed = static_cast<const uint8_t*>(W);
    s.a_group_bytes = static_cast<int64_t>(O) * Kd;
    s.a_groups = groups;
    s.a_boxes = 1;
    s.a_rows = 0;
    set_fp8_records(s, W, groups, O, Kd);
    return MOE_OK;
  }
  if (layout == MOE_WEIGHTS_PACKED) {
    s.a_packed = static_cast<const uint8_t*>(W);
    s.a_group_bytes = static_cast<int64_t>(O) * Kd * 2;
    s.a_groups = groups;
    s.a_boxes = 1;
    s.a_rows = 0;
    return MOE_OK;
  }
  if (encode_tmap_weights_3d(&s.tmA, W, groups, O, Kd, 128) != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed for weights");
  s.a_boxes = 1;
  s.a_rows = 0;
  return MOE_OK;
}

void clear(GemmSegment& s) { memset(&s, 0, sizeof(s)); }

// Expert passes shared by moe_grouped_swiglu and moe_layer_forward.
struct ExpertIO {
  const void* x_e;       // [T, d_e]
  const int32_t* offsets;
  const int32_t* perm;
  const float* topk_w;   // may be null
  const void* W_gate_up;
  const void* W_down;
  const void* x_shared;  // [T, d] or null
  const void* Ws_gate_up;
  const void* Ws_down;
  void* Y;               // [T*K, d_e]
  void* Y_shared;        // [S, T, d] or null
  // the routing in token order (both or neither): lets the bf16 gather read
  // each token row once and write its K copies
  const int32_t* topk_idx = nullptr;
  const int32_t* inv = nullptr;
};

// The shared experts' gate/up pass as a GEMM segment: every token of x
// against each shared expert, SwiGLU outputs into the packed planes Hs.
int32_t shared_gate_up_segment(GemmSegment& s, const moe_config* c, int64_t T, const void* x,
                               const void* Ws_gate_up, const Layout& L, void* ws, int packed) {
  clear(s);
  int32_t e;
  if ((e = set_gate_up_A(s, Ws_gate_up, c->E_shared, c->d_ff_shared, c->d_model, packed)) != MOE_OK)
    return e;
  if ((e = set_B(s, x, T, c->d_model, token_tile(T))) != MOE_OK) return e;
  s.a128 = c->d_ff_shared / 64;
  s.groups = c->E_shared;
  s.rows = static_cast<int>(T);
  s.b_group_stride = 0;
  s.out_group_stride = L.Ts;
  s.out = at<__nv_bfloat16>(ws, L.Hs);
  s.out_packed = 1;
  s.out_plane_rows = L.plane_rows_s;
  s.own_mode = 1;
  s.mode = kModeSwiGLU;
  s.nt = token_tile(T);
  s.b_major = prefer_b_major(4ll * c->E_shared * c->d_ff_shared * c->d_model,
                             2ll * T * c->d_model);
  return MOE_OK;
}

// weights_in_Y: scale the routed rows of Y by their routing weights (the
// moe_grouped_swiglu contract); the layer forward leaves Y unscaled and
// weights the rows in its combine instead, which keeps the scale out of the
// GEMM epilogues.
int32_t run_experts(const moe_config* c, int64_t T, const ExpertIO& io, void* ws,
                    cudaEvent_t ev_up, cudaEvent_t ev_down, cudaStream_t st, bool weights_in_Y) {
  const Layout L = layout(c, T);
  const int E = c->E_routed, K = c->K, F = c->d_ff, de = d_expert(c);
  const int S = io.x_shared ? c->E_shared : 0;
  const int Fs = c->d_ff_shared, d = c->d_model;
  const int64_t TK = T * K;
  int* status = at<int>(ws, L.status);
  RowTile* tiles = at<RowTile>(ws, L.tiles);
  int* ntiles = at<int>(ws, L.ntiles);
  float* w_perm = weights_in_Y && io.topk_w ? at<float>(ws, L.w_perm) : nullptr;
  void* Xp = at<void>(ws, L.Xp);
  void* H = at<void>(ws, L.H);
  void* Hs = at<void>(ws, L.Hs);
  const bool bf16 = c->dtype == MOE_BF16;
  const int packed = c->weight_layout;  // moe_weight_layout of the expert banks
  const int nt = bf16 ? token_tile(T) : kSimtTile;
  const int nt_down = bf16 ? token_tile(T, true) : kSimtTile;
  RowTile* tiles_down = tiles;
  int* ntiles_down = ntiles;

  int32_t* poffsets = at<int32_t>(ws, L.poffsets);
  MOE_CUDA(launch_build_tiles(io.offsets, E, nt, tiles, ntiles, poffsets, st));
  if (nt_down != nt) {
    tiles_down = at<RowTile>(ws, L.tiles_down);
    ntiles_down = ntiles + 1;
    MOE_CUDA(launch_build_tiles(io.offsets, E, nt_down, tiles_down, ntiles_down, nullptr, st));
  }
  if (bf16 && io.topk_idx && io.inv) {
    MOE_CUDA(launch_gather_tokens_packed(io.x_e, T, K, de, io.topk_idx, io.inv, io.offsets,
                                         poffsets, E, io.topk_w, Xp, L.plane_rows, w_perm, st));
  } else if (bf16) {
    MOE_CUDA(launch_gather_packed(io.x_e, K, de, io.perm, io.offsets, poffsets, E, io.topk_w, Xp,
                                  L.plane_rows, w_perm, st));
  } else {
    MOE_CUDA(launch_gather(io.x_e, T, K, de, elem_bytes(c), io.perm, io.offsets, E, io.topk_w,
                           Xp, w_perm, st));
  }
  if (ev_up) MOE_CUDA(cudaEventRecord(ev_up, st));

  if (bf16) {
    GemmParams p;
    memset(&p, 0, sizeof(p));
    p.mode = kModeSwiGLU;
    p.nt = nt;
    p.a_per_unit = gate_up_a_per_unit();
    p.status = status;
    p.nseg = S ? 2 : 1;
    // gate/up: routed experts over the gathered rows
    GemmSegment& r = p.seg[0];
    clear(r);
    int32_t e;
    if ((e = set_gate_up_A(r, io.W_gate_up, E, F, de, packed)) != MOE_OK) return e;
    set_B_packed(r, Xp, L.plane_rows, de);
    r.a128 = F / 64;
    r.tiles = tiles;
    r.ntiles = ntiles;
    r.out = static_cast<__nv_bfloat16*>(H);
    r.out_packed = 1;
    r.out_plane_rows = L.plane_rows;
    if (p.nseg == 2 &&
        (e = shared_gate_up_segment(p.seg[1], c, T, io.x_shared, io.Ws_gate_up, L, ws, packed)) !=
            MOE_OK)
      return e;
    p.pair = use_pairs(false);
    MOE_CUDA(launch_tc_gemm(p, num_sms(), st));
    if (ev_down) MOE_CUDA(cudaEventRecord(ev_down, st));

    // down: routed rows (scaled by their gate weight when weights_in_Y) and
    // the shared experts' rows, one launch
    p.mode = kModeStore;
    p.nt = nt_down;
    p.nseg = S ? 2 : 1;
    p.a_per_unit = down_a_per_unit();
    GemmSegment& r2 = p.seg[0];
    clear(r2);
    if ((e = set_store_A(r2, io.W_down, E, de, F, packed)) != MOE_OK) return e;
    set_B_packed(r2, H, L.plane_rows, F);
    r2.a128 = de / 128;
    r2.o_limit = de;
    r2.tiles = tiles_down;
    r2.ntiles = ntiles_down;
    r2.out = static_cast<__nv_bfloat16*>(io.Y);
    r2.out_ld = de;
    r2.row_scale = w_perm;  // null unless the weights go into Y
    if (S) {
      GemmSegment& s2 = p.seg[1];
      clear(s2);
      if ((e = set_store_A(s2, io.Ws_down, S, d, Fs, packed)) != MOE_OK) return e;
      set_B_packed(s2, Hs, L.plane_rows_s, Fs);
      s2.a128 = d / 128;
      s2.o_limit = d;
      s2.groups = S;
      s2.rows = static_cast<int>(T);
      s2.b_group_stride = L.Ts;
      s2.out_group_stride = T;
      s2.out = static_cast<__nv_bfloat16*>(io.Y_shared);
      s2.out_ld = d;
      s2.b_major = prefer_b_major(2ll * S * d * Fs, 2ll * T * Fs);
    }
    p.pair = use_pairs(true);
    MOE_CUDA(launch_tc_gemm(p, num_sms(), st));
    return MOE_OK;
  }

  // fp32 CUDA-core path
  const int64_t bound_r = TK / kSimtTile + E;
  SimtGemm g;
  g.B = static_cast<const float*>(Xp);
  g.W = static_cast<const float*>(io.W_gate_up);
  g.w_group_stride = 2ll * F * de;
  g.Kdim = de;
  g.O = F;
  g.swiglu = true;
  g.tiles = tiles;
  g.ntiles = ntiles;
  g.out = static_cast<float*>(H);
  MOE_CUDA(launch_simt_gemm(g, bound_r, st));
  SimtGemm gs;
  const int64_t bound_s = S * ((T + kSimtTile - 1) / kSimtTile);
  if (S) {
    gs.B = static_cast<const float*>(io.x_shared);
    gs.W = static_cast<const float*>(io.Ws_gate_up);
    gs.w_group_stride = 2ll * Fs * d;
    gs.Kdim = d;
    gs.O = Fs;
    gs.swiglu = true;
    gs.groups = S;
    gs.rows = static_cast<int>(T);
    gs.b_group_stride = 0;
    gs.out_group_stride = T;
    gs.out = static_cast<float*>(Hs);
    MOE_CUDA(launch_simt_gemm(gs, bound_s, st));
  }
  if (ev_down) MOE_CUDA(cudaEventRecord(ev_down, st));
  SimtGemm g2;
  g2.B = static_cast<const float*>(H);
  g2.W = static_cast<const float*>(io.W_down);
  g2.w_group_stride = static_cast<int64_t>(de) * F;
  g2.Kdim = F;
  g2.O = de;
  g2.tiles = tiles;
  g2.ntiles = ntiles;
  g2.out = static_cast<float*>(io.Y);
  g2.row_scale = w_perm;
  MOE_CUDA(launch_simt_gemm(g2, bound_r, st));
  if (S) {
    SimtGemm g3;
    g3.B = static_cast<const float*>(Hs);
    g3.W = static_cast<const float*>(io.Ws_down);
    g3.w_group_stride = static_cast<int64_t>(d) * Fs;
    g3.Kdim = Fs;
    g3.O = d;
    g3.groups = S;
    g3.rows = static_cast<int>(T);
    g3.b_group_stride = T;
    g3.out_group_stride = T;
    g3.out = static_cast<float*>(io.Y_shared);
    MOE_CUDA(launch_simt_gemm(g3, bound_s, st));
  }
  (void)status;
  return MOE_OK;
}

// The K3 latent projections are bf16 whatever the expert banks are: packed
// when the banks are packed (bf16 or FP8), natural otherwise.
int latent_layout(const moe_config* c) {
  return c->weight_layout == MOE_WEIGHTS_NATURAL ? MOE_WEIGHTS_NATURAL : MOE_WEIGHTS_PACKED;
}

int32_t run_linear(int64_t T, int in_f, int out_f, const void* x, const void* W, const void* add,
                   void* y, int* status, cudaStream_t st, int packed = MOE_WEIGHTS_NATURAL) {
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.mode = kModeStore;
  p.nt = token_tile(T);
  p.status = status;
  p.nseg = 1;
  GemmSegment& s = p.seg[0];
  clear(s);
  int32_t e;
  if ((e = set_store_A(s, W, 1, out_f, in_f, packed)) != MOE_OK) return e;
  if ((e = set_B(s, x, T, in_f, p.nt)) != MOE_OK) return e;
  s.a128 = out_f / 128;
  s.o_limit = out_f;
  s.groups = 1;
  s.rows = static_cast<int>(T);
  s.out = static_cast<__nv_bfloat16*>(y);
  s.out_ld = out_f;
  s.add = static_cast<const __nv_bfloat16*>(add);
  s.add_ld = out_f;
  s.b_major = prefer_b_major(2ll * out_f * in_f, 2ll * T * in_f);
  MOE_CUDA(launch_tc_gemm(p, num_sms(), st));
  return MOE_OK;
}

// The router logits GEMM: partial logits part j = x W_split^T over k steps
// [j K / P, (j + 1) K / P) of K = d / 64, where W_split [E, 3 d] holds the
// hi, mid and lo bf16 pieces of W_r side by side; the three pieces of a
// k step accumulate into the unit's one accumulator, so each token tile in
// shared memory feeds all three.
int32_t router_gemm(const void* x, const void* w_split, int64_t T, int d, int E, int parts,
                    float* logits, int* status, cudaStream_t st) {
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.mode = kModeStore;
  p.nt = router_tile(T);
  p.a_per_unit = 1;
  p.pieces = 3;
  p.status = status;
  p.nseg = 1;
  GemmSegment& g = p.seg[0];
  clear(g);
  if (encode_tmap_weights_3d(&g.tmA, w_split, 1, E, 3ll * d, 128) != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed for the split router weight");
  int32_t e;
  if ((e = set_B(g, x, T, d, p.nt)) != MOE_OK) return e;
  g.k_steps = d / 64;
  g.a_piece_cols = d;
  g.a128 = (E + 127) / 128;
  g.o_limit = E;
  g.groups = 1;
  g.rows = static_cast<int>(T);
  g.out_f32 = logits;
  g.out_ld = E;
  g.ksplit = parts;
  g.b_major = prefer_b_major(6ll * E * d, 2ll * T * d);
  g.out_split_stride = T * E;
  MOE_CUDA(launch_tc_gemm(p, num_sms(), st));
  return MOE_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// Fixed scratch for moe_router_noalloc: some callers may not allocate device
// memory at the moment they route tokens, so this one entry point takes its
// scratch from a statically sized device array that exists for as long as
// the library is loaded on a device.
constexpr size_t kNoAllocScratchBytes = 64ull << 20;  // 64 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_noalloc_mutex;
// Per device: the context the address was looked up in, and the address.
struct NoAllocSlot {
  unsigned long long ctx_id = 0;
  void* ptr = nullptr;
};
NoAllocSlot g_noalloc_slot[64];

// Identity of the calling thread's current CUDA context (0 when there is
// none yet, or when the driver entry points are unavailable).  A context
// that is torn down (cudaDeviceReset) and created again gets a new id.
unsigned long long current_context_id() {
  typedef CUresult (*GetCurrent)(CUcontext*);
  typedef CUresult (*GetId)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) ==
            cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
            cudaSuccess &&
        qb == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<GetCurrent>(a);
      get_id = reinterpret_cast<GetId>(b);
    }
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_noalloc_scratch in the current device's context.  In
// host code the array's name is only a stand-in for the device object, so
// kernels must be given this address instead.  It is looked up once per
// device and context: again after the context was torn down and created
// anew, and on every call when the context cannot be identified.
int32_t noalloc_scratch(void** out) {
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(MOE_ERR_CUDA, "device ordinal beyond 63");
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoAllocSlot& slot = g_noalloc_slot[dev];
  unsigned long long id = current_context_id();
  if (id == 0 || id != slot.ctx_id || !slot.ptr) {
    void* p = nullptr;
    MOE_CUDA(cudaGetSymbolAddress(&p, g_noalloc_scratch));
    if (id == 0) id = current_context_id();  // the lookup made the context current
    slot.ctx_id = id;
    slot.ptr = p;
  }
  *out = slot.ptr;
  return MOE_OK;
}

// Scratch bytes moe_router_noalloc needs with P K parts: the status word,
// the split router weight (unless the caller passes it) and P partial
// logit arrays.
size_t noalloc_need(int64_t T, int d, int E, bool presplit, int parts) {
  return kWsHeader + (presplit ? 0 : round256(3ull * E * d * 2)) +
         round256(4ull * parts * T * E);
}

// K parts of the allocation-free router GEMM: moe_router's own count when
// that fits the static scratch, else the largest smaller count that fits;
// 0 when none does.
int noalloc_ksplit(int64_t T, int d, int E, bool presplit) {
  for (int c = router_ksplit(T, d, E); c >= 1; --c)
    if (noalloc_need(T, d, E, presplit, c) <= kNoAllocScratchBytes) return c;
  return 0;
}

}  // namespace

extern "C" {

int32_t moe_version(void) { return 100; }

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* moe_status_string(int32_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_TIMEOUT: return "bounded device wait expired";
    case MOE_ERR_DEVICE_INDEX: return "expert index out of range";
    default: return "unknown status";
  }
}

const char* moe_last_error_detail(void) { return g_detail; }

int32_t moe_validate_config(const moe_config* cfg, int64_t T) {
  if (cfg && cfg->d_ff > 0) return check_layer_cfg(cfg, T);
  return check_router_cfg(cfg, T);
}

size_t moe_workspace_size(const moe_config* cfg, int64_t T) {
  if (moe_validate_config(cfg, T) != MOE_OK) return 0;
  return layout(cfg, T).total;
}

namespace fgs {
namespace {

// One thread waits, through the library's bounded mbarrier wait, on a
// barrier that nothing arrives at: the wait gives up after its time limit,
// records MOE_ERR_TIMEOUT in the status word and the kernel returns.
__global__ void bounded_wait_probe_kernel(int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait_bounded(smem_u32(&bar), 0u, &abort_flag, status);
    if (ok) record_status(status, MOE_ERR_INVALID_ARG);  // cannot happen: nothing arrives
  }
}

}  // namespace
}  // namespace fgs

int32_t moe_selftest_bounded_wait(void* workspace, void* stream) {
  if (!workspace) return fail(MOE_ERR_WORKSPACE, "workspace is null");
  fgs::note_launch();
  fgs::bounded_wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<int*>(workspace));
  MOE_CUDA(cudaGetLastError());
  return MOE_OK;
}

int32_t moe_get_device_status(void* workspace, void* stream) {
  if (!workspace) return fail(MOE_ERR_WORKSPACE, "workspace is null");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_CUDA(cudaStreamSynchronize(st));
  int v = 0;
  MOE_CUDA(cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost));
  MOE_CUDA(cudaMemset(workspace, 0, sizeof(int)));
  return v;
}

int32_t moe_router(const moe_config* cfg, int64_t T, const void* x, const float* W_r,
                   const float* bias, int32_t* topk_idx, float* topk_w, void* workspace,
                   size_t ws_bytes, void* stream) {
  int32_t st = check_router_cfg(cfg, T);
  if (st != MOE_OK) return st;
  if (!x || !W_r || !bias || !topk_idx || !topk_w) return fail(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(x) || !aligned16(W_r) || !aligned16(bias) || !aligned16(topk_idx) ||
      !aligned16(topk_w) || (workspace && !aligned16(workspace)))
    return fail(MOE_ERR_ALIGNMENT, "pointer not 16-byte aligned");
  const bool presplit = cfg->router_weight == MOE_ROUTER_WEIGHT_SPLIT;
  if (presplit && !(workspace && cfg->dtype == MOE_BF16 && cfg->d_model % 64 == 0))
    return fail(MOE_ERR_UNSUPPORTED_SHAPE,
                "a split router weight needs bf16 x, d_model % 64 == 0 and a workspace");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  RouterArgs a;
  a.W_r = W_r;
  a.bias = bias;
  a.T = T;
  a.d = cfg->d_model;
  a.E = cfg->E_routed;
  a.K = cfg->K;
  a.G = cfg->n_group;
  a.Gk = cfg->topk_group;
  a.scale = cfg->routed_scaling_factor;
  a.norm = cfg->norm_topk_prob;
  a.x_bf16 = cfg->dtype == MOE_BF16;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  if (workspace && cfg->dtype == MOE_BF16 && cfg->d_model % 64 == 0) {
    const Layout L = layout(cfg, T);
    if (ws_bytes < L.total) return fail(MOE_ERR_WORKSPACE, "workspace too small");
    // logits = x (W_hi + W_mid + W_lo)^T on the tensor cores
    const void* w_split = presplit ? static_cast<const void*>(W_r)
                                   : at<__nv_bfloat16>(workspace, L.w_split);
    float* logits = at<float>(workspace, L.logits);
    const int d = cfg->d_model, E = cfg->E_routed;
    if (!presplit)
      MOE_CUDA(launch_split_router_weight(W_r, E, d, at<__nv_bfloat16>(workspace, L.w_split), s));
    const int parts = router_ksplit(T, d, E);
    const int32_t e =
        router_gemm(x, w_split, T, d, E, parts, logits, at<int>(workspace, L.status), s);
    if (e != MOE_OK) return e;
    a.logits = logits;
    a.logit_parts = parts;
    a.logit_part_stride = T * E;
  } else {
    a.x = x;
  }
  MOE_CUDA(launch_router(a, s));
  return MOE_OK;
}

int32_t moe_dense_gates(const moe_config* cfg, int64_t T, const int32_t* topk_idx,
                        const float* topk_w, float* G, void* stream) {
  int32_t st = check_router_cfg(cfg, T);
  if (st != MOE_OK) return st;
  if (!topk_idx || !topk_w || !G) return fail(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(G))
    return fail(MOE_ERR_ALIGNMENT, "pointer not 16-byte aligned");
  MOE_CUDA(launch_dense_gates(topk_idx, topk_w, T, cfg->K, cfg->E_routed, G,
                              static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int32_t moe_update_bias(const moe_config* cfg, int64_t T, const int32_t* counts, float gamma,
                        float* bias, void* stream) {
  int32_t st = check_router_cfg(cfg, T);
  if (st != MOE_OK) return st;
  if (!counts || !bias) return fail(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(counts) || !aligned16(bias))
    return fail(MOE_ERR_ALIGNMENT, "pointer not 16-byte aligned");
  if (!(gamma >= 0.0f) || !(gamma < 1.0f)) return fail(MOE_ERR_INVALID_ARG, "gamma not in [0, 1)");
  MOE_CUDA(launch_bias_update(counts, T, cfg->K, cfg->E_routed, gamma, bias,
                              static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int32_t moe_quantile_bias_update(const moe_config* cfg, int64_t T, const float* logits, float rate,
                                 float* theta, float* bias, void* stream) {
  int32_t st = check_router_cfg(cfg, T);
  if (st != MOE_OK) return st;
  if (!logits || !theta || !bias) return fail(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(logits) || !aligned16(theta) || !aligned16(bias))
    return fail(MOE_ERR_ALIGNMENT, "pointer not 16-byte aligned");
  if (!(rate >= 0.0f) || !(rate <= 1.0f)) return fail(MOE_ERR_INVALID_ARG, "rate not in [0, 1]");
  MOE_CUDA(launch_quantile_bias(logits, T, cfg->K, cfg->E_routed, rate, theta, bias,
                                static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int32_t moe_router_from_logits(const moe_config* cfg, int64_t T, const float* logits,
                               const float* bias, int32_t* topk_idx, float* topk_w,
                               void* stream) {
  int32_t st = check_router_cfg(cfg, T);
  if (st != MOE_OK) return st;
  if (!logits || !bias || !topk_idx || !topk_w) return fail(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(logits) || !aligned16(bias) || !aligned16(topk_idx) || !aligned16(topk_w))
    return fail(MOE_ERR_ALIGNMENT, "pointer not 16-byte aligned");
  RouterArgs a;
  a.logits = logits;
  a.bias = bias;
  a.T = T;
  a.E = cfg->E_routed;
  a.K = cfg->K;
  a.G = cfg->n_group;
  a.Gk = cfg->topk_group;
  a.scale = cfg->routed_scaling_factor;
  a.norm = cfg->norm_topk_prob;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  MOE_CUDA(launch_router(a, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int32_t moe_permute(const moe_config* cfg, int64_t T, const int32_t* topk_idx, int32_t* counts,
                    int32_t* offsets, int32_t* perm, int32_t* inv, void* workspace,
                    size_t ws_bytes, void* stream) {
  int32_t st = check_router_cfg(cfg, T);
  if (st != MOE_OK) return st;
  if (!topk_idx || !counts || !offsets || !perm || !inv) return fail(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(topk_idx) || !aligned16(counts) || !aligned16(offsets) || !aligned16(perm) ||
      !aligned16(inv))
    return fail(MOE_ERR_ALIGNMENT, "pointer not 16-byte aligned");
  // status word, then the per-chunk counts
  const size_t need = kWsHeader + 4 * static_cast<size_t>(permute_chunks(T * cfg->K)) *
                                      static_cast<size_t>(cfg->E_routed);
  if (!workspace || ws_bytes < need) return fail(MOE_ERR_WORKSPACE, "workspace too small");
  if (!aligned16(workspace)) return fail(MOE_ERR_ALIGNMENT, "workspace not aligned");
  MOE_CUDA(launch_permute(topk_idx, T, cfg->K, cfg->E_routed, counts, offsets, perm, inv,
                          at<int32_t>(workspace, kWsHeader), static_cast<int*>(workspace),
                          static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int32_t moe_grouped_swiglu(const moe_config* cfg, int64_t T, const void* x_e,
                           const int32_t* offsets, const int32_t* perm, const float* topk_w,
                           const void* W_gate_up, const void* W_down, const void* x_shared,
                           const void* Ws_gate_up, const void* Ws_down, void* Y, void* Y_shared,
                           void* workspace, size_t ws_bytes, void* stream) {
  int32_t st = check_layer_cfg(cfg, T);
  if (st != MOE_OK) return st;
  if (!x_e || !offsets || !perm || !W_gate_up || !W_down || !Y)
    return fail(MOE_ERR_INVALID_ARG, "null pointer");
  const bool shared = x_shared != nullptr && cfg->E_shared > 0;
  if (shared && (!Ws_gate_up || !Ws_down || !Y_shared))
    return fail(MOE_ERR_INVALID_ARG, "shared expert pointers missing");
  const void* ptrs[] = {x_e, offsets, perm, topk_w, W_gate_up, W_down, x_shared, Ws_gate_up,
                        Ws_down, Y, Y_shared, workspace};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return fail(MOE_ERR_ALIGNMENT, "pointer not 16-byte aligned");
  if (!workspace || ws_bytes < layout(cfg, T).total) return fail(MOE_ERR_WORKSPACE, "workspace too small");
  ExpertIO io = {x_e, offsets, perm, topk_w, W_gate_up, W_down, shared ? x_shared : nullptr,
                 Ws_gate_up, Ws_down, Y, Y_shared};
  return run_experts(cfg, T, io, workspace, nullptr, nullptr, static_cast<cudaStream_t>(stream),
                     true);
}

int32_t moe_combine(const moe_config* cfg, int64_t T, const void* Y, const int32_t* inv,
                    const float* topk_w, const void* Y_shared, void* y, void* stream) {
  int32_t st = check_layer_cfg(cfg, T);
  if (st != MOE_OK) return st;
  if (!Y || !inv || !y) return fail(MOE_ERR_INVALID_ARG, "null pointer");
  if (Y_shared && cfg->d_latent) return fail(MOE_ERR_INVALID_ARG, "Y_shared with d_latent");
  if (!aligned16(Y) || !aligned16(inv) || !aligned16(y) || (Y_shared && !aligned16(Y_shared)) ||
      (topk_w && !aligned16(topk_w)))
    return fail(MOE_ERR_ALIGNMENT, "pointer not 16-byte aligned");
  const int D = d_expert(cfg);
  if (D % 8) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "width % 8 != 0");
  MOE_CUDA(launch_combine(Y, inv, topk_w, T, cfg->K, D, Y_shared, Y_shared ? cfg->E_shared : 0, T,
                          y, cfg->dtype == MOE_BF16, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int32_t moe_pack_weights(int32_t kind, int64_t groups, int64_t rows, int64_t cols,
                         const void* src, void* dst, void* stream) {
  if (kind != MOE_PACK_GATE_UP && kind != MOE_PACK_PLAIN) return fail(MOE_ERR_INVALID_ARG, "kind");
  if (groups < 1 || rows < 128 || cols < 64) return fail(MOE_ERR_INVALID_ARG, "sizes");
  if (rows % 128 || cols % 64) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "rows % 128 or cols % 64");
  if (!src || !dst) return fail(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(src) || !aligned16(dst)) return fail(MOE_ERR_ALIGNMENT, "pointer not 16-byte aligned");
  const size_t bytes = static_cast<size_t>(groups * rows * cols) * 2;
  const char* a = static_cast<const char*>(src);
  const char* b = static_cast<const char*>(dst);
  if (a < b + bytes && b < a + bytes) return fail(MOE_ERR_INVALID_ARG, "src and dst overlap");
  MOE_CUDA(launch_pack_weights(kind, groups, rows, cols, src, dst, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int64_t moe_packed_fp8_bytes(int64_t groups, int64_t rows, int64_t cols) {
  if (groups < 1 || rows < 128 || cols < 128 || rows % 128 || cols % 128) return -1;
  return packed_fp8_bytes(groups, rows, cols);
}

int32_t moe_pack_weights_fp8(int32_t kind, int64_t groups, int64_t rows, int64_t cols,
                             const void* codes, const float* scales, void* dst, void* stream) {
  if (kind != MOE_PACK_GATE_UP && kind != MOE_PACK_PLAIN) return fail(MOE_ERR_INVALID_ARG, "kind");
  if (groups < 1 || rows < 128 || cols < 128) return fail(MOE_ERR_INVALID_ARG, "sizes");
  if (rows % 128 || cols % 128) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "rows % 128 or cols % 128");
  if (!codes || !scales || !dst) return fail(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(codes) || !aligned16(dst) || reinterpret_cast<uintptr_t>(scales) % 4)
    return fail(MOE_ERR_ALIGNMENT, "codes or dst not 16-byte aligned, or scales not 4-byte aligned");
  const char* a = static_cast<const char*>(codes);
  const char* b = static_cast<const char*>(dst);
  const size_t na = static_cast<size_t>(groups * rows * cols);
  const size_t nb = static_cast<size_t>(packed_fp8_bytes(groups, rows, cols));
  if (a < b + nb && b < a + na) return fail(MOE_ERR_INVALID_ARG, "codes and dst overlap");
  MOE_CUDA(launch_pack_weights_fp8(kind, groups, rows, cols, codes, scales, dst,
                                   static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int32_t moe_linear(int64_t T, int32_t in_features, int32_t out_features, const void* x,
                   const void* W, const void* add, void* y, void* workspace, size_t ws_bytes,
                   void* stream) {
  if (T < 1 || T > (1ll << 30)) return fail(MOE_ERR_INVALID_ARG, "T out of range");
  if (in_features < 128 || out_features < 128 || in_features % 128 || out_features % 128)
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "in/out features must be multiples of 128");
  if (!x || !W || !y) return fail(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(x) || !aligned16(W) || !aligned16(y) || (add && !aligned16(add)))
    return fail(MOE_ERR_ALIGNMENT, "pointer not 16-byte aligned");
  if (!workspace || ws_bytes < kWsHeader) return fail(MOE_ERR_WORKSPACE, "workspace too small");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return run_linear(T, in_features, out_features, x, W, add, y, static_cast<int*>(workspace), st);
}

int32_t moe_layer_forward(const moe_config* cfg, int64_t T, const void* x, const float* W_r,
                          const float* bias, const void* W_gate_up, const void* W_down,
                          const void* Ws_gate_up, const void* Ws_down, const void* W_lat_down,
                          const void* W_lat_up, void* y, int32_t* topk_idx_out,
                          float* topk_w_out, int32_t* counts_out, void* workspace,
                          size_t ws_bytes, void* const* stage_events, void* stream) {
  int32_t st = check_layer_cfg(cfg, T);
  if (st != MOE_OK) return st;
  const int S = cfg->E_shared;
  if (!x || !W_r || !bias || !W_gate_up || !W_down || !y) return fail(MOE_ERR_INVALID_ARG, "null pointer");
  if (S && (!Ws_gate_up || !Ws_down)) return fail(MOE_ERR_INVALID_ARG, "shared expert weights missing");
  if (cfg->d_latent && (!W_lat_down || !W_lat_up)) return fail(MOE_ERR_INVALID_ARG, "latent projections missing");
  const void* ptrs[] = {x, W_r, bias, W_gate_up, W_down, Ws_gate_up, Ws_down, W_lat_down,
                        W_lat_up, y, topk_idx_out, topk_w_out, counts_out, workspace};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return fail(MOE_ERR_ALIGNMENT, "pointer not 16-byte aligned");
  const Layout L = layout(cfg, T);
  if (!workspace || ws_bytes < L.total) return fail(MOE_ERR_WORKSPACE, "workspace too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto ev = [&](int i) -> cudaEvent_t {
    return stage_events ? static_cast<cudaEvent_t>(stage_events[i]) : nullptr;
  };
  void* ws = workspace;
  int* status = at<int>(ws, L.status);
  int32_t* idx = topk_idx_out ? topk_idx_out : at<int32_t>(ws, L.topk_idx);
  float* w = topk_w_out ? topk_w_out : at<float>(ws, L.topk_w);
  int32_t* counts = counts_out ? counts_out : at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* perm = at<int32_t>(ws, L.perm);
  int32_t* inv = at<int32_t>(ws, L.inv);
  const bool bf16 = cfg->dtype == MOE_BF16;

  if (ev(0)) MOE_CUDA(cudaEventRecord(ev(0), s));
  st = moe_router(cfg, T, x, W_r, bias, idx, w, ws, ws_bytes, s);
  if (st != MOE_OK) return st;
  if (ev(1)) MOE_CUDA(cudaEventRecord(ev(1), s));
  MOE_CUDA(launch_permute(idx, T, cfg->K, cfg->E_routed, counts, offsets, perm, inv,
                          at<int32_t>(ws, L.ccount), status, s));
  const void* x_e = x;
  if (cfg->d_latent) {
    st = run_linear(T, cfg->d_model, cfg->d_latent, x, W_lat_down, nullptr, at<void>(ws, L.x_lat),
                    status, s, latent_layout(cfg));
    if (st != MOE_OK) return st;
    x_e = at<void>(ws, L.x_lat);
  }
  ExpertIO io = {x_e, offsets, perm, w, W_gate_up, W_down, S ? x : nullptr, Ws_gate_up, Ws_down,
                 at<void>(ws, L.Y), S ? at<void>(ws, L.Ysh) : nullptr};
  io.topk_idx = idx;
  io.inv = inv;
  st = run_experts(cfg, T, io, ws, ev(2), ev(3), s, false);
  if (st != MOE_OK) return st;
  if (ev(4)) MOE_CUDA(cudaEventRecord(ev(4), s));
  if (!cfg->d_latent) {
    MOE_CUDA(launch_combine(at<void>(ws, L.Y), inv, w, T, cfg->K, cfg->d_model,
                            at<void>(ws, L.Ysh), S, T, y, bf16, s));
  } else {
    // routed sum in latent space, project back, add the shared experts
    MOE_CUDA(launch_combine(at<void>(ws, L.Y), inv, w, T, cfg->K, cfg->d_latent, nullptr, 0, 0,
                            at<void>(ws, L.r_lat), bf16, s));
    st = run_linear(T, cfg->d_latent, cfg->d_model, at<void>(ws, L.r_lat), W_lat_up, nullptr,
                    at<void>(ws, L.U), status, s, latent_layout(cfg));
    if (st != MOE_OK) return st;
    MOE_CUDA(launch_combine(nullptr, nullptr, nullptr, T, 0, cfg->d_model, at<void>(ws, L.U), 1 + S,
                            T, y, bf16, s));
  }
  if (ev(5)) MOE_CUDA(cudaEventRecord(ev(5), s));
  return MOE_OK;
}

namespace {

// Per-workspace state of the pipelined host-buffer forward: which staging
// buffer the next call takes, and the events that order the copy stream and
// the caller's stream around each buffer.
struct HostPipe {
  cudaEvent_t copied[2] = {nullptr, nullptr};  // x landed in staging buffer b
  cudaEvent_t read[2] = {nullptr, nullptr};    // the forward that read buffer b finished
  cudaEvent_t landed[2] = {nullptr, nullptr};  // y of buffer b copied out (pipelined calls)
  bool used[2] = {false, false};
  bool y_out[2] = {false, false};  // a copy-out of y buffer b was enqueued
  int next = 0;
  int last = -1;  // buffer of the latest pipelined call, until its y is waited for
};

std::mutex g_pipe_mutex;
std::unordered_map<void*, HostPipe> g_pipes;
cudaStream_t g_copy_stream[64] = {nullptr};  // x in
cudaStream_t g_out_stream[64] = {nullptr};   // y out (pipelined calls)

// The host-buffer forward, synchronous (y_host valid once `stream` is
// synchronised) or pipelined (y_host of this call valid once `stream` has
// passed the next pipelined call on the workspace, or a flush).
int32_t forward_host(const moe_config* cfg, int64_t T, const void* x_host, const float* W_r,
                     const float* bias, const void* W_gate_up, const void* W_down,
                     const void* Ws_gate_up, const void* Ws_down, const void* W_lat_down,
                     const void* W_lat_up, void* y_host, void* workspace, size_t ws_bytes,
                     void* stream, bool pipelined) {
  int32_t st = check_layer_cfg(cfg, T);
  if (st != MOE_OK) return st;
  if (!x_host || !y_host) return fail(MOE_ERR_INVALID_ARG, "null host pointer");
  const Layout L = layout(cfg, T);
  if (!workspace || ws_bytes < L.total) return fail(MOE_ERR_WORKSPACE, "workspace too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = static_cast<size_t>(T) * cfg->d_model * elem_bytes(cfg);
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  if (dev >= 64) return fail(MOE_ERR_INVALID_ARG, "device index above 63");
  HostPipe* hp;
  cudaStream_t cs, os;
  int b;
  {
    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    if (!g_copy_stream[dev])
      MOE_CUDA(cudaStreamCreateWithFlags(&g_copy_stream[dev], cudaStreamNonBlocking));
    if (!g_out_stream[dev])
      MOE_CUDA(cudaStreamCreateWithFlags(&g_out_stream[dev], cudaStreamNonBlocking));
    cs = g_copy_stream[dev];
    os = g_out_stream[dev];
    hp = &g_pipes[workspace];
    for (int i = 0; i < 2; ++i) {
      if (!hp->copied[i]) MOE_CUDA(cudaEventCreateWithFlags(&hp->copied[i], cudaEventDisableTiming));
      if (!hp->read[i]) MOE_CUDA(cudaEventCreateWithFlags(&hp->read[i], cudaEventDisableTiming));
      if (!hp->landed[i]) MOE_CUDA(cudaEventCreateWithFlags(&hp->landed[i], cudaEventDisableTiming));
    }
    b = hp->next;
    hp->next ^= 1;
  }
  void* xd = at<void>(workspace, L.x_stage + b * round256(bytes));
  void* yd = at<void>(workspace, L.y_stage + b * round256(bytes));
  // synchronous form: y_host pinned and mapped into this device's address
  // space is written by the layer's last kernel itself (over the host link),
  // so no staging copy delays the next call's forward on `stream`
  bool y_direct = false;
  static const int direct_ok = env_int("FGS_Y_DIRECT", 1);  // 0: always stage and copy
  if (!pipelined && direct_ok) {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, y_host) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
        pa.devicePointer && aligned16(pa.devicePointer) && pa.device == dev) {
      yd = pa.devicePointer;
      y_direct = true;
    } else {
      cudaGetLastError();  // an unregistered pointer leaves an error to clear
    }
  }
  // the buffer is free once the forward that last read it has finished
  if (hp->used[b]) MOE_CUDA(cudaStreamWaitEvent(cs, hp->read[b], 0));
  MOE_CUDA(cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, cs));
  MOE_CUDA(cudaEventRecord(hp->copied[b], cs));
  MOE_CUDA(cudaStreamWaitEvent(s, hp->copied[b], 0));
  // y buffer b is free once its last copy-out has finished (two calls ago)
  if (hp->y_out[b]) MOE_CUDA(cudaStreamWaitEvent(s, hp->landed[b], 0));
  st = moe_layer_forward(cfg, T, xd, W_r, bias, W_gate_up, W_down, Ws_gate_up, Ws_down,
                         W_lat_down, W_lat_up, yd, nullptr, nullptr, nullptr, workspace, ws_bytes,
                         nullptr, stream);
  if (st != MOE_OK) return st;
  MOE_CUDA(cudaEventRecord(hp->read[b], s));
  hp->used[b] = true;
  if (!pipelined) {
    if (!y_direct) MOE_CUDA(cudaMemcpyAsync(y_host, yd, bytes, cudaMemcpyDeviceToHost, s));
    return MOE_OK;
  }
  // pipelined: y goes out on the output stream while the next call's forward
  // runs; `stream` waits for the previous pipelined call's copy-out only now,
  // after this call's forward (by then that copy has long finished)
  MOE_CUDA(cudaStreamWaitEvent(os, hp->read[b], 0));
  MOE_CUDA(cudaMemcpyAsync(y_host, yd, bytes, cudaMemcpyDeviceToHost, os));
  MOE_CUDA(cudaEventRecord(hp->landed[b], os));
  hp->y_out[b] = true;
  if (hp->last >= 0 && hp->last != b) MOE_CUDA(cudaStreamWaitEvent(s, hp->landed[hp->last], 0));
  hp->last = b;
  return MOE_OK;
}

}  // namespace

int32_t moe_layer_forward_host(const moe_config* cfg, int64_t T, const void* x_host,
                               const float* W_r, const float* bias, const void* W_gate_up,
                               const void* W_down, const void* Ws_gate_up, const void* Ws_down,
                               const void* W_lat_down, const void* W_lat_up, void* y_host,
                               void* workspace, size_t ws_bytes, void* stream) {
  return forward_host(cfg, T, x_host, W_r, bias, W_gate_up, W_down, Ws_gate_up, Ws_down,
                      W_lat_down, W_lat_up, y_host, workspace, ws_bytes, stream, false);
}

int32_t moe_layer_forward_host_pipelined(const moe_config* cfg, int64_t T, const void* x_host,
                                         const float* W_r, const float* bias,
                                         const void* W_gate_up, const void* W_down,
                                         const void* Ws_gate_up, const void* Ws_down,
                                         const void* W_lat_down, const void* W_lat_up,
                                         void* y_host, void* workspace, size_t ws_bytes,
                                         void* stream) {
  return forward_host(cfg, T, x_host, W_r, bias, W_gate_up, W_down, Ws_gate_up, Ws_down,
                      W_lat_down, W_lat_up, y_host, workspace, ws_bytes, stream, true);
}

int32_t moe_layer_forward_host_flush(void* workspace, void* stream) {
  if (!workspace) return fail(MOE_ERR_INVALID_ARG, "workspace is null");
  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  auto it = g_pipes.find(workspace);
  if (it == g_pipes.end() || it->second.last < 0) return MOE_OK;
  MOE_CUDA(cudaStreamWaitEvent(static_cast<cudaStream_t>(stream),
                               it->second.landed[it->second.last], 0));
  it->second.last = -1;
  return MOE_OK;
}

int32_t moe_layer_forward_host_release(void* workspace) {
  if (!workspace) return fail(MOE_ERR_INVALID_ARG, "workspace is null");
  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  auto it = g_pipes.find(workspace);
  if (it == g_pipes.end()) return MOE_OK;
  // an event whose recorded work is still pending is released once that
  // work completes; waits already enqueued on it are unaffected
  cudaError_t first = cudaSuccess;
  for (int i = 0; i < 2; ++i) {
    for (cudaEvent_t e : {it->second.copied[i], it->second.read[i], it->second.landed[i]}) {
      if (!e) continue;
      const cudaError_t r = cudaEventDestroy(e);
      if (first == cudaSuccess) first = r;
    }
  }
  g_pipes.erase(it);
  if (first != cudaSuccess) return cuda_fail(first, "cudaEventDestroy");
  return MOE_OK;
}

size_t moe_router_weight_split_bytes(const moe_config* cfg) {
  if (!cfg || cfg->E_routed < 1 || cfg->E_routed > 1024 || cfg->d_model < 64 ||
      cfg->d_model % 64)
    return 0;
  return 6ull * cfg->E_routed * cfg->d_model;
}

int32_t moe_split_router_weight(const moe_config* cfg, const float* W_r, void* W_split,
                                void* stream) {
  if (!cfg) return fail(MOE_ERR_INVALID_ARG, "cfg is null");
  if (cfg->E_routed < 1 || cfg->E_routed > 1024)
    return fail(MOE_ERR_INVALID_ARG, "E_routed not in [1, 1024]");
  if (cfg->d_model < 64 || cfg->d_model % 64)
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "d_model % 64 != 0");
  if (!W_r || !W_split) return fail(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(W_r) || !aligned16(W_split)) return fail(MOE_ERR_ALIGNMENT, "pointer not 16-byte aligned");
  const uint8_t* a = reinterpret_cast<const uint8_t*>(W_r);
  const uint8_t* b = static_cast<const uint8_t*>(W_split);
  const size_t na = 4ull * cfg->E_routed * cfg->d_model, nb = 6ull * cfg->E_routed * cfg->d_model;
  if (a < b + nb && b < a + na) return fail(MOE_ERR_INVALID_ARG, "W_r and W_split overlap");
  MOE_CUDA(launch_split_router_weight(W_r, cfg->E_routed, cfg->d_model,
                                      static_cast<__nv_bfloat16*>(W_split),
                                      static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int32_t moe_router_noalloc(const moe_config* cfg, int64_t T, const void* x, const float* W_r,
                           const float* bias, int32_t* topk_idx, float* topk_w, void* stream) {
  int32_t st = check_router_cfg(cfg, T);
  if (st != MOE_OK) return st;
  if (cfg->dtype != MOE_BF16 || cfg->d_model % 64)
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "moe_router_noalloc needs bf16 x and d_model % 64 == 0");
  if (!x || !W_r || !bias || !topk_idx || !topk_w) return fail(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(x) || !aligned16(W_r) || !aligned16(bias) || !aligned16(topk_idx) ||
      !aligned16(topk_w))
    return fail(MOE_ERR_ALIGNMENT, "pointer not 16-byte aligned");
  const int d = cfg->d_model, E = cfg->E_routed;
  // scratch: status word | split router weight (unless the caller passes
  // it) | partial logits
  const bool presplit = cfg->router_weight == MOE_ROUTER_WEIGHT_SPLIT;
  const int ksplit = noalloc_ksplit(T, d, E, presplit);
  if (ksplit == 0) {
    snprintf(g_detail, sizeof(g_detail),
             "moe_router_noalloc needs %zu bytes of scratch; its static scratch holds %zu",
             noalloc_need(T, d, E, presplit, 1), kNoAllocScratchBytes);
    return MOE_ERR_WORKSPACE;
  }
  const size_t split_off = kWsHeader;
  const size_t logits_off = split_off + (presplit ? 0 : round256(3ull * E * d * 2));
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = at<int>(scratch, 0);
  __nv_bfloat16* w_scratch = at<__nv_bfloat16>(scratch, split_off);
  const void* w_split = presplit ? static_cast<const void*>(W_r) : w_scratch;
  float* logits = at<float>(scratch, logits_off);
  // the array keeps the previous call's contents: only the status word must
  // start at zero (the split weight and every partial logit are rewritten)
  MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(int), s));
  if (!presplit) MOE_CUDA(launch_split_router_weight(W_r, E, d, w_scratch, s));
  if ((st = router_gemm(x, w_split, T, d, E, ksplit, logits, status, s)) != MOE_OK) return st;
  RouterArgs a;
  a.logits = logits;
  a.logit_parts = ksplit;
  a.logit_part_stride = T * E;
  a.bias = bias;
  a.T = T;
  a.d = d;
  a.E = E;
  a.K = cfg->K;
  a.G = cfg->n_group;
  a.Gk = cfg->topk_group;
  a.scale = cfg->routed_scaling_factor;
  a.norm = cfg->norm_topk_prob;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  MOE_CUDA(launch_router(a, s));
  return MOE_OK;
}

}  // extern "C"
