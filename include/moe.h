/*
 * fine_grained_sparse_gb300 -- C ABI of the fine-grained MoE layer forward
 * (Kimi-K2 / Kimi-K3 shape) on one GB300 (sm_103a).
 *
 * The layer, as the pages state it:
 *   - "Kimi K2 · Router · OpenModelAtlas", equations under "All 4 steps":
 *       z = x_ffn W_r,  s = sigmoid(z),  E_sel = [i in top_K(s + b)],
 *       G_i = 2.827 s_i E_sel_i / sum_j s_j E_sel_j
 *     and its MoEGate listing (fp32 gate GEMM, noaux_tc biased selection with
 *     n_group / topk_group group limiting, renormalisation + 1e-20,
 *     routed_scaling_factor).
 *   - "Kimi K2 MoE", sections 2-3: output = shared_expert(x) + sum over the
 *     selected experts of G_i f_i(x); SwiGLU experts of 3 d d_ff parameters.
 *   - "Kimi K3's router picks 16 of 896 experts", K3 table and the Stable
 *     LatentMoE paragraph: routed experts work on a 7168 -> 3584 projection
 *     of x, their combined output is projected back, 2 shared experts stay
 *     at 7168.
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers unless a parameter says "host".  All
 *     buffers are owned by the caller; no call allocates device memory.
 *   - Matrices are dense row-major.  Batch and sequence are flattened:
 *     T = B * seq_len rows.  Weights follow nn.Linear (out x in).
 *   - Element type of activations, expert weights and layer outputs is
 *     cfg->dtype: MOE_BF16 (tensor-core path, fp32 accumulation) or MOE_F32
 *     (CUDA-core path).  The router weight, bias, logits and gate weights
 *     are always fp32; expert indices are int32.
 *   - Every pointer must be 16-byte aligned (MOE_ERR_ALIGNMENT otherwise).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Argument errors are reported by the return value
 *     before anything is enqueued.  Errors found on the device (an expert
 *     index out of range, a bounded wait that expired) are written to the
 *     status word at the start of the workspace; read them with
 *     moe_get_device_status().  No exception crosses this interface.
 *   - The same workspace may not be used by two calls that run concurrently.
 *     moe_workspace_size(cfg, T) bytes suffice for every call below with
 *     that cfg and a row count <= T.
 */
#ifndef FINE_GRAINED_SPARSE_GB300_MOE_H
#define FINE_GRAINED_SPARSE_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,       /* null pointer, T < 1, K > E, ...        */
  MOE_ERR_UNSUPPORTED_SHAPE = 2, /* shape the chosen path does not cover   */
  MOE_ERR_ALIGNMENT = 3,         /* a pointer is not 16-byte aligned       */
  MOE_ERR_WORKSPACE = 4,         /* workspace missing or too small         */
  MOE_ERR_CUDA = 5,              /* a CUDA runtime/driver call failed      */
  MOE_ERR_TIMEOUT = 6,           /* a bounded device wait expired          */
  MOE_ERR_DEVICE_INDEX = 7       /* an expert index outside [0, E_routed)  */
} moe_status;

typedef enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Layer configuration.  Field names follow the gate config of the
 * "Kimi K2 · Router" MoEGate listing where it has one. */
typedef struct moe_config {
  int32_t d_model;      /* hidden_size d (7168 for K2 and K3)                  */
  int32_t d_ff;         /* routed expert intermediate width F (K2 2048, K3 3072)*/
  int32_t E_routed;     /* n_routed_experts E (K2 384, K3 896), <= 1024         */
  int32_t E_shared;     /* always-on shared experts S (K2 1, K3 2), may be 0    */
  int32_t d_ff_shared;  /* shared expert intermediate width F_s                 */
  int32_t K;            /* num_experts_per_tok (K2 8, K3 16), 1 <= K <= E       */
  int32_t n_group;      /* n_group G, E % G == 0, G <= 32                       */
  int32_t topk_group;   /* topk_group, 1 <= topk_group <= G                     */
  float routed_scaling_factor; /* 2.827                                         */
  int32_t norm_topk_prob;      /* renormalise the K weights when K > 1 (1)      */
  int32_t d_latent;     /* K3 latent width L (3584); 0 = K2 form (no projection)*/
  int32_t dtype;        /* moe_dtype of activations, expert weights, outputs    */
  int32_t weight_layout;/* moe_weight_layout of the expert, shared-expert and
                           latent-projection weights                           */
  int32_t router_weight;/* moe_router_weight_form of the W_r argument          */
} moe_config;

/* Forms of the router weight W_r passed to moe_router and the layer forwards.
 *   MOE_ROUTER_WEIGHT_F32: fp32 [E, d_model], as the model stores gate.weight.
 *   MOE_ROUTER_WEIGHT_SPLIT: the same weight as three bf16 terms, written
 *     once by moe_split_router_weight() (a load step, like the packing of the
 *     expert weights): bf16 [E, 3 d_model], row e = hi | mid | lo with
 *     hi = bf16(W_r[e]), mid = bf16(W_r[e] - hi), lo = bf16(W_r[e] - hi - mid)
 *     elementwise.  The tensor-core router GEMM reads it as it is instead of
 *     splitting W_r on every call; the logits are bit-identical.  Needs bf16
 *     x, d_model % 64 == 0 and a workspace (the CUDA-core path reads fp32);
 *     the pointer is still passed as the W_r argument. */
typedef enum moe_router_weight_form {
  MOE_ROUTER_WEIGHT_F32 = 0,
  MOE_ROUTER_WEIGHT_SPLIT = 1
} moe_router_weight_form;

/* Layouts of the weight matrices the expert GEMMs stream.
 *   MOE_WEIGHTS_NATURAL: bf16, row-major [G, O, K] as documented per argument.
 *   MOE_WEIGHTS_PACKED:  the same values rearranged by moe_pack_weights()
 *     into the order the tensor cores consume them, so that every pipeline
 *     stage of a GEMM is one contiguous bulk copy (see moe_pack_weights).
 *   MOE_WEIGHTS_PACKED_FP8: the routed and shared experts' W_gate_up and
 *     W_down are FP8 E4M3 with one fp32 multiplier per 128 x 128 block,
 *     packed by moe_pack_weights_fp8 (each bank one buffer: tiles, then the
 *     block-scale records); the latent projections stay bf16, packed by
 *     moe_pack_weights.  Needs bf16 activations and d_model, d_ff,
 *     d_ff_shared, d_latent multiples of 128.  ("Kimi K2 · Router ·
 *     OpenModelAtlas", Parameters: the checkpoint's tensors carry FP8 block
 *     scales.  The encoding, the block shape and the scale's type are not on
 *     the page; E4M3, 128 x 128 and an fp32 multiplier are this library's
 *     reading.)  Activations, H and the accumulation stay as in the bf16
 *     form; each weight enters the tensor cores as bf16(code value x scale). */
typedef enum moe_weight_layout {
  MOE_WEIGHTS_NATURAL = 0,
  MOE_WEIGHTS_PACKED = 1,
  MOE_WEIGHTS_PACKED_FP8 = 2
} moe_weight_layout;

/* Kinds of packed matrices. */
typedef enum moe_pack_kind {
  MOE_PACK_GATE_UP = 0, /* [G, 2F, K]: rows 0..F-1 gate, F..2F-1 up (W_gate_up) */
  MOE_PACK_PLAIN = 1    /* [G, O, K] (W_down, Ws_down, W_lat_down, W_lat_up)     */
} moe_pack_kind;

/*
 * Rearrange a bf16 weight bank into MOE_WEIGHTS_PACKED order (no call of the
 * forward pass needs it: it is a one-time load step).  src and dst are
 * device buffers of groups * rows * cols bf16 (the same size); they must not
 * overlap.  rows % 128 == 0 (MOE_PACK_GATE_UP: F = rows / 2, F % 64 == 0),
 * cols % 64 == 0.
 * Packed order, per group g: the 128-row tiles along O are taken in pairs
 * (u = 0, 1, ...; the last "pair" may hold one tile), and for each pair and
 * each 64-column step k of K the pair's tiles follow each other, each tile
 * 128 rows x 64 columns = 16 KB.  Inside a tile, row r occupies bytes
 * [128 r, 128 r + 128) and its 16-byte chunk c (columns 8c..8c+7) sits at
 * chunk position c XOR (r mod 8) -- the 128-byte swizzle of the tensor
 * cores' shared-memory operand layout.  For MOE_PACK_GATE_UP tile t of a
 * group holds, in rows 32 q + 16 h + i (q < 4, h < 2, i < 16), row
 * h * F + 64 t + 16 q + i of the source: the gate and up rows of 16 features
 * side by side. */
int32_t moe_pack_weights(int32_t kind, int64_t groups, int64_t rows, int64_t cols,
                         const void* src, void* dst, void* stream);

/* Bytes of a bank packed by moe_pack_weights_fp8:
 * groups * rows * cols (the codes) + groups * ceil(rows / 256) * (cols / 64)
 * * 16 (the records); -1 for sizes moe_pack_weights_fp8 rejects. */
int64_t moe_packed_fp8_bytes(int64_t groups, int64_t rows, int64_t cols);

/*
 * Rearrange an FP8 E4M3 weight bank and its block scales into
 * MOE_WEIGHTS_PACKED_FP8 order (a one-time load step, like
 * moe_pack_weights).
 *   codes  [groups, rows, cols] uint8, device, E4M3 codes (row-major)
 *   scales [groups, rows / 128, cols / 128] fp32, device: weight (g, r, c) =
 *          value(codes[g][r][c]) * scales[g][r / 128][c / 128]
 *   dst    device buffer of moe_packed_fp8_bytes(groups, rows, cols) bytes,
 *          not overlapping codes
 * rows % 128 == 0 and cols % 128 == 0 (MOE_PACK_GATE_UP: rows = 2 F, the
 * gate rows then the up rows).  codes and dst 16-byte aligned, scales 4-byte
 * aligned.  The tiles take the order and row interleave of moe_pack_weights
 * with one byte per element: a tile is 128 rows x 64 columns = 8 KB, row r
 * at bytes [64 r, 64 r + 64), its 8-byte chunk c (columns 8c..8c+7) at
 * chunk position c XOR (r mod 8).  After all tiles, one 16-byte record per
 * (group, tile pair u, k step), in that order: four fp32 scales, those of
 * tile 2u's rows (its gate rows, then its up rows; for MOE_PACK_PLAIN its one
 * row block twice) and of tile 2u + 1's (zero when the pair has one tile),
 * each at the k step's 128-column block.  Asynchronous on `stream`;
 * MOE_ERR_INVALID_ARG / UNSUPPORTED_SHAPE / ALIGNMENT before any launch. */
int32_t moe_pack_weights_fp8(int32_t kind, int64_t groups, int64_t rows, int64_t cols,
                             const void* codes, const float* scales, void* dst, void* stream);

/*
 * Self-test of the library's failure detection, with no counterpart on the
 * pages: every device wait of the library is a bounded mbarrier wait that
 * gives up after 2 s of %globaltimer, records MOE_ERR_TIMEOUT in the
 * workspace status word and lets its kernel return.  This enqueues one
 * such wait on a barrier that nothing arrives at (about 2 s on `stream`);
 * moe_get_device_status(workspace) then reads MOE_ERR_TIMEOUT, and the
 * context stays usable.  Returns MOE_ERR_WORKSPACE for a null workspace. */
int32_t moe_selftest_bounded_wait(void* workspace, void* stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t moe_version(void);

/* Number of kernels the library has enqueued in this process since it was
 * loaded, on every device, stream and thread; counted on the host when each
 * launch is issued (a launch that CUDA rejects is counted too).  The paper
 * has no counterpart: it lets a caller check how many kernels one call
 * enqueues.  Never fails. */
uint64_t moe_launch_count(void);

/* Static text for a moe_status value. */
const char* moe_status_string(int32_t status);

/* Text describing the most recent failing call on the calling thread (the
 * failed check or the CUDA error).  Valid until the next failing call on
 * that thread. */
const char* moe_last_error_detail(void);

/* Check cfg and T against the rules every call applies; makes no CUDA call.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED_SHAPE.  The
 * MOE_BF16 path needs d_model and d_latent to be multiples of 128 and
 * d_ff and d_ff_shared multiples of 64; MOE_F32 takes any positive sizes. */
int32_t moe_validate_config(const moe_config* cfg, int64_t T);

/* Bytes of device workspace any call below needs for (cfg, T); 0 if the
 * configuration is invalid.  Makes no CUDA call. */
size_t moe_workspace_size(const moe_config* cfg, int64_t T);

/* Read and clear the device status word of `workspace` (synchronises
 * `stream` first).  Returns MOE_OK or the first device-side error recorded
 * since the last read. */
int32_t moe_get_device_status(void* workspace, void* stream);

/* Bytes of the split router weight: 6 * E_routed * d_model; 0 for a NULL
 * cfg or sizes moe_split_router_weight rejects. */
size_t moe_router_weight_split_bytes(const moe_config* cfg);

/*
 * Write the MOE_ROUTER_WEIGHT_SPLIT form of an fp32 router weight (see
 * moe_router_weight_form): W_r fp32 [E, d_model] in, W_split bf16
 * [E, 3 d_model] out, both device buffers, 16-byte aligned, not overlapping.
 * Needs 1 <= E_routed <= 1024 and d_model % 64 == 0.  Asynchronous on stream. */
int32_t moe_split_router_weight(const moe_config* cfg, const float* W_r, void* W_split,
                                void* stream);

/*
 * Router, all four steps ("Kimi K2 · Router", "All 4 steps"; MoEGate):
 *   z = x W_r^T in fp32 (x upcast from cfg->dtype), s = sigmoid(z),
 *   c = s + bias, optional group limiting (G > 1: keep the topk_group groups
 *   with the largest sum of their two best c, set c of every other expert to
 *   0.0), then the K largest c.
 *   x        [T, d_model]  cfg->dtype
 *   W_r      [E, d_model]  fp32 (gate.weight), or [E, 3 d_model] bf16 when
 *                          cfg->router_weight is MOE_ROUTER_WEIGHT_SPLIT
 *   bias     [E]           fp32 (e_score_correction_bias)
 *   topk_idx [T, K] int32  out: selected experts, ordered by c descending,
 *                          equal c by smaller expert index first
 *   topk_w   [T, K] fp32   out: routed_scaling_factor * s_i / (sum s + 1e-20)
 *                          (no renormalisation when K == 1 or
 *                          norm_topk_prob == 0)
 * The selection is decided on fp32 values with s rounded once from the
 * exact sigmoid of the fp32 logit.
 *   workspace: NULL, or moe_workspace_size(cfg, T) bytes (ws_bytes).  With a
 *   workspace and bf16 x (d_model % 64 == 0) the logits come from a
 *   tensor-core GEMM against a three-way bf16 split of W_r (hi + mid + lo
 *   carries W_r to ~2^-24 relative; bf16 x bf16 products are exact and the
 *   sums fp32); otherwise from a fused fp32 CUDA-core kernel. */
int32_t moe_router(const moe_config* cfg, int64_t T, const void* x, const float* W_r,
                   const float* bias, int32_t* topk_idx, float* topk_w, void* workspace,
                   size_t ws_bytes, void* stream);

/* Router steps 2-4 from given fp32 logits z [T, E] (the parity entry point:
 * identical logits give identical expert indices on every implementation
 * that follows the rule above).  Other arguments as moe_router. */
int32_t moe_router_from_logits(const moe_config* cfg, int64_t T, const float* logits,
                               const float* bias, int32_t* topk_idx, float* topk_w,
                               void* stream);

/*
 * Dense gate matrix ("Kimi K2 · Router · OpenModelAtlas": "out: G [B batch,
 * T positions, 384 experts]"; its Explanation: G spreads each position's K
 * weights over all experts, zero for the others):
 *   G[t, e] = topk_w[t, k] where topk_idx[t, k] == e, else 0.
 *   topk_idx [T, K] int32, topk_w [T, K] fp32 in (moe_router's outputs);
 *   G [T, E] fp32 out, every entry written.  Indices outside [0, E) are
 *   ignored.  Needs no workspace. */
int32_t moe_dense_gates(const moe_config* cfg, int64_t T, const int32_t* topk_idx,
                        const float* topk_w, float* G, void* stream);

/*
 * One aux-loss-free update of the selection bias ("Kimi K2 MoE",
 * "Routing-distribution diagnostics": DeepSeek V3's schedule, gamma = 1e-3,
 * sign-only) from one batch's per-expert loads:
 *   bias[e] += gamma * sign(T*K/E - counts[e])
 * the comparison with the mean load made in integers (E*counts[e] against
 * T*K), the step one fp32 addition.  counts [E] int32 (moe_permute's output
 * for that batch), bias [E] fp32 updated in place.  Needs no workspace. */
int32_t moe_update_bias(const moe_config* cfg, int64_t T, const int32_t* counts, float gamma,
                        float* bias, void* stream);

/*
 * One Quantile Balancing update of the selection bias ("Kimi K3's router
 * picks 16 of 896 experts", "The router trains inside the main run": a
 * per-expert threshold at which the expert receives its target number of
 * tokens, from a quantile of the router scores, updates the bias; training
 * only).  The page gives no formula; this library's reading:
 *   target load n* = T K / E; s = sigmoid(z) rounded once to fp32;
 *   theta[e] = the ceil(n*)-th largest s[t, e] over the batch (an order
 *     statistic: the (1 - K/E) quantile of expert e's scores);
 *   tau = (sum_e theta[e]) / E, summed in fp64 in expert order;
 *   bias[e] = fp32(b + rate ((tau - theta[e]) - b)), b = bias[e], each step
 *     an fp64 operation in that order, so that rate = 1 puts every expert's
 *     biased score at its threshold on the common cut-off tau.
 *   logits [T, E] fp32 in (the router GEMM's z for the batch), rate in
 *   [0, 1], theta [E] fp32 out, bias [E] fp32 updated in place.  Needs no
 *   workspace. */
int32_t moe_quantile_bias_update(const moe_config* cfg, int64_t T, const float* logits, float rate,
                                 float* theta, float* bias, void* stream);

/*
 * Dispatch: group the T*K (token, slot) pairs by expert ("Kimi K2 MoE",
 * section 3, dispatch_and_combine; its body is not given).  Order: expert
 * major, ascending token index within an expert.  Pair j = t * K + k.
 *   topk_idx [T, K] int32  in
 *   counts   [E]    int32  out: pairs routed to each expert
 *   offsets  [E+1]  int32  out: exclusive prefix sum of counts
 *   perm     [T*K]  int32  out: perm[offsets[e] + r] = j of the r-th pair of e
 *   inv      [T*K]  int32  out: inv[j] = the slot of pair j
 * An index outside [0, E) records MOE_ERR_DEVICE_INDEX in the workspace
 * status; its pair is left out of counts and perm, and its inv entry is -1. */
int32_t moe_permute(const moe_config* cfg, int64_t T, const int32_t* topk_idx,
                    int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                    void* workspace, size_t ws_bytes, void* stream);

/*
 * Grouped SwiGLU experts ("Kimi K2 MoE", section 2: SwiGLU experts,
 * 3 d d_ff parameters each): for every slot r of expert e,
 *   Y[r] = w_r * W_down[e] (SiLU(W_gate[e] u) * (W_up[e] u)),  u = x_e[perm[r] / K]
 * with w_r = topk_w[perm[r]] (or 1 when topk_w is NULL); and for every shared
 * expert s and token t, Y_shared[s, t] = f_s(x_shared[t]) with weight 1.
 *   x_e        [T, d_e]        rows the routed experts read (d_e = d_latent if
 *                              set, else d_model)
 *   offsets    [E+1], perm [T*K] from moe_permute
 *   topk_w     [T, K] fp32 or NULL
 *   W_gate_up  [E, 2F, d_e]    rows 0..F-1 = W_gate, rows F..2F-1 = W_up
 *   W_down     [E, d_e, F]
 *   x_shared   [T, d_model] or NULL (then the shared arguments are ignored)
 *   Ws_gate_up [S, 2F_s, d_model], Ws_down [S, d_model, F_s]
 *   Y          [T*K, d_e]      out, slot order
 *   Y_shared   [S, T, d_model] out (may be NULL when x_shared is NULL)
 * Intermediates (the gathered rows and SwiGLU activations, rounded to
 * cfg->dtype) live in the workspace. */
int32_t moe_grouped_swiglu(const moe_config* cfg, int64_t T, const void* x_e,
                           const int32_t* offsets, const int32_t* perm, const float* topk_w,
                           const void* W_gate_up, const void* W_down, const void* x_shared,
                           const void* Ws_gate_up, const void* Ws_down, void* Y, void* Y_shared,
                           void* workspace, size_t ws_bytes, void* stream);

/*
 * Weighted combine ("Kimi K2 MoE", section 3: shared_expert(x) + routed;
 * the routed part is the gate-weighted sum of the selected experts):
 *   y[t] = sum_{k=0..K-1} w[t, k] Y[inv[t*K + k]] + sum_s Y_shared[s, t]
 * summed in fp32 in that fixed order, w[t, k] = topk_w[t*K + k], or 1 when
 * topk_w is NULL (the weights are already in Y: moe_grouped_swiglu was
 * given topk_w).  Passing topk_w here and NULL to moe_grouped_swiglu is
 * what moe_layer_forward does: the weight is applied in fp32 after Y was
 * rounded to cfg->dtype, instead of before.
 *   Y        [T*K, D], inv [T*K], topk_w [T, K] fp32 or NULL,
 *   Y_shared [S, T, D] or NULL, y [T, D] out; D = d_e.  For the K3 form
 *   (d_latent != 0) Y_shared must be NULL: the routed sum is in latent space.
 * An inv entry outside [0, T*K) -- moe_permute writes -1 for a pair whose
 * expert index it rejected, and reports MOE_ERR_DEVICE_INDEX itself --
 * adds nothing to y[t]; no read leaves Y. */
int32_t moe_combine(const moe_config* cfg, int64_t T, const void* Y, const int32_t* inv,
                    const float* topk_w, const void* Y_shared, void* y, void* stream);

/*
 * Plain projection y = x W^T (+ add) for the K3 latent maps ("Kimi K3's
 * router picks 16 of 896 experts", Stable LatentMoE: 7168 -> 3584 before
 * the routed experts, 3584 -> 7168 after their combine).  MOE_BF16 only.
 *   x [T, in] bf16, W [out, in] bf16, add [T, out] bf16 or NULL, y [T, out].
 * in and out must be multiples of 128. */
int32_t moe_linear(int64_t T, int32_t in_features, int32_t out_features, const void* x,
                   const void* W, const void* add, void* y, void* workspace, size_t ws_bytes,
                   void* stream);

/*
 * The whole layer forward, one stream:
 *   K2 form: y = sum_s f_s(x) + sum_k w_k f_{idx_k}(x)
 *   K3 form: y = sum_s f_s(x) + W_lat_up (sum_k w_k f_{idx_k}(W_lat_down x))
 * (router on x in both forms).
 *   x [T, d], W_r [E, d] fp32, bias [E] fp32, W_gate_up/W_down as in
 *   moe_grouped_swiglu, Ws_gate_up/Ws_down (NULL when E_shared == 0),
 *   W_lat_down [L, d] and W_lat_up [d, L] (NULL unless d_latent != 0),
 *   y [T, d] out.
 *   topk_idx_out [T, K], topk_w_out [T, K], counts_out [E]: optional copies
 *   of the routing (NULL to skip).
 *   stage_events: NULL, or MOE_STAGE_COUNT + 1 cudaEvent_t handles recorded
 *   on `stream` before each stage and after the last (router, dispatch,
 *   expert gate/up, expert down, combine and projections); a NULL entry is
 *   not recorded.  A recorded event keeps the kernels on its two sides from
 *   overlapping (the library launches successive kernels so that the next
 *   one's set-up runs while the previous one drains). */
#define MOE_STAGE_COUNT 5
int32_t moe_layer_forward(const moe_config* cfg, int64_t T, const void* x, const float* W_r,
                          const float* bias, const void* W_gate_up, const void* W_down,
                          const void* Ws_gate_up, const void* Ws_down, const void* W_lat_down,
                          const void* W_lat_up, void* y, int32_t* topk_idx_out,
                          float* topk_w_out, int32_t* counts_out, void* workspace,
                          size_t ws_bytes, void* const* stage_events, void* stream);

/*
 * moe_layer_forward with x and y in HOST memory (pinned for asynchronous
 * copies; pageable memory works but the copies then block).  The call
 * enqueues the host-to-device copy of x into the workspace, the forward and
 * the device-to-host copy of y, and returns without waiting: y_host is valid
 * after `stream` has been synchronised.  Weights stay device pointers.
 * Successive calls on one workspace are pipelined: x is copied on a copy
 * stream of the library into one of two staging buffers, alternating, so
 * the copy for one call overlaps the forward of the call before it.  That
 * copy therefore does not wait for work enqueued earlier on `stream`: x_host
 * must hold its values when the call is made (host writes, or device work
 * already synchronised).  When y_host is pinned host memory mapped into the
 * current device's address space (cudaHostAlloc / cudaHostRegister on a
 * unified-addressing system) and 16-byte aligned, the layer's last kernel
 * writes y straight into it over the host link instead of staging y in the
 * workspace and copying it, so no copy stands between this call's forward and
 * the next one on `stream`; y_host is valid at the same point either way. */
int32_t moe_layer_forward_host(const moe_config* cfg, int64_t T, const void* x_host,
                               const float* W_r, const float* bias, const void* W_gate_up,
                               const void* W_down, const void* Ws_gate_up, const void* Ws_down,
                               const void* W_lat_down, const void* W_lat_up, void* y_host,
                               void* workspace, size_t ws_bytes, void* stream);

/*
 * moe_layer_forward_host for a stream of batches, with the copy of y out of
 * the device overlapped with the next batch's forward.  Arguments, errors and
 * the handling of x are those of moe_layer_forward_host; y is always staged
 * in the workspace (one of two buffers, alternating with x's) and copied to
 * y_host on a second copy stream of the library once this call's forward has
 * finished.  y_host of this call is therefore valid once `stream` has passed
 * the NEXT moe_layer_forward_host_pipelined call on the same workspace (that
 * call makes `stream` wait for this copy after enqueueing its own forward),
 * or moe_layer_forward_host_flush(workspace, stream); until then the caller
 * must neither read nor reuse y_host.  Successive calls may pass the same
 * y_host: its copies are made in call order.  No counterpart on the pages:
 * it keeps the host link (about 0.2 TB/s each way on one GB300) off the
 * critical path of a batch stream. */
int32_t moe_layer_forward_host_pipelined(const moe_config* cfg, int64_t T, const void* x_host,
                                         const float* W_r, const float* bias,
                                         const void* W_gate_up, const void* W_down,
                                         const void* Ws_gate_up, const void* Ws_down,
                                         const void* W_lat_down, const void* W_lat_up,
                                         void* y_host, void* workspace, size_t ws_bytes,
                                         void* stream);

/*
 * Make `stream` wait for the copy of y of the latest
 * moe_layer_forward_host_pipelined call on `workspace` (after this, a
 * synchronisation of `stream` leaves that y in its y_host).  Nothing pending
 * (or a workspace never used by that call): no effect.  MOE_ERR_INVALID_ARG
 * for a NULL workspace; MOE_ERR_CUDA if the wait cannot be enqueued. */
int32_t moe_layer_forward_host_flush(void* workspace, void* stream);

/*
 * Release the library's per-workspace state of moe_layer_forward_host and
 * moe_layer_forward_host_pipelined: the six CUDA events that order their
 * staging copies, kept from the first host-buffer call on `workspace` until
 * this call (the paper has no
 * counterpart; it bounds what a caller that cycles through workspaces
 * holds).  Work already enqueued is not waited for.  A later host-buffer
 * call on the same workspace starts afresh; it must not be enqueued before
 * the earlier calls on that workspace have completed (their staging buffers
 * are no longer tracked).  A workspace without such state is accepted.
 * MOE_ERR_INVALID_ARG for a NULL workspace. */
int32_t moe_layer_forward_host_release(void* workspace);

/*
 * moe_router without a caller-provided workspace.  This entry point has no
 * counterpart on the pages: it exists for callers that cannot allocate
 * device memory when they route tokens -- for example code running inside
 * an allocator-free runtime or a plugin interface that hands over only its
 * input and output buffers.  It computes what moe_router computes with a
 * workspace and bf16 x (the split-bf16 tensor-core router), taking its
 * scratch (the three-way split of W_r and the partial logits) from a static
 * device array of 64 MiB that every GPU loading this library holds until
 * the process exits; it calls no allocating routine.
 *   Arguments as moe_router.  cfg->dtype must be MOE_BF16 and d_model a
 *   multiple of 64 (MOE_ERR_UNSUPPORTED_SHAPE otherwise).
 *   Scratch for P K parts: 256 + S + 4 T E P bytes (each term rounded up
 *   to 256), S = 6 E d, or 0 when cfg->router_weight is
 *   MOE_ROUTER_WEIGHT_SPLIT.  P is moe_router's own count of K parts when
 *   that fits the array; otherwise the largest smaller count that fits, and
 *   the logits are then summed in a different grouping than moe_router's:
 *   they may differ from it in the last bit, and so may a selection whose
 *   deciding margin is of that size.  The call is rejected with
 *   MOE_ERR_WORKSPACE, before anything is enqueued, only when even P = 1
 *   does not fit: 256 + S + 4 T E > 64 MiB, which holds for every T above a
 *   bound (K2 router, E = 384, d = 7168: T > 32938, or T > 43690 with the
 *   split weight; K3, E = 896: T > 7972, or T > 18724 with the split
 *   weight).
 *   The call looks up the array's device address in the current context
 *   the first time it runs in that context (again after the context was
 *   destroyed and created anew); make that first call before any stream
 *   capture.  All calls on a device share the array, which keeps the
 *   previous call's contents: calls whose work overlaps on the GPU (other
 *   streams, other threads) race and must be serialised by the caller.  A
 *   bounded device wait that expires leaves the outputs incomplete and is
 *   not reported by this entry point. */
int32_t moe_router_noalloc(const moe_config* cfg, int64_t T, const void* x, const float* W_r,
                           const float* bias, int32_t* topk_idx, float* topk_w, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FINE_GRAINED_SPARSE_GB300_MOE_H */
