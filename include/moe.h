/*
 * moe.h - C ABI of the GB300 (sm_103a) top-k routed Mixture-of-Experts
 * feed-forward layer forward pass.
 *
 * The layer, step by step (sources are the page titles and sections that define
 * each operation):
 *
 *   route        router projection of every token to one score per expert with a
 *                fixed reduction order, FP32 softmax, top-k, left-to-right
 *                renormalisation, experts sorted by probability
 *                ("0 train-infer mismatch for open-weight MoE RL", section
 *                 "Mixture-of-experts layers / The router")
 *   load stats   routed-token count per expert and its exclusive prefix sum
 *                ("RoutePack", section 2.2 "Routing replay", Eq. 1)
 *   permute      dispatch: stable permutation of token rows into expert-contiguous
 *                rows ("FlexFloor", Figure 1: token -> dispatch -> experts;
 *                 "RoutePack", section 2.3: a rank's local experts run as one
 *                 grouped operation)
 *   expert FFN   grouped SwiGLU expert GEMMs with one BF16 rounding of the
 *                intermediate ("0 train-infer mismatch", section "SwiGLU: rounding
 *                after the multiply")
 *   combine      per token, the routing slots accumulated in FP32 in slot order,
 *                rounded once to BF16 ("0 train-infer mismatch", sections
 *                "Sharding the experts" and "The experts: keeping the route weight
 *                inside the accumulator")
 *
 * Every token is routed to exactly k distinct experts; nothing is dropped
 * ("HARTS", section "MoE semantics without expert expansion": deterministic,
 * no-token-drop top-k routing).
 *
 * Conventions for every call
 * --------------------------
 *  - All tensor pointers are DEVICE pointers, owned by the caller, 16-byte
 *    aligned, dense and row-major.  bf16 tensors are passed as void*.  The
 *    library never allocates, frees or keeps device memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls are stream-ordered and asynchronous: they return once the work is
 *    enqueued.
 *  - Host-side validation happens before anything is launched; a non-OK status
 *    means nothing was enqueued, except MOE_ERR_CUDA, which reports a failed
 *    launch or runtime call.
 *  - Kernels that read indices or offsets from memory check them against the
 *    dimensions.  A failed check skips the offending access and records
 *    MOE_ERR_DEVICE_CHECK in the workspace status word; a bounded device-side
 *    wait that runs out records MOE_ERR_TIMEOUT.  Read (and clear) it with
 *    moe_read_device_status.  Calls without a workspace argument (moe_route,
 *    moe_combine) take no status word: moe_combine skips out-of-range rows.
 *  - Dimensions (moe_dims): T tokens (T >= 0; T = 0 is a no-op), H hidden size,
 *    E experts, k experts per token, I expert intermediate size.
 *    Limits: 1 <= E <= 256, 1 <= k <= min(E, 16), H and I multiples of 128,
 *    H <= 16384, I <= 16384, T*k < 2^31.
 *  - Batch invariance: no kernel's reduction order, tile shape or launch shape
 *    depends on T, so a token's output bytes do not depend on which batch it
 *    is in.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer where one is required, bad dimension */
  MOE_ERR_UNSUPPORTED = 2,  /* dimension outside the limits above, or no sm_103a device */
  MOE_ERR_MISALIGNED = 3,   /* pointer not 16-byte aligned (workspace: 256-byte) */
  MOE_ERR_WORKSPACE = 4,    /* workspace or packed-weight buffer too small */
  MOE_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 6,      /* device: a bounded wait ran out (read via moe_read_device_status) */
  MOE_ERR_DEVICE_CHECK = 7  /* device: an index or offset read from memory was out of range */
} moe_status;

typedef struct {
  int32_t T, H, E, k, I;
} moe_dims;

/* Router variants ("0 train-infer mismatch for open-weight MoE RL"). */
typedef enum {
  /* FP32 softmax over the logits (plus the optional per-expert bias), top-k by
   * logit, ties to the lower expert, left-to-right renormalisation
   * (section "The router"). */
  MOE_ROUTER_SOFTMAX = 0,
  /* GLM's rule (section "Choosing GLM's eight experts"): scores s = sigmoid(l);
   * the FP32 correction bias is added only to choose the top k (ties to the lower
   * expert); the weights are the chosen pre-bias scores divided by their sum
   * (added left to right, FP32).  The exponential is Cody & Waite reduction with a
   * degree-7 Taylor polynomial in FP32 fused multiply-adds, so the choice is
   * reproducible bit for bit on any implementation of the same steps. */
  MOE_ROUTER_SIGMOID_BIAS_SELECT = 1
} moe_router_kind;

typedef struct {
  int32_t kind;          /* moe_router_kind */
  int32_t weights_bf16;  /* nonzero: every routing weight is rounded to bf16 (section
                            "The router": the renormalised weights are cast to BF16) */
  float route_scale;     /* > 0: multiplies every routing weight in FP32 inside the
                            combine (GLM applies 2.5 inside the expert kernel); 1 = none */
} moe_router_opts;

/* Bytes of device workspace that every call taking a workspace needs for these
 * dimensions (the full layer's need; each step uses a part of the same layout).
 * The workspace must be 256-byte aligned and its first 256 bytes (the status
 * word) zero before first use; moe_read_device_status clears them.  The rest is
 * scratch.  Two calls in flight at once must not share a workspace. */
size_t moe_workspace_bytes(moe_dims d);

/* Bytes of the packed expert-weight buffer written by moe_prepack_expert_weights:
 * E * 3 * H * I bf16 values. */
size_t moe_packed_weight_bytes(moe_dims d);

/* Step: router.  For every token t:
 *   l[t,e] = ((sum over h = 0..H-1, as an FP32 fused multiply-add chain from 0,
 *              of float(x[t,h]) * w_router[h,e])) + bias[e]
 *   p = softmax(l) in FP32; the k experts with the largest l (ties: lower expert
 *   index first) become slots j = 0..k-1 in that order; S = sum of their p added
 *   left to right; topk_w[t,j] = p[e_j] / S.
 *   x        [T, H] bf16
 *   w_router [H, E] fp32
 *   bias     [E] fp32 or NULL (a per-expert popularity bias added to the logits)
 *   topk_idx [T, k] int32 out (expert ids), topk_w [T, k] fp32 out.
 * The indices are bit-reproducible against a CPU FMA chain; the weights agree
 * with it to a few FP32 ulp (the exponential differs between math libraries). */
moe_status moe_route(const void* x, const float* w_router, const float* bias, moe_dims d,
                     int32_t* topk_idx, float* topk_w, void* stream);

/* moe_route with a router variant (opts NULL: softmax, FP32 weights).
 * opts->route_scale is not used here (it belongs to the combine).  An unknown
 * kind or a scale that is not a positive finite number: MOE_ERR_INVALID_ARG. */
moe_status moe_route_ex(const void* x, const float* w_router, const float* bias,
                        const moe_router_opts* opts, moe_dims d, int32_t* topk_idx, float* topk_w,
                        void* stream);

/* Step: per-expert load.  counts[e] = number of (t, j) with topk_idx[t,j] = e;
 * offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e] (so offsets[E] = T*k).
 *   topk_idx [T, k] int32 in; counts [E] int32 out; offsets [E+1] int32 out.
 * Out-of-range ids are skipped and flagged (MOE_ERR_DEVICE_CHECK). */
moe_status moe_load_stats(const int32_t* topk_idx, moe_dims d, int32_t* counts, int32_t* offsets,
                          void* workspace, size_t ws_bytes, void* stream);

/* Host-side summary of counts already copied to the host: imbalance
 * max/mean - 1 ("HARTS", Eq. 23, taken over experts) and the coefficient of
 * variation std/mean ("RoutePack", Eq. 22 form, one layer, over experts).
 * Either output pointer may be NULL. */
moe_status moe_load_summary_host(const int32_t* counts_host, int32_t E, double* imbalance,
                                 double* cv);

/* moe_load_stats with two options:
 *   slot_of_expert [E] (device, or NULL): "RoutePack" section 3.3 / Figure 4, the
 *     dispatcher's map from the router's logical expert e to physical slot
 *     slot_of_expert[e] (a permutation of 0..E-1, e.g. from
 *     moe_lpt_placement_host).  counts and offsets are then indexed by physical
 *     slot, the grouping the expert FFN runs in when its weights were packed with
 *     the same map (moe_prepack_expert_weights_ex).  A map that is not a
 *     permutation yields repeated slots within a token: flagged
 *     (MOE_ERR_DEVICE_CHECK), rows stay inside [0, T*k).
 *   q [T] int32 (device) and weighted_counts [E] int64 (device), both or neither:
 *     "HARTS" Eq. 20, a compact row t standing for q[t] >= 0 tokens counts q[t]
 *     times: weighted_counts[e] = sum of q[t] over the (t, j) routed to logical
 *     expert e (integer atomics, exact).  Routing and compute are unaffected. */
moe_status moe_load_stats_ex(const int32_t* topk_idx, const int32_t* slot_of_expert,
                             const int32_t* q, moe_dims d, int32_t* counts, int32_t* offsets,
                             int64_t* weighted_counts, void* workspace, size_t ws_bytes,
                             void* stream);

/* Host: "RoutePack" Algorithm 1, layer-local LPT expert placement.  Experts in
 * order of (load descending, index ascending) each go to the least-loaded of the
 * P ranks that still has a free slot (ties: lower rank), into that rank's next
 * slot: slot_of_expert[e] = p * (E/P) + n_p.  rank_loads [P] (optional) receives
 * the rank loads G_p of Eq. 10.  E must be a multiple of P and at most 256.
 * All pointers are host pointers. */
moe_status moe_lpt_placement_host(const int64_t* loads, int32_t E, int32_t P,
                                  int32_t* slot_of_expert, int64_t* rank_loads);

/* Host: balance of P rank loads ("RoutePack" Eq. 22, one layer: population
 * std/mean; Eq. 23 for one row, layer and shard: mean/max).  Outputs may be NULL. */
moe_status moe_rank_load_summary_host(const int64_t* rank_loads, int32_t P, double* cv,
                                      double* eta_ep);

/* moe_permute with the dispatcher's logical -> physical slot map (NULL: identity):
 * rows are grouped by physical slot, stable within a slot; offsets are indexed
 * by slot (as moe_load_stats_ex writes them with the same map). */
moe_status moe_permute_ex(const void* x, const int32_t* topk_idx, const int32_t* slot_of_expert,
                          const int32_t* offsets, moe_dims d, void* x_perm, int32_t* row_of_slot,
                          int32_t* slot_of_row, void* workspace, size_t ws_bytes, void* stream);

/* Step: dispatch.  Stable permutation into expert-contiguous rows: slot
 * s = t*k + j with expert e goes to row
 *   r = offsets[e] + #{ t' < t : token t' chose e },
 * row_of_slot[s] = r, slot_of_row[r] = s, and x_perm[r, :] = x[t, :] (bytes).
 *   x [T, H] bf16; topk_idx [T, k]; offsets [E+1] (as moe_load_stats writes them)
 *   x_perm [T*k, H] bf16 out; row_of_slot [T*k] out; slot_of_row [T*k] out.
 * Offsets that disagree with topk_idx are flagged (MOE_ERR_DEVICE_CHECK) and
 * rows that would fall outside [0, T*k) are not written. */
moe_status moe_permute(const void* x, const int32_t* topk_idx, const int32_t* offsets, moe_dims d,
                       void* x_perm, int32_t* row_of_slot, int32_t* slot_of_row, void* workspace,
                       size_t ws_bytes, void* stream);

/* One-time weight preparation (not part of a forward).  Reads the logical
 * layouts and writes the K-major tiles the grouped GEMMs stream with TMA:
 *   w_gate [E, H, I] bf16, w_up [E, H, I] bf16, w_down [E, I, H] bf16
 *   packed: moe_packed_weight_bytes(d) bytes, 16-byte aligned. */
moe_status moe_prepack_expert_weights(const void* w_gate, const void* w_up, const void* w_down,
                                      moe_dims d, void* packed, size_t packed_bytes, void* stream);

/* moe_prepack_expert_weights with expert e packed into physical slot
 * slot_of_expert[e] (device, or NULL for the identity): "RoutePack" Figure 4,
 * each expert's weights materialised in its destination slot.  Slots outside
 * [0, E) are not written. */
moe_status moe_prepack_expert_weights_ex(const void* w_gate, const void* w_up,
                                         const void* w_down, const int32_t* slot_of_expert,
                                         moe_dims d, void* packed, size_t packed_bytes,
                                         void* stream);

/* Step: grouped SwiGLU experts.  For each expert e and each row r in
 * [offsets[e], offsets[e+1]):
 *   g = x_perm[r] . W_gate[e], u = x_perm[r] . W_up[e]   (BF16 products, FP32 accumulation)
 *   h[r] = bf16(silu(g) * u)                             (the only rounding)
 *   y[r] = h[r] . W_down[e]                              (FP32 accumulation, FP32 output)
 *   x_perm [T*k, H] bf16; offsets [E+1] int32; packed weights from
 *   moe_prepack_expert_weights; y [T*k, H] fp32 out.  h lives in the workspace.
 * Offsets that are not a non-decreasing sequence from 0 to T*k are flagged
 * (MOE_ERR_DEVICE_CHECK) and no row is written. */
moe_status moe_expert_ffn(const void* x_perm, const int32_t* offsets, const void* packed_weights,
                          moe_dims d, float* y, void* workspace, size_t ws_bytes, void* stream);

/* Which form of the grouped GEMMs moe_expert_ffn (and every layer call) runs for
 * these dims on the current device: 0 = tile kernels (128 token rows per MMA),
 * 1 = swapped kernels (128 weight rows per MMA, up to 64 token rows on N; chosen
 * while experts hold at most 8 rows on average and the gate/up work units number
 * at most four per SM).  Both forms give the same bits for every row.
 * Negative: minus a moe_status (invalid dims, no usable device). */
int moe_expert_ffn_form(moe_dims d);

/* Step: combine.  out[t, c] = bf16(acc), acc = 0, then for j = 0..k-1:
 *   acc = fmaf(topk_w[t,j], y[row_of_slot[t*k+j], c], acc).
 *   y [T*k, H] fp32; topk_w [T, k] fp32; row_of_slot [T*k] int32; out [T, H] bf16.
 * Rows outside [0, T*k) contribute nothing. */
moe_status moe_combine(const float* y, const float* topk_w, const int32_t* row_of_slot, moe_dims d,
                       void* out, void* stream);

/* moe_combine with every routing weight multiplied by route_scale (FP32, one
 * rounding) before the slot-order chain; route_scale = 1 is moe_combine. */
moe_status moe_combine_ex(const float* y, const float* topk_w, const int32_t* row_of_slot,
                          float route_scale, moe_dims d, void* out, void* stream);

/* Combine as G expert ranks would do it, without the exchange ("0 train-infer
 * mismatch for open-weight MoE RL", section "Sharding the experts").  owner [E]
 * int32 (device) gives the rank in [0, G) that owns each logical expert; a slot
 * whose expert has an owner outside [0, G) contributes to no rank.  For token t,
 * column c and rank g = 0..G-1:
 *   acc = 0; for j = 0..k-1:
 *     acc = fmaf(route_scale * topk_w[t,j], owner[topk_idx[t,j]] == g ? y[row, c] : 0.0f, acc)
 *   acc = acc + shared[g, t, c]          (if shared != NULL: [G, T, H] fp32, e.g.
 *                                         from moe_shared_expert)
 *   partial[g, t, c] = bf16(acc)         (round to nearest even)
 * out[t, c] = bf16 of the FP64 pairwise tree over partial[0..G-1, t, c] (below).
 *   partials [G, T, H] bf16 is optional (NULL: kept in registers only).
 *   1 <= G <= 16; route_scale > 0 and finite.  Other arguments as moe_combine. */
moe_status moe_combine_sharded(const float* y, const float* topk_w, const int32_t* topk_idx,
                               const int32_t* row_of_slot, const int32_t* owner, int32_t G,
                               float route_scale, const float* shared, moe_dims d, void* partials,
                               void* out, void* stream);

/* Shared expert ("0 train-infer mismatch for open-weight MoE RL", section
 * "Mixture-of-experts layers": the fixed-K projections and SwiGLU of the dense
 * FFN; each expert rank holds one shard of it).  W_gate, W_up [H, Is] and W_down
 * [Is, H] bf16, row-major.  Rank g's shard is intermediate columns
 * [g*Is/G, (g+1)*Is/G) of W_gate and W_up and the same rows of W_down.
 * Limits: Is % G == 0, (Is / G) % 128 == 0, H % 128 == 0, both <= 16384. */
size_t moe_shared_packed_bytes(int32_t H, int32_t Is);

/* One-time packing of the shared expert's G shards into the K-major layout of
 * the grouped GEMMs (packed: moe_shared_packed_bytes, 16-byte aligned). */
moe_status moe_prepack_shared_expert(const void* w_gate, const void* w_up, const void* w_down,
                                     int32_t H, int32_t Is, int32_t G, void* packed,
                                     size_t packed_bytes, void* stream);

/* Workspace of moe_shared_expert (0: dimensions outside the limits). */
size_t moe_shared_expert_workspace_bytes(int32_t T, int32_t H, int32_t Is, int32_t G);

/* shared_out[g, t, :] = rank g's shard of the shared expert for token t:
 *   gate = x[t] . W_gate[:, shard g], up = x[t] . W_up[:, shard g]   (FP32 accumulation)
 *   h = bf16(silu(gate) * up)                                       (the only rounding)
 *   shared_out[g, t] = h . W_down[shard g, :]                       (FP32 accumulation)
 * x [T, H] bf16; shared_packed from moe_prepack_shared_expert; shared_out
 * [G, T, H] fp32, ready for moe_combine_sharded.  Workspace 256-byte aligned,
 * its first word the device status (moe_read_device_status). */
moe_status moe_shared_expert(const void* x, const void* shared_packed, int32_t T, int32_t H,
                             int32_t Is, int32_t G, float* shared_out, void* workspace,
                             size_t ws_bytes, void* stream);

/* The fixed expert-output reduction (same section): for every n in [0, N),
 * v = partials[0..G-1][n] (bf16, logical rank order) widened exactly to FP64;
 * each level adds adjacent pairs (v0+v1, v2+v3, ...) in FP64 and carries an odd
 * last value unchanged; the last value is rounded once, FP64 -> bf16, to nearest
 * even.  partials [G][N] and out [N] bf16 on the device, 2-byte aligned
 * (16-byte alignment and N % 8 == 0 take the vector path); 1 <= G <= 16. */
moe_status moe_tree_reduce_bf16(const void* partials, int32_t G, int64_t N, void* out,
                                void* stream);

/* Workspace of moe_layer_fwd_sharded (Is = 0: no shared expert; 0: dimensions
 * outside the limits). */
size_t moe_sharded_workspace_bytes(moe_dims d, int32_t G, int32_t Is);

/* The layer as G expert ranks compute it, on one GPU: moe_layer_fwd_ex up to the
 * expert FFN, then (shared_packed != NULL, Is > 0) moe_shared_expert, then
 * moe_combine_sharded with owner [E] (device) and the fixed FP64 tree.
 * 1 <= G <= 16.  Workspace: moe_sharded_workspace_bytes. */
moe_status moe_layer_fwd_sharded(const void* x, const float* w_router, const float* bias,
                                 const moe_router_opts* opts, const void* packed_weights,
                                 const int32_t* owner, int32_t G, const void* shared_packed,
                                 int32_t Is, moe_dims d, void* out, int32_t* topk_idx_out,
                                 float* topk_w_out, int32_t* counts_out, void* workspace,
                                 size_t ws_bytes, void* stream);

/* moe_layer_fwd_sharded recording 7 events on `stream` (as moe_layer_fwd_profiled:
 * before route, after route, after load stats, after permute, after the gate/up
 * GEMM, after the down GEMM and the shared expert, after the sharded combine). */
moe_status moe_layer_fwd_sharded_profiled(
    const void* x, const float* w_router, const float* bias, const moe_router_opts* opts,
    const void* packed_weights, const int32_t* owner, int32_t G, const void* shared_packed,
    int32_t Is, moe_dims d, void* out, int32_t* topk_idx_out, float* topk_w_out,
    int32_t* counts_out, void* workspace, size_t ws_bytes, void* stream, void* const* events,
    int32_t n_events);

/* The whole layer forward: route -> load stats -> permute -> expert FFN ->
 * combine, enqueued on one stream with no host synchronisation.
 *   x [T, H] bf16; w_router [H, E] fp32; bias [E] fp32 or NULL; packed_weights
 *   from moe_prepack_expert_weights; out [T, H] bf16.
 *   topk_idx_out [T, k], topk_w_out [T, k] and counts_out [E] are optional
 *   (NULL: kept in the workspace only).
 * Stream order is that of ordinary launches for every other kernel: the layer's
 * own kernels may start while the previous one of them runs (programmatic
 * dependent launch) but touch its outputs only after it has finished.  For a
 * one-token batch the small-batch expert GEMMs run before the load statistics
 * (their rows follow from the token's expert ids); every output is the same. */
moe_status moe_layer_fwd(const void* x, const float* w_router, const float* bias,
                         const void* packed_weights, moe_dims d, void* out, int32_t* topk_idx_out,
                         float* topk_w_out, int32_t* counts_out, void* workspace, size_t ws_bytes,
                         void* stream);

/* moe_layer_fwd with a router variant and routing scale (opts NULL: the defaults
 * of moe_layer_fwd).  For MOE_ROUTER_SIGMOID_BIAS_SELECT, `bias` is the
 * selection-only correction bias. */
moe_status moe_layer_fwd_ex(const void* x, const float* w_router, const float* bias,
                            const moe_router_opts* opts, const void* packed_weights, moe_dims d,
                            void* out, int32_t* topk_idx_out, float* topk_w_out,
                            int32_t* counts_out, void* workspace, size_t ws_bytes, void* stream);

/* moe_layer_fwd that also records caller-created CUDA events (cudaEvent_t
 * passed as void*) on `stream` at the step boundaries, for per-step timing:
 *   events[0] before the router, [1] after it, [2] after the load statistics,
 *   [3] after the permutation, [4] after the grouped gate/up GEMM (SwiGLU),
 *   [5] after the grouped down GEMM, [6] after the combine.
 * n_events must be 7 (or 0 with events NULL, which is moe_layer_fwd).  The work
 * enqueued is identical to moe_layer_fwd's. */
moe_status moe_layer_fwd_profiled(const void* x, const float* w_router, const float* bias,
                                  const void* packed_weights, moe_dims d, void* out,
                                  int32_t* topk_idx_out, float* topk_w_out, int32_t* counts_out,
                                  void* workspace, size_t ws_bytes, void* stream,
                                  void* const* events, int32_t n_events);

/* moe_load_stats for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point: it exists for callers that run where
 * calling cudaMalloc (or taking memory from an allocator) is not allowed, such as
 * code inside a host framework whose device memory is owned by its own pool, or
 * a serving loop that must not allocate after start-up because an allocation can
 * synchronise the device.  It computes exactly what moe_load_stats computes
 * (counts [E], offsets [E+1]) from the same inputs, but keeps the per-block
 * partial counts in a 2 MiB scratch array compiled into the library (one per GPU
 * that loads it, held until the process exits) instead of a caller workspace.
 *   Limit: 2 * ceil(T / 256) * E <= 524288 (for E = 256: T <= 262144); larger
 *   sizes return MOE_ERR_UNSUPPORTED before anything is launched.
 *   device_status: optional device int32 (NULL: not reported); receives
 *   MOE_ERR_DEVICE_CHECK if an expert id is out of range or repeated within a
 *   token (the caller zeroes it beforehand).
 * Arguments are checked as moe_load_stats checks them (dims, non-null 16-byte
 * aligned pointers, an sm_103 device), and device_status too when given.
 * The first call on each device looks up the scratch array's device address
 * (cudaGetSymbolAddress) and keeps it for the process; make that first call
 * before any stream capture, and do not call this entry point again on a device
 * after cudaDeviceReset on it (the kept address belonged to the old context).
 * All calls on a device share the one scratch array, and each call overwrites the
 * part of it that it reads, so calls whose kernels can overlap on the GPU (other
 * streams, other host threads) race: serialise them.  Nothing is allocated or
 * freed. */
moe_status moe_load_stats_noalloc(const int32_t* topk_idx, moe_dims d, int32_t* counts,
                                  int32_t* offsets, int32_t* device_status, void* stream);

/* Synchronises `stream`, returns the workspace status word in *status_out
 * (MOE_OK or the first device-side error recorded since the last read) and
 * clears it. */
moe_status moe_read_device_status(void* workspace, int32_t* status_out, void* stream);

/* Diagnostics: the limit, in SM clock cycles, of every bounded wait inside the
 * grouped GEMM kernels of calls launched afterwards (process-wide; cycles <= 0
 * restores the default of 4e9, about 2 s).  A wait that runs out records
 * MOE_ERR_TIMEOUT in the workspace status word; the kernel then waits for its own
 * copies and MMAs in flight (always with the default limit), releases its tensor
 * memory and exits, leaving the outputs of that call undefined and the CUDA
 * context usable.  Meant for exercising that path, not for production. */
moe_status moe_set_wait_limit(long long cycles);

/* Static text for a status code. */
const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
