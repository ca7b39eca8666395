// Internal launchers of the sm_103a kernels (one translation unit each); the
// C ABI in moe_api.cu validates arguments and calls these.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Host-side argument checks of the C ABI (moe_api.cu), for entry points defined
// in other translation units: dims within the library's limits, a non-null
// 16-byte-aligned pointer, a current device that is sm_103.
moe_status validate_dims(const moe_dims& d);
moe_status validate_ptr(const void* p);
moe_status validate_device();

constexpr int kMaxE = 256;
constexpr int kMaxK = 16;
constexpr int kMaxShards = 16;  // expert ranks of the sharded combine / tree
constexpr int kPermBlock = 256;  // tokens per ranking block of the permutation
constexpr long long kSpinLimitCycles = 4000000000LL;  // ~2 s at 2 GHz
constexpr int kRouteSmallMaxT = 64;  // batches up to this size use the small-T router kernel
constexpr int kRouteClusterMaxT = 1024;  // and up to this size its eight-token clusters

// router: projection (FP32 FMA chain), then kind 0: softmax, top-k (bias joins the
// logits); kind 1: sigmoid scores, top-k on score + correction bias, weights from
// the scores.  weights_bf16 rounds every weight to bf16.
cudaError_t launch_route(const void* x, const float* w_router, const float* bias, int T, int H,
                         int E, int k, int kind, int weights_bf16, int32_t* topk_idx,
                         float* topk_w, cudaStream_t s);

// per-block expert counts: blk_counts [nb, E], nb = ceil(T / kPermBlock)
// (remap: optional logical expert -> physical slot map; counts then per slot)
cudaError_t launch_block_counts(const int32_t* topk_idx, int T, int k, int E, int32_t* blk_counts,
                                int32_t* status, cudaStream_t s, const int32_t* remap = nullptr);

// counts [E] (nullable), offsets [E+1] (written, or read and checked if given),
// blk_base [nb, E] = first row of each (block, expert)
cudaError_t launch_scan(const int32_t* blk_counts, int nb, int E, int R, int32_t* counts,
                        int32_t* offsets, bool offsets_given, int32_t* blk_base, int32_t* status,
                        cudaStream_t s);

// stable ranks: row_of_slot [T*k], slot_of_row [T*k]
cudaError_t launch_rank(const int32_t* topk_idx, int T, int k, int E, const int32_t* blk_base,
                        int32_t* row_of_slot, int32_t* slot_of_row, int32_t* status,
                        cudaStream_t s, const int32_t* remap = nullptr);

// out[e] (int64, zeroed here) = sum of q[t] over the (t, j) with topk_idx[t,j] = e
cudaError_t launch_weighted_counts(const int32_t* topk_idx, const int32_t* q, int T, int k, int E,
                                   int64_t* out, int32_t* status, cudaStream_t s);

// offsets[g] = g * T for g = 0..G (G groups of T rows each)
cudaError_t launch_uniform_offsets(int32_t* offsets, int G, int T, cudaStream_t s);

// T <= kPermBlock: counts, offsets, row_of_slot, slot_of_row and the permuted
// rows x_perm in one launch
// x_perm == nullptr (late): the indices only, computed before the kernel waits for
// its predecessor (which must neither read nor write them); the kernel then waits, so
// its completion implies the predecessor's
cudaError_t launch_dispatch_small(const int32_t* topk_idx, int T, int k, int E, const void* x,
                                  int H, int32_t* counts, int32_t* offsets, int32_t* row_of_slot,
                                  int32_t* slot_of_row, void* x_perm, int32_t* status,
                                  cudaStream_t s);

// x_perm[row_of_slot[t*k+j]] = x[t]
cudaError_t launch_copy_rows(const void* x, const int32_t* row_of_slot, int T, int H, int k,
                             void* x_perm, int32_t* status, cudaStream_t s);

// packed weights: [E][2I][H] (gate/up interleaved in 128-row halves of 256-row
// tiles) followed by [E][H][I] (down, transposed)
cudaError_t launch_prepack(const void* w_gate, const void* w_up, const void* w_down, int E, int H,
                           int I, void* packed, cudaStream_t s,
                           const int32_t* slot_of_expert = nullptr);

// A shared expert (W_gate, W_up [H, Is], W_down [Is, H]) packed as G experts of
// intermediate size Is/G: expert g holds columns [g*Is/G, (g+1)*Is/G) of the gate
// and up projections and the same rows of the down projection (layout as above).
cudaError_t launch_prepack_shared(const void* w_gate, const void* w_up, const void* w_down, int H,
                                  int Is, int G, void* packed, cudaStream_t s);

// A bf16 row-major operand [rows, cols] of a grouped GEMM.  encode() writes a TMA
// map of it with boxes of 64 columns x box_rows rows and 128-byte swizzle
// (defined with the ABI, which owns the driver entry point).
struct GemmOperand {
  const void* ptr;
  uint64_t cols, rows;
  bool encode(CUtensorMap* map, uint32_t box_rows) const;
};

// A row-major 2D tensor [rows, cols] of FP32 (fp32) or BF16 elements, boxes of
// box_cols x box_rows without swizzle, zeros outside; false if the driver
// refuses it (base not 16-byte aligned, row stride not a multiple of 16 bytes).
bool encode_rowmajor_2d(CUtensorMap* map, const void* ptr, uint64_t cols, uint64_t rows, bool fp32,
                        uint32_t box_cols, uint32_t box_rows);

// grouped GEMM-1 with the SwiGLU epilogue: a = x_perm [R, H], b = packed W1
// [E*2I, H] -> h [R, I] bf16.  a_local: every group reads rows of `a` from 0
// (one token matrix for all groups, e.g. the column shards of a shared expert).
cudaError_t launch_gemm_gate_up(const GemmOperand& a, const GemmOperand& b,
                                const int32_t* offsets, int E, int R, int H, int I, void* h,
                                int32_t* status, long long spin_limit, cudaStream_t s,
                                bool a_local = false);

// grouped GEMM-2: a = h [R, I], b = packed W2 [E*H, I] -> y [R, H] fp32
cudaError_t launch_gemm_down(const GemmOperand& a, const GemmOperand& b,
                             const int32_t* offsets, int E, int R, int H, int I, float* y,
                             int32_t* status, long long spin_limit, cudaStream_t s);

// N tile width of the down projection for this H (fixed per model shape)
int gemm_down_bn(int H);

// The same two GEMMs with the weight rows on the MMA's M side and up to 64 token
// rows on N (small batches); outputs bit-identical to the tile kernels above.
// use_swap_gemm: at most kSwapRowsPerExpert rows per expert on average and at
// most four gate/up work units per SM (experts with rows <= min(E, R)).
constexpr int kSwapRowsPerExpert = 8;
bool use_swap_gemm(int E, int R, int H, int I);
// one_token_ids (a batch of one token, R = k): the schedule comes from the token's
// k expert ids instead of `offsets` (the same rows: expert e's row is the number of
// chosen experts below e), so the GEMMs need not wait for the dispatch; the gate/up
// GEMM then reads the token row itself (a = x [1, H]).
cudaError_t launch_gemm_gate_up_swap(const GemmOperand& a, const GemmOperand& b,
                                     const int32_t* offsets, int E, int R, int H, int I, void* h,
                                     int32_t* status, long long spin_limit, cudaStream_t s,
                                     bool a_local = false, const int32_t* one_token_ids = nullptr);
cudaError_t launch_gemm_down_swap(const GemmOperand& a, const GemmOperand& b,
                                  const int32_t* offsets, int E, int R, int H, int I, float* y,
                                  int32_t* status, long long spin_limit, cudaStream_t s,
                                  const int32_t* one_token_ids = nullptr);

// out[t] = bf16(slot-order FMA chain of (scale * topk_w[t,j]) * y[row_of_slot[t*k+j]])
// slots_final: topk_w and row_of_slot were complete before the kernel that writes
// y began (so they may be read before the kernel waits for y)
cudaError_t launch_combine(const float* y, const float* topk_w, const int32_t* row_of_slot, int T,
                           int H, int k, float scale, void* out, cudaStream_t s,
                           bool slots_final = false);

// Sharded combine: G per-rank BF16 partials (slot-order FP32 chains, other ranks'
// slots as exact zeros, optional shared [G][T][H] FP32 added before the rounding)
// reduced by the fixed FP64 pairwise tree.  partials [G][T][H] bf16 is optional.
cudaError_t launch_combine_sharded(const float* y, const float* topk_w, const int32_t* topk_idx,
                                   const int32_t* row_of_slot, const int32_t* owner, int G, int T,
                                   int H, int E, int k, float scale, const float* shared,
                                   void* partials, void* out, cudaStream_t s);

// out[n] = bf16(FP64 pairwise tree over partials[0..G-1][n]); vec: 16-byte vectors
// (N a multiple of 8, all rows 16-byte aligned).
cudaError_t launch_tree_reduce(const void* partials, int G, long long N, void* out, bool vec,
                               cudaStream_t s);

// number of SMs of the current device (cached per device)
int device_sm_count();

}  // namespace moe
