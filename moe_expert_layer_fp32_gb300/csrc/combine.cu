// Combine: the weighted sum of a token's k expert outputs, in slot order.
//
// "0 train-infer mismatch for open-weight MoE RL", section "Sharding the
// experts": every routing slot is accumulated in FP32 in slot order and rounded
// once to BF16; section "The experts: keeping the route weight inside the
// accumulator": the route weight multiplies the FP32 down-projection value
// before the single rounding.  Here: acc = 0, acc = fmaf(w[t,j], y[row_j, c], acc)
// for j = 0..k-1, out = bf16(acc).
//
// An optional routing scale (GLM applies 2.5 inside the expert kernel) multiplies
// each weight once in FP32 before the chain; a scale of 1 leaves the weights, and
// so the result, unchanged.
//
// Memory-bound gather: one CTA per token and column block, 16-byte loads of the k
// FP32 rows (all issued before the FMA chain), 8-byte stores of four bf16 outputs.
// Column blocks are split across CTAs (gridDim.y) when T alone would leave SMs
// idle; every element's chain is the same either way.
#include "common.cuh"
#include "kernels.cuh"
#include "pdl.cuh"

namespace moe {
namespace {

// SPLIT: gridDim.y CTAs share a token's columns.  Both forms are held to five CTAs
// per SM (at most 96 registers) by the launch bound.
// A programmatic dependent of the down GEMM: y is read (and out written) only after
// that kernel has finished.  EARLY: the weights and rows were final before the
// down GEMM started (the layer's own chain), so they are read before the wait.
template <bool SPLIT, bool EARLY>
__global__ void __launch_bounds__(128, 5) combine_kernel(const float* __restrict__ y,
                                                      const float* __restrict__ topk_w,
                                                      const int32_t* __restrict__ row_of_slot,
                                                      int T, int H, int k, float scale,
                                                      uint16_t* __restrict__ out) {
  __shared__ int s_row[kMaxK];
  __shared__ float s_w[kMaxK];
  const int t = blockIdx.x;
  const long long R = (long long)T * k;
  auto load_slots = [&]() {
    if (threadIdx.x < k) {
      const int r = row_of_slot[(size_t)t * k + threadIdx.x];
      s_row[threadIdx.x] = (r >= 0 && r < R) ? r : -1;
      s_w[threadIdx.x] = __fmul_rn(scale, topk_w[(size_t)t * k + threadIdx.x]);
    }
  };
  if (EARLY) load_slots();
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  if (!EARLY) load_slots();
  __syncthreads();
  int row[kMaxK];
  float w[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    row[j] = (j < k) ? s_row[j] : -1;
    w[j] = (j < k) ? s_w[j] : 0.0f;
  }
  // this CTA's column block (a multiple of 4 * blockDim.x columns)
  const int cols = SPLIT ? H / gridDim.y : H;
  const int cb = SPLIT ? blockIdx.y * cols : 0;
  const float* yb = y + cb;
  for (int c = threadIdx.x * 4; c < cols; c += blockDim.x * 4) {
    float4 v[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (row[j] >= 0) v[j] = __ldg(reinterpret_cast<const float4*>(yb + (size_t)row[j] * H + c));
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (row[j] >= 0) {
        a0 = fmaf(w[j], v[j].x, a0);
        a1 = fmaf(w[j], v[j].y, a1);
        a2 = fmaf(w[j], v[j].z, a2);
        a3 = fmaf(w[j], v[j].w, a3);
      }
    }
    uint2 o;
    o.x = pack_bf16x2(a0, a1);
    o.y = pack_bf16x2(a2, a3);
    // (the output address is formed here: a pointer hoisted out of the loop
    // costs about 40 registers and two CTAs per SM)
    *reinterpret_cast<uint2*>(out + (size_t)t * H + cb + c) = o;
  }
}

}  // namespace

cudaError_t launch_combine(const float* y, const float* topk_w, const int32_t* row_of_slot, int T,
                           int H, int k, float scale, void* out, cudaStream_t s,
                           bool slots_final) {
  if (T == 0) return cudaSuccess;
  // split the columns of each token over up to H / 512 CTAs while the grid stays
  // within four CTAs per SM (one wave)
  int split = 1;
  while (split * 2 <= H / 512 && H % (split * 2 * 512) == 0 &&
         (long long)T * split * 2 <= 4LL * device_sm_count())
    split *= 2;
  auto go = [&](auto kern, dim3 grid) {
    return launch_pdl(kern, grid, dim3(128), 0, s, y, topk_w, row_of_slot, T, H, k, scale,
                      static_cast<uint16_t*>(out));
  };
  if (split > 1)
    return slots_final ? go(combine_kernel<true, true>, dim3(T, split))
                       : go(combine_kernel<true, false>, dim3(T, split));
  return slots_final ? go(combine_kernel<false, true>, dim3(T))
                     : go(combine_kernel<false, false>, dim3(T));
}

}  // namespace moe
