// Router: fixed-order FP32 projection, FP32 softmax, top-k, renormalisation.
//
// "0 train-infer mismatch for open-weight MoE RL", section "Mixture-of-experts
// layers / The router": every token is projected to one score per expert with a
// fixed-K matrix multiplication, FP32 softmax is applied, the top-k
// probabilities are selected and renormalised by adding them left to right and
// dividing each by the sum; experts are returned sorted by probability.
//
// Kernel shape.  One CTA = 32 tokens x all E experts (E padded to EP in
// {32, 64, 128, 256}); 128 threads = 4 warps, four CTAs per SM.  Warp w owns
// tokens 8w..8w+7; lane i owns EP/32 experts (4i + 128g + jj for EP >= 128, else
// EP/32 consecutive).  Each logit is ONE thread's fused multiply-add chain over
// h = 0, 1, ..., H-1 starting from 0 (no split of K, no tree), then one FP32 add
// of the bias: the same bits as a CPU FMA chain, and independent of T.
//
// Data movement: 16-column chunks of W_r (FP32) and x (bf16) are copied into a
// double-buffered shared-memory ring with cp.async while the previous chunk is
// multiplied; x is then widened once to FP32 into a transposed buffer, so a
// warp's eight token values for one h are two broadcast loads.  Small CTAs (32
// tokens) keep each SM's share of T within a few percent of the mean.
//
// Epilogue: logits go to shared memory; one warp per token runs k rounds of a
// warp-wide argmax under the key (logit desc, expert asc), then the softmax
// denominator (lane partial sums in ascending expert order, then an xor
// butterfly: identical bits on every lane and for every T).  Selection uses the
// FP32 logit, which orders experts exactly as the probabilities do.
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int BT = 32;       // tokens per CTA
constexpr int HK = 16;       // hidden columns per chunk
constexpr int XLD = BT + 4;  // row stride of the transposed FP32 x chunk
constexpr int NTHR = 128;

template <int EP>
struct RouteSmem {
  static constexpr int w_floats = 2 * HK * EP;         // W_r ring
  static constexpr int xst_halves = 2 * BT * HK;       // bf16 x ring
  static constexpr int xs_floats = HK * XLD;           // FP32 transposed x
  static constexpr int ring_bytes = 4 * w_floats + 2 * xst_halves + 4 * xs_floats;
  static constexpr int logit_bytes = 4 * BT * (EP + 1);
  static constexpr int bytes = ring_bytes > logit_bytes ? ring_bytes : logit_bytes;
};

template <int EP>
__device__ __forceinline__ int expert_of(int lane, int jj) {
  constexpr int TE = EP / 32;
  if constexpr (TE >= 4) {
    return (jj >> 2) * 128 + lane * 4 + (jj & 3);
  } else {
    return lane * TE + jj;
  }
}

template <int EP>
__global__ void __launch_bounds__(NTHR, 4) route_kernel(const uint16_t* __restrict__ x,
                                                        const float* __restrict__ wr,
                                                        const float* __restrict__ bias, int T,
                                                        int H, int E, int k,
                                                        int32_t* __restrict__ topk_idx,
                                                        float* __restrict__ topk_w) {
  constexpr int TE = EP / 32;  // experts per thread
  constexpr int TT = 8;        // tokens per thread (one warp = 8 tokens)
  extern __shared__ float4 smem_f4[];
  float* ws = reinterpret_cast<float*>(smem_f4);                      // [2][HK][EP]
  uint16_t* xst = reinterpret_cast<uint16_t*>(ws + 2 * HK * EP);      // [2][BT][HK]
  float* xs = reinterpret_cast<float*>(xst + 2 * BT * HK);            // [HK][XLD]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * BT;
  const int nchunks = H / HK;
  const bool vec_w = (E % 4) == 0;

  // Padding experts (E..EP-1) read zeros from both ring buffers for the whole kernel.
  if (E < EP) {
    for (int i = tid; i < 2 * HK * EP; i += NTHR)
      if ((i % EP) >= E) ws[i] = 0.0f;
  }

  auto issue_chunk = [&](int c, int buf) {
    const int h0 = c * HK;
    float* wdst = ws + buf * HK * EP;
    if (E == EP) {
      // W_r rows h0..h0+HK-1 are contiguous and unpadded: a flat 16-byte copy
      const float* src = wr + (size_t)h0 * E;
#pragma unroll
      for (int i = tid; i < HK * EP / 4; i += NTHR) cp_async_16(wdst + 4 * i, src + 4 * i, 16);
    } else if (vec_w) {
      const int n4 = HK * E / 4;  // 16-byte pieces
      const float* src = wr + (size_t)h0 * E;
      for (int i = tid; i < n4; i += NTHR) {
        const int f = 4 * i;
        cp_async_16(wdst + (f / E) * EP + (f % E), src + f, 16);
      }
    } else {
      const float* src = wr + (size_t)h0 * E;
      for (int i = tid; i < HK * E; i += NTHR) cp_async_4(wdst + (i / E) * EP + (i % E), src + i);
    }
    // x chunk: BT rows x HK bf16 = two 16-byte pieces per row; rows past T are zero
    uint16_t* xdst = xst + buf * BT * HK;
    if (tid < 2 * BT) {
      const int r = tid >> 1, half = tid & 1;
      const int t = t0 + r;
      const uint16_t* src = (t < T) ? x + (size_t)t * H + h0 + 8 * half : x;
      cp_async_16(xdst + r * HK + 8 * half, src, (t < T) ? 16 : 0);
    }
    cp_async_commit();
  };

  float acc[TT][TE];
#pragma unroll
  for (int i = 0; i < TT; ++i)
#pragma unroll
    for (int j = 0; j < TE; ++j) acc[i][j] = 0.0f;

  issue_chunk(0, 0);
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    if (c + 1 < nchunks) {
      issue_chunk(c + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    // widen the x chunk to FP32, transposed: xs[h][token]
    {
      const int r = tid >> 2, hq = (tid & 3) * 4;  // 32 rows x 4 groups of 4 columns
      const uint2 v = *reinterpret_cast<const uint2*>(xst + buf * BT * HK + r * HK + hq);
      xs[(hq + 0) * XLD + r] = bf16_lo(v.x);
      xs[(hq + 1) * XLD + r] = bf16_hi(v.x);
      xs[(hq + 2) * XLD + r] = bf16_lo(v.y);
      xs[(hq + 3) * XLD + r] = bf16_hi(v.y);
    }
    __syncthreads();
    const float* wsb = ws + buf * HK * EP;
#pragma unroll
    for (int hh = 0; hh < HK; ++hh) {
      const float4 xa = *reinterpret_cast<const float4*>(xs + hh * XLD + warp * TT);
      const float4 xb = *reinterpret_cast<const float4*>(xs + hh * XLD + warp * TT + 4);
      const float xv[TT] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      float wv[TE];
      if constexpr (TE >= 4) {
#pragma unroll
        for (int g = 0; g < TE / 4; ++g) {
          const float4 w4 = *reinterpret_cast<const float4*>(wsb + hh * EP + g * 128 + lane * 4);
          wv[4 * g + 0] = w4.x;
          wv[4 * g + 1] = w4.y;
          wv[4 * g + 2] = w4.z;
          wv[4 * g + 3] = w4.w;
        }
      } else if constexpr (TE == 2) {
        const float2 w2 = *reinterpret_cast<const float2*>(wsb + hh * EP + lane * 2);
        wv[0] = w2.x;
        wv[1] = w2.y;
      } else {
        wv[0] = wsb[hh * EP + lane];
      }
#pragma unroll
      for (int i = 0; i < TT; ++i)
#pragma unroll
        for (int j = 0; j < TE; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }

  // ---- epilogue: logits (+ bias) to shared memory --------------------------
  constexpr int LLD = EP + 1;
  float* ls = reinterpret_cast<float*>(smem_f4);  // [BT][LLD], over the drained ring
#pragma unroll
  for (int j = 0; j < TE; ++j) {
    const int e = expert_of<EP>(lane, j);
    const float b = (bias != nullptr && e < E) ? __ldg(bias + e) : 0.0f;
#pragma unroll
    for (int i = 0; i < TT; ++i) {
      float l = acc[i][j];
      if (bias != nullptr) l = __fadd_rn(l, b);
      ls[(warp * TT + i) * LLD + e] = l;
    }
  }
  __syncthreads();

  // ---- softmax / top-k / renormalise: warp w handles its 8 tokens ----------
  constexpr int NV = EP / 32;
  for (int i = 0; i < TT; ++i) {
    const int tl = warp * TT + i;
    const int t = t0 + tl;
    if (t >= T) break;
    float v[NV];
    unsigned taken = 0;
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      const int e = lane + 32 * q;
      v[q] = (e < E) ? ls[tl * LLD + e] : -INFINITY;
      if (e >= E) taken |= 1u << q;
    }
    float sel_l[kMaxK];
    int sel_e[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k) {
        float bv = -INFINITY;
        int be = 0x7FFFFFFF;
#pragma unroll
        for (int q = 0; q < NV; ++q) {
          const int e = lane + 32 * q;
          if (!((taken >> q) & 1u) && (v[q] > bv || (v[q] == bv && e < be))) {
            bv = v[q];
            be = e;
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
          const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, off);
          if (ov > bv || (ov == bv && oe < be)) {
            bv = ov;
            be = oe;
          }
        }
        sel_l[j] = bv;
        sel_e[j] = be;
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
      }
    }
    // softmax denominator over all E experts, max-shifted
    const float m = sel_l[0];
    float z = 0.0f;
#pragma unroll
    for (int q = 0; q < NV; ++q)
      if (lane + 32 * q < E) z = __fadd_rn(z, expf(v[q] - m));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z = __fadd_rn(z, __shfl_xor_sync(0xFFFFFFFFu, z, off));
    // selected probabilities, their left-to-right sum, renormalised weights
    float p[kMaxK];
    float S = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k) {
        p[j] = __fdiv_rn(expf(sel_l[j] - m), z);
        S = __fadd_rn(S, p[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k && lane == j) {
        topk_idx[(size_t)t * k + j] = sel_e[j];
        topk_w[(size_t)t * k + j] = __fdiv_rn(p[j], S);
      }
    }
  }
}

template <int EP>
cudaError_t launch_ep(const void* x, const float* wr, const float* bias, int T, int H, int E, int k,
                      int32_t* idx, float* w, cudaStream_t s) {
  constexpr int smem = RouteSmem<EP>::bytes;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(route_kernel<EP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  dim3 grid((T + BT - 1) / BT);
  route_kernel<EP><<<grid, NTHR, smem, s>>>(static_cast<const uint16_t*>(x), wr, bias, T, H, E,
                                            k, idx, w);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const void* x, const float* w_router, const float* bias, int T, int H,
                         int E, int k, int32_t* topk_idx, float* topk_w, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (E <= 32) return launch_ep<32>(x, w_router, bias, T, H, E, k, topk_idx, topk_w, s);
  if (E <= 64) return launch_ep<64>(x, w_router, bias, T, H, E, k, topk_idx, topk_w, s);
  if (E <= 128) return launch_ep<128>(x, w_router, bias, T, H, E, k, topk_idx, topk_w, s);
  return launch_ep<256>(x, w_router, bias, T, H, E, k, topk_idx, topk_w, s);
}

}  // namespace moe
