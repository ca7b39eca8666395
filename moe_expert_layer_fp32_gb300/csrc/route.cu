// Router: fixed-order FP32 projection, FP32 softmax, top-k, renormalisation.
//
// "0 train-infer mismatch for open-weight MoE RL", section "Mixture-of-experts
// layers / The router": every token is projected to one score per expert with a
// fixed-K matrix multiplication, FP32 softmax is applied, the top-k
// probabilities are selected and renormalised by adding them left to right and
// dividing each by the sum; experts are returned sorted by probability.
//
// Kernel shape.  One CTA = 64 tokens x all E experts (E padded to EP in
// {32, 64, 128, 256}); 256 threads = 8 warps.  Warp w owns tokens 8w..8w+7; lane
// i owns EP/32 experts (4i + 128g + jj for EP >= 128, else EP/32 consecutive).
// Each logit is ONE thread's fused multiply-add chain over h = 0, 1, ..., H-1
// starting from 0 (no split of K, no tree), then one FP32 add of the bias: the
// same bits as the CPU reference FMA chain, and independent of T.  x is widened
// to FP32 once per 32-column chunk into shared memory (transposed, so a warp's
// token reads are broadcasts); W_r chunks are staged beside it.
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

constexpr int BT = 64;       // tokens per CTA
constexpr int HK = 32;       // hidden columns per chunk
constexpr int XLD = BT + 4;  // row stride of the transposed x chunk (16-byte aligned rows)

template <int EP>
struct RouteSmem {
  static constexpr int chunk_floats = HK * XLD + HK * EP;
  static constexpr int logit_floats = BT * (EP + 1);
  static constexpr int bytes =
      4 * (chunk_floats > logit_floats ? chunk_floats : logit_floats);
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
__global__ void __launch_bounds__(256) route_kernel(const uint16_t* __restrict__ x,
                                                    const float* __restrict__ wr,
                                                    const float* __restrict__ bias, int T, int H,
                                                    int E, int k, int32_t* __restrict__ topk_idx,
                                                    float* __restrict__ topk_w) {
  constexpr int TE = EP / 32;   // experts per thread
  constexpr int TT = 8;         // tokens per thread
  constexpr int WPT = EP / 8;   // W_r chunk elements loaded per thread (HK*EP/256)
  extern __shared__ float4 smem_f4[];
  float* smem = reinterpret_cast<float*>(smem_f4);
  float* xs = smem;             // [HK][XLD]   x chunk, transposed, FP32
  float* ws = smem + HK * XLD;  // [HK][EP]    W_r chunk, zero beyond E

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * BT;

  float acc[TT][TE];
#pragma unroll
  for (int i = 0; i < TT; ++i)
#pragma unroll
    for (int j = 0; j < TE; ++j) acc[i][j] = 0.0f;

  // global -> register staging of one chunk
  const int xr = tid >> 2, xc = (tid & 3) * 8;  // 64 rows x 4 pieces of 8 bf16
  const int xt = t0 + xr;
  uint4 xreg;
  float wreg[WPT];
  auto load_chunk = [&](int h0) {
    xreg = make_uint4(0, 0, 0, 0);
    if (xt < T) xreg = __ldg(reinterpret_cast<const uint4*>(x + (size_t)xt * H + h0 + xc));
#pragma unroll
    for (int i = 0; i < WPT; ++i) {
      int f = tid + i * 256;
      int r = f / EP, c = f % EP;
      wreg[i] = (c < E) ? __ldg(wr + (size_t)(h0 + r) * E + c) : 0.0f;
    }
  };
  auto store_chunk = [&]() {
    const uint32_t xw[4] = {xreg.x, xreg.y, xreg.z, xreg.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      xs[(xc + 2 * q) * XLD + xr] = bf16_lo(xw[q]);
      xs[(xc + 2 * q + 1) * XLD + xr] = bf16_hi(xw[q]);
    }
#pragma unroll
    for (int i = 0; i < WPT; ++i) {
      int f = tid + i * 256;
      ws[(f / EP) * EP + (f % EP)] = wreg[i];
    }
  };

  load_chunk(0);
  for (int h0 = 0; h0 < H; h0 += HK) {
    __syncthreads();
    store_chunk();
    __syncthreads();
    if (h0 + HK < H) load_chunk(h0 + HK);
#pragma unroll 4
    for (int hh = 0; hh < HK; ++hh) {
      const float4 xa = *reinterpret_cast<const float4*>(xs + hh * XLD + warp * TT);
      const float4 xb = *reinterpret_cast<const float4*>(xs + hh * XLD + warp * TT + 4);
      const float xv[TT] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      float wv[TE];
      if constexpr (TE >= 4) {
#pragma unroll
        for (int g = 0; g < TE / 4; ++g) {
          const float4 w4 = *reinterpret_cast<const float4*>(ws + hh * EP + g * 128 + lane * 4);
          wv[4 * g + 0] = w4.x;
          wv[4 * g + 1] = w4.y;
          wv[4 * g + 2] = w4.z;
          wv[4 * g + 3] = w4.w;
        }
      } else if constexpr (TE == 2) {
        const float2 w2 = *reinterpret_cast<const float2*>(ws + hh * EP + lane * 2);
        wv[0] = w2.x;
        wv[1] = w2.y;
      } else {
        wv[0] = ws[hh * EP + lane];
      }
#pragma unroll
      for (int i = 0; i < TT; ++i)
#pragma unroll
        for (int j = 0; j < TE; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
    }
  }

  // ---- epilogue: logits (+ bias) to shared memory --------------------------
  __syncthreads();
  constexpr int LLD = EP + 1;
  float* ls = smem;  // [BT][LLD]
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
  route_kernel<EP><<<grid, 256, smem, s>>>(static_cast<const uint16_t*>(x), wr, bias, T, H, E, k,
                                           idx, w);
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
