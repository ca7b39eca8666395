// Router: fixed-order FP32 projection, FP32 softmax, top-k, renormalisation.
//
// "0 train-infer mismatch for open-weight MoE RL", section "Mixture-of-experts
// layers / The router": every token is projected to one score per expert with a
// fixed-K matrix multiplication, FP32 softmax is applied, the top-k
// probabilities are selected and renormalised by adding them left to right and
// dividing each by the sum; experts are returned sorted by probability.
//
// In both kernels below each logit is ONE thread's fused multiply-add chain over
// h = 0, 1, ..., H-1 starting from 0 (no split of K, no tree), then one FP32 add
// of the bias, and both finish with the same per-token epilogue: the routing of
// a token is the same bits whichever kernel runs and whatever T is.
//
// route_kernel (T > 1024): one CTA = 32 tokens x all E experts (E padded to EP
// in {32, 64, 128, 256}); 128 threads = 4 warps, up to four CTAs per SM.  Warp w
// owns tokens 8w..8w+7; lane i owns EP/32 experts (4i + 128g + jj for EP >= 128,
// else EP/32 consecutive).  Chunks of HK = max(2048/EP, 16) hidden columns (8-16
// KB of W_r) and the matching x columns are copied by cp.async into a 3-stage
// ring while earlier chunks are multiplied (four CTAs fit on an SM); x is widened
// once to FP32 into a transposed buffer (two of them, so each chunk costs two CTA
// barriers), and a warp's eight token values for one h are two broadcast loads.
//
// route_cluster_kernel (T <= 1024): a cluster of eight CTAs (sixteen for T <= 8
// and 64 experts or more) per 1, 2, 4 or 8 tokens, each CTA owning its share of
// the experts and streaming only those columns of W_r; logits meet in the first
// CTA's shared memory (see below).
//
// route_tile_kernel (256 experts, large T): 2D warp tiles (see below).
//
// Epilogue (shared): logits go to shared memory; one warp per token runs k
// rounds of a warp-wide selection under the key (logit desc, expert asc), each
// a redux.sync max over a monotone integer key and a min over the expert, then the
// softmax denominator (lane partial sums in ascending expert order, then an xor
// butterfly: identical bits on every lane and for every T).  Selection uses the
// FP32 logit, which orders experts exactly as the probabilities do.
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int BT = 32;       // tokens per CTA (large-T kernel)
constexpr int NTHR = 128;
constexpr int NST = 3;       // cp.async ring depth

constexpr int XLD = BT + 4;  // row stride of the transposed FP32 x chunk

template <int EP>
struct RouteCfg {
  static constexpr int HK = (2048 / EP > 16) ? 2048 / EP : 16;  // 8-16 KB of W_r per chunk
  static constexpr int w_floats = NST * HK * EP;        // W_r ring
  static constexpr int xst_halves = NST * BT * HK;      // bf16 x ring
  static constexpr int xs_floats = 2 * HK * XLD;        // FP32 transposed x, two chunks
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

// exp(x) in FP32 by Cody & Waite argument reduction and a Taylor polynomial of
// degree 7 (Horner, fused multiply-adds), scaled by 2^n: n = rint(x log2 e),
// r = x - n ln2 with ln2 split into a 16-bit high part and its remainder.  Every
// step is one IEEE FP32 operation, so any implementation of the same steps gives
// the same bits (used where the exponential decides which experts are chosen).
__device__ __forceinline__ float exp_cw(float x) {
  x = fminf(fmaxf(x, -104.0f), 89.0f);
  const float LOG2E = 1.44269502162933349609375f;
  const float LN2_HI = 0.693145751953125f;
  const float LN2_LO = 1.428606765330187e-06f;
  const float n = rintf(__fmul_rn(x, LOG2E));
  float r = fmaf(-n, LN2_HI, x);
  r = fmaf(-n, LN2_LO, r);
  float p = 1.0f / 5040.0f;
  p = fmaf(p, r, 1.0f / 720.0f);
  p = fmaf(p, r, 1.0f / 120.0f);
  p = fmaf(p, r, 1.0f / 24.0f);
  p = fmaf(p, r, 1.0f / 6.0f);
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  return ldexpf(p, (int)n);
}

// The large-T kernels advance two experts' chains per instruction: FFMA2 on
// (x, x) * (w_e, w_e+1) + (acc_e, acc_e+1).  Each lane is the same IEEE
// round-to-nearest fused multiply-add as fmaf, so every logit is the same chain
// as one FFMA per step would give; the packed form halves the FMA issue slots of
// these issue-bound loops.  Measured on GB300 (router stage): large 1.59 -> 1.43-
// 1.47 ms, packed_rl 255 -> 236 us, ling3_tiny 198 -> 186 us, fine_grained T = 4096
// 73 -> 70 us.  Storing every token value twice in shared memory, so a 16-byte
// load gives two ready pairs, was slower than either (large 1.71 ms).
__device__ __forceinline__ float2 ffma2(float2 x, float2 w, float2 acc) {
  return __ffma2_rn(x, w, acc);
}

__device__ __forceinline__ float round_bf16(float f) {
  return __bfloat162float(__float2bfloat16_rn(f));
}

// One warp routes token t from its E logits lrow[0..E) (shared memory).
//   KIND 0 (softmax): top-k by (logit desc, expert asc), FP32 softmax over all E,
//     selected probabilities renormalised left to right.
//   KIND 1 (sigmoid, "0 train-infer mismatch", section "Choosing GLM's eight
//     experts"): scores s = sigmoid(l); the correction bias joins only the
//     selection key s + b (ties to the lower expert); weights = selected s over
//     their left-to-right sum.
// wbf16 rounds every final weight to bf16.
template <int EP, int KIND>
__device__ __forceinline__ void route_one_token(const float* lrow, const float* corr_bias, int E,
                                                int k, int wbf16, int lane, int t,
                                                int32_t* __restrict__ topk_idx,
                                                float* __restrict__ topk_w) {
  constexpr int NV = EP / 32;
  float v[NV];   // selection key
  float sc[NV];  // KIND 1: pre-bias scores
  unsigned taken = 0;
#pragma unroll
  for (int q = 0; q < NV; ++q) {
    const int e = lane + 32 * q;
    if (e < E) {
      if constexpr (KIND == 0) {
        v[q] = lrow[e];
        sc[q] = 0.0f;
      } else {
        sc[q] = __fdiv_rn(1.0f, __fadd_rn(1.0f, exp_cw(-lrow[e])));
        v[q] = (corr_bias != nullptr) ? __fadd_rn(sc[q], __ldg(corr_bias + e)) : sc[q];
      }
    } else {
      v[q] = -INFINITY;
      sc[q] = 0.0f;
      taken |= 1u << q;
    }
  }
  // Selection keys as unsigned integers in the order (value desc): the value
  // plus 0.0f (so -0 and +0 become one key and tie, as in a float comparison),
  // its bits made monotone; NaN sorts below every number and padding experts
  // below everything.  Each round takes the largest key over the warp with one
  // reduction and, among the lanes holding it, the lowest expert with another:
  // the order (value desc, expert asc) of the shuffle argmax it replaced, in two
  // dependent warp operations per round instead of ten.
  uint32_t key[NV];
#pragma unroll
  for (int q = 0; q < NV; ++q) {
    if ((taken >> q) & 1u) {
      key[q] = 0u;
    } else {
      const float f = __fadd_rn(v[q], 0.0f);
      const uint32_t u = __float_as_uint(f);
      key[q] = (f != f) ? 1u : ((u & 0x80000000u) ? ~u : (u | 0x80000000u));
    }
  }
  float sel_l[kMaxK];
  int sel_e[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    if (j < k) {
      uint32_t bk = 0u;
      int bq = 0;
#pragma unroll
      for (int q = 0; q < NV; ++q) {
        if (!((taken >> q) & 1u) && key[q] > bk) {
          bk = key[q];
          bq = q;
        }
      }
      const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, bk);
      const uint32_t cand = (bk == m && !((taken >> bq) & 1u)) ? (uint32_t)(lane + 32 * bq) : 0xFFFFFFFFu;
      const int be = (int)__reduce_min_sync(0xFFFFFFFFu, cand);
      float bv;
      if constexpr (KIND == 1) {
        // the winner's pre-bias score, from the lane that owns expert be
        float mine = 0.0f;
#pragma unroll
        for (int q = 0; q < NV; ++q)
          if (q == (be >> 5)) mine = sc[q];
        bv = __shfl_sync(0xFFFFFFFFu, mine, be & 31);
      } else {
        // the logit back from its key (for -0 this gives +0, which the softmax
        // below treats identically)
        bv = __uint_as_float((m & 0x80000000u) ? (m & 0x7FFFFFFFu) : ~m);
      }
      sel_l[j] = bv;
      sel_e[j] = be;
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
    }
  }
  float p[kMaxK];
  float S = 0.0f;
  if constexpr (KIND == 0) {
    // softmax denominator over all E experts, max-shifted
    const float m = sel_l[0];
    float z = 0.0f;
#pragma unroll
    for (int q = 0; q < NV; ++q)
      if (lane + 32 * q < E) z = __fadd_rn(z, expf(v[q] - m));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z = __fadd_rn(z, __shfl_xor_sync(0xFFFFFFFFu, z, off));
    // lane j < k divides its own p_j = exp(l_j - m) / z; every lane then adds
    // p_0 .. p_{k-1} left to right
    float lj = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < k && j == lane) lj = sel_l[j];
    const float pl = __fdiv_rn(expf(lj - m), z);
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k) {
        p[j] = __shfl_sync(0xFFFFFFFFu, pl, j);
        S = __fadd_rn(S, p[j]);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k) {
        p[j] = sel_l[j];
        S = __fadd_rn(S, p[j]);
      }
    }
  }
  // lane j < k writes slot j (the k divisions run side by side)
  float pj = 0.0f;
  int ej = 0;
#pragma unroll
  for (int j = 0; j < kMaxK; ++j)
    if (j < k && j == lane) {
      pj = p[j];
      ej = sel_e[j];
    }
  if (lane < k) {
    float wj = __fdiv_rn(pj, S);
    if (wbf16) wj = round_bf16(wj);
    topk_idx[(size_t)t * k + lane] = ej;
    topk_w[(size_t)t * k + lane] = wj;
  }
}

// Eight token values of one hidden row as (x, x) pairs for FFMA2: two runs of
// four tokens, `gap` tokens apart in the transposed x chunk.
__device__ __forceinline__ void load_x8(const float* src, int gap, float2 (&xp)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(src);
  const float4 b = *reinterpret_cast<const float4*>(src + gap);
  const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) xp[i] = make_float2(v[i], v[i]);
}

template <int EP, int KIND>
__global__ void __launch_bounds__(NTHR, 4) route_kernel(const uint16_t* __restrict__ x,
                                                        const float* __restrict__ wr,
                                                        const float* __restrict__ bias, int T,
                                                        int H, int E, int k, int wbf16,
                                                        int32_t* __restrict__ topk_idx,
                                                        float* __restrict__ topk_w) {
  using C = RouteCfg<EP>;
  constexpr int HK = C::HK;
  constexpr int TE = EP / 32;  // experts per thread
  constexpr int TT = 8;        // tokens per thread (one warp = 8 tokens)
  extern __shared__ float4 smem_f4[];
  float* ws = reinterpret_cast<float*>(smem_f4);                      // [NST][HK][EP]
  uint16_t* xst = reinterpret_cast<uint16_t*>(ws + NST * HK * EP);    // [NST][BT][HK]
  float* xs = reinterpret_cast<float*>(xst + NST * BT * HK);          // [HK][XLD]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * BT;
  const int nchunks = H / HK;
  const bool vec_w = (E % 4) == 0;

  // Padding experts (E..EP-1) read zeros from every ring buffer for the whole kernel.
  if (E < EP) {
    for (int i = tid; i < NST * HK * EP; i += NTHR)
      if ((i % EP) >= E) ws[i] = 0.0f;
  }

  auto issue_chunk = [&](int c) {
    if (c < nchunks) {
      const int buf = c % NST;
      const int h0 = c * HK;
      float* wdst = ws + buf * HK * EP;
      const float* wsrc = wr + (size_t)h0 * E;
      if (E == EP) {
        // W_r rows h0..h0+HK-1 are contiguous and unpadded: a flat 16-byte copy
#pragma unroll
        for (int i = tid; i < HK * EP / 4; i += NTHR) cp_async_16(wdst + 4 * i, wsrc + 4 * i, 16);
      } else if (vec_w) {
        for (int i = tid; i < HK * E / 4; i += NTHR) {
          const int f = 4 * i;
          cp_async_16(wdst + (f / E) * EP + (f % E), wsrc + f, 16);
        }
      } else {
        for (int i = tid; i < HK * E; i += NTHR)
          cp_async_4(wdst + (i / E) * EP + (i % E), wsrc + i);
      }
      // x chunk: BT rows x HK bf16 in 16-byte pieces; rows past T are zero
      uint16_t* xdst = xst + buf * BT * HK;
      constexpr int PPR = HK / 8;  // pieces per row
      for (int i = tid; i < BT * PPR; i += NTHR) {
        const int r = i / PPR, pc = i % PPR;
        const int t = t0 + r;
        const uint16_t* src = (t < T) ? x + (size_t)t * H + h0 + 8 * pc : x;
        cp_async_16(xdst + r * HK + 8 * pc, src, (t < T) ? 16 : 0);
      }
    }
    cp_async_commit();  // one group per chunk slot, empty past the end
  };

  float acc[TT][TE];
#pragma unroll
  for (int i = 0; i < TT; ++i)
#pragma unroll
    for (int j = 0; j < TE; ++j) acc[i][j] = 0.0f;

#pragma unroll
  for (int c = 0; c < NST - 1; ++c) issue_chunk(c);
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c % NST;
    // chunk c has landed; every thread is past chunk c-1, so its ring slot is free
    cp_async_wait<NST - 2>();
    __syncthreads();
    issue_chunk(c + NST - 1);
    // widen the x chunk to FP32, transposed: xsc[h][token] (two buffers: chunk c-1's
    // may still be read by other warps)
    float* xsc = xs + (c & 1) * HK * XLD;
    for (int i = tid; i < BT * HK / 4; i += NTHR) {
      const int r = i / (HK / 4), hq = (i % (HK / 4)) * 4;
      const uint2 v = *reinterpret_cast<const uint2*>(xst + buf * BT * HK + r * HK + hq);
      xsc[(hq + 0) * XLD + r] = bf16_lo(v.x);
      xsc[(hq + 1) * XLD + r] = bf16_hi(v.x);
      xsc[(hq + 2) * XLD + r] = bf16_lo(v.y);
      xsc[(hq + 3) * XLD + r] = bf16_hi(v.y);
    }
    __syncthreads();
    const float* wsb = ws + buf * HK * EP;
#pragma unroll (HK > 16 ? 8 : HK)
    for (int hh = 0; hh < HK; ++hh) {
      float2 xp[TT];
      load_x8(xsc + hh * XLD + warp * TT, 4, xp);
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
      if constexpr (TE == 1) {
#pragma unroll
        for (int i = 0; i < TT; ++i) acc[i][0] = fmaf(xp[i].x, wv[0], acc[i][0]);
      } else {
#pragma unroll
        for (int i = 0; i < TT; ++i) {
#pragma unroll
          for (int j = 0; j < TE; j += 2) {
            const float2 r = ffma2(xp[i], make_float2(wv[j], wv[j + 1]),
                                   make_float2(acc[i][j], acc[i][j + 1]));
            acc[i][j] = r.x;
            acc[i][j + 1] = r.y;
          }
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // the logits below overwrite the ring

  // ---- epilogue: logits (+ bias for the softmax router) to shared memory ---
  constexpr int LLD = EP + 1;
  const bool add_bias = KIND == 0 && bias != nullptr;
  float* ls = reinterpret_cast<float*>(smem_f4);  // [BT][LLD], over the drained ring
#pragma unroll
  for (int j = 0; j < TE; ++j) {
    const int e = expert_of<EP>(lane, j);
    const float b = (add_bias && e < E) ? __ldg(bias + e) : 0.0f;
#pragma unroll
    for (int i = 0; i < TT; ++i) {
      float l = acc[i][j];
      if (add_bias) l = __fadd_rn(l, b);
      ls[(warp * TT + i) * LLD + e] = l;
    }
  }
  __syncthreads();
  for (int i = 0; i < TT; ++i) {
    const int tl = warp * TT + i;
    const int t = t0 + tl;
    if (t >= T) break;
    route_one_token<EP, KIND>(ls + tl * LLD, KIND == 1 ? bias : nullptr, E, k, wbf16, lane, t,
                              topk_idx, topk_w);
  }
}

// --------------------------------------------------- large T, 2D warp tiles ---
// route_tile_kernel: one CTA = BT = 8192/EP tokens x EP experts, 128 threads, each
// thread an 8-token x 8-expert block of logits.  A warp covers LT*8 tokens x
// LE*8 experts (LE = 8 lanes along experts when EP >= 64); a lane's tokens and
// experts are two runs of four, so each of its four 16-byte shared-memory loads
// per hidden column reads one contiguous run with the other lanes (no bank
// conflicts) and every W_r value is read by a quarter of the lanes the 1D layout
// needs.  Used for 256 experts once T gives every SM a CTA; the logits are the
// same FMA chains as in route_kernel, so the bits do not depend on the kernel
// chosen.
template <int EP>
struct TileCfg {
  static constexpr int BT = 8192 / EP;
  static constexpr int HK = (EP >= 256) ? 16 : 32;
  static constexpr int XL = BT + 4;
  static constexpr int LE = (EP / 8 < 8) ? EP / 8 : 8;  // lanes along experts
  static constexpr int LT = 32 / LE;                    // lanes along tokens
  static constexpr int WE = (EP / 8) / LE;              // warps along experts
  static constexpr int WT = (NTHR / 32) / WE;           // warps along tokens
  static_assert(WT * LT * 8 == BT, "tile");
  static constexpr int w_floats = NST * HK * EP;
  static constexpr int xst_halves = NST * BT * HK;
  static constexpr int xs_floats = 2 * HK * XL;  // two widened chunks
  static constexpr int ring_bytes = 4 * w_floats + 2 * xst_halves + 4 * xs_floats;
  static constexpr int logit_bytes = 4 * BT * (EP + 1);
  static constexpr int bytes = ring_bytes > logit_bytes ? ring_bytes : logit_bytes;
};

template <int EP, int KIND>
__global__ void __launch_bounds__(NTHR, 4) route_tile_kernel(const uint16_t* __restrict__ x,
                                                             const float* __restrict__ wr,
                                                             const float* __restrict__ bias, int T,
                                                             int H, int E, int k, int wbf16,
                                                             int32_t* __restrict__ topk_idx,
                                                             float* __restrict__ topk_w) {
  using C = TileCfg<EP>;
  constexpr int BTT = C::BT, HK = C::HK, XL = C::XL, LE = C::LE, LT = C::LT, WE = C::WE;
  extern __shared__ float4 smem_f4[];
  float* ws = reinterpret_cast<float*>(smem_f4);                      // [NST][HK][EP]
  uint16_t* xst = reinterpret_cast<uint16_t*>(ws + NST * HK * EP);    // [NST][BTT][HK]
  float* xs = reinterpret_cast<float*>(xst + NST * BTT * HK);         // [HK][XL]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * BTT;
  const int nchunks = H / HK;
  // this thread's tokens: tb + tok(i); experts: eb + exp(j)
  const int tb = (warp / WE) * (LT * 8) + (lane / LE) * 4;
  const int eb = (warp % WE) * (LE * 8) + (lane % LE) * 4;
  auto tok = [](int i) { return i < 4 ? i : 4 * LT + i - 4; };
  auto ex = [](int j) { return j < 4 ? j : 4 * LE + j - 4; };

  if (E < EP) {
    for (int i = tid; i < NST * HK * EP; i += NTHR)
      if ((i % EP) >= E) ws[i] = 0.0f;
  }
  auto issue_chunk = [&](int c) {
    if (c < nchunks) {
      const int buf = c % NST;
      const int h0 = c * HK;
      float* wdst = ws + buf * HK * EP;
      const float* wsrc = wr + (size_t)h0 * E;
      if (E == EP) {
#pragma unroll
        for (int i = tid; i < HK * EP / 4; i += NTHR) cp_async_16(wdst + 4 * i, wsrc + 4 * i, 16);
      } else if ((E % 4) == 0) {
        for (int i = tid; i < HK * E / 4; i += NTHR) {
          const int f = 4 * i;
          cp_async_16(wdst + (f / E) * EP + (f % E), wsrc + f, 16);
        }
      } else {
        for (int i = tid; i < HK * E; i += NTHR)
          cp_async_4(wdst + (i / E) * EP + (i % E), wsrc + i);
      }
      uint16_t* xdst = xst + buf * BTT * HK;
      constexpr int PPR = HK / 8;
      for (int i = tid; i < BTT * PPR; i += NTHR) {
        const int r = i / PPR, pc = i % PPR;
        const int t = t0 + r;
        const uint16_t* src = (t < T) ? x + (size_t)t * H + h0 + 8 * pc : x;
        cp_async_16(xdst + r * HK + 8 * pc, src, (t < T) ? 16 : 0);
      }
    }
    cp_async_commit();
  };

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

#pragma unroll
  for (int c = 0; c < NST - 1; ++c) issue_chunk(c);
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c % NST;
    // chunk c has landed; every thread is past chunk c-1, so its ring slot is free
    cp_async_wait<NST - 2>();
    __syncthreads();
    issue_chunk(c + NST - 1);
    float* xsc = xs + (c & 1) * HK * XL;  // two widened chunks (see route_kernel)
    for (int i = tid; i < BTT * HK / 4; i += NTHR) {
      const int r = i / (HK / 4), hq = (i % (HK / 4)) * 4;
      const uint2 v = *reinterpret_cast<const uint2*>(xst + buf * BTT * HK + r * HK + hq);
      xsc[(hq + 0) * XL + r] = bf16_lo(v.x);
      xsc[(hq + 1) * XL + r] = bf16_hi(v.x);
      xsc[(hq + 2) * XL + r] = bf16_lo(v.y);
      xsc[(hq + 3) * XL + r] = bf16_hi(v.y);
    }
    __syncthreads();
    const float* wsb = ws + buf * HK * EP;
#pragma unroll
    for (int hh = 0; hh < HK; ++hh) {
      float2 xp[8];
      load_x8(xsc + hh * XL + tb, 4 * LT, xp);
      const float4 wa = *reinterpret_cast<const float4*>(wsb + hh * EP + eb);
      const float4 wb = *reinterpret_cast<const float4*>(wsb + hh * EP + eb + 4 * LE);
      const float2 wp[4] = {make_float2(wa.x, wa.y), make_float2(wa.z, wa.w),
                            make_float2(wb.x, wb.y), make_float2(wb.z, wb.w)};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const float2 r = ffma2(xp[i], wp[p], make_float2(acc[i][2 * p], acc[i][2 * p + 1]));
          acc[i][2 * p] = r.x;
          acc[i][2 * p + 1] = r.y;
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // the logits below overwrite the ring

  constexpr int LLD = EP + 1;
  const bool add_bias = KIND == 0 && bias != nullptr;
  float* ls = reinterpret_cast<float*>(smem_f4);  // [BTT][LLD], over the drained ring
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = eb + ex(j);
    const float b = (add_bias && e < E) ? __ldg(bias + e) : 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float l = acc[i][j];
      if (add_bias) l = __fadd_rn(l, b);
      ls[(tb + tok(i)) * LLD + e] = l;
    }
  }
  __syncthreads();
  for (int tl = warp; tl < BTT; tl += NTHR / 32) {
    const int t = t0 + tl;
    if (t >= T) break;
    route_one_token<EP, KIND>(ls + tl * LLD, KIND == 1 ? bias : nullptr, E, k, wbf16, lane, t,
                              topk_idx, topk_w);
  }
}

// ------------------------------------------------ small T, CTA clusters ---
// route_cluster_kernel: a cluster of CC CTAs routes TSV tokens; CTA r owns the
// EC = EP / CC experts [r*EC, (r+1)*EC) and streams only those columns of W_r
// (EC*4 contiguous bytes per hidden row), so CC SMs share the weight traffic that
// one CTA carried alone.  Thread (tok, el) runs the FMA chain of token tok and
// expert r*EC + el over h = 0..H-1 (the same chain as the other router kernels),
// reading W_r and x from a cp.async ring (16-byte copies; x read eight hidden
// values per 16-byte load).  The logits go into the first CTA's
// shared memory (distributed shared memory), and after a cluster barrier its warps
// run the shared per-token epilogue.
constexpr int kCC = 8;       // CTAs per cluster (16, non-portable, up to 64 tokens)

template <int EP, int TSV, int CC = kCC>
struct ClusterCfg {
  static constexpr int EC = EP / CC;                   // experts per CTA
  static constexpr int HC = (EP >= 256) ? 128 : 256;   // hidden rows per stage
  static constexpr int CNST = (EP <= 64) ? 6 : 4;      // ring depth: 40-64 KB of W_r in flight
  static constexpr int NCMP = EC * TSV;                // computing threads
  static constexpr int NTH = NCMP < 128 ? 128 : NCMP;  // all of them copy
  static constexpr int LLD = EP + 1;
  static constexpr int ring = CNST * (HC * EC * 4 + TSV * HC * 2);
  static constexpr int bytes = ring + TSV * LLD * 4;
};

template <int EP, int TSV, int KIND, int CC>
__global__ void __launch_bounds__(ClusterCfg<EP, TSV, CC>::NTH)
    route_cluster_kernel(const uint16_t* __restrict__ x, const float* __restrict__ wr,
                         const float* __restrict__ bias, int T, int H, int E, int k, int wbf16,
                         int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  using C = ClusterCfg<EP, TSV, CC>;
  constexpr int EC = C::EC, HC = C::HC, NTH = C::NTH, LLD = C::LLD, CNST = C::CNST;
  extern __shared__ float4 smem_f4[];
  float* ws = reinterpret_cast<float*>(smem_f4);                    // [CNST][HC][EC]
  uint16_t* xst = reinterpret_cast<uint16_t*>(ws + CNST * HC * EC); // [CNST][TSV][HC]
  float* ls = reinterpret_cast<float*>(xst + CNST * TSV * HC);      // [TSV][LLD], CTA 0's used
  const int tid = threadIdx.x;
  const int rank = (int)cluster_ctarank();
  const int e0 = rank * EC;                  // this CTA's first expert
  const int t0 = (blockIdx.x / CC) * TSV;   // the cluster's first token
  const int nchunks = (H + HC - 1) / HC;  // the last one may hold fewer rows (H % 128 == 0)
  const int ecols = max(0, min(EC, E - e0));  // valid experts of this CTA
  // a programmatic dependent launch: x (often the previous kernel's output), the
  // router weights and the outputs are touched only after that kernel finished
  pdl_wait();
  if (tid == 0) pdl_launch_dependents();

  if (ecols < EC) {  // experts past E read zeros for the whole kernel
    for (int i = tid; i < CNST * HC * EC; i += NTH)
      if ((i % EC) >= ecols) ws[i] = 0.0f;
  }
  auto issue_chunk = [&](int c) {
    if (c < nchunks) {
      const int buf = c % CNST;
      const int h0 = c * HC;
      const int rows = min(HC, H - h0);
      float* wdst = ws + buf * HC * EC;
      if (ecols == EC && (E % 4) == 0) {
        constexpr int PPR = EC / 4;  // 16-byte pieces per hidden row
        for (int i = tid; i < rows * PPR; i += NTH) {
          const int r = i / PPR, pc = i % PPR;
          cp_async_16(wdst + r * EC + 4 * pc, wr + (size_t)(h0 + r) * E + e0 + 4 * pc, 16);
        }
      } else {
        for (int i = tid; i < rows * ecols; i += NTH) {
          const int r = i / ecols, c2 = i % ecols;
          cp_async_4(wdst + r * EC + c2, wr + (size_t)(h0 + r) * E + e0 + c2);
        }
      }
      const int XPR = rows / 8;  // 16-byte pieces per x row
      uint16_t* xdst = xst + buf * TSV * HC;
      for (int i = tid; i < TSV * XPR; i += NTH) {
        const int r = i / XPR, pc = i % XPR;
        const int t = t0 + r;
        const uint16_t* src = (t < T) ? x + (size_t)t * H + h0 + 8 * pc : x;
        cp_async_16(xdst + r * HC + 8 * pc, src, (t < T) ? 16 : 0);
      }
    }
    cp_async_commit();
  };

  const int el = tid % EC, tok = tid / EC;  // computing threads: tid < NCMP
  float acc = 0.0f;
#pragma unroll
  for (int c = 0; c < CNST - 1; ++c) issue_chunk(c);
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c % CNST;
    const int rows = min(HC, H - c * HC);
    issue_chunk(c + CNST - 1);
    cp_async_wait<CNST - 1>();
    __syncthreads();
    if (tid < C::NCMP) {
      const float* wsb = ws + buf * HC * EC + el;
      const uint16_t* xsb = xst + buf * TSV * HC + tok * HC;
      // eight hidden rows of the chain: the same FMAs in the same order either way
      auto step8 = [&](int hh) {
        const uint4 xv = *reinterpret_cast<const uint4*>(xsb + hh);
        acc = fmaf(bf16_lo(xv.x), wsb[(hh + 0) * EC], acc);
        acc = fmaf(bf16_hi(xv.x), wsb[(hh + 1) * EC], acc);
        acc = fmaf(bf16_lo(xv.y), wsb[(hh + 2) * EC], acc);
        acc = fmaf(bf16_hi(xv.y), wsb[(hh + 3) * EC], acc);
        acc = fmaf(bf16_lo(xv.z), wsb[(hh + 4) * EC], acc);
        acc = fmaf(bf16_hi(xv.z), wsb[(hh + 5) * EC], acc);
        acc = fmaf(bf16_lo(xv.w), wsb[(hh + 6) * EC], acc);
        acc = fmaf(bf16_hi(xv.w), wsb[(hh + 7) * EC], acc);
      };
      if (rows == HC) {
        // a whole chunk unrolled: every load is visible to the scheduler (an
        // isolated probe ran this loop at 6.2 instead of 6.9 cycles per FMA)
#pragma unroll
        for (int hh = 0; hh < HC; hh += 8) step8(hh);
      } else {
#pragma unroll 4
        for (int hh = 0; hh < rows; hh += 8) step8(hh);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  // logits (+ bias for the softmax router) into CTA 0's shared memory
  if (tid < C::NCMP && el < ecols) {
    const int e = e0 + el;
    float l = acc;
    if (KIND == 0 && bias != nullptr) l = __fadd_rn(l, __ldg(bias + e));
    const uint32_t dst = mapa_shared(smem_u32(ls + tok * LLD + e), 0);
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst), "f"(l) : "memory");
  }
  cluster_sync();
  if (rank == 0) {
    const int lane = tid & 31, warp = tid >> 5;
    for (int tl = warp; tl < TSV; tl += NTH / 32) {
      const int t = t0 + tl;
      if (t < T)
        route_one_token<EP, KIND>(ls + tl * LLD, KIND == 1 ? bias : nullptr, E, k, wbf16, lane,
                                  t, topk_idx, topk_w);
    }
  }
}

// ------------------------------------------------ decode (T <= 8): TMA ring ---
// route_decode_kernel: the sixteen-CTA cluster form for at most eight tokens with
// the W_r and x copies moved to the tensor memory accelerator.  CTA r owns the
// EC = EP/16 experts from r*EC; one thread streams boxes of HC hidden rows x EC
// experts of W_r and HC columns x TSV rows of x into a ring of CNST stages, each
// completing on its own mbarrier.  The computing threads (one per expert and
// token) wait on that barrier alone and free a stage with one arrival per warp:
// no CTA-wide barrier sits inside the FMA chains.  Each logit is the same chain
// over h = 0..H-1 as in the other kernels, then the bias add; the logits meet in
// CTA 0, which runs the shared epilogue.  Measured on GB300 against the
// cp.async form (per-thread 16-byte copies, two CTA barriers per chunk), whose
// time grew with a deeper ring: see the launcher.
template <int EP, int TSV>
struct DecodeCfg {
  static constexpr int CC = 16;
  static constexpr int EC = EP / CC;
  static constexpr int BR = 256;                     // hidden rows per box (the TMA maximum)
  static constexpr int NB = 2;                       // boxes per stage
  static constexpr int HC = NB * BR;                 // hidden rows per stage
  static constexpr int NCMP = EC * TSV;              // computing threads
  static constexpr int CW = (NCMP + 31) / 32;        // computing warps
  static constexpr int NTH = 32 * (1 + CW);          // + the copy warp
  static constexpr int WB_BYTES = BR * EC * 4;       // one W_r box [BR][EC]
  static constexpr int XB_BYTES = TSV * BR * 2;      // one x box [TSV][BR]
  static constexpr int W_BYTES = NB * WB_BYTES;
  static constexpr int X_BYTES = NB * XB_BYTES;
  static constexpr int STAGE = W_BYTES + X_BYTES;
  static constexpr int CNST = (160 * 1024 / STAGE) < 16 ? 160 * 1024 / STAGE : 16;
  static constexpr int LLD = EP + 1;
  static constexpr int bytes = 128 + CNST * STAGE + 2 * CNST * 8 + 16 + TSV * LLD * 4;
  static_assert(EC >= 4 && WB_BYTES % 128 == 0 && XB_BYTES % 128 == 0, "TMA boxes");
  static_assert(bytes <= 227 * 1024, "shared memory");
};

struct DecodeMaps {
  CUtensorMap w;  // W_r [H][E] FP32, box EC x BR
  CUtensorMap x;  // x [T][H] BF16, box BR x TSV
};

// Bounded parity wait without a status word (the router has none): false once
// *abort is raised or `limit` cycles pass (then it raises *abort).
__device__ __forceinline__ bool route_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                           long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      *abort = 1;
      return false;
    }
  }
}

template <int EP, int TSV, int KIND>
__global__ void __launch_bounds__(DecodeCfg<EP, TSV>::NTH)
    route_decode_kernel(const __grid_constant__ DecodeMaps maps, const float* __restrict__ bias,
                        int T, int H, int E, int k, int wbf16, int32_t* __restrict__ topk_idx,
                        float* __restrict__ topk_w, long long spin_limit) {
  using C = DecodeCfg<EP, TSV>;
  constexpr int EC = C::EC, HC = C::HC, CNST = C::CNST, LLD = C::LLD;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  uint8_t* sW = base;                                   // [CNST][HC][EC] FP32
  uint8_t* sX = base + CNST * C::W_BYTES;               // [CNST][TSV][HC] BF16
  uint64_t* full = reinterpret_cast<uint64_t*>(sX + CNST * C::X_BYTES);
  uint64_t* empty = full + CNST;
  int* s_err = reinterpret_cast<int*>(empty + CNST);    // CTA 0's: the cluster's error flag
  volatile int* abort_flag = s_err + 1;                 // this CTA's
  float* ls = reinterpret_cast<float*>(s_err + 4);      // [TSV][LLD], CTA 0's used
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)cluster_ctarank();
  const int e0 = rank * EC;
  const int t0 = (blockIdx.x / C::CC) * TSV;
  // a CTA whose experts all lie past E copies and computes nothing
  const int nchunks = e0 < E ? (H + HC - 1) / HC : 0;

  if (tid == 0) {
    for (int s = 0; s < CNST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::CW);
    }
    *s_err = 0;
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&maps.w);
    prefetch_tensormap(&maps.x);
  }
  __syncthreads();
  // first cluster phase: every CTA's flag is initialised before any remote write
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  // a programmatic dependent launch: x, W_r and the outputs are touched after the
  // previous kernel finished
  pdl_wait();
  if (tid == 0) pdl_launch_dependents();

  float acc = 0.0f;
  const int ct = tid - 32;
  const int el = ct % EC, tok = ct / EC;
  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- copies
      int c = 0;
      for (; c < nchunks; ++c) {
        const int s = c % CNST;
        const uint32_t ph = (c / CNST) & 1;
        if (!route_wait(&empty[s], ph ^ 1, abort_flag, spin_limit)) break;
        // boxes that start inside H (none lies wholly past the tensor)
        const int nbx = min(C::NB, (H - c * HC + C::BR - 1) / C::BR);
        mbar_arrive_expect_tx(&full[s], nbx * (C::WB_BYTES + C::XB_BYTES));
        for (int b = 0; b < nbx; ++b) {
          tma_load_2d(&maps.w, sW + s * C::W_BYTES + b * C::WB_BYTES, &full[s], e0,
                      c * HC + b * C::BR);
          tma_load_2d(&maps.x, sX + s * C::X_BYTES + b * C::XB_BYTES, &full[s], c * HC + b * C::BR,
                      t0);
        }
      }
      if (*abort_flag) {  // let the copies in flight land before the CTA exits
        for (int i = (c > CNST ? c - CNST : 0); i < c; ++i)
          wait_drain(&full[i % CNST], (i / CNST) & 1, kSpinLimitCycles);
      }
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------------- chains
    const bool active = ct < C::NCMP;
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % CNST;
      const uint32_t ph = (c / CNST) & 1;
      const bool ok = __all_sync(0xFFFFFFFFu, route_wait(&full[s], ph, abort_flag, spin_limit));
      if (!ok) break;
      if (active) {
        const int rows = min(HC, H - c * HC);
        // the stage's W_r rows are contiguous over its boxes; its x holds one
        // [TSV][BR] box after the other
        const float* wsb = reinterpret_cast<const float*>(sW + s * C::W_BYTES) + el;
        const uint16_t* xs0 = reinterpret_cast<const uint16_t*>(sX + s * C::X_BYTES) + tok * C::BR;
        const uint16_t* xsb = xs0;
        auto step8 = [&](int hh) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xsb + hh);
          acc = fmaf(bf16_lo(xv.x), wsb[(hh + 0) * EC], acc);
          acc = fmaf(bf16_hi(xv.x), wsb[(hh + 1) * EC], acc);
          acc = fmaf(bf16_lo(xv.y), wsb[(hh + 2) * EC], acc);
          acc = fmaf(bf16_hi(xv.y), wsb[(hh + 3) * EC], acc);
          acc = fmaf(bf16_lo(xv.z), wsb[(hh + 4) * EC], acc);
          acc = fmaf(bf16_hi(xv.z), wsb[(hh + 5) * EC], acc);
          acc = fmaf(bf16_lo(xv.w), wsb[(hh + 6) * EC], acc);
          acc = fmaf(bf16_hi(xv.w), wsb[(hh + 7) * EC], acc);
        };
        // step8(hh) reads x at xsb + hh: box b's x starts at xs0 + b * (XB - BR) elements
        // before row b * BR, so xsb moves back by that much for each later box
        if (rows == HC) {
#pragma unroll
          for (int b = 0; b < C::NB; ++b) {
            xsb = xs0 + b * (C::XB_BYTES / 2 - C::BR);
#pragma unroll
            for (int hh = b * C::BR; hh < (b + 1) * C::BR; hh += 8) step8(hh);
          }
        } else {
          for (int b = 0; b < C::NB && b * C::BR < rows; ++b) {
            xsb = xs0 + b * (C::XB_BYTES / 2 - C::BR);
            const int hend = min(rows, (b + 1) * C::BR);
#pragma unroll 4
            for (int hh = b * C::BR; hh < hend; hh += 8) step8(hh);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (*abort_flag) {
    if (tid == 0) {
      const uint32_t dst = mapa_shared(smem_u32(s_err), 0);
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(dst), "r"(1) : "memory");
    }
  } else if (warp > 0 && ct < C::NCMP && e0 + el < E) {
    const int e = e0 + el;
    float l = acc;
    if (KIND == 0 && bias != nullptr) l = __fadd_rn(l, __ldg(bias + e));
    const uint32_t dst = mapa_shared(smem_u32(ls + tok * LLD + e), 0);
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst), "f"(l) : "memory");
  }
  cluster_sync();
  if (rank == 0) {
    for (int tl = warp; tl < TSV; tl += C::NTH / 32) {
      const int t = t0 + tl;
      if (t >= T) continue;
      if (*s_err) {  // a wait ran out: no routing (the dispatch rejects index -1)
        if (lane < k) {
          topk_idx[(size_t)t * k + lane] = -1;
          topk_w[(size_t)t * k + lane] = 0.0f;
        }
      } else {
        route_one_token<EP, KIND>(ls + tl * LLD, KIND == 1 ? bias : nullptr, E, k, wbf16, lane,
                                  t, topk_idx, topk_w);
      }
    }
  }
}

template <int EP, int TSV, int KIND, int CC = kCC>
cudaError_t launch_cluster(const void* x, const float* wr, const float* bias, int T, int H, int E,
                           int k, int wbf16, int32_t* idx, float* w, cudaStream_t s) {
  using C = ClusterCfg<EP, TSV, CC>;
  auto kern = route_cluster_kernel<EP, TSV, KIND, CC>;
  static int ok[64] = {};  // 0: unknown, 1: launchable, -1: this cluster size does not fit
  int dv = 0;
  cudaGetDevice(&dv);
  const int known = dv < 64 ? ok[dv] : 0;
  if constexpr (CC > kCC) {  // only a non-portable size can be refused
    if (known < 0)
      return launch_cluster<EP, TSV, KIND, kCC>(x, wr, bias, T, H, E, k, wbf16, idx, w, s);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  pdl_attr(attr[1]);
  cfg.gridDim = dim3(CC * ((T + TSV - 1) / TSV));
  cfg.blockDim = dim3(C::NTH);
  cfg.dynamicSmemBytes = C::bytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (known == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::bytes);
    if (e != cudaSuccess) return e;
    if constexpr (CC > 8) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      int clusters = 0;
      cfg.numAttrs = 1;  // the query takes the cluster shape alone
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
      cfg.numAttrs = 2;
      if (e != cudaSuccess || clusters < 1) {
        (void)cudaGetLastError();
        if (dv < 64) ok[dv] = -1;
        return launch_cluster<EP, TSV, KIND, kCC>(x, wr, bias, T, H, E, k, wbf16, idx, w, s);
      }
    }
    if (dv < 64) ok[dv] = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const uint16_t*>(x), wr, bias, T, H, E, k,
                            wbf16, idx, w);
}

template <int EP, int TSV, int KIND>
cudaError_t launch_decode(const void* x, const float* wr, const float* bias, int T, int H, int E,
                          int k, int wbf16, int32_t* idx, float* w, cudaStream_t s) {
  using C = DecodeCfg<EP, TSV>;
  auto kern = route_decode_kernel<EP, TSV, KIND>;
  static int ok[64] = {};  // 0: unknown, 1: launchable, -1: a 16-CTA cluster does not fit
  int dv = 0;
  cudaGetDevice(&dv);
  const int known = dv < 64 ? ok[dv] : 0;
  DecodeMaps m;
  if (known < 0 || (E % 4) != 0 ||
      !encode_rowmajor_2d(&m.w, wr, (uint64_t)E, (uint64_t)H, true, C::EC, C::BR) ||
      !encode_rowmajor_2d(&m.x, x, (uint64_t)H, (uint64_t)T, false, C::BR, TSV))
    return launch_cluster<EP, TSV, KIND, 16>(x, wr, bias, T, H, E, k, wbf16, idx, w, s);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C::CC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  pdl_attr(attr[1]);
  cfg.gridDim = dim3(C::CC * ((T + TSV - 1) / TSV));
  cfg.blockDim = dim3(C::NTH);
  cfg.dynamicSmemBytes = C::bytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (known == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::bytes);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    int clusters = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess || clusters < 1) {
      (void)cudaGetLastError();
      if (dv < 64) ok[dv] = -1;
      return launch_cluster<EP, TSV, KIND, 16>(x, wr, bias, T, H, E, k, wbf16, idx, w, s);
    }
    if (dv < 64) ok[dv] = 1;
  }
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, m, bias, T, H, E, k, wbf16, idx, w, kSpinLimitCycles);
}

template <int EP, int KIND>
cudaError_t launch_ep(const void* x, const float* wr, const float* bias, int T, int H, int E, int k,
                      int wbf16, int32_t* idx, float* w, cudaStream_t s) {
  if (T <= kRouteSmallMaxT) {
    // one cluster holds every token (T <= 8) and there are 64 experts or more:
    // sixteen CTAs, four or more experts each.  Measured on GB300 (router stage,
    // L2 flushed): large T = 8 38 against 46 us, T = 1 33 against 34 us;
    // fine_grained T = 1 17 against 18 us; at T = 64 eight CTAs were 2 us faster.
    if constexpr (EP >= 64) {
      if (T == 1) return launch_decode<EP, 1, KIND>(x, wr, bias, T, H, E, k, wbf16, idx, w, s);
      if (T == 2) return launch_decode<EP, 2, KIND>(x, wr, bias, T, H, E, k, wbf16, idx, w, s);
      if (T <= 4) return launch_decode<EP, 4, KIND>(x, wr, bias, T, H, E, k, wbf16, idx, w, s);
      if (T <= 8) return launch_decode<EP, 8, KIND>(x, wr, bias, T, H, E, k, wbf16, idx, w, s);
    }
    if (T == 1) return launch_cluster<EP, 1, KIND>(x, wr, bias, T, H, E, k, wbf16, idx, w, s);
    if (T == 2) return launch_cluster<EP, 2, KIND>(x, wr, bias, T, H, E, k, wbf16, idx, w, s);
    if (T <= 4) return launch_cluster<EP, 4, KIND>(x, wr, bias, T, H, E, k, wbf16, idx, w, s);
    if (T <= 8) return launch_cluster<EP, 8, KIND>(x, wr, bias, T, H, E, k, wbf16, idx, w, s);
    return launch_cluster<EP, 8, KIND>(x, wr, bias, T, H, E, k, wbf16, idx, w, s);
  }
  // Clusters of eight tokens up to kRouteClusterMaxT.  Measured on GB300 (router
  // stage, L2 flushed): fine_grained T = 128 / 512: 27 / 49 us against 77 / 78 us
  // for route_kernel; large T = 256: 84 against 314 us.  From about 1000 tokens
  // route_kernel (all experts of 32 tokens per CTA) is faster: fine_grained
  // T = 2048: 79 against 137 us; large T = 2048: 321 against 537 us.
  if (T <= kRouteClusterMaxT)
    return launch_cluster<EP, 8, KIND>(x, wr, bias, T, H, E, k, wbf16, idx, w, s);
  if constexpr (EP == 256) {
    // 2D tiles once T gives every SM at least one CTA.  Measured on GB300: 5% faster
    // than route_kernel for 256 experts; for 64 and 128 experts (fewer experts per
    // token, larger token tiles) it was 15-45% slower, so those keep route_kernel.
    using TC = TileCfg<EP>;
    int sms = device_sm_count();
    if ((long long)T >= (long long)sms * TC::BT) {
      static bool tattr[64] = {};
      int dv = 0;
      cudaGetDevice(&dv);
      if (dv < 64 && !tattr[dv]) {
        cudaError_t e = cudaFuncSetAttribute(route_tile_kernel<EP, KIND>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, TC::bytes);
        if (e != cudaSuccess) return e;
        tattr[dv] = true;
      }
      route_tile_kernel<EP, KIND><<<(T + TC::BT - 1) / TC::BT, NTHR, TC::bytes, s>>>(
          static_cast<const uint16_t*>(x), wr, bias, T, H, E, k, wbf16, idx, w);
      return cudaGetLastError();
    }
  }
  constexpr int smem = RouteCfg<EP>::bytes;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(route_kernel<EP, KIND>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  dim3 grid((T + BT - 1) / BT);
  route_kernel<EP, KIND><<<grid, NTHR, smem, s>>>(static_cast<const uint16_t*>(x), wr, bias, T, H,
                                                  E, k, wbf16, idx, w);
  return cudaGetLastError();
}

template <int KIND>
cudaError_t launch_kind(const void* x, const float* w_router, const float* bias, int T, int H,
                        int E, int k, int wbf16, int32_t* topk_idx, float* topk_w, cudaStream_t s) {
  if (E <= 32) return launch_ep<32, KIND>(x, w_router, bias, T, H, E, k, wbf16, topk_idx, topk_w, s);
  if (E <= 64) return launch_ep<64, KIND>(x, w_router, bias, T, H, E, k, wbf16, topk_idx, topk_w, s);
  if (E <= 128)
    return launch_ep<128, KIND>(x, w_router, bias, T, H, E, k, wbf16, topk_idx, topk_w, s);
  return launch_ep<256, KIND>(x, w_router, bias, T, H, E, k, wbf16, topk_idx, topk_w, s);
}

}  // namespace

cudaError_t launch_route(const void* x, const float* w_router, const float* bias, int T, int H,
                         int E, int k, int kind, int weights_bf16, int32_t* topk_idx,
                         float* topk_w, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (kind == 1)
    return launch_kind<1>(x, w_router, bias, T, H, E, k, weights_bf16, topk_idx, topk_w, s);
  return launch_kind<0>(x, w_router, bias, T, H, E, k, weights_bf16, topk_idx, topk_w, s);
}

}  // namespace moe
