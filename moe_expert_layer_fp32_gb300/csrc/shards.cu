// Expert ranks without the exchange: per-rank BF16 partials and the fixed FP64
// expert-output reduction, on one GPU.
//
// "0 train-infer mismatch for open-weight MoE RL", section "Sharding the experts":
// a rank accumulates every routing slot of a token in FP32 in slot order (slots
// whose expert another rank owns add exact zeros), adds its shard of the shared
// expert, and rounds once to BF16.  The G partials are then placed in logical
// rank order and reduced by adjacent pairs in FP64, an odd last partial carried
// to the next level unchanged, with one BF16 rounding at the end.
//
// combine_sharded_kernel runs all G ranks of one token in one CTA: the k gathered
// FP32 rows are read once, the G chains, the G roundings and the tree all stay in
// registers, and only the final BF16 row (plus the partials, when asked for) is
// written.  tree_reduce_kernel is the reduction alone, for partials that another
// engine delivered: G BF16 rows in, one BF16 row out, 16-byte vectors.
//
// Format conversions are integer bit manipulation: bf16 -> f64 widens exactly, and
// f64 -> bf16 rounds once to nearest even from the full 52-bit fraction, so no
// value passes through FP32 on its way out (that would round twice).
//
// FP64 is a narrow pipe on this GPU, so the tree runs in FP32 wherever that is
// provably the same.  Every leaf is a bf16 value (8 significant bits).  A group of
// leaves whose exponents lie within W = 16 - ceil(log2 G) binades of each other
// sums exactly in FP32 (the sum of their magnitudes stays below 2^24 units of the
// smallest one), in any order.  The leaves are split at W binades below the
// largest exponent into two such groups, H and L; if the smallest non-zero leaf is
// within 2W + 1 binades of the largest, both sums are exact and H + L is the exact
// sum of all leaves.  So is the FP64 tree's result: every node of it is a partial
// sum of fewer than 2^53 units, hence exact.  H + L is rounded once to bf16:
// s = fl(H + L) plus its exact TwoSum error decides the one case where s alone
// cannot, a tie.  Both accumulators start at -0, so an all -0 input gives -0 and
// any exact zero sum of other leaves +0, as IEEE addition in the tree gives it.
// Wider spreads, leaves from 2^124 up (no FP32 overflow), infinities and NaNs take
// the FP64 tree itself.
//
// The per-rank chains: a slot whose expert another rank owns adds w * 0 = +-0 to
// that rank's accumulator, which changes nothing except -0 + +0 = +0 when w has a
// clear sign bit.  Per token (the same for every column) the CTA works out, for
// each slot, whether its owner's accumulator must first be normalised (acc + 0.0f)
// because such a slot came after the owner's previous FMA, and for each rank
// whether it needs that at the end.  Each slot then costs one FMA into its own
// rank's accumulator instead of G masked FMAs.  A token with a non-finite weight
// runs the chains literally.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

// Exact widening of bf16 bits to FP64.
__device__ __forceinline__ double bf16_bits_to_f64(uint32_t b) {
  const uint32_t s = (b & 0x8000u) << 16;
  const uint32_t e = (b >> 7) & 0xFFu;
  const uint32_t m = b & 0x7Fu;
  uint32_t hi;
  if (e == 0xFFu) {
    hi = s | 0x7FF00000u | (m << 13);  // inf / NaN
  } else if (e != 0u) {
    hi = s | ((e + 896u) << 20) | (m << 13);  // rebias 127 -> 1023
  } else if (m == 0u) {
    hi = s;  // signed zero
  } else {
    // subnormal m * 2^-133: leading bit p of m becomes the implicit one
    const uint32_t p = 31u - __clz(m);
    hi = s | ((p + 890u) << 20) | ((m ^ (1u << p)) << (20u - p));
  }
  return __hiloint2double((int)hi, 0);
}

// FP64 -> bf16 bits, one rounding to nearest even (NaN -> 0x7FC0).
__device__ __forceinline__ uint32_t f64_to_bf16_bits(double x) {
  const uint32_t hi = (uint32_t)__double2hiint(x), lo = (uint32_t)__double2loint(x);
  const uint32_t s = (hi >> 16) & 0x8000u;
  const int ex = (int)((hi >> 20) & 0x7FFu);
  const uint32_t mh = hi & 0xFFFFFu;  // top 20 fraction bits
  if (ex == 0x7FF) return (mh | lo) ? 0x7FC0u : (s | 0x7F80u);
  const int E = ex - 1023;
  if (E >= -126) {
    // keep 7 fraction bits; the discarded part is mh[12:0] and lo
    const uint32_t rh = mh & 0x1FFFu;
    const bool above = rh > 0x1000u || (rh == 0x1000u && lo != 0u);
    const bool tie = rh == 0x1000u && lo == 0u;
    uint32_t r = ((uint32_t)(E + 127) << 7) | (mh >> 13);  // a carry moves into the exponent
    if (above || (tie && (r & 1u))) r += 1u;
    return r >= 0x7F80u ? (s | 0x7F80u) : (s | r);
  }
  if (ex == 0) return s;  // FP64 subnormals are far below half the smallest bf16
  // bf16 subnormal range: units of 2^-133; value = full * 2^(E-52), so the unit
  // count is full >> (-(E + 81)) with full the 53-bit significand
  const int rsh = -(E + 81);  // >= 46 here
  if (rsh > 63) return s;
  const unsigned long long full = (1ull << 52) | ((unsigned long long)mh << 32) | lo;
  unsigned long long q = full >> rsh;
  const unsigned long long rem = full & ((1ull << rsh) - 1ull);
  const unsigned long long half = 1ull << (rsh - 1);
  if (rem > half || (rem == half && (q & 1ull))) q += 1ull;
  return s | (uint32_t)q;  // q = 128 is the smallest normal, which this encodes
}

// In-place fixed tree over v[0..N): adjacent pairs per level, odd last carried.
template <int N>
__device__ __forceinline__ void fp64_tree(double* v) {
  if constexpr (N > 1) {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) v[i] = __dadd_rn(v[2 * i], v[2 * i + 1]);
    if constexpr ((N & 1) != 0) v[N / 2] = v[N - 1];
    fp64_tree<(N + 1) / 2>(v);
  }
}

__host__ __device__ constexpr int ceil_log2(int n) { return n <= 1 ? 0 : 1 + ceil_log2((n + 1) / 2); }

__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// bf16 bits of s + err, rounded to nearest even, where s = fl(H + L) and err is
// its exact rounding error (|err| <= half an FP32 ulp of s).
__device__ __forceinline__ uint32_t round_pair_to_bf16(float s, float err) {
  const uint32_t u = __float_as_uint(s);
  const uint32_t low = u & 0xFFFFu;
  uint32_t b = u >> 16;  // truncated towards zero (sign-magnitude)
  if (low > 0x8000u) {
    b += 1u;
  } else if (low == 0x8000u) {  // s is a tie: err breaks it, else the even side
    if (err == 0.0f) b += b & 1u;
    else if ((__float_as_uint(err) ^ u) >> 31 == 0u) b += 1u;  // err points away from zero
  }
  // low < 0x8000: s + err stays below the tie (err is under half an FP32 ulp)
  return b;
}

// bf16(FP64 tree over the G bf16 leaves `b`).  active: leaves that may be non-zero;
// the others are known to be +0 (a rank that owns no slot of the token).
template <int G>
__device__ __forceinline__ uint32_t reduce_leaves(const uint32_t* b, uint32_t active) {
  if constexpr (G == 1) {  // no addition: the value itself (NaN as the FP64 path gives it)
    return ((b[0] & 0x7F80u) == 0x7F80u && (b[0] & 0x7Fu)) ? 0x7FC0u : b[0];
  }
  constexpr int kW = 16 - ceil_log2(G);
  constexpr uint32_t kAll = (1u << G) - 1u;
  int e_max = 0, e_min = 255;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if ((active >> g) & 1u) {
      const int e = (int)((b[g] >> 7) & 0xFFu);
      const bool nz = (b[g] & 0x7FFFu) != 0u;
      e_max = max(e_max, e);
      e_min = nz ? min(e_min, max(e, 1)) : e_min;  // subnormals: the spacing of e = 1
    }
  }
  // e_max <= 250: leaves below 2^124; e = 255 (inf / NaN) fails it too
  if (e_max <= 250 && e_max - e_min <= 2 * kW + 1) {
    const int split = e_max - kW;  // H: e >= split (within kW of e_max), L: the rest
    float h = ((active & kAll) == kAll) ? -0.0f : 0.0f;  // a known +0 leaf joins as +0
    float l = -0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if ((active >> g) & 1u) {
        const float v = __uint_as_float(b[g] << 16);
        const bool hi = (int)((b[g] >> 7) & 0xFFu) >= split;
        h = __fadd_rn(h, hi ? v : -0.0f);
        l = __fadd_rn(l, hi ? -0.0f : v);
      }
    }
    const float s = __fadd_rn(h, l);
    const float bv = __fsub_rn(s, h);
    const float err = __fadd_rn(__fsub_rn(h, __fsub_rn(s, bv)), __fsub_rn(l, bv));
    return round_pair_to_bf16(s, err);
  }
  double d[G];
#pragma unroll
  for (int g = 0; g < G; ++g) d[g] = bf16_bits_to_f64(((active >> g) & 1u) ? b[g] : 0u);
  fp64_tree<G>(d);
  return f64_to_bf16_bits(d[0]);
}

// Per-token chain schedule (see the header).  norm_pre bit j: normalise slot j's
// owner before its FMA; norm_end bit g: normalise rank g after the last slot;
// literal: a weight is not finite, run the chains as written.
struct ChainPlan {
  uint32_t norm_pre, norm_end;
  uint32_t active;  // ranks owning at least one slot (all ranks when shards are added)
  int literal;
};

// Slots with an invalid row contribute nothing to any rank and are left out.
__device__ __forceinline__ ChainPlan plan_chains(const int* row, const int* own, const float* w,
                                                 int k, int G) {
  ChainPlan p{0u, 0u, 0u, 0};
  uint32_t started = 0u, pending = 0u;
  const uint32_t all = (G >= 32) ? 0xFFFFFFFFu : ((1u << G) - 1u);
  for (int j = 0; j < k; ++j) {
    if (row[j] < 0) continue;
    if (!isfinite(w[j])) p.literal = 1;
    const int o = own[j];
    const uint32_t ob = (o >= 0) ? (1u << o) : 0u;
    if (started & pending & ob) p.norm_pre |= 1u << j;
    started |= ob;
    pending &= ~ob;
    if (!signbit(w[j])) pending |= all & ~ob;  // w * 0 = +0: -0 becomes +0 in the others
  }
  p.norm_end = started & pending;
  p.active = started;
  return p;
}

__device__ __forceinline__ float norm0(float a) { return __fadd_rn(a, 0.0f); }

// One CTA per token, CPT consecutive columns per thread.
template <int G, int CPT>
__global__ void __launch_bounds__(128) combine_sharded_kernel(
    const float* __restrict__ y, const float* __restrict__ topk_w,
    const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ row_of_slot,
    const int32_t* __restrict__ owner, int T, int H, int E, int k, float scale,
    const float* __restrict__ shared, uint16_t* __restrict__ partials, uint16_t* __restrict__ out) {
  __shared__ int s_row[kMaxK];
  __shared__ int s_own[kMaxK];
  __shared__ float s_w[kMaxK];
  __shared__ ChainPlan s_plan;
  const int t = blockIdx.x;
  const long long R = (long long)T * k;
  if (threadIdx.x < k) {
    const int j = threadIdx.x;
    const int r = row_of_slot[(size_t)t * k + j];
    const int e = topk_idx[(size_t)t * k + j];
    const int o = (e >= 0 && e < E) ? owner[e] : -1;
    s_row[j] = (r >= 0 && r < R) ? r : -1;
    s_own[j] = (o >= 0 && o < G) ? o : -1;  // -1: no rank owns the slot
    s_w[j] = __fmul_rn(scale, topk_w[(size_t)t * k + j]);
  }
  __syncthreads();
  if (threadIdx.x == 0) s_plan = plan_chains(s_row, s_own, s_w, k, G);
  __syncthreads();
  const ChainPlan plan = s_plan;
  // with shards added every rank's partial may be non-zero; a literal token keeps all
  const uint32_t active = (shared != nullptr || plan.literal) ? 0xFFFFu : plan.active;
  int row[kMaxK], own[kMaxK];
  float w[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    row[j] = (j < k) ? s_row[j] : -1;
    own[j] = (j < k) ? s_own[j] : -1;
    w[j] = (j < k) ? s_w[j] : 0.0f;
  }
  for (int c0 = threadIdx.x * CPT; c0 < H; c0 += blockDim.x * CPT) {
    float v[kMaxK][CPT];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (row[j] >= 0) {
        const float* src = y + (size_t)row[j] * H + c0;
        if constexpr (CPT == 4) {
          const float4 q = __ldg(reinterpret_cast<const float4*>(src));
          v[j][0] = q.x; v[j][1] = q.y; v[j][2] = q.z; v[j][3] = q.w;
        } else {
          const float2 q = __ldg(reinterpret_cast<const float2*>(src));
          v[j][0] = q.x; v[j][1] = q.y;
        }
      } else {
#pragma unroll
        for (int c = 0; c < CPT; ++c) v[j][c] = 0.0f;
      }
    }
    float acc[G][CPT];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int c = 0; c < CPT; ++c) acc[g][c] = 0.0f;
    if (!plan.literal) {
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k && row[j] >= 0) {
          const bool pre = (plan.norm_pre >> j) & 1u;
          switch (own[j]) {  // the same value in every thread of the CTA
#define MOE_SLOT_CASE(n)                                                     \
  case n:                                                                    \
    if constexpr (n < G) {                                                   \
      _Pragma("unroll") for (int c = 0; c < CPT; ++c) {                      \
        const float a = pre ? norm0(acc[n][c]) : acc[n][c];                  \
        acc[n][c] = fmaf(w[j], v[j][c], a);                                  \
      }                                                                      \
    }                                                                        \
    break;
            MOE_SLOT_CASE(0) MOE_SLOT_CASE(1) MOE_SLOT_CASE(2) MOE_SLOT_CASE(3)
            MOE_SLOT_CASE(4) MOE_SLOT_CASE(5) MOE_SLOT_CASE(6) MOE_SLOT_CASE(7)
            MOE_SLOT_CASE(8) MOE_SLOT_CASE(9) MOE_SLOT_CASE(10) MOE_SLOT_CASE(11)
            MOE_SLOT_CASE(12) MOE_SLOT_CASE(13) MOE_SLOT_CASE(14) MOE_SLOT_CASE(15)
#undef MOE_SLOT_CASE
            default:
              break;
          }
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g)
        if ((plan.norm_end >> g) & 1u)
#pragma unroll
          for (int c = 0; c < CPT; ++c) acc[g][c] = norm0(acc[g][c]);
    } else {
      // the chains as written: every rank, every slot, y or an exact zero
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < kMaxK; ++j)
          if (row[j] >= 0)
#pragma unroll
            for (int c = 0; c < CPT; ++c)
              acc[g][c] = fmaf(w[j], own[j] == g ? v[j][c] : 0.0f, acc[g][c]);
    }
    uint32_t pb[CPT][G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (shared != nullptr) {
        const float* sp = shared + ((size_t)g * T + t) * H + c0;
        if constexpr (CPT == 4) {
          const float4 q = __ldg(reinterpret_cast<const float4*>(sp));
          acc[g][0] = __fadd_rn(acc[g][0], q.x); acc[g][1] = __fadd_rn(acc[g][1], q.y);
          acc[g][2] = __fadd_rn(acc[g][2], q.z); acc[g][3] = __fadd_rn(acc[g][3], q.w);
        } else {
          const float2 q = __ldg(reinterpret_cast<const float2*>(sp));
          acc[g][0] = __fadd_rn(acc[g][0], q.x); acc[g][1] = __fadd_rn(acc[g][1], q.y);
        }
      }
#pragma unroll
      for (int c = 0; c < CPT; ++c) pb[c][g] = f32_to_bf16_bits(acc[g][c]);
      if (partials != nullptr) {
        uint16_t* pp = partials + ((size_t)g * T + t) * H + c0;
        if constexpr (CPT == 4) {
          *reinterpret_cast<uint2*>(pp) =
              make_uint2(pb[0][g] | (pb[1][g] << 16), pb[2][g] | (pb[3][g] << 16));
        } else {
          *reinterpret_cast<uint32_t*>(pp) = pb[0][g] | (pb[1][g] << 16);
        }
      }
    }
    uint32_t ob[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) ob[c] = reduce_leaves<G>(pb[c], active);
    uint16_t* op = out + (size_t)t * H + c0;
    if constexpr (CPT == 4) {
      *reinterpret_cast<uint2*>(op) = make_uint2(ob[0] | (ob[1] << 16), ob[2] | (ob[3] << 16));
    } else {
      *reinterpret_cast<uint32_t*>(op) = ob[0] | (ob[1] << 16);
    }
  }
}

// out[n] = bf16(tree(partials[0..G-1][n])).  VEC: 8 elements per 16-byte vector
// (every row base 16-byte aligned), else one element per step.
template <int G, bool VEC>
__global__ void __launch_bounds__(256) tree_reduce_kernel(const uint16_t* __restrict__ partials,
                                                          long long N, uint16_t* __restrict__ out) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long first = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if constexpr (VEC) {
    const long long nv = N / 8;
    for (long long i = first; i < nv; i += stride) {
      uint4 q[G];
#pragma unroll
      for (int g = 0; g < G; ++g)
        q[g] = __ldg(reinterpret_cast<const uint4*>(partials + (size_t)g * N) + i);
      uint32_t o[4];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        uint32_t b[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const uint32_t word = (&q[g].x)[h >> 1];
          b[g] = (h & 1) ? (word >> 16) : (word & 0xFFFFu);
        }
        const uint32_t r = reduce_leaves<G>(b, 0xFFFFu);
        if (h & 1) o[h >> 1] |= r << 16;
        else o[h >> 1] = r;
      }
      reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  } else {
    for (long long n = first; n < N; n += stride) {
      uint32_t b[G];
#pragma unroll
      for (int g = 0; g < G; ++g) b[g] = __ldg(partials + (size_t)g * N + n);
      out[n] = (uint16_t)reduce_leaves<G>(b, 0xFFFFu);
    }
  }
}

template <int G>
cudaError_t launch_tree_g(const uint16_t* p, long long N, uint16_t* out, bool vec, cudaStream_t s) {
  const long long units = vec ? N / 8 : N;
  if (units == 0) return cudaSuccess;
  const long long want = (units + 255) / 256;
  const int cap = device_sm_count() * 8;
  const int grid = (int)(want < cap ? want : cap);
  if (vec) tree_reduce_kernel<G, true><<<grid, 256, 0, s>>>(p, N, out);
  else tree_reduce_kernel<G, false><<<grid, 256, 0, s>>>(p, N, out);
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_combine_sharded_g(const float* y, const float* topk_w, const int32_t* topk_idx,
                                     const int32_t* row_of_slot, const int32_t* owner, int T, int H,
                                     int E, int k, float scale, const float* shared,
                                     uint16_t* partials, uint16_t* out, cudaStream_t s) {
  constexpr int CPT = G <= 8 ? 4 : 2;  // fewer columns per thread keep G > 8 in registers
  combine_sharded_kernel<G, CPT><<<T, 128, 0, s>>>(y, topk_w, topk_idx, row_of_slot, owner, T, H,
                                                   E, k, scale, shared, partials, out);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tree_reduce(const void* partials, int G, long long N, void* out, bool vec,
                               cudaStream_t s) {
  const uint16_t* p = static_cast<const uint16_t*>(partials);
  uint16_t* o = static_cast<uint16_t*>(out);
  switch (G) {
#define MOE_TREE_CASE(n) \
  case n:                \
    return launch_tree_g<n>(p, N, o, vec, s);
    MOE_TREE_CASE(1) MOE_TREE_CASE(2) MOE_TREE_CASE(3) MOE_TREE_CASE(4)
    MOE_TREE_CASE(5) MOE_TREE_CASE(6) MOE_TREE_CASE(7) MOE_TREE_CASE(8)
    MOE_TREE_CASE(9) MOE_TREE_CASE(10) MOE_TREE_CASE(11) MOE_TREE_CASE(12)
    MOE_TREE_CASE(13) MOE_TREE_CASE(14) MOE_TREE_CASE(15) MOE_TREE_CASE(16)
#undef MOE_TREE_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine_sharded(const float* y, const float* topk_w, const int32_t* topk_idx,
                                   const int32_t* row_of_slot, const int32_t* owner, int G, int T,
                                   int H, int E, int k, float scale, const float* shared,
                                   void* partials, void* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  uint16_t* p = static_cast<uint16_t*>(partials);
  uint16_t* o = static_cast<uint16_t*>(out);
  switch (G) {
#define MOE_SHARD_CASE(n)                                                                      \
  case n:                                                                                      \
    return launch_combine_sharded_g<n>(y, topk_w, topk_idx, row_of_slot, owner, T, H, E, k, \
                                       scale, shared, p, o, s);
    MOE_SHARD_CASE(1) MOE_SHARD_CASE(2) MOE_SHARD_CASE(3) MOE_SHARD_CASE(4)
    MOE_SHARD_CASE(5) MOE_SHARD_CASE(6) MOE_SHARD_CASE(7) MOE_SHARD_CASE(8)
    MOE_SHARD_CASE(9) MOE_SHARD_CASE(10) MOE_SHARD_CASE(11) MOE_SHARD_CASE(12)
    MOE_SHARD_CASE(13) MOE_SHARD_CASE(14) MOE_SHARD_CASE(15) MOE_SHARD_CASE(16)
#undef MOE_SHARD_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace moe
