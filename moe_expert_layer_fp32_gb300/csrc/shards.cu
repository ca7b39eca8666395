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
// FP32 rows are read once, the chains, the G roundings and the reduction stay in
// registers, and only the final BF16 row (plus the partials, when asked for) is
// written.  tree_reduce_kernel is the reduction alone, for partials that another
// engine delivered: G BF16 rows in, one BF16 row out.
//
// FP64 is a narrow pipe on this GPU, so the reduction runs in FP32 wherever that
// is provably the same.  Every leaf is a bf16 value (8 significant bits).  A group
// of at most G leaves whose exponents lie within W = 16 - ceil(log2 G) binades of
// each other sums exactly in FP32 (the sum of their magnitudes stays below 2^24
// units of the smallest one), in any order.  The leaves are split at W binades
// below the largest exponent into two such groups, H and L; if the smallest
// non-zero leaf is within 2W + 1 binades of the largest, both sums are exact and
// H + L is the exact sum of all leaves.  So is the FP64 tree's result: every node
// of it is a partial sum of fewer than 2^53 units, hence exact.  H + L is rounded
// once to bf16: s = fl(H + L) plus its exact TwoSum error decides the one case s
// alone cannot, a tie.  Both accumulators start at -0, so an all -0 input gives
// -0 and any exact zero sum of other leaves +0, as IEEE addition in the tree gives
// it.  Wider spreads, leaves from 2^124 up (no FP32 overflow), infinities and NaNs
// take the FP64 tree itself, in a separate routine.
//
// The per-rank chains: a slot whose expert another rank owns adds w * 0 = +-0 to
// that rank's accumulator, which changes nothing except -0 + +0 = +0 when w has a
// clear sign bit.  Per token (the same for every column) one thread orders the
// owned slots rank by rank, slot order within a rank, and marks where a rank's
// accumulator must first be normalised (acc + 0.0f) because such a slot came after
// its previous FMA, and where at the end.  One running accumulator then does one
// FMA per slot, and each rank's bf16 partial comes out at the end of its run.
// The sum above does not depend on the order of its leaves, so the run order can
// stand in for the rank order.  A token with a non-finite weight runs the chains
// literally.
//
// Conversions to and from FP64 are integer bit manipulation: bf16 -> f64 widens
// exactly, and f64 -> bf16 rounds once to nearest even from the full 52-bit
// fraction, never through FP32 (that would round twice).
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

// The fixed tree over d[0..n): adjacent pairs per level in FP64, odd last carried;
// the bf16 of the last value.
__device__ __forceinline__ uint32_t fp64_tree_to_bf16(double* d, int n) {
  while (n > 1) {
    int m = 0;
    for (int i = 0; i + 1 < n; i += 2) d[m++] = __dadd_rn(d[i], d[i + 1]);
    if (n & 1) d[m++] = d[n - 1];
    n = m;
  }
  return f64_to_bf16_bits(d[0]);
}

__host__ __device__ constexpr int ceil_log2(int n) { return n <= 1 ? 0 : 1 + ceil_log2((n + 1) / 2); }

__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// f rounded to bf16 (nearest even), as an FP32 value.
__device__ __forceinline__ float round_bf16_f32(float f) {
  return __uint_as_float(f32_to_bf16_bits(f) << 16);
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

// One column of the exact path.  mx, mn1: the largest |leaf| bits and the
// smallest (|leaf| bits - 1) over the present leaves (so 0xFFFF: no non-zero
// leaf); returns false where the FP64 tree itself must decide.
template <int kW>
__device__ __forceinline__ bool exact_window(uint32_t mx, uint32_t mn1, uint32_t& thr) {
  const int e_max = (int)(mx >> 7);
  const int e_min = mn1 == 0xFFFFu ? 255 : max((int)((mn1 + 1u) >> 7), 1);  // subnormals: e = 1
  // e_max <= 250: leaves below 2^124; e = 255 (inf / NaN) fails it too
  if (!(e_max <= 250 && e_max - e_min <= 2 * kW + 1)) return false;
  thr = (uint32_t)max(e_max - kW, 0) << 7;  // H: |leaf| bits >= thr (within kW of e_max)
  return true;
}

// The exact path for both columns of the packed leaves words[i] (column 0 in the
// low half) with bit i of `mask` set.  Any order: the sums are exact.  kW: the
// window of one FP32 group for the largest number of leaves present.
// no_pos_zero: no leaf outside the mask is a known +0.  Returns bit c set where
// column c could not take the exact path (the FP64 tree must decide it).
template <int N, int kW>
__device__ __forceinline__ uint32_t exact_pair_sum(const uint32_t* words, uint32_t mask,
                                                   bool no_pos_zero, uint32_t& out) {
  uint32_t mx = 0u, mn1 = 0xFFFFFFFFu;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    if ((mask >> i) & 1u) {
      const uint32_t ab = words[i] & 0x7FFF7FFFu;  // |leaf| bits, both columns
      mx = __vmaxu2(mx, ab);
      mn1 = __vminu2(mn1, __vsub2(ab, 0x00010001u));  // 0 wraps to 0xFFFF
    }
  }
  uint32_t thr0 = 0u, thr1 = 0u;
  const bool ok0 = exact_window<kW>(mx & 0xFFFFu, mn1 & 0xFFFFu, thr0);
  const bool ok1 = exact_window<kW>(mx >> 16, mn1 >> 16, thr1);
  const uint32_t thr = thr0 | (thr1 << 16);
  const float z = no_pos_zero ? -0.0f : 0.0f;  // a known +0 leaf joins as +0
  float h0 = z, h1 = z, l0 = -0.0f, l1 = -0.0f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    if ((mask >> i) & 1u) {
      const uint32_t w = words[i];
      const uint32_t m = __vcmpgeu2(w & 0x7FFF7FFFu, thr);  // 0xFFFF where the leaf is in H
      const uint32_t m0 = (uint32_t)((int32_t)(m << 16) >> 16), m1 = (uint32_t)((int32_t)m >> 16);
      const uint32_t v0 = w << 16, v1 = w & 0xFFFF0000u;
      // in the group: the leaf; out of it: -0 (the identity of IEEE addition)
      h0 = __fadd_rn(h0, __uint_as_float((v0 & m0) | (0x80000000u & ~m0)));
      l0 = __fadd_rn(l0, __uint_as_float((v0 & ~m0) | (0x80000000u & m0)));
      h1 = __fadd_rn(h1, __uint_as_float((v1 & m1) | (0x80000000u & ~m1)));
      l1 = __fadd_rn(l1, __uint_as_float((v1 & ~m1) | (0x80000000u & m1)));
    }
  }
  uint32_t r[2];
  const float hs[2] = {h0, h1}, ls[2] = {l0, l1};
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const float sum = __fadd_rn(hs[c], ls[c]);
    const float bv = __fsub_rn(sum, hs[c]);
    const float err = __fadd_rn(__fsub_rn(hs[c], __fsub_rn(sum, bv)), __fsub_rn(ls[c], bv));
    r[c] = round_pair_to_bf16(sum, err);
  }
  out = r[0] | (r[1] << 16);
  return (ok0 ? 0u : 1u) | (ok1 ? 0u : 2u);
}

// The common case first: all present leaves non-zero and within one window of
// S = 16 - ceil(log2 G) binades (max|leaf| < min|leaf| * 2^S), so their plain FP32
// sum is exact in any order and rounds once to bf16.  Returns bit c set where
// column c needs exact_pair_sum instead (a zero leaf, a wider spread, inf, NaN).
template <int N, int kW>
__device__ __forceinline__ uint32_t fast_pair_sum(const uint32_t* words, uint32_t mask,
                                                  bool no_pos_zero, uint32_t& out) {
  constexpr float kScale = (float)(1u << kW);
  const float z = no_pos_zero ? -0.0f : 0.0f;
  float s0 = z, s1 = z, mx0 = 0.0f, mx1 = 0.0f;
  float mn0 = __int_as_float(0x7F800000), mn1 = mn0;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    if ((mask >> i) & 1u) {
      const float v0 = __uint_as_float(words[i] << 16);
      const float v1 = __uint_as_float(words[i] & 0xFFFF0000u);
      s0 = __fadd_rn(s0, v0);
      s1 = __fadd_rn(s1, v1);
      mx0 = fmaxf(mx0, fabsf(v0));
      mx1 = fmaxf(mx1, fabsf(v1));
      mn0 = fminf(mn0, fabsf(v0));
      mn1 = fminf(mn1, fabsf(v1));
    }
  }
  // mx < 2^124: no FP32 overflow, no inf; mn > 0: no zero leaf; a NaN leaf makes s NaN
  const bool ok0 = mx0 < __int_as_float(0x7D800000) && mn0 > 0.0f && mx0 < mn0 * kScale && s0 == s0;
  const bool ok1 = mx1 < __int_as_float(0x7D800000) && mn1 > 0.0f && mx1 < mn1 * kScale && s1 == s1;
  const __nv_bfloat162 r = __floats2bfloat162_rn(s0, s1);
  out = *reinterpret_cast<const uint32_t*>(&r);
  return (ok0 ? 0u : 1u) | (ok1 ? 0u : 2u);
}

// fast_pair_sum, then exact_pair_sum for the columns it could not take.  Returns
// bit c set where column c needs the FP64 tree itself.
template <int N, int kW>
__device__ __forceinline__ uint32_t leaf_pair_sum(const uint32_t* words, uint32_t mask,
                                                  bool no_pos_zero, uint32_t& out) {
  uint32_t fast;
  const uint32_t miss = fast_pair_sum<N, kW>(words, mask, no_pos_zero, fast);
  if (miss == 0u) {
    out = fast;
    return 0u;
  }
  uint32_t ex;
  const uint32_t bad = exact_pair_sum<N, kW>(words, mask, no_pos_zero, ex);
  const uint32_t keep = (miss & 1u ? 0u : 0xFFFFu) | (miss & 2u ? 0u : 0xFFFF0000u);
  out = (fast & keep) | (ex & ~keep);
  return bad & miss;
}

// Per-token schedule, the same for every column.  The owned slots visited rank
// by rank, in slot order within a rank ("positions" p); bits over positions:
// first of its rank's run, last of it, normalise before the FMA, normalise at the
// end of the run.  has_run: ranks owning at least one slot.  literal: a weight is
// not finite, run the chains as written.
struct TokenPlan {
  int n_pos, literal;
  uint32_t first, last, norm_pre, norm_end, has_run;
  int row[kMaxK];
  int rank[kMaxK];
  float w[kMaxK];
};

// Slots with an invalid row contribute nothing to any rank and are left out.
__device__ void build_plan(TokenPlan& P, const int* row, const int* own, const float* w, int k,
                           int G) {
  const uint32_t all = (G >= 32) ? 0xFFFFFFFFu : ((1u << G) - 1u);
  uint32_t started = 0u, pending = 0u, pre_slot = 0u;
  int literal = 0;
  for (int j = 0; j < k; ++j) {  // slot order: where a -0 must become +0
    if (row[j] < 0) continue;
    if (!isfinite(w[j])) literal = 1;
    const uint32_t ob = own[j] >= 0 ? (1u << own[j]) : 0u;
    if (started & pending & ob) pre_slot |= 1u << j;
    started |= ob;
    pending &= ~ob;
    if (!signbit(w[j])) pending |= all & ~ob;  // w * 0 = +0 reaches every other rank
  }
  const uint32_t end_rank = started & pending;
  uint32_t first = 0u, last = 0u, norm_pre = 0u, norm_end = 0u;
  int n = 0;
  for (int g = 0; g < G; ++g) {
    int lastp = -1;
    for (int j = 0; j < k; ++j) {
      if (row[j] < 0 || own[j] != g) continue;
      const int p = n++;
      P.row[p] = row[j];
      P.rank[p] = g;
      P.w[p] = w[j];
      if (lastp < 0) first |= 1u << p;
      else if ((pre_slot >> j) & 1u) norm_pre |= 1u << p;
      lastp = p;
    }
    if (lastp >= 0) {
      last |= 1u << lastp;
      if ((end_rank >> g) & 1u) norm_end |= 1u << lastp;
    }
  }
  P.n_pos = n;
  P.literal = literal;
  P.first = first;
  P.last = last;
  P.norm_pre = norm_pre;
  P.norm_end = norm_end;
  P.has_run = started;
}

// One output element the way the section writes it: every rank's chain over all
// slots with exact zeros, the shard, one rounding, the FP64 tree.  Used for tokens
// with a non-finite weight and for the rare element the exact path cannot take.
__device__ __noinline__ uint32_t literal_element(const float* __restrict__ y, const int* row,
                                                 const int* own, const float* w, int k, int G,
                                                 const float* __restrict__ shared, int T, int H,
                                                 int t, int c, uint16_t* partials) {
  double d[kMaxShards];
  for (int g = 0; g < G; ++g) {
    float acc = 0.0f;
    for (int j = 0; j < k; ++j)
      if (row[j] >= 0) acc = fmaf(w[j], own[j] == g ? y[(size_t)row[j] * H + c] : 0.0f, acc);
    if (shared != nullptr) acc = __fadd_rn(acc, shared[((size_t)g * T + t) * H + c]);
    const uint32_t b = f32_to_bf16_bits(acc);
    if (partials != nullptr) partials[((size_t)g * T + t) * H + c] = (uint16_t)b;
    d[g] = bf16_bits_to_f64(b);
  }
  return fp64_tree_to_bf16(d, G);
}

// One warp per token (kWarps tokens per CTA), two consecutive columns per lane
// (a leaf's two columns share one 32-bit register).  GM >= G bounds the ranks,
// KP >= k the slots, SHARED says whether shard outputs are added.  Column pairs
// that the exact path cannot take are marked in shared memory and redone after
// the main loop, so the rare FP64 routine stays out of it.  Warps synchronise
// only among their own lanes.
constexpr int kShardWarps = 4;

struct WarpToken {
  int row[kMaxK];
  int own[kMaxK];
  float w[kMaxK];
  TokenPlan plan;
  int any_redo;
  uint32_t redo[16384 / 2 / 32];  // one bit per column pair (H <= 16384)
};

template <int GM, int KP, bool SHARED>
__global__ void __launch_bounds__(kShardWarps * 32, 4) combine_sharded_kernel(
    const float* __restrict__ y, const float* __restrict__ topk_w,
    const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ row_of_slot,
    const int32_t* __restrict__ owner, int G, int T, int H, int E, int k, float scale,
    const float* __restrict__ shared, uint16_t* __restrict__ partials, uint16_t* __restrict__ out) {
  constexpr int kW = 16 - ceil_log2(GM);  // one leaf per rank, at most GM
  __shared__ WarpToken s_tok[kShardWarps];
  // with shards: each lane's run-end values by rank
  __shared__ float2 s_end[kShardWarps][SHARED ? GM : 1][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kShardWarps + warp;
  if (t >= T) return;
  WarpToken& W = s_tok[warp];
  const long long R = (long long)T * k;
  if (lane < k) {
    const int r = row_of_slot[(size_t)t * k + lane];
    const int e = topk_idx[(size_t)t * k + lane];
    const int o = (e >= 0 && e < E) ? owner[e] : -1;
    W.row[lane] = (r >= 0 && r < R) ? r : -1;
    W.own[lane] = (o >= 0 && o < G) ? o : -1;  // -1: no rank owns the slot
    W.w[lane] = __fmul_rn(scale, topk_w[(size_t)t * k + lane]);
  }
  for (int i = lane; i < H / 64; i += 32) W.redo[i] = 0u;
  if (lane == 0) W.any_redo = 0;
  __syncwarp();
  if (lane == 0) build_plan(W.plan, W.row, W.own, W.w, k, G);
  __syncwarp();
  const float* sh = SHARED ? shared : nullptr;
  if (W.plan.literal) {
    for (int c0 = lane * 2; c0 < H; c0 += 64) {
      const uint32_t o0 = literal_element(y, W.row, W.own, W.w, k, G, sh, T, H, t, c0, partials);
      const uint32_t o1 = literal_element(y, W.row, W.own, W.w, k, G, sh, T, H, t, c0 + 1, partials);
      *reinterpret_cast<uint32_t*>(out + (size_t)t * H + c0) = o0 | (o1 << 16);
    }
    return;
  }
  const int n_pos = W.plan.n_pos;
  const uint32_t first = W.plan.first, last = W.plan.last;
  const uint32_t norm_pre = W.plan.norm_pre, norm_end = W.plan.norm_end;
  const uint32_t has_run = W.plan.has_run;
  const uint32_t all = (1u << G) - 1u;
  const uint32_t no_run = all & ~has_run;
  int prow[KP];
  float pw[KP];
#pragma unroll
  for (int p = 0; p < KP; ++p) {
    prow[p] = (p < n_pos) ? W.plan.row[p] : 0;
    pw[p] = (p < n_pos) ? W.plan.w[p] : 0.0f;
  }
  // leaves: with shards one per rank (index = rank), else the run ends (index = position)
  constexpr int NL = SHARED ? GM : KP;
  const uint32_t mask = SHARED ? all : last;
  const bool no_pos_zero = SHARED || no_run == 0u;
  // the rows of the next column pair are in flight while this one is computed
  float2 vn[KP];
#pragma unroll
  for (int p = 0; p < KP; ++p)
    if (p < n_pos) vn[p] = __ldg(reinterpret_cast<const float2*>(y + (size_t)prow[p] * H + lane * 2));
  for (int c0 = lane * 2; c0 < H; c0 += 64) {
    float2 v[KP];
#pragma unroll
    for (int p = 0; p < KP; ++p) v[p] = vn[p];
    if (c0 + 64 < H) {
#pragma unroll
      for (int p = 0; p < KP; ++p)
        if (p < n_pos)
          vn[p] = __ldg(reinterpret_cast<const float2*>(y + (size_t)prow[p] * H + c0 + 64));
    }
    // shard values: issued with the rows for up to 8 ranks, later for more (registers)
    constexpr bool kEarlyShards = SHARED && GM <= 8;
    float2 shv[kEarlyShards ? GM : 1];
    if constexpr (kEarlyShards) {
#pragma unroll
      for (int g = 0; g < GM; ++g)
        if (g < G) shv[g] = __ldg(reinterpret_cast<const float2*>(shared + ((size_t)g * T + t) * H + c0));
    }
    uint32_t lf[NL];  // bf16 leaves, column c0 in the low half
    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
    for (int p = 0; p < KP; ++p) {
      if (p < n_pos) {
        // a run starts from +0; adding +0 normalises -0, adding -0 changes nothing
        const bool fst = (first >> p) & 1u;
        const float nz = ((norm_pre >> p) & 1u) ? 0.0f : -0.0f;
        a0 = fmaf(pw[p], v[p].x, __fadd_rn(fst ? 0.0f : a0, nz));
        a1 = fmaf(pw[p], v[p].y, __fadd_rn(fst ? 0.0f : a1, nz));
        if ((last >> p) & 1u) {
          const float ne = ((norm_end >> p) & 1u) ? 0.0f : -0.0f;
          const float r0 = __fadd_rn(a0, ne), r1 = __fadd_rn(a1, ne);
          if constexpr (SHARED) {
            s_end[warp][W.plan.rank[p]][lane] = make_float2(r0, r1);
          } else {
            const __nv_bfloat162 b = __floats2bfloat162_rn(r0, r1);
            lf[p] = *reinterpret_cast<const uint32_t*>(&b);
            if (partials != nullptr)
              *reinterpret_cast<uint32_t*>(partials + ((size_t)W.plan.rank[p] * T + t) * H + c0) =
                  lf[p];
          }
        }
      }
    }
    if constexpr (SHARED) {
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        if (g < G) {
          // +0 for a rank without a slot, then its shard: one FP32 add, one rounding
          const float2 e = ((has_run >> g) & 1u) ? s_end[warp][g][lane] : make_float2(0.0f, 0.0f);
          float2 q;
          if constexpr (kEarlyShards) q = shv[g];
          else q = __ldg(reinterpret_cast<const float2*>(shared + ((size_t)g * T + t) * H + c0));
          const __nv_bfloat162 b = __floats2bfloat162_rn(__fadd_rn(e.x, q.x), __fadd_rn(e.y, q.y));
          lf[g] = *reinterpret_cast<const uint32_t*>(&b);
          if (partials != nullptr)
            *reinterpret_cast<uint32_t*>(partials + ((size_t)g * T + t) * H + c0) = lf[g];
        }
      }
    } else if (partials != nullptr) {
#pragma unroll
      for (int g = 0; g < GM; ++g)
        if ((no_run >> g) & 1u)  // a rank without a slot: +0
          *reinterpret_cast<uint32_t*>(partials + ((size_t)g * T + t) * H + c0) = 0u;
    }
    uint32_t o = 0u;
    if (leaf_pair_sum<NL, kW>(lf, mask, no_pos_zero, o) != 0u) {
      atomicOr(&W.redo[c0 >> 6], 1u << ((c0 >> 1) & 31));
      W.any_redo = 1;
    }
    *reinterpret_cast<uint32_t*>(out + (size_t)t * H + c0) = o;
  }
  __syncwarp();
  if (W.any_redo) {
    for (int c0 = lane * 2; c0 < H; c0 += 64) {
      if ((W.redo[c0 >> 6] >> ((c0 >> 1) & 31)) & 1u) {
        const uint32_t o0 = literal_element(y, W.row, W.own, W.w, k, G, sh, T, H, t, c0, nullptr);
        const uint32_t o1 =
            literal_element(y, W.row, W.own, W.w, k, G, sh, T, H, t, c0 + 1, nullptr);
        *reinterpret_cast<uint32_t*>(out + (size_t)t * H + c0) = o0 | (o1 << 16);
      }
    }
  }
}

// The layer's sharded combine, when no partials are asked for: one CTA per token
// and column block, four columns per thread per step, the k rows read with
// 16-byte loads as in the plain combine.  The per-token schedule (positions in
// rank order, a mask that restarts the chain at each run's first position, the
// run ends) is built by one warp in parallel (lane = slot), sits in registers
// before the column loop, and the run-end test is a branch that is the same for
// the whole CTA.
//
// The chains here leave out the signed-zero adds of the plan: they change a
// run's value only while it is exactly zero (once a chain is non-zero its later
// values do not depend on the sign of an earlier zero), and a zero leaf sends its
// column to the literal routine below.  Per column: when every leaf is non-zero,
// below 2^124, and within one window of 16 - ceil(log2 GM) binades, their plain
// FP32 sum is exact in any order and equals the FP64 tree's value, rounded once
// to bf16; any other column (a zero, inf or NaN leaf, a wider spread) is marked
// and, after the streaming loop, computed by literal_element, the definition itself.
template <int GM, int KP, bool SHARED>
__global__ void __launch_bounds__(128) combine_sharded_fast_kernel(
    const float* __restrict__ y, const float* __restrict__ topk_w,
    const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ row_of_slot,
    const int32_t* __restrict__ owner, int G, int T, int H, int E, int k, float scale,
    const float* __restrict__ shared, uint16_t* __restrict__ out) {
  constexpr float kScale = (float)(1u << (16 - ceil_log2(GM)));
  __shared__ int s_row[kMaxK];
  __shared__ int s_own[kMaxK];
  __shared__ float s_w[kMaxK];
  __shared__ TokenPlan s_plan;
  __shared__ uint32_t s_redo[16384 / 32];  // columns for the literal routine (H <= 16384)
  __shared__ int s_owner[kMaxE];            // the owner table, read with the slots
  const int t = blockIdx.x;
  const long long R = (long long)T * k;
  for (int i = threadIdx.x; i < H / gridDim.y / 32; i += blockDim.x) s_redo[i] = 0u;
  // the slots' loads and the owner table's go out together (one round trip)
  int r = -1, e = -1;
  float wraw = 0.0f;
  if (threadIdx.x < k) {
    r = row_of_slot[(size_t)t * k + threadIdx.x];
    e = topk_idx[(size_t)t * k + threadIdx.x];
    wraw = topk_w[(size_t)t * k + threadIdx.x];
  }
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_owner[i] = __ldg(owner + i);
  __syncthreads();
  if (threadIdx.x < 32) {
    // the schedule, warp-parallel: lane j is slot j.  Positions are the owned slots
    // sorted by rank, slot order within a rank (build_plan's order); the run of a
    // rank starts at its first position and ends at its last.
    const int j = threadIdx.x;
    int o = -1;
    float wj = 0.0f;
    if (j < k) {
      o = (e >= 0 && e < E) ? s_owner[e] : -1;
      r = (r >= 0 && r < R) ? r : -1;
      o = (o >= 0 && o < G) ? o : -1;  // -1: no rank owns the slot
      wj = __fmul_rn(scale, wraw);
      s_row[j] = r;
      s_own[j] = o;
      s_w[j] = wj;
    }
    const bool pos = j < k && r >= 0 && o >= 0;  // the slot joins its rank's run
    int before = 0, same_before = 0, same_after = 0;
#pragma unroll
    for (int i = 0; i < kMaxK; ++i) {
      const int oi = __shfl_sync(0xFFFFFFFFu, pos ? o : -1, i);
      if (i < k && oi >= 0) {
        before += (oi < o) || (oi == o && i < j);
        same_before += oi == o && i < j;
        same_after += oi == o && i > j;
      }
    }
    const unsigned first = __reduce_or_sync(0xFFFFFFFFu, pos && same_before == 0 ? 1u << before : 0u);
    const unsigned last = __reduce_or_sync(0xFFFFFFFFu, pos && same_after == 0 ? 1u << before : 0u);
    const unsigned runs = __reduce_or_sync(0xFFFFFFFFu, pos ? 1u << o : 0u);
    const unsigned npos = __popc(__ballot_sync(0xFFFFFFFFu, pos));
    const bool bad_w = __any_sync(0xFFFFFFFFu, j < k && r >= 0 && !isfinite(wj));
    if (pos) {
      s_plan.row[before] = r;
      s_plan.rank[before] = o;
      s_plan.w[before] = wj;
    }
    if (j == 0) {
      s_plan.n_pos = (int)npos;
      s_plan.literal = bad_w ? 1 : 0;
      s_plan.first = first;
      s_plan.last = last;
      s_plan.has_run = runs;
    }
  }
  __syncthreads();
  const int cols = H / gridDim.y;
  const int cb = blockIdx.y * cols;
  const float* sh = SHARED ? shared : nullptr;
  uint16_t* orow = out + (size_t)t * H;
  if (s_plan.literal) {
    for (int c = cb + threadIdx.x; c < cb + cols; c += blockDim.x)
      orow[c] = (uint16_t)literal_element(y, s_row, s_own, s_w, k, G, sh, T, H, t, c, nullptr);
    return;
  }
  const int n_pos = s_plan.n_pos;
  const uint32_t last = s_plan.last;
  const uint32_t no_run = ((1u << G) - 1u) & ~s_plan.has_run;
  int prow[KP], prank[KP];
  float pw[KP];
  uint32_t keep[KP];  // 0: the position starts its rank's run (the chain restarts at +0)
#pragma unroll
  for (int p = 0; p < KP; ++p) {
    prow[p] = (p < n_pos) ? s_plan.row[p] : 0;
    prank[p] = (p < n_pos) ? s_plan.rank[p] : 0;
    pw[p] = (p < n_pos) ? s_plan.w[p] : 0.0f;
    keep[p] = ((s_plan.first >> p) & 1u) ? 0u : 0xFFFFFFFFu;
  }
  // a rank without a slot contributes +0 (no shard) or bf16(+0 + its shard)
  const float s0 = no_run != 0u ? 0.0f : -0.0f;
  int any_redo = 0;
  // the rows of the next step are in flight while this one is computed
  float4 vn[KP];
  const int cstart = cb + threadIdx.x * 4, cend = cb + cols, cstep = blockDim.x * 4;
#pragma unroll
  for (int p = 0; p < KP; ++p)
    if (p < n_pos && cstart < cend)
      vn[p] = __ldg(reinterpret_cast<const float4*>(y + (size_t)prow[p] * H + cstart));
  for (int c = cstart; c < cend; c += cstep) {
    float4 v[KP];
#pragma unroll
    for (int p = 0; p < KP; ++p) v[p] = vn[p];
    if (c + cstep < cend) {
#pragma unroll
      for (int p = 0; p < KP; ++p)
        if (p < n_pos) vn[p] = __ldg(reinterpret_cast<const float4*>(y + (size_t)prow[p] * H + c + cstep));
    }
    float4 q[SHARED ? KP : 1];
    if constexpr (SHARED) {
#pragma unroll
      for (int p = 0; p < KP; ++p)
        if (p < n_pos && ((last >> p) & 1u))
          q[p] = __ldg(reinterpret_cast<const float4*>(shared + ((size_t)prank[p] * T + t) * H + c));
    }
    float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    float sum[4] = {s0, s0, s0, s0};
    float mx[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    float mn[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) mn[i] = __int_as_float(0x7F800000);
#pragma unroll
    for (int p = 0; p < KP; ++p) {
      if (p < n_pos) {
        const float vv[4] = {v[p].x, v[p].y, v[p].z, v[p].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          a[i] = fmaf(pw[p], vv[i], __uint_as_float(__float_as_uint(a[i]) & keep[p]));
        if ((last >> p) & 1u) {
          float qq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          if constexpr (SHARED) {
            qq[0] = q[p].x;
            qq[1] = q[p].y;
            qq[2] = q[p].z;
            qq[3] = q[p].w;
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float lf = round_bf16_f32(SHARED ? __fadd_rn(a[i], qq[i]) : a[i]);
            sum[i] = __fadd_rn(sum[i], lf);
            mx[i] = fmaxf(mx[i], fabsf(lf));
            mn[i] = fminf(mn[i], fabsf(lf));
          }
        }
      }
    }
    if constexpr (SHARED) {
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        if (g < G && ((no_run >> g) & 1u)) {
          const float4 qg = __ldg(reinterpret_cast<const float4*>(shared + ((size_t)g * T + t) * H + c));
          const float qv[4] = {qg.x, qg.y, qg.z, qg.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float lf = round_bf16_f32(__fadd_rn(0.0f, qv[i]));
            sum[i] = __fadd_rn(sum[i], lf);
            mx[i] = fmaxf(mx[i], fabsf(lf));
            mn[i] = fminf(mn[i], fabsf(lf));
          }
        }
      }
    }
    uint32_t o[4];
    uint32_t bad = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool ok = mx[i] < __int_as_float(0x7D800000) && mn[i] > 0.0f &&
                      mx[i] < mn[i] * kScale && sum[i] == sum[i];
      o[i] = f32_to_bf16_bits(sum[i]);
      if (!ok) bad |= 1u << i;
    }
    *reinterpret_cast<uint2*>(orow + c) = make_uint2(o[0] | (o[1] << 16), o[2] | (o[3] << 16));
    if (bad != 0u) {  // redone below by this thread, outside the streaming loop
      atomicOr(&s_redo[(c - cb) >> 5], bad << ((c - cb) & 31));
      any_redo = 1;
    }
  }
  // the rare columns one window could not take: their leaves again (the chains from
  // L2), then the exact two-window sum of exact_pair_sum, and where that cannot
  // decide either (a zero leaf, whose sign the chains above do not settle, a spread
  // beyond two windows, inf, NaN) the definition itself
  if (__syncthreads_or(any_redo)) {
    constexpr int kW = 16 - ceil_log2(GM);
    for (int c = cstart; c < cend; c += cstep) {
      const uint32_t bad = (s_redo[(c - cb) >> 5] >> ((c - cb) & 31)) & 0xFu;
      for (int i = 0; i < 4; ++i) {
        if (!((bad >> i) & 1u)) continue;
        const int col = c + i;
        uint32_t words[KP];
        bool zero_leaf = false;
        float a = 0.0f;
#pragma unroll
        for (int p = 0; p < KP; ++p) {
          words[p] = 0u;
          if (p < n_pos) {
            a = fmaf(pw[p], __ldg(y + (size_t)prow[p] * H + col),
                     __uint_as_float(__float_as_uint(a) & keep[p]));
            if ((last >> p) & 1u) {
              const uint32_t lb = f32_to_bf16_bits(a);
              words[p] = lb | (lb << 16);
              zero_leaf |= (lb & 0x7FFFu) == 0u;
            }
          }
        }
        uint32_t o = 0u;
        if (zero_leaf || (exact_pair_sum<KP, kW>(words, last, no_run == 0u, o) & 1u))
          o = literal_element(y, s_row, s_own, s_w, k, G, sh, T, H, t, col, nullptr);
        orow[col] = (uint16_t)(o & 0xFFFFu);
      }
    }
  }
}

// The FP64 tree over element n of the G rows, from memory.
__device__ __forceinline__ uint32_t tree_element_fp64(const uint16_t* __restrict__ partials, int G,
                                                   long long N, long long n) {
  double d[kMaxShards];
  for (int g = 0; g < G; ++g) d[g] = bf16_bits_to_f64(partials[(size_t)g * N + n]);
  return fp64_tree_to_bf16(d, G);
}

// out[n] = bf16(tree(partials[0..G-1][n])), GM >= G (FULL: G == GM).  VEC: 8
// elements per 16-byte vector (every row base 16-byte aligned), else one element
// per step.
template <int GM, bool FULL, bool VEC>
__global__ void __launch_bounds__(256) tree_reduce_kernel(const uint16_t* __restrict__ partials,
                                                          int G, long long N,
                                                          uint16_t* __restrict__ out) {
  constexpr int kW = 16 - ceil_log2(GM);
  const uint32_t mask = FULL ? (1u << GM) - 1u : (1u << G) - 1u;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long first = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if constexpr (VEC) {
    const long long nv = N / 8;
    for (long long i = first; i < nv; i += stride) {
      uint4 q[GM];
#pragma unroll
      for (int g = 0; g < GM; ++g)
        if (FULL || g < G) q[g] = __ldg(reinterpret_cast<const uint4*>(partials + (size_t)g * N) + i);
      uint32_t o[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t words[GM];
#pragma unroll
        for (int g = 0; g < GM; ++g) words[g] = (&q[g].x)[w];
        const uint32_t bad = leaf_pair_sum<GM, kW>(words, mask, true, o[w]);
        if (bad != 0u) {
          const long long n = 8 * i + 2 * w;
          uint32_t lo = o[w] & 0xFFFFu, hi = o[w] >> 16;
          if (bad & 1u) lo = tree_element_fp64(partials, G, N, n);
          if (bad & 2u) hi = tree_element_fp64(partials, G, N, n + 1);
          o[w] = lo | (hi << 16);
        }
      }
      reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  } else {
    for (long long n = first; n < N; n += stride) {
      uint32_t words[GM];
#pragma unroll
      for (int g = 0; g < GM; ++g) words[g] = (FULL || g < G) ? partials[(size_t)g * N + n] : 0u;
      uint32_t r;
      if (leaf_pair_sum<GM, kW>(words, mask, true, r) & 1u) r = tree_element_fp64(partials, G, N, n);
      out[n] = (uint16_t)r;
    }
  }
}

template <int GM>
cudaError_t launch_tree_gm(const uint16_t* p, int G, long long N, uint16_t* out, bool vec,
                           cudaStream_t s) {
  const long long units = vec ? N / 8 : N;
  if (units == 0) return cudaSuccess;
  const long long want = (units + 255) / 256;
  const int cap = device_sm_count() * 8;
  const int grid = (int)(want < cap ? want : cap);
  const bool full = G == GM;
  if (vec && full) tree_reduce_kernel<GM, true, true><<<grid, 256, 0, s>>>(p, G, N, out);
  else if (vec) tree_reduce_kernel<GM, false, true><<<grid, 256, 0, s>>>(p, G, N, out);
  else if (full) tree_reduce_kernel<GM, true, false><<<grid, 256, 0, s>>>(p, G, N, out);
  else tree_reduce_kernel<GM, false, false><<<grid, 256, 0, s>>>(p, G, N, out);
  return cudaGetLastError();
}

template <int GM, int KP>
cudaError_t launch_combine_gm(const float* y, const float* topk_w, const int32_t* topk_idx,
                              const int32_t* row_of_slot, const int32_t* owner, int G, int T, int H,
                              int E, int k, float scale, const float* shared, uint16_t* partials,
                              uint16_t* out, cudaStream_t s) {
  if (partials == nullptr && shared == nullptr) {
    // split each token's columns over up to H / 512 CTAs while the grid stays within
    // four CTAs per SM (as the plain combine does)
    int split = 1;
    while (split * 2 <= H / 512 && H % (split * 2 * 512) == 0 &&
           (long long)T * split * 2 <= 4LL * device_sm_count())
      split *= 2;
    combine_sharded_fast_kernel<GM, KP, false><<<dim3(T, split), 128, 0, s>>>(
        y, topk_w, topk_idx, row_of_slot, owner, G, T, H, E, k, scale, nullptr, out);
    return cudaGetLastError();
  }
  const int grid = (T + kShardWarps - 1) / kShardWarps;
  if (shared != nullptr)
    combine_sharded_kernel<GM, KP, true><<<grid, kShardWarps * 32, 0, s>>>(
        y, topk_w, topk_idx, row_of_slot, owner, G, T, H, E, k, scale, shared, partials, out);
  else
    combine_sharded_kernel<GM, KP, false><<<grid, kShardWarps * 32, 0, s>>>(
        y, topk_w, topk_idx, row_of_slot, owner, G, T, H, E, k, scale, nullptr, partials, out);
  return cudaGetLastError();
}

template <int KP>
cudaError_t launch_combine_kp(const float* y, const float* topk_w, const int32_t* topk_idx,
                              const int32_t* row_of_slot, const int32_t* owner, int G, int T, int H,
                              int E, int k, float scale, const float* shared, uint16_t* partials,
                              uint16_t* out, cudaStream_t s) {
  if (G <= 2)
    return launch_combine_gm<2, KP>(y, topk_w, topk_idx, row_of_slot, owner, G, T, H, E, k, scale,
                                    shared, partials, out, s);
  if (G <= 4)
    return launch_combine_gm<4, KP>(y, topk_w, topk_idx, row_of_slot, owner, G, T, H, E, k, scale,
                                    shared, partials, out, s);
  if (G <= 8)
    return launch_combine_gm<8, KP>(y, topk_w, topk_idx, row_of_slot, owner, G, T, H, E, k, scale,
                                    shared, partials, out, s);
  return launch_combine_gm<16, KP>(y, topk_w, topk_idx, row_of_slot, owner, G, T, H, E, k, scale,
                                   shared, partials, out, s);
}

}  // namespace

cudaError_t launch_tree_reduce(const void* partials, int G, long long N, void* out, bool vec,
                               cudaStream_t s) {
  const uint16_t* p = static_cast<const uint16_t*>(partials);
  uint16_t* o = static_cast<uint16_t*>(out);
  if (G < 1 || G > kMaxShards) return cudaErrorInvalidValue;
  if (G <= 2) return launch_tree_gm<2>(p, G, N, o, vec, s);
  if (G <= 4) return launch_tree_gm<4>(p, G, N, o, vec, s);
  if (G <= 8) return launch_tree_gm<8>(p, G, N, o, vec, s);
  return launch_tree_gm<16>(p, G, N, o, vec, s);
}

cudaError_t launch_combine_sharded(const float* y, const float* topk_w, const int32_t* topk_idx,
                                   const int32_t* row_of_slot, const int32_t* owner, int G, int T,
                                   int H, int E, int k, float scale, const float* shared,
                                   void* partials, void* out, cudaStream_t s) {
  if (G < 1 || G > kMaxShards) return cudaErrorInvalidValue;
  if (T == 0) return cudaSuccess;
  uint16_t* p = static_cast<uint16_t*>(partials);
  uint16_t* o = static_cast<uint16_t*>(out);
  if (k <= 8)
    return launch_combine_kp<8>(y, topk_w, topk_idx, row_of_slot, owner, G, T, H, E, k, scale,
                                shared, p, o, s);
  return launch_combine_kp<kMaxK>(y, topk_w, topk_idx, row_of_slot, owner, G, T, H, E, k, scale,
                                  shared, p, o, s);
}

}  // namespace moe
