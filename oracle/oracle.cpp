// CPU ORACLE for the top-k routed MoE feed-forward layer forward pass.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, plain definition that the
// CUDA path is checked against.  Only the tests, the smoke check and the
// benchmark's CPU-baseline leg may load it; the library never does.  It shares
// no code, header, table or helper with the CUDA path.
//
// Sources (page title, section):
//  * "0 train-infer mismatch for open-weight MoE RL", section "Mixture-of-experts
//    layers / The router": fixed-K projection of each token to one score per
//    expert, FP32 softmax, top-k selection, the k selected probabilities added
//    left to right, each divided by that sum, experts returned sorted by
//    probability.  Same page, "Selecting sparse-attention positions": the lower
//    position wins a tie (used here for equal logits).
//  * same page, "SwiGLU: rounding after the multiply": inputs to FP32, SiLU and
//    the product in FP32, a single cast to BF16.
//  * same page, "The experts: keeping the route weight inside the accumulator"
//    and "Sharding the experts": every routing slot is accumulated in FP32 in
//    slot order and rounded once to BF16.
//  * "RoutePack: Expert Placement and Attention-Aware Data Packing for MoE RL",
//    section 2.2 "Routing replay" (Eq. 1: per-expert assignment counts) and
//    section 2.3 (grouped-GEMM execution of a rank's local experts).
//  * "FlexFloor", Figure 1: token -> dispatch -> experts -> combine.
//  * "HARTS", section 3.4 "MoE semantics without expert expansion":
//    deterministic, no-token-drop top-k routing; Eq. 23 imbalance max/mean - 1.
//  * RoutePack, section 6 Eq. 22: coefficient of variation of loads.
//  * "0 train-infer mismatch for open-weight MoE RL", section "Sharding the
//    experts": each expert rank ends with one BF16 partial per token (slots it
//    does not own add exact zeros; its shared-expert shard is added before the
//    rounding); the partials are summed in a fixed logical order by adjacent
//    pairs in FP64, an odd last one carried up a level unchanged, one BF16
//    rounding at the end.  Section "Mixture-of-experts layers" (shared expert):
//    the fixed-K projections and SwiGLU of the dense case.
//
// Readings where the pages leave a step open (each stated again where used):
//  R1 router dot product: FP32 fused multiply-add chain over ascending h from 0,
//     then one FP32 add of the optional per-expert bias;
//  R2 selection key: the FP32 logit (softmax is monotone), ties to the lower
//     expert index; slot order = selection order;
//  R3 softmax: subtract the max logit, exp in FP32, sum over ascending e;
//  R4 routing weights stay FP32;
//  R5 permutation: stable, rows of one expert in ascending token order;
//  R6 expert GEMMs: FP32 accumulation over ascending K; only h = SwiGLU output is
//     rounded to BF16; y stays FP32;
//  R7 combine: FMA chain over slots j = 0..k-1 from 0, one BF16 round.
//  R8 sharded combine: rank g's partial is the same chain with y replaced by an
//     exact 0.0f in the slots whose expert another rank owns, then one FP32 add
//     of g's shared-expert shard output (if any), then one BF16 round;
//  R9 the FP64 tree's final rounding goes straight from FP64 to BF16 (round to
//     nearest, ties to even), not through FP32;
//  R10 shared expert sharded G ways: rank g holds intermediate columns
//     [g*Is/G, (g+1)*Is/G) of the gate/up projections and the same rows of the
//     down projection, and computes them as one expert over all tokens.
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off (no contraction: every a*b+c below
// rounds twice unless written as std::fma).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

namespace {

// bf16 -> f32 is exact: the bf16 bits are the top half of the f32 bits.
inline float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// f32 -> bf16, round to nearest, ties to even (NaN stays NaN).
inline uint16_t f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

// f64 -> bf16 in one rounding (reading R9).  Definition: of the two bf16 values
// next to |x| at the bf16 spacing of its binade, the nearer; on a tie the one
// whose last mantissa bit is even; beyond the largest finite bf16 (after
// rounding) infinity.  NaN -> 0x7FC0.
inline uint16_t f64_to_bf16(double x) {
  if (std::isnan(x)) return 0x7FC0;
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  const double a = std::fabs(x);
  if (std::isinf(a)) return sign | 0x7F80;
  if (a == 0.0) return sign;
  int ex;
  std::frexp(a, &ex);                           // a in [2^(ex-1), 2^ex)
  const int e = std::max(ex - 1, -126);         // bf16 subnormals share 2^-126's spacing
  const double ulp = std::ldexp(1.0, e - 7);    // 7 stored mantissa bits
  const double n = std::floor(a / ulp);         // exact: ulp is a power of two
  const double lo = n * ulp, hi = lo + ulp;     // both exact
  const double dlo = a - lo, dhi = hi - a;      // both exact (Sterbenz, or lo = 0)
  double r;
  if (dlo < dhi) r = lo;
  else if (dhi < dlo) r = hi;
  else r = (std::fmod(n, 2.0) == 0.0) ? lo : hi;
  if (r >= std::ldexp(1.0, 128)) return sign | 0x7F80;
  const float f = (float)r;  // exact: r is a bf16 value
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return sign | (uint16_t)(u >> 16);
}

// The fixed expert-output reduction: v holds the contributors in logical order,
// widened to FP64.  Each level adds adjacent pairs in FP64 and carries an odd
// last value unchanged, until one value remains.
double fp64_pairwise_tree(std::vector<double>& v) {
  size_t n = v.size();
  while (n > 1) {
    size_t m = 0;
    for (size_t i = 0; i + 1 < n; i += 2) v[m++] = v[i] + v[i + 1];
    if (n & 1) v[m++] = v[n - 1];
    n = m;
  }
  return n == 1 ? v[0] : 0.0;
}

// Run body(i) for i in [0, n) on up to nthreads threads (contiguous chunks).
void parallel_for(int64_t n, int nthreads, const std::function<void(int64_t)>& body) {
  if (n <= 0) return;
  if (nthreads <= 0) nthreads = (int)std::thread::hardware_concurrency();
  if (nthreads < 1) nthreads = 1;
  if (nthreads > n) nthreads = (int)n;
  if (nthreads == 1) {
    for (int64_t i = 0; i < n; ++i) body(i);
    return;
  }
  std::vector<std::thread> pool;
  for (int w = 0; w < nthreads; ++w) {
    int64_t b = n * w / nthreads, e = n * (w + 1) / nthreads;
    pool.emplace_back([b, e, &body] {
      for (int64_t i = b; i < e; ++i) body(i);
    });
  }
  for (auto& t : pool) t.join();
}

// Router logits of one token (reading R1).
void token_logits(const uint16_t* x_row, const float* wr, const float* bias, int H, int E,
                  float* l) {
  for (int e = 0; e < E; ++e) l[e] = 0.0f;
  for (int h = 0; h < H; ++h) {
    float xf = bf16_to_f32(x_row[h]);
    const float* wrow = wr + (int64_t)h * E;
    for (int e = 0; e < E; ++e) l[e] = std::fma(xf, wrow[e], l[e]);
  }
  if (bias)
    for (int e = 0; e < E; ++e) l[e] = l[e] + bias[e];
}

// Route one token: FP32 softmax, top-k by (logit desc, index asc), renormalise.
void route_token(const float* l, int E, int k, int32_t* idx, float* w) {
  // softmax (reading R3)
  float m = l[0];
  for (int e = 1; e < E; ++e) m = std::max(m, l[e]);
  std::vector<float> z(E);
  float Z = 0.0f;
  for (int e = 0; e < E; ++e) {
    z[e] = std::exp(l[e] - m);
    Z = Z + z[e];
  }
  // selection (reading R2): order experts by the key (logit descending, index ascending)
  std::vector<int> order(E);
  for (int e = 0; e < E; ++e) order[e] = e;
  std::sort(order.begin(), order.end(), [&](int a, int b) {
    if (l[a] != l[b]) return l[a] > l[b];
    return a < b;
  });
  // renormalisation: add the k selected probabilities left to right, divide each by the sum
  std::vector<float> p(k);
  float S = 0.0f;
  for (int j = 0; j < k; ++j) {
    p[j] = z[order[j]] / Z;
    S = S + p[j];
  }
  for (int j = 0; j < k; ++j) {
    idx[j] = order[j];
    w[j] = p[j] / S;
  }
}

inline float silu(float g) { return g / (1.0f + std::exp(-g)); }

// exp(x) in FP32 by Cody & Waite argument reduction and a Taylor polynomial:
//   n = rint(x * log2 e),  r = x - n*ln2 (ln2 split in a high part with 16 significant
//   bits, so n*LN2_HI is exact, plus the low remainder),  exp(r) = sum_{i<=7} r^i/i!
//   evaluated by Horner with fused multiply-adds,  result = exp(r) * 2^n.
// Every step is an IEEE FP32 operation, so the result is the same bits on any
// machine that computes it the same way.  |r| <= ln2/2 keeps the truncated
// series below half an FP32 ulp.
float exp_cw(float x) {
  if (x > 89.0f) x = 89.0f;
  if (x < -104.0f) x = -104.0f;
  const float LOG2E = 1.44269502162933349609375f;  // log2(e) rounded to FP32
  const float LN2_HI = 0.693145751953125f;         // ln 2 to 16 significant bits
  const float LN2_LO = 1.428606765330187e-06f;     // ln 2 - LN2_HI
  const float n = std::rint(x * LOG2E);
  float r = std::fma(-n, LN2_HI, x);
  r = std::fma(-n, LN2_LO, r);
  const float c[8] = {1.0f, 1.0f, 1.0f / 2, 1.0f / 6, 1.0f / 24, 1.0f / 120, 1.0f / 720,
                      1.0f / 5040};
  float p = c[7];
  for (int i = 6; i >= 0; --i) p = std::fma(p, r, c[i]);
  return std::ldexp(p, (int)n);
}

// Logistic sigmoid built on exp_cw: 1 / (1 + exp(-l)).
inline float sigmoid_cw(float l) { return 1.0f / (1.0f + exp_cw(-l)); }

// Round an FP32 value to bf16 (nearest, ties to even) and widen it back.
inline float round_bf16(float f) { return bf16_to_f32(f32_to_bf16(f)); }

// Router variant with GLM's choice rule ("0 train-infer mismatch", section
// "Choosing GLM's eight experts"): sigmoid scores s_e = sigmoid(l_e); the FP32
// correction bias joins only the selection key s_e + b_e (ties to the lower
// index); the weights are the selected pre-bias scores divided by their sum
// (added left to right, FP32).
void route_token_sigmoid(const float* l, const float* corr_bias, int E, int k, int32_t* idx,
                         float* w) {
  std::vector<float> sc(E), key(E);
  for (int e = 0; e < E; ++e) {
    sc[e] = sigmoid_cw(l[e]);
    key[e] = corr_bias ? sc[e] + corr_bias[e] : sc[e];
  }
  std::vector<int> order(E);
  for (int e = 0; e < E; ++e) order[e] = e;
  std::sort(order.begin(), order.end(), [&](int a, int b) {
    if (key[a] != key[b]) return key[a] > key[b];
    return a < b;
  });
  float S = 0.0f;
  for (int j = 0; j < k; ++j) S = S + sc[order[j]];
  for (int j = 0; j < k; ++j) {
    idx[j] = order[j];
    w[j] = sc[order[j]] / S;
  }
}

}  // namespace

extern "C" {

// Router logits l[t, e] (reading R1), for inspection by tests.
int oracle_router_logits(const uint16_t* x, const float* wr, const float* bias, int T, int H, int E,
                         float* logits, int nthreads) {
  if (T < 0 || H <= 0 || E <= 0) return 1;
  parallel_for(T, nthreads, [&](int64_t t) {
    token_logits(x + t * H, wr, bias, H, E, logits + t * E);
  });
  return 0;
}

// Step 1-2: router projection, softmax, top-k, renormalisation.
// x [T, H] bf16 bits; wr [H, E] f32; bias [E] f32 or null -> idx [T, k] int32, w [T, k] f32.
int oracle_route(const uint16_t* x, const float* wr, const float* bias, int T, int H, int E, int k,
                 int32_t* idx, float* w, int nthreads) {
  if (T < 0 || H <= 0 || E <= 0 || k < 1 || k > E) return 1;
  parallel_for(T, nthreads, [&](int64_t t) {
    std::vector<float> l(E);
    token_logits(x + t * H, wr, bias, H, E, l.data());
    route_token(l.data(), E, k, idx + t * k, w + t * k);
  });
  return 0;
}

// exp_cw for tests (pinned against the float64 exponential).
float oracle_exp_cw(float x) { return exp_cw(x); }

// Router with options:
//   kind 0: softmax router (as oracle_route; `bias` joins the logits);
//   kind 1: sigmoid scores, `bias` is GLM's correction bias used only for selection,
//           weights = selected scores over their sum.
//   weights_bf16 != 0: each final weight is rounded to bf16 (stored as its FP32 value).
int oracle_route_ex(const uint16_t* x, const float* wr, const float* bias, int kind,
                    int weights_bf16, int T, int H, int E, int k, int32_t* idx, float* w,
                    int nthreads) {
  if (T < 0 || H <= 0 || E <= 0 || k < 1 || k > E || kind < 0 || kind > 1) return 1;
  parallel_for(T, nthreads, [&](int64_t t) {
    std::vector<float> l(E);
    if (kind == 0) {
      token_logits(x + t * H, wr, bias, H, E, l.data());
      route_token(l.data(), E, k, idx + t * k, w + t * k);
    } else {
      token_logits(x + t * H, wr, nullptr, H, E, l.data());
      route_token_sigmoid(l.data(), bias, E, k, idx + t * k, w + t * k);
    }
    if (weights_bf16)
      for (int j = 0; j < k; ++j) w[t * k + j] = round_bf16(w[t * k + j]);
  });
  return 0;
}

// Step 3-4: per-expert assignment counts (RoutePack Eq. 1 summed over tokens),
// exclusive prefix offsets [E+1], imbalance max/mean - 1 (HARTS Eq. 23 over
// experts) and coefficient of variation (RoutePack Eq. 22 form over experts).
int oracle_load_stats(const int32_t* idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
                      double* imbalance, double* cv) {
  if (T < 0 || k < 1 || E <= 0) return 1;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t s = 0; s < (int64_t)T * k; ++s) {
    int e = idx[s];
    if (e < 0 || e >= E) return 2;
    counts[e] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  double mean = (double)T * k / E;
  double mx = 0.0, var = 0.0;
  for (int e = 0; e < E; ++e) {
    mx = std::max(mx, (double)counts[e]);
    var += ((double)counts[e] - mean) * ((double)counts[e] - mean);
  }
  var /= E;
  if (imbalance) *imbalance = mean > 0 ? mx / mean - 1.0 : 0.0;
  if (cv) *cv = mean > 0 ? std::sqrt(var) / mean : 0.0;
  return 0;
}

// "HARTS", Eq. 20 and section "MoE execution and objectives": compact row t stands
// for q[t] semantic tokens; its assignments count q[t] times in the expert loads
// while routing and compute run once.  out[e] = sum over (t, j) with idx[t,j] = e
// of q[t] (int64).
int oracle_weighted_counts(const int32_t* idx, const int32_t* q, int T, int k, int E,
                           int64_t* out) {
  if (T < 0 || k < 1 || E <= 0) return 1;
  for (int e = 0; e < E; ++e) out[e] = 0;
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      int e = idx[t * k + j];
      if (e < 0 || e >= E) return 2;
      out[e] += q[t];
    }
  return 0;
}

// "RoutePack", Algorithm 1 (layer-local LPT expert placement): experts in order
// of (load descending, index ascending); each goes to the least-loaded rank
// (ties: lower rank id) among ranks with a free slot; pi(e) = p*Hs + n_p, the
// next slot of that rank.  P ranks of Hs = E/P slots.  Also returns the rank
// loads G_p (Eq. 10).
int oracle_lpt_placement(const int64_t* loads, int E, int P, int32_t* slot_of_expert,
                         int64_t* rank_loads) {
  if (E <= 0 || P <= 0 || E % P != 0) return 1;
  const int Hs = E / P;
  std::vector<int64_t> G(P, 0);
  std::vector<int> n(P, 0);
  std::vector<int> order(E);
  for (int e = 0; e < E; ++e) order[e] = e;
  std::sort(order.begin(), order.end(), [&](int a, int b) {
    if (loads[a] != loads[b]) return loads[a] > loads[b];
    return a < b;
  });
  for (int e : order) {
    int best = -1;
    for (int p = 0; p < P; ++p) {
      if (n[p] >= Hs) continue;
      if (best < 0 || G[p] < G[best]) best = p;  // ties keep the lower rank id
    }
    slot_of_expert[e] = best * Hs + n[best];
    G[best] += loads[e];
    n[best] += 1;
  }
  if (rank_loads)
    for (int p = 0; p < P; ++p) rank_loads[p] = G[p];
  return 0;
}

// Rank-load balance of one layer: coefficient of variation ("RoutePack", Eq. 22,
// population form over the P ranks) and EP balance efficiency (Eq. 23 for one
// row, layer and shard: mean rank load over the largest).
int oracle_rank_metrics(const int64_t* G, int P, double* cv, double* eta) {
  if (P <= 0) return 1;
  double mean = 0.0, mx = 0.0;
  for (int p = 0; p < P; ++p) {
    mean += (double)G[p];
    mx = std::max(mx, (double)G[p]);
  }
  mean /= P;
  double var = 0.0;
  for (int p = 0; p < P; ++p) var += ((double)G[p] - mean) * ((double)G[p] - mean);
  var /= P;
  *cv = mean > 0 ? std::sqrt(var) / mean : 0.0;
  *eta = mx > 0 ? mean / mx : 1.0;
  return 0;
}

// Step 5: stable permutation into expert-contiguous rows (reading R5).
// Walk slots in token order, then slot order; each takes the next free row of its
// expert.  slot s = t*k + j.  x_perm[r] is a byte copy of x[slot_of_row[r] / k].
int oracle_permute(const uint16_t* x, const int32_t* idx, const int32_t* offsets, int T, int H,
                   int E, int k, uint16_t* x_perm, int32_t* row_of_slot, int32_t* slot_of_row) {
  if (T < 0 || H <= 0 || E <= 0 || k < 1) return 1;
  std::vector<int32_t> next(offsets, offsets + E);
  for (int64_t t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j) {
      int64_t s = t * k + j;
      int e = idx[s];
      if (e < 0 || e >= E) return 2;
      int32_t r = next[e]++;
      if (r >= offsets[e + 1]) return 3;
      row_of_slot[s] = r;
      slot_of_row[r] = (int32_t)s;
      if (x_perm) std::memcpy(x_perm + (int64_t)r * H, x + t * H, sizeof(uint16_t) * H);
    }
  }
  return 0;
}

// Step 5 with "RoutePack"'s dispatcher remap (section 3.3, Figure 4): the router's
// logical expert e is dispatched to physical slot slot_of_expert[e]; rows are
// grouped by physical slot (offsets indexed by slot), stable within a slot.
int oracle_permute_remap(const uint16_t* x, const int32_t* idx, const int32_t* slot_of_expert,
                         const int32_t* offsets, int T, int H, int E, int k, uint16_t* x_perm,
                         int32_t* row_of_slot, int32_t* slot_of_row) {
  std::vector<int32_t> phys((size_t)T * k);
  for (int64_t s2 = 0; s2 < (int64_t)T * k; ++s2) {
    int e = idx[s2];
    if (e < 0 || e >= E) return 2;
    phys[s2] = slot_of_expert[e];
  }
  return oracle_permute(x, phys.data(), offsets, T, H, E, k, x_perm, row_of_slot, slot_of_row);
}

// Steps 6-7: per expert e, rows [offsets[e], offsets[e+1]) of x_perm [R, H]:
//   g = x W_gate[e], u = x W_up[e]   (FP32 accumulation, ascending h)
//   h = bf16(silu(g) * u)            (the only rounding, reading R6)
//   y = h W_down[e]                  (FP32 accumulation, ascending i; FP32 output)
// W_gate, W_up [E, H, I] and W_down [E, I, H], bf16 bits, row-major.
// h_out [R, I] (bf16 bits) is optional.
int oracle_expert_ffn(const uint16_t* x_perm, const int32_t* offsets, const uint16_t* wg,
                      const uint16_t* wu, const uint16_t* wd, int E, int H, int I, uint16_t* h_out,
                      float* y, int nthreads) {
  if (E <= 0 || H <= 0 || I <= 0) return 1;
  int64_t R = offsets[E];
  // Each row is independent; expert of row r found by scanning offsets.
  std::vector<int32_t> expert_of_row(R);
  for (int e = 0; e < E; ++e)
    for (int64_t r = offsets[e]; r < offsets[e + 1]; ++r) expert_of_row[r] = e;
  parallel_for(R, nthreads, [&](int64_t r) {
    int e = expert_of_row[r];
    const uint16_t* xr = x_perm + r * H;
    const uint16_t* Wg = wg + (int64_t)e * H * I;
    const uint16_t* Wu = wu + (int64_t)e * H * I;
    const uint16_t* Wd = wd + (int64_t)e * I * H;
    std::vector<float> g(I, 0.0f), u(I, 0.0f), hf(I);
    for (int h = 0; h < H; ++h) {
      float xv = bf16_to_f32(xr[h]);
      const uint16_t* grow = Wg + (int64_t)h * I;
      const uint16_t* urow = Wu + (int64_t)h * I;
      for (int i = 0; i < I; ++i) {
        g[i] = g[i] + xv * bf16_to_f32(grow[i]);
        u[i] = u[i] + xv * bf16_to_f32(urow[i]);
      }
    }
    for (int i = 0; i < I; ++i) {
      uint16_t hb = f32_to_bf16(silu(g[i]) * u[i]);
      if (h_out) h_out[r * I + i] = hb;
      hf[i] = bf16_to_f32(hb);
    }
    float* yr = y + r * H;
    for (int c = 0; c < H; ++c) yr[c] = 0.0f;
    for (int i = 0; i < I; ++i) {
      float hv = hf[i];
      const uint16_t* drow = Wd + (int64_t)i * H;
      for (int c = 0; c < H; ++c) yr[c] = yr[c] + hv * bf16_to_f32(drow[c]);
    }
  });
  return 0;
}

// Step 8: out[t, c] = bf16(acc), acc = 0; for j = 0..k-1: acc = fma(w[t,j], y[row_of_slot[t*k+j], c], acc)
// (reading R7).
int oracle_combine(const float* y, const float* w, const int32_t* row_of_slot, int T, int H, int k,
                   uint16_t* out, int nthreads) {
  if (T < 0 || H <= 0 || k < 1) return 1;
  parallel_for(T, nthreads, [&](int64_t t) {
    for (int c = 0; c < H; ++c) {
      float acc = 0.0f;
      for (int j = 0; j < k; ++j) {
        int64_t r = row_of_slot[t * k + j];
        acc = std::fma(w[t * k + j], y[r * H + c], acc);
      }
      out[t * H + c] = f32_to_bf16(acc);
    }
  });
  return 0;
}

// Combine with a routing scale (GLM's factor applied inside the expert kernel):
// each slot's weight is first multiplied by `scale` in FP32 (one rounding), then
// the slot-order FMA chain runs as in oracle_combine.
int oracle_combine_scaled(const float* y, const float* w, const int32_t* row_of_slot, float scale,
                          int T, int H, int k, uint16_t* out, int nthreads) {
  if (T < 0 || H <= 0 || k < 1) return 1;
  parallel_for(T, nthreads, [&](int64_t t) {
    for (int c = 0; c < H; ++c) {
      float acc = 0.0f;
      for (int j = 0; j < k; ++j) {
        int64_t r = row_of_slot[t * k + j];
        acc = std::fma(scale * w[t * k + j], y[r * H + c], acc);
      }
      out[t * H + c] = f32_to_bf16(acc);
    }
  });
  return 0;
}

uint16_t oracle_f64_to_bf16(double x) { return f64_to_bf16(x); }

// Fixed expert-output reduction of G BF16 partials: partials [G][N] (logical
// order g = 0..G-1), out [N] = bf16(tree(partials[.][n])) (reading R9).
int oracle_tree_reduce(const uint16_t* partials, int G, int64_t N, uint16_t* out) {
  if (G < 1 || N < 0) return 1;
  std::vector<double> v(G);
  for (int64_t n = 0; n < N; ++n) {
    for (int g = 0; g < G; ++g) v[g] = (double)bf16_to_f32(partials[(int64_t)g * N + n]);
    out[n] = f64_to_bf16(fp64_pairwise_tree(v));
  }
  return 0;
}

// Sharded combine (reading R8): owner[e] in [0, G) is the rank that owns logical
// expert e.  For every token t, column c and rank g:
//   acc = 0; for j = 0..k-1: acc = fma(scale * w[t,j], owner[idx[t,j]] == g ? y[row,c] : 0, acc)
//   if shared (shared [G][T][H] FP32): acc = acc + shared[g,t,c]
//   partial[g,t,c] = bf16(acc)
// out[t,c] = bf16(FP64 tree over partial[0..G-1,t,c]).  partials_out is optional.
int oracle_combine_sharded(const float* y, const float* w, const int32_t* idx,
                           const int32_t* row_of_slot, const int32_t* owner, int G, float scale,
                           const float* shared, int T, int H, int E, int k, uint16_t* partials_out,
                           uint16_t* out, int nthreads) {
  if (T < 0 || H <= 0 || E <= 0 || k < 1 || G < 1) return 1;
  for (int e = 0; e < E; ++e)
    if (owner[e] < 0 || owner[e] >= G) return 1;
  parallel_for(T, nthreads, [&](int64_t t) {
    std::vector<double> v(G);
    for (int c = 0; c < H; ++c) {
      for (int g = 0; g < G; ++g) {
        float acc = 0.0f;
        for (int j = 0; j < k; ++j) {
          const int e = idx[t * k + j];
          const int64_t r = row_of_slot[t * k + j];
          const float val = (owner[e] == g) ? y[r * H + c] : 0.0f;
          acc = std::fma(scale * w[t * k + j], val, acc);
        }
        if (shared) acc = acc + shared[((int64_t)g * T + t) * H + c];
        const uint16_t p = f32_to_bf16(acc);
        if (partials_out) partials_out[((int64_t)g * T + t) * H + c] = p;
        v[g] = (double)bf16_to_f32(p);
      }
      out[t * H + c] = f64_to_bf16(fp64_pairwise_tree(v));
    }
  });
  return 0;
}

// Shared expert sharded G ways (reading R10): W_gate, W_up [H, Is], W_down [Is, H]
// (bf16 bits, row-major).  Rank g takes intermediate columns [g*Is/G, (g+1)*Is/G)
// and runs them as one expert over all T tokens (oracle_expert_ffn with E = 1).
// shared [G][T][H] FP32.
int oracle_shared_expert(const uint16_t* x, const uint16_t* wg, const uint16_t* wu,
                         const uint16_t* wd, int T, int H, int Is, int G, float* shared,
                         int nthreads) {
  if (T < 0 || H <= 0 || Is <= 0 || G < 1 || Is % G != 0) return 1;
  const int Ig = Is / G;
  std::vector<uint16_t> sg((size_t)H * Ig), su((size_t)H * Ig);
  const int32_t offsets[2] = {0, T};
  for (int g = 0; g < G; ++g) {
    for (int h = 0; h < H; ++h)
      for (int i = 0; i < Ig; ++i) {
        sg[(size_t)h * Ig + i] = wg[(size_t)h * Is + (size_t)g * Ig + i];
        su[(size_t)h * Ig + i] = wu[(size_t)h * Is + (size_t)g * Ig + i];
      }
    const uint16_t* sd = wd + (size_t)g * Ig * H;  // rows g*Ig .. (g+1)*Ig - 1
    const int rc = oracle_expert_ffn(x, offsets, sg.data(), su.data(), sd, 1, H, Ig, nullptr,
                                     shared + (size_t)g * T * H, nthreads);
    if (rc) return rc;
  }
  return 0;
}

// The whole layer: steps 1-8 in order.  Outputs idx/w/counts are optional.
int oracle_layer_fwd(const uint16_t* x, const float* wr, const float* bias, const uint16_t* wg,
                     const uint16_t* wu, const uint16_t* wd, int T, int H, int E, int k, int I,
                     uint16_t* out, int32_t* idx_out, float* w_out, int32_t* counts_out,
                     int nthreads) {
  if (T < 0 || H <= 0 || E <= 0 || I <= 0 || k < 1 || k > E) return 1;
  int64_t R = (int64_t)T * k;
  std::vector<int32_t> idx(R), counts(E), offsets(E + 1), row_of_slot(R), slot_of_row(R);
  std::vector<float> w(R);
  int rc = oracle_route(x, wr, bias, T, H, E, k, idx.data(), w.data(), nthreads);
  if (rc) return rc;
  rc = oracle_load_stats(idx.data(), T, k, E, counts.data(), offsets.data(), nullptr, nullptr);
  if (rc) return rc;
  std::vector<uint16_t> x_perm((size_t)R * H);
  rc = oracle_permute(x, idx.data(), offsets.data(), T, H, E, k, x_perm.data(), row_of_slot.data(),
                      slot_of_row.data());
  if (rc) return rc;
  std::vector<float> y((size_t)R * H);
  rc = oracle_expert_ffn(x_perm.data(), offsets.data(), wg, wu, wd, E, H, I, nullptr, y.data(),
                         nthreads);
  if (rc) return rc;
  rc = oracle_combine(y.data(), w.data(), row_of_slot.data(), T, H, k, out, nthreads);
  if (rc) return rc;
  if (idx_out) std::memcpy(idx_out, idx.data(), sizeof(int32_t) * R);
  if (w_out) std::memcpy(w_out, w.data(), sizeof(float) * R);
  if (counts_out) std::memcpy(counts_out, counts.data(), sizeof(int32_t) * E);
  return 0;
}

}  // extern "C"
