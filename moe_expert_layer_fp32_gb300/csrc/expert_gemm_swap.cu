// Grouped expert GEMMs for small batches: the weight rows on the MMA's M side.
//
// "RoutePack", section 2.3 (a rank's experts run as one grouped operation);
// "0 train-infer mismatch for open-weight MoE RL", sections "SwiGLU: rounding
// after the multiply" and "Matrix multiplication: the same reduction along K".
// The same two GEMMs as the tile kernels in expert_gemm.cu:
//   gate/up: h[r, :] = bf16(silu(x_perm[r] Wg_e) * (x_perm[r] Wu_e))
//   down:    y[r, :] = h[r] Wd_e                              (FP32 out)
//
// When experts hold a handful of rows (decode), a 128-row token tile is almost
// empty and each MMA of N = 256 weight columns costs the full tensor time for a
// few useful rows.  Here the transposed product is formed instead:
//   D^T[w, r] = sum_k W[w, k] X[r, k]
// with M = 128 weight rows per MMA and N = 16, 32 or 64 token rows, so the MMAs
// are short and the kernel is bound by streaming the weights from HBM.
//
// Work unit: (expert e, one packed 256-row weight box column, up to 64 of e's
// rows).  The box's two 128-row halves are the two M = 128 operands: for gate/up
// the gate and the up rows of the same 128 intermediate columns (the packed
// interleave), for down two 128-column halves of the output.  Per stage the
// producer loads one 256 x 64 weight box (32 KB, contiguous in the box-tiled
// packing) and one N x 64 token box; the MMA issuer runs, per 16-wide K step,
// one MMA per half into two TMEM accumulators of N columns (double-buffered).
// Units are numbered expert-major, then weight column, then token tile, so the
// token tiles of one weight column run side by side and share its L2 lines.
// When whole-box units would fill at most half of the SMs, units shrink so that
// twice as many SMs stream the weights, with the same chain and epilogue per
// element:
//   down (HV = 1): one 128-row half of a box, one MMA per K step;
//   gate/up (HV = 4): 64 gate rows and the matching 64 up rows of a box, loaded
//     as two 64-row boxes into one 128-row operand, one MMA per K step; TMEM
//     lanes 0-63 then hold gate and 64-127 up, so the two epilogue warps that own
//     the up lanes pass their values to the gate warps through shared memory.
//
// Each output element is the same K order (64-wide k-blocks ascending, 16-wide
// MMAs ascending, FP32 accumulation from zero) over the same BF16 products as in
// the tile kernels, and the epilogue applies the same operations (silu_f32, one
// FP32 product, one BF16 rounding; or the FP32 value as it is).  A layer test
// checks that rows computed here and by the tile kernels are bit-identical, which
// keeps the output batch-invariant when the host switches forms with the number
// of rows.
//
// Roles and bounded waits are those of the tile kernels: warp 0 lane 0 TMA
// producer, warp 1 lane 0 MMA issuer, warps 2..5 epilogue (TMEM lane quarter =
// warp % 4); every wait has a clock limit and an abort path that drains this
// CTA's own copies and MMAs before tensor memory is freed.
//
// Both GEMMs are programmatic dependent launches (pdl.cuh).  The gate/up GEMM
// waits for its predecessor (the dispatch) before reading the offsets; the down
// GEMM reads the offsets at once, builds its schedule and issues its first weight
// stages, and waits for the gate/up GEMM only before its first token (h) copy.
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int SK = 64;                       // k-block: one 128-byte swizzle row
constexpr int SUK = 16;                      // MMA K
constexpr int WROWS = 256;                   // rows of one packed weight box
constexpr int HALF = 128;                    // MMA M
constexpr int kTT = 64;                      // token rows per unit at most (MMA N <= 64)

// HV selects the unit: 2 = a whole packed box (two M = 128 MMAs per K step; gate
// and up meet in one CTA), 1 = one 128-row half of a box (down only), 4 = 64 gate
// rows + the matching 64 up rows of a box in one M = 128 operand (gate/up only).
// TT: token rows per unit at most: 64, or 16 when the whole batch has at most 16
// rows (T <= 2 for k = 8).  The down GEMM is a programmatic dependent launch of
// the gate/up GEMM: its CTAs start on SMs with room while the gate/up GEMM runs
// and stream their first weight stages before they wait for h.  The TT = 16
// quarter and half units hold five and six stages of 16 KB + a 2 KB token box
// (about 100 and 115 KB), so a gate/up CTA and a down CTA fit on one SM together.
template <int HV, int TT = kTT>
struct SwapCfg {
  static constexpr int UROWS = HV == 2 ? 2 * HALF : HALF;  // weight rows per unit
  static constexpr int NMMA = HV == 2 ? 2 : 1;             // M = 128 MMAs per K step
  static constexpr int X_BYTES = TT * SK * 2;              // token box (N = TT)
  // TT = 16: five stages for gate/up units, six for half (down) units, so the
  // down CTA holds more of its weights before its wait (the pair still fits)
  static constexpr int STAGES = HV == 2 ? 5 : (TT == 16 ? (HV == 1 ? 6 : 5) : 8);
  static constexpr int W_BYTES = UROWS * SK * 2;           // 32 or 16 KB
  static constexpr int HOFF = TT < 32 ? 32 : TT;           // TMEM columns per half (32-aligned)
  static constexpr int ACC_COLS = NMMA * HOFF;             // one accumulator buffer
  static constexpr int TMEM_COLS = 2 * ACC_COLS;           // double-buffered
  static constexpr int NBAR = 2 * STAGES + 2 + 2 + 1;
  // HV = 4: up values of 64 weight rows x TT token rows, passed to the gate warps
  static constexpr int XCH_BYTES = HV == 4 ? 64 * (TT + 1) * 4 : 0;
  static constexpr int SMEM_BYTES = 1024 + STAGES * (W_BYTES + X_BYTES) + XCH_BYTES + NBAR * 8 +
                                    16 + 3 * (kMaxE + 1) * 4;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};
// a gate/up quarter-unit CTA and a down half-unit CTA on one SM (228 KB, 1 KB each
// reserved)
static_assert(SwapCfg<4, 16>::SMEM_BYTES + SwapCfg<1, 16>::SMEM_BYTES + 2048 <= 228 * 1024,
              "co-resident TT = 16 units");

// Weight boxes (UROWS rows; 64 for HV = 4) and token boxes of 16, 32 and 64 rows;
// all 64 columns.
struct SwapMaps {
  CUtensorMap w, x16, x32, x64;
};

struct SwapWork {
  int e, wt;       // expert, weight box column (256 output rows of the transposed tile)
  int row0, rows;  // first token row (output row) and rows that belong to e (<= TT)
  int nb;          // MMA N = token box rows: 16, 32 or 64
  int x_load_row;  // first row of the token box
  int w_load_row;  // box row of k-block 0 in the packed weights
};

template <int HV, int TT>
__device__ __forceinline__ SwapWork swap_decode(int u, const int* s_prefix, const int* s_off,
                                                const int* s_tt, int E, int NTW, int KB,
                                                int a_local) {
  // largest e with s_prefix[e] <= u (experts without rows share the next prefix)
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  const int local = u - s_prefix[lo];
  const int tt = s_tt[lo];
  SwapWork w;
  w.e = lo;
  w.wt = local / tt;
  const int ti = local - w.wt * tt;
  w.row0 = s_off[lo] + ti * TT;
  w.rows = min(TT, s_off[lo + 1] - w.row0);
  w.nb = (TT == 16 || w.rows <= 16) ? 16 : (w.rows <= 32 ? 32 : 64);
  w.x_load_row = w.row0 - (a_local ? s_off[lo] : 0);
  // box row of (expert, box, k-block 0), plus the unit's rows within the box:
  // HV = 1 its 128-row half, HV = 4 its 64 gate rows (its up rows are 128 further)
  if constexpr (HV == 2) {
    w.w_load_row = (lo * NTW + w.wt) * KB * WROWS;
  } else {
    const int NTB = NTW / 2;  // packed boxes per expert
    w.w_load_row = (lo * NTB + (w.wt >> 1)) * KB * WROWS + (w.wt & 1) * (HV == 1 ? HALF : 64);
  }
  return w;
}

// 32 lanes x 16 consecutive 32-bit columns: thread i gets lane (base + i).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

template <bool SWIGLU, int HV, int TT, bool DEP>
__global__ void __launch_bounds__(192, 1)
    grouped_gemm_swap_kernel(const __grid_constant__ SwapMaps maps,
                             const int32_t* __restrict__ offsets, int E, int R, int n_per_expert,
                             int K, void* __restrict__ out, int out_ld, int32_t* status,
                             long long spin_limit, int a_local, const int32_t* one_token_ids,
                             int k_ids) {
  using C = SwapCfg<HV, TT>;
  static_assert(SWIGLU ? HV != 1 : HV != 4, "gate and up rows of a unit must meet in one CTA");
  constexpr int STAGES = C::STAGES, W_BYTES = C::W_BYTES, ACC_COLS = C::ACC_COLS;
  constexpr int X_BYTES = C::X_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sW = base;
  uint8_t* sX = base + STAGES * W_BYTES;
  float* s_xch = reinterpret_cast<float*>(sX + STAGES * X_BYTES);  // HV = 4 only
  uint64_t* bars = reinterpret_cast<uint64_t*>(sX + STAGES * X_BYTES + C::XCH_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_prefix = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_off = s_prefix + (kMaxE + 1);
  int* s_tt = s_off + (kMaxE + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NTW = n_per_expert / C::UROWS;  // units per expert (and token tile)
  const int KB = K / SK;

  // prologue that touches no memory the previous kernel writes: barriers, tensor
  // maps (kernel parameters), tensor memory
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&maps.w);
    prefetch_tensormap(&maps.x16);
    prefetch_tensormap(&maps.x32);
    prefetch_tensormap(&maps.x64);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  // The gate/up GEMM waits here for the kernel that wrote the offsets and the
  // token rows, then lets the down GEMM start.  The down GEMM (DEP) reads the
  // offsets at once (their writer finished before the gate/up GEMM passed this
  // point) and waits only before its first load of h, the gate/up output.
  if constexpr (!DEP) {
    pdl_wait();
    if (threadIdx.x == 0) pdl_launch_dependents();
  }
  if (one_token_ids == nullptr) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = __ldg(offsets + e);
  } else if (warp == 0) {
    // one token (R = k_ids rows): the offsets of the stable permutation follow from
    // its k distinct expert ids, o_e = #{j : id_j < e}; a bad or repeated id
    // leaves o_E = 0 != R, which the check below rejects
    const int id = lane < k_ids ? __ldg(one_token_ids + lane) : -1;
    bool bad = lane < k_ids && (id < 0 || id >= E);
    int ids[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      ids[j] = __shfl_sync(0xFFFFFFFFu, id, j);
      if (j < k_ids && j != lane && lane < k_ids && ids[j] == id) bad = true;
    }
    bad = __any_sync(0xFFFFFFFFu, bad);
    for (int e = lane; e <= E; e += 32) {
      int c = 0;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) c += (j < k_ids && ids[j] < e) ? 1 : 0;
      s_off[e] = bad ? 0 : c;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // schedule, one warp: validate offsets (0 = o_0 <= o_1 <= ... <= o_E = R),
    // token tiles per expert and the exclusive prefix of work units, 32 experts
    // per step (a scan over the lanes)
    bool ok = true;
    int carry = 0;
    for (int eb = 0; eb < E; eb += 32) {
      const int e = eb + lane;
      int cnt = 0;
      if (e < E) {
        const int a = s_off[e], b = s_off[e + 1];
        if (b < a) ok = false;
        const int tt = b > a ? (b - a + TT - 1) / TT : 0;
        s_tt[e] = tt;
        cnt = tt * NTW;
      }
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += n;
      }
      if (e < E) s_prefix[e] = carry + incl - cnt;
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    ok = __all_sync(0xFFFFFFFFu, ok) && s_off[0] == 0 && s_off[E] == R;
    if (!ok) {
      for (int e = lane; e < E; e += 32) s_prefix[e] = 0;
      carry = 0;
      if (lane == 0) flag_error(status, MOE_ERR_DEVICE_CHECK);
    }
    if (lane == 0) s_prefix[E] = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = s_prefix[E];

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int it = 0;
      bool aborted = false;
      bool first = true;
      for (int u = blockIdx.x; u < total && !aborted; u += gridDim.x, first = false) {
        const SwapWork w = swap_decode<HV, TT>(u, s_prefix, s_off, s_tt, E, NTW, KB, a_local);
        const CUtensorMap* xm = w.nb == 16 ? &maps.x16 : (w.nb == 32 ? &maps.x32 : &maps.x64);
        const uint32_t bytes = W_BYTES + w.nb * SK * 2;
        // DEP (a dependent launch): the first unit's first stages get their weight
        // boxes now and their token boxes (rows of the previous grid's output) only
        // after griddepcontrol.wait, i.e. once that grid has finished and its
        // writes are visible
        const int ndefer = (DEP && first) ? min(STAGES, KB) : 0;
        const int it0 = it;
        // (also on an abort: every armed stage then still receives its bytes, so
        // the drain below ends)
        auto load_deferred = [&](int n) {
          pdl_wait();
          pdl_launch_dependents();  // the combine may start; it waits for this grid
          for (int j = 0; j < n; ++j) {
            const int sj = (it0 + j) % STAGES;
            tma_load_2d(xm, sX + sj * X_BYTES, &full[sj], j * SK, w.x_load_row);
          }
        };
        for (int kb = 0; kb < KB; ++kb, ++it) {
          if (kb == ndefer && ndefer > 0) load_deferred(ndefer);
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, status, spin_limit)) {
            if (kb < ndefer) load_deferred(kb);
            aborted = true;
            break;
          }
          mbar_arrive_expect_tx(&full[s], bytes);
          tma_load_2d(&maps.w, sW + s * W_BYTES, &full[s], 0, w.w_load_row + kb * WROWS);
          if constexpr (HV == 4)  // the matching up rows, into operand rows 64..127
            tma_load_2d(&maps.w, sW + s * W_BYTES + 64 * 128, &full[s], 0,
                        w.w_load_row + HALF + kb * WROWS);
          if (kb >= ndefer) tma_load_2d(xm, sX + s * X_BYTES, &full[s], kb * SK, w.x_load_row);
        }
        if (ndefer > 0 && ndefer == KB && !aborted) load_deferred(ndefer);
      }
      if (aborted) {
        for (int i = (it > STAGES ? it - STAGES : 0); i < it; ++i)
          wait_drain(&full[i % STAGES], (i / STAGES) & 1, kSpinLimitCycles);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      int it = 0, tcount = 0;
      for (int u = blockIdx.x; u < total; u += gridDim.x, ++tcount) {
        const SwapWork w = swap_decode<HV, TT>(u, s_prefix, s_off, s_tt, E, NTW, KB, a_local);
        const uint32_t idesc = idesc_bf16_f32(HALF, w.nb);
        const int acc = tcount & 1;
        const uint32_t aph = (tcount >> 1) & 1;
        if (!mbar_wait_bounded(&tempty[acc], aph ^ 1, abort_flag, status, spin_limit)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + acc * ACC_COLS;  // half 0; half 1 at + HOFF
        bool aborted = false;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait_bounded(&full[s], ph, abort_flag, status, spin_limit)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          const uint32_t w_addr = smem_u32(sW + s * W_BYTES);
          const uint32_t x_addr = smem_u32(sX + s * X_BYTES);
#pragma unroll
          for (int kk = 0; kk < SK / SUK; ++kk) {
            const uint64_t xd = sdesc_k_major_sw128(x_addr + kk * SUK * 2);
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            mma_bf16(d0, sdesc_k_major_sw128(w_addr + kk * SUK * 2), xd, idesc, accum);
            if constexpr (HV == 2)
              mma_bf16(d0 + C::HOFF, sdesc_k_major_sw128(w_addr + HALF * 128 + kk * SUK * 2), xd,
                       idesc, accum);
          }
          mma_commit(&empty[s]);
        }
        if (aborted) break;
        mma_commit(&tfull[acc]);
      }
      mma_commit(mma_done);
      wait_drain(mma_done, 0, kSpinLimitCycles);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    // TMEM lane (32 q + lane) = weight row of each half; column j = token row0 + j.
    const int q = warp & 3;
    int tcount = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++tcount) {
      const SwapWork w = swap_decode<HV, TT>(u, s_prefix, s_off, s_tt, E, NTW, KB, a_local);
      const int acc = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&tfull[acc], aph, abort_flag, status, spin_limit);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      // HV = 4: the four warps meet at barriers below, so they go on or stop together
      if constexpr (HV == 4) ok = named_barrier_and(1, 128, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS);
      if constexpr (HV == 4) {
        // lanes 0-63: gate, 64-127: up, of intermediate column wt * 64 + (lane % 64);
        // warps owning the up lanes (q = 2, 3) hand them to the gate warps (q = 0, 1)
        float* xr = s_xch + (q & 1) * 32 * (TT + 1) + lane * (TT + 1);
        if (q >= 2) {
          for (int j0 = 0; j0 < w.nb; j0 += 16) {
            uint32_t uu[16];
            tmem_ld_32x32b_x16(taddr + j0, uu);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) xr[j0 + i] = __uint_as_float(uu[i]);
          }
        }
        named_barrier_sync(1, 128);
        if (q < 2) {
          uint16_t* h = static_cast<uint16_t*>(out) + (size_t)w.wt * 64 + q * 32 + lane;
          for (int j0 = 0; j0 < w.nb; j0 += 16) {
            uint32_t g[16];
            tmem_ld_32x32b_x16(taddr + j0, g);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int j = j0 + i;
              if (j < w.rows) {
                const float hv = __fmul_rn(silu_f32(__uint_as_float(g[i])), xr[j]);
                h[(size_t)(w.row0 + j) * out_ld] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
              }
            }
          }
        }
        named_barrier_sync(1, 128);  // the exchange buffer is free for the next unit
      } else if constexpr (SWIGLU) {
        // half 0: gate, half 1: up, of intermediate column wt * 128 + 32 q + lane
        uint16_t* h = static_cast<uint16_t*>(out) + (size_t)w.wt * HALF + q * 32 + lane;
        for (int j0 = 0; j0 < w.nb; j0 += 16) {
          uint32_t g[16], uu[16];
          tmem_ld_32x32b_x16(taddr + j0, g);
          tmem_ld_32x32b_x16(taddr + C::HOFF + j0, uu);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int j = j0 + i;
            if (j < w.rows) {
              const float hv =
                  __fmul_rn(silu_f32(__uint_as_float(g[i])), __uint_as_float(uu[i]));
              h[(size_t)(w.row0 + j) * out_ld] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
            }
          }
        }
      } else {
        // half c: output columns wt * UROWS + 128 c + 32 q + lane
        float* y = static_cast<float*>(out) + (size_t)w.wt * C::UROWS + q * 32 + lane;
#pragma unroll
        for (int c = 0; c < C::NMMA; ++c) {
          for (int j0 = 0; j0 < w.nb; j0 += 16) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(taddr + c * C::HOFF + j0, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int j = j0 + i;
              if (j < w.rows) y[(size_t)(w.row0 + j) * out_ld + c * HALF] = __uint_as_float(v[i]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <bool SWIGLU, int HV, int TT>
cudaError_t launch_swap_tt(const GemmOperand& a, const GemmOperand& b, const int32_t* offsets,
                           int E, int R, int n_per_expert, int K, void* out, int out_ld,
                           int32_t* status, long long spin_limit, cudaStream_t s, int a_local,
                           const int32_t* one_token_ids) {
  SwapMaps m;
  using C = SwapCfg<HV, TT>;
  // both GEMMs are programmatic dependent launches; the down GEMM (DEP) streams
  // weights before it waits
  constexpr bool DEP = !SWIGLU;
  auto kern = grouped_gemm_swap_kernel<SWIGLU, HV, TT, DEP>;
  if (!b.encode(&m.w, HV == 4 ? 64 : C::UROWS) || !a.encode(&m.x16, 16) || !a.encode(&m.x32, 32) ||
      !a.encode(&m.x64, 64))
    return cudaErrorInvalidValue;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64 || !attr_set[dev]) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    if (dev < 64) attr_set[dev] = true;
  }
  // units <= weight columns x (experts with rows + R / TT): one CTA per unit up to
  // one per SM (the kernel is persistent beyond that)
  const long long units =
      (long long)(n_per_expert / C::UROWS) * (std::min<long long>(E, R) + R / TT);
  const int grid = (int)std::max<long long>(1, std::min<long long>(device_sm_count(), units));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  pdl_attr(attr[0]);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // one token: k_ids = R
  return cudaLaunchKernelEx(&cfg, kern, m, offsets, E, R, n_per_expert, K, out, out_ld, status,
                            spin_limit, a_local, one_token_ids, R);
}

// TT = 16 when the whole batch has at most 16 rows (every expert then has at most
// 16): the same N = 16 MMAs per row as with TT = 64.
template <bool SWIGLU, int HV>
cudaError_t launch_swap(const GemmOperand& a, const GemmOperand& b, const int32_t* offsets, int E,
                        int R, int n_per_expert, int K, void* out, int out_ld, int32_t* status,
                        long long spin_limit, cudaStream_t s, int a_local,
                        const int32_t* one_token_ids = nullptr) {
  if (R <= 16)
    return launch_swap_tt<SWIGLU, HV, 16>(a, b, offsets, E, R, n_per_expert, K, out, out_ld,
                                          status, spin_limit, s, a_local, one_token_ids);
  return launch_swap_tt<SWIGLU, HV, kTT>(a, b, offsets, E, R, n_per_expert, K, out, out_ld, status,
                                         spin_limit, s, a_local, one_token_ids);
}

}  // namespace

// Measured on GB300 (L2 flushed, CUDA graph): the swapped form is 2-10% faster for
// fine_grained at T <= 64 and ling3_tiny at T <= 64, where the tile kernels' units
// are few and bound by one SM's tensor time per 128-row tile.  It is 4% slower for
// fine_grained at T >= 128 and for `large` at T = 64, where experts hold more rows
// or the units run many waves and both forms stream the weights at the HBM rate.
bool use_swap_gemm(int E, int R, int H, int I) {
  if ((2 * I) % WROWS != 0 || H % WROWS != 0) return false;
  if ((long long)R > (long long)kSwapRowsPerExpert * E) return false;
  const long long units = (long long)(2 * I / WROWS) * std::min(E, R);
  return units <= 4LL * device_sm_count();
}

cudaError_t launch_gemm_gate_up_swap(const GemmOperand& a, const GemmOperand& b,
                                     const int32_t* offsets, int E, int R, int H, int I, void* h,
                                     int32_t* status, long long spin_limit, cudaStream_t s,
                                     bool a_local, const int32_t* one_token_ids) {
  if (R == 0) return cudaSuccess;
  // one token: every expert's single row is the token itself (A rows from 0)
  const int al = (a_local || one_token_ids != nullptr) ? 1 : 0;
  // quarter units (64 gate + 64 up rows) while whole-box units would fill at most
  // half of the SMs (experts with rows <= min(E, R)); each element's chain and
  // epilogue arithmetic are the same
  if (2LL * (2 * I / WROWS) * std::min(E, R) <= device_sm_count())
    return launch_swap<true, 4>(a, b, offsets, E, R, 2 * I, H, h, I, status, spin_limit, s, al,
                                one_token_ids);
  return launch_swap<true, 2>(a, b, offsets, E, R, 2 * I, H, h, I, status, spin_limit, s, al,
                              one_token_ids);
}

cudaError_t launch_gemm_down_swap(const GemmOperand& a, const GemmOperand& b,
                                  const int32_t* offsets, int E, int R, int H, int I, float* y,
                                  int32_t* status, long long spin_limit, cudaStream_t s,
                                  const int32_t* one_token_ids) {
  if (R == 0) return cudaSuccess;
  // half-box units while whole-box units would fill at most half of the SMs
  // (experts with rows <= min(E, R)); each row's chain and epilogue are the same
  if (2LL * (H / WROWS) * std::min(E, R) <= device_sm_count())
    return launch_swap<false, 1>(a, b, offsets, E, R, H, I, y, H, status, spin_limit, s, 0,
                                 one_token_ids);
  return launch_swap<false, 2>(a, b, offsets, E, R, H, I, y, H, status, spin_limit, s, 0,
                               one_token_ids);
}

}  // namespace moe
