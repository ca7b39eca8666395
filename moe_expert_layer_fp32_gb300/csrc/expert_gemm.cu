// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// "RoutePack", section 2.3: a rank's local experts execute as one grouped
// operation.  "0 train-infer mismatch for open-weight MoE RL", section "SwiGLU:
// rounding after the multiply": gate and up in FP32, SiLU(gate)*up in FP32, one
// cast to BF16; section "Matrix multiplication: the same reduction along K": a
// reduction order that does not change with the number of rows.
//
//   GEMM-1 (gate/up, SwiGLU epilogue): h[r, :] = bf16(silu(x_perm[r] Wg_e) * (x_perm[r] Wu_e))
//   GEMM-2 (down):                     y[r, :] = h[r] Wd_e            (FP32 out)
//
// Design (one persistent CTA per SM, 192 threads, warp-specialised):
//   warp 0 lane 0   TMA producer: 128x64 A tile + BNx64 B tile per stage into a
//                   STAGES-deep ring of 128-byte-swizzled shared-memory buffers.
//   warp 1 lane 0   MMA issuer: tcgen05.mma kind::f16, M=128, N=BN, K=16, four
//                   per 64-wide k-block, accumulating in TMEM; tcgen05.commit
//                   frees each stage and signals a finished accumulator.
//   warps 2..5      epilogue: tcgen05.ld of their 32 TMEM lanes (= tile rows),
//                   SwiGLU or FP32 pass-through, 16-byte global stores of the
//                   rows that belong to the tile's expert.
// Two TMEM accumulators (2*BN columns) let the epilogue of tile i overlap the
// main loop of tile i+1.
//
// Tiles: for each expert e, ceil(M_e/128) row tiles x (N/BN) column tiles,
// numbered expert-major, row-tile, column-tile; CTA c takes tiles c, c+grid, ...
// The schedule is built on the device from `offsets`, so no host round trip.
// A row tile may run past its expert's last row into the next expert's rows or
// past the end (TMA fills zeros there); those rows are computed but never
// stored, and a row's result does not depend on the other rows of its tile.
// The tile shape, K order (k-blocks ascending, 16-wide MMAs ascending) and N
// split depend only on H and I, never on T: batch-invariant by construction.
//
// Every wait is bounded (clock64 limit); a wait that runs out raises a CTA-wide
// abort flag and records MOE_ERR_TIMEOUT; the roles then drain their own
// in-flight TMA copies and MMAs (bounded again) before TMEM is released.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int GM = 128;  // tile rows (MMA M)
constexpr int GK = 64;   // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int UK = 16;   // MMA K

template <int BN>
struct Cfg {
  static constexpr int STAGES = (BN == 256) ? 4 : 6;
  static constexpr int A_BYTES = GM * GK * 2;
  static constexpr int B_BYTES = BN * GK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int NBAR = 2 * STAGES + 2 + 2 + 1;
  // epilogue staging: per epilogue warp a 32 x 32-word tile (row stride 36 words)
  static constexpr int EPI_LD = 36;
  static constexpr int EPI_BYTES = 4 * 32 * EPI_LD * 4;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + NBAR * 8 + 16 +
                                    2 * (kMaxE + 1) * 4;
};

struct Tile {
  int e, nt, a_row0, rows;
};

__device__ __forceinline__ Tile decode_tile(int t, const int* s_prefix, const int* s_off, int E,
                                            int NT) {
  // largest e with s_prefix[e] <= t (experts without tiles share the next prefix)
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  const int local = t - s_prefix[lo];
  const int mt = local / NT;
  Tile ti;
  ti.e = lo;
  ti.nt = local - mt * NT;
  ti.a_row0 = s_off[lo] + mt * GM;
  ti.rows = min(GM, s_off[lo + 1] - ti.a_row0);
  return ti;
}

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, long long limit) {
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}

__device__ __forceinline__ float silu_f32(float g) { return __fdiv_rn(g, __fadd_rn(1.0f, expf(-g))); }

// One warp writes a 32-row x 128-byte block whose row i (i = lane) it holds in
// registers: the rows go through shared memory so that every global store
// instruction writes four whole 128-byte row segments instead of 32 scattered
// 16-byte pieces.  Row r of the block goes to dst + r * ld_bytes; rows >= nrows
// are skipped.
__device__ __forceinline__ void store_rows_128b(const uint32_t (&w)[32], uint32_t* stile, int lane,
                                                uint8_t* dst, size_t ld_bytes, int nrows) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    *reinterpret_cast<uint4*>(stile + lane * 36 + 4 * q) =
        make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  __syncwarp();
  const int cb = lane & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = i * 4 + (lane >> 3);
    const uint4 v = *reinterpret_cast<const uint4*>(stile + r * 36 + 4 * cb);
    if (r < nrows) *reinterpret_cast<uint4*>(dst + r * ld_bytes + 16 * cb) = v;
  }
  __syncwarp();
}

template <int BN, bool SWIGLU>
__global__ void __launch_bounds__(192, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const int32_t* __restrict__ offsets, int E, int R, int n_per_expert, int K,
                        void* __restrict__ out, int out_ld, int32_t* status,
                        long long spin_limit) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + C::STAGES * C::A_BYTES;
  uint32_t* s_epi = reinterpret_cast<uint32_t*>(sB + C::STAGES * C::B_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(s_epi) + C::EPI_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* tfull = bars + 2 * C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_prefix = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_off = s_prefix + (kMaxE + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = n_per_expert / BN;
  const int KB = K / GK;

  if (threadIdx.x == 0) {
    // schedule: validate offsets (0 = o_0 <= o_1 <= ... <= o_E = R), tile prefix
    bool ok = __ldg(offsets) == 0 && __ldg(offsets + E) == R;
    int p = 0;
    for (int e = 0; e < E; ++e) {
      const int a = __ldg(offsets + e), b = __ldg(offsets + e + 1);
      if (b < a) ok = false;
      s_off[e] = a;
      s_prefix[e] = p;
      if (b > a) p += ((b - a + GM - 1) / GM) * NT;
    }
    s_off[E] = __ldg(offsets + E);
    if (!ok) {
      flag_error(status, MOE_ERR_DEVICE_CHECK);
      for (int e = 0; e < E; ++e) s_prefix[e] = 0;
      p = 0;
    }
    s_prefix[E] = p;
    *abort_flag = 0;
    for (int s = 0; s < C::STAGES; ++s) {
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
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = s_prefix[E];

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int it = 0;  // k-blocks issued
      bool aborted = false;
      for (int t = blockIdx.x; t < total && !aborted; t += gridDim.x) {
        const Tile ti = decode_tile(t, s_prefix, s_off, E, NT);
        const int b_row0 = ti.e * n_per_expert + ti.nt * BN;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, status, spin_limit)) {
            aborted = true;
            break;
          }
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          tma_load_2d(&tmA, sA + s * C::A_BYTES, &full[s], kb * GK, ti.a_row0);
          tma_load_2d(&tmB, sB + s * C::B_BYTES, &full[s], kb * GK, b_row0);
        }
      }
      if (aborted) {
        // the copies issued into the last STAGES slots may still be in flight
        for (int i = (it > C::STAGES ? it - C::STAGES : 0); i < it; ++i)
          wait_drain(&full[i % C::STAGES], (i / C::STAGES) & 1, spin_limit);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t IDESC = idesc_bf16_f32(GM, BN);
      int it = 0, tcount = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x, ++tcount) {
        const int acc = tcount & 1;
        const uint32_t aph = (tcount >> 1) & 1;
        if (!mbar_wait_bounded(&tempty[acc], aph ^ 1, abort_flag, status, spin_limit)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool aborted = false;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait_bounded(&full[s], ph, abort_flag, status, spin_limit)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + s * C::A_BYTES);
          const uint32_t b_addr = smem_u32(sB + s * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < GK / UK; ++kk) {
            mma_bf16(d_tmem, sdesc_k_major_sw128(a_addr + kk * UK * 2),
                     sdesc_k_major_sw128(b_addr + kk * UK * 2), IDESC,
                     (kb > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
        if (aborted) break;
        mma_commit(&tfull[acc]);
      }
      // every MMA this thread issued completes before TMEM is released
      mma_commit(mma_done);
      wait_drain(mma_done, 0, spin_limit);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int tcount = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++tcount) {
      const Tile ti = decode_tile(t, s_prefix, s_off, E, NT);
      const int acc = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&tfull[acc], aph, abort_flag, status, spin_limit);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      // rows of this warp's 32-row block that belong to the tile's expert
      const int nrows = min(32, max(0, ti.rows - q * 32));
      uint32_t* stile = s_epi + q * 32 * C::EPI_LD;
      if constexpr (SWIGLU) {
        // accumulator columns [0, BN/2) = gate, [BN/2, BN) = up, same intermediate index;
        // 64 intermediate columns (128 bytes of h per row) per pass
        uint8_t* dst = static_cast<uint8_t*>(out) +
                       ((size_t)(ti.a_row0 + q * 32) * out_ld + ti.nt * (BN / 2)) * 2;
#pragma unroll 1
        for (int c0 = 0; c0 < BN / 2; c0 += 64) {
          uint32_t hp[32];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t g[32], u[32];
            tmem_ld_32x32b_x32(taddr + c0 + 32 * half, g);
            tmem_ld_32x32b_x32(taddr + BN / 2 + c0 + 32 * half, u);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float h0 =
                  __fmul_rn(silu_f32(__uint_as_float(g[2 * i])), __uint_as_float(u[2 * i]));
              const float h1 = __fmul_rn(silu_f32(__uint_as_float(g[2 * i + 1])),
                                         __uint_as_float(u[2 * i + 1]));
              hp[16 * half + i] = pack_bf16x2(h0, h1);
            }
          }
          store_rows_128b(hp, stile, lane, dst + c0 * 2, (size_t)out_ld * 2, nrows);
        }
      } else {
        uint8_t* dst = static_cast<uint8_t*>(out) +
                       ((size_t)(ti.a_row0 + q * 32) * out_ld + ti.nt * BN) * 4;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + c0, v);
          tmem_ld_wait();
          store_rows_128b(v, stile, lane, dst + c0 * 4, (size_t)out_ld * 4, nrows);
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

template <int BN, bool SWIGLU>
cudaError_t launch_grouped(const CUtensorMap& a, const CUtensorMap& b, const int32_t* offsets,
                           int E, int R, int n_per_expert, int K, void* out, int out_ld,
                           int32_t* status, long long spin_limit, cudaStream_t s) {
  using C = Cfg<BN>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && !attr_set[dev]) {
    err = cudaFuncSetAttribute(grouped_gemm_kernel<BN, SWIGLU>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  const int grid = device_sm_count();
  grouped_gemm_kernel<BN, SWIGLU><<<grid, 192, C::SMEM_BYTES, s>>>(
      a, b, offsets, E, R, n_per_expert, K, out, out_ld, status, spin_limit);
  return cudaGetLastError();
}

}  // namespace

int gemm_down_bn(int H) { return (H % 256 == 0) ? 256 : 128; }

cudaError_t launch_gemm_gate_up(const CUtensorMap& a_xperm, const CUtensorMap& b_w1,
                                const int32_t* offsets, int E, int R, int H, int I, void* h,
                                int32_t* status, long long spin_limit, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  return launch_grouped<256, true>(a_xperm, b_w1, offsets, E, R, 2 * I, H, h, I, status,
                                   spin_limit, s);
}

cudaError_t launch_gemm_down(const CUtensorMap& a_h, const CUtensorMap& b_w2,
                             const int32_t* offsets, int E, int R, int H, int I, float* y,
                             int32_t* status, long long spin_limit, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  if (gemm_down_bn(H) == 256)
    return launch_grouped<256, false>(a_h, b_w2, offsets, E, R, H, I, y, H, status, spin_limit, s);
  return launch_grouped<128, false>(a_h, b_w2, offsets, E, R, H, I, y, H, status, spin_limit, s);
}

}  // namespace moe
