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
// Design (persistent CTAs, one per SM, 192 threads, warp-specialised):
//   warp 0 lane 0   TMA producer: 128x64 A tile + BNx64 B tile per stage into a
//                   STAGES-deep ring of 128-byte-swizzled shared-memory buffers.
//   warp 1 lane 0   MMA issuer: tcgen05.mma kind::f16, M=128, N=BN, K=16, four
//                   per 64-wide k-block, accumulating in TMEM; tcgen05.commit
//                   frees each stage and signals a finished accumulator.
//   warps 2..5      epilogue: tcgen05.ld of their 32 TMEM lanes (= tile rows),
//                   SwiGLU or FP32 pass-through, rows staged through shared
//                   memory so every global store writes whole 128-byte segments.
// Two TMEM accumulators (2*BN columns) let the epilogue of tile i overlap the
// main loop of tile i+1.
//
// Tiles: for each expert e, ceil(M_e/128) row tiles x (N/BN) column tiles, built
// on the device from `offsets` (no host round trip).  A row tile may run past
// its expert's last row into the next expert's rows or past the end (TMA fills
// zeros there); those rows are computed but never stored, and a row's result
// does not depend on the other rows of its tile.
//
// A pair variant (grouped_gemm_pair_kernel, below) runs one M=256 MMA across the
// two CTAs of a cluster (cta_group::2); the launchers use it where it measured
// faster.  Every TMA load of both kernels writes only the issuing CTA's own shared
// memory (no cluster multicast).
//
// The tile shape, K order (k-blocks ascending, 16-wide MMAs ascending) and N
// split depend only on H and I, never on T: batch-invariant by construction.
//
// Every wait is bounded (clock64 limit, spin_limit); a wait that runs out raises a
// CTA-wide abort flag and records MOE_ERR_TIMEOUT; the roles then drain their own
// in-flight TMA copies and MMAs (bounded by the fixed default limit, whatever
// spin_limit is) before TMEM is released, and
// the two CTAs of a pair meet at a cluster barrier before either exits.
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

// Tensor maps of one grouped GEMM: A (rows of x_perm or h) in boxes of 128 rows,
// B (packed weight rows) in boxes of BN rows (single-CTA kernel) or BN/2 rows (one
// CTA's half of the pair kernel's tile); all 64 columns.
struct Maps {
  CUtensorMap a128, b_tile;
};

// One work unit of the single-CTA kernel: one 128-row tile of one expert's rows
// times one BN-column tile.
struct Work {
  int e, nt;       // expert, column tile
  int a_row0;      // first output row of the tile
  int rows;        // rows of the tile that belong to expert e
  int a_load_row;  // first row of the A box
  int b_load_row;  // box row of k-block 0 in the packed weights
};

// Units are numbered expert-major, then row tile, then column tile.
// a_local: every group reads A rows from 0 (one A operand shared by all groups,
// e.g. the token rows of a shared expert split into column shards); otherwise a
// group's A rows are its output rows.
template <int BN>
__device__ __forceinline__ Work decode(int u, const int* s_prefix, const int* s_off, int E, int NT,
                                       int KB, int a_local) {
  // largest e with s_prefix[e] <= u (experts without work share the next prefix)
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  const int local = u - s_prefix[lo];
  const int mt = local / NT;
  Work w;
  w.e = lo;
  w.nt = local - mt * NT;
  w.a_row0 = s_off[lo] + mt * GM;
  w.rows = min(GM, s_off[lo + 1] - w.a_row0);
  w.a_load_row = w.a_row0 - (a_local ? s_off[lo] : 0);
  // B is packed box by box: (expert, column tile, k-block) -> BN contiguous rows of
  // 64 K values; this is the box row of k-block 0 (k-block kb adds kb * BN)
  w.b_load_row = (lo * NT + w.nt) * KB * BN;
  return w;
}

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

// Epilogue of one warp's 32-row block of an accumulator: TMEM columns at taddr
// (this warp's lane quarter), output rows row0 .. row0 + nrows - 1, column tile nt.
// SWIGLU: columns [0, BN/2) are gate and [BN/2, BN) up for the same intermediate
// index; h = bf16(silu(gate) * up), 64 intermediate columns (128 bytes) per pass.
// Otherwise the FP32 accumulator is stored as it is.
template <int BN, bool SWIGLU>
__device__ __forceinline__ void epilogue_block(uint32_t taddr, int row0, int nt, int nrows,
                                               uint32_t* stile, int lane, void* out, int out_ld) {
  if constexpr (SWIGLU) {
    uint8_t* dst = static_cast<uint8_t*>(out) + ((size_t)row0 * out_ld + nt * (BN / 2)) * 2;
#pragma unroll 1
    for (int c0 = 0; c0 < BN / 2; c0 += 64) {
      uint32_t hp[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t g[32], uu[32];
        tmem_ld_32x32b_x32(taddr + c0 + 32 * half, g);
        tmem_ld_32x32b_x32(taddr + BN / 2 + c0 + 32 * half, uu);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float h0 =
              __fmul_rn(silu_f32(__uint_as_float(g[2 * i])), __uint_as_float(uu[2 * i]));
          const float h1 =
              __fmul_rn(silu_f32(__uint_as_float(g[2 * i + 1])), __uint_as_float(uu[2 * i + 1]));
          hp[16 * half + i] = pack_bf16x2(h0, h1);
        }
      }
      store_rows_128b(hp, stile, lane, dst + c0 * 2, (size_t)out_ld * 2, nrows);
    }
  } else {
    uint8_t* dst = static_cast<uint8_t*>(out) + ((size_t)row0 * out_ld + nt * BN) * 4;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      uint32_t v[32];
      tmem_ld_32x32b_x32(taddr + c0, v);
      tmem_ld_wait();
      store_rows_128b(v, stile, lane, dst + c0 * 4, (size_t)out_ld * 4, nrows);
    }
  }
}

template <int BN, bool SWIGLU>
__global__ void __launch_bounds__(192, 1)
    grouped_gemm_kernel(const __grid_constant__ Maps maps, const int32_t* __restrict__ offsets,
                        int E, int R, int n_per_expert, int K, void* __restrict__ out, int out_ld,
                        int32_t* status, long long spin_limit, int a_local) {
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

  // all threads bring the offsets in at once; thread 0 then builds the schedule from
  // shared memory (a serial walk over global memory would cost E load latencies)
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = __ldg(offsets + e);
  __syncthreads();
  if (threadIdx.x == 0) {
    // schedule: validate offsets (0 = o_0 <= o_1 <= ... <= o_E = R), work prefix
    bool ok = s_off[0] == 0 && s_off[E] == R;
    int p = 0;
    for (int e = 0; e < E; ++e) {
      const int a = s_off[e], b = s_off[e + 1];
      if (b < a) ok = false;
      s_prefix[e] = p;
      p += (b > a ? (b - a + GM - 1) / GM : 0) * NT;
    }
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
    prefetch_tensormap(&maps.a128);
    prefetch_tensormap(&maps.b_tile);
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
      for (int u = blockIdx.x; u < total && !aborted; u += gridDim.x) {
        const Work w = decode<BN>(u, s_prefix, s_off, E, NT, KB, a_local);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, status, spin_limit)) {
            aborted = true;
            break;
          }
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          tma_load_2d(&maps.a128, sA + s * C::A_BYTES, &full[s], kb * GK, w.a_load_row);
          tma_load_2d(&maps.b_tile, sB + s * C::B_BYTES, &full[s], 0, w.b_load_row + kb * BN);
        }
      }
      if (aborted) {
        // the copies issued into the last STAGES slots may still be in flight
        for (int i = (it > C::STAGES ? it - C::STAGES : 0); i < it; ++i)
          wait_drain(&full[i % C::STAGES], (i / C::STAGES) & 1, kSpinLimitCycles);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t IDESC = idesc_bf16_f32(GM, BN);
      int it = 0, tcount = 0;
      for (int u = blockIdx.x; u < total; u += gridDim.x, ++tcount) {
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
      wait_drain(mma_done, 0, kSpinLimitCycles);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int tcount = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++tcount) {
      const Work w = decode<BN>(u, s_prefix, s_off, E, NT, KB, a_local);
      const int acc = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&tfull[acc], aph, abort_flag, status, spin_limit);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      // rows of this warp's 32-row block that belong to the tile's expert
      const int nrows = min(32, max(0, w.rows - q * 32));
      epilogue_block<BN, SWIGLU>(taddr, w.a_row0 + q * 32, w.nt, nrows,
                                 s_epi + q * 32 * C::EPI_LD, lane, out, out_ld);
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

// --------------------------------------------------------------------------
// Pair variant: two CTAs of a cluster run one tcgen05 MMA of M = 256 rows
// (cta_group::2).  Each CTA holds its own 128 rows of A and one half of the B
// tile, so per SM each MMA reads half of the B bytes the single-CTA form reads
// from shared memory, and TMA writes half as many B bytes there.
//   both CTAs, warp 0 lane 0   TMA producer: its 128 A rows and its BN/2 B rows
//                              per stage; completion counted on the even CTA's
//                              `full` barrier (the only full barriers in use).
//   even CTA, warp 1 lane 0    MMA issuer (M=256, N=BN, K=16); commits free the
//                              stage and signal the accumulator in both CTAs.
//   both CTAs, warps 2..5      epilogue of their own 128 rows (their own TMEM);
//                              one arrival per warp on the even CTA's `tempty`.
// Tiles: for each expert e, ceil(M_e/256) row tiles x (N/BN) column tiles; the odd
// CTA's rows past the expert's end are computed but never stored.  The K order and
// tile shape depend only on H and I.
template <int BN>
struct PairCfg {
  static constexpr int STAGES = (BN == 256) ? 6 : 8;
  static constexpr int A_BYTES = GM * GK * 2;         // this CTA's 128 rows
  static constexpr int B_BYTES = (BN / 2) * GK * 2;   // this CTA's half of the B tile
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int NBAR = 2 * STAGES + 2 + 2 + 1;
  static constexpr int EPI_LD = 36;
  static constexpr int EPI_BYTES = 4 * 32 * EPI_LD * 4;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + NBAR * 8 + 16 +
                                    3 * (kMaxE + 1) * 4;
};

struct PairWork {
  int nt;          // column tile
  int a_row0;      // first output row of this CTA's 128 rows
  int rows;        // of those, rows that belong to the expert
  int a_load_row;  // first A row this CTA loads
  int b_load_row;  // first B row this CTA loads (its half of the column tile)
};

template <int BN>
__device__ __forceinline__ PairWork decode_pair(int u, int rank, const int* s_prefix,
                                                const int* s_off, int E, int NT, int KB,
                                                int a_local) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  const int local = u - s_prefix[lo];
  const int mt = local / NT;
  PairWork w;
  w.nt = local - mt * NT;
  w.a_row0 = s_off[lo] + mt * (2 * GM) + rank * GM;
  w.rows = min(GM, max(0, s_off[lo + 1] - w.a_row0));
  w.a_load_row = w.a_row0 - (a_local ? s_off[lo] : 0);
  w.b_load_row = (lo * NT + w.nt) * KB * BN + rank * (BN / 2);  // k-block kb adds kb * BN
  return w;
}

template <int BN, bool SWIGLU>
__global__ void __launch_bounds__(192, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ Maps maps, const int32_t* __restrict__ offsets,
                             int E, int R, int n_per_expert, int K, void* __restrict__ out,
                             int out_ld, int32_t* status, long long spin_limit, int a_local) {
  using C = PairCfg<BN>;
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
  const int rank = (int)cluster_ctarank();
  const int unit0 = blockIdx.x / 2, unit_step = gridDim.x / 2;

  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = __ldg(offsets + e);
  __syncthreads();
  if (threadIdx.x == 0) {
    // schedule: validate offsets (0 = o_0 <= o_1 <= ... <= o_E = R), work prefix
    bool ok = s_off[0] == 0 && s_off[E] == R;
    int p = 0;
    for (int e = 0; e < E; ++e) {
      const int a = s_off[e], b = s_off[e + 1];
      if (b < a) ok = false;
      s_prefix[e] = p;
      p += (b > a ? (b - a + 2 * GM - 1) / (2 * GM) : 0) * NT;
    }
    if (!ok) {
      flag_error(status, MOE_ERR_DEVICE_CHECK);
      for (int e = 0; e < E; ++e) s_prefix[e] = 0;
      p = 0;
    }
    s_prefix[E] = p;
    *abort_flag = 0;
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);   // the even CTA's producer; bytes from both CTAs
      mbar_init(&empty[s], 1);  // the pair MMA's commit, multicast
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);   // the pair MMA's commit, multicast
      mbar_init(&tempty[a], 8);  // four epilogue warps of each CTA
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&maps.a128);
    prefetch_tensormap(&maps.b_tile);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers and tensor memory exist before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = s_prefix[E];

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int it = 0;
      bool aborted = false;
      for (int u = unit0; u < total && !aborted; u += unit_step) {
        const PairWork w = decode_pair<BN>(u, rank, s_prefix, s_off, E, NT, KB, a_local);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, status, spin_limit)) {
            aborted = true;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * C::STAGE_BYTES);
          const uint32_t bar = mapa_shared(smem_u32(&full[s]), 0);
          tma_load_2d_pair(&maps.a128, sA + s * C::A_BYTES, bar, kb * GK, w.a_load_row);
          tma_load_2d_pair(&maps.b_tile, sB + s * C::B_BYTES, bar, 0, w.b_load_row + kb * BN);
        }
      }
      if (aborted && rank == 0) {
        // copies into the last STAGES slots (both CTAs' bytes count here) may be in flight
        for (int i = (it > C::STAGES ? it - C::STAGES : 0); i < it; ++i)
          wait_drain(&full[i % C::STAGES], (i / C::STAGES) & 1, kSpinLimitCycles);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t IDESC = idesc_bf16_f32(2 * GM, BN);
      int it = 0, tcount = 0;
      for (int u = unit0; u < total; u += unit_step, ++tcount) {
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
            mma_bf16_pair(d_tmem, sdesc_k_major_sw128(a_addr + kk * UK * 2),
                          sdesc_k_major_sw128(b_addr + kk * UK * 2), IDESC,
                          (kb > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_pair(&empty[s], 0x3);
        }
        if (aborted) break;
        mma_commit_pair(&tfull[acc], 0x3);
      }
      // every MMA this thread issued completes before tensor memory is released
      mma_commit_pair(mma_done, 0x1);
      wait_drain(mma_done, 0, kSpinLimitCycles);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int tcount = 0;
    for (int u = unit0; u < total; u += unit_step, ++tcount) {
      const PairWork w = decode_pair<BN>(u, rank, s_prefix, s_off, E, NT, KB, a_local);
      const int acc = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&tfull[acc], aph, abort_flag, status, spin_limit);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      const int nrows = min(32, max(0, w.rows - q * 32));
      epilogue_block<BN, SWIGLU>(taddr, w.a_row0 + q * 32, w.nt, nrows,
                                 s_epi + q * 32 * C::EPI_LD, lane, out, out_ld);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&tempty[acc]), 0));
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves or frees tensor memory while the pair may still use it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

// Per device and kernel: the shared-memory opt-in and the grid (one CTA per SM).
template <int BN, bool SWIGLU>
cudaError_t kernel_grid(int* grid) {
  using C = Cfg<BN>;
  static int cache[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && cache[dev] > 0) {
    *grid = cache[dev];
    return cudaSuccess;
  }
  err = cudaFuncSetAttribute(grouped_gemm_kernel<BN, SWIGLU>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  const int g = device_sm_count();
  if (dev < 64) cache[dev] = g;
  *grid = g;
  return cudaSuccess;
}

template <int BN, bool SWIGLU>
cudaError_t launch_grouped(const Maps& maps, const int32_t* offsets, int E, int R,
                           int n_per_expert, int K, void* out, int out_ld, int32_t* status,
                           long long spin_limit, cudaStream_t s, int a_local) {
  using C = Cfg<BN>;
  int grid = 0;
  cudaError_t err = kernel_grid<BN, SWIGLU>(&grid);
  if (err != cudaSuccess) return err;
  grouped_gemm_kernel<BN, SWIGLU><<<grid, 192, C::SMEM_BYTES, s>>>(
      maps, offsets, E, R, n_per_expert, K, out, out_ld, status, spin_limit, a_local);
  return cudaGetLastError();
}

// Grid of the pair kernel: twice the number of co-resident two-CTA clusters.
template <int BN, bool SWIGLU>
cudaError_t pair_grid(int* grid) {
  using C = PairCfg<BN>;
  static int cache[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && cache[dev] > 0) {
    *grid = cache[dev];
    return cudaSuccess;
  }
  auto kern = grouped_gemm_pair_kernel<BN, SWIGLU>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * device_sm_count(), 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
  if (err != cudaSuccess) return err;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  if (dev < 64) cache[dev] = 2 * clusters;
  *grid = 2 * clusters;
  return cudaSuccess;
}

template <int BN, bool SWIGLU>
cudaError_t launch_pair(const Maps& maps, const int32_t* offsets, int E, int R, int n_per_expert,
                        int K, void* out, int out_ld, int32_t* status, long long spin_limit,
                        cudaStream_t s, int a_local) {
  using C = PairCfg<BN>;
  int grid = 0;
  cudaError_t err = pair_grid<BN, SWIGLU>(&grid);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<BN, SWIGLU>, maps, offsets, E, R,
                            n_per_expert, K, out, out_ld, status, spin_limit, a_local);
}

}  // namespace

// The pair kernel and the single-CTA kernel give the same bits for every row (the
// same MMA shape per row, K order and epilogue), so the choice may depend on the
// number of rows without breaking batch invariance.  The pair form halves each
// SM's B traffic from L2 and shared memory; it pays when experts hold many rows
// (few half-empty 256-row tiles) and K is not short (both CTAs' epilogues gate
// every accumulator).
bool use_pair_gemm(int E, int R, int K) { return K >= 768 && (long long)R >= 512LL * E; }

int gemm_down_bn(int H) { return (H % 256 == 0) ? 256 : 128; }

cudaError_t launch_gemm_gate_up(const GemmOperand& a, const GemmOperand& b, const int32_t* offsets,
                                int E, int R, int H, int I, void* h, int32_t* status,
                                long long spin_limit, cudaStream_t s, bool a_local) {
  if (R == 0) return cudaSuccess;
  const bool pair = use_pair_gemm(E, R, H);
  Maps m;
  if (!a.encode(&m.a128, 128) || !b.encode(&m.b_tile, pair ? 128 : 256))
    return cudaErrorInvalidValue;
  if (pair)
    return launch_pair<256, true>(m, offsets, E, R, 2 * I, H, h, I, status, spin_limit, s,
                                  a_local ? 1 : 0);
  return launch_grouped<256, true>(m, offsets, E, R, 2 * I, H, h, I, status, spin_limit, s,
                                   a_local ? 1 : 0);
}

cudaError_t launch_gemm_down(const GemmOperand& a, const GemmOperand& b, const int32_t* offsets,
                             int E, int R, int H, int I, float* y, int32_t* status,
                             long long spin_limit, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const int bn = gemm_down_bn(H);
  const bool pair = use_pair_gemm(E, R, I);
  Maps m;
  if (!a.encode(&m.a128, 128) || !b.encode(&m.b_tile, pair ? bn / 2 : bn))
    return cudaErrorInvalidValue;
  if (pair) {
    if (bn == 256)
      return launch_pair<256, false>(m, offsets, E, R, H, I, y, H, status, spin_limit, s, 0);
    return launch_pair<128, false>(m, offsets, E, R, H, I, y, H, status, spin_limit, s, 0);
  }
  if (bn == 256)
    return launch_grouped<256, false>(m, offsets, E, R, H, I, y, H, status, spin_limit, s, 0);
  return launch_grouped<128, false>(m, offsets, E, R, H, I, y, H, status, spin_limit, s, 0);
}

}  // namespace moe
