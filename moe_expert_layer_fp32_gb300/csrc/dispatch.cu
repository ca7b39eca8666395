// Load statistics and dispatch: per-expert counts, exclusive offsets, and the
// stable permutation of token rows into expert-contiguous rows.
//
// "RoutePack", section 2.2 "Routing replay" (Eq. 1): the load of expert e is the
// number of token->expert assignments.  Section 2.3: a rank's local experts run
// as one grouped operation, which needs each expert's rows contiguous.
// "FlexFloor", Figure 1: token -> dispatch -> experts -> combine.
//
// Determinism without float atomics or sorting.  Tokens are cut into blocks of
// 256 (8 warps x 32 lanes, one token per lane).  For each warp and expert a
// 32-bit mask of the lanes whose token chose that expert is built with integer
// atomicOr (order-free).  A token's stable rank inside its block is then
//   popc(mask[w][e] & lanes_below) + sum_{w' < w} popc(mask[w'][e]),
// the block's count of e is sum_w popc(mask[w][e]), and one scan kernel turns
// per-block counts into per-(block, expert) first rows.  Every quantity is an
// integer function of topk_idx alone: bit-identical on every run and for every T.
#include "common.cuh"
#include "kernels.cuh"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int PB = kPermBlock;  // 256 tokens, 8 warps

// Builds masks[w][e] for the block's tokens; returns nothing but fills smem.
// sidx holds the block's topk_idx rows.  Invalid ids and repeated experts within
// one token are flagged and left out.
// With `remap` (RoutePack's dispatcher map, logical expert -> physical slot),
// sidx holds physical slots; out-of-range slots are flagged like bad ids.
__device__ __forceinline__ void build_masks(const int32_t* __restrict__ topk_idx, int T, int k,
                                            int E, int t0, uint32_t* masks, int32_t* sidx,
                                            int32_t* status,
                                            const int32_t* __restrict__ remap = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ntok = min(PB, T - t0);
  const int n = ntok * k;
  const int32_t* src = topk_idx + (size_t)t0 * k;
  for (int i = tid; i < n; i += blockDim.x) {
    int e = __ldg(src + i);
    if (remap != nullptr && e >= 0 && e < E) e = __ldg(remap + e);
    sidx[i] = e;
  }
  for (int i = tid; i < 8 * E; i += blockDim.x) masks[i] = 0u;
  __syncthreads();
  const int tl = warp * 32 + lane;
  if (tl < ntok) {
    for (int j = 0; j < k; ++j) {
      const int e = sidx[tl * k + j];
      if (e < 0 || e >= E) {
        flag_error(status, MOE_ERR_DEVICE_CHECK);
        continue;
      }
      const uint32_t old = atomicOr(&masks[warp * E + e], 1u << lane);
      if (old & (1u << lane)) flag_error(status, MOE_ERR_DEVICE_CHECK);  // expert repeated
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(PB) block_counts_kernel(const int32_t* __restrict__ topk_idx,
                                                          int T, int k, int E,
                                                          int32_t* __restrict__ blk_counts,
                                                          int32_t* status,
                                                          const int32_t* __restrict__ remap) {
  extern __shared__ uint32_t smem_u[];
  uint32_t* masks = smem_u;                               // [8][E]
  int32_t* sidx = reinterpret_cast<int32_t*>(smem_u + 8 * E);  // [PB*k]
  const int b = blockIdx.x;
  build_masks(topk_idx, T, k, E, b * PB, masks, sidx, status, remap);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) c += __popc(masks[w * E + e]);
    blk_counts[(size_t)b * E + e] = c;
  }
}

// One CTA, one thread per expert: running sums over blocks, then an exclusive
// scan over experts for the offsets.
__global__ void __launch_bounds__(kMaxE) scan_kernel(const int32_t* __restrict__ blk_counts, int nb,
                                                     int E, int R, int32_t* __restrict__ counts,
                                                     int32_t* __restrict__ offsets,
                                                     int offsets_given,
                                                     int32_t* __restrict__ blk_base,
                                                     int32_t* status) {
  __shared__ int s_scan[kMaxE];
  __shared__ int s_bad;
  const int e = threadIdx.x;
  if (e == 0) s_bad = 0;
  int running = 0;
  if (e < E) {
    for (int b = 0; b < nb; ++b) {
      const int c = blk_counts[(size_t)b * E + e];
      blk_base[(size_t)b * E + e] = running;
      running += c;
    }
  }
  // inclusive Hillis-Steele scan over the (padded) expert axis
  s_scan[e] = (e < E) ? running : 0;
  __syncthreads();
  for (int off = 1; off < kMaxE; off <<= 1) {
    const int v = (e >= off) ? s_scan[e - off] : 0;
    __syncthreads();
    s_scan[e] += v;
    __syncthreads();
  }
  const int excl = s_scan[e] - ((e < E) ? running : 0);
  const int total = s_scan[kMaxE - 1];
  int base = excl;
  if (offsets_given) {
    if (e < E) {
      const int a = offsets[e], bnext = offsets[e + 1];
      if (a != excl || bnext - a != running) atomicOr(&s_bad, 1);
    }
    if (e == 0 && (offsets[0] != 0 || offsets[E] != R)) atomicOr(&s_bad, 1);
  } else {
    if (e < E) offsets[e] = excl;
    if (e == 0) offsets[E] = total;
  }
  if (e == 0 && total != R) atomicOr(&s_bad, 1);
  if (counts != nullptr && e < E) counts[e] = running;
  __syncthreads();
  if (e == 0 && s_bad) flag_error(status, MOE_ERR_DEVICE_CHECK);
  if (e < E) {
    for (int b = 0; b < nb; ++b) blk_base[(size_t)b * E + e] += base;
  }
}

__global__ void __launch_bounds__(PB) rank_kernel(const int32_t* __restrict__ topk_idx, int T,
                                                  int k, int E,
                                                  const int32_t* __restrict__ blk_base,
                                                  int32_t* __restrict__ row_of_slot,
                                                  int32_t* __restrict__ slot_of_row,
                                                  int32_t* status,
                                                  const int32_t* __restrict__ remap) {
  extern __shared__ uint32_t smem_u[];
  uint32_t* masks = smem_u;
  int32_t* sidx = reinterpret_cast<int32_t*>(smem_u + 8 * E);
  const int b = blockIdx.x, t0 = b * PB;
  build_masks(topk_idx, T, k, E, t0, masks, sidx, status, remap);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tl = warp * 32 + lane;
  const int t = t0 + tl;
  if (t >= T) return;
  const long long R = (long long)T * k;
  const uint32_t below = (1u << lane) - 1u;
  for (int j = 0; j < k; ++j) {
    const int e = sidx[tl * k + j];
    const size_t s = (size_t)t * k + j;
    if (e < 0 || e >= E) {
      row_of_slot[s] = -1;
      continue;
    }
    int rank = __popc(masks[warp * E + e] & below);
    for (int w = 0; w < warp; ++w) rank += __popc(masks[w * E + e]);
    const long long row = (long long)blk_base[(size_t)b * E + e] + rank;
    if (row < 0 || row >= R) {
      flag_error(status, MOE_ERR_DEVICE_CHECK);
      row_of_slot[s] = -1;
      continue;
    }
    row_of_slot[s] = (int32_t)row;
    slot_of_row[row] = (int32_t)s;
  }
}

// T <= 256 (a single ranking block): masks, counts, offsets, stable ranks and the
// row copy in one launch, the work of block_counts + scan + rank + copy_rows.
// CTA (b, c) ranks all T tokens (at most 256 x k ids, from L2) and then copies
// column slice c (of gridDim.y) of tokens 8b..8b+7, one warp per token; the CTAs
// of slice 0 write the rows, CTA (0, 0) counts and offsets.
// LATE: no row copy; the indices are computed first and the kernel waits for its
// predecessor only at the end (so its completion implies the predecessor's).
template <bool LATE>
__global__ void __launch_bounds__(PB) dispatch_small_kernel(const int32_t* __restrict__ topk_idx,
                                                            int T, int k, int E,
                                                            const uint16_t* __restrict__ x, int H,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ row_of_slot,
                                                            int32_t* __restrict__ slot_of_row,
                                                            uint16_t* __restrict__ x_perm,
                                                            int32_t* status) {
  extern __shared__ uint32_t smem_u[];
  uint32_t* masks = smem_u;
  int32_t* sidx = reinterpret_cast<int32_t*>(smem_u + 8 * E);
  __shared__ int s_scan[kMaxE];
  __shared__ int s_wsum[PB / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = blockIdx.x * 8 + warp;  // this warp's token (copy phase)
  const bool lead = blockIdx.y == 0;
  // The token's source row does not depend on the routing: the first 32 x U
  // 16-byte vectors of this CTA's slice are loaded now, and land while it ranks.
  constexpr int U = 8;
  const int nvs = H / 8 / gridDim.y;  // 16-byte vectors of the slice
  const int cb = blockIdx.y * nvs;    // its first vector
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(t < T ? t : 0) * H) + cb;
  uint4 v0[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int cc = u * 32 + lane;
    if (!LATE && t < T && cc < nvs) v0[u] = __ldg(src + cc);
  }
  // a programmatic dependent of the router: the routing is read, and every
  // output written, after it has finished (x was final before the router began)
  if constexpr (!LATE) {
    pdl_wait();
    if (tid == 0) pdl_launch_dependents();
  }
  // every CTA ranks the whole (single) block; each then copies its own 8 tokens
  build_masks(topk_idx, T, k, E, 0, masks, sidx, blockIdx.x == 0 && lead ? status : nullptr);
  int c = 0;
  if (tid < E) {
#pragma unroll
    for (int w = 0; w < 8; ++w) c += __popc(masks[w * E + tid]);
  }
  // exclusive scan over the experts (blockDim == kMaxE): within each warp by
  // shuffles, then over the eight warp totals
  int incl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += n;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  int total = 0;
#pragma unroll
  for (int w = 0; w < PB / 32; ++w) {
    const int sw = s_wsum[w];
    if (w < warp) incl += sw;
    total += sw;
  }
  const int excl = incl - c;
  if (blockIdx.x == 0 && lead) {
    if (tid < E) {
      counts[tid] = c;
      offsets[tid] = excl;
    }
    if (tid == 0) offsets[E] = total;
  }
  s_scan[tid] = excl;  // first row of each expert
  __syncthreads();
  if (t >= T) return;
  const long long R = (long long)T * k;
  // lane j < k ranks slot (t, j): the token sits in mask word t / 32, bit t % 32
  int my_row = -1;
  if (lane < k) {
    const int e = sidx[t * k + lane];
    const size_t sl = (size_t)t * k + lane;
    if (e >= 0 && e < E) {
      const int tw = t >> 5;
      int rank = __popc(masks[tw * E + e] & ((1u << (t & 31)) - 1u));
      for (int w = 0; w < tw; ++w) rank += __popc(masks[w * E + e]);
      const long long row = (long long)s_scan[e] + rank;
      if (row >= 0 && row < R) my_row = (int)row;
      else if (lead) flag_error(status, MOE_ERR_DEVICE_CHECK);
    }
    if (lead) {
      row_of_slot[sl] = my_row;
      if (my_row >= 0) slot_of_row[my_row] = (int32_t)sl;
    }
  }
  if constexpr (LATE) {
    pdl_wait();
    if (tid == 0) pdl_launch_dependents();
  } else {
    for (int c0 = 0; c0 < nvs; c0 += 32 * U) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int cc = c0 + u * 32 + lane;
        if (c0 == 0) v[u] = v0[u];
        else if (cc < nvs) v[u] = __ldg(src + cc);
      }
      for (int j = 0; j < k; ++j) {
        const int r = __shfl_sync(0xFFFFFFFFu, my_row, j);
        if (r < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)r * H) + cb;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int cc = c0 + u * 32 + lane;
          if (cc < nvs) dst[cc] = v[u];
        }
      }
    }
  }
}

// "HARTS", Eq. 20: compact row t counts q[t] times in the expert loads.  Integer
// additions only (order-free): shared-memory partial sums per block, then one
// global atomic per expert and block.  out (int64 [E]) must start at zero.
__global__ void __launch_bounds__(PB) weighted_counts_kernel(const int32_t* __restrict__ topk_idx,
                                                             const int32_t* __restrict__ q, int T,
                                                             int k, int E,
                                                             unsigned long long* __restrict__ out,
                                                             int32_t* status) {
  __shared__ unsigned long long acc[kMaxE];
  for (int e = threadIdx.x; e < E; e += blockDim.x) acc[e] = 0ull;
  __syncthreads();
  const int t = blockIdx.x * PB + threadIdx.x;
  if (t < T) {
    const int qt = __ldg(q + t);
    if (qt < 0) flag_error(status, MOE_ERR_DEVICE_CHECK);
    for (int j = 0; j < k; ++j) {
      const int e = __ldg(topk_idx + (size_t)t * k + j);
      if (e < 0 || e >= E || qt < 0) {
        flag_error(status, MOE_ERR_DEVICE_CHECK);
        continue;
      }
      atomicAdd(&acc[e], (unsigned long long)qt);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (acc[e] != 0ull) atomicAdd(out + e, acc[e]);
}

// One warp per token: read the row once (16-byte vectors), write it to its k rows.
__global__ void __launch_bounds__(256) copy_rows_kernel(const uint16_t* __restrict__ x,
                                                        const int32_t* __restrict__ row_of_slot,
                                                        int T, int H, int k,
                                                        uint16_t* __restrict__ x_perm,
                                                        int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const long long R = (long long)T * k;
  int my_row = -1;
  if (lane < k) {
    const int r = row_of_slot[(size_t)t * k + lane];
    if (r >= 0 && r < R) my_row = r;
    else flag_error(status, MOE_ERR_DEVICE_CHECK);
  }
  const int nv = H / 8;  // 16-byte vectors per row
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  constexpr int U = 8;
  for (int c0 = 0; c0 < nv; c0 += 32 * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * 32 + lane;
      if (c < nv) v[u] = __ldg(src + c);
    }
    for (int j = 0; j < k; ++j) {
      const int r = __shfl_sync(0xFFFFFFFFu, my_row, j);
      if (r < 0) continue;
      uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)r * H);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < nv) dst[c] = v[u];
      }
    }
  }
}

size_t mask_smem_bytes(int E, int k) { return (size_t)8 * E * 4 + (size_t)PB * k * 4; }

}  // namespace

cudaError_t launch_block_counts(const int32_t* topk_idx, int T, int k, int E, int32_t* blk_counts,
                                int32_t* status, cudaStream_t s, const int32_t* remap) {
  if (T == 0) return cudaSuccess;
  const int nb = (T + PB - 1) / PB;
  block_counts_kernel<<<nb, PB, mask_smem_bytes(E, k), s>>>(topk_idx, T, k, E, blk_counts, status,
                                                           remap);
  return cudaGetLastError();
}

cudaError_t launch_scan(const int32_t* blk_counts, int nb, int E, int R, int32_t* counts,
                        int32_t* offsets, bool offsets_given, int32_t* blk_base, int32_t* status,
                        cudaStream_t s) {
  scan_kernel<<<1, kMaxE, 0, s>>>(blk_counts, nb, E, R, counts, offsets, offsets_given ? 1 : 0,
                                  blk_base, status);
  return cudaGetLastError();
}

cudaError_t launch_rank(const int32_t* topk_idx, int T, int k, int E, const int32_t* blk_base,
                        int32_t* row_of_slot, int32_t* slot_of_row, int32_t* status,
                        cudaStream_t s, const int32_t* remap) {
  if (T == 0) return cudaSuccess;
  const int nb = (T + PB - 1) / PB;
  rank_kernel<<<nb, PB, mask_smem_bytes(E, k), s>>>(topk_idx, T, k, E, blk_base, row_of_slot,
                                                    slot_of_row, status, remap);
  return cudaGetLastError();
}

cudaError_t launch_weighted_counts(const int32_t* topk_idx, const int32_t* q, int T, int k, int E,
                                   int64_t* out, int32_t* status, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(out, 0, (size_t)E * sizeof(int64_t), s);
  if (err != cudaSuccess || T == 0) return err;
  weighted_counts_kernel<<<(T + PB - 1) / PB, PB, 0, s>>>(
      topk_idx, q, T, k, E, reinterpret_cast<unsigned long long*>(out), status);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_small(const int32_t* topk_idx, int T, int k, int E, const void* x,
                                  int H, int32_t* counts, int32_t* offsets, int32_t* row_of_slot,
                                  int32_t* slot_of_row, void* x_perm, int32_t* status,
                                  cudaStream_t s) {
  const int nb = T > 0 ? (T + 7) / 8 : 1;
  if (x_perm == nullptr)
    return launch_pdl(dispatch_small_kernel<true>, dim3(nb, 1), dim3(PB), mask_smem_bytes(E, k),
                      s, topk_idx, T, k, E, static_cast<const uint16_t*>(x), H, counts, offsets,
                      row_of_slot, slot_of_row, static_cast<uint16_t*>(x_perm), status);
  // column slices of at least 32 vectors (one per lane) while the grid stays
  // within two CTAs per SM
  int split = 1;
  const int nv = H / 8;
  while (split < 16 && nv % (2 * split) == 0 && nv / (2 * split) >= 32 &&
         (long long)nb * 2 * split <= 2LL * device_sm_count())
    split *= 2;
  return launch_pdl(dispatch_small_kernel<false>, dim3(nb, split), dim3(PB),
                    mask_smem_bytes(E, k), s, topk_idx, T, k, E, static_cast<const uint16_t*>(x),
                    H, counts, offsets, row_of_slot, slot_of_row, static_cast<uint16_t*>(x_perm),
                    status);
}

namespace {
__global__ void uniform_offsets_kernel(int32_t* offsets, int G, int T) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g <= G) offsets[g] = g * T;
}
}  // namespace

cudaError_t launch_uniform_offsets(int32_t* offsets, int G, int T, cudaStream_t s) {
  uniform_offsets_kernel<<<(G + 1 + 255) / 256, 256, 0, s>>>(offsets, G, T);
  return cudaGetLastError();
}

cudaError_t launch_copy_rows(const void* x, const int32_t* row_of_slot, int T, int H, int k,
                             void* x_perm, int32_t* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  copy_rows_kernel<<<(T + 7) / 8, 256, 0, s>>>(static_cast<const uint16_t*>(x), row_of_slot, T, H,
                                              k, static_cast<uint16_t*>(x_perm), status);
  return cudaGetLastError();
}

}  // namespace moe
