// One-time expert-weight preparation: logical row-major weights -> the K-major
// boxes the grouped GEMMs stream with TMA.
//
//   W1 (gate/up): output column tiles of 256 rows; in tile n, rows 0..127 are gate
//                 columns 128n..128n+127 and rows 128..255 the matching up columns,
//                 each a row over h (K-major).  One MMA tile then holds a gate block
//                 and its up block, so SwiGLU runs in the epilogue.
//   W2 (down):    output column tiles of BN2 = 256 rows (128 when H % 256 != 0), row
//                 c = down-projection column c over i (K-major).
//
// Both are stored box by box: for expert e, column tile n and k-block b (64 K
// values), the BN x 64 box is contiguous (BN rows of 128 bytes), boxes ordered
// (e, n, b).  A TMA box of the GEMM is then one sequential read of 16-32 KB instead
// of 128 bytes from each of BN rows a K-row apart.
//
// 32x32 tiles through shared memory; reads and writes are both coalesced.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

// src: per expert a [rows x cols] matrix with row stride `ld`, expert e starting
// `estride` elements after expert e - 1.  Source row r is K index r; source column
// c becomes output row map(c) of the expert's column tiles.
// mode 0: gate half of W1, mode 1: up half of W1, mode 2: W2 (tiles of bn2 rows).
// slot_of_expert (optional): expert e is written to physical slot slot_of_expert[e]
// (RoutePack's materialisation of a placement: each expert's weights move into the
// tensors of its destination slot).
__global__ void __launch_bounds__(256) transpose_pack_kernel(const uint16_t* __restrict__ src,
                                                             int rows, int cols, size_t ld,
                                                             size_t estride, int mode, int I,
                                                             int H, int bn2,
                                                             uint16_t* __restrict__ dst,
                                                             const int32_t* __restrict__ slot_of_expert) {
  __shared__ uint16_t tile[32][33];
  const int e = blockIdx.z;
  const int de = slot_of_expert != nullptr ? __ldg(slot_of_expert + e) : e;
  if (de < 0 || de >= (int)gridDim.z) return;  // a slot outside [0, E) is not written
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const uint16_t* s = src + (size_t)e * estride;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[i][threadIdx.x] = s[(size_t)r * ld + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i;          // source column -> destination row
    const int r = r0 + threadIdx.x;  // source row -> destination column
    if (r >= rows || c >= cols) continue;
    // (column tile, row in tile), K extent of the expert
    int tn, tr, bn, K, ntiles;
    if (mode < 2) {
      tn = c / 128;
      tr = (c % 128) + (mode == 1 ? 128 : 0);
      bn = 256;
      K = H;
      ntiles = (2 * I) / 256;
    } else {
      tn = c / bn2;
      tr = c % bn2;
      bn = bn2;
      K = I;
      ntiles = H / bn2;
    }
    const size_t box = ((size_t)de * ntiles + tn) * (K / 64) + (r / 64);
    dst[(box * bn + tr) * 64 + (r % 64)] = tile[threadIdx.x][i];
  }
}

}  // namespace

cudaError_t launch_prepack(const void* w_gate, const void* w_up, const void* w_down, int E, int H,
                           int I, void* packed, cudaStream_t s, const int32_t* slot_of_expert) {
  uint16_t* w1 = static_cast<uint16_t*>(packed);
  uint16_t* w2 = w1 + (size_t)E * 2 * I * H;
  dim3 block(32, 8);
  dim3 g1((I + 31) / 32, (H + 31) / 32, E);  // gate/up: [H x I] per expert
  const size_t e1 = (size_t)H * I, e2 = (size_t)I * H;
  const int bn2 = gemm_down_bn(H);
  transpose_pack_kernel<<<g1, block, 0, s>>>(static_cast<const uint16_t*>(w_gate), H, I, I, e1, 0,
                                             I, H, bn2, w1, slot_of_expert);
  transpose_pack_kernel<<<g1, block, 0, s>>>(static_cast<const uint16_t*>(w_up), H, I, I, e1, 1, I,
                                             H, bn2, w1, slot_of_expert);
  dim3 g2((H + 31) / 32, (I + 31) / 32, E);  // down: [I x H] per expert
  transpose_pack_kernel<<<g2, block, 0, s>>>(static_cast<const uint16_t*>(w_down), I, H, H, e2, 2,
                                             I, H, bn2, w2, slot_of_expert);
  return cudaGetLastError();
}

cudaError_t launch_prepack_shared(const void* w_gate, const void* w_up, const void* w_down, int H,
                                  int Is, int G, void* packed, cudaStream_t s) {
  const int Ig = Is / G;
  uint16_t* w1 = static_cast<uint16_t*>(packed);
  uint16_t* w2 = w1 + (size_t)G * 2 * Ig * H;
  dim3 block(32, 8);
  dim3 g1((Ig + 31) / 32, (H + 31) / 32, G);  // shard g: columns [g*Ig, (g+1)*Ig) of [H x Is]
  const int bn2 = gemm_down_bn(H);
  transpose_pack_kernel<<<g1, block, 0, s>>>(static_cast<const uint16_t*>(w_gate), H, Ig, Is, Ig,
                                             0, Ig, H, bn2, w1, nullptr);
  transpose_pack_kernel<<<g1, block, 0, s>>>(static_cast<const uint16_t*>(w_up), H, Ig, Is, Ig, 1,
                                             Ig, H, bn2, w1, nullptr);
  dim3 g2((H + 31) / 32, (Ig + 31) / 32, G);  // shard g: rows [g*Ig, (g+1)*Ig) of [Is x H]
  transpose_pack_kernel<<<g2, block, 0, s>>>(static_cast<const uint16_t*>(w_down), Ig, H, H,
                                             (size_t)Ig * H, 2, Ig, H, bn2, w2, nullptr);
  return cudaGetLastError();
}

}  // namespace moe
