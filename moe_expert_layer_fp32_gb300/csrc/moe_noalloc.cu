// moe_load_stats_noalloc: the per-expert load statistics for callers that cannot
// allocate device memory.
//
// Some callers of this library cannot call cudaMalloc or take memory from an
// allocator at the point where they need the expert counts: code running inside
// a host framework whose device memory is owned entirely by its own pool, or a
// latency-critical serving loop that must not allocate after start-up (a
// cudaMalloc can synchronise the device).  moe_load_stats needs a workspace for
// its per-block partial counts; this variant keeps that scratch in a fixed array
// compiled into the library instead, so the caller passes only the inputs and
// outputs.
//
// The scratch is the file-scope array below (2 MiB per GPU that loads the
// library, held until the process exits).  Host code cannot use the array's
// name as a device address: it is looked up once per device with
// cudaGetSymbolAddress and that address is what the kernels receive.  The cached
// address belongs to the device's current context: after cudaDeviceReset on a
// device, this entry point must not be called on that device again in the same
// process.
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

// Two int32 tables of nb*E entries each (per-block counts, per-block first rows),
// nb = ceil(T / 256).
constexpr size_t kNoAllocScratchInts = 524288;  // 2 MiB
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per
// device).  Returns nullptr on failure.
int32_t* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_load_stats_noalloc(const int32_t* topk_idx, moe_dims d, int32_t* counts,
                                             int32_t* offsets, int32_t* device_status,
                                             void* stream) {
  // the checks of moe_load_stats: dims, pointers (16-byte aligned), sm_103 device
  moe_status st = validate_dims(d);
  if (st != MOE_OK) return st;
  const long long nb = ((long long)d.T + kPermBlock - 1) / kPermBlock;
  if (2 * nb * d.E > (long long)kNoAllocScratchInts) return MOE_ERR_UNSUPPORTED;
  if (d.T > 0 && (st = validate_ptr(topk_idx)) != MOE_OK) return st;
  if ((st = validate_ptr(counts)) != MOE_OK) return st;
  if ((st = validate_ptr(offsets)) != MOE_OK) return st;
  if (device_status != nullptr && (st = validate_ptr(device_status)) != MOE_OK) return st;
  if ((st = validate_device()) != MOE_OK) return st;
  int32_t* scratch = scratch_on_current_device();
  if (scratch == nullptr) return MOE_ERR_CUDA;
  int32_t* blk_counts = scratch;
  int32_t* blk_base = scratch + nb * d.E;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Every entry of the two tables that the scan reads is written first by this
  // call, so nothing left by an earlier call needs clearing.
  if (launch_block_counts(topk_idx, d.T, d.k, d.E, blk_counts, device_status, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_scan(blk_counts, (int)nb, d.E, d.T * d.k, counts, offsets, false, blk_base,
                  device_status, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
