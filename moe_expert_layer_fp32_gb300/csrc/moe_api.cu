// C ABI of the routed MoE layer forward (declared in include/moe.h): host-side
// argument validation, the workspace layout, TMA tensor maps, and the launch
// sequence route -> load stats -> permute -> grouped expert GEMMs -> combine.
// No call allocates device memory or synchronises the stream (except
// moe_read_device_status, whose job is to synchronise).
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {

int device_sm_count() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 1;
  if (dev < 64) cache[dev] = n;
  return n;
}

namespace {

// Limit of the GEMM kernels' bounded waits, in SM clock cycles (diagnostics knob).
std::atomic<long long> g_wait_limit{kSpinLimitCycles};

// ------------------------------------------------------------------ layout ---
constexpr size_t kAlign = 256;
inline size_t up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t status, idx, w, counts, offsets, blk_counts, blk_base, row_of_slot, slot_of_row, x_perm,
      h, y, total;
};

Layout layout(const moe_dims& d) {
  const size_t T = (size_t)d.T, R = (size_t)d.T * d.k, E = (size_t)d.E;
  const size_t nb = (T + kPermBlock - 1) / kPermBlock;
  Layout L;
  size_t o = 0;
  L.status = o;       o += up(kAlign);
  L.idx = o;          o += up(R * 4);
  L.w = o;            o += up(R * 4);
  L.counts = o;       o += up(E * 4);
  L.offsets = o;      o += up((E + 1) * 4);
  L.blk_counts = o;   o += up(nb * E * 4);
  L.blk_base = o;     o += up(nb * E * 4);
  L.row_of_slot = o;  o += up(R * 4);
  L.slot_of_row = o;  o += up(R * 4);
  L.x_perm = o;       o += up(R * (size_t)d.H * 2);
  L.h = o;            o += up(R * (size_t)d.I * 2);
  L.y = o;            o += up(R * (size_t)d.H * 4);
  L.total = o;
  return L;
}

// Workspace of the sharded shared expert: status word, group offsets, h [G*T, Is/G].
struct SharedLayout {
  size_t status, offsets, h, total;
};

SharedLayout shared_layout(int T, int G, int Is) {
  SharedLayout L;
  size_t o = 0;
  L.status = o;   o += up(kAlign);
  L.offsets = o;  o += up(((size_t)G + 1) * 4);
  L.h = o;        o += up((size_t)T * Is * 2);  // G * T rows of Is / G
  L.total = o;
  return L;
}

template <typename T>
inline T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// -------------------------------------------------------------- validation ---
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_dims(const moe_dims& d) {
  if (d.T < 0 || d.H <= 0 || d.E <= 0 || d.k <= 0 || d.I <= 0) return MOE_ERR_INVALID_ARG;
  if (d.k > d.E) return MOE_ERR_INVALID_ARG;
  if (d.E > kMaxE || d.k > kMaxK) return MOE_ERR_UNSUPPORTED;
  if (d.H % 128 != 0 || d.I % 128 != 0 || d.H > 16384 || d.I > 16384) return MOE_ERR_UNSUPPORTED;
  if ((long long)d.T * d.k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status check_shared(int T, int H, int Is, int G) {
  if (T < 0 || H <= 0 || Is <= 0 || G < 1) return MOE_ERR_INVALID_ARG;
  if (Is % G != 0) return MOE_ERR_INVALID_ARG;
  const int Ig = Is / G;
  if (H % 128 != 0 || Ig % 128 != 0 || H > 16384 || Ig > 16384 || G > kMaxE)
    return MOE_ERR_UNSUPPORTED;
  if ((long long)G * T >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status need(const void* p) {
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(p)) return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

moe_status check_ws(const moe_dims& d, const void* ws, size_t ws_bytes) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_MISALIGNED;
  if (ws_bytes < layout(d).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

#define MOE_TRY(expr)                 \
  do {                                \
    moe_status _s = (expr);           \
    if (_s != MOE_OK) return _s;      \
  } while (0)

#define MOE_CUDA(expr)                          \
  do {                                          \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

moe_status device_ok() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  static int cc_cache[64] = {};
  int cc = dev < 64 ? cc_cache[dev] : 0;
  if (cc == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    cc = major * 10 + minor;
    if (dev < 64) cc_cache[dev] = cc;
  }
  return cc == 103 ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

// ------------------------------------------------------------- tensor maps ---
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

moe_status validate_dims(const moe_dims& d) { return check_dims(d); }
moe_status validate_ptr(const void* p) { return need(p); }
moe_status validate_device() { return device_ok(); }

bool GemmOperand::encode(CUtensorMap* m, uint32_t box_rows) const {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_rowmajor_2d(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, bool fp32,
                        uint32_t box_cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr || rows == 0) return false;
  const uint64_t es = fp32 ? 4 : 2;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * es};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

// ------------------------------------------------------------ step bodies ---
moe_status do_load_stats(const int32_t* idx, const moe_dims& d, int32_t* counts,
                         int32_t* offsets, bool offsets_given, void* ws, cudaStream_t s,
                         const int32_t* remap = nullptr) {
  const Layout L = layout(d);
  const int nb = (d.T + kPermBlock - 1) / kPermBlock;
  int32_t* status = at<int32_t>(ws, L.status);
  MOE_CUDA(launch_block_counts(idx, d.T, d.k, d.E, at<int32_t>(ws, L.blk_counts), status, s,
                               remap));
  MOE_CUDA(launch_scan(at<int32_t>(ws, L.blk_counts), nb, d.E, d.T * d.k, counts, offsets,
                       offsets_given, at<int32_t>(ws, L.blk_base), status, s));
  return MOE_OK;
}

moe_status do_permute_rows(const void* x, const int32_t* idx, const moe_dims& d, void* x_perm,
                           int32_t* ros, int32_t* sor, void* ws, cudaStream_t s,
                           const int32_t* remap = nullptr) {
  const Layout L = layout(d);
  int32_t* status = at<int32_t>(ws, L.status);
  MOE_CUDA(launch_rank(idx, d.T, d.k, d.E, at<int32_t>(ws, L.blk_base), ros, sor, status, s,
                       remap));
  MOE_CUDA(launch_copy_rows(x, ros, d.T, d.H, d.k, x_perm, status, s));
  return MOE_OK;
}

// token_ids (one token, the swapped form): the GEMMs take their rows from the
// token's k expert ids and the gate/up GEMM reads the token row x_token itself, so
// neither x_perm nor offsets is read
moe_status do_expert_ffn(const void* x_perm, const int32_t* offsets, const void* packed,
                         const moe_dims& d, float* y, void* ws, cudaStream_t s,
                         cudaEvent_t after_gate_up = nullptr, const void* x_token = nullptr,
                         const int32_t* token_ids = nullptr) {
  const Layout L = layout(d);
  const int R = d.T * d.k;
  if (R == 0) return MOE_OK;
  int32_t* status = at<int32_t>(ws, L.status);
  void* h = at<void>(ws, L.h);
  const uint16_t* w1 = static_cast<const uint16_t*>(packed);
  const uint16_t* w2 = w1 + (size_t)d.E * 2 * d.I * d.H;
  const GemmOperand ma{token_ids != nullptr ? x_token : x_perm, (uint64_t)d.H,
                       (uint64_t)(token_ids != nullptr ? d.T : R)};
  // packed weights are box-tiled: 64 K values per row, (expert, column tile, k-block) boxes
  const GemmOperand mb{w1, 64, (uint64_t)d.E * 2 * d.I * (d.H / 64)};
  const GemmOperand mh{h, (uint64_t)d.I, (uint64_t)R};
  const GemmOperand md{w2, 64, (uint64_t)d.E * d.H * (d.I / 64)};
  // few rows per expert: weight rows on the MMA's M side (same bits as the tiles)
  const bool swap = use_swap_gemm(d.E, R, d.H, d.I);
  const long long lim = g_wait_limit.load();
  if (token_ids != nullptr && !(swap && d.T == 1)) return MOE_ERR_INVALID_ARG;
  if (swap)
    MOE_CUDA(launch_gemm_gate_up_swap(ma, mb, offsets, d.E, R, d.H, d.I, h, status, lim, s, false,
                                      token_ids));
  else
    MOE_CUDA(launch_gemm_gate_up(ma, mb, offsets, d.E, R, d.H, d.I, h, status, lim, s));
  if (after_gate_up != nullptr) MOE_CUDA(cudaEventRecord(after_gate_up, s));
  if (swap)
    MOE_CUDA(launch_gemm_down_swap(mh, md, offsets, d.E, R, d.H, d.I, y, status, lim, s,
                                   token_ids));
  else
    MOE_CUDA(launch_gemm_down(mh, md, offsets, d.E, R, d.H, d.I, y, status, lim, s));
  return MOE_OK;
}

// Shared expert split into G column shards: gate/up GEMM over the same token rows
// for every shard (a_local), then the down GEMM into shared_out [G, T, H] fp32.
// status: the device status word the GEMMs report into.
moe_status do_shared_expert(const void* x, const void* packed, int T, int H, int Is, int G,
                            float* shared_out, void* ws, int32_t* status, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const SharedLayout L = shared_layout(T, G, Is);
  const int Ig = Is / G, R = G * T;
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  void* h = at<void>(ws, L.h);
  const uint16_t* w1 = static_cast<const uint16_t*>(packed);
  const uint16_t* w2 = w1 + (size_t)G * 2 * Ig * H;
  MOE_CUDA(launch_uniform_offsets(offsets, G, T, s));
  const GemmOperand ma{x, (uint64_t)H, (uint64_t)T};
  const GemmOperand mb{w1, 64, (uint64_t)G * 2 * Ig * (H / 64)};
  const GemmOperand mh{h, (uint64_t)Ig, (uint64_t)R};
  const GemmOperand md{w2, 64, (uint64_t)G * H * (Ig / 64)};
  const long long lim = g_wait_limit.load();
  if (use_swap_gemm(G, R, H, Ig)) {
    MOE_CUDA(launch_gemm_gate_up_swap(ma, mb, offsets, G, R, H, Ig, h, status, lim, s, true));
    MOE_CUDA(launch_gemm_down_swap(mh, md, offsets, G, R, H, Ig, shared_out, status, lim, s));
  } else {
    MOE_CUDA(launch_gemm_gate_up(ma, mb, offsets, G, R, H, Ig, h, status, lim, s, true));
    MOE_CUDA(launch_gemm_down(mh, md, offsets, G, R, H, Ig, shared_out, status, lim, s));
  }
  return MOE_OK;
}

// Expert ranks on one GPU: owner map, rank count, optional shared expert (packed
// by moe_prepack_shared_expert, intermediate size Is, 0: none).
struct ShardArgs {
  const int32_t* owner;
  int G;
  const void* shared_packed;
  int Is;
};

size_t sharded_extra_bytes(const moe_dims& d, const ShardArgs& a) {
  if (a.Is <= 0) return 0;
  return shared_layout(d.T, a.G, a.Is).total + up((size_t)a.G * d.T * d.H * 4);
}

moe_status check_opts(const moe_router_opts& o) {
  if (o.kind != MOE_ROUTER_SOFTMAX && o.kind != MOE_ROUTER_SIGMOID_BIAS_SELECT)
    return MOE_ERR_INVALID_ARG;
  if (!(o.route_scale > 0.0f) || !isfinite(o.route_scale)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

constexpr moe_router_opts kDefaultOpts = {MOE_ROUTER_SOFTMAX, 0, 1.0f};

moe_status layer_fwd(const void* x, const float* w_router, const float* bias,
                     const moe_router_opts& opts, const void* packed_weights, const moe_dims& d,
                     void* out, int32_t* topk_idx_out, float* topk_w_out, int32_t* counts_out,
                     void* workspace, size_t ws_bytes, cudaStream_t s, cudaEvent_t* ev,
                     const ShardArgs* shard = nullptr) {
  MOE_TRY(check_dims(d));
  MOE_TRY(check_opts(opts));
  MOE_TRY(check_ws(d, workspace, ws_bytes));
  if (shard != nullptr) {
    if (shard->G < 1 || shard->G > kMaxShards) return MOE_ERR_UNSUPPORTED;
    MOE_TRY(need(shard->owner));
    if (shard->Is > 0) {
      MOE_TRY(check_shared(d.T, d.H, shard->Is, shard->G));
      MOE_TRY(need(shard->shared_packed));
    }
    if (ws_bytes < layout(d).total + sharded_extra_bytes(d, *shard)) return MOE_ERR_WORKSPACE;
  }
  MOE_TRY(need(w_router));
  if (bias != nullptr) MOE_TRY(need(bias));
  MOE_TRY(need(packed_weights));
  if (topk_idx_out != nullptr) MOE_TRY(need(topk_idx_out));
  if (topk_w_out != nullptr) MOE_TRY(need(topk_w_out));
  if (counts_out != nullptr) MOE_TRY(need(counts_out));
  if (d.T > 0) {
    MOE_TRY(need(x));
    MOE_TRY(need(out));
  }
  MOE_TRY(device_ok());
  const Layout L = layout(d);
  int32_t* idx = topk_idx_out ? topk_idx_out : at<int32_t>(workspace, L.idx);
  float* w = topk_w_out ? topk_w_out : at<float>(workspace, L.w);
  int32_t* counts = counts_out ? counts_out : at<int32_t>(workspace, L.counts);
  int32_t* offsets = at<int32_t>(workspace, L.offsets);
  int32_t* ros = at<int32_t>(workspace, L.row_of_slot);
  int32_t* sor = at<int32_t>(workspace, L.slot_of_row);
  void* x_perm = at<void>(workspace, L.x_perm);
  float* y = at<float>(workspace, L.y);
  auto mark = [&](int i) -> moe_status {
    if (ev != nullptr && cudaEventRecord(ev[i], s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  };
  MOE_TRY(mark(0));
  MOE_CUDA(launch_route(x, w_router, bias, d.T, d.H, d.E, d.k, opts.kind, opts.weights_bf16, idx,
                        w, s));
  MOE_TRY(mark(1));
  if (d.T == 1 && ev == nullptr && shard == nullptr && use_swap_gemm(d.E, d.k, d.H, d.I)) {
    // One token: both GEMMs take their rows from the token's expert ids and the
    // gate/up GEMM reads the token row itself, so the dispatch (indices only) runs
    // after them and off their path; the combine then reads the rows after its wait.
    MOE_TRY(do_expert_ffn(nullptr, offsets, packed_weights, d, y, workspace, s, nullptr, x, idx));
    MOE_CUDA(launch_dispatch_small(idx, d.T, d.k, d.E, x, d.H, counts, offsets, ros, sor, nullptr,
                                   at<int32_t>(workspace, L.status), s));
    MOE_CUDA(launch_combine(y, w, ros, d.T, d.H, d.k, opts.route_scale, out, s, false));
    return MOE_OK;
  }
  if (d.T > 0 && d.T <= kPermBlock) {
    // one ranking block: counts, offsets, ranks and the row copy in a single
    // launch (the load-statistics stage holds the permute; mark 2 closes both)
    MOE_CUDA(launch_dispatch_small(idx, d.T, d.k, d.E, x, d.H, counts, offsets, ros, sor, x_perm,
                                   at<int32_t>(workspace, L.status), s));
    MOE_TRY(mark(2));
  } else {
    MOE_TRY(do_load_stats(idx, d, counts, offsets, false, workspace, s));
    MOE_TRY(mark(2));
    if (d.T > 0) MOE_TRY(do_permute_rows(x, idx, d, x_perm, ros, sor, workspace, s));
  }
  MOE_TRY(mark(3));
  if (d.T > 0)
    MOE_TRY(do_expert_ffn(x_perm, offsets, packed_weights, d, y, workspace, s,
                          ev != nullptr ? ev[4] : nullptr));
  else
    MOE_TRY(mark(4));
  if (shard != nullptr) {
    float* shared_out = nullptr;
    if (shard->Is > 0 && d.T > 0) {
      void* sws = at<void>(workspace, L.total);
      shared_out = at<float>(workspace, L.total + shared_layout(d.T, shard->G, shard->Is).total);
      MOE_TRY(do_shared_expert(x, shard->shared_packed, d.T, d.H, shard->Is, shard->G, shared_out,
                               sws, at<int32_t>(workspace, L.status), s));
    }
    MOE_TRY(mark(5));
    if (d.T > 0)
      MOE_CUDA(launch_combine_sharded(y, w, idx, ros, shard->owner, shard->G, d.T, d.H, d.E, d.k,
                                      opts.route_scale, shared_out, nullptr, out, s));
    MOE_TRY(mark(6));
    return MOE_OK;
  }
  MOE_TRY(mark(5));
  // the routing and the rows were written before the expert GEMMs began
  if (d.T > 0)
    MOE_CUDA(launch_combine(y, w, ros, d.T, d.H, d.k, opts.route_scale, out, s, true));
  MOE_TRY(mark(6));
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(moe_dims d) {
  if (check_dims(d) != MOE_OK) return 0;
  return layout(d).total;
}

size_t moe_packed_weight_bytes(moe_dims d) {
  if (check_dims(d) != MOE_OK) return 0;
  return (size_t)d.E * 3 * d.H * d.I * 2;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported dimensions or device";
    case MOE_ERR_MISALIGNED: return "misaligned pointer";
    case MOE_ERR_WORKSPACE: return "workspace or packed buffer too small";
    case MOE_ERR_CUDA: return "CUDA runtime or launch error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device-side index or offset check failed";
  }
  return "unknown status";
}

moe_status moe_route_ex(const void* x, const float* w_router, const float* bias,
                        const moe_router_opts* opts, moe_dims d, int32_t* topk_idx, float* topk_w,
                        void* stream) {
  const moe_router_opts o = opts ? *opts : kDefaultOpts;
  MOE_TRY(check_dims(d));
  MOE_TRY(check_opts(o));
  if (d.T == 0) return MOE_OK;
  MOE_TRY(need(x));
  MOE_TRY(need(w_router));
  if (bias != nullptr) MOE_TRY(need(bias));
  MOE_TRY(need(topk_idx));
  MOE_TRY(need(topk_w));
  MOE_TRY(device_ok());
  MOE_CUDA(launch_route(x, w_router, bias, d.T, d.H, d.E, d.k, o.kind, o.weights_bf16, topk_idx,
                        topk_w, as_stream(stream)));
  return MOE_OK;
}

moe_status moe_route(const void* x, const float* w_router, const float* bias, moe_dims d,
                     int32_t* topk_idx, float* topk_w, void* stream) {
  return moe_route_ex(x, w_router, bias, nullptr, d, topk_idx, topk_w, stream);
}

moe_status moe_load_stats(const int32_t* topk_idx, moe_dims d, int32_t* counts, int32_t* offsets,
                          void* workspace, size_t ws_bytes, void* stream) {
  MOE_TRY(check_dims(d));
  if (d.T > 0) MOE_TRY(need(topk_idx));
  MOE_TRY(need(counts));
  MOE_TRY(need(offsets));
  MOE_TRY(check_ws(d, workspace, ws_bytes));
  MOE_TRY(device_ok());
  return do_load_stats(topk_idx, d, counts, offsets, false, workspace, as_stream(stream));
}

moe_status moe_load_summary_host(const int32_t* counts_host, int32_t E, double* imbalance,
                                 double* cv) {
  if (counts_host == nullptr || E <= 0) return MOE_ERR_INVALID_ARG;
  double sum = 0.0, mx = 0.0;
  for (int e = 0; e < E; ++e) {
    sum += counts_host[e];
    mx = fmax(mx, (double)counts_host[e]);
  }
  const double mean = sum / E;
  double var = 0.0;
  for (int e = 0; e < E; ++e) var += (counts_host[e] - mean) * (counts_host[e] - mean);
  var /= E;
  if (imbalance) *imbalance = mean > 0 ? mx / mean - 1.0 : 0.0;
  if (cv) *cv = mean > 0 ? sqrt(var) / mean : 0.0;
  return MOE_OK;
}

moe_status moe_load_stats_ex(const int32_t* topk_idx, const int32_t* slot_of_expert,
                             const int32_t* q, moe_dims d, int32_t* counts, int32_t* offsets,
                             int64_t* weighted_counts, void* workspace, size_t ws_bytes,
                             void* stream) {
  MOE_TRY(check_dims(d));
  if (d.T > 0) MOE_TRY(need(topk_idx));
  MOE_TRY(need(counts));
  MOE_TRY(need(offsets));
  if (slot_of_expert != nullptr) MOE_TRY(need(slot_of_expert));
  if (weighted_counts != nullptr) {
    MOE_TRY(need(weighted_counts));
    if (q == nullptr) return MOE_ERR_INVALID_ARG;
    if (d.T > 0) MOE_TRY(need(q));
  }
  MOE_TRY(check_ws(d, workspace, ws_bytes));
  MOE_TRY(device_ok());
  cudaStream_t s = as_stream(stream);
  MOE_TRY(do_load_stats(topk_idx, d, counts, offsets, false, workspace, s, slot_of_expert));
  if (weighted_counts != nullptr)
    MOE_CUDA(launch_weighted_counts(topk_idx, q, d.T, d.k, d.E, weighted_counts,
                                    at<int32_t>(workspace, layout(d).status), s));
  return MOE_OK;
}

moe_status moe_lpt_placement_host(const int64_t* loads, int32_t E, int32_t P,
                                  int32_t* slot_of_expert, int64_t* rank_loads) {
  if (loads == nullptr || slot_of_expert == nullptr || E <= 0 || P <= 0 || E % P != 0 ||
      E > kMaxE)
    return MOE_ERR_INVALID_ARG;
  const int Hs = E / P;
  int64_t G[kMaxE] = {};
  int n[kMaxE] = {};
  int order[kMaxE];
  for (int e = 0; e < E; ++e) order[e] = e;
  // experts by (load descending, index ascending); insertion sort keeps it plain
  for (int i = 1; i < E; ++i) {
    const int v = order[i];
    int j = i - 1;
    while (j >= 0 && (loads[order[j]] < loads[v] || (loads[order[j]] == loads[v] && order[j] > v))) {
      order[j + 1] = order[j];
      --j;
    }
    order[j + 1] = v;
  }
  for (int i = 0; i < E; ++i) {
    const int e = order[i];
    int best = -1;
    for (int p = 0; p < P; ++p)
      if (n[p] < Hs && (best < 0 || G[p] < G[best])) best = p;  // ties: lower rank
    slot_of_expert[e] = best * Hs + n[best];
    G[best] += loads[e];
    n[best] += 1;
  }
  if (rank_loads != nullptr)
    for (int p = 0; p < P; ++p) rank_loads[p] = G[p];
  return MOE_OK;
}

moe_status moe_rank_load_summary_host(const int64_t* rank_loads, int32_t P, double* cv,
                                      double* eta_ep) {
  if (rank_loads == nullptr || P <= 0) return MOE_ERR_INVALID_ARG;
  double mean = 0.0, mx = 0.0;
  for (int p = 0; p < P; ++p) {
    mean += (double)rank_loads[p];
    mx = fmax(mx, (double)rank_loads[p]);
  }
  mean /= P;
  double var = 0.0;
  for (int p = 0; p < P; ++p) var += ((double)rank_loads[p] - mean) * ((double)rank_loads[p] - mean);
  var /= P;
  if (cv) *cv = mean > 0 ? sqrt(var) / mean : 0.0;
  if (eta_ep) *eta_ep = mx > 0 ? mean / mx : 1.0;
  return MOE_OK;
}

moe_status moe_permute_ex(const void* x, const int32_t* topk_idx, const int32_t* slot_of_expert,
                          const int32_t* offsets, moe_dims d, void* x_perm, int32_t* row_of_slot,
                          int32_t* slot_of_row, void* workspace, size_t ws_bytes, void* stream) {
  MOE_TRY(check_dims(d));
  MOE_TRY(need(offsets));
  MOE_TRY(check_ws(d, workspace, ws_bytes));
  if (slot_of_expert != nullptr) MOE_TRY(need(slot_of_expert));
  if (d.T == 0) return MOE_OK;
  MOE_TRY(need(x));
  MOE_TRY(need(topk_idx));
  MOE_TRY(need(x_perm));
  MOE_TRY(need(row_of_slot));
  MOE_TRY(need(slot_of_row));
  MOE_TRY(device_ok());
  cudaStream_t s = as_stream(stream);
  MOE_TRY(do_load_stats(topk_idx, d, nullptr, const_cast<int32_t*>(offsets), true, workspace, s,
                        slot_of_expert));
  return do_permute_rows(x, topk_idx, d, x_perm, row_of_slot, slot_of_row, workspace, s,
                         slot_of_expert);
}

moe_status moe_permute(const void* x, const int32_t* topk_idx, const int32_t* offsets, moe_dims d,
                       void* x_perm, int32_t* row_of_slot, int32_t* slot_of_row, void* workspace,
                       size_t ws_bytes, void* stream) {
  MOE_TRY(check_dims(d));
  MOE_TRY(need(offsets));
  MOE_TRY(check_ws(d, workspace, ws_bytes));
  if (d.T == 0) return MOE_OK;
  MOE_TRY(need(x));
  MOE_TRY(need(topk_idx));
  MOE_TRY(need(x_perm));
  MOE_TRY(need(row_of_slot));
  MOE_TRY(need(slot_of_row));
  MOE_TRY(device_ok());
  cudaStream_t s = as_stream(stream);
  MOE_TRY(do_load_stats(topk_idx, d, nullptr, const_cast<int32_t*>(offsets), true, workspace, s));
  return do_permute_rows(x, topk_idx, d, x_perm, row_of_slot, slot_of_row, workspace, s);
}

moe_status moe_prepack_expert_weights_ex(const void* w_gate, const void* w_up,
                                         const void* w_down, const int32_t* slot_of_expert,
                                         moe_dims d, void* packed, size_t packed_bytes,
                                         void* stream) {
  MOE_TRY(check_dims(d));
  MOE_TRY(need(w_gate));
  MOE_TRY(need(w_up));
  MOE_TRY(need(w_down));
  MOE_TRY(need(packed));
  if (slot_of_expert != nullptr) MOE_TRY(need(slot_of_expert));
  if (packed_bytes < moe_packed_weight_bytes(d)) return MOE_ERR_WORKSPACE;
  MOE_TRY(device_ok());
  MOE_CUDA(launch_prepack(w_gate, w_up, w_down, d.E, d.H, d.I, packed, as_stream(stream),
                          slot_of_expert));
  return MOE_OK;
}

moe_status moe_prepack_expert_weights(const void* w_gate, const void* w_up, const void* w_down,
                                      moe_dims d, void* packed, size_t packed_bytes,
                                      void* stream) {
  MOE_TRY(check_dims(d));
  MOE_TRY(need(w_gate));
  MOE_TRY(need(w_up));
  MOE_TRY(need(w_down));
  MOE_TRY(need(packed));
  if (packed_bytes < moe_packed_weight_bytes(d)) return MOE_ERR_WORKSPACE;
  MOE_TRY(device_ok());
  MOE_CUDA(launch_prepack(w_gate, w_up, w_down, d.E, d.H, d.I, packed, as_stream(stream)));
  return MOE_OK;
}

moe_status moe_expert_ffn(const void* x_perm, const int32_t* offsets, const void* packed_weights,
                          moe_dims d, float* y, void* workspace, size_t ws_bytes, void* stream) {
  MOE_TRY(check_dims(d));
  MOE_TRY(check_ws(d, workspace, ws_bytes));
  if (d.T == 0) return MOE_OK;
  MOE_TRY(need(x_perm));
  MOE_TRY(need(offsets));
  MOE_TRY(need(packed_weights));
  MOE_TRY(need(y));
  MOE_TRY(device_ok());
  return do_expert_ffn(x_perm, offsets, packed_weights, d, y, workspace, as_stream(stream));
}

int moe_expert_ffn_form(moe_dims d) {
  moe_status st = check_dims(d);
  if (st == MOE_OK) st = device_ok();
  if (st != MOE_OK) return -(int)st;
  return use_swap_gemm(d.E, d.T * d.k, d.H, d.I) ? 1 : 0;
}

moe_status moe_combine_ex(const float* y, const float* topk_w, const int32_t* row_of_slot,
                          float route_scale, moe_dims d, void* out, void* stream) {
  MOE_TRY(check_dims(d));
  if (!(route_scale > 0.0f) || !isfinite(route_scale)) return MOE_ERR_INVALID_ARG;
  if (d.T == 0) return MOE_OK;
  MOE_TRY(need(y));
  MOE_TRY(need(topk_w));
  MOE_TRY(need(row_of_slot));
  MOE_TRY(need(out));
  MOE_TRY(device_ok());
  MOE_CUDA(launch_combine(y, topk_w, row_of_slot, d.T, d.H, d.k, route_scale, out,
                          as_stream(stream)));
  return MOE_OK;
}

moe_status moe_combine(const float* y, const float* topk_w, const int32_t* row_of_slot, moe_dims d,
                       void* out, void* stream) {
  return moe_combine_ex(y, topk_w, row_of_slot, 1.0f, d, out, stream);
}

size_t moe_shared_packed_bytes(int32_t H, int32_t Is) {
  if (H <= 0 || Is <= 0) return 0;
  return (size_t)3 * H * Is * 2;
}

size_t moe_shared_expert_workspace_bytes(int32_t T, int32_t H, int32_t Is, int32_t G) {
  if (check_shared(T, H, Is, G) != MOE_OK) return 0;
  return shared_layout(T, G, Is).total;
}

moe_status moe_prepack_shared_expert(const void* w_gate, const void* w_up, const void* w_down,
                                     int32_t H, int32_t Is, int32_t G, void* packed,
                                     size_t packed_bytes, void* stream) {
  MOE_TRY(check_shared(0, H, Is, G));
  MOE_TRY(need(w_gate));
  MOE_TRY(need(w_up));
  MOE_TRY(need(w_down));
  MOE_TRY(need(packed));
  if (packed_bytes < moe_shared_packed_bytes(H, Is)) return MOE_ERR_WORKSPACE;
  MOE_TRY(device_ok());
  MOE_CUDA(launch_prepack_shared(w_gate, w_up, w_down, H, Is, G, packed, as_stream(stream)));
  return MOE_OK;
}

moe_status moe_shared_expert(const void* x, const void* shared_packed, int32_t T, int32_t H,
                             int32_t Is, int32_t G, float* shared_out, void* workspace,
                             size_t ws_bytes, void* stream) {
  MOE_TRY(check_shared(T, H, Is, G));
  if (workspace == nullptr) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return MOE_ERR_MISALIGNED;
  if (ws_bytes < shared_layout(T, G, Is).total) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  MOE_TRY(need(x));
  MOE_TRY(need(shared_packed));
  MOE_TRY(need(shared_out));
  MOE_TRY(device_ok());
  return do_shared_expert(x, shared_packed, T, H, Is, G, shared_out, workspace,
                          at<int32_t>(workspace, shared_layout(T, G, Is).status), as_stream(stream));
}

size_t moe_sharded_workspace_bytes(moe_dims d, int32_t G, int32_t Is) {
  if (check_dims(d) != MOE_OK || G < 1 || G > kMaxShards) return 0;
  if (Is > 0 && check_shared(d.T, d.H, Is, G) != MOE_OK) return 0;
  const ShardArgs a{nullptr, G, nullptr, Is};
  return layout(d).total + sharded_extra_bytes(d, a);
}

moe_status moe_layer_fwd_sharded(const void* x, const float* w_router, const float* bias,
                                 const moe_router_opts* opts, const void* packed_weights,
                                 const int32_t* owner, int32_t G, const void* shared_packed,
                                 int32_t Is, moe_dims d, void* out, int32_t* topk_idx_out,
                                 float* topk_w_out, int32_t* counts_out, void* workspace,
                                 size_t ws_bytes, void* stream) {
  const ShardArgs a{owner, G, shared_packed, Is};
  return layer_fwd(x, w_router, bias, opts ? *opts : kDefaultOpts, packed_weights, d, out,
                   topk_idx_out, topk_w_out, counts_out, workspace, ws_bytes, as_stream(stream),
                   nullptr, &a);
}

moe_status moe_combine_sharded(const float* y, const float* topk_w, const int32_t* topk_idx,
                               const int32_t* row_of_slot, const int32_t* owner, int32_t G,
                               float route_scale, const float* shared, moe_dims d, void* partials,
                               void* out, void* stream) {
  MOE_TRY(check_dims(d));
  if (G < 1 || G > kMaxShards) return MOE_ERR_UNSUPPORTED;
  if (!(route_scale > 0.0f) || !isfinite(route_scale)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(need(owner));
  if (d.T == 0) return MOE_OK;
  MOE_TRY(need(y));
  MOE_TRY(need(topk_w));
  MOE_TRY(need(topk_idx));
  MOE_TRY(need(row_of_slot));
  MOE_TRY(need(out));
  if (shared != nullptr) MOE_TRY(need(shared));
  if (partials != nullptr) MOE_TRY(need(partials));
  MOE_TRY(device_ok());
  MOE_CUDA(launch_combine_sharded(y, topk_w, topk_idx, row_of_slot, owner, G, d.T, d.H, d.E, d.k,
                                  route_scale, shared, partials, out, as_stream(stream)));
  return MOE_OK;
}

moe_status moe_tree_reduce_bf16(const void* partials, int32_t G, int64_t N, void* out,
                                void* stream) {
  if (G < 1 || N < 0) return MOE_ERR_INVALID_ARG;
  if (G > kMaxShards) return MOE_ERR_UNSUPPORTED;
  if (N == 0) return MOE_OK;
  if (partials == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(partials) & 1) || (reinterpret_cast<uintptr_t>(out) & 1))
    return MOE_ERR_MISALIGNED;
  MOE_TRY(device_ok());
  const bool vec = (N % 8 == 0) && aligned16(partials) && aligned16(out);
  MOE_CUDA(launch_tree_reduce(partials, G, (long long)N, out, vec, as_stream(stream)));
  return MOE_OK;
}

moe_status moe_layer_fwd(const void* x, const float* w_router, const float* bias,
                         const void* packed_weights, moe_dims d, void* out, int32_t* topk_idx_out,
                         float* topk_w_out, int32_t* counts_out, void* workspace, size_t ws_bytes,
                         void* stream) {
  return layer_fwd(x, w_router, bias, kDefaultOpts, packed_weights, d, out, topk_idx_out, topk_w_out,
                   counts_out, workspace, ws_bytes, as_stream(stream), nullptr);
}

moe_status moe_layer_fwd_ex(const void* x, const float* w_router, const float* bias,
                            const moe_router_opts* opts, const void* packed_weights, moe_dims d,
                            void* out, int32_t* topk_idx_out, float* topk_w_out,
                            int32_t* counts_out, void* workspace, size_t ws_bytes, void* stream) {
  return layer_fwd(x, w_router, bias, opts ? *opts : kDefaultOpts, packed_weights, d, out,
                   topk_idx_out, topk_w_out, counts_out, workspace, ws_bytes, as_stream(stream),
                   nullptr);
}

moe_status moe_layer_fwd_profiled(const void* x, const float* w_router, const float* bias,
                                  const void* packed_weights, moe_dims d, void* out,
                                  int32_t* topk_idx_out, float* topk_w_out, int32_t* counts_out,
                                  void* workspace, size_t ws_bytes, void* stream,
                                  void* const* events, int32_t n_events) {
  if (n_events == 0 && events == nullptr)
    return moe_layer_fwd(x, w_router, bias, packed_weights, d, out, topk_idx_out, topk_w_out,
                         counts_out, workspace, ws_bytes, stream);
  if (n_events != 7 || events == nullptr) return MOE_ERR_INVALID_ARG;
  cudaEvent_t ev[7];
  for (int i = 0; i < 7; ++i) {
    if (events[i] == nullptr) return MOE_ERR_INVALID_ARG;
    ev[i] = static_cast<cudaEvent_t>(events[i]);
  }
  return layer_fwd(x, w_router, bias, kDefaultOpts, packed_weights, d, out, topk_idx_out, topk_w_out,
                   counts_out, workspace, ws_bytes, as_stream(stream), ev);
}

moe_status moe_layer_fwd_sharded_profiled(
    const void* x, const float* w_router, const float* bias, const moe_router_opts* opts,
    const void* packed_weights, const int32_t* owner, int32_t G, const void* shared_packed,
    int32_t Is, moe_dims d, void* out, int32_t* topk_idx_out, float* topk_w_out,
    int32_t* counts_out, void* workspace, size_t ws_bytes, void* stream, void* const* events,
    int32_t n_events) {
  if (n_events != 7 || events == nullptr) return MOE_ERR_INVALID_ARG;
  cudaEvent_t ev[7];
  for (int i = 0; i < 7; ++i) {
    if (events[i] == nullptr) return MOE_ERR_INVALID_ARG;
    ev[i] = static_cast<cudaEvent_t>(events[i]);
  }
  const ShardArgs a{owner, G, shared_packed, Is};
  return layer_fwd(x, w_router, bias, opts ? *opts : kDefaultOpts, packed_weights, d, out,
                   topk_idx_out, topk_w_out, counts_out, workspace, ws_bytes, as_stream(stream),
                   ev, &a);
}

moe_status moe_set_wait_limit(long long cycles) {
  g_wait_limit.store(cycles > 0 ? cycles : kSpinLimitCycles);
  return MOE_OK;
}

moe_status moe_read_device_status(void* workspace, int32_t* status_out, void* stream) {
  if (workspace == nullptr || status_out == nullptr) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return MOE_ERR_MISALIGNED;
  cudaStream_t s = as_stream(stream);
  int32_t v = 0;
  MOE_CUDA(cudaMemcpyAsync(&v, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  MOE_CUDA(cudaStreamSynchronize(s));
  MOE_CUDA(cudaMemsetAsync(workspace, 0, sizeof(int32_t), s));
  MOE_CUDA(cudaStreamSynchronize(s));
  *status_out = v;
  return MOE_OK;
}

}  // extern "C"
