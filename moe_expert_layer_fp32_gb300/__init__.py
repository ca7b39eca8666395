"""GB300 (sm_103a) top-k routed MoE feed-forward layer forward.

Thin binding over the C ABI in ``include/moe.h`` (``libmoe_gb300.so``): the
functions below carry the same names and only marshal arguments (torch tensors
-> device pointers, the current CUDA stream).  Every step runs in the library's
CUDA kernels; there is no CPU path.  Importing fails loudly when the library has
not been built (``python moe_expert_layer_fp32_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python moe_expert_layer_fp32_gb300/build.py)")

_lib = ctypes.CDLL(LIB_PATH)

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_MISALIGNED",
          4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_TIMEOUT",
          7: "MOE_ERR_DEVICE_CHECK"}

# Every symbol include/moe.h declares.
ABI_SYMBOLS = ("moe_workspace_bytes", "moe_packed_weight_bytes", "moe_route", "moe_load_stats",
               "moe_load_summary_host", "moe_permute", "moe_prepack_expert_weights",
               "moe_expert_ffn", "moe_combine", "moe_layer_fwd", "moe_layer_fwd_profiled",
               "moe_read_device_status", "moe_status_string", "moe_load_stats_noalloc",
               "moe_set_wait_limit", "moe_route_ex", "moe_combine_ex", "moe_layer_fwd_ex",
               "moe_load_stats_ex", "moe_lpt_placement_host", "moe_rank_load_summary_host",
               "moe_permute_ex", "moe_prepack_expert_weights_ex", "moe_combine_sharded",
               "moe_tree_reduce_bf16", "moe_shared_packed_bytes", "moe_prepack_shared_expert",
               "moe_shared_expert_workspace_bytes", "moe_shared_expert",
               "moe_sharded_workspace_bytes", "moe_layer_fwd_sharded",
               "moe_layer_fwd_sharded_profiled", "moe_expert_ffn_form")


class moe_dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("I", ctypes.c_int32)]

    def __repr__(self):
        return f"moe_dims(T={self.T}, H={self.H}, E={self.E}, k={self.k}, I={self.I})"


def dims(T, H, E, k, I) -> moe_dims:
    return moe_dims(T, H, E, k, I)


MOE_ROUTER_SOFTMAX, MOE_ROUTER_SIGMOID_BIAS_SELECT = 0, 1


class moe_router_opts(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("weights_bf16", ctypes.c_int32),
                ("route_scale", ctypes.c_float)]


def router_opts(kind=MOE_ROUTER_SOFTMAX, weights_bf16=False, route_scale=1.0) -> moe_router_opts:
    return moe_router_opts(int(kind), int(bool(weights_bf16)), float(route_scale))


def _opts(o):
    return None if o is None else ctypes.byref(o)


_vp, _sz, _i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
_sig = {
    "moe_workspace_bytes": (_sz, [moe_dims]),
    "moe_packed_weight_bytes": (_sz, [moe_dims]),
    "moe_route": (ctypes.c_int, [_vp, _vp, _vp, moe_dims, _vp, _vp, _vp]),
    "moe_load_stats": (ctypes.c_int, [_vp, moe_dims, _vp, _vp, _vp, _sz, _vp]),
    "moe_load_summary_host": (ctypes.c_int, [_vp, _i32, _vp, _vp]),
    "moe_permute": (ctypes.c_int, [_vp, _vp, _vp, moe_dims, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_prepack_expert_weights": (ctypes.c_int, [_vp, _vp, _vp, moe_dims, _vp, _sz, _vp]),
    "moe_expert_ffn": (ctypes.c_int, [_vp, _vp, _vp, moe_dims, _vp, _vp, _sz, _vp]),
    "moe_combine": (ctypes.c_int, [_vp, _vp, _vp, moe_dims, _vp, _vp]),
    "moe_layer_fwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, moe_dims, _vp, _vp, _vp, _vp, _vp, _sz,
                                     _vp]),
    "moe_layer_fwd_profiled": (ctypes.c_int, [_vp, _vp, _vp, _vp, moe_dims, _vp, _vp, _vp, _vp,
                                              _vp, _sz, _vp, _vp, _i32]),
    "moe_read_device_status": (ctypes.c_int, [_vp, _vp, _vp]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_load_stats_noalloc": (ctypes.c_int, [_vp, moe_dims, _vp, _vp, _vp, _vp]),
    "moe_set_wait_limit": (ctypes.c_int, [ctypes.c_longlong]),
    "moe_route_ex": (ctypes.c_int, [_vp, _vp, _vp, _vp, moe_dims, _vp, _vp, _vp]),
    "moe_combine_ex": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_float, moe_dims, _vp, _vp]),
    "moe_layer_fwd_ex": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, moe_dims, _vp, _vp, _vp, _vp,
                                        _vp, _sz, _vp]),
    "moe_load_stats_ex": (ctypes.c_int, [_vp, _vp, _vp, moe_dims, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_lpt_placement_host": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp]),
    "moe_rank_load_summary_host": (ctypes.c_int, [_vp, _i32, _vp, _vp]),
    "moe_permute_ex": (ctypes.c_int, [_vp, _vp, _vp, _vp, moe_dims, _vp, _vp, _vp, _vp, _sz,
                                      _vp]),
    "moe_prepack_expert_weights_ex": (ctypes.c_int, [_vp, _vp, _vp, _vp, moe_dims, _vp, _sz,
                                                     _vp]),
    "moe_combine_sharded": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i32, ctypes.c_float, _vp,
                                           moe_dims, _vp, _vp, _vp]),
    "moe_tree_reduce_bf16": (ctypes.c_int, [_vp, _i32, ctypes.c_int64, _vp, _vp]),
    "moe_shared_packed_bytes": (_sz, [_i32, _i32]),
    "moe_expert_ffn_form": (ctypes.c_int, [moe_dims]),
    "moe_prepack_shared_expert": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _sz, _vp]),
    "moe_shared_expert_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32]),
    "moe_shared_expert": (ctypes.c_int, [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _sz, _vp]),
    "moe_sharded_workspace_bytes": (_sz, [moe_dims, _i32, _i32]),
    "moe_layer_fwd_sharded": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32,
                                             moe_dims, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_layer_fwd_sharded_profiled": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp,
                                                      _i32, moe_dims, _vp, _vp, _vp, _vp, _vp,
                                                      _sz, _vp, _vp, _i32]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class MoEError(RuntimeError):
    def __init__(self, name, code):
        self.code = code
        super().__init__(f"{name}: {STATUS.get(code, code)} "
                         f"({_lib.moe_status_string(code).decode()})")


def _check(name, code):
    if code != MOE_OK:
        raise MoEError(name, code)


def _ptr(t):
    """Device address of a tensor (None -> NULL); an int is taken as an address."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ws(ws):
    return (_ptr(ws), ws.numel() * ws.element_size()) if isinstance(ws, torch.Tensor) else ws


# ------------------------------------------------------------ raw ABI calls ---
def moe_workspace_bytes(d: moe_dims) -> int:
    return int(_lib.moe_workspace_bytes(d))


def moe_packed_weight_bytes(d: moe_dims) -> int:
    return int(_lib.moe_packed_weight_bytes(d))


def moe_route(x, w_router, bias, d, topk_idx, topk_w, stream=None):
    _check("moe_route", _lib.moe_route(_ptr(x), _ptr(w_router), _ptr(bias), d, _ptr(topk_idx),
                                       _ptr(topk_w), _stream(stream)))


def moe_route_ex(x, w_router, bias, opts, d, topk_idx, topk_w, stream=None):
    _check("moe_route_ex", _lib.moe_route_ex(_ptr(x), _ptr(w_router), _ptr(bias), _opts(opts), d,
                                             _ptr(topk_idx), _ptr(topk_w), _stream(stream)))


def moe_combine_ex(y, topk_w, row_of_slot, route_scale, d, out, stream=None):
    _check("moe_combine_ex", _lib.moe_combine_ex(_ptr(y), _ptr(topk_w), _ptr(row_of_slot),
                                                 float(route_scale), d, _ptr(out),
                                                 _stream(stream)))


def moe_layer_fwd_ex(x, w_router, bias, opts, packed_weights, d, out, topk_idx_out, topk_w_out,
                     counts_out, workspace, stream=None):
    wp, wb = _ws(workspace)
    _check("moe_layer_fwd_ex", _lib.moe_layer_fwd_ex(
        _ptr(x), _ptr(w_router), _ptr(bias), _opts(opts), _ptr(packed_weights), d, _ptr(out),
        _ptr(topk_idx_out), _ptr(topk_w_out), _ptr(counts_out), wp, wb, _stream(stream)))


def moe_load_stats(topk_idx, d, counts, offsets, workspace, stream=None):
    wp, wb = _ws(workspace)
    _check("moe_load_stats", _lib.moe_load_stats(_ptr(topk_idx), d, _ptr(counts), _ptr(offsets),
                                                 wp, wb, _stream(stream)))


def moe_load_stats_noalloc(topk_idx, d, counts, offsets, device_status=None, stream=None):
    """moe_load_stats without a workspace, for callers that cannot allocate: the
    library's own fixed scratch array holds the partial counts (see include/moe.h
    for the size limit and the rule that overlapping calls race)."""
    _check("moe_load_stats_noalloc", _lib.moe_load_stats_noalloc(
        _ptr(topk_idx), d, _ptr(counts), _ptr(offsets), _ptr(device_status), _stream(stream)))


def moe_load_stats_ex(topk_idx, slot_of_expert, q, d, counts, offsets, weighted_counts,
                      workspace, stream=None):
    wp, wb = _ws(workspace)
    _check("moe_load_stats_ex", _lib.moe_load_stats_ex(
        _ptr(topk_idx), _ptr(slot_of_expert), _ptr(q), d, _ptr(counts), _ptr(offsets),
        _ptr(weighted_counts), wp, wb, _stream(stream)))


def moe_lpt_placement_host(loads, P):
    """(slot_of_expert [E] int32, rank_loads [P] int64) from host loads (RoutePack Alg. 1)."""
    import numpy as np
    L = np.ascontiguousarray(loads, dtype=np.int64)
    pi = np.empty(L.size, dtype=np.int32)
    G = np.empty(P, dtype=np.int64)
    _check("moe_lpt_placement_host", _lib.moe_lpt_placement_host(
        L.ctypes.data, int(L.size), int(P), pi.ctypes.data, G.ctypes.data))
    return pi, G


def moe_rank_load_summary_host(rank_loads):
    """(cv, eta_ep) of host rank loads."""
    import numpy as np
    G = np.ascontiguousarray(rank_loads, dtype=np.int64)
    cv, eta = ctypes.c_double(), ctypes.c_double()
    _check("moe_rank_load_summary_host", _lib.moe_rank_load_summary_host(
        G.ctypes.data, int(G.size), ctypes.addressof(cv), ctypes.addressof(eta)))
    return cv.value, eta.value


def moe_permute_ex(x, topk_idx, slot_of_expert, offsets, d, x_perm, row_of_slot, slot_of_row,
                   workspace, stream=None):
    wp, wb = _ws(workspace)
    _check("moe_permute_ex", _lib.moe_permute_ex(
        _ptr(x), _ptr(topk_idx), _ptr(slot_of_expert), _ptr(offsets), d, _ptr(x_perm),
        _ptr(row_of_slot), _ptr(slot_of_row), wp, wb, _stream(stream)))


def moe_prepack_expert_weights_ex(w_gate, w_up, w_down, slot_of_expert, d, packed, stream=None):
    nbytes = packed.numel() * packed.element_size() if isinstance(packed, torch.Tensor) else 1 << 62
    _check("moe_prepack_expert_weights_ex", _lib.moe_prepack_expert_weights_ex(
        _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(slot_of_expert), d, _ptr(packed), nbytes,
        _stream(stream)))


def moe_combine_sharded(y, topk_w, topk_idx, row_of_slot, owner, G, route_scale, shared, d, out,
                        partials=None, stream=None):
    """Per-rank BF16 partials (slots of other ranks as exact zeros, optional
    shared-expert shards [G, T, H] fp32) reduced by the fixed FP64 pairwise tree."""
    _check("moe_combine_sharded", _lib.moe_combine_sharded(
        _ptr(y), _ptr(topk_w), _ptr(topk_idx), _ptr(row_of_slot), _ptr(owner), int(G),
        float(route_scale), _ptr(shared), d, _ptr(partials), _ptr(out), _stream(stream)))


def moe_tree_reduce_bf16(partials, G, N, out, stream=None):
    """out [N] = bf16(FP64 pairwise tree over partials [G, N]) (bf16 tensors)."""
    _check("moe_tree_reduce_bf16", _lib.moe_tree_reduce_bf16(_ptr(partials), int(G), int(N),
                                                             _ptr(out), _stream(stream)))


def moe_shared_packed_bytes(H, Is) -> int:
    return int(_lib.moe_shared_packed_bytes(int(H), int(Is)))


def moe_shared_expert_workspace_bytes(T, H, Is, G) -> int:
    return int(_lib.moe_shared_expert_workspace_bytes(int(T), int(H), int(Is), int(G)))


def moe_prepack_shared_expert(w_gate, w_up, w_down, H, Is, G, packed, stream=None):
    nbytes = packed.numel() * packed.element_size() if isinstance(packed, torch.Tensor) else 1 << 62
    _check("moe_prepack_shared_expert", _lib.moe_prepack_shared_expert(
        _ptr(w_gate), _ptr(w_up), _ptr(w_down), int(H), int(Is), int(G), _ptr(packed), nbytes,
        _stream(stream)))


def moe_shared_expert(x, shared_packed, T, H, Is, G, shared_out, workspace, stream=None):
    wp, wb = _ws(workspace)
    _check("moe_shared_expert", _lib.moe_shared_expert(
        _ptr(x), _ptr(shared_packed), int(T), int(H), int(Is), int(G), _ptr(shared_out), wp, wb,
        _stream(stream)))


def moe_sharded_workspace_bytes(d, G, Is=0) -> int:
    return int(_lib.moe_sharded_workspace_bytes(d, int(G), int(Is)))


def moe_layer_fwd_sharded(x, w_router, bias, opts, packed_weights, owner, G, shared_packed, Is, d,
                          out, topk_idx_out, topk_w_out, counts_out, workspace, stream=None):
    wp, wb = _ws(workspace)
    _check("moe_layer_fwd_sharded", _lib.moe_layer_fwd_sharded(
        _ptr(x), _ptr(w_router), _ptr(bias), _opts(opts), _ptr(packed_weights), _ptr(owner),
        int(G), _ptr(shared_packed), int(Is), d, _ptr(out), _ptr(topk_idx_out), _ptr(topk_w_out),
        _ptr(counts_out), wp, wb, _stream(stream)))


def _event_array(events, stream):
    for e in events:
        if e.cuda_event == 0:  # torch creates the CUDA event on its first record
            e.record(torch.cuda.current_stream() if stream is None else stream)
    return (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])


def moe_layer_fwd_sharded_profiled(x, w_router, bias, opts, packed_weights, owner, G,
                                   shared_packed, Is, d, out, topk_idx_out, topk_w_out, counts_out,
                                   workspace, events, stream=None):
    """moe_layer_fwd_sharded with 7 torch.cuda.Event(enable_timing=True) recorded at
    the step boundaries (as moe_layer_fwd_profiled)."""
    wp, wb = _ws(workspace)
    arr = _event_array(events, stream)
    _check("moe_layer_fwd_sharded_profiled", _lib.moe_layer_fwd_sharded_profiled(
        _ptr(x), _ptr(w_router), _ptr(bias), _opts(opts), _ptr(packed_weights), _ptr(owner),
        int(G), _ptr(shared_packed), int(Is), d, _ptr(out), _ptr(topk_idx_out), _ptr(topk_w_out),
        _ptr(counts_out), wp, wb, _stream(stream), arr, len(events)))


def moe_load_summary_host(counts_host):
    """(imbalance max/mean - 1, cv) from host counts (sequence or numpy array)."""
    import numpy as np
    c = np.ascontiguousarray(counts_host, dtype=np.int32)
    imb, cv = ctypes.c_double(), ctypes.c_double()
    _check("moe_load_summary_host", _lib.moe_load_summary_host(
        c.ctypes.data, int(c.size), ctypes.addressof(imb), ctypes.addressof(cv)))
    return imb.value, cv.value


def moe_permute(x, topk_idx, offsets, d, x_perm, row_of_slot, slot_of_row, workspace, stream=None):
    wp, wb = _ws(workspace)
    _check("moe_permute", _lib.moe_permute(_ptr(x), _ptr(topk_idx), _ptr(offsets), d, _ptr(x_perm),
                                           _ptr(row_of_slot), _ptr(slot_of_row), wp, wb,
                                           _stream(stream)))


def moe_prepack_expert_weights(w_gate, w_up, w_down, d, packed, stream=None):
    nbytes = packed.numel() * packed.element_size() if isinstance(packed, torch.Tensor) else 1 << 62
    _check("moe_prepack_expert_weights", _lib.moe_prepack_expert_weights(
        _ptr(w_gate), _ptr(w_up), _ptr(w_down), d, _ptr(packed), nbytes, _stream(stream)))


def moe_expert_ffn(x_perm, offsets, packed_weights, d, y, workspace, stream=None):
    wp, wb = _ws(workspace)
    _check("moe_expert_ffn", _lib.moe_expert_ffn(_ptr(x_perm), _ptr(offsets), _ptr(packed_weights),
                                                 d, _ptr(y), wp, wb, _stream(stream)))


def moe_expert_ffn_form(d):
    """0: tile GEMMs, 1: swapped GEMMs (weight rows on the MMA's M side)."""
    r = _lib.moe_expert_ffn_form(d)
    if r < 0:
        raise MoEError("moe_expert_ffn_form", -r)
    return r


def moe_combine(y, topk_w, row_of_slot, d, out, stream=None):
    _check("moe_combine", _lib.moe_combine(_ptr(y), _ptr(topk_w), _ptr(row_of_slot), d, _ptr(out),
                                           _stream(stream)))


def moe_layer_fwd(x, w_router, bias, packed_weights, d, out, topk_idx_out, topk_w_out, counts_out,
                  workspace, stream=None):
    wp, wb = _ws(workspace)
    _check("moe_layer_fwd", _lib.moe_layer_fwd(
        _ptr(x), _ptr(w_router), _ptr(bias), _ptr(packed_weights), d, _ptr(out),
        _ptr(topk_idx_out), _ptr(topk_w_out), _ptr(counts_out), wp, wb, _stream(stream)))


def moe_layer_fwd_profiled(x, w_router, bias, packed_weights, d, out, topk_idx_out, topk_w_out,
                           counts_out, workspace, events, stream=None):
    """``events``: 7 torch.cuda.Event(enable_timing=True) recorded at the step
    boundaries (before route, after route, load stats, permute, gate/up GEMM,
    down GEMM, combine)."""
    wp, wb = _ws(workspace)
    arr = _event_array(events, stream)
    _check("moe_layer_fwd_profiled", _lib.moe_layer_fwd_profiled(
        _ptr(x), _ptr(w_router), _ptr(bias), _ptr(packed_weights), d, _ptr(out),
        _ptr(topk_idx_out), _ptr(topk_w_out), _ptr(counts_out), wp, wb, _stream(stream), arr,
        len(events)))


def moe_set_wait_limit(cycles: int) -> None:
    """Diagnostics: bounded-wait limit of the GEMM kernels (<= 0: default)."""
    _check("moe_set_wait_limit", _lib.moe_set_wait_limit(int(cycles)))


def moe_read_device_status(workspace, stream=None) -> int:
    v = ctypes.c_int32()
    wp, _ = _ws(workspace)
    _check("moe_read_device_status", _lib.moe_read_device_status(wp, ctypes.addressof(v),
                                                                 _stream(stream)))
    return v.value


# ------------------------------------------------- allocation conveniences ---
# (torch's allocator supplies the memory; the library itself allocates nothing)
def new_workspace(d: moe_dims, device="cuda") -> torch.Tensor:
    """Zeroed workspace of moe_workspace_bytes(d) bytes (256-byte aligned by torch)."""
    n = moe_workspace_bytes(d)
    if n == 0:
        raise MoEError("moe_workspace_bytes", 2)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def prepack(w_gate, w_up, w_down, d, stream=None) -> torch.Tensor:
    packed = torch.empty(moe_packed_weight_bytes(d) // 2, dtype=torch.bfloat16,
                         device=w_gate.device)
    moe_prepack_expert_weights(w_gate, w_up, w_down, d, packed, stream)
    return packed


def layer_forward(x, w_router, bias, packed, d, workspace, stream=None, want_routing=False,
                  opts=None):
    """out [T, H] bf16 (and topk_idx, topk_w, counts if want_routing).  opts: a
    moe_router_opts (router variant, bf16 weights, routing scale) or None."""
    dev = x.device
    out = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev)
    idx = w = counts = None
    if want_routing:
        idx = torch.empty((d.T, d.k), dtype=torch.int32, device=dev)
        w = torch.empty((d.T, d.k), dtype=torch.float32, device=dev)
        counts = torch.empty(d.E, dtype=torch.int32, device=dev)
    moe_layer_fwd_ex(x, w_router, bias, opts, packed, d, out, idx, w, counts, workspace, stream)
    return (out, idx, w, counts) if want_routing else out


def layer_forward_host_batches(x_host_batches, w_router, bias, packed, d, out_host_batches,
                               workspace, stream=None, layer=None):
    """Forward a sequence of token batches that live in pinned host memory, writing each
    batch's output back to pinned host memory.

    Transfers overlap compute: batch i+1 is copied to the device on one copy stream
    while batch i runs (moe_layer_fwd on `stream`, default the current stream), and
    batch i's output is copied back on a second copy stream while batch i+1 runs.
    Two device buffers per direction rotate.  Every batch must have d.T tokens.
    layer: optional callable (x_dev, out_dev, stream) that runs one forward in place
    of moe_layer_fwd (e.g. moe_layer_fwd_sharded with its own arguments bound).
    Returns once all work is enqueued; synchronise `stream` (or the last event) to
    read the outputs.
    """
    compute = torch.cuda.current_stream() if stream is None else stream
    dev = torch.device("cuda", torch.cuda.current_device())
    h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    h2d.wait_stream(compute)  # nothing starts before work already queued on the caller's stream
    x_dev = [torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    o_dev = [torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    copied_in = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    copied_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]
    for i, (xh, oh) in enumerate(zip(x_host_batches, out_host_batches)):
        b = i & 1
        if used[b]:
            h2d.wait_event(computed[b])        # batch i-2 no longer reads x_dev[b]
        with torch.cuda.stream(h2d):
            x_dev[b].copy_(xh, non_blocking=True)
            copied_in[b].record(h2d)
        compute.wait_event(copied_in[b])
        if used[b]:
            compute.wait_event(copied_out[b])  # batch i-2's output has left o_dev[b]
        if layer is None:
            moe_layer_fwd(x_dev[b], w_router, bias, packed, d, o_dev[b], None, None, None,
                          workspace, compute)
        else:
            layer(x_dev[b], o_dev[b], compute)
        computed[b].record(compute)
        d2h.wait_event(computed[b])
        with torch.cuda.stream(d2h):
            oh.copy_(o_dev[b], non_blocking=True)
            copied_out[b].record(d2h)
        used[b] = True
    for e in copied_out:
        compute.wait_event(e)                  # the caller's stream covers the last copies
    for t in x_dev + o_dev:
        t.record_stream(h2d)
        t.record_stream(d2h)
    return compute
