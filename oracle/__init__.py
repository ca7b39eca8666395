"""CPU oracle for the top-k routed MoE feed-forward layer (TEST INFRASTRUCTURE).

A plain, slow, obviously correct C++ implementation (``oracle.cpp``) of what the
layer computes, wrapped for numpy.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg use it; the library never imports it, and it shares
no code with the CUDA path.  Every function follows the passage cited in
``oracle.cpp``.

Parity pins (what fixes this oracle independently of itself) live in
``tests/test_oracle_pins.py`` and ``tests/golden/``.  The absolute layer values
have no worked example on the pages: they are pinned only through closed forms,
special cases and brute force (the pins file lists which).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (g++, no CUDA, no contraction)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                        os.path.getmtime(__file__))):
            return _LIB_PATH
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O3", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", _SRC, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        lib.oracle_router_logits.argtypes = [vp, vp, vp, i32, i32, i32, vp, i32]
        lib.oracle_route.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, i32]
        lib.oracle_load_stats.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
        lib.oracle_permute.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp]
        lib.oracle_expert_ffn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp, vp, i32]
        lib.oracle_combine.argtypes = [vp, vp, vp, i32, i32, i32, vp, i32]
        lib.oracle_layer_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp,
                                         vp, vp, i32]
        lib.oracle_route_ex.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, i32]
        lib.oracle_combine_scaled.argtypes = [vp, vp, vp, ctypes.c_float, i32, i32, i32, vp, i32]
        lib.oracle_weighted_counts.argtypes = [vp, vp, i32, i32, i32, vp]
        lib.oracle_lpt_placement.argtypes = [vp, i32, i32, vp, vp]
        lib.oracle_rank_metrics.argtypes = [vp, i32, vp, vp]
        lib.oracle_permute_remap.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp]
        for f in ("oracle_weighted_counts", "oracle_lpt_placement", "oracle_rank_metrics",
                  "oracle_permute_remap"):
            getattr(lib, f).restype = ctypes.c_int
        lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        lib.oracle_tree_reduce.argtypes = [vp, i32, ctypes.c_int64, vp]
        lib.oracle_combine_sharded.argtypes = [vp, vp, vp, vp, vp, i32, ctypes.c_float, vp, i32,
                                               i32, i32, i32, vp, vp, i32]
        lib.oracle_shared_expert.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, i32]
        for f in ("oracle_tree_reduce", "oracle_combine_sharded", "oracle_shared_expert"):
            getattr(lib, f).restype = ctypes.c_int
        lib.oracle_exp_cw.argtypes = [ctypes.c_float]
        lib.oracle_exp_cw.restype = ctypes.c_float
        for f in ("oracle_router_logits", "oracle_route", "oracle_load_stats", "oracle_permute",
                  "oracle_expert_ffn", "oracle_combine", "oracle_layer_fwd", "oracle_route_ex",
                  "oracle_combine_scaled"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a):
    return None if a is None else a.ctypes.data


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name}: invalid input (code {rc})")


def router_logits(x, wr, bias=None, nthreads=0):
    """l [T, E] fp32: FP32 FMA chain over ascending h, plus bias (one add)."""
    x = _c(x, np.uint16)
    wr = _c(wr, np.float32)
    bias = None if bias is None else _c(bias, np.float32)
    T, H = x.shape
    E = wr.shape[1]
    out = np.empty((T, E), dtype=np.float32)
    _check(_L().oracle_router_logits(_p(x), _p(wr), _p(bias), T, H, E, _p(out), nthreads),
           "router_logits")
    return out


def route(x, wr, bias, k, nthreads=0):
    """(idx [T, k] int32, w [T, k] fp32)."""
    x = _c(x, np.uint16)
    wr = _c(wr, np.float32)
    bias = None if bias is None else _c(bias, np.float32)
    T, H = x.shape
    E = wr.shape[1]
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    _check(_L().oracle_route(_p(x), _p(wr), _p(bias), T, H, E, k, _p(idx), _p(w), nthreads),
           "route")
    return idx, w


ROUTER_SOFTMAX, ROUTER_SIGMOID = 0, 1


def route_ex(x, wr, bias, k, kind=ROUTER_SOFTMAX, weights_bf16=False, nthreads=0):
    """Router variants: kind 0 softmax (bias joins the logits); kind 1 sigmoid
    scores with `bias` as a selection-only correction bias.  weights_bf16 rounds
    every weight to bf16."""
    x = _c(x, np.uint16)
    wr = _c(wr, np.float32)
    bias = None if bias is None else _c(bias, np.float32)
    T, H = x.shape
    E = wr.shape[1]
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    _check(_L().oracle_route_ex(_p(x), _p(wr), _p(bias), int(kind), int(bool(weights_bf16)), T, H,
                                E, k, _p(idx), _p(w), nthreads), "route_ex")
    return idx, w


def weighted_counts(idx, q, E):
    """int64 [E]: assignments of expert e counted q[t] times (multiplicity weights)."""
    idx = _c(idx, np.int32)
    q = _c(q, np.int32)
    T, k = idx.shape
    out = np.empty(E, dtype=np.int64)
    _check(_L().oracle_weighted_counts(_p(idx), _p(q), T, k, E, _p(out)), "weighted_counts")
    return out


def lpt_placement(loads, P):
    """(slot_of_expert [E] int32, rank_loads [P] int64): layer-local LPT placement."""
    loads = _c(loads, np.int64)
    E = loads.shape[0]
    pi = np.empty(E, dtype=np.int32)
    G = np.empty(P, dtype=np.int64)
    _check(_L().oracle_lpt_placement(_p(loads), E, P, _p(pi), _p(G)), "lpt_placement")
    return pi, G


def rank_metrics(G):
    """(cv, eta_ep) of rank loads."""
    G = _c(G, np.int64)
    cv, eta = ctypes.c_double(), ctypes.c_double()
    _check(_L().oracle_rank_metrics(_p(G), G.shape[0], ctypes.addressof(cv),
                                    ctypes.addressof(eta)), "rank_metrics")
    return cv.value, eta.value


def permute_remap(x, idx, slot_of_expert, offsets, E, with_x_perm=True):
    """permute with logical expert e dispatched to physical slot slot_of_expert[e]."""
    x = _c(x, np.uint16)
    idx = _c(idx, np.int32)
    pi = _c(slot_of_expert, np.int32)
    offsets = _c(offsets, np.int32)
    T, H = x.shape
    k = idx.shape[1]
    R = T * k
    x_perm = np.empty((R, H), dtype=np.uint16) if with_x_perm else None
    ros = np.empty(R, dtype=np.int32)
    sor = np.empty(R, dtype=np.int32)
    _check(_L().oracle_permute_remap(_p(x), _p(idx), _p(pi), _p(offsets), T, H, E, k, _p(x_perm),
                                     _p(ros), _p(sor)), "permute_remap")
    return x_perm, ros, sor


def f64_to_bf16(x: float) -> int:
    """bf16 bits of x rounded once, to nearest even, straight from FP64."""
    return int(_L().oracle_f64_to_bf16(float(x)))


def tree_reduce(partials):
    """out [N] bf16 bits: the fixed FP64 pairwise tree over partials [G, ...] (bf16 bits)."""
    p = _c(partials, np.uint16)
    G = p.shape[0]
    flat = p.reshape(G, -1)
    out = np.empty(flat.shape[1], dtype=np.uint16)
    _check(_L().oracle_tree_reduce(_p(flat), G, flat.shape[1], _p(out)), "tree_reduce")
    return out.reshape(p.shape[1:])


def combine_sharded(y, w, idx, row_of_slot, owner, G, scale=1.0, shared=None, want_partials=False,
                    nthreads=0):
    """out [T, H] bf16 bits (and partials [G, T, H] if want_partials): per-rank
    slot-order chains over the experts each rank owns, FP64 tree across ranks."""
    y = _c(y, np.float32)
    w = _c(w, np.float32)
    idx = _c(idx, np.int32)
    ros = _c(row_of_slot, np.int32).reshape(-1)
    owner = _c(owner, np.int32)
    T, k = w.shape
    H = y.shape[1]
    sh = None if shared is None else _c(shared, np.float32)
    out = np.empty((T, H), dtype=np.uint16)
    parts = np.empty((G, T, H), dtype=np.uint16) if want_partials else None
    _check(_L().oracle_combine_sharded(_p(y), _p(w), _p(idx), _p(ros), _p(owner), int(G),
                                       float(scale), _p(sh), T, H, owner.shape[0], k, _p(parts),
                                       _p(out), nthreads), "combine_sharded")
    return (out, parts) if want_partials else out


def shared_expert(x, wg, wu, wd, G, nthreads=0):
    """shared [G, T, H] FP32: the shared expert's G intermediate-column shards."""
    x = _c(x, np.uint16)
    wg, wu, wd = _c(wg, np.uint16), _c(wu, np.uint16), _c(wd, np.uint16)
    T, H = x.shape
    Is = wg.shape[1]
    out = np.empty((G, T, H), dtype=np.float32)
    _check(_L().oracle_shared_expert(_p(x), _p(wg), _p(wu), _p(wd), T, H, Is, int(G), _p(out),
                                     nthreads), "shared_expert")
    return out


def exp_cw(x: float) -> float:
    return float(_L().oracle_exp_cw(float(x)))


def combine_scaled(y, w, row_of_slot, scale, nthreads=0):
    """out [T, H] bf16 bits, every routing weight multiplied by `scale` first."""
    y = _c(y, np.float32)
    w = _c(w, np.float32)
    ros = _c(row_of_slot, np.int32).reshape(-1)
    T, k = w.shape
    H = y.shape[1]
    out = np.empty((T, H), dtype=np.uint16)
    _check(_L().oracle_combine_scaled(_p(y), _p(w), _p(ros), float(scale), T, H, k, _p(out),
                                      nthreads), "combine_scaled")
    return out


def load_stats(idx, E):
    """(counts [E], offsets [E+1], imbalance max/mean-1, cv)."""
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    imb = ctypes.c_double()
    cv = ctypes.c_double()
    _check(_L().oracle_load_stats(_p(idx), T, k, E, _p(counts), _p(offsets),
                                  ctypes.addressof(imb), ctypes.addressof(cv)), "load_stats")
    return counts, offsets, imb.value, cv.value


def permute(x, idx, offsets, E, with_x_perm=True):
    """(x_perm [T*k, H] bf16 bits or None, row_of_slot [T*k], slot_of_row [T*k])."""
    x = _c(x, np.uint16)
    idx = _c(idx, np.int32)
    offsets = _c(offsets, np.int32)
    T, H = x.shape
    k = idx.shape[1]
    R = T * k
    x_perm = np.empty((R, H), dtype=np.uint16) if with_x_perm else None
    ros = np.empty(R, dtype=np.int32)
    sor = np.empty(R, dtype=np.int32)
    _check(_L().oracle_permute(_p(x), _p(idx), _p(offsets), T, H, E, k, _p(x_perm), _p(ros),
                               _p(sor)), "permute")
    return x_perm, ros, sor


def expert_ffn(x_perm, offsets, wg, wu, wd, want_h=False, nthreads=0):
    """y [R, H] fp32 (and h [R, I] bf16 bits if want_h)."""
    x_perm = _c(x_perm, np.uint16)
    offsets = _c(offsets, np.int32)
    wg, wu, wd = _c(wg, np.uint16), _c(wu, np.uint16), _c(wd, np.uint16)
    E, H, I = wg.shape
    R = int(offsets[E])
    y = np.empty((R, H), dtype=np.float32)
    h = np.empty((R, I), dtype=np.uint16) if want_h else None
    _check(_L().oracle_expert_ffn(_p(x_perm), _p(offsets), _p(wg), _p(wu), _p(wd), E, H, I, _p(h),
                                  _p(y), nthreads), "expert_ffn")
    return (y, h) if want_h else y


def combine(y, w, row_of_slot, nthreads=0):
    """out [T, H] bf16 bits."""
    y = _c(y, np.float32)
    w = _c(w, np.float32)
    ros = _c(row_of_slot, np.int32).reshape(-1)
    T, k = w.shape
    H = y.shape[1]
    out = np.empty((T, H), dtype=np.uint16)
    _check(_L().oracle_combine(_p(y), _p(w), _p(ros), T, H, k, _p(out), nthreads), "combine")
    return out


def layer_fwd(x, wr, bias, wg, wu, wd, k, nthreads=0):
    """(out [T, H] bf16 bits, idx [T, k], w [T, k], counts [E])."""
    x = _c(x, np.uint16)
    wr = _c(wr, np.float32)
    bias = None if bias is None else _c(bias, np.float32)
    wg, wu, wd = _c(wg, np.uint16), _c(wu, np.uint16), _c(wd, np.uint16)
    T, H = x.shape
    E, _, I = wg.shape
    out = np.empty((T, H), dtype=np.uint16)
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    counts = np.empty(E, dtype=np.int32)
    _check(_L().oracle_layer_fwd(_p(x), _p(wr), _p(bias), _p(wg), _p(wu), _p(wd), T, H, E, k, I,
                                 _p(out), _p(idx), _p(w), _p(counts), nthreads), "layer_fwd")
    return out, idx, w, counts
