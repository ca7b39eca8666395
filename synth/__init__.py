"""Seeded synthetic inputs for the top-k routed MoE feed-forward layer.

This module holds random-number generation and the workload recipes only; it
contains none of the layer's arithmetic.  It is the one module that serves both
the CPU oracle (via the tests) and the CUDA path (via the tests, the smoke check
and the benchmark).  The generator itself is ``synth.c`` (counter-based
SplitMix64 + Box-Muller), compiled here on first use.

Workloads (shapes and value distributions of the synthetic MoE layers):

* ``tiny``          T=256,  H=128,  E=8,   k=2, I=256, weights ~N(0, 0.02), uniform router
* ``fine_grained``  T=4096, H=2048, E=64,  k=8, I=1024, weights ~N(0, 0.02),
                    router logits plus a Zipf(s=1.0) per-expert bias
* ``packed_rl``     T=16384 (one packed row of lognormal-length sequences),
                    H=2048, E=128, k=8, I=768, Zipf(s=1.2) bias
* ``large``         T=32768, H=4096, E=256, k=8, I=2048, weights ~N(0, 0.01), uniform router
* ``decode``        the ``fine_grained`` layer at T in {1, 8, 64, 512, 4096}; each
                    batch is a prefix of the T=4096 tokens

In all of them x ~ N(0, 1) in bf16 and the router weight W_r ~ N(0, 0.02) in fp32.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

# Counter streams, one per tensor.
TID_X, TID_WR, TID_WG, TID_WU, TID_WD, TID_LENGTHS = 1, 2, 3, 4, 5, 6
# Streams used only by tests that drive one step in isolation.
TID_Y, TID_TOPK_W, TID_TOPK_IDX, TID_X_PERM, TID_MISC = 7, 8, 9, 10, 11
TID_SWG, TID_SWU, TID_SWD = 12, 13, 14  # shared-expert weights


def build(force: bool = False) -> str:
    """Compile libsynth.so next to its source (gcc, no CUDA)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                        os.path.getmtime(__file__))):
            return _LIB_PATH
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, u32, i32, i64, dbl, vp = (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32,
                                       ctypes.c_int64, ctypes.c_double, ctypes.c_void_p)
        lib.synth_normal_bf16.argtypes = [u64, u32, u64, u64, dbl, vp, ctypes.c_int]
        lib.synth_normal_f32.argtypes = [u64, u32, u64, u64, dbl, vp, ctypes.c_int]
        lib.synth_uniform_f32.argtypes = [u64, u32, u64, u64, dbl, dbl, vp, ctypes.c_int]
        lib.synth_uniform_i32.argtypes = [u64, u32, u64, u64, i64, i64, vp, ctypes.c_int]
        lib.synth_zipf_bias.argtypes = [i32, dbl, dbl, vp]
        lib.synth_packed_lengths.argtypes = [u64, u32, dbl, dbl, i32, i32, i32, vp, i32]
        lib.synth_packed_lengths.restype = i32
        for f in ("synth_normal_bf16", "synth_normal_f32", "synth_uniform_f32",
                  "synth_uniform_i32", "synth_zipf_bias"):
            getattr(lib, f).restype = None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------- raw fills ---
def fill_normal_bf16(addr: int, seed: int, tid: int, start: int, count: int, std: float,
                     nthreads: int = 0) -> None:
    """Write ``count`` bf16 bit patterns to host address ``addr``."""
    _L().synth_normal_bf16(seed, tid, start, count, std, addr, nthreads)


def normal_bf16(seed: int, tid: int, shape, std: float, start: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    _L().synth_normal_bf16(seed, tid, start, out.size, std, _ptr(out), 0)
    return out


def normal_f32(seed: int, tid: int, shape, std: float, start: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _L().synth_normal_f32(seed, tid, start, out.size, std, _ptr(out), 0)
    return out


def uniform_f32(seed: int, tid: int, shape, lo: float, hi: float, start: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _L().synth_uniform_f32(seed, tid, start, out.size, lo, hi, _ptr(out), 0)
    return out


def uniform_i32(seed: int, tid: int, shape, lo: int, hi: int, start: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.int32)
    _L().synth_uniform_i32(seed, tid, start, out.size, lo, hi, _ptr(out), 0)
    return out


def zipf_bias(E: int, s: float, coef: float = 1.5) -> np.ndarray:
    out = np.empty(E, dtype=np.float32)
    _L().synth_zipf_bias(E, s, coef, _ptr(out))
    return out


def packed_lengths(seed: int, row_tokens: int, mu: float = 7.0, sigma: float = 1.0,
                   lo: int = 64, hi: int = 8192) -> np.ndarray:
    """cu_seqlens of one packed row (metadata only: the MoE layer is token-wise)."""
    cu = np.empty(row_tokens + 1, dtype=np.int32)
    n = _L().synth_packed_lengths(seed, TID_LENGTHS, mu, sigma, lo, hi, row_tokens, _ptr(cu),
                                  row_tokens)
    if n < 0:
        raise RuntimeError("packed_lengths: too many sequences")
    return cu[: n + 1].copy()


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (a reinterpretation, no rounding)."""
    return (u16.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- workloads ---
@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    w_std: float           # expert weights W_gate, W_up, W_down
    wr_std: float = 0.02   # router weight
    zipf_s: float = 0.0    # 0: no bias; otherwise b_e = 1.5*ln(Zipf(s) rank weight)
    zipf_coef: float = 1.5
    seed: int = 0
    packed: bool = False   # tokens form one packed row of lognormal-length sequences

    def dims(self, T: int | None = None):
        return dict(T=self.T if T is None else T, H=self.H, E=self.E, k=self.k, I=self.I)


WORKLOADS = {
    "tiny": Workload("tiny", T=256, H=128, E=8, k=2, I=256, w_std=0.02),
    "fine_grained": Workload("fine_grained", T=4096, H=2048, E=64, k=8, I=1024, w_std=0.02,
                             zipf_s=1.0),
    "packed_rl": Workload("packed_rl", T=16384, H=2048, E=128, k=8, I=768, w_std=0.02,
                          zipf_s=1.2, packed=True),
    "large": Workload("large", T=32768, H=4096, E=256, k=8, I=2048, w_std=0.01),
    # the MoE layer of Ling-3.0-tiny (HARTS, Table 1): hidden 1,536, 128 experts,
    # top-8, expert intermediate 512; a packed RL micro-batch of 16,384 rows; no
    # popularity bias (HARTS keeps expert loads balanced through its loss and bias
    # updates)
    "ling3_tiny": Workload("ling3_tiny", T=16384, H=1536, E=128, k=8, I=512, w_std=0.02,
                           packed=True),
}
DECODE_T = (1, 8, 64, 512, 4096)   # the fine_grained layer at these batch sizes


def tokens(wl: Workload, T: int | None = None, rows: np.ndarray | None = None) -> np.ndarray:
    """x [T, H] bf16 bits (or only the given token rows).  Token t of any batch is
    the same bytes, so smaller batches are prefixes of larger ones."""
    H = wl.H
    if rows is None:
        T = wl.T if T is None else T
        return normal_bf16(wl.seed, TID_X, (T, H), 1.0)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((len(rows), H), dtype=np.uint16)
    for i, t in enumerate(rows):
        _L().synth_normal_bf16(wl.seed, TID_X, int(t) * H, H, 1.0, _ptr(out[i]), 1)
    return out


def router(wl: Workload):
    """(W_r [H, E] fp32, bias [E] fp32 or None)."""
    wr = normal_f32(wl.seed, TID_WR, (wl.H, wl.E), wl.wr_std)
    bias = zipf_bias(wl.E, wl.zipf_s, wl.zipf_coef) if wl.zipf_s > 0 else None
    return wr, bias


def expert_weights(wl: Workload, experts=None):
    """(W_gate [n, H, I], W_up [n, H, I], W_down [n, I, H]) bf16 bits for the given
    experts (all E by default), in the logical row-major layouts."""
    E, H, I = wl.E, wl.H, wl.I
    experts = list(range(E)) if experts is None else [int(e) for e in experts]
    n = len(experts)
    wg = np.empty((n, H, I), dtype=np.uint16)
    wu = np.empty((n, H, I), dtype=np.uint16)
    wd = np.empty((n, I, H), dtype=np.uint16)
    contiguous = experts == list(range(experts[0], experts[0] + n)) if n else True
    if contiguous and n:
        e0 = experts[0]
        _L().synth_normal_bf16(wl.seed, TID_WG, e0 * H * I, n * H * I, wl.w_std, _ptr(wg), 0)
        _L().synth_normal_bf16(wl.seed, TID_WU, e0 * H * I, n * H * I, wl.w_std, _ptr(wu), 0)
        _L().synth_normal_bf16(wl.seed, TID_WD, e0 * I * H, n * I * H, wl.w_std, _ptr(wd), 0)
    else:
        for i, e in enumerate(experts):
            _L().synth_normal_bf16(wl.seed, TID_WG, e * H * I, H * I, wl.w_std, _ptr(wg[i]), 0)
            _L().synth_normal_bf16(wl.seed, TID_WU, e * H * I, H * I, wl.w_std, _ptr(wu[i]), 0)
            _L().synth_normal_bf16(wl.seed, TID_WD, e * I * H, I * H, wl.w_std, _ptr(wd[i]), 0)
    return wg, wu, wd


def shared_expert_weights(wl: Workload, Is: int, std: float | None = None):
    """(W_gate [H, Is], W_up [H, Is], W_down [Is, H]) bf16 bits of a shared expert
    of intermediate size Is for the workload's hidden size."""
    std = wl.w_std if std is None else std
    return (normal_bf16(wl.seed, TID_SWG, (wl.H, Is), std),
            normal_bf16(wl.seed, TID_SWU, (wl.H, Is), std),
            normal_bf16(wl.seed, TID_SWD, (Is, wl.H), std))


def layer_inputs(wl: Workload, T: int | None = None) -> dict:
    """Every input of one layer forward as host numpy arrays (bf16 as uint16 bits)."""
    wr, bias = router(wl)
    wg, wu, wd = expert_weights(wl)
    out = dict(x=tokens(wl, T), wr=wr, bias=bias, wg=wg, wu=wu, wd=wd)
    if wl.packed:
        out["cu_seqlens"] = packed_lengths(wl.seed, wl.T if T is None else T)
    return out
