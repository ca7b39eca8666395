"""Helpers for the GPU tests: move synthetic host inputs to the device, build
packed weights through the library, compare against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import synth

# Layer-output tolerance against the FP32-accumulated oracle.
MAX_ABS = 2e-2
REL_L2 = 5e-3


def dev_bf16(u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).cuda().view(torch.bfloat16)


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 device tensor -> host uint16 bit patterns."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32(u16: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(u16)


def assert_close(got_bits: np.ndarray, ref_bits: np.ndarray, max_abs=MAX_ABS, rel_l2=REL_L2):
    g = f32(got_bits).astype(np.float64)
    r = f32(ref_bits).astype(np.float64)
    err = np.abs(g - r)
    rl2 = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    assert err.max() <= max_abs, f"max-abs {err.max():.3e} > {max_abs}"
    assert rl2 <= rel_l2, f"rel-L2 {rl2:.3e} > {rel_l2}"
    return err.max(), rl2


def assert_close_f32(got: np.ndarray, ref: np.ndarray, max_abs=MAX_ABS, rel_l2=REL_L2):
    g = got.astype(np.float64)
    r = ref.astype(np.float64)
    err = np.abs(g - r)
    rl2 = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    assert err.max() <= max_abs, f"max-abs {err.max():.3e} > {max_abs}"
    assert rl2 <= rel_l2, f"rel-L2 {rl2:.3e} > {rel_l2}"
    return err.max(), rl2


class DeviceWeights:
    """Expert weights of a workload on the device in the logical layouts, uploaded
    a few experts at a time (host memory stays bounded), plus the packed copy."""

    def __init__(self, wl: synth.Workload, keep_logical: bool = False, chunk: int = 16):
        import moe_expert_layer_fp32_gb300 as moe
        E, H, I = wl.E, wl.H, wl.I
        self.wg = torch.empty((E, H, I), dtype=torch.bfloat16, device="cuda")
        self.wu = torch.empty((E, H, I), dtype=torch.bfloat16, device="cuda")
        self.wd = torch.empty((E, I, H), dtype=torch.bfloat16, device="cuda")
        for e0 in range(0, E, chunk):
            ex = list(range(e0, min(E, e0 + chunk)))
            g, u, d = synth.expert_weights(wl, ex)
            self.wg[e0:e0 + len(ex)].copy_(dev_bf16(g))
            self.wu[e0:e0 + len(ex)].copy_(dev_bf16(u))
            self.wd[e0:e0 + len(ex)].copy_(dev_bf16(d))
        self.dims = moe.dims(wl.T, H, E, wl.k, I)
        self.packed = moe.prepack(self.wg, self.wu, self.wd, self.dims)
        torch.cuda.synchronize()
        if not keep_logical:
            del self.wg, self.wu, self.wd
            torch.cuda.empty_cache()


_cache: dict = {}


def weights(wl: synth.Workload) -> DeviceWeights:
    """Packed device weights of a workload, kept for the next caller with the same
    (E, H, I, w_std, seed); at most one set is held at a time."""
    key = (wl.E, wl.H, wl.I, wl.w_std, wl.seed)
    if key not in _cache:
        _cache.clear()
        torch.cuda.empty_cache()
        _cache[key] = DeviceWeights(wl)
    return _cache[key]
