"""Helpers for the GPU tests: move synthetic host inputs to the device, build
packed weights through the library, compare against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import synth

# Layer-output tolerance against the FP32-accumulated oracle.
MAX_ABS = 2e-2
REL_L2 = 5e-3


def routing_weight_rtol(k: int) -> float:
    """Relative bound on |w_gpu - w_oracle| for the softmax router's weights.

    Both sides compute w_j = p_j / S with p_j = exp(l_j - m) / Z and S the left-to-
    right sum of the k selected p.  The logits, m and l_j - m are the same bits on
    both sides.  Z cancels out of the ratio up to the rounding of each p_j, so
    its summation order (lane sums and an xor butterfly on the GPU, ascending on
    the host) does not enter the bound.  With u = 2^-24 (half an ulp, relative), the
    CUDA expf within 2 ulp (4u) and the host exp within 1 ulp (2u), each side's w_j
    is within (e_j + e_max + (k - 1) + 1) u of the exact ratio, where e = exp error
    + the division by Z: GPU (4+1)+(4+1)+k = k + 10, host (2+1)+(2+1)+k = k + 6.
    The two sides differ by at most (2k + 16) u: 1.9e-6 for k = 8, 2.9e-6 for
    k = 16."""
    return (2 * k + 16) * 2.0 ** -24


def assert_routing_weights_close(w: np.ndarray, w_ref: np.ndarray, k: int) -> None:
    w = np.asarray(w, dtype=np.float64)
    w_ref = np.asarray(w_ref, dtype=np.float64)
    bound = routing_weight_rtol(k) * np.abs(w_ref)
    err = np.abs(w - w_ref)
    worst = float((err / np.maximum(np.abs(w_ref), 1e-300)).max()) if err.size else 0.0
    assert np.all(err <= bound), f"routing weight rel. error {worst:.3e} > {routing_weight_rtol(k):.3e}"


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
