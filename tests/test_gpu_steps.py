"""Per-step parity of the CUDA path (through the C ABI) against the CPU oracle on
the synthetic workloads.  Each step gets the same seeded inputs on both sides;
no oracle input comes from the GPU.

  route       indices bit-exact, weights within a few FP32 ulp
  load stats  counts and offsets bit-exact
  permute     x_perm, row_of_slot, slot_of_row bit-exact
  expert FFN  y within the layer tolerance (max-abs 2e-2, rel-L2 5e-3)
  combine     bit-exact given the same y
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (DeviceWeights, assert_close_f32, assert_routing_weights_close, bits, dev,
                      dev_bf16, weights)

pytestmark = pytest.mark.gpu

NAMES = ["tiny", "fine_grained", "packed_rl", "large"]


@pytest.fixture(scope="module")
def moe(cuda_ok):
    import moe_expert_layer_fp32_gb300 as m
    return m


@pytest.fixture(scope="module", params=NAMES)
def case(request, moe):
    wl = synth.WORKLOADS[request.param]
    x = synth.tokens(wl)
    wr, bias = synth.router(wl)
    idx, w = oracle.route(x, wr, bias, wl.k)
    counts, offsets, _, _ = oracle.load_stats(idx, wl.E)
    yield dict(wl=wl, x=x, wr=wr, bias=bias, idx=idx, w=w, counts=counts, offsets=offsets,
               d=moe.dims(wl.T, wl.H, wl.E, wl.k, wl.I))
    torch.cuda.empty_cache()


def test_route(moe, case):
    wl, d = case["wl"], case["d"]
    idx = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, wl.k), dtype=torch.float32, device="cuda")
    bias = None if case["bias"] is None else dev(case["bias"])
    moe.moe_route(dev_bf16(case["x"]), dev(case["wr"]), bias, d, idx, w)
    np.testing.assert_array_equal(idx.cpu().numpy(), case["idx"])
    assert_routing_weights_close(w.cpu().numpy(), case["w"], wl.k)


def test_load_stats(moe, case):
    wl, d = case["wl"], case["d"]
    ws = moe.new_workspace(d)
    counts = torch.empty(wl.E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(wl.E + 1, dtype=torch.int32, device="cuda")
    moe.moe_load_stats(dev(case["idx"]), d, counts, offsets, ws)
    np.testing.assert_array_equal(counts.cpu().numpy(), case["counts"])
    np.testing.assert_array_equal(offsets.cpu().numpy(), case["offsets"])
    assert moe.moe_read_device_status(ws) == 0
    imb, cv = moe.moe_load_summary_host(counts.cpu().numpy())
    _, _, imb_o, cv_o = oracle.load_stats(case["idx"], wl.E)
    assert imb == pytest.approx(imb_o, rel=1e-12) and cv == pytest.approx(cv_o, rel=1e-12)


def test_permute(moe, case):
    wl, d = case["wl"], case["d"]
    R = wl.T * wl.k
    ws = moe.new_workspace(d)
    xp = torch.empty((R, wl.H), dtype=torch.bfloat16, device="cuda")
    ros = torch.empty(R, dtype=torch.int32, device="cuda")
    sor = torch.empty(R, dtype=torch.int32, device="cuda")
    moe.moe_permute(dev_bf16(case["x"]), dev(case["idx"]), dev(case["offsets"]), d, xp, ros, sor, ws)
    xp_o, ros_o, sor_o = oracle.permute(case["x"], case["idx"], case["offsets"], wl.E)
    np.testing.assert_array_equal(ros.cpu().numpy(), ros_o)
    np.testing.assert_array_equal(sor.cpu().numpy(), sor_o)
    np.testing.assert_array_equal(bits(xp), xp_o)
    assert moe.moe_read_device_status(ws) == 0


def _ffn_subproblem(case, experts):
    """Rows of the given experts as a self-contained grouped problem."""
    offs = case["offsets"]
    sizes = [int(offs[e + 1] - offs[e]) for e in experts]
    sub_off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = np.concatenate([np.arange(offs[e], offs[e + 1]) for e in experts]).astype(np.int64)
    return rows, sub_off


def test_expert_ffn(moe, case):
    wl, d = case["wl"], case["d"]
    R = wl.T * wl.k
    ws = moe.new_workspace(d)
    W = weights(wl)
    xp = synth.normal_bf16(wl.seed, synth.TID_X_PERM, (R, wl.H), 1.0)
    y = torch.empty((R, wl.H), dtype=torch.float32, device="cuda")
    moe.moe_expert_ffn(dev_bf16(xp), dev(case["offsets"]), W.packed, d, y, ws)
    assert moe.moe_read_device_status(ws) == 0
    counts = case["counts"]
    active = [e for e in range(wl.E) if counts[e] > 0]
    if wl.name in ("tiny", "fine_grained"):
        experts = list(range(wl.E))
    else:  # the busiest, a median and the last active expert: every row of each
        by_load = sorted(active, key=lambda e: -counts[e])
        experts = sorted({by_load[0], by_load[len(by_load) // 2], active[-1]})
        if wl.name == "packed_rl":
            experts = sorted({by_load[1], by_load[len(by_load) // 2], active[-1]})
    rows, sub_off = _ffn_subproblem(case, experts)
    wg, wu, wd = synth.expert_weights(wl, experts)
    y_o = oracle.expert_ffn(xp[rows], sub_off, wg, wu, wd)
    y_g = y[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert_close_f32(y_g, y_o)
    # per-row relative error stays small too (no row silently wrong)
    rel = np.linalg.norm(y_g - y_o, axis=1) / np.maximum(np.linalg.norm(y_o, axis=1), 1e-30)
    assert rel.max() < 2e-2


def test_combine(moe, case):
    wl, d = case["wl"], case["d"]
    R = wl.T * wl.k
    y = synth.normal_f32(wl.seed, synth.TID_Y, (R, wl.H), 1.0)
    _, ros_o, _ = oracle.permute(case["x"], case["idx"], case["offsets"], wl.E, with_x_perm=False)
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(dev(y), dev(case["w"]), dev(ros_o), d, out)
    np.testing.assert_array_equal(bits(out), oracle.combine(y, case["w"], ros_o))


def test_route_kernels_agree_bitwise(moe):
    """Three router kernels: CTA clusters (1 to 8 tokens each) up to 1024 tokens,
    1D tiles, and (256 experts) 2D tiles once every SM gets a CTA (T >= 32 x SMs,
    4864 on 152 SMs).  Every logit is the same FMA chain in all of them, so a
    token's experts and weights must be the same bits whichever kernel ran."""
    wl = synth.WORKLOADS["large"]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Ts = (5, 64, 65, 1024, 1025, 32 * sms - 1, 32 * sms + 96)
    x = synth.tokens(wl, Ts[-1])
    wr, bias = synth.router(wl)
    got = []
    for T in Ts:
        d = moe.dims(T, wl.H, wl.E, wl.k, wl.I)
        idx = torch.empty((T, wl.k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, wl.k), dtype=torch.float32, device="cuda")
        moe.moe_route(dev_bf16(x[:T]), dev(wr), None if bias is None else dev(bias), d, idx, w)
        got.append((idx.cpu().numpy(), w.cpu().numpy()))
    big_idx, big_w = got[-1]
    for T, (idx, w) in zip(Ts[:-1], got[:-1]):
        np.testing.assert_array_equal(idx, big_idx[:T])
        np.testing.assert_array_equal(w.view(np.uint32), big_w[:T].view(np.uint32))



@pytest.mark.parametrize("E,H", [(64, 1024), (68, 1024), (100, 1024), (200, 1024), (66, 1024),
                                 (64, 1152), (256, 640)])
def test_decode_router_matches_cluster_router(moe, E, H):
    """Up to eight tokens run the sixteen-CTA router fed by tensor copies; expert
    counts that leave the last CTAs partly or wholly past E (68, 100, 200), one
    whose W_r rows are not 16-byte multiples (66: the cp.async form) and hidden
    sizes whose last stage is short (1152, 640) must give the bits of the cluster
    router that runs from nine tokens, and the oracle's."""
    wl = synth.Workload("decode_route", T=64, H=H, E=E, k=8, I=128, w_std=0.05)
    x = synth.tokens(wl)
    wr, bias = synth.router(wl)
    def route(T):
        d = moe.dims(T, wl.H, wl.E, wl.k, wl.I)
        idx = torch.empty((T, wl.k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, wl.k), dtype=torch.float32, device="cuda")
        moe.moe_route(dev_bf16(x[:T]), dev(wr), None if bias is None else dev(bias), d, idx, w)
        return idx.cpu().numpy(), w.cpu().numpy()
    ref_idx, ref_w = route(64)
    for T in (1, 2, 3, 5, 8):
        idx, w = route(T)
        np.testing.assert_array_equal(idx, ref_idx[:T])
        np.testing.assert_array_equal(w.view(np.uint32), ref_w[:T].view(np.uint32))
    idx_o, w_o = oracle.route(x[:8], wr, bias, wl.k)
    np.testing.assert_array_equal(route(8)[0], idx_o)
