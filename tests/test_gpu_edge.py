"""Edge cases and device-side checks of the CUDA path: empty batches, a single
token, ragged tails, degenerate expert counts (E = 1, k = E), the largest E, k
and H, caller-supplied routing, and malformed indices/offsets that the kernels must
flag instead of touching memory out of range."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (DeviceWeights, assert_close, assert_routing_weights_close, bits, dev,
                      dev_bf16, weights)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_ok):
    import moe_expert_layer_fp32_gb300 as m
    return m


def layer_vs_oracle(moe, wl, T=None):
    W = weights(wl)
    x = synth.tokens(wl, T)
    wr, bias = synth.router(wl)
    d = moe.dims(x.shape[0], wl.H, wl.E, wl.k, wl.I)
    ws = moe.new_workspace(d)
    out, idx, w, counts = moe.layer_forward(dev_bf16(x), dev(wr),
                                            None if bias is None else dev(bias), W.packed, d, ws,
                                            want_routing=True)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    wg, wu, wd = synth.expert_weights(wl)
    out_o, idx_o, w_o, counts_o = oracle.layer_fwd(x, wr, bias, wg, wu, wd, wl.k)
    np.testing.assert_array_equal(idx.cpu().numpy(), idx_o)
    np.testing.assert_array_equal(counts.cpu().numpy(), counts_o)
    assert_close(bits(out), out_o)
    return w.cpu().numpy(), w_o


def test_empty_batch_is_noop(moe):
    d = moe.dims(0, 128, 8, 2, 256)
    ws = moe.new_workspace(d)
    wl = synth.Workload("e", T=0, H=128, E=8, k=2, I=256, w_std=0.02)
    W = DeviceWeights(synth.Workload("e", T=1, H=128, E=8, k=2, I=256, w_std=0.02))
    wr, _ = synth.router(wl)
    counts = torch.full((8,), 7, dtype=torch.int32, device="cuda")
    out = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    moe.moe_layer_fwd(None, dev(wr), None, W.packed, d, out, None, None, counts, ws)
    torch.cuda.synchronize()
    assert counts.cpu().tolist() == [0] * 8
    offsets = torch.full((9,), 7, dtype=torch.int32, device="cuda")
    moe.moe_load_stats(None, d, counts, offsets, ws)
    assert offsets.cpu().tolist() == [0] * 9
    assert moe.moe_read_device_status(ws) == 0


@pytest.mark.parametrize("T", [1, 3, 300])
def test_single_token_and_ragged_tails(moe, T):
    wl = synth.Workload("ragged", T=T, H=256, E=16, k=4, I=384, w_std=0.05, zipf_s=1.0)
    layer_vs_oracle(moe, wl)


def test_single_expert_is_dense_ffn(moe):
    wl = synth.Workload("dense", T=200, H=128, E=1, k=1, I=256, w_std=0.05)
    w, _ = layer_vs_oracle(moe, wl)
    assert np.all(w == 1.0)


def test_k_equals_E(moe):
    wl = synth.Workload("all", T=130, H=128, E=8, k=8, I=128, w_std=0.05)
    w, w_o = layer_vs_oracle(moe, wl)
    assert_routing_weights_close(w, w_o, wl.k)


def test_max_experts_and_k(moe):
    wl = synth.Workload("max", T=777, H=128, E=256, k=16, I=128, w_std=0.05, wr_std=0.5)
    layer_vs_oracle(moe, wl)


@pytest.mark.parametrize("name,T,E,k", [("one_expert", 5, 1, 1), ("k_is_E", 2, 8, 8),
                                        ("max_E_k", 8, 256, 16)])
def test_degenerate_shapes_in_swapped_form(moe, name, T, E, k):
    """The same degenerate expert counts at H = 256, where small batches run the
    GEMMs with the weight rows on the MMA's M side."""
    wl = synth.Workload(name, T=T, H=256, E=E, k=k, I=128, w_std=0.05, wr_std=0.5)
    assert moe.moe_expert_ffn_form(moe.dims(T, wl.H, E, k, wl.I)) == 1
    layer_vs_oracle(moe, wl)


@pytest.mark.parametrize("T", [2, 300])
def test_largest_hidden_size(moe, T):
    """H = 16384, the library's largest hidden size: 256 k-blocks per GEMM tile and
    the router's longest FMA chains, in the swapped form (T = 2) and the tile form
    (T = 300)."""
    wl = synth.Workload("wide_h", T=T, H=16384, E=4, k=2, I=256, w_std=0.01, wr_std=0.01)
    assert moe.moe_expert_ffn_form(moe.dims(T, wl.H, wl.E, wl.k, wl.I)) == (1 if T == 2 else 0)
    layer_vs_oracle(moe, wl)


def test_caller_supplied_routing(moe):
    """Router replay: permute, expert FFN and combine driven by indices and
    weights that did not come from moe_route (here: uniform random distinct
    experts, random weights)."""
    T, H, E, k, I = 500, 256, 12, 3, 256
    wl = synth.Workload("replay", T=T, H=H, E=E, k=k, I=I, w_std=0.05)
    keys = synth.uniform_f32(3, synth.TID_TOPK_IDX, (T, E), 0.0, 1.0)
    idx = np.argsort(keys, axis=1)[:, :k].astype(np.int32)
    w = synth.uniform_f32(3, synth.TID_TOPK_W, (T, k), 0.0, 1.0)
    x = synth.tokens(wl)
    counts, offsets, _, _ = oracle.load_stats(idx, E)
    xp_o, ros_o, _ = oracle.permute(x, idx, offsets, E)
    wg, wu, wd = synth.expert_weights(wl)
    y_o = oracle.expert_ffn(xp_o, offsets, wg, wu, wd)
    out_o = oracle.combine(y_o, w, ros_o)
    d = moe.dims(T, H, E, k, I)
    ws = moe.new_workspace(d)
    W = weights(wl)
    R = T * k
    xp = torch.empty((R, H), dtype=torch.bfloat16, device="cuda")
    ros = torch.empty(R, dtype=torch.int32, device="cuda")
    sor = torch.empty(R, dtype=torch.int32, device="cuda")
    moe.moe_permute(dev_bf16(x), dev(idx), dev(offsets), d, xp, ros, sor, ws)
    y = torch.empty((R, H), dtype=torch.float32, device="cuda")
    moe.moe_expert_ffn(xp, dev(offsets), W.packed, d, y, ws)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(y, dev(w), ros, d, out)
    assert moe.moe_read_device_status(ws) == 0
    np.testing.assert_array_equal(ros.cpu().numpy(), ros_o)
    assert_close(bits(out), out_o)


def test_bad_indices_are_flagged_not_followed(moe):
    """An out-of-range expert id and a repeated expert in one token: counted out,
    flagged as MOE_ERR_DEVICE_CHECK, no out-of-range access."""
    T, H, E, k, I = 64, 128, 8, 2, 128
    d = moe.dims(T, H, E, k, I)
    idx = np.tile(np.array([[0, 1]], np.int32), (T, 1))
    idx[5, 1] = 99
    ws = moe.new_workspace(d)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    moe.moe_load_stats(dev(idx), d, counts, offsets, ws)
    assert moe.moe_read_device_status(ws) == 7
    assert counts.cpu().tolist()[:2] == [64, 63]
    idx[5, 1] = 0  # repeated expert
    moe.moe_load_stats(dev(idx), d, counts, offsets, ws)
    assert moe.moe_read_device_status(ws) == 7


def test_bad_offsets_are_flagged_and_nothing_written(moe):
    T, H, E, k, I = 64, 128, 4, 2, 128
    wl = synth.Workload("bad", T=T, H=H, E=E, k=k, I=I, w_std=0.05)
    d = moe.dims(T, H, E, k, I)
    W = weights(wl)
    ws = moe.new_workspace(d)
    R = T * k
    xp = dev_bf16(synth.normal_bf16(0, synth.TID_X_PERM, (R, H), 1.0))
    sentinel = 12345.0
    for bad in ([0, 40, 30, 100, R], [0, 40, 80, 100, R + 500], [5, 40, 80, 100, R]):
        y = torch.full((R, H), sentinel, dtype=torch.float32, device="cuda")
        moe.moe_expert_ffn(xp, dev(np.array(bad, np.int32)), W.packed, d, y, ws)
        assert moe.moe_read_device_status(ws) == 7
        assert bool((y == sentinel).all())


def test_combine_skips_rows_out_of_range(moe):
    T, H, k = 8, 128, 2
    d = moe.dims(T, H, 4, k, 128)
    y = synth.normal_f32(1, synth.TID_Y, (T * k, H), 1.0)
    ros = np.arange(T * k, dtype=np.int32)
    ros[3] = T * k + 1000
    ros[4] = -7
    w = np.ones((T, k), np.float32)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(dev(y), dev(w), dev(ros), d, out)
    ros_ok = ros.copy()
    y_ext = np.concatenate([y, np.zeros((1, H), np.float32)])
    ros_ok[3] = ros_ok[4] = T * k  # the zero row
    np.testing.assert_array_equal(bits(out), oracle.combine(y_ext, w, ros_ok))
