"""Router variants and the routing scale on the GPU against the oracle.

  sigmoid router (GLM's rule: correction bias only selects, weights from the
  pre-bias scores): indices AND weights bit-exact in both router kernels (the
  exponential is the same Cody-Waite/Taylor steps on both sides);
  bf16 weight cast: indices bit-exact; softmax weights within one bf16 ulp
  (the FP32 softmax weights already differ by a few FP32 ulp);
  routing scale in the combine: bit-exact given the same y;
  whole layer with GLM options: indices bit-exact, output within tolerance,
  bitwise batch-invariant across T.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close, bits, dev, dev_bf16, weights

pytestmark = pytest.mark.gpu

SIG = oracle.ROUTER_SIGMOID


@pytest.fixture(scope="module")
def moe(cuda_ok):
    import moe_expert_layer_fp32_gb300 as m
    return m


def corr_bias(E, seed=7):
    return synth.uniform_f32(seed, synth.TID_MISC, (E,), -0.05, 0.05)


def gpu_route(moe, x, wr, bias, d, opts):
    idx = torch.empty((d.T, d.k), dtype=torch.int32, device="cuda")
    w = torch.empty((d.T, d.k), dtype=torch.float32, device="cuda")
    moe.moe_route_ex(dev_bf16(x), dev(wr), None if bias is None else dev(bias), opts, d, idx, w)
    return idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("name,T", [("fine_grained", 4096), ("fine_grained", 700),
                                    ("fine_grained", 64), ("fine_grained", 3), ("large", 2048),
                                    ("large", 5000), ("tiny", 256)])
@pytest.mark.parametrize("wbf16", [False, True])
def test_sigmoid_router_bit_exact(moe, name, T, wbf16):
    wl = synth.WORKLOADS[name]
    x = synth.tokens(wl, T)
    wr, _ = synth.router(wl)
    b = corr_bias(wl.E)
    d = moe.dims(T, wl.H, wl.E, wl.k, wl.I)
    idx, w = gpu_route(moe, x, wr, b, d, moe.router_opts(moe.MOE_ROUTER_SIGMOID_BIAS_SELECT, wbf16))
    idx_o, w_o = oracle.route_ex(x, wr, b, wl.k, kind=SIG, weights_bf16=wbf16)
    np.testing.assert_array_equal(idx, idx_o)
    np.testing.assert_array_equal(w.view(np.uint32), w_o.view(np.uint32))


def test_sigmoid_router_bias_flips_choice_on_gpu(moe):
    """The hand-built case of the oracle pins: logits 0..3, bias [1,0,0,0]."""
    x = np.full((1, 128), 0, np.uint16)
    x[0, 0] = 0x3F80  # 1.0
    wr = np.zeros((128, 32), np.float32)
    wr[0, :4] = [0.0, 1.0, 2.0, 3.0]
    wr[0, 4:] = -20.0
    b = np.zeros(32, np.float32)
    b[0] = 1.0
    d = moe.dims(1, 128, 32, 2, 128)
    idx, w = gpu_route(moe, x, wr, b, d, moe.router_opts(moe.MOE_ROUTER_SIGMOID_BIAS_SELECT))
    assert idx.tolist() == [[0, 3]]
    idx_o, w_o = oracle.route_ex(x, wr, b, 2, kind=SIG)
    np.testing.assert_array_equal(w.view(np.uint32), w_o.view(np.uint32))


@pytest.mark.parametrize("T", [64, 4096])
def test_softmax_router_bf16_weights(moe, T):
    wl = synth.WORKLOADS["fine_grained"]
    x = synth.tokens(wl, T)
    wr, bias = synth.router(wl)
    d = moe.dims(T, wl.H, wl.E, wl.k, wl.I)
    idx, w = gpu_route(moe, x, wr, bias, d, moe.router_opts(weights_bf16=True))
    idx_o, w_o = oracle.route_ex(x, wr, bias, wl.k, weights_bf16=True)
    np.testing.assert_array_equal(idx, idx_o)
    assert np.all((w.view(np.uint32) & 0xFFFF) == 0)  # bf16 values
    np.testing.assert_allclose(w, w_o, rtol=2.0 ** -7, atol=0)  # one bf16 ulp


def test_combine_route_scale_bit_exact(moe):
    wl = synth.WORKLOADS["packed_rl"]
    T, R = 2048, 2048 * wl.k
    y = synth.normal_f32(2, synth.TID_Y, (R, wl.H), 1.0)
    w = synth.uniform_f32(2, synth.TID_TOPK_W, (T, wl.k), 0.0, 1.0)
    ros = np.random.default_rng(3).permutation(R).astype(np.int32)
    d = moe.dims(T, wl.H, wl.E, wl.k, wl.I)
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine_ex(dev(y), dev(w), dev(ros), 2.5, d, out)
    np.testing.assert_array_equal(bits(out), oracle.combine_scaled(y, w, ros.reshape(T, -1), 2.5))


def _glm_layer_oracle(wl, x, wr, b, opts_bf16=False):
    idx, w = oracle.route_ex(x, wr, b, wl.k, kind=SIG, weights_bf16=opts_bf16)
    counts, offs, _, _ = oracle.load_stats(idx, wl.E)
    experts = np.flatnonzero(counts)
    wg, wu, wd = synth.expert_weights(wl, experts)
    remap = np.full(wl.E, -1, np.int64)
    remap[experts] = np.arange(len(experts))
    sidx = remap[idx].astype(np.int32)
    _, soffs, _, _ = oracle.load_stats(sidx, len(experts))
    xp, ros, _ = oracle.permute(x, sidx, soffs, len(experts))
    y = oracle.expert_ffn(xp, soffs, wg, wu, wd)
    return oracle.combine_scaled(y, w, ros, 2.5), idx


def test_glm_layer_and_batch_invariance(moe):
    wl = synth.WORKLOADS["fine_grained"]
    W = weights(wl)
    wr, _ = synth.router(wl)
    b = corr_bias(wl.E)
    opts = moe.router_opts(moe.MOE_ROUTER_SIGMOID_BIAS_SELECT, False, 2.5)
    outs = {}
    for T in (1, 64, 1024):
        x = synth.tokens(wl, T)
        d = moe.dims(T, wl.H, wl.E, wl.k, wl.I)
        ws = moe.new_workspace(d)
        out, idx, w, counts = moe.layer_forward(dev_bf16(x), dev(wr), dev(b), W.packed, d, ws,
                                                want_routing=True, opts=opts)
        torch.cuda.synchronize()
        assert moe.moe_read_device_status(ws) == 0
        outs[T] = bits(out)
        if T == 64:
            out_o, idx_o = _glm_layer_oracle(wl, x, wr, b)
            np.testing.assert_array_equal(idx.cpu().numpy(), idx_o)
            assert_close(outs[T], out_o)
    np.testing.assert_array_equal(outs[1], outs[1024][:1])
    np.testing.assert_array_equal(outs[64], outs[1024][:64])
