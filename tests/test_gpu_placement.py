"""Placement-aware dispatch and multiplicity-weighted loads on the GPU.

  "RoutePack" Algorithm 1 (host LPT placement from measured expert loads) feeds
  the dispatcher's logical -> physical slot map; counts, offsets and the
  permutation by physical slot must equal the oracle's bit for bit, and a layer
  run with the weights packed into their physical slots must give the same
  output bytes as the identity placement (every row's arithmetic is unchanged).
  "HARTS" Eq. 20 multiplicity-weighted counts: bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import DeviceWeights, bits, dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_ok):
    import moe_expert_layer_fp32_gb300 as m
    return m


@pytest.mark.parametrize("name,P", [("fine_grained", 8), ("packed_rl", 16)])
def test_placed_dispatch_matches_oracle(moe, name, P):
    wl = synth.WORKLOADS[name]
    x = synth.tokens(wl)
    wr, bias = synth.router(wl)
    idx, _ = oracle.route(x, wr, bias, wl.k)
    counts, _, _, _ = oracle.load_stats(idx, wl.E)
    pi, G = moe.moe_lpt_placement_host(counts.astype(np.int64), P)
    cv0, eta0 = moe.moe_rank_load_summary_host(
        np.bincount(np.arange(wl.E) // (wl.E // P), weights=counts, minlength=P).astype(np.int64))
    cv1, eta1 = moe.moe_rank_load_summary_host(G)
    assert cv1 <= cv0 and eta1 >= eta0  # LPT balances the ranks at least as well
    d = moe.dims(wl.T, wl.H, wl.E, wl.k, wl.I)
    ws = moe.new_workspace(d)
    pc = torch.empty(wl.E, dtype=torch.int32, device="cuda")
    po = torch.empty(wl.E + 1, dtype=torch.int32, device="cuda")
    moe.moe_load_stats_ex(dev(idx), dev(pi), None, d, pc, po, None, ws)
    phys = np.zeros(wl.E, np.int32)
    phys[pi] = counts
    np.testing.assert_array_equal(pc.cpu().numpy(), phys)
    poff = np.concatenate([[0], np.cumsum(phys)]).astype(np.int32)
    np.testing.assert_array_equal(po.cpu().numpy(), poff)
    R = wl.T * wl.k
    xp = torch.empty((R, wl.H), dtype=torch.bfloat16, device="cuda")
    ros = torch.empty(R, dtype=torch.int32, device="cuda")
    sor = torch.empty(R, dtype=torch.int32, device="cuda")
    moe.moe_permute_ex(dev_bf16(x), dev(idx), dev(pi), po, d, xp, ros, sor, ws)
    xp_o, ros_o, sor_o = oracle.permute_remap(x, idx, pi, poff, wl.E)
    np.testing.assert_array_equal(ros.cpu().numpy(), ros_o)
    np.testing.assert_array_equal(sor.cpu().numpy(), sor_o)
    np.testing.assert_array_equal(bits(xp), xp_o)
    assert moe.moe_read_device_status(ws) == 0


def test_placed_layer_is_bitwise_the_identity_layer(moe):
    """Rows regrouped by physical slot, weights packed into their slots: the
    layer output bytes do not change."""
    wl = synth.WORKLOADS["fine_grained"]
    T, E, H, I, k = 2048, wl.E, wl.H, wl.I, wl.k
    x = synth.tokens(wl, T)
    wr, bias = synth.router(wl)
    d = moe.dims(T, H, E, k, I)
    ws = moe.new_workspace(d)
    W = DeviceWeights(wl, keep_logical=True)
    xd, wrd, bd = dev_bf16(x), dev(wr), dev(bias)
    out_id, idx, w, counts = moe.layer_forward(xd, wrd, bd, W.packed, d, ws, want_routing=True)
    pi, _ = moe.moe_lpt_placement_host(counts.cpu().numpy().astype(np.int64), 8)
    pid = dev(pi)
    packed_pl = torch.empty_like(W.packed)
    moe.moe_prepack_expert_weights_ex(W.wg, W.wu, W.wd, pid, d, packed_pl)
    pc = torch.empty(E, dtype=torch.int32, device="cuda")
    po = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    moe.moe_load_stats_ex(idx, pid, None, d, pc, po, None, ws)
    R = T * k
    xp = torch.empty((R, H), dtype=torch.bfloat16, device="cuda")
    ros = torch.empty(R, dtype=torch.int32, device="cuda")
    sor = torch.empty(R, dtype=torch.int32, device="cuda")
    moe.moe_permute_ex(xd, idx, pid, po, d, xp, ros, sor, ws)
    y = torch.empty((R, H), dtype=torch.float32, device="cuda")
    moe.moe_expert_ffn(xp, po, packed_pl, d, y, ws)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(y, w, ros, d, out)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    np.testing.assert_array_equal(bits(out), bits(out_id))


@pytest.mark.parametrize("name", ["tiny", "fine_grained", "large"])
def test_weighted_counts_bit_exact(moe, name):
    wl = synth.WORKLOADS[name]
    T = min(wl.T, 8192)
    x = synth.tokens(wl, T)
    wr, bias = synth.router(wl)
    idx, _ = oracle.route(x, wr, bias, wl.k)
    q = synth.uniform_i32(4, synth.TID_MISC, (T,), 1, 50)
    d = moe.dims(T, wl.H, wl.E, wl.k, wl.I)
    ws = moe.new_workspace(d)
    c = torch.empty(wl.E, dtype=torch.int32, device="cuda")
    o = torch.empty(wl.E + 1, dtype=torch.int32, device="cuda")
    wc = torch.full((wl.E,), -1, dtype=torch.int64, device="cuda")
    moe.moe_load_stats_ex(dev(idx), None, dev(q), d, c, o, wc, ws)
    np.testing.assert_array_equal(wc.cpu().numpy(), oracle.weighted_counts(idx, q, wl.E))
    np.testing.assert_array_equal(c.cpu().numpy(), oracle.load_stats(idx, wl.E)[0])
    assert moe.moe_read_device_status(ws) == 0
