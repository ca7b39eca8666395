"""Shared expert in G column shards and the whole layer as G expert ranks.

  "0 train-infer mismatch for open-weight MoE RL", sections "Mixture-of-experts
  layers" (shared expert: fixed-K projections and SwiGLU of the dense case; each
  rank adds its shard before the ranks combine) and "Sharding the experts".

  Shards vs the oracle within the GEMM tolerance (the K order of the tensor-core
  sums differs from the oracle's ascending sum); shards bit-exact against the
  routed expert path run on G copies of the token rows (the same GEMM and tiles
  per row, so the same bits); the sharded layer bit-exact against its steps and
  batch-invariant; the sharded layer against the full oracle within tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close, assert_close_f32, bits, dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_ok):
    import moe_expert_layer_fp32_gb300 as m
    return m


def packed_shared(moe, wl, Is, G):
    wg, wu, wd = synth.shared_expert_weights(wl, Is)
    p = torch.empty(moe.moe_shared_packed_bytes(wl.H, Is) // 2, dtype=torch.bfloat16,
                    device="cuda")
    moe.moe_prepack_shared_expert(dev_bf16(wg), dev_bf16(wu), dev_bf16(wd), wl.H, Is, G, p)
    return p, (wg, wu, wd)


def run_shared(moe, x, p, T, H, Is, G):
    ws = torch.zeros(moe.moe_shared_expert_workspace_bytes(T, H, Is, G), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((G, T, H), dtype=torch.float32, device="cuda")
    moe.moe_shared_expert(dev_bf16(x), p, T, H, Is, G, out, ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    return out


@pytest.mark.parametrize("Is,G,T", [(1024, 8, 300), (1024, 2, 129), (2048, 16, 64),
                                    (256, 1, 1)])
def test_shared_expert_vs_oracle(moe, Is, G, T):
    wl = synth.WORKLOADS["ling3_tiny"]
    x = synth.tokens(wl, T)
    p, (wg, wu, wd) = packed_shared(moe, wl, Is, G)
    got = run_shared(moe, x, p, T, wl.H, Is, G).cpu().numpy()
    ref = oracle.shared_expert(x, wg, wu, wd, G)
    assert_close_f32(got, ref)


@pytest.mark.parametrize("T", [333, 5])
def test_shared_expert_equals_routed_path_on_copies(moe, T):
    """Shard g of the shared expert, computed with the token rows read in place,
    equals the grouped expert FFN over G copies of the rows with the same packed
    weights (E = G experts of intermediate Is / G), bit for bit.  T = 5 runs the
    GEMMs in their swapped form on both sides."""
    wl = synth.WORKLOADS["ling3_tiny"]
    Is, G = 1024, 8
    x = synth.tokens(wl, T)
    p, _ = packed_shared(moe, wl, Is, G)
    got = run_shared(moe, x, p, T, wl.H, Is, G)
    d_rows = moe.dims(G * T, wl.H, G, 1, Is // G)  # G "experts" of Is / G, G * T rows
    assert moe.moe_expert_ffn_form(d_rows) == (1 if T == 5 else 0)
    ws = moe.new_workspace(d_rows)
    xp = dev_bf16(np.tile(x, (G, 1)))
    offsets = dev(np.arange(G + 1, dtype=np.int32) * T)
    y = torch.empty((G * T, wl.H), dtype=torch.float32, device="cuda")
    moe.moe_expert_ffn(xp, offsets, p, d_rows, y, ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    np.testing.assert_array_equal(got.view(-1, wl.H).cpu().numpy().view(np.uint32),
                                  y.cpu().numpy().view(np.uint32))


def test_shared_expert_rejects_bad_shapes(moe):
    x = torch.zeros((4, 1536), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty((8, 4, 1536), dtype=torch.float32, device="cuda")
    for Is, G, code in [(1000, 7, 1), (1000, 8, 2), (512, 8, 2), (0, 1, 1)]:
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_shared_expert(x, x, 4, 1536, Is, G, out, ws)
        assert ei.value.code == code
    assert moe.moe_shared_expert_workspace_bytes(4, 1536, 512, 8) == 0


def _owner(E, G):
    return (np.arange(E) * G // E).astype(np.int32)  # contiguous blocks, every rank < G


def sharded_layer(moe, wl, T, G, Is, p_shared, W_packed, opts=None):
    x = synth.tokens(wl, T)
    wr, bias = synth.router(wl)
    d = moe.dims(T, wl.H, wl.E, wl.k, wl.I)
    ws = torch.zeros(moe.moe_sharded_workspace_bytes(d, G, Is), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, wl.k), dtype=torch.float32, device="cuda")
    counts = torch.empty(wl.E, dtype=torch.int32, device="cuda")
    owner = dev(_owner(wl.E, G))
    moe.moe_layer_fwd_sharded(dev_bf16(x), dev(wr), None if bias is None else dev(bias), opts,
                              W_packed, owner, G, p_shared, Is, d, out, idx, w, counts, ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    return x, out, idx, w, owner, d


@pytest.fixture(scope="module")
def ling(moe):
    from gpu_util import DeviceWeights
    wl = synth.WORKLOADS["ling3_tiny"]
    return wl, DeviceWeights(wl)


@pytest.mark.parametrize("G,Is", [(8, 1024), (8, 0), (16, 2048), (3, 384)])
def test_sharded_layer_equals_its_steps(moe, ling, G, Is):
    wl, W = ling
    T = 700
    p = packed_shared(moe, wl, Is, G)[0] if Is else None
    x, out, idx, w, owner, d = sharded_layer(moe, wl, T, G, Is, p, W.packed)
    # the same steps through the step entry points
    ws = moe.new_workspace(d)
    R = T * wl.k
    c = torch.empty(wl.E, dtype=torch.int32, device="cuda")
    o = torch.empty(wl.E + 1, dtype=torch.int32, device="cuda")
    moe.moe_load_stats(idx, d, c, o, ws)
    xp = torch.empty((R, wl.H), dtype=torch.bfloat16, device="cuda")
    ros = torch.empty(R, dtype=torch.int32, device="cuda")
    sor = torch.empty(R, dtype=torch.int32, device="cuda")
    moe.moe_permute(dev_bf16(x), idx, o, d, xp, ros, sor, ws)
    y = torch.empty((R, wl.H), dtype=torch.float32, device="cuda")
    moe.moe_expert_ffn(xp, o, W.packed, d, y, ws)
    sh = run_shared(moe, x, p, T, wl.H, Is, G) if Is else None
    ref = torch.empty_like(out)
    moe.moe_combine_sharded(y, w, idx, ros, owner, G, 1.0, sh, d, ref)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(out), bits(ref))
    # and the combine bit-exact against the oracle on these same inputs
    ref_o = oracle.combine_sharded(y.cpu().numpy(), w.cpu().numpy(), idx.cpu().numpy(),
                                   ros.cpu().numpy().reshape(T, -1), owner.cpu().numpy(), G, 1.0,
                                   None if sh is None else sh.cpu().numpy())
    np.testing.assert_array_equal(bits(out), ref_o)


def test_sharded_layer_batch_invariant(moe, ling):
    wl, W = ling
    G, Is = 8, 1024
    p = packed_shared(moe, wl, Is, G)[0]
    outs = {T: bits(sharded_layer(moe, wl, T, G, Is, p, W.packed)[1]) for T in (1, 64, 777)}
    np.testing.assert_array_equal(outs[1], outs[777][:1])
    np.testing.assert_array_equal(outs[64], outs[777][:64])


def test_sharded_layer_vs_full_oracle(moe, ling):
    """Route, permute, experts, shared expert shards and the sharded combine, all
    from the oracle, against the GPU layer: indices bit-exact, output within the
    layer tolerance."""
    wl, W = ling
    T, G, Is = 96, 8, 1024
    p, (swg, swu, swd) = packed_shared(moe, wl, Is, G)
    x, out, idx, w, owner, d = sharded_layer(moe, wl, T, G, Is, p, W.packed)
    wr, bias = synth.router(wl)
    idx_o, w_o = oracle.route(x, wr, bias, wl.k)
    np.testing.assert_array_equal(idx.cpu().numpy(), idx_o)
    counts, offs, _, _ = oracle.load_stats(idx_o, wl.E)
    experts = np.flatnonzero(counts)
    wg, wu, wd = synth.expert_weights(wl, experts)
    remap = np.full(wl.E, -1, np.int64)
    remap[experts] = np.arange(len(experts))
    sidx = remap[idx_o].astype(np.int32)
    _, soffs, _, _ = oracle.load_stats(sidx, len(experts))
    xp, ros, _ = oracle.permute(x, sidx, soffs, len(experts))
    y = oracle.expert_ffn(xp, soffs, wg, wu, wd)
    sh = oracle.shared_expert(x, swg, swu, swd, G)
    ref = oracle.combine_sharded(y, w_o, idx_o, ros, _owner(wl.E, G), G, 1.0, sh)
    assert_close(bits(out), ref)
