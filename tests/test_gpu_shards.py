"""Expert ranks on one GPU: sharded combine and the fixed FP64 tree, bit-exact
against the oracle.

  "0 train-infer mismatch for open-weight MoE RL", section "Sharding the experts":
  per-rank BF16 partials (other ranks' slots as exact zeros, shared-expert shard
  added before the rounding), reduced by adjacent pairs in FP64 with the odd
  contributor carried, one BF16 rounding.  Every output bit must equal the
  oracle's: the chains, the roundings and the tree are fixed operations.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close, bits, dev, dev_bf16, weights

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def moe(cuda_ok):
    import moe_expert_layer_fp32_gb300 as m
    return m


def random_bf16_bits(seed, shape):
    """Finite bf16 bit patterns of every exponent (zeros, subnormals, huge and
    tiny values, both signs): exercises every branch of both conversions."""
    u = synth.uniform_i32(seed, synth.TID_MISC, shape, 0, 65535).astype(np.uint32)
    u = np.where((u & 0x7F80) == 0x7F80, u & 0x807F, u)  # no inf / NaN inputs
    return u.astype(np.uint16)


def gpu_tree(moe, p, N=None):
    G = p.shape[0]
    N = p.shape[1] if N is None else N
    pd = dev_bf16(p)
    out = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    moe.moe_tree_reduce_bf16(pd, G, N, out)
    return bits(out)


@pytest.mark.parametrize("G", list(range(1, 17)))
def test_tree_reduce_all_exponents(moe, G):
    N = 4096 + 8  # vector path
    p = random_bf16_bits(100 + G, (G, N))
    np.testing.assert_array_equal(gpu_tree(moe, p), oracle.tree_reduce(p))


@pytest.mark.parametrize("G,N", [(3, 1001), (8, 77777), (16, 5)])
def test_tree_reduce_ragged_scalar_path(moe, G, N):
    p = random_bf16_bits(200 + G, (G, N))
    np.testing.assert_array_equal(gpu_tree(moe, p), oracle.tree_reduce(p))


def test_tree_reduce_near_ties_and_cancellation(moe):
    """Partials built so that the FP64 sums land on, just above and just below
    bf16 ties, cancel to signed zeros, overflow to infinity, or lose a term in
    FP64: the cases where a second rounding or another order shows."""
    rng = np.random.default_rng(3)
    rows = []
    for _ in range(3000):
        a = rng.integers(0x3F00, 0x4100)           # around 1
        b = rng.integers(0x3A00, 0x3C00)           # around 2^-8 .. 2^-7
        c = rng.integers(0x2000, 0x3000) | (rng.integers(0, 2) << 15)  # tiny, either sign
        rows.append([a, b, c, rng.choice([0, 0x8000])])
    rows += [[0x5D80, 0x3F80, 0xDD80, 0x3F80], [0x7F7F, 0x7F7F, 0, 0], [0xFF7F, 0x7F7F, 0x8000, 0],
             [0x8000, 0x8000, 0x8000, 0x8000], [0x0001, 0x0001, 0x8001, 0x0000]]
    p = np.array(rows, np.uint16).T.copy()
    np.testing.assert_array_equal(gpu_tree(moe, p), oracle.tree_reduce(p))
    with open(os.path.join(GOLDEN, "fp64_tree.json")) as f:
        for c in json.load(f)["cases"]:
            q = np.array(c["partials_bf16_bits"], np.uint16).reshape(-1, 1)
            assert int(gpu_tree(moe, q)[0]) == c["expected_bf16_bits"], c["name"]


def test_tree_reduce_rejects_bad_arguments(moe):
    out = torch.empty(8, dtype=torch.bfloat16, device="cuda")
    p = torch.zeros((17, 8), dtype=torch.bfloat16, device="cuda")
    for G, N, code in [(0, 8, 1), (17, 8, 2), (2, -1, 1)]:
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_tree_reduce_bf16(p, G, N, out)
        assert ei.value.code == code
    moe.moe_tree_reduce_bf16(p, 2, 0, out)  # empty: nothing to do


def _case(wl, T, seed):
    x = synth.tokens(wl, T)
    wr, bias = synth.router(wl)
    idx, w = oracle.route(x, wr, bias, wl.k)
    R = T * wl.k
    y = synth.normal_f32(seed, synth.TID_Y, (R, wl.H), 0.05)
    ros = np.random.default_rng(seed).permutation(R).astype(np.int32).reshape(T, wl.k)
    return idx, w, y, ros


def _owners(E, G, kind, counts=None, moe=None):
    if kind == "contiguous":
        return (np.arange(E) // -(-E // G)).astype(np.int32)
    if kind == "strided":
        return (np.arange(E) % G).astype(np.int32)
    pi, _ = moe.moe_lpt_placement_host(counts.astype(np.int64), G)  # RoutePack LPT
    return (pi // (E // G)).astype(np.int32)


@pytest.mark.parametrize("G,kind,with_shared,scale", [
    (1, "contiguous", False, 1.0), (2, "strided", True, 1.0), (3, "contiguous", False, 2.5),
    (8, "lpt", False, 1.0), (8, "contiguous", True, 2.5), (16, "lpt", True, 1.0),
    (5, "strided", True, 1.0)])
def test_combine_sharded_bit_exact(moe, G, kind, with_shared, scale):
    wl = synth.WORKLOADS["fine_grained"]
    T = 777  # several CTAs' worth and a ragged count
    idx, w, y, ros = _case(wl, T, 30 + G)
    counts = np.bincount(idx.ravel(), minlength=wl.E)
    owner = _owners(wl.E, G, kind, counts, moe)
    sh = synth.normal_f32(40 + G, synth.TID_MISC, (G, T, wl.H), 0.02) if with_shared else None
    d = moe.dims(T, wl.H, wl.E, wl.k, wl.I)
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
    parts = torch.empty((G, T, wl.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine_sharded(dev(y), dev(w), dev(idx), dev(ros), dev(owner), G, scale,
                            None if sh is None else dev(sh), d, out, partials=parts)
    ref, ref_parts = oracle.combine_sharded(y, w, idx, ros, owner, G, scale, sh,
                                            want_partials=True)
    np.testing.assert_array_equal(bits(parts), ref_parts)
    np.testing.assert_array_equal(bits(out), ref)
    out2 = torch.empty_like(out)  # without the partials output: same bits
    moe.moe_combine_sharded(dev(y), dev(w), dev(idx), dev(ros), dev(owner), G, scale,
                            None if sh is None else dev(sh), d, out2)
    np.testing.assert_array_equal(bits(out2), ref)


def test_combine_sharded_golden_cases(moe):
    """The hand-derived cases, padded to H = 128 (column 0 holds the case)."""
    with open(os.path.join(GOLDEN, "sharded_combine.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        G = c["G"]
        owner = np.array(c["owner"], np.int32)
        idx = np.array(c["idx"], np.int32)
        w = np.array(c["w"], np.float32)
        ros = np.array(c["row_of_slot"], np.int32)
        T, k = w.shape
        y = np.zeros((T * k, 128), np.float32)
        y[:, 0] = np.array(c["y"], np.float32)[:, 0]
        sh = None
        if c["shared"] is not None:
            sh = np.zeros((G, T, 128), np.float32)
            sh[:, :, 0] = np.array(c["shared"], np.float32)[:, :, 0]
        d = moe.dims(T, 128, len(owner), k, 128)
        out = torch.empty((T, 128), dtype=torch.bfloat16, device="cuda")
        parts = torch.empty((G, T, 128), dtype=torch.bfloat16, device="cuda")
        moe.moe_combine_sharded(dev(y), dev(w), dev(idx), dev(ros), dev(owner), G, 1.0,
                                None if sh is None else dev(sh), d, out, partials=parts)
        assert bits(out)[:, 0].tolist() == [v[0] for v in c["expected_out_bf16_bits"]], c["name"]
        np.testing.assert_array_equal(bits(parts)[:, :, :1],
                                      np.array(c["expected_partials_bf16_bits"]))
        out2 = torch.empty_like(out)  # the layer's form (no partials written)
        moe.moe_combine_sharded(dev(y), dev(w), dev(idx), dev(ros), dev(owner), G, 1.0,
                                None if sh is None else dev(sh), d, out2)
        assert bits(out2)[:, 0].tolist() == [v[0] for v in c["expected_out_bf16_bits"]], c["name"]


def test_sharded_layer_on_gpu_expert_outputs(moe):
    """The real path: GPU route, permute and expert FFN, then the sharded combine
    over 8 contiguous expert ranks.  Bit-exact against the oracle's sharded
    combine of the same y; within tolerance of the unsharded layer."""
    wl = synth.WORKLOADS["fine_grained"]
    T = 512
    W = weights(wl)
    x = synth.tokens(wl, T)
    wr, bias = synth.router(wl)
    d = moe.dims(T, wl.H, wl.E, wl.k, wl.I)
    ws = moe.new_workspace(d)
    xd = dev_bf16(x)
    R = T * wl.k
    idx = torch.empty((T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, wl.k), dtype=torch.float32, device="cuda")
    moe.moe_route(xd, dev(wr), dev(bias), d, idx, w)
    c = torch.empty(wl.E, dtype=torch.int32, device="cuda")
    o = torch.empty(wl.E + 1, dtype=torch.int32, device="cuda")
    moe.moe_load_stats(idx, d, c, o, ws)
    xp = torch.empty((R, wl.H), dtype=torch.bfloat16, device="cuda")
    ros = torch.empty(R, dtype=torch.int32, device="cuda")
    sor = torch.empty(R, dtype=torch.int32, device="cuda")
    moe.moe_permute(xd, idx, o, d, xp, ros, sor, ws)
    y = torch.empty((R, wl.H), dtype=torch.float32, device="cuda")
    moe.moe_expert_ffn(xp, o, W.packed, d, y, ws)
    owner = _owners(wl.E, 8, "contiguous")
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine_sharded(y, w, idx, ros, dev(owner), 8, 1.0, None, d, out)
    plain = torch.empty_like(out)
    moe.moe_combine(y, w, ros, d, plain)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    ref = oracle.combine_sharded(y.cpu().numpy(), w.cpu().numpy(), idx.cpu().numpy(),
                                 ros.cpu().numpy().reshape(T, -1), owner, 8)
    np.testing.assert_array_equal(bits(out), ref)
    assert_close(bits(out), bits(plain))


@pytest.mark.parametrize("G", [2, 3, 8, 16])
def test_combine_sharded_signed_zeros_and_fallback(moe, G):
    """Inputs built so that the chain order shows in the sign of zero (products
    that underflow to -0, weights of both signs, exact zeros), and shard outputs
    spread over 40 binades so that part of the tree falls back to FP64.  Partials
    and outputs bit-exact, with and without the partials output (two kernels)."""
    T, H, E, k = 300, 128, 16, 8
    rng = np.random.default_rng(G)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    R = T * k
    choices = np.array([-2.0 ** -100, 2.0 ** -100, -0.0, 0.0, -1.5, 0.75, -2.0 ** -140],
                       np.float32)
    y = choices[rng.integers(0, len(choices), (R, H))].astype(np.float32)
    wch = np.array([2.0 ** -100, -2.0 ** -100, 0.5, -0.25, 0.0, -0.0], np.float32)
    w = wch[rng.integers(0, len(wch), (T, k))].astype(np.float32)
    ros = rng.permutation(R).astype(np.int32).reshape(T, k)
    owner = rng.integers(0, G, E).astype(np.int32)
    sh = (rng.standard_normal((G, T, H)) * 10.0 ** rng.integers(-20, 20, (G, T, 1))).astype(
        np.float32)
    sh[:, ::3] = 0.0  # some tokens without a shared contribution: zeros reach the tree
    d = moe.dims(T, H, E, k, 128)
    for shared in (None, sh):
        out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        parts = torch.empty((G, T, H), dtype=torch.bfloat16, device="cuda")
        moe.moe_combine_sharded(dev(y), dev(w), dev(idx), dev(ros), dev(owner), G, 1.0,
                                None if shared is None else dev(shared), d, out, partials=parts)
        ref, ref_parts = oracle.combine_sharded(y, w, idx, ros, owner, G, 1.0, shared,
                                                want_partials=True)
        np.testing.assert_array_equal(bits(parts), ref_parts)
        np.testing.assert_array_equal(bits(out), ref)
        out2 = torch.empty_like(out)  # the layer's form (no partials written)
        moe.moe_combine_sharded(dev(y), dev(w), dev(idx), dev(ros), dev(owner), G, 1.0,
                                None if shared is None else dev(shared), d, out2)
        np.testing.assert_array_equal(bits(out2), ref)
