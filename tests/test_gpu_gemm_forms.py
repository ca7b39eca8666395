"""The three forms of the grouped expert GEMMs give the same bits.

  "0 train-infer mismatch for open-weight MoE RL", section "Matrix
  multiplication: the same reduction along K": a row's result must not depend
  on how many rows the batch holds.

The tile kernels put token rows on the MMA's M side (128 per tile); the swapped
kernels, used for small batches, put weight rows on M and up to 64 token rows on
N; the pair kernels, used from 512 rows per expert on average, run one M = 256
MMA over two CTAs.  All of them sum the same BF16 products in the same K order,
so every row of h and y must be bit-identical.  moe_expert_ffn picks the form
from the dims alone (moe_expert_ffn_form): the same expert rows are run with few
rows in total (swapped form), with more rows added to the last expert (single-CTA
tiles) and with many more (pairs), and the shared rows are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close_f32, dev, dev_bf16, weights

pytestmark = pytest.mark.gpu

# rows of the experts that have any (every fifth expert): one row, the 16/32/64
# token-box edges, two and three token tiles of 64 (469 rows), and 3 rows in the
# last expert
PATTERN = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 130]


@pytest.fixture(scope="module")
def moe(cuda_ok):
    import moe_expert_layer_fp32_gb300 as m
    return m


def ffn(moe, wl, W, x, counts, form):
    offsets = np.zeros(wl.E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    R = int(offsets[-1])
    d = moe.dims(R, wl.H, wl.E, 1, wl.I)  # k = 1: R rows
    assert moe.moe_expert_ffn_form(d) == form
    ws = moe.new_workspace(d)
    y = torch.empty((R, wl.H), dtype=torch.float32, device="cuda")
    moe.moe_expert_ffn(dev_bf16(x[:R]), dev(offsets), W.packed, d, y, ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    return y.cpu().numpy(), offsets


@pytest.mark.parametrize("name", ["fine_grained", "ling3_tiny"])
def test_swapped_and_tile_forms_bit_identical(moe, name):
    wl = synth.WORKLOADS[name]
    W = weights(wl)
    counts_small = np.zeros(wl.E, dtype=np.int64)
    counts_small[0:5 * len(PATTERN):5] = PATTERN
    counts_small[-1] = 3
    R_small = int(counts_small.sum())
    counts_big = counts_small.copy()
    counts_big[-1] += 64 * wl.E  # the last expert's first rows are shared
    x = synth.tokens(wl, int(counts_big.sum()))
    y_small, offs = ffn(moe, wl, W, x, counts_small, form=1)
    y_big, _ = ffn(moe, wl, W, x, counts_big, form=0)
    np.testing.assert_array_equal(y_small.view(np.uint32), y_big[:R_small].view(np.uint32))

    # and the swapped form within tolerance of the oracle on a few experts
    experts = np.array([e for e in range(30) if counts_small[e] > 0])
    wg, wu, wd = synth.expert_weights(wl, experts)
    rows = np.concatenate([np.arange(offs[e], offs[e + 1]) for e in experts])
    sub_off = np.zeros(len(experts) + 1, dtype=np.int32)
    sub_off[1:] = np.cumsum(counts_small[experts])
    ref = oracle.expert_ffn(x[rows], sub_off, wg, wu, wd)
    assert_close_f32(y_small[rows], ref)


@pytest.mark.parametrize("name", ["fine_grained", "packed_rl"])
def test_single_cta_and_pair_forms_bit_identical(moe, name):
    """Expert row counts around the 128- and 256-row tile edges (odd last tiles,
    an expert whose rows end inside the odd CTA's half, empty experts): the same
    rows through the single-CTA tile kernels (under 512 rows per expert on
    average) and through the pair kernels (above) give the same bits."""
    wl = synth.WORKLOADS[name]
    W = weights(wl)
    counts_mid = np.zeros(wl.E, dtype=np.int64)
    edges = [1, 127, 128, 129, 255, 256, 257, 383, 384, 385, 511, 640]
    counts_mid[0:3 * len(edges):3] = edges
    counts_mid[-1] = 5
    R_mid = int(counts_mid.sum())
    counts_big = counts_mid.copy()
    counts_big[-1] += 512 * wl.E  # the last expert's first rows are shared
    x = synth.tokens(wl, int(counts_big.sum()))
    y_mid, _ = ffn(moe, wl, W, x, counts_mid, form=0)
    y_big, _ = ffn(moe, wl, W, x, counts_big, form=0)
    np.testing.assert_array_equal(y_mid.view(np.uint32), y_big[:R_mid].view(np.uint32))


@pytest.mark.parametrize("name", ["fine_grained", "ling3_tiny"])
def test_quarter_and_half_box_units_bit_identical(moe, name):
    """Decode-sized batches (at most a few experts with rows): the swapped gate/up
    GEMM splits each packed box into 64-gate + 64-up-row units and the down GEMM
    into 128-row halves.  Those rows must equal the tile kernels' bits."""
    wl = synth.WORKLOADS[name]
    W = weights(wl)
    counts_small = np.zeros(wl.E, dtype=np.int64)
    counts_small[[0, 5, 17, wl.E - 1]] = [1, 2, 3, 2]  # 8 rows in 4 experts
    R_small = int(counts_small.sum())
    counts_big = counts_small.copy()
    counts_big[-1] += 64 * wl.E
    x = synth.tokens(wl, int(counts_big.sum()))
    y_small, offs = ffn(moe, wl, W, x, counts_small, form=1)
    y_big, _ = ffn(moe, wl, W, x, counts_big, form=0)
    np.testing.assert_array_equal(y_small.view(np.uint32), y_big[:R_small].view(np.uint32))
    experts = np.nonzero(counts_small)[0]
    wg, wu, wd = synth.expert_weights(wl, experts)
    sub_off = np.zeros(len(experts) + 1, dtype=np.int32)
    sub_off[1:] = np.cumsum(counts_small[experts])
    ref = oracle.expert_ffn(x[:R_small], sub_off, wg, wu, wd)
    assert_close_f32(y_small, ref)
