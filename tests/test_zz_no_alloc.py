"""moe_load_stats_noalloc: the load statistics for callers that cannot allocate
device memory (its scratch is a fixed array inside the library rather than a
caller workspace).  Called through the C ABI twice in a row on different inputs,
its counts and offsets must equal those of moe_load_stats on the same inputs and
those of the CPU oracle (bit-exact, like every integer output of the library),
with no device-side error.  An empty batch gives all-zero counts and offsets, and
a token that names one expert twice is reported through the device status word.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_ok):
    import moe_expert_layer_fp32_gb300 as m
    return m


def routed_idx(wl):
    wr, bias = synth.router(wl)
    idx, _ = oracle.route(synth.tokens(wl), wr, bias, wl.k)
    return idx


def random_distinct_idx(T, E, k, seed):
    keys = synth.uniform_f32(seed, synth.TID_TOPK_IDX, (T, E), 0.0, 1.0)
    return np.argsort(keys, axis=1)[:, :k].astype(np.int32)


def test_noalloc_matches_workspace_version_twice(moe):
    cases = [(synth.WORKLOADS["fine_grained"], routed_idx(synth.WORKLOADS["fine_grained"])),
             (synth.Workload("wide", T=777, H=128, E=256, k=16, I=128, w_std=0.02),
              random_distinct_idx(777, 256, 16, seed=5))]
    for wl, idx in cases:  # two calls in a row, different shapes and inputs
        d = moe.dims(idx.shape[0], wl.H, wl.E, wl.k, wl.I)
        idx_d = torch.from_numpy(idx).cuda()
        counts = torch.full((wl.E,), -1, dtype=torch.int32, device="cuda")
        offsets = torch.full((wl.E + 1,), -1, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        moe.moe_load_stats_noalloc(idx_d, d, counts, offsets, status)

        ws = moe.new_workspace(d)
        counts_ref = torch.empty(wl.E, dtype=torch.int32, device="cuda")
        offsets_ref = torch.empty(wl.E + 1, dtype=torch.int32, device="cuda")
        moe.moe_load_stats(idx_d, d, counts_ref, offsets_ref, ws)
        torch.cuda.synchronize()
        assert moe.moe_read_device_status(ws) == 0
        assert int(status.item()) == 0
        np.testing.assert_array_equal(counts.cpu().numpy(), counts_ref.cpu().numpy())
        np.testing.assert_array_equal(offsets.cpu().numpy(), offsets_ref.cpu().numpy())
        assert int(offsets[-1].item()) == idx.size
        counts_o, offsets_o, _, _ = oracle.load_stats(idx, wl.E)
        np.testing.assert_array_equal(counts.cpu().numpy(), counts_o)
        np.testing.assert_array_equal(offsets.cpu().numpy(), offsets_o)


def test_noalloc_empty_batch_and_repeated_expert(moe):
    E = 16
    # T = 0: nothing to count; every count and offset is written as 0
    d = moe.dims(0, 128, E, 2, 128)
    counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_load_stats_noalloc(torch.empty((0, 2), dtype=torch.int32, device="cuda"), d, counts,
                               offsets, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert not counts.any().item() and not offsets.any().item()

    # token 3 names expert 5 twice: flagged, never a silent count
    idx = random_distinct_idx(300, E, 2, seed=9)
    idx[3] = [5, 5]
    d = moe.dims(300, 128, E, 2, 128)
    status.zero_()
    moe.moe_load_stats_noalloc(torch.from_numpy(idx).cuda(), d, counts, offsets, status)
    torch.cuda.synchronize()
    assert moe.STATUS[int(status.item())] == "MOE_ERR_DEVICE_CHECK"


def test_noalloc_rejects_sizes_beyond_its_scratch(moe):
    # 2 * ceil(T/256) * E must stay within 524288 int32 entries
    d = moe.dims(262144 + 256, 128, 256, 1, 128)
    counts = torch.empty(256, dtype=torch.int32, device="cuda")
    offsets = torch.empty(257, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_load_stats_noalloc(16, d, counts, offsets)
    assert moe.STATUS[ei.value.code] == "MOE_ERR_UNSUPPORTED"
