"""Failure detection on the GPU without a fault: the grouped GEMMs' bounded waits
are given a limit far below a TMA round trip, so a wait runs out; the kernel
must record MOE_ERR_TIMEOUT in the workspace status word, drain its own copies
and return, and the same context must then run a correct forward.

The shape has one column tile per GEMM (H = I = 128), which selects the
single-CTA kernels: no copy of one CTA targets another CTA's shared memory."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close, bits, dev, dev_bf16, weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_ok):
    import moe_expert_layer_fp32_gb300 as m
    return m


def test_wait_timeout_is_reported_and_context_survives(moe):
    wl = synth.Workload("timeout", T=256, H=128, E=4, k=2, I=128, w_std=0.05)
    W = weights(wl)
    x = synth.tokens(wl)
    wr, _ = synth.router(wl)
    idx, w = oracle.route(x, wr, None, wl.k)
    counts, offsets, _, _ = oracle.load_stats(idx, wl.E)
    xp, ros, _ = oracle.permute(x, idx, offsets, wl.E)
    d = moe.dims(wl.T, wl.H, wl.E, wl.k, wl.I)
    ws = moe.new_workspace(d)
    R = wl.T * wl.k
    y = torch.zeros((R, wl.H), dtype=torch.float32, device="cuda")
    statuses = []
    try:
        moe.moe_set_wait_limit(16)
        for _ in range(3):
            moe.moe_expert_ffn(dev_bf16(xp), dev(offsets), W.packed, d, y, ws)
            statuses.append(moe.moe_read_device_status(ws))
    finally:
        moe.moe_set_wait_limit(0)
    assert moe.STATUS[6] == "MOE_ERR_TIMEOUT"
    assert 6 in statuses, statuses
    assert set(statuses) <= {0, 6}
    # the context is intact: the default limit gives the right answer again
    moe.moe_expert_ffn(dev_bf16(xp), dev(offsets), W.packed, d, y, ws)
    assert moe.moe_read_device_status(ws) == 0
    wg, wu, wdn = synth.expert_weights(wl)
    y_o = oracle.expert_ffn(xp, offsets, wg, wu, wdn)
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(y, dev(w), dev(ros), d, out)
    assert_close(bits(out), oracle.combine(y_o, w, ros))
