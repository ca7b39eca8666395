"""The C-ABI library loads and exports every symbol include/moe.h declares, and
its host-side validation rejects bad arguments before touching the GPU.  CPU only
(no compute call reaches a device here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "moe_build", os.path.join(ROOT, "moe_expert_layer_fp32_gb300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    b.build()
    import moe_expert_layer_fp32_gb300 as m
    return m


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(moe):
    names = header_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/moe.h but not exported"
    assert set(names) == set(moe.ABI_SYMBOLS)


def test_sizes(moe):
    d = moe.dims(4096, 2048, 64, 8, 1024)
    assert moe.moe_packed_weight_bytes(d) == 64 * 3 * 2048 * 1024 * 2
    ws = moe.moe_workspace_bytes(d)
    R = 4096 * 8
    # x_perm + h + y dominate
    assert ws >= R * 2048 * 2 + R * 1024 * 2 + R * 2048 * 4
    assert ws % 256 == 0
    assert moe.moe_workspace_bytes(moe.dims(0, 128, 8, 2, 256)) > 0
    assert moe.moe_workspace_bytes(moe.dims(8, 100, 8, 2, 256)) == 0  # H not a multiple of 128


@pytest.mark.parametrize("T,H,E,k,I,code", [
    (16, 128, 8, 9, 256, "MOE_ERR_INVALID_ARG"),    # k > E
    (16, 128, 8, 0, 256, "MOE_ERR_INVALID_ARG"),    # k = 0
    (-1, 128, 8, 2, 256, "MOE_ERR_INVALID_ARG"),    # T < 0
    (16, 128, 300, 2, 256, "MOE_ERR_UNSUPPORTED"),  # E > 256
    (16, 128, 32, 17, 256, "MOE_ERR_UNSUPPORTED"),  # k > 16
    (16, 96, 8, 2, 256, "MOE_ERR_UNSUPPORTED"),     # H % 128
    (16, 128, 8, 2, 200, "MOE_ERR_UNSUPPORTED"),    # I % 128
    (1 << 28, 128, 16, 8, 256, "MOE_ERR_UNSUPPORTED"),  # T*k >= 2^31
])
def test_bad_dims_rejected_before_launch(moe, T, H, E, k, I, code):
    d = moe.dims(T, H, E, k, I)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_layer_fwd(16, 16, None, 16, d, 16, None, None, None, (256, 1 << 40), stream=0)
    assert moe.STATUS[ei.value.code] == code
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_route(16, 16, None, d, 16, 16, stream=0)
    assert moe.STATUS[ei.value.code] == code
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_expert_ffn_form(d)
    assert moe.STATUS[ei.value.code] == code


def test_pointer_and_workspace_checks(moe):
    d = moe.dims(64, 128, 8, 2, 256)
    need = moe.moe_workspace_bytes(d)
    call = lambda **kw: moe.moe_layer_fwd(
        kw.get("x", 4096), 4096, None, 4096, d, 4096, None, None, None,
        kw.get("ws", (1 << 20, need)), stream=0)
    with pytest.raises(moe.MoEError) as ei:
        call(x=None)
    assert moe.STATUS[ei.value.code] == "MOE_ERR_INVALID_ARG"
    with pytest.raises(moe.MoEError) as ei:
        call(x=4100)
    assert moe.STATUS[ei.value.code] == "MOE_ERR_MISALIGNED"
    with pytest.raises(moe.MoEError) as ei:
        call(ws=((1 << 20) + 16, need))
    assert moe.STATUS[ei.value.code] == "MOE_ERR_MISALIGNED"
    with pytest.raises(moe.MoEError) as ei:
        call(ws=(1 << 20, need - 1))
    assert moe.STATUS[ei.value.code] == "MOE_ERR_WORKSPACE"


def test_load_summary_host(moe):
    assert moe.moe_load_summary_host([5, 5, 5, 5]) == (0.0, 0.0)
    imb, cv = moe.moe_load_summary_host([8, 0, 0, 0])
    assert imb == pytest.approx(3.0) and cv == pytest.approx(3 ** 0.5)
    with pytest.raises(moe.MoEError):
        moe.moe_load_summary_host([])


def test_status_strings(moe):
    for code in range(8):
        assert moe._lib.moe_status_string(code)


def test_lpt_placement_host_matches_oracle(moe):
    """The library's host LPT planner and rank metrics equal the oracle's."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(5)
    for E, P in [(8, 2), (64, 8), (256, 16), (128, 4)]:
        loads = (rng.zipf(1.4, E) * 37 + rng.integers(0, 9, E)).astype(np.int64)
        loads[: E // 4] = loads[E // 4: E // 2]  # equal loads exercise the tie rules
        pi, G = moe.moe_lpt_placement_host(loads, P)
        pi_o, G_o = oracle.lpt_placement(loads, P)
        np.testing.assert_array_equal(pi, pi_o)
        np.testing.assert_array_equal(G, G_o)
        assert moe.moe_rank_load_summary_host(G) == pytest.approx(oracle.rank_metrics(G),
                                                                   rel=1e-12)
    with pytest.raises(moe.MoEError):
        moe.moe_lpt_placement_host(np.ones(10, np.int64), 3)  # E not a multiple of P
