"""Pins for the CPU oracle: checks against facts fixed by the pages and by
mathematics (hand-derived fixtures, closed forms, special cases, brute force),
never against the oracle itself.  CPU only.

Each test names the plausible oracle mistake it would catch.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def f32_to_bf16_bits(a):
    """Round-to-nearest-even float32 -> bf16 bits, written here independently."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits(a):
    """Exact bf16 bits of values that bf16 represents exactly."""
    a = np.asarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "fixture value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def f32(u16):
    return synth.bf16_bits_to_f32(np.asarray(u16, dtype=np.uint16))


def silu64(g):
    return g / (1.0 + np.exp(-g))


def key_order(lrow):
    """Expert order by (logit descending, index ascending)."""
    return sorted(range(len(lrow)), key=lambda e: (-float(lrow[e]), e))


# ------------------------------------------------------------------ router ---
def test_router_fma_order_golden():
    """Pins reading R1 (ascending-h FMA chain). Catches a reversed, pairwise or
    split reduction order and a dropped term."""
    g = load("router_fma_order.json")
    x = bf16_bits(g["x"])
    wr = np.array(g["w_router"], dtype=np.float32)
    l = oracle.router_logits(x, wr)
    np.testing.assert_array_equal(l, np.array(g["expected_logits"], dtype=np.float32))
    idx, w = oracle.route(x, wr, None, g["k"])
    np.testing.assert_array_equal(idx, g["expected_idx"])
    np.testing.assert_array_equal(w, np.array(g["expected_w"], dtype=np.float32))


@pytest.mark.parametrize("H,E", [(16, 8), (128, 8), (64, 64), (96, 256)])
def test_router_logits_match_exact_dot_product(H, E):
    """|l - exact| <= H*u*sum|x*w| (FP32 summation error bound, u = 2^-24).
    Catches a transposed W_r, a wrong stride, a dropped or doubled term."""
    T = 37
    x = synth.normal_bf16(5, synth.TID_MISC, (T, H), 1.0)
    wr = synth.normal_f32(5, synth.TID_WR, (H, E), 0.02)
    l = oracle.router_logits(x, wr).astype(np.float64)
    xf = f32(x).astype(np.float64)
    exact = xf @ wr.astype(np.float64)
    bound = H * 2.0 ** -24 * (np.abs(xf) @ np.abs(wr.astype(np.float64))) + 1e-30
    assert np.all(np.abs(l - exact) <= bound)


def test_router_bias_is_one_fp32_add():
    """The per-expert bias is added once to the finished FP32 logit.
    Catches a bias added per term, scaled, or to the probabilities."""
    T, H, E = 19, 32, 16
    x = synth.normal_bf16(1, synth.TID_MISC, (T, H), 1.0)
    wr = synth.normal_f32(1, synth.TID_WR, (H, E), 0.02)
    b = synth.zipf_bias(E, 1.0)
    l0 = oracle.router_logits(x, wr)
    l1 = oracle.router_logits(x, wr, b)
    np.testing.assert_array_equal(l1, (l0 + b).astype(np.float32))


def test_router_tie_rule_golden():
    """Ties go to the lower expert index; slots ordered by probability.
    Catches selection by higher index, unstable ordering, or an unsorted output."""
    g = load("router_ties.json")
    x = bf16_bits(g["x"])
    wr = np.array(g["w_router"], dtype=np.float32)
    idx, w = oracle.route(x, wr, None, g["k"])
    np.testing.assert_array_equal(idx, g["expected_idx"])
    np.testing.assert_allclose(w, g["expected_w_closed_form"], rtol=3e-7, atol=0)


def _tie_heavy_router(T, H, E, seed):
    """x and W_r on coarse grids so equal logits are common (exact FP32 sums)."""
    x = synth.uniform_i32(seed, synth.TID_MISC, (T, H), -2, 3).astype(np.float32)
    wr = synth.uniform_i32(seed, synth.TID_WR, (H, E), -2, 3).astype(np.float32) * 0.25
    return bf16_bits(x), wr


@pytest.mark.parametrize("E,k", [(8, 2), (8, 1), (8, 8), (6, 3), (5, 4), (8, 5)])
def test_topk_bruteforce_exhaustive(E, k):
    """Brute force over all C(E, k) subsets: exactly one subset has every member
    beating every non-member under (logit desc, index asc); it must be the
    oracle's, in key order.  Catches wrong tie rule, wrong slot order, selection
    on a wrong key, off-by-one in k."""
    T, H = 200, 3
    x, wr = _tie_heavy_router(T, H, E, seed=E * 10 + k)
    l = oracle.router_logits(x, wr)
    idx, _ = oracle.route(x, wr, None, k)
    n_ties = 0
    for t in range(T):
        beats = lambda a, b: (l[t, a] > l[t, b]) or (l[t, a] == l[t, b] and a < b)
        winners = [S for S in itertools.combinations(range(E), k)
                   if all(beats(a, b) for a in S for b in range(E) if b not in S)]
        assert len(winners) == 1
        assert sorted(idx[t].tolist()) == list(winners[0])
        assert idx[t].tolist() == [e for e in key_order(l[t]) if e in winners[0]]
        n_ties += len(set(l[t].tolist())) < E
    assert n_ties > T // 4, "fixture should exercise ties"


def test_weights_closed_form_and_invariants():
    """w_j = exp(l_j - m) / sum_sel exp(l - m) (to FP32 rounding); weights sum to 1
    within k*2^-23 and are non-increasing.  Catches renormalising over all
    experts, a missing max shift, weights in the wrong slot."""
    wl = synth.Workload("pin", T=300, H=64, E=32, k=6, I=64, w_std=0.02)
    x = synth.tokens(wl)
    wr, _ = synth.router(wl)
    wr = wr * 20  # spread logits so weights differ
    l = oracle.router_logits(x, wr).astype(np.float64)
    idx, w = oracle.route(x, wr, None, wl.k)
    sel = np.take_along_axis(l, idx.astype(np.int64), axis=1)
    m = l.max(axis=1, keepdims=True)
    ref = np.exp(sel - m) / np.exp(sel - m).sum(axis=1, keepdims=True)
    np.testing.assert_allclose(w, ref, rtol=2e-6, atol=0)
    assert np.all(np.abs(w.astype(np.float64).sum(axis=1) - 1.0) <= wl.k * 2.0 ** -23)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_k_equals_E_weights_equal_full_softmax():
    """With k = E the renormalised weights are the full softmax in key order."""
    T, H, E = 50, 32, 8
    x = synth.normal_bf16(3, synth.TID_MISC, (T, H), 1.0)
    wr = synth.normal_f32(3, synth.TID_WR, (H, E), 0.3)
    l = oracle.router_logits(x, wr).astype(np.float64)
    idx, w = oracle.route(x, wr, None, E)
    p = np.exp(l - l.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    np.testing.assert_allclose(w, np.take_along_axis(p, idx.astype(np.int64), 1), rtol=2e-6)
    for t in range(T):
        assert idx[t].tolist() == key_order(l[t].astype(np.float32))


def test_one_hot_router_closed_form():
    """Designed router: x[t] = e_{t mod E}, W_r = 10*I, so expert t mod E wins by
    a margin and the rest tie at 0 (lower indices next).  Routing, counts and the
    permutation all have closed forms."""
    T, E, k = 40, 8, 3
    H = E
    x = np.zeros((T, H), dtype=np.float32)
    x[np.arange(T), np.arange(T) % E] = 1.0
    x = bf16_bits(x)
    wr = (10.0 * np.eye(E)).astype(np.float32)
    idx, w = oracle.route(x, wr, None, k)
    for t in range(T):
        top = t % E
        rest = [e for e in range(E) if e != top][: k - 1]
        assert idx[t].tolist() == [top] + rest
    a = math.exp(-10.0)
    np.testing.assert_allclose(w[:, 0], 1 / (1 + (k - 1) * a), rtol=1e-6)
    np.testing.assert_allclose(w[:, 1:], a / (1 + (k - 1) * a), rtol=1e-5)
    counts, offsets, _, _ = oracle.load_stats(idx, E)
    expect = np.zeros(E, np.int64)
    for t in range(T):
        for e in idx[t]:
            expect[e] += 1
    np.testing.assert_array_equal(counts, expect)
    _, ros, sor = oracle.permute(synth.normal_bf16(0, 1, (T, 4), 1.0), idx, offsets, E)
    # closed form: row of (t, j) = offsets[e] + number of earlier tokens that chose e
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            assert ros[t * k + j] == offsets[e] + int((idx[:t] == e).any(axis=1).sum())


# ------------------------------------------------------- load statistics ---
def test_counts_offsets_and_sum():
    """counts = bincount of idx, sum = T*k, offsets = exclusive prefix."""
    T, E, k = 513, 16, 4
    wl = synth.Workload("pin", T=T, H=32, E=E, k=k, I=32, w_std=0.02, zipf_s=1.0)
    wr, b = synth.router(wl)
    idx, _ = oracle.route(synth.tokens(wl), wr * 30, b, k)
    counts, offsets, _, _ = oracle.load_stats(idx, E)
    np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert counts.sum() == T * k
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))


def test_load_stats_closed_forms():
    """Imbalance max/mean - 1 and CV: 0 for perfectly even loads; E-1 and
    sqrt(E-1) when one expert takes everything."""
    E, k = 8, 1
    even = np.arange(64, dtype=np.int32).reshape(64, 1) % E
    _, _, imb, cv = oracle.load_stats(even, E)
    assert imb == 0.0 and cv == 0.0
    one = np.zeros((64, 1), dtype=np.int32)
    _, _, imb, cv = oracle.load_stats(one, E)
    assert imb == pytest.approx(E - 1) and cv == pytest.approx(math.sqrt(E - 1))
    two = np.array([[0], [0], [0], [1]], dtype=np.int32)  # counts [3, 1, 0, 0]
    _, _, imb, cv = oracle.load_stats(two, 4)
    assert imb == pytest.approx(3 / 1 - 1)
    assert cv == pytest.approx(math.sqrt(((3 - 1) ** 2 + 0 + 1 + 1) / 4) / 1)


# ------------------------------------------------------------- permutation ---
@pytest.mark.parametrize("T,E,k", [(1, 4, 2), (97, 8, 2), (300, 64, 8), (64, 5, 5)])
def test_permutation_is_stable_bijection(T, E, k):
    """Bijection on [0, T*k); each token appears k times; rows of each expert in
    ascending token order; x_perm[r] is a byte copy of x[token]; brute-force row
    formula.  Catches an unstable order, overlapping rows, a wrong source row."""
    H = 24
    x = synth.normal_bf16(7, synth.TID_X, (T, H), 1.0)
    wr = synth.normal_f32(7, synth.TID_WR, (H, E), 1.0)
    idx, _ = oracle.route(x, wr, None, k)
    counts, offsets, _, _ = oracle.load_stats(idx, E)
    x_perm, ros, sor = oracle.permute(x, idx, offsets, E)
    R = T * k
    assert sorted(ros.tolist()) == list(range(R))
    np.testing.assert_array_equal(sor[ros], np.arange(R))
    np.testing.assert_array_equal(np.bincount(sor // k, minlength=T), np.full(T, k))
    for e in range(E):
        toks = sor[offsets[e]:offsets[e + 1]] // k
        assert np.all(np.diff(toks) > 0)
        assert np.all(idx[toks].__eq__(e).any(axis=1))
    np.testing.assert_array_equal(x_perm, x[sor // k])
    flat = idx.reshape(-1)
    for s in range(0, R, max(1, R // 200)):
        t, e = s // k, flat[s]
        assert ros[s] == offsets[e] + int((idx[:t] == e).any(axis=1).sum())


@pytest.mark.parametrize("E,k", [(8, 2), (64, 8), (128, 8), (256, 16)])
def test_one_token_rows_follow_from_its_expert_ids(E, k):
    """For a batch of one token the stable permutation is fixed by the token's k
    distinct expert ids alone: offsets[e] = #{j : id_j < e} and the row of slot j
    is offsets[id_j].  The one-token decode path schedules both expert GEMMs by
    this formula before the dispatch has run; here it is checked against the
    oracle's load statistics and permutation."""
    H = 16
    for seed in range(5):
        x = synth.normal_bf16(11 + seed, synth.TID_X, (1, H), 1.0)
        wr = synth.normal_f32(11 + seed, synth.TID_WR, (H, E), 1.0)
        idx, _ = oracle.route(x, wr, None, k)
        ids = idx[0]
        assert len(set(ids.tolist())) == k
        counts, offsets, _, _ = oracle.load_stats(idx, E)
        _, ros, _ = oracle.permute(x, idx, offsets, E, with_x_perm=False)
        formula = np.array([int((ids < e).sum()) for e in range(E + 1)], dtype=np.int32)
        np.testing.assert_array_equal(offsets, formula)
        np.testing.assert_array_equal(ros, formula[ids])


# ------------------------------------------------------------- expert FFN ---
def test_swiglu_one_round_golden():
    """silu(g)*u in FP32, one BF16 round, identity down projection.  Catches gate
    and up swapped, a transposed weight, a second rounding, a wrong activation."""
    g = load("swiglu_one_round.json")
    y, h = oracle.expert_ffn(bf16_bits(g["x_perm"]), np.array(g["offsets"], np.int32),
                             bf16_bits(g["w_gate"]), bf16_bits(g["w_up"]), bf16_bits(g["w_down"]),
                             want_h=True)
    np.testing.assert_array_equal(f32(h), np.array(g["expected_h"], np.float32))
    np.testing.assert_array_equal(y, np.array(g["expected_y"], np.float32))


def _ffn64(xp, offsets, wg, wu, wd):
    """float64 reference with h rounded to bf16 as the pages require."""
    E = wg.shape[0]
    xf = f32(xp).astype(np.float64)
    y = np.zeros((xp.shape[0], wd.shape[2]))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r0 == r1:
            continue
        gg = xf[r0:r1] @ f32(wg[e]).astype(np.float64)
        uu = xf[r0:r1] @ f32(wu[e]).astype(np.float64)
        hh = f32(f32_to_bf16_bits((silu64(gg) * uu).astype(np.float32))).astype(np.float64)
        y[r0:r1] = hh @ f32(wd[e]).astype(np.float64)
    return y


def test_expert_ffn_matches_float64_grouped_reference():
    """Per-expert row groups against a float64 grouped SwiGLU FFN (H != I so a
    transposed operand cannot line up; an empty expert included)."""
    E, H, I = 5, 48, 80
    counts = np.array([7, 0, 13, 1, 9], np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(offsets[-1])
    xp = synth.normal_bf16(2, synth.TID_X_PERM, (R, H), 1.0)
    wg = synth.normal_bf16(2, synth.TID_WG, (E, H, I), 0.2)
    wu = synth.normal_bf16(2, synth.TID_WU, (E, H, I), 0.2)
    wd = synth.normal_bf16(2, synth.TID_WD, (E, I, H), 0.2)
    y = oracle.expert_ffn(xp, offsets, wg, wu, wd)
    ref = _ffn64(xp, offsets, wg, wu, wd)
    err = np.abs(y - ref)
    scale = np.abs(ref).max()
    # FP32 accumulation error plus rare BF16 rounding flips of h
    assert err.max() <= 2e-2 * scale
    assert np.linalg.norm(y - ref) <= 2e-3 * np.linalg.norm(ref)


def _dense_layer64(x, wg, wu, wd):
    xf = f32(x).astype(np.float64)
    gg = xf @ f32(wg).astype(np.float64)
    uu = xf @ f32(wu).astype(np.float64)
    return (silu64(gg) * uu) @ f32(wd).astype(np.float64)


def test_single_expert_layer_is_dense_swiglu_ffn():
    """E = 1, k = 1: the routed layer is the textbook dense SwiGLU FFN and the
    routing weight is exactly 1 (torch-free float64 reference)."""
    wl = synth.Workload("dense", T=33, H=64, E=1, k=1, I=96, w_std=0.1)
    inp = synth.layer_inputs(wl)
    out, idx, w, counts = oracle.layer_fwd(inp["x"], inp["wr"], None, inp["wg"], inp["wu"],
                                           inp["wd"], 1)
    assert np.all(idx == 0) and np.all(w == 1.0) and counts.tolist() == [33]
    ref = _dense_layer64(inp["x"], inp["wg"][0], inp["wu"][0], inp["wd"][0])
    o = f32(out).astype(np.float64)
    assert np.abs(o - ref).max() <= 2e-2
    assert np.linalg.norm(o - ref) <= 5e-3 * np.linalg.norm(ref)


def test_identical_experts_give_dense_ffn_for_any_routing():
    """All experts share one weight set: routing weights sum to 1, so the layer
    equals the dense FFN whatever the routing."""
    T, H, E, k, I = 64, 32, 6, 3, 48
    x = synth.normal_bf16(4, synth.TID_X, (T, H), 1.0)
    wr = synth.normal_f32(4, synth.TID_WR, (H, E), 0.5)
    wg1 = synth.normal_bf16(4, synth.TID_WG, (1, H, I), 0.15)
    wu1 = synth.normal_bf16(4, synth.TID_WU, (1, H, I), 0.15)
    wd1 = synth.normal_bf16(4, synth.TID_WD, (1, I, H), 0.15)
    rep = lambda a: np.repeat(a, E, axis=0)
    out, _, _, _ = oracle.layer_fwd(x, wr, None, rep(wg1), rep(wu1), rep(wd1), k)
    ref = _dense_layer64(x, wg1[0], wu1[0], wd1[0])
    o = f32(out).astype(np.float64)
    assert np.linalg.norm(o - ref) <= 5e-3 * np.linalg.norm(ref)


# ----------------------------------------------------------------- combine ---
def test_combine_slot_order_and_fma_golden():
    """Slot-order FMA chain from 0, one BF16 round, rows through row_of_slot.
    Catches reversed slot order, separate multiply and add, a wrong row."""
    g = load("combine_order.json")
    out = oracle.combine(np.array(g["y"], np.float32), np.array(g["w"], np.float32),
                         np.array(g["row_of_slot"], np.int32))
    np.testing.assert_array_equal(out, np.array(g["expected_out_bf16_bits"], np.uint16))


def test_combine_single_slot_is_rounding_of_y():
    """k = 1, w = 1: out = bf16(y[row_of_slot])."""
    T, H = 17, 40
    y = synth.normal_f32(9, synth.TID_Y, (T, H), 3.0)
    perm = synth.uniform_i32(9, synth.TID_MISC, (T,), 0, 1 << 30).argsort().astype(np.int32)
    out = oracle.combine(y, np.ones((T, 1), np.float32), perm)
    np.testing.assert_array_equal(out, f32_to_bf16_bits(y[perm]))


def test_combine_matches_float64_weighted_sum():
    """Weighted sum of k gathered rows within FP32 + one BF16 rounding."""
    T, H, k, R = 40, 32, 4, 160
    y = synth.normal_f32(8, synth.TID_Y, (R, H), 1.0)
    w = synth.uniform_f32(8, synth.TID_TOPK_W, (T, k), 0.0, 1.0)
    ros = np.random.default_rng(0).permutation(R).astype(np.int32).reshape(T, k)
    out = f32(oracle.combine(y, w, ros)).astype(np.float64)
    ref = np.einsum("tk,tkh->th", w.astype(np.float64), y[ros].astype(np.float64))
    assert np.all(np.abs(out - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


# ------------------------------------------------------------ whole layer ---
def test_layer_equals_composition_and_tiny_workload_sane():
    """layer_fwd = route -> load_stats -> permute -> expert_ffn -> combine, and
    on the tiny workload it matches a float64 per-token reference."""
    wl = synth.WORKLOADS["tiny"]
    inp = synth.layer_inputs(wl)
    out, idx, w, counts = oracle.layer_fwd(inp["x"], inp["wr"], inp["bias"], inp["wg"],
                                           inp["wu"], inp["wd"], wl.k)
    i2, w2 = oracle.route(inp["x"], inp["wr"], inp["bias"], wl.k)
    np.testing.assert_array_equal(idx, i2)
    np.testing.assert_array_equal(w, w2)
    c2, off, _, _ = oracle.load_stats(idx, wl.E)
    np.testing.assert_array_equal(counts, c2)
    xp, ros, _ = oracle.permute(inp["x"], idx, off, wl.E)
    y = oracle.expert_ffn(xp, off, inp["wg"], inp["wu"], inp["wd"])
    np.testing.assert_array_equal(out, oracle.combine(y, w, ros))
    # float64 per-token reference
    xf = f32(inp["x"]).astype(np.float64)
    ref = np.zeros((wl.T, wl.H))
    for t in range(wl.T):
        for j in range(wl.k):
            e = idx[t, j]
            gg = xf[t] @ f32(inp["wg"][e]).astype(np.float64)
            uu = xf[t] @ f32(inp["wu"][e]).astype(np.float64)
            ref[t] += float(w[t, j]) * ((silu64(gg) * uu) @ f32(inp["wd"][e]).astype(np.float64))
    o = f32(out).astype(np.float64)
    assert np.abs(o - ref).max() <= 2e-2
    assert np.linalg.norm(o - ref) <= 5e-3 * np.linalg.norm(ref)


# ------------------------------------------------------ router variants ---
def test_exp_cw_matches_float64_exp():
    """Cody-Waite + degree-7 Taylor exp: within 2^-23 relative of the float64
    exponential over the range sigmoid scores use; exact at 0."""
    import math
    assert oracle.exp_cw(0.0) == 1.0
    for v in np.linspace(-80.0, 80.0, 4001):
        v = float(np.float32(v))
        ref = math.exp(v)
        assert abs(oracle.exp_cw(v) - ref) <= 2.0 ** -23 * ref, v


def test_sigmoid_router_bias_only_selects():
    """GLM's rule: the correction bias changes which experts are chosen but the
    weights come from the pre-bias sigmoid scores, normalised over the chosen.
    Catches a bias added to the weights, a softmax instead of the sigmoid, a
    missing renormalisation."""
    import math
    x = bf16_bits([[1.0]])
    wr = np.array([[0.0, 1.0, 2.0, 3.0]], np.float32)  # logits 0, 1, 2, 3
    sig = [1 / (1 + math.exp(-v)) for v in (0.0, 1.0, 2.0, 3.0)]
    idx, w = oracle.route_ex(x, wr, None, 2, kind=oracle.ROUTER_SIGMOID)
    assert idx.tolist() == [[3, 2]]
    np.testing.assert_allclose(w[0], [sig[3] / (sig[3] + sig[2]), sig[2] / (sig[3] + sig[2])],
                               rtol=1e-6)
    bias = np.array([1.0, 0.0, 0.0, 0.0], np.float32)
    idx, w = oracle.route_ex(x, wr, bias, 2, kind=oracle.ROUTER_SIGMOID)
    assert idx.tolist() == [[0, 3]]  # keys 1.5, .73, .88, .95
    np.testing.assert_allclose(w[0], [sig[0] / (sig[0] + sig[3]), sig[3] / (sig[0] + sig[3])],
                               rtol=1e-6)
    # the softmax router instead adds the bias to the logits: 1, 1, 2, 3 -> [3, 2]
    idx, _ = oracle.route_ex(x, wr, bias, 2, kind=oracle.ROUTER_SOFTMAX)
    assert idx.tolist() == [[3, 2]]


def test_sigmoid_router_ties_and_sums():
    """Equal keys go to the lower index; weights sum to one; random inputs agree
    with a float64 restatement of the rule up to FP32 rounding."""
    T, H, E, k = 200, 32, 16, 4
    x, wr = _tie_heavy_router(T, H, E, seed=3)
    l = oracle.router_logits(x, wr).astype(np.float64)
    bias = (synth.uniform_i32(3, synth.TID_MISC, (E,), -2, 3) * 0.125).astype(np.float32)
    idx, w = oracle.route_ex(x, wr, bias, k, kind=oracle.ROUTER_SIGMOID)
    s = 1.0 / (1.0 + np.exp(-l))
    for t in range(T):
        key = s[t] + bias
        order = sorted(range(E), key=lambda e: (-key[e], e))
        # keys equal in float64 are equal in FP32 here (coarse grids), so the order is pinned
        if len(set(np.round(key, 6))) == E:
            assert idx[t].tolist() == order[:k]
        sel = s[t][idx[t]]
        np.testing.assert_allclose(w[t], sel / sel.sum(), rtol=2e-6)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1) <= k * 2.0 ** -23)


def test_weights_bf16_flag_rounds_each_weight():
    """weights_bf16: every weight is the round-to-nearest-even bf16 of the FP32
    weight (for both router kinds)."""
    wl = synth.Workload("p", T=64, H=64, E=16, k=4, I=64, w_std=0.02, zipf_s=1.0)
    x = synth.tokens(wl)
    wr, b = synth.router(wl)
    for kind in (oracle.ROUTER_SOFTMAX, oracle.ROUTER_SIGMOID):
        i32, w32 = oracle.route_ex(x, wr * 10, b, wl.k, kind=kind)
        i16, w16 = oracle.route_ex(x, wr * 10, b, wl.k, kind=kind, weights_bf16=True)
        np.testing.assert_array_equal(i16, i32)
        np.testing.assert_array_equal(w16, f32(f32_to_bf16_bits(w32)))


def test_combine_scaled_closed_form():
    """Scale 1 reproduces the plain combine; scale 2.5 with k = 1, w = 1 gives
    bf16(2.5 y); the scale multiplies each weight before the FMA chain."""
    T, H, k, R = 16, 24, 3, 48
    y = synth.normal_f32(4, synth.TID_Y, (R, H), 1.0)
    w = synth.uniform_f32(4, synth.TID_TOPK_W, (T, k), 0.0, 1.0)
    ros = np.random.default_rng(1).permutation(R).astype(np.int32).reshape(T, k)
    np.testing.assert_array_equal(oracle.combine_scaled(y, w, ros, 1.0), oracle.combine(y, w, ros))
    one = oracle.combine_scaled(y[:T], np.ones((T, 1), np.float32), np.arange(T, dtype=np.int32),
                                2.5)
    np.testing.assert_array_equal(one, f32_to_bf16_bits((np.float32(2.5) * y[:T]).astype(np.float32)))
    ref = np.einsum("tk,tkh->th", 2.5 * w.astype(np.float64), y[ros].astype(np.float64))
    got = f32(oracle.combine_scaled(y, w, ros, 2.5)).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


# ------------------------------------- placement, rank loads, multiplicity ---
def test_lpt_placement_hand_example():
    """Algorithm 1 traced by hand: loads [10,9,8,7,1,1,1,1], 2 ranks of 4 slots.
    Order e0..e7; e0->r0 (10), e1->r1 (9), e2->r1 (17), e3->r0 (17), e4 ties ->
    r0 (18), e5->r1 (18), e6 ties -> r0 (19), e7->r1 (19).  Catches a wrong sort
    key, a wrong tie rule, slots filled out of order, a missing capacity check."""
    pi, G = oracle.lpt_placement([10, 9, 8, 7, 1, 1, 1, 1], 2)
    assert pi.tolist() == [0, 4, 5, 1, 2, 6, 3, 7]
    assert G.tolist() == [19, 19]


def test_lpt_placement_invariants():
    """Random loads: a permutation of slots, exactly E/P experts per rank, rank
    loads = sums of their experts' loads (Eq. 10), the classic LPT bound
    max G <= sum L / P + max L, and no worse than identity placement."""
    rng = np.random.default_rng(0)
    for E, P in [(64, 8), (128, 16), (256, 8), (12, 3)]:
        loads = rng.zipf(1.5, E).astype(np.int64) * 100 + rng.integers(0, 50, E)
        pi, G = oracle.lpt_placement(loads, P)
        assert sorted(pi.tolist()) == list(range(E))
        owner = pi // (E // P)
        assert np.all(np.bincount(owner, minlength=P) == E // P)
        np.testing.assert_array_equal(G, np.bincount(owner, weights=loads, minlength=P))
        assert G.max() <= loads.sum() / P + loads.max()
        ident = np.bincount(np.arange(E) // (E // P), weights=loads, minlength=P)
        assert G.max() <= ident.max()


def test_rank_metrics_closed_forms():
    assert oracle.rank_metrics([5, 5, 5, 5]) == (0.0, 1.0)
    cv, eta = oracle.rank_metrics([6, 2])  # mean 4, std 2, max 6
    assert cv == pytest.approx(0.5) and eta == pytest.approx(4 / 6)


def test_weighted_counts():
    """q = 1 gives the plain counts; sum = k * sum(q); brute force."""
    T, E, k = 100, 16, 4
    idx = np.argsort(synth.uniform_f32(1, synth.TID_TOPK_IDX, (T, E), 0, 1), axis=1)[:, :k]
    idx = idx.astype(np.int32)
    c, _, _, _ = oracle.load_stats(idx, E)
    np.testing.assert_array_equal(oracle.weighted_counts(idx, np.ones(T, np.int32), E), c)
    q = synth.uniform_i32(1, synth.TID_MISC, (T,), 1, 9)
    wc = oracle.weighted_counts(idx, q, E)
    assert wc.sum() == k * q.sum()
    ref = np.zeros(E, np.int64)
    for t in range(T):
        for e in idx[t]:
            ref[e] += q[t]
    np.testing.assert_array_equal(wc, ref)


def test_permute_remap_groups_by_physical_slot():
    """The dispatcher remap: rows grouped by physical slot pi(e), stable within a
    slot; with the identity map it is the plain permutation."""
    T, H, E, k = 90, 16, 8, 2
    x = synth.normal_bf16(2, synth.TID_X, (T, H), 1.0)
    wr = synth.normal_f32(2, synth.TID_WR, (H, E), 1.0)
    idx, _ = oracle.route(x, wr, None, k)
    c, off, _, _ = oracle.load_stats(idx, E)
    ident = np.arange(E, dtype=np.int32)
    a = oracle.permute(x, idx, off, E)
    b = oracle.permute_remap(x, idx, ident, off, E)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)
    pi, _ = oracle.lpt_placement(c.astype(np.int64), 2)
    phys_counts = np.zeros(E, np.int64)
    phys_counts[pi] = c
    poff = np.concatenate([[0], np.cumsum(phys_counts)]).astype(np.int32)
    xp, ros, sor = oracle.permute_remap(x, idx, pi, poff, E)
    for slot in range(E):
        toks = sor[poff[slot]:poff[slot + 1]] // k
        e = int(np.flatnonzero(pi == slot)[0])
        assert np.all(np.diff(toks) > 0) and np.all((idx[toks] == e).any(axis=1))
    np.testing.assert_array_equal(xp, x[sor // k])


# ------------------------------------------- sharded experts: FP64 tree ---
from fractions import Fraction  # noqa: E402


def bf16_value(bits):
    """Exact value of bf16 bits as a Fraction (finite values only)."""
    bits = int(bits)
    sign = -1 if bits & 0x8000 else 1
    ex = (bits >> 7) & 0xFF
    man = bits & 0x7F
    assert ex != 0xFF
    if ex == 0:
        return sign * Fraction(man) * Fraction(2) ** -133
    return sign * (Fraction(128 + man) * Fraction(2) ** (ex - 134))


def is_nearest_even_bf16(q, bits):
    """bits is the round-to-nearest-even bf16 of the exact value q: no finite bf16
    neighbour is nearer, and on a tie the kept mantissa is even."""
    bits = int(bits)
    if (bits & 0x7FFF) == 0x7F80:  # infinity: q at or beyond max + half a spacing
        return abs(q) >= bf16_value(0x7F7F) + Fraction(2) ** (127 - 8)
    v = bf16_value(bits)
    if v != 0 and (v > 0) != (q > 0):
        return False
    mag = bits & 0x7FFF
    s = bits & 0x8000
    d = abs(q - v)
    for nb in (mag - 1, mag + 1):
        if nb < 0:
            continue
        if nb >= 0x7F80:
            continue
        dn = abs(q - bf16_value(s | nb))
        if dn < d:
            return False
        if dn == d and (mag & 1):
            return False
    if mag == 0 and q != 0:  # rounded to zero: the zero keeps the sign of q
        return (q < 0) == bool(s)
    return True


def test_f64_to_bf16_is_round_to_nearest_even():
    """Catches double rounding through FP32, truncation, a wrong tie rule, a
    wrong subnormal spacing and a missed overflow: each result is checked against
    its exact neighbours."""
    rng = np.random.default_rng(11)
    xs = [1 + 2 ** -8 + 2 ** -40, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8 + 2 ** -60),
          2 ** -134, 3 * 2 ** -135, 2 ** -133 * 1.5, 2 ** -140, 2 ** -127 * 1.75,
          3.3895313892515355e38, 3.39e38, 3.4e38, -1e300, 1e-300, 0.0, -0.0]
    xs += list(rng.standard_normal(2000) * 10.0 ** rng.integers(-40, 38, 2000))
    # values at and near every kind of bf16 tie
    for b in rng.integers(0x0001, 0x7F7F, 500):
        lo, hi = bf16_value(int(b)), bf16_value(int(b) + 1)
        mid = (lo + hi) / 2
        xs += [float(mid), float(mid) * (1 + 2 ** -45), float(mid) * (1 - 2 ** -45)]
    for x in xs:
        bits = oracle.f64_to_bf16(x)
        if x == 0.0:
            assert bits == (0x8000 if math.copysign(1, x) < 0 else 0)
            continue
        assert is_nearest_even_bf16(Fraction(x), bits), (x, hex(bits))
        assert (bits >> 15) == (1 if x < 0 else 0)


def test_f64_to_bf16_equals_library_rounding_on_f32_values():
    """Values that FP32 holds exactly: one rounding from FP64 equals torch's
    float32 -> bfloat16 (round to nearest even)."""
    import torch
    f = synth.normal_f32(5, synth.TID_MISC, (4000,), 3.0)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f64_to_bf16(float(v)) for v in f], np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_fp64_tree_golden():
    """Hand-derived cases: pairs vs left-to-right, the odd carry at 3 and 5
    contributors, FP64 vs FP32 accumulation, one final rounding, signed zeros."""
    fx = load("fp64_tree.json")
    for c in fx["cases"]:
        p = np.array(c["partials_bf16_bits"], np.uint16).reshape(-1, 1)
        assert int(oracle.tree_reduce(p)[0]) == c["expected_bf16_bits"], c["name"]


def test_fp64_tree_is_rounded_exact_sum_when_fp64_holds_every_node():
    """Partials within a 2^20 range: every FP64 partial sum is exact, so the
    tree's result is the exact sum rounded once.  Catches a dropped contributor,
    a wrong carry, FP32 accumulation and a second rounding, for G = 1..16."""
    rng = np.random.default_rng(12)
    for G in range(1, 17):
        vals = rng.standard_normal((G, 300)) * 2.0 ** rng.integers(-10, 10, (G, 300))
        p = f32_to_bf16_bits(vals.astype(np.float32))
        out = oracle.tree_reduce(p)
        for n in range(p.shape[1]):
            q = sum(bf16_value(b) for b in p[:, n])
            assert is_nearest_even_bf16(q, out[n]) or (q == 0 and out[n] in (0, 0x8000)), (G, n)


def test_sharded_combine_golden():
    fx = load("sharded_combine.json")
    for c in fx["cases"]:
        sh = None if c["shared"] is None else np.array(c["shared"], np.float32)
        out, parts = oracle.combine_sharded(np.array(c["y"], np.float32),
                                            np.array(c["w"], np.float32),
                                            np.array(c["idx"], np.int32),
                                            np.array(c["row_of_slot"], np.int32),
                                            np.array(c["owner"], np.int32), c["G"], 1.0, sh,
                                            want_partials=True)
        np.testing.assert_array_equal(parts, np.array(c["expected_partials_bf16_bits"]),
                                      err_msg=c["name"])
        np.testing.assert_array_equal(out, np.array(c["expected_out_bf16_bits"]),
                                      err_msg=c["name"])


def _sharded_case(T=40, H=24, E=12, k=4, seed=13):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ros = rng.permutation(T * k).astype(np.int32).reshape(T, k)
    y = synth.normal_f32(seed, synth.TID_Y, (T * k, H), 1.0)
    w = synth.uniform_f32(seed, synth.TID_TOPK_W, (T, k), 0.0, 1.0)
    return idx, ros, y, w


def test_sharded_combine_one_rank_is_the_combine():
    """G = 1 (or every expert on rank 0 of G = 4, the other partials +0): the
    output is the pinned slot-order combine, bit for bit."""
    idx, ros, y, w = _sharded_case()
    E = 12
    ref = oracle.combine_scaled(y, w, ros, 2.5)
    for G in (1, 4):
        out = oracle.combine_sharded(y, w, idx, ros, np.zeros(E, np.int32), G, 2.5)
        np.testing.assert_array_equal(out, ref)


def test_sharded_partials_are_combines_of_owned_rows():
    """Rank g's partial equals the plain combine of y with every row whose expert
    another rank owns replaced by zeros.  Catches owner looked up by slot instead
    of by expert, and a partial that skips the rounding."""
    idx, ros, y, w = _sharded_case()
    E, G, T, k = 12, 3, 40, 4
    owner = (np.arange(E) * 7 % G).astype(np.int32)
    out, parts = oracle.combine_sharded(y, w, idx, ros, owner, G, 1.0, want_partials=True)
    for g in range(G):
        yg = y.copy()
        for t in range(T):
            for j in range(k):
                if owner[idx[t, j]] != g:
                    yg[ros[t, j]] = 0.0
        np.testing.assert_array_equal(parts[g], oracle.combine(yg, w, ros))
    np.testing.assert_array_equal(out, oracle.tree_reduce(parts))


def test_sharded_combine_close_to_float64_sum():
    idx, ros, y, w = _sharded_case(T=64, H=32, E=16, k=6, seed=14)
    owner = (np.arange(16) // 4).astype(np.int32)
    sh = synth.normal_f32(15, synth.TID_MISC, (4, 64, 32), 0.5)
    out = f32(oracle.combine_sharded(y, w, idx, ros, owner, 4, 1.0, sh))
    ref = np.einsum("tj,tjc->tc", w.astype(np.float64), y[ros].astype(np.float64)) + sh.sum(0)
    bound = 2.0 ** -8 * (np.abs(y[ros]).max() * w.sum(1, keepdims=True) * 1.0 + np.abs(sh).sum(0)) \
        + 2.0 ** -8 * np.abs(ref)
    assert np.all(np.abs(out - ref) <= bound)


def _swiglu_f64(x, wg, wu, wd):
    g = x @ wg
    u = x @ wu
    h = f32(f32_to_bf16_bits((silu64(g) * u).astype(np.float32)))
    return h.astype(np.float64) @ wd


def test_shared_expert_shards():
    """Shard g uses intermediate columns [g*Is/G, (g+1)*Is/G) only (changing
    another shard's columns leaves it unchanged), each shard is the dense SwiGLU
    FFN of its slice, and the shards add up to the dense FFN over all of Is."""
    T, H, Is, G = 20, 32, 48, 4
    x = synth.normal_bf16(16, synth.TID_X, (T, H), 1.0)
    wg = synth.normal_bf16(16, synth.TID_WG, (H, Is), 0.2)
    wu = synth.normal_bf16(16, synth.TID_WU, (H, Is), 0.2)
    wd = synth.normal_bf16(16, synth.TID_WD, (Is, H), 0.2)
    ys = oracle.shared_expert(x, wg, wu, wd, G)
    X = f32(x).astype(np.float64)
    Wg, Wu, Wd = (f32(a).astype(np.float64) for a in (wg, wu, wd))
    Ig = Is // G
    for g in range(G):
        sl = slice(g * Ig, (g + 1) * Ig)
        ref = _swiglu_f64(X, Wg[:, sl], Wu[:, sl], Wd[sl])
        np.testing.assert_allclose(ys[g], ref, rtol=0, atol=2e-3 * np.abs(ref).max() + 1e-6)
    dense = _swiglu_f64(X, Wg, Wu, Wd)
    np.testing.assert_allclose(ys.astype(np.float64).sum(0), dense, rtol=0,
                               atol=2e-3 * np.abs(dense).max() + 1e-6)
    wg2 = wg.copy()
    wg2[:, Ig:2 * Ig] ^= 0x0040  # change shard 1's gate columns
    ys2 = oracle.shared_expert(x, wg2, wu, wd, G)
    np.testing.assert_array_equal(ys2[[0, 2, 3]], ys[[0, 2, 3]])
    assert not np.array_equal(ys2[1], ys[1])
