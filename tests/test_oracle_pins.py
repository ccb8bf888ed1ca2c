"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks one part of ``oracle`` against a closed form, an invariant
the pages state, an independent brute-force or native-fp32 restatement, or a
printed worked example, so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small_layer(out=8, K=256, n=64, seed=3, outliers=(5, 130), factor=25.0, w_std=0.02):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((out, K)) * w_std).astype(np.float32)
    X = rng.standard_normal((n, K)).astype(np.float32)
    for c in outliers:
        X[:, c] *= factor
    return W.astype(np.float64), workloads.round_to_bf16(X).astype(np.float64)


# ---------------------------------------------------------------- rounding helpers


def test_f32_rounds_ties_to_even():
    one = 1.0
    ulp = 2.0**-23
    assert O.f32(one + ulp / 2) == one  # tie -> even (1.0)
    assert O.f32(one + 1.5 * ulp) == one + 2 * ulp  # tie -> even mantissa
    assert O.f32(one + 0.75 * ulp) == one + ulp
    assert O.f32(-(one + ulp / 2)) == -one


def test_fp16_storage_rounds_ties_to_even():
    # 1 + 2^-11 is halfway between fp16 1.0 and 1 + 2^-10: ties go to 1.0.
    vals = np.array([1 + 2.0**-11, 1 + 3 * 2.0**-11, 2.0**-20, 65504.0, 3.0], dtype=np.float32)
    h = vals.astype(np.float16).astype(np.float64)
    assert h[0] == 1.0
    assert h[1] == 1 + 2 * 2.0**-10
    assert h[2] == 2.0**-20  # fp16 subnormal, exact
    assert h[3] == 65504.0
    assert h[4] == 3.0


# ---------------------------------------------------------------- statistics


def test_channel_importance_brute_force():
    rng = np.random.default_rng(0)
    X = rng.standard_normal((5, 7))
    got = O.channel_importance(X)
    for j in range(7):
        acc = 0.0
        for t in range(5):
            acc += abs(float(X[t, j]))
        assert got[j] == pytest.approx(acc / 5, rel=1e-15)


def test_alpha_grid_endpoints():
    g = O.alpha_grid(20)
    assert len(g) == 20 and g[0] == 0.0 and g[-1] == pytest.approx(0.95)
    assert np.all(np.diff(g) > 0)


def test_alpha_zero_gives_unit_scale_exactly():
    sx = np.array([1e-7, 0.3, 7.0, 55.0])
    for norm in (False, True):
        s = O.awq_scales(sx, 0.0, normalize=norm)
        assert np.all(s == 1.0)


def test_scale_clamp_and_power_closed_form():
    sx = np.array([1e-6, 0.5, 2.0, 40.0])
    s = O.awq_scales(sx, 0.5, normalize=False)
    expect = np.sqrt(np.array([O.CLAMP_MIN, 0.5, 2.0, 40.0]))
    np.testing.assert_allclose(s, expect, rtol=1e-15)
    sn = O.awq_scales(sx, 0.5, normalize=True)
    c = math.sqrt(expect.max() * expect.min())
    np.testing.assert_allclose(sn, expect / c, rtol=1e-15)
    assert sn.max() * sn.min() == pytest.approx(1.0, rel=1e-14)


# ---------------------------------------------------------------- quantiser


def _native_fp32_rtn_group(vals, floor=np.float32(1e-5), levels=15):
    """Independent per-group asymmetric RTN in native fp32 scalar arithmetic
    (`levels` = 2^b - 1 steps across the group's range)."""
    v = [np.float32(x) for x in vals]
    hi, lo = max(v), min(v)
    d = np.float32(np.float32(hi - lo) / np.float32(levels))
    if d < floor:
        d = floor
    z = np.float32(np.rint(np.float32(-lo / d)))
    codes = []
    for x in v:
        c = np.float32(np.rint(np.float32(x / d))) + z
        codes.append(min(max(float(c), 0.0), float(levels)))
    return codes, float(d), float(z)


def test_alpha_zero_is_plain_rtn_native_fp32():
    """alpha = 0 gives s = 1, so the search's quantiser is plain group RTN."""
    W, X = _small_layer(out=6, K=256)
    s = O.awq_scales(O.channel_importance(X), 0.0)
    W_hat = O.fake_quantize(W, s)
    for r in range(W.shape[0]):
        for g in range(W.shape[1] // 128):
            vals = W[r, g * 128:(g + 1) * 128]
            codes, d, z = _native_fp32_rtn_group(vals)
            expect = [(c - z) * d for c in codes]
            np.testing.assert_array_equal(W_hat[r, g * 128:(g + 1) * 128], expect)


def test_pinned_quantizer_matches_native_fp32_with_scales():
    W, X = _small_layer(out=6, K=256, seed=11)
    sx = O.channel_importance(X)
    for alpha in (0.25, 0.6, 0.95):
        s32 = O.f32(O.awq_scales(sx, alpha))
        V = O.f32(W * s32[None, :])
        q, d, z = O.quantize_groups(V)
        for r in range(W.shape[0]):
            for g in range(2):
                vals = [np.float32(W[r, k]) * np.float32(s32[k]) for k in range(g * 128, (g + 1) * 128)]
                codes, dn, zn = _native_fp32_rtn_group(vals)
                assert d[r, g] == dn and z[r, g] == zn
                np.testing.assert_array_equal(q[r, g * 128:(g + 1) * 128], codes)


def test_scaling_cancels_without_rounding():
    """Scaling identity: with rounding removed, Q(W*s)/s gives back W."""
    W, X = _small_layer(out=5, K=256, seed=4)
    sx = O.channel_importance(X)
    ident = lambda a: np.asarray(a, dtype=np.float64)  # noqa: E731
    for alpha in (0.0, 0.3, 0.9):
        s = O.awq_scales(sx, alpha)
        W_hat = O.fake_quantize(W, s, pinned=False, round_fn=ident)
        np.testing.assert_allclose(W_hat, W, rtol=1e-12, atol=1e-15)
        # pinned (fp32) steps leave only fp32-rounding residue
        W_hat32 = O.fake_quantize(W, s, pinned=True, round_fn=ident)
        np.testing.assert_allclose(W_hat32, W, rtol=0, atol=1e-6 * np.abs(W).max())


def test_error_at_most_half_a_step_and_codes_in_range():
    W, X = _small_layer(out=16, K=384, seed=5)
    sx = O.channel_importance(X)
    for alpha in O.alpha_grid(20):
        s32 = O.f32(O.awq_scales(sx, alpha))
        V = O.f32(W * s32[None, :])
        q, d, z = O.quantize_groups(V, group=128)
        assert q.min() >= 0 and q.max() <= 15
        assert np.all(z == np.round(z))
        assert np.all(q == np.round(q))
        dq = O.dequantize_groups(q, d, z, 128)
        err = np.abs(V - dq).reshape(16, 3, 128)
        bound = d[:, :, None] * (0.5 + 1e-5)
        assert np.all(err <= bound)


def test_hand_built_groups():
    # all-zero group: delta hits the floor, zero point 0, codes 0, exact zeros back
    V = np.zeros((1, 128))
    q, d, z = O.quantize_groups(V)
    assert d[0, 0] == O.f32(1e-5) and z[0, 0] == 0 and np.all(q == 0)
    # exact ties: range [0, 15] gives delta = 1, z = 0; 2.5 -> 2, 3.5 -> 4 (half to even)
    vals = np.zeros(128)
    vals[1] = 15.0
    vals[2] = 2.5
    vals[3] = 3.5
    vals[4] = 0.5
    q, d, z = O.quantize_groups(vals[None, :])
    assert d[0, 0] == 1.0 and z[0, 0] == 0.0
    assert q[0, 1] == 15 and q[0, 2] == 2 and q[0, 3] == 4 and q[0, 4] == 0
    # one-sign group: all positive, so the zero point is negative; codes still in range
    vals = np.linspace(1.0, 2.0, 128)
    q, d, z = O.quantize_groups(vals[None, :])
    assert z[0, 0] < 0 and q.min() == 0 and q.max() == 15
    dq = O.dequantize_groups(q, d, z)
    assert np.all(np.abs(dq - vals) <= d[0, 0] * 0.5 * (1 + 1e-6))
    # constant nonzero group: floor step, value recovered to within half a step
    vals = np.full(128, 0.02)
    q, d, z = O.quantize_groups(vals[None, :])
    dq = O.dequantize_groups(q, d, z)
    assert np.all(np.abs(dq - 0.02) <= d[0, 0] * 0.5)


# ---------------------------------------------------------------- loss and search


def test_loss_brute_force_tiny():
    rng = np.random.default_rng(9)
    X = rng.standard_normal((3, 128))
    W = rng.standard_normal((4, 128)) * 0.02
    W_hat = O.fake_quantize(W, np.ones(128))
    acc = 0.0
    for t in range(3):
        for r in range(4):
            y = sum(X[t, k] * W_hat[r, k] for k in range(128))
            y0 = sum(X[t, k] * W[r, k] for k in range(128))
            acc += (y - y0) ** 2
    assert O.output_mse(X, W, W_hat) == pytest.approx(acc / 12, rel=1e-10)


def test_literal_and_residual_loss_forms_agree():
    L = workloads.make_layer("tiny")
    W, X = L["W"].astype(np.float64), L["X"].astype(np.float64)
    sx = O.channel_importance(X)
    for alpha in (0.0, 0.5, 0.95):
        W_hat = O.fake_quantize(W, O.awq_scales(sx, alpha))
        a = O.output_mse(X, W, W_hat)
        b = O.output_sq_err_sum(X, W, W_hat) / (X.shape[0] * W.shape[0])
        assert a == pytest.approx(b, rel=1e-12)


def test_normalisation_leaves_losses_unchanged():
    W, X = _small_layer(out=8, K=256, seed=6)
    sx = O.channel_importance(X)
    a = O.search_scale(W, X, sx, normalize=True, pinned=False)
    b = O.search_scale(W, X, sx, normalize=False, pinned=False)
    np.testing.assert_allclose(a["losses"], b["losses"], rtol=1e-10)
    assert a["best_idx"] == b["best_idx"]
    # the pinned (fp32) quantiser moves at most a few codes at rounding ties
    c = O.search_scale(W, X, sx, normalize=True, pinned=True)
    d = O.search_scale(W, X, sx, normalize=False, pinned=True)
    np.testing.assert_allclose(c["losses"], d["losses"], rtol=1e-3)


def test_search_beats_rtn_with_interior_optimum():
    L = workloads.make_layer("tiny")
    W, X = L["W"].astype(np.float64), L["X"].astype(np.float64)
    res = O.search_scale(W, X, O.channel_importance(X))
    losses = res["losses"]
    assert losses[res["best_idx"]] == losses.min()
    assert res["best_idx"] > 0 and losses.min() < 0.9 * losses[0]
    assert res["best_idx"] == int(np.argmin(losses))


def test_first_strict_minimum_wins():
    W, X = _small_layer(out=2, K=128, n=8, outliers=(5, 70))
    res = O.search_scale(W, X, O.channel_importance(X), n_grid=5, loss=lambda X, W, Wh: 1.0)
    assert res["best_idx"] == 0
    vals = iter([3.0, 2.0, 1.0, 1.0, 5.0])
    res = O.search_scale(W, X, O.channel_importance(X), n_grid=5, loss=lambda X, W, Wh: next(vals))
    assert res["best_idx"] == 2


def test_activation_salience_beats_weight_salience():
    """Protecting the high-activation channel lowers output error more than
    protecting the largest-weight channel, and the best single channel to
    protect is an activation outlier (AWQ-devto, "How does AWQ decide which
    weights to protect?")."""
    rng = np.random.default_rng(21)
    out, K, n = 8, 128, 64
    W = rng.standard_normal((out, K)) * 0.02
    X = rng.standard_normal((n, K))
    act_out = [17, 90]
    X[:, act_out] *= 30.0
    big_w = 40  # a channel with large weights but ordinary activations
    W[:, big_w] *= 4.0

    def mse_protect(j, k):
        s = np.ones(K)
        s[j] = k
        return O.output_mse(X, W, O.fake_quantize(W, s, pinned=False))

    base = O.output_mse(X, W, O.fake_quantize(W, np.ones(K), pinned=False))
    best = {}
    for j in range(K):
        best[j] = min(mse_protect(j, k) for k in (1.0, 2.0, 4.0, 8.0))
    j_star = min(best, key=best.get)
    assert j_star in act_out
    act_rank = np.argsort(-np.abs(X).mean(axis=0))[0]
    w_rank = np.argsort(-np.abs(W).mean(axis=0))[0]
    assert act_rank in act_out and w_rank == big_w
    assert best[act_rank] < best[w_rank] and best[act_rank] < base


# ---------------------------------------------------------------- packing


def test_pack_nibble_order_golden():
    cases = json.load(open(os.path.join(GOLDEN, "pack_order.json")))["cases"]
    for c in cases:
        w = O.pack_words(np.array([c["codes"]]))
        assert int(w.view(np.uint32)[0, 0]) == int(c["word_hex"], 16)


def test_pack_roundtrip_and_dequant_bound():
    W, X = _small_layer(out=9, K=256, seed=8)
    s = O.awq_scales(O.channel_importance(X), 0.55)
    p = O.quantize_pack(W, s)
    assert p["qweight"].dtype == np.int32 and p["qweight"].shape == (9, 32)
    np.testing.assert_array_equal(O.unpack_words(p["qweight"], 256), p["codes"])
    V = O.f32(W * O.f32(s)[None, :])
    sc = p["scales"].astype(np.float64)
    zz = p["zeros"].astype(np.float64)
    dq = O.dequantize_groups(p["codes"], sc, zz)
    delta = p["delta"]
    bound = (delta * 0.5 + delta * 2.0**-11 * 15)[:, :, None]
    assert np.all(np.abs(V - dq).reshape(9, 2, 128) <= bound * (1 + 1e-6))


def test_memory_arithmetic_13b_golden():
    g = json.load(open(os.path.join(GOLDEN, "memory_13b.json")))
    rows = g["weights"] // g["group"]
    b = O.packed_bytes(rows, g["group"], group=g["group"])
    assert rows * g["group"] * 2 == g["fp16_bytes"]
    assert b["codes"] == g["int4_code_bytes"]
    assert b["scales"] == pytest.approx(g["scale_bytes_approx"], rel=0.02)
    assert b["codes"] + b["scales"] == pytest.approx(g["total_approx"], rel=0.005)
    assert b["zeros"] == b["scales"]


def test_generator_is_deterministic():
    a = workloads.make_layer("tiny")
    b = workloads.make_layer("tiny")
    np.testing.assert_array_equal(a["W"], b["W"])
    np.testing.assert_array_equal(a["X"], b["X"])
    assert len(a["outlier_channels"]) == 3
    # bf16-exact activations
    workloads.bf16_bits(a["X"])


# ---------------------------------------------------------------- packed-layer product (w4a16)


def test_w4a16_linear_brute_force_from_words():
    # codes read straight from the words with integer shifts, sums by loops
    rng = np.random.default_rng(11)
    M, N, K = 2, 3, 256
    words = rng.integers(0, 2**32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32).view(np.int32)
    sc = rng.uniform(0.001, 0.02, size=(N, K // 128)).astype(np.float16)
    zr = rng.integers(0, 16, size=(N, K // 128)).astype(np.float16)
    x = rng.standard_normal((M, K))
    got = O.w4a16_linear(x, words, sc, zr)
    for m in range(M):
        for r in range(N):
            acc = 0.0
            for k in range(K):
                word = int(words[r, k // 8]) & 0xFFFFFFFF
                q = (word >> (4 * (k % 8))) & 0xF
                acc += x[m, k] * (q - float(zr[r, k // 128])) * float(sc[r, k // 128])
            assert got[m, r] == pytest.approx(acc, rel=1e-12, abs=1e-12)


def test_w4a16_linear_matches_the_searched_weight():
    # the packed layer applied to x / s reproduces x @ W_hat^T of the search's
    # fake-quant (scaling equation), up to the fp16 storage of each step:
    # |fp16(delta) - delta| <= 2^-11 delta, so every product term moves by at
    # most 2^-11 of its size
    W, X = _small_layer(out=16, K=512, n=8)
    sx = O.channel_importance(X)
    s = O.f32(O.awq_scales(sx, 0.55))
    pk = O.quantize_pack(W, s)
    got = O.w4a16_linear(X / s[None, :], pk["qweight"], pk["scales"], pk["zeros"])
    W_hat = O.fake_quantize(W, s)
    ref = X @ W_hat.T
    bound = 2.0**-11 * (np.abs(X) @ np.abs(W_hat).T) + 1e-12
    assert np.all(np.abs(got - ref) <= bound)
    # and it is not trivially close: the quantisation error itself is much larger
    assert np.max(np.abs(X @ W.T - ref)) > 50 * np.max(np.abs(got - ref))


def test_block_search_is_the_output_weighted_mean_of_the_linears():
    # three linears sharing X, searched separately with the same statistic:
    # the block loss of each alpha is their losses weighted by output count
    rng = np.random.default_rng(21)
    K, n = 256, 48
    Ws = [(rng.standard_normal((r, K)) * 0.02) for r in (24, 8, 8)]
    X = rng.standard_normal((n, K))
    X[:, 17] *= 30.0
    X = workloads.round_to_bf16(X.astype(np.float32)).astype(np.float64)
    sx = O.channel_importance(X)
    blk = O.search_scale_block(Ws, X, sx)
    parts = [O.search_scale(W, X, sx)["losses"] for W in Ws]
    outs = np.array([W.shape[0] for W in Ws], dtype=np.float64)
    ref = sum(o * l for o, l in zip(outs, parts)) / outs.sum()
    np.testing.assert_allclose(blk["losses"], ref, rtol=1e-12)
    assert blk["best_idx"] == int(np.argmin(ref))


# ---------------------------------------------------------------- symmetric quantiser (zero point off)


def test_symmetric_quantizer_matches_native_fp32_restatement():
    # "Why does naive 4-bit quantization wreck LLM accuracy?": delta = max|w| / 2^(N-1),
    # Q(w) = delta * round(w / delta); 4-bit storage clamps the rounded value to [-8, 7]
    rng = np.random.default_rng(13)
    V = (rng.standard_normal((6, 256)) * 0.05).astype(np.float32)
    V[2, :128] = np.abs(V[2, :128])  # one-sign group
    V[3, 128:] = -np.abs(V[3, 128:])
    q, delta, z = O.quantize_groups(V.astype(np.float64), zero_point=False)
    assert np.all(z == 8.0)
    for r in range(V.shape[0]):
        for g in range(2):
            grp = V[r, 128 * g:128 * g + 128]
            amax = np.float32(np.max(np.abs(grp)))
            d = np.float32(amax / np.float32(8.0))
            assert delta[r, g] == float(d)
            codes = np.clip(np.rint(grp / d), -8, 7)  # fp32 division, ties to even
            np.testing.assert_array_equal(q[r, 128 * g:128 * g + 128] - 8.0, codes.astype(np.float64))


def test_symmetric_error_bound_and_range():
    rng = np.random.default_rng(14)
    V = rng.standard_normal((5, 384)) * 0.02
    q, delta, z = O.quantize_groups(V, zero_point=False)
    assert q.min() >= 0 and q.max() <= 15
    err = np.abs(V - O.dequantize_groups(q, delta, z))
    d = np.repeat(delta, 128, axis=1)
    top = q == 15  # the positive maximum may clamp from +8 to +7 steps: error up to one step
    assert np.all(err[~top] <= d[~top] / 2 * (1 + 1e-6))
    assert np.all(err[top] <= d[top] * (1 + 1e-6))


# ---------------------------------------------------------------- group sizes and code widths (the quantiser's knobs)


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("w_bit", [2, 3, 4, 8])
def test_group_size_and_width_match_native_fp32(group, w_bit):
    # "AWQ > Salient Weight Preservation", step-size equation: the range over 2^b - 1 levels, for any b;
    # the first page's deployment notes: finer groups carry their own step. Checked group by group
    # against the scalar fp32 restatement, which walks the row in slices of `group`.
    rng = np.random.default_rng(100 * group + w_bit)
    W = O.f32(rng.standard_normal((4, 256)) * 0.02)  # fp32 weights, as the kernels read them
    s32 = O.f32(rng.uniform(0.3, 3.0, 256))
    V = O.f32(W * s32[None, :])
    q, d, z = O.quantize_groups(V, w_bit=w_bit, group=group)
    assert d.shape == (4, 256 // group)
    for r in range(4):
        for g in range(256 // group):
            vals = [np.float32(W[r, k]) * np.float32(s32[k]) for k in range(g * group, (g + 1) * group)]
            codes, dn, zn = _native_fp32_rtn_group(vals, levels=2**w_bit - 1)
            assert d[r, g] == dn and z[r, g] == zn, (r, g)
            np.testing.assert_array_equal(q[r, g * group:(g + 1) * group], codes)


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("w_bit", [2, 3, 4, 8])
def test_symmetric_group_size_and_width_match_native_fp32(group, w_bit):
    # "Why does naive 4-bit quantization wreck LLM accuracy?": delta = max|w| / 2^(N-1); b bits hold
    # -2^(b-1) .. 2^(b-1) - 1 steps
    rng = np.random.default_rng(200 * group + w_bit)
    V = (rng.standard_normal((3, 256)) * 0.05).astype(np.float32)
    half = np.float32(2 ** (w_bit - 1))
    q, delta, z = O.quantize_groups(V.astype(np.float64), w_bit=w_bit, group=group, zero_point=False)
    assert np.all(z == float(half))
    for r in range(3):
        for g in range(256 // group):
            grp = V[r, g * group:(g + 1) * group]
            d = np.float32(np.float32(np.max(np.abs(grp))) / half)
            assert delta[r, g] == float(d)
            codes = np.clip(np.rint(grp / d), -half, half - 1)
            np.testing.assert_array_equal(q[r, g * group:(g + 1) * group] - float(half), codes.astype(np.float64))


@pytest.mark.parametrize("w_bit", [2, 3, 4, 5, 8])
def test_group_of_exact_levels_is_reproduced(w_bit):
    """Closed form: a group whose values are 2^b evenly spaced levels (power-of-two spacing, the zero at
    level z0) has step = the spacing, zero point z0 and codes = the level indices, and dequantises
    exactly. A wrong level count (2^b or 2^b - 2) or a wrong zero point breaks it."""
    levels = 2**w_bit
    group = 128
    rng = np.random.default_rng(w_bit)
    for z0 in (0, 1, levels // 2, levels - 1):
        spacing = 2.0**-7
        idx = np.concatenate([[0, levels - 1], rng.integers(0, levels, group - 2)])
        vals = (idx - z0) * spacing
        q, d, z = O.quantize_groups(vals[None, :], w_bit=w_bit, group=group)
        assert d[0, 0] == spacing and z[0, 0] == z0
        np.testing.assert_array_equal(q[0], idx)
        np.testing.assert_array_equal(O.dequantize_groups(q, d, z, group)[0], vals)


def test_finer_groups_never_widen_the_step():
    """A group of g weights inside a group of 2g has a range no wider than the larger group's, so its
    step is at most the larger group's step (the pages' accuracy/overhead trade-off of finer groups):
    the step of group j at size g is bounded by that of group j // 2 at size 2g."""
    rng = np.random.default_rng(21)
    V = O.f32(rng.standard_normal((8, 512)) * 0.03)
    V[:, 7] = 2.0  # an outlier column widens only the groups that hold it
    steps = {g: O.quantize_groups(V, group=g)[1] for g in (32, 64, 128)}
    for g in (32, 64):
        fine, coarse = steps[g], steps[2 * g]
        assert np.all(fine <= np.repeat(coarse, 2, axis=1))
    # the outlier's 32-group step is far above the others', and only its own groups carry it
    assert steps[32][:, 0].min() > 10 * steps[32][:, 1:].max()
    assert np.all(steps[64][:, 1:] < steps[64][:, :1])


@pytest.mark.parametrize("group", [32, 64])
def test_pack_and_w4a16_with_finer_groups(group):
    """Packed layer with groups of 32 or 64: one fp16 scale and zero per group, codes unchanged by the
    storage, and the product over the words equals the dequantised weight's (brute force)."""
    rng = np.random.default_rng(group)
    W = rng.standard_normal((6, 256)) * 0.02
    s = O.f32(rng.uniform(0.5, 2.0, 256))
    pk = O.quantize_pack(W, s, group=group)
    assert pk["scales"].shape == (6, 256 // group) and pk["zeros"].shape == (6, 256 // group)
    np.testing.assert_array_equal(O.unpack_words(pk["qweight"], 256), pk["codes"])
    x = rng.standard_normal((3, 256))
    y = O.w4a16_linear(x, pk["qweight"], pk["scales"], pk["zeros"], group=group)
    ref = np.zeros((3, 6))
    for t in range(3):
        for r in range(6):
            acc = 0.0
            for k in range(256):
                word = int(pk["qweight"][r, k // 8]) & 0xFFFFFFFF
                code = (word >> (4 * (k % 8))) & 0xF
                gi = k // group
                acc += x[t, k] * (code - float(pk["zeros"][r, gi])) * float(pk["scales"][r, gi])
            ref[t, r] = acc
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- bf16 weight of the prefill product


def test_bf16_rounding_matches_torch_conversion():
    """The oracle's own bf16 rounding against torch's float32 -> bfloat16 conversion (a library routine),
    on random values, exact ties (both directions), signed zeros and values near the bf16 limits."""
    import torch

    rng = np.random.default_rng(3)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-20, 20, 20000),
        # fp32 values exactly halfway between two bf16 values: low 16 bits 0x8000, odd and even bf16 lsb
        (np.arange(1, 2001, dtype=np.uint32) * 0x20000 + 0x3F808000).view(np.float32),
        (np.arange(1, 2001, dtype=np.uint32) * 0x20000 + 0x3F818000).view(np.float32),
        np.array([0.0, -0.0, 1e-38, -1e-38, 3.3e38, -3.3e38], dtype=np.float32),
    ]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16(vals.astype(np.float64))
    np.testing.assert_array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))


def test_expanded_weight_is_the_rounded_dequantised_weight():
    """w4a16_expand_bf16 equals bf16 of (q - z) * scale computed element by element from the words."""
    rng = np.random.default_rng(8)
    W = rng.standard_normal((5, 256)) * 0.02
    pk = O.quantize_pack(W, O.f32(rng.uniform(0.5, 2.0, 256)), group=64)
    Wb = O.w4a16_expand_bf16(pk["qweight"], pk["scales"], pk["zeros"], group=64)
    for r in range(5):
        for k in range(0, 256, 7):
            code = (int(pk["qweight"][r, k // 8]) & 0xFFFFFFFF) >> (4 * (k % 8)) & 0xF
            v = (code - float(pk["zeros"][r, k // 64])) * float(pk["scales"][r, k // 64])
            assert Wb[r, k] == O.bf16(np.array([v]))[0]
    # and it is within half a bf16 step (8 significant bits: 2^-8 relative) of the exact dequantised weight
    exact = O.dequantize_groups(O.unpack_words(pk["qweight"], 256), pk["scales"].astype(np.float64),
                                pk["zeros"].astype(np.float64), 64)
    assert np.all(np.abs(Wb - exact) <= 2.0**-8 * np.abs(exact))
    assert np.any(np.abs(Wb - exact) > 2.0**-9 * np.abs(exact))  # and the bound is not loose by a factor 2


# ---------------------------------------------------------------- randomised pin of the quantiser


def test_quantizer_against_scalar_restatement_randomised():
    """Many random groups (sizes 32/64/128, 2-8 bits, normal, heavy-tailed, one-sign, near-constant and
    tie-laden values) against the scalar fp32 restatement, group by group."""
    rng = np.random.default_rng(99)
    for trial in range(60):
        group = int(rng.choice([32, 64, 128]))
        w_bit = int(rng.integers(2, 9))
        kind = trial % 5
        n = group * 2
        if kind == 0:
            v = rng.standard_normal(n) * 0.05
        elif kind == 1:
            v = rng.standard_t(2, n) * 0.01
        elif kind == 2:
            v = np.abs(rng.standard_normal(n)) + 3.0
        elif kind == 3:
            v = 0.7 + rng.standard_normal(n) * 1e-6
        else:
            levels = 2**w_bit - 1
            v = (rng.integers(0, levels, n) + 0.5) / levels  # exact-tie candidates on a unit range
            v[0], v[1] = 0.0, 1.0
        V = O.f32(v)[None, :]
        q, d, z = O.quantize_groups(V, w_bit=w_bit, group=group)
        for g in range(2):
            vals = V[0, g * group:(g + 1) * group]
            codes, dn, zn = _native_fp32_rtn_group(vals, levels=2**w_bit - 1)
            assert d[0, g] == dn and z[0, g] == zn, (trial, g)
            np.testing.assert_array_equal(q[0, g * group:(g + 1) * group], codes)


# ---------------------------------------------------------------- 2- and 8-bit packing


@pytest.mark.parametrize("w_bit", [2, 8])
def test_pack_order_for_other_widths(w_bit):
    """Hand-written words: column (32/b)*j + k sits in bits [b*k, b*k + b) of word j."""
    per = 32 // w_bit
    q = np.zeros((1, 2 * per), dtype=np.int64)
    q[0, 0] = 1                 # lowest bits of word 0
    q[0, per - 1] = 2**w_bit - 1  # highest bits of word 0
    q[0, per + 1] = 2           # second code of word 1
    words = O.pack_words(q, w_bit).view(np.uint32)
    assert int(words[0, 0]) == 1 | ((2**w_bit - 1) << (32 - w_bit))
    assert int(words[0, 1]) == 2 << w_bit
    np.testing.assert_array_equal(O.unpack_words(O.pack_words(q, w_bit), 2 * per, w_bit), q)


@pytest.mark.parametrize("w_bit", [2, 8])
def test_quantize_pack_other_widths_round_trip(w_bit):
    rng = np.random.default_rng(w_bit)
    W = rng.standard_normal((5, 256)) * 0.02
    s = O.f32(rng.uniform(0.5, 2.0, 256))
    pk = O.quantize_pack(W, s, w_bit=w_bit, group=64)
    assert pk["qweight"].shape == (5, 256 * w_bit // 32)
    np.testing.assert_array_equal(O.unpack_words(pk["qweight"], 256, w_bit), pk["codes"])
    q, d, z = O.quantize_groups(O.f32(W * s[None, :]), w_bit=w_bit, group=64)
    np.testing.assert_array_equal(pk["codes"], q)
    with pytest.raises(ValueError):
        O.quantize_pack(W, s, w_bit=3)


def test_memory_arithmetic_70b_golden():
    """The 70B deployment figure: 140 GB of fp16 weights, 35 GB of 4-bit codes; with one fp16 scale and
    one fp16 zero per 128 weights the reduction lies between the page's 72% and the codes' 75%."""
    g = json.load(open(os.path.join(GOLDEN, "memory_70b.json")))
    rows, cols = 175000, 400000  # 7e10 weights, rows of whole groups of 128 (the counts are per weight)
    assert rows * cols == g["weights"] and cols % 128 == 0
    b = O.packed_bytes(rows, cols, group=128)
    assert rows * cols * 2 == g["fp16_bytes"]
    assert b["codes"] == g["int4_bytes"]
    reduction = 1.0 - b["total"] / g["fp16_bytes"]
    assert g["stated_reduction"] <= reduction <= 0.75


# ---------------------------------------------------------------- the composed search, restated independently


def _torch_group_rtn(V, group=128, qmax=15.0, floor=1e-5):
    """Asymmetric min/max group quantise-dequantise in torch float64, written
    from the step-size equation of "AWQ > Salient Weight Preservation" and the
    zero point of the deployment quant_config, independently of the oracle:
    step = max((max - min) / (2^b - 1), floor), zero = round(-min / step),
    code = clamp(round(v / step) + zero, 0, 2^b - 1), value = (code - zero) * step
    (torch.round rounds half to even)."""
    import torch

    rows, K = V.shape
    g = V.reshape(rows, K // group, group)
    hi = g.amax(dim=2, keepdim=True)
    lo = g.amin(dim=2, keepdim=True)
    step = torch.clamp((hi - lo) / qmax, min=floor)
    zero = torch.round(-lo / step)
    code = torch.clamp(torch.round(g / step) + zero, 0.0, qmax)
    return ((code - zero) * step).reshape(rows, K)


def _torch_search(W, X, n_grid=20):
    """The per-layer grid search of "AWQ: How Activation-Aware Quantization
    Saves 4-bit LLMs" ("How does AWQ protect channels without mixed
    precision?"), step by step in torch float64: the statistic is the mean
    |x| per input channel; for alpha = i / n_grid the scale is the clamped
    statistic to the power alpha; the weight's columns are multiplied by it,
    quantised with the group quantiser, and divided by it again; the error is
    the mean of the squared difference between the quantised layer's output
    and the unquantised layer's output; a later alpha replaces the best only if
    its error is strictly lower."""
    import torch

    Wt = torch.from_numpy(np.asarray(W, dtype=np.float64))
    Xt = torch.from_numpy(np.asarray(X, dtype=np.float64))
    sx = Xt.abs().mean(dim=0)
    y_ref = Xt @ Wt.T
    errs, best, best_err, best_s = [], -1, float("inf"), None
    for i in range(n_grid):
        s = sx.clamp(min=1e-4) ** (i / n_grid)
        w_q = _torch_group_rtn(Wt * s) / s
        err = float(((Xt @ w_q.T - y_ref) ** 2).mean())
        errs.append(err)
        if err < best_err:
            best, best_err, best_s = i, err, s
    return np.array(errs), best, best_s.numpy()


@pytest.mark.parametrize("layer", ["tiny", "square1024"])
def test_search_matches_an_independent_restatement(layer):
    """The oracle's composed search (fp64 quantiser, no normalisation, as the
    pages' search is written) equals an independent torch float64 statement
    of the same steps: every per-alpha loss to 1e-12 relative, the same first
    minimum and the same scale. With the normalisation on, the losses move by
    rounding only (the normaliser cancels in exact arithmetic)."""
    if layer == "tiny":
        L = workloads.make_layer("tiny")
    else:
        L = workloads.make_layer("llama7b_q_proj", n_tok=256, out_features=1024, in_features=1024, seed=11)
    W, X = L["W"].astype(np.float64), L["X"].astype(np.float64)
    sx = O.channel_importance(X)
    assert sx.min() > 1e-4  # the clamp constant (1e-4 here, its fp32 value in the oracle) never binds
    ref_losses, ref_best, ref_s = _torch_search(W, X)
    res = O.search_scale(W, X, sx, normalize=False, pinned=False)
    np.testing.assert_allclose(res["losses"], ref_losses, rtol=1e-12)
    assert res["best_idx"] == ref_best
    np.testing.assert_allclose(res["s_best"], ref_s, rtol=1e-14)
    norm = O.search_scale(W, X, sx, normalize=True, pinned=False)
    np.testing.assert_allclose(norm["losses"], ref_losses, rtol=1e-10)
    assert norm["best_idx"] == ref_best


@pytest.mark.parametrize("layer", ["tiny", "square1024"])
def test_fp32_decided_search_tracks_the_fp64_search(layer):
    """The search whose codes are decided in fp32 (the precision the kernels
    decide them in) against the same search in fp64: per-alpha losses within
    1e-3 relative, and the same chosen alpha. A code can differ only where
    v / step lies within an fp32 rounding of a half-integer."""
    if layer == "tiny":
        L = workloads.make_layer("tiny")
    else:
        L = workloads.make_layer("llama7b_q_proj", n_tok=256, out_features=1024, in_features=1024, seed=11)
    W, X = L["W"].astype(np.float64), L["X"].astype(np.float64)
    sx = O.channel_importance(X)
    a = O.search_scale(W, X, sx, pinned=True)
    b = O.search_scale(W, X, sx, pinned=False)
    np.testing.assert_allclose(a["losses"], b["losses"], rtol=1e-3)
    assert a["best_idx"] == b["best_idx"]
