"""Stage-by-stage parity of the CUDA path against the CPU oracle.

Every input comes from the seeded generator or from the oracle; no expected
value comes from the CUDA path. Calls go through the C ABI (ctypes).
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads
from gpu_util import dev_bf16, dev_f32, dev_weight, host_bf16_to_f64, save_debug
from post_bit_weight_awq_b300 import build, capi, capi_testing

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    capi.lib()


def _rand_bf16(rng, shape, scale=1.0):
    return workloads.round_to_bf16((rng.standard_normal(shape) * scale).astype(np.float32))


# ------------------------------------------------------------------ statistics


@pytest.mark.parametrize("n,K", [(1, 128), (129, 256), (257, 384), (128, 256), (1000, 11008), (4096, 4096)])
def test_act_stats_matches_oracle(n, K):
    rng = np.random.default_rng(n * 7919 + K)
    X = _rand_bf16(rng, (n, K), 3.0)
    X[:, ::97] *= 40.0
    X = workloads.round_to_bf16(X)
    Xd = dev_bf16(X)
    mean = torch.empty(K, dtype=torch.float32, device="cuda")
    ws = torch.empty(capi.awq_act_stats_workspace_size(n, K), dtype=torch.uint8, device="cuda")
    capi.awq_act_stats(Xd, mean, ws)
    m1 = mean.cpu().numpy().copy()
    capi.awq_act_stats(Xd, mean, ws)
    m2 = mean.cpu().numpy()
    ref = O.channel_importance(X)
    # fp32 partial sums of at most 128 tokens (bound 128 * 2^-24), compensated across chunks
    np.testing.assert_allclose(m1, ref, rtol=1e-5, atol=0)
    np.testing.assert_array_equal(m1, m2)  # deterministic


# ------------------------------------------------------------------ alpha scales


@pytest.mark.parametrize("normalize", [1, 0])
def test_alpha_scales_match_oracle(normalize):
    L = workloads.make_layer("tiny")
    sx32 = O.f32(O.channel_importance(L["X"]))
    sx32[5] = 1e-7  # below the clamp
    K = sx32.size
    cfg = capi.config(normalize=normalize)
    G = cfg.n_grid
    s = torch.empty(G, K, dtype=torch.float32, device="cuda")
    inv = torch.empty_like(s)
    capi_testing.awq_alpha_scales(dev_f32(sx32), cfg, s, inv)
    s_h, inv_h = s.cpu().numpy().astype(np.float64), inv.cpu().numpy().astype(np.float64)
    assert np.all(s_h[0] == 1.0) and np.all(inv_h[0] == 1.0)
    for i, a in enumerate(O.alpha_grid(G)):
        ref = O.f32(O.awq_scales(sx32, a, normalize=bool(normalize)))
        # both sides form s in fp64 and round once to fp32: equal except where
        # the two pow implementations straddle an fp32 rounding boundary
        ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(s_h[i] - ref) <= ulp)
        assert np.mean(s_h[i] == ref) >= 0.999
        np.testing.assert_array_equal(inv_h[i], O.f32(1.0 / s_h[i]))


# ------------------------------------------------------------------ fake-quant


def _oracle_scales32(sx, G):
    s32 = np.stack([O.f32(O.awq_scales(sx, a)) for a in O.alpha_grid(G)])
    inv32 = O.f32(1.0 / s32)
    return s32, inv32


@pytest.mark.parametrize("layer,rows", [("tiny", None), ("llama7b_q_proj", 300)])
@pytest.mark.parametrize("form", [capi.AWQ_LOSS_RESIDUAL, capi.AWQ_LOSS_REFERENCE])
def test_fakequant_codes_and_values(layer, rows, form):
    kw = {} if rows is None else dict(out_features=rows, in_features=1024, n_tok=256)
    L = workloads.make_layer(layer, **kw)
    W, X = L["W"].astype(np.float64), L["X"]
    N, K = W.shape
    cfg = capi.config(loss_form=form)
    G = cfg.n_grid
    s32, inv32 = _oracle_scales32(O.channel_importance(X), G)
    slots = G + 1 if form == capi.AWQ_LOSS_REFERENCE else G
    op = torch.empty(slots, N, K, dtype=torch.bfloat16, device="cuda")
    capi_testing.awq_fakequant(dev_weight(L), dev_f32(s32), dev_f32(inv32), cfg, op)
    got = host_bf16_to_f64(op)
    for i in range(G):
        W_hat = O.fake_quantize(W, s32[i])
        ref = W_hat - W if form == capi.AWQ_LOSS_RESIDUAL else W_hat
        # same fp32 codes; then three fp32 roundings and one bf16 rounding
        tol = 2.0**-8 * np.abs(ref) + 1e-6 * (np.abs(W) + np.abs(W_hat)) + 1e-30
        bad = np.abs(got[i] - ref) > tol
        if bad.any():
            save_debug(f"fakequant_{layer}_{form}_{i}", got=got[i], ref=ref, W=W, s=s32[i])
        assert not bad.any(), f"alpha {i}: {bad.sum()} elements off"
    if form == capi.AWQ_LOSS_REFERENCE:
        np.testing.assert_array_equal(got[G], workloads.round_to_bf16(L["W"]).astype(np.float64))


# ------------------------------------------------------------------ search product


@pytest.mark.parametrize("single_cta", [0, 1])  # 0: the default CTA-pair kernel
@pytest.mark.parametrize("n,N,K,G", [(128, 256, 128, 1), (300, 520, 384, 3), (1, 7, 128, 2), (257, 130, 256, 2),
                                     (512, 1024, 1024, 2)])
def test_search_gemm_products_and_partials(n, N, K, G, single_cta):
    rng = np.random.default_rng(n + 31 * N + 7 * K + G)
    A = _rand_bf16(rng, (n, K))
    B = _rand_bf16(rng, (G, N, K), 0.05)
    cfg = capi.config(n_grid=G)
    mt, nt, tm, tn = capi_testing.awq_search_tiles(n, N, cfg)
    partials = torch.zeros(G, mt, nt, 4, dtype=torch.float32, device="cuda")
    dump = torch.zeros(G, n, N, dtype=torch.float32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    capi_testing.awq_search_gemm_dump(dev_bf16(A), dev_bf16(B.reshape(G * N, K)), cfg, partials, status, dump,
                              n_tok=n, in_features=K, out_features=N, single_cta=single_cta)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    D = dump.cpu().numpy().astype(np.float64)
    P = partials.cpu().numpy().astype(np.float64)
    A64 = A.astype(np.float64)
    for i in range(G):
        ref = A64 @ B[i].astype(np.float64).T
        scale = np.sqrt(K) * 0.05
        ok = np.allclose(D[i], ref, rtol=1e-5, atol=1e-5 * scale)
        if not ok:
            save_debug(f"gemm_{n}_{N}_{K}_{G}_{i}_c{single_cta}", got=D[i], ref=ref, A=A, B=B[i])
        assert ok, f"product of alpha {i} differs: max err {np.abs(D[i] - ref).max()}"
        sq = ref * ref
        for mb in range(mt):
            for nb in range(nt):
                for q in range(4):
                    r0, r1 = mb * tm + q * 32, min(mb * tm + q * 32 + 32, n)
                    c0, c1 = nb * tn, min(nb * tn + tn, N)
                    expect = sq[r0:r1, c0:c1].sum() if r0 < n else 0.0
                    assert P[i, mb, nb, q] == pytest.approx(expect, rel=1e-4, abs=1e-6)
    # the production entry point (the CTA-pair kernel) gives the same partials
    partials2 = torch.zeros_like(partials)
    capi_testing.awq_search_gemm(dev_bf16(A), dev_bf16(B.reshape(G * N, K)), cfg, partials2, status, n_tok=n,
                         in_features=K, out_features=N)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    if single_cta == 0:
        assert torch.equal(partials, partials2)
    else:
        np.testing.assert_allclose(partials2.cpu().numpy(), partials.cpu().numpy(), rtol=1e-5, atol=1e-6)


# ------------------------------------------------------------------ fused fake-quant + search product


@pytest.mark.parametrize("layer,kw", [("tiny", {}),
                                      ("llama7b_q_proj", dict(out_features=300, in_features=640, n_tok=257)),
                                      ("llama7b_q_proj", dict(out_features=1024, in_features=1024, n_tok=512)),
                                      ("70b_mlp", dict(out_features=520, in_features=8192, n_tok=130))])
def test_fused_search_matches_separate_stages(layer, kw):
    """The quantiser warps of the fused kernel write exactly the operand that
    awq_fakequant writes, and the products consume it only once it is
    complete: op and the partial sums equal the two-launch path bit for bit
    (ragged operand tiles, a partial channel strip, fp32 weights included)."""
    L = workloads.make_layer(layer, **kw)
    N, K = L["W"].shape
    n = L["X"].shape[0]
    W, X = dev_weight(L), dev_bf16(L["X"])
    cfg = capi.config()
    G = cfg.n_grid
    s = torch.empty(G, K, dtype=torch.float32, device="cuda")
    inv = torch.empty_like(s)
    capi_testing.awq_alpha_scales(dev_f32(O.f32(O.channel_importance(L["X"]))), cfg, s, inv)
    op_ref = torch.empty(G, N, K, dtype=torch.bfloat16, device="cuda")
    capi_testing.awq_fakequant(W, s, inv, cfg, op_ref)
    mt, nt, _, _ = capi_testing.awq_search_tiles(n, N, cfg)
    p_ref = torch.zeros(G, mt, nt, 4, dtype=torch.float32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    capi_testing.awq_search_gemm(X, op_ref, cfg, p_ref, status, n_tok=n, in_features=K, out_features=N)
    op = torch.full_like(op_ref, float("nan"))
    parts = torch.full_like(p_ref, float("nan"))
    ready = torch.full((G * (nt + 1) + 1,), 7, dtype=torch.int32, device="cuda")  # the call zeroes it
    for _ in range(2):  # twice: ready counters and op are reset / rewritten by each call
        capi_testing.awq_search_fused(W, X, s, inv, cfg, op, parts, ready, status)
        torch.cuda.synchronize()
        assert int(status[0]) == 0
        assert torch.equal(op.view(torch.int16), op_ref.view(torch.int16))
        assert torch.equal(parts, p_ref)
        strips8 = ((K + 511) // 512) * 8
        assert torch.all(ready[:G * nt] == strips8)  # every tile, every strip, every quantiser warp
        assert torch.all(ready[G * nt:G * (nt + 1)] == nt * strips8)
        assert int(ready[-1]) == G  # the search started every alpha


# ------------------------------------------------------------------ loss + argmin


def test_loss_select_sums_argmin_and_copy():
    rng = np.random.default_rng(5)
    n, N, K, G = 300, 520, 256, 6
    cfg = capi.config(n_grid=G)
    mt, nt, _, _ = capi_testing.awq_search_tiles(n, N, cfg)
    parts = rng.uniform(0.0, 1.0, (G, mt, nt, 4)).astype(np.float32)
    parts[3] *= 0.25  # alpha 3 smallest
    parts[4] = parts[3]  # tie with 3: the first one wins
    s = rng.uniform(0.5, 2.0, (G, K)).astype(np.float32)
    losses = torch.empty(G, dtype=torch.float32, device="cuda")
    best = torch.empty(1, dtype=torch.int32, device="cuda")
    s_best = torch.empty(K, dtype=torch.float32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    capi_testing.awq_loss_select(dev_f32(parts), dev_f32(s), cfg, losses, best, s_best, status, n_tok=n, out_features=N,
                         in_features=K)
    torch.cuda.synchronize()
    ref = parts.astype(np.float64).reshape(G, -1).sum(axis=1) / (n * N)
    np.testing.assert_allclose(losses.cpu().numpy(), ref, rtol=1e-6)
    assert int(best[0]) == 3
    np.testing.assert_array_equal(s_best.cpu().numpy(), s[3])
    assert int(status[0]) == 0
    parts[1, 0, 0, 0] = np.nan
    capi_testing.awq_loss_select(dev_f32(parts), dev_f32(s), cfg, losses, best, s_best, status, n_tok=n, out_features=N,
                         in_features=K)
    torch.cuda.synchronize()
    assert int(status[0]) == capi.AWQ_ERR_NONFINITE


# ------------------------------------------------------------------ pack


@pytest.mark.parametrize("layer,kw", [("tiny", {}), ("llama7b_q_proj", dict(out_features=200, in_features=1024,
                                                                          n_tok=64)),
                                      ("70b_mlp", dict(out_features=64, in_features=8192, n_tok=64))])
def test_pack_bit_exact_with_oracle_scale(layer, kw):
    L = workloads.make_layer(layer, **kw)
    W, X = L["W"], L["X"]
    N, K = W.shape
    sx = O.channel_importance(X)
    for alpha in (0.0, 0.35, 0.9):
        s32 = O.f32(O.awq_scales(sx, alpha))
        ref = O.quantize_pack(W.astype(np.float64), s32)
        qw = torch.empty(N, K // 8, dtype=torch.int32, device="cuda")
        sc = torch.empty(N, K // 128, dtype=torch.float16, device="cuda")
        zr = torch.empty(N, K // 128, dtype=torch.float16, device="cuda")
        capi.awq_quantize_pack(dev_weight(L), dev_f32(s32), capi.config(), qw, sc, zr)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(qw.cpu().numpy(), ref["qweight"])
        np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint16), ref["scales"].view(np.uint16))
        np.testing.assert_array_equal(zr.cpu().numpy().view(np.uint16), ref["zeros"].view(np.uint16))


def test_pack_hand_built_groups():
    # constant, all-zero, tie-laden and one-sign groups in one layer, fp32 weights
    K = 512
    W = np.zeros((3, K), dtype=np.float32)
    W[0, 128:256] = 0.02
    W[0, 256:384] = np.linspace(1.0, 2.0, 128)
    W[0, 384] = 15.0
    W[0, 385:388] = [2.5, 3.5, 0.5]
    W[1] = np.linspace(-1, 1, K)
    W[2] = np.float32(-0.75)
    s32 = np.ones(K, dtype=np.float32)
    ref = O.quantize_pack(W.astype(np.float64), s32.astype(np.float64))
    qw = torch.empty(3, K // 8, dtype=torch.int32, device="cuda")
    sc = torch.empty(3, K // 128, dtype=torch.float16, device="cuda")
    zr = torch.empty(3, K // 128, dtype=torch.float16, device="cuda")
    capi.awq_quantize_pack(dev_f32(W), dev_f32(s32), capi.config(), qw, sc, zr)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(qw.cpu().numpy(), ref["qweight"])
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint16), ref["scales"].view(np.uint16))
    np.testing.assert_array_equal(zr.cpu().numpy().view(np.uint16), ref["zeros"].view(np.uint16))


# ------------------------------------------------------------------ symmetric quantiser (zero point off)


@pytest.mark.parametrize("layer,kw", [("tiny", {}), ("llama7b_q_proj", dict(out_features=200, in_features=1024,
                                                                          n_tok=64))])
def test_symmetric_pack_and_fakequant_bit_exact(layer, kw):
    L = workloads.make_layer(layer, **kw)
    W, X = L["W"], L["X"]
    N, K = W.shape
    cfg = capi.config(zero_point=0)
    sx = O.channel_importance(X)
    for alpha in (0.0, 0.45, 0.9):
        s32 = O.f32(O.awq_scales(sx, alpha))
        ref = O.quantize_pack(W.astype(np.float64), s32, zero_point=False)
        qw = torch.empty(N, K // 8, dtype=torch.int32, device="cuda")
        sc = torch.empty(N, K // 128, dtype=torch.float16, device="cuda")
        zr = torch.empty(N, K // 128, dtype=torch.float16, device="cuda")
        capi.awq_quantize_pack(dev_weight(L), dev_f32(s32), cfg, qw, sc, zr)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(qw.cpu().numpy(), ref["qweight"])
        np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint16), ref["scales"].view(np.uint16))
        assert np.all(zr.cpu().numpy() == 8.0)
    # the search operand of every alpha, as in test_fakequant_codes_and_values
    G = cfg.n_grid
    s32, inv32 = _oracle_scales32(sx, G)
    op = torch.empty(G, N, K, dtype=torch.bfloat16, device="cuda")
    capi_testing.awq_fakequant(dev_weight(L), dev_f32(s32), dev_f32(inv32), cfg, op)
    got = host_bf16_to_f64(op)
    W64 = W.astype(np.float64)
    for i in range(G):
        W_hat = O.fake_quantize(W64, s32[i], zero_point=False)
        ref = W_hat - W64
        tol = 2.0**-8 * np.abs(ref) + 1e-6 * (np.abs(W64) + np.abs(W_hat)) + 1e-30
        assert not (np.abs(got[i] - ref) > tol).any(), f"alpha {i}"


# ------------------------------------------------------------------ group sizes and code widths


@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("zero_point", [1, 0])
@pytest.mark.parametrize("w_dtype_layer,kw", [("tiny", {}),
                                              ("llama7b_q_proj", dict(out_features=130, in_features=640, n_tok=64))])
def test_finer_groups_pack_bit_exact(group, zero_point, w_dtype_layer, kw):
    """Groups of 32 and 64: codes, fp16 scales and zeros equal the oracle's bit for bit (fp32 and bf16
    weights, a partial 512-channel strip at in = 640)."""
    L = workloads.make_layer(w_dtype_layer, **kw)
    W, X = L["W"], L["X"]
    N, K = W.shape
    cfg = capi.config(group=group, zero_point=zero_point)
    sx = O.channel_importance(X)
    for alpha in (0.0, 0.5, 0.95):
        s32 = O.f32(O.awq_scales(sx, alpha))
        ref = O.quantize_pack(W.astype(np.float64), s32, group=group, zero_point=bool(zero_point))
        qw = torch.empty(N, K // 8, dtype=torch.int32, device="cuda")
        sc = torch.full((N, K // group), float("nan"), dtype=torch.float16, device="cuda")
        zr = torch.full((N, K // group), float("nan"), dtype=torch.float16, device="cuda")
        capi.awq_quantize_pack(dev_weight(L), dev_f32(s32), cfg, qw, sc, zr)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(qw.cpu().numpy(), ref["qweight"])
        np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint16), ref["scales"].view(np.uint16))
        np.testing.assert_array_equal(zr.cpu().numpy().view(np.uint16), ref["zeros"].view(np.uint16))


@pytest.mark.parametrize("group,w_bit,zero_point", [(32, 4, 1), (64, 4, 1), (128, 3, 1), (64, 2, 1), (32, 8, 1),
                                                    (128, 8, 0), (32, 3, 0)])
def test_group_and_width_fakequant_values(group, w_bit, zero_point):
    """The search operand for other group sizes and code widths, every alpha, against the oracle's
    fake-quant with the same knobs (the tolerance of test_fakequant_codes_and_values)."""
    L = workloads.make_layer("llama7b_q_proj", out_features=96, in_features=640, n_tok=128, seed=group + w_bit)
    W, X = L["W"].astype(np.float64), L["X"]
    N, K = W.shape
    cfg = capi.config(group=group, w_bit=w_bit, zero_point=zero_point)
    G = cfg.n_grid
    s32, inv32 = _oracle_scales32(O.channel_importance(X), G)
    op = torch.empty(G, N, K, dtype=torch.bfloat16, device="cuda")
    capi_testing.awq_fakequant(dev_weight(L), dev_f32(s32), dev_f32(inv32), cfg, op)
    got = host_bf16_to_f64(op)
    for i in range(G):
        W_hat = O.fake_quantize(W, s32[i], w_bit=w_bit, group=group, zero_point=bool(zero_point))
        ref = W_hat - W
        tol = 2.0**-8 * np.abs(ref) + 1e-6 * (np.abs(W) + np.abs(W_hat)) + 1e-30
        bad = np.abs(got[i] - ref) > tol
        assert not bad.any(), f"alpha {i}: {bad.sum()} elements off"


@pytest.mark.parametrize("group,w_bit,zero_point", [(32, 4, 1), (64, 3, 1), (64, 4, 0)])
def test_fused_search_matches_separate_stages_other_quantisers(group, w_bit, zero_point):
    """The fused kernel's quantiser warps with other group sizes and widths write the operand the
    fake-quant kernel writes, bit for bit, and the partial sums are identical."""
    L = workloads.make_layer("llama7b_q_proj", out_features=300, in_features=640, n_tok=257)
    N, K = L["W"].shape
    n = L["X"].shape[0]
    W, X = dev_weight(L), dev_bf16(L["X"])
    cfg = capi.config(group=group, w_bit=w_bit, zero_point=zero_point)
    G = cfg.n_grid
    s = torch.empty(G, K, dtype=torch.float32, device="cuda")
    inv = torch.empty_like(s)
    capi_testing.awq_alpha_scales(dev_f32(O.f32(O.channel_importance(L["X"]))), cfg, s, inv)
    op_ref = torch.empty(G, N, K, dtype=torch.bfloat16, device="cuda")
    capi_testing.awq_fakequant(W, s, inv, cfg, op_ref)
    mt, nt, _, _ = capi_testing.awq_search_tiles(n, N, cfg)
    p_ref = torch.zeros(G, mt, nt, 4, dtype=torch.float32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    capi_testing.awq_search_gemm(X, op_ref, cfg, p_ref, status, n_tok=n, in_features=K, out_features=N)
    op = torch.full_like(op_ref, float("nan"))
    parts = torch.full_like(p_ref, float("nan"))
    ready = torch.zeros((G * (nt + 1) + 1,), dtype=torch.int32, device="cuda")
    capi_testing.awq_search_fused(W, X, s, inv, cfg, op, parts, ready, status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    assert torch.equal(op.view(torch.int16), op_ref.view(torch.int16))
    assert torch.equal(parts, p_ref)


# ------------------------------------------------------------------ near-tie code decisions


def _near_tie_rows(step, rows=8, K=512, seed=0):
    """fp32 rows whose groups of 128 span [0, 15 * step] and otherwise hold values a few ulps either side of
    the exact ties (k + 1/2) * step, where the fast code decision must hand over to the IEEE division."""
    rng = np.random.default_rng(seed)
    W = np.zeros((rows, K), dtype=np.float32)
    for r in range(rows):
        for g in range(K // 128):
            vals = np.empty(128, dtype=np.float32)
            vals[0], vals[1] = np.float32(0.0), np.float32(15.0 * step)
            for i in range(2, 128):
                k = rng.integers(0, 15)
                tie = np.float32((k + 0.5) * step)
                vals[i] = tie + np.float32(rng.integers(-3, 4)) * np.spacing(tie)
            W[r, g * 128:(g + 1) * 128] = rng.permutation(vals)
    return W


@pytest.mark.parametrize("step", [1.0, 1.0 / 15.0, 0.013, 3.3e-3])
@pytest.mark.parametrize("zero_point", [1, 0])
def test_pack_decides_near_ties_exactly(step, zero_point):
    W = _near_tie_rows(step, seed=int(step * 1e6) + zero_point)
    rows, K = W.shape
    cfg = capi.config(zero_point=zero_point)
    for s32 in (np.ones(K, dtype=np.float32), np.full(K, 1.5, dtype=np.float32)):
        ref = O.quantize_pack(W.astype(np.float64), s32.astype(np.float64), zero_point=bool(zero_point))
        qw = torch.empty(rows, K // 8, dtype=torch.int32, device="cuda")
        sc = torch.empty(rows, K // 128, dtype=torch.float16, device="cuda")
        zr = torch.empty(rows, K // 128, dtype=torch.float16, device="cuda")
        capi.awq_quantize_pack(dev_f32(W), dev_f32(s32), cfg, qw, sc, zr)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(qw.cpu().numpy(), ref["qweight"])
        np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint16), ref["scales"].view(np.uint16))
        np.testing.assert_array_equal(zr.cpu().numpy().view(np.uint16), ref["zeros"].view(np.uint16))


@pytest.mark.parametrize("w_bit", [2, 8])
@pytest.mark.parametrize("group,zero_point", [(128, 1), (64, 0), (32, 1)])
@pytest.mark.parametrize("layer,kw", [("tiny", {}),
                                      ("llama7b_q_proj", dict(out_features=130, in_features=640, n_tok=64))])
def test_pack_other_widths_bit_exact(w_bit, group, zero_point, layer, kw):
    """2-bit (16 per word) and 8-bit (4 per word) packing: words, scales and zeros equal the oracle's."""
    L = workloads.make_layer(layer, **kw)
    W, X = L["W"], L["X"]
    N, K = W.shape
    cfg = capi.config(w_bit=w_bit, group=group, zero_point=zero_point)
    sx = O.channel_importance(X)
    for alpha in (0.0, 0.6):
        s32 = O.f32(O.awq_scales(sx, alpha))
        ref = O.quantize_pack(W.astype(np.float64), s32, w_bit=w_bit, group=group, zero_point=bool(zero_point))
        qw = torch.full((N, K * w_bit // 32), -1, dtype=torch.int32, device="cuda")
        sc = torch.empty(N, K // group, dtype=torch.float16, device="cuda")
        zr = torch.empty(N, K // group, dtype=torch.float16, device="cuda")
        capi.awq_quantize_pack(dev_weight(L), dev_f32(s32), cfg, qw, sc, zr)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(qw.cpu().numpy(), ref["qweight"])
        np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint16), ref["scales"].view(np.uint16))
        np.testing.assert_array_equal(zr.cpu().numpy().view(np.uint16), ref["zeros"].view(np.uint16))
