"""The GRAM loss form on the GPU against the CPU oracle and against the
direct product.

The form scores alpha_i by sum_r D_i[r] (X^T X) D_i[r]^T (D_i = W_hat_i - W),
equal in exact arithmetic to the search_scale listing's sum over tokens and
output rows of (X W_hat_i^T - X W^T)^2 ("AWQ: How Activation-Aware
Quantization Saves 4-bit LLMs"); the identity itself is checked on the CPU
in test_gram_identity.py. Here:
  * awq_gram_matrix: the transposed copy of X bit for bit, and H's blocks on
    and below the diagonal against X^T X formed in fp64 from the same bf16
    values, within the rounding the kernel's arithmetic allows;
  * awq_gram_loss: the per-alpha sums against the direct products' sums on
    the same operand, and against the oracle;
  * awq_search_layer / awq_search_block with loss_form GRAM: levels 2 and 3
    of the library's contract (per-alpha losses within 1e-2 of the oracle's,
    the chosen alpha's oracle loss within 0.5% of the minimum) on small,
    ragged and degenerate layers and on the full-size layers, row losses,
    determinism.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
import workloads
from gpu_util import dev_bf16, dev_f32, dev_weight, host_bf16_to_f64
from post_bit_weight_awq_b300 import build, capi, capi_testing, layer
from test_gpu_layers import (LOSS_RTOL, _arithmetic_bound, _check_levels, _check_pack, _oracle_losses,
                             _search_with_statistic)

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "oracle_losses.json")
GRAM = capi.AWQ_LOSS_GRAM


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    capi.lib()


def _gram_bound(L, sx32):
    """Per-alpha |L_gpu - L_oracle| the GRAM form's arithmetic allows: the
    RESIDUAL operand's rounding (as for the direct product), plus X^T X held
    as bf16 after fp32 accumulation over the tokens (2^-8 relative per entry
    plus n 2^-24 of sum_t |x x|), plus the fp32 accumulation of P = D H^T
    over up to `in` terms and of the epilogue's sums; all bounded through
    sum_t sum_r (|X_t| . |E_r|)^2."""
    res = _arithmetic_bound(L, sx32, capi.AWQ_LOSS_RESIDUAL)
    W = L["W"].astype(np.float64)
    X = L["X"].astype(np.float64)
    n, K = X.shape
    N = W.shape[0]
    ax = np.abs(X)
    out = []
    for i, a in enumerate(O.alpha_grid(20)):
        E = O.fake_quantize(W, O.f32(O.awq_scales(sx32, a))) - W
        m = ax @ np.abs(E).T
        out.append(res[i] + 1.05 * (2.0**-8 + (n + K + 1024) * 2.0**-24) * np.sum(m * m) / (n * N))
    return np.array(out)


def _sizes(n, N, K):
    return capi_testing.awq_gram_sizes(n, N, K)


def _gram_matrix(X, n, K, cfg):
    xt_elems, h_elems, _ = _sizes(n, 1, K)
    xt = torch.full((xt_elems,), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    H = torch.zeros(h_elems, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    capi_testing.awq_gram_matrix(X, xt, H, cfg, status, n_tok=n, in_features=K)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    return xt, H.view(K, K)


@pytest.mark.parametrize("n,K", [(37, 128), (64, 256), (129, 384), (300, 640), (1000, 1024), (4096, 4096)])
def test_gram_matrix_blocks(n, K):
    L = workloads.make_layer("llama7b_q_proj", n_tok=n, out_features=8, in_features=K, seed=n + K)
    X32 = L["X"]
    xt, H = _gram_matrix(dev_bf16(X32), n, K, capi.config(loss_form=GRAM))
    n_pad = (n + 63) // 64 * 64
    # the transposed copy: X^T bit for bit, zeros past the last token
    xt64 = host_bf16_to_f64(xt).reshape(K, n_pad)
    np.testing.assert_array_equal(xt64[:, :n], X32.T.astype(np.float64))
    assert not xt64[:, n:].any()
    # H on and below the block diagonal
    X = X32.astype(np.float64)
    C = X.T @ X
    A = np.abs(X).T @ np.abs(X)
    jb = np.arange(K) // 256
    below = jb[None, :] < jb[:, None]
    same = jb[None, :] == jb[:, None]
    f = np.where(below, 2.0, 1.0)
    keep = below | same
    Hg = host_bf16_to_f64(H.reshape(-1)).reshape(K, K)
    err = np.abs(Hg - f * C)
    bound = f * (2.0**-8 * np.abs(C) + n * 2.0**-24 * A) * 1.01 + 1e-30
    assert np.all(err[keep] <= bound[keep]), f"max excess {np.max((err / bound)[keep]):.3f}"


def _stage_losses(L, cfg):
    """Alpha scales, fake-quant, then the GRAM stages and the direct products on the same operand:
    (GRAM per-alpha sums, direct per-alpha sums), both / (n N)."""
    W, X = dev_weight(L), dev_bf16(L["X"])
    N, K = L["W"].shape
    n = L["X"].shape[0]
    G = cfg.n_grid
    sx = dev_f32(O.f32(O.channel_importance(L["X"])))
    s = torch.empty(G, K, dtype=torch.float32, device="cuda")
    inv = torch.empty_like(s)
    capi_testing.awq_alpha_scales(sx, cfg, s, inv)
    xt, H = _gram_matrix(X, n, K, cfg)
    op = torch.empty(G, N, K, dtype=torch.bfloat16, device="cuda")
    capi_testing.awq_fakequant(W, s, inv, cfg, op)
    _, _, per_alpha = _sizes(n, N, K)
    parts = torch.full((G, per_alpha), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    capi_testing.awq_gram_loss(op, H, cfg, parts, status)
    mt, nt, _, _ = capi_testing.awq_search_tiles(n, N, cfg)
    dparts = torch.empty(G, mt, nt, 4, dtype=torch.float32, device="cuda")
    capi_testing.awq_search_gemm(X, op, capi.config(), dparts, status, n_tok=n, in_features=K, out_features=N)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    gp = parts.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(gp)), "a partial sum was left unwritten"
    dp = dparts.cpu().numpy().astype(np.float64).reshape(G, -1)
    return gp.sum(axis=1) / (n * N), dp.sum(axis=1) / (n * N)


@pytest.mark.parametrize("n,N,K", [(128, 256, 256), (300, 520, 384), (1, 7, 128), (257, 130, 640), (512, 2100, 1024),
                                   (1000, 300, 2048)])
def test_gram_loss_against_direct_products_and_oracle(n, N, K):
    L = workloads.make_layer("llama7b_q_proj", n_tok=n, out_features=N, in_features=K, seed=3 * n + N)
    cfg = capi.config(loss_form=GRAM)
    g, d = _stage_losses(L, cfg)
    sx32 = O.f32(O.channel_importance(L["X"]))
    res = _oracle_losses(L["W"], L["X"], sx=sx32)
    bound = _gram_bound(L, sx32)
    lo = np.asarray(res["losses"])
    assert np.all(np.abs(g - lo) <= np.maximum(LOSS_RTOL * lo, bound))
    # the two forms on one operand differ only by the rounding of X^T X and the summation order
    if n >= 128 and N >= 128:
        np.testing.assert_allclose(g, d, rtol=2e-3)


@pytest.mark.parametrize("n,N,K", [(1, 7, 128), (129, 130, 256), (257, 300, 384), (64, 1, 128), (300, 520, 1024)])
def test_gram_search_layer_ragged(n, N, K):
    L = workloads.make_layer("llama7b_q_proj", n_tok=n, out_features=N, in_features=K, seed=n + N)
    sx32 = O.f32(O.channel_importance(L["X"]))
    res = _oracle_losses(L["W"], L["X"], sx=sx32)
    cfg = capi.config(loss_form=GRAM)
    ws = torch.empty(capi.awq_workspace_size(n, N, K, cfg), dtype=torch.uint8, device="cuda")
    losses = torch.empty(cfg.n_grid, dtype=torch.float32, device="cuda")
    best = torch.empty(1, dtype=torch.int32, device="cuda")
    s_best = torch.empty(K, dtype=torch.float32, device="cuda")
    capi.awq_search_layer(dev_weight(L), dev_bf16(L["X"]), dev_f32(sx32), cfg, losses, best, s_best, ws)
    assert capi.awq_get_device_status(ws) == capi.AWQ_OK
    degenerate = n == 1 or N == 1
    _check_levels(losses.cpu().numpy(), int(best[0]), res["losses"],
                  bound=_gram_bound(L, sx32) if degenerate else None)
    if int(best[0]) == res["best_idx"]:
        np.testing.assert_array_equal(s_best.cpu().numpy(), O.f32(res["s_best"]))


@pytest.mark.parametrize("kw", [dict(group=64), dict(group=32), dict(w_bit=3), dict(group=64, w_bit=2),
                                dict(zero_point=0)])
def test_gram_search_other_quantisers(kw):
    """The GRAM form with the other quantiser settings (groups of 64 and 32, 3 and 2 bits, the symmetric
    quantiser): levels 2 and 3 against the oracle run with the same settings."""
    L = workloads.make_layer("llama7b_q_proj", n_tok=1024, out_features=640, in_features=1024,
                             seed=17 + sum(kw.values()))
    sx32 = O.f32(O.channel_importance(L["X"]))
    okw = {k: (bool(v) if k == "zero_point" else v) for k, v in kw.items()}
    res = _oracle_losses(L["W"], L["X"], sx=sx32, **okw)
    losses, best, _ = _search_with_statistic(L, sx32, capi.config(loss_form=GRAM, **kw))
    _check_levels(losses, best, res["losses"])


def test_gram_tiny_layer_all_levels():
    L = workloads.make_layer("tiny")
    res = _oracle_losses(L["W"], L["X"])
    q = layer.quantize_layer(dev_weight(L), dev_bf16(L["X"]), capi.config(loss_form=GRAM))
    torch.cuda.synchronize()
    _check_levels(q.losses.cpu().numpy(), int(q.best_idx[0]), res["losses"])
    _check_pack(L, O.f32(res["s_best"]))


def test_gram_dead_channels_and_zero_rows():
    L = workloads.make_layer("llama7b_q_proj", n_tok=256, out_features=384, in_features=640, seed=11)
    L["X"] = L["X"].copy()
    L["X"][:, [3, 200, 201, 639]] = 0.0
    L["W"] = L["W"].copy()
    L["W"][5, :] = 0.0
    L["W"][7, 128:256] = 0.0
    res = _oracle_losses(L["W"], L["X"])
    q = layer.quantize_layer(dev_weight(L), dev_bf16(L["X"]), capi.config(loss_form=GRAM))
    torch.cuda.synchronize()
    _check_levels(q.losses.cpu().numpy(), int(q.best_idx[0]), res["losses"])
    _check_pack(L, O.f32(res["s_best"]))


def test_gram_deterministic_and_row_losses():
    L = workloads.make_layer("llama7b_q_proj", n_tok=1024, out_features=1100, in_features=1280, seed=4)
    cfg = capi.config(loss_form=GRAM)
    a = layer.quantize_layer(dev_weight(L), dev_bf16(L["X"]), cfg, row_losses=True)
    b = layer.quantize_layer(dev_weight(L), dev_bf16(L["X"]), cfg)
    torch.cuda.synchronize()
    assert torch.equal(a.losses, b.losses) and torch.equal(a.qweight, b.qweight)
    rl = a.row_losses.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(rl.sum(axis=1), a.losses.cpu().numpy().astype(np.float64), rtol=1e-4)
    # sampled rows against the oracle's exact per-row loss
    sx = O.channel_importance(L["X"])
    X64 = L["X"].astype(np.float64)
    n, N = L["X"].shape[0], L["W"].shape[0]
    rows = np.array([0, 1, 517, N - 1])
    for i in (0, 9, 19):
        s32 = O.f32(O.awq_scales(sx, O.alpha_grid(20)[i]))
        Wr = L["W"][rows].astype(np.float64)
        D = X64 @ (O.fake_quantize(Wr, s32) - Wr).T
        np.testing.assert_allclose(rl[i, rows], (D * D).sum(axis=0) / (n * N), rtol=LOSS_RTOL)


def test_gram_block_search_shared_input():
    K, n = 1024, 256
    base = workloads.make_layer("llama7b_q_proj", n_tok=n, out_features=768, in_features=K, seed=5)
    X = base["X"]
    Ws32 = [workloads.round_to_bf16(base["W"][a:b]) for a, b in ((0, 512), (512, 640), (640, 768))]
    sx32 = O.f32(O.channel_importance(X))
    res = O.search_scale_block([W.astype(np.float64) for W in Ws32], X.astype(np.float64), sx32)
    cfg = capi.config(loss_form=GRAM)
    outs = [W.shape[0] for W in Ws32]
    ws = torch.empty(capi.awq_search_block_workspace_size(n, outs, K, cfg), dtype=torch.uint8, device="cuda")
    losses = torch.empty(cfg.n_grid, dtype=torch.float32, device="cuda")
    best = torch.empty(1, dtype=torch.int32, device="cuda")
    s_best = torch.empty(K, dtype=torch.float32, device="cuda")
    capi.awq_search_block([dev_bf16(W) for W in Ws32], dev_bf16(X), dev_f32(sx32), cfg, losses, best, s_best, ws)
    assert capi.awq_get_device_status(ws) == capi.AWQ_OK
    _check_levels(losses.cpu().numpy(), int(best[0]), res["losses"])


@pytest.mark.parametrize("name", ["llama7b_q_proj", "13b_up_proj", "70b_mlp"])
def test_gram_full_size_layer(name):
    """Levels 2 and 3 on the full-size layers through the one-call path, against the stored oracle losses
    (written by tests/golden/make_oracle_losses.py from the oracle alone), and sampled output rows against the
    oracle's exact per-row losses."""
    g = json.load(open(GOLDEN))[name]
    L = workloads.make_layer(name)
    W, X = L["W"], L["X"]
    n, K = X.shape
    N = W.shape[0]
    assert (g["n_tok"], g["out_features"], g["in_features"]) == (n, N, K)
    q = layer.quantize_layer(dev_weight(L), dev_bf16(X), capi.config(loss_form=GRAM), row_losses=True)
    torch.cuda.synchronize()
    rel = _check_levels(q.losses.cpu().numpy(), int(q.best_idx[0]), g["losses"])
    print(f"{name} GRAM: max rel loss err {rel:.2e}, gpu best {int(q.best_idx[0])}, oracle best {g['best_idx']}")
    rl = q.row_losses.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(rl.sum(axis=1), q.losses.cpu().numpy().astype(np.float64), rtol=1e-4)
    sx = O.channel_importance(X)
    rows = np.array([0, N // 3, N - 1])
    X64 = X.astype(np.float64)
    for i in sorted({0, g["best_idx"], 19}):
        s32 = O.f32(O.awq_scales(sx, O.alpha_grid(20)[i]))
        Wr = W[rows].astype(np.float64)
        D = X64 @ (O.fake_quantize(Wr, s32) - Wr).T
        np.testing.assert_allclose(rl[i, rows], (D * D).sum(axis=0) / (n * N), rtol=LOSS_RTOL)
