"""Failure detection on the GPU without a fault.

A wait that can never complete (one pipeline stage is never filled) must end
after the configured limit with AWQ_ERR_TIMEOUT in the status word, and the
device, including tensor memory, must be usable by the next launch.
"""
import time

import numpy as np
import pytest
import torch

import workloads
from gpu_util import dev_bf16
from post_bit_weight_awq_b300 import build, capi, capi_testing

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    capi.lib()


def test_stuck_wait_ends_with_timeout_status_and_device_stays_usable():
    n, N, K, G = 512, 1024, 512, 2
    rng = np.random.default_rng(3)
    A = workloads.round_to_bf16(rng.standard_normal((n, K)).astype(np.float32))
    B = workloads.round_to_bf16((rng.standard_normal((G, N, K)) * 0.05).astype(np.float32))
    Ad, Bd = dev_bf16(A), dev_bf16(B.reshape(G * N, K))
    cfg = capi.config(n_grid=G, wait_timeout_ms=100)
    mt, nt, tm, tn = capi_testing.awq_search_tiles(n, N, cfg)
    partials = torch.zeros(G, mt, nt, 4, dtype=torch.float32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    capi_testing.awq_search_gemm_withhold_fill(Ad, Bd, cfg, partials, status, n_tok=n, in_features=K, out_features=N)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status[0]) == capi.AWQ_ERR_TIMEOUT
    assert elapsed < 5.0
    # the next launch on the same device is correct
    status.zero_()
    capi_testing.awq_search_gemm(Ad, Bd, cfg, partials, status, n_tok=n, in_features=K, out_features=N)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    P = partials.cpu().numpy().astype(np.float64).sum(axis=(1, 2, 3))
    for i in range(G):
        ref = ((A.astype(np.float64) @ B[i].astype(np.float64).T) ** 2).sum()
        assert P[i] == pytest.approx(ref, rel=1e-4)


def test_gram_loss_stuck_wait_ends_with_timeout_and_device_stays_usable():
    """The GRAM form's products with every CTA's first ring stage left unfilled: the MMA issuer's wait runs
    out after the limit, the kernel reports AWQ_ERR_TIMEOUT and returns, and the next launch on the same
    device gives the right sums (checked against sum_r D[r] X^T X D[r]^T in fp64)."""
    n, N, K, G = 512, 640, 768, 2
    rng = np.random.default_rng(5)
    X = workloads.round_to_bf16(rng.standard_normal((n, K)).astype(np.float32))
    D = workloads.round_to_bf16((rng.standard_normal((G, N, K)) * 0.01).astype(np.float32))
    Xd, Dd = dev_bf16(X), dev_bf16(D.reshape(G * N, K))
    cfg = capi.config(n_grid=G, wait_timeout_ms=100, loss_form=capi.AWQ_LOSS_GRAM)
    xt_elems, h_elems, per_alpha = capi_testing.awq_gram_sizes(n, N, K)
    xt = torch.empty(xt_elems, dtype=torch.bfloat16, device="cuda")
    H = torch.empty(h_elems, dtype=torch.bfloat16, device="cuda")
    partials = torch.zeros(G, per_alpha, dtype=torch.float32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    capi_testing.awq_gram_matrix(Xd, xt, H, cfg, status, n_tok=n, in_features=K)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    t0 = time.perf_counter()
    capi_testing.awq_gram_loss_withhold_fill(Dd, H, cfg, partials, status, out_features=N, in_features=K)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status[0]) == capi.AWQ_ERR_TIMEOUT
    assert elapsed < 5.0
    status.zero_()
    capi_testing.awq_gram_loss(Dd, H, cfg, partials, status, out_features=N, in_features=K)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    C = X.astype(np.float64).T @ X.astype(np.float64)
    P = partials.cpu().numpy().astype(np.float64).sum(axis=1)
    for i in range(G):
        Di = D[i].astype(np.float64)
        ref = float(np.einsum("rc,cj,rj->", Di, C, Di))
        assert P[i] == pytest.approx(ref, rel=1e-3)


def test_fused_search_stuck_tile_ends_with_timeout_and_device_stays_usable():
    """The cross-CTA wait of the fused search: one quantiser unit is never
    published, so the producers needing its tile wait until the limit; the
    kernel reports AWQ_ERR_TIMEOUT and the next launch is correct."""
    n, N, K = 512, 1024, 512
    rng = np.random.default_rng(4)
    X = dev_bf16(workloads.round_to_bf16(rng.standard_normal((n, K)).astype(np.float32)))
    W = dev_bf16(workloads.round_to_bf16((rng.standard_normal((N, K)) * 0.02).astype(np.float32)))
    cfg = capi.config(n_grid=3, wait_timeout_ms=100)
    G = cfg.n_grid
    s = torch.empty(G, K, dtype=torch.float32, device="cuda")
    inv = torch.empty_like(s)
    mean = X.float().abs().mean(0).contiguous()
    capi_testing.awq_alpha_scales(mean, cfg, s, inv)
    mt, nt, _, _ = capi_testing.awq_search_tiles(n, N, cfg)
    op = torch.empty(G, N, K, dtype=torch.bfloat16, device="cuda")
    parts = torch.zeros(G, mt, nt, 4, dtype=torch.float32, device="cuda")
    ready = torch.zeros(G * (nt + 1) + 1, dtype=torch.int32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    capi_testing.awq_search_fused_withhold_unit(W, X, s, inv, cfg, op, parts, ready, status)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status[0]) == capi.AWQ_ERR_TIMEOUT
    assert elapsed < 5.0
    # the next launch on the same device is correct: it equals the two separate launches
    status.zero_()
    capi_testing.awq_search_fused(W, X, s, inv, cfg, op, parts, ready, status)
    op_ref = torch.empty_like(op)
    p_ref = torch.zeros_like(parts)
    capi_testing.awq_fakequant(W, s, inv, cfg, op_ref)
    capi_testing.awq_search_gemm(X, op_ref, cfg, p_ref, status, n_tok=n, in_features=K, out_features=N)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    assert torch.equal(op.view(torch.int16), op_ref.view(torch.int16))
    assert torch.equal(parts, p_ref)
