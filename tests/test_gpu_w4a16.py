"""The packed layer applied to a few tokens (awq_w4a16_gemv) against the CPU
oracle: element by element, within the bound of its fp32 arithmetic, on
ragged and full-size shapes, and end to end from a layer packed on the GPU.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads
from gpu_util import dev_bf16, dev_f32, dev_weight
from post_bit_weight_awq_b300 import build, capi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    capi.lib()


def _bound(x, W_hat):
    # exact products (bf16 x times small integers), then fp32 sums. Groups of
    # 32 or 64: pair sums over 16 terms, one pair add, one fused scale per 32
    # columns, at most K/1024 chunk sums per lane and a 5-level lane tree.
    # Groups of 128: eight tensor-core accumulations per group, one fused
    # scale into one of four running sums (at most a third of the K/128
    # groups each), three final adds and the split sums of a tile cut
    # between warps. Either way under max(64, 24 + K/384) roundings of 2^-24
    # of sum |x| |w|.
    n_round = max(64, 24 + x.shape[1] // 384)
    return n_round * 2.0**-24 * (np.abs(x) @ np.abs(W_hat).T) + 1e-30


def _random_packed(rng, N, K, group=128):
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float64)
    s = O.f32(rng.uniform(0.5, 2.0, K))
    return O.quantize_pack(W, s, group=group)


def _run(x32, pk, group=128):
    M, K = x32.shape
    N = pk["qweight"].shape[0]
    y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    capi.awq_w4a16_gemv(dev_bf16(x32), torch.from_numpy(pk["qweight"]).cuda(),
                        torch.from_numpy(pk["scales"].view(np.int16)).cuda(),
                        torch.from_numpy(pk["zeros"].view(np.int16)).cuda(), capi.config(group=group), y)
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,N,K", [(1, 7, 128), (3, 300, 1024), (8, 130, 4096), (4, 1000, 11008), (2, 4096, 4096),
                                   (1, 4096, 4096), (5, 520, 8192), (5, 2, 640)])
def test_w4a16_matches_oracle(M, N, K):
    rng = np.random.default_rng(M * 1000 + N + K)
    pk = _random_packed(rng, N, K)
    x = workloads.round_to_bf16((rng.standard_normal((M, K)) * 2.0).astype(np.float32)).astype(np.float64)
    got = _run(x.astype(np.float32), pk)
    ref = O.w4a16_linear(x, pk["qweight"], pk["scales"], pk["zeros"])
    W_hat = O.dequantize_groups(O.unpack_words(pk["qweight"], K), pk["scales"].astype(np.float64),
                                pk["zeros"].astype(np.float64))
    bad = np.abs(got - ref) > _bound(x, W_hat)
    assert not bad.any(), f"{bad.sum()} outputs off, max err {np.abs(got - ref).max():.3e}"


def _at_offset(a16, elems):
    """The fp16 array on the device `elems` values (2 bytes each) past an 8-byte boundary."""
    flat = torch.from_numpy(a16.view(np.int16).reshape(-1)).cuda()
    big = torch.empty(flat.numel() + 4, dtype=torch.int16, device="cuda")
    big[elems:elems + flat.numel()] = flat
    view = big[elems:elems + flat.numel()].view(a16.shape)
    assert view.data_ptr() % 8 == 2 * elems
    return view


@pytest.mark.parametrize("elems", [1, 2])
@pytest.mark.parametrize("M,N,K", [(2, 300, 4096), (4, 130, 8192)])
def test_w4a16_steps_and_zeros_at_unaligned_offsets(M, N, K, elems):
    """Steps and zeros only 2- or 4-byte aligned (the call requires 2): the product is still right. The
    tensor-core kernel reads both groups' values of a step in one 4-byte load, so 2-byte aligned pointers
    take the fp32 kernel and 4-byte aligned ones the tensor-core kernel."""
    rng = np.random.default_rng(M * 5 + N + K)
    pk = _random_packed(rng, N, K)
    x = workloads.round_to_bf16((rng.standard_normal((M, K)) * 2.0).astype(np.float32)).astype(np.float64)
    y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    capi.awq_w4a16_gemv(dev_bf16(x.astype(np.float32)), torch.from_numpy(pk["qweight"]).cuda(),
                        _at_offset(pk["scales"], elems), _at_offset(pk["zeros"], elems), capi.config(), y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    ref = O.w4a16_linear(x, pk["qweight"], pk["scales"], pk["zeros"])
    W_hat = O.dequantize_groups(O.unpack_words(pk["qweight"], K), pk["scales"].astype(np.float64),
                                pk["zeros"].astype(np.float64))
    bad = np.abs(got - ref) > _bound(x, W_hat)
    assert not bad.any(), f"{bad.sum()} outputs off, max err {np.abs(got - ref).max():.3e}"


@pytest.mark.parametrize("M,N,K", [(3, 300, 4096), (1, 4096, 2048), (8, 130, 5632)])
def test_w4a16_zero_points_far_outside_the_code_range(M, N, K):
    """Groups offset far from 0 (one-signed groups): the zero point is not
    clamped, so stored zeros reach the thousands and the group-128 kernel
    takes its split z = z_lo + 256 k. Its two partial sums carry at most
    |q - z_lo| + 256 |k| <= |q - z| + 256 per product, under 4 times |q - z|
    for |z| > 128, so the bound is widened by 4."""
    rng = np.random.default_rng(M * 7 + N + K)
    W = rng.standard_normal((N, K)) * 0.02
    offsets = rng.choice([0.0, 0.5, -0.5, 2.0, -2.0, 20.0, -20.0], size=(N, K // 128))
    W = W + np.repeat(offsets, 128, axis=1)
    s = O.f32(rng.uniform(0.999, 1.001, K))  # a near-flat scale keeps each offset group narrow
    pk = O.quantize_pack(W, s)
    z = pk["zeros"].astype(np.float64)
    assert np.isfinite(z).all() and (z < -128).any() and (z > 127).any() and (np.abs(z) > 2048).any()
    x = workloads.round_to_bf16((rng.standard_normal((M, K)) * 2.0).astype(np.float32)).astype(np.float64)
    got = _run(x.astype(np.float32), pk)
    ref = O.w4a16_linear(x, pk["qweight"], pk["scales"], pk["zeros"])
    W_hat = O.dequantize_groups(O.unpack_words(pk["qweight"], K), pk["scales"].astype(np.float64), z)
    bad = np.abs(got - ref) > 4 * _bound(x, W_hat)
    assert not bad.any(), f"{bad.sum()} outputs off, max err {np.abs(got - ref).max():.3e}"


@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("M,N,K", [(1, 300, 1024), (4, 130, 640), (8, 520, 4096), (1, 4096, 4096)])
def test_w4a16_finer_groups_match_oracle(group, M, N, K):
    """Groups of 32 and 64: one stored step and zero per 32 or 64 columns."""
    rng = np.random.default_rng(group * 7 + M * 1000 + N + K)
    pk = _random_packed(rng, N, K, group)
    x = workloads.round_to_bf16((rng.standard_normal((M, K)) * 2.0).astype(np.float32)).astype(np.float64)
    got = _run(x.astype(np.float32), pk, group)
    ref = O.w4a16_linear(x, pk["qweight"], pk["scales"], pk["zeros"], group=group)
    W_hat = O.dequantize_groups(O.unpack_words(pk["qweight"], K), pk["scales"].astype(np.float64),
                                pk["zeros"].astype(np.float64), group)
    bad = np.abs(got - ref) > _bound(x, W_hat)
    assert not bad.any(), f"{bad.sum()} outputs off, max err {np.abs(got - ref).max():.3e}"


@pytest.mark.parametrize("M,K", [(1, 45056), (8, 5632), (2, 22528)])
def test_w4a16_at_the_largest_token_channel_count(M, K):
    """n_tok * in at AWQ_W4A16_MAX_TOKEN_CHANNELS (the activations fill the kernel's shared memory)."""
    assert M * K == capi.AWQ_W4A16_MAX_TOKEN_CHANNELS
    rng = np.random.default_rng(K + M)
    N = 130
    pk = _random_packed(rng, N, K)
    x = workloads.round_to_bf16((rng.standard_normal((M, K)) * 2.0).astype(np.float32)).astype(np.float64)
    got = _run(x.astype(np.float32), pk)
    ref = O.w4a16_linear(x, pk["qweight"], pk["scales"], pk["zeros"])
    W_hat = O.dequantize_groups(O.unpack_words(pk["qweight"], K), pk["scales"].astype(np.float64),
                                pk["zeros"].astype(np.float64))
    assert not (np.abs(got - ref) > _bound(x, W_hat)).any()


@pytest.mark.parametrize("M,N,K", [(1, 28672, 8192), (4, 28672, 8192), (8, 28672, 5632), (1, 16400, 8192)])
def test_w4a16_full_size_sampled_rows(M, N, K):
    """70B-class MLP shapes in the launch configuration the benchmark times
    (one token on a layer above the single-token size threshold takes the
    tensor-core kernel), on random codes, steps and zero points (a tenth of
    them far outside the code range), checked on 512 sampled rows, the first
    and the last row tile included."""
    rng = np.random.default_rng(M * 7 + N + K)
    G = K // 128
    qweight = rng.integers(-2**31, 2**31, size=(N, K // 8), dtype=np.int64).astype(np.int32)
    scales = rng.uniform(1e-3, 1e-2, size=(N, G)).astype(np.float16)
    zeros = rng.integers(0, 16, size=(N, G)).astype(np.float64)
    far = rng.random((N, G)) < 0.1
    zeros[far] = rng.integers(-3000, 3000, size=far.sum())
    zeros = zeros.astype(np.float16)
    x = workloads.round_to_bf16((rng.standard_normal((M, K)) * 2.0).astype(np.float32)).astype(np.float64)
    y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    capi.awq_w4a16_gemv(dev_bf16(x.astype(np.float32)), torch.from_numpy(qweight).cuda(),
                        torch.from_numpy(scales.view(np.int16)).cuda(), torch.from_numpy(zeros.view(np.int16)).cuda(),
                        capi.config(), y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    # the order of every sum is fixed: a second call gives the same bits
    y2 = torch.empty_like(y)
    capi.awq_w4a16_gemv(dev_bf16(x.astype(np.float32)), torch.from_numpy(qweight).cuda(),
                        torch.from_numpy(scales.view(np.int16)).cuda(), torch.from_numpy(zeros.view(np.int16)).cuda(),
                        capi.config(), y2)
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))
    rows = np.unique(np.concatenate([np.arange(16), np.arange(N - 16, N), rng.choice(N, 480, replace=False)]))
    ref = O.w4a16_linear(x, qweight[rows], scales[rows], zeros[rows])
    W_hat = O.dequantize_groups(O.unpack_words(qweight[rows], K), scales[rows].astype(np.float64),
                                zeros[rows].astype(np.float64))
    # far zero points: the split z = z_lo + 256 k widens the bound by 4 (see the far-zero-point test)
    bad = np.abs(got[:, rows] - ref) > 4 * _bound(x, W_hat)
    assert not bad.any(), f"{bad.sum()} outputs off, max err {np.abs(got[:, rows] - ref).max():.3e}"


def test_layer_packed_on_gpu_reproduces_the_searched_weight():
    """Search-side weight and inference-side packed layer agree: the GPU pack
    of W * diag(s) applied to x / s equals x W_hat^T of the fake-quant, up to
    the fp16 storage of each group's step (2^-11) and the fp32 sums."""
    L = workloads.make_layer("llama7b_q_proj", n_tok=64, out_features=384, in_features=2048)
    W, X = L["W"].astype(np.float64), L["X"]
    N, K = W.shape
    s32 = O.f32(O.awq_scales(O.channel_importance(X), 0.4))
    qw = torch.empty(N, K // 8, dtype=torch.int32, device="cuda")
    sc = torch.empty(N, K // 128, dtype=torch.float16, device="cuda")
    zr = torch.empty(N, K // 128, dtype=torch.float16, device="cuda")
    capi.awq_quantize_pack(dev_weight(L), dev_f32(s32), capi.config(), qw, sc, zr)
    x = workloads.round_to_bf16((X[:4] / s32[None, :]).astype(np.float32)).astype(np.float64)
    y = torch.empty(4, N, dtype=torch.float32, device="cuda")
    capi.awq_w4a16_gemv(dev_bf16(x.astype(np.float32)), qw, sc, zr, capi.config(), y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    W_hat = O.fake_quantize(W, s32)
    ref = x @ (W_hat * s32[None, :]).T  # x already carries 1/s
    bound = 2.0**-11 * (np.abs(x) @ np.abs(W_hat * s32[None, :]).T) + _bound(x, W_hat * s32[None, :])
    assert np.all(np.abs(got - ref) <= bound)


# ------------------------------------------------------------------ prefill: expanded weight on the tensor cores


def _run_gemm(x32, pk, group=128):
    M, K = x32.shape
    N = pk["qweight"].shape[0]
    cfg = capi.config(group=group)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(capi.awq_w4a16_gemm_workspace_size(M, K, N, cfg), dtype=torch.uint8, device="cuda")
    capi.awq_w4a16_gemm(dev_bf16(x32), torch.from_numpy(pk["qweight"]).cuda(),
                        torch.from_numpy(pk["scales"].view(np.int16)).cuda(),
                        torch.from_numpy(pk["zeros"].view(np.int16)).cuda(), cfg, y, ws)
    assert capi.awq_get_device_status(ws) == capi.AWQ_OK
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,N,K,group", [(16, 300, 1024, 128), (129, 520, 640, 64), (1000, 4096, 4096, 128),
                                         (300, 130, 8192, 32), (9, 7, 128, 128)])
def test_w4a16_gemm_matches_oracle(M, N, K, group):
    """The prefill product: against x times the oracle's bf16 weight within the fp32 accumulation bound,
    and against the exact packed layer within the bf16 rounding of the weight."""
    rng = np.random.default_rng(M + N + K + group)
    pk = _random_packed(rng, N, K, group)
    x = workloads.round_to_bf16((rng.standard_normal((M, K)) * 2.0).astype(np.float32)).astype(np.float64)
    got = _run_gemm(x.astype(np.float32), pk, group)
    Wb = O.w4a16_expand_bf16(pk["qweight"], pk["scales"], pk["zeros"], group)
    ref = x @ Wb.T
    mag = np.abs(x) @ np.abs(Wb).T
    bad = np.abs(got - ref) > K * 2.0**-24 * mag + 1e-30
    assert not bad.any(), f"{bad.sum()} outputs off, max err {np.abs(got - ref).max():.3e}"
    exact = O.w4a16_linear(x, pk["qweight"], pk["scales"], pk["zeros"], group=group)
    assert np.all(np.abs(got - exact) <= (2.0**-8 + K * 2.0**-24) * mag + 1e-30)
