"""The allocation-free statistics entry point, checked against the regular one
and against the oracle.

awq_act_stats_noalloc serves callers that cannot call cudaMalloc or pass a
scratch buffer (a plugin that only receives its inputs and outputs from the
engine owning device memory, or a path where an allocation would synchronise
the device). It keeps its partial sums in a fixed library-owned device array,
so two calls in a row must each match awq_act_stats, which takes a caller
workspace, and the oracle's mean |x| per channel. This file is collected last
so that a failure here leaves every other test already run.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads
from gpu_util import dev_bf16
from post_bit_weight_awq_b300 import build, capi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    capi.lib()


def _stats_with_workspace(X):
    n, K = X.shape
    out = torch.empty(K, dtype=torch.float32, device="cuda")
    ws = torch.empty(capi.awq_act_stats_workspace_size(n, K), dtype=torch.uint8, device="cuda")
    capi.awq_act_stats(X, out, ws)
    return out


def test_noalloc_stats_match_workspace_entry_point_twice():
    rng = np.random.default_rng(77)
    shapes = [(4096, 4096), (1000, 11008)]  # the second call reuses the array with another shape
    for n, K in shapes:
        X32 = workloads.round_to_bf16((rng.standard_normal((n, K)) * 2.0).astype(np.float32))
        X32[:, ::53] *= 25.0
        X32 = workloads.round_to_bf16(X32)  # the values the device holds
        X = dev_bf16(X32)
        got = torch.empty(K, dtype=torch.float32, device="cuda")
        capi.awq_act_stats_noalloc(X, got)
        ref = _stats_with_workspace(X)
        torch.cuda.synchronize()
        got = got.cpu().numpy()
        np.testing.assert_allclose(got, ref.cpu().numpy(), rtol=1e-5, atol=0)
        np.testing.assert_allclose(got, O.channel_importance(X32), rtol=1e-5, atol=0)


def test_noalloc_stats_reject_sizes_beyond_the_fixed_scratch():
    # one chunk of 2^20 + 128 channels is more partial sums than the fixed array holds: refused on the host,
    # nothing launched
    with pytest.raises(capi.AwqError) as e:
        capi.awq_act_stats_noalloc(0x1000, 0x2000, 0, n_tok=16384, in_features=(1 << 20) + 128,
                                   x_dtype=capi.AWQ_BF16)
    assert e.value.status == capi.AWQ_ERR_WORKSPACE
