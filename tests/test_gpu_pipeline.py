"""Layers streamed from host memory (awq_quantize_layers): every output equals
the one-layer-at-a-time device path bit for bit, whatever the order of layer
sizes and however many layers reuse the two device slots; the losses meet the
oracle's levels; a device-side error in any layer stays in the status word.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads
from gpu_util import dev_bf16, dev_weight
from post_bit_weight_awq_b300 import build, capi, layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    capi.lib()


def _host_inputs(L):
    W = workloads.bf16_bits(L["W"]).view(np.int16) if L["w_dtype"] == "bf16" else L["W"].astype(np.float32)
    Wh = torch.from_numpy(np.ascontiguousarray(W)).pin_memory()
    Xh = torch.from_numpy(workloads.bf16_bits(L["X"]).view(np.int16)).pin_memory()
    return Wh, Xh


def _host_outputs(N, K, cfg):
    pin = dict(pin_memory=True)
    return dict(qweight=torch.zeros(N, K * cfg.w_bit // 32, dtype=torch.int32, **pin),
                scales=torch.zeros(N, K // cfg.group, dtype=torch.int16, **pin),
                zeros=torch.zeros(N, K // cfg.group, dtype=torch.int16, **pin),
                losses=torch.zeros(cfg.n_grid, dtype=torch.float32, **pin),
                best=torch.zeros(1, dtype=torch.int32, **pin),
                s_best=torch.zeros(K, dtype=torch.float32, **pin),
                mean=torch.zeros(K, dtype=torch.float32, **pin))


def _run_pipeline(Ls, cfg, w_dtype):
    ins = [_host_inputs(L) for L in Ls]
    outs = [_host_outputs(*L["W"].shape, cfg) for L in Ls]
    ios = [capi.layer_io(Wh, Xh, o["qweight"], o["scales"], o["zeros"], o["losses"], o["best"], o["s_best"],
                         o["mean"], n_tok=L["X"].shape[0], out=L["W"].shape[0], in_features=L["W"].shape[1])
           for L, (Wh, Xh), o in zip(Ls, ins, outs)]
    dims = np.array([[L["X"].shape[0], *L["W"].shape] for L in Ls]).max(axis=0)
    ws = torch.empty(capi.awq_pipeline_workspace_size(int(dims[0]), int(dims[1]), int(dims[2]), w_dtype, cfg),
                     dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    capi.awq_quantize_layers(ios, w_dtype, cfg, ws, stream)
    status = capi.awq_get_device_status(ws, stream)
    torch.cuda.synchronize()
    return outs, status


def _device_path(L, cfg):
    q = layer.quantize_layer(dev_weight(L), dev_bf16(L["X"]), cfg)
    torch.cuda.synchronize()
    return q


def _assert_same(o, q):
    assert torch.equal(o["qweight"], q.qweight.cpu())
    assert torch.equal(o["scales"], q.scales.cpu().view(torch.int16))
    assert torch.equal(o["zeros"], q.zeros.cpu().view(torch.int16))
    assert torch.equal(o["losses"], q.losses.cpu())
    assert int(o["best"][0]) == int(q.best_idx[0])
    assert torch.equal(o["s_best"], q.s_best.cpu())
    assert torch.equal(o["mean"], q.mean_abs.cpu())


@pytest.mark.parametrize("w_dtype_name", ["bf16", "fp32"])
def test_layers_from_host_equal_the_device_path(w_dtype_name):
    """Five layers of mixed sizes (the largest in the middle, ragged tiles) pass through the two slots;
    each equals awq_act_stats + awq_search_layer + awq_quantize_pack on device copies, bit for bit."""
    shapes = [(257, 300, 640), (64, 130, 256), (512, 1024, 1024), (129, 7, 384), (300, 520, 1024)]
    Ls = []
    for i, (n, N, K) in enumerate(shapes):
        L = workloads.make_layer("llama7b_q_proj", n_tok=n, out_features=N, in_features=K, seed=10 + i)
        if w_dtype_name == "fp32":
            L = dict(L, w_dtype="fp32", W=L["W"].astype(np.float32))
        Ls.append(L)
    cfg = capi.config()
    w_dtype = capi.AWQ_BF16 if w_dtype_name == "bf16" else capi.AWQ_FP32
    outs, status = _run_pipeline(Ls, cfg, w_dtype)
    assert status == capi.AWQ_OK
    for L, o in zip(Ls, outs):
        _assert_same(o, _device_path(L, cfg))


def test_layers_of_both_loss_forms_in_one_call():
    """AUTO resolves per layer: GRAM for layers with in < 2 n_tok and many rows, RESIDUAL for the others. A
    pipeline call mixing both (the largest dimensions come from different layers) equals the device path bit
    for bit; its workspace holds either form's scratch for every layer."""
    shapes = [(2048, 1024, 1024), (300, 520, 1024), (1024, 1536, 768), (64, 256, 2048)]
    cfg = capi.config()
    forms = [capi.awq_search_form(n, N, K, cfg) for n, N, K in shapes]
    assert forms == [capi.AWQ_LOSS_GRAM, capi.AWQ_LOSS_RESIDUAL, capi.AWQ_LOSS_GRAM, capi.AWQ_LOSS_RESIDUAL]
    Ls = [workloads.make_layer("llama7b_q_proj", n_tok=n, out_features=N, in_features=K, seed=40 + i)
          for i, (n, N, K) in enumerate(shapes)]
    outs, status = _run_pipeline(Ls, cfg, capi.AWQ_BF16)
    assert status == capi.AWQ_OK
    for L, o in zip(Ls, outs):
        _assert_same(o, _device_path(L, cfg))


def test_layers_from_host_meet_the_oracle_levels():
    """Levels 2 and 3 (losses within 1e-2, argmin within 0.5%) and level 1 (the pack with the oracle's
    scale, where the GPU chose the same alpha) for two layers with other quantiser knobs."""
    Ls = [workloads.make_layer("llama7b_q_proj", n_tok=512, out_features=640, in_features=1024, seed=s)
          for s in (21, 22)]
    cfg = capi.config(group=64)
    outs, status = _run_pipeline(Ls, cfg, capi.AWQ_BF16)
    assert status == capi.AWQ_OK
    for L, o in zip(Ls, outs):
        sx32 = O.f32(O.channel_importance(L["X"]))
        np.testing.assert_allclose(o["mean"].numpy(), sx32, rtol=1e-5)
        res = O.search_scale(L["W"].astype(np.float64), L["X"].astype(np.float64), sx32, group=64)
        lo = res["losses"]
        lg = o["losses"].numpy().astype(np.float64)
        assert np.all(np.abs(lg - lo) <= 1e-2 * lo)
        assert lo[int(o["best"][0])] <= 1.005 * lo.min()
        s32 = o["s_best"].numpy().astype(np.float64)
        ref = O.quantize_pack(L["W"].astype(np.float64), s32, group=64)
        np.testing.assert_array_equal(o["qweight"].numpy(), ref["qweight"])
        np.testing.assert_array_equal(o["scales"].numpy().view(np.uint16), ref["scales"].view(np.uint16))
        np.testing.assert_array_equal(o["zeros"].numpy().view(np.uint16), ref["zeros"].view(np.uint16))


def test_error_in_one_layer_stays_in_the_status_word():
    """A non-finite activation in the second of three layers: the status word reports it after the call
    (later layers do not clear it), and the other layers' outputs are still exact."""
    Ls = [workloads.make_layer("llama7b_q_proj", n_tok=128, out_features=256, in_features=512, seed=s)
          for s in (31, 32, 33)]
    X = Ls[1]["X"].copy()
    X[5, 40] = np.inf
    Ls[1] = dict(Ls[1], X=X)
    cfg = capi.config()
    outs, status = _run_pipeline(Ls, cfg, capi.AWQ_BF16)
    assert status == capi.AWQ_ERR_NONFINITE
    for i in (0, 2):
        _assert_same(outs[i], _device_path(Ls[i], cfg))


@pytest.mark.parametrize("kw", [dict(loss_form=capi.AWQ_LOSS_REFERENCE), dict(zero_point=0, group=32),
                                dict(w_bit=8, group=64)])
def test_layers_from_host_with_other_configurations(kw):
    """The REFERENCE loss form, and the symmetric quantiser with groups of 32, through the pipeline: the
    same outputs as the one-layer device path."""
    Ls = [workloads.make_layer("llama7b_q_proj", n_tok=n, out_features=N, in_features=K, seed=40 + i)
          for i, (n, N, K) in enumerate([(200, 300, 512), (129, 130, 768), (64, 260, 512)])]
    cfg = capi.config(**kw)
    outs, status = _run_pipeline(Ls, cfg, capi.AWQ_BF16)
    assert status == capi.AWQ_OK
    for L, o in zip(Ls, outs):
        _assert_same(o, _device_path(L, cfg))


def test_layers_from_pageable_host_memory():
    """Unpinned host buffers: the copies lose their overlap but not their correctness."""
    Ls = [workloads.make_layer("llama7b_q_proj", n_tok=128, out_features=256, in_features=512, seed=s)
          for s in (51, 52, 53)]
    cfg = capi.config()
    ins = []
    outs = []
    for L in Ls:
        Wh = torch.from_numpy(np.ascontiguousarray(workloads.bf16_bits(L["W"]).view(np.int16)))
        Xh = torch.from_numpy(np.ascontiguousarray(workloads.bf16_bits(L["X"]).view(np.int16)))
        ins.append((Wh, Xh))
        N, K = L["W"].shape
        outs.append(dict(qweight=torch.zeros(N, K // 8, dtype=torch.int32),
                         scales=torch.zeros(N, K // 128, dtype=torch.int16),
                         zeros=torch.zeros(N, K // 128, dtype=torch.int16),
                         losses=torch.zeros(cfg.n_grid), best=torch.zeros(1, dtype=torch.int32),
                         s_best=torch.zeros(K), mean=torch.zeros(K)))
    ios = [capi.layer_io(Wh, Xh, o["qweight"], o["scales"], o["zeros"], o["losses"], o["best"], o["s_best"], o["mean"],
                         n_tok=128, out=256, in_features=512) for (Wh, Xh), o in zip(ins, outs)]
    ws = torch.empty(capi.awq_pipeline_workspace_size(128, 256, 512, capi.AWQ_BF16, cfg), dtype=torch.uint8,
                     device="cuda")
    capi.awq_quantize_layers(ios, capi.AWQ_BF16, cfg, ws, torch.cuda.current_stream())
    assert capi.awq_get_device_status(ws) == capi.AWQ_OK
    torch.cuda.synchronize()
    for L, o in zip(Ls, outs):
        _assert_same(o, _device_path(L, cfg))


def test_two_host_threads_enqueue_pipelines_at_once():
    """Two threads run the pipeline on their own streams and workspaces at the same time; the shared copy
    streams and events are taken in turn, and both threads get exactly the device path's outputs."""
    import threading

    cfg = capi.config()
    sets = [[workloads.make_layer("llama7b_q_proj", n_tok=128, out_features=256, in_features=512, seed=60 + 10 * t + i)
             for i in range(3)] for t in range(2)]
    results = [None, None]
    errors = []

    def work(t):
        try:
            with torch.cuda.stream(torch.cuda.Stream()):
                results[t] = _run_pipeline(sets[t], cfg, capi.AWQ_BF16)
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for t in range(2):
        outs, status = results[t]
        assert status == capi.AWQ_OK
        for L, o in zip(sets[t], outs):
            _assert_same(o, _device_path(L, cfg))
