"""C-ABI checks that need no GPU: the library loads, exports exactly what
include/awq.h declares, and rejects bad arguments on the host before any
CUDA call (every call below passes stream 0 and fake pointers, so reaching a
launch would fail loudly on a machine without a driver)."""
import ctypes
import os
import re

import pytest

import oracle as O
from post_bit_weight_awq_b300 import build, capi, capi_testing

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "awq.h")
STAGES_HEADER = os.path.join(ROOT, "include", "awq_stages.h")
TESTING_HEADER = os.path.join(ROOT, "include", "awq_testing.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return capi_testing.lib()


def header_functions(path=HEADER):
    text = open(path).read()
    return sorted(set(re.findall(r"^AWQ_API\s+[\w\s\*]+?\b(awq_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_list():
    """The product header declares exactly the product binding; the stage calls and the test aids live in
    their own headers and their own binding module."""
    assert header_functions() == sorted(capi.EXPORTED)
    assert header_functions(STAGES_HEADER) == sorted(capi_testing.STAGE_EXPORTED)
    assert header_functions(TESTING_HEADER) == sorted(capi_testing.TESTING_EXPORTED)
    assert not set(capi.EXPORTED) & set(capi_testing.STAGE_EXPORTED + capi_testing.TESTING_EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    declared = header_functions() + header_functions(STAGES_HEADER) + header_functions(TESTING_HEADER)
    for name in declared:
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {capi.LIB_PATH}").read()
    exported = sorted(set(re.findall(r"\bT (awq_\w+)", out)))
    assert exported == sorted(declared)


def test_product_binding_loads_without_the_test_aids():
    """The product binding sets the signatures of the product calls only."""
    import inspect

    src = inspect.getsource(capi)
    for name in capi_testing.STAGE_EXPORTED + capi_testing.TESTING_EXPORTED:
        assert f'"{name}"' not in src, name


def test_library_is_built_for_sm_103a_only():
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_config_default(lib):
    c = capi.config()
    assert (c.w_bit, c.group, c.n_grid, c.zero_point, c.normalize) == (4, 128, 20, 1, 1)
    assert c.sx_clamp_min == pytest.approx(1e-4) and c.delta_floor == pytest.approx(1e-5)
    assert c.loss_form == capi.AWQ_LOSS_AUTO
    assert ctypes.sizeof(capi.AwqConfig) == 36


@pytest.mark.parametrize("shape,form", [
    ((128, 256, 256), "RESIDUAL"),         # tiny linear: X^T X costs more than the products it saves
    ((4096, 4096, 4096), "GRAM"),         # Llama-7B q_proj: in == n_tok, about half the flops
    ((4096, 11008, 4096), "GRAM"),        # Llama-7B up
    ((4096, 4096, 11008), "RESIDUAL"),    # Llama-7B down: in > n_tok, the Gram form costs more
    ((16384, 13824, 5120), "GRAM"),       # 13B-class up_proj
    ((16384, 28672, 8192), "GRAM"),       # 70B-class MLP
])
def test_auto_form_resolution(lib, shape, form):
    """AUTO picks the GRAM form exactly when its tensor-core flops (X^T X over the tiles on and below the block
    diagonal, then per alpha each 128-row block over its prefix of 256-channel blocks) are below 0.7 of the
    direct product's 2 n_grid n_tok out in; the workspace is sized for the form it picks."""
    n, N, K = shape
    cfg = capi.config()
    assert capi.awq_search_form(n, N, K, cfg) == getattr(capi, "AWQ_LOSS_" + form)
    assert capi.awq_workspace_size(n, N, K, cfg) == capi.awq_workspace_size(
        n, N, K, capi.config(loss_form=getattr(capi, "AWQ_LOSS_" + form)))
    for f in (capi.AWQ_LOSS_RESIDUAL, capi.AWQ_LOSS_REFERENCE, capi.AWQ_LOSS_GRAM):
        assert capi.awq_search_form(n, N, K, capi.config(loss_form=f)) == f
    # the rule written out from the tiling
    ct = K // 128
    m, b = ct // 2, ct % 2
    n_pad = (n + 63) // 64 * 64
    h = 2.0 * (m + 1) * (m + b) * 128 * 256 * n_pad
    nC, nR = (K + 255) // 256, (N + 127) // 128
    loss = 2.0 * 20 * nR * 128 * 256 * sum(min(256 * (c + 1), K) for c in range(nC))
    assert (h + loss < 0.7 * 2.0 * 20 * n * N * K) == (form == "GRAM")


def test_gram_form_channel_limit(lib):
    """The GRAM form's transpose takes in / 64 rows of tiles on one grid axis (at most 65535): past
    65535 * 64 channels AUTO keeps the direct form and an explicit GRAM request is refused up front."""
    n, N, K = 1 << 23, 128, 65536 * 64
    assert capi.awq_search_form(n, N, K, capi.config()) == capi.AWQ_LOSS_RESIDUAL
    gram = capi.config(loss_form=capi.AWQ_LOSS_GRAM)
    for fn in (lambda: capi.awq_search_form(n, N, K, gram), lambda: capi.awq_workspace_size(n, N, K, gram),
               lambda: capi.awq_pipeline_workspace_size(n, N, K, capi.AWQ_BF16, gram)):
        with pytest.raises(capi.AwqError) as e:
            fn()
        assert e.value.status == capi.AWQ_ERR_UNSUPPORTED
    # just inside the limit the explicit form is accepted
    assert capi.awq_search_form(1 << 16, N, 65535 * 64 - 64, gram) == capi.AWQ_LOSS_GRAM


def test_auto_form_rejects_unknown_forms(lib):
    with pytest.raises(capi.AwqError):
        capi.awq_search_form(128, 256, 256, capi.config(loss_form=4))


def test_status_strings(lib):
    for code in range(8):
        assert capi.status_string(code)
    assert capi.status_string(123) == "unknown status"


def test_packed_bytes_matches_13b_arithmetic(lib):
    cfg = capi.config()
    rows = 13_000_000_000 // 128
    b = capi.awq_packed_bytes(rows, 128, cfg)
    assert b == 6_500_000_000 + 2 * (13_000_000_000 // 128) * 2


def test_workspace_sizes(lib):
    cfg = capi.config()
    n, N, K = 4096, 4096, 4096
    ws = capi.awq_workspace_size(n, N, K, capi.config(loss_form=capi.AWQ_LOSS_RESIDUAL))
    assert ws >= 20 * N * K * 2 + 2 * 20 * K * 4
    ref = capi.awq_workspace_size(n, N, K, capi.config(loss_form=capi.AWQ_LOSS_REFERENCE))
    assert ref >= ws + N * K * 2
    # the GRAM form adds X^T X (bf16 [in][in]); X^T itself shares the operands' space
    gram = capi.awq_workspace_size(n, N, K, capi.config(loss_form=capi.AWQ_LOSS_GRAM))
    assert gram >= ws + K * K * 2
    assert capi.awq_workspace_size(n, N, K, cfg) == gram  # AUTO picks GRAM here
    assert capi.awq_act_stats_workspace_size(n, K) >= (n // 128) * K * 4
    mt, nt, tm, tn = capi_testing.awq_search_tiles(n, N, cfg)
    assert (mt, nt) == ((n + tm - 1) // tm, (N + tn - 1) // tn)


def _status_of(fn, *a, **k):
    try:
        fn(*a, **k)
    except capi.AwqError as e:
        return e.status
    return capi.AWQ_OK


def test_host_validation_of_act_stats(lib):
    A, B, C = 0x1000, 0x2000, 0x3000
    f = capi.awq_act_stats
    kw = dict(n_tok=64, in_features=128, x_dtype=capi.AWQ_BF16, ws_bytes=1 << 20)
    assert _status_of(f, 0, B, C, 0, **kw) == capi.AWQ_ERR_INVALID_ARG
    assert _status_of(f, A, 0, C, 0, **kw) == capi.AWQ_ERR_INVALID_ARG
    assert _status_of(f, A + 8, B, C, 0, **kw) == capi.AWQ_ERR_MISALIGNED
    assert _status_of(f, A, B, C, 0, **{**kw, "x_dtype": capi.AWQ_FP32}) == capi.AWQ_ERR_UNSUPPORTED
    assert _status_of(f, A, B, C, 0, **{**kw, "x_dtype": 7}) == capi.AWQ_ERR_INVALID_ARG
    assert _status_of(f, A, B, C, 0, **{**kw, "in_features": 100}) == capi.AWQ_ERR_INVALID_ARG
    assert _status_of(f, A, B, C, 0, **{**kw, "n_tok": 0}) == capi.AWQ_ERR_INVALID_ARG
    assert _status_of(f, A, B, C, 0, **{**kw, "ws_bytes": 16}) == capi.AWQ_ERR_WORKSPACE


def test_host_validation_of_search_and_pack(lib):
    A, B, C, D = 0x1000, 0x2000, 0x3000, 0x4000
    cfg = capi.config()
    kw = dict(out_features=256, in_features=256, n_tok=128, w_dtype=capi.AWQ_BF16, x_dtype=capi.AWQ_BF16)
    need = capi.awq_workspace_size(128, 256, 256, cfg)
    s = capi.awq_search_layer
    assert _status_of(s, A, B, C, cfg, D, D, D, 0, 0, ws_bytes=need, **kw) == capi.AWQ_ERR_INVALID_ARG
    assert _status_of(s, A, B, C, cfg, D, D, D, D, 0, ws_bytes=need - 1, **kw) == capi.AWQ_ERR_WORKSPACE
    # groups of 32, 64 and 128 and codes of 2 to 8 bits are built; others are refused before any launch
    for bad in (dict(group=256), dict(group=16), dict(group=96), dict(w_bit=9), dict(w_bit=1)):
        assert _status_of(s, A, B, C, capi.config(**bad), D, D, D, D, 0, ws_bytes=need, **kw) == \
            capi.AWQ_ERR_UNSUPPORTED, bad
    assert _status_of(s, A, B, C, capi.config(w_bit=0), D, D, D, D, 0, ws_bytes=need, **kw) == \
        capi.AWQ_ERR_INVALID_ARG
    assert _status_of(s, A, B, C, capi.config(n_grid=65), D, D, D, D, 0, ws_bytes=need, **kw) == \
        capi.AWQ_ERR_INVALID_ARG
    assert _status_of(s, A, B, C, capi.config(zero_point=2), D, D, D, D, 0, ws_bytes=need, **kw) == \
        capi.AWQ_ERR_INVALID_ARG
    assert _status_of(s, A, B, C, capi.config(loss_form=5), D, D, D, D, 0, ws_bytes=need, **kw) == \
        capi.AWQ_ERR_INVALID_ARG
    assert _status_of(s, A, B, C, cfg, D, D, D, D + 4, 0, ws_bytes=need, **kw) == capi.AWQ_ERR_MISALIGNED
    assert _status_of(s, A, B, C, cfg, D, D, D, D, 0, ws_bytes=need, **{**kw, "in_features": 200}) == \
        capi.AWQ_ERR_INVALID_ARG
    p = capi.awq_quantize_pack
    pkw = dict(out_features=4, in_features=128, w_dtype=capi.AWQ_FP32)
    assert _status_of(p, A, B, cfg, C, D, 0, 0, **pkw) == capi.AWQ_ERR_INVALID_ARG
    assert _status_of(p, A, B, cfg, C + 4, D, D, 0, **pkw) == capi.AWQ_ERR_MISALIGNED
    assert _status_of(p, A, B, cfg, C, D + 1, D, 0, **pkw) == capi.AWQ_ERR_MISALIGNED
    # codes are packed for 2, 4 and 8 bits (widths that divide a 32-bit word), at any built group size
    for bad in (dict(w_bit=3), dict(w_bit=6), dict(w_bit=3, group=32), dict(group=256)):
        assert _status_of(p, A, B, capi.config(**bad), C, D, D, 0, **pkw) == capi.AWQ_ERR_UNSUPPORTED, bad
    assert _status_of(p, A, B, cfg, C, D, D, 0, **{**pkw, "w_dtype": 3}) == capi.AWQ_ERR_INVALID_ARG


def test_host_validation_of_fused_search(lib):
    A, B, C, D = 0x1000, 0x2000, 0x3000, 0x4000
    f = capi_testing.awq_search_fused
    kw = dict(out_features=256, in_features=256, n_tok=128, w_dtype=capi.AWQ_BF16)
    cfg = capi.config()
    assert _status_of(f, A, B, C, C, capi.config(loss_form=capi.AWQ_LOSS_REFERENCE), D, D, D, D, 0, **kw) == \
        capi.AWQ_ERR_UNSUPPORTED
    assert _status_of(f, A, B, C, C, cfg, D, D, 0, D, 0, **kw) == capi.AWQ_ERR_INVALID_ARG
    assert _status_of(f, A, B, C, C, cfg, D, D, D + 4, D, 0, **kw) == capi.AWQ_ERR_MISALIGNED
    assert _status_of(f, A, B, C, C, cfg, D, D, D, D, 0, **{**kw, "w_dtype": 9}) == capi.AWQ_ERR_INVALID_ARG


def test_host_validation_of_w4a16(lib):
    f = capi.awq_w4a16_gemv
    A, B, C, D, E = 0x1000, 0x2000, 0x3000, 0x4000, 0x5000
    kw = dict(n_tok=2, in_features=256, out_features=4, x_dtype=capi.AWQ_BF16)
    cfg = capi.config()
    assert _status_of(f, A, B, C, D, cfg, E, 0, **{**kw, "n_tok": 9}) == capi.AWQ_ERR_UNSUPPORTED
    assert _status_of(f, A, B, C, D, cfg, E, 0, **{**kw, "n_tok": 8, "in_features": 8192}) == \
        capi.AWQ_ERR_UNSUPPORTED
    assert _status_of(f, A, B, C, D, cfg, 0, 0, **kw) == capi.AWQ_ERR_INVALID_ARG
    assert _status_of(f, A, B + 4, C, D, cfg, E, 0, **kw) == capi.AWQ_ERR_MISALIGNED
    assert _status_of(f, A, B, C + 1, D, cfg, E, 0, **kw) == capi.AWQ_ERR_MISALIGNED
    assert _status_of(f, A, B, C, D, cfg, E, 0, **{**kw, "in_features": 200}) == capi.AWQ_ERR_INVALID_ARG
    for bad in (dict(group=256), dict(w_bit=2), dict(w_bit=8, group=64)):
        assert _status_of(f, A, B, C, D, capi.config(**bad), E, 0, **kw) == capi.AWQ_ERR_UNSUPPORTED, bad


def test_host_validation_of_block_search(lib):
    cfg = capi.config()
    with pytest.raises(capi.AwqError) as e:
        capi.awq_search_block_workspace_size(128, [], 256, cfg)
    assert e.value.status == capi.AWQ_ERR_INVALID_ARG
    with pytest.raises(capi.AwqError) as e:
        capi.awq_search_block_workspace_size(128, [8] * 17, 256, cfg)
    assert e.value.status == capi.AWQ_ERR_INVALID_ARG
    one = capi.awq_search_block_workspace_size(128, [512], 256, cfg)
    three = capi.awq_search_block_workspace_size(128, [256, 128, 128], 256, cfg)
    assert three == one == capi.awq_workspace_size(128, 512, 256, cfg) + 512 * 256 * 2
    f = capi.awq_search_block
    A, B, C, D = 0x1000, 0x2000, 0x3000, 0x4000
    kw = dict(outs=[64, 64], in_features=256, n_tok=128, w_dtype=capi.AWQ_BF16, x_dtype=capi.AWQ_BF16,
              ws_bytes=1 << 30)
    assert _status_of(f, [A, 0], B, C, cfg, D, D, D, D, 0, **kw) == capi.AWQ_ERR_INVALID_ARG
    assert _status_of(f, [A, A + 8], B, C, cfg, D, D, D, D, 0, **kw) == capi.AWQ_ERR_MISALIGNED
    assert _status_of(f, [A, A], B, C, cfg, D, D, D, D, 0, **{**kw, "ws_bytes": 1024}) == capi.AWQ_ERR_WORKSPACE
    assert _status_of(f, [A, A], B, C, cfg, D, D, D, D, 0, **{**kw, "outs": [64, 0]}) == capi.AWQ_ERR_INVALID_ARG


def test_host_validation_of_layer_pipeline(lib):
    cfg = capi.config()
    need = capi.awq_pipeline_workspace_size(128, 256, 512, capi.AWQ_BF16, cfg)
    # two slots of inputs and outputs on top of the search workspace and the statistics scratch
    slot = 256 * 512 * 2 + 128 * 512 * 2 + 256 * 512 // 2 + 2 * 256 * 4 * 2 + 2 * 512 * 4
    assert need >= capi.awq_workspace_size(128, 256, 512, cfg) + 2 * slot
    assert capi.awq_pipeline_workspace_size(128, 256, 512, capi.AWQ_FP32, cfg) > need
    with pytest.raises(capi.AwqError) as e:
        capi.awq_pipeline_workspace_size(128, 256, 512, capi.AWQ_BF16, capi.config(w_bit=3))
    assert e.value.status == capi.AWQ_ERR_UNSUPPORTED
    A = 0x10000
    io = capi.AwqLayerIO(A, A, 128, 256, 512, A, A, A, A, A, A, 0)
    f = capi.lib().awq_quantize_layers

    def call(layers, count, w_dtype=capi.AWQ_BF16, c=cfg, ws=0x100000, ws_bytes=need):
        arr = (capi.AwqLayerIO * max(1, len(layers)))(*layers)
        return f(ctypes.cast(arr, ctypes.c_void_p) if layers else None, count, w_dtype, ctypes.byref(c), ws,
                 ws_bytes, None)

    assert call([], 0) == capi.AWQ_ERR_INVALID_ARG
    assert call([io], 0) == capi.AWQ_ERR_INVALID_ARG
    assert call([io], 1, ws=0) == capi.AWQ_ERR_INVALID_ARG
    assert call([io], 1, ws=0x100004) == capi.AWQ_ERR_MISALIGNED
    assert call([io], 1, ws_bytes=need - 1) == capi.AWQ_ERR_WORKSPACE
    assert call([io], 1, c=capi.config(w_bit=3)) == capi.AWQ_ERR_UNSUPPORTED  # 3-bit codes are not packed
    assert call([io], 1, w_dtype=7) == capi.AWQ_ERR_INVALID_ARG
    bad = capi.AwqLayerIO(A, A, 128, 256, 200, A, A, A, A, A, A, 0)  # in not a multiple of 128
    assert call([io, bad], 2) == capi.AWQ_ERR_INVALID_ARG
    null = capi.AwqLayerIO(A, A, 128, 256, 512, 0, A, A, A, A, A, 0)
    assert call([io, null], 2) == capi.AWQ_ERR_INVALID_ARG
    big = capi.AwqLayerIO(A, A, 129, 256, 512, A, A, A, A, A, A, 0)  # more tokens than the workspace was sized for
    assert call([io, big], 2) == capi.AWQ_ERR_WORKSPACE


def test_bounds_checks_are_absent_from_the_release_library(lib):
    f, u, ln, off = ctypes.c_uint64(), ctypes.c_int32(), ctypes.c_uint64(), ctypes.c_uint64()
    assert lib.awq_bounds_report(ctypes.byref(f), ctypes.byref(u), ctypes.byref(ln), ctypes.byref(off)) == \
        capi.AWQ_ERR_UNSUPPORTED
    assert lib.awq_bounds_selftest(ctypes.c_void_p(0x1000), 4, None) == capi.AWQ_ERR_UNSUPPORTED
    assert lib.awq_bounds_report(None, ctypes.byref(u), ctypes.byref(ln), ctypes.byref(off)) == \
        capi.AWQ_ERR_INVALID_ARG


def test_checked_library_builds_and_exports_the_same_calls():
    path = build.build(checked=True)
    checked = ctypes.CDLL(path)
    for name in capi.EXPORTED + capi_testing.STAGE_EXPORTED + capi_testing.TESTING_EXPORTED:
        assert hasattr(checked, name), name


def test_binding_constants_match_the_header():
    for path, mod, names in ((HEADER, capi, ("AWQ_W4A16_MAX_TOKENS", "AWQ_W4A16_MAX_TOKEN_CHANNELS",
                                             "AWQ_BLOCK_MAX_LINEARS")),
                             (STAGES_HEADER, capi_testing, ("AWQ_SEARCH_FUSED_MAX_FLOPS",))):
        text = open(path).read()
        for name in names:
            m = re.search(r"#define\s+" + name + r"\s+(.+)", text)
            assert m, name
            assert eval(m.group(1).split("/*")[0].strip()) == getattr(mod, name), name


def test_host_validation_of_w4a16_gemm(lib):
    f = capi.awq_w4a16_gemm
    A, B, C, D, E, F = 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000
    cfg = capi.config()
    need = capi.awq_w4a16_gemm_workspace_size(64, 256, 128, cfg)
    assert need >= 128 * 256 * 2  # the bf16 weight
    kw = dict(n_tok=64, in_features=256, out_features=128, x_dtype=capi.AWQ_BF16, ws_bytes=need)
    assert _status_of(f, A, B, C, D, cfg, 0, F, 0, **kw) == capi.AWQ_ERR_INVALID_ARG
    assert _status_of(f, A, B, C, D, cfg, E + 4, F, 0, **kw) == capi.AWQ_ERR_MISALIGNED
    assert _status_of(f, A, B, C, D, cfg, E, F, 0, **{**kw, "ws_bytes": need - 1}) == capi.AWQ_ERR_WORKSPACE
    assert _status_of(f, A, B, C, D, capi.config(w_bit=3), E, F, 0, **kw) == capi.AWQ_ERR_UNSUPPORTED
    assert _status_of(f, A, B, C, D, cfg, E, F, 0, **{**kw, "in_features": 200}) == capi.AWQ_ERR_INVALID_ARG
    assert _status_of(f, A, B, C, D, cfg, E, F, 0, **{**kw, "x_dtype": capi.AWQ_FP32}) == capi.AWQ_ERR_UNSUPPORTED


@pytest.mark.parametrize("w_bit", [2, 4, 8])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("zero_point", [0, 1])
def test_packed_bytes_matches_the_oracle_for_every_layout(lib, w_bit, group, zero_point):
    cfg = capi.config(w_bit=w_bit, group=group, zero_point=zero_point)
    for out, inf in ((4096, 4096), (28672, 8192), (7, 128)):
        ref = O.packed_bytes(out, inf, group=group, w_bit=w_bit, zero_point=bool(zero_point))
        assert capi.awq_packed_bytes(out, inf, cfg) == ref["total"]


def test_workspace_sizes_grow_with_every_dimension(lib):
    cfg = capi.config()
    base = (1024, 1024, 1024)
    for fn in (lambda n, N, K: capi.awq_workspace_size(n, N, K, cfg),
               lambda n, N, K: capi.awq_pipeline_workspace_size(n, N, K, capi.AWQ_BF16, cfg),
               lambda n, N, K: capi.awq_w4a16_gemm_workspace_size(n, K, N, cfg)):
        b = fn(*base)
        for i in range(3):
            dims = list(base)
            dims[i] *= 2
            assert fn(*dims) >= b
    # the search workspace holds the G operand copies; the prefill scratch holds the bf16 weight
    assert capi.awq_workspace_size(1024, 1024, 1024, cfg) >= 20 * 1024 * 1024 * 2
    assert capi.awq_w4a16_gemm_workspace_size(1024, 1024, 1024, cfg) >= 1024 * 1024 * 2
    # more alphas, more operand copies
    assert capi.awq_workspace_size(256, 256, 256, capi.config(n_grid=64)) > \
        capi.awq_workspace_size(256, 256, 256, capi.config(n_grid=20))


def test_every_status_has_its_own_message(lib):
    codes = [capi.AWQ_OK, capi.AWQ_ERR_INVALID_ARG, capi.AWQ_ERR_UNSUPPORTED, capi.AWQ_ERR_MISALIGNED,
             capi.AWQ_ERR_WORKSPACE, capi.AWQ_ERR_CUDA, capi.AWQ_ERR_TIMEOUT, capi.AWQ_ERR_NONFINITE]
    msgs = [capi.status_string(c) for c in codes]
    assert len(set(msgs)) == len(codes)
    assert "unknown" in capi.status_string(99)


def test_layer_api_rejects_bad_inputs_before_the_library():
    import torch

    from post_bit_weight_awq_b300 import layer

    W = torch.zeros(4, 128, dtype=torch.bfloat16)
    X = torch.zeros(8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        layer.quantize_layer(W, X)  # host tensors


def test_header_is_plain_c_and_links(lib, tmp_path):
    """include/awq.h compiles as C99 with warnings as errors, and a C program linked against libawq.so runs
    the host-only entry points."""
    import shutil
    import subprocess

    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = os.path.join(os.path.dirname(__file__), "c_abi_check.c")
    exe = str(tmp_path / "c_abi_check")
    libdir = os.path.dirname(capi.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), src,
                    "-o", exe, "-L", libdir, "-lawq", "-Wl,-rpath," + libdir], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert "c abi ok" in r.stdout
