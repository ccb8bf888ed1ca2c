"""Benchmark: AWQ per-layer search + INT4 pack on B300, one JSON line.

A step is one pass of the whole path over one synthetic layer through the
library's public calls: awq_act_stats (activation statistics),
awq_search_layer (alpha scales, fake-quant, the tcgen05 products of the
loss form the library picks for the shape, loss + argmin) and
awq_quantize_pack (final codes).
The headline layer is the 70B-class MLP projection (W 28672 x 8192 bf16,
X 16384 x 8192 bf16, 20 alphas), the largest workload of the suite. Inputs
are resident in HBM when the timed region starts; they are larger than L2,
and L2 is flushed (a 512 MiB write, then a 512 MiB read) between steps
anyway, outside the timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, bounded sample

With N > 1 (torchrun) every rank quantises its own copy of the layer
(independent layers, no collective on the data path); value is the job's
milliseconds per layer = max-over-ranks time / layers processed.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ms per layer AWQ search+pack (20-pt α grid); % BF16 TC peak and % HBM BW"
DEFAULT_WORKLOAD = "70b_mlp"
# the other workloads of the suite, each timed through the same calls (one entry per layer, not the headline)
SIDE_WORKLOADS = ("tiny", "llama7b_q_proj", "llama7b_mlp", "13b_up_proj")
RUN_AHEAD_CYCLES = 4_000_000  # GPU spin before each timed step so the host enqueues the whole step first
FLUSH_BYTES = 512 << 20


class L2Flush:
    """Between timed launches: write a 512 MiB buffer (more than the 126 MB L2), then read another 512 MiB
    buffer. The write evicts every cached input; the read then evicts the write's dirty lines, so the next
    timed kernel does not pay for writing the flush buffer back to HBM (126 MB of write-back, which costs
    the statistics kernel 8 of its 55 microseconds on the 70B-class X). Both run outside the timed events."""

    def __init__(self, dev):
        import torch

        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty(1, dtype=torch.int64, device=dev)

    def run(self):
        import torch

        self.w.zero_()
        torch.sum(self.r, dim=0, keepdim=True, out=self.sink)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


GEMM_SOURCES = ["post_bit_weight_awq_b300/csrc/awq_search_gemm.cu", "post_bit_weight_awq_b300/csrc/awq_device.cuh",
                "post_bit_weight_awq_b300/csrc/awq_quant.cuh"]
GRAM_SOURCES = ["post_bit_weight_awq_b300/csrc/awq_gram.cu", "post_bit_weight_awq_b300/csrc/awq_device.cuh",
                "post_bit_weight_awq_b300/csrc/awq_launch.h"]


def gram_prefix_area(K):
    """S = sum over 256-channel blocks cb of (channels in cb) x (channels in blocks 0..cb): the entries of
    X^T X on and below the block diagonal."""
    nC = (K + 255) // 256
    return sum(min(256, K - 256 * c) * min(256 * (c + 1), K) for c in range(nC))


def search_flops(n, N, K, G, form):
    """Algorithmic tensor-core flops of one search: the direct products 2 G n N K, or for the GRAM form X^T X
    on and below the block diagonal (2 n S) plus the alphas' products over the block prefixes (2 G N S)."""
    if form == "gram":
        return 2.0 * gram_prefix_area(K) * (n + G * N)
    return 2.0 * G * n * N * K


def profiled_traffic(kernel_tag, workload):
    """DRAM bytes per launch of the search kernel from the committed ncu summary
    profiles/search_<kernel_tag>_<workload>.md, if it was taken on the current
    kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"search_{kernel_tag}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch\s*=\s*(\d+).*?workload\s*=\s*(\w+).*?source_sha256_16\s*=\s*(\w+)",
                  text, flags=re.S)
    if not m:
        return None
    sources = GRAM_SOURCES if kernel_tag == "gram" else GEMM_SOURCES
    if m.group(2) != workload or m.group(3) != source_digest(sources):
        return None
    return int(m.group(1))


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.out_path = os.path.join("/tmp", f"awq_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.out_path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.out_path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.out_path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_median": statistics.median(pw) if pw else None,
                "power_w_max": max(pw, default=None)}


# ------------------------------------------------------------------ oracle arm


def oracle_sample(L, rows, X64=None):
    """Run the oracle's statistics over all of X, then its search and pack on
    the first ``rows`` output rows of layer ``L`` (all tokens, all input
    channels). The loss is a sum over output rows and s depends only on X, so
    the sample is the oracle's exact work for those rows. Returns the seconds
    of the statistics, the seconds of the row sample and the factor out/rows
    that scales the row sample to the whole layer."""
    import numpy as np

    import oracle as O

    W = L["W"][:rows].astype(np.float64)
    X = L["X"].astype(np.float64) if X64 is None else X64
    N = L["W"].shape[0]
    t0 = time.perf_counter()
    sx = O.channel_importance(X)
    t1 = time.perf_counter()
    res = O.search_scale(W, X, sx)
    O.quantize_pack(W, O.f32(res["s_best"]))
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1, N / rows


def blas_threads():
    try:
        from threadpoolctl import threadpool_info

        return max((p.get("num_threads", 1) for p in threadpool_info()), default=1)
    except Exception:
        return len(os.sched_getaffinity(0))


def reference_arm(args, rank):
    """The CPU oracle as it stands on this host's cores, on a bounded row sample of the same layer per step."""
    if rank != 0:
        return
    import numpy as np

    import workloads

    name = workloads.WORKLOADS[args.workload][0]
    L = workloads.make_layer(name)
    X64 = L["X"].astype(np.float64)
    rows = args.reference_rows
    for _ in range(args.warmup):
        oracle_sample(L, rows, X64)
    stats_s, rows_s = [], []
    scale = 1.0
    t_run = time.perf_counter()
    for _ in range(args.steps):
        ts, tr, scale = oracle_sample(L, rows, X64)
        stats_s.append(ts)
        rows_s.append(tr)
    wall = time.perf_counter() - t_run
    sample_ms = (statistics.mean(stats_s) + statistics.mean(rows_s)) * 1e3
    ms = (statistics.mean(stats_s) + statistics.mean(rows_s) * scale) * 1e3
    cores = blas_threads()
    sample = (f"oracle statistics over all {L['X'].shape[0]} tokens ({statistics.mean(stats_s):.2f} s) + search and "
              f"pack of output rows [0,{rows}) of the {name} layer ({statistics.mean(rows_s):.2f} s) per step; "
              f"value = statistics + rows time x out/rows = {scale:g}, one layer")
    line = {"impl": "reference", "metric": METRIC, "value": round(ms, 1), "unit": "ms", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sample_ms, 1),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "layer": name, "W": list(L["W"].shape), "X": list(L["X"].shape),
                       "n_grid": 20, "group": 128},
            "cpu_baseline": {"value": round(ms, 1), "unit": "ms", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(ms, 1), "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s_timed_steps": round(wall, 2)}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm


def timed(fn, flush, reps, warm=0):
    """Median CUDA-event time (ms) of fn() over reps runs, L2 flushed before each, after `warm` untimed runs."""
    import torch

    for _ in range(warm):
        fn()
    ts = []
    for _ in range(reps):
        flush.run()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def hbm_bytes(n, N, K, G, wbytes):
    """Algorithmic bytes of the bandwidth kernels: the statistics read X once; the fake-quant reads W once and
    writes G bf16 operands; the pack reads W and writes the codes, fp16 scales and zeros."""
    return {"stats": 2.0 * n * K, "fakequant": wbytes * N * K + G * 2.0 * N * K,
            "pack": wbytes * N * K + N * K / 2 + 4.0 * N * K / 128}


class LayerRun:
    """One layer resident on the device with the buffers of the three public calls."""

    def __init__(self, name, dev, cfg, rows=None):
        import numpy as np
        import torch

        import workloads
        from post_bit_weight_awq_b300 import capi

        self.name = name
        L = workloads.make_layer(name, out_features=rows)
        self.L = L
        W32, X32 = L["W"], L["X"]
        self.N, self.K = W32.shape
        self.n = X32.shape[0]
        self.cfg = cfg
        self.G = cfg.n_grid
        self.wbytes = 2 if L["w_dtype"] == "bf16" else 4

        def to_dev_bf16(a):
            return torch.from_numpy(workloads.bf16_bits(a).view(np.int16)).to(dev).view(torch.bfloat16)

        self.W = to_dev_bf16(W32) if L["w_dtype"] == "bf16" else torch.from_numpy(W32).to(dev)
        self.X = to_dev_bf16(X32)
        n, N, K, G = self.n, self.N, self.K, self.G
        f32 = torch.float32
        self.mean_abs = torch.empty(K, dtype=f32, device=dev)
        self.ws = torch.empty(max(capi.awq_workspace_size(n, N, K, cfg), capi.awq_act_stats_workspace_size(n, K)),
                              dtype=torch.uint8, device=dev)
        self.losses = torch.empty(G, dtype=f32, device=dev)
        self.best = torch.empty(1, dtype=torch.int32, device=dev)
        self.s_best = torch.empty(K, dtype=f32, device=dev)
        self.qw = torch.empty(N, K // 8, dtype=torch.int32, device=dev)
        self.sc = torch.empty(N, K // 128, dtype=torch.float16, device=dev)
        self.zr = torch.empty(N, K // 128, dtype=torch.float16, device=dev)
        forms = {capi.AWQ_LOSS_RESIDUAL: "residual", capi.AWQ_LOSS_REFERENCE: "reference", capi.AWQ_LOSS_GRAM: "gram"}
        self.form = forms[capi.awq_search_form(n, N, K, cfg)]
        self.flops = search_flops(n, N, K, G, self.form)
        # the dominant kernel's flops: the GRAM form's alpha products, else the whole direct search
        self.loss_flops = 2.0 * G * N * gram_prefix_area(K) if self.form == "gram" else self.flops

    def step(self, ev=None):
        """awq_act_stats, awq_search_layer, awq_quantize_pack on the current stream (events between the calls)."""
        import torch

        from post_bit_weight_awq_b300 import capi

        st = torch.cuda.current_stream()
        if ev:
            ev[0].record(st)
        capi.awq_act_stats(self.X, self.mean_abs, self.ws, st)
        if ev:
            ev[1].record(st)
        capi.awq_search_layer(self.W, self.X, self.mean_abs, self.cfg, self.losses, self.best, self.s_best, self.ws,
                              st)
        if ev:
            ev[2].record(st)
        capi.awq_quantize_pack(self.W, self.s_best, self.cfg, self.qw, self.sc, self.zr, st)
        if ev:
            ev[3].record(st)

    def parity(self):
        """Per-alpha losses of the last step against the stored oracle losses of this layer."""
        import numpy as np

        gpath = os.path.join(ROOT, "tests", "golden", "oracle_losses.json")
        if not os.path.exists(gpath):
            return None
        g = json.load(open(gpath)).get(self.name)
        if not g or g["out_features"] != self.N:
            return None
        lo = np.array(g["losses"])
        lg = self.losses.cpu().numpy().astype(np.float64)
        b = int(self.best[0])
        return {"max_rel_loss_err": float(np.max(np.abs(lg - lo) / lo)), "gpu_best_idx": b,
                "oracle_best_idx": g["best_idx"], "oracle_loss_at_gpu_best_over_min": float(lo[b] / lo.min())}


def stage_kernels(R, flush, reps):
    """Each kernel awq_search_layer may run, launched alone through the stage calls, plus the statistics and
    pack calls: median CUDA-event ms per launch, L2 flushed before each. The short bandwidth- and
    latency-bound kernels go first, after two seconds of rest: right after a seconds-long search the GPU sits
    at its power limit, at about half its top SM clock, and these kernels issue at that clock; the step's own
    per-call times (``calls``) show them in that state."""
    import torch

    from post_bit_weight_awq_b300 import capi, capi_testing

    dev = R.W.device
    G, N, K, n = R.G, R.N, R.K, R.n
    s = torch.empty(G, K, dtype=torch.float32, device=dev)
    inv = torch.empty_like(s)
    op = torch.empty(G, N, K, dtype=torch.bfloat16, device=dev)
    mt, nt, _, _ = capi_testing.awq_search_tiles(n, N, R.cfg)
    parts = torch.zeros(G, mt, nt, 4, dtype=torch.float32, device=dev)  # loss_select may run before the products
    ready = torch.zeros(G * (nt + 1) + 1, dtype=torch.int32, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    losses = torch.empty(G, dtype=torch.float32, device=dev)
    best = torch.empty(1, dtype=torch.int32, device=dev)
    s_best = torch.empty(K, dtype=torch.float32, device=dev)
    capi_testing.awq_alpha_scales(R.mean_abs, R.cfg, s, inv)
    gcfg = capi.config(loss_form=capi.AWQ_LOSS_GRAM)
    xt_elems, h_elems, per_alpha = capi_testing.awq_gram_sizes(n, N, K)
    xt = torch.empty(xt_elems, dtype=torch.bfloat16, device=dev)
    H = torch.empty(h_elems, dtype=torch.bfloat16, device=dev)
    gparts = torch.empty(G, per_alpha, dtype=torch.float32, device=dev)
    capi_testing.awq_gram_matrix(R.X, xt, H, gcfg, status)
    calls = {
        # short kernels first, rested
        "stats": lambda: capi.awq_act_stats(R.X, R.mean_abs, R.ws),
        "alpha_scales": lambda: capi_testing.awq_alpha_scales(R.mean_abs, R.cfg, s, inv),
        "fakequant": lambda: capi_testing.awq_fakequant(R.W, s, inv, R.cfg, op),
        "pack": lambda: capi.awq_quantize_pack(R.W, R.s_best, R.cfg, R.qw, R.sc, R.zr),
        "gram_matrix": lambda: capi_testing.awq_gram_matrix(R.X, xt, H, gcfg, status),
        "loss_select": lambda: capi_testing.awq_loss_select(parts, s, R.cfg, losses, best, s_best, status, n_tok=n,
                                                            out_features=N, in_features=K),
        # then the products: the GRAM form's, then the direct form's two kernels for comparison
        "gram_loss": lambda: capi_testing.awq_gram_loss(op, H, gcfg, gparts, status),
        "search_gemm": lambda: capi_testing.awq_search_gemm(R.X, op, R.cfg, parts, status, n_tok=n, in_features=K,
                                                            out_features=N),
        "fused_search": lambda: capi_testing.awq_search_fused(R.W, R.X, s, inv, R.cfg, op, parts, ready, status),
    }
    out = {}
    torch.cuda.synchronize()
    time.sleep(2.0)
    for nm, fn in calls.items():
        fn()
        torch.cuda.synchronize()
        short = nm not in ("search_gemm", "fused_search", "gram_loss")
        # the short kernels: a few untimed launches bring the clock up from idle, then the median of many
        out[nm] = timed(fn, flush, max(reps, 15) if short else reps, warm=5 if short else 0)
    if int(status[0]) != 0:
        raise RuntimeError("device status " + capi.status_string(int(status[0])))
    del op, xt, H
    return out


def fractions(R, ms, pk):
    """Per-kernel achieved rates and fractions of the measured peaks."""
    hb = hbm_bytes(R.n, R.N, R.K, R.G, R.wbytes)
    d = {}
    for nm, t in ms.items():
        e = {"ms": round(t, 4)}
        if nm in hb:
            gbs = hb[nm] / (t * 1e-3) / 1e9
            e.update({"bytes": hb[nm], "gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 3)})
        if nm in ("fused_search", "search_gemm", "gram_loss", "gram_matrix"):
            f = {"gram_loss": 2.0 * R.G * R.N * gram_prefix_area(R.K), "gram_matrix": 2.0 * R.n * gram_prefix_area(R.K)}
            tf = f.get(nm, 2.0 * R.G * R.n * R.N * R.K) / (t * 1e-3) / 1e12
            e.update({"tflops": round(tf, 1), "frac_bf16_burst": round(tf / pk["bf16_tflops"], 3)})
            if pk.get("bf16_tflops_sustained"):
                e["frac_bf16_sustained"] = round(tf / pk["bf16_tflops_sustained"], 3)
        d[nm] = e
    return d


def search_path(R):
    """What awq_search_layer runs for this layer (the form AUTO resolved to, then the kernels)."""
    from post_bit_weight_awq_b300 import capi_testing

    if R.form == "gram":
        return "gram: X^T X, fake-quant launch, D H^T products over block prefixes"
    if R.flops < capi_testing.AWQ_SEARCH_FUSED_MAX_FLOPS:
        return f"{R.form}: fused fake-quant + CTA-pair products"
    return f"{R.form}: fake-quant launch + single-CTA products"


def side_workload(name, dev, flush, pk, reps):
    """Statistics, search and pack of each layer of a smaller workload through the public calls (eager, L2
    flushed before each step), with the search's fraction of the tensor peak and the oracle parity."""
    import torch

    import workloads
    from post_bit_weight_awq_b300 import capi, capi_testing

    out = []
    for layer in workloads.WORKLOADS[name]:
        R = LayerRun(layer, dev, capi.config())
        for _ in range(2):
            R.step()
        torch.cuda.synchronize()
        evs = []
        for _ in range(reps):
            flush.run()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            R.step(ev)
            evs.append(ev)
        torch.cuda.synchronize()
        assert capi.awq_get_device_status(R.ws) == capi.AWQ_OK
        st = [statistics.median(e[i].elapsed_time(e[i + 1]) for e in evs) for i in range(3)]
        hb = hbm_bytes(R.n, R.N, R.K, R.G, R.wbytes)
        tf = R.flops / (st[1] * 1e-3) / 1e12
        out.append({
            "layer": layer, "W": [R.N, R.K], "X": [R.n, R.K], "ms_per_layer": round(sum(st), 4),
            "stats_ms": round(st[0], 4), "stats_frac_hbm": round(hb["stats"] / (st[0] * 1e-3) / 1e9 / pk["hbm_gbs"], 3),
            "search_ms": round(st[1], 4), "search_tflops": round(tf, 1),
            "search_frac_bf16_burst": round(tf / pk["bf16_tflops"], 3),
            "search_path": search_path(R), "search_flops": R.flops,
            "pack_ms": round(st[2], 4), "pack_frac_hbm": round(hb["pack"] / (st[2] * 1e-3) / 1e9 / pk["hbm_gbs"], 3),
            "parity_vs_oracle": R.parity()})
        del R
        torch.cuda.empty_cache()
    return out


def decode_line(R, dev, flush, pk, reps):
    """awq_w4a16_gemv on the packed layer of the step, for one and for four tokens: enough copies of the layer
    to exceed L2, applied one after another (a decode step running through layers), L2 flushed before each
    pass."""
    import torch

    from post_bit_weight_awq_b300 import capi

    N, K = R.N, R.K
    layer_bytes = N * K // 2 + 2 * 2 * N * (K // 128)
    copies = max(3, int((256 << 20) // layer_bytes) + 1)
    packs = [(R.qw.clone(), R.sc.clone(), R.zr.clone()) for _ in range(copies)]
    out = {"layer": [N, K], "tokens": {},
           "timing": f"{copies} distinct copies per CUDA graph (> L2), L2 flushed before each graph"}
    for M in (1, 4):
        if M * K > capi.AWQ_W4A16_MAX_TOKEN_CHANNELS:
            continue
        xg = torch.randn(M, K, device=dev).to(torch.bfloat16)
        yg = torch.empty(M, N, dtype=torch.float32, device=dev)

        def one_pass():
            for q_, s_, z_ in packs:
                capi.awq_w4a16_gemv(xg, q_, s_, z_, R.cfg, yg)

        one_pass()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            one_pass()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        ms = timed(g.replay, flush, reps) / copies
        gbytes = layer_bytes + 2 * M * K + 4 * M * N
        # groups of 128: the tensor-core kernel for two or more tokens and for one token on 3 * 2^24 weights or more
        kernel = "w4a16_mma_kernel" if (M >= 2 or N * K >= 3 << 24) else f"w4a16_gemv_kernel<{M}, R>"
        out["tokens"][str(M)] = {"kernel": kernel, "ms_per_layer": round(ms, 5), "bytes_per_layer": gbytes,
                                 "gbs": round(gbytes / (ms * 1e-3) / 1e9, 1),
                                 "frac_hbm": round(gbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 3)}
        del g
    del packs
    return out if out["tokens"] else None


def prefill_line(R, dev, flush, pk, reps):
    """awq_w4a16_gemm on the packed layer of the step, 2048 prompt tokens (expansion + tensor-core product)."""
    import torch

    from post_bit_weight_awq_b300 import capi

    N, K = R.N, R.K
    Mp = 2048
    xp = torch.randn(Mp, K, device=dev).to(torch.bfloat16)
    yp = torch.empty(Mp, N, dtype=torch.float32, device=dev)
    gws = torch.empty(capi.awq_w4a16_gemm_workspace_size(Mp, K, N, R.cfg), dtype=torch.uint8, device=dev)

    def call():
        capi.awq_w4a16_gemm(xp, R.qw, R.sc, R.zr, R.cfg, yp, gws)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    ms = timed(call, flush, reps)
    assert capi.awq_get_device_status(gws) == capi.AWQ_OK
    pflops = 2.0 * Mp * N * K
    del gws, xp, yp
    return {"call": "awq_w4a16_gemm (bf16 expansion of the packed layer + tcgen05 CTA-pair product)", "tokens": Mp,
            "layer": [N, K], "ms": round(ms, 5), "tflops": round(pflops / (ms * 1e-3) / 1e12, 1),
            "frac_bf16_burst": round(pflops / (ms * 1e-3) / 1e12 / pk["bf16_tflops"], 3),
            "timing": "median of CUDA-event timed calls, L2 flushed before each"}


def gpu_arm(args, rank, world, local_rank):
    import torch

    import workloads
    from post_bit_weight_awq_b300 import build, capi, capi_testing, multi

    build.build()
    capi.lib()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    pk = peaks()
    name = workloads.WORKLOADS[args.workload][0]
    cfg = capi.config()
    R = LayerRun(name, dev, cfg, rows=args.rows)
    n, N, K, G = R.n, R.N, R.K, R.G
    flops = R.flops
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        flush.run()
        R.step()
    torch.cuda.synchronize()
    assert capi.awq_get_device_status(R.ws, stream) == capi.AWQ_OK

    # the whole step as one CUDA graph (no host launch gaps between kernels)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        R.step()
    for _ in range(args.warmup):
        flush.run()
        graph.replay()
    torch.cuda.synchronize()
    # the replayed graph must reproduce the eager step's results
    losses_eager = R.losses.clone()
    R.losses.zero_()
    graph.replay()
    torch.cuda.synchronize()
    if not torch.equal(R.losses, losses_eager):
        raise RuntimeError("graph replay does not reproduce the eager step")

    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    for k in range(args.steps):
        flush.run()
        torch.cuda._sleep(RUN_AHEAD_CYCLES)
        gev[k][0].record(stream)
        graph.replay()
        gev[k][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    assert capi.awq_get_device_status(R.ws, stream) == capi.AWQ_OK
    step_ms = [a.elapsed_time(b) for a, b in gev]
    ms_step = statistics.mean(step_ms)
    t_total = sum(step_ms)
    if dist:
        t_total = multi.max_over_ranks(t_total, device=dev)
    value = t_total / (args.steps * world)
    parity = R.parity()

    # the three public calls of the step, timed one by one (eager, events between the calls)
    evs = []
    for _ in range(args.steps):
        flush.run()
        torch.cuda._sleep(RUN_AHEAD_CYCLES)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        R.step(ev)
        evs.append(ev)
    torch.cuda.synchronize()
    calls_ms = {nm: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs)
                for i, nm in enumerate(("awq_act_stats", "awq_search_layer", "awq_quantize_pack"))}

    # each kernel alone (stage calls), for the per-kernel rooflines
    kern = fractions(R, stage_kernels(R, flush, max(3, args.steps // 4)), pk)
    fused_path = R.form != "gram" and flops < capi_testing.AWQ_SEARCH_FUSED_MAX_FLOPS
    search_kernel = "gram_loss" if R.form == "gram" else ("fused_search" if fused_path else "search_gemm")
    traffic_tag = "gram" if R.form == "gram" else ("fused" if fused_path else "single")
    search_ms = kern[search_kernel]["ms"]
    kernel_flops = R.loss_flops
    achieved = kernel_flops / (search_ms * 1e-3) / 1e12
    form, path = R.form, search_path(R)
    long_step = ms_step > 100.0  # a timed region of seconds settles at the power cap
    sustained = pk.get("bf16_tflops_sustained")
    peak, peak_kind = (sustained, "sustained") if (long_step and sustained) else (pk["bf16_tflops"], "burst")

    L = R.L
    e2e, gemv, gemm, side = None, None, None, None
    if not args.no_extras:
        e2e = end_to_end(R, args, cfg, dev, flush, stream, world, dist)
        gemv = decode_line(R, dev, flush, pk, max(3, args.steps // 2))
        gemm = prefill_line(R, dev, flush, pk, max(3, args.steps // 2))
    del R, graph
    torch.cuda.empty_cache()
    if not args.no_side and world == 1:
        side = {w: side_workload(w, dev, flush, pk, 5) for w in SIDE_WORKLOADS}

    if dist:
        dist.destroy_process_group()
    if rank != 0:
        return

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        ts, tr, scale = oracle_sample(L, args.oracle_rows)
        cpu = {"value": round((ts + tr * scale) * 1e3, 1), "unit": "ms", "cores": blas_threads(), "kind": "oracle",
               "sample": f"oracle statistics over all {n} tokens ({ts:.1f} s) + search and pack of output rows "
                         f"[0,{args.oracle_rows}) ({tr:.1f} s), the rows scaled by out/rows = {scale:g} to one layer"}

    kernel_names = {"fused_search": "search_gemm_pair_kernel<fused> (quantiser warps + tcgen05 pair products)",
                    "search_gemm": "search_gemm_kernel (tcgen05 single-CTA products; fake-quant launched before it)",
                    "gram_loss": "gram_kernel<LOSS> (tcgen05 single-CTA D_i H^T tiles over channel-block prefixes, lockstep "
                                 "column-block pair items; fake-quant and X^T X launched before it)"}
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "layer": name, "W": [N, K], "X": [n, K], "w_dtype": L["w_dtype"],
                   "n_grid": G, "group": 128, "loss_form": f"auto -> {form}", "search_path": path,
                   "search_flops": flops, "parallelism": f"replicas{world}",
                   "calls": "awq_act_stats + awq_search_layer + awq_quantize_pack",
                   "launch": "the three calls captured as one CUDA graph and replayed",
                   "l2": "inputs larger than L2, and L2 flushed between steps outside the timed events (a 512 MiB "
                         "write, then a 512 MiB read so that no dirty flush lines are left for the timed kernels)"},
        "roofline": {"bound": "tensor", "kernel": kernel_names[search_kernel], "achieved": round(achieved, 1),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 3),
                     "traffic": profiled_traffic(traffic_tag, args.workload),
                     "peak_source": f"{pk['source']} bf16 {peak_kind}", "algorithmic_flops_per_launch": kernel_flops,
                     "direct_form_flops": 2.0 * G * n * N * K,
                     "note": ("GRAM form: the same per-alpha loss as sum_r D[r] (X^T X) D[r]^T; the launch's flops are "
                              "2 n_grid out S (S = entries of X^T X on and below the 256-channel block diagonal), "
                              "not the direct form's 2 n_grid n_tok out in" if form == "gram" else None),
                     "launch_ms": search_ms},
        "calls": {k: round(v, 4) for k, v in calls_ms.items()},
        "kernels": kern,
        "e2e": e2e,
        # stats, alpha scales, [fake-quant,] search product, loss reduce, select, pack; the GRAM form adds
        # the transpose and X^T X
        "gpu_launches": (9 if form == "gram" else (6 if fused_path else 7)) * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 4),
        "parity_vs_oracle": parity,
        "w4a16_gemv": gemv,
        "w4a16_gemm_prefill": gemm,
        "other_workloads": side,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def end_to_end(R, args, cfg, dev, flush, stream, world, dist):
    """The public layer pipeline (awq_quantize_layers): K layers whose W and X sit in pinned host memory, each
    copied in, searched, packed and copied out; the copies of one layer overlap the search of the next."""
    import numpy as np
    import torch

    import workloads
    from post_bit_weight_awq_b300 import capi, multi

    L = R.L
    n, N, K, G = R.n, R.N, R.K, R.G
    pin = dict(pin_memory=True)
    Wh = (torch.from_numpy(workloads.bf16_bits(L["W"]).view(np.int16)).view(torch.bfloat16) if L["w_dtype"] == "bf16"
          else torch.from_numpy(L["W"])).pin_memory()
    Xh = torch.from_numpy(workloads.bf16_bits(L["X"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    outs_h = {"qweight": torch.empty(N, K // 8, dtype=torch.int32, **pin),
              "scales": torch.empty(N, K // 128, dtype=torch.float16, **pin),
              "zeros": torch.empty(N, K // 128, dtype=torch.float16, **pin),
              "losses": torch.empty(G, dtype=torch.float32, **pin),
              "best_idx": torch.empty(1, dtype=torch.int32, **pin),
              "s_best": torch.empty(K, dtype=torch.float32, **pin)}
    wcode = capi.AWQ_BF16 if L["w_dtype"] == "bf16" else capi.AWQ_FP32
    pipe_ws = torch.empty(capi.awq_pipeline_workspace_size(n, N, K, wcode, cfg), dtype=torch.uint8, device=dev)
    h2d = Wh.numel() * Wh.element_size() + Xh.numel() * Xh.element_size()
    d2h = sum(t.numel() * t.element_size() for t in outs_h.values())
    io = capi.layer_io(Wh, Xh, outs_h["qweight"], outs_h["scales"], outs_h["zeros"], outs_h["losses"],
                       outs_h["best_idx"], outs_h["s_best"])
    capi.awq_quantize_layers([io] * 3, wcode, cfg, pipe_ws, stream)
    torch.cuda.synchronize()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush.run()
    ea.record(stream)
    capi.awq_quantize_layers([io] * args.steps, wcode, cfg, pipe_ws, stream)
    eb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = ea.elapsed_time(eb) / args.steps
    if dist:
        e2e_ms = multi.max_over_ranks(e2e_ms, device=dev) / world
    assert capi.awq_get_device_status(pipe_ws, stream) == capi.AWQ_OK
    assert int(outs_h["best_idx"][0]) == int(R.best[0])  # the streamed layer chose what the device path chose
    assert torch.equal(outs_h["qweight"], R.qw.cpu())  # and packed the same codes
    del pipe_ws, Wh, Xh
    return {"value": round(e2e_ms, 4), "unit": "ms", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "awq_quantize_layers: steps layers in one call, each layer's W and X copied in from pinned host "
                   "memory and its packed outputs, losses and s_best copied out, copies overlapping the previous "
                   "layer's search (no L2 flush inside the call)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--oracle-rows", type=int, default=512, help="output rows of the cpu_baseline sample (about 10 s)")
    ap.add_argument("--reference-rows", type=int, default=64, help="output rows per step of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side", action="store_true", help="skip the entries of the other workloads")
    ap.add_argument("--no-extras", action="store_true", help="skip the end-to-end, decode and prefill timings")
    ap.add_argument("--rows", type=int, default=None,
                    help="output rows of the layer (default: the workload's); a smaller case for profiler captures")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        reference_arm(args, rank)
        return
    gpu_arm(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
