"""Benchmark: AWQ per-layer search + INT4 pack on B300, one JSON line.

A step is one pass of the whole path over one synthetic layer, through the C
ABI: activation statistics, the 20-point alpha search (scales, fake-quant,
tcgen05 search product with fused squared-error epilogue, loss + argmin) and
the final pack. Inputs are resident in HBM when the timed region starts; L2
is flushed (a 512 MiB write) between steps, outside the timed events.

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
DEFAULT_WORKLOAD = "llama7b_q_proj"
KERNELS_PER_STEP = 6  # stats, alpha scales, fused fake-quant + search product, loss reduce + select, pack
RUN_AHEAD_CYCLES = 4_000_000  # GPU spin before each timed step so the host enqueues the whole step first
FLUSH_BYTES = 512 << 20


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


def profiled_traffic(workload):
    """DRAM bytes per launch of the fused search kernel from the committed ncu
    summary of this workload, if it was taken on the current kernel source;
    else None."""
    path = os.path.join(ROOT, "profiles", f"search_fused_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch\s*=\s*(\d+).*?workload\s*=\s*(\w+).*?source_sha256_16\s*=\s*(\w+)",
                  text, flags=re.S)
    if not m:
        return None
    if m.group(2) != workload or m.group(3) != source_digest(GEMM_SOURCES):
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
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows if r[3].replace(".", "").isdigit()), default=None)}


# ------------------------------------------------------------------ oracle arm


def oracle_layer(workload):
    import workloads

    return workloads.make_layer(workloads.WORKLOADS[workload][0])


def oracle_sample(L, rows):
    """Run the oracle's statistics, search and pack on the first ``rows``
    output rows of layer ``L`` (all tokens, all input channels). Returns the
    seconds taken and the factor that scales the sample to the whole layer."""
    import numpy as np

    import oracle as O

    W = L["W"][:rows].astype(np.float64)
    X = L["X"].astype(np.float64)
    N = L["W"].shape[0]
    t0 = time.perf_counter()
    sx = O.channel_importance(X)
    res = O.search_scale(W, X, sx)
    O.quantize_pack(W, O.f32(res["s_best"]))
    dt = time.perf_counter() - t0
    return dt, N / rows


def blas_threads():
    try:
        from threadpoolctl import threadpool_info

        return max((p.get("num_threads", 1) for p in threadpool_info()), default=1)
    except Exception:
        return len(os.sched_getaffinity(0))


def reference_arm(args, rank):
    if rank != 0:
        return
    rows = args.oracle_rows
    L = oracle_layer(args.workload)
    for _ in range(args.warmup):
        oracle_sample(L, rows)
    times = []
    scale = 1.0
    for _ in range(args.steps):
        dt, scale = oracle_sample(L, rows)
        times.append(dt * scale * 1e3)
    ms = statistics.mean(times)
    cores = blas_threads()
    sample = (f"oracle statistics+search+pack on output rows [0,{rows}) of the layer (all tokens), "
              f"time scaled by out/rows = {scale:g} to one layer")
    line = {"impl": "reference", "metric": METRIC, "value": ms, "unit": "ms", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "n_grid": 20, "group": 128},
            "cpu_baseline": {"value": ms, "unit": "ms", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": ms, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm


def gpu_arm(args, rank, world, local_rank):
    import numpy as np
    import torch

    import workloads
    from post_bit_weight_awq_b300 import build, capi, multi

    build.build()
    capi.lib()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    name = workloads.WORKLOADS[args.workload][0]
    L = workloads.make_layer(name)
    W32, X32 = L["W"], L["X"]
    N, K = W32.shape
    n = X32.shape[0]
    cfg = capi.config()
    G = cfg.n_grid

    def to_dev_bf16(a):
        return torch.from_numpy(workloads.bf16_bits(a).view(np.int16)).to(dev).view(torch.bfloat16)

    Wd = to_dev_bf16(W32) if L["w_dtype"] == "bf16" else torch.from_numpy(W32).to(dev)
    Xd = to_dev_bf16(X32)
    f32, i32, u8 = torch.float32, torch.int32, torch.uint8
    mean_abs = torch.empty(K, dtype=f32, device=dev)
    stats_ws = torch.empty(capi.awq_act_stats_workspace_size(n, K), dtype=u8, device=dev)
    s = torch.empty(G, K, dtype=f32, device=dev)
    inv = torch.empty_like(s)
    op = torch.empty(G, N, K, dtype=torch.bfloat16, device=dev)
    mt, nt, _, _ = capi.awq_search_tiles(n, N, cfg)
    parts = torch.empty(G, mt, nt, 4, dtype=f32, device=dev)
    ready = torch.zeros(G * (nt + 1) + 1, dtype=i32, device=dev)
    status = torch.zeros(4, dtype=i32, device=dev)
    losses = torch.empty(G, dtype=f32, device=dev)
    best = torch.empty(1, dtype=i32, device=dev)
    s_best = torch.empty(K, dtype=f32, device=dev)
    qw = torch.empty(N, K // 8, dtype=i32, device=dev)
    sc = torch.empty(N, K // 128, dtype=torch.float16, device=dev)
    zr = torch.empty(N, K // 128, dtype=torch.float16, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=u8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        # the same kernels, in the same order, as awq_act_stats + awq_search_layer + awq_quantize_pack;
        # launched on the current stream (the capture stream while a CUDA graph is recorded)
        st = torch.cuda.current_stream(dev)
        if ev:
            ev[0].record(st)
        capi.awq_act_stats(Xd, mean_abs, stats_ws, st)
        if ev:
            ev[1].record(st)
        capi.awq_alpha_scales(mean_abs, cfg, s, inv, st)
        if ev:
            ev[2].record(st)
        capi.awq_search_fused(Wd, Xd, s, inv, cfg, op, parts, ready, status, st)
        if ev:
            ev[3].record(st)
        capi.awq_loss_select(parts, s, cfg, losses, best, s_best, status, st, n_tok=n, out_features=N,
                             in_features=K)
        if ev:
            ev[4].record(st)
        capi.awq_quantize_pack(Wd, s_best, cfg, qw, sc, zr, st)
        if ev:
            ev[5].record(st)

    def unfused(ev):
        # the fake-quant and the search product as separate launches (what the fused kernel overlaps)
        st = torch.cuda.current_stream(dev)
        ev[0].record(st)
        capi.awq_fakequant(Wd, s, inv, cfg, op, st)
        ev[1].record(st)
        capi.awq_search_gemm(Xd, op, cfg, parts, status, st, n_tok=n, in_features=K, out_features=N)
        ev[2].record(st)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert int(status[0]) == 0, capi.status_string(int(status[0]))

    # the whole step as one CUDA graph (no host launch gaps between kernels)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(args.warmup):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize()
    # the replayed graph must reproduce the eager step's results
    losses_eager = losses.clone()
    losses.zero_()
    graph.replay()
    torch.cuda.synchronize()
    if not torch.equal(losses, losses_eager):
        raise RuntimeError("graph replay does not reproduce the eager step")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    uevents = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    for k in range(args.steps):
        flush.zero_()
        torch.cuda._sleep(RUN_AHEAD_CYCLES)
        gev[k][0].record(stream)
        graph.replay()
        gev[k][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    # per-stage device times: the same step launched eagerly, host run ahead of the GPU
    for k in range(args.steps):
        flush.zero_()
        torch.cuda._sleep(RUN_AHEAD_CYCLES)
        step(events[k])
    torch.cuda.synchronize()
    if int(status[0]) != 0:
        raise RuntimeError("device status " + capi.status_string(int(status[0])))
    for k in range(args.steps):
        flush.zero_()
        torch.cuda._sleep(RUN_AHEAD_CYCLES)
        unfused(uevents[k])
    torch.cuda.synchronize()
    if int(status[0]) != 0:
        raise RuntimeError("device status " + capi.status_string(int(status[0])))

    stage_names = ["stats", "alpha_scales", "search", "loss_select", "pack"]
    per_stage = {nm: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in events) for i, nm in enumerate(stage_names)}
    alone = {"fakequant": statistics.mean(e[0].elapsed_time(e[1]) for e in uevents),
             "search_gemm": statistics.mean(e[1].elapsed_time(e[2]) for e in uevents)}
    step_ms = [a.elapsed_time(b) for a, b in gev]
    ms_step = statistics.mean(step_ms)
    ms_step_eager = statistics.mean(e[0].elapsed_time(e[5]) for e in events)
    t_total = sum(step_ms)
    if dist:
        t_total = multi.max_over_ranks(t_total, device=dev)
    layers = args.steps * world
    value = t_total / layers

    # ---------------------------------------------------------- end to end (host buffers)
    # the public layer pipeline (awq_quantize_layers): K layers whose W and X sit in pinned host memory, each
    # copied in, searched, packed and copied out; the copies of one layer overlap the search of the next
    pin = dict(pin_memory=True)
    Wh = (torch.from_numpy(workloads.bf16_bits(W32).view(np.int16)).view(torch.bfloat16) if L["w_dtype"] == "bf16"
          else torch.from_numpy(W32)).clone().pin_memory()
    Xh = torch.from_numpy(workloads.bf16_bits(X32).view(np.int16)).view(torch.bfloat16).clone().pin_memory()
    outs_h = {"qweight": torch.empty(N, K // 8, dtype=i32, **pin), "scales": torch.empty(N, K // 128,
                                                                                      dtype=torch.float16, **pin),
              "zeros": torch.empty(N, K // 128, dtype=torch.float16, **pin), "losses": torch.empty(G, dtype=f32, **pin),
              "best_idx": torch.empty(1, dtype=i32, **pin), "s_best": torch.empty(K, dtype=f32, **pin)}
    del op
    wcode = capi.AWQ_BF16 if L["w_dtype"] == "bf16" else capi.AWQ_FP32
    pipe_ws = torch.empty(capi.awq_pipeline_workspace_size(n, N, K, wcode, cfg), dtype=u8, device=dev)
    h2d = Wh.numel() * Wh.element_size() + Xh.numel() * Xh.element_size()
    d2h = sum(t.numel() * t.element_size() for t in outs_h.values())
    io = capi.layer_io(Wh, Xh, outs_h["qweight"], outs_h["scales"], outs_h["zeros"], outs_h["losses"],
                       outs_h["best_idx"], outs_h["s_best"])
    capi.awq_quantize_layers([io] * max(3, args.warmup), wcode, cfg, pipe_ws, stream)
    torch.cuda.synchronize()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush.zero_()
    ea.record(stream)
    capi.awq_quantize_layers([io] * args.steps, wcode, cfg, pipe_ws, stream)
    eb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = ea.elapsed_time(eb) / args.steps
    if dist:
        e2e_ms = multi.max_over_ranks(e2e_ms, device=dev) / world
    assert capi.awq_get_device_status(pipe_ws, stream) == capi.AWQ_OK
    assert int(outs_h["best_idx"][0]) == int(best[0])  # the streamed layer chose what the device path chose
    del pipe_ws

    # ---------------------------------------------------------- the packed layer in use (w4a16 decode product)
    # copies of the packed layer, more bytes than L2, applied one after another to one token (a decode step
    # running through layers): HBM bandwidth of awq_w4a16_gemv
    gemv = None
    if K * 4 <= 50 * 1024:
        layer_bytes = N * K // 2 + 2 * 2 * N * (K // 128)
        copies = max(4, int((256 << 20) // layer_bytes) + 1)
        packs = [(qw.clone(), sc.clone(), zr.clone()) for _ in range(copies)]
        xg = torch.randn(1, K, device=dev).to(torch.bfloat16)
        yg = torch.empty(1, N, dtype=f32, device=dev)
        gcfg = capi.config()

        def gemv_pass():
            st = torch.cuda.current_stream(dev)
            for q_, s_, z_ in packs:
                capi.awq_w4a16_gemv(xg, q_, s_, z_, gcfg, yg, st)

        gemv_pass()
        gg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gg):
            gemv_pass()
        for _ in range(3):
            gg.replay()
        torch.cuda.synchronize()
        gt = []
        for _ in range(max(3, args.steps // 2)):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            gg.replay()
            b.record(stream)
            torch.cuda.synchronize()
            gt.append(a.elapsed_time(b) / copies)
        ms_g = statistics.median(gt)
        gbytes = layer_bytes + K * 2 + N * 4
        gemv = {"kernel": "w4a16_gemv_kernel<1, R> (R rows per warp, chosen by the launcher)", "tokens": 1, "layer": [N, K], "ms_per_layer": round(ms_g, 5),
                "bytes_per_layer": gbytes, "gbs": round(gbytes / (ms_g * 1e-3) / 1e9, 1),
                "frac_hbm": round(gbytes / (ms_g * 1e-3) / 1e9 / peaks()["hbm_gbs"], 3),
                "timing": f"{copies} distinct copies per CUDA graph (> L2), L2 flushed before each graph"}
        del packs

    # ---------------------------------------------------------- the packed layer in a prefill (2048 prompt tokens)
    # expand to bf16 in the workspace, then the tensor-core product (awq_w4a16_gemm); L2 flushed before each run
    gemm = None
    Mp = 2048
    xp = torch.randn(Mp, K, device=dev).to(torch.bfloat16)
    yp = torch.empty(Mp, N, dtype=f32, device=dev)
    gws = torch.empty(capi.awq_w4a16_gemm_workspace_size(Mp, K, N, cfg), dtype=u8, device=dev)
    for _ in range(3):
        capi.awq_w4a16_gemm(xp, qw, sc, zr, cfg, yp, gws, stream)
    torch.cuda.synchronize()
    pt = []
    for _ in range(max(3, args.steps // 2)):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        capi.awq_w4a16_gemm(xp, qw, sc, zr, cfg, yp, gws, stream)
        b.record(stream)
        torch.cuda.synchronize()
        pt.append(a.elapsed_time(b))
    assert capi.awq_get_device_status(gws, stream) == capi.AWQ_OK
    ms_p = statistics.median(pt)
    pflops = 2.0 * Mp * N * K
    gemm = {"call": "awq_w4a16_gemm (bf16 expansion of the packed layer + tcgen05 CTA-pair product)", "tokens": Mp,
            "layer": [N, K], "ms": round(ms_p, 5), "tflops": round(pflops / (ms_p * 1e-3) / 1e12, 1),
            "frac_bf16_burst": round(pflops / (ms_p * 1e-3) / 1e12 / peaks()["bf16_tflops"], 3),
            "timing": "median of CUDA-event timed calls, L2 flushed before each"}
    del gws, xp, yp

    # ---------------------------------------------------------- bandwidth kernels on the largest layer
    # the statistics, fake-quant and pack kernels move 33-700 MB on the benchmark layer, a few microseconds of
    # work beside a few microseconds of launch and ramp; on the 70B-class MLP layer they move 0.27-9.9 GB
    large = None if args.no_large else large_layer_rates(dev, flush, peaks()["hbm_gbs"])

    # ---------------------------------------------------------- parity spot check vs stored oracle losses
    parity = None
    gpath = os.path.join(ROOT, "tests", "golden", "oracle_losses.json")
    if os.path.exists(gpath):
        g = json.load(open(gpath)).get(name)
        if g:
            lo = np.array(g["losses"])
            lg = outs_h["losses"].numpy().astype(np.float64)
            parity = {"max_rel_loss_err": float(np.max(np.abs(lg - lo) / lo)),
                      "gpu_best_idx": int(outs_h["best_idx"][0]), "oracle_best_idx": g["best_idx"],
                      "oracle_loss_at_gpu_best_over_min": float(lo[int(outs_h["best_idx"][0])] / lo.min())}

    if dist:
        dist.destroy_process_group()
    if rank != 0:
        return

    pk = peaks()
    flops = G * 2.0 * n * K * N
    search_ms = per_stage["search"]
    achieved = flops / (search_ms * 1e-3) / 1e12
    traffic = profiled_traffic(args.workload)
    wbytes = 2 if L["w_dtype"] == "bf16" else 4
    hbm_bytes = {
        "stats": 2.0 * n * K,
        "fakequant": wbytes * N * K + G * 2.0 * N * K,
        "pack": wbytes * N * K + N * K / 2 + 4.0 * N * K / 128,
    }

    def tensor_fracs(tf):
        d = {"tflops": round(tf, 1), "frac_bf16_burst": round(tf / pk["bf16_tflops"], 3)}
        if pk.get("bf16_tflops_sustained"):
            d["frac_bf16_sustained"] = round(tf / pk["bf16_tflops_sustained"], 3)
        return d

    def hbm_fracs(nm, ms):
        gbs = hbm_bytes[nm] / (ms * 1e-3) / 1e9
        return {"gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 3)}

    stages = {}
    for nm, ms in per_stage.items():
        d = {"ms": round(ms, 4)}
        if nm in hbm_bytes:
            d.update(hbm_fracs(nm, ms))
        if nm == "search":
            d["kernel"] = "search_gemm_pair_kernel<fused> (fake-quant warps + tcgen05 pair products)"
            d.update(tensor_fracs(achieved))
        stages[nm] = d
    # the two halves of the fused stage launched separately, for the per-kernel rooflines
    separate = {"fakequant": {"ms": round(alone["fakequant"], 4), **hbm_fracs("fakequant", alone["fakequant"])},
                "search_gemm": {"ms": round(alone["search_gemm"], 4),
                                **tensor_fracs(flops / (alone["search_gemm"] * 1e-3) / 1e12)}}

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        dt, scale = oracle_sample(L, args.oracle_rows)
        cpu = {"value": dt * scale * 1e3, "unit": "ms", "cores": blas_threads(), "kind": "oracle",
               "sample": f"oracle search+pack on output rows [0,{args.oracle_rows}) of the layer (all tokens), "
                         f"{dt:.1f} s, scaled by out/rows = {scale:g} to one layer"}

    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "layer": name, "W": [N, K], "X": [n, K], "w_dtype": L["w_dtype"],
                   "n_grid": G, "group": 128, "loss_form": "residual", "parallelism": f"replicas{world}",
                   "launch": "whole step replayed as one CUDA graph",
                   "l2": "flushed between steps (512 MiB write outside the timed events)"},
        "ms_per_step_eager": round(ms_step_eager, 4),
        "roofline": {"bound": "tensor", "kernel": "search_gemm_pair_kernel<fused>", "achieved": round(achieved, 1),
                     "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": round(achieved / pk["bf16_tflops"], 3),
                     "traffic": traffic, "peak_source": f"{pk['source']} bf16 burst",
                     "algorithmic_flops_per_launch": flops},
        "stages": stages,
        "stages_unfused": separate,
        "w4a16_gemv": gemv,
        "w4a16_gemm_prefill": gemm,
        "bandwidth_kernels_70b_layer": large,
        "e2e": {"value": round(e2e_ms, 4), "unit": "ms", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "awq_quantize_layers: steps layers in one call, each layer's W and X copied in from pinned "
                       "host memory and its packed outputs, losses and s_best copied out, copies overlapping the "
                       "previous layer's search (no L2 flush inside the call)"},
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 4),
        "parity_vs_oracle": parity,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def large_layer_rates(dev, flush, hbm_gbs):
    """Time the statistics, fake-quant and pack kernels alone on the 70B-class MLP shape (W 28672 x 8192
    bf16, X 16384 x 8192 bf16, 20 alphas; random data, timing only), L2 flushed before each launch."""
    import torch

    from post_bit_weight_awq_b300 import capi

    n, N, K = 16384, 28672, 8192
    cfg = capi.config()
    G = cfg.n_grid
    X = torch.randn(n, K, device=dev).to(torch.bfloat16)
    W = (torch.randn(N, K, device=dev) * 0.01).to(torch.bfloat16)
    mean = torch.empty(K, dtype=torch.float32, device=dev)
    sws = torch.empty(capi.awq_act_stats_workspace_size(n, K), dtype=torch.uint8, device=dev)
    s = torch.empty(G, K, dtype=torch.float32, device=dev)
    inv = torch.empty_like(s)
    op = torch.empty(G, N, K, dtype=torch.bfloat16, device=dev)
    qw = torch.empty(N, K // 8, dtype=torch.int32, device=dev)
    sc = torch.empty(N, K // 128, dtype=torch.float16, device=dev)
    zr = torch.empty(N, K // 128, dtype=torch.float16, device=dev)
    capi.awq_act_stats(X, mean, sws)
    capi.awq_alpha_scales(mean, cfg, s, inv)
    calls = {
        "stats": (lambda: capi.awq_act_stats(X, mean, sws), 2.0 * n * K),
        "fakequant": (lambda: capi.awq_fakequant(W, s, inv, cfg, op), 2.0 * N * K + G * 2.0 * N * K),
        "pack": (lambda: capi.awq_quantize_pack(W, s[7], cfg, qw, sc, zr), 2.0 * N * K + N * K / 2 + 4.0 * N * K / 128),
    }
    out = {"layer": {"W": [N, K], "X": [n, K], "n_grid": G}, "data": "random, timing only"}
    for name, (fn, nbytes) in calls.items():
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(5):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ms = statistics.median(ts)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": round(ms, 4), "bytes": nbytes, "gbs": round(gbs, 1), "frac_hbm": round(gbs / hbm_gbs, 3)}
    del op, X, W
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--oracle-rows", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-large", action="store_true", help="skip the 70B-class bandwidth-kernel timings")
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
