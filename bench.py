"""Benchmark: concurrent decode attention (Hogwild! Inference) on GB300.

One step = one decode token for every worker through the whole layer stack:
64 sequential hw_attn_decode calls (one per layer, each layer with its own K/V
pools) on the 32B-shaped 4-worker 16K-context workload.  The metric is KV HBM
GB/s (algorithmic bytes: every K and V row of the step read once, shared by all
workers and query heads) and worker-tokens/s per layer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  --impl reference times the float64 CPU oracle on the
same workload (a bounded sample of layers per step) on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "concurrent decode attention: KV HBM GB/s vs 8 TB/s peak; worker-tokens/s per layer"
NOMINAL_HBM_GBS = 8000.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--config", default="C3", choices=["C2", "C3", "C4", "C5", "W8"],
                   help="W8: the C3 shape with eight workers (40 query columns a block)")
    p.add_argument("--eager", action="store_true", help="time eager launches instead of a CUDA graph")
    p.add_argument("--layout", default="combined", choices=["combined", "interleaved", "contiguous"],
                   help="views of the cache layout (the combined layout is the method's own)")
    p.add_argument("--append", action="store_true",
                   help="each layer first writes every worker's new token (the last position of "
                        "its block) and then decodes, in one hw_attn_append_decode_planned launch")
    p.add_argument("--chunk", type=int, default=0,
                   help="T > 0: T query tokens per worker, each seeing its own block up to its own "
                        "token (hw_views_chunked + hw_attn_plan_limited)")
    p.add_argument("--kv", default="bf16", choices=["bf16", "fp8"],
                   help="fp8: the K/V pools as E4M3 codes with per-kv-head scales "
                        "(hw_attn_decode_planned_fp8)")
    p.add_argument("--commit-all", action="store_true",
                   help="C4: every worker's finished block joins the history each step, all in "
                        "one hw_block_commit_many launch (the common block gets room for them)")
    p.add_argument("--unplanned", action="store_true",
                   help="one hw_attn_decode per layer instead of hw_attn_plan once per step "
                        "plus hw_attn_decode_planned per layer")
    p.add_argument("--no-early", action="store_true",
                   help="never pass the early-loads promise (HW_DESC_EARLY_LOADS)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    p.add_argument("--layers", type=int, default=0,
                   help="time only the first N layers (profiling of a small case); 0 = all")
    return p.parse_args()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


class ClockSampler:
    """nvidia-smi samples during the timed region (SM clock, throttle reasons)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_traffic(kernel: str, workload_key: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's sources changed since the counters were taken (or none exist)."""
    import hashlib
    root = os.path.dirname(os.path.abspath(__file__))
    path = os.path.join(root, "profiles", f"{kernel}_{workload_key}_traffic.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if line.startswith("#") or ":" not in line:
            continue
        k, v = line.split(":", 1)
        kv[k.strip()] = v.strip()
    h = hashlib.sha256()
    try:
        for src in kv["sources"].split():
            h.update(open(os.path.join(root, src), "rb").read())
    except (KeyError, OSError):
        return None
    if h.hexdigest()[:16] != kv.get("sources_sha256_16"):
        return None
    return int(kv["dram_bytes_per_launch"])


def workload_config(w, config: str, layout: str = "combined", layers=None) -> dict:
    """The keys that name the timed workload, the same in both arms' lines."""
    if layers is None:
        layers = w.layers if config != "C5" else 64  # C5: one layer timed x64
    return {"workload": w.name, "layers_per_step": layers,
            "problems": w.n_problems, "workers": w.n_workers, "q_heads": w.n_q_heads,
            "kv_heads": w.n_kv_heads, "head_dim": w.head_dim,
            "kv_tokens_per_layer": w.kv_tokens(), "layout": layout}


def max_over_ranks(t: float, device) -> float:
    """The slowest rank's time (every rank gets it): replicas run the same
    work, so the job takes as long as its slowest one.  Identity without a
    process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return t
    tt = torch.tensor([t], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def replica_value(units_per_rank: float, t_max: float, world: int) -> float:
    """Whole-job throughput of `world` replicas: all ranks' units over the
    slowest rank's time."""
    return units_per_rank * world / t_max


def reference_arm(args):
    """The float64 oracle on the host cores, on the same workload and metric:
    each step runs the oracle over every layer of the step (the 16-problem
    serving shape: 2 of its 16 problems of its one timed layer, scaled), and
    ms_per_step is the time the steps actually took.  Nothing here loads the
    CUDA library: the views come from the oracle's own builder."""
    import oracle
    from concurrent_shared_kv_gb300 import workloads as wl

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = {**wl.ALL, **wl.EXTRA}[args.config]()
    o = oracle.get()
    lens, starts = w.block_lengths(), w.block_starts()
    vb, vo, qp = oracle.combined_views(lens, w.n_problems, w.n_workers)
    cores = len(os.sched_getaffinity(0))
    serving = args.config == "C5"
    rows = None if not serving else list(range(0, 4)) + list(range(60, 64))
    frac_rows = 1.0 if rows is None else len(rows) / w.n_rows
    layers = w.layers if not serving else 1
    if args.layers > 0:
        layers = min(layers, args.layers)
    # four distinct layers cycled through the step's calls (64 layers of host
    # inputs would take gigabytes; the oracle's time does not depend on the values)
    inputs = [wl.draw_host(w, l) for l in range(min(layers, 4))]
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        for l in range(layers):
            q, k, v = inputs[l % len(inputs)]
            o.attn_decode(q=q, k_cache=k, v_cache=v, block_start=starts, block_len=lens,
                          view_block=vb, view_offset=vo, q_pos=qp, n_kv_heads=w.n_kv_heads,
                          rope_theta=w.rope_theta, scale=w.scale,
                          dtype=oracle.F32 if w.dtype == "f32" else oracle.BF16, rows=rows,
                          n_threads=cores)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    t_step = statistics.median(times)
    done_bytes = w.kv_bytes_per_layer() * layers * frac_rows
    gbs = done_bytes / t_step / 1e9
    t_layer = t_step / layers / frac_rows
    sample = (f"{layers} layer calls per step (4 distinct layers' inputs cycled), all rows and heads, "
              f"float64 oracle, {cores} threads"
              if rows is None else
              f"problems 0 and 15 of the one timed layer per step (2 of 16), float64 oracle, "
              f"{cores} threads; GB/s of the KV those rows read")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_step * 1e3,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.config, layers=layers),
        "worker_tokens_per_s_per_layer": w.n_rows / t_layer,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
        return
    import numpy as np
    import torch
    import torch.distributed as dist

    from concurrent_shared_kv_gb300 import api, engine
    from concurrent_shared_kv_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    w = {**wl.ALL, **wl.EXTRA}[args.config]()
    commit_all = args.commit_all and args.config == "C4"
    if commit_all:
        w = dataclasses.replace(w, name=w.name + ", all 4 workers' blocks committed per step",
                                common_extra=w.n_workers * w.commit_tokens)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    L = w.layers if args.config != "C5" else 1
    if args.layers > 0:
        L = min(L, args.layers)
    lens, starts = w.block_lengths(), w.block_starts()
    chunk = args.chunk
    fp8 = args.kv == "fp8"
    if fp8:
        assert not args.unplanned, "--kv fp8 runs planned decodes"
        assert w.dtype == "bf16" and w.head_dim == 128, "E4M3 caches: the bf16 head_dim-128 shapes"
    if chunk > 0:
        assert not (args.append or args.unplanned), "--chunk runs planned decodes without appends"
        vb, vo, vl, qp = api.views_chunked(args.layout, lens, w.n_problems, w.n_workers, chunk)
        vl_dev = torch.from_numpy(vl).to(dev)  # uploaded once (the graph replays the plan)
    else:
        vb, vo, qp = api.views(args.layout, lens, w.n_problems, w.n_workers)
    n_rows = vb.shape[0]
    sess = engine.DecodeSession(n_rows=n_rows, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                                head_dim=w.head_dim, n_blocks=w.n_blocks,
                                max_view_blocks=w.n_workers + 1, capacity=w.capacity, dtype=tdt,
                                rope_theta=w.rope_theta, scale=w.scale, device=dev,
                                view_limits=chunk > 0, kv_fp8=fp8)
    sess.set_metadata(starts, lens, vb, vo, qp)
    qs, ks, vs = [], [], []
    kscale, vscale = [], []  # E4M3: per layer, the per-kv-head scales
    commit = w.commit_tokens > 0 and args.config == "C4"
    if commit:
        # one [layers][Hkv][cap][D] pool per K and V, so that one commit launch
        # covers every layer
        k_all = torch.empty((L, w.n_kv_heads, w.capacity, w.head_dim),
                            dtype=torch.uint8 if fp8 else tdt, device=dev)
        v_all = torch.empty_like(k_all)
    for l in range(L):
        q, k, v = wl.draw_device_layer(w, l, dev)
        if fp8:  # the layer's pools packed as E4M3 codes, one scale per kv head
            k, ksc = wl.e4m3_pack(k, lens, starts)
            v, vsc = wl.e4m3_pack(v, lens, starts)
            kscale.append(ksc)
            vscale.append(vsc)
        if chunk > 0:  # one query per chunk token
            gq = torch.Generator(device=dev)
            gq.manual_seed(7000 + l)
            q = torch.randn((n_rows, w.n_q_heads, w.head_dim), generator=gq, device=dev).to(tdt)
        if commit:
            k_all[l].copy_(k)
            v_all[l].copy_(v)
            k, v = k_all[l], v_all[l]
        qs.append(q)
        ks.append(k)
        vs.append(v)
    outs = [torch.empty_like(qs[0]) for _ in range(L)]
    lses = [torch.empty((n_rows, w.n_q_heads), dtype=torch.float32, device=dev) for _ in range(L)]
    calls_per_step = L if args.config != "C5" else 64  # C5: one layer timed x64
    kernel = "decode_tc_kernel" if (w.dtype == "bf16" and w.head_dim == 128) else "decode_simt_kernel"
    stream = torch.cuda.Stream(device=dev)

    planned = not args.unplanned
    # hw_attn_decode (unplanned) keeps the plan of the metadata it last saw.
    # A model's metadata changes every step (positions and lengths grow), so
    # the steps alternate between this metadata and an equivalent copy with
    # every view offset and position one higher (i_q - offset, and with it
    # every result, unchanged): the first layer of each step rebuilds the
    # plan, like the planned steps' hw_attn_plan.
    metas = [sess.meta]
    if not planned:
        alt = dict(sess.meta)
        alt["view_offset"] = sess.meta["view_offset"] + 1
        alt["q_pos"] = sess.meta["q_pos"] + 1
        metas.append(alt)

    append = args.append and planned and kernel == "decode_tc_kernel"
    if append:
        # every worker's new token at the last position of its own block (the
        # block lengths count it); the same rows are rewritten every step
        ab = np.full(w.n_rows, -1, np.int32)
        ap = np.zeros(w.n_rows, np.int32)
        for r in range(w.n_rows):
            pb, wk = divmod(r, w.n_workers)
            b = pb * (w.n_workers + 1) + 1 + wk
            if lens[b] > 0:
                ab[r], ap[r] = b, lens[b] - 1
        ab = torch.from_numpy(ab).to(dev)  # uploaded once (the graph replays the plan)
        ap = torch.from_numpy(ap).to(dev)
        gn = torch.Generator(device=dev)
        gn.manual_seed(4321)
        new_k = [torch.randn((w.n_rows, w.n_kv_heads, w.head_dim), generator=gn, device=dev).to(tdt)
                 for _ in range(L)]
        new_v = [torch.randn((w.n_rows, w.n_kv_heads, w.head_dim), generator=gn, device=dev).to(tdt)
                 for _ in range(L)]

    def layer_calls(qsrc, osrc=outs, lsrc=lses):
        # a decode step: the views are planned once, then every layer runs
        if planned and append:
            sess.plan_append(ab, ap, stream=stream)
        elif chunk > 0:
            sess.plan_limited(vl_dev, stream=stream)
        elif planned:
            sess.plan(stream=stream)
        for i in range(calls_per_step):
            l = i % L
            # The early-loads promise (HW_DESC_EARLY_LOADS): the call before
            # this one writes neither its pools nor the plan.  Not for the
            # first layer (it follows the plan, or the previous step's commit),
            # nor when the layers repeat one pool that the appends write.
            early = not args.no_early and i > 0 and not (append and L < calls_per_step)
            if append and fp8:
                sess.append_decode_planned_fp8(qsrc[l], new_k[l], new_v[l], ks[l], vs[l], kscale[l],
                                               vscale[l], out=osrc[l], lse=lsrc[l], stream=stream,
                                               early=early)
            elif append:
                sess.append_decode_planned(qsrc[l], new_k[l], new_v[l], ks[l], vs[l], out=osrc[l],
                                           lse=lsrc[l], stream=stream, early=early)
            elif planned and fp8:
                sess.decode_planned_fp8(qsrc[l], ks[l], vs[l], kscale[l], vscale[l], out=osrc[l],
                                        lse=lsrc[l], stream=stream, early=early)
            elif planned:
                sess.decode_planned(qsrc[l], ks[l], vs[l], out=osrc[l], lse=lsrc[l], stream=stream,
                                    early=early)
            else:
                sess.decode(qsrc[l], ks[l], vs[l], out=osrc[l], lse=lsrc[l], stream=stream,
                            early=early)

    step_no = [0]

    def commit_call():
        # a worker's finished step joins the common history: its block is
        # rotated by the position change and written after the common tokens
        # (the decode's views keep reading [0, common_len), so every rep times
        # the same work)
        if commit_all:
            n, c0 = w.commit_tokens, int(w.common_len[0])
            commits = [(int(starts[1 + k]), n, int(starts[0]) + c0 + k * n, c0 + k * n)
                       for k in range(w.n_workers)]
            engine.block_commit_many(k_all, v_all, commits, k_all, v_all, w.rope_theta, stream=stream)
            return
        wk = step_no[0] % w.n_workers
        step_no[0] += 1
        src = int(starts[1 + wk])
        engine.block_commit(k_all, v_all, src, w.commit_tokens, k_all, v_all,
                            int(starts[0]) + int(w.common_len[0]), int(w.common_len[0]),
                            w.rope_theta, stream=stream)

    def step(k=0):
        sess.meta = metas[k % len(metas)]
        layer_calls(qs)
        if commit:
            commit_call()

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for k in range(max(args.warmup, 3)):
            step(k)
    stream.synchronize()
    graphs = None
    if not args.eager:
        graphs = []
        for k in range(len(metas)):  # one graph per metadata set, replayed in turn
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(k)
            graphs.append(g)
        stream.synchronize()
        for k in range(2):
            graphs[k % len(graphs)].replay()
        stream.synchronize()
    flags = sess.device_flags()
    assert flags == 0, f"device flags {flags}"

    def run_timed(n):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            start.record(stream)
            for k in range(n):
                if graphs is not None:
                    graphs[k % len(graphs)].replay()
                else:
                    step(k)
            end.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        return start.elapsed_time(end) / 1e3

    with ClockSampler(local) as clk:
        t = run_timed(args.steps)
    t = max_over_ranks(t, dev)

    # algorithmic bytes: E4M3 codes are one byte where bf16 takes two
    div = 2 if fp8 else 1
    kv_layer = w.kv_bytes_per_layer() // div
    commit_bytes = (w.commit_bytes_per_layer() // div * L * (w.n_workers if commit_all else 1)
                    if commit else 0)
    step_bytes = kv_layer * calls_per_step + commit_bytes
    per_step = t / args.steps
    gbs_rank = step_bytes / per_step / 1e9
    value = replica_value(step_bytes / 1e9, per_step, world)  # replicas: each streams its own copy
    per_launch = per_step / calls_per_step
    achieved = kv_layer / per_launch / 1e9
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["hbm_gbs"])

    def run_e2e():
        # End to end through the public API with host buffers, as a serving
        # loop would run it: each step uploads the step's metadata and every
        # layer's query from pinned host memory (one packed copy), replays the
        # step's API calls (plan + every layer, captured once like the timed
        # region's), and reads every layer's output and lse back (one packed
        # copy each); the KV pools are the resident cache state.
        q_host = torch.stack([q for q in qs]).cpu().pin_memory()
        qdev_all = torch.empty(q_host.shape, dtype=q_host.dtype, device=dev)
        qdev = [qdev_all[l] for l in range(L)]
        outs_all = torch.empty((L,) + tuple(outs[0].shape), dtype=outs[0].dtype, device=dev)
        lses_all = torch.empty((L,) + tuple(lses[0].shape), dtype=lses[0].dtype, device=dev)
        o_host = torch.empty(outs_all.shape, dtype=outs_all.dtype, pin_memory=True)
        l_host = torch.empty(lses_all.shape, dtype=lses_all.dtype, pin_memory=True)
        # (unplanned: the steps upload the two equivalent metadata sets in turn)
        meta_hosts = [[torch.from_numpy(np.ascontiguousarray(x, np.int32)).pin_memory()
                       for x in (starts, lens, vb, np.asarray(vo) + k, np.asarray(qp) + k)]
                      for k in range(len(metas))]
        sess.meta = metas[0]
        meta_dev = [sess.meta[name] for name in ("block_start", "block_len", "view_block",
                                                 "view_offset", "q_pos")]
        if chunk > 0:
            meta_hosts[0].append(torch.from_numpy(np.ascontiguousarray(vl, np.int32)).pin_memory())
            meta_dev.append(vl_dev)
        h2d = q_host.numel() * q_host.element_size() + sum(m.numel() * 4 for m in meta_hosts[0])
        d2h = o_host.numel() * o_host.element_size() + l_host.numel() * 4

        def calls():
            layer_calls(qdev, [outs_all[l] for l in range(L)], [lses_all[l] for l in range(L)])
            if commit:
                commit_call()

        with torch.cuda.stream(stream):
            calls()
        stream.synchronize()
        g_e2e = None
        if graphs is not None:
            g_e2e = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_e2e, stream=stream):
                calls()
            stream.synchronize()

        def e2e_step(k):  # noqa: E306
            with torch.cuda.stream(stream):
                for m, md in zip(meta_hosts[k % len(meta_hosts)], meta_dev):
                    md.copy_(m, non_blocking=True)
                qdev_all.copy_(q_host, non_blocking=True)
                if g_e2e is not None:
                    g_e2e.replay()
                else:
                    calls()
                o_host.copy_(outs_all, non_blocking=True)
                l_host.copy_(lses_all, non_blocking=True)

        for k in range(3):
            e2e_step(k)
        stream.synchronize()
        e2e_steps = max(3, min(args.steps, 10))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for k in range(e2e_steps):
            e2e_step(k)
            stream.synchronize()
        t_e2e = (time.perf_counter() - t0) / e2e_steps
        assert torch.isfinite(o_host.float()).all(), "e2e outputs"
        t_e2e = max_over_ranks(t_e2e, dev)
        e2e_gbs = replica_value(step_bytes / 1e9, t_e2e, world)
        return {"value": e2e_gbs, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3,
                "how": "per step: metadata + packed queries H2D from pinned memory, the step's "
                       "API calls (captured once), packed outputs + lse D2H; host-timed with a "
                       "stream sync per step"}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e()

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 kv, bf16 q" if fp8 else w.dtype,
        "data": "synthetic",
        "config": {
            **workload_config(w, args.config, args.layout, calls_per_step),
            "kv_bytes_per_step": step_bytes, "commit_bytes_per_step": commit_bytes,
            "parallelism": f"replicas x{world}", "kv": args.kv,
            "query_rows": n_rows, "chunk": chunk if chunk > 0 else None,
            "mode": "eager" if graphs is None else "cuda-graph",
            "calls": (f"hw_attn_plan_append once per step + hw_attn_append_decode_planned"
                      f"{'_fp8' if fp8 else ''} per layer (each worker's new token written, then "
                      "decoded)" if append else
                      f"hw_attn_plan_limited once per step + hw_attn_decode_planned{'_fp8' if fp8 else ''} "
                      f"per layer ({chunk}-token chunks, causal within each worker's own block)"
                      if chunk > 0 else
                      "hw_attn_plan once per step + hw_attn_decode_planned_fp8 per layer (E4M3 "
                      "K/V codes, per-kv-head scales)" if fp8 else
                      "hw_attn_plan once per step + hw_attn_decode_planned per layer" if planned
                      else "hw_attn_decode per layer"),
            "l2": "inputs larger than L2: each step reads every layer's own KV pools "
                  f"({step_bytes / 1e9:.2f} GB per step vs 0.13 GB of L2)",
        },
        "frac_of_8TBps": gbs_rank / NOMINAL_HBM_GBS,
        "worker_tokens_per_s_per_layer": n_rows / per_launch,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": (measured_traffic(kernel, "qwq32b_w4_fp8" if fp8 else "qwq32b_w4")
                                 if args.config == "C3" and planned and not (append or chunk)
                                 and args.layout == "combined" else None),
                     "peak_kind": peak_kind,
                     "kernel": f"{'hw_attn_decode_planned' if planned else 'hw_attn_decode'} ({kernel})",
                     "per_launch": "step time / layers per step (the plan launch included)"},
        # every rank's launches in the timed region (replicas: the same on each)
        "gpu_launches": (calls_per_step + (1 if planned else 0) + (1 if commit else 0)) * args.steps * world,
        "clocks": clk.summary(),
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and chunk == 0 and not fp8:
        line["cpu_baseline"] = timed_oracle(w, qs, ks, vs, starts, lens, args.layout)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def timed_oracle(w, qs, ks, vs, starts, lens, layout, budget_s=12.0):
    """The oracle, as it stands, over whole layers of the same workload on the
    host cores for about budget_s seconds (at least one layer); GB/s of KV."""
    import numpy as np
    import torch
    import oracle

    # the timed step's views, from the oracle's own builders
    build_views = {"combined": oracle.combined_views, "interleaved": oracle.interleaved_views,
                   "contiguous": oracle.contiguous_views}[layout]
    vb, vo, qp = build_views(lens, w.n_problems, w.n_workers)

    def host(t):
        t = t.detach().cpu().contiguous()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    cores = len(os.sched_getaffinity(0))
    rows = None if w.n_problems == 1 else list(range(0, w.n_workers))  # one problem of the batch
    done, spent = 0, 0.0
    while True:
        l = done % len(qs)
        q, k, v = host(qs[l]), host(ks[l]), host(vs[l])
        t0 = time.perf_counter()
        oracle.get().attn_decode(q=q, k_cache=k, v_cache=v, block_start=starts, block_len=lens,
                                 view_block=vb, view_offset=vo, q_pos=qp,
                                 n_kv_heads=w.n_kv_heads, rope_theta=w.rope_theta, scale=w.scale,
                                 dtype=oracle.F32 if w.dtype == "f32" else oracle.BF16, rows=rows,
                                 n_threads=cores)
        spent += time.perf_counter() - t0
        done += 1
        if spent >= budget_s or done >= 4096:  # (the layers repeat past the stack)
            break
    if rows is None:
        nbytes = w.kv_bytes_per_layer() * done
        what = f"{done} whole layer(s), all rows and heads"
    else:
        per_problem = (w.common_len[0] + sum(w.worker_len[0])) * w.n_kv_heads * w.head_dim * 2 * w.elem_bytes
        nbytes = per_problem * done
        what = f"{done} layer(s) of problem 0 only"
    return {"value": nbytes / spent / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{what}, float64, {cores} threads, {spent:.1f} s"}


if __name__ == "__main__":
    main()
