"""Layer timeline of the tensor-core decode: consecutive layers of a decode
step (the same launches bench.py times, replayed from a CUDA graph) run
through the HW_TRACE build of the library, and the globaltimer stamps of
every CTA are summarised per layer - when the CTAs enter, when the wait on
the previous layer returns, when the first and last scores come, when the
records, arrivals and merges finish - and how the layers overlap: how many
of a layer's CTAs start before the previous layer has finished.

    python -m concurrent_shared_kv_gb300.trace --config C3 [--unplanned]
        [--kv fp8] [--no-early] [--layers 8] [--out FILE]

Prints a markdown summary (and writes it to FILE).  Needs a GPU; builds
_build_trace/libhogwild_trace.so first.
"""
from __future__ import annotations

import argparse
import sys

import numpy as np

from . import api, build


POINTS = [(0, "entry"), (1, "pre-wait done"), (2, "wait returned"), (3, "queries ready"),
          (4, "first scores"), (5, "last scores"), (6, "records stored"), (7, "arrivals"),
          (8, "merge phase"), (10, "item's records in"), (11, "item merged"), (12, "exit")]


def main(argv=None) -> int:
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--config", default="C3", choices=["C2", "C3", "C4", "C5", "W8"])
    p.add_argument("--layers", type=int, default=8, help="layers per step (at most 8 are kept)")
    p.add_argument("--unplanned", action="store_true", help="hw_attn_decode instead of the planned calls")
    p.add_argument("--no-early", action="store_true", help="without the early-loads promise")
    p.add_argument("--kv", default="bf16", choices=["bf16", "fp8"],
                   help="fp8: E4M3 pools with per-kv-head scales (planned calls)")
    p.add_argument("--out", default=None)
    args = p.parse_args(argv)
    fp8 = args.kv == "fp8"
    if fp8 and args.unplanned:
        p.error("E4M3 pools are decoded by the planned calls")
    api.use_library(build.build(trace=True))
    import torch
    from . import engine
    from . import workloads as wl
    w = {**wl.ALL, **wl.EXTRA}[args.config]()
    n = min(args.layers, 8)
    lens, starts = w.block_lengths(), w.block_starts()
    vb, vo, qp = api.views_combined(lens, w.n_problems, w.n_workers)
    s = engine.DecodeSession(n_rows=w.n_rows, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                             head_dim=w.head_dim, n_blocks=w.n_blocks,
                             max_view_blocks=w.n_workers + 1, capacity=w.capacity,
                             dtype=torch.bfloat16, rope_theta=w.rope_theta, scale=w.scale,
                             kv_fp8=fp8)
    s.set_metadata(starts, lens, vb, vo, qp)
    layers = []
    for l in range(n):
        q, k, v = wl.draw_device_layer(w, l, "cuda")
        if fp8:  # the layer's pools as E4M3 codes, one scale per kv head
            k, ks = wl.e4m3_pack(k, lens, starts)
            v, vs = wl.e4m3_pack(v, lens, starts)
            layers.append((q, k, v, ks, vs))
        else:
            layers.append((q, k, v, None, None))
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())

    def step():
        if not args.unplanned:
            s.plan(stream=st)
        for i, (q, k, v, ks, vs) in enumerate(layers):
            early = i > 0 and not args.no_early
            if args.unplanned:
                s.decode(q, k, v, stream=st, early=early)
            elif fp8:
                s.decode_planned_fp8(q, k, v, ks, vs, stream=st, early=early)
            else:
                s.decode_planned(q, k, v, stream=st, early=early)

    with torch.cuda.stream(st):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        step()
    with torch.cuda.stream(st):
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    api.trace_clear()
    with torch.cuda.stream(st):
        g.replay()
    torch.cuda.synchronize()
    assert s.device_flags() == 0
    T = api.trace_read().astype(np.int64)
    grid = engine_grid = int((T[:, :, 12] > 0).sum(axis=1).max())
    # the calls of the last replay, in launch order (by their wait's return)
    calls = [c for c in range(8) if (T[c, :grid, 2] > 0).any()]
    calls.sort(key=lambda c: T[c, :grid, 2][T[c, :grid, 2] > 0].min())
    lines = []
    mode = ("hw_attn_decode" if args.unplanned else "hw_attn_plan + hw_attn_decode_planned" +
            ("_fp8 (E4M3 pools)" if fp8 else "")) + \
        (", no early loads" if args.no_early else ", early loads after the first layer")
    lines.append(f"Layer timeline: {w.name}; {mode}; {engine_grid} CTAs; one step of {n} layers "
                 "from a CUDA graph (4th replay).  Times in us from the layer's first "
                 "griddepcontrol.wait return (t0): median / last CTA.")
    lines.append("")
    lines.append("| layer | t0 - previous t0 | " + " | ".join(nm for _, nm in POINTS) + " |")
    lines.append("|---" * (len(POINTS) + 2) + "|")
    prev_t0, periods = None, []
    for li, c in enumerate(calls):
        X = T[c, :grid]
        t0 = X[:, 2][X[:, 2] > 0].min()
        cells = []
        for k, _ in POINTS:
            x = X[:, k]
            x = x[x > 0]
            cells.append("-" if len(x) == 0 else f"{np.median(x - t0) / 1e3:.2f} / {(x.max() - t0) / 1e3:.2f}")
        per = "" if prev_t0 is None else f"{(t0 - prev_t0) / 1e3:.2f}"
        if prev_t0 is not None:
            periods.append((t0 - prev_t0) / 1e3)
        prev_t0 = t0
        lines.append(f"| {li} | {per} | " + " | ".join(cells) + " |")
    lines.append("")
    # overlap: CTAs of layer L+1 that entered before the last CTA of layer L exited
    lines.append("| layers | CTAs of L+1 entered before L's last exit | of them, past their "
                 "early work by then | entry - exit of L's CTA on the same SM, median (us) |")
    lines.append("|---|---|---|---|")
    for li in range(len(calls) - 1):
        A, B = T[calls[li], :grid], T[calls[li + 1], :grid]
        last_exit = A[:, 12].max()
        early_in = int((B[:, 0] < last_exit).sum())
        ready = int(((B[:, 1] > 0) & (B[:, 1] < last_exit)).sum())
        exit_by_sm = {int(A[c, 22]): A[c, 12] for c in range(grid)}
        gaps = [(B[c, 0] - exit_by_sm[int(B[c, 22])]) / 1e3 for c in range(grid)
                if int(B[c, 22]) in exit_by_sm]
        lines.append(f"| {li} -> {li + 1} | {early_in} / {grid} | {ready} | "
                     f"{np.median(gaps):.2f} |")
    if periods:
        lines.append("")
        lines.append(f"Median layer period (t0 to t0): {np.median(periods):.2f} us.")
    text = "\n".join(lines)
    print(text)
    if args.out:
        with open(args.out, "w") as f:
            f.write(text + "\n")
    return 0


if __name__ == "__main__":
    sys.exit(main())
