"""The early-loads promise (HW_DESC_EARLY_LOADS): with it a decode reads its
plan (or metadata) and starts its first K/V tiles before the previous kernel
on the stream has completed.  Results must be bit for bit those of the same
calls without the promise, back to back on one stream and replayed from a CUDA
graph (where consecutive layers overlap), and match the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from concurrent_shared_kv_gb300 import workloads as wl
from tests import harness as H

pytestmark = pytest.mark.gpu


def _layers(w, n):
    return [H.device_case(w, l) for l in range(n)]


def _step(s, cases, outs, lses, planned, early, stream):
    if planned:
        s.plan(stream=stream)
    for i, c in enumerate(cases):
        e = early and i > 0
        if planned:
            s.decode_planned(c.q, c.k, c.v, out=outs[i], lse=lses[i], stream=stream, early=e)
        else:
            s.decode(c.q, c.k, c.v, out=outs[i], lse=lses[i], stream=stream, early=e)


def _buffers(w, n):
    outs = [torch.empty((w.n_rows, w.n_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
            for _ in range(n)]
    lses = [torch.empty((w.n_rows, w.n_q_heads), device="cuda") for _ in range(n)]
    return outs, lses


@pytest.mark.parametrize("planned", [True, False])
def test_early_loads_change_no_bit(planned):
    w = wl.qwq32b_w4()
    n = 6
    cases = _layers(w, n)
    s = cases[0].session()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    ref_o, ref_l = _buffers(w, n)
    with torch.cuda.stream(st):
        _step(s, cases, ref_o, ref_l, planned, early=False, stream=st)
    st.synchronize()
    # eagerly, then from a graph (replayed twice into fresh buffers)
    o1, l1 = _buffers(w, n)
    with torch.cuda.stream(st):
        _step(s, cases, o1, l1, planned, early=True, stream=st)
    st.synchronize()
    o2, l2 = _buffers(w, n)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        _step(s, cases, o2, l2, planned, early=True, stream=st)
    for _ in range(2):
        for t in o2 + l2:
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for i in range(n):
            assert torch.equal(o2[i].view(torch.int16), ref_o[i].view(torch.int16)), f"graph layer {i}"
            assert torch.equal(l2[i], ref_l[i]), f"graph lse layer {i}"
    for i in range(n):
        assert torch.equal(o1[i].view(torch.int16), ref_o[i].view(torch.int16)), f"layer {i}"
        assert torch.equal(l1[i], ref_l[i])
    assert s.device_flags() == 0
    for i in (0, n - 1):
        ro, rl = cases[i].run_oracle()
        H.compare(w.dtype, ref_o[i], ref_l[i], ro, rl, what=f"early layer {i}")


def test_early_loads_on_the_serving_workload():
    # 16 ragged problems: more items than CTAs, so every CTA merges
    w = wl.serve_ragged()
    cases = [H.device_case(w, 0), H.device_case(w, 1)]
    s = cases[0].session()
    outs, lses = _buffers(w, 2)
    ref_o, ref_l = _buffers(w, 2)
    _step(s, cases, ref_o, ref_l, True, early=False, stream=None)
    _step(s, cases, outs, lses, True, early=True, stream=None)
    torch.cuda.synchronize()
    for i in range(2):
        assert torch.equal(outs[i].view(torch.int16), ref_o[i].view(torch.int16))
        assert torch.equal(lses[i], ref_l[i])
    rows = list(range(0, 4)) + list(range(60, 64))
    ro, rl = cases[1].run_oracle(rows=rows)
    H.compare(w.dtype, outs[1], lses[1], ro, rl, rows=rows, what="early serving layer 1")
