"""hw_attn_decode's plan cache.  The layers of a step share their metadata, so
a workspace keeps the plan of the metadata it last saw and a call rebuilds it
only when its metadata differs.  Every result must be bit for bit the one of
hw_attn_plan + hw_attn_decode_planned on the same metadata, whatever the
sequence: the same metadata again, new contents in the same arrays, the old
contents back, with and without the early-loads promise, replayed from a CUDA
graph across a change, and through the no-allocation entry point with its
description changing between calls."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from concurrent_shared_kv_gb300 import api
from concurrent_shared_kv_gb300 import workloads as wl
from tests import harness as H
from tests.test_parity_gpu import small

pytestmark = pytest.mark.gpu


def metadata_b(c):
    """Other metadata of the same shapes: worker block 1 one tile shorter and
    the interleaved views (each worker sees the common block and its own)."""
    w = c.w
    bl = c.block_len.copy()
    bl[2] = max(int(bl[2]) - 128, 1)
    vb, vo, qp = api.views("interleaved", bl, w.n_problems, w.n_workers)
    return c.block_start.copy(), bl, vb, vo, qp


def planned(c, meta):
    """The planned path on its own workspace."""
    s = c.session()
    s.set_metadata(*meta)
    s.plan()
    out, lse = s.decode_planned(c.q, c.k, c.v)
    torch.cuda.synchronize()
    assert s.device_flags() == 0
    return out, lse


def same(a, b):
    (o1, l1), (o2, l2) = a, b
    return torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def write_meta(s, meta):
    for key, x in zip(("block_start", "block_len", "view_block", "view_offset", "q_pos"), meta):
        s.meta[key].copy_(torch.as_tensor(np.ascontiguousarray(x, dtype=np.int32)))


def test_changes_in_place_and_back():
    w = wl.qwq32b_w4()
    c = H.device_case(w, 0)
    meta_a = (c.block_start, c.block_len, c.view_block, c.view_offset, c.q_pos)
    meta_b = metadata_b(c)
    ref_a, ref_b = planned(c, meta_a), planned(c, meta_b)
    assert not same(ref_a, ref_b)
    s = c.session()
    seq = [("a", False), ("a", True), ("a", True), ("b", False), ("b", True), ("a", False),
           ("a", True), ("b", False), ("b", False), ("b", True)]
    cur = "a"
    for i, (m, early) in enumerate(seq):
        if m != cur:
            write_meta(s, meta_a if m == "a" else meta_b)  # (a new step: no promise on this call)
            cur = m
        got = s.decode(c.q, c.k, c.v, early=early)
        torch.cuda.synchronize()
        assert same(got, ref_a if m == "a" else ref_b), (i, m, early)
    assert s.device_flags() == 0
    # and the planned path's results are the oracle's
    c_b = H.Case(w, c.q, c.k, c.v, block_start=meta_b[0], block_len=meta_b[1],
                 views=(meta_b[2], meta_b[3], meta_b[4]))
    ro, rl = c_b.run_oracle()
    H.compare("bf16", ref_b[0], ref_b[1], ro, rl, what="metadata b")


def test_graph_replay_across_a_change():
    w = wl.qwq32b_w4()
    layers = [H.device_case(w, l) for l in range(3)]
    c = layers[0]
    meta_a = (c.block_start, c.block_len, c.view_block, c.view_offset, c.q_pos)
    meta_b = metadata_b(c)
    refs = {m: [planned(x, meta) for x in layers] for m, meta in (("a", meta_a), ("b", meta_b))}
    s = c.session()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    outs = [torch.empty((w.n_rows, w.n_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
            for _ in layers]
    lses = [torch.empty((w.n_rows, w.n_q_heads), device="cuda") for _ in layers]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for i, x in enumerate(layers):
            s.decode(x.q, x.k, x.v, out=outs[i], lse=lses[i], stream=st, early=i > 0)
    for m in ("a", "b", "b", "a"):
        write_meta(s, meta_a if m == "a" else meta_b)
        torch.cuda.synchronize()
        for t in outs + lses:
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for i in range(len(layers)):
            assert same((outs[i], lses[i]), refs[m][i]), (m, i)
    assert s.device_flags() == 0


def test_noalloc_alternating_descriptions():
    # the scratch's layout follows the description: calls alternating between
    # two of them must each rebuild a plan of their own
    c1 = H.device_case(wl.qwq32b_w4(), 0)
    c2 = H.device_case(small(P=2, W=3, Hq=8, Hkv=2, common=(700, 300),
                             blocks=((129, 64, 1), (5, 0, 300))), 0)
    refs = []
    for c in (c1, c2):
        refs.append(planned(c, (c.block_start, c.block_len, c.view_block, c.view_offset, c.q_pos)))
    api.noalloc_status()
    for k in range(5):
        c = (c1, c2)[k % 2]
        s = c.session()
        m = s.meta
        w = c.w
        out = torch.empty((w.n_rows, w.n_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.n_rows, w.n_q_heads), device="cuda")
        for _ in range(2):  # the second call finds its plan cached
            api.attn_decode_noalloc(s.desc, c.q, c.k, c.v, m["block_start"], m["block_len"],
                                    m["view_block"], m["view_offset"], m["q_pos"], out, lse,
                                    q_to_kv=m["q_to_kv"])
            torch.cuda.synchronize()
            assert same((out, lse), refs[k % 2]), k
    assert api.noalloc_status() == 0
