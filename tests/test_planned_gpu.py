"""hw_attn_plan + hw_attn_decode_planned: the step's metadata planned once,
then one call per layer.  A planned call must give exactly what
hw_attn_decode gives on the same metadata (the plan is the same computation,
moved out of the layer loop), on the tensor-core and the CUDA-core paths; it
must keep serving after the caller's metadata arrays change; and a missing or
mismatched plan must be reported (HW_DEV_BAD_PLAN) without touching the
outputs."""
import numpy as np
import pytest
import torch

from concurrent_shared_kv_gb300 import api
from concurrent_shared_kv_gb300 import workloads as wl
from tests import harness as H
from tests.test_parity_gpu import small

pytestmark = pytest.mark.gpu


def planned_vs_plain(c: H.Case):
    s = c.session()
    ref_out, ref_lse = s.decode(c.q, c.k, c.v)
    s.plan()
    out, lse = s.decode_planned(c.q, c.k, c.v)
    torch.cuda.synchronize()
    assert s.device_flags() == 0
    assert torch.equal(out.view(torch.int16) if out.dtype == torch.bfloat16 else out,
                       ref_out.view(torch.int16) if ref_out.dtype == torch.bfloat16 else ref_out)
    assert torch.equal(lse, ref_lse)
    return s, out, lse


@pytest.mark.parametrize("make", [wl.tiny_f32, wl.qwq32b_w4, wl.serve_ragged],
                         ids=["tiny-f32", "qwq32b-w4", "serve-ragged"])
def test_planned_equals_unplanned(make):
    w = make()
    c = H.host_case(w) if w.dtype == "f32" else H.device_case(w, 0)
    _, out, lse = planned_vs_plain(c)
    if w.dtype == "f32":
        ro, rl = c.run_oracle()
        H.compare(w.dtype, out, lse, ro, rl, what="planned f32")


@pytest.mark.parametrize("case", ["head-map", "empty-rows", "offsets", "many"])
def test_planned_edge_cases(case):
    if case == "head-map":
        w = small(Hq=8, Hkv=2)
        c = H.host_case(w, q_to_kv=np.array([1, 0, 0, 1, 1, 0, 1, 0], np.int32))
    elif case == "empty-rows":
        w = small(blocks=((0, 5, 0),), common=(77,))
        c = H.host_case(w)
        vb = c.view_block.copy()
        vb[1] = -1
        c.view_block = vb
    elif case == "offsets":
        w = small(W=3, blocks=((129, 64, 10),))
        rng = np.random.default_rng(3)
        vb = np.stack([rng.permutation(4) for _ in range(3)]).astype(np.int32)
        vo = rng.integers(-10 ** 6, 10 ** 6, size=vb.shape).astype(np.int32)
        qp = rng.integers(0, 2 * 10 ** 6, size=3).astype(np.int32)
        c = H.host_case(w, views=(vb, vo, qp))
    else:
        rng = np.random.default_rng(9)
        P, W = 24, 3
        common = [int(x) for x in rng.integers(1, 700, size=P)]
        blocks = [[int(x) for x in rng.integers(0, 200, size=W)] for _ in range(P)]
        w = wl.Workload("many", "bf16", P, W, 8, 2, 128, 1e6, 1, common, blocks, seed=13)
        c = H.host_case(w)
    _, out, lse = planned_vs_plain(c)
    ro, rl = c.run_oracle()
    H.compare(w.dtype, out, lse, ro, rl, what=f"planned {case}")


def test_one_plan_serves_every_layer_and_owns_its_metadata():
    w = wl.qwq32b_w2()
    c0 = H.device_case(w, 0)
    s = c0.session()
    s.plan()
    # the caller's arrays may change after planning: the plan keeps its copy
    saved = {k: v.clone() for k, v in s.meta.items() if v is not None}
    for v in s.meta.values():
        if v is not None:
            v.fill_(-7)
    outs = []
    for layer in (0, 1, w.layers - 1):
        c = H.device_case(w, layer)
        out, lse = s.decode_planned(c.q, c.k, c.v)
        outs.append((c, out.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert s.device_flags() == 0
    s.meta.update(saved)
    for c, out, lse in outs:
        ref_out, ref_lse = s.decode(c.q, c.k, c.v)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse, ref_lse)


def test_missing_or_mismatched_plan_is_reported():
    w = wl.qwq32b_w4()
    c = H.device_case(w, 0)
    s = c.session()
    # no plan in a fresh workspace
    out = torch.full((w.n_rows, w.n_q_heads, w.head_dim), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    lse = torch.full((w.n_rows, w.n_q_heads), float("nan"), device="cuda")
    s.decode_planned(c.q, c.k, c.v, out=out, lse=lse)
    torch.cuda.synchronize()
    assert s.device_flags() & 32  # HW_DEV_BAD_PLAN
    assert torch.isnan(out.float()).all() and torch.isnan(lse).all()
    # a plan made for another description
    s.plan()
    d2 = api.make_desc(w.n_rows, w.n_q_heads, w.n_kv_heads, w.head_dim, s.desc.n_blocks,
                       s.desc.max_view_blocks, s.desc.cache_capacity // 2, api.HW_BF16,
                       w.rope_theta, w.scale)
    assert api.attn_decode_workspace_size(d2) <= s.ws_bytes
    api.attn_decode_planned(d2, c.q, c.k, c.v, out, lse, s.workspace, s.ws_bytes)
    torch.cuda.synchronize()
    assert s.device_flags() & 32
    assert torch.isnan(out.float()).all()
    # and the right description still works afterwards
    o2, l2 = s.decode_planned(c.q, c.k, c.v)
    torch.cuda.synchronize()
    assert s.device_flags() == 0 and torch.isfinite(o2.float()).all()
