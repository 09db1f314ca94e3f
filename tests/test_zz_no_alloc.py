"""hw_attn_decode_noalloc: decode attention for callers that cannot allocate.

Code running inside a memory pool or allocator, plugins whose host runtime owns
every device buffer, and processes that forbid allocation after start-up cannot
hand hw_attn_decode a freshly allocated workspace.  The no-allocation entry
point runs the same kernels on a fixed scratch array the library holds.  These
tests call it through the C ABI and check it against the workspace entry point,
twice in a row (the scratch keeps the previous call's contents), within the
tolerances of the parity tests.  The file sorts last so that a run stopping at
its first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from concurrent_shared_kv_gb300 import api
from concurrent_shared_kv_gb300 import workloads as wl
from tests import harness as H

pytestmark = pytest.mark.gpu


def _tolerances(dtype):
    return (H.F32_TOL, H.F32_TOL) if dtype == "f32" else (H.BF16_MAX, H.BF16_MEAN)


@pytest.mark.parametrize("make", [wl.tiny_f32, wl.qwq32b_w4], ids=["tiny-f32", "qwq32b-w4"])
def test_noalloc_matches_workspace_entry_point(make):
    w = make()
    c = H.host_case(w) if w.dtype == "f32" else H.device_case(w, 0)
    s = c.session()
    ref_out, ref_lse = s.decode(c.q, c.k, c.v)  # hw_attn_decode with a workspace
    torch.cuda.synchronize()
    m = s.meta
    max_tol, mean_tol = _tolerances(w.dtype)
    for call in range(2):  # the scratch keeps the last call's contents
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        api.attn_decode_noalloc(s.desc, c.q, c.k, c.v, m["block_start"], m["block_len"],
                                m["view_block"], m["view_offset"], m["q_pos"], out, lse,
                                q_to_kv=m["q_to_kv"])
        torch.cuda.synchronize()
        err = (out.double() - ref_out.double()).abs()
        assert torch.isfinite(out).all(), call
        assert err.max().item() <= max_tol and err.mean().item() <= mean_tol, (call, err.max().item())
        lerr = (lse.double() - ref_lse.double()).abs().max().item()
        assert lerr <= H.LSE_TOL[w.dtype], (call, lerr)


def test_noalloc_rejects_descriptions_beyond_the_scratch():
    # 256 blocks x 8 kv heads of partial-record slots need more than 32 MiB
    d = api.make_desc(4, 40, 8, 128, 256, 5, 1 << 20, api.HW_BF16, 1e6, 128 ** -0.5)
    need = api.attn_decode_workspace_size(d)
    assert need > (32 << 20)
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    st = api.lib().hw_attn_decode_noalloc(ctypes.byref(d), *([dummy.data_ptr()] * 12), None)
    assert st == -3  # HW_ERR_WORKSPACE, nothing enqueued


def test_noalloc_status_reports_device_errors():
    # seven workers at five query heads per kv head put 35 query columns on
    # every block (two column groups): the no-allocation call matches the
    # oracle and leaves no error bit.  A view naming a block that does not
    # exist then records HW_DEV_BAD_BLOCK, which the no-allocation status
    # call reads (and clears) without a workspace.
    w = wl.Workload("wide", "bf16", 1, 7, 40, 8, 128, 1e6, 1, [512], [[64] * 7], seed=21)
    c = H.device_case(w, 0)
    s = c.session()
    m = s.meta
    api.noalloc_status()  # start from a clear word (earlier calls may have left bits)
    out = torch.empty((w.n_rows, w.n_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.n_rows, w.n_q_heads), device="cuda")
    api.attn_decode_noalloc(s.desc, c.q, c.k, c.v, m["block_start"], m["block_len"],
                            m["view_block"], m["view_offset"], m["q_pos"], out, lse,
                            q_to_kv=m["q_to_kv"])
    assert api.noalloc_status() == 0
    ro, rl = c.run_oracle()
    H.compare("bf16", out, lse, ro, rl, what="noalloc 35 columns")
    bad = m["view_block"].clone()
    bad[0, 1] = w.n_blocks + 5  # no such block
    api.attn_decode_noalloc(s.desc, c.q, c.k, c.v, m["block_start"], m["block_len"], bad,
                            m["view_offset"], m["q_pos"], out, lse, q_to_kv=m["q_to_kv"])
    assert api.noalloc_status() & 1  # HW_DEV_BAD_BLOCK
    assert api.noalloc_status() == 0  # read and cleared
