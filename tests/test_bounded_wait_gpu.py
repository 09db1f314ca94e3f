"""A bounded wait made to run out, with no fault and no hang: the merge of one
(row, q head) item is made to wait for one partial result more than any CTA
delivers (its arrival counter starts at -1 instead of 0), under a wait bound
of 10^5 cycles.  The call must return, report HW_DEV_TIMEOUT, leave that
item's rows untouched and merge every other item correctly; an ordinary call
on a fresh workspace afterwards must match the oracle."""
import numpy as np
import pytest
import torch

from concurrent_shared_kv_gb300 import api
from concurrent_shared_kv_gb300 import workloads as wl
from tests import harness as H
from tests.test_parity_gpu import small

pytestmark = pytest.mark.gpu

COUNTERS_INT32 = 256 // 4  # the arrival counters follow the 256-byte error word


def run_with_unreachable_item(c, planned, item=0):
    w = c.w
    s = c.session()
    ws = s.workspace.view(torch.int32)
    ws[COUNTERS_INT32 + item] = -1  # one arrival short, whatever the CTAs deliver
    out = torch.full((c.q.shape[0], w.n_q_heads, w.head_dim), float("nan"), dtype=c.q.dtype,
                     device="cuda")
    lse = torch.full((c.q.shape[0], w.n_q_heads), float("nan"), device="cuda")
    api.test_set_merge_wait_limit(100000)
    try:
        if planned:
            s.plan()
            s.decode_planned(c.q, c.k, c.v, out=out, lse=lse)
        else:
            s.decode(c.q, c.k, c.v, out=out, lse=lse)
        torch.cuda.synchronize()
    finally:
        api.test_set_merge_wait_limit(0)
    return s, out, lse


@pytest.mark.parametrize("planned", [True, False])
def test_merge_wait_gives_up_and_reports_timeout(planned):
    w = wl.qwq32b_w4()
    c = H.device_case(w, 0)
    s, out, lse = run_with_unreachable_item(c, planned, item=0)
    assert s.device_flags() & 16  # HW_DEV_TIMEOUT
    o = out.float().view(-1, w.head_dim)
    assert torch.isnan(o[0]).all() and torch.isnan(lse.view(-1)[0])  # the item given up
    assert torch.isfinite(o[1:]).all() and torch.isfinite(lse.view(-1)[1:]).all()
    # every other item is the oracle's
    ro, rl = c.run_oracle()
    g = H.out_f64(out).reshape(-1, w.head_dim)[1:]
    r = ro.reshape(-1, w.head_dim)[1:]
    assert np.abs(g - r).max() <= H.BF16_MAX
    # a fresh workspace works as before
    c2 = H.device_case(w, 1)
    s2 = c2.session()
    if planned:
        s2.plan()
        o2, l2 = s2.decode_planned(c2.q, c2.k, c2.v)
    else:
        o2, l2 = s2.decode(c2.q, c2.k, c2.v)
    torch.cuda.synchronize()
    assert s2.device_flags() == 0
    ro2, rl2 = c2.run_oracle()
    H.compare(w.dtype, o2, l2, ro2, rl2, what="after a timed-out call")


def test_merge_wait_gives_up_on_the_fp32_kernel():
    w = small(P=1, W=2, common=(256,), blocks=((32, 40),), dtype="f32", D=64)
    c = H.host_case(w)
    s, out, lse = run_with_unreachable_item(c, planned=False, item=3)
    assert s.device_flags() & 16
    o = out.float().view(-1, w.head_dim)
    assert torch.isnan(o[3]).all()
    keep = [i for i in range(o.shape[0]) if i != 3]
    assert torch.isfinite(o[keep]).all()
