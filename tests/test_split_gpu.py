"""The tensor-core kernel's integer work list, exported from the plan
(hw_plan_export) and compared bit for bit with the oracle's restatement of
the split's definition (stream-K over a weighted line of 128-token tiles):
every CTA's unit range and the coordinates and segment flags of its first
tiles.  The ranges must also tile [0, U) with no gap or overlap."""
import numpy as np
import pytest

import oracle
from concurrent_shared_kv_gb300 import api
from concurrent_shared_kv_gb300 import workloads as wl
from tests import harness as H
from tests.test_parity_gpu import small

pytestmark = pytest.mark.gpu


def check_split(c, what):
    s = c.session()
    s.plan()
    got = api.plan_export(s.desc, s.workspace, s.ws_bytes)
    w = c.w
    want = oracle.stream_k_split(c.block_start, c.block_len, c.view_block, w.n_q_heads,
                                 w.n_kv_heads, grid=len(got))
    assert np.array_equal(got, want), (what, np.argwhere(got != want)[:5])
    # the ranges tile the units
    u0, u1 = got[:, 0], got[:, 1]
    assert u0[0] == 0 and np.all(u0[1:] == u1[:-1]) and np.all(u1 >= u0), what
    return got


@pytest.mark.parametrize("cfg", ["C2", "C3", "C4"])
def test_split_of_the_configs(cfg):
    w = wl.ALL[cfg]()
    c = H.device_case(w, 0)
    got = check_split(c, cfg)
    assert got[:, 1].max() > 0


def test_split_of_ragged_serving_and_edges():
    check_split(H.device_case(wl.serve_ragged()), "ragged")
    w = small(P=2, W=3, common=(300, 77), blocks=((129, 64, 1), (128, 0, 33)))
    check_split(H.host_case(w), "small edges")
    # interleaved views: each worker block is referenced by its own row only
    w = wl.qwq32b_w4()
    check_split(H.device_case(w, 0, views=api.views("interleaved", w.block_lengths(), 1, 4)),
                "interleaved")
