"""Cache layouts of the Hogwild! notes' layout ablation (combined,
interleaved, contiguous) and the batched commit's host-side checks, without a
GPU.  The oracle's views are pinned against arrays written out by hand from
the definitions; the library's hw_views must then equal the oracle's."""
import numpy as np
import pytest

import oracle
from concurrent_shared_kv_gb300 import api

# one problem, three workers: common 10 tokens, worker blocks 4, 5 and 6
LENS = [10, 4, 5, 6]


def test_oracle_interleaved_views_written_out():
    # a worker sees the history and its own unfinished step, nothing else
    vb, vo, qp = oracle.interleaved_views(LENS, 1, 3)
    assert vb.tolist() == [[0, 1, -1, -1], [0, 2, -1, -1], [0, 3, -1, -1]]
    assert vo.tolist() == [[0, 10, 0, 0], [0, 10, 0, 0], [0, 10, 0, 0]]
    assert qp.tolist() == [14, 15, 16]


@pytest.mark.parametrize("layout", ["combined", "contiguous"])
def test_oracle_combined_order_written_out(layout):
    # common, the other workers in id order, itself
    vb, vo, qp = oracle.layout_views(layout, LENS, 1, 3)
    assert vb.tolist() == [[0, 2, 3, 1], [0, 1, 3, 2], [0, 1, 2, 3]]
    assert vo.tolist() == [[0, 10, 15, 21], [0, 10, 14, 20], [0, 10, 14, 19]]
    assert qp.tolist() == [25, 25, 25]


def test_oracle_layouts_second_problem_uses_its_own_blocks():
    lens = LENS + [7, 1, 2, 3]
    vb, vo, qp = oracle.interleaved_views(lens, 2, 3)
    assert vb[3:].tolist() == [[4, 5, -1, -1], [4, 6, -1, -1], [4, 7, -1, -1]]
    assert qp[3:].tolist() == [8, 9, 10]


@pytest.mark.parametrize("layout", ["combined", "interleaved", "contiguous"])
@pytest.mark.parametrize("P,W", [(1, 1), (2, 2), (3, 4), (16, 4)])
def test_library_views_equal_the_oracle(layout, P, W):
    rng = np.random.default_rng(100 * P + W)
    lens = rng.integers(0, 3000, size=P * (W + 1)).astype(np.int32)
    got = api.views(layout, lens, P, W)
    want = oracle.layout_views(layout, lens, P, W)
    for g, w_ in zip(got, want):
        assert np.array_equal(g, w_)
    if layout == "combined":
        for g, w_ in zip(api.views_combined(lens, P, W), want):
            assert np.array_equal(g, w_)


def test_views_reject_an_unknown_layout():
    with pytest.raises(api.HwError) as e:
        api.views(7, LENS, 1, 3)
    assert e.value.status == -1


# ---------------------------------------------------------------------------
# hw_block_commit_many: every error is found before anything is enqueued
# ---------------------------------------------------------------------------

KS, VS, KD, VD = 1 << 30, 2 << 30, 3 << 30, 4 << 30  # aligned, far apart, never dereferenced


def many(commits, cap_src=1000, cap_dst=1000, k_dst=KD, v_dst=VD, k_src=KS, v_src=VS):
    cols = list(zip(*commits)) if commits else [(), (), (), ()]
    try:
        return api.block_commit_many(api.HW_BF16, 2, 8, 128, 1e6, k_src, v_src, cap_src, k_dst, v_dst,
                                     cap_dst, *cols)
    except api.HwError as e:
        return e.status


def test_commit_many_errors_before_launch():
    assert many([]) == 0  # nothing to do: no launch
    assert many([(0, 0, 5, 5)]) == 0  # an empty commit: no launch
    assert many([(0, 10, 0, 0), (20, 10, 5, 5)]) == -5  # destinations meet
    assert many([(0, 10, 995, 995)]) == -4  # past the destination pool
    assert many([(995, 10, 0, 0)]) == -4  # past the source pool
    assert many([(-1, 10, 0, 0)]) == -1
    assert many([(0, 1, 2 * i, 0) for i in range(api.HW_MAX_COMMITS + 1)]) == -1
    # the same pool: a destination range may not meet any source range
    assert many([(0, 10, 100, 100), (100, 10, 200, 100)], k_dst=KS, v_dst=VS) == -5
    with pytest.raises(ValueError):
        api.block_commit_many(api.HW_BF16, 1, 8, 128, 1e6, KS, VS, 10, KD, VD, 10, [0, 1], [1], [0], [0])
