"""View limits and query chunks without a GPU: the oracle's chunk views
written out by hand from their definition (T query rows per worker, each
seeing its own block up to its own token), the library's hw_views_chunked
equal to them, and the C ABI's argument checks, which run before anything is
enqueued."""
import numpy as np
import pytest

import oracle
from concurrent_shared_kv_gb300 import api

LENS = [10, 4, 5, 6]  # one problem: common 10, worker blocks 4, 5, 6


def test_oracle_chunk_views_written_out():
    vb, vo, lim, qp = oracle.chunk_views("combined", LENS, 1, 3, 2)
    # rows (w, t): worker 0's view is common, w1, w2, itself at offset 21
    assert vb.tolist() == [[0, 2, 3, 1]] * 2 + [[0, 1, 3, 2]] * 2 + [[0, 1, 2, 3]] * 2
    assert vo.tolist() == [[0, 10, 15, 21]] * 2 + [[0, 10, 14, 20]] * 2 + [[0, 10, 14, 19]] * 2
    # own block of 4, chunk of 2: its tokens at positions 2 and 3 see 3 and 4
    assert lim.tolist() == [[-1, -1, -1, 3], [-1, -1, -1, 4], [-1, -1, -1, 4], [-1, -1, -1, 5],
                            [-1, -1, -1, 5], [-1, -1, -1, 6]]
    assert qp.tolist() == [23, 24, 23, 24, 23, 24]
    vb, vo, lim, qp = oracle.chunk_views("interleaved", LENS, 1, 3, 3)
    assert vb[3].tolist() == [0, 2, -1, -1] and vo[3].tolist() == [0, 10, 0, 0]
    assert lim[3:6].tolist() == [[-1, 3, -1, -1], [-1, 4, -1, -1], [-1, 5, -1, -1]]
    assert qp[3:6].tolist() == [12, 13, 14]


def test_chunk_of_one_is_the_layout_view_at_the_last_token():
    # T = 1: the row is the layout's row, its own block whole, the query at
    # its block's last token (one before the layout's q_pos, which sits after
    # the view)
    lens = [300, 7, 129, 64, 1]
    for layout in ("combined", "interleaved"):
        vb1, vo1, qp1 = oracle.layout_views(layout, lens, 1, 4)
        vb, vo, lim, qp = oracle.chunk_views(layout, lens, 1, 4, 1)
        assert np.array_equal(vb, vb1) and np.array_equal(vo, vo1)
        assert np.array_equal(qp, qp1 - 1)
        for r in range(4):
            v = int(np.where(vb[r] == 1 + r)[0][0])
            assert lim[r, v] == lens[1 + r]


@pytest.mark.parametrize("layout", ["combined", "interleaved", "contiguous"])
@pytest.mark.parametrize("P,W,T", [(1, 1, 1), (2, 2, 3), (3, 4, 2), (16, 4, 4)])
def test_library_chunk_views_equal_the_oracle(layout, P, W, T):
    rng = np.random.default_rng(10 * P + W + T)
    lens = rng.integers(T, 3000, size=P * (W + 1)).astype(np.int32)
    got = api.views_chunked(layout, lens, P, W, T)
    want = oracle.chunk_views(layout, lens, P, W, T)
    for g, w_ in zip(got, want):
        assert np.array_equal(g, w_)


def test_chunk_views_reject_bad_arguments():
    for args in [(7, LENS, 1, 3, 2), ("combined", LENS, 1, 3, 0), ("combined", LENS, 1, 3, 5)]:
        with pytest.raises(api.HwError) as e:
            api.views_chunked(*args)  # unknown layout; empty chunk; a block shorter than it
        assert e.value.status == -1


FAKE = 1 << 20


def desc(**kw):
    base = dict(n_rows=2, n_q_heads=4, n_kv_heads=2, head_dim=128, n_blocks=3, max_view_blocks=3,
                cache_capacity=400, dtype=api.HW_BF16, rope_theta=1e6, scale=0.088)
    base.update(kw)
    return api.make_desc(**base)


def status(fn, *args, **kw):
    try:
        return fn(*args, **kw)
    except api.HwError as e:
        return e.status


LIM = api.HW_DESC_VIEW_LIMITS


def test_plan_limited_needs_the_flag_the_limits_and_the_tensor_core_path():
    # (these checks come before the workspace's, so no device is needed)
    call = lambda d, vl=FAKE: status(api.attn_plan_limited, d, FAKE, FAKE, FAKE, FAKE, vl, FAKE,
                                     FAKE, 0)
    assert call(desc(flags=LIM), vl=None) == -1
    assert call(desc()) == -1                          # a descriptor without the flag
    assert call(desc(flags=LIM, dtype=api.HW_F32)) == -2
    assert call(desc(flags=LIM, head_dim=64)) == -2
    assert call(desc(flags=64)) == -1                  # an unknown flag


def test_a_limited_descriptor_is_only_planned_with_limits():
    d = desc(flags=LIM)
    assert status(api.attn_plan, d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == -2
    assert status(api.attn_plan_append, d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0) == -2
    assert status(api.attn_append_decode_planned, d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                  FAKE, 0) == -2
    assert status(api.attn_decode, d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                  FAKE, 0) == -2
    assert status(api.attn_decode_noalloc, d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                  None) == -2


def test_views_reject_more_rows_on_a_block_than_a_plan_ranks():
    # a block named by more than HW_MAX_REFS_PER_BLOCK = 255 view entries is
    # skipped by the decode; the host builders refuse such tables up front
    with pytest.raises(api.HwError) as e:
        api.views_combined(np.full(257, 10, np.int32), 1, 256)  # 256 rows on the common block
    assert e.value.status == -2
    with pytest.raises(api.HwError) as e:
        api.views_chunked("combined", np.full(5, 300, np.int32), 1, 4, 64)  # 4 x 64 rows
    assert e.value.status == -2
    # at the limit: 255 rows
    vb, vo, qp = api.views_combined(np.full(256, 10, np.int32), 1, 255)
    assert (vb[:, 0] == 0).all()
