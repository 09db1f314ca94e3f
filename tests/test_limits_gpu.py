"""GPU parity of view limits (hw_attn_plan_limited + hw_attn_decode_planned,
through the C ABI) against the float64 oracle: query chunks, each row seeing
its own block only up to its own token (causal order inside the chunk) and the
other blocks whole, and limits anywhere in a block - mid-tile, on tile edges,
zero, past the end - including blocks split over many CTAs, whose later
partials then hold no token of a limited row."""
import numpy as np
import pytest
import torch

import oracle
from concurrent_shared_kv_gb300 import api
from concurrent_shared_kv_gb300 import workloads as wl
from tests import harness as H
from tests.test_parity_gpu import small

pytestmark = pytest.mark.gpu


def chunk_case(w, T, layout="combined", seed=31, device=False):
    """The workload's caches with T query rows per worker (chunk views)."""
    vb, vo, vl, qp = api.views_chunked(layout, w.block_lengths(), w.n_problems, w.n_workers, T)
    rows = vb.shape[0]
    if device:
        _, k, v = wl.draw_device_layer(w, 0, "cuda")
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)
        q = torch.randn((rows, w.n_q_heads, w.head_dim), generator=g, device="cuda").to(k.dtype)
    else:
        _, k, v = wl.draw_host(w, 0)
        rng = np.random.default_rng(seed)
        q = wl.to_storage(rng.standard_normal((rows, w.n_q_heads, w.head_dim)), w.dtype)
        q, k, v = (H.from_storage_np(x, w.dtype) for x in (q, k, v))
    return H.Case(w, q, k, v, views=(vb, vo, qp)), vl


def oracle_limited(c, vl, rows=None):
    w = c.w
    return oracle.get().attn_decode(
        q=H.to_storage_np(c.q), k_cache=H.to_storage_np(c.k), v_cache=H.to_storage_np(c.v),
        block_start=c.block_start, block_len=c.block_len, view_block=c.view_block,
        view_offset=c.view_offset, q_pos=c.q_pos, n_kv_heads=w.n_kv_heads,
        rope_theta=w.rope_theta, scale=w.scale, dtype=oracle.BF16, rows=rows, view_limit=vl)


def run_limited(c, vl):
    s = c.session(view_limits=True)
    s.plan_limited(vl)
    out, lse = s.decode_planned(c.q, c.k, c.v)
    torch.cuda.synchronize()
    assert s.device_flags() == 0
    return out, lse, s


def check(c, vl, what, rows=None):
    out, lse, s = run_limited(c, vl)
    ro, rl = oracle_limited(c, vl, rows)
    H.compare("bf16", out, lse, ro, rl, rows=rows, what=what)
    return out, lse, s


@pytest.mark.parametrize("layout", ["combined", "interleaved"])
def test_chunks_across_tile_edges(layout):
    # own blocks 129 (chunk tokens 126..128: the last one opens the second
    # tile), 64, 3 (the whole block is the chunk); 130, 5, 256
    w = small(P=2, W=3, Hq=4, Hkv=2, common=(300, 77), blocks=((129, 64, 3), (130, 5, 256)))
    c, vl = chunk_case(w, 3, layout)
    assert {127, 128, 129, 1, 3, 254, 256} <= set(vl[vl >= 0].tolist())
    check(c, vl, f"chunks {layout}")


def test_no_limit_is_the_plain_plan_bit_for_bit():
    w = small(P=2, W=3, Hq=4, Hkv=2, common=(3000, 77), blocks=((129, 64, 3), (130, 5, 256)))
    c = H.host_case(w)
    s = c.session()
    s.plan()
    out0, lse0 = s.decode_planned(c.q, c.k, c.v)
    torch.cuda.synchronize()
    lens = c.block_len
    none = np.full(c.view_block.shape, -1, np.int32)
    past = np.where(c.view_block >= 0, lens[np.maximum(c.view_block, 0)] + 7, -1).astype(np.int32)
    for vl in (none, past):
        out, lse, _ = run_limited(c, vl)
        assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
        assert torch.equal(lse, lse0)


def test_limits_anywhere_on_blocks_split_over_many_ctas():
    # a 40000-token common block is cut into many CTAs' shares; rows limited
    # to a prefix of it leave the later shares' partials empty for their
    # columns, and a row limited to nothing at all gives zero and -inf
    w = small(P=1, W=3, Hq=8, Hkv=2, common=(40000,), blocks=((700, 129, 128),))
    c = H.host_case(w)
    vl = np.full(c.view_block.shape, -1, np.int32)
    own = lambda r: int(np.where(c.view_block[r] == 1 + r)[0][0])
    vl[0, 0] = 300            # common: a prefix inside the third tile
    vl[0, own(0)] = 128       # own block: exactly one tile
    vl[1, 0] = 0              # common dropped
    vl[1, 1] = 1              # one token of worker 0's block
    vl[2, :] = 0              # nothing at all
    out, lse, _ = check(c, vl, "limits anywhere")
    assert torch.all(out[2] == 0) and torch.all(torch.isneginf(lse[2]))


def test_random_limits():
    w = small(P=2, W=4, Hq=8, Hkv=2, common=(5000, 900),
              blocks=((129, 64, 1, 300), (2, 700, 256, 255)))
    c = H.host_case(w)
    rng = np.random.default_rng(17)
    lens = c.block_len[np.maximum(c.view_block, 0)]
    vl = (rng.random(c.view_block.shape) * (lens + 2)).astype(np.int32) - 1
    vl[rng.random(vl.shape) < 0.3] = -1
    check(c, vl, "random limits")


def test_chunks_qwen3_8b_shape_w4_t2():
    # 32K common, four 1024-token worker blocks, two query rows per worker:
    # 8 rows x 4 query heads per kv head = the tile's 32 columns on every block
    w = wl.qwen3_8b_w4()
    c, vl = chunk_case(w, 2, device=True)
    check(c, vl, "qwen3-8b W4 chunks of 2")
