"""GPU parity of E4M3 KV caches with per-kv-head scales (hw_attn_plan +
hw_attn_decode_planned_fp8, and hw_block_commit on E4M3 pools, through the C
ABI) against the float64 oracle on the same codes and scales.  The caches'
quantisation is part of the inputs - both sides attend the decoded, scaled
codes - so the bar is the bf16 path's: the kernel's own arithmetic (queries
in four E4M3 parts, about 16 significant bits; P in f16) is no coarser than
the bf16 path's (queries in two bf16 parts; P in bf16).  A first build with
three parts (about 13 bits) missed the lse bar on large queries."""
import numpy as np
import pytest
import torch

import oracle
from concurrent_shared_kv_gb300 import api, engine
from concurrent_shared_kv_gb300 import workloads as wl
from tests import harness as H
from tests.test_parity_gpu import small

pytestmark = pytest.mark.gpu


class Fp8Case:
    """A workload's bf16 queries and its caches packed as E4M3 codes."""

    def __init__(self, c: H.Case, q=None, poison_code=None):
        self.c = c
        w = c.w
        self.q = c.q if q is None else q
        lens, starts = c.block_len, c.block_start
        self.kc, self.ks = wl.e4m3_pack(c.k, lens, starts)
        self.vc, self.vs = wl.e4m3_pack(c.v, lens, starts)
        if poison_code is not None:  # rows outside every block: never read
            used = torch.zeros(self.kc.shape[1], dtype=torch.bool, device=self.kc.device)
            for s_, n in zip(starts, lens):
                used[int(s_):int(s_) + int(n)] = True
            self.kc[:, ~used] = poison_code
            self.vc[:, ~used] = poison_code

    def run(self):
        c, w = self.c, self.c.w
        s = engine.DecodeSession(n_rows=self.q.shape[0], n_q_heads=w.n_q_heads,
                                 n_kv_heads=w.n_kv_heads, head_dim=w.head_dim,
                                 n_blocks=len(c.block_len), max_view_blocks=c.view_block.shape[1],
                                 capacity=c.capacity, dtype=torch.bfloat16, rope_theta=w.rope_theta,
                                 scale=w.scale, kv_fp8=True)
        s.set_metadata(c.block_start, c.block_len, c.view_block, c.view_offset, c.q_pos, c.q_to_kv)
        s.plan()
        out, lse = s.decode_planned_fp8(self.q, self.kc, self.vc, self.ks, self.vs)
        torch.cuda.synchronize()
        assert s.device_flags() == 0
        return out, lse, s

    def oracle(self, rows=None):
        c, w = self.c, self.c.w
        return oracle.get().attn_decode(
            q=H.to_storage_np(self.q), k_cache=self.kc.cpu().numpy(), v_cache=self.vc.cpu().numpy(),
            k_scale=self.ks.cpu().numpy(), v_scale=self.vs.cpu().numpy(), block_start=c.block_start,
            block_len=c.block_len, view_block=c.view_block, view_offset=c.view_offset, q_pos=c.q_pos,
            n_kv_heads=w.n_kv_heads, rope_theta=w.rope_theta, scale=w.scale, dtype=oracle.FP8,
            q_to_kv=c.q_to_kv, rows=rows)

    def check(self, what, rows=None):
        out, lse, s = self.run()
        ro, rl = self.oracle(rows)
        H.compare("bf16", out, lse, ro, rl, rows=rows, what=what)
        return out, lse


def test_fp8_small_edges():
    # ragged tiles (129, 64, 1, 128, 33), an empty block, two problems
    w = small(P=2, W=3, common=(300, 77), blocks=((129, 64, 1), (128, 0, 33)))
    Fp8Case(H.host_case(w)).check("fp8 small")


def test_fp8_codes_outside_the_blocks_are_never_read():
    w = small(extra=37, blocks=((129, 64, 10),))
    Fp8Case(H.host_case(w), poison_code=0x7F).check("fp8 NaN codes in the slack")


@pytest.mark.parametrize("qscale", [1e-3, 1.0, 300.0])
def test_fp8_query_magnitudes(qscale):
    # the query parts' scale is a power of two per segment: tiny and large
    # queries, and one q head far smaller than the others of its segment
    w = small(P=1, W=3, common=(700,), blocks=((129, 64, 40),))
    c = H.host_case(w)
    q = (c.q.float() * qscale)
    q[:, 1] *= 1e-3
    Fp8Case(c, q=q.to(torch.bfloat16)).check(f"fp8 q x{qscale}")


def test_fp8_qwq32b_w4_layer():
    w = wl.qwq32b_w4()
    Fp8Case(H.device_case(w, 0)).check("fp8 C3 layer", rows=[0, 1, 2, 3])


def test_fp8_serving_ragged_many_segments_per_cta():
    w = wl.serve_ragged()
    Fp8Case(H.device_case(w)).check("fp8 serving ragged", rows=list(range(0, 4)) + list(range(60, 64)))


def test_fp8_is_deterministic():
    w = small(P=2, W=3, common=(3000, 77), blocks=((129, 64, 1), (128, 5, 33)))
    f = Fp8Case(H.host_case(w))
    o1, l1, _ = f.run()
    o2, l2, _ = f.run()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_fp8_commit_against_the_oracle():
    # two layers x 8 heads: 300 tokens rotated by 1000 positions into another
    # range of the same pool, codes rounded from the fp32 rotation
    rng = np.random.default_rng(4)
    L_, Hkv, cap, D = 2, 8, 2000, 128
    x = rng.standard_normal((L_ * Hkv, cap, D))
    codes, _ = wl.e4m3_pack(x)
    k = torch.from_numpy(codes).view(L_, Hkv, cap, D).cuda()
    v = torch.from_numpy(codes[::-1].copy()).view(L_, Hkv, cap, D).cuda()
    k0, v0 = k.cpu().numpy().copy(), v.cpu().numpy().copy()
    engine.block_commit(k, v, 100, 300, k, v, 1500, 1000, 1e6)
    torch.cuda.synchronize()
    kg, vg = k.cpu().numpy(), v.cpu().numpy()
    for l in range(L_):
        kd, vd = oracle.get().block_commit(dtype=oracle.FP8, rope_theta=1e6, k_src=k0[l], v_src=v0[l],
                                           src_begin=100, n_tokens=300, k_dst=k0[l], v_dst=v0[l],
                                           dst_offset=1500, pos_delta=1000)
        assert np.array_equal(vg[l], vd)
        same = kg[l] == kd
        # the kernel rotates in fp32: a value next to a rounding boundary may
        # land on the neighbouring code; every other code is the oracle's
        assert same.mean() > 0.995, same.mean()
        got, want = wl.e4m3_values(kg[l][~same]), wl.e4m3_values(kd[~same])
        step = np.maximum(np.abs(want), 2.0 ** -6) * 2.0 ** -3
        assert np.all(np.abs(got - want) <= step * 1.0001)


def test_fp8_interleaved_layout():
    # views [common, own]: each worker block is read for one row only
    w = small(P=2, W=3, common=(1000, 77), blocks=((129, 64, 1), (128, 5, 33)))
    c = H.host_case(w, views=api.views("interleaved", w.block_lengths(), w.n_problems, w.n_workers))
    Fp8Case(c).check("fp8 interleaved")


def test_fp8_commit_many_equals_the_commits_in_turn():
    # three finished steps of one layer committed in one launch
    rng = np.random.default_rng(6)
    Hkv, cap, D = 4, 3000, 128
    codes, _ = wl.e4m3_pack(rng.standard_normal((Hkv, cap, D)))
    k = torch.from_numpy(codes).cuda()
    v = torch.from_numpy(codes[:, ::-1].copy()).cuda()
    k0, v0 = k.cpu().numpy().copy(), v.cpu().numpy().copy()
    commits = [(0, 200, 1000, 1000), (200, 150, 1200, 1200), (350, 77, 1350, 1350)]
    engine.block_commit_many(k, v, commits, k, v, 1e6)
    torch.cuda.synchronize()
    kd, vd = k0, v0
    for sb, n, dst, delta in commits:
        kd, vd = oracle.get().block_commit(dtype=oracle.FP8, rope_theta=1e6, k_src=k0, v_src=v0,
                                           src_begin=sb, n_tokens=n, k_dst=kd, v_dst=vd,
                                           dst_offset=dst, pos_delta=delta)
    kg, vg = k.cpu().numpy(), v.cpu().numpy()
    assert np.array_equal(vg, vd)
    same = kg == kd
    assert same.mean() > 0.998, same.mean()


def test_fp8_full_tile_of_columns():
    # 256 query heads over 8 kv heads: every block's tile carries 32 columns,
    # the Q~ buffer all four parts x 32 rows; one row viewing 20 blocks
    rng = np.random.default_rng(29)
    nb, Hq, Hkv, D = 20, 256, 8, 128
    lens = rng.integers(1, 300, size=nb).astype(np.int32)
    w = wl.Workload("fp8 columns", "bf16", 1, 1, Hq, Hkv, D, 1e6, 1, [0], [[0]], seed=6)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int32)
    cap = int(lens.sum())
    k = wl.to_storage(rng.standard_normal((Hkv, cap, D)), "bf16")
    v = wl.to_storage(rng.standard_normal((Hkv, cap, D)), "bf16")
    q = wl.to_storage(rng.standard_normal((1, Hq, D)), "bf16")
    vb = np.arange(nb, dtype=np.int32)[None, :]
    vo = np.concatenate([[0], np.cumsum(lens)[:-1]])[None, :].astype(np.int32)
    qp = np.array([cap], np.int32)
    c = H.Case(w, H.from_storage_np(q, "bf16"), H.from_storage_np(k, "bf16"),
               H.from_storage_np(v, "bf16"), block_start=starts, block_len=lens, views=(vb, vo, qp))
    Fp8Case(c).check("fp8 32 columns")


def test_fp8_with_query_chunks():
    # view limits over E4M3 caches: three-token chunks causal in their own
    # blocks, against the oracle with the same limits, codes and scales
    w = small(P=2, W=3, Hq=4, Hkv=2, common=(300, 77), blocks=((129, 64, 3), (130, 5, 256)))
    vb, vo, vl, qp = api.views_chunked("combined", w.block_lengths(), w.n_problems, w.n_workers, 3)
    rng = np.random.default_rng(41)
    _, k, v = wl.draw_host(w, 0)
    q = wl.to_storage(rng.standard_normal((vb.shape[0], w.n_q_heads, w.head_dim)), "bf16")
    c = H.Case(w, H.from_storage_np(q, "bf16"), H.from_storage_np(k, "bf16"),
               H.from_storage_np(v, "bf16"), views=(vb, vo, qp))
    f = Fp8Case(c)
    s = engine.DecodeSession(n_rows=vb.shape[0], n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                             head_dim=w.head_dim, n_blocks=len(c.block_len),
                             max_view_blocks=vb.shape[1], capacity=c.capacity, dtype=torch.bfloat16,
                             rope_theta=w.rope_theta, scale=w.scale, kv_fp8=True, view_limits=True)
    s.set_metadata(c.block_start, c.block_len, vb, vo, qp)
    s.plan_limited(vl)
    out, lse = s.decode_planned_fp8(f.q, f.kc, f.vc, f.ks, f.vs)
    torch.cuda.synchronize()
    assert s.device_flags() == 0
    ro, rl = oracle.get().attn_decode(
        q=H.to_storage_np(f.q), k_cache=f.kc.cpu().numpy(), v_cache=f.vc.cpu().numpy(),
        k_scale=f.ks.cpu().numpy(), v_scale=f.vs.cpu().numpy(), block_start=c.block_start,
        block_len=c.block_len, view_block=vb, view_offset=vo, q_pos=qp, n_kv_heads=w.n_kv_heads,
        rope_theta=w.rope_theta, scale=w.scale, dtype=oracle.FP8, view_limit=vl)
    H.compare("bf16", out, lse, ro, rl, what="fp8 chunks")


def _fp8_append_check(c, what, rows=None):
    from tests.test_append_gpu import last_position_appends, new_tokens
    w = c.w
    f = Fp8Case(c)
    ab, ap = last_position_appends(c)
    kn, vn = new_tokens(w, 12)
    kc0, vc0 = f.kc.cpu().numpy().copy(), f.vc.cpu().numpy().copy()
    s = engine.DecodeSession(n_rows=w.n_rows, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                             head_dim=w.head_dim, n_blocks=len(c.block_len),
                             max_view_blocks=c.view_block.shape[1], capacity=c.capacity,
                             dtype=torch.bfloat16, rope_theta=w.rope_theta, scale=w.scale,
                             kv_fp8=True)
    s.set_metadata(c.block_start, c.block_len, c.view_block, c.view_offset, c.q_pos)
    s.plan_append(ab, ap)
    out, lse = s.append_decode_planned_fp8(f.q, kn, vn, f.kc, f.vc, f.ks, f.vs)
    torch.cuda.synchronize()
    assert s.device_flags() == 0
    ks, vs = f.ks.cpu().numpy(), f.vs.cpu().numpy()
    kd, vd, _ = oracle.append_tokens_e4m3(oracle.get(), rope_theta=w.rope_theta, k_cache=kc0,
                                          v_cache=vc0, k_new=H.to_storage_np(kn),
                                          v_new=H.to_storage_np(vn), k_scale=ks, v_scale=vs,
                                          block_start=c.block_start, append_block=ab, append_pos=ap)
    kg, vg = f.kc.cpu().numpy(), f.vc.cpu().numpy()
    # untouched rows bit for bit; the new codes the oracle's, or one code step
    # away where the fp32 rotation and reciprocal meet a rounding boundary
    for got, want in ((kg, kd), (vg, vd)):
        diff = got != want
        assert diff.mean() < 1e-3, (what, diff.mean())
        a_, b_ = wl.e4m3_values(got[diff]), wl.e4m3_values(want[diff])
        assert np.all(np.abs(a_ - b_) <= np.maximum(np.abs(b_), 2.0 ** -6) * 2.0 ** -3 * 1.0001), what
    ro, rl = oracle.get().attn_decode(
        q=H.to_storage_np(f.q), k_cache=kg, v_cache=vg, k_scale=ks, v_scale=vs,
        block_start=c.block_start, block_len=c.block_len, view_block=c.view_block,
        view_offset=c.view_offset, q_pos=c.q_pos, n_kv_heads=w.n_kv_heads,
        rope_theta=w.rope_theta, scale=w.scale, dtype=oracle.FP8, rows=rows)
    H.compare("bf16", out, lse, ro, rl, rows=rows, what=what)


def test_fp8_append_small_edges():
    w = small(P=2, W=3, common=(300, 77), blocks=((129, 64, 1), (128, 0, 33)))
    _fp8_append_check(H.host_case(w), "fp8 append small")


def test_fp8_append_qwq32b_w4_layer():
    _fp8_append_check(H.device_case(wl.qwq32b_w4(), 0), "fp8 append C3 layer", rows=[0, 1, 2, 3])
