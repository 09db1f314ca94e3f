"""GPU parity for the layout ablation's layouts and the batched commit,
through the C ABI against the float64 oracle: decoding over interleaved views
(each worker sees the history and its own step only), hw_block_commit_many
against the oracle's single commits applied in order, and one interleaved
step after several workers' steps were committed in one launch."""
import numpy as np
import pytest
import torch

import oracle
from concurrent_shared_kv_gb300 import api, engine
from concurrent_shared_kv_gb300 import workloads as wl
from tests import harness as H
from tests.test_parity_gpu import run_and_compare, small

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_interleaved_views_small(dtype):
    w = small(dtype=dtype, P=2, W=3, common=(300, 77), blocks=((129, 64, 1), (0, 200, 33)))
    lens = w.block_lengths()
    c = H.host_case(w, views=api.views("interleaved", lens, w.n_problems, w.n_workers))
    assert (c.view_block[:, 2:] == -1).all()
    run_and_compare(c, f"interleaved {dtype}")


def test_interleaved_views_qwq32b_w4_layer():
    w = wl.qwq32b_w4()
    c = H.device_case(w, 0, views=api.views("interleaved", w.block_lengths(), 1, 4))
    _, _, s = run_and_compare(c, "interleaved C3 layer 0")
    assert s.device_flags() == 0
    # the planned path reads the same views from its plan
    s.plan()
    out, lse = s.decode_planned(c.q, c.k, c.v)
    ref_out, ref_lse = s.decode(c.q, c.k, c.v)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse, ref_lse)


def commit_oracle_in_order(dtype, theta, k, v, commits):
    """The oracle's single commits applied one after the other (each sees the
    previous one's writes), on [Hkv][cap][D] storage arrays."""
    kd, vd = k, v
    exact = []
    for (src, n, dst, delta) in commits:
        kd, vd, ex = oracle.get().block_commit(dtype=dtype, rope_theta=theta, k_src=kd, v_src=vd,
                                               src_begin=src, n_tokens=n, k_dst=kd, v_dst=vd,
                                               dst_offset=dst, pos_delta=delta, want_exact=True)
        exact.append(ex)
    return kd, vd, exact


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_commit_many_equals_single_commits(dtype):
    L, Hkv, cap, D, theta = 3, 4, 700, 128, 1e6
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    k = torch.randn((L, Hkv, cap, D), generator=g, device="cuda").to(tdt)
    v = torch.randn((L, Hkv, cap, D), generator=g, device="cuda").to(tdt)
    # three workers' finished steps (blocks at 450.., 500.., 600..) join the
    # history after its 300 tokens, in worker order; plus an empty commit
    commits = [(450, 37, 300, 300), (500, 64, 337, 337), (600, 1, 401, 401), (650, 0, 0, 0)]
    before = [(H.to_storage_np(k[l]), H.to_storage_np(v[l])) for l in range(L)]
    engine.block_commit_many(k, v, commits, k, v, theta)
    torch.cuda.synchronize()
    odt = oracle.F32 if dtype == "f32" else oracle.BF16
    for l in range(L):
        kd, vd, exact = commit_oracle_in_order(odt, theta, *before[l], commits)
        kg, vg = H.to_storage_np(k[l]), H.to_storage_np(v[l])
        assert np.array_equal(vg, vd), l  # V: bit copies, nothing else written
        mask = np.zeros(cap, bool)
        for (src, n, dst, _), ex in zip(commits, exact):
            mask[dst:dst + n] = True
        assert np.array_equal(kg[:, ~mask], kd[:, ~mask]), l
        for (src, n, dst, _), ex in zip(commits, exact):
            if n == 0:
                continue
            got = wl.storage_to_f64(kg[:, dst:dst + n], dtype)
            if dtype == "f32":
                assert np.max(np.abs(got - ex)) < 1e-5
            else:
                src_vals = wl.storage_to_f64(before[l][0][:, src:src + n], dtype)
                half = D // 2
                mag = np.abs(src_vals) + np.abs(np.concatenate([src_vals[..., half:], src_vals[..., :half]], -1))
                assert (np.abs(got - ex) <= np.abs(ex) * 2.0 ** -7 + mag * 2.0 ** -20).all(), l
                assert np.mean(kg[:, dst:dst + n] == kd[:, dst:dst + n]) > 0.99


def test_interleaved_step_after_a_batched_commit():
    """Step 1 over interleaved views; workers 0 and 2 finish their steps and
    join the history in one launch; step 2's views see them in the common
    block (and worker 1's unfinished step still only in its own view)."""
    w = small(dtype="bf16", P=1, W=3, common=(300,), blocks=((129, 64, 40),), extra=200)
    c1 = H.host_case(w, views=api.views("interleaved", w.block_lengths(), 1, 3))
    run_and_compare(c1, "interleaved step 1")
    starts, lens = c1.block_start.copy(), c1.block_len.copy()
    k0, v0 = H.to_storage_np(c1.k), H.to_storage_np(c1.v)
    common = int(lens[0])
    commits = [(int(starts[1]), int(lens[1]), common, common),
               (int(starts[3]), int(lens[3]), common + int(lens[1]), common + int(lens[1]))]
    engine.block_commit_many(c1.k, c1.v, commits, c1.k, c1.v, w.rope_theta)
    torch.cuda.synchronize()
    kd, vd, _ = commit_oracle_in_order(oracle.BF16, w.rope_theta, k0, v0, commits)
    lens2 = lens.copy()
    lens2[0] = common + lens[1] + lens[3]
    lens2[1] = lens2[3] = 0
    views2 = api.views("interleaved", lens2, 1, 3)
    c2 = H.Case(w, c1.q, c1.k, c1.v, block_len=lens2, views=views2)
    out, lse, s = c2.run_gpu()
    # the oracle decodes its own committed caches
    ro, rl = oracle.get().attn_decode(
        q=H.to_storage_np(c1.q), k_cache=kd, v_cache=vd, block_start=c2.block_start,
        block_len=lens2, view_block=views2[0], view_offset=views2[1], q_pos=views2[2],
        n_kv_heads=w.n_kv_heads, rope_theta=w.rope_theta, scale=w.scale, dtype=oracle.BF16)
    H.compare("bf16", out, lse, ro, rl, what="interleaved step 2")
    assert s.device_flags() == 0
