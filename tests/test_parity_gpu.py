"""GPU parity: hw_attn_decode and hw_block_commit (through the C ABI) against
the float64 oracle on the same seeded inputs, for all five workload shapes and
the edge cases.  Tolerances: fp32 max-abs 1e-5; bf16 max-abs 2e-2 and
mean-abs 1e-2 (fp32 accumulation); indexing and placement bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from concurrent_shared_kv_gb300 import api, engine
from concurrent_shared_kv_gb300 import workloads as wl
from tests import harness as H

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------------------
# the five workload shapes
# ---------------------------------------------------------------------------

def test_tiny_f32_all_rows():
    w = wl.tiny_f32()
    c = H.host_case(w)
    out, lse, s = c.run_gpu()
    ro, rl = c.run_oracle()
    bo, bl = c.run_oracle(brute=True)
    assert np.max(np.abs(ro - bo)) < 1e-12  # the oracle's two forms agree here too
    H.compare(w.dtype, out, lse, ro, rl, what="tiny f32")
    assert s.device_flags() == 0


def test_tiny_f32_commit_then_decode():
    w = wl.tiny_f32()
    c = H.host_case(w)
    starts, lens = c.block_start, c.block_len
    cap_common = w.common_len[0] + w.common_extra  # 288
    k0, v0 = H.to_storage_np(c.k), H.to_storage_np(c.v)
    # worker 0's step (block 1) moves to the end of the common history
    src, n, dst = int(starts[1]), int(lens[1]), int(lens[0])
    engine.block_commit(c.k, c.v, src, n, c.k, c.v, dst, dst, w.rope_theta)
    torch.cuda.synchronize()
    kd, vd, exact = oracle.get().block_commit(dtype=oracle.F32, rope_theta=w.rope_theta, k_src=k0,
                                              v_src=v0, src_begin=src, n_tokens=n, k_dst=k0,
                                              v_dst=v0, dst_offset=dst, pos_delta=dst,
                                              want_exact=True)
    kg, vg = H.to_storage_np(c.k), H.to_storage_np(c.v)
    assert np.array_equal(vg, vd)  # V bit copy, nothing else moved
    mask = np.zeros(kg.shape[1], bool)
    mask[dst:dst + n] = True
    assert np.array_equal(kg[:, ~mask], kd[:, ~mask])
    assert np.max(np.abs(kg[:, mask].astype(np.float64) - exact)) < 1e-5
    assert dst + n <= cap_common
    # next step: common grew by n, worker 0's block is empty
    lens2 = lens.copy()
    lens2[0] += n
    lens2[1] = 0
    c2 = H.Case(w, c.q, c.k, c.v, block_len=lens2)
    out, lse, _ = c2.run_gpu()
    ro, rl = c2.run_oracle()
    H.compare(w.dtype, out, lse, ro, rl, what="after commit")


@pytest.mark.parametrize("cfg", ["C2", "C3", "C4"])
def test_bf16_stack_first_and_last_layer(cfg):
    w = wl.ALL[cfg]()
    sess = None
    for layer in (0, w.layers - 1):
        c = H.device_case(w, layer)
        out, lse, sess = c.run_gpu(sess)
        ro, rl = c.run_oracle()
        H.compare(w.dtype, out, lse, ro, rl, what=f"{cfg} layer {layer}")
        del c
    assert sess.device_flags() == 0


def test_serving_ragged_problems_0_and_15():
    w = wl.serve_ragged()
    c = H.device_case(w)
    out, lse, s = c.run_gpu()
    rows = list(range(0, 4)) + list(range(60, 64))
    ro, rl = c.run_oracle(rows=rows)
    H.compare(w.dtype, out, lse, ro, rl, rows=rows, what="serving ragged")
    assert s.device_flags() == 0


def test_qwen3_commit_all_layers_one_launch():
    w = wl.qwen3_8b_w4()
    L, Hkv, cap, D = w.layers, w.n_kv_heads, w.capacity, w.head_dim
    g = torch.Generator(device="cuda")
    g.manual_seed(4242)
    k = torch.empty((L, Hkv, cap, D), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    for l in range(L):
        k[l] = torch.randn((Hkv, cap, D), generator=g, device="cuda").to(torch.bfloat16)
        v[l] = torch.randn((Hkv, cap, D), generator=g, device="cuda").to(torch.bfloat16)
    starts = w.block_starts()
    worker = 2  # the commit of step 2 (step mod 4)
    src, n, dst = int(starts[1 + worker]), 1024, w.common_len[0]
    before = {l: (H.to_storage_np(k[l]), H.to_storage_np(v[l])) for l in (0, L - 1)}
    engine.block_commit(k, v, src, n, k, v, dst, dst, w.rope_theta)
    torch.cuda.synchronize()
    for l in (0, L - 1):
        k0, v0 = before[l]
        kd, vd, exact = oracle.get().block_commit(dtype=oracle.BF16, rope_theta=w.rope_theta,
                                                  k_src=k0, v_src=v0, src_begin=src, n_tokens=n,
                                                  k_dst=k0, v_dst=v0, dst_offset=dst,
                                                  pos_delta=dst, want_exact=True)
        kg, vg = H.to_storage_np(k[l]), H.to_storage_np(v[l])
        assert np.array_equal(vg, vd), l
        mask = np.zeros(cap, bool)
        mask[dst:dst + n] = True
        assert np.array_equal(kg[:, ~mask], kd[:, ~mask]), l
        got = wl.storage_to_f64(kg[:, mask], "bf16")
        # one bf16 unit in the last place of the exact value, plus the fp32
        # rotation's own error where the two products cancel (a few fp32 ulps
        # of the pair's magnitude)
        src_pair = wl.storage_to_f64(k0[:, src:src + n], "bf16")
        half = D // 2
        mag = np.abs(src_pair) + np.abs(np.concatenate([src_pair[..., half:], src_pair[..., :half]], -1))
        bound = np.abs(exact) * 2.0 ** -7 + mag * 2.0 ** -20
        bad = np.abs(got - exact) > bound
        assert not bad.any(), (l, got[bad][:5], exact[bad][:5], bound[bad][:5])
        # most values are the correctly rounded bf16 of the exact rotation
        assert np.mean(kg[:, mask] == kd[:, mask]) > 0.99


# ---------------------------------------------------------------------------
# bit-exact indexing: a saturating one-hot score returns one V row exactly
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_one_hot_returns_exact_v_row(dtype):
    w = wl.Workload("one-hot", dtype, 1, 3, 8, 2, 128, 1e6, 1, [300], [[129, 64, 1]], sink=False,
                    seed=77)
    q, k, v = wl.draw_host(w)
    k[:] = 0
    starts, lens = w.block_starts(), w.block_lengths()
    vb, vo, qp = api.views_combined(lens, 1, 3)
    o = oracle.get()
    rng = np.random.default_rng(5)
    checks = []
    qf = wl.storage_to_f64(q, dtype)
    for (row, head, block, t) in [(0, 0, 0, 0), (0, 3, 0, 127), (1, 4, 0, 128), (2, 7, 0, 299),
                                  (1, 1, 1, 63), (2, 5, 1, 128), (0, 6, 2, 0), (1, 2, 3, 0),
                                  (2, 0, 2, 64)]:
        g = head // 4
        kt = rng.standard_normal(128)
        kt_s = wl.to_storage(kt, dtype)
        k[g, starts[block] + t] = kt_s
        ktd = wl.storage_to_f64(kt_s, dtype)
        v_idx = int(np.where(vb[row] == block)[0][0])
        rel = int(qp[row]) - int(vo[row, v_idx])
        lam = 400.0 / (np.dot(ktd, ktd) * w.scale)
        qf[row, head] = o.rope(lam * ktd, w.rope_theta, -rel)  # rho(q, rel) = lam * k_t
        checks.append((row, head, g, starts[block] + t))
    # only one hot key per (kv head, row view): keep the ones that do not share a kv head
    q = wl.to_storage(qf, dtype)
    c = H.Case(w, H.from_storage_np(q, dtype), H.from_storage_np(k, dtype),
               H.from_storage_np(v, dtype), views=(vb, vo, qp))
    out, _, s = c.run_gpu()
    got = H.to_storage_np(out)
    ro, _ = c.run_oracle()
    for (row, head, g, tok) in checks:
        # the planted key is the largest score by >= 300 nats among the view
        # only when no other planted key of kv head g is in the view; the oracle
        # says which rows are saturated
        want = v[g, tok]
        if np.array_equal(wl.to_storage(ro[row, head], dtype), want):
            assert np.array_equal(got[row, head], want), (row, head, tok)
    n_sat = sum(np.array_equal(wl.to_storage(ro[r, h], dtype), v[g, t]) for r, h, g, t in checks)
    assert n_sat >= 6


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

def small(dtype="bf16", P=1, W=3, Hq=8, Hkv=2, D=128, common=(300,), blocks=((129, 64, 1),),
          extra=0, seed=11, theta=1e6):
    return wl.Workload("edge", dtype, P, W, Hq, Hkv, D, theta, 1, list(common),
                       [list(b) for b in blocks], common_extra=extra, sink=True, seed=seed)


def run_and_compare(c: H.Case, what: str, rows=None):
    out, lse, s = c.run_gpu()
    ro, rl = c.run_oracle(rows=rows)
    H.compare(c.w.dtype, out, lse, ro, rl, rows=rows, what=what)
    return out, lse, s


def test_nan_in_unused_capacity_is_never_read():
    for dtype in ("f32", "bf16"):
        w = small(dtype=dtype, extra=37)
        c = H.host_case(w, poison=float("nan"))
        run_and_compare(c, f"poison {dtype}")


def test_empty_views_and_zero_length_blocks():
    w = small(blocks=((0, 5, 0),), common=(77,))
    c = H.host_case(w)
    vb = c.view_block.copy()
    vb[1] = -1  # row 1 sees nothing at all
    c.view_block = vb
    out, lse, s = run_and_compare(c, "empty")
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    w = small(blocks=((0, 0, 0),), common=(0,))
    c = H.host_case(w)
    out, lse, s = c.run_gpu()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 2), (40, 8), (32, 8)])
def test_group_sizes(Hq, Hkv):
    w = small(Hq=Hq, Hkv=Hkv, W=2, blocks=((200, 77),))
    run_and_compare(H.host_case(w), f"G={Hq // Hkv}")


def test_custom_head_map():
    w = small(Hq=8, Hkv=2)
    qmap = np.array([1, 0, 0, 1, 1, 0, 1, 0], np.int32)
    run_and_compare(H.host_case(w, q_to_kv=qmap), "head map")


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f32", 128), ("f32", 64)])
def test_head_dims(dtype, D):
    w = small(dtype=dtype, D=D)
    run_and_compare(H.host_case(w), f"{dtype} D={D}")


def test_arbitrary_orders_and_large_offsets():
    w = small(W=3, blocks=((129, 64, 10),))
    rng = np.random.default_rng(3)
    vb = np.stack([rng.permutation(4) for _ in range(3)]).astype(np.int32)
    vo = rng.integers(-10 ** 6, 10 ** 6, size=vb.shape).astype(np.int32)
    qp = rng.integers(0, 2 * 10 ** 6, size=3).astype(np.int32)
    run_and_compare(H.host_case(w, views=(vb, vo, qp)), "arbitrary offsets")


def test_many_problems_many_merges():
    rng = np.random.default_rng(9)
    P, W = 24, 3
    common = [int(x) for x in rng.integers(1, 700, size=P)]
    blocks = [[int(x) for x in rng.integers(0, 200, size=W)] for _ in range(P)]
    w = wl.Workload("many", "bf16", P, W, 8, 2, 128, 1e6, 1, common, blocks, seed=13)
    run_and_compare(H.host_case(w), "many problems")


def test_block_shared_by_two_problems():
    # one prompt block referenced by rows of two problems: 2 problems x 2 workers,
    # G = 4 -> 16 query heads on the shared block
    w = small(P=2, W=2, Hq=8, Hkv=2, common=(200, 50), blocks=((30, 40), (20, 10)))
    lens = w.block_lengths()
    vb, vo, qp = api.views_combined(lens, 2, 2)
    vb[2:, 0] = 0  # problem 1 also reads problem 0's common block
    vo[2:, 1:] += int(lens[0]) - int(lens[3])
    qp[2:] += int(lens[0]) - int(lens[3])
    run_and_compare(H.host_case(w, views=(vb, vo, qp)), "shared block")


def test_device_flags_without_faults():
    w = small()
    c = H.host_case(w)
    vb = c.view_block.copy()
    vb[0, 1] = 99  # no such block
    c.view_block = vb
    out, lse, s = c.run_gpu()
    assert s.device_flags() & 1
    c = H.host_case(w)
    bl = c.block_len.copy()
    bl[2] = 10 ** 6  # past the pool
    c.block_len = bl
    out, lse, s = c.run_gpu()
    assert s.device_flags() & 2
    # more query columns on a block than a tile serves (5 views x G = 8):
    # column groups, no flag, the oracle's results
    w = small(W=5, Hq=16, Hkv=2, blocks=((10, 10, 10, 10, 10),))
    out, lse, s = run_and_compare(H.host_case(w), "40 columns")
    assert s.device_flags() == 0


def test_deterministic_and_metadata_reuse():
    w = wl.qwq32b_w4()
    c0 = H.device_case(w, 0)
    c1 = H.device_case(w, 1)
    s = c0.session()
    a, la = s.decode(c0.q, c0.k, c0.v)
    b, lb = s.decode(c1.q, c1.k, c1.v)
    a2, la2 = s.decode(c0.q, c0.k, c0.v)
    torch.cuda.synchronize()
    assert torch.equal(a, a2) and torch.equal(la, la2)
    assert not torch.equal(a, b)
    ro, rl = c1.run_oracle()
    H.compare("bf16", b, lb, ro, rl, what="layer 1 through a reused session")


def test_maximum_sizes():
    # at the interface's limits at once: 256 blocks in the pool (HW_MAX_BLOCKS),
    # one row whose view holds 64 of them (HW_MAX_VIEW_BLOCKS, some empty),
    # 256 query heads over 8 kv heads (HW_MAX_Q_HEADS; G = 32 fills the
    # tile's 32 columns on every block), planned and unplanned
    rng = np.random.default_rng(23)
    nb, V, Hq, Hkv, D = 256, 64, 256, 8, 128
    lens = rng.integers(0, 90, size=nb).astype(np.int32)
    lens[[3, 17]] = 0
    w = wl.Workload("max", "bf16", 1, 1, Hq, Hkv, D, 1e6, 1, [0], [[0]], seed=5)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int32)
    cap = int(lens.sum()) + 8
    k = wl.to_storage(rng.standard_normal((Hkv, cap, D)), "bf16")
    v = wl.to_storage(rng.standard_normal((Hkv, cap, D)), "bf16")
    q = wl.to_storage(rng.standard_normal((1, Hq, D)), "bf16")
    chosen = np.sort(rng.choice(nb, size=V, replace=False))
    chosen[:2] = [3, 17]  # two empty blocks in the view
    chosen = np.sort(chosen)
    vb = chosen[None, :].astype(np.int32)
    vo = np.concatenate([[0], np.cumsum(lens[chosen])[:-1]])[None, :].astype(np.int32)
    qp = np.array([int(lens[chosen].sum())], np.int32)
    c = H.Case(w, H.from_storage_np(q, "bf16"), H.from_storage_np(k, "bf16"),
               H.from_storage_np(v, "bf16"), block_start=starts, block_len=lens, views=(vb, vo, qp))
    ro, rl = c.run_oracle()
    out, lse, s = c.run_gpu()
    assert s.device_flags() == 0
    H.compare("bf16", out, lse, ro, rl, what="maximum sizes")
    s.plan()
    out2, lse2 = s.decode_planned(c.q, c.k, c.v)
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16)) and torch.equal(lse2, lse)
