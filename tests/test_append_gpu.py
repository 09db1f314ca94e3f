"""GPU parity of the fused KV append (hw_attn_plan_append +
hw_attn_append_decode_planned, through the C ABI) against the float64 oracle:
the oracle appends each row's new token (its key rotated at its block-local
position) and then decodes; the kernel must give the same outputs and leave
the same cache - values and untouched rows bit for bit, appended keys within
one bf16 unit of the exact rotation (fp32 arithmetic, one rounding)."""
import numpy as np
import pytest
import torch

import oracle
from concurrent_shared_kv_gb300 import workloads as wl
from tests import harness as H
from tests.test_parity_gpu import small

pytestmark = pytest.mark.gpu


def new_tokens(w, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    shape = (w.n_rows, w.n_kv_heads, w.head_dim)
    kn = torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)
    vn = torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)
    return kn, vn


def last_position_appends(c, skip=()):
    """Row r = (p, w) appends its token at the end of its own block (block_len
    already counts it); rows in `skip` and rows with an empty block append
    nothing."""
    w = c.w
    ab = np.full(w.n_rows, -1, np.int32)
    ap = np.zeros(w.n_rows, np.int32)
    for r in range(w.n_rows):
        p, wk = divmod(r, w.n_workers)
        b = p * (w.n_workers + 1) + 1 + wk
        if r in skip or c.block_len[b] == 0:
            continue
        ab[r], ap[r] = b, c.block_len[b] - 1
    return ab, ap


def check_append_decode(c, ab, ap, kn, vn, what, rows=None):
    k0, v0 = H.to_storage_np(c.k), H.to_storage_np(c.v)
    s = c.session()
    s.plan_append(ab, ap)
    out, lse = s.append_decode_planned(c.q, kn, vn, c.k, c.v)
    torch.cuda.synchronize()
    assert s.device_flags() == 0
    w = c.w
    kd, vd, exact = oracle.get().append_tokens(
        dtype=oracle.BF16, rope_theta=w.rope_theta, k_cache=k0, v_cache=v0,
        k_new=H.to_storage_np(kn), v_new=H.to_storage_np(vn), block_start=c.block_start,
        append_block=ab, append_pos=ap, want_exact=True)
    # the cache: values and every untouched key row bit for bit
    kg, vg = H.to_storage_np(c.k), H.to_storage_np(c.v)
    assert np.array_equal(vg, vd), what
    touched = np.zeros(kg.shape[1], bool)
    for r in exact:
        touched[c.block_start[ab[r]] + ap[r]] = True
    assert np.array_equal(kg[:, ~touched], kd[:, ~touched]), what
    for r, ex in exact.items():
        got = wl.storage_to_f64(kg[:, c.block_start[ab[r]] + ap[r]], "bf16")
        src = wl.storage_to_f64(H.to_storage_np(kn)[r], "bf16")
        half = w.head_dim // 2
        mag = np.abs(src) + np.abs(np.concatenate([src[..., half:], src[..., :half]], -1))
        assert (np.abs(got - ex) <= np.abs(ex) * 2.0 ** -8 + mag * 2.0 ** -20).all(), (what, r)
    # the decode saw the new tokens
    ro, rl = oracle.get().attn_decode(
        q=H.to_storage_np(c.q), k_cache=kd, v_cache=vd, block_start=c.block_start,
        block_len=c.block_len, view_block=c.view_block, view_offset=c.view_offset, q_pos=c.q_pos,
        n_kv_heads=w.n_kv_heads, rope_theta=w.rope_theta, scale=w.scale, dtype=oracle.BF16,
        rows=rows)
    H.compare("bf16", out, lse, ro, rl, rows=rows, what=what)
    # the same plan without the append reads the same cache: the same result
    out2, lse2 = s.decode_planned(c.q, c.k, c.v)
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16)), what
    assert torch.equal(lse2, lse), what
    return s


def test_append_decode_small_edges():
    # worker blocks 129 (token in the second tile), 64, 1 (position 0); 128
    # (last row of a tile), an empty block, 33; row 1 appends nothing
    w = small(P=2, W=3, common=(300, 77), blocks=((129, 64, 1), (128, 0, 33)))
    c = H.host_case(w)
    ab, ap = last_position_appends(c, skip=(1,))
    assert sorted(ap[ab >= 0].tolist()) == [0, 32, 127, 128]
    kn, vn = new_tokens(w, 5)
    check_append_decode(c, ab, ap, kn, vn, "append small")


def test_append_decode_qwq32b_w4_layer():
    w = wl.qwq32b_w4()
    c = H.device_case(w, 0)
    ab, ap = last_position_appends(c)
    kn, vn = new_tokens(w, 6)
    check_append_decode(c, ab, ap, kn, vn, "append C3 layer 0")


def test_append_position_outside_its_block_is_reported_and_skipped():
    w = small(P=1, W=3, common=(300,), blocks=((129, 64, 40),))
    c = H.host_case(w)
    ab, ap = last_position_appends(c)
    ap[1] = c.block_len[ab[1]]  # one past the block's length: the next block's first row
    kn, vn = new_tokens(w, 7)
    k0 = H.to_storage_np(c.k)
    s = c.session()
    s.plan_append(ab, ap)
    s.append_decode_planned(c.q, kn, vn, c.k, c.v)
    torch.cuda.synchronize()
    assert s.device_flags() & 2  # HW_DEV_BAD_RANGE
    kg = H.to_storage_np(c.k)
    bad_row = c.block_start[ab[1]] + ap[1]
    assert np.array_equal(kg[:, bad_row], k0[:, bad_row])  # not written
    good_row = c.block_start[ab[0]] + ap[0]
    assert not np.array_equal(kg[:, good_row], k0[:, good_row])  # the others were


def test_append_decode_serving_ragged_uses_the_scan_beyond_the_plan_list():
    # 16 problems x 4 workers: CTAs that cross many short worker blocks own
    # more new tokens than the plan lists and find the rest by scanning
    w = wl.serve_ragged()
    c = H.device_case(w)
    ab, ap = last_position_appends(c)
    kn, vn = new_tokens(w, 8)
    check_append_decode(c, ab, ap, kn, vn, "append serving ragged", rows=list(range(0, 4)) + list(range(60, 64)))


def test_append_decode_beyond_the_plan_list():
    # a long common block makes each CTA's share of the split large, so the
    # CTAs that cross the 30 one-to-three-token worker blocks own up to 11 new
    # tokens (host replica of the split: four CTAs above the plan's list of 8)
    w = wl.Workload("scan", "bf16", 1, 30, 2, 2, 128, 1e6, 1, [400000],
                    [[1 + (i % 3) for i in range(30)]], seed=21)
    c = H.device_case(w)
    ab, ap = last_position_appends(c)
    kn, vn = new_tokens(w, 9)
    check_append_decode(c, ab, ap, kn, vn, "append beyond the list", rows=[0, 13, 29])
