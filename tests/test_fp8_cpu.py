"""E4M3 caches without a GPU: the C ABI's argument checks (which run before
anything is enqueued) and the E4M3 packing of the synthetic inputs."""
import numpy as np

import oracle
from concurrent_shared_kv_gb300 import api
from concurrent_shared_kv_gb300 import workloads as wl

FAKE = 1 << 20
F8 = api.HW_FP8_E4M3


def desc(**kw):
    base = dict(n_rows=2, n_q_heads=4, n_kv_heads=2, head_dim=128, n_blocks=3, max_view_blocks=3,
                cache_capacity=400, dtype=F8, rope_theta=1e6, scale=0.088)
    base.update(kw)
    return api.make_desc(**base)


def status(fn, *args, **kw):
    try:
        return fn(*args, **kw)
    except api.HwError as e:
        return e.status


def test_fp8_append_entry_checks():
    call = lambda d, ks=FAKE, vs=FAKE: status(api.attn_append_decode_planned_fp8, d, FAKE, FAKE, FAKE,
                                              FAKE, FAKE, ks, vs, FAKE, None, FAKE, 0)
    assert call(desc(), ks=None) == -1
    assert call(desc(dtype=api.HW_BF16)) == -1
    assert call(desc(flags=api.HW_DESC_VIEW_LIMITS)) == -2


def test_fp8_decode_entry_checks():
    call = lambda d, ks=FAKE, vs=FAKE: status(api.attn_decode_planned_fp8, d, FAKE, FAKE, FAKE, ks, vs,
                                              FAKE, None, FAKE, 0)
    assert call(desc(), ks=None) == -1
    assert call(desc(), vs=None) == -1
    assert call(desc(dtype=api.HW_BF16)) == -1  # another dtype: the plain planned call
    assert call(desc(head_dim=64)) == -2


def test_fp8_descriptor_is_refused_by_the_other_decode_calls():
    d = desc()
    assert status(api.attn_decode, d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                  FAKE, 0) == -2
    assert status(api.attn_decode_noalloc, d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                  None) == -2
    assert status(api.attn_decode_planned, d, FAKE, FAKE, FAKE, FAKE, None, FAKE, 0) == -2
    # (E4M3 with appends is planned by hw_attn_plan_append: past its checks)
    assert status(api.attn_plan_append, d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                  0) not in (-1, -2)
    assert status(api.attn_append_decode_planned, d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                  FAKE, 0) == -2
    # E4M3 with view limits is planned by hw_attn_plan_limited: the call gets
    # past the descriptor and argument checks (and stops at the workspace,
    # which needs a device)
    assert status(api.attn_plan_limited, desc(flags=api.HW_DESC_VIEW_LIMITS), FAKE, FAKE, FAKE,
                  FAKE, FAKE, FAKE, FAKE, 0) not in (-1, -2)


def test_fp8_commit_checks():
    KS, VS, KD, VD = 1 << 30, 2 << 30, 3 << 30, 4 << 30
    c = lambda D, ks=KS: status(api.block_commit, F8, 1, 8, D, 1e6, ks, VS, 1000, 0, 10, KD, VD,
                                1000, 100, 100)
    assert c(16) == -2        # head_dim: a multiple of 32 (two 16-code chunks per half row)
    assert c(128, ks=KS + 8) == -1  # 16-byte aligned pools


def test_e4m3_packing_of_the_inputs():
    # one scale per kv head, max |x| / 448; every decoded value within half
    # an E4M3 step of the scaled input
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 40, 32)) * np.array([1.0, 0.01, 50.0])[:, None, None]
    codes, scale = wl.e4m3_pack(x)
    assert np.allclose(scale, np.abs(x).reshape(3, -1).max(1) / 448, rtol=1e-6)
    z = x / scale[:, None, None]
    got = wl.e4m3_values(codes)
    assert np.max(np.abs(got)) <= 448
    half = np.maximum(np.abs(z), 2.0 ** -6) * 2.0 ** -4
    assert np.all(np.abs(got - z) <= half * 1.0001)
    o = oracle.get()
    assert all(o.e4m3_to_double(int(b)) == g for b, g in zip(codes.ravel()[:500], got.ravel()[:500]))


def test_oracle_e4m3_append():
    # the new token's key rotated at its position, divided by the head scale,
    # rounded to the nearest code; position 0 and power-of-two scales: the
    # codes of the scaled raw values; a rotated key decodes (x scale) back,
    # rotated by -p, to the raw key within E4M3's half-step
    o = oracle.get()
    rng = np.random.default_rng(3)
    Hkv, D = 2, 16
    raw = rng.standard_normal((2, Hkv, D))
    kn = wl.to_storage(raw, "bf16")
    vn = wl.to_storage(raw[::-1].copy(), "bf16")
    k = np.zeros((Hkv, 40, D), np.uint8)
    v = np.zeros_like(k)
    ks, vs = np.array([0.5, 2.0]), np.array([0.25, 1.0])
    kd, vd, ex = oracle.append_tokens_e4m3(o, rope_theta=1e4, k_cache=k, v_cache=v, k_new=kn,
                                          v_new=vn, k_scale=ks, v_scale=vs, block_start=[0, 20],
                                          append_block=[0, 1], append_pos=[0, 9])
    kb, vb_ = wl.storage_to_f64(kn, "bf16"), wl.storage_to_f64(vn, "bf16")
    for h in range(Hkv):
        assert [o.e4m3_from_double(x / ks[h]) for x in kb[0, h]] == kd[h, 0].tolist()
        assert [o.e4m3_from_double(x / vs[h]) for x in vb_[1, h]] == vd[h, 29].tolist()
        back = o.rope(wl.e4m3_values(kd[h, 29]) * ks[h], 1e4, -9.0)
        step = (np.abs(kb[1, h]) + 2.0 ** -6 * ks[h]) * 2.0 ** -3
        assert np.all(np.abs(back - kb[1, h]) <= np.max(step) * 2)
    untouched = np.ones(40, bool)
    untouched[[0, 29]] = False
    assert not kd[:, untouched].any() and not vd[:, untouched].any()
