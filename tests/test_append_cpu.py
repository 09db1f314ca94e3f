"""The fused KV append without a GPU: the oracle's append pinned against
what the cache convention fixes (a key stored at block-local position p is the
raw key rotated by p: position 0 is a bit copy, rotating the stored key back
by -p returns the raw key, the value is a bit copy, nothing else moves), and
the C ABI's argument checks, which run before anything is enqueued."""
import numpy as np
import pytest

import oracle
from concurrent_shared_kv_gb300 import api
from concurrent_shared_kv_gb300 import workloads as wl

THETA = 1e6


def caches(dtype, Hkv=2, cap=50, D=128, seed=3):
    rng = np.random.default_rng(seed)
    k = wl.to_storage(rng.standard_normal((Hkv, cap, D)), dtype)
    v = wl.to_storage(rng.standard_normal((Hkv, cap, D)), dtype)
    kn = wl.to_storage(rng.standard_normal((3, Hkv, D)), dtype)
    vn = wl.to_storage(rng.standard_normal((3, Hkv, D)), dtype)
    return k, v, kn, vn


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_oracle_append_stores_the_key_at_its_block_position(dtype):
    odt = oracle.F32 if dtype == "f32" else oracle.BF16
    k, v, kn, vn = caches(dtype)
    starts = np.array([0, 20, 30, 40], np.int32)  # four blocks in one pool
    blocks = np.array([1, -1, 3], np.int32)  # row 1 appends nothing
    pos = np.array([7, 0, 0], np.int32)
    kd, vd, exact = oracle.get().append_tokens(dtype=odt, rope_theta=THETA, k_cache=k, v_cache=v,
                                               k_new=kn, v_new=vn, block_start=starts,
                                               append_block=blocks, append_pos=pos, want_exact=True)
    rows = {0: 20 + 7, 2: 40 + 0}
    touched = np.zeros(k.shape[1], bool)
    touched[list(rows.values())] = True
    assert np.array_equal(kd[:, ~touched], k[:, ~touched])  # nothing else moves
    assert np.array_equal(vd[:, ~touched], v[:, ~touched])
    for r, row in rows.items():
        assert np.array_equal(vd[:, row], vn[r])  # the value as it is
    # position 0: the raw key, bit for bit
    assert np.array_equal(kd[:, 40], kn[2])
    # position 7: rotating the stored key back by -7 returns the raw key (to the
    # storage rounding), and the stored key is the rounded exact rotation
    raw = wl.storage_to_f64(kn[0], dtype)
    back = np.stack([oracle.get().rope(wl.storage_to_f64(kd[h, 27], dtype), THETA, -7.0)
                     for h in range(k.shape[0])])
    tol = 1e-6 if dtype == "f32" else 2.0 ** -7
    assert np.max(np.abs(back - raw)) <= tol * np.max(np.abs(raw))
    assert np.max(np.abs(wl.storage_to_f64(kd[:, 27], dtype) - exact[0])) <= tol * np.max(np.abs(exact[0]))
    # and it is not the unrotated key: a dropped rotation would pass the copy checks
    assert np.max(np.abs(wl.storage_to_f64(kd[:, 27], dtype) - raw)) > 0.1


# ---------------------------------------------------------------------------
# C ABI checks (no launch)
# ---------------------------------------------------------------------------

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


def test_plan_append_needs_both_arrays_and_the_tensor_core_path():
    # (these checks come before the workspace's, so no device is needed)
    d = desc()
    assert status(api.attn_plan_append, d, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 0) == -1
    assert status(api.attn_plan_append, d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 0) == -1
    assert status(api.attn_plan_append, desc(dtype=api.HW_F32), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                  FAKE, FAKE, 0) == -2


def test_append_decode_checks():
    d = desc()
    call = lambda dd, kn=FAKE, vn=FAKE: status(api.attn_append_decode_planned, dd, FAKE, kn, vn,
                                              FAKE, FAKE, FAKE, None, FAKE, 0)
    assert call(d, kn=None) == -1
    assert call(d, vn=None) == -1
    assert call(d, kn=FAKE + 2) == -1          # 16-byte loads of the new rows
    assert call(desc(dtype=api.HW_F32)) == -2  # bf16 head_dim 128 only
    assert call(desc(head_dim=64)) == -2
