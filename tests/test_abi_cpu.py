"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and rejects bad arguments on the host before anything is enqueued.
Every call here fails its host checks, so none of them reaches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from concurrent_shared_kv_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return api.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "hogwild.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(hw_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(L):
    names = header_functions()
    assert len(names) >= 8, names
    for n in names:
        assert hasattr(L, n), n
    assert sorted(api.EXPORTS) == names


def test_status_strings(L):
    assert api.status_string(0) == "ok"
    assert "overlap" in api.status_string(-5)


def desc(**kw):
    base = dict(n_rows=2, n_q_heads=4, n_kv_heads=2, head_dim=64, n_blocks=3, max_view_blocks=3,
                cache_capacity=400, dtype=api.HW_F32, rope_theta=1e4, scale=0.125)
    base.update(kw)
    return api.make_desc(**base)


FAKE = 1 << 20  # a non-null, aligned address: never dereferenced, the calls fail first


def call_decode(d, **ptrs):
    p = dict(q=FAKE, k=FAKE, v=FAKE, bs=FAKE, bl=FAKE, vb=FAKE, vo=FAKE, qp=FAKE, qmap=None,
             out=FAKE, lse=None, ws=None, wsb=0)
    p.update(ptrs)
    return api.lib().hw_attn_decode(ctypes.byref(d), p["q"], p["k"], p["v"], p["bs"], p["bl"],
                                     p["vb"], p["vo"], p["qp"], p["qmap"], p["out"], p["lse"],
                                     p["ws"], p["wsb"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), -2), (dict(head_dim=0), -2), (dict(n_q_heads=5), -1),
    (dict(n_kv_heads=0), -1), (dict(dtype=7), -1), (dict(rope_theta=0.5), -1),
    (dict(rope_theta=float("nan")), -1), (dict(scale=float("inf")), -1),
    (dict(n_blocks=257), -2), (dict(max_view_blocks=65), -2), (dict(n_rows=-1), -1),
    (dict(n_rows=100, max_view_blocks=64), -2), (dict(n_q_heads=66, n_kv_heads=2), -2),
    (dict(cache_capacity=1 << 31), -2),
])
def test_decode_rejects_bad_desc(L, kw, status):
    assert call_decode(desc(**kw)) == status
    n = ctypes.c_size_t(0)
    assert L.hw_attn_decode_workspace_size(ctypes.byref(desc(**kw)), ctypes.byref(n)) == status


def test_decode_rejects_null_and_workspace(L):
    d = desc()
    assert call_decode(d, q=None) == -1
    assert call_decode(d, out=None) == -1
    assert call_decode(d, qp=None) == -1
    assert call_decode(d, vb=None) == -1
    assert call_decode(d, k=None) == -1
    assert call_decode(d, ws=None) == -3          # no workspace
    assert call_decode(d, ws=FAKE + 16) == -3     # not 256-byte aligned
    assert call_decode(desc(n_rows=0), q=None, out=None) == 0  # nothing to do


COMMIT = dict(dtype=api.HW_BF16, n_layers=2, n_kv_heads=8, head_dim=128, rope_theta=1e6,
              k_src=FAKE, v_src=FAKE * 64, src_capacity=1024, src_begin=0, n_tokens=512,
              k_dst=FAKE * 128, v_dst=FAKE * 256, dst_capacity=4096, dst_offset=0, pos_delta=7)


def call_commit(**kw):
    a = dict(COMMIT)
    a.update(kw)
    return api.lib().hw_block_commit(a["dtype"], a["n_layers"], a["n_kv_heads"], a["head_dim"],
                                     a["rope_theta"], a["k_src"], a["v_src"], a["src_capacity"],
                                     a["src_begin"], a["n_tokens"], a["k_dst"], a["v_dst"],
                                     a["dst_capacity"], a["dst_offset"], a["pos_delta"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=3), -1), (dict(n_kv_heads=0), -1), (dict(n_tokens=-1), -1),
    (dict(src_begin=-1), -1), (dict(head_dim=100), -2), (dict(head_dim=8), -2),
    (dict(rope_theta=1.0), -1), (dict(k_src=None), -1), (dict(k_dst=FAKE * 128 + 8), -1),
    # ranges leaving their pools
    (dict(src_begin=600), -4), (dict(dst_offset=3585), -4),
    # destination overlapping a source: same pool, overlapping token ranges
    (dict(k_dst=FAKE, src_capacity=4096, dst_capacity=4096, src_begin=100, dst_offset=300), -5),
    # same pool but different capacities (different layouts)
    (dict(k_dst=FAKE, dst_capacity=2048, dst_offset=1024), -5),
    # V destination inside the K source pool
    (dict(v_dst=FAKE + 4096), -5),
    # both destinations overlapping each other
    (dict(v_dst=FAKE * 128 + 1024), -5),
])
def test_commit_host_checks(L, kw, status):
    assert call_commit(**kw) == status


def test_commit_noop(L):
    assert call_commit(n_tokens=0) == 0
    assert call_commit(n_layers=0) == 0


def test_views_combined_matches_oracle(L):
    rng = np.random.default_rng(0)
    for P, W in [(1, 2), (1, 4), (3, 3), (16, 4), (2, 1)]:
        lens = rng.integers(0, 3000, size=P * (W + 1))
        got = api.views_combined(lens, P, W)
        want = oracle.combined_views(lens, P, W)
        for g, w in zip(got, want):
            assert np.array_equal(g, w)


def test_phase_table_source_is_integer_exact():
    # the fixed-point RoPE phase: p * F mod 2^64 as an angle in turns.  Checked
    # here on the host with Python integers against the double-precision angle
    # p * w mod 2pi (the oracle's own definition of the angle).
    import math
    from fractions import Fraction
    theta, D = 1e6, 128
    for i in (0, 1, 17, 63):
        w = theta ** (-2.0 * i / D)
        F = round(Fraction(w) / Fraction(2 * math.pi) % 1 * 2 ** 64) % 2 ** 64
        for p in (1, 7, 328, 65536 + 2048, -5):
            turns = ((p * F) % 2 ** 64) / 2 ** 64
            ang = (p * w) % (2 * math.pi)
            diff = (turns * 2 * math.pi - ang + math.pi) % (2 * math.pi) - math.pi
            assert abs(diff) < 1e-9, (i, p, diff)



def test_early_loads_flag_is_accepted_and_unknown_flags_are_not(L):
    # the flag passes the description checks: the call gets as far as its
    # null workspace (HW_ERR_WORKSPACE); an unknown bit is an invalid argument
    assert call_decode(desc(dtype=api.HW_BF16, head_dim=128, flags=api.HW_DESC_EARLY_LOADS)) == -3
    assert call_decode(desc(flags=api.HW_DESC_EARLY_LOADS)) == -3
    assert call_decode(desc(flags=64)) == -1


def test_trace_calls_are_absent_from_the_normal_build(L):
    # the layer timeline needs the HW_TRACE build; the normal library carries
    # no stamps and says so before touching the device
    dst = np.zeros((8, 160, 24), np.uint64)
    assert L.hw_trace_read(dst.ctypes.data) == -2   # HW_ERR_UNSUPPORTED
    assert L.hw_trace_clear() == -2
