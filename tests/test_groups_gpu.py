"""GPU parity of column groups against the float64 oracle, through the C ABI.
A tile serves 32 query columns (view references x GQA group); a block named
by more references is read once per group of 32 // G of them (key design 1
of the Hogwild! notes: every worker attends the common block, however many
there are).  Covered: eight workers at G = 5 (40 columns on every block),
the four-worker QwQ-32B shape with two-token query chunks (eight rows on the
common block), one reference per group (G = 32), the SIMT kernel, appends and
E4M3 caches over grouped blocks, and the split's export against the oracle's."""
import numpy as np
import pytest
import torch

import oracle
from concurrent_shared_kv_gb300 import api
from concurrent_shared_kv_gb300 import workloads as wl
from tests import harness as H
from tests.test_append_gpu import check_append_decode, last_position_appends, new_tokens
from tests.test_fp8_gpu import Fp8Case
from tests.test_limits_gpu import check as check_limited, chunk_case
from tests.test_parity_gpu import run_and_compare, small
from tests.test_split_gpu import check_split

pytestmark = pytest.mark.gpu


def planned(c):
    s = c.session()
    s.plan()
    out, lse = s.decode_planned(c.q, c.k, c.v)
    torch.cuda.synchronize()
    assert s.device_flags() == 0
    return out, lse


def test_eight_workers_g5_small_ragged():
    # 40 columns on every block: two groups (6 + 2 references); ragged tiles,
    # an empty worker block and blocks shorter than a tile
    w = small(P=2, W=8, Hq=40, Hkv=8, common=(3000, 77),
              blocks=((129, 64, 1, 128, 0, 33, 300, 256), (5, 200, 128, 127, 1, 0, 64, 900)))
    c = H.host_case(w)
    out, lse, s = run_and_compare(c, "W8 G5 unplanned")
    assert s.device_flags() == 0
    ro, rl = c.run_oracle()
    po, pl = planned(c)
    H.compare("bf16", po, pl, ro, rl, what="W8 G5 planned")
    check_split(c, "W8 G5")


def test_eight_workers_g5_full_size():
    # the QwQ-32B shape with eight workers, 16K common tokens: every row whole
    w = wl.qwq32b_w8()
    c = H.device_case(w, 0)
    ro, rl = c.run_oracle()
    po, pl = planned(c)
    H.compare("bf16", po, pl, ro, rl, what="W8 full planned")
    out, lse, s = c.run_gpu()
    assert s.device_flags() == 0
    H.compare("bf16", out, lse, ro, rl, what="W8 full unplanned")
    got = check_split(c, "W8 full")
    assert set(got[:, 12:15][got[:, 2:3] > np.arange(3)].tolist()) == {0, 1}


def test_qwq32b_w4_chunk_2():
    # two-token chunks: 8 rows name the common block (40 columns, two groups)
    # and each worker block (its own two rows see it up to their own token)
    w = wl.qwq32b_w4()
    c, vl = chunk_case(w, 2, device=True)
    assert c.view_block.shape[0] == 8
    check_limited(c, vl, "C3 chunk 2")


def test_one_reference_per_group():
    # G = 32: a tile's columns are one reference's q heads, so every reference
    # to a block is its own group (three readers of each block)
    w = small(P=1, W=3, Hq=64, Hkv=2, common=(700,), blocks=((129, 64, 300),))
    c = H.host_case(w)
    run_and_compare(c, "G32 unplanned")
    ro, rl = c.run_oracle()
    po, pl = planned(c)
    H.compare("bf16", po, pl, ro, rl, what="G32 planned")


def test_simt_kernel_groups():
    # the f32 SIMT kernel (head_dim 64): nine workers at G = 8, three groups
    # (4 + 4 + 1 references) on every block
    w = small(dtype="f32", P=1, W=9, Hq=16, Hkv=2, D=64, common=(300,),
              blocks=((65, 64, 1, 0, 130, 7, 64, 200, 3),))
    c = H.host_case(w)
    out, lse, s = run_and_compare(c, "SIMT groups")
    assert s.device_flags() == 0


def test_appends_into_grouped_blocks():
    # the new token of a worker lies in a tile that both groups read, possibly
    # on different CTAs: each writes it before its own copy of the tile
    w = small(P=1, W=8, Hq=40, Hkv=8, common=(2000,),
              blocks=((129, 64, 1, 128, 300, 33, 257, 256),))
    c = H.device_case(w, 0)
    ab, ap = last_position_appends(c, skip=(3,))
    kn, vn = new_tokens(w, 5)
    check_append_decode(c, ab, ap, kn, vn, "appends W8 G5")


def test_e4m3_grouped_blocks():
    w = small(P=1, W=8, Hq=40, Hkv=8, common=(3000,),
              blocks=((129, 64, 1, 128, 300, 33, 257, 256),))
    f = Fp8Case(H.device_case(w, 0))
    out, lse, s = f.run()
    ro, rl = f.oracle()
    H.compare("bf16", out, lse, ro, rl, what="E4M3 W8 G5")


def test_too_many_references_flagged_without_faults():
    # 128 rows, each naming block 0 twice: 256 references to one block, more
    # than a plan ranks; the block is skipped and HW_DEV_TOO_MANY_REFS set
    w = small(P=32, W=4, Hq=8, Hkv=2, common=(100,) * 32, blocks=((10, 10, 10, 10),) * 32)
    c = H.host_case(w)
    vb = c.view_block.copy()
    vb[:, 0] = 0
    vb[:, 1] = 0
    c.view_block = vb
    out, lse, s = c.run_gpu()
    assert s.device_flags() & 8
