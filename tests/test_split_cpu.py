"""The oracle's restatement of the work split, pinned by a case worked out by
hand from the definition and by invariants that any correct split keeps."""
import numpy as np

import oracle


def test_split_worked_by_hand():
    # one kv head (one q head), blocks of 256 and 128 tokens (2 and 1 tiles),
    # both viewed.  Weights: block 0's tiles at 0 + 3*1 + t = 3, 4; block 1's
    # tile at 2 + 3*2 = 8.  W = 3 + 3*2 = 9, C = min(3, 9 // 4) = 2 CTAs:
    # CTA 0 takes weights [0, 4) -> unit 0; CTA 1 [4, 9) -> units 1, 2; CTA 2 none.
    got = oracle.stream_k_split(block_start=[0, 1000], block_len=[256, 128],
                                view_block=[[0, 1]], n_q_heads=1, n_kv_heads=1, grid=3,
                                seg_weight=3)
    want = np.zeros((3, 12), np.int64)
    want[0, :3] = (0, 1, 1)
    want[0, 3], want[0, 6], want[0, 9] = 0, 0, 3            # row 0, head 0, starts and ends here
    want[1, :3] = (1, 3, 2)
    want[1, 3:5], want[1, 6:8], want[1, 9:11] = (128, 1000), (0, 0), (3, 3)
    want[2, :3] = (3, 3, 0)
    assert np.array_equal(got, want), got


def test_split_worked_by_hand_segment_weight_2():
    # the kernel's weights (a segment start weighs 2 tiles): one kv head, blocks
    # of 384 and 128 tokens (3 and 1 tiles), and a third of 128 tokens no view
    # references.  Weights: block 0's tiles at 0 + 2*1 + t = 2, 3, 4; block 1's
    # tile at 3 + 2*2 = 7.  W = 4 + 2*2 = 8, C = min(4, 8 // 3) = 2 CTAs:
    # CTA 0 takes weights [0, 4) -> units 0, 1; CTA 1 [4, 8) -> units 2, 3.
    # Flags: 1 = the CTA's first tile of the segment, 2 = its last one.
    got = oracle.stream_k_split(block_start=[0, 500, 1000], block_len=[384, 128, 128],
                                view_block=[[0, 2]], n_q_heads=1, n_kv_heads=1, grid=4)
    want = np.zeros((4, 12), np.int64)
    want[0, :3] = (0, 2, 2)
    want[0, 3:5], want[0, 9:11] = (0, 128), (1, 2)          # CTA 0's share of block 0
    want[1, :3] = (2, 4, 2)
    want[1, 3:5], want[1, 9:11] = (256, 1000), (3, 3)       # the rest of block 0, block 2 whole
    want[2, :3] = want[3, :3] = (4, 4, 0)
    assert np.array_equal(got, want), got


def test_split_invariants():
    rng = np.random.default_rng(4)
    lens = rng.integers(0, 3000, size=9).tolist()
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).tolist()
    vb = np.array([[0, 1, 2, 3], [0, 4, 5, -1], [6, 7, 8, 2]], np.int32)
    G, Hkv = 4, 3
    got = oracle.stream_k_split(starts, lens, vb, G * Hkv, Hkv, grid=152)
    tiles = [(l + 127) // 128 for l in lens]
    U = sum(tiles) * Hkv
    u0, u1 = got[:, 0], got[:, 1]
    assert u0[0] == 0 and u1[-1] == U and np.all(u0[1:] == u1[:-1])
    # every working CTA owns a unit; the first tiles lie inside their blocks
    C = np.sum(u1 > u0)
    assert np.all(u1[:C] > u0[:C])
    for c in range(C):
        for i in range(got[c, 2]):
            row = got[c, 3 + i]
            b = max(bb for bb in range(len(lens)) if starts[bb] <= row and tiles[bb] > 0)
            assert (row - starts[b]) % 128 == 0 and row - starts[b] < lens[b]
