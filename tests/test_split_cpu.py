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
    want = np.zeros((3, 15), np.int64)
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
    want = np.zeros((4, 15), np.int64)
    want[0, :3] = (0, 2, 2)
    want[0, 3:5], want[0, 9:11] = (0, 128), (1, 2)          # CTA 0's share of block 0
    want[1, :3] = (2, 4, 2)
    want[1, 3:5], want[1, 9:11] = (256, 1000), (3, 3)       # the rest of block 0, block 2 whole
    want[2, :3] = want[3, :3] = (4, 4, 0)
    assert np.array_equal(got, want), got


def test_split_worked_by_hand_column_groups():
    # one kv head of G = 16 q heads: a tile serves 32 columns, i.e. two view
    # references.  Block 0 (256 tokens, 2 tiles) is referenced by three rows,
    # so its references form groups {0, 1} and {2}; block 1 (128 tokens) by
    # one.  Units (block, group, tile): (0,0,0) (0,0,1) (0,1,0) (0,1,1) (1,0,0);
    # UH = 5, NSH = 3 segments.  Weights (a segment start weighs 2):
    # 0 + 2*1 = 2, 3; 2 + 2*2 = 6, 7; 4 + 2*3 = 10.  W = 5 + 2*3 = 11,
    # C = min(3, 11 // 3) = 3; CTA bounds 0, 3, 7, 11: CTA 0 takes unit 0,
    # CTA 1 units 1, 2 and CTA 2 units 3, 4.
    got = oracle.stream_k_split(block_start=[0, 1000], block_len=[256, 128],
                                view_block=[[0, 1], [0, -1], [0, -1]], n_q_heads=16,
                                n_kv_heads=1, grid=3)
    want = np.zeros((3, 15), np.int64)
    want[0, :3] = (0, 1, 1)
    want[0, 3], want[0, 9], want[0, 12] = 0, 3, 0
    want[1, :3] = (1, 3, 2)
    want[1, 3:5], want[1, 9:11], want[1, 12:14] = (128, 0), (3, 3), (0, 1)
    want[2, :3] = (3, 5, 2)
    want[2, 3:5], want[2, 9:11], want[2, 12:14] = (128, 1000), (3, 3), (1, 0)
    assert np.array_equal(got, want), got


def test_split_groups_read_every_tile_once_per_group():
    # G = 5: six references a group.  Eight rows on a common block of 1000
    # tokens (8 tiles) make two groups, so the common block's 8 tiles appear
    # twice per kv head; each row's own block one group.
    lens = [1000] + [200] * 8
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).tolist()
    vb = np.array([[0, 1 + r] for r in range(8)], np.int32)
    got = oracle.stream_k_split(starts, lens, vb, 40, 8, grid=152)
    U = (8 * 2 + 8 * 2) * 8
    assert got[:, 1].max() == U and got[0, 0] == 0
    assert np.all(got[1:, 0] == got[:-1, 1])
    # a CTA's first tiles: a group index below the block's group count
    for c in range(152):
        for i in range(got[c, 2]):
            row, g = got[c, 3 + i], got[c, 12 + i]
            assert g < (2 if row < 1000 else 1)


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
