"""Host logic of the verification step (no GPU): the attention split count
chosen when the tree is built in one launch and the attention streams its
prefix beside it."""
from speculative_decoding_eagle_gb300 import step as S


def test_overlap_splits_takes_the_fewest_splits_that_end_before_the_tree():
    # 7B heads, prefix 1024 (16 + 1 tiles), depth 6: one split streams 17
    # tiles in 23.8 us < 0.8 * 6 * 7 us; 32 blocks fit in 128 free slots
    assert S.overlap_splits(17, 6, 4, 32, 128) == 1
    # 13B heads, prefix 4096 (64 + 1 tiles): 3 splits of 22 tiles (30.8 us), 120 blocks
    assert S.overlap_splits(65, 6, 6, 40, 128) == 3


def test_overlap_splits_falls_back_to_the_standalone_plan():
    # 70B GQA, prefix 8192: 5 splits would stream in time, but 240 blocks do not fit in 160 slots
    assert S.overlap_splits(130, 8, 5, 48, 160) == 5
    # a prefix too long for any split count within the standalone plan's
    assert S.overlap_splits(1000, 2, 8, 4, 1000) == 8
    # no room beside the tree at all
    assert S.overlap_splits(17, 6, 4, 32, 0) == 4


def test_overlap_splits_never_exceeds_the_standalone_plan():
    for tiles in (1, 5, 17, 65, 257):
        for auto in (1, 2, 4, 8):
            s = S.overlap_splits(tiles, 6, auto, 8, 1000)
            assert 1 <= s <= auto
