"""The token-tile rule against the candle page's printed decisions (tests/golden/candle_pr4056_tile_rule.json):
the 64-token tile is used only where it pads no more tokens than the 32-token tile; this library extends
the same rule to a 128-token tile."""
import json
import os

import pytest

import weight_quantized_matmul_fly_gb300 as qmm

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "candle_pr4056_tile_rule.json")))


def pad(M, T):
    return -(-M // T) * T - M


def two_tile(M):
    """The library's rule restricted to the page's two tiles {32, 64}. A pick of 128 implies the 64-tile pads
    no more than the 32-tile too (its padding lies between theirs), so it maps to 64."""
    t = qmm.qmm_pick_tile(M)
    return 64 if t == 128 else t


@pytest.fixture(scope="module", autouse=True)
def _lib():
    qmm.build()


def test_page_table_chosen_column():
    for M, chosen in GOLD["chosen"]:
        assert two_tile(M) == chosen, M


def test_pinned_counts_and_strict_rule():
    s = GOLD["strict_rule_failure"]
    assert two_tile(s["tokens"]) == s["correct"]
    # the strict form (< instead of <=) never picks the wider tile, so it disagrees exactly where the page says
    assert s["strict"] == 32


def test_three_tile_rule():
    want = {2: 32, 32: 32, 33: 64, 64: 64, 96: 32, 100: 128, 128: 128, 136: 32, 2048: 128}
    for M in GOLD["pinned_counts"]:
        assert qmm.qmm_pick_tile(M) == want[M], M


def test_never_pads_more_than_32_tile():
    for M in range(1, 5000):
        T = qmm.qmm_pick_tile(M)
        assert T in (32, 64, 128)
        assert pad(M, T) == pad(M, 32)
        # and it is the largest such tile
        for bigger in (64, 128):
            if bigger > T:
                assert pad(M, bigger) != pad(M, 32)


def test_up_to_32_tokens_is_32():
    assert all(qmm.qmm_pick_tile(M) == 32 for M in range(1, 33))
