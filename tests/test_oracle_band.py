"""Pins for the oracle's band predicate: the hand-derived visible sets of
tests/golden/window_visible_sets.txt (OpenVINO PR #37423, "Sliding window"; tract PR #2645,
"What changed") and the set construction of the pure-Python brute force."""
import os

import pytest

import brute_force
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "window_visible_sets.txt")


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, tail = line.split(":")
            past, curr, window, causal, i = map(int, head.split())
            rows.append((past, curr, window, causal, i, sorted(map(int, tail.split()))))
    return rows


@pytest.mark.parametrize("row", _golden_rows())
def test_visible_sets_match_golden(row):
    past, curr, window, causal, i, want = row
    total = past + curr
    got = [j for j in range(total + 4) if oracle.visible(past + i, j, total, bool(causal), window)]
    assert got == want


def test_visible_sets_match_brute_force_exhaustive():
    for past in range(0, 9):
        for curr in range(1, 4):
            for window in (-1, 1, 2, 3, 5, 50):
                for causal in (0, 1):
                    for i in range(curr):
                        total = past + curr
                        got = {j for j in range(-2, total + 3)
                               if oracle.visible(past + i, j, total, bool(causal), window)}
                        assert got == brute_force.visible_set(past, curr, i, window, causal)


def test_window_one_is_self_only_and_large_window_is_causal():
    for past in range(0, 20, 3):
        for curr in (1, 2, 3):
            total = past + curr
            for i in range(curr):
                qa = past + i
                assert [j for j in range(total) if oracle.visible(qa, j, total, True, 1)] == [qa]
                big = [j for j in range(total) if oracle.visible(qa, j, total, True, total + 5)]
                nowin = [j for j in range(total) if oracle.visible(qa, j, total, True, -1)]
                assert big == nowin == list(range(qa + 1))


def test_sequence_status():
    # valid; negative past; overflowing capacity; separate past too long; rope out of range
    assert oracle.sequence_status(10, 1, 16, 16, False, False, 0) == 0
    assert oracle.sequence_status(-1, 1, 16, 16, False, False, 0) == 1
    assert oracle.sequence_status(15, 2, 16, 16, False, False, 0) == 1
    assert oracle.sequence_status(15, 1, 16, 16, False, False, 0) == 0
    assert oracle.sequence_status(9, 1, 8, 16, True, False, 0) == 1
    assert oracle.sequence_status(9, 1, 8, 16, False, False, 0) == 0
    assert oracle.sequence_status(10, 2, 16, 16, False, True, 11) == 2
    assert oracle.sequence_status(10, 2, 16, 16, False, True, 12) == 0
