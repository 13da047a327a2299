"""Host logic of bench.py that decides how steps are timed (no GPU needed).

Timing rule: between timed steps either flush L2 or use inputs larger than
L2.  Block timing (K steps back to back between one pair of events, no flush)
is chosen only when the step's inputs exceed L2; otherwise every step is
preceded by a flush."""
import os
import sys
from types import SimpleNamespace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

L2 = 136 * 10**6


@pytest.fixture(autouse=True)
def fake_l2(monkeypatch):
    monkeypatch.setattr(bench, "_l2_bytes", lambda dev: L2)


def _mode(timing, input_bytes):
    return bench._timing_mode(SimpleNamespace(timing=timing), input_bytes, None)


def test_auto_picks_block_only_for_inputs_larger_than_l2():
    x_training_profile = 2 * 4096 * 20480          # 168 MB of BF16 X
    x_edge = 2 * 1000 * 20480                      # 41 MB
    assert _mode("auto", x_training_profile) == "block"
    assert _mode("auto", x_edge) == "flushed"
    assert _mode("auto", L2) == "flushed"          # not larger: flush


def test_explicit_modes():
    assert _mode("flushed", 10 * L2) == "flushed"
    assert _mode("block", L2 + 1) == "block"
    with pytest.raises(SystemExit):
        _mode("block", L2 // 2)                     # would time L2-resident inputs


def test_l2_note_names_the_rule_used():
    assert "not flushed" in bench._l2_note("block", 2 * L2, None)
    assert "flushed before every timed step" in bench._l2_note("flushed", 1, None)
