"""Clock arithmetic of the oracle against the values the pages print."""
import json
import os

import pytest

from oracle import clock


@pytest.fixture(scope="module")
def table(golden_dir):
    with open(os.path.join(golden_dir, "clock_table.json")) as f:
        return json.load(f)


def test_frame_len_to_clock(table):
    assert clock.FRAME_MS == table["tower_frame_ms"]
    for row in table["rows"]:
        assert clock.clock_ms(row["frame_len"]) == row["clock_ms"]


def test_decisions_per_second_as_printed(table):
    for row in table["rows"]:
        printed = row["decisions_per_s_printed"]
        digits = len(printed.split(".")[1])
        assert f"{float(clock.decisions_per_second(row['clock_ms'])):.{digits}f}" == printed


def test_left_pad_and_operating_points(table):
    for row in table["rows"]:
        assert clock.LEFT_PAD_TOKENS[row["frame_len"]] == row["streaming_n_left_pad_tokens"]
        for d in row["post_trained_delays_ms"]:
            assert clock.is_post_trained(row["clock_ms"], d)
            assert clock.num_delay_tokens(d, row["clock_ms"]) * row["clock_ms"] == d
    # derived invariant: every clock looks back the same 1440 ms of left context
    assert {r["streaming_n_left_pad_tokens"] * r["clock_ms"] for r in table["rows"]} == {1440}


def test_delay_tokens_example(table):
    ex = table["delay_example"]
    assert clock.num_delay_tokens(ex["target_delay_ms"], ex["clock_ms"]) == ex["num_delay_tokens"]


def test_samples_per_token_example(table):
    ex = table["usage_example"]
    assert clock.samples_per_token(80) == ex["raw_audio_samples_per_token"]
    assert clock.SAMPLE_RATE_HZ == ex["sampling_rate"]
    assert clock.LEFT_PAD_TOKENS[4] == ex["streaming_n_left_pad_tokens"]


def test_windows(table):
    # 30 s of steps: 375 and 250 exactly, 187.5 rounded up at 160 ms
    assert [clock.window_steps(r["clock_ms"]) for r in table["rows"]] == [375, 250, 188]
    assert clock.NATIVE_CONTEXT_MS == table["native_context_ms"]


def test_delay_must_be_multiple():
    with pytest.raises(clock.ClockError):
        clock.num_delay_tokens(500, 80)
    with pytest.raises(clock.ClockError):
        clock.num_delay_tokens(0, 80)
    # longer delays stay available when they are multiples, even if not post-trained
    assert clock.num_delay_tokens(640, 80) == 8 and not clock.is_post_trained(80, 640)
    with pytest.raises(clock.ClockError):
        clock.clock_ms(5)


def test_resolve():
    r = clock.resolve(6, 480)
    assert r == {"clock_ms": 120, "window": 250, "num_delay_tokens": 4, "left_pad_tokens": 12,
                 "samples_per_token": 1920, "decisions_per_s": 1000 / 120, "post_trained": True}
