"""Audio clock, window and delay-token arithmetic.

Sources (both pages print the same table):
  * Edge0/Audio8-ASR-Infinite model card and README, "Optimized operation
    points": clock 80/120/160 ms <-> frame_len 4/6/8, streaming_n_left_pad_tokens
    18/12/9, post-trained target_delay_ms 240/320/480/560, 240/480, 320/480;
    target_delay_ms must be an integer multiple of the clock.
  * Audio8 ASR Infinite 无限长转写原理, "三档音频时钟": the tower frame is
    20 ms and frame_len frames are packed per step; 12.5 / 8.3 / 6.25
    decisions per second.  "可配置转写延迟": num_delay_tokens =
    target_delay_ms / clock (480 ms at 80 ms -> 6).
  * Model card "使用" (usage) example: 1280 raw samples per token at 80 ms,
    16 kHz.
  * Native context 30 s (model card, "查看 ... 运行演示"; explainer 第 1 步);
    the rolling window holds the last 30 s of clock steps.  30000/160 is
    187.5; the window is rounded up to 188.
"""
from __future__ import annotations

from fractions import Fraction

FRAME_MS = 20
SAMPLE_RATE_HZ = 16000
NATIVE_CONTEXT_MS = 30000
FRAME_LENS = (4, 6, 8)
LEFT_PAD_TOKENS = {4: 18, 6: 12, 8: 9}
POST_TRAINED_DELAYS_MS = {80: (240, 320, 480, 560), 120: (240, 480), 160: (320, 480)}


class ClockError(ValueError):
    pass


def clock_ms(frame_len: int) -> int:
    if frame_len not in FRAME_LENS:
        raise ClockError(f"frame_len must be one of {FRAME_LENS}, got {frame_len}")
    return FRAME_MS * frame_len


def decisions_per_second(clock: int) -> Fraction:
    return Fraction(1000, clock)


def window_steps(clock: int) -> int:
    """Clock steps in the 30 s native context, rounded up."""
    return -(-NATIVE_CONTEXT_MS // clock)


def num_delay_tokens(target_delay_ms: int, clock: int) -> int:
    if target_delay_ms <= 0 or target_delay_ms % clock != 0:
        raise ClockError(f"target_delay_ms={target_delay_ms} is not a positive multiple of {clock} ms")
    return target_delay_ms // clock


def samples_per_token(clock: int) -> int:
    return SAMPLE_RATE_HZ * clock // 1000


def is_post_trained(clock: int, target_delay_ms: int) -> bool:
    return target_delay_ms in POST_TRAINED_DELAYS_MS.get(clock, ())


def resolve(frame_len: int, target_delay_ms: int) -> dict:
    """Everything the clock fixes, after validation."""
    c = clock_ms(frame_len)
    return {
        "clock_ms": c,
        "window": window_steps(c),
        "num_delay_tokens": num_delay_tokens(target_delay_ms, c),
        "left_pad_tokens": LEFT_PAD_TOKENS[frame_len],
        "samples_per_token": samples_per_token(c),
        "decisions_per_s": float(decisions_per_second(c)),
        "post_trained": is_post_trained(c, target_delay_ms),
    }
