"""CUDA path against the fp64 oracle (max |out error| <= 2e-2, |lse error| <= 1e-3 max(1, |lse|)).

Small cases compare every output of every step; full-size workloads run in the
shape the benchmark times and compare sampled stream-layer-steps.
"""
import numpy as np
import pytest

import synth
from rkv_harness import compare, run_gpu

pytestmark = pytest.mark.gpu

SMALL = {
    # several pages of 64 slots with a ragged tail (150 = 2 * 64 + 22), window rolls
    "tiny_exact": ("tiny", dict(n_layers=2, n_streams=3, extra={"window": 150}), 190),
    "tiny_exact_interval5": ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 150}, rebase_interval=5), 190),
    "tiny_offset_large_p0": ("tiny", dict(n_layers=1, n_streams=3, extra={"window": 150}, scheme=0,
                                          p0_high=2 ** 41), 190),
    "voxtral_shape": ("voxtral", dict(n_layers=1, n_streams=2, extra={"window": 130}), 150),
    "encoder_q4": ("encoder", dict(n_layers=1, n_streams=3, extra={"window": 70}), 30),
    "encoder_q4_exact": ("encoder", dict(n_layers=1, n_streams=2, extra={"window": 70}, scheme=1), 30),
    "qwen_scaled": ("qwen", dict(n_layers=2, n_streams=3, extra={"window": 100}), 120),
    "mixed_small": ("mixed", dict(n_layers=1, n_streams=9, extra={}), 60),
    # exact re-base applied as attention reads the pre-RoPE keys (no stored re-based copy)
    "tiny_on_read": ("tiny", dict(n_layers=2, n_streams=3, extra={"window": 150}, scheme=2), 190),
    "tiny_on_read_interval5": ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 150}, scheme=2,
                                            rebase_interval=5), 190),
    "encoder_q4_on_read": ("encoder", dict(n_layers=1, n_streams=2, extra={"window": 70}, scheme=2), 30),
    "qwen_on_read_p0": ("qwen", dict(n_layers=2, n_streams=3, extra={"window": 100}, scheme=2), 120),
    # the whole step (all layers per launch) through rkv_step
    "qwen_whole_step": ("qwen", dict(n_layers=3, n_streams=3, extra={"window": 100}), 120, True),
    "voxtral_whole_step": ("voxtral", dict(n_layers=2, n_streams=2, extra={"window": 130}), 150, True),
    "encoder_whole_step": ("encoder", dict(n_layers=2, n_streams=2, extra={"window": 70}), 30, True),
    "mixed_whole_step_on_read": ("mixed", dict(n_layers=2, n_streams=9, extra={}, scheme=2), 60, True),
    # page sizes other than one stage (16 slots: four pages per stage; 128: half a page per stage)
    "tiny_page16": ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 150, "page_size": 16}), 190),
    "tiny_page128_on_read": ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 150, "page_size": 128},
                                          scheme=2), 190),
    "tiny_page32": ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 100, "page_size": 32}, scheme=0), 130),
    # 16 query rows per kv head: GQA group 16, and group 4 with 4 queries per step
    "gqa16_exact": ("tiny", dict(n_layers=1, n_streams=2, n_q_heads=16, n_kv_heads=1, extra={"window": 150}),
                    190),
    "gqa16_on_read": ("tiny", dict(n_layers=1, n_streams=2, n_q_heads=16, n_kv_heads=1, extra={"window": 150},
                                   scheme=2), 190),
    "gqa4_q4_d64": ("encoder", dict(n_layers=1, n_streams=2, n_q_heads=8, n_kv_heads=2, extra={"window": 90}), 40),
    "gqa4_q4_d64_on_read": ("encoder", dict(n_layers=1, n_streams=2, n_q_heads=8, n_kv_heads=2,
                                            extra={"window": 90}, scheme=2), 40),
    "gqa16_whole_step": ("tiny", dict(n_layers=2, n_streams=3, n_q_heads=16, n_kv_heads=1, extra={"window": 150}),
                         170, True),
    # degenerate windows: one key (the current token only), two keys, and W = Q for the encoder
    # (each step evicts everything before it)
    "tiny_w1": ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 1}), 20),
    "tiny_w2_on_read": ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 2}, scheme=2), 20),
    "tiny_w2_exact": ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 2}), 20),
    "encoder_w4": ("encoder", dict(n_layers=1, n_streams=2, extra={"window": 4}), 12),
    # head_dim 64 with GQA, one query per step
    "d64_gqa4": ("tiny", dict(n_layers=1, n_streams=2, n_q_heads=8, n_kv_heads=2, head_dim=64,
                              extra={"window": 150}), 190),
    # append fused into the attention launch (rkv_append_decode_attn): every scheme, the 4-query
    # step whose new tokens straddle stages and wrap the ring, small pages, mixed clocks
    "tiny_exact_fused": ("tiny", dict(n_layers=2, n_streams=3, extra={"window": 150}), 190, "fused"),
    "tiny_offset_fused": ("tiny", dict(n_layers=1, n_streams=3, extra={"window": 150}, scheme=0,
                                       p0_high=2 ** 41), 190, "fused"),
    "qwen_on_read_fused": ("qwen", dict(n_layers=2, n_streams=3, extra={"window": 100}, scheme=2), 120,
                           "fused"),
    "encoder_q4_fused": ("encoder", dict(n_layers=1, n_streams=3, extra={"window": 70}), 30, "fused"),
    "encoder_q4_on_read_fused": ("encoder", dict(n_layers=1, n_streams=2, extra={"window": 66}, scheme=2), 40,
                                 "fused"),
    "tiny_page16_fused": ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 150, "page_size": 16}), 190,
                          "fused"),
    "mixed_small_fused": ("mixed", dict(n_layers=1, n_streams=9, extra={}, scheme=2), 60, "fused"),
    "gqa16_fused": ("tiny", dict(n_layers=1, n_streams=2, n_q_heads=16, n_kv_heads=1, extra={"window": 150}),
                    190, "fused"),
    "tiny_w1_fused": ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 1}), 20, "fused"),
    # eviction in batches: a ring of capacity W + slack, cut back to the last W when a step would
    # overflow it, so the window length varies in [W, C] (every scheme; C = W + 8 and C = 2W)
    "tiny_exact_slack8": ("tiny", dict(n_layers=2, n_streams=3, extra={"window": 150}, window_slack=8), 200),
    "tiny_exact_slack_2w": ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 150}, window_slack=150), 420),
    "tiny_on_read_slack_2w_fused": ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 150}, scheme=2,
                                                 window_slack=150), 420, "fused"),
    "tiny_offset_slack8_fused": ("tiny", dict(n_layers=1, n_streams=3, extra={"window": 150}, scheme=0,
                                              window_slack=8, p0_high=2 ** 41), 200, "fused"),
    "encoder_q4_slack8": ("encoder", dict(n_layers=1, n_streams=2, extra={"window": 70}, window_slack=8), 45),
    "encoder_q4_on_read_slack_2w": ("encoder", dict(n_layers=1, n_streams=2, extra={"window": 70}, scheme=2,
                                                    window_slack=70), 60),
    "qwen_whole_step_slack": ("qwen", dict(n_layers=3, n_streams=3, extra={"window": 100}, window_slack=40),
                              200, True),
    "mixed_small_slack_on_read": ("mixed", dict(n_layers=1, n_streams=9, extra={}, scheme=2, window_slack=20),
                                  120, "fused"),
    # the fp8 (e4m3) store, against the oracle's model of it: keys quantised after their rotation at
    # the stored position, values quantised, power-of-two row scales
    "tiny_offset_fp8": ("tiny", dict(n_layers=1, n_streams=3, extra={"window": 150}, scheme=0, kv_format=1,
                                     p0_high=2 ** 41), 190),
    "tiny_on_read_fp8": ("tiny", dict(n_layers=2, n_streams=3, extra={"window": 150}, scheme=2, kv_format=1), 190),
    "tiny_on_read_fp8_fused": ("tiny", dict(n_layers=1, n_streams=3, extra={"window": 150}, scheme=2,
                                            kv_format=1), 190, "fused"),
    "tiny_offset_fp8_static": ("tiny", dict(n_layers=1, n_streams=3, extra={"window": 150}, scheme=0,
                                            kv_format=1), 190, "static"),
    "qwen_on_read_fp8_whole_step": ("qwen", dict(n_layers=2, n_streams=3, extra={"window": 100}, scheme=2,
                                                 kv_format=1), 120, True),
    "encoder_q4_fp8": ("encoder", dict(n_layers=1, n_streams=3, extra={"window": 70}, kv_format=1), 30),
    "encoder_q4_on_read_fp8_fused": ("encoder", dict(n_layers=1, n_streams=2, extra={"window": 66}, scheme=2,
                                                     kv_format=1), 40, "fused"),
    "tiny_page16_fp8": ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 150, "page_size": 16}, scheme=2,
                                     kv_format=1), 190),
    "tiny_on_read_slack_fp8": ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 150}, scheme=2,
                                            window_slack=40, kv_format=1), 230, "fused"),
    "mixed_whole_step_fp8": ("mixed", dict(n_layers=2, n_streams=9, extra={}, scheme=2, kv_format=1), 60, True),
    "d64_gqa4_fp8": ("tiny", dict(n_layers=1, n_streams=2, n_q_heads=8, n_kv_heads=2, head_dim=64,
                                  extra={"window": 150}, scheme=0, kv_format=1), 190),
}


@pytest.mark.parametrize("case", sorted(SMALL))
def test_small_every_output(case):
    name, over, ticks, *opt = SMALL[case]
    wl = synth.workload(name, **over)
    want = set()
    w = wl.windows()
    fill = wl.initial_fill()
    counts = fill.copy()
    for t in range(ticks):
        counts[wl.active_at_tick(t)] += 1
    for s in range(wl.n_streams):
        for layer in range(wl.n_layers):
            for n_old in range(int(fill[s]) * wl.q_per_step, int(counts[s]) * wl.q_per_step, wl.q_per_step):
                want.add((s, layer, n_old))
    mode = opt[0] if opt else False
    run = run_gpu(wl, ticks, want, whole_step=mode is True, attn=mode if isinstance(mode, str) else "regular")
    assert len(run.samples) == len(want)
    e_o, e_l = compare(run, wl)
    print(case, "max out err", e_o, "max lse err", e_l)


def final_counts(wl, n_ticks):
    """Token count of every stream after the harness's initial fill and `n_ticks` ticks."""
    counts = wl.initial_fill().copy()
    for t in range(n_ticks):
        counts[wl.active_at_tick(t)] += 1
    return counts * wl.q_per_step


FULL = {
    "tiny": ("tiny", dict(), 1000, [0, 1, 374, 375, 376, 998, 999], [0]),
    "qwen": ("qwen", dict(), 1000, [0, 1, 374, 375, 376, 999], [0, 17, 40, 63]),
    "encoder": ("encoder", dict(), 200, [0, 4, 744, 748, 752, 796], [0, 31]),
    "mixed": ("mixed", dict(), 400, None, [0, 1, 2, 3]),
    "voxtral": ("voxtral", dict(), 8200, [0, 8191, 8192, 8193, 8199], [0, 15]),
    # one stream, a long window: each kv head's window splits over a cluster of 8 CTAs
    "long_window_cluster8": ("tiny", dict(n_streams=1, extra={"window": 2000}), 2050, [0, 999, 1999, 2000, 2049],
                             [0]),
    # the most streams a handle takes (RKV_MAX_STREAMS)
    "max_streams": ("qwen", dict(n_layers=1, n_streams=1024, extra={"window": 40}), 50, [0, 39, 40, 49],
                    [0, 511, 1023]),
    # the timed path itself: rkv_step over every layer (the persistent all-layers launches after the
    # re-base in reverse layer order), at the benchmark's shapes
    "qwen_step": ("qwen", dict(), 1000, [0, 374, 375, 376, 999], [0, 17, 40, 63], True),
    "qwen_step_on_read": ("qwen", dict(scheme=2), 1000, [0, 374, 375, 376, 999], [0, 17, 40, 63], True),
    # mixed clocks: windows of 375 / 250 / 188 filled from ragged starts, then two 12-tick schedule
    # periods more; one stream of each clock and one more 80 ms stream
    "mixed_step": ("mixed", dict(), 510, "schedule", [0, 1, 2, 3], True),
    # the benchmark's headline: the same ticks with the exact re-base applied on read
    "mixed_step_on_read": ("mixed", dict(scheme=2), 510, "schedule", [0, 1, 2, 3, 4], True),
    # the same batch read the other way: all 256 streams step on every call (no scheduler tick)
    "mixed_all_streams_step_on_read": ("mixed", dict(scheme=2, tick_ms=0), 400, "schedule", [0, 1, 2, 3], True),
    # the per-layer calls over keys stored at their ring slot
    "qwen_on_read": ("qwen", dict(scheme=2), 1000, [0, 374, 375, 376, 999], [0, 40, 63]),
    "encoder_step": ("encoder", dict(), 200, [0, 4, 744, 748, 752, 796], [0, 31], True),
    # the fp8 store at the benchmark's shape, through rkv_step
    "qwen_step_on_read_fp8": ("qwen", dict(scheme=2, kv_format=1), 1000, [0, 374, 375, 376, 999], [0, 17, 63],
                              True),
    # the append fused into the per-layer attention launch (rkv_append_decode_attn): one unit per
    # CTA at the Qwen shape and on the mixed schedule; several units per CTA at 1024 streams
    "qwen_fused": ("qwen", dict(), 1000, [0, 374, 375, 376, 999], [0, 17, 40, 63], "fused"),
    "mixed_fused_on_read": ("mixed", dict(scheme=2), 510, "schedule", [0, 1, 2, 3, 4], "fused"),
    "max_streams_fused": ("qwen", dict(n_layers=1, n_streams=1024, extra={"window": 40}, scheme=2), 50,
                          [0, 39, 40, 49], [0, 511, 1023], "fused"),
}


@pytest.mark.slow
@pytest.mark.parametrize("case", sorted(FULL))
def test_full_size_sampled(case):
    name, over, ticks, steps, streams, *opt = FULL[case]
    whole_step = bool(opt and opt[0] is True)
    attn = opt[0] if opt and isinstance(opt[0], str) else "regular"
    wl = synth.workload(name, **over)
    layers = sorted({0, wl.n_layers // 2, wl.n_layers - 1})
    final = final_counts(wl, ticks)
    fill = wl.initial_fill() * wl.q_per_step
    w = wl.windows()
    want = set()
    for s in streams:
        if steps is None:        # mixed clocks: every 37th token of the chosen streams
            mine = range(0, 500, 37)
        elif steps == "schedule":  # the fill, the window's edge and the last two steps the run reaches
            mine = {0, int(fill[s]) - 1, int(fill[s]), int(w[s]) - 1, int(w[s]), int(w[s]) + 1,
                    int(final[s]) - 2, int(final[s]) - 1}
        else:
            mine = steps
        for layer in layers:
            for n_old in mine:
                if 0 <= n_old < final[s] and n_old % wl.q_per_step == 0:
                    want.add((s, layer, n_old))
    if steps == "schedule":
        assert all(final[s] >= w[s] + 2 for s in streams)   # every chosen window filled and rolled
    run = run_gpu(wl, ticks, want, streams_of_interest=streams, whole_step=whole_step, attn=attn)
    assert set(run.samples) == want
    e_o, e_l = compare(run, wl)
    for s in streams:
        assert list(run.states[s].values()) == run.ring[s].state()
    print(case, len(run.samples), "samples; max out err", e_o, "max lse err", e_l)
