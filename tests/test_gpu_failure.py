"""Failure detection on the device: a bounded wait that runs out, and recovery afterwards.

Every wait of the attention kernel on its shared-memory stages is bounded.  The
failure-detection test hook (rkv_set_wait_test) shortens the limit to 2 ms and
makes each CTA's producer skip the copy of one stage, so the consumers' wait for
that stage runs out: nothing faults or hangs.  The kernel must record
RKV_ERR_TIMEOUT, return within milliseconds, leave later launches of the handle
skipping their copies until rkv_sync_status has read the status, and the
handle must then run clean again: its ring state and pages were kept by the
other kernels of the step, so the next steps match the fp64 oracle.
"""
import time

import numpy as np
import pytest

import synth
from rkv_harness import LSE_TOL, OUT_TOL, oracle_step

pytestmark = pytest.mark.gpu

WAIT_NS = 2_000_000


def _bufs(wl, layers):
    import torch
    S, Q, hq, hkv, d = wl.n_streams, wl.q_per_step, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    q = torch.empty(layers, S, Q, hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(layers, S, Q, hkv, d, dtype=torch.bfloat16, device="cuda")
    return q, k, torch.empty_like(k), torch.empty_like(q), torch.empty(layers, S, Q, hq, dtype=torch.float32,
                                                                         device="cuda")


def _check_against_oracle(wl, n_old, out, lse, layers, streams):
    for layer in layers:
        for s in streams:
            o_ref, l_ref = oracle_step(wl, s, layer, n_old)
            o = out[layer, s].float().cpu().numpy()
            lv = lse[layer, s].cpu().numpy()
            assert np.abs(o - o_ref).max() <= OUT_TOL, (layer, s, n_old)
            assert (np.abs(lv - l_ref) / np.maximum(1.0, np.abs(l_ref))).max() <= LSE_TOL, (layer, s, n_old)


def _handle(rkv, wl):
    return rkv.RollingKV(wl.windows().tolist(), wl.start_offsets().tolist(), n_layers=wl.n_layers,
                         n_streams=wl.n_streams, n_q_heads=wl.n_q_heads, n_kv_heads=wl.n_kv_heads,
                         head_dim=wl.head_dim, q_per_step=wl.q_per_step, scheme=wl.scheme,
                         rope_theta=wl.rope_theta)


@pytest.mark.parametrize("path,withhold", [
    ("per_layer", 0),      # few units: each window split over a cluster of CTAs merged in shared memory
    ("static", 0),         # the scratch form: per-split partials and a merge kernel
    ("fused", 0),          # the append fused into the launch: the appender warp still writes the tokens
    ("whole_step", 4),     # many units: persistent CTAs, the stage withheld in a CTA's second unit
    ("whole_step_on_read", 4),  # the same over keys at their ring slot (next unit's query staged)
])
def test_bounded_wait_runs_out_and_the_handle_recovers(path, withhold):
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv

    whole = path.startswith("whole_step")
    n_streams = 64 if whole else 3
    wl = synth.workload("tiny", n_layers=3, n_streams=n_streams, extra={"window": 150},
                        scheme=2 if path.endswith("on_read") else 1)
    S, L = wl.n_streams, wl.n_layers
    h = _handle(rkv, wl)
    q, k, v, out, lse = _bufs(wl, L)
    active = list(range(S))

    def step(n_old, fail_layer=None):
        if whole:
            h.gen_next_inputs(wl.seed, active, wl.input_scale, q, k, v)
            h.step(active, q, k, v, out, lse)
            return
        h.begin_step(active)
        for layer in range(L):
            h.gen_step_inputs(wl.seed, layer, wl.input_scale, q[layer], k[layer], v[layer])
            h.rebase(layer)
            if path != "fused":
                h.append_rope(layer, k[layer], v[layer])
            if layer == fail_layer:
                rkv.rkv_set_wait_test(h.handle, withhold, WAIT_NS)
            if path == "fused":
                h.append_decode_attn(layer, q[layer], k[layer], v[layer], out[layer], lse[layer])
            elif path == "static":
                rkv.rkv_decode_attn_static(h.handle, layer, q[layer], out[layer], lse[layer])
            else:
                h.decode_attn(layer, q[layer], out[layer], lse[layer])
            if layer == fail_layer:
                # two more launches while the status reports the timeout: they skip their copies
                h.decode_attn(layer, q[layer], out[layer], lse[layer])
                h.decode_attn(layer, q[layer], out[layer], lse[layer])
                rkv.rkv_set_wait_test(h.handle, -1, 0)

    n = 0
    for _ in range(155):                       # the windows fill and roll
        step(n)
        n += 1
    h.sync_status()
    torch.cuda.synchronize()

    t0 = time.perf_counter()
    if whole:
        rkv.rkv_set_wait_test(h.handle, withhold, WAIT_NS)
        step(n)
        rkv.rkv_set_wait_test(h.handle, -1, 0)
        h.decode_attn_layers(0, L, q, out, lse)   # skips its copies too
    else:
        step(n, fail_layer=1)
    n += 1
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 1.0      # the waits gave up after milliseconds
    with pytest.raises(rkv.RkvError) as e:
        h.sync_status()
    assert e.value.code == rkv.RKV_ERR_TIMEOUT and "timed-out wait" in str(e.value)
    h.sync_status()                            # read and cleared

    # the same handle runs clean: outputs of the next steps against the oracle, state bit-exact
    streams = [0, S - 1]
    for _ in range(3):
        step(n)
        torch.cuda.synchronize()
        _check_against_oracle(wl, n, out, lse, range(L), streams)
        n += 1
    h.sync_status()
    assert h.stream_state(0)["n"] == n
    h.close()

    # and so does a fresh handle
    h2 = _handle(rkv, wl)
    h = h2
    n = 0
    for _ in range(3):
        step(n)
        n += 1
    torch.cuda.synchronize()
    _check_against_oracle(wl, n - 1, out, lse, range(L), streams)
    h2.sync_status()
    h2.close()


def test_wait_test_hook_validates_its_arguments():
    import rolling_kv_sliding_rkv_b300 as rkv

    wl = synth.workload("tiny", n_layers=1, n_streams=1, extra={"window": 8})
    h = _handle(rkv, wl)
    for bad in ((-2, 0), (0, 10), (0, 2_000_000_000)):
        with pytest.raises(rkv.RkvError) as e:
            rkv.rkv_set_wait_test(h.handle, *bad)
        assert e.value.code == rkv.RKV_ERR_INVALID_ARG
    h.close()
