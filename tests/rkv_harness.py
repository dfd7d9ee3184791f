"""Drive the CUDA path through the C ABI and compare sampled outputs with the oracle.

The GPU run draws its inputs on the device (rkv_gen_step_inputs); the oracle
regenerates the same tokens on the host (synth.token_tensor), so nothing the
GPU computes ever feeds the oracle.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

import synth
from oracle.attention import attention_step
from oracle.fp8 import quantize_rows, rotate_fp32
from oracle.ring import StreamRing
from oracle.schemes import stored_key_attention_step

OUT_TOL = 2e-2
LSE_TOL = 1e-3


@dataclass
class Run:
    """Outputs copied back from the GPU at sampled (stream step index, stream, layer)."""
    samples: dict = field(default_factory=dict)   # (stream, layer, n_old) -> (out [Q][Hq][d], lse [Q][Hq])
    states: dict = field(default_factory=dict)    # stream -> final device state
    ring: dict = field(default_factory=dict)      # stream -> oracle StreamRing after the run


def run_gpu(wl: synth.Workload, n_ticks: int, want: set, streams_of_interest=None, whole_step=False,
            attn="regular"):
    """Run `n_ticks` steps (ticks for the mixed-clock workload) and copy sampled outputs.

    want: set of (stream, layer, n_old) to record, n_old = the stream's token
    count before the step.  A mixed-clock workload first brings every stream
    to its initial fill with extra steps of the lagging streams.
    whole_step: drive rkv_step (all layers per launch) instead of the
    per-layer calls; the inputs are the same generator draws
    (rkv_gen_next_inputs, every layer of the step in one launch).
    attn: the per-layer calls: "regular" (rkv_append_rope, rkv_decode_attn),
    "static" (rkv_append_rope, rkv_decode_attn_static) or "fused"
    (rkv_append_decode_attn).
    """
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv

    dev = torch.device("cuda")
    windows = wl.windows()
    p0 = wl.start_offsets()
    h = rkv.RollingKV(windows.tolist(), p0.tolist(), device=dev, n_layers=wl.n_layers, n_streams=wl.n_streams,
                      n_q_heads=wl.n_q_heads, n_kv_heads=wl.n_kv_heads, head_dim=wl.head_dim,
                      q_per_step=wl.q_per_step, scheme=wl.scheme, rebase_interval=wl.rebase_interval,
                      rope_theta=wl.rope_theta, page_size=int(wl.extra.get("page_size", 64)),
                      window_slack=wl.window_slack, kv_format=wl.kv_format)
    S, L, Q, hq, hkv, d = wl.n_streams, wl.n_layers, wl.q_per_step, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    q = torch.empty(S * Q * hq * d, dtype=torch.bfloat16, device=dev)
    k = torch.empty(S * Q * hkv * d, dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    out = torch.empty_like(q)
    lse = torch.empty(S * Q * hq, dtype=torch.float32, device=dev)
    exact = wl.scheme in (rkv.RKV_SCHEME_EXACT_REBASE, rkv.RKV_SCHEME_EXACT_ON_READ)
    # both exact schemes keep the same bookkeeping; they differ only in what the pool stores
    ring_scheme = rkv.RKV_SCHEME_EXACT_REBASE if exact else rkv.RKV_SCHEME_OFFSET_ONLY
    rings = {s: StreamRing(int(windows[s]), int(p0[s]), Q, ring_scheme, wl.rebase_interval,
                           capacity=int(windows[s]) + wl.window_slack) for s in range(S)}
    run = Run()
    want_streams = {s for s, _, _ in want}
    if whole_step:
        qa = torch.empty(L * S * Q * hq * d, dtype=torch.bfloat16, device=dev)
        ka = torch.empty(L * S * Q * hkv * d, dtype=torch.bfloat16, device=dev)
        va = torch.empty_like(ka)
        outa = torch.empty_like(qa)
        lsea = torch.empty(L * S * Q * hq, dtype=torch.float32, device=dev)

    def record(active, n_old, layer, o_all, l_all):
        a = len(active)
        for idx, s in enumerate(active):
            if s in want_streams and (s, layer, n_old[s]) in want:
                o = o_all[: a * Q * hq * d].view(a, Q, hq, d)[idx].float().cpu().numpy()
                lv = l_all[: a * Q * hq].view(a, Q, hq)[idx].cpu().numpy()
                run.samples[(s, layer, n_old[s])] = (o, lv)

    def one_whole_step(active):
        a = len(active)
        n_old = {s: rings[s].n for s in active}
        for s in active:
            rings[s].step()
        nqe, nke = a * Q * hq * d, a * Q * hkv * d
        h.gen_next_inputs(wl.seed, active, wl.input_scale, qa, ka, va)
        h.step(active, qa[: L * nqe], ka[: L * nke], va[: L * nke], outa[: L * nqe], lsea[: L * a * Q * hq])
        for layer in range(L):
            record(active, n_old, layer, outa[layer * nqe:], lsea[layer * a * Q * hq:])

    def one_step(active):
        if whole_step:
            return one_whole_step(active)
        a = len(active)
        h.begin_step(active)
        n_old = {s: rings[s].n for s in active}
        for s in active:
            rings[s].step()
        for layer in range(L):
            h.gen_step_inputs(wl.seed, layer, wl.input_scale, q, k, v)
            if exact:
                h.rebase(layer)
            if attn == "fused":
                h.append_decode_attn(layer, q, k, v, out, lse)
            else:
                h.append_rope(layer, k, v)
                if attn == "static":
                    rkv.rkv_decode_attn_static(h.handle, layer, q, out, lse)
                else:
                    h.decode_attn(layer, q, out, lse)
            record(active, n_old, layer, out, lse)

    # initial fill (ragged), one extra step at a time for the streams still short of it
    fill = wl.initial_fill()
    for r in range(int(fill.max()) if len(fill) else 0):
        active = [s for s in range(S) if fill[s] > r]
        if active:
            one_step(active)
    for tick in range(n_ticks):
        active = wl.active_at_tick(tick).tolist()
        if active:
            one_step(active)
    h.sync_status()
    for s in (streams_of_interest if streams_of_interest is not None else range(S)):
        run.states[s] = h.stream_state(s)
        run.ring[s] = rings[s]
    h.close()
    return run


def evicted_after(wl: synth.Workload, stream: int, n_new: int) -> int:
    """Tokens out of the window once the stream holds n_new tokens (the oracle's ring model)."""
    w = int(wl.windows()[stream])
    ring = StreamRing(w, 0, wl.q_per_step, capacity=w + wl.window_slack)
    while ring.n < n_new:
        ring.step()
    return ring.evicted


def oracle_step(wl: synth.Workload, stream: int, layer: int, n_old: int, p0: int | None = None):
    """Oracle outputs of one stream-layer-step, from regenerated inputs (p0: the stream's start
    offset, by default the workload's)."""
    Q, hq, hkv, d = wl.q_per_step, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    w = int(wl.windows()[stream])
    p0 = int(wl.start_offsets()[stream]) if p0 is None else int(p0)
    n_new = n_old + Q
    first = evicted_after(wl, stream, n_new) if wl.window_slack else None
    toks = np.arange(max(0, n_new - w) if first is None else first, n_new)
    sc = wl.input_scale
    qb = synth.token_tensor(wl.seed, synth.TAG_Q, stream, layer, np.arange(n_old, n_new), hq, d, sc)
    kb = synth.token_tensor(wl.seed, synth.TAG_K, stream, layer, toks, hkv, d, sc)
    vb = synth.token_tensor(wl.seed, synth.TAG_V, stream, layer, toks, hkv, d, sc)
    q, k, v = synth.bf16_bits_to_f64(qb), synth.bf16_bits_to_f64(kb), synth.bf16_bits_to_f64(vb)
    if wl.kv_format == 1:
        # the fp8 store: keys rotated at the position the scheme stores them at (P0 + j offset-only,
        # the ring slot j mod C on read), then quantised, as are the values
        C = w + wl.window_slack
        spos = (lambda j: j % C) if wl.scheme == 2 else (lambda j: p0 + j)
        return stored_key_attention_step(q, k, v, toks, n_old, w, 1.0 / math.sqrt(d), wl.rope_theta, spos,
                                         quantize=quantize_rows, first_key=first,
                                         rotate_keys=lambda kk, pos: rotate_fp32(kk, pos, wl.rope_theta))
    return attention_step(q, k, v, toks, n_old, p0, w, 1.0 / math.sqrt(d), wl.rope_theta, first_key=first)


def compare(run: Run, wl: synth.Workload):
    """Max errors over all samples; asserts the tolerances."""
    worst_o = worst_l = 0.0
    for (s, layer, n_old), (o, lv) in sorted(run.samples.items()):
        o_ref, l_ref = oracle_step(wl, s, layer, n_old)
        e_o = float(np.abs(o - o_ref).max())
        e_l = float((np.abs(lv - l_ref) / np.maximum(1.0, np.abs(l_ref))).max())
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(lv))
        assert e_o <= OUT_TOL, f"out error {e_o:.3g} at stream {s} layer {layer} n_old {n_old}"
        assert e_l <= LSE_TOL, f"lse error {e_l:.3g} at stream {s} layer {layer} n_old {n_old}"
        worst_o, worst_l = max(worst_o, e_o), max(worst_l, e_l)
    return worst_o, worst_l
