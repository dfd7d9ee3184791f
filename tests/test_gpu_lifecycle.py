"""Stream lifecycle: rkv_reset_stream starts a new history in a stream slot.

voxtral.c's continuous mode restarts the decoder cache while audio keeps
flowing (voxtral.c rolling-KV article §四), and a serving loop hands a slot to
a new audio stream.  After the reset the stream must behave exactly like a
fresh stream with the new start offset (outputs against the fp64 oracle, ring
state against the integer model), and the other streams must not notice.
"""
import math

import numpy as np
import pytest

import synth
from oracle.attention import attention_step
from oracle.ring import StreamRing
from rkv_harness import LSE_TOL, OUT_TOL

pytestmark = pytest.mark.gpu


def _oracle(wl, stream, layer, n_old, p0):
    Q, hq, hkv, d = wl.q_per_step, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    w = int(wl.windows()[stream])
    toks = np.arange(max(0, n_old + Q - w), n_old + Q)
    sc = wl.input_scale
    qb = synth.token_tensor(wl.seed, synth.TAG_Q, stream, layer, np.arange(n_old, n_old + Q), hq, d, sc)
    kb = synth.token_tensor(wl.seed, synth.TAG_K, stream, layer, toks, hkv, d, sc)
    vb = synth.token_tensor(wl.seed, synth.TAG_V, stream, layer, toks, hkv, d, sc)
    return attention_step(synth.bf16_bits_to_f64(qb), synth.bf16_bits_to_f64(kb), synth.bf16_bits_to_f64(vb),
                          toks, n_old, p0, w, 1.0 / math.sqrt(d), wl.rope_theta)


@pytest.mark.parametrize("scheme", [0, 1, 2])
def test_reset_stream_starts_a_fresh_history(scheme):
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv

    wl = synth.workload("qwen", n_layers=2, n_streams=3, extra={"window": 100}, scheme=scheme)
    S, L, hq, hkv, d = wl.n_streams, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    p0 = wl.start_offsets().tolist()
    h = rkv.RollingKV(wl.windows().tolist(), p0, n_layers=L, n_streams=S, n_q_heads=hq, n_kv_heads=hkv,
                      head_dim=d, q_per_step=1, scheme=scheme, rope_theta=wl.rope_theta)
    q = torch.empty(S, 1, hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(S, 1, hkv, d, dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    out = torch.empty_like(q)
    lse = torch.empty(S, 1, hq, dtype=torch.float32, device="cuda")
    new_p0, reset_at, steps = 777_777, 130, 170
    rings = {s: StreamRing(100, p0[s], 1, 1 if scheme else 0) for s in range(S)}
    checked = 0
    for step in range(steps):
        if step == reset_at:
            h.reset_stream(1, new_p0)
            rings[1] = StreamRing(100, new_p0, 1, 1 if scheme else 0)
        n_old = {s: rings[s].n for s in range(S)}
        h.begin_step(list(range(S)))
        for s in range(S):
            rings[s].step()
        for layer in range(L):
            h.gen_step_inputs(wl.seed, layer, wl.input_scale, q, k, v)
            if scheme:
                h.rebase(layer)
            h.append_rope(layer, k, v)
            h.decode_attn(layer, q, out, lse)
            # the reset stream every 7th step of its new history (its pages still hold the old
            # history beyond the new length); stream 0 every 41st step
            for s in (0, 1):
                if (s == 1 and step >= reset_at and (step - reset_at) % 7 == 0) or (s == 0 and step % 41 == 0):
                    o_ref, l_ref = _oracle(wl, s, layer, n_old[s], new_p0 if (s == 1 and step >= reset_at) else p0[s])
                    o = out[s].float().cpu().numpy()
                    lv = lse[s].cpu().numpy()
                    assert np.abs(o - o_ref).max() <= OUT_TOL, (s, step, layer)
                    assert (np.abs(lv - l_ref) / np.maximum(1.0, np.abs(l_ref))).max() <= LSE_TOL, (s, step, layer)
                    checked += 1
    h.sync_status()
    for s in range(S):
        assert list(h.stream_state(s).values()) == rings[s].state(), f"stream {s}"
    assert checked > 20
    h.close()


def test_reset_stream_validates_arguments():
    import rolling_kv_sliding_rkv_b300 as rkv

    h = rkv.RollingKV([8, 8], [0, 0], n_layers=1, n_streams=2, n_q_heads=4, n_kv_heads=2, head_dim=64,
                      q_per_step=1, scheme=0, page_size=16)
    with pytest.raises(rkv.RkvError) as e:
        h.reset_stream(2, 0)
    assert e.value.code == rkv.RKV_ERR_INVALID_ARG
    with pytest.raises(rkv.RkvError) as e:
        h.reset_stream(0, -1)
    assert e.value.code == rkv.RKV_ERR_CONFIG
    h.close()


def _drive(h, wl, steps, q, k, v, out, lse, record_stream=None):
    """Run `steps` steps of all streams with the generator's inputs; return the recorded outputs."""
    rec = []
    S, L = wl.n_streams, wl.n_layers
    for _ in range(steps):
        h.begin_step(list(range(S)))
        for layer in range(L):
            h.gen_step_inputs(wl.seed, layer, wl.input_scale, q, k, v)
            if wl.scheme:
                h.rebase(layer)
            h.append_rope(layer, k, v)
            h.decode_attn(layer, q, out, lse)
            if record_stream is not None:
                rec.append((out[record_stream].clone(), lse[record_stream].clone()))
    return rec


@pytest.mark.parametrize("scheme,where,kv_format", [(1, "device", 0), (2, "host", 0), (0, "device", 0),
                                                   (2, "device", 1), (0, "host", 1)])
def test_snapshot_resumes_a_stream_exactly(scheme, where, kv_format):
    """A stream saved from one handle and loaded into another continues bit for bit (also from
    the fp8 store: its key, value and scale planes)."""
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv

    wl = synth.workload("qwen", n_layers=2, n_streams=3, extra={"window": 100}, scheme=scheme)
    S, L, hq, hkv, d = wl.n_streams, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim

    def handle():
        return rkv.RollingKV(wl.windows().tolist(), wl.start_offsets().tolist(), n_layers=L, n_streams=S,
                             n_q_heads=hq, n_kv_heads=hkv, head_dim=d, q_per_step=1, scheme=scheme,
                             rope_theta=wl.rope_theta, kv_format=kv_format)

    q = torch.empty(S, 1, hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(S, 1, hkv, d, dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    out = torch.empty_like(q)
    lse = torch.empty(S, 1, hq, dtype=torch.float32, device="cuda")
    a = handle()
    _drive(a, wl, 130, q, k, v, out, lse)
    snap = a.save_stream(1)
    if where == "host":
        snap = snap.cpu()
    state_a = a.stream_state(1)
    ref = _drive(a, wl, 20, q, k, v, out, lse, record_stream=1)

    b = handle()
    _drive(b, wl, 7, q, k, v, out, lse)          # b's other streams are elsewhere in their histories
    b.load_stream(1, snap)
    assert b.stream_state(1) == state_a
    got = _drive(b, wl, 20, q, k, v, out, lse, record_stream=1)
    for (o_ref, l_ref), (o, lv) in zip(ref, got):
        assert torch.equal(o_ref, o) and torch.equal(l_ref, lv)
    assert b.stream_state(1) == a.stream_state(1)
    a.sync_status()
    b.sync_status()

    # a slot with another window cannot take the snapshot
    c = rkv.RollingKV([100, 90, 100], wl.start_offsets().tolist(), n_layers=L, n_streams=S, n_q_heads=hq,
                      n_kv_heads=hkv, head_dim=d, q_per_step=1, scheme=scheme, rope_theta=wl.rope_theta,
                      kv_format=kv_format)
    with pytest.raises(rkv.RkvError) as e:
        c.load_stream(1, snap)
    assert e.value.code == rkv.RKV_ERR_CONFIG
    # nor can a handle in the middle of a step save or load
    b.begin_step(list(range(S)))
    with pytest.raises(rkv.RkvError) as e:
        b.save_stream(0)
    assert e.value.code == rkv.RKV_ERR_STATE
    for hh in (a, b, c):
        hh.close()
