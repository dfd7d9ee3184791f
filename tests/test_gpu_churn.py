"""Streams leaving and joining a live mixed-clock batch (voxtral.c rolling-KV article §四: the
continuous-mode restart, applied to a serving loop that hands a stream slot to a new stream).

Every few ticks some slots are reset from a device-side list (rkv_reset_streams) with new start
offsets, between whole steps (rkv_step).  A slot's new stream starts an empty history at its new
P0 while the other streams keep theirs; sampled outputs of the streams that joined, before and
after the handover, and of streams that never left, match the fp64 oracle, and every slot's ring
state matches the integer model.
"""
import numpy as np
import pytest

import synth
from oracle.ring import StreamRing
from rkv_harness import LSE_TOL, OUT_TOL, oracle_step

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("scheme,slack", [(1, 0), (2, 0), (2, 24), (0, 0)])
def test_join_and_leave_between_steps(scheme, slack):
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv

    wl = synth.workload("mixed", n_layers=2, n_streams=24, extra={"window": 40}, scheme=scheme,
                        window_slack=slack, ragged_fill=False)
    S, L, hq, hkv, d = wl.n_streams, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    W = 40
    p0 = wl.start_offsets().astype(np.int64).copy()
    h = rkv.RollingKV([W] * S, p0.tolist(), n_layers=L, n_streams=S, n_q_heads=hq, n_kv_heads=hkv, head_dim=d,
                      q_per_step=1, scheme=scheme, rope_theta=wl.rope_theta, window_slack=slack)
    q = torch.empty(L * S * hq * d, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(L * S * hkv * d, dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    out = torch.empty_like(q)
    lse = torch.empty(L * S * hq, dtype=torch.float32, device="cuda")
    ring_scheme = 1 if scheme else 0
    rings = [StreamRing(W, int(p0[s]), 1, ring_scheme, 1, capacity=W + slack) for s in range(S)]
    joined = {}          # stream -> tick of its last join
    checked = {"joined_before": 0, "joined_after": 0, "stayed": 0}
    rng = np.random.default_rng(5 + scheme + slack)
    for tick in range(260):
        if tick % 9 == 4:        # two streams leave, new ones take their slots
            ids = rng.choice(S, size=2, replace=False).astype(np.int32)
            new_p0 = rng.integers(0, 2 ** 40, size=2).astype(np.int64)
            ids_d = torch.from_numpy(ids).cuda()
            p0_d = torch.from_numpy(new_p0).cuda()
            h.reset_streams(ids_d, p0_d)
            for s, p in zip(ids.tolist(), new_p0.tolist()):
                rings[s] = StreamRing(W, int(p), 1, ring_scheme, 1, capacity=W + slack)
                p0[s] = p
                joined[s] = tick
        active = wl.active_at_tick(tick).tolist()
        if not active:
            continue
        a = len(active)
        n_old = {s: rings[s].n for s in active}
        for s in active:
            rings[s].step()
        h.gen_next_inputs(wl.seed, active, wl.input_scale, q, k, v)
        h.step(active, q[: L * a * hq * d], k[: L * a * hkv * d], v[: L * a * hkv * d], out[: L * a * hq * d],
               lse[: L * a * hq])
        if tick % 5 == 0 or tick > 250:
            torch.cuda.synchronize()
            for idx, s in enumerate(active):
                n = n_old[s]
                if s in joined:
                    kind = "joined_after" if n >= W else "joined_before"
                elif tick % 10 == 0:
                    kind = "stayed"
                else:
                    continue
                for layer in range(L):
                    o_ref, l_ref = oracle_step(wl, s, layer, n, p0=int(p0[s]))
                    o = out[layer * a * hq * d:][: a * hq * d].view(a, 1, hq, d)[idx].float().cpu().numpy()
                    lv = lse[layer * a * hq:][: a * hq].view(a, 1, hq)[idx].cpu().numpy()
                    assert np.abs(o - o_ref).max() <= OUT_TOL, (s, layer, n, tick)
                    assert (np.abs(lv - l_ref) / np.maximum(1.0, np.abs(l_ref))).max() <= LSE_TOL, (s, layer, n)
                checked[kind] += 1
    h.sync_status()
    for s in range(S):
        assert list(h.stream_state(s).values()) == rings[s].state(), s
    assert min(checked.values()) > 5, checked
    h.close()


def test_reset_streams_reports_bad_entries():
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv

    h = rkv.RollingKV([8, 8], [0, 0], n_layers=1, n_streams=2, n_q_heads=4, n_kv_heads=2, head_dim=64,
                      q_per_step=1, scheme=0, page_size=16)
    ids = torch.tensor([-1, 1, 5], dtype=torch.int32, device="cuda")
    p0 = torch.tensor([0, 7, 0], dtype=torch.int64, device="cuda")
    h.reset_streams(ids, p0)
    with pytest.raises(rkv.RkvError) as e:
        h.sync_status()
    assert e.value.code == rkv.RKV_ERR_DEVICE_BOUNDS
    assert h.stream_state(1)["P0"] == 7 and h.stream_state(0)["P0"] == 0
    h.close()
