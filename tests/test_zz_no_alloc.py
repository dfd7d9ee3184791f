"""rkv_decode_attn_static: decode attention for callers that may not allocate.

A real-time audio callback cannot risk an allocator call inside its clock
step, and a plug-in inside a serving engine may find the free HBM already
held by the engine's allocator.  The static entry point keeps its split-K
scratch in a fixed array inside the library; here it must give the same
outputs as rkv_decode_attn, call after call, through the C ABI.
"""
import pytest

import synth

pytestmark = pytest.mark.gpu

OUT_TOL, LSE_TOL = 2e-2, 1e-3


def _close(a_out, a_lse, b_out, b_lse):
    e_o = (a_out.float() - b_out.float()).abs().max().item()
    e_l = ((a_lse - b_lse).abs() / b_lse.abs().clamp(min=1.0)).max().item()
    assert e_o <= OUT_TOL and e_l <= LSE_TOL, (e_o, e_l)


def test_static_scratch_matches_regular_entry_point():
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv

    dev = torch.device("cuda")
    wl = synth.workload("qwen", n_layers=2, n_streams=8, extra={"window": 150})
    h = rkv.RollingKV(wl.windows().tolist(), wl.start_offsets().tolist(), device=dev, n_layers=wl.n_layers,
                      n_streams=wl.n_streams, n_q_heads=wl.n_q_heads, n_kv_heads=wl.n_kv_heads,
                      head_dim=wl.head_dim, q_per_step=wl.q_per_step, scheme=wl.scheme, rope_theta=wl.rope_theta)
    S, L, hq, hkv, d = wl.n_streams, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    q = torch.empty(S, 1, hq, d, dtype=torch.bfloat16, device=dev)
    k = torch.empty(S, 1, hkv, d, dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    out_ref, out_a, out_b = (torch.empty_like(q) for _ in range(3))
    lse_ref, lse_a, lse_b = (torch.empty(S, 1, hq, dtype=torch.float32, device=dev) for _ in range(3))
    active = list(range(S))
    compared = 0
    for step in range(160):          # the window of 150 fills and rolls
        h.begin_step(active)
        for layer in range(L):
            h.gen_step_inputs(wl.seed, layer, wl.input_scale, q, k, v)
            h.rebase(layer)
            h.append_rope(layer, k, v)
            h.decode_attn(layer, q, out_ref, lse_ref)
            if step in (0, 149, 158, 159):
                # two calls in a row of the static entry point, each against the regular one
                rkv.rkv_decode_attn_static(h.handle, layer, q, out_a, lse_a)
                rkv.rkv_decode_attn_static(h.handle, layer, q, out_b, lse_b)
                torch.cuda.synchronize()
                _close(out_a, lse_a, out_ref, lse_ref)
                _close(out_b, lse_b, out_ref, lse_ref)
                compared += 2
    h.sync_status()
    assert compared == 16
    h.close()


def test_static_scratch_rejects_oversized_calls():
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv

    dev = torch.device("cuda")
    # 1024 streams x 16 query heads x (128 + 2) floats of partials is above 8 MiB; with 1024
    # (stream, kv head) units there are more than enough CTAs, so the window is never split
    S = 1024
    h = rkv.RollingKV([8] * S, [0] * S, device=dev, n_layers=1, n_streams=S, n_q_heads=16, n_kv_heads=1,
                      head_dim=128, q_per_step=1, scheme=0, page_size=16)
    q = torch.zeros(S, 1, 16, 128, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(S, 1, 1, 128, dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    h.begin_step(list(range(S)))
    h.append_rope(0, k, k)
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_decode_attn_static(h.handle, 0, q, out)
    assert e.value.code == rkv.RKV_ERR_CAPACITY and "fixed array" in str(e.value)
    h.decode_attn(0, q, out)          # the regular entry point still serves this size
    h.sync_status()
    h.close()
