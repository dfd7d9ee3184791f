"""Ring state on the device against the integer model, and the call-order rules."""
import numpy as np
import pytest

import synth
from rkv_harness import run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,overrides", [
    ("tiny", dict(extra={"window": 7}, n_kv_heads=2)),
    ("tiny", dict(extra={"window": 5}, rebase_interval=3)),
    ("encoder", dict(n_layers=1, n_streams=3, extra={"window": 10})),
    ("mixed", dict(n_layers=1, n_streams=12)),
    # eviction in batches (ring capacity above the window)
    ("tiny", dict(extra={"window": 7}, window_slack=5)),
    ("encoder", dict(n_layers=1, n_streams=3, extra={"window": 10}, window_slack=10)),
    ("mixed", dict(n_layers=1, n_streams=12, window_slack=3, scheme=2)),
])
def test_state_bit_exact(name, overrides):
    wl = synth.workload(name, **overrides)
    run = run_gpu(wl, 40, set())
    for s, st in run.states.items():
        assert list(st.values()) == run.ring[s].state(), f"stream {s}"


def _small(rkv, scheme=1, n_layers=2):
    import torch
    h = rkv.RollingKV([8, 8], [0, 5], n_layers=n_layers, n_streams=2, n_q_heads=4, n_kv_heads=2, head_dim=64,
                      q_per_step=1, scheme=scheme, page_size=16)
    q = torch.zeros(2, 1, 4, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(2, 1, 2, 64, dtype=torch.bfloat16, device="cuda")
    return h, q, k, k.clone(), q.clone()


def test_call_order_errors():
    import rolling_kv_sliding_rkv_b300 as rkv
    h, q, k, v, out = _small(rkv)
    with pytest.raises(rkv.RkvError) as e:
        h.append_rope(0, k, v)                         # no step open
    assert e.value.code == rkv.RKV_ERR_STATE
    with pytest.raises(rkv.RkvError) as e:
        h.begin_step([0, 0])                              # duplicate id
    assert e.value.code == rkv.RKV_ERR_INVALID_ARG
    with pytest.raises(rkv.RkvError) as e:
        h.begin_step([2])                                 # id out of range
    assert e.value.code == rkv.RKV_ERR_INVALID_ARG
    h.begin_step([0, 1])
    with pytest.raises(rkv.RkvError) as e:
        h.decode_attn(0, q, out)                          # before append
    assert e.value.code == rkv.RKV_ERR_STATE
    h.rebase(0)
    h.append_rope(0, k, v)
    with pytest.raises(rkv.RkvError) as e:
        h.append_rope(0, k, v)                         # twice
    assert e.value.code == rkv.RKV_ERR_STATE
    with pytest.raises(rkv.RkvError) as e:
        h.rebase(0)                                       # twice
    assert e.value.code == rkv.RKV_ERR_STATE
    h.decode_attn(0, q, out)
    with pytest.raises(rkv.RkvError) as e:
        h.begin_step([0, 1])                              # layer 1 never appended
    assert e.value.code == rkv.RKV_ERR_STATE
    with pytest.raises(rkv.RkvError) as e:
        h.append_rope(2, k, v)                         # layer out of range
    assert e.value.code == rkv.RKV_ERR_INVALID_ARG
    h.rebase(1)
    h.append_rope(1, k, v)
    h.begin_step([1])
    h.sync_status()
    h.close()
    h, q, k, v, out = _small(rkv, scheme=0, n_layers=1)
    h.begin_step([0])
    with pytest.raises(rkv.RkvError) as e:
        h.rebase(0)                                       # offset-only has no re-base
    assert e.value.code == rkv.RKV_ERR_STATE
    h.close()


def test_create_errors():
    import torch
    import rolling_kv_sliding_rkv_b300 as rkv
    cfg = rkv.make_config(n_layers=1, n_streams=2, n_q_heads=4, n_kv_heads=2, head_dim=64, q_per_step=1)
    pool_b, state_b = rkv.rkv_required_bytes(cfg, [8, 8])
    pool = torch.empty(pool_b, dtype=torch.uint8, device="cuda")
    state = torch.empty(state_b, dtype=torch.uint8, device="cuda")
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_create(cfg, [8, 8], [0, 0], pool, pool_b - 1, state, state_b)
    assert e.value.code == rkv.RKV_ERR_CAPACITY
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_create(cfg, [8, 8], [0, -1], pool, pool_b, state, state_b)
    assert e.value.code == rkv.RKV_ERR_CONFIG
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_create(cfg, [8, 8], [0, 0], pool.data_ptr() + 16, pool_b - 16, state, state_b)
    assert e.value.code == rkv.RKV_ERR_INVALID_ARG
    h = rkv.rkv_create(cfg, [8, 8], [0, 0], pool, pool_b, state, state_b)
    rkv.rkv_destroy(h)


def test_memory_constant_over_steps():
    import torch
    import rolling_kv_sliding_rkv_b300 as rkv
    h, q, k, v, out = _small(rkv, scheme=1, n_layers=1)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for i in range(3000):
        h.begin_step([0, 1])
        h.rebase(0)
        h.append_rope(0, k, v)
        h.decode_attn(0, q, out)
        if i in (10, 2999):
            torch.cuda.synchronize()
            assert torch.cuda.mem_get_info()[0] == free0
    h.sync_status()
    h.close()


def test_decode_attn_layers_matches_per_layer_calls():
    """rkv_decode_attn_layers (several layers in one launch) gives the per-layer results."""
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv

    wl = synth.workload("qwen", n_layers=3, n_streams=4, extra={"window": 100})
    S, L, hq, hkv, d = wl.n_streams, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    h = rkv.RollingKV(wl.windows().tolist(), wl.start_offsets().tolist(), n_layers=L, n_streams=S, n_q_heads=hq,
                      n_kv_heads=hkv, head_dim=d, q_per_step=1, scheme=1, rope_theta=wl.rope_theta)
    q = torch.randn(L, S, 1, hq, d, device="cuda").mul_(0.1).to(torch.bfloat16)
    k = torch.randn(L, S, 1, hkv, d, device="cuda").mul_(0.1).to(torch.bfloat16)
    v = torch.randn(L, S, 1, hkv, d, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(q)
    lse = torch.empty(L, S, 1, hq, device="cuda")
    act = list(range(S))
    for _ in range(120):
        h.step(act, q, k, v, out, lse)
    h.begin_step(act)
    with pytest.raises(rkv.RkvError) as e:
        h.decode_attn_layers(0, L, q, out, lse)        # before the layers are appended
    assert e.value.code == rkv.RKV_ERR_STATE
    for layer in range(L):
        h.rebase(layer)
        h.append_rope(layer, k[layer], v[layer])
    out_a, lse_a = torch.empty_like(out), torch.empty_like(lse)
    for layer in range(L):
        h.decode_attn(layer, q[layer], out_a[layer], lse_a[layer])
    h.decode_attn_layers(0, L, q, out, lse)
    h.decode_attn_layers(1, 2, q[1:], out[1:], lse[1:])  # a sub-range
    h.sync_status()
    assert (out.float() - out_a.float()).abs().max().item() <= 1e-2
    assert (lse - lse_a).abs().max().item() <= 1e-4
    for bad in ((-1, 1), (0, L + 1), (2, 2), (0, 0)):
        with pytest.raises(rkv.RkvError) as e:
            h.decode_attn_layers(bad[0], bad[1], q, out, lse)
        assert e.value.code == rkv.RKV_ERR_INVALID_ARG
    h.close()


@pytest.mark.parametrize("scheme", [0, 1, 2])
def test_key_outside_fp16_range_is_reported(scheme):
    """A rotated key that cannot be stored in fp16 is reported by rkv_sync_status, once."""
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv
    h, q, k, v, out = _small(rkv, scheme=scheme, n_layers=1)
    h.begin_step([0, 1])
    k.fill_(1.0e5)          # |R(p) k| >= 1e5 > 65504 in at least one element of every pair
    if scheme:
        h.rebase(0)
    h.append_rope(0, k, v)
    h.decode_attn(0, q, out)
    with pytest.raises(rkv.RkvError) as e:
        h.sync_status()
    assert e.value.code == rkv.RKV_ERR_DEVICE_RANGE
    h.sync_status()         # the status word was cleared
    h.close()


def test_device_memory_is_constant_over_steps():
    """Memory does not grow with the stream's length: no allocation after create (T8)."""
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv
    wl = synth.workload("qwen", n_layers=2, n_streams=8, extra={"window": 64})
    S, L, hq, hkv, d = wl.n_streams, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    h = rkv.RollingKV(wl.windows().tolist(), wl.start_offsets().tolist(), n_layers=L, n_streams=S, n_q_heads=hq,
                      n_kv_heads=hkv, head_dim=d, q_per_step=1, scheme=1, rope_theta=wl.rope_theta)
    q = torch.zeros(L, S, 1, hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(L, S, 1, hkv, d, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    act = list(range(S))
    for _ in range(5):
        h.step(act, q, k, k, out)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(600):            # ~9 windows
        h.step(act, q, k, k, out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert h.stream_state(0)["n"] == 605
    h.sync_status()
    h.close()
