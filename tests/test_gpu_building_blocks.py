"""Device building blocks against their host definitions: input generator, RoPE angles."""
import numpy as np
import pytest

import synth
from oracle.rope import cos_sin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rkv():
    import rolling_kv_sliding_rkv_b300 as m
    return m


def test_generator_bit_identical(rkv):
    import torch
    cases = [(20260101, synth.TAG_Q, 0, 0, 0, 3, 16 * 128, 1.0),
             (20260102, synth.TAG_K, 63, 35, 4999, 2, 2 * 128, float(np.float32(1 / np.sqrt(128)))),
             (20260104, synth.TAG_V, 255, 7, 2 ** 40 + 3, 4, 20 * 64, 1.0),
             (1, 17, 5, 2, 123456789, 1, 1000, 0.37)]
    for seed, tag, s, layer, tok0, nt, width, scale in cases:
        out = torch.empty(nt * width, dtype=torch.bfloat16, device="cuda")
        rkv.rkv_gen_tokens(seed, tag, s, layer, tok0, nt, width, scale, out)
        dev = out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(nt, width)
        key = synth.counter_key(seed, tag, s, layer, np.arange(tok0, tok0 + nt))
        host = synth.normal_bf16_bits(key, width, scale)
        assert np.array_equal(dev, host)


@pytest.mark.parametrize("head_dim", [64, 128])
def test_rope_cos_sin_exact_at_large_positions(rkv, head_dim):
    import torch
    rng = np.random.default_rng(3)
    pos = np.concatenate([[0, 1, 374, 375, 1_079_999, 2_000_000, 2 ** 31 + 5, 2 ** 40, 2 ** 52 - 1, -7],
                          rng.integers(0, 2 ** 52, 40)]).astype(np.int64)
    pos_d = torch.from_numpy(pos).cuda()
    cs = torch.empty(len(pos), head_dim // 2, 2, dtype=torch.float32, device="cuda")
    rkv.rkv_rope_cossin(pos_d, len(pos), head_dim, 1e6, cs)
    got = cs.cpu().numpy().astype(np.float64)
    c, s = cos_sin(pos, head_dim, 1e6)
    # fp32 rounding of an fp64 value accurate to ~1e-15: within 2^-24 relative plus a hair
    assert np.abs(got[..., 0] - c).max() < 1.2e-7
    assert np.abs(got[..., 1] - s).max() < 1.2e-7


def test_next_step_generator_bit_identical(rkv):
    """rkv_gen_next_inputs: every layer of the next step of a subset of streams, in rkv_step's layout,
    with each stream's token index read from the device state (streams at different counts)."""
    import torch
    L, S, hq, hkv, d, Q = 3, 5, 8, 2, 64, 2
    h = rkv.RollingKV([16] * S, [0] * S, n_layers=L, n_streams=S, n_q_heads=hq, n_kv_heads=hkv, head_dim=d,
                      q_per_step=Q, scheme=0, page_size=16)
    zq = torch.zeros(S, Q, hq, d, dtype=torch.bfloat16, device="cuda")
    zk = torch.zeros(S, Q, hkv, d, dtype=torch.bfloat16, device="cuda")
    counts = [0] * S
    for active in ([0, 1, 2, 3, 4], [1, 3], [3]):     # streams 0..4 at 2, 4, 2, 6, 2 tokens
        h.begin_step(active)
        for layer in range(L):
            h.append_rope(layer, zk, zk)
        for s in active:
            counts[s] += Q
    h.sync_status()
    active = [3, 0, 1]
    seed, scale = 99, 0.5
    q = torch.empty(L, len(active), Q, hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(L, len(active), Q, hkv, d, dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    h.gen_next_inputs(seed, active, scale, q, k, v)
    torch.cuda.synchronize()
    for tag, buf, heads in ((synth.TAG_Q, q, hq), (synth.TAG_K, k, hkv), (synth.TAG_V, v, hkv)):
        got = buf.view(torch.int16).cpu().numpy().view(np.uint16)
        for layer in range(L):
            for a, s in enumerate(active):
                want = synth.token_tensor(seed, tag, s, layer, range(counts[s], counts[s] + Q), heads, d, scale)
                assert np.array_equal(got[layer, a], np.asarray(want).reshape(Q, heads, d)), (tag, layer, s)
    h.close()
