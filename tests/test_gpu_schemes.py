"""The two exact schemes against each other, far tighter than either against the oracle.

The materialised exact re-base (rkv_rebase writes every retained key rotated by R(j - rope_base),
Audio8 ASR Infinite 无限长转写原理, 第 2 步) and the same re-base applied while the attention
kernel reads the keys place every key at the same window-relative position and round it once to
fp16; their cos/sin differ only by the ~1e-6 of the recurrences along a run of 8 ring slots.
So their outputs agree to the rounding of the bf16 output itself, and their logsumexps to 1e-4
(relative): a misplaced, mis-signed or stale rotation in either path would show far above that, even
where it could hide under the oracle tolerances of 2e-2 / 1e-3.
"""
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,over", [
    ("qwen", dict(n_layers=2, n_streams=5, extra={"window": 100})),
    # d = 64, Q = 4; inputs scaled by 1/sqrt(d) like the Qwen-shaped ones, so that one fp16
    # rounding step of a unit-size key does not move a score by ~1e-3 on its own
    ("encoder", dict(n_layers=1, n_streams=3, extra={"window": 70}, scale_inputs=True)),
    ("tiny", dict(n_layers=1, n_streams=2, extra={"window": 150}, rebase_interval=5)),
])
def test_exact_schemes_agree(name, over):
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv

    runs = {}
    for scheme in (1, 2):
        wl = synth.workload(name, scheme=scheme, **over)
        S, L, Q, hq, hkv, d = wl.n_streams, wl.n_layers, wl.q_per_step, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
        h = rkv.RollingKV(wl.windows().tolist(), wl.start_offsets().tolist(), n_layers=L, n_streams=S,
                          n_q_heads=hq, n_kv_heads=hkv, head_dim=d, q_per_step=Q, scheme=scheme,
                          rebase_interval=wl.rebase_interval, rope_theta=wl.rope_theta)
        q = torch.empty(S, Q, hq, d, dtype=torch.bfloat16, device="cuda")
        k = torch.empty(S, Q, hkv, d, dtype=torch.bfloat16, device="cuda")
        v = torch.empty_like(k)
        out = torch.empty_like(q)
        lse = torch.empty(S, Q, hq, dtype=torch.float32, device="cuda")
        rec = []
        W = int(wl.windows().max())
        steps = (W + 40) // Q            # the windows fill, then roll for 40 tokens
        for step in range(steps):
            h.begin_step(list(range(S)))
            for layer in range(L):
                h.gen_step_inputs(wl.seed, layer, wl.input_scale, q, k, v)
                h.rebase(layer)          # a no-op launch-wise when rotating on read
                h.append_rope(layer, k, v)
                h.decode_attn(layer, q, out, lse)
                if step % max(1, 9 // Q) == 0 or step >= steps - 3:
                    rec.append((out.float().clone(), lse.clone()))
        h.sync_status()
        h.close()
        runs[scheme] = rec
    worst_l = 0.0
    for (o1, l1), (o2, l2) in zip(runs[1], runs[2]):
        # one bf16 rounding step of the output (at most 2^-7 relative), plus 5e-4
        bound = torch.maximum(o1.abs(), o2.abs()) * 2.0 ** -7 + 5e-4
        assert ((o1 - o2).abs() <= bound).all(), (o1 - o2).abs().max().item()
        worst_l = max(worst_l, ((l1 - l2).abs() / l1.abs().clamp(min=1.0)).max().item())
    assert worst_l <= 1e-4, worst_l
    assert len(runs[1]) == len(runs[2]) > 10
