"""rkv_decode_attn_static: decode attention for callers that may not allocate.

A real-time audio callback cannot risk an allocator call inside its clock
step, and a plug-in inside a serving engine may find the free HBM already
held by the engine's allocator.  The static entry point keeps the partial
results of a split window in a fixed array inside the library.  Here it is
checked through the C ABI against the fp64 oracle, and against
rkv_decode_attn call after call: when neither call splits the windows the two
run the same launch and agree bit for bit; when they split, they merge in a
different order and agree to the rounding of the bf16 output.
"""
import pytest

import synth
from rkv_harness import compare, run_gpu

pytestmark = pytest.mark.gpu


def _close_to_rounding(a_out, a_lse, b_out, b_lse):
    """Outputs within one bf16 rounding step of each other plus 1e-4, logsumexps within 1e-5.

    With the same split plan the two calls differ only in the fp32 order of the merge.  With
    different plans (a long window: 8 splits in a cluster against 32 with the merge kernel) each
    split also rounds its softmax weights to bf16 against its own running maximum, so the
    weights differ by up to 2^-9 relative; over the 2000 keys of a window that moves an output of
    unit-scale values by a few 1e-5 at most (3.1e-5 measured on the B300).
    """
    a, b = a_out.float(), b_out.float()
    bound = a.abs().maximum(b.abs()) * 2.0 ** -7 + 1e-4
    assert ((a - b).abs() <= bound).all(), (a - b).abs().max().item()
    e_l = ((a_lse - b_lse).abs() / b_lse.abs().clamp(min=1.0)).max().item()
    assert e_l <= 1e-5, e_l


@pytest.mark.parametrize("n_streams,window", [(8, 150), (1, 2000)])
def test_static_scratch_matches_regular_entry_point(n_streams, window):
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv

    dev = torch.device("cuda")
    wl = synth.workload("qwen", n_layers=2, n_streams=n_streams, extra={"window": window})
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
    checkpoints = {0, window - 1, window + 8, window + 9}
    for step in range(window + 10):          # the window fills and rolls
        h.begin_step(active)
        for layer in range(L):
            h.gen_step_inputs(wl.seed, layer, wl.input_scale, q, k, v)
            h.rebase(layer)
            h.append_rope(layer, k, v)
            h.decode_attn(layer, q, out_ref, lse_ref)
            if step in checkpoints:
                # two calls in a row of the static entry point, each against the regular one
                rkv.rkv_decode_attn_static(h.handle, layer, q, out_a, lse_a)
                rkv.rkv_decode_attn_static(h.handle, layer, q, out_b, lse_b)
                torch.cuda.synchronize()
                _close_to_rounding(out_a, lse_a, out_ref, lse_ref)
                assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)
                compared += 2
    h.sync_status()
    assert compared == 2 * len(checkpoints) * L
    h.close()


@pytest.mark.parametrize("case", ["split3", "split32"])
def test_static_scratch_against_oracle(case):
    """The split-K partials and their merge kernel, every output of every step, against the oracle."""
    over = (dict(n_layers=1, n_streams=3, extra={"window": 150}) if case == "split3"
            else dict(n_layers=1, n_streams=1, extra={"window": 2000}))
    wl = synth.workload("tiny", **over)
    ticks = int(wl.windows()[0]) + 12
    samples = {(s, 0, n) for s in range(wl.n_streams) for n in range(0, ticks, 1 if case == "split3" else 97)}
    run = run_gpu(wl, ticks, samples, attn="static")
    assert set(run.samples) == samples
    compare(run, wl)


def test_static_scratch_unsplit_large_batch():
    """1024 streams: more (stream, kv head) units than CTA slots, so nothing splits; the static call
    then touches no scratch, takes the same launch as rkv_decode_attn and gives the same bits."""
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv

    dev = torch.device("cuda")
    S = 1024
    wl = synth.workload("qwen", n_layers=1, n_streams=S, n_q_heads=16, n_kv_heads=1, extra={"window": 40})
    h = rkv.RollingKV(wl.windows().tolist(), wl.start_offsets().tolist(), device=dev, n_layers=1, n_streams=S,
                      n_q_heads=16, n_kv_heads=1, head_dim=128, q_per_step=1, scheme=1, rope_theta=wl.rope_theta)
    q = torch.empty(S, 1, 16, 128, dtype=torch.bfloat16, device=dev)
    k = torch.empty(S, 1, 1, 128, dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    out_ref, out_a = torch.empty_like(q), torch.empty_like(q)
    lse_ref, lse_a = (torch.empty(S, 1, 16, dtype=torch.float32, device=dev) for _ in range(2))
    for step in range(45):
        h.begin_step(list(range(S)))
        h.gen_step_inputs(wl.seed, 0, wl.input_scale, q, k, v)
        h.rebase(0)
        h.append_rope(0, k, v)
        h.decode_attn(0, q, out_ref, lse_ref)
        if step in (0, 39, 44):
            for _ in range(2):
                rkv.rkv_decode_attn_static(h.handle, 0, q, out_a, lse_a)
                torch.cuda.synchronize()
                assert torch.equal(out_a, out_ref) and torch.equal(lse_a, lse_ref)
    h.sync_status()
    h.close()
