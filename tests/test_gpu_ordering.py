"""Queries written by the kernel launched just before rkv_decode_attn.

The attention kernel is launched with programmatic dependent launch, so it may
start while its predecessor still runs.  rkv_decode_attn promises to read q only
after that predecessor has completed; here the predecessor is a generator
kernel that lets its dependents launch before it writes q (as a caller's q-norm
kernel with programmatic launch might), and the buffer held zeros until then.
A read of q before the dependency wait would attend with a zero query (the
mean of the window's values), far outside the oracle tolerance.
"""
import numpy as np
import pytest

import synth
from rkv_harness import LSE_TOL, OUT_TOL, oracle_step

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("scheme", [0, 1, 2])
def test_q_written_by_the_immediate_predecessor(scheme):
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv

    wl = synth.workload("tiny", n_layers=2, n_streams=3, extra={"window": 150}, scheme=scheme)
    S, L, hq, hkv, d = wl.n_streams, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    h = rkv.RollingKV(wl.windows().tolist(), wl.start_offsets().tolist(), n_layers=L, n_streams=S, n_q_heads=hq,
                      n_kv_heads=hkv, head_dim=d, q_per_step=1, scheme=scheme, rope_theta=wl.rope_theta)
    q = torch.empty(S, 1, hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(S, 1, hkv, d, dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    kk, vv = torch.empty_like(k), torch.empty_like(k)
    out = torch.empty_like(q)
    lse = torch.empty(S, 1, hq, dtype=torch.float32, device="cuda")
    checked = 0
    for step in range(160):
        h.begin_step(list(range(S)))
        for layer in range(L):
            h.gen_step_inputs(wl.seed, layer, wl.input_scale, q, k, v)
            kk.copy_(k)
            vv.copy_(v)
            if scheme:
                h.rebase(layer)
            h.append_rope(layer, kk, vv)
            q.zero_()
            h.gen_step_inputs(wl.seed, layer, wl.input_scale, q, k, v)   # writes q; the next launch
            h.decode_attn(layer, q, out, lse)                            # is the attention
            if step % 13 == 0 or step >= 157:
                torch.cuda.synchronize()
                for s in range(S):
                    o_ref, l_ref = oracle_step(wl, s, layer, step)
                    o = out[s].float().cpu().numpy()
                    lv = lse[s].cpu().numpy()
                    assert np.abs(o - o_ref).max() <= OUT_TOL, (step, layer, s)
                    assert (np.abs(lv - l_ref) / np.maximum(1.0, np.abs(l_ref))).max() <= LSE_TOL
                    checked += 1
    h.sync_status()
    h.close()
    assert checked == 2 * 3 * 16
