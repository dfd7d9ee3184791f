"""Negative controls: shortcuts the design rejects must fail the parity tolerance.

Both simulate, in numpy, what a GPU kernel would do with the shortcut and
compare with the fp64 oracle.  Tolerances are those the CUDA path is held to:
max |out error| <= 2e-2 and |lse error| <= 1e-3 * max(1, |lse|).
"""
import math

import numpy as np
import pytest

import synth
from oracle.attention import attention_step
from oracle.rope import cos_sin, omegas
from synth import generator as g

OUT_TOL, LSE_TOL = 2e-2, 1e-3


def _bf16(x):
    return g.bf16_bits_to_f64(g.f32_to_bf16_bits(np.asarray(x, dtype=np.float32)))


def _rotate_f32(x, c, s):
    x = np.asarray(x, dtype=np.float32)
    h = x.shape[-1] // 2
    a, b = x[..., :h], x[..., h:]
    return np.concatenate([a * c - b * s, a * s + b * c], -1).astype(np.float32)


def _attend(qr, kr, v, scale):
    s = kr @ qr * scale
    m = s.max()
    e = np.exp(s - m)
    return e @ v / e.sum(), m + math.log(e.sum())


def _errors(o, lse, o_ref, lse_ref):
    return np.abs(o - o_ref).max(), np.abs(lse - lse_ref).max() / max(1.0, np.abs(lse_ref).max())


def test_fp32_angles_drift_at_large_positions():
    d, theta = 128, 1e6
    w = omegas(d, theta).astype(np.float32)
    # cos/sin level: at 2e6 (about 44 h at 12.5 Hz) an fp32 product p*omega is off by up to ulp/2 = 0.06 rad
    p = np.arange(2_000_000, 2_000_064)
    c_exact, _ = cos_sin(p, d, theta)
    c32 = np.cos((p.astype(np.float32)[:, None] * w[None, :]).astype(np.float32))
    assert np.abs(c32 - c_exact).max() > 1e-2
    # attention level, one Qwen-shaped head group of the unscaled tiny workload at P0 = 2^31 + 5
    hq, hkv, win, n, p0 = 16, 2, 375, 400, 2 ** 31 + 5
    toks = np.arange(n - win + 1, n + 1)
    q = g.bf16_bits_to_f64(synth.token_tensor(1, synth.TAG_Q, 0, 0, [n], hq, d))
    k = g.bf16_bits_to_f64(synth.token_tensor(1, synth.TAG_K, 0, 0, toks, hkv, d))
    v = g.bf16_bits_to_f64(synth.token_tensor(1, synth.TAG_V, 0, 0, toks, hkv, d))
    o_ref, lse_ref = attention_step(q, k, v, toks, n, p0, win, 1 / math.sqrt(d), theta)
    ang_k = ((p0 + toks).astype(np.float32)[:, None] * w[None, :]).astype(np.float32)
    ang_q = np.float32(p0 + n) * w
    kr = _bf16(_rotate_f32(k, np.cos(ang_k)[:, None], np.sin(ang_k)[:, None]))
    qr = _bf16(_rotate_f32(q[0], np.cos(ang_q), np.sin(ang_q)))
    o = np.zeros((hq, d))
    lse = np.zeros(hq)
    for h in range(hq):
        o[h], lse[h] = _attend(qr[h], kr[:, h // 8], v[:, h // 8], 1 / math.sqrt(d))
    e_out, e_lse = _errors(o, lse, o_ref[0], lse_ref[0])
    assert e_out > OUT_TOL or e_lse > LSE_TOL


@pytest.mark.slow
def test_in_place_bf16_rebase_drifts_but_rederivation_does_not():
    """Rotating stored bf16 keys by R(-1) on every roll compounds W-1 roundings.

    Tiny workload shape (W = 375, unscaled, one KV head with its 8 query heads,
    1000 steps, exact re-base every step once full).  Re-deriving each stored
    key from its pre-RoPE copy at the new window-relative position, which is
    what the library does, keeps a single rounding.
    """
    d, hq, win, steps, theta = 128, 8, 375, 1000, 1e6
    seed = synth.workload("tiny").seed
    k = g.bf16_bits_to_f64(synth.token_tensor(seed, synth.TAG_K, 0, 0, np.arange(steps), 1, d))[:, 0]
    v = g.bf16_bits_to_f64(synth.token_tensor(seed, synth.TAG_V, 0, 0, np.arange(steps), 1, d))[:, 0]
    c_tab, s_tab = (x.astype(np.float32) for x in cos_sin(np.arange(win), d, theta))
    c_m1, s_m1 = (x.astype(np.float32)[0] for x in cos_sin([-1], d, theta))
    stored = np.zeros((steps, d), dtype=np.float64)     # in-place scheme, by token index
    worst_inplace = worst_rederive = 0.0
    evicted = 0
    for t in range(steps):
        n = t + 1
        ev = max(0, n - win)
        if ev > evicted:                                 # roll: R(-1) on every retained key
            stored[ev:t] = _bf16(_rotate_f32(stored[ev:t], c_m1, s_m1))
        evicted = ev
        rel = t - ev
        stored[t] = _bf16(_rotate_f32(k[t], c_tab[rel], s_tab[rel]))
        if t in (350, 600, 800, 999):
            q = g.bf16_bits_to_f64(synth.token_tensor(seed, synth.TAG_Q, 0, 0, [t], hq, d))
            toks = np.arange(ev, t + 1)
            o_ref, lse_ref = attention_step(q, k[toks, None], v[toks, None], toks, t, 0, win,
                                            1 / math.sqrt(d), theta)
            qr = _bf16(_rotate_f32(q[0], c_tab[rel], s_tab[rel]))
            rederived = _bf16(_rotate_f32(k[toks], c_tab[toks - ev], s_tab[toks - ev]))
            for keys, tag in ((stored[toks], "inplace"), (rederived, "rederive")):
                o = np.zeros((hq, d))
                lse = np.zeros(hq)
                for h in range(hq):
                    o[h], lse[h] = _attend(qr[h], keys, v[toks], 1 / math.sqrt(d))
                e_out, e_lse = _errors(o, lse, o_ref[0], lse_ref[0])
                score = max(e_out / OUT_TOL, e_lse / LSE_TOL)
                if tag == "inplace":
                    worst_inplace = max(worst_inplace, score)
                else:
                    worst_rederive = max(worst_rederive, score)
    print("worst in-place / re-derived, in units of the tolerance:", worst_inplace, worst_rederive)
    assert worst_inplace > 1.0          # compounded roundings break the tolerance
    assert worst_rederive < 0.5         # one rounding stays well inside it
