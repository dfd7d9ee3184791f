"""Windowed attention for one stream and one layer, in fp64.

Definition (the result the rolling cache is meant to reproduce exactly):

* Token j of a stream has absolute position P0 + j (voxtral.c rolling-KV
  article, §二: logical position = physical index + kv_pos_offset, i.e. the
  token's place in the whole sequence).
* A step appends Q tokens n .. n+Q-1 (Q = 1 for the decoder, one text token
  per clock step: model card "亮点"; Q = frame_len = 4 for the audio tower's
  incremental step: voxtral.c article §三).  The window keeps the last W
  tokens (explainer, "Rolling KV Cache 三步拆解", 第 1 步; voxtral.c article
  §二 keeps the last VOX_DEC_WINDOW positions).
* Query token n+i attends key tokens j with lo <= j <= n+i, where
  lo = max(0, n+Q-W) (for Q = 1 this is t-W < j <= t).  All queries of a
  multi-query step share the cache as it stands after the step's append, with
  a causal mask inside the step (reading of voxtral.c §三: compact when
  cache length + new length exceeds the window, then encode the new
  positions against the cache).  ``per_query_window=True`` selects the
  alternative reading t-W < j <= t for every query.  With eviction in
  batches (a ring of capacity above W, oracle/ring.py), the shared cache
  starts at the first retained token instead: ``first_key`` = evicted after
  the step, which replaces n+Q-W as the lower bound.
* q head h reads kv head floor(h / G), G = Hq / Hkv (contiguous GQA groups;
  Qwen2.5-3B has 16 query / 2 KV heads, model card "架构").
* s_j = <R(p_t) q, R(p_j) k_j> * scale; o = sum_j softmax(s)_j v_j;
  lse = ln sum_j exp(s_j) (natural log of the scaled scores).
"""
from __future__ import annotations

import math

import numpy as np

from .rope import rotate


def visible_keys(n: int, q_per_step: int, window: int, per_query_window: bool = False,
                 first_key: int | None = None):
    """For each query i < Q: (lo, hi) inclusive token range it attends."""
    out = []
    for i in range(q_per_step):
        t = n + i
        if first_key is not None:
            lo = first_key
        else:
            lo = t - window + 1 if per_query_window else n + q_per_step - window
        out.append((max(0, lo), t))
    return out


def attention_step(q_new, k_tok, v_tok, key_tokens, n: int, p0: int, window: int,
                   scale: float, theta: float, pairing: str = "half",
                   per_query_window: bool = False, first_key: int | None = None):
    """Outputs of one step.

    q_new   [Q][Hq][d]   raw (pre-RoPE) queries of tokens n .. n+Q-1
    k_tok   [T][Hkv][d]  raw keys of the tokens listed in key_tokens
    v_tok   [T][Hkv][d]  values of the same tokens
    key_tokens           token indices of k_tok/v_tok rows; must contain every
                         token some query attends
    Returns o [Q][Hq][d] and lse [Q][Hq] in fp64.
    """
    q_new = np.asarray(q_new, dtype=np.float64)
    k_tok = np.asarray(k_tok, dtype=np.float64)
    v_tok = np.asarray(v_tok, dtype=np.float64)
    key_tokens = np.asarray(key_tokens, dtype=np.int64)
    n_q, hq, d = q_new.shape
    hkv = k_tok.shape[1]
    group = hq // hkv
    ranges = visible_keys(n, n_q, window, per_query_window, first_key)
    lo_all = min(r[0] for r in ranges)
    hi_all = max(r[1] for r in ranges)
    keep = (key_tokens >= lo_all) & (key_tokens <= hi_all)
    toks = key_tokens[keep]
    if len(set((lo_all + np.arange(hi_all - lo_all + 1)).tolist()) - set(toks.tolist())):
        raise ValueError("key_tokens does not cover the attended range")
    k_rot = rotate(k_tok[keep], [p0 + int(j) for j in toks], theta, pairing)
    q_rot = rotate(q_new, [p0 + n + i for i in range(n_q)], theta, pairing)
    vv = v_tok[keep]
    o = np.zeros((n_q, hq, d))
    lse = np.zeros((n_q, hq))
    for i, (lo, hi) in enumerate(ranges):
        sel = (toks >= lo) & (toks <= hi)
        for h in range(hq):
            g = h // group
            s = (k_rot[sel, g, :] @ q_rot[i, h, :]) * scale
            m = s.max()
            e = np.exp(s - m)
            z = e.sum()
            o[i, h] = (e @ vv[sel, g, :]) / z
            lse[i, h] = m + math.log(z)
    return o, lse


def attention_step_bruteforce(q_new, k_tok, v_tok, key_tokens, n: int, p0: int, window: int,
                              scale: float, theta: float, per_query_window: bool = False,
                              first_key: int | None = None):
    """Second formulation: explicit loops, angles by math.cos(p * omega) (small p only).

    Half-split pairing.  Written without numpy linear algebra and without the
    exact angle reduction, so that it shares no arithmetic path with
    ``attention_step`` beyond the definition itself.
    """
    n_q, hq, d = len(q_new), len(q_new[0]), len(q_new[0][0])
    hkv = len(k_tok[0])
    half = d // 2
    omega = [theta ** (-2.0 * i / d) for i in range(half)]

    def rot(vec, p):
        out = [0.0] * d
        for i in range(half):
            a, b = float(vec[i]), float(vec[i + half])
            c, s = math.cos(p * omega[i]), math.sin(p * omega[i])
            out[i] = a * c - b * s
            out[i + half] = a * s + b * c
        return out

    row_of = {int(t): r for r, t in enumerate(key_tokens)}
    o = [[[0.0] * d for _ in range(hq)] for _ in range(n_q)]
    lse = [[0.0] * hq for _ in range(n_q)]
    for i in range(n_q):
        t = n + i
        if first_key is not None:
            lo = max(0, first_key)
        else:
            lo = max(0, t - window + 1) if per_query_window else max(0, n + n_q - window)
        for h in range(hq):
            g = h // (hq // hkv)
            qr = rot(q_new[i][h], p0 + t)
            scores, vals = [], []
            for j in range(lo, t + 1):
                kr = rot(k_tok[row_of[j]][g], p0 + j)
                scores.append(sum(a * b for a, b in zip(qr, kr)) * scale)
                vals.append([float(x) for x in v_tok[row_of[j]][g]])
            m = max(scores)
            w = [math.exp(s - m) for s in scores]
            z = sum(w)
            for c in range(d):
                o[i][h][c] = sum(wj * vj[c] for wj, vj in zip(w, vals)) / z
            lse[i][h] = m + math.log(z)
    return np.array(o), np.array(lse)
