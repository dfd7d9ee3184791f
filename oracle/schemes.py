"""fp64 mirrors of the two storage schemes (invariance checks only).

Offset-only (voxtral.c rolling-KV article, §二): RoPE is applied once, when a
key is written, at its logical position P0 + j; keys are never re-encoded.

Exact re-base (Audio8 ASR Infinite 无限长转写原理, "Rolling KV Cache 三步拆解",
第 2 步): on every roll all retained keys are rotated by R(-delta), delta the
number of positions evicted since the last re-base, so the stored positions
restart inside the window; the new query and key use window-relative
positions too.

Both are evaluated in fp64 against a stored-key cache and must equal
``oracle.attention.attention_step`` (absolute positions) up to rounding,
because RoPE scores depend only on position differences.
"""
from __future__ import annotations

import math

import numpy as np

from .ring import SCHEME_EXACT_REBASE, SCHEME_OFFSET_ONLY, StreamRing
from .rope import rotate


class StoredKeyCache:
    """One stream, one layer: a ring of stored (rotated) keys and values."""

    def __init__(self, ring: StreamRing, n_kv_heads: int, head_dim: int, theta: float):
        self.ring = ring
        self.theta = theta
        self.k = np.zeros((ring.C, n_kv_heads, head_dim))
        self.v = np.zeros((ring.C, n_kv_heads, head_dim))

    def step(self, q_new, k_new, v_new, scale: float):
        """Advance the ring by Q tokens and return (o [Q][Hq][d], lse [Q][Hq])."""
        r = self.ring
        n_old = r.n
        r.step()
        if r.scheme == SCHEME_EXACT_REBASE and r.last_delta:
            for j in range(r.evicted, n_old):              # retained old tokens
                s = r.slot(j)
                self.k[s] = rotate(self.k[s][None], [-r.last_delta], self.theta)[0]
        toks = list(range(n_old, r.n))
        pos = [r.rope_position(j) for j in toks]
        k_rot = rotate(np.asarray(k_new, dtype=np.float64), pos, self.theta)
        q_rot = rotate(np.asarray(q_new, dtype=np.float64), pos, self.theta)
        for i, j in enumerate(toks):
            self.k[r.slot(j)] = k_rot[i]
            self.v[r.slot(j)] = np.asarray(v_new[i], dtype=np.float64)
        n_q, hq, d = q_rot.shape
        group = hq // self.k.shape[1]
        o = np.zeros((n_q, hq, d))
        lse = np.zeros((n_q, hq))
        for i, t in enumerate(toks):
            keys = [j for j in r.retained() if j <= t]
            slots = [r.slot(j) for j in keys]
            for h in range(hq):
                s = (self.k[slots, h // group, :] @ q_rot[i, h]) * scale
                m = s.max()
                e = np.exp(s - m)
                o[i, h] = e @ self.v[slots, h // group, :] / e.sum()
                lse[i, h] = m + math.log(e.sum())
        return o, lse


__all__ = ["StoredKeyCache", "SCHEME_OFFSET_ONLY", "SCHEME_EXACT_REBASE"]
