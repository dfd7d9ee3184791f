"""fp64 mirrors of the storage schemes (invariance checks only).

Offset-only (voxtral.c rolling-KV article, §二): RoPE is applied once, when a
key is written, at its logical position P0 + j; keys are never re-encoded.

Exact re-base (Audio8 ASR Infinite 无限长转写原理, "Rolling KV Cache 三步拆解",
第 2 步): on every roll all retained keys are rotated by R(-delta), delta the
number of positions evicted since the last re-base, so the stored positions
restart inside the window; the new query and key use window-relative
positions too.

The exact re-base applied on read (RingSlotKeyCache below) stores each key
once at its ring slot and rotates the query instead.

All are evaluated in fp64 against a stored-key cache and must equal
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


class RingSlotKeyCache:
    """One stream, one layer: keys stored rotated by their ring slot, the exact re-base on read.

    The stored key of token j is R(j mod C) k_j, written once; nothing is
    re-rotated when the window rolls.  Window positions then stay below C
    however long the stream runs, like the exact re-base's window-relative
    positions (explainer, "Rolling KV Cache 三步拆解", 第 2 步), and the
    re-base moves to the query: with E = floor(evicted / C), the retained
    tokens j in [evicted, n) have floor(j / C) = E in ring slots >= evicted
    mod C and E + 1 below, so query token t is rotated to t - C*E against the
    first group and to t - C*(E + 1) against the second.  Each score is then
    <R(t - j) q, k_j>, the definition's.
    """

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
        C = r.C
        toks = list(range(n_old, r.n))
        k_rot = rotate(np.asarray(k_new, dtype=np.float64), [r.slot(j) for j in toks], self.theta)
        for i, j in enumerate(toks):
            self.k[r.slot(j)] = k_rot[i]
            self.v[r.slot(j)] = np.asarray(v_new[i], dtype=np.float64)
        lap = r.evicted // C
        first_slot = r.evicted % C
        q_new = np.asarray(q_new, dtype=np.float64)
        n_q, hq, d = q_new.shape
        group = hq // self.k.shape[1]
        o = np.zeros((n_q, hq, d))
        lse = np.zeros((n_q, hq))
        for i, t in enumerate(toks):
            q_cur = rotate(q_new[i][None], [t - C * lap], self.theta)[0]         # slots >= first_slot
            q_next = rotate(q_new[i][None], [t - C * (lap + 1)], self.theta)[0]  # slots < first_slot
            keys = [j for j in r.retained() if j <= t]
            slots = [r.slot(j) for j in keys]
            for h in range(hq):
                s = np.array([self.k[sl, h // group, :] @ (q_cur[h] if sl >= first_slot else q_next[h])
                              for sl in slots]) * scale
                m = s.max()
                e = np.exp(s - m)
                o[i, h] = e @ self.v[slots, h // group, :] / e.sum()
                lse[i, h] = m + math.log(e.sum())
        return o, lse


def stored_key_attention_step(q_new, k_tok, v_tok, key_tokens, n: int, window: int, scale: float,
                              theta: float, stored_pos, quantize=None, first_key: int | None = None,
                              rotate_keys=None):
    """One step's outputs over keys as a store holds them, without the store's state.

    Key token j is stored rotated by R(s_j), s_j = stored_pos(j) (P0 + j offset-only; j mod C
    with the exact re-base applied on read), then passed through ``quantize`` (rows of d, e.g.
    ``oracle.fp8.quantize_rows``); values through the same.  Query token t meets key j rotated
    by R(t - j + s_j), so every score is <R(t - j) q, k_j> up to the store's rounding: with no
    quantisation this is the definition (``oracle.attention.attention_step``) exactly, and the
    fp8 store's error is modelled by quantising what the store would hold.  ``rotate_keys(k,
    positions)`` replaces the fp64 rotation of the stored keys (``oracle.fp8.rotate_fp32``: the
    store's own fp32 arithmetic, in which its quantisation decisions are taken).
    Arguments as ``attention_step`` (q_new [Q][Hq][d] raw, k_tok / v_tok [T][Hkv][d] raw)."""
    from .attention import visible_keys
    q_new = np.asarray(q_new, dtype=np.float64)
    k_tok = np.asarray(k_tok, dtype=np.float64)
    v_tok = np.asarray(v_tok, dtype=np.float64)
    key_tokens = [int(j) for j in key_tokens]
    row = {j: r for r, j in enumerate(key_tokens)}
    spos = [int(stored_pos(j)) for j in key_tokens]
    if rotate_keys is None:
        k_st = np.stack([rotate(k_tok[r][None], [spos[r]], theta)[0] for r in range(len(key_tokens))])
    else:
        k_st = rotate_keys(k_tok, spos)
    v_st = v_tok
    if quantize is not None:
        k_st, v_st = quantize(k_st), quantize(v_st)
    n_q, hq, d = q_new.shape
    group = hq // k_tok.shape[1]
    o = np.zeros((n_q, hq, d))
    lse = np.zeros((n_q, hq))
    for i, (lo, hi) in enumerate(visible_keys(n, n_q, window, first_key=first_key)):
        t = n + i
        rows = [row[j] for j in range(lo, hi + 1)]
        qpos = [t - key_tokens[r] + spos[r] for r in rows]
        q_rot = {p: rotate(q_new[i][None], [p], theta)[0] for p in set(qpos)}
        for h in range(hq):
            s = np.array([k_st[r, h // group] @ q_rot[p][h] for r, p in zip(rows, qpos)]) * scale
            m = s.max()
            e = np.exp(s - m)
            o[i, h] = e @ v_st[rows, h // group] / e.sum()
            lse[i, h] = m + math.log(e.sum())
    return o, lse


__all__ = ["StoredKeyCache", "RingSlotKeyCache", "stored_key_attention_step", "SCHEME_OFFSET_ONLY",
           "SCHEME_EXACT_REBASE"]
