"""Integer model of one stream's rolling window, and the compaction it replaces.

State fields, in the order the CUDA library reports them:
  n              tokens appended so far
  len            tokens in the window, min(n, W)
  evicted        tokens pushed out of the window, n - len
  kv_pos_offset  P0 + evicted: added to a token's physical index (its place
                 inside the window, 0 = oldest retained) to get its logical
                 RoPE position (voxtral.c rolling-KV article, §二
                 "RoPE 逻辑位置修正": logical_pos = kv_pos_offset + pos)
  rope_base      exact re-base scheme: the origin the stored keys are rotated
                 against (stored K of token j is R(j - rope_base) k_j); moved
                 to `evicted` on every roll (explainer, "Rolling KV Cache
                 三步拆解", 第 2 步), or once `rebase_interval` tokens have been
                 evicted since the last re-base.  0 in the offset-only scheme.
  head_slot      ring slot of the oldest retained token, evicted mod C
  W              window
  P0             logical position of token 0

Eviction: a step of Q tokens keeps the last W tokens (explainer 第 1 步;
voxtral.c article §二 keeps the last VOX_DEC_WINDOW positions, §三 compacts
when cache length + new length exceeds the window).  The ring stores token j
in slot j mod C, so eviction moves no data.

Capacity C >= W (default C = W, the plain sliding window above): the window
may grow to C tokens and is cut back to the last W only when a step would
exceed C, i.e. eviction in batches.  This is the reading of the explainer's
"oldest batch" (第 1 步: 最老的一批) and of voxtral.c's trigger (article §二:
compaction only once the position reaches kv_cache_max, down to the
window); the window length then varies in [W, C] once filled.
"""
from __future__ import annotations

SCHEME_OFFSET_ONLY = 0
SCHEME_EXACT_REBASE = 1

FIELDS = ("n", "len", "evicted", "kv_pos_offset", "rope_base", "head_slot", "W", "P0")


class StreamRing:
    def __init__(self, window: int, p0: int = 0, q_per_step: int = 1,
                 scheme: int = SCHEME_OFFSET_ONLY, rebase_interval: int = 1, capacity: int | None = None):
        capacity = window if capacity is None else capacity
        if window < 1 or q_per_step < 1 or q_per_step > window or rebase_interval < 1 or capacity < window:
            raise ValueError("bad ring parameters")
        self.W = int(window)
        self.C = int(capacity)
        self.P0 = int(p0)
        self.Q = int(q_per_step)
        self.scheme = scheme
        self.interval = int(rebase_interval)
        self.n = 0
        self.len = 0
        self.evicted = 0
        self.rope_base = 0
        self.last_delta = 0

    @property
    def kv_pos_offset(self) -> int:
        return self.P0 + self.evicted

    @property
    def head_slot(self) -> int:
        return self.evicted % self.C

    def step(self) -> None:
        """Append Q tokens: advance n, evict down to W once past the capacity, schedule a re-base."""
        self.n += self.Q
        if self.n - self.evicted > self.C:
            self.evicted = self.n - self.W
        self.len = self.n - self.evicted
        self.last_delta = 0
        if self.scheme == SCHEME_EXACT_REBASE and self.evicted - self.rope_base >= self.interval:
            self.last_delta = self.evicted - self.rope_base
            self.rope_base = self.evicted

    def slot(self, j: int) -> int:
        return j % self.C

    def physical(self, j: int) -> int:
        return j - self.evicted

    def logical(self, j: int) -> int:
        return self.physical(j) + self.kv_pos_offset

    def rope_position(self, j: int) -> int:
        """Position the stored key of token j (or the query of token j) is rotated to."""
        if self.scheme == SCHEME_EXACT_REBASE:
            return j - self.rope_base
        return self.logical(j)

    def retained(self) -> range:
        return range(self.evicted, self.n)

    def state(self) -> list:
        return [self.n, self.len, self.evicted, self.kv_pos_offset, self.rope_base,
                self.head_slot, self.W, self.P0]


class CompactingCache:
    """The voxtral.c formulation: a growable buffer compacted by memmove.

    Before appending `new_len` tokens, if length + new_len exceeds the
    compaction threshold (`compact_at`, voxtral's kv_cache_max; by default the
    window itself), the oldest entries are dropped so that exactly `window`
    remain after the append, the rest move to index 0 (memmove), and the
    dropped count is added to kv_pos_offset (voxtral.c article §二, §三).
    Kept only to pin the ring model: both must agree on which tokens are
    retained and on their logical positions.
    """

    def __init__(self, window: int, p0: int = 0, compact_at: int | None = None):
        self.window = window
        self.compact_at = window if compact_at is None else compact_at
        self.buf: list = []          # token ids, physical index = list index
        self.kv_pos_offset = p0

    def append(self, tokens: list) -> None:
        new_len = len(tokens)
        if len(self.buf) + new_len > self.compact_at:
            drop = len(self.buf) + new_len - self.window
            self.buf = self.buf[drop:]
            self.kv_pos_offset += drop
        self.buf.extend(tokens)

    def logical_positions(self) -> list:
        return [self.kv_pos_offset + pos for pos in range(len(self.buf))]
