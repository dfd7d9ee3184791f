"""The five synthetic workloads: shapes, windows, schemes, start offsets, schedules.

Each workload stands in for a deployment the pages describe (a Qwen2.5-3B
decoder with 16 query / 2 KV heads of dim 128 under a 30 s window; the
voxtral.c decoder window of 8192 positions; the causal audio tower's 750-frame
window with frame_len 4 new positions per step; a mixed-clock serving batch).
No dataset or trained weight is involved: q, k and v are the generator's
N(0, 1) draws, optionally scaled by fp32(1/sqrt(head_dim)).
"""
from __future__ import annotations

from dataclasses import dataclass, field
import math

import numpy as np

from .generator import TAG_CLOCK, TAG_FILL, TAG_P0, TAG_PHASE, uniform_int

SCHEME_OFFSET_ONLY = 0
SCHEME_EXACT_REBASE = 1


@dataclass
class Workload:
    name: str
    index: int
    n_layers: int
    n_streams: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    q_per_step: int
    steps: int
    scheme: int
    scale_inputs: bool
    rope_theta: float = 1.0e6
    p0_high: int = 0          # start offsets uniform in [0, p0_high); 0 -> all zero
    clocks_ms: tuple = (80,)  # clock per stream drawn uniformly from this tuple
    tick_ms: int = 0          # >0: mixed-clock schedule on a tick of this length
    ragged_fill: bool = False
    rebase_interval: int = 1
    window_slack: int = 0     # ring capacity beyond the window (eviction in batches); 0: every step
    kv_format: int = 0        # 0: fp16 keys / bf16 values; 1: the fp8 (e4m3) store
    extra: dict = field(default_factory=dict)

    @property
    def seed(self) -> int:
        return 20260101 + self.index

    @property
    def input_scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.head_dim))) if self.scale_inputs else 1.0

    def window_for_clock(self, clock_ms: int) -> int:
        # 30 s of clock steps, rounded up (160 ms gives 187.5 -> 188)
        return -(-30000 // clock_ms) if self.q_per_step == 1 else self.extra["window"]

    def stream_clocks(self) -> np.ndarray:
        if len(self.clocks_ms) == 1:
            return np.full(self.n_streams, self.clocks_ms[0], dtype=np.int64)
        pick = uniform_int(self.seed, TAG_CLOCK, np.arange(self.n_streams), len(self.clocks_ms))
        return np.asarray(self.clocks_ms, dtype=np.int64)[pick]

    def windows(self) -> np.ndarray:
        if "window" in self.extra:
            return np.full(self.n_streams, self.extra["window"], dtype=np.int32)
        return np.array([self.window_for_clock(int(c)) for c in self.stream_clocks()], dtype=np.int32)

    def start_offsets(self) -> np.ndarray:
        if self.p0_high <= 0:
            return np.zeros(self.n_streams, dtype=np.int64)
        return uniform_int(self.seed, TAG_P0, np.arange(self.n_streams), self.p0_high)

    def phases(self) -> np.ndarray:
        """Tick phase of each stream in [0, clock/tick)."""
        period = self.stream_clocks() // max(self.tick_ms, 1)
        raw = uniform_int(self.seed, TAG_PHASE, np.arange(self.n_streams), 1 << 30)
        return raw % np.maximum(period, 1)

    def initial_fill(self) -> np.ndarray:
        """Tokens each stream has appended before the measured ticks start."""
        if not self.ragged_fill:
            return np.zeros(self.n_streams, dtype=np.int64)
        w = self.windows().astype(np.int64)
        raw = uniform_int(self.seed, TAG_FILL, np.arange(self.n_streams), 1 << 30)
        return raw % (w + 1)

    def active_at_tick(self, tick: int) -> np.ndarray:
        """Stream ids that take a step at this tick (all streams when there is no tick)."""
        if self.tick_ms <= 0:
            return np.arange(self.n_streams, dtype=np.int32)
        period = self.stream_clocks() // self.tick_ms
        return np.nonzero((tick + self.phases()) % period == 0)[0].astype(np.int32)


WORKLOADS = {
    "tiny": Workload("tiny", 0, n_layers=1, n_streams=1, n_q_heads=16, n_kv_heads=2, head_dim=128,
                     q_per_step=1, steps=1000, scheme=SCHEME_EXACT_REBASE, scale_inputs=False),
    "qwen": Workload("qwen", 1, n_layers=36, n_streams=64, n_q_heads=16, n_kv_heads=2, head_dim=128,
                     q_per_step=1, steps=5000, scheme=SCHEME_EXACT_REBASE, scale_inputs=True,
                     p0_high=1_080_000),
    "voxtral": Workload("voxtral", 2, n_layers=26, n_streams=16, n_q_heads=32, n_kv_heads=8, head_dim=128,
                        q_per_step=1, steps=20000, scheme=SCHEME_OFFSET_ONLY, scale_inputs=False,
                        extra={"window": 8192}),
    "encoder": Workload("encoder", 3, n_layers=32, n_streams=32, n_q_heads=20, n_kv_heads=20, head_dim=64,
                        q_per_step=4, steps=2000, scheme=SCHEME_OFFSET_ONLY, scale_inputs=False,
                        extra={"window": 750}),
    "mixed": Workload("mixed", 4, n_layers=36, n_streams=256, n_q_heads=16, n_kv_heads=2, head_dim=128,
                      q_per_step=1, steps=10000, scheme=SCHEME_EXACT_REBASE, scale_inputs=True,
                      p0_high=2_000_000, clocks_ms=(80, 120, 160), tick_ms=40, ragged_fill=True),
}


def workload(name: str, **overrides) -> Workload:
    """A copy of a named workload with fields replaced (e.g. smaller step counts)."""
    import dataclasses
    return dataclasses.replace(WORKLOADS[name], **overrides)
