"""Rolling KV cache for unbounded streaming attention on one B300.

The compute runs in librkv.so (hand-written CUDA for sm_103a, C ABI in
include/rkv.h).  This package is its Python binding: the functions in
``_abi`` carry the C names, and ``RollingKV`` owns the two device buffers a
handle needs (allocated with PyTorch) and forwards calls.  Nothing here
computes; without the built library the import fails.
"""
from __future__ import annotations

from . import _abi
from ._abi import (  # noqa: F401
    RKV_ERR_CAPACITY, RKV_ERR_CONFIG, RKV_ERR_CUDA, RKV_ERR_DEVICE_BOUNDS, RKV_ERR_DEVICE_RANGE, RKV_ERR_INVALID_ARG,
    RKV_ERR_STATE, RKV_ERR_TIMEOUT, RKV_KV_E4M3, RKV_KV_F16, RKV_OK, RKV_SCHEME_EXACT_ON_READ, RKV_SCHEME_EXACT_REBASE, RKV_SCHEME_OFFSET_ONLY,
    STATE_FIELDS, RkvError, make_config, rkv_append_decode_attn, rkv_append_rope, rkv_begin_step, rkv_check_stream_state, rkv_clock_resolve,
    rkv_create, rkv_decode_attn, rkv_decode_attn_layers, rkv_decode_attn_static, rkv_destroy, rkv_gen_next_inputs, rkv_gen_step_inputs, rkv_gen_tokens,
    rkv_get_stream_state, rkv_last_error, rkv_load_stream, rkv_rebase, rkv_required_bytes, rkv_reset_stream, rkv_reset_streams,
    rkv_rope_cossin, rkv_save_stream, rkv_set_wait_test, rkv_stream_snapshot_bytes,
    rkv_step, rkv_sync_status,
)

__all__ = [n for n in dir(_abi) if n.startswith("rkv_")] + ["RollingKV", "make_config", "RkvError"]


class RollingKV:
    """A handle plus the caller-owned pool and state buffers it runs on."""

    def __init__(self, windows, start_offsets=None, device="cuda", stream=None, **config):
        import torch

        self.cfg = make_config(**config)
        self.windows = [int(w) for w in windows]
        self.start_offsets = [int(p) for p in (start_offsets if start_offsets is not None
                                               else [0] * len(self.windows))]
        self.pool_bytes, self.state_bytes = rkv_required_bytes(self.cfg, self.windows)
        self.pool = torch.empty(max(self.pool_bytes, 1), dtype=torch.uint8, device=device)
        self.state = torch.empty(max(self.state_bytes, 1), dtype=torch.uint8, device=device)
        self.handle = rkv_create(self.cfg, self.windows, self.start_offsets, self.pool, self.pool_bytes,
                                 self.state, self.state_bytes, stream)

    # per-step calls, in the order the ABI requires
    def begin_step(self, active_ids, stream=None):
        rkv_begin_step(self.handle, active_ids, stream)

    def append_rope(self, layer, k, v, stream=None):
        rkv_append_rope(self.handle, layer, k, v, stream)

    def rebase(self, layer, stream=None):
        rkv_rebase(self.handle, layer, stream)

    def decode_attn(self, layer, q, out, lse=None, stream=None):
        rkv_decode_attn(self.handle, layer, q, out, lse, stream)

    def append_decode_attn(self, layer, q, k, v, out, lse=None, stream=None):
        rkv_append_decode_attn(self.handle, layer, q, k, v, out, lse, stream)

    def decode_attn_layers(self, layer0, n_layers, q, out, lse=None, stream=None):
        rkv_decode_attn_layers(self.handle, layer0, n_layers, q, out, lse, stream)

    def step(self, active_ids, q, k, v, out, lse=None, stream=None):
        rkv_step(self.handle, active_ids, q, k, v, out, lse, stream)

    def gen_step_inputs(self, seed, layer, scale, q, k, v, stream=None):
        rkv_gen_step_inputs(self.handle, seed, layer, scale, q, k, v, stream)

    def gen_next_inputs(self, seed, active_ids, scale, q, k, v, stream=None):
        rkv_gen_next_inputs(self.handle, seed, active_ids, scale, q, k, v, stream)

    def reset_stream(self, stream_id, start_offset=0, stream=None):
        rkv_reset_stream(self.handle, stream_id, start_offset, stream)

    def reset_streams(self, ids_dev, p0_dev, stream=None):
        rkv_reset_streams(self.handle, ids_dev, p0_dev, ids_dev.numel(), stream)

    def save_stream(self, stream_id, stream=None):
        """The stream's snapshot as a uint8 tensor on the handle's device."""
        import torch
        n = rkv_stream_snapshot_bytes(self.handle, stream_id)
        buf = torch.empty(n, dtype=torch.uint8, device=self.pool.device)
        rkv_save_stream(self.handle, stream_id, buf, n, stream)
        return buf

    def load_stream(self, stream_id, snapshot, stream=None):
        rkv_load_stream(self.handle, stream_id, snapshot, snapshot.numel() * snapshot.element_size(), stream)

    def stream_state(self, stream_id, stream=None) -> dict:
        return dict(zip(STATE_FIELDS, rkv_get_stream_state(self.handle, stream_id, stream)))

    def sync_status(self, stream=None):
        rkv_sync_status(self.handle, stream)

    def close(self):
        if getattr(self, "handle", None):
            rkv_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
