"""ctypes binding of librkv.so (include/rkv.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
computation of its own: tensors become raw pointers, Python sequences become
C arrays, a non-zero status becomes an RkvError.  There is no fallback: if
the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "librkv.so")

RKV_OK = 0
RKV_ERR_INVALID_ARG = -1
RKV_ERR_CONFIG = -2
RKV_ERR_CUDA = -3
RKV_ERR_CAPACITY = -4
RKV_ERR_TIMEOUT = -5
RKV_ERR_STATE = -6
RKV_ERR_DEVICE_BOUNDS = -7
RKV_ERR_DEVICE_RANGE = -8
RKV_KV_F16 = 0
RKV_KV_E4M3 = 1
RKV_SCHEME_OFFSET_ONLY = 0
RKV_SCHEME_EXACT_REBASE = 1
RKV_SCHEME_EXACT_ON_READ = 2
RKV_MAX_STREAMS = 1024
RKV_STATE_FIELDS = 8
STATE_FIELDS = ("n", "len", "evicted", "kv_pos_offset", "rope_base", "head_slot", "W", "P0")


class RkvError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"rkv error {code}: {msg}")
        self.code = code


class rkv_config(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("n_streams", C.c_int32), ("n_q_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("q_per_step", C.c_int32),
                ("page_size", C.c_int32), ("scheme", C.c_int32), ("rebase_interval", C.c_int32),
                ("window_slack", C.c_int32), ("kv_format", C.c_int32), ("reserved", C.c_int32),
                ("rope_theta", C.c_double), ("softmax_scale", C.c_double)]


class rkv_clock(C.Structure):
    _fields_ = [("clock_ms", C.c_int32), ("window", C.c_int32), ("num_delay_tokens", C.c_int32),
                ("left_pad_tokens", C.c_int32), ("samples_per_token", C.c_int32),
                ("post_trained", C.c_int32), ("decisions_per_s", C.c_double)]


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run `python rolling_kv_sliding_rkv_b300/build.py`")
_lib = C.CDLL(LIB_PATH)

_vp, _i32, _i64, _u64, _u32, _f32, _f64, _sz = (C.c_void_p, C.c_int32, C.c_int64, C.c_uint64, C.c_uint32,
                                                 C.c_float, C.c_double, C.c_size_t)
_SIGS = {
    "rkv_clock_resolve": [_i32, _i32, C.POINTER(rkv_clock)],
    "rkv_required_bytes": [C.POINTER(rkv_config), C.POINTER(_i32), C.POINTER(_sz), C.POINTER(_sz)],
    "rkv_create": [C.POINTER(rkv_config), C.POINTER(_i32), C.POINTER(_i64), _vp, _sz, _vp, _sz, _vp,
                   C.POINTER(_vp)],
    "rkv_begin_step": [_vp, C.POINTER(_i32), _i32, _vp],
    "rkv_append_rope": [_vp, _i32, _vp, _vp, _vp],
    "rkv_rebase": [_vp, _i32, _vp],
    "rkv_decode_attn": [_vp, _i32, _vp, _vp, _vp, _vp],
    "rkv_decode_attn_static": [_vp, _i32, _vp, _vp, _vp, _vp],
    "rkv_append_decode_attn": [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp],
    "rkv_decode_attn_layers": [_vp, _i32, _i32, _vp, _vp, _vp, _vp],
    "rkv_step": [_vp, C.POINTER(_i32), _i32, _vp, _vp, _vp, _vp, _vp, _vp],
    "rkv_get_stream_state": [_vp, _i32, C.POINTER(_i64), _vp],
    "rkv_check_stream_state": [C.POINTER(rkv_config), C.POINTER(_i64)],
    "rkv_reset_stream": [_vp, _i32, _i64, _vp],
    "rkv_reset_streams": [_vp, _vp, _vp, _i32, _vp],
    "rkv_stream_snapshot_bytes": [_vp, _i32, C.POINTER(_sz)],
    "rkv_save_stream": [_vp, _i32, _vp, _sz, _vp],
    "rkv_load_stream": [_vp, _i32, _vp, _sz, _vp],
    "rkv_sync_status": [_vp, _vp],
    "rkv_set_wait_test": [_vp, _i32, _u64],
    "rkv_destroy": [_vp],
    "rkv_rope_cossin": [_vp, _i32, _i32, _f64, _vp, _vp],
    "rkv_gen_tokens": [_u64, _u32, _i32, _i32, _i64, _i32, _i32, _f32, _vp, _vp],
    "rkv_gen_step_inputs": [_vp, _u64, _i32, _f32, _vp, _vp, _vp, _vp],
    "rkv_gen_next_inputs": [_vp, _u64, C.POINTER(_i32), _i32, _f32, _vp, _vp, _vp, _vp],
}
for _name, _args in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = C.c_int
_lib.rkv_last_error.argtypes = [_vp]
_lib.rkv_last_error.restype = C.c_char_p


def lib() -> C.CDLL:
    return _lib


def _ptr(x) -> int | None:
    """Device or host address of a tensor, or an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def rkv_last_error(h=None) -> str:
    m = _lib.rkv_last_error(h)
    return m.decode() if m else ""


def _check(rc: int, h=None) -> None:
    if rc != RKV_OK:
        raise RkvError(rc, rkv_last_error(h))


def make_config(**kw) -> rkv_config:
    c = rkv_config()
    c.page_size = 64
    c.rebase_interval = 1
    c.rope_theta = 1e6
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _i32_array(xs):
    xs = [int(x) for x in xs]
    return (_i32 * len(xs))(*xs), len(xs)


def rkv_clock_resolve(frame_len: int, target_delay_ms: int) -> dict:
    out = rkv_clock()
    _check(_lib.rkv_clock_resolve(frame_len, target_delay_ms, C.byref(out)))
    return {f: getattr(out, f) for f, _ in rkv_clock._fields_}


def rkv_required_bytes(cfg: rkv_config, windows) -> tuple:
    w, n = _i32_array(windows)
    if n != cfg.n_streams:
        raise ValueError("one window per stream expected")
    pool, state = _sz(), _sz()
    _check(_lib.rkv_required_bytes(C.byref(cfg), w, C.byref(pool), C.byref(state)))
    return pool.value, state.value


def rkv_create(cfg: rkv_config, windows, start_offsets, pool, pool_bytes: int, state, state_bytes: int,
               stream=None) -> int:
    w, n = _i32_array(windows)
    offs = [int(x) for x in start_offsets]
    if n != cfg.n_streams or len(offs) != cfg.n_streams:
        raise ValueError("one window and one start offset per stream expected")
    p0 = (_i64 * n)(*offs)
    h = _vp()
    _check(_lib.rkv_create(C.byref(cfg), w, p0, _ptr(pool), pool_bytes, _ptr(state), state_bytes,
                           _stream(stream), C.byref(h)))
    return h.value


def rkv_begin_step(h: int, active_ids, stream=None) -> None:
    ids, n = _i32_array(active_ids)
    _check(_lib.rkv_begin_step(h, ids, n, _stream(stream)), h)


def rkv_append_rope(h: int, layer: int, k, v, stream=None) -> None:
    _check(_lib.rkv_append_rope(h, layer, _ptr(k), _ptr(v), _stream(stream)), h)


def rkv_rebase(h: int, layer: int, stream=None) -> None:
    _check(_lib.rkv_rebase(h, layer, _stream(stream)), h)


def rkv_decode_attn(h: int, layer: int, q, out, lse=None, stream=None) -> None:
    _check(_lib.rkv_decode_attn(h, layer, _ptr(q), _ptr(out), _ptr(lse), _stream(stream)), h)


def rkv_append_decode_attn(h: int, layer: int, q, k, v, out, lse=None, stream=None) -> None:
    _check(_lib.rkv_append_decode_attn(h, layer, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _stream(stream)), h)


def rkv_decode_attn_static(h: int, layer: int, q, out, lse=None, stream=None) -> None:
    _check(_lib.rkv_decode_attn_static(h, layer, _ptr(q), _ptr(out), _ptr(lse), _stream(stream)), h)


def rkv_decode_attn_layers(h: int, layer0: int, n_layers: int, q, out, lse=None, stream=None) -> None:
    _check(_lib.rkv_decode_attn_layers(h, layer0, n_layers, _ptr(q), _ptr(out), _ptr(lse), _stream(stream)), h)


def rkv_step(h: int, active_ids, q, k, v, out, lse=None, stream=None) -> None:
    ids, n = _i32_array(active_ids)
    _check(_lib.rkv_step(h, ids, n, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _stream(stream)), h)


def rkv_reset_stream(h: int, stream_id: int, start_offset: int, stream=None) -> None:
    _check(_lib.rkv_reset_stream(h, stream_id, start_offset, _stream(stream)), h)


def rkv_reset_streams(h: int, ids_dev, p0_dev, n: int, stream=None) -> None:
    _check(_lib.rkv_reset_streams(h, _ptr(ids_dev), _ptr(p0_dev), n, _stream(stream)), h)


def rkv_stream_snapshot_bytes(h: int, stream_id: int) -> int:
    n = _sz()
    _check(_lib.rkv_stream_snapshot_bytes(h, stream_id, C.byref(n)))
    return n.value


def rkv_save_stream(h: int, stream_id: int, dst, nbytes: int, stream=None) -> None:
    _check(_lib.rkv_save_stream(h, stream_id, _ptr(dst), nbytes, _stream(stream)), h)


def rkv_load_stream(h: int, stream_id: int, src, nbytes: int, stream=None) -> None:
    _check(_lib.rkv_load_stream(h, stream_id, _ptr(src), nbytes, _stream(stream)), h)


def rkv_get_stream_state(h: int, stream_id: int, stream=None) -> list:
    out = (_i64 * RKV_STATE_FIELDS)()
    _check(_lib.rkv_get_stream_state(h, stream_id, out, _stream(stream)), h)
    return list(out)


def rkv_check_stream_state(cfg: rkv_config, state) -> None:
    vals = [int(x) for x in state]
    if len(vals) != RKV_STATE_FIELDS:
        raise ValueError(f"{RKV_STATE_FIELDS} state fields expected")
    _check(_lib.rkv_check_stream_state(C.byref(cfg), (_i64 * RKV_STATE_FIELDS)(*vals)))


def rkv_sync_status(h: int, stream=None) -> None:
    _check(_lib.rkv_sync_status(h, _stream(stream)), h)


def rkv_set_wait_test(h: int, withhold_stage: int, wait_ns: int) -> None:
    _check(_lib.rkv_set_wait_test(h, withhold_stage, wait_ns), h)


def rkv_destroy(h: int) -> None:
    _check(_lib.rkv_destroy(h))


def rkv_rope_cossin(pos, n: int, head_dim: int, theta: float, cs, stream=None) -> None:
    _check(_lib.rkv_rope_cossin(_ptr(pos), n, head_dim, theta, _ptr(cs), _stream(stream)))


def rkv_gen_tokens(seed: int, tag: int, stream_id: int, layer: int, token0: int, n_tokens: int, width: int,
                   scale: float, out, stream=None) -> None:
    _check(_lib.rkv_gen_tokens(seed, tag, stream_id, layer, token0, n_tokens, width, scale, _ptr(out),
                               _stream(stream)))


def rkv_gen_step_inputs(h: int, seed: int, layer: int, scale: float, q, k, v, stream=None) -> None:
    _check(_lib.rkv_gen_step_inputs(h, seed, layer, scale, _ptr(q), _ptr(k), _ptr(v), _stream(stream)), h)


def rkv_gen_next_inputs(h: int, seed: int, active_ids, scale: float, q, k, v, stream=None) -> None:
    ids, n = _i32_array(active_ids)
    _check(_lib.rkv_gen_next_inputs(h, seed, ids, n, scale, _ptr(q), _ptr(k), _ptr(v), _stream(stream)), h)
