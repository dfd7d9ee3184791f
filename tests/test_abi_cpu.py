"""The C ABI without a GPU: exported symbols, host-side validation, clock arithmetic.

The clock logic of the library (C) is compared with the oracle's (Python);
the two are separate implementations of the same page-printed table.
"""
import os
import re
import subprocess

import pytest

import rolling_kv_sliding_rkv_b300 as rkv
from oracle import clock as oclock

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            with open(os.path.join(ROOT, "include", fn)) as f:
                names += re.findall(r"^RKV_API\s+[\w\s\*]+?\b(rkv_\w+)\s*\(", f.read(), re.M)
    return names


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert len(names) >= 15
    out = subprocess.run(["nm", "-D", "--defined-only", rkv._abi.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r" T (rkv_\w+)", out))
    assert set(names) <= exported, set(names) - exported
    for n in names:
        getattr(rkv._abi.lib(), n)


@pytest.mark.parametrize("frame_len", [3, 4, 5, 6, 8, 10])
def test_clock_resolve_matches_oracle(frame_len):
    for delay in list(range(-80, 1000, 40)) + [1, 50, 100]:
        try:
            ref = oclock.resolve(frame_len, delay)
        except oclock.ClockError:
            ref = None
        if ref is None:
            with pytest.raises(rkv.RkvError) as e:
                rkv.rkv_clock_resolve(frame_len, delay)
            assert e.value.code == rkv.RKV_ERR_CONFIG
        else:
            got = rkv.rkv_clock_resolve(frame_len, delay)
            assert got == {**ref, "post_trained": int(ref["post_trained"])}


def _cfg(**kw):
    base = dict(n_layers=36, n_streams=64, n_q_heads=16, n_kv_heads=2, head_dim=128, q_per_step=1, scheme=1)
    base.update(kw)
    return rkv.make_config(**base)


def test_required_bytes_closed_form():
    pool, state = rkv.rkv_required_bytes(_cfg(), [375] * 64)
    # 6 pages of 64 slots per stream, three regions (rotated K, V, pre-RoPE K), bf16
    assert pool == 36 * 64 * 6 * 2 * 64 * 128 * 2 * 3
    pool0, _ = rkv.rkv_required_bytes(_cfg(scheme=0), [375] * 64)
    assert pool0 * 3 == pool * 2
    pool_l1, _ = rkv.rkv_required_bytes(_cfg(n_layers=1), [375] * 64)
    assert pool_l1 * 36 == pool
    assert state < 8 << 20
    # fp8 store: one byte per key and value element, plus a (key, value) pair of float scales per row
    rows = 36 * 64 * 6 * 2 * 64
    for scheme in (0, 2):
        pool8, _ = rkv.rkv_required_bytes(_cfg(scheme=scheme, kv_format=rkv.RKV_KV_E4M3), [375] * 64)
        assert pool8 == rows * 128 * 2 + rows * 8


@pytest.mark.parametrize("bad", [dict(n_layers=0), dict(n_streams=0), dict(n_streams=2000),
                                 dict(n_q_heads=15), dict(head_dim=96), dict(q_per_step=0),
                                 dict(q_per_step=9), dict(n_q_heads=32, n_kv_heads=1), dict(page_size=48),
                                 dict(scheme=3), dict(rebase_interval=0), dict(rope_theta=1.0),
                                 dict(window_slack=-1), dict(softmax_scale=-1.0), dict(kv_format=2),
                                 dict(reserved=1), dict(kv_format=1, scheme=1),
                                 dict(kv_format=1, scheme=2, n_q_heads=16, n_kv_heads=1)])
def test_invalid_configs(bad):
    cfg = _cfg(**bad)
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_required_bytes(cfg, [375] * cfg.n_streams)
    assert e.value.code in (rkv.RKV_ERR_CONFIG, rkv.RKV_ERR_INVALID_ARG)


def test_invalid_windows():
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_required_bytes(_cfg(n_streams=2, q_per_step=4, n_q_heads=4, n_kv_heads=4), [375, 3])
    assert e.value.code == rkv.RKV_ERR_CONFIG
    with pytest.raises(rkv.RkvError):
        rkv.rkv_required_bytes(_cfg(n_streams=1), [(1 << 20) + 1])


def test_create_rejects_before_touching_the_device():
    cfg = _cfg(n_streams=2)
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_create(cfg, [8, 8], [0, 0], 0, 1 << 30, 0, 1 << 30, 0)
    assert e.value.code == rkv.RKV_ERR_INVALID_ARG
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_create(cfg, [8, 8], [0, 2 ** 52], 256, 1 << 30, 512, 1 << 30, 0)
    assert e.value.code == rkv.RKV_ERR_CONFIG
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_create(cfg, [8, 8], [0, 0], 256, 16, 512, 16, 0)
    assert e.value.code == rkv.RKV_ERR_CAPACITY
    assert "rkv_required_bytes" in rkv.rkv_last_error()


def test_null_handle_is_rejected():
    for call in (lambda: rkv.rkv_begin_step(None, [0], 0), lambda: rkv.rkv_rebase(None, 0, 0),
                 lambda: rkv.rkv_append_rope(None, 0, 16, 16, 0), lambda: rkv.rkv_sync_status(None, 0)):
        with pytest.raises(rkv.RkvError) as e:
            call()
        assert e.value.code == rkv.RKV_ERR_INVALID_ARG


@pytest.mark.parametrize("scheme,interval,q,slack", [(0, 1, 1, 0), (1, 1, 1, 0), (1, 5, 1, 0), (2, 3, 1, 0),
                                                     (0, 1, 4, 0), (1, 1, 1, 5), (2, 2, 4, 9), (0, 1, 4, 12)])
def test_stream_state_check(scheme, interval, q, slack):
    """States the integer ring model reaches are accepted; one field off by one is rejected."""
    from oracle.ring import StreamRing
    cfg = _cfg(n_streams=1, scheme=scheme, rebase_interval=interval, q_per_step=q,
               n_q_heads=4 if q > 1 else 16, n_kv_heads=4 if q > 1 else 2, window_slack=slack)
    w, p0 = 12, 2 ** 40 + 3
    ring = StreamRing(w, p0, q, 1 if scheme else 0, interval, capacity=w + slack)
    checked = 0
    for _ in range(60):
        st = ring.state()
        rkv.rkv_check_stream_state(cfg, st)
        for i in range(len(st)):
            for dlt in (-1, 1):
                bad = list(st)
                bad[i] += dlt
                if i == 4 and scheme and 0 <= bad[4] <= bad[2] and bad[2] - bad[4] < interval:
                    continue        # rope_base has slack of its own between re-bases
                if i == 6 and (st[0] <= w or slack):
                    continue        # W is fixed by the stream's pages (rkv_load_stream checks it); the
                    #                 state pins it only for a full plain sliding window
                with pytest.raises(rkv.RkvError) as e:
                    rkv.rkv_check_stream_state(cfg, bad)
                assert e.value.code == rkv.RKV_ERR_CONFIG
                checked += 1
        ring.step()
    assert checked > 600
    for bad in ([0, 0, 0, -1, 0, 0, w, -1], [0, 0, 0, 2 ** 52, 0, 0, w, 2 ** 52]):   # P0 outside [0, 2^52)
        with pytest.raises(rkv.RkvError):
            rkv.rkv_check_stream_state(cfg, bad)


@pytest.mark.parametrize("struct", ["rkv_config", "rkv_clock"])
def test_struct_layout_matches_the_header(tmp_path, struct):
    """The ctypes mirrors of the ABI's structs have the C structs' sizes and field offsets (gcc)."""
    import ctypes
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    cls = getattr(rkv._abi, struct)
    fields = [f for f, _ in cls._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "rkv.h"\nint main(void) {\n'
                   f'  printf("%zu\\n", sizeof({struct}));\n' +
                   "".join(f'  printf("%zu\\n", offsetof({struct}, {f}));\n' for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(cls)
    assert got[1:] == [getattr(cls, f).offset for f in fields]
