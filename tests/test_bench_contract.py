"""bench.py's JSON line: the contract keys and the roofline arithmetic (no GPU needed)."""
import json
import os
import subprocess
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402

REQUIRED = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks")


def _fake_measurement(wl, steps, ms_per_step, attn_us):
    lens = [int(w) for w in wl.windows()]
    per_layer = bench.algorithmic_attn_bytes(wl, lens)
    return {"value": wl.n_streams * steps / (ms_per_step * steps / 1000.0), "ms": ms_per_step * steps,
            "stream_steps": wl.n_streams * steps, "launches": 4 * steps, "attn_all_ms": attn_us / 1000.0,
            "attn_layer_ms": attn_us / 1000.0 / wl.n_layers * 3.0, "attn_bytes_layer": per_layer,
            "attn_bytes": per_layer * wl.n_layers, "attn_streams": wl.n_streams,
            "clocks": {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": []}}


def test_line_has_the_contract_keys_and_the_roofline_arithmetic():
    wl = synth.workload("qwen")
    args = types.SimpleNamespace(steps=100, warmup=20)
    m = _fake_measurement(wl, 100, 0.343, 148.0)
    e2e = {"value": 1.0, "unit": bench.UNIT, "h2d_bytes_per_step": 1, "d2h_bytes_per_step": 1}
    cpu = {"value": 1.0, "unit": bench.UNIT, "cores": 16, "kind": "oracle", "sample": "x"}
    line = bench.bench_line(wl, "exact re-base", args, 1, m, 6492.7, "measured", e2e=e2e, cpu=cpu)
    json.dumps(line)                                   # serialisable
    for key in REQUIRED:
        assert key in line, key
    assert line["metric"] == "stream-steps/sec (all layers) and decode-attn HBM GB/s as % of B300 peak"
    assert line["unit"] == "stream-steps/s" and line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["ms_per_step"] == pytest.approx(0.343)
    assert line["value"] == pytest.approx(64 / 0.343e-3)
    r = line["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6492.7
    # Qwen-shaped layer: 64 streams x 392256 algorithmic bytes; 36 layers per launch
    assert r["algorithmic_bytes_per_launch"] == 36 * 64 * 392256
    assert r["achieved"] == pytest.approx(36 * 64 * 392256 / 148e-6 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6492.7)
    assert set(line["e2e"]) >= {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert set(line["cpu_baseline"]) >= {"value", "unit", "cores", "kind", "sample"}


def test_algorithmic_bytes_of_one_stream_layer_step():
    # K + V of the window, q in, out, lse: 2*375*2*128*2 + 16*128*2*2 + 16*4
    wl = synth.workload("qwen")
    assert bench.algorithmic_attn_bytes(wl, [375]) == 392256


def test_rebase_share_of_the_step():
    # exact step 0.336 ms, offset-only step 0.154 ms: the re-base costs 182 us per step and moves
    # 64 streams x 36 layers x 2 kv heads x 374 retained keys x 128 x 2 bytes, read and written
    wl = synth.workload("qwen")
    args = types.SimpleNamespace(steps=100, warmup=20)
    m = _fake_measurement(wl, 100, 0.336, 145.0)
    m["plan"] = [list(range(wl.n_streams))]
    variants = {"offset-only": {"value": 1.0, "unit": bench.UNIT, "ms_per_step": 0.154}}
    line = bench.bench_line(wl, "exact re-base", args, 1, m, 6492.7, "measured", variants=variants)
    rb = line["rebase_in_step"]
    assert rb["algorithmic_bytes_per_step"] == 64 * 36 * 2 * 374 * 128 * 2 * 2
    assert rb["us_per_step"] == pytest.approx(182.0)
    assert rb["achieved_gbs"] == pytest.approx(64 * 36 * 2 * 374 * 128 * 4 / 182e-6 / 1e9)
    assert rb["frac"] == pytest.approx(rb["achieved_gbs"] / 6492.7)
    # no offset-only timing, or another scheme: no derived figure
    assert "rebase_in_step" not in bench.bench_line(wl, "exact re-base", args, 1, m, 6492.7, "measured",
                                                     variants={"x": {"ms_per_step": 0.1}})
    off = synth.workload("qwen", scheme=0)
    assert bench.rebase_in_step(off, m, variants, 100, 6492.7) is None


def test_code_digest_ignores_comments_and_layout_only(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    a.write_text("// header\nint f(int x) {\n  return x + 1;  /* one */\n}\n")
    b.write_text("/* another\n header */ int f(int x) { return x + 1; }  // trailing\n")
    c.write_text("int f(int x) { return x + 2; }\n")
    assert bench.code_digest(a) == bench.code_digest(b)
    assert bench.code_digest(a) != bench.code_digest(c)
    # a kernel source other than the profiled one reports no traffic
    wl = synth.workload("qwen", n_layers=8)
    assert bench.profiled_traffic(wl) is None


def test_traffic_table_is_for_the_current_attention_source():
    """The committed DRAM-traffic figures are those of the attention source as it stands: a change
    to its code must come with a new launch-list capture (else the bench line reports null)."""
    digest = bench.code_digest(os.path.join(ROOT, "rolling_kv_sliding_rkv_b300", "csrc", "rkv_attn.cu"))
    assert {t["attn_code_sha256_16"] for t in bench.TRAFFIC} == {digest}
    for name, scheme in (("mixed", 2), ("qwen", 2), ("qwen", 1), ("voxtral", 0), ("encoder", 0)):
        t = bench.profiled_traffic(synth.workload(name, scheme=scheme))
        lens = [int(w) for w in synth.workload(name).windows()]
        algo = bench.algorithmic_attn_bytes(synth.workload(name), lens) * synth.workload(name).n_layers
        if name != "mixed":   # every stream active: within a few % above the algorithmic bytes
            assert algo <= t <= 1.05 * algo, (name, t, algo)


def test_reference_arm_prints_one_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                          "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "stream-steps/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    # the same workload description as the GPU arm's line, and a per-step time of the steps it ran
    import argparse
    wl, _ = bench.bench_workload(argparse.Namespace(workload="tiny", scheme=None, layers=None))
    assert wl.scheme == 2        # an exact re-base workload is run with the re-base applied on read
    assert line["config"]["workload"] == bench.describe(wl, bench.SCHEME_NAMES[wl.scheme])
    assert 0 < line["ms_per_step"] * line["steps"] < 600e3


def test_rebase_share_with_the_re_base_applied_on_read_as_headline():
    # the headline runs the re-base on read; the materialised scheme's step comes from `schemes`
    wl = synth.workload("qwen", scheme=2)
    m = _fake_measurement(wl, 100, 0.160, 145.0)
    m["plan"] = [list(range(wl.n_streams))]
    variants = {"offset-only": {"ms_per_step": 0.154}, "exact re-base": {"ms_per_step": 0.336}}
    rb = bench.rebase_in_step(wl, m, variants, 100, 6492.7)
    assert rb["us_per_step"] == pytest.approx(182.0)
    assert bench.rebase_in_step(wl, m, {"offset-only": {"ms_per_step": 0.154}}, 100, 6492.7) is None
