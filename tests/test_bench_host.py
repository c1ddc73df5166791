"""Host-side pieces of bench.py that need no GPU: the clock sampler (against
a fake nvidia-smi) and the reference arm's JSON line (the fp64 oracle on a
small workload)."""
import json
import os
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

FAKE = r'''#!{python}
import datetime, sys, time
args = sys.argv[1:]
sm, state = {sm}, "{state}"
row = [str(sm), "2070", "1000.5", "0x0", "Not Active", "Not Active", "Not Active", state]
if "-lms" in args:
    period = int(args[args.index("-lms") + 1]) / 1000.0
    try:
        while True:
            ts = datetime.datetime.now().strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
            sys.stdout.write(", ".join([ts] + row) + "\n")
            {flush}
            time.sleep(period)
    except KeyboardInterrupt:
        sys.exit(0)
print(", ".join(row))
'''


def _fake(tmp_path, sm=2070, state="Not Active", flush=True):
    p = tmp_path / "nvidia-smi"
    p.write_text(FAKE.format(python=sys.executable, sm=sm, state=state,
                             flush="sys.stdout.flush()" if flush else "pass"))
    p.chmod(0o755)
    return str(p)


def _region(sampler, seconds):
    with sampler:
        time.sleep(seconds)
    return sampler.summary()


def test_clock_sampler_takes_samples_inside_the_region(tmp_path):
    s = bench.ClockSampler(0, exe=_fake(tmp_path))
    c = _region(s, 0.3)
    # a sample every 20 ms over 0.3 s (the fake's own startup aside)
    assert c is not None and c["samples"] >= 6
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0 and c["reasons"] == []
    # every kept sample but the last lies inside the region
    ts = sorted(t for t, _ in s.lines)
    assert sum(1 for t in ts if s.t0 <= t <= s.t1) == c["samples"] - 1


def test_clock_sampler_reports_throttle_reasons(tmp_path):
    c = _region(bench.ClockSampler(0, exe=_fake(tmp_path, sm=1545, state="Active")), 0.2)
    assert c["sm_mhz"] == 1545.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]


def test_clock_sampler_with_block_buffered_output(tmp_path):
    # nothing arrives until the loop exits on SIGINT; the timestamps still
    # place the samples inside the region
    c = _region(bench.ClockSampler(0, exe=_fake(tmp_path, flush=False)), 0.3)
    assert c is not None and c["samples"] >= 6


def test_clock_sampler_without_nvidia_smi(tmp_path):
    s = bench.ClockSampler(0, exe=str(tmp_path / "missing"))
    assert _region(s, 0.01) is None


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_swiglu", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["value"] > 0
    assert d["config"]["workload"] == "tiny_swiglu"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


@pytest.mark.parametrize("world", [2])
def test_reference_arm_runs_on_rank_zero_only(world):
    env = dict(os.environ, RANK="1", WORLD_SIZE=str(world), LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_swiglu", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


# Per-config work of one step (GEMM flops = 2 x multiply-adds), as the scope
# table states them: fwd, bwd (incl. any recompute GEMM), and the model
# flops of fwd + bwd without the recompute.
STATED_TFLOP = {
    "tiny_swiglu": (17.3e-6, 34.6e-6, 51.9e-6),
    "llama7b_swiglu": (0.554, 1.108, 1.662),
    "falcon_h1_swiglu": (0.490, 0.979, 1.469),
    "nanogpt_relu_sq": (0.464, 1.160, 1.392),
    "llama3_8b_swiglu": (2.886, 7.697, 8.659),
}


@pytest.mark.parametrize("name", sorted(STATED_TFLOP))
def test_step_flops_match_the_stated_work(name):
    from activated_mlp_gemms_gb300.workloads import WORKLOADS
    w = WORKLOADS[name]
    fwd, bwd, model = STATED_TFLOP[name]
    got_fwd = bench.flops_of(w, "fwd") / 1e12
    got_bwd = bench.flops_of(w, bench.mode_of(w)) / 1e12
    got_model = (bench.flops_of(w, "fwd") + bench.flops_of(w, "bwd")) / 1e12
    for got, want in ((got_fwd, fwd), (got_bwd, bwd), (got_model, model)):
        assert abs(got - want) <= 0.0011 * want, (name, got, want)


@pytest.mark.parametrize("name", sorted(STATED_TFLOP))
def test_kernel_flops_add_up_to_the_step(name):
    # the kernels one step launches, each once (the recompute backward runs
    # the gated gate/up kernel a second time; the non-gated one fuses it)
    from activated_mlp_gemms_gb300.workloads import WORKLOADS
    w = WORKLOADS[name]
    k = bench.kernel_flops(w)
    step = bench.flops_of(w, "fwd") + bench.flops_of(w, bench.mode_of(w))
    # the gated forward runs as one fused launch or as two
    forwards = [["gate_up_act", "down_proj"]] + ([["fwd_fused"]] if w.gated else [])
    for fwd in forwards:
        launched = fwd + ["dx", "wgrad"]
        if w.recompute and not w.gated:
            launched.append("dact_recompute")
        else:
            launched.append("dgated")
            if w.recompute:
                launched.append("gate_up_act")
        assert sum(k[n] for n in launched) == pytest.approx(step, rel=1e-12), launched


def test_device_code_hash_ignores_comments_only(tmp_path):
    d = tmp_path / "csrc"
    d.mkdir()
    (d / "k.cu").write_text("int f(int x) {  // doubles\n  return 2 * x; /* plain */\n}\n")
    (d / "mlp_api.cu").write_text("host code\n")
    h0 = bench.csrc_hash(str(d))
    (d / "k.cu").write_text("// a header\nint f(int x) {\n    return 2 * x;\n}\n")
    (d / "mlp_api.cu").write_text("other host code\n")
    assert bench.csrc_hash(str(d)) == h0
    (d / "k.cu").write_text("int f(int x) { return 3 * x; }\n")
    assert bench.csrc_hash(str(d)) != h0
