"""bench.py's host logic on the CPU: the algorithmic work model (bytes and FLOPs per
launch, stated per token-head in the design notes), the kernel each workload is
dispatched to, and the JSON line of the reference arm (the fp64 oracle)."""
import json
import os
import subprocess
import sys

import pytest

import bench
from test_sequence_layers_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_linear_work_model_per_token_head():
    inp = synth.workload("linear_125m", T=64)
    B, H, T, d, b = inp.B, inp.H, inp.T, inp.d, inp.b
    # E = K W, the update and Q W (2 d^2 each) plus the masked scores over (b + 1)/2 pairs
    assert bench.flops_per_token_head(inp) == 6 * d * d + 2 * (b + 1) * d == 26752
    # q, k, v read and z written (bf16), W0 per head read, final W per chain written
    assert bench.bytes_per_launch(inp) == B * H * T * d * 2 * 4 + H * d * d * 4 + B * H * d * d * 4


def test_mlp_and_gate_work_models():
    inp = synth.workload("mlp_125m", T=32)
    d, m, b = inp.d, inp.m, inp.b
    assert bench.flops_per_token_head(inp) == 14 * d * m + 2 * (b + 1) * (d + m) == 240256
    g = synth.workload("linear_long_gate_x", T=128, B=1, H=4)
    dm = g.H * g.d
    assert g.gate_x.shape == (1, 128, dm) and g.gate_theta.shape == (4, dm) and g.eta is None
    plain = g.B * g.H * g.T * g.d * 2 * 4 + g.H * g.d * g.d * 4 + g.B * g.H * g.d * g.d * 4
    assert bench.bytes_per_launch(g) == plain + g.B * g.T * dm * 2 + g.H * dm * 2 + 2 * g.B * g.H * g.T * 4
    assert bench.flops_per_token_head(g) == 2 * dm + 6 * g.d * g.d + 2 * (g.b + 1) * g.d


def test_gate_alone_work_model_and_reference_sample():
    g = synth.workload("eta_gate_long", T=96, B=1, H=4)
    dm = g.H * g.d
    assert g.kind == "gate" and g.q.shape == (1, 96, dm) and g.k is None
    assert bench.bytes_per_launch(g) == 96 * dm * 2 + 4 * dm * 2 + 4 * 96 * 4
    assert bench.flops_per_token_head(g) == 2 * dm
    assert bench.kernel_name(g) == "ttt_eta_gate_kernel"
    v, cores, desc = bench.oracle_sample(g, 0.05)
    assert v > 0 and cores == 1 and "tokens" in desc


@pytest.mark.parametrize("name,kernel", [
    ("linear_125m", "ttt_linear_b16_kernel"), ("linear_125m_b1", "ttt_linear_b16_kernel"),
    ("vision_linear", "ttt_linear_fb_tc_kernel"), ("vision_linear_dot", "ttt_linear_fb_tc_kernel"),
    ("vision_linear_3ep", "ttt_linear_fb_kernel"), ("mlp_125m", "ttt_mlp_w8_kernel"),
    ("vision_mlp", "ttt_mlp_fb_tc_kernel"), ("vision_dwconv", "ttt_dwconv_kernel"),
    ("linear_tiny_f32", "ttt_linear_f32_kernel")])
def test_kernel_names_follow_the_dispatch(name, kernel):
    small = {"T": 196} if name.startswith("vision") else {"T": 64}
    small.update(B=1)
    assert bench.kernel_name(synth.workload(name, **small)) == kernel


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "linear_tiny_f32", "--steps", "2", "--warmup", "3", "--cpu-budget", "0.2"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["unit"] == "tokens/s" and j["higher_is_better"] is True
    assert j["value"] > 0 and j["steps"] == 2 and j["warmup"] == 3
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["value"] == j["value"]
    assert j["e2e"] == {"value": j["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert j["config"]["workload"] == "linear_tiny_f32"


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "linear_tiny_f32", "--warmup", "2"], capture_output=True, text=True, timeout=300,
                       cwd=ROOT)
    assert r.returncode != 0


def _peaks():
    return {"hbm_gbs": 6771.5, "bf16_tflops": 1922.2, "bf16_tflops_sustained": 1710.2, "source": "measured"}


def test_roofline_bound_is_the_attainable_minimum():
    """The bound is min(tensor peak, AI x bandwidth) per workload, not per kind: the
    full-batch MLP's required final weights (about 203 MB) make it HBM-bound, the
    causal MLP stays tensor-bound, TTT-Linear is HBM-bound."""
    pk = _peaks()
    vm = synth.workload("vision_mlp")
    flops = bench.flops_per_token_head(vm) * vm.token_heads
    nbytes = bench.bytes_per_launch(vm)
    assert 3.4e8 < nbytes < 3.7e8 and 6.5e10 < flops < 7.2e10
    r = bench.roofline_bound(flops, nbytes, 0.5, pk)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["frac"] - nbytes / 0.5e-3 / 1e9 / pk["hbm_gbs"]) < 1e-12
    assert abs(r["bound_ms"] - nbytes / (pk["hbm_gbs"] * 1e9) * 1e3) < 1e-12
    m = synth.workload("mlp_125m", T=2048)
    r = bench.roofline_bound(bench.flops_per_token_head(m) * m.token_heads, bench.bytes_per_launch(m), 0.4, pk)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    lin = synth.workload("linear_125m")
    r = bench.roofline_bound(bench.flops_per_token_head(lin) * lin.token_heads, bench.bytes_per_launch(lin),
                             0.0374, pk)
    assert r["bound"] == "hbm" and abs(r["frac"] - 0.4045) < 2e-3
