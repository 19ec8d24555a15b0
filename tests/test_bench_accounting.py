"""bench.py's host-side accounting without a GPU: kernels per forward, the live count of a capacity
point, and the algorithmic work the roofline divides by."""

import types

import numpy as np
import pytest

import synth

bench = pytest.importorskip("bench")


@pytest.mark.parametrize("name,M,n,launches", [
    ("decode", 32, 32, 5),          # single-CTA alignment, small-batch GEMMs
    ("mid", 8192, 8192, 7),         # counting + placement alignment, separate SwiGLU kernel
    ("glm_slice", 4096, 4096, 7),
    ("padded", 4096, 4096, 6),      # block-scaled GEMMs keep SwiGLU in FC1's epilogue
    ("padded", 512, 16, 5),         # capacity 4096 pairs: one alignment CTA, UE8M0 tiles
    ("padded_fp32", 512, 16, 6),    # FP32 tiles at the same capacity: separate SwiGLU kernel
])
def test_launches_per_forward(lib, name, M, n, launches):
    case = types.SimpleNamespace(shape=synth.SHAPES[name], M_cap=M, n=n)   # no weights needed
    assert bench.launches_per_forward(case) == launches


def test_capacity_points_default_to_their_live_count():
    assert dict(synth.SWEEPS["padded"])[512] == 16
    assert dict(synth.SWEEPS["padded_fp32"])[512] == 16
    assert bench.workload_name(synth.SHAPES["padded"], 512, 16).endswith("capacity 512, 16 live")
    assert bench.workload_name(synth.SHAPES["decode"], 32, 32).endswith("M=32")


def test_layer_work_counts_live_pairs_and_occupied_experts():
    case = synth.make_case("decode", 32, 5)
    sh = case.shape
    w = bench.layer_work(case)
    ids = case.topk_ids[:5].ravel()
    assert w["pairs"] == ids.size == 5 * sh.topk
    assert w["occupied_experts"] == np.unique(ids).size
    assert w["flops"] == 6.0 * w["pairs"] * sh.H * sh.I
    assert w["fc1_flops"] == 4.0 * w["pairs"] * sh.H * sh.I
    per_expert = 3 * sh.H * sh.I + 4 * ((2 * sh.I // 128) * (sh.H // 128) + (sh.H // 128) * (sh.I // 128))
    assert w["layer_bytes"] == w["occupied_experts"] * per_expert + 4 * 5 * sh.H + 8 * 5 * sh.topk


def test_default_headline_is_the_largest_layer_and_sweep_keeps_decode():
    shape = synth.SHAPES[bench.WORKLOAD]
    assert (shape.E, shape.H, shape.I, shape.topk) == (32, 7168, 2048, 8)
    assert shape.weight_fmt == shape.act_fmt == synth.SCALE_UE8M0
    pts = set(bench.SWEEP_POINTS)
    assert {("decode", 1, 1), ("decode", 4, 4), ("decode", 32, 32), ("padded", 512, 16),
            ("padded_fp32", 4096, 4096)} <= pts
    cfg = bench.bench_config(shape, 4096, 4096, 1)
    assert cfg["workload"] == "padded MoE layer E=32 H=7168 I=2048 top-8 M=4096"


def test_reference_arm_reports_the_same_config():
    args = types.SimpleNamespace(workload="tiny", M=16, n=16, steps=1, warmup=1, gpus=1)
    line = bench.reference_arm(args)
    assert line["impl"] == "reference"
    assert line["config"] == bench.bench_config(synth.SHAPES["tiny"], 16, 16, 1)
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # a step is one sampled token: its wall time, not the layer time it scales to
    assert line["ms_per_step"] * 1e3 * 16 == pytest.approx(line["value"])
