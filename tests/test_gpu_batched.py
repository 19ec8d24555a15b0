"""GPU parity of the batched-expert layout (per-expert rows with masked counts) against the
oracle's batched_forward: both GEMM schedules, empty, partial and full experts, clamped counts,
and rows past each count left untouched."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from moe_testutil import assert_layer_close, bf16_tensor_to_f32

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def _run(shape, max_m, counts, seed, weights=None):
    import torch
    import block_fp8_mixture_gb300 as moe
    w = weights or synth.make_weights(shape)
    rng = np.random.Generator(np.random.PCG64(seed))
    xb = rng.standard_normal((shape.E, max_m, shape.H), dtype=np.float32)
    bits, vals = synth._to_bf16(xb)
    dev = lambda a: torch.from_numpy(a).cuda()
    x = dev(bits.view(np.int16)).view(torch.bfloat16)
    out = torch.empty_like(x)
    out.view(torch.int16).fill_(-1)
    ws = moe.alloc_batched_workspace(shape.E, max_m, shape.H, shape.I, shape.act_fmt)
    ws.fill_(0xFF)
    d_counts = dev(np.asarray(counts, np.int32))
    moe.batched_forward(x, d_counts, dev(w.w13), dev(w.s13), dev(w.w2), dev(w.s2), out, ws,
                        weight_fmt=shape.weight_fmt, act_fmt=shape.act_fmt,
                        clamp_mode=shape.clamp_mode, clamp_limit=shape.limit,
                        numerics=shape.numerics)
    torch.cuda.synchronize()
    assert moe.last_device_status(ws) == 0
    ref, live = oracle.batched_forward(vals, counts, w.w13, w.s13, w.w2, w.s2,
                                       act_fmt=shape.act_fmt, weight_fmt=shape.weight_fmt,
                                       clamp_mode=shape.clamp_mode, limit=shape.limit,
                                       numerics=shape.numerics)
    got = bf16_tensor_to_f32(out)
    raw = out.view(torch.int16).cpu().numpy()
    assert np.all(raw[~live] == -1), "rows past an expert's count were written"
    if live.any():
        assert_layer_close(got[live], ref[live], "batched")
    return got, ref, live


SMALL = synth.small_shape("batched_small", E=8, H=512, I=256, topk=1)


@pytest.mark.parametrize("max_m,counts", [
    (128, [0, 128, 3, 1, 50, 128, 33, 97]),          # small-batch schedule (swap-AB chunks)
    (256, [256, 0, 0, 255, 32, 31, 1, 129]),
    (512, [0, 512, 130, 1, 256, 300, 7, 511]),       # 128-row tile schedule
    (384, [-5, 1000, 128, 129, 0, 383, 64, 2]),      # counts clamped to [0, max_m]
])
def test_batched_layer(lib, max_m, counts):
    _run(SMALL, max_m, counts, seed=100 + max_m)


def test_batched_all_empty(lib):
    _run(SMALL, 128, [0] * SMALL.E, seed=7)


@pytest.mark.parametrize("max_m", [128, 512])
def test_batched_ue8m0_clamp_reciprocal(lib, max_m):
    sh = synth.small_shape("batched_ue8m0", E=4, H=384, I=384, topk=1,
                           act_fmt=synth.SCALE_UE8M0, weight_fmt=synth.SCALE_UE8M0,
                           clamp_mode=synth.CLAMP_BEFORE_SILU, limit=0.05, numerics=1)
    counts = [max_m, max_m // 2 + 3, 0, 17]
    _run(sh, max_m, counts, seed=3 + max_m)


def test_batched_matches_routed_layer(lib):
    """The same rows through the routed forward with one expert per token and weight 1 give the
    same BF16 outputs up to the accumulation order of the two GEMM schedules."""
    import torch
    import block_fp8_mixture_gb300 as moe
    from moe_testutil import run_forward
    max_m, counts = 128, [5, 0, 128, 40, 1, 77, 2, 64]
    got, _, live = _run(SMALL, max_m, counts, seed=55)
    rng = np.random.Generator(np.random.PCG64(55))
    xb = rng.standard_normal((SMALL.E, max_m, SMALL.H), dtype=np.float32)
    bits, vals = synth._to_bf16(xb)
    rows_bits, rows = bits[live], vals[live]
    ids = np.repeat(np.arange(SMALL.E), counts)[:, None].astype(np.int32)
    case = synth.LayerCase(SMALL, rows.shape[0], rows.shape[0], rows_bits, rows, ids,
                           np.ones(ids.shape, np.float32), synth.make_weights(SMALL))
    out, _, _ = run_forward(case)
    torch.cuda.synchronize()
    routed = bf16_tensor_to_f32(out)
    assert_layer_close(got[live], routed, "batched vs routed")
    assert np.mean(routed == got[live]) > 0.99
