"""The forward that needs no workspace and allocates nothing (moe_fp8_block_forward_static).

It exists for callers that cannot allocate device memory when they run the layer, so it keeps its
scratch in a fixed array inside the library.  Called through the C ABI, it runs the same kernels on
the same plan as moe_fp8_block_forward with a caller workspace, so its output must equal that
forward's bit for bit, on consecutive calls that reuse the array (whatever an earlier call left
there), and it must reject layers too large for the array before launching anything.  This file is
collected last on purpose.
"""

import ctypes

import numpy as np
import pytest

import synth
from moe_testutil import device_case

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import block_fp8_mixture_gb300 as moe  # noqa: E402


def _args(case, dev, out):
    sh = case.shape
    return moe.make_args(dev["x"], dev["ids"], dev["w"], dev["w13"], dev["s13"], dev["w2"], dev["s2"],
                         out, E=sh.E, H=sh.H, I=sh.I, topk=sh.topk, M_cap=case.M_cap,
                         d_num_tokens=dev["n"], weight_fmt=sh.weight_fmt, act_fmt=sh.act_fmt,
                         clamp_mode=sh.clamp_mode, clamp_limit=sh.limit)


def _poisoned_out(case):
    out = torch.empty((case.M_cap, case.shape.H), dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)
    return out


def _reference(case, dev):
    sh = case.shape
    ws = moe.alloc_workspace(case.M_cap, sh.E, sh.H, sh.I, sh.topk, sh.act_fmt)
    out = _poisoned_out(case)
    moe.forward(_args(case, dev, out), ws)
    torch.cuda.synchronize()
    assert moe.last_device_status(ws) == moe.MOE_OK
    return out.view(torch.int16).cpu().numpy()


def _static(case, dev):
    lib = moe.load_library(build_if_missing=True)
    out = _poisoned_out(case)
    args = _args(case, dev, out)
    status = lib.moe_fp8_block_forward_static(ctypes.byref(args),
                                              torch.cuda.current_stream().cuda_stream)
    assert status == moe.MOE_OK, moe.status_str(status)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy()


def _same(got, ref, n):
    """BF16 outputs equal bit for bit on the live rows; rows past the live count keep the poison."""
    assert np.array_equal(got[:n], ref[:n])
    assert np.all(got[n:] == -1)


def _small_case(name, E, H, I, topk, M, n=None):
    return synth.make_case(name, M, n, shape=synth.small_shape(name, E=E, H=H, I=I, topk=topk))


def test_static_forward_matches_workspace_forward_twice():
    moe.load_library(build_if_missing=True)
    tiny = synth.make_case("tiny", 16)
    dev_t = device_case(tiny)
    ref_t = _reference(tiny, dev_t)
    # two calls in a row on the shared array
    _same(_static(tiny, dev_t), ref_t, tiny.n)
    _same(_static(tiny, dev_t), ref_t, tiny.n)
    # a different layer in between, then the first one again: the array keeps the previous
    # call's contents, which must not leak into the next result
    dec = synth.make_case("decode", 1)
    dev_d = device_case(dec)
    ref_d = _reference(dec, dev_d)
    _same(_static(dec, dev_d), ref_d, dec.n)
    partial = synth.make_case("tiny", 16, 9)
    dev_p = device_case(partial)
    _same(_static(partial, dev_p), _reference(partial, dev_p), partial.n)
    _same(_static(tiny, dev_t), ref_t, tiny.n)


def test_static_forward_resets_split_k_counters_and_alignment_counts():
    """The two pieces of array state that must start from zero on every call: the split-K arrival
    counters (a plan whose FC1 splits K eight ways) and the per-CTA expert counts of the multi-CTA
    alignment (4800 pairs).  Each runs after a different layer has left the array dirty, twice."""
    ksplit = _small_case("nz_ksplit", 2, 4096, 128, 1, 8)
    multi = _small_case("nz_align", 16, 256, 256, 8, 600, 590)
    plan_k = moe.workspace_plan(8, 2, 4096, 128, 1)
    plan_m = moe.workspace_plan(600, 16, 256, 256, 8)
    assert plan_k["fc1_ksplit"] > 1 and plan_k["total_bytes"] <= moe.STATIC_SCRATCH_BYTES
    assert plan_m["align_ctas"] > 1 and plan_m["total_bytes"] <= moe.STATIC_SCRATCH_BYTES
    tiny = synth.make_case("tiny", 16)
    dev_t, dev_k, dev_m = device_case(tiny), device_case(ksplit), device_case(multi)
    ref_t, ref_k, ref_m = _reference(tiny, dev_t), _reference(ksplit, dev_k), _reference(multi, dev_m)
    for _ in range(2):
        _same(_static(multi, dev_m), ref_m, multi.n)
        _same(_static(ksplit, dev_k), ref_k, ksplit.n)
        _same(_static(tiny, dev_t), ref_t, tiny.n)


def test_static_forward_rejects_layers_beyond_the_array():
    lib = moe.load_library(build_if_missing=True)
    sh = synth.SHAPES["decode"]
    need = moe.workspace_bytes(32, sh.E, sh.H, sh.I, sh.topk, sh.act_fmt)
    assert need > moe.STATIC_SCRATCH_BYTES
    # pointers are never dereferenced: the size check comes before any launch
    args = moe.FwdArgs(256, 256, 256, None, 256, 256, 256, 256, 256, 32, sh.E, sh.H, sh.I,
                       sh.topk, sh.weight_fmt, sh.act_fmt, sh.clamp_mode, sh.limit)
    status = lib.moe_fp8_block_forward_static(ctypes.byref(args), None)
    assert status == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_fp8_block_forward_static(None, None) == moe.MOE_ERR_INVALID_ARG
