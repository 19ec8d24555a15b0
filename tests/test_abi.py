"""The C-ABI library without a GPU: it builds, loads, exports every symbol the header declares, and
its host-side plan and argument checks answer before anything is launched."""

import ctypes
import os
import re

import pytest

import block_fp8_mixture_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_fp8.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(moe_[a-z0-9_]+)\s*\(", text, re.M)
    return sorted(set(names))


def test_header_lists_entry_points():
    names = header_functions()
    for want in ("moe_align", "moe_quant_act", "moe_fp8_block_forward", "moe_workspace_bytes",
                 "moe_status_str", "moe_last_device_status"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    assert set(header_functions()) <= set(moe.SIGNATURES)


def test_version_and_status_strings(lib):
    assert b"sm_103a" in lib.moe_version()
    assert moe.status_str(moe.MOE_ERR_WORKSPACE_TOO_SMALL) == "workspace too small"
    assert moe.status_str(99) == "unknown status"


def test_plan_sizes():
    p = moe.workspace_plan(32, 288, 4096, 512, 8)
    assert p["P_cap"] == 256
    assert p["R_cap"] == 256 + 256 * 127 + (128 - (256 + 256 * 127) % 128) % 128
    assert p["T_cap"] == p["R_cap"] // 128
    offs = [p[k] for k in ("status", "num_tiles", "seg_start", "live_end", "sorted_pair",
                           "pair_row", "tile_expert", "a1_q", "a1_s", "a2_q", "a2_s", "y")]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert p["y"] + p["R_cap"] * 4096 * 2 <= p["total_bytes"]
    assert moe.workspace_bytes(32, 288, 4096, 512, 8) == p["total_bytes"]
    # small batches split FC1's K; large ones do not
    assert moe.workspace_plan(1, 288, 4096, 512, 8)["fc1_ksplit"] == 4
    assert moe.workspace_plan(32, 288, 4096, 512, 8)["fc1_ksplit"] == 1
    assert moe.workspace_plan(32, 288, 4096, 512, 8)["small_batch"] == 1
    assert moe.workspace_plan(32, 288, 4096, 512, 8)["align_ctas"] == 1
    assert moe.workspace_plan(8192, 128, 2048, 768, 8)["align_ctas"] == 64
    assert moe.workspace_plan(4096, 32, 7168, 2048, 8)["fc1_ksplit"] == 1
    # UE8M0 scales take one byte
    p8 = moe.workspace_plan(32, 288, 4096, 512, 8, moe.SCALE_UE8M0)
    assert p8["a2_q"] - p8["a1_s"] < p["a2_q"] - p["a1_s"]


@pytest.mark.parametrize("shape,status", [
    ((16, 8, 500, 256, 2), moe.MOE_ERR_UNSUPPORTED_SHAPE),     # H % 128
    ((16, 8, 512, 200, 2), moe.MOE_ERR_UNSUPPORTED_SHAPE),     # I % 128
    ((16, 2000, 512, 256, 2), moe.MOE_ERR_UNSUPPORTED_SHAPE),  # E > 1024
    ((16, 8, 512, 256, 17), moe.MOE_ERR_UNSUPPORTED_SHAPE),    # topk > 16
    ((1 << 18, 8, 512, 256, 8), moe.MOE_ERR_UNSUPPORTED_SHAPE),
    ((-1, 8, 512, 256, 2), moe.MOE_ERR_INVALID_ARG),
    ((16, 0, 512, 256, 2), moe.MOE_ERR_INVALID_ARG),
])
def test_plan_rejects_bad_shapes(lib, shape, status):
    plan = moe.WsPlan()
    assert lib.moe_workspace_plan(*shape, 0, ctypes.byref(plan)) == status
    assert lib.moe_workspace_bytes(*shape, 0) == 0


def _args(**kw):
    base = dict(x=256, topk_ids=256, topk_weights=256, d_num_tokens=None, w13=256, s13=256, w2=256,
                s2=256, out=256, M_cap=16, E=8, H=512, I=256, topk=2, weight_scale_fmt=0,
                act_scale_fmt=0, clamp_mode=0, clamp_limit=0.0)
    base.update(kw)
    return moe.FwdArgs(**base)


def test_forward_validates_before_launch(lib):
    """Every rejection below happens on the host: no device, no launch."""
    need = lib.moe_workspace_bytes(16, 8, 512, 256, 2, 0)
    ws = 1 << 20    # a fake, 256-aligned device address: never dereferenced on these paths
    fwd = lib.moe_fp8_block_forward
    assert fwd(None, ws, need, None) == moe.MOE_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_args()), ws, need - 1, None) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    assert fwd(ctypes.byref(_args()), ws + 16, need, None) == moe.MOE_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_args()), None, need, None) == moe.MOE_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_args(x=None)), ws, need, None) == moe.MOE_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_args(x=258)), ws, need, None) == moe.MOE_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_args(w13=264)), ws, need, None) == moe.MOE_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_args(out=None)), ws, need, None) == moe.MOE_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_args(clamp_mode=3)), ws, need, None) == moe.MOE_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_args(clamp_mode=1, clamp_limit=-1.0)), ws, need, None) == moe.MOE_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_args(act_scale_fmt=7)), ws, need, None) == moe.MOE_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_args(H=300)), ws, need, None) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert fwd(ctypes.byref(_args(weight_scale_fmt=0, s13=258)), ws, need, None) == moe.MOE_ERR_INVALID_ARG
    # zero-capacity layer: valid, nothing to do
    assert fwd(ctypes.byref(_args(M_cap=0)), ws, lib.moe_workspace_bytes(0, 8, 512, 256, 2, 0), None) == moe.MOE_OK
    assert lib.moe_align(None, None, 16, 2, 8, 0, 512, 256, 0, ws, need, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_quant_act(None, None, 16, 8, 512, 256, 2, 0, 0, ws, need, None) == moe.MOE_ERR_INVALID_ARG
    assert fwd(ctypes.byref(_args(numerics=2)), ws, need, None) == moe.MOE_ERR_INVALID_ARG
    wt = lib.moe_selftest_wait_timeout
    assert wt(None, 100, None) == moe.MOE_ERR_INVALID_ARG
    assert wt(ws + 16, 100, None) == moe.MOE_ERR_INVALID_ARG
    assert wt(ws, 0, None) == moe.MOE_ERR_INVALID_ARG
    assert wt(ws, 1000001, None) == moe.MOE_ERR_INVALID_ARG


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(moe, "_LIB", None)
    monkeypatch.setattr(moe, "LIBPATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        moe.load_library()


def test_expert_slices_partition_the_experts():
    for E in (1, 7, 16, 288):
        for world in (1, 2, 3, 8):
            spans = [moe.expert_slice(E, world, r) for r in range(world)]
            covered = [e for first, count in spans for e in range(first, first + count)]
            assert covered == list(range(E))
            assert max(c for _, c in spans) - min(c for _, c in spans) <= 1


def test_weight_bytes_per_expert_match_printed_figure():
    """The byte count of the roofline (bench.layer_work) charges each occupied expert its W13 and W2
    codes plus block scales; for two experts of H=7168, I=2048 the pages print about 88 MB of
    weights (tests/golden/expert_weight_bytes.json)."""
    import json
    import types

    import numpy as np

    import bench
    import synth
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "expert_weight_bytes.json")))
    shape = synth.LayerShape("g", 32, g["H"], g["I"], 8)
    case = types.SimpleNamespace(shape=shape, n=1,
                                 topk_ids=np.arange(g["experts"], dtype=np.int32)[None, :])
    work = bench.layer_work(case)
    assert work["occupied_experts"] == g["experts"]
    weights = work["layer_bytes"] - 4 * g["H"] - 8 * shape.topk
    codes = g["experts"] * 3 * g["H"] * g["I"]
    assert round(codes / 1e6) == g["printed_mb"]
    assert codes <= weights <= codes * 1.001       # the block scales add under 0.1%
