"""Shared helpers of the GPU parity tests: move a synthetic case to the device, run the library
through its C ABI, and build the oracle's expectations for the same inputs."""

from __future__ import annotations

import numpy as np

import oracle
import synth

# layer outputs: |gpu - oracle| <= REL_TOL * max|oracle| per element (accumulation order differs)
REL_TOL = 1e-2
# share of FC2-input FP8 codes that must be identical to the oracle's
CODE_MATCH_MIN = 0.999


def device_case(case: synth.LayerCase, device="cuda"):
    import torch
    w = case.weights
    d = {
        "x": torch.from_numpy(case.x_bits.view(np.int16)).to(device).view(torch.bfloat16),
        "ids": torch.from_numpy(case.topk_ids).to(device),
        "w": torch.from_numpy(case.topk_weights).to(device),
        "w13": torch.from_numpy(w.w13).to(device),
        "s13": torch.from_numpy(w.s13).to(device),
        "w2": torch.from_numpy(w.w2).to(device),
        "s2": torch.from_numpy(w.s2).to(device),
        "n": torch.tensor([case.n], dtype=torch.int32, device=device),
    }
    return d


def run_forward(case: synth.LayerCase, dev=None, *, poison=True, use_device_n=True, ws=None,
                out=None, stream=None):
    """Run moe_fp8_block_forward on the case; returns (out, workspace, views)."""
    import torch
    import block_fp8_mixture_gb300 as moe
    sh = case.shape
    dev = dev or device_case(case)
    if ws is None:
        ws = moe.alloc_workspace(case.M_cap, sh.E, sh.H, sh.I, sh.topk, sh.act_fmt)
        if poison:
            ws.fill_(0xFF)
    if out is None:
        out = torch.empty((case.M_cap, sh.H), dtype=torch.bfloat16, device="cuda")
        if poison:
            out.view(torch.int16).fill_(-1)
    args = moe.make_args(dev["x"], dev["ids"], dev["w"], dev["w13"], dev["s13"], dev["w2"], dev["s2"],
                         out, E=sh.E, H=sh.H, I=sh.I, topk=sh.topk, M_cap=case.M_cap,
                         d_num_tokens=dev["n"] if use_device_n else None,
                         weight_fmt=sh.weight_fmt, act_fmt=sh.act_fmt, clamp_mode=sh.clamp_mode,
                         clamp_limit=sh.limit, numerics=sh.numerics)
    moe.forward(args, ws, stream)
    views = moe.workspace_views(ws, case.M_cap, sh.E, sh.H, sh.I, sh.topk, sh.act_fmt)
    return out, ws, views


def oracle_forward(case: synth.LayerCase, tokens=None, return_pairs=False):
    sh = case.shape
    w = case.weights
    tokens = np.arange(case.n) if tokens is None else np.asarray(tokens)
    return oracle.moe_forward(case.x, case.topk_ids, case.topk_weights, w.w13, w.s13, w.w2, w.s2,
                              act_fmt=sh.act_fmt, weight_fmt=sh.weight_fmt,
                              clamp_mode=sh.clamp_mode, limit=sh.limit, tokens=tokens,
                              return_pairs=return_pairs, numerics=sh.numerics)


def bf16_tensor_to_f32(t) -> np.ndarray:
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32).__lshift__(16).view(np.float32)


def assert_layer_close(gpu: np.ndarray, ref: np.ndarray, what=""):
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite outputs"
    bound = REL_TOL * float(np.abs(ref).max())
    err = np.abs(gpu.astype(np.float64) - ref.astype(np.float64))
    assert err.max() <= bound, f"{what}: max err {err.max():.3e} > {bound:.3e}"
    return err.max() / max(float(np.abs(ref).max()), 1e-30)


def scale_values(arr, act_fmt) -> np.ndarray:
    a = np.asarray(arr)
    if act_fmt == oracle.SCALE_UE8M0:
        return oracle.ue8m0_to_f32(a.astype(np.uint8))
    return a.astype(np.float32)


def check_a2_codes(case, views, pairs) -> float:
    """Share of FC2-input codes identical to the oracle's, over all live pairs compared."""
    pair_row = views["pair_row"].cpu().numpy()
    a2q = views["a2_q"]
    same = total = 0
    k = case.shape.topk
    for (t, j), (_, inter) in pairs.items():
        row = int(pair_row[t * k + j])
        assert row >= 0
        got = a2q[row].cpu().numpy()
        same += int(np.count_nonzero(got == inter["a2_q"]))
        total += got.size
    return same / max(total, 1)


def check_untouched(case, views):
    """Rows outside the live part of every expert segment keep the 0xFF poison."""
    seg = views["seg_start"].cpu().numpy()
    live = views["live_end"].cpu().numpy()
    R = views["plan"]["R_cap"]
    dead = np.ones(R, bool)
    for e in range(case.shape.E):
        dead[seg[e]:live[e]] = False
    rows = np.nonzero(dead)[0]
    if rows.size > 4096:
        rows = np.random.default_rng(0).choice(rows, 4096, replace=False)
    import torch
    idx = torch.from_numpy(rows).to(views["a1_q"].device)
    for name in ("a1_q", "a2_q"):
        assert bool((views[name].index_select(0, idx) == 0xFF).all()), f"{name} padding written"
    assert bool((views["y"].index_select(0, idx) == -1).all()), "y padding written"
    if views.get("g1") is not None:
        assert bool((views["g1"].index_select(0, idx) == -1).all()), "FC1 output padding written"
