"""Block-FP8 mixture-of-experts layer forward on one GB300 (sm_103a).

Thin Python binding of the C ABI in include/moe_fp8.h (libmoe_fp8.so, built in-tree by
block_fp8_mixture_gb300.build).  The functions here only marshal arguments: every step of the layer
runs in the library's CUDA kernels.  PyTorch supplies device memory and streams.  If the library is
missing, loading fails loudly; there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import build as _build

SCALE_FP32 = 0
SCALE_FP32_POW2 = 1
SCALE_UE8M0 = 2
CLAMP_NONE = 0
CLAMP_BEFORE_SILU = 1
CLAMP_AFTER_SILU = 2
NUMERICS_DIVIDE = 0
NUMERICS_RECIPROCAL = 1

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_TIMEOUT = 5

LIBPATH = _build.LIBPATH


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} (status {status})")


class WsPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "status", "num_tiles", "seg_start", "live_end", "sorted_pair", "pair_row", "tile_expert",
        "num_chunks", "chunk_row0", "align_hist", "a1_q", "a1_s", "a2_q", "a2_s", "y", "g1",
        "splitk_partial", "splitk_count", "total_bytes")] + [
        ("R_cap", ctypes.c_int32), ("T_cap", ctypes.c_int32), ("C_cap", ctypes.c_int32),
        ("P_cap", ctypes.c_int32), ("fc1_ksplit", ctypes.c_int32), ("small_batch", ctypes.c_int32),
        ("align_ctas", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class FwdArgs(ctypes.Structure):
    _fields_ = [
        ("x", ctypes.c_void_p), ("topk_ids", ctypes.c_void_p), ("topk_weights", ctypes.c_void_p),
        ("d_num_tokens", ctypes.c_void_p), ("w13", ctypes.c_void_p), ("s13", ctypes.c_void_p),
        ("w2", ctypes.c_void_p), ("s2", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("M_cap", ctypes.c_int), ("E", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
        ("topk", ctypes.c_int), ("weight_scale_fmt", ctypes.c_int), ("act_scale_fmt", ctypes.c_int),
        ("clamp_mode", ctypes.c_int), ("clamp_limit", ctypes.c_float), ("numerics", ctypes.c_int),
        ("expert_offset", ctypes.c_int), ("out_fp32", ctypes.c_int),
    ]


class BatchedArgs(ctypes.Structure):
    _fields_ = [
        ("x", ctypes.c_void_p), ("d_counts", ctypes.c_void_p), ("w13", ctypes.c_void_p),
        ("s13", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("s2", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("E", ctypes.c_int), ("max_m", ctypes.c_int),
        ("H", ctypes.c_int), ("I", ctypes.c_int), ("weight_scale_fmt", ctypes.c_int),
        ("act_scale_fmt", ctypes.c_int), ("clamp_mode", ctypes.c_int),
        ("clamp_limit", ctypes.c_float), ("numerics", ctypes.c_int),
    ]


_LIB = None
# every function the header declares, with its ctypes signature (restype, argtypes)
_VP, _SZ, _I, _P = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.POINTER
SIGNATURES = {
    "moe_workspace_plan": (_I, [_I, _I, _I, _I, _I, _I, _P(WsPlan)]),
    "moe_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moe_align": (_I, [_VP, _VP, _I, _I, _I, _I, _I, _I, _I, _VP, _SZ, _VP]),
    "moe_quant_act": (_I, [_VP, _VP, _I, _I, _I, _I, _I, _I, _I, _VP, _SZ, _VP]),
    "moe_fc1_swiglu_quant": (_I, [_P(FwdArgs), _VP, _SZ, _VP]),
    "moe_fc2": (_I, [_P(FwdArgs), _VP, _SZ, _VP]),
    "moe_topk_reduce": (_I, [_P(FwdArgs), _VP, _SZ, _VP]),
    "moe_fp8_block_forward": (_I, [_P(FwdArgs), _VP, _SZ, _VP]),
    "moe_fp8_block_forward_static": (_I, [_P(FwdArgs), _VP]),
    "moe_batched_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_fp8_batched_forward": (_I, [_P(BatchedArgs), _VP, _SZ, _VP]),
    "moe_last_device_status": (_I, [_VP, _VP]),
    "moe_selftest_wait_timeout": (_I, [_VP, _I, _VP]),
    "moe_status_str": (ctypes.c_char_p, [_I]),
    "moe_version": (ctypes.c_char_p, []),
}


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libmoe_fp8.so (building it first when asked); raises if it is unavailable."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if build_if_missing:
        _build.build()
    if not os.path.exists(LIBPATH):
        raise RuntimeError(
            f"{LIBPATH} is missing: build it with `python -m block_fp8_mixture_gb300.build` "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(LIBPATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def status_str(status: int) -> str:
    return load_library().moe_status_str(status).decode()


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def workspace_plan(M_cap: int, E: int, H: int, I: int, topk: int, act_fmt: int = SCALE_FP32) -> dict:
    plan = WsPlan()
    _check(load_library().moe_workspace_plan(M_cap, E, H, I, topk, act_fmt, ctypes.byref(plan)),
           "moe_workspace_plan")
    return plan.as_dict()


def workspace_bytes(M_cap: int, E: int, H: int, I: int, topk: int, act_fmt: int = SCALE_FP32) -> int:
    return load_library().moe_workspace_bytes(M_cap, E, H, I, topk, act_fmt)


def alloc_workspace(M_cap: int, E: int, H: int, I: int, topk: int, act_fmt: int = SCALE_FP32,
                    device="cuda"):
    """A caller-owned workspace tensor (uint8) of the size the plan asks for."""
    import torch
    return torch.empty(max(1, workspace_bytes(M_cap, E, H, I, topk, act_fmt)), dtype=torch.uint8,
                       device=device)


def workspace_views(ws, M_cap: int, E: int, H: int, I: int, topk: int, act_fmt: int = SCALE_FP32):
    """Typed views of the workspace sub-buffers (for inspecting intermediates)."""
    import torch
    p = workspace_plan(M_cap, E, H, I, topk, act_fmt)
    R, T, P = p["R_cap"], p["T_cap"], p["P_cap"]
    sdt, ssz = (torch.uint8, 1) if act_fmt == SCALE_UE8M0 else (torch.float32, 4)

    def view(off, count, dtype, size):
        return ws[off: off + count * size].view(dtype)

    return {
        "plan": p,
        "status": view(p["status"], 1, torch.int32, 4),
        "num_tiles": view(p["num_tiles"], 1, torch.int32, 4),
        "seg_start": view(p["seg_start"], E + 1, torch.int32, 4),
        "live_end": view(p["live_end"], E, torch.int32, 4),
        "sorted_pair": view(p["sorted_pair"], R, torch.int32, 4),
        "pair_row": view(p["pair_row"], P, torch.int32, 4),
        "tile_expert": view(p["tile_expert"], T, torch.int32, 4),
        "num_chunks": view(p["num_chunks"], 1, torch.int32, 4),
        "chunk_row0": view(p["chunk_row0"], p["C_cap"], torch.int32, 4),
        "a1_q": view(p["a1_q"], R * H, torch.uint8, 1).view(R, H),
        "a1_s": view(p["a1_s"], (H // 128) * R, sdt, ssz).view(H // 128, R),
        "a2_q": view(p["a2_q"], R * I, torch.uint8, 1).view(R, I),
        "a2_s": view(p["a2_s"], (I // 128) * R, sdt, ssz).view(I // 128, R),
        "y": view(p["y"], R * H, torch.int16, 2).view(R, H),
        "g1": view(p["g1"], R * 2 * I, torch.int16, 2).view(R, 2 * I) if p["g1"] else None,
    }


def make_args(x, topk_ids, topk_weights, w13, s13, w2, s2, out, *, E, H, I, topk, M_cap=None,
              d_num_tokens=None, weight_fmt=SCALE_FP32, act_fmt=SCALE_FP32,
              clamp_mode=CLAMP_NONE, clamp_limit=0.0, numerics=NUMERICS_DIVIDE, expert_offset=0,
              out_fp32=False) -> FwdArgs:
    if M_cap is None:
        M_cap = x.shape[0] if x is not None else topk_ids.shape[0]
    return FwdArgs(_ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(d_num_tokens), _ptr(w13),
                   _ptr(s13), _ptr(w2), _ptr(s2), _ptr(out), M_cap, E, H, I, topk, weight_fmt,
                   act_fmt, clamp_mode, float(clamp_limit), numerics, expert_offset,
                   1 if out_fp32 else 0)


def align(topk_ids, E: int, H: int, I: int, workspace, *, d_num_tokens=None,
          act_fmt: int = SCALE_FP32, expert_offset: int = 0, stream=None):
    M_cap, topk = topk_ids.shape
    _check(load_library().moe_align(_ptr(topk_ids), _ptr(d_num_tokens), M_cap, topk, E, expert_offset,
                                    H, I, act_fmt, _ptr(workspace), workspace.numel(),
                                    _stream(stream)), "moe_align")


def expert_slice(num_experts: int, world: int, rank: int):
    """(first expert, expert count) of `rank` when `world` ranks split the experts into contiguous,
    near-equal slices (the first num_experts % world ranks hold one more)."""
    base, extra = divmod(num_experts, world)
    count = base + (1 if rank < extra else 0)
    first = rank * base + min(rank, extra)
    return first, count


def quant_act(x, topk: int, E: int, I: int, workspace, *, d_num_tokens=None,
              act_fmt: int = SCALE_FP32, numerics: int = NUMERICS_DIVIDE, stream=None):
    M_cap, H = x.shape
    _check(load_library().moe_quant_act(_ptr(x), _ptr(d_num_tokens), M_cap, E, H, I, topk, act_fmt,
                                        numerics, _ptr(workspace), workspace.numel(),
                                        _stream(stream)),
           "moe_quant_act")


def _run(name: str, args: FwdArgs, workspace, stream):
    fn = getattr(load_library(), name)
    _check(fn(ctypes.byref(args), _ptr(workspace), workspace.numel(), _stream(stream)), name)


def fc1_swiglu_quant(args: FwdArgs, workspace, stream=None):
    _run("moe_fc1_swiglu_quant", args, workspace, stream)


def fc2(args: FwdArgs, workspace, stream=None):
    _run("moe_fc2", args, workspace, stream)


def topk_reduce(args: FwdArgs, workspace, stream=None):
    _run("moe_topk_reduce", args, workspace, stream)


def forward(args: FwdArgs, workspace, stream=None):
    """The whole layer (moe_fp8_block_forward) on `stream` (default: torch's current stream)."""
    _run("moe_fp8_block_forward", args, workspace, stream)


def forward_static(args: FwdArgs, stream=None):
    """The whole layer without a caller workspace (moe_fp8_block_forward_static): for callers that
    cannot allocate device memory; small layers only (workspace <= STATIC_SCRATCH_BYTES)."""
    _check(load_library().moe_fp8_block_forward_static(ctypes.byref(args), _stream(stream)),
           "moe_fp8_block_forward_static")


STATIC_SCRATCH_BYTES = 32 << 20


def batched_workspace_bytes(E: int, max_m: int, H: int, I: int, act_fmt: int = SCALE_FP32) -> int:
    n = load_library().moe_batched_workspace_bytes(E, max_m, H, I, act_fmt)
    if n == 0:
        raise MoeError(MOE_ERR_UNSUPPORTED_SHAPE, "moe_batched_workspace_bytes")
    return n


def alloc_batched_workspace(E: int, max_m: int, H: int, I: int, act_fmt: int = SCALE_FP32,
                            device="cuda"):
    import torch
    return torch.empty(batched_workspace_bytes(E, max_m, H, I, act_fmt), dtype=torch.uint8,
                       device=device)


def batched_forward(x, d_counts, w13, s13, w2, s2, out, workspace, *, weight_fmt=SCALE_FP32,
                    act_fmt=SCALE_FP32, clamp_mode=CLAMP_NONE, clamp_limit=0.0,
                    numerics=NUMERICS_DIVIDE, stream=None):
    """The batched-expert layer (moe_fp8_batched_forward): x and out [E, max_m, H] BF16, d_counts
    device int32 [E]; rows r >= counts[e] of out are left as they were."""
    E, max_m, H = x.shape
    a = BatchedArgs(_ptr(x), _ptr(d_counts), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), _ptr(out),
                    E, max_m, H, w13.shape[1] // 2, weight_fmt, act_fmt, clamp_mode, clamp_limit,
                    numerics)
    _check(load_library().moe_fp8_batched_forward(ctypes.byref(a), _ptr(workspace),
                                                  workspace.numel(), _stream(stream)),
           "moe_fp8_batched_forward")


def last_device_status(workspace, stream=None) -> int:
    return load_library().moe_last_device_status(_ptr(workspace), _stream(stream))


def selftest_wait_timeout(workspace, limit_us: int, stream=None):
    """Run the bounded-wait diagnostic: a device wait that nothing completes runs out after
    `limit_us` and records MOE_ERR_DEVICE_TIMEOUT in the workspace status word."""
    _check(load_library().moe_selftest_wait_timeout(_ptr(workspace), int(limit_us), _stream(stream)),
           "moe_selftest_wait_timeout")


class MoELayer:
    """A block-FP8 MoE layer with resident weights and a caller-owned workspace.

    Weights are device tensors: w13 E4M3 codes [E, 2I, H] (uint8 or float8_e4m3fn), s13 block scales
    [E, 2I/128, H/128] (fp32, or uint8 UE8M0), w2 [E, H, I], s2 [E, H/128, I/128].
    """

    def __init__(self, w13, s13, w2, s2, *, weight_fmt=SCALE_FP32, act_fmt=SCALE_FP32,
                 clamp_mode=CLAMP_NONE, clamp_limit=0.0, max_tokens: int, topk: int,
                 numerics=NUMERICS_DIVIDE, expert_offset: int = 0, out_fp32: bool = False):
        self.w13, self.s13, self.w2, self.s2 = w13, s13, w2, s2
        self.E, two_i, self.H = w13.shape
        self.I = two_i // 2
        self.topk = topk
        self.M_cap = max_tokens
        self.weight_fmt, self.act_fmt = weight_fmt, act_fmt
        self.clamp_mode, self.clamp_limit = clamp_mode, clamp_limit
        self.numerics = numerics
        self.expert_offset, self.out_fp32 = expert_offset, out_fp32
        self.workspace = alloc_workspace(max_tokens, self.E, self.H, self.I, topk, act_fmt,
                                         device=w13.device)

    def args(self, x, topk_ids, topk_weights, out, d_num_tokens=None) -> FwdArgs:
        return make_args(x, topk_ids, topk_weights, self.w13, self.s13, self.w2, self.s2, out,
                         E=self.E, H=self.H, I=self.I, topk=self.topk, M_cap=x.shape[0],
                         d_num_tokens=d_num_tokens, weight_fmt=self.weight_fmt,
                         act_fmt=self.act_fmt, clamp_mode=self.clamp_mode,
                         clamp_limit=self.clamp_limit, numerics=self.numerics,
                         expert_offset=self.expert_offset, out_fp32=self.out_fp32)

    def __call__(self, x, topk_ids, topk_weights, out=None, d_num_tokens=None, stream=None):
        import torch
        if x.shape[0] > self.M_cap:
            raise ValueError(f"{x.shape[0]} tokens exceed the layer's capacity {self.M_cap}")
        if out is None:
            out = torch.empty(x.shape, dtype=torch.float32 if self.out_fp32 else x.dtype,
                              device=x.device)
        forward(self.args(x, topk_ids, topk_weights, out, d_num_tokens), self.workspace, stream)
        return out
