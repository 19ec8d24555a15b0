"""Seeded synthetic inputs for the block-FP8 MoE layer (shared by the CUDA-path
tests, the oracle tests, the smoke check and the benchmark).

This module holds input recipes only: token activations, router outputs and
block-quantized expert weights.  The weights stand in for an FP8 checkpoint
with 128x128 block scales; their E4M3 codes come from torch's own
float32 -> float8_e4m3fn conversion and their scales are amax/448 per block
(rounded up to a power of two for UE8M0 checkpoints).  Nothing here computes
any step of the layer.

Workload shapes follow the pages' benchmark shapes, scaled to synthetic data:
  tiny       E=8   H=512  I=256  k=2  M=16
  decode     E=288 H=4096 I=512  k=8  M in {1,4,32}, SwiGLU clamp 7.0
  padded     E=32  H=7168 I=2048 k=8  capacity 512 / 16 live, 4096 / 4096 live, UE8M0
  glm_slice  E=256 H=6144 I=256  k=8  M in {1,8,64,256,1024,4096}, Zipf(1.2) routing
  mid        E=128 H=2048 I=768  k=8  M in {1,8,32,128,512,2048,8192}, 1% outliers x10
  glm_slice_pow2  glm_slice with power-of-two-rounded fp32 activation scales
  mid_empty       mid with every fourth expert never routed to
"""

from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os
from typing import Optional

import numpy as np

SCALE_FP32 = 0
SCALE_FP32_POW2 = 1
SCALE_UE8M0 = 2
CLAMP_NONE = 0
CLAMP_BEFORE_SILU = 1
CLAMP_AFTER_SILU = 2

BLOCK = 128


@dataclasses.dataclass
class LayerShape:
    name: str
    E: int
    H: int
    I: int
    topk: int
    act_fmt: int = SCALE_FP32
    weight_fmt: int = SCALE_FP32
    clamp_mode: int = CLAMP_NONE
    limit: float = 0.0
    routing: str = "softmax"       # softmax | zipf | softmax_empty4
    outliers: float = 0.0          # fraction of x elements multiplied by 10
    cfg_id: int = 0
    numerics: int = 0              # 0: divide by the scale; 1: multiply by RN(448/amax)


SHAPES = {
    "tiny": LayerShape("tiny", 8, 512, 256, 2, cfg_id=1),
    "decode": LayerShape("decode", 288, 4096, 512, 8, clamp_mode=CLAMP_BEFORE_SILU,
                         limit=7.0, cfg_id=2),
    "padded": LayerShape("padded", 32, 7168, 2048, 8, act_fmt=SCALE_UE8M0,
                         weight_fmt=SCALE_UE8M0, cfg_id=3),
    # the same layer with FP32 128x128 weight scales and FP32 1x128 activation scales (the pages
    # also time this shape with plain FP32 scales)
    "padded_fp32": LayerShape("padded_fp32", 32, 7168, 2048, 8, cfg_id=3),
    "glm_slice": LayerShape("glm_slice", 256, 6144, 256, 8, routing="zipf", cfg_id=4),
    "mid": LayerShape("mid", 128, 2048, 768, 8, routing="softmax", outliers=0.01, cfg_id=5),
    # the variants the two swept configurations also name: power-of-two-rounded activation scales,
    # and routing with forced-empty experts (every fourth expert never chosen)
    "glm_slice_pow2": LayerShape("glm_slice_pow2", 256, 6144, 256, 8, act_fmt=SCALE_FP32_POW2,
                                 routing="zipf", cfg_id=4),
    "mid_empty": LayerShape("mid_empty", 128, 2048, 768, 8, routing="softmax_empty4",
                            outliers=0.01, cfg_id=5),
}

# M values of each workload (capacity, live) pairs
SWEEPS = {
    "tiny": [(16, 16)],
    "decode": [(1, 1), (4, 4), (32, 32)],
    "padded": [(512, 16), (4096, 4096)],
    "padded_fp32": [(512, 16), (4096, 4096)],
    "glm_slice": [(m, m) for m in (1, 8, 64, 256, 1024, 4096)],
    "mid": [(m, m) for m in (1, 8, 32, 128, 512, 2048, 8192)],
    "glm_slice_pow2": [(m, m) for m in (1, 8, 64, 256, 1024, 4096)],
    "mid_empty": [(m, m) for m in (1, 8, 32, 128, 512, 2048, 8192)],
}


@dataclasses.dataclass
class Weights:
    w13: np.ndarray   # uint8 E4M3 codes [E, 2I, H]
    s13: np.ndarray   # fp32 or uint8 UE8M0 [E, 2I/128, H/128]
    w2: np.ndarray    # uint8 [E, H, I]
    s2: np.ndarray    # [E, H/128, I/128]


@dataclasses.dataclass
class LayerCase:
    shape: LayerShape
    M_cap: int
    n: int
    x_bits: np.ndarray        # uint16 BF16 patterns [M_cap, H]
    x: np.ndarray             # fp32 values of the same BF16 numbers
    topk_ids: np.ndarray      # int32 [M_cap, k]
    topk_weights: np.ndarray  # fp32 [M_cap, k]
    weights: Weights


def _to_bf16(v: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16).copy()
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    return bits, vals


def _quantize_blocks(w: np.ndarray, fmt: int):
    """Checkpoint-style 128x128 block quantization of one expert matrix [N, K]."""
    import torch
    n, k = w.shape
    blocks = w.reshape(n // BLOCK, BLOCK, k // BLOCK, BLOCK)
    amax = np.abs(blocks).max(axis=(1, 3)).astype(np.float32)
    amax = np.where(amax > 0, amax, np.float32(1.0))
    s = (amax / np.float32(448.0)).astype(np.float32)
    if fmt == SCALE_UE8M0:
        mant, ex = np.frexp(s.astype(np.float64))          # s = mant * 2^ex, mant in [0.5, 1)
        ex = np.where(mant == 0.5, ex - 1, ex)               # exact powers of two stay
        s = np.ldexp(np.float64(1.0), ex).astype(np.float32)
        stored = (ex + 127).astype(np.uint8)
    else:
        stored = s
    scaled = blocks / s[:, None, :, None]
    codes = torch.from_numpy(np.ascontiguousarray(scaled.reshape(n, k), np.float32))
    codes = codes.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    return codes, stored


def _expert_weights(seed_seq, H, I, fmt):
    rng = np.random.Generator(np.random.PCG64(seed_seq))
    w13 = rng.standard_normal((2 * I, H), dtype=np.float32) * np.float32(0.02)
    w2 = rng.standard_normal((H, I), dtype=np.float32) * np.float32(0.02)
    q13, s13 = _quantize_blocks(w13, fmt)
    q2, s2 = _quantize_blocks(w2, fmt)
    return q13, s13, q2, s2


_WEIGHT_CACHE: dict = {}


def make_weights(shape: LayerShape, seed: Optional[int] = None) -> Weights:
    """Block-quantized expert weights N(0, 0.02), one independent stream per expert."""
    seed = 1000 * shape.cfg_id if seed is None else seed
    key = (shape.name, shape.E, shape.H, shape.I, shape.weight_fmt, seed)
    if key in _WEIGHT_CACHE:
        return _WEIGHT_CACHE[key]
    E, H, I = shape.E, shape.H, shape.I
    sdt = np.uint8 if shape.weight_fmt == SCALE_UE8M0 else np.float32
    w13 = np.empty((E, 2 * I, H), np.uint8)
    s13 = np.empty((E, 2 * I // BLOCK, H // BLOCK), sdt)
    w2 = np.empty((E, H, I), np.uint8)
    s2 = np.empty((E, H // BLOCK, I // BLOCK), sdt)
    children = np.random.SeedSequence(seed).spawn(E)

    def one(e):
        q13, a, q2, b = _expert_weights(children[e], H, I, shape.weight_fmt)
        w13[e], s13[e], w2[e], s2[e] = q13, a, q2, b

    workers = max(1, min(16, os.cpu_count() or 1))
    with _cf.ThreadPoolExecutor(workers) as pool:
        list(pool.map(one, range(E)))
    out = Weights(w13, s13, w2, s2)
    _WEIGHT_CACHE[key] = out
    return out


def _softmax(z):
    z = z - z.max(axis=-1, keepdims=True)
    p = np.exp(z)
    return p / p.sum(axis=-1, keepdims=True)


def make_routing(kind: str, M: int, E: int, topk: int, rng: np.random.Generator):
    """Router outputs: expert ids int32 [M, k] and renormalized fp32 weights [M, k]."""
    if kind in ("softmax", "softmax_empty4"):
        logits = rng.standard_normal((M, E))
        if kind == "softmax_empty4":
            logits[:, ::4] = -np.inf
        p = _softmax(logits)
        ids = np.argsort(-p, axis=1, kind="stable")[:, :topk]
        w = np.take_along_axis(p, ids, axis=1)
    elif kind == "zipf":
        perm = np.random.Generator(np.random.PCG64(4242)).permutation(E)
        pop = np.empty(E)
        pop[perm] = 1.0 / np.arange(1, E + 1) ** 1.2
        logp = np.log(pop / pop.sum())
        gumbel = -np.log(-np.log(rng.uniform(size=(M, E))))
        ids = np.argsort(-(logp[None, :] + gumbel), axis=1, kind="stable")[:, :topk]
        w = _softmax(rng.standard_normal((M, topk)))
    else:
        raise ValueError(kind)
    w = w / w.sum(axis=1, keepdims=True)
    return ids.astype(np.int32), w.astype(np.float32)


def make_case(name: str, M_cap: int, n: Optional[int] = None, *,
              routing: Optional[str] = None, seed: Optional[int] = None,
              shape: Optional[LayerShape] = None, weights: Optional[Weights] = None) -> LayerCase:
    """A full layer input: x, routing and weights for one workload point."""
    shape = shape or SHAPES[name]
    n = M_cap if n is None else n
    seed = 1000 * shape.cfg_id + M_cap if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((M_cap, shape.H), dtype=np.float32)
    if shape.outliers > 0:
        mask = rng.uniform(size=x.shape) < shape.outliers
        x = np.where(mask, x * np.float32(10.0), x).astype(np.float32)
    x_bits, x_vals = _to_bf16(x)
    ids, w = make_routing(routing or shape.routing, M_cap, shape.E, shape.topk, rng)
    weights = weights if weights is not None else make_weights(shape)
    return LayerCase(shape, M_cap, n, x_bits, x_vals, ids, w, weights)


def small_shape(name="small", E=8, H=512, I=256, topk=2, **kw) -> LayerShape:
    """A reduced shape for fast tests (same recipe as the workloads above)."""
    return LayerShape(name, E, H, I, topk, **kw)
