"""Plain CPU oracle of the block-FP8 mixture-of-experts layer forward.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU-baseline
leg of the benchmark import this module. It shares no code with the CUDA path.

The layer (composite of the three pages; step names follow the pages):

1. routing alignment -- (token, expert) pairs sorted by expert, each expert's
   segment padded to a multiple of the tile height, per-expert prefix-sum
   endpoints (vLLM "Skip padded work in block-FP8 DeepGemmExperts", Purpose;
   TensorRT-LLM "Triton FP8-activation MoE for decode-sized batches on Hopper",
   description: "single-program moe_align").
2. per-1x128 FP8 E4M3 activation quantization (TensorRT-LLM page, description;
   vLLM "per-layer activation scale format + fused SiLU+quant", Details:
   scale = max(amax/448, 1/(448*512)), then x/scale).
3. FC1 (gate+up) grouped FP8 x FP8 GEMM with 128x128 weight block scales,
   partial sums promoted once per 128-wide K block with the scale product
   a_scale*b_scale formed first (TensorRT-LLM page, human review on the scale
   product and on DeepGEMM's promotion).
4. SwiGLU (SiLU(gate)*up, optionally clamped) in fp32 without intermediate
   BF16 rounding, fused with the 1x128 requantization (vLLM per-layer scale
   page, Details, sorted-A bullet; TensorRT-LLM page, SiLU as 1/(1+exp(-x))
   with IEEE division).
5. FC2 grouped GEMM, BF16 output per pair row; routing weights NOT applied here.
6. top-k weighted unpermute/sum: the routing weights scale the BF16 expert
   outputs in fp32 (TensorRT-LLM page, rounding-fix commit message).

Readings where the pages are silent (each is listed with its reason in the
design notes): FC1 outputs are rounded to BF16 before the SwiGLU (the unfused
pipelines the pages describe write a BF16 gate/up workspace); gate rows are
[0, I) of W13 and up rows [I, 2I); the promotion acc += p*(sa*sb) is one fused
multiply-add, as the compiled kernels on the pages do; pairs inside an expert
segment are in ascending pair order; ids outside [0, E) are dropped; power-of-
two scales round up; E4M3 conversion saturates to +-448.

Everything is numpy. fp32 steps are numpy float32 operations (IEEE round to
nearest even); the 128-wide block dots are formed exactly in float64 (every
product of two E4M3 values is a multiple of 2^-18 below 2^18, so any partial
sum of 128 of them is an integer number of 2^-18 units below 2^43 < 2^53).
"""

import numpy as np

from .formats import (
    bf16_round,
    e4m3_decode,
    e4m3_encode,
    f32_exponent_field,
    fma_f32,
    pow2_ceil,
    ue8m0_to_f32,
)

# scale formats of activations and weights (vLLM per-layer scale page, Overview
# and Details; vLLM padded-work page, Purpose)
SCALE_FP32 = 0
SCALE_FP32_POW2 = 1
SCALE_UE8M0 = 2

CLAMP_NONE = 0
CLAMP_BEFORE_SILU = 1
CLAMP_AFTER_SILU = 2

# quantizer / epilogue numerics
NUMERICS_DIVIDE = 0      # vLLM fused SiLU+mul+quant: x / scale, fp32 SwiGLU output
NUMERICS_RECIPROCAL = 1  # TensorRT-LLM fused op: x * RN(448/amax), reciprocal stored as the scale,
                         # SwiGLU output rounded to BF16 before its quantization

GROUP = 128      # 1x128 activation quantization group and 128x128 weight block
ALIGN = 128      # expert segment alignment (= GEMM tile height)
F32 = np.float32
SCALE_FLOOR = F32(1.0) / F32(448.0 * 512.0)   # RN32(1/229376)


# ---------------------------------------------------------------- alignment
def align(topk_ids, n_tokens, num_experts, align_to=ALIGN, chunk_rows=32, expert_offset=0):
    """Routing alignment into per-expert prefix-sum endpoints.

    Pairs p = t*topk + j for t < n_tokens; a pair is valid when its id is in
    [0, E).  Valid pairs are stably sorted by expert (ascending p inside an
    expert).  Expert e's segment starts at seg_start[e], a multiple of
    align_to, and its live rows end at live_end[e]; the padded segment ends at
    seg_start[e+1].  Row-tile i covers rows [i*align_to, (i+1)*align_to) and
    belongs to the expert whose segment holds it; only tiles that start below
    the expert's live end exist (vLLM padded-work page, Purpose and SM90
    section: whole padded tiles are skipped, padding inside a tile remains).

    Returns a dict of int32 arrays: seg_start[E+1], live_end[E],
    pair_row[n*topk] (row of each pair, -1 when dropped), sorted_pair[rows]
    (pair of each live row, -1 on padding rows), tile_expert[num_tiles],
    num_tiles, and the small-batch work list: chunk_row0 = the first row of each
    chunk_rows-row piece of every expert's live rows (experts ascending), num_chunks.
    With expert_offset, this call holds experts [offset, offset + num_experts) of a larger set:
    ids are rebased by the offset and the others dropped (expert-parallel slice).
    """
    topk_ids = np.asarray(topk_ids, np.int64) - expert_offset   # local expert ids
    topk = topk_ids.shape[1]
    num_pairs = n_tokens * topk
    ids = topk_ids.reshape(-1)[:num_pairs]
    valid = (ids >= 0) & (ids < num_experts)
    counts = np.bincount(ids[valid], minlength=num_experts).astype(np.int64)
    padded = -(-counts // align_to) * align_to
    seg_start = np.zeros(num_experts + 1, np.int64)
    seg_start[1:] = np.cumsum(padded)
    live_end = seg_start[:-1] + counts
    rows = int(seg_start[-1])
    pair_row = np.full(num_pairs, -1, np.int64)
    sorted_pair = np.full(rows, -1, np.int64)
    for e in range(num_experts):
        pairs = np.nonzero(valid & (ids == e))[0]        # ascending pair index
        r = seg_start[e] + np.arange(pairs.size)
        pair_row[pairs] = r
        sorted_pair[r] = pairs
    num_tiles = rows // align_to
    tile_expert = np.empty(num_tiles, np.int64)
    for e in range(num_experts):
        tile_expert[seg_start[e] // align_to: seg_start[e + 1] // align_to] = e
    chunk_row0 = [int(seg_start[e]) + c * chunk_rows
                  for e in range(num_experts)
                  for c in range(-(-int(counts[e]) // chunk_rows))]
    return {
        "chunk_row0": np.asarray(chunk_row0, np.int32),
        "num_chunks": len(chunk_row0),
        "seg_start": seg_start.astype(np.int32),
        "live_end": live_end.astype(np.int32),
        "pair_row": pair_row.astype(np.int32),
        "sorted_pair": sorted_pair.astype(np.int32),
        "tile_expert": tile_expert.astype(np.int32),
        "num_tiles": int(num_tiles),
    }


# ---------------------------------------------------------- quantization
def group_scale(amax, fmt):
    """Scale of a 1x128 group from its amax: max(RN32(amax/448), RN32(1/229376)),
    rounded up to a power of two for the POW2 and UE8M0 formats."""
    amax = np.asarray(amax, F32)
    s = np.maximum(amax / F32(448.0), SCALE_FLOOR).astype(F32)
    if fmt in (SCALE_FP32_POW2, SCALE_UE8M0):
        s = pow2_ceil(s)
    return s


def quant_1x128(v, fmt, numerics=NUMERICS_DIVIDE):
    """Per-1x128-group FP8 E4M3 quantization along the last axis.

    v: fp32 [..., K] with K % 128 == 0.
    Returns (codes uint8 [..., K], scales fp32 [..., K/128]); for UE8M0 the
    scale bytes are f32_exponent_field(scales).

    NUMERICS_DIVIDE (vLLM per-layer scale page, Details): s = max(RN(amax/448),
    RN(1/229376)), codes = q8(RN(v / s)).
    NUMERICS_RECIPROCAL with fp32 scales (TensorRT-LLM page, rounding-fix
    commit: multiply by 448/amax, both correctly rounded, store the reciprocal):
    inv = min(RN(448/amax), 448*512), codes = q8(RN(v * inv)), s = RN(1/inv).
    The cap keeps the same scale floor (and handles amax = 0).  Power-of-two
    formats quantize identically in both modes (v/s = v*(1/s) exactly).
    """
    v = np.asarray(v, F32)
    k = v.shape[-1]
    g = v.reshape(v.shape[:-1] + (k // GROUP, GROUP))
    amax = np.abs(g).max(axis=-1)
    if numerics == NUMERICS_RECIPROCAL and fmt == SCALE_FP32:
        with np.errstate(divide="ignore"):
            inv = np.minimum(F32(448.0) / amax, F32(448.0 * 512.0)).astype(F32)
        q = e4m3_encode((g * inv[..., None]).astype(F32))
        s = (F32(1.0) / inv).astype(F32)
        return q.reshape(v.shape), s
    s = group_scale(amax, fmt)
    q = e4m3_encode(g / s[..., None])           # fp32 IEEE division
    return q.reshape(v.shape), s


def scale_bytes(scales):
    """fp32 power-of-two scales -> UE8M0 bytes."""
    return f32_exponent_field(scales)


def weight_scales_f32(scales, fmt):
    """Weight block scales as fp32 values (UE8M0 bytes are 2^(b-127))."""
    if fmt == SCALE_UE8M0:
        return ue8m0_to_f32(scales)
    return np.asarray(scales, F32)


# ------------------------------------------------------------- block GEMM
def block_gemm(a_q, a_s, w_q, w_s):
    """FP8 x FP8 GEMM with per-128 K-block promotion.

    a_q: uint8 [R, K] activation codes, a_s: fp32 [R, K/128] activation scales,
    w_q: uint8 [N, K] weight codes (K-major), w_s: fp32 [N/128, K/128] weight
    block scales.  For each K block kb (ascending):
        d   = exact sum of the 128 products of decoded codes
        p   = RN32(d)
        sab = RN32(a_s[r, kb] * w_s[c // 128, kb])
        acc = RN32(acc + p * sab)          (one fused multiply-add)
    Returns acc, fp32 [R, N].
    """
    r, k = a_q.shape
    n = w_q.shape[0]
    acc = np.zeros((r, n), F32)
    a_s = np.asarray(a_s, F32)
    w_s = np.asarray(w_s, F32)
    for kb in range(k // GROUP):
        cols = slice(kb * GROUP, (kb + 1) * GROUP)
        d = e4m3_decode(a_q[:, cols]) @ e4m3_decode(w_q[:, cols]).T   # exact in f64
        p = d.astype(F32)
        sw = np.repeat(w_s[:, kb], GROUP)[None, :]
        sab = (a_s[:, kb][:, None] * sw).astype(F32)
        acc = fma_f32(p, sab, acc)
    return acc


# ---------------------------------------------------------------- SwiGLU
def swiglu(gate, up, clamp_mode=CLAMP_NONE, limit=0.0):
    """SiLU(gate) * up in fp32 with the optional scalar clamp.

    sig  = RN32(1 / RN32(1 + RN32(exp(-gate))))   (IEEE division)
    silu = RN32(gate * sig);  h = RN32(silu * up)
    CLAMP_BEFORE_SILU: gate <- min(gate, L), up <- clamp(up, -L, L) first.
    CLAMP_AFTER_SILU:  silu <- min(silu, L), up <- clamp(up, -L, L).
    """
    g = np.asarray(gate, F32)
    u = np.asarray(up, F32)
    lim = F32(limit)
    if clamp_mode == CLAMP_BEFORE_SILU:
        g = np.minimum(g, lim)
        u = np.clip(u, -lim, lim)
    with np.errstate(over="ignore"):
        e = np.exp(-g.astype(np.float64)).astype(F32)
    sig = (F32(1.0) / (F32(1.0) + e)).astype(F32)
    silu = (g * sig).astype(F32)
    if clamp_mode == CLAMP_AFTER_SILU:
        silu = np.minimum(silu, lim)
        u = np.clip(u, -lim, lim)
    return (silu * u).astype(F32)


# ------------------------------------------------------------ expert FFN
def expert_rows(x_rows, w13_q, s13, w2_q, s2, act_fmt, weight_fmt,
                clamp_mode=CLAMP_NONE, limit=0.0, intermediates=False,
                numerics=NUMERICS_DIVIDE):
    """One expert applied to a set of BF16 token rows (fp32 holding BF16 values).

    Returns Y (fp32 holding BF16 values, [R, H]); with intermediates=True also
    a dict with A1 codes/scales, G1, A2 codes/scales.
    """
    inter = w13_q.shape[0] // 2
    a1_q, a1_s = quant_1x128(x_rows, act_fmt, numerics)
    g1 = bf16_round(block_gemm(a1_q, a1_s, w13_q, weight_scales_f32(s13, weight_fmt)))
    h = swiglu(g1[:, :inter], g1[:, inter:], clamp_mode, limit)
    if numerics == NUMERICS_RECIPROCAL:
        h = bf16_round(h)
    a2_q, a2_s = quant_1x128(h, act_fmt, numerics)
    y = bf16_round(block_gemm(a2_q, a2_s, w2_q, weight_scales_f32(s2, weight_fmt)))
    if intermediates:
        return y, {"a1_q": a1_q, "a1_s": a1_s, "g1": g1, "h": h, "a2_q": a2_q, "a2_s": a2_s}
    return y


# ---------------------------------------------------------------- reduce
def topk_reduce(y_pairs, weights, present, out_fp32=False):
    """out = RNbf16(sum_j RN32(w_j * y_j)) accumulated in fp32, j ascending,
    over the pairs that are present (valid ids); out_fp32 returns the fp32 sum unrounded."""
    topk = weights.shape[-1]
    acc = np.zeros(y_pairs.shape[:1] + y_pairs.shape[2:], F32)
    for j in range(topk):
        term = (np.asarray(weights[:, j], F32)[:, None] * y_pairs[:, j]).astype(F32)
        acc = np.where(present[:, j][:, None], (acc + term).astype(F32), acc)
    return acc if out_fp32 else bf16_round(acc)


# ------------------------------------------------------------------ layer
def moe_forward(x, topk_ids, topk_weights, w13_q, s13, w2_q, s2, *,
                act_fmt=SCALE_FP32, weight_fmt=SCALE_FP32,
                clamp_mode=CLAMP_NONE, limit=0.0, tokens=None,
                return_pairs=False, numerics=NUMERICS_DIVIDE, expert_offset=0, out_fp32=False):
    """Full layer forward for the selected tokens (default: all rows of x).

    x: fp32 [M, H] holding BF16 values; topk_ids int [M, k]; topk_weights fp32
    [M, k]; w13_q uint8 [E, 2I, H]; s13 [E, 2I/128, H/128] (fp32, or UE8M0
    bytes); w2_q uint8 [E, H, I]; s2 [E, H/128, I/128].
    Returns out (fp32 holding BF16 values) [len(tokens), H]; with
    return_pairs=True also the per-pair dict {(t, j): (Y row, intermediates)}.
    expert_offset: the weights hold experts [offset, offset + E) of a larger set (an
    expert-parallel slice); other ids are dropped.  out_fp32: return the fp32 sum (the
    partial output a rank contributes before the cross-rank sum) instead of BF16.
    """
    x = np.asarray(x, F32)
    num_experts = w13_q.shape[0]
    hidden = x.shape[1]
    if tokens is None:
        tokens = np.arange(x.shape[0])
    tokens = np.asarray(tokens, np.int64)
    topk = topk_ids.shape[1]
    ids = np.asarray(topk_ids, np.int64)[tokens] - expert_offset
    present = (ids >= 0) & (ids < num_experts)
    y_pairs = np.zeros((tokens.size, topk, hidden), F32)
    pairs = {}
    for e in np.unique(ids[present]):
        sel_t, sel_j = np.nonzero(ids == e)
        y, inter = expert_rows(x[tokens[sel_t]], w13_q[e], s13[e], w2_q[e], s2[e],
                               act_fmt, weight_fmt, clamp_mode, limit, intermediates=True,
                               numerics=numerics)
        y_pairs[sel_t, sel_j] = y
        if return_pairs:
            for i, (ti, j) in enumerate(zip(sel_t, sel_j)):
                pairs[(int(tokens[ti]), int(j))] = (
                    y[i], {k: v[i] for k, v in inter.items()})
    out = topk_reduce(y_pairs, np.asarray(topk_weights, F32)[tokens], present, out_fp32)
    if return_pairs:
        return out, pairs
    return out


# ------------------------------------------------------- batched experts
def batched_forward(x, counts, w13_q, s13, w2_q, s2, *, act_fmt=SCALE_FP32,
                    weight_fmt=SCALE_FP32, clamp_mode=CLAMP_NONE, limit=0.0,
                    numerics=NUMERICS_DIVIDE):
    """Batched-expert layout (vLLM per-layer activation scale page, Details:
    batched experts with masked per-expert counts).

    x: fp32 [E, max_m, H] holding BF16 values; counts int [E].  Expert e runs
    on its rows r < counts[e] (clamped to [0, max_m]) with no routing weight:
    out[e, r] = expert_rows(x[e, r]).  Returns (out fp32 [E, max_m, H] holding
    BF16 values, with NaN in the rows that are not live, and live mask [E, max_m]).
    """
    x = np.asarray(x, F32)
    num_experts, max_m, hidden = x.shape
    out = np.full((num_experts, max_m, hidden), np.nan, F32)
    live = np.zeros((num_experts, max_m), bool)
    for e in range(num_experts):
        c = int(min(max(int(counts[e]), 0), max_m))
        if c == 0:
            continue
        out[e, :c] = expert_rows(x[e, :c], w13_q[e], s13[e], w2_q[e], s2[e], act_fmt,
                                 weight_fmt, clamp_mode, limit, numerics=numerics)
        live[e, :c] = True
    return out, live
