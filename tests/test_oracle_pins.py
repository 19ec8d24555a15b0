"""Pins of the CPU oracle to things other than itself.

Each test ties one oracle function to a format definition, a closed form,
brute force on tiny inputs, exact rational arithmetic, a library routine or a
layer invariant, so that a plausible mistake (a dropped term, a wrong sign or
index, a transposed operand, a wrong rounding) fails at least one of them.
"""

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import formats as fm
import synth

F32 = np.float32


# ------------------------------------------------------------------ helpers
def exact_round_f32(q: Fraction) -> float:
    """Round a rational to the nearest fp32 (ties to even), by integer search.

    Written from the definition: find the binade, scale to a 24-bit integer
    significand, round the remainder half to even.  Normal range only.
    """
    if q == 0:
        return 0.0
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    # adjust so that 2^e <= a < 2^(e+1)
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    scaled = a / Fraction(2) ** (e - 23)          # in [2^23, 2^24)
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    return sign * float(m) * 2.0 ** (e - 23)


def brute_nearest_e4m3(v: float) -> int:
    """Nearest E4M3 code by exhaustive search over the finite codes; ties to even code;
    saturating at 448; sign of zero kept."""
    best = None
    for code in range(256):
        val = fm.E4M3_VALUES[code]
        if np.isnan(val):
            continue
        if (code & 0x80) != (0x80 if math.copysign(1.0, v) < 0 else 0):
            continue      # only codes of the same sign (so -0 is kept)
        d = abs(val - v)
        key = (d, code & 1)
        if best is None or key < best[0]:
            best = (key, code)
    return best[1]


# ----------------------------------------------------------- E4M3 format
def test_e4m3_table_definition_points():
    t = fm.E4M3_VALUES
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert t[0x08] == 2.0 ** -6            # smallest normal
    assert t[0x01] == 2.0 ** -9            # smallest subnormal
    assert t[0x07] == 7 / 8 * 2.0 ** -6    # largest subnormal
    assert t[0x38] == 1.0                  # exponent field 7 = bias
    assert t[0x00] == 0.0 and t[0x80] == 0.0 and math.copysign(1, t[0x80]) < 0
    assert np.isfinite(t).sum() == 254
    assert np.all(np.diff(t[:0x7F]) > 0)


def test_e4m3_table_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = fm.E4M3_VALUES
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], ours[fin])


def test_e4m3_encode_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = fm.E4M3_VALUES[codes].astype(F32)
    assert np.array_equal(fm.e4m3_encode(vals), codes)


def _midpoint_probes():
    pos = fm.E4M3_VALUES[:0x7F]
    mids = ((pos[:-1] + pos[1:]) / 2).astype(F32)
    probes = [mids, np.nextafter(mids, F32(np.inf)), np.nextafter(mids, F32(0))]
    probes.append(pos.astype(F32))
    v = np.concatenate(probes)
    return np.concatenate([v, -v]).astype(F32)


def test_e4m3_encode_brute_force():
    rng = np.random.default_rng(1)
    rand = np.concatenate([
        rng.uniform(-464, 464, 3000),
        rng.standard_normal(2000) * 2.0 ** rng.integers(-12, 9, 2000),
        [449.0, 463.9, 464.0, 465.0, 1e6, -1e-12, 1e-12, 0.0, -0.0],
    ]).astype(F32)
    v = np.concatenate([_midpoint_probes(), rand])
    ours = fm.e4m3_encode(v)
    ref = np.array([brute_nearest_e4m3(float(x)) for x in v], np.uint8)
    assert np.array_equal(ours, ref)


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(2)
    v = np.concatenate([_midpoint_probes(),
                        rng.uniform(-448, 448, 200000).astype(F32),
                        (rng.standard_normal(200000) * 0.01).astype(F32)])
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fm.e4m3_encode(v), ref)


def test_e4m3_saturation_and_nan():
    v = np.array([448.5, 464.0, 480.0, 1e30, -500.0, np.inf, -np.inf, np.nan], F32)
    assert list(fm.e4m3_encode(v)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE, 0x7F]


# ---------------------------------------------------------------- BF16
def test_bf16_round_matches_torch():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, 500000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(F32)
    v = v[np.isfinite(v)]
    ties = (((rng.integers(0, 2 ** 16, 1000).astype(np.uint32) << 16) | 0x8000)).view(F32)
    v = np.concatenate([v, ties[np.isfinite(ties)], np.array([0.0, -0.0, 3.3895314e38], F32)])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    ours = fm.bf16_round(v)
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------ pow2 / UE8M0
def test_pow2_ceil_against_frexp():
    rng = np.random.default_rng(4)
    s = (rng.uniform(0.5, 1.0, 20000) * 2.0 ** rng.integers(-30, 30, 20000)).astype(F32)
    s = np.concatenate([s, (2.0 ** np.arange(-30, 30)).astype(F32)])
    ours = fm.pow2_ceil(s)
    for a, b in zip(s[::50].tolist() + s[-60:].tolist(), ours[::50].tolist() + ours[-60:].tolist()):
        m, e = math.frexp(a)               # a = m * 2^e, m in [0.5, 1)
        want = 2.0 ** (e - 1) if m == 0.5 else 2.0 ** e
        assert b == want
    assert np.all(ours >= s) and np.all(ours < 2 * s)
    assert np.all((ours.view(np.uint32) & 0x7FFFFF) == 0)


def test_ue8m0_bytes():
    assert fm.ue8m0_to_f32(np.array([127, 128, 126, 110], np.uint8)).tolist() == [1.0, 2.0, 0.5, 2.0 ** -17]
    assert fm.f32_exponent_field(np.array([1.0, 0.25, 2.0 ** -17], F32)).tolist() == [127, 125, 110]


# --------------------------------------------------------------- fp32 FMA
def test_fma_f32_exact_rational():
    rng = np.random.default_rng(5)
    a = (rng.standard_normal(3000) * 2.0 ** rng.integers(-20, 20, 3000)).astype(F32)
    b = (rng.standard_normal(3000) * 2.0 ** rng.integers(-20, 20, 3000)).astype(F32)
    c = (rng.standard_normal(3000) * 2.0 ** rng.integers(-20, 20, 3000)).astype(F32)
    got = fm.fma_f32(a, b, c)
    for x, y, z, g in zip(a.tolist(), b.tolist(), c.tolist(), got.tolist()):
        want = exact_round_f32(Fraction(x) * Fraction(y) + Fraction(z))
        assert g == want


def test_fma_f32_double_rounding_case():
    # exact value sits just below the tie between 1+2^-23 (odd) and 1+2^-22 (even);
    # rounding through float64 first would land on the tie and pick the even side
    a = F32(1 + 2.0 ** -23)
    b = F32(2.0 ** -24 * (1 - 2.0 ** -23))
    c = F32(1 + 2.0 ** -23)
    want = exact_round_f32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))
    assert want == 1 + 2.0 ** -23
    assert fm.fma_f32(a, b, c) == F32(want)
    naive = F32(float(a) * float(b) + float(c))
    assert naive != F32(want)          # the emulation matters here
    # exact ties resolve to even
    assert fm.fma_f32(F32(2.0 ** -12), F32(2.0 ** -12), F32(1.0)) == F32(1.0)


# ------------------------------------------------------------------ scales
def test_group_scale_closed_form():
    amax = np.array([0.0, 448.0, 896.0, 1.0, 1e-9, 3.0], F32)
    s = oracle.group_scale(amax, oracle.SCALE_FP32)
    floor = F32(1.0) / F32(229376.0)
    assert s[0] == floor and s[4] == floor
    assert s[1] == 1.0 and s[2] == 2.0
    assert s[3] == F32(1.0) / F32(448.0)
    assert s[5] == F32(3.0) / F32(448.0)
    p = oracle.group_scale(amax, oracle.SCALE_FP32_POW2)
    assert p[1] == 1.0 and p[2] == 2.0
    assert p[3] == 2.0 ** -8            # 1/448 = 2^-8.8 -> 2^-8
    assert p[0] == 2.0 ** -17           # floor 2^-17.8 -> 2^-17
    assert np.all(amax / p <= 448.0)


def test_quant_1x128_properties():
    rng = np.random.default_rng(6)
    v = (rng.standard_normal((7, 512)) * 3).astype(F32)
    v[2, 128:256] = 0.0
    for fmt in (oracle.SCALE_FP32, oracle.SCALE_FP32_POW2, oracle.SCALE_UE8M0):
        q, s = oracle.quant_1x128(v, fmt)
        assert q.dtype == np.uint8 and s.shape == (7, 4)
        assert np.all(q[2, 128:256] == 0) and s[2, 1] == oracle.group_scale(F32(0), fmt)
        # each group: codes are the nearest E4M3 of v/s, the largest |code| <= 448
        deq = oracle.e4m3_decode(q).reshape(7, 4, 128) * s[..., None]
        g = v.reshape(7, 4, 128)
        err = np.abs(deq - g)
        assert np.all(err <= s[..., None] * np.maximum(np.abs(g / s[..., None]) * 2.0 ** -4, 2.0 ** -10) + 1e-30)
        if fmt == oracle.SCALE_FP32:
            # the group maximum maps to exactly 448 when the floor is not hit
            top = np.abs(oracle.e4m3_decode(q)).reshape(7, 4, 128).max(-1)
            assert np.all(top[s > oracle.SCALE_FLOOR] == 448.0)


# ---------------------------------------------- quantizer, element by element
def _expected_scale(amax: float, fmt) -> float:
    """The group scale from its definition, in exact rationals: max(RN32(amax/448), RN32(1/229376)),
    then, for the power-of-two formats, the smallest power of two that is >= it."""
    s = max(exact_round_f32(Fraction(amax) / 448), exact_round_f32(Fraction(1, 229376)))
    if fmt in (oracle.SCALE_FP32_POW2, oracle.SCALE_UE8M0):
        e = 0
        while Fraction(2) ** e < Fraction(s):
            e += 1
        while Fraction(2) ** (e - 1) >= Fraction(s):
            e -= 1
        s = 2.0 ** e
    return s


def _nearest_code(q: Fraction, sign_of: float) -> int:
    """E4M3 code of RN32(q): the quotient or product rounded once to fp32, then to the nearest code."""
    r = exact_round_f32(q)
    if r == 0.0:
        r = math.copysign(0.0, sign_of)
    return brute_nearest_e4m3(r)


def _quant_pin_inputs():
    """BF16 groups of 128 chosen to expose the quantizer's arithmetic.

    Midpoint groups: amax = 448 * c * 2^j makes the scale exactly c * 2^j, and every other element
    is c * 2^j times an E4M3 midpoint (all BF16 values), so x / scale lands exactly on a tie, which
    goes to the even code; with c = 7 the product x * RN32(1/scale) is one fp32 ulp off the tie for
    about a quarter of them and picks the other code (the TensorRT-LLM page's reason for correctly
    rounded division: BF16 inputs that sit on E4M3 midpoints).  Then random BF16 groups, a group
    with 1% outliers x10, an all-zero group and a tiny group (both at the scale floor)."""
    pos = fm.E4M3_VALUES[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2.0                    # 126 positive midpoints
    groups = []
    for c, j in ((7, -8), (7, 3), (3, -5), (5, 0)):
        unit = c * 2.0 ** j
        for sign in (1.0, -1.0):
            g = np.zeros(128, np.float64)
            g[0] = 448.0 * unit
            g[1:127] = sign * mids * unit
            g[127] = -sign * mids[60] * unit
            groups.append(g)
    rng = np.random.default_rng(31)
    for _ in range(8):
        groups.append(rng.standard_normal(128) * 3.0)
    out = rng.standard_normal(128)
    out[rng.uniform(size=128) < 0.05] *= 10.0
    groups.append(out)
    groups.append(np.zeros(128))
    groups.append(rng.standard_normal(128) * 1e-6)
    v = np.stack(groups).astype(F32)
    bv = fm.bf16_round(v)
    assert np.array_equal(bv[:8], v[:8])                # the designed groups are BF16 exactly
    return bv


def _quant_mismatches(quant, v, fmt, numerics=oracle.NUMERICS_DIVIDE):
    """Elements whose code or group scale differs from the definition evaluated in exact rationals."""
    q, s = quant(v, fmt, numerics)
    bad = 0
    for gi in range(v.shape[0]):
        row = v[gi].tolist()
        amax = max(abs(x) for x in row)
        if numerics == oracle.NUMERICS_RECIPROCAL and fmt == oracle.SCALE_FP32:
            inv = 448.0 * 512.0 if amax == 0 else min(exact_round_f32(Fraction(448) / Fraction(amax)),
                                                      448.0 * 512.0)
            want_s = exact_round_f32(1 / Fraction(inv))
            codes = [_nearest_code(Fraction(x) * Fraction(inv), x) for x in row]
        else:
            want_s = _expected_scale(amax, fmt)
            codes = [_nearest_code(Fraction(x) / Fraction(want_s), x) for x in row]
        bad += int(float(s[gi, 0]) != want_s) * 128
        bad += sum(int(a != b) for a, b in zip(q[gi].tolist(), codes))
    return bad


@pytest.mark.parametrize("fmt", [oracle.SCALE_FP32, oracle.SCALE_FP32_POW2, oracle.SCALE_UE8M0])
def test_quant_1x128_element_by_element(fmt):
    """Every code is the nearest E4M3 (ties to even) of x / scale correctly rounded to fp32, and
    every scale is max(RN32(amax/448), RN32(1/229376)) (power of two rounded up for POW2/UE8M0),
    both evaluated in exact rationals (vLLM per-layer scale page, Details: x/scale; TensorRT-LLM
    page, rounding-fix commit: correctly rounded division)."""
    v = _quant_pin_inputs()
    assert _quant_mismatches(oracle.quant_1x128, v, fmt) == 0
    if fmt == oracle.SCALE_UE8M0:
        _, s = oracle.quant_1x128(v, fmt)
        assert np.array_equal(oracle.scale_bytes(s),
                              np.array([[127 + int(math.log2(float(x)))] for x in s[:, 0]], np.uint8))


def test_quant_1x128_reciprocal_element_by_element():
    """The TensorRT-LLM numerics: codes are the nearest E4M3 of x * RN32(448/amax) rounded once to
    fp32, the stored scale is RN32(1/inv), with inv capped at 448*512 (the scale floor)."""
    v = _quant_pin_inputs()
    assert _quant_mismatches(oracle.quant_1x128, v, oracle.SCALE_FP32, oracle.NUMERICS_RECIPROCAL) == 0


def test_quant_pin_catches_reciprocal_multiply():
    """A quantizer that multiplies by RN32(1/scale) instead of dividing by the scale (the mistake the
    TensorRT-LLM page's rounding fix removes) fails the element-by-element pin."""
    def planted(v, fmt, numerics=0):
        g = np.asarray(v, F32).reshape(v.shape[0], -1, 128)
        s = oracle.group_scale(np.abs(g).max(-1), fmt)
        inv = (F32(1.0) / s).astype(F32)
        return fm.e4m3_encode((g * inv[..., None]).astype(F32)).reshape(v.shape), s
    v = _quant_pin_inputs()
    assert _quant_mismatches(planted, v, oracle.SCALE_FP32) > 0


def test_quant_scaling_by_power_of_two():
    rng = np.random.default_rng(7)
    v = rng.standard_normal((3, 256)).astype(F32)
    for fmt in (oracle.SCALE_FP32, oracle.SCALE_FP32_POW2):
        q1, s1 = oracle.quant_1x128(v, fmt)
        q2, s2 = oracle.quant_1x128(v * F32(8.0), fmt)
        assert np.array_equal(q1, q2) and np.array_equal(s2, s1 * 8)


# --------------------------------------------------------------- alignment
def test_align_brute_force():
    rng = np.random.default_rng(8)
    for trial in range(60):
        E = int(rng.integers(1, 12))
        k = int(rng.integers(1, 5))
        M = int(rng.integers(0, 40))
        n = int(rng.integers(0, M + 1))
        A = int(rng.choice([4, 8, 128]))
        ids = rng.integers(-2, E + 2, (M, k)).astype(np.int32)
        r = oracle.align(ids, n, E, A)
        pairs = [(int(ids.reshape(-1)[p]), p) for p in range(n * k)
                 if 0 <= ids.reshape(-1)[p] < E]
        order = sorted(pairs)                         # by expert, then pair index
        # rebuild expected layout by walking experts
        seg, row = [], 0
        exp_rows = {}
        for e in range(E):
            mine = [p for (ee, p) in order if ee == e]
            seg.append(row)
            for i, p in enumerate(mine):
                exp_rows[p] = row + i
            row += -(-len(mine) // A) * A
        seg.append(row)
        assert r["seg_start"].tolist() == seg
        for p in range(n * k):
            assert r["pair_row"][p] == exp_rows.get(p, -1)
        for p, rr in exp_rows.items():
            assert r["sorted_pair"][rr] == p
        assert r["num_tiles"] == row // A
        for i in range(r["num_tiles"]):
            e = r["tile_expert"][i]
            assert seg[e] <= i * A < seg[e + 1]
        assert np.all(r["seg_start"] % A == 0)
        assert (r["live_end"] - r["seg_start"][:-1]).sum() == len(pairs)
        # 32-row chunks cover every live row exactly once and never cross a segment
        covered = []
        for c0 in r["chunk_row0"]:
            e = [ee for ee in range(E) if seg[ee] <= c0 < r["live_end"][ee]]
            assert len(e) == 1 and (c0 - seg[e[0]]) % 32 == 0
            covered += list(range(c0, min(c0 + 32, r["live_end"][e[0]])))
        assert sorted(covered) == sorted(exp_rows.values())
        assert r["num_chunks"] == len(r["chunk_row0"])


def test_align_edge_cases():
    ids = np.array([[-1, 5], [7, -3]], np.int32)
    r = oracle.align(ids, 2, 4)
    assert r["num_tiles"] == 0 and r["pair_row"].tolist() == [-1, -1, -1, -1]
    r = oracle.align(np.zeros((0, 8), np.int32), 0, 72)
    assert r["num_tiles"] == 0 and r["seg_start"].sum() == 0
    # 128-pair threshold (16x8) and above (24x8), 72 experts (not a power of two)
    rng = np.random.default_rng(9)
    for M in (16, 24):
        ids = np.stack([rng.permutation(72)[:8] for _ in range(M)]).astype(np.int32)
        r = oracle.align(ids, M, 72)
        assert (r["live_end"] - r["seg_start"][:-1]).sum() == M * 8
        assert r["num_tiles"] == np.count_nonzero(np.bincount(ids.reshape(-1), minlength=72))


# ------------------------------------------------------------- block GEMM
def test_block_gemm_exact_integer_dot():
    rng = np.random.default_rng(10)
    aq = rng.integers(0, 256, (3, 128)).astype(np.uint8)
    wq = rng.integers(0, 256, (128, 128)).astype(np.uint8)
    aq[aq & 0x7F == 0x7F] = 0
    wq[wq & 0x7F == 0x7F] = 0
    acc = oracle.block_gemm(aq, np.ones((3, 1), F32), wq, np.ones((1, 1), F32))
    # brute force: each E4M3 value times 2^9 is an integer
    ia = np.rint(fm.E4M3_VALUES[aq] * 512).astype(object)
    iw = np.rint(fm.E4M3_VALUES[wq] * 512).astype(object)
    for r in range(3):
        for c in range(0, 128, 7):
            d = sum(int(x) * int(y) for x, y in zip(ia[r], iw[c]))
            assert acc[r, c] == exact_round_f32(Fraction(d, 2 ** 18))


def _int_codes(codes):
    """E4M3 codes as integers: value * 2^9 (every E4M3 value is an integer multiple of 2^-9)."""
    return np.rint(fm.E4M3_VALUES[np.asarray(codes, np.uint8)] * 512).astype(np.int64)


def _block_gemm_steps(aq, a_s, wq, w_s, accumulate="fused"):
    """The per-128-K promotion evaluated in exact rationals: d = exact block dot, p = RN32(d),
    sab = RN32(sa*sw), acc = RN32(acc + p*sab) with one rounding (a fused multiply-add; TensorRT-LLM
    page, human review: the scale product is formed first).  `accumulate` selects a planted
    variant: "separate" rounds p*sab before the add, "unrounded_sab" skips the scale-product
    rounding."""
    ia, iw = _int_codes(aq), _int_codes(wq)
    R, K = aq.shape
    N = wq.shape[0]
    out = np.zeros((R, N), F32)
    for r in range(R):
        for c in range(N):
            acc = Fraction(0)
            for kb in range(K // 128):
                sl = slice(kb * 128, (kb + 1) * 128)
                d = Fraction(int(np.dot(ia[r, sl], iw[c, sl])), 2 ** 18)
                p = Fraction(exact_round_f32(d))
                sa, sw = Fraction(float(a_s[r, kb])), Fraction(float(w_s[c // 128, kb]))
                if accumulate == "unrounded_sab":
                    acc = Fraction(exact_round_f32(acc + p * sa * sw))
                    continue
                sab = Fraction(exact_round_f32(sa * sw))
                if accumulate == "separate":
                    acc = Fraction(exact_round_f32(acc + Fraction(exact_round_f32(p * sab))))
                else:
                    acc = Fraction(exact_round_f32(acc + p * sab))
            out[r, c] = float(acc)
    return out


def test_block_gemm_promotion_step_by_step():
    """Several K blocks with scales that are not powers of two: every output equals the stated
    promotion sequence in exact rationals, and the two plausible misreadings (rounding p*sab before
    the add; not rounding the scale product) each change some outputs."""
    rng = np.random.default_rng(17)
    R, N, K = 3, 256, 384
    aq = fm.e4m3_encode(rng.standard_normal((R, K)).astype(F32) * 60)
    wq = fm.e4m3_encode(rng.standard_normal((N, K)).astype(F32) * 60)
    a_s = (rng.uniform(0.5, 1.0, (R, K // 128)) * 2.0 ** -9).astype(F32)
    w_s = (rng.uniform(0.5, 1.0, (N // 128, K // 128)) * 2.0 ** -7).astype(F32)
    got = oracle.block_gemm(aq, a_s, wq, w_s)
    want = _block_gemm_steps(aq, a_s, wq, w_s)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    for variant in ("separate", "unrounded_sab"):
        bad = _block_gemm_steps(aq, a_s, wq, w_s, variant)
        assert not np.array_equal(bad.view(np.uint32), want.view(np.uint32)), variant


def test_block_gemm_vs_dequantized_matmul():
    rng = np.random.default_rng(11)
    R, N, K = 5, 256, 512
    aq = fm.e4m3_encode(rng.standard_normal((R, K)).astype(F32) * 100)
    wq = fm.e4m3_encode(rng.standard_normal((N, K)).astype(F32) * 100)
    a_s = rng.uniform(1e-3, 1e-2, (R, K // 128)).astype(F32)
    w_s = rng.uniform(1e-3, 1e-2, (N // 128, K // 128)).astype(F32)
    acc = oracle.block_gemm(aq, a_s, wq, w_s)
    a_deq = fm.e4m3_decode(aq) * np.repeat(a_s.astype(np.float64), 128, axis=1)
    w_deq = fm.e4m3_decode(wq) * np.repeat(np.repeat(w_s.astype(np.float64), 128, axis=0), 128, axis=1)
    exact = a_deq @ w_deq.T
    absterms = np.abs(fm.e4m3_decode(aq) * np.repeat(a_s.astype(np.float64), 128, 1)) @ \
        np.abs(w_deq).T
    bound = (K // 128 + 2) * 2.0 ** -23 * absterms
    assert np.all(np.abs(acc - exact) <= bound)
    # a transposed weight operand or a misplaced scale block breaks the match
    w_s_t = np.ascontiguousarray(w_s[::-1])
    bad = oracle.block_gemm(aq, a_s, wq, w_s_t)
    assert np.any(np.abs(bad - exact) > bound)


# ------------------------------------------------------------------ SwiGLU
def test_swiglu_against_high_precision():
    import mpmath
    mpmath.mp.prec = 100
    rng = np.random.default_rng(12)
    g = fm.bf16_round((rng.standard_normal(400) * 4).astype(F32))
    u = fm.bf16_round((rng.standard_normal(400) * 4).astype(F32))
    h = oracle.swiglu(g, u)
    for gi, ui, hi in zip(g.tolist(), u.tolist(), h.tolist()):
        exact = mpmath.mpf(gi) / (1 + mpmath.exp(-mpmath.mpf(gi))) * ui
        assert abs(hi - float(exact)) <= 4 * 2.0 ** -24 * abs(float(exact)) + 1e-45


def _mp_fraction(x) -> Fraction:
    """An mpmath number as an exact rational (mantissa * 2^exponent)."""
    import mpmath
    man, exp = mpmath.mpf(x).man_exp
    return Fraction(int(man)) * Fraction(2) ** int(exp)


def _swiglu_steps(g: float, u: float, clamp_mode=0, limit=0.0) -> float:
    """SiLU(g)*up, each stated step rounded once to fp32, in exact rationals: e = RN32(exp(-g)) (exp
    to 120 bits, then rounded), d = RN32(1 + e), sig = RN32(1/d) (IEEE division), silu = RN32(g*sig),
    h = RN32(silu*u); the clamps are exact (TensorRT-LLM page, human review: 1/(1+expf(-x)) with
    IEEE division)."""
    import mpmath
    mpmath.mp.prec = 120
    if clamp_mode == oracle.CLAMP_BEFORE_SILU:
        g = min(g, limit)
        u = min(max(u, -limit), limit)
    e = exact_round_f32(_mp_fraction(mpmath.exp(-mpmath.mpf(g))))
    d = exact_round_f32(1 + Fraction(e))
    sig = exact_round_f32(1 / Fraction(d))
    silu = exact_round_f32(Fraction(g) * Fraction(sig))
    if clamp_mode == oracle.CLAMP_AFTER_SILU:
        silu = min(silu, limit)
        u = min(max(u, -limit), limit)
    return exact_round_f32(Fraction(silu) * Fraction(u))


def _swiglu_pin_inputs():
    rng = np.random.default_rng(41)
    g = fm.bf16_round((rng.standard_normal(1500) * 4).astype(F32))
    u = fm.bf16_round((rng.standard_normal(1500) * 4).astype(F32))
    return g, u


def _swiglu_mismatches(fn, g, u, clamp_mode=0, limit=0.0):
    h = fn(g, u, clamp_mode, limit)
    return sum(int(float(hi) != _swiglu_steps(gi, ui, clamp_mode, limit))
               for gi, ui, hi in zip(g.tolist(), u.tolist(), h.tolist()))


@pytest.mark.parametrize("clamp_mode,limit", [(0, 0.0), (1, 1.5), (2, 1.5)])
def test_swiglu_step_by_step(clamp_mode, limit):
    """Each fp32 step of the SwiGLU equals its exact-rational evaluation, bit for bit."""
    g, u = _swiglu_pin_inputs()
    assert _swiglu_mismatches(oracle.swiglu, g, u, clamp_mode, limit) == 0


def test_swiglu_pin_catches_a_once_rounded_sigmoid():
    """A sigmoid formed in float64 and rounded once (instead of the stated fp32 steps) fails the
    step-by-step pin."""
    def planted(gate, up, clamp_mode=0, limit=0.0):
        g = np.asarray(gate, F32)
        sig = (1.0 / (1.0 + np.exp(-g.astype(np.float64)))).astype(F32)
        return ((g * sig).astype(F32) * np.asarray(up, F32)).astype(F32)
    g, u = _swiglu_pin_inputs()
    assert _swiglu_mismatches(planted, g, u) > 0


def test_swiglu_clamp_semantics():
    g = np.array([10.0, -10.0, 3.0, 9.0], F32)
    u = np.array([-9.0, 9.0, 2.0, 1.0], F32)
    L = 7.0
    sil = lambda z: z / (1 + math.exp(-z))
    before = oracle.swiglu(g, u, oracle.CLAMP_BEFORE_SILU, L)
    want_b = [sil(7.0) * -7.0, sil(-10.0) * 7.0, sil(3.0) * 2.0, sil(7.0) * 1.0]
    after = oracle.swiglu(g, u, oracle.CLAMP_AFTER_SILU, L)
    want_a = [min(sil(10.0), 7.0) * -7.0, sil(-10.0) * 7.0, sil(3.0) * 2.0, min(sil(9.0), 7.0) * 1.0]
    none = oracle.swiglu(g, u, oracle.CLAMP_NONE, L)
    want_n = [sil(10.0) * -9.0, sil(-10.0) * 9.0, sil(3.0) * 2.0, sil(9.0)]
    np.testing.assert_allclose(before, want_b, rtol=1e-6)
    np.testing.assert_allclose(after, want_a, rtol=1e-6)
    np.testing.assert_allclose(none, want_n, rtol=1e-6)


# ---------------------------------------------------------------- reduce
def test_topk_reduce_hand_example():
    y = np.array([[[1.0, 2.0], [4.0, -8.0], [100.0, 100.0]]], F32)
    w = np.array([[0.5, 0.25, 0.125]], F32)
    present = np.array([[True, True, False]])
    out = oracle.topk_reduce(y, w, present)
    assert out.tolist() == [[1.5, -1.0]]
    # fp32 accumulation then one BF16 rounding: 1 + 2^-9 is not a BF16 value
    y = np.array([[[1.0], [2.0 ** -9]]], F32)
    out = oracle.topk_reduce(y, np.ones((1, 2), F32), np.ones((1, 2), bool))
    assert out[0, 0] == 1.0


def _reduce_steps(y, w, present, out_fp32=False):
    """out = RNbf16(acc), acc = 0; for j ascending over present pairs acc = RN32(acc + RN32(w*y)),
    evaluated with exact rationals (TensorRT-LLM page, rounding-fix commit: the finalize step scales
    the BF16 expert outputs in fp32)."""
    T, K, H = y.shape
    out = np.zeros((T, H), F32)
    for t in range(T):
        for h in range(H):
            acc = 0.0
            for j in range(K):
                if present[t, j]:
                    term = exact_round_f32(Fraction(float(w[t, j])) * Fraction(float(y[t, j, h])))
                    acc = exact_round_f32(Fraction(acc) + Fraction(term))
            out[t, h] = acc
    return out if out_fp32 else fm.bf16_round(out)


def _reduce_pin_case():
    """Terms chosen so that the order and the rounding of the fp32 accumulation decide the result.

    Column 0: 1+2^-8 (a BF16 tie), then 2^-24 twice.  In ascending order each 2^-24 is half an fp32
    ulp of the running sum and ties back to it, so the sum stays on the BF16 tie and rounds to 1.0;
    summed in reverse, or in float64 and rounded once, the two small terms survive as 2^-23 and the
    BF16 result is 1 + 2^-7.  Column 1: a product w*y that is not an fp32 number (its per-term
    rounding matters), on token 1.  A dropped pair between live ones carries a large value that must not count.
    Further columns: random BF16 outputs and fp32 weights."""
    T, K, H = 3, 4, 6
    rng = np.random.default_rng(43)
    y = fm.bf16_round(rng.standard_normal((T, K, H)).astype(F32))
    w = rng.uniform(0.05, 1.0, (T, K)).astype(F32)
    present = np.ones((T, K), bool)
    y[0, :, 0] = [1.0, 2.0 ** -24, 1e4, 2.0 ** -24]
    w[0] = [F32(1 + 2.0 ** -8), 1.0, 1.0, 1.0]
    present[0, 2] = False
    y[1, :, 1] = [1.0, fm.bf16_round(np.array([1 + 2.0 ** -7], F32))[0], 3.0, 0.0]
    w[1, 1] = F32(1 + 2.0 ** -20)
    present[2, 0] = False
    return y, w, present


def test_topk_reduce_step_by_step():
    y, w, present = _reduce_pin_case()
    for out_fp32 in (False, True):
        got = oracle.topk_reduce(y, w, present, out_fp32)
        want = _reduce_steps(y, w, present, out_fp32)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), out_fp32
    assert oracle.topk_reduce(y, w, present)[0, 0] == 1.0


def test_topk_reduce_pin_catches_order_and_fused_accumulation():
    """Summing j descending, or accumulating in float64 and rounding once, fails the pin."""
    y, w, present = _reduce_pin_case()
    want = _reduce_steps(y, w, present)

    def descending(y, w, present):
        acc = np.zeros((y.shape[0], y.shape[2]), F32)
        for j in reversed(range(w.shape[1])):
            term = (w[:, j][:, None] * y[:, j]).astype(F32)
            acc = np.where(present[:, j][:, None], (acc + term).astype(F32), acc)
        return fm.bf16_round(acc)

    def fused64(y, w, present):
        acc = np.zeros((y.shape[0], y.shape[2]), np.float64)
        for j in range(w.shape[1]):
            acc += np.where(present[:, j][:, None],
                            w[:, j][:, None].astype(np.float64) * y[:, j].astype(np.float64), 0.0)
        return fm.bf16_round(acc.astype(F32))

    for planted in (descending, fused64):
        assert not np.array_equal(planted(y, w, present), want), planted.__name__


def test_expert_rows_wiring_exact():
    """One expert end to end (H = 256, I = 256, two rows), every step from its stated definition in
    exact rationals: 1x128 quantization of x, the FC1 promotion, BF16 rounding of the gate/up sums,
    the SwiGLU steps, requantization of h, the FC2 promotion and the final BF16 rounding.  Pins which
    intermediate feeds which step (a dropped BF16 rounding of the FC1 sums, or gate and up swapped,
    fails it)."""
    rng = np.random.default_rng(23)
    H = I = 256
    x = fm.bf16_round(rng.standard_normal((2, H)).astype(F32))
    w13 = fm.e4m3_encode(rng.standard_normal((2 * I, H)).astype(F32) * 100)
    w2 = fm.e4m3_encode(rng.standard_normal((H, I)).astype(F32) * 100)
    s13 = (rng.uniform(0.5, 1.0, (2 * I // 128, H // 128)) * 2.0 ** -8).astype(F32)
    s2 = (rng.uniform(0.5, 1.0, (H // 128, I // 128)) * 2.0 ** -8).astype(F32)

    def quant_rows(v):
        q = np.zeros(v.shape, np.uint8)
        sc = np.zeros((v.shape[0], v.shape[1] // 128), F32)
        for r in range(v.shape[0]):
            for g in range(v.shape[1] // 128):
                grp = v[r, g * 128:(g + 1) * 128].tolist()
                s = _expected_scale(max(abs(t) for t in grp), oracle.SCALE_FP32)
                sc[r, g] = s
                q[r, g * 128:(g + 1) * 128] = [_nearest_code(Fraction(t) / Fraction(s), t) for t in grp]
        return q, sc

    def run(round_g1=True, swap=False):
        a1q, a1s = quant_rows(x)
        g1 = _block_gemm_steps(a1q, a1s, w13, s13)
        if round_g1:
            g1 = fm.bf16_round(g1)
        gate, up = (g1[:, I:], g1[:, :I]) if swap else (g1[:, :I], g1[:, I:])
        h = np.array([[_swiglu_steps(float(gv), float(uv)) for gv, uv in zip(gr, ur)]
                      for gr, ur in zip(gate, up)], F32)
        a2q, a2s = quant_rows(h)
        return fm.bf16_round(_block_gemm_steps(a2q, a2s, w2, s2))

    got = oracle.expert_rows(x, w13, s13, w2, s2, oracle.SCALE_FP32, oracle.SCALE_FP32)
    want = run()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert not np.array_equal(run(round_g1=False).view(np.uint32), want.view(np.uint32))
    assert not np.array_equal(run(swap=True).view(np.uint32), want.view(np.uint32))


# ----------------------------------------------------------- layer pins
@pytest.fixture(scope="module")
def small_case():
    shape = synth.small_shape(E=6, H=256, I=256, topk=2)
    return synth.make_case("small", 12, shape=shape)


def _fwd(case, **kw):
    w = case.weights
    sh = case.shape
    args = dict(act_fmt=sh.act_fmt, weight_fmt=sh.weight_fmt,
                clamp_mode=sh.clamp_mode, limit=sh.limit)
    args.update(kw)
    return oracle.moe_forward(case.x, case.topk_ids, case.topk_weights,
                              w.w13, w.s13, w.w2, w.s2, **args)


def dense_reference(case, clamp_mode=0, limit=0.0):
    """Unquantized-activation layer in float64 with the dequantized weights."""
    w = case.weights
    out = np.zeros(case.x.shape, np.float64)
    I = w.w13.shape[1] // 2
    for t in range(case.x.shape[0]):
        for j in range(case.topk_ids.shape[1]):
            e = case.topk_ids[t, j]
            if not (0 <= e < w.w13.shape[0]):
                continue
            w13 = fm.e4m3_decode(w.w13[e]) * np.kron(oracle.weight_scales_f32(w.s13[e], case.shape.weight_fmt), np.ones((128, 128)))
            w2 = fm.e4m3_decode(w.w2[e]) * np.kron(oracle.weight_scales_f32(w.s2[e], case.shape.weight_fmt), np.ones((128, 128)))
            g1 = w13 @ case.x[t].astype(np.float64)
            g, u = g1[:I], g1[I:]
            if clamp_mode == 1:
                g = np.minimum(g, limit); u = np.clip(u, -limit, limit)
            h = g / (1 + np.exp(-g))
            if clamp_mode == 2:
                h = np.minimum(h, limit); u = np.clip(u, -limit, limit)
            out[t] += case.topk_weights[t, j] * (w2 @ (h * u))
    return out


def test_layer_close_to_dense_reference(small_case):
    out = _fwd(small_case)
    ref = dense_reference(small_case)
    rel = np.linalg.norm(out - ref) / np.linalg.norm(ref)
    # FP8 activation rounding (3 mantissa bits) dominates: a few percent
    assert 0.002 < rel < 0.1, rel


def test_layer_invariants(small_case):
    c = small_case
    base = _fwd(c)
    # doubling the routing weights doubles the output exactly
    w2x = synth.LayerCase(c.shape, c.M_cap, c.n, c.x_bits, c.x, c.topk_ids,
                          c.topk_weights * 2, c.weights)
    assert np.array_equal(_fwd(w2x), base * 2)
    # all ids dropped -> zero output
    dropped = synth.LayerCase(c.shape, c.M_cap, c.n, c.x_bits, c.x,
                              np.full_like(c.topk_ids, -1), c.topk_weights, c.weights)
    assert np.all(_fwd(dropped) == 0)
    # experts that no pair routes to contribute nothing: change their weights
    used = set(c.topk_ids.reshape(-1).tolist())
    unused = [e for e in range(c.shape.E) if e not in used]
    if unused:
        w = c.weights
        w13 = w.w13.copy(); w13[unused] = 0x38
        alt = synth.LayerCase(c.shape, c.M_cap, c.n, c.x_bits, c.x, c.topk_ids, c.topk_weights,
                              synth.Weights(w13, w.s13, w.w2, w.s2))
        assert np.array_equal(_fwd(alt), base)
    # token order does not matter
    perm = np.random.default_rng(0).permutation(c.M_cap)
    pc = synth.LayerCase(c.shape, c.M_cap, c.n, c.x_bits[perm], c.x[perm], c.topk_ids[perm],
                         c.topk_weights[perm], c.weights)
    assert np.array_equal(_fwd(pc), base[perm])


def test_one_live_row_single_expert(small_case):
    """topk = 1 with weight 1: the output is the BF16 expert output itself,
    and equals the dequantized-weight dense FFN to within FP8 activation error."""
    c = small_case
    ids = c.topk_ids[:1, :1].copy()
    one = synth.LayerCase(c.shape, 1, 1, c.x_bits[:1], c.x[:1], ids,
                          np.ones((1, 1), F32), c.weights)
    out = _fwd(one)
    ref = dense_reference(one)
    assert np.linalg.norm(out - ref) / np.linalg.norm(ref) < 0.1
    w = c.weights
    e = ids[0, 0]
    y = oracle.expert_rows(c.x[:1], w.w13[e], w.s13[e], w.w2[e], w.s2[e], 0, 0)
    assert np.array_equal(out, y)


def test_clamp_modes_against_dense(small_case):
    c = small_case
    for mode in (1, 2):
        out = _fwd(c, clamp_mode=mode, limit=0.05)
        ref = dense_reference(c, mode, 0.05)
        assert np.linalg.norm(out - ref) / np.linalg.norm(ref) < 0.1
    # a limit that clamps does change the result
    assert not np.array_equal(_fwd(c, clamp_mode=1, limit=0.05), _fwd(c))


def test_pow2_scales_no_better_than_fp32(small_case):
    """Power-of-two activation scales add rounding error (vLLM per-layer scale
    page, Claims): on average the layer error is not lower than with fp32 scales."""
    c = small_case
    ref = dense_reference(c)
    e32 = np.linalg.norm(_fwd(c, act_fmt=0) - ref)
    ep2 = np.linalg.norm(_fwd(c, act_fmt=1) - ref)
    assert ep2 >= 0.9 * e32


def test_planted_mistakes_are_caught(monkeypatch, small_case):
    """A mistake planted in the oracle (on the CPU) must fail a pin."""
    from oracle import moe_ref
    c = small_case
    ref = dense_reference(c)
    good = np.linalg.norm(_fwd(c) - ref) / np.linalg.norm(ref)
    # swapped gate/up halves
    orig = moe_ref.swiglu
    monkeypatch.setattr(moe_ref, "swiglu", lambda g, u, m=0, l=0.0: orig(u, g, m, l))
    bad = np.linalg.norm(_fwd(c) - ref) / np.linalg.norm(ref)
    monkeypatch.setattr(moe_ref, "swiglu", orig)
    assert good < 0.1 <= bad          # the dense-reference pin's bound
    # weight scale block indexed transposed
    orig_ws = moe_ref.weight_scales_f32
    monkeypatch.setattr(moe_ref, "weight_scales_f32",
                        lambda s, f: np.ascontiguousarray(np.asarray(orig_ws(s, f))[::-1, ::-1]))
    bad = np.linalg.norm(_fwd(c) - ref) / np.linalg.norm(ref)
    monkeypatch.setattr(moe_ref, "weight_scales_f32", orig_ws)
    assert good < 0.1 <= bad


# ------------------------------------------- reciprocal (TensorRT-LLM) numerics
def test_reciprocal_quant_closed_form():
    R = oracle.NUMERICS_RECIPROCAL
    amax = np.array([448.0, 896.0, 3.0, 0.0, 1e-9], F32)
    v = np.zeros((5, 128), F32)
    v[:, 0] = amax
    q, s = oracle.quant_1x128(v, oracle.SCALE_FP32, R)
    inv3 = F32(448.0) / F32(3.0)
    assert s[0, 0] == 1.0 and s[1, 0] == 2.0
    assert s[2, 0] == F32(1.0) / inv3
    assert s[3, 0] == oracle.SCALE_FLOOR and s[4, 0] == F32(1.0) / F32(229376.0)
    assert np.all(q[3] == 0)
    # the group maximum maps to the nearest E4M3 of amax * RN(448/amax) (448 or a neighbour)
    assert fm.E4M3_VALUES[q[2, 0]] == fm.E4M3_VALUES[fm.e4m3_encode(np.array([F32(3.0) * inv3]))[0]]


def test_reciprocal_quant_differs_from_division_on_bf16_inputs():
    """The two quantizers disagree on some BF16 inputs that sit on E4M3 midpoints (the reason the
    TensorRT-LLM page gives for matching the fused op), and each is its own nearest rounding."""
    rng = np.random.default_rng(21)
    v = fm.bf16_round((rng.standard_normal((4000, 128)) * 3).astype(F32))
    qd, sd = oracle.quant_1x128(v, oracle.SCALE_FP32, oracle.NUMERICS_DIVIDE)
    qr, sr = oracle.quant_1x128(v, oracle.SCALE_FP32, oracle.NUMERICS_RECIPROCAL)
    assert np.count_nonzero(qd != qr) > 0
    inv = F32(448.0) / np.abs(v).max(axis=1)
    assert np.array_equal(qr, fm.e4m3_encode((v * inv[:, None]).astype(F32)))
    assert np.array_equal(sr[:, 0], (F32(1.0) / inv).astype(F32))
    # power-of-two formats: the two numerics coincide
    for fmt in (oracle.SCALE_FP32_POW2, oracle.SCALE_UE8M0):
        a = oracle.quant_1x128(v[:50], fmt, oracle.NUMERICS_DIVIDE)
        b = oracle.quant_1x128(v[:50], fmt, oracle.NUMERICS_RECIPROCAL)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_reciprocal_numerics_rounds_swiglu_output_to_bf16(small_case):
    c = small_case
    w = c.weights
    e = int(c.topk_ids[0, 0])
    _, inter = oracle.expert_rows(c.x[:3], w.w13[e], w.s13[e], w.w2[e], w.s2[e], 0, 0,
                                  intermediates=True, numerics=oracle.NUMERICS_RECIPROCAL)
    assert np.array_equal(inter["h"], fm.bf16_round(inter["h"]))
    _, inter0 = oracle.expert_rows(c.x[:3], w.w13[e], w.s13[e], w.w2[e], w.s2[e], 0, 0,
                                   intermediates=True)
    assert not np.array_equal(inter0["h"], fm.bf16_round(inter0["h"]))
    ref = dense_reference(c)
    out = _fwd(c, numerics=oracle.NUMERICS_RECIPROCAL)
    assert np.linalg.norm(out - ref) / np.linalg.norm(ref) < 0.1


# --------------------------------------------------------- expert-parallel slice
def test_expert_slices_sum_to_the_whole_layer(small_case):
    """Ranks holding contiguous expert slices produce fp32 partials whose sum, rounded once to
    BF16, is the whole layer up to the order of the fp32 additions."""
    c = small_case
    w = c.weights
    full32 = _fwd(c, out_fp32=True)
    E = c.shape.E
    for world in (2, 3):
        total = np.zeros_like(full32)
        terms = np.zeros_like(full32)
        for r in range(world):
            base, extra = divmod(E, world)
            cnt = base + (1 if r < extra else 0)
            first = r * base + min(r, extra)
            part = oracle.moe_forward(c.x, c.topk_ids, c.topk_weights, w.w13[first:first + cnt],
                                      w.s13[first:first + cnt], w.w2[first:first + cnt],
                                      w.s2[first:first + cnt], expert_offset=first, out_fp32=True)
            total = (total + part).astype(F32)
            terms += np.abs(part)
        bound = 4 * 2.0 ** -23 * (terms + np.abs(full32))
        assert np.all(np.abs(total - full32) <= bound + 1e-30)
        assert np.mean(fm.bf16_round(total) == fm.bf16_round(full32)) > 0.99


def test_expert_offset_drops_ids_outside_the_slice(small_case):
    c = small_case
    w = c.weights
    first, cnt = 2, 3
    part = oracle.moe_forward(c.x, c.topk_ids, c.topk_weights, w.w13[first:first + cnt],
                              w.s13[first:first + cnt], w.w2[first:first + cnt],
                              w.s2[first:first + cnt], expert_offset=first)
    ids = c.topk_ids.copy()
    ids[(ids < first) | (ids >= first + cnt)] = -1
    masked = synth.LayerCase(c.shape, c.M_cap, c.n, c.x_bits, c.x, ids, c.topk_weights, c.weights)
    assert np.array_equal(part, _fwd(masked))
    a = oracle.align(c.topk_ids, c.n, cnt, expert_offset=first)
    assert (a["live_end"] - a["seg_start"][:-1]).sum() == np.count_nonzero(ids >= 0)


def test_batched_experts_match_the_routed_layer_and_the_dense_ffn(small_case):
    """Batched-expert layout: expert e on its first counts[e] rows equals the routed layer with
    one expert per token and weight 1 (out = the BF16 expert output), each live row is within FP8
    error of the dequantized dense FFN, and rows past the count stay out of the result."""
    c = small_case
    w = c.weights
    E, H = c.shape.E, c.shape.H
    max_m = 8
    counts = np.array([0, 8, 3, 1, 5, 8, 2, 7][:E], np.int64)
    rng = np.random.default_rng(11)
    xb = fm.bf16_round(rng.standard_normal((E, max_m, H)).astype(F32))
    out, live = oracle.batched_forward(xb, counts, w.w13, w.s13, w.w2, w.s2)
    assert live.sum() == counts.sum()
    assert np.all(np.isnan(out[~live])) and np.all(np.isfinite(out[live]))
    rows = xb[live]
    ids = np.repeat(np.arange(E), counts)[:, None].astype(np.int32)
    routed = oracle.moe_forward(rows, ids, np.ones_like(ids, dtype=F32), w.w13, w.s13, w.w2, w.s2)
    assert np.array_equal(out[live], routed)
    one = synth.LayerCase(c.shape, rows.shape[0], rows.shape[0], fm.bf16_bits(rows), rows, ids,
                          np.ones(ids.shape, F32), w)
    ref = dense_reference(one)
    assert np.linalg.norm(out[live] - ref) / np.linalg.norm(ref) < 0.1
    # counts are clamped to [0, max_m]; dead rows never influence live ones
    xb2 = xb.copy()
    xb2[~live] = 1e4
    wild = counts.copy()
    wild[0], wild[1] = -3, 99                 # clamp to 0 and to max_m
    out2, live2 = oracle.batched_forward(xb2, wild, w.w13, w.s13, w.w2, w.s2)
    assert np.array_equal(live2, live)
    assert np.array_equal(out2[live], out[live])
