"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs.

Bars: alignment arrays and FC1-input codes/scales bit-exact; layer outputs within
1e-2 * max|oracle| per element; >= 99.9% of FC2-input codes identical; padded workspace rows and
output rows t >= n untouched.
"""

import numpy as np
import pytest

import oracle
import synth
from moe_testutil import (CODE_MATCH_MIN, assert_layer_close, bf16_tensor_to_f32, check_a2_codes,
                          check_untouched, device_case, oracle_forward, run_forward, scale_values)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import block_fp8_mixture_gb300 as moe  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    moe.load_library(build_if_missing=True)


# ------------------------------------------------------------------ align
ALIGN_CASES = [
    # (E, topk, M_cap, n, id_low, id_high)
    (8, 2, 16, 16, 0, 8),
    (72, 8, 16, 16, 0, 72),       # 128-pair threshold, non-power-of-two expert count
    (72, 8, 24, 24, 0, 72),       # above it
    (288, 8, 32, 32, -1, 290),    # invalid ids dropped
    (32, 8, 512, 16, 0, 32),      # device token count below capacity
    (128, 8, 8192, 8192, 0, 128),
    (1024, 4, 300, 257, -3, 1030),
    (5, 3, 0, 0, 0, 5),           # no tokens
    (16, 1, 64, 0, 0, 16),        # capacity but zero live tokens
    (64, 4, 2000, 1500, -1, 66),  # multi-CTA alignment, device count below capacity
    (16, 8, 1024, 3, 0, 16),      # multi-CTA alignment with fewer live pairs than CTAs
    (256, 8, 4096, 4096, 0, 256), # 32768 pairs
]


@pytest.mark.parametrize("E,topk,M_cap,n,lo,hi", ALIGN_CASES)
def test_align_bit_exact(E, topk, M_cap, n, lo, hi):
    rng = np.random.default_rng(E * 1000 + M_cap)
    ids = rng.integers(lo, hi, (M_cap, topk)).astype(np.int32)
    H, I = 256, 256
    ws = moe.alloc_workspace(M_cap, E, H, I, topk)
    ws.fill_(0xFF)
    d_ids = torch.from_numpy(ids).cuda()
    d_n = torch.tensor([n], dtype=torch.int32, device="cuda")
    moe.align(d_ids, E, H, I, ws, d_num_tokens=d_n)
    torch.cuda.synchronize()
    v = moe.workspace_views(ws, M_cap, E, H, I, topk)
    ref = oracle.align(ids, n, E)
    assert np.array_equal(v["seg_start"].cpu().numpy(), ref["seg_start"])
    assert np.array_equal(v["live_end"].cpu().numpy(), ref["live_end"])
    assert int(v["num_tiles"].item()) == ref["num_tiles"]
    assert np.array_equal(v["pair_row"].cpu().numpy()[: n * topk], ref["pair_row"])
    nt = ref["num_tiles"]
    assert np.array_equal(v["tile_expert"].cpu().numpy()[:nt], ref["tile_expert"])
    assert int(v["num_chunks"].item()) == ref["num_chunks"]
    assert np.array_equal(v["chunk_row0"].cpu().numpy()[: ref["num_chunks"]], ref["chunk_row0"])
    sp = v["sorted_pair"].cpu().numpy()
    live = ref["sorted_pair"] >= 0
    assert np.array_equal(sp[: live.size][live], ref["sorted_pair"][live])
    assert moe.last_device_status(ws) == moe.MOE_OK


# ------------------------------------------------------------------ quant
@pytest.mark.parametrize("fmt,numerics", [(moe.SCALE_FP32, 0), (moe.SCALE_FP32_POW2, 0),
                                          (moe.SCALE_UE8M0, 0), (moe.SCALE_FP32, 1)])
@pytest.mark.parametrize("H,M_cap,n,outliers", [(512, 16, 16, 0.0), (7168, 64, 40, 0.0),
                                                (2048, 300, 300, 0.01), (4096, 3, 1, 0.0)])
def test_quant_bit_exact(fmt, numerics, H, M_cap, n, outliers):
    E, topk, I = 16, 4, 256
    rng = np.random.default_rng(H + M_cap + fmt)
    x = rng.standard_normal((M_cap, H)).astype(np.float32)
    if outliers:
        x = np.where(rng.uniform(size=x.shape) < outliers, x * 10, x).astype(np.float32)
    x[0, :128] = 0.0                       # an all-zero group hits the scale floor
    x[min(1, M_cap - 1), 128:256] *= 1e-6  # tiny group
    xt = torch.from_numpy(x).to(torch.bfloat16)
    x_f = xt.float().numpy()
    ids = np.stack([rng.permutation(E)[:topk] for _ in range(M_cap)]).astype(np.int32)
    ids[0, 0] = -1
    ws = moe.alloc_workspace(M_cap, E, H, I, topk, fmt)
    ws.fill_(0xFF)
    d_n = torch.tensor([n], dtype=torch.int32, device="cuda")
    moe.align(torch.from_numpy(ids).cuda(), E, H, I, ws, d_num_tokens=d_n, act_fmt=fmt)
    moe.quant_act(xt.cuda(), topk, E, I, ws, d_num_tokens=d_n, act_fmt=fmt, numerics=numerics)
    torch.cuda.synchronize()
    v = moe.workspace_views(ws, M_cap, E, H, I, topk, fmt)
    pair_row = v["pair_row"].cpu().numpy()
    a1q = v["a1_q"].cpu().numpy()
    a1s = v["a1_s"].cpu().numpy()
    q_ref, s_ref = oracle.quant_1x128(x_f[:n], fmt, numerics)
    for t in range(n):
        for j in range(topk):
            row = pair_row[t * topk + j]
            if ids[t, j] < 0:
                assert row == -1
                continue
            assert np.array_equal(a1q[row], q_ref[t]), (t, j)
            got_s = a1s[:, row]
            if fmt == moe.SCALE_UE8M0:
                assert np.array_equal(got_s, oracle.scale_bytes(s_ref[t]))
            else:
                assert np.array_equal(got_s.view(np.uint32), s_ref[t].view(np.uint32))


# ------------------------------------------------------------------ layer
def _layer_check(case, *, tokens=None, check_codes=True, check_poison=True):
    out, ws, views = run_forward(case)
    torch.cuda.synchronize()
    assert moe.last_device_status(ws) == moe.MOE_OK
    gpu = bf16_tensor_to_f32(out)
    sel = np.arange(case.n) if tokens is None else np.asarray(tokens)
    ref, pairs = oracle_forward(case, sel, return_pairs=True)
    rel = assert_layer_close(gpu[sel], ref, case.shape.name)
    if check_codes and pairs:
        share = check_a2_codes(case, views, pairs)
        assert share >= 0.999, share
    if check_poison:
        if case.n < case.M_cap:
            assert bool((out[case.n:].view(torch.int16) == -1).all()), "rows t >= n written"
        check_untouched(case, views)
    return rel, out


def test_layer_tiny():
    _layer_check(synth.make_case("tiny", 16))


@pytest.mark.parametrize("clamp_mode,limit", [(0, 0.0), (1, 0.02), (2, 0.01)])
@pytest.mark.parametrize("act_fmt", [0, 1, 2])
def test_layer_small_variants(clamp_mode, limit, act_fmt):
    shape = synth.small_shape("small_v", E=12, H=512, I=384, topk=3, act_fmt=act_fmt,
                              clamp_mode=clamp_mode, limit=limit)
    _layer_check(synth.make_case("small_v", 40, 33, shape=shape))


@pytest.mark.parametrize("E,H,I,topk,M,n", [
    (12, 384, 384, 3, 40, 37),    # small-batch: odd 128-column block counts in H (FC2's last item
                                  # has one weight half) and in I (FC1 column blocks)
    (24, 640, 128, 1, 96, 90),    # top-1 routing, one FC1 column block, five FC2 blocks
    (64, 256, 256, 16, 48, 45),   # the largest supported top-k (16 pairs a token)
    (20, 384, 640, 16, 96, 96),   # top-16 on the 128-row tiles (1536 pairs > 16 E)
])
def test_layer_odd_blocks_and_topk_extremes(E, H, I, topk, M, n):
    shape = synth.small_shape("edge", E=E, H=H, I=I, topk=topk)
    case = synth.make_case("edge", M, n, shape=shape)
    small = moe.workspace_plan(M, E, H, I, topk)["small_batch"]
    assert small == (1 if M * topk <= 16 * E else 0)
    _layer_check(case)


@pytest.mark.parametrize("name,M", [("decode", 32), ("mid", 512)])
def test_layer_zero_and_duplicate_tokens(name, M):
    """Degenerate tokens, exactly: an all-zero x row quantizes to the floor scale and zero codes and
    gives an all-zero output row; two tokens with the same x and the same routing give identical
    output rows although their pairs sit in different rows of the expert segments."""
    case = synth.make_case(name, M)
    case.x_bits[3] = 0
    case.x[3] = 0.0
    case.x_bits[7] = case.x_bits[11]
    case.x[7] = case.x[11]
    case.topk_ids[7] = case.topk_ids[11]
    case.topk_weights[7] = case.topk_weights[11]
    _, out = _layer_check(case, tokens=[0, 3, 7, 11, M - 1])
    rows = out.view(torch.int16).cpu().numpy()
    assert not rows[3].any()
    assert np.array_equal(rows[7], rows[11])


@pytest.mark.parametrize("E,H,I,topk,M,n,small,ksplit", [
    (2, 32768, 128, 1, 8, 8, 1, 8),       # largest H: 256 K blocks, FC1 split 8 ways (the most)
    (2, 32768, 128, 1, 64, 60, 0, 1),     # largest H on the 128-row tiles
    (2, 128, 16384, 1, 8, 7, 1, 1),       # largest I: 128 FC1 column blocks, FC2 K = 16384
    (2, 128, 16384, 1, 64, 64, 0, 1),     # largest I on the 128-row tiles
    (1024, 256, 128, 8, 16, 16, 1, 1),    # largest expert count
])
def test_layer_maximum_dimensions(E, H, I, topk, M, n, small, ksplit):
    plan = moe.workspace_plan(M, E, H, I, topk)
    assert (plan["small_batch"], plan["fc1_ksplit"]) == (small, ksplit)
    shape = synth.small_shape("maxd", E=E, H=H, I=I, topk=topk)
    _layer_check(synth.make_case("maxd", M, n, shape=shape))


@pytest.mark.parametrize("clamp_mode,limit", [(0, 0.0), (1, 0.02), (2, 0.01)])
@pytest.mark.parametrize("act_fmt,weight_fmt", [(0, 0), (1, 0), (2, 2), (0, 2), (2, 0)])
def test_layer_tile_kernel_variants(clamp_mode, limit, act_fmt, weight_fmt):
    """128-row-tile schedule (P_cap > 16 E): odd K-block counts (I = 384), a hidden size that
    ends on half an output tile (H = 384), and a device token count below capacity."""
    shape = synth.small_shape("tile_v", E=4, H=384, I=384, topk=2, act_fmt=act_fmt,
                              weight_fmt=weight_fmt, clamp_mode=clamp_mode, limit=limit)
    case = synth.make_case("tile_v", 96, 80, shape=shape)
    assert moe.workspace_plan(96, 4, 384, 384, 2, act_fmt)["small_batch"] == 0
    _layer_check(case)


@pytest.mark.parametrize("shape_kw,M,n", [
    (dict(E=12, H=512, I=384, topk=3), 40, 33),                     # small-batch schedule
    (dict(E=4, H=384, I=384, topk=2), 96, 80),                      # 128-row-tile schedule
    (dict(E=4, H=384, I=384, topk=2, clamp_mode=1, limit=0.02), 96, 96),
])
def test_layer_reciprocal_numerics(shape_kw, M, n):
    """TensorRT-LLM fused-op numerics: multiply by RN(448/amax), BF16-rounded SwiGLU output."""
    shape = synth.small_shape("recip", numerics=1, **shape_kw)
    _layer_check(synth.make_case("recip", M, n, shape=shape))


def test_layer_decode_reciprocal_numerics():
    base = synth.SHAPES["decode"]
    shape = synth.LayerShape("decode_r", base.E, base.H, base.I, base.topk,
                             clamp_mode=base.clamp_mode, limit=base.limit, cfg_id=2, numerics=1)
    _layer_check(synth.make_case("decode_r", 4, shape=shape))


@pytest.mark.parametrize("act_fmt,weight_fmt", [(2, 2), (0, 2), (2, 0), (1, 2)])
def test_layer_small_ue8m0_weights(act_fmt, weight_fmt):
    """Small-batch schedule with UE8M0 block scales on either operand (byte scales: 16 to a
    16-byte scale box) and mixed with fp32 or power-of-two fp32 scales on the other."""
    shape = synth.small_shape("small_u", E=10, H=1024, I=256, topk=4, act_fmt=act_fmt,
                              weight_fmt=weight_fmt)
    _layer_check(synth.make_case("small_u", 64, shape=shape))


@pytest.mark.parametrize("M", [1, 4, 32])
def test_layer_decode(M):
    _layer_check(synth.make_case("decode", M))


@pytest.mark.parametrize("name", ["padded", "padded_fp32"])
def test_layer_padded_16_live(name):
    _layer_check(synth.make_case(name, 512, 16))


def test_layer_empty_and_dropped():
    shape = synth.small_shape("small_e", E=8, H=256, I=256, topk=2)
    case = synth.make_case("small_e", 20, shape=shape)
    case.topk_ids[:] = -1
    case.topk_ids[3, 1] = 5           # a single live pair
    _layer_check(case)
    zero = synth.make_case("small_e", 20, 0, shape=shape)
    out, ws, views = run_forward(zero)
    torch.cuda.synchronize()
    assert bool((out.view(torch.int16) == -1).all())


@pytest.mark.parametrize("name,M", [("glm_slice", 1), ("glm_slice", 8), ("glm_slice", 64),
                                    ("mid", 1), ("mid", 8), ("mid", 32), ("mid", 128)])
def test_layer_mid_sizes_full(name, M):
    """Every sweep point of the two swept workloads up to M=128, all tokens checked."""
    _layer_check(synth.make_case(name, M))


def covering_tokens(case):
    """Tokens whose pairs sit on the first and the last live row of every expert segment and of every
    live 128-row tile (so every tile of every expert, including each expert's partial last tile,
    and every position of the persistent GEMMs' work lists is checked), found from the oracle's
    alignment of the same routing."""
    a = oracle.align(case.topk_ids, case.n, case.shape.E)
    k = case.shape.topk
    seg, live, sp = a["seg_start"], a["live_end"], a["sorted_pair"]
    toks = set()
    for e in range(case.shape.E):
        for m0 in range(int(seg[e]), int(live[e]), oracle.ALIGN):
            last = min(m0 + oracle.ALIGN, int(live[e])) - 1
            toks.add(int(sp[m0]) // k)
            toks.add(int(sp[last]) // k)
    return np.array(sorted(toks), np.int64)


def check_a1_bit_exact(case, views, tokens):
    """FC1-input codes and scales of every pair of the given tokens equal the oracle's, bit for bit."""
    sh = case.shape
    k = sh.topk
    pair_row = views["pair_row"].cpu().numpy()
    q_ref, s_ref = oracle.quant_1x128(case.x[tokens], sh.act_fmt, sh.numerics)
    rows, want_q, want_s = [], [], []
    for i, t in enumerate(tokens):
        for j in range(k):
            r = int(pair_row[t * k + j])
            if 0 <= case.topk_ids[t, j] < sh.E:
                rows.append(r)
                want_q.append(q_ref[i])
                want_s.append(s_ref[i])
            else:
                assert r == -1
    idx = torch.from_numpy(np.array(rows, np.int64)).to(views["a1_q"].device)
    got_q = views["a1_q"].index_select(0, idx).cpu().numpy()
    got_s = views["a1_s"].index_select(1, idx).cpu().numpy().T
    assert np.array_equal(got_q, np.stack(want_q))
    want_s = np.stack(want_s)
    if sh.act_fmt == oracle.SCALE_UE8M0:
        assert np.array_equal(got_s, oracle.scale_bytes(want_s))
    else:
        assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32))
    return len(rows)


@pytest.mark.parametrize("name,M_cap,n", [("padded", 4096, 4096), ("padded_fp32", 4096, 4096),
                                          ("glm_slice", 4096, 4096),
                                          ("mid", 8192, 8192), ("glm_slice", 1024, 1024),
                                          ("mid", 2048, 2048), ("glm_slice", 256, 256),
                                          ("mid", 512, 512)])
def test_layer_large_every_tile(name, M_cap, n):
    """Full-size layers, checked on the tokens that cover the first and last live row of every 128-row
    tile and every expert segment; their FC1-input codes and scales bit-exact, their FC2-input codes
    >= 99.9% identical, their outputs within the layer tolerance, and the padding untouched."""
    case = synth.make_case(name, M_cap, n)
    tokens = covering_tokens(case)
    out, ws, views = run_forward(case)
    torch.cuda.synchronize()
    assert moe.last_device_status(ws) == moe.MOE_OK
    assert check_a1_bit_exact(case, views, tokens) > 0
    gpu = bf16_tensor_to_f32(out)
    ref, pairs = oracle_forward(case, tokens, return_pairs=True)
    assert_layer_close(gpu[tokens], ref, f"{name} {M_cap}")
    assert check_a2_codes(case, views, pairs) >= CODE_MATCH_MIN
    check_untouched(case, views)


def _embed(case, M_big, seed):
    """The same n live tokens (x rows, ids, routing weights) at a larger token capacity; the rows
    past n hold other tokens that must never be read."""
    rng = np.random.default_rng(seed)
    sh = case.shape
    big = synth.make_case(sh.name, M_big, case.n, shape=sh, seed=seed, weights=case.weights)
    big.x_bits[: case.M_cap] = case.x_bits
    big.x[: case.M_cap] = case.x
    big.topk_ids[: case.M_cap] = case.topk_ids
    big.topk_weights[: case.M_cap] = case.topk_weights
    big.x_bits[case.n:] = rng.integers(0, 2 ** 16, big.x_bits[case.n:].shape).astype(np.uint16)
    return big


@pytest.mark.parametrize("name,M_small,M_big,n", [("padded_fp32", 4096, 8192, 4096),
                                                  ("padded", 512, 4096, 16),
                                                  ("decode", 16, 48, 16)])
def test_capacity_invariance(name, M_small, M_big, n):
    """The padded capacity never reaches the result (vLLM padded-work page, Validation: outputs
    identical between schedules, poisoned workspaces): the same live tokens at two capacities that
    take the same GEMM schedule give byte-identical outputs, and both workspaces keep their
    poisoned padding."""
    small = synth.make_case(name, M_small, n)
    big = _embed(small, M_big, seed=99)
    sh = small.shape
    p_s = moe.workspace_plan(M_small, sh.E, sh.H, sh.I, sh.topk, sh.act_fmt)
    p_b = moe.workspace_plan(M_big, sh.E, sh.H, sh.I, sh.topk, sh.act_fmt)
    assert (p_s["small_batch"], p_s["fc1_ksplit"]) == (p_b["small_batch"], p_b["fc1_ksplit"])
    assert p_b["R_cap"] > p_s["R_cap"]
    out_s, ws_s, v_s = run_forward(small)
    out_b, ws_b, v_b = run_forward(big)
    torch.cuda.synchronize()
    assert moe.last_device_status(ws_s) == moe.MOE_OK and moe.last_device_status(ws_b) == moe.MOE_OK
    assert torch.equal(out_s[:n].view(torch.int16), out_b[:n].view(torch.int16))
    assert bool((out_s[n:].view(torch.int16) == -1).all())
    assert bool((out_b[n:].view(torch.int16) == -1).all())
    check_untouched(small, v_s)
    check_untouched(big, v_b)


@pytest.mark.parametrize("name,M", [("decode", 32), ("tiny", 16), ("mid", 512)])
def test_layer_zero_routing_weights(name, M):
    """Zero routing weights (TensorRT-LLM page, human review): a zero-weight pair still runs through
    the experts but contributes exactly nothing; a token whose weights are all zero gets a zero row."""
    case = synth.make_case(name, M)
    case.topk_weights[1, :] = 0.0
    case.topk_weights[2, ::2] = 0.0
    case.topk_weights[M - 1, -1] = 0.0
    rel, out = _layer_check(case, tokens=[0, 1, 2, 5, M - 1])
    rows = out.view(torch.int16).cpu().numpy()
    assert not rows[1].any()


def test_layer_forced_empty_experts():
    case = synth.make_case("mid", 512, routing="softmax_empty4")
    assert not np.any(case.topk_ids % 4 == 0)
    tokens = np.random.default_rng(3).choice(512, 16, replace=False)
    _layer_check(case, tokens=tokens)


def test_pow2_activation_scales_glm():
    shape = synth.LayerShape("glm_pow2", 256, 6144, 256, 8, act_fmt=synth.SCALE_FP32_POW2,
                             routing="zipf", cfg_id=4)
    case = synth.make_case("glm_pow2", 256, shape=shape)
    tokens = np.random.default_rng(5).choice(256, 12, replace=False)
    _layer_check(case, tokens=tokens)


def test_deterministic():
    case = synth.make_case("decode", 4)
    o1, _, _ = run_forward(case)
    o2, _, _ = run_forward(case)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


@pytest.mark.parametrize("name,M,n", [("decode", 1, 1), ("decode", 4, 4), ("decode", 32, 29),
                                      ("mid", 128, 128), ("glm_slice", 1024, 1000),
                                      ("padded", 512, 16)])
def test_step_entry_points_match_forward(name, M, n):
    """The five per-step entry points run back to back give the whole-layer forward's output bit for
    bit (small-batch schedule for the decode and mid cases, 128-row tiles for glm_slice, block-scaled
    128-row tiles for padded, where the standalone FC2 also checks FC1's per-tile counters)."""
    case = synth.make_case(name, M, n)
    sh = case.shape
    dev = device_case(case)
    o_fwd, ws_fwd, _ = run_forward(case, dev)
    ws = moe.alloc_workspace(M, sh.E, sh.H, sh.I, sh.topk, sh.act_fmt)
    ws.fill_(0xFF)
    out = torch.empty((M, sh.H), dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)
    args = moe.make_args(dev["x"], dev["ids"], dev["w"], dev["w13"], dev["s13"], dev["w2"], dev["s2"],
                         out, E=sh.E, H=sh.H, I=sh.I, topk=sh.topk, M_cap=M, d_num_tokens=dev["n"],
                         weight_fmt=sh.weight_fmt, act_fmt=sh.act_fmt, clamp_mode=sh.clamp_mode,
                         clamp_limit=sh.limit, numerics=sh.numerics)
    moe.align(dev["ids"], sh.E, sh.H, sh.I, ws, d_num_tokens=dev["n"], act_fmt=sh.act_fmt)
    moe.quant_act(dev["x"], sh.topk, sh.E, sh.I, ws, d_num_tokens=dev["n"], act_fmt=sh.act_fmt,
                  numerics=sh.numerics)
    moe.fc1_swiglu_quant(args, ws)
    moe.fc2(args, ws)
    moe.topk_reduce(args, ws)
    torch.cuda.synchronize()
    assert moe.last_device_status(ws_fwd) == 0 and moe.last_device_status(ws) == 0
    assert torch.equal(o_fwd[:n].view(torch.int16), out[:n].view(torch.int16))


def test_bounded_wait_expiry_reported_and_context_usable():
    """A device wait that nothing completes runs out (the pipelines' bounded-wait helper with a 2 ms
    limit), the status word reads MOE_ERR_DEVICE_TIMEOUT, and the next forward on the same
    workspace runs, resets the word and reproduces the earlier output."""
    case = synth.make_case("decode", 4)
    dev = device_case(case)
    o1, ws, _ = run_forward(case, dev)
    torch.cuda.synchronize()
    assert moe.last_device_status(ws) == moe.MOE_OK
    moe.selftest_wait_timeout(ws, 2000)
    assert moe.last_device_status(ws) == moe.MOE_ERR_DEVICE_TIMEOUT
    o2, _, _ = run_forward(case, dev, ws=ws, poison=False)
    torch.cuda.synchronize()
    assert moe.last_device_status(ws) == moe.MOE_OK
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_tile_ready_wait_expiry_reported_and_context_usable():
    """The block-scaled FC2 of a routed layer waits, per row tile, for FC1's completion counters
    instead of the whole FC1 grid.  Run right after the alignment reset those counters, with no FC1
    in between, its bounded wait runs out (1 s), the status word reads MOE_ERR_DEVICE_TIMEOUT, and
    the next forward on the same workspace runs normally and reproduces the earlier output."""
    shape = synth.small_shape("tile_to", E=4, H=384, I=256, topk=2, act_fmt=2, weight_fmt=2)
    case = synth.make_case("tile_to", 96, 80, shape=shape)
    sh = case.shape
    assert moe.workspace_plan(96, sh.E, sh.H, sh.I, sh.topk, sh.act_fmt)["small_batch"] == 0
    dev = device_case(case)
    o1, ws, _ = run_forward(case, dev)
    torch.cuda.synchronize()
    assert moe.last_device_status(ws) == moe.MOE_OK
    moe.align(dev["ids"], sh.E, sh.H, sh.I, ws, d_num_tokens=dev["n"], act_fmt=sh.act_fmt)
    out = torch.empty((96, sh.H), dtype=torch.bfloat16, device="cuda")
    args = moe.make_args(dev["x"], dev["ids"], dev["w"], dev["w13"], dev["s13"], dev["w2"], dev["s2"],
                         out, E=sh.E, H=sh.H, I=sh.I, topk=sh.topk, M_cap=96, d_num_tokens=dev["n"],
                         weight_fmt=sh.weight_fmt, act_fmt=sh.act_fmt)
    moe.fc2(args, ws)
    torch.cuda.synchronize()
    assert moe.last_device_status(ws) == moe.MOE_ERR_DEVICE_TIMEOUT
    o2, _, _ = run_forward(case, dev, ws=ws, poison=False)
    torch.cuda.synchronize()
    assert moe.last_device_status(ws) == moe.MOE_OK
    assert torch.equal(o1[:80].view(torch.int16), o2[:80].view(torch.int16))


def test_graph_replay_changing_routing():
    """Capture once, then change routing and the live-token count in place between replays."""
    shape = synth.small_shape("graph", E=16, H=512, I=256, topk=4)
    case = synth.make_case("graph", 48, 48, shape=shape)
    dev = device_case(case)
    ws = moe.alloc_workspace(48, 16, 512, 256, 4)
    out = torch.empty((48, 512), dtype=torch.bfloat16, device="cuda")
    args = moe.make_args(dev["x"], dev["ids"], dev["w"], dev["w13"], dev["s13"], dev["w2"], dev["s2"],
                         out, E=16, H=512, I=256, topk=4, M_cap=48, d_num_tokens=dev["n"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        moe.forward(args, ws, s)           # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.forward(args, ws, s)
    rng = np.random.default_rng(77)
    for n in (48, 17, 1):
        ids, w = synth.make_routing("softmax", 48, 16, 4, rng)
        case.topk_ids[:] = ids
        case.topk_weights[:] = w
        case.n = n
        dev["ids"].copy_(torch.from_numpy(ids))
        dev["w"].copy_(torch.from_numpy(w))
        dev["n"].fill_(n)
        out.view(torch.int16).fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        gpu = bf16_tensor_to_f32(out)
        ref = oracle_forward(case)
        assert_layer_close(gpu[:n], ref, f"replay n={n}")
        assert bool((out[n:].view(torch.int16) == -1).all())


def test_graph_replay_changing_routing_block_scaled_tiles():
    """The block-scaled 128-row-tile schedule, whose FC2 starts on row tiles once FC1's per-tile
    counters are complete: one captured forward replayed with new routing and live-token counts
    (the alignment resets the counters on every replay) matches the oracle every time."""
    E, H, I, k, M = 8, 512, 256, 4, 96
    shape = synth.small_shape("graph_bs", E=E, H=H, I=I, topk=k, act_fmt=2, weight_fmt=2)
    assert moe.workspace_plan(M, E, H, I, k, 2)["small_batch"] == 0
    case = synth.make_case("graph_bs", M, M, shape=shape)
    dev = device_case(case)
    ws = moe.alloc_workspace(M, E, H, I, k, 2)
    out = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    args = moe.make_args(dev["x"], dev["ids"], dev["w"], dev["w13"], dev["s13"], dev["w2"], dev["s2"],
                         out, E=E, H=H, I=I, topk=k, M_cap=M, d_num_tokens=dev["n"], weight_fmt=2,
                         act_fmt=2)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        moe.forward(args, ws, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.forward(args, ws, s)
    rng = np.random.default_rng(78)
    for n in (96, 41, 3, 96):
        ids, w = synth.make_routing("softmax", M, E, k, rng)
        case.topk_ids[:] = ids
        case.topk_weights[:] = w
        case.n = n
        dev["ids"].copy_(torch.from_numpy(ids))
        dev["w"].copy_(torch.from_numpy(w))
        dev["n"].fill_(n)
        out.view(torch.int16).fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert moe.last_device_status(ws) == moe.MOE_OK
        gpu = bf16_tensor_to_f32(out)
        assert_layer_close(gpu[:n], oracle_forward(case), f"block-scaled replay n={n}")
        assert bool((out[n:].view(torch.int16) == -1).all())


@pytest.mark.parametrize("world,fmt", [(2, 0), (3, 0), (2, 2)])
def test_expert_parallel_virtual_ranks(world, fmt):
    """Expert-parallel slices run one after another on one GPU ("virtual ranks"): each rank's fp32
    partial matches the oracle's partial, rows t >= n stay untouched, and the rank-ordered fp32 sum
    rounded once to BF16 matches the whole layer.  With UE8M0 scales and 256 pairs on 16 experts the
    slices run the block-scaled 128-row tiles (FC2 starting on FC1's finished tiles)."""
    E, H, I, k = 16, 512, 256, 4
    M, n = (64, 50) if fmt == 0 else (256, 250)
    shape = synth.small_shape("ep_gpu", E=E, H=H, I=I, topk=k, act_fmt=fmt, weight_fmt=fmt)
    case = synth.make_case("ep_gpu", M, n, shape=shape)
    dev = device_case(case)
    w = case.weights
    total = torch.zeros((M, H), dtype=torch.float32, device="cuda")
    whole = oracle_forward(case)
    for r in range(world):
        first, cnt = moe.expert_slice(E, world, r)
        sl = slice(first, first + cnt)
        if fmt == 2:
            assert moe.workspace_plan(M, cnt, H, I, k, fmt)["small_batch"] == 0
        ws = moe.alloc_workspace(M, cnt, H, I, k, fmt)
        out = torch.full((M, H), float("nan"), dtype=torch.float32, device="cuda")
        args = moe.make_args(dev["x"], dev["ids"], dev["w"], dev["w13"][sl], dev["s13"][sl],
                             dev["w2"][sl], dev["s2"][sl], out, E=cnt, H=H, I=I, topk=k, M_cap=M,
                             d_num_tokens=dev["n"], expert_offset=first, out_fp32=True,
                             weight_fmt=fmt, act_fmt=fmt)
        moe.forward(args, ws)
        torch.cuda.synchronize()
        assert moe.last_device_status(ws) == moe.MOE_OK
        part = out.cpu().numpy()
        ref = oracle.moe_forward(case.x, case.topk_ids, case.topk_weights, w.w13[sl], w.s13[sl],
                                 w.w2[sl], w.s2[sl], expert_offset=first, out_fp32=True,
                                 tokens=np.arange(n), act_fmt=fmt, weight_fmt=fmt)
        assert np.all(np.isnan(part[n:]))
        assert np.abs(part[:n] - ref).max() <= 1e-2 * float(np.abs(whole).max())
        total += out.nan_to_num(0.0)
    got = oracle.bf16_round(total.cpu().numpy()[:n])
    assert_layer_close(got, whole, f"expert parallel x{world}")
