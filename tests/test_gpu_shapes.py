"""GPU parity at the edges of the supported shapes, through both GEMM schedules: a single 128-wide K
block (the two-K-block copies then deliver one block of zeros), odd K-block counts, the largest
top-k, a single expert, the largest expert count, and the largest FC1 K split."""

from __future__ import annotations

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import block_fp8_mixture_gb300 as moe  # noqa: E402
from test_gpu_parity import _layer_check  # noqa: E402


def _plan(case):
    sh = case.shape
    return moe.workspace_plan(case.M_cap, sh.E, sh.H, sh.I, sh.topk, sh.act_fmt)


@pytest.mark.parametrize("name,shape_kw,M,n,small", [
    ("k1_small", dict(E=4, H=128, I=128, topk=2), 8, 7, 1),          # one K block, one N block
    ("k1_tile", dict(E=2, H=128, I=128, topk=2), 128, 101, 0),
    ("k3_small", dict(E=8, H=384, I=256, topk=2), 16, 16, 1),       # odd K blocks, small schedule
    ("top16_small", dict(E=32, H=256, I=256, topk=16), 8, 8, 1),    # largest top-k
    ("top16_tile", dict(E=32, H=256, I=256, topk=16), 64, 50, 0),
    ("one_expert", dict(E=1, H=256, I=256, topk=1), 300, 300, 0),   # three tiles, ragged tail
    ("e1024", dict(E=1024, H=128, I=128, topk=8), 4, 4, 1),         # largest expert count
])
def test_layer_edge_shapes(name, shape_kw, M, n, small):
    shape = synth.small_shape(name, **shape_kw)
    case = synth.make_case(name, M, n, shape=shape)
    assert _plan(case)["small_batch"] == small
    _layer_check(case)


@pytest.mark.parametrize("act_fmt,weight_fmt", [(0, 0), (2, 2)])
def test_layer_largest_k_split(act_fmt, weight_fmt):
    """One token, two FC1 column blocks and a long K: the plan splits FC1's K eight ways and the
    last split to arrive sums the fp32 partials in split order."""
    shape = synth.small_shape("ks8", E=8, H=8192, I=256, topk=1, act_fmt=act_fmt,
                              weight_fmt=weight_fmt)
    case = synth.make_case("ks8", 1, 1, shape=shape)
    assert _plan(case)["fc1_ksplit"] == 8
    _layer_check(case)


@pytest.mark.parametrize("M,n", [(4, 4), (24, 19), (64, 64)])
def test_layer_decode_shaped(M, n):
    """Decode-shaped layers (K = 32 blocks, 64 experts) at batch sizes whose (chunk, column block)
    units leave the SMs partly idle, fill them, or give a ragged last round."""
    shape = synth.small_shape("dec_shape", E=64, H=4096, I=512, topk=8, clamp_mode=1, limit=7.0)
    case = synth.make_case("dec_shape", M, n, shape=shape)
    assert _plan(case)["small_batch"] == 1
    _layer_check(case)


def test_layer_ue8m0_tile_k1():
    """Block-scaled MMA path with a single K block per GEMM."""
    shape = synth.small_shape("bs_k1", E=2, H=128, I=128, topk=2, act_fmt=2, weight_fmt=2)
    case = synth.make_case("bs_k1", 128, 128, shape=shape)
    assert _plan(case)["small_batch"] == 0
    _layer_check(case)
