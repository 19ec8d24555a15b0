"""Expert-parallel layer across two processes (gloo on CPU): contiguous expert slices, fp32 partial
outputs, one all-reduce, one BF16 rounding -- compared with the whole layer."""

import multiprocessing as mp
import socket

import numpy as np

import oracle
import synth
from oracle import formats as fm


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_rank_expert_parallel_matches_whole_layer(tmp_path):
    import ep_gloo_worker
    ctx = mp.get_context("spawn")
    port = _free_port()
    out = str(tmp_path / "sum.npy")
    procs = [ctx.Process(target=ep_gloo_worker.run, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        assert p.exitcode == 0
    total = np.load(out)
    shape = synth.small_shape("ep", E=6, H=256, I=256, topk=3)
    case = synth.make_case("ep", 12, shape=shape)
    w = case.weights
    whole = oracle.moe_forward(case.x, case.topk_ids, case.topk_weights, w.w13, w.s13, w.w2, w.s2,
                               out_fp32=True)
    assert np.allclose(total, whole, rtol=0, atol=4 * 2.0 ** -23 * float(np.abs(whole).max()))
    assert np.mean(fm.bf16_round(total) == fm.bf16_round(whole)) > 0.99
