"""Worker of the two-process expert-parallel test: each rank computes its experts' fp32 partial
with the CPU oracle and the ranks all-reduce the partials over gloo."""

import os
import sys

import numpy as np


def run(rank, world, port, result_path):
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch
    import torch.distributed as dist

    import oracle
    import synth
    from block_fp8_mixture_gb300 import expert_slice

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    shape = synth.small_shape("ep", E=6, H=256, I=256, topk=3)
    case = synth.make_case("ep", 12, shape=shape)
    w = case.weights
    first, cnt = expert_slice(shape.E, world, rank)
    part = oracle.moe_forward(case.x, case.topk_ids, case.topk_weights, w.w13[first:first + cnt],
                              w.s13[first:first + cnt], w.w2[first:first + cnt],
                              w.s2[first:first + cnt], expert_offset=first, out_fp32=True)
    t = torch.from_numpy(part.copy())
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    if rank == 0:
        np.save(result_path, t.numpy())
    dist.barrier()
    dist.destroy_process_group()
