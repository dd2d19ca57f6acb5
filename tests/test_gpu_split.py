"""Split send / receive phases with one EP rank per workspace, through the C
ABI, against the CPU oracle bit for bit (MORI-EP User Guide, section 3,
"Split dispatch/combine (send + recv)").

Each rank's receive rows, src_token_pos, scales, weights, ids and combine
outputs must equal that rank's part of the oracle's dispatch and combine
on the whole group's inputs. In one process every rank is a handle and the
peers are the other handles' workspaces (one stream orders the phases);
across processes every rank is a process on the same GPU, the peers are
mapped with CUDA IPC and a gloo group carries the handles and the phase
barriers (no kernel waits on another rank)."""
import os
import socket

import numpy as np
import pytest
import torch

from gen import WORKLOADS
from split_worker import DEV, Group, config, run_process_rank

pytestmark = pytest.mark.gpu


def run_inprocess(wl, seed=0, ragged=False, zero_copy=False, rounds=1, streams=False,
                  **cfg_over):
    """Every rank a handle. One stream orders the phases, or (streams=True)
    every rank runs on a stream of its own and a phase ends when all ranks'
    streams have finished it, as ranks on separate GPUs would run."""
    from combine_route_layout_gb300.ranks import EpRankOp
    R = wl.world_size
    ops = [EpRankOp(config(wl, **cfg_over), r) for r in range(R)]
    ptrs = [op.workspace.data_ptr() for op in ops]
    for op in ops:
        op.set_peers(ptrs)
    lanes = [torch.cuda.Stream() for _ in range(R)] if streams else None

    def phase(fn):
        if not streams:
            return [fn(r, op) for r, op in enumerate(ops)]
        cur = torch.cuda.current_stream()
        out = []
        for r, op in enumerate(ops):
            lanes[r].wait_stream(cur)
            with torch.cuda.stream(lanes[r]):
                out.append(fn(r, op))
        for ln in lanes:
            cur.wait_stream(ln)
        return out

    for it in range(rounds):
        g = Group(wl, seed + it, ragged)
        ins = [g.inputs(r) for r in range(R)]
        views = phase(lambda r, op: op.dispatch_send(ins[r][0], ins[r][1], None, ins[r][2],
                                                     int(g.ntok[r])))
        phase(lambda r, op: op.dispatch_recv())
        torch.cuda.synchronize()
        for r, op in enumerate(ops):
            g.check_dispatch(r, views[r], op.get_dispatch_src_token_pos())
        ys = [torch.from_numpy(g.yb[r].view(np.int16)).to(DEV).view(torch.bfloat16)
              for r in range(R)]
        if zero_copy:
            for r, op in enumerate(ops):
                n = int(g.recv[r])
                op.get_registered_combine_input_buffer()[:n].copy_(ys[r][:n])
        outs = phase(lambda r, op: op.combine_send(None if zero_copy else ys[r], views[r][1]))
        phase(lambda r, op: op.combine_recv(call_reset=True))
        for op in ops:
            op.sync()
        for s in range(R):
            g.check_combine(s, *outs[s])


@pytest.mark.parametrize("name,over,seed,ragged", [
    ("tiny", dict(), 0, False),
    ("tiny", dict(), 1, True),
    ("ds_v3_latency", dict(tokens_per_rank=64, hidden=1024), 2, True),             # FP8
    ("ds_v3_latency", dict(tokens_per_rank=300, hidden=2048), 3, True),            # several chunks
    ("ds_v3_latency", dict(tokens_per_rank=48, hidden=1056, dispatch_dtype="fp4"), 4, True),
    ("mid_masked", dict(tokens_per_rank=100, hidden=512), 5, True),                # dropped slots
    ("mid_masked", dict(tokens_per_rank=100, hidden=512, weighted=True,
                        combine_out_dtype="fp32"), 6, True),                       # weighted
    ("tiny", dict(world_size=1, experts_per_rank=8), 7, False),
    ("tiny", dict(world_size=16, experts_per_rank=2, topk=8, tokens_per_rank=24), 8, True),
])
def test_split_phases_in_one_process(name, over, seed, ragged):
    run_inprocess(WORKLOADS[name].with_(**over), seed, ragged)


def test_split_phases_zero_copy_and_repeated_rounds():
    """Experts writing the registered combine input in place, and three
    rounds on the same handles with different routings and token counts."""
    wl = WORKLOADS["ds_v3_latency"].with_(tokens_per_rank=80, hidden=1024)
    run_inprocess(wl, seed=11, ragged=True, zero_copy=True, rounds=3)


@pytest.mark.parametrize("name,over,seed,zero_copy", [
    ("ds_v3_latency", dict(), 12, True),                                     # FP8, decode shape
    ("mid_masked", dict(tokens_per_rank=300, hidden=1024, weighted=True,
                        combine_out_dtype="fp32"), 13, False),
])
def test_split_phases_one_stream_per_rank(name, over, seed, zero_copy):
    """Every rank's phase on its own stream, the ranks' kernels running side
    by side (as bench.py --split times them); two rounds."""
    run_inprocess(WORKLOADS[name].with_(**over), seed=seed, ragged=True, zero_copy=zero_copy,
                  rounds=2, streams=True)


def test_split_phases_decode_shape():
    """The DeepSeek-V3 decode shape (8 ranks x 32 experts, 128 tokens/rank,
    H 7168, top-8, FP8 dispatch, bf16 combine) through the split phases."""
    run_inprocess(WORKLOADS["ds_v3_latency"], seed=0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


@pytest.mark.parametrize("world,name,over,zero_copy", [
    (2, "ds_v3_latency", dict(tokens_per_rank=64, hidden=1024, experts_per_rank=8), False),
    (4, "mid_masked", dict(tokens_per_rank=100, hidden=512, experts_per_rank=4), True),
])
def test_split_phases_one_process_per_rank(world, name, over, zero_copy):
    """Every rank a process on cuda:0, peers' workspaces mapped with CUDA IPC,
    phases separated by host barriers; two rounds."""
    import torch.multiprocessing as mp
    mp.spawn(run_process_rank,
             args=(world, _free_port(), name, over, 21, True, zero_copy, 2),
             nprocs=world, join=True)
