"""One EP rank of a split-phase group, checked against the oracle.

Used by tests/test_gpu_split.py both in one process (every rank a handle,
peers are the other handles' workspaces) and as one process per rank (peers
mapped with CUDA IPC over a gloo group). Every rank draws the whole group's
seeded inputs (so each process can run the oracle on them) and feeds its own
rank's part to the library.
"""
from __future__ import annotations

import os
from datetime import timedelta

import numpy as np
import torch

import oracle
from gen import WORKLOADS, make_expert_outputs, make_indices, make_num_tokens, make_tokens, \
    make_weights

DEV = "cuda"


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def out_bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) if a.dtype == np.float32 else a


def config(wl, **over):
    from combine_route_layout_gb300 import EpDispatchCombineConfig
    kw = dict(
        data_type=torch.bfloat16, world_size=wl.world_size, hidden_dim=wl.hidden, scale_dim=0,
        scale_type_size=4, max_token_type_size=4, max_num_inp_token_per_rank=wl.tokens_per_rank,
        num_experts_per_rank=wl.experts_per_rank, num_experts_per_token=wl.topk,
        quant_type={"fp8": "fp8_e4m3_block128", "fp4": "fp4_e2m1_block32"}.get(wl.dispatch_dtype,
                                                                            "none"),
        combine_dtype=torch.bfloat16,
        combine_out_dtype=torch.float32 if wl.combine_out_dtype == "fp32" else torch.bfloat16,
        weighted_combine=wl.weighted)
    kw.update(over)
    return EpDispatchCombineConfig(**kw)


class Group:
    """The whole group's seeded inputs and the oracle's results on them."""

    def __init__(self, wl, seed: int, ragged: bool):
        self.wl = wl
        self.idx = make_indices(wl, seed)
        self.w = make_weights(wl, seed)
        self.ntok = make_num_tokens(wl, ragged=ragged, seed=seed)
        xt = make_tokens(wl, seed)
        self.x = xt
        self.xb = xt.view(torch.int16).numpy().view(np.uint16)
        R, T = wl.world_size, wl.tokens_per_rank
        self.cap = R * T
        self.y = make_expert_outputs(wl, self.cap, seed)                 # [R][cap][H] bf16
        self.yb = self.y.view(torch.int16).numpy().view(np.uint16)
        self.recv, self.src_pos, self.slot = oracle.route(self.idx, self.ntok, wl.experts_per_rank)
        if wl.dispatch_dtype == "fp8":
            q, sc = oracle.quant_tokens(self.xb)
        elif wl.dispatch_dtype == "fp4":
            q, sc = oracle.quant_tokens_fp4(self.xb)
        else:
            q, sc = self.xb, None
        self.x_ref = oracle.place_rows(q, self.ntok, self.slot)
        self.sc_ref = oracle.place_rows(sc, self.ntok, self.slot) if sc is not None else None
        self.w_ref = oracle.place_rows(self.w, self.ntok, self.slot)
        self.idx_ref = oracle.place_rows(self.idx, self.ntok, self.slot)
        od = "fp32" if wl.combine_out_dtype == "fp32" else "bf16"
        self.out_ref, self.outw_ref = oracle.combine(self.yb, self.idx, self.ntok, self.slot,
                                                     wl.experts_per_rank, w_recv=self.w_ref,
                                                     weighted=wl.weighted, out_dtype=od)

    def inputs(self, r: int):
        x = self.x[r].to(DEV)
        w = torch.from_numpy(self.w[r]).to(DEV)
        idx = torch.from_numpy(self.idx[r]).to(DEV)
        return x, w, idx

    def check_dispatch(self, r: int, views, src_pos_d):
        x, w, sc, idx, recv = views
        n = int(self.recv[r])
        assert int(host(recv)[0]) == n, f"recv_num_token rank {r}"
        assert np.array_equal(host(src_pos_d)[:n], self.src_pos[r, :n]), f"src_token_pos rank {r}"
        assert np.array_equal(host(x)[:n], self.x_ref[r, :n]), f"payload rank {r}"
        if self.sc_ref is not None:
            assert np.array_equal(host(sc)[:n].view(np.uint32),
                                  self.sc_ref[r, :n].view(np.uint32)), f"scales rank {r}"
        assert np.array_equal(host(w)[:n].view(np.uint32), self.w_ref[r, :n].view(np.uint32))
        assert np.array_equal(host(idx)[:n], self.idx_ref[r, :n])

    def check_combine(self, s: int, out, out_w):
        n = int(self.ntok[s])
        assert np.array_equal(out_bits(host(out)[:n]), out_bits(self.out_ref[s, :n])), \
            f"combine rank {s}"
        if out_w is not None:
            assert np.array_equal(host(out_w)[:n].view(np.uint32),
                                  self.outw_ref[s, :n].view(np.uint32)), f"combine weights {s}"


def run_process_rank(rank: int, world: int, port: int, name: str, over: dict, seed: int,
                     ragged: bool, zero_copy: bool, rounds: int) -> None:
    """Body of one process of the multi-process test: gloo group for the
    workspace exchange and the phase barriers, CUDA IPC for the peers."""
    import torch.distributed as dist
    from combine_route_layout_gb300.ranks import EpRankOp, phase_barrier
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=timedelta(seconds=120))
    torch.cuda.set_device(0)
    try:
        wl = WORKLOADS[name].with_(world_size=world, **over)
        op = EpRankOp(config(wl), rank)
        op.connect()
        for it in range(rounds):
            g = Group(wl, seed + it, ragged)
            x, w, idx = g.inputs(rank)
            views = op.dispatch_send(x, w, None, idx, int(g.ntok[rank]))
            phase_barrier()
            op.dispatch_recv()
            phase_barrier()
            g.check_dispatch(rank, views, op.get_dispatch_src_token_pos())
            n = int(g.recv[rank])
            y = torch.from_numpy(g.yb[rank].view(np.int16)).to(DEV).view(torch.bfloat16)
            if zero_copy:
                op.get_registered_combine_input_buffer()[:n].copy_(y[:n])
                out, out_w = op.combine_send(None, views[1])
            else:
                out, out_w = op.combine_send(y, views[1])
            phase_barrier()
            op.combine_recv(call_reset=True)
            phase_barrier()
            op.sync()
            g.check_combine(rank, out, out_w)
        dist.barrier()                    # nobody unmaps while a peer may still read
        op._mapped.clear()
        torch.cuda.synchronize()
        dist.barrier()
    finally:
        dist.destroy_process_group()
