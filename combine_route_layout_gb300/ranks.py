"""One EP rank per workspace with split send / receive phases (binding).

Mirrors the split operator API of the MORI-EP User Guide, section 3
("Split dispatch/combine (send + recv)"): dispatch_send returns the five
dispatch outputs, dispatch_recv completes them; combine_send returns the
combine outputs, combine_recv completes them. Every step runs in libep's
kernels (include/ep.h, ep_rank_*); this module only marshals pointers and
builds tensor views.

Each rank owns one workspace (a torch allocation here). The ranks see each
other's workspaces as device pointers: in one process, the other handles'
workspaces; across processes, peers' memory mapped into this process.
`connect` exchanges the mappings over a torch.distributed group, by
default with torch's CUDA IPC sharing (the process group carries only the
handles). The caller orders the phases across ranks: all ranks finish a
send phase (stream synchronised) before any rank starts the following
receive phase, e.g. with `phase_barrier`.
"""
from __future__ import annotations

import torch

from . import ep as E


def _stream():
    return torch.cuda.current_stream().cuda_stream


class EpRankOp:
    """Rank `rank` of a world_size-rank EP group (config.world_size ranks).

    Inputs of dispatch_send are this rank's tokens only: input [Tmax, H],
    weights [Tmax, k], indices [Tmax, k]; num_tokens <= Tmax."""

    def __init__(self, config: "E.EpDispatchCombineConfig", rank: int,
                 device: torch.device | str = "cuda"):
        self.config = config
        self.rank = int(rank)
        self.c = config.to_c()
        nbytes = E.ep_rank_workspace_size(self.c)
        if nbytes == 0:
            raise E.EpError(E.EP_ERR_INVALID_ARG, E.ep_last_error())
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self._handle = E.ep_rank_create(self.c, self.rank, self.workspace.data_ptr(), nbytes)
        self.cap = config.world_size * config.max_num_inp_token_per_rank
        self._mapped = []        # peers' workspaces mapped into this process (kept alive)
        self._views = None

    def __del__(self):
        h = getattr(self, "_handle", None)
        if h:
            E.ep_rank_destroy(h)
            self._handle = None

    # peers ---------------------------------------------------------------------
    def set_peers(self, peer_workspaces) -> None:
        """peer_workspaces: device pointers (ints) of every rank's workspace as
        this process sees them, in rank order (this rank's own included)."""
        E.ep_rank_set_peers(self._handle, list(peer_workspaces))

    def export_workspace(self):
        """A picklable handle another process can map with `open_peer`
        (torch's CUDA IPC sharing of the workspace tensor)."""
        from torch.multiprocessing.reductions import reduce_tensor
        fn, args = reduce_tensor(self.workspace)
        return (fn, args)

    def open_peer(self, exported) -> int:
        fn, args = exported
        t = fn(*args)
        self._mapped.append(t)
        return t.data_ptr()

    def connect(self, group=None, export=None, open_peer=None) -> list[int]:
        """Exchange workspaces with the other ranks of `group` (group rank =
        EP rank) and set the peer table. export / open_peer default to CUDA
        IPC; returns the peer pointers."""
        import torch.distributed as dist
        if dist.get_world_size(group) != self.config.world_size:
            raise E.EpError(E.EP_ERR_INVALID_ARG, "group size differs from world_size")
        ptrs = exchange_workspaces(self.rank, self.workspace.data_ptr(),
                                   export or self.export_workspace, open_peer or self.open_peer,
                                   group)
        self.set_peers(ptrs)
        return ptrs

    # views into the workspace -----------------------------------------------------
    def _view(self, ptr: int, dtype: torch.dtype, shape) -> torch.Tensor:
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        off = ptr - self.workspace.data_ptr()
        assert 0 <= off and off + nbytes <= self.workspace.numel()
        return self.workspace[off:off + nbytes].view(dtype).view(*shape)

    def _payload(self):
        cfg = self.config
        H = cfg.hidden_dim
        if cfg.quant_type == "fp8_e4m3_block128":
            return torch.float8_e4m3fn, H, H // 128
        if cfg.quant_type == "fp4_e2m1_block32":
            return torch.uint8, H // 2, H // 32
        if E._FP4X2 is not None and cfg.data_type == E._FP4X2:
            return cfg.data_type, H // 2, None
        return cfg.data_type, H, None

    def _dispatch_views(self, o):
        k = self.config.num_experts_per_token
        dt, cols, nsc = self._payload()
        x = self._view(o.x, dt, (self.cap, cols))
        if o.scales:
            sc = (self._view(o.scales, torch.float32, (self.cap, nsc)) if nsc is not None
                  else self._view(o.scales, torch.uint8, (self.cap, o.scale_row_bytes)))
        else:
            sc = None
        w = self._view(o.weights, torch.float32, (self.cap, k))
        idx = self._view(o.indices, torch.int32, (self.cap, k))
        recv = self._view(o.recv_num_token, torch.int32, (1,))
        return x, w, sc, idx, recv

    # phases --------------------------------------------------------------------------
    def dispatch_send(self, input, weights, scales, indices, num_tokens=None):
        """Returns (dispatch_output, dispatch_weights, dispatch_scales,
        dispatch_indices, recv_num_token), valid after dispatch_recv."""
        n = self.config.max_num_inp_token_per_rank if num_tokens is None else int(num_tokens)
        o = E.ep_dispatch_send(self._handle, E._ptr(input), E._ptr(weights), E._ptr(scales),
                               E._ptr(indices), n, _stream())
        if self._views is None:
            self._views = self._dispatch_views(o)
        return self._views

    def dispatch_recv(self) -> None:
        E.ep_dispatch_recv(self._handle, _stream())

    def combine_send(self, input, weights, indices=None, out=None, out_weights=None,
                     want_weights=True):
        """input: expert outputs [cap, H] in receive order, or None when the
        experts wrote get_registered_combine_input_buffer(). Returns
        (combine_output [Tmax, H], combine_weights [Tmax, k] or None), valid
        after combine_recv. `indices` is accepted for API parity."""
        cfg = self.config
        T, H, k = cfg.max_num_inp_token_per_rank, cfg.hidden_dim, cfg.num_experts_per_token
        dev = self.workspace.device
        if out is None:
            out = torch.empty((T, H), dtype=cfg.combine_out_dtype, device=dev)
        if out_weights is None and want_weights and weights is not None:
            out_weights = torch.empty((T, k), dtype=torch.float32, device=dev)
        E.ep_combine_send(self._handle, E._ptr(input), E._ptr(weights), E._ptr(out),
                          E._ptr(out_weights), _stream())
        return out, out_weights

    def combine_recv(self, call_reset: bool = False) -> None:
        E.ep_combine_recv(self._handle, call_reset, _stream())

    def reset(self) -> None:
        E.ep_rank_reset(self._handle)

    def get_registered_combine_input_buffer(self) -> torch.Tensor:
        cfg = self.config
        p = E.ep_rank_get_registered_combine_input_buffer(self._handle)
        return self._view(p, cfg.combine_dtype, (self.cap, cfg.hidden_dim))

    def get_dispatch_src_token_pos(self) -> torch.Tensor:
        p = E.ep_rank_get_dispatch_src_token_pos(self._handle)
        return self._view(p, torch.int32, (self.cap,))

    def sync(self) -> None:
        E.ep_rank_sync(self._handle, _stream())


def exchange_workspaces(rank: int, own_ptr: int, export, open_peer, group=None) -> list[int]:
    """Every rank's workspace pointer as this process sees it, in rank order:
    each rank publishes export() to the group (all_gather_object) and maps
    the others' with open_peer(handle); its own entry is own_ptr."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    allx = [None] * world
    dist.all_gather_object(allx, export(), group=group)
    return [int(own_ptr) if r == rank else int(open_peer(allx[r])) for r in range(world)]


def phase_barrier(group=None) -> None:
    """End of a phase on every rank: this rank's stream is drained, then all
    ranks meet (host barrier), so the next phase may read peers' buffers."""
    import torch.distributed as dist
    torch.cuda.current_stream().synchronize()
    dist.barrier(group=group)
