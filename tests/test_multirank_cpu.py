"""Multi-rank plumbing on CPU with gloo ranks: bench.py's barrier and
max-over-ranks timing (each rank runs an independent replica; no collective
touches the data path), and the EP rank handles' workspace exchange and
phase state machine (every rank of the group a process; the exchange only
carries workspace handles, no data)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier_fn(w)()
    mx = bench.reduce_max(float(10 + 5 * rank), w)
    q.put((rank, mx))
    dist.destroy_process_group()


def test_two_rank_max_timing():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 15.0), (1, 15.0)]


def test_reference_arm_single_rank_line():
    """The reference arm prints one line with the contract keys."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "2", "--warmup", "3",
                          "--ref-tokens", "16"], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "impl", "cpu_baseline", "e2e", "higher_is_better"):
        assert key in line
    assert line["impl"] == "reference" and line["value"] > 0


FAKE = 1 << 40   # aligned addresses that these tests never dereference


def _rank_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from combine_route_layout_gb300 import ep
    from combine_route_layout_gb300.ranks import exchange_workspaces
    c = ep.ep_config()
    for k, v in dict(world_size=world, hidden_dim=512, scale_dim=0, scale_type_size=4,
                     max_token_type_size=4, max_num_inp_token_per_rank=64,
                     num_experts_per_rank=4, num_experts_per_token=4,
                     data_type=ep.EP_DTYPE_BF16, quant_type=ep.EP_QUANT_FP8_E4M3_BLOCK128,
                     combine_dtype=ep.EP_DTYPE_BF16, combine_out_dtype=ep.EP_DTYPE_BF16,
                     use_external_inp_buf=1).items():
        setattr(c, k, v)
    n = ep.ep_rank_workspace_size(c)
    sizes = [None] * world
    dist.all_gather_object(sizes, n)            # same config: same carve on every rank
    mine = FAKE + (rank << 32)
    h = ep.ep_rank_create(c, rank, mine, n)
    opened = []
    ptrs = exchange_workspaces(rank, mine, export=lambda: mine,
                               open_peer=lambda x: opened.append(x) or x)
    ep.ep_rank_set_peers(h, ptrs)
    # the receive phases are refused until a send phase ran on this rank
    errs = []
    for call in (lambda: ep.ep_dispatch_recv(h, None), lambda: ep.ep_combine_recv(h, 0, None)):
        try:
            call()
        except ep.EpError as e:
            errs.append(e.status)
    ep.ep_rank_destroy(h)
    dist.barrier()
    q.put((rank, sizes, ptrs, sorted(opened), errs))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_rank_workspace_exchange(world):
    """Each rank publishes its workspace and opens every other rank's: the
    peer tables agree, in rank order, with the own entry in place, and the
    rank handles accept them."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted((q.get(timeout=10) for _ in range(world)), key=lambda t: t[0])
    want = [FAKE + (r << 32) for r in range(world)]
    for rank, sizes, ptrs, opened, errs in got:
        assert len(set(sizes)) == 1 and sizes[0] > 0
        assert ptrs == want
        assert opened == [p for r, p in enumerate(want) if r != rank]
        assert errs == [-2, -2]                      # EP_ERR_STATE
