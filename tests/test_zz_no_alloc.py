"""The routing-layout entry point that allocates nothing.

Callers that cannot call cudaMalloc -- plugins and embedded engines whose
host application has reserved all device memory in its own pool, and code
paths that must not enter a device allocator -- call
ep_routing_layout_noalloc, whose scratch is a static device array inside
libep. This file runs last (pytest collects it after the others) and checks,
through the C ABI, that two calls in a row reproduce ep_dispatch's layout
exactly; the second call uses a different geometry so stale scratch from the
first would show.
"""
import numpy as np
import pytest
import torch

from combine_route_layout_gb300 import EpDispatchCombineOp, EpError
from combine_route_layout_gb300 import ep as E
from gen import WORKLOADS, make_indices, make_num_tokens

pytestmark = pytest.mark.gpu


def _via_dispatch(wl, idx_d, ntok):
    from ep_harness import make_config
    op = EpDispatchCombineOp(make_config(wl, quant_type="none", combine_dtype=torch.bfloat16))
    x = torch.zeros((wl.world_size, wl.tokens_per_rank, wl.hidden), dtype=torch.bfloat16,
                    device="cuda")
    w = torch.zeros((wl.world_size, wl.tokens_per_rank, wl.topk), dtype=torch.float32,
                    device="cuda")
    d = op.dispatch(x, w, None, idx_d, ntok)
    op.sync()
    recv = d[4].cpu().numpy().copy()
    src = op.get_dispatch_src_token_pos().cpu().numpy().copy()
    op.reset()
    return recv, src


def _via_noalloc(wl, idx_d, ntok):
    """Run the entry point into outputs allocated beforehand; returns its
    results and the device memory it took (free memory before minus after)."""
    R, T = wl.world_size, wl.tokens_per_rank
    recv = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    src = torch.full((R, R * T), -7, dtype=torch.int32, device="cuda")
    slot = torch.full((R, T, R), -7, dtype=torch.int32, device="cuda")
    err = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    E.ep_routing_layout_noalloc(R, T, wl.experts_per_rank, wl.topk, idx_d.data_ptr(),
                                list(ntok), recv.data_ptr(), src.data_ptr(), slot.data_ptr(),
                                err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    took = free0 - torch.cuda.mem_get_info()[0]
    return recv.cpu().numpy(), src.cpu().numpy(), slot.cpu().numpy(), int(err.item()), took


def test_noalloc_layout_matches_dispatch_on_two_calls():
    cases = [(WORKLOADS["ds_v3_throughput"].with_(hidden=256), 0, False),
             (WORKLOADS["mid_masked"].with_(hidden=256, tokens_per_rank=1500), 1, True)]
    for call, (wl, seed, ragged) in enumerate(cases):
        R, T = wl.world_size, wl.tokens_per_rank
        idx = make_indices(wl, seed)
        ntok = make_num_tokens(wl, ragged=ragged, seed=seed)
        idx_d = torch.from_numpy(idx).cuda()
        recv_ref, src_ref = _via_dispatch(wl, idx_d, ntok)
        recv, src, slot, err, took = _via_noalloc(wl, idx_d, ntok)
        if call > 0:   # the first call may commit the static array; later ones take nothing
            assert took == 0, f"second call took {took} bytes of device memory"
        assert err == 0
        assert np.array_equal(recv, recv_ref)
        for r in range(R):
            assert np.array_equal(src[r, :recv[r]], src_ref[r, :recv[r]]), r
        # slot_map is the inverse of src_token_pos: row i of rank r holds (s, t)
        for s in range(R):
            for r in range(R):
                sl = slot[s, :ntok[s], r]
                sent = sl >= 0
                assert np.array_equal(src[r, sl[sent]], s * R * T + np.nonzero(sent)[0])
                assert np.all(sl[~sent] == -1)
                owned = ((idx[s, :ntok[s]] >= 0) & (idx[s, :ntok[s]] // wl.experts_per_rank == r))
                assert np.array_equal(sent, owned.any(-1))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    idx_d = torch.zeros((8, 8193, 8), dtype=torch.int32, device="cuda")
    out = torch.empty(8 * 8 * 8193 * 8, dtype=torch.int32, device="cuda")
    with pytest.raises(EpError) as ei:
        E.ep_routing_layout_noalloc(8, 8193, 32, 8, idx_d.data_ptr(), [1] * 8, out.data_ptr(),
                                    out.data_ptr(), out.data_ptr(), None,
                                    torch.cuda.current_stream().cuda_stream)
    assert ei.value.status == E.EP_ERR_INVALID_ARG
    assert "EP_NOALLOC_MAX_TOKENS" in str(ei.value)
