"""GPU parity: libep (through its C ABI) against the CPU oracle, bit for bit.

Workload shapes follow the MORI-EP User Guide's DeepSeek-V3 example and
benchmark tables; the small variants keep several 256-token chunks and a
ragged tail so every tile path runs. The full-size workloads are compared
whole (every row, scale and token); the forced-kernel variants at full size
compare all routing metadata and a seeded sample of rows and tokens.
"""
import json

import numpy as np
import pytest
import torch

import oracle
from combine_route_layout_gb300 import EpDispatchCombineOp, EpError
from combine_route_layout_gb300 import ep as E
from gen import WORKLOADS, make_expert_outputs
from ep_harness import (DEV, Inputs, bits16, check_route, host, make_config, oracle_quant,
                        oracle_rows_to_pool, pool_to_ranks, sample_rows, sample_tokens, std_pcap,
                        std_pool_rows)

pytestmark = pytest.mark.gpu


def _out_bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) if a.dtype == np.float32 else a


def run_2d(wl, seed=None, ragged=False, full=True, nsample=192, cfg_over=None,
           y_dtype=torch.bfloat16, want_weights=True):
    cfg_over = dict(cfg_over or {})
    inp = Inputs(wl, seed, ragged)
    cfg = make_config(wl, combine_dtype=y_dtype, **cfg_over)
    op = EpDispatchCombineOp(cfg)
    R, T, H, Er = wl.world_size, wl.tokens_per_rank, wl.hidden, wl.experts_per_rank
    cap = R * T
    d_x, d_w, d_sc, d_idx, recv_d = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)
    torch.cuda.synchronize()
    op.sync()
    recv, src_pos, slot = check_route(inp, recv_d, op.get_dispatch_src_token_pos())
    quant = cfg.quant_type != "none"

    # weights and indices of every received row
    w_ref = oracle.place_rows(inp.w, inp.ntok, slot)
    idx_ref = oracle.place_rows(inp.idx, inp.ntok, slot)
    gw, gi = host(d_w), host(d_idx)
    for r in range(R):
        n = recv[r]
        assert np.array_equal(gw[r, :n].view(np.uint32), w_ref[r, :n].view(np.uint32)), r
        assert np.array_equal(gi[r, :n], idx_ref[r, :n]), r

    # payload (and FP8 scales)
    if full:
        xb = inp.x_bits()
        if quant:
            q, sc = oracle_quant(cfg, xb)
            x_ref, sc_ref = oracle.place_rows(q, inp.ntok, slot), oracle.place_rows(sc, inp.ntok, slot)
        else:
            x_ref, sc_ref = oracle.place_rows(xb, inp.ntok, slot), None
        gx = host(d_x)
        gsc = host(d_sc) if quant else None
        for r in range(R):
            n = recv[r]
            assert np.array_equal(gx[r, :n], x_ref[r, :n]), f"payload rank {r}"
            if quant:
                assert np.array_equal(gsc[r, :n].view(np.uint32), sc_ref[r, :n].view(np.uint32))
    else:
        rows = sample_rows(recv, nsample, seed=int(seed or 0))
        rr = np.array([r for r, _ in rows])
        ii = np.array([i for _, i in rows])
        st = np.array([divmod(int(src_pos[r, i]), cap) for r, i in rows])
        xb = inp.x_bits((st[:, 0], st[:, 1]))
        gx = host(d_x[torch.as_tensor(rr, device=DEV), torch.as_tensor(ii, device=DEV)])
        if quant:
            q, sc = oracle_quant(cfg, xb)
            gsc = host(d_sc[torch.as_tensor(rr, device=DEV), torch.as_tensor(ii, device=DEV)])
            assert np.array_equal(gx, q), "sampled FP8 codes"
            assert np.array_equal(gsc.view(np.uint32), sc.view(np.uint32)), "sampled scales"
        else:
            assert np.array_equal(gx, xb), "sampled payload"

    # combine
    if wl.expert_output == "identity":
        assert not quant
        y_d = d_x
        y_ref = x_ref if full else None
    else:
        y_d = make_expert_outputs(wl, cap, seed, device=DEV, dtype=y_dtype)
        y_ref = host(y_d)
    od = "fp32" if cfg.combine_out_dtype == torch.float32 else "bf16"
    out_d, outw_d = op.combine(y_d, d_w, inp.idx_d, call_reset=True, want_weights=want_weights)
    op.sync()
    go = host(out_d)
    if y_ref is None:
        y_ref = host(y_d)
    if full:
        out_ref, outw_ref = oracle.combine(y_ref, inp.idx, inp.ntok, slot, Er, w_recv=w_ref,
                                           weighted=cfg.weighted_combine, out_dtype=od)
        gow = host(outw_d) if outw_d is not None else None
        for s in range(R):
            n = inp.ntok[s]
            assert np.array_equal(_out_bits(go[s, :n]), _out_bits(out_ref[s, :n])), f"combine rank {s}"
            if gow is not None:
                assert np.array_equal(gow[s, :n].view(np.uint32), outw_ref[s, :n].view(np.uint32))
    else:
        toks = sample_tokens(wl, inp.ntok, 4 * nsample, seed=int(seed or 0))
        out_ref, outw_ref = oracle.combine_tokens(toks, y_ref, inp.idx, slot, Er, w_recv=w_ref,
                                                  weighted=cfg.weighted_combine, out_dtype=od)
        s_, t_ = toks // T, toks % T
        got = go[s_, t_]
        assert np.array_equal(_out_bits(got), _out_bits(out_ref)), "sampled combine"
        if outw_d is not None:
            gow = host(outw_d)[s_, t_]
            assert np.array_equal(gow.view(np.uint32), outw_ref.view(np.uint32))
    return op


# ------------------------------------------------------------- small shapes

@pytest.mark.parametrize("seed,ragged", [(0, False), (1, True), (2, False)])
def test_tiny_identity(seed, ragged):
    run_2d(WORKLOADS["tiny"], seed=seed, ragged=ragged)


@pytest.mark.parametrize("impl", ["auto", "vector"])
def test_ds_v3_latency_full(impl):
    """The decode shape whole, with the automatic and the forced-vector
    dispatch choice."""
    run_2d(WORKLOADS["ds_v3_latency"], cfg_over=dict(dispatch_impl=impl))


@pytest.mark.parametrize("seed", [1, 2])
def test_ds_v3_latency_seeds(seed):
    run_2d(WORKLOADS["ds_v3_latency"], seed=seed, ragged=True)


def test_throughput_shape_small_ragged():
    wl = WORKLOADS["ds_v3_throughput"].with_(tokens_per_rank=300)
    run_2d(wl, seed=3, ragged=True)


def test_mid_shape_small_ragged():
    wl = WORKLOADS["mid_masked"].with_(tokens_per_rank=600)
    run_2d(wl, seed=4, ragged=True)


@pytest.mark.parametrize("over", [
    dict(world_size=1, experts_per_rank=8, topk=4),
    dict(world_size=32, experts_per_rank=2, topk=8, tokens_per_rank=40),
    dict(world_size=4, experts_per_rank=3, topk=1),
    dict(world_size=8, experts_per_rank=4, topk=16),
    dict(hidden=384),
    dict(hidden=264),
    dict(mask_prob=1.0),
    dict(mask_prob=0.6, tokens_per_rank=257),
])
def test_edge_shapes(over):
    wl = WORKLOADS["tiny"].with_(**over)
    run_2d(wl, seed=5, ragged=True)


def test_empty_ranks():
    wl = WORKLOADS["tiny"]
    inp_ntok = np.zeros(wl.world_size, np.int32)
    inp = Inputs(wl, 0)
    op = EpDispatchCombineOp(make_config(wl))
    d_x, d_w, _, _, recv = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp_ntok)
    out, _ = op.combine(d_x, d_w, None, call_reset=True)
    op.sync()
    assert int(recv.sum()) == 0


@pytest.mark.parametrize("yd,od", [(torch.float32, torch.float32), (torch.float32, torch.bfloat16),
                                   (torch.bfloat16, torch.bfloat16)])
def test_combine_dtypes(yd, od):
    wl = WORKLOADS["mid_masked"].with_(tokens_per_rank=100, hidden=512, expert_output="random")
    run_2d(wl, seed=6, ragged=True, y_dtype=yd, cfg_over=dict(combine_out_dtype=od))


@pytest.mark.parametrize("fp8", [False, True])
def test_weighted_2d_combine(fp8):
    wl = WORKLOADS["mid_masked"].with_(tokens_per_rank=130, hidden=1024, weighted=True,
                                       dispatch_dtype="fp8" if fp8 else "bf16")
    run_2d(wl, seed=7, ragged=True)


def test_fp8_passthrough_with_scales():
    """Dispatch carries already-quantised FP8 payloads and their scales
    ("Choosing an EP API and backend", EP paths table)."""
    wl = WORKLOADS["ds_v3_latency"].with_(tokens_per_rank=70, hidden=1024)
    R, T, H, k = wl.world_size, wl.tokens_per_rank, wl.hidden, wl.topk
    inp = Inputs(wl, 8, ragged=True)
    codes = torch.randint(0, 256, (R, T, H), dtype=torch.uint8, device=DEV)
    codes[codes == 0x7F] = 0
    codes[codes == 0xFF] = 0
    xq = codes.view(torch.float8_e4m3fn)
    scales = torch.rand((R, T, H // 128), device=DEV, dtype=torch.float32)
    cfg = make_config(wl, data_type=torch.float8_e4m3fn, quant_type="none", scale_dim=H // 128,
                      scale_type_size=4)
    op = EpDispatchCombineOp(cfg)
    d_x, d_w, d_sc, d_idx, recv_d = op.dispatch(xq, inp.w_d, scales, inp.idx_d, inp.ntok)
    op.sync()
    recv, src_pos, slot = check_route(inp, recv_d, op.get_dispatch_src_token_pos())
    x_ref = oracle.place_rows(host(codes), inp.ntok, slot)
    sc_ref = oracle.place_rows(host(scales), inp.ntok, slot)
    gx, gs = host(d_x), host(d_sc).view(np.float32)
    for r in range(R):
        n = recv[r]
        assert np.array_equal(gx[r, :n], x_ref[r, :n])
        assert np.array_equal(gs[r, :n].reshape(n, -1).view(np.uint32),
                              sc_ref[r, :n].view(np.uint32))
    op.reset()


# --------------------------------------------------------------- full sizes

@pytest.mark.slow
def test_ds_v3_throughput_full_size():
    """The 4096-token DeepSeek-V3 shape whole: every receive row's FP8 codes,
    block scales, weights and ids, all routing metadata, and every combined
    token and weight row against the oracle."""
    run_2d(WORKLOADS["ds_v3_throughput"], full=True)


@pytest.mark.slow
def test_mid_masked_full_size():
    """The mid-size masked workload whole (every row and token)."""
    run_2d(WORKLOADS["mid_masked"], full=True)


@pytest.mark.slow
def test_tiny_full_size_seed0():
    run_2d(WORKLOADS["tiny"])


# ------------------------------------------------------------ standard MoE

def _pool_y(wl, rows, seed, dtype=torch.bfloat16):
    """Stand-in expert outputs for every row of the packed pool, [rows, H]."""
    return make_expert_outputs(wl.with_(world_size=1), rows, seed, device=DEV, dtype=dtype)[0]


def run_std(wl, seed=None, ragged=False, full=True, nsample=256, cfg_over=None):
    cfg_over = dict(cfg_over or {})
    inp = Inputs(wl, seed, ragged)
    cfg = make_config(wl, standard_moe=True, **cfg_over)
    op = EpDispatchCombineOp(cfg)
    R, T, H, Er = wl.world_size, wl.tokens_per_rank, wl.hidden, wl.experts_per_rank
    v = op.dispatch_standard_moe(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)
    op.sync()
    assert op.pcap == std_pool_rows(wl) or cfg.max_packed_rows_per_rank > 0
    pcap = std_pcap(wl)                 # the oracle's per-rank capacity
    ref = oracle.std_layout(inp.idx, inp.ntok, Er, pcap)
    assert np.array_equal(host(v["packed_recv_count"]), ref["count"])
    assert np.array_equal(host(v["expert_offset"]), ref["seg_off"])
    assert np.array_equal(host(v["rank_rows"]), ref["rank_rows"])
    assert np.array_equal(host(v["packed_recv_layout_range"]), ref["layout_range"])
    base = host(v["rank_base"]).astype(np.int64)
    assert np.array_equal(base, np.concatenate([[0], np.cumsum(ref["rank_rows"])[:-1]]))
    gsi = host(v["packed_recv_src_info"])
    for r in range(R):
        n = ref["rank_rows"][r]
        assert np.array_equal(gsi[base[r]:base[r] + n], ref["src_info"][r, :n]), f"src_info rank {r}"
    quant = cfg.quant_type != "none"
    data = [(r, i) for r in range(R) for i in np.nonzero(ref["src_info"][r] >= 0)[0]]
    if not full:
        rng = np.random.default_rng(1)
        data = [data[j] for j in np.sort(rng.choice(len(data), size=min(len(data), 8 * nsample),
                                                    replace=False))]
    gi = torch.as_tensor(np.array([base[r] + i for r, i in data], np.int64), device=DEV)
    st = np.array([divmod(int(ref["src_info"][r, i]), R * T) for r, i in data])
    xb = inp.x_bits((st[:, 0], st[:, 1]))
    gx = host(v["packed_recv_x"][gi])
    if quant:
        q, sc = oracle_quant(cfg, xb)
        gsc = host(v["packed_recv_scales"][gi])
        assert np.array_equal(gx, q)
        assert np.array_equal(gsc.view(np.uint32), sc.view(np.uint32))
    else:
        assert np.array_equal(gx, xb), "packed payload"

    # combine_standard_moe on random expert outputs over the whole pool
    Y = _pool_y(wl, op.pcap, seed, dtype=cfg.combine_dtype)
    out_d = op.combine_standard_moe(Y, inp.w_d, inp.idx_d, call_reset=True)
    op.sync()
    od = "fp32" if cfg.combine_out_dtype == torch.float32 else "bf16"
    toks = (np.array([s * T + t for s in range(R) for t in range(int(inp.ntok[s]))], np.int64)
            if full else sample_tokens(wl, inp.ntok, 4 * nsample))
    # gather the rows the tokens use (oracle layout) into a compact Y
    rm = ref["row_map"].reshape(-1, wl.topk)[toks]
    used = np.unique(rm[rm >= 0])
    remap = np.full(R * pcap, -1, np.int64)
    remap[used] = np.arange(len(used))
    Ysub = host(Y[torch.as_tensor(oracle_rows_to_pool(used, base, pcap), device=DEV)])
    rm_sub = np.full((R * T, wl.topk), -1, np.int32)
    rm_sub[toks] = np.where(rm >= 0, remap[np.maximum(rm, 0)], -1)
    out_ref = oracle.std_combine_tokens(toks, Ysub, inp.idx, rm_sub.reshape(R, T, wl.topk), Er,
                                        w=inp.w, weighted=cfg.weighted_combine, out_dtype=od)
    got = host(out_d)[toks // T, toks % T]
    assert np.array_equal(_out_bits(got), _out_bits(out_ref)), "combine_standard_moe"
    return op


def test_skewed_std_small():
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(tokens_per_rank=300)
    run_std(wl, seed=1, ragged=True)


@pytest.mark.parametrize("over", [dict(router="uniform", mask_prob=0.2),
                                  dict(dispatch_dtype="fp8", tokens_per_rank=90),
                                  dict(weighted=False, combine_out_dtype="bf16"),
                                  dict(world_size=4, experts_per_rank=5, topk=3, hidden=384)])
def test_std_variants(over):
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(tokens_per_rank=200, hidden=1024).with_(**over)
    run_std(wl, seed=2, ragged=True)


@pytest.mark.slow
def test_skewed_std_full_size():
    """The Zipf-skewed standard-MoE workload whole: every packed row, the
    layout, and every token of the weighted f32 combine."""
    run_std(WORKLOADS["skewed_zipf_std_moe"], full=True)


# ------------------------------------------------------------- conversions

def run_convert(wl, seed, impl="auto", dtype=torch.bfloat16):
    """dispatch -> convert_dispatch_output -> convert_combine_input -> combine
    (and combine_standard_moe on the converted layout), every row against the
    oracle. impl picks the convert_combine_input kernel (combine phase)."""
    R, T, H, Er, k = wl.world_size, wl.tokens_per_rank, wl.hidden, wl.experts_per_rank, wl.topk
    inp = Inputs(wl, seed, ragged=True)
    cfg = make_config(wl, standard_moe=2, combine_dtype=dtype,
                      combine_out_dtype=torch.float32, weighted_combine=False)
    op = EpDispatchCombineOp(cfg)
    op.set_launch_config(E.EP_PHASE_COMBINE, impl)
    d_x, d_w, _, d_idx, recv_d = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)
    px, pcount, psrc, prange = op.convert_dispatch_output(d_x, d_idx)
    op.sync()
    assert op.pcap == std_pool_rows(wl)
    pcap = std_pcap(wl)
    ref = oracle.std_dispatch(inp.x_bits(), inp.idx, inp.ntok, Er, pcap)
    assert np.array_equal(host(pcount), ref["count"])
    assert np.array_equal(host(prange), ref["layout_range"])
    base = np.concatenate([[0], np.cumsum(ref["rank_rows"])[:-1]]).astype(np.int64)
    gsi = pool_to_ranks(host(psrc), base, ref["rank_rows"], pcap, fill=-2)
    gx = pool_to_ranks(host(px), base, ref["rank_rows"], pcap)
    for r in range(R):
        n = ref["rank_rows"][r]
        assert np.array_equal(gsi[r, :n], ref["src_info"][r, :n])
        used = ref["src_info"][r, :n] >= 0
        assert np.array_equal(gx[r, :n][used], ref["x"][r, :n][used])

    recv, src_pos, slot = oracle.route(inp.idx, inp.ntok, Er)
    Y = _pool_y(wl, op.pcap, seed, dtype=dtype)
    y2d = op.convert_combine_input(Y, psrc, prange)
    op.sync()
    Yh = pool_to_ranks(host(Y), base, ref["rank_rows"], pcap)
    y2d_ref = oracle.convert_combine_input(Yh, recv, src_pos, inp.idx, ref["row_map"], Er,
                                           out_dtype="bf16" if dtype == torch.bfloat16 else "fp32")
    gy = host(y2d)
    for r in range(R):
        assert np.array_equal(gy[r, :recv[r]], y2d_ref[r, :recv[r]]), f"convert_combine_input {r}"
    out_d, _ = op.combine(y2d, d_w, None)
    out_ref, _ = oracle.combine(y2d_ref, inp.idx, inp.ntok, slot, Er, out_dtype="fp32")
    go = host(out_d)
    for s in range(R):
        n = inp.ntok[s]
        assert np.array_equal(go[s, :n].view(np.uint32), out_ref[s, :n].view(np.uint32))
    # the packed layout from the conversion also feeds combine_standard_moe
    out_std = op.combine_standard_moe(Y, None, None, call_reset=True)
    ref_std = oracle.std_combine(Yh, inp.idx, inp.ntok, ref["row_map"], Er, weighted=False,
                                 out_dtype="fp32")
    gs = host(out_std)
    for s in range(R):
        n = inp.ntok[s]
        assert np.array_equal(gs[s, :n].view(np.uint32), ref_std[s, :n].view(np.uint32))


@pytest.mark.parametrize("impl,hidden,dtype,seed", [
    ("auto", 1024, torch.bfloat16, 3),
    ("vector", 1024, torch.bfloat16, 3),
    ("bulk", 1056, torch.bfloat16, 4),     # a ragged last column chunk
    ("vector", 1056, torch.bfloat16, 4),
    ("bulk", 2080, torch.float32, 5),      # f32 rows, three chunks
    ("vector", 2080, torch.float32, 5),
])
def test_convert_round_trip(impl, hidden, dtype, seed):
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(tokens_per_rank=260, hidden=hidden, mask_prob=0.1)
    run_convert(wl, seed, impl, dtype)


def test_convert_round_trip_top2_sixteen_ranks():
    """Few slots per token over many ranks: many receive rows with one
    packed row each and rows with none on a rank."""
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(world_size=16, experts_per_rank=4, topk=2,
                                               tokens_per_rank=150, hidden=512, mask_prob=0.2)
    run_convert(wl, 6, "bulk")


def test_convert_round_trip_top12():
    """More than 8 slots per token: convert_combine_input falls back from the
    bulk ring (8 rows per unit) to the vector kernel under AUTO."""
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(topk=12, tokens_per_rank=120, hidden=768,
                                               mask_prob=0.1)
    run_convert(wl, 8, "auto")


@pytest.mark.slow
def test_convert_full_size():
    """The skewed shape whole (8 x 4096 tokens, H 7168) through both
    conversions, every receive row and packed row compared."""
    run_convert(WORKLOADS["skewed_zipf_std_moe"], 7, "auto")


# ------------------------------------------------------------ error flags

def test_invalid_index_sets_error_flag():
    wl = WORKLOADS["tiny"]
    inp = Inputs(wl, 0)
    idx = inp.idx.copy()
    idx[2, 3, 1] = wl.num_experts          # out of range
    op = EpDispatchCombineOp(make_config(wl))
    op.dispatch(inp.x, inp.w_d, None, torch.from_numpy(idx).to(DEV), inp.ntok)
    with pytest.raises(EpError) as ei:
        op.sync()
    assert ei.value.status == E.EP_ERR_INVALID_INDEX
    op.sync()                               # flag cleared
    op.reset()


def test_bounded_wait_timeout_is_reported_and_the_handle_stays_usable():
    """Failure detection without a GPU fault: a kernel waits on a barrier that
    nothing completes; its bounded wait gives up after about a second and
    sets the timeout flag, ep_sync reports EP_ERR_TIMEOUT once, and the same
    handle then dispatches correctly."""
    wl = WORKLOADS["tiny"]
    inp = Inputs(wl, 0)
    op = EpDispatchCombineOp(make_config(wl))
    E.ep_selftest_bounded_wait(op._handle, torch.cuda.current_stream().cuda_stream)
    with pytest.raises(EpError) as ei:
        op.sync()
    assert ei.value.status == E.EP_ERR_TIMEOUT
    op.sync()                               # flag cleared
    d_x, _, _, _, recv_d = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)
    op.sync()
    recv, src_pos, slot = check_route(inp, recv_d, op.get_dispatch_src_token_pos())
    x_ref = oracle.place_rows(inp.x_bits(), inp.ntok, slot)
    gx = host(d_x)
    for r in range(wl.world_size):
        assert np.array_equal(gx[r, :recv[r]], x_ref[r, :recv[r]])
    op.reset()


def test_std_capacity_overflow_flagged():
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(tokens_per_rank=100, hidden=256)
    inp = Inputs(wl, 0)
    op = EpDispatchCombineOp(make_config(wl, standard_moe=True, max_packed_rows_per_rank=256))
    op.dispatch_standard_moe(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)
    with pytest.raises(EpError) as ei:
        op.sync()
    assert ei.value.status == E.EP_ERR_CAPACITY
    op.reset()


def test_std_duplicate_ids_flagged():
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(tokens_per_rank=20, hidden=256)
    inp = Inputs(wl, 0)
    idx = inp.idx.copy()
    idx[1, 2, 3] = idx[1, 2, 0]
    op = EpDispatchCombineOp(make_config(wl, standard_moe=True))
    op.dispatch_standard_moe(inp.x, inp.w_d, None, torch.from_numpy(idx).to(DEV), inp.ntok)
    with pytest.raises(EpError) as ei:
        op.sync()
    assert ei.value.status == E.EP_ERR_INVALID_INDEX
    op.reset()


# ------------------------------------------- invariants and repeated rounds

def test_identity_invariant_bf16_dispatch():
    """Identity experts: combine returns the token times its number of
    distinct destination ranks (exact in f32 since |D| <= 8)."""
    wl = WORKLOADS["mid_masked"].with_(tokens_per_rank=512, combine_out_dtype="fp32")
    inp = Inputs(wl, 9, ragged=True)
    op = EpDispatchCombineOp(make_config(wl))
    d_x, d_w, _, _, _ = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)
    out, _ = op.combine(d_x, d_w, None, call_reset=True)
    owners = torch.where(inp.idx_d >= 0, inp.idx_d // wl.experts_per_rank, -1)
    nD = torch.zeros(owners.shape[:2], dtype=torch.float32, device=DEV)
    for r in range(wl.world_size):
        nD += (owners == r).any(-1).float()
    exp = inp.x.float() * nD[..., None]
    for s in range(wl.world_size):
        n = int(inp.ntok[s])
        assert torch.equal(out[s, :n], exp[s, :n])


def test_repeated_rounds_random_shapes():
    """500 dispatch -> combine -> reset rounds with changing token counts on
    one handle (the tuning guide's 500-round verification)."""
    wl = WORKLOADS["tiny"].with_(tokens_per_rank=64, hidden=256)
    inp = Inputs(wl, 0)
    op = EpDispatchCombineOp(make_config(wl))
    rng = np.random.default_rng(0)
    R, T = wl.world_size, wl.tokens_per_rank
    owners = torch.where(inp.idx_d >= 0, inp.idx_d // wl.experts_per_rank, -1)
    nD = torch.zeros(owners.shape[:2], dtype=torch.float32, device=DEV)
    for r in range(R):
        nD += (owners == r).any(-1).float()
    exp = inp.x.float() * nD[..., None]
    for it in range(500):
        ntok = rng.integers(0, T + 1, size=R).astype(np.int32)
        d_x, d_w, _, _, recv = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, ntok)
        out, _ = op.combine(d_x, d_w, None, call_reset=True)
        if it % 50 == 0:
            op.sync()
            for s in range(R):
                assert torch.equal(out[s, :ntok[s]], exp[s, :ntok[s]].to(out.dtype))
    op.sync()


def test_cuda_graph_capture_replay():
    """Dispatch + combine make no host synchronisation, so they capture into a
    CUDA graph and replay with the same results."""
    wl = WORKLOADS["ds_v3_latency"].with_(tokens_per_rank=64)
    inp = Inputs(wl, 0)
    op = EpDispatchCombineOp(make_config(wl))
    cap = wl.world_size * wl.tokens_per_rank
    y = make_expert_outputs(wl, cap, 0, device=DEV)
    out = torch.empty((wl.world_size, wl.tokens_per_rank, wl.hidden), dtype=torch.bfloat16,
                      device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, None)   # warm-up (first-call set-up)
        op.combine(y, d[1], None, out=out, call_reset=True)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        d = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, None)
        op.combine(y, d[1], None, out=out, call_reset=True)
    for _ in range(3):
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_fp8_quotients_on_e4m3_midpoints():
    """Blocks whose amax is 448*c (so the scale is exactly c) and whose other
    elements are c times an E4M3 midpoint (or one bf16 step away): x / scale
    lands exactly on a rounding boundary, where the reciprocal-multiply fast
    path must hand over to the IEEE division. Codes must still match the
    oracle bit for bit."""
    wl = WORKLOADS["ds_v3_latency"].with_(tokens_per_rank=48, hidden=1024)
    R, T, H = wl.world_size, wl.tokens_per_rank, wl.hidden
    codes = np.array([c for c in range(0x7F) if c != 0x7F], np.uint8)
    vals = oracle.e4m3_to_f32(codes).astype(np.float64)
    mids = np.concatenate([(vals[1:] + vals[:-1]) / 2, vals])
    mults = np.array([3, 5, 7, 0.75, 1.5, 2.5, 3.5, 0.375, 1.25, 96, 0.0234375, 6], np.float64)
    rng = np.random.default_rng(11)
    x = np.empty((R, T, H), np.float32)
    for s in range(R):
        for t in range(T):
            for b in range(H // 128):
                c = mults[rng.integers(len(mults))]
                blk = c * rng.choice(mids, size=128) * rng.choice([-1.0, 1.0], size=128)
                blk[rng.integers(128)] = 448.0 * c * rng.choice([-1.0, 1.0])
                x[s, t, b * 128:(b + 1) * 128] = blk
    xb = torch.from_numpy(x).to(torch.bfloat16)
    nudge = rng.random(xb.shape) < 0.2          # some elements one bf16 step off the midpoint
    xi = xb.view(torch.int16)
    xi[torch.from_numpy(nudge)] += torch.from_numpy(rng.choice([-1, 1], size=int(nudge.sum()))
                                                    ).to(torch.int16)
    inp = Inputs(wl, 0)
    inp.x = xb.to(DEV)
    cfg = make_config(wl)
    op = EpDispatchCombineOp(cfg)
    d_x, d_w, d_sc, _, recv_d = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)
    op.sync()
    recv, src_pos, slot = check_route(inp, recv_d, op.get_dispatch_src_token_pos())
    q, sc = oracle.quant_tokens(bits16(xb))
    x_ref, sc_ref = oracle.place_rows(q, inp.ntok, slot), oracle.place_rows(sc, inp.ntok, slot)
    gx, gsc = host(d_x), host(d_sc)
    for r in range(R):
        n = recv[r]
        assert np.array_equal(gsc[r, :n].view(np.uint32), sc_ref[r, :n].view(np.uint32))
        assert np.array_equal(gx[r, :n], x_ref[r, :n]), f"codes rank {r}"
    op.reset()


# ------------------------------------------- bulk-copy (TMA) combine kernels

@pytest.mark.parametrize("name,over,seed,ragged", [
    ("tiny", {}, 0, False),
    ("tiny", {}, 1, True),
    ("ds_v3_latency", {}, 0, False),
    ("ds_v3_throughput", dict(tokens_per_rank=300), 3, True),
    ("mid_masked", dict(tokens_per_rank=600), 4, True),
    ("mid_masked", dict(tokens_per_rank=130, hidden=1032, weighted=True), 7, True),
    ("tiny", dict(hidden=264), 5, True),
    ("tiny", dict(world_size=32, experts_per_rank=2, topk=8, tokens_per_rank=40), 5, True),
])
def test_bulk_combine_2d(name, over, seed, ragged):
    run_2d(WORKLOADS[name].with_(**over), seed=seed, ragged=ragged,
           cfg_over=dict(combine_impl="bulk"))


@pytest.mark.parametrize("yd,od", [(torch.float32, torch.float32), (torch.float32, torch.bfloat16),
                                   (torch.bfloat16, torch.float32)])
def test_bulk_combine_dtypes(yd, od):
    wl = WORKLOADS["mid_masked"].with_(tokens_per_rank=100, hidden=2056)
    run_2d(wl, seed=6, ragged=True, y_dtype=yd, cfg_over=dict(combine_out_dtype=od,
                                                              combine_impl="bulk"))


@pytest.mark.parametrize("over", [dict(tokens_per_rank=300),
                                  dict(router="uniform", mask_prob=0.2, tokens_per_rank=200),
                                  dict(weighted=False, combine_out_dtype="bf16", hidden=1032),
                                  dict(world_size=4, experts_per_rank=5, topk=3, hidden=384)])
def test_bulk_combine_std(over):
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(hidden=1024).with_(**over)
    run_std(wl, seed=2, ragged=True, cfg_over=dict(combine_impl="bulk"))


@pytest.mark.slow
def test_bulk_combine_full_size():
    run_2d(WORKLOADS["ds_v3_throughput"], full=False, cfg_over=dict(combine_impl="bulk"))
    run_std(WORKLOADS["skewed_zipf_std_moe"], full=False, cfg_over=dict(combine_impl="bulk"))


# ------------------------------------------------------------- codec sweeps

@pytest.mark.parametrize("impl", ["auto", "vector"])
def test_gpu_e4m3_codes_for_every_bf16_value(impl):
    """Every finite bf16 value with |x| <= 448 passes through the FP8 dispatch
    with a block scale of exactly 1 (each block holds 448), so the codes are
    E4M3(x) and must equal the oracle's encoder."""
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = (allb.astype(np.uint32) << 16).view(np.float32)
    keep = np.isfinite(vals) & (np.abs(vals) <= 448.0)
    bits = allb[keep]
    per_block = 127
    nblk = -(-len(bits) // per_block)
    H = 1024
    tokens = -(-nblk // (H // 128))
    R, T = 1, tokens
    x = np.zeros((R, T, H), np.uint16)
    flat = x.reshape(-1, 128)
    flat[:, 127] = 0x43E0                        # bf16 448.0 in every block: scale 1
    for b in range(nblk):
        chunk = bits[b * per_block:(b + 1) * per_block]
        flat[b, :len(chunk)] = chunk
    wl = WORKLOADS["tiny"].with_(world_size=R, experts_per_rank=1, topk=1, tokens_per_rank=T,
                                 hidden=H, dispatch_dtype="fp8", expert_output="random")
    idx = np.zeros((R, T, 1), np.int32)
    w = np.ones((R, T, 1), np.float32)
    op = EpDispatchCombineOp(make_config(wl, dispatch_impl=impl))
    xd = torch.from_numpy(x.view(np.int16)).to(DEV).view(torch.bfloat16)
    d_x, _, d_sc, _, recv = op.dispatch(xd, torch.from_numpy(w).to(DEV), None,
                                         torch.from_numpy(idx).to(DEV), [T])
    op.sync()
    q_ref, sc_ref = oracle.quant_tokens(x)
    assert np.all(sc_ref == 1.0)
    assert np.array_equal(host(d_x)[0, :T], q_ref[0])
    op.reset()


def test_gpu_bf16_rounding_sweep():
    """A million random f32 bit patterns through an f32-in / bf16-out combine
    with one copy per token: the output is the GPU's bf16 rounding of +0 + y,
    compared with the oracle's."""
    rng = np.random.default_rng(3)
    H, T = 1024, 1024
    u = rng.integers(0, 2**32, size=(T, H), dtype=np.uint64).astype(np.uint32)
    u[:, :64] = (rng.integers(0, 2**16, size=(T, 64), dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    y = u.view(np.float32)
    y[~np.isfinite(y)] = 1.0
    wl = WORKLOADS["tiny"].with_(world_size=1, experts_per_rank=1, topk=1, tokens_per_rank=T,
                                 hidden=H, combine_out_dtype="bf16")
    idx = np.zeros((1, T, 1), np.int32)
    w = np.ones((1, T, 1), np.float32)
    op = EpDispatchCombineOp(make_config(wl, combine_dtype=torch.float32))
    x = torch.zeros((1, T, H), dtype=torch.bfloat16, device=DEV)
    d = op.dispatch(x, torch.from_numpy(w).to(DEV), None, torch.from_numpy(idx).to(DEV), [T])
    yd = torch.from_numpy(y.reshape(1, T, H).copy()).to(DEV)
    out, _ = op.combine(yd, d[1], None, call_reset=True)
    op.sync()
    recv, src_pos, slot = oracle.route(idx, np.array([T], np.int32), 1)
    ref, _ = oracle.combine(y.reshape(1, T, H), idx, np.array([T], np.int32), slot, 1,
                            out_dtype="bf16")
    assert np.array_equal(host(out), ref)


def test_registered_combine_input_buffer_zero_copy():
    """Zero-copy mode (use_external_inp_buf = 0): experts write into the
    library's registered buffer and combine reads it in place."""
    wl = WORKLOADS["ds_v3_latency"].with_(tokens_per_rank=100)
    R, T = wl.world_size, wl.tokens_per_rank
    inp = Inputs(wl, 1, ragged=True)
    op = EpDispatchCombineOp(make_config(wl, use_external_inp_buf=False))
    d_x, d_w, _, _, recv_d = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)
    buf = op.get_registered_combine_input_buffer()
    y = make_expert_outputs(wl, R * T, 1, device=DEV)
    buf.copy_(y)
    out, outw = op.combine(None, d_w, None, call_reset=True)
    op.sync()
    recv, src_pos, slot = oracle.route(inp.idx, inp.ntok, wl.experts_per_rank)
    w_ref = oracle.place_rows(inp.w, inp.ntok, slot)
    ref, ref_w = oracle.combine(host(y), inp.idx, inp.ntok, slot, wl.experts_per_rank,
                                w_recv=w_ref, out_dtype="bf16")
    go, gw = host(out), host(outw)
    for s in range(R):
        n = inp.ntok[s]
        assert np.array_equal(go[s, :n], ref[s, :n])
        assert np.array_equal(gw[s, :n].view(np.uint32), ref_w[s, :n].view(np.uint32))


# ------------------------------------------ bulk-copy (TMA) dispatch kernels

@pytest.mark.parametrize("name,over,seed,ragged", [
    ("tiny", {}, 0, False),
    ("tiny", {}, 1, True),
    ("mid_masked", dict(tokens_per_rank=600), 4, True),
    ("mid_masked", dict(tokens_per_rank=300, hidden=1032, mask_prob=0.9), 2, True),
    ("tiny", dict(world_size=32, experts_per_rank=2, topk=8, tokens_per_rank=40), 5, True),
    ("tiny", dict(world_size=1, experts_per_rank=8, topk=4), 5, True),
])
def test_bulk_dispatch_2d(name, over, seed, ragged):
    run_2d(WORKLOADS[name].with_(**over), seed=seed, ragged=ragged,
           cfg_over=dict(dispatch_impl="bulk", combine_impl="bulk"))


@pytest.mark.parametrize("over", [dict(tokens_per_rank=300),
                                  dict(router="uniform", mask_prob=0.2, tokens_per_rank=200),
                                  dict(world_size=4, experts_per_rank=5, topk=3, hidden=384)])
def test_bulk_dispatch_std(over):
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(hidden=1024).with_(**over)
    run_std(wl, seed=2, ragged=True, cfg_over=dict(dispatch_impl="bulk"))


def test_bulk_dispatch_fp8_passthrough_with_scales():
    wl = WORKLOADS["ds_v3_latency"].with_(tokens_per_rank=70, hidden=1024)
    R, T, H = wl.world_size, wl.tokens_per_rank, wl.hidden
    inp = Inputs(wl, 8, ragged=True)
    codes = torch.randint(0, 126, (R, T, H), dtype=torch.uint8, device=DEV)
    scales = torch.rand((R, T, H // 128), device=DEV, dtype=torch.float32)
    cfg = make_config(wl, data_type=torch.float8_e4m3fn, quant_type="none", scale_dim=H // 128,
                      scale_type_size=4, dispatch_impl="bulk")
    op = EpDispatchCombineOp(cfg)
    d_x, d_w, d_sc, d_idx, recv_d = op.dispatch(codes.view(torch.float8_e4m3fn), inp.w_d, scales,
                                                inp.idx_d, inp.ntok)
    op.sync()
    recv, src_pos, slot = check_route(inp, recv_d, op.get_dispatch_src_token_pos())
    x_ref = oracle.place_rows(host(codes), inp.ntok, slot)
    sc_ref = oracle.place_rows(host(scales), inp.ntok, slot)
    w_ref = oracle.place_rows(inp.w, inp.ntok, slot)
    gx, gs, gw = host(d_x), host(d_sc).view(np.float32), host(d_w)
    for r in range(R):
        n = recv[r]
        assert np.array_equal(gx[r, :n], x_ref[r, :n])
        assert np.array_equal(gs[r, :n].reshape(n, -1).view(np.uint32), sc_ref[r, :n].view(np.uint32))
        assert np.array_equal(gw[r, :n].view(np.uint32), w_ref[r, :n].view(np.uint32))
    op.reset()


@pytest.mark.slow
def test_bulk_dispatch_full_size():
    run_2d(WORKLOADS["mid_masked"], full=False, cfg_over=dict(dispatch_impl="bulk"))
    run_std(WORKLOADS["skewed_zipf_std_moe"], full=False, cfg_over=dict(dispatch_impl="bulk"))


# --------------------------------------------------------------- FP4 dispatch

@pytest.mark.parametrize("impl", ["auto", "vector"])
@pytest.mark.parametrize("over,seed", [(dict(), 0), (dict(tokens_per_rank=300, hidden=1056), 1),
                                       (dict(tokens_per_rank=70, hidden=224), 2)])
def test_fp4_dispatch(over, seed, impl):
    """FP4 E2M1 block-32 quantisation in dispatch: codes, nibble order and
    scales bit-exact against the oracle (2D layout), automatic and forced-vector
    dispatch choice."""
    wl = WORKLOADS["ds_v3_latency"].with_(dispatch_dtype="fp4").with_(**over)
    run_2d(wl, seed=seed, ragged=bool(seed), cfg_over=dict(dispatch_impl=impl))


def test_fp4_dispatch_standard_moe():
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(tokens_per_rank=150, hidden=1024,
                                               dispatch_dtype="fp4")
    run_std(wl, seed=3, ragged=True)


def test_fp4_quant_signed_zero_blocks():
    wl = WORKLOADS["ds_v3_latency"].with_(tokens_per_rank=8, hidden=256, dispatch_dtype="fp4")
    inp = Inputs(wl, 4)
    x = inp.x.clone()
    x[0, 0, :32] = 0.0
    x[0, 1, 32:64] = -0.0
    x[1, 2, :32] = torch.tensor(1e-38).to(torch.bfloat16)
    inp.x = x
    op = EpDispatchCombineOp(make_config(wl))
    d_x, _, d_sc, _, recv_d = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)
    op.sync()
    recv, src_pos, slot = check_route(inp, recv_d, op.get_dispatch_src_token_pos())
    q, sc = oracle.quant_tokens_fp4(bits16(x))
    x_ref, sc_ref = oracle.place_rows(q, inp.ntok, slot), oracle.place_rows(sc, inp.ntok, slot)
    gx, gs = host(d_x), host(d_sc)
    for r in range(wl.world_size):
        n = recv[r]
        assert np.array_equal(gx[r, :n], x_ref[r, :n])
        assert np.array_equal(gs[r, :n].view(np.uint32), sc_ref[r, :n].view(np.uint32))
    op.reset()


def test_fp4_quotients_on_e2m1_midpoints():
    """As the E4M3 midpoint test, for FP4: blocks of 32 with amax 6*c, the
    other elements c times an E2M1 midpoint (0.25 sits on a binade start) or
    one bf16 step away."""
    wl = WORKLOADS["ds_v3_latency"].with_(tokens_per_rank=40, hidden=1024, dispatch_dtype="fp4")
    R, T, H = wl.world_size, wl.tokens_per_rank, wl.hidden
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    mids = np.concatenate([(mags[1:] + mags[:-1]) / 2, mags])
    mults = np.array([3, 5, 7, 0.75, 1.5, 2.5, 3.5, 0.375, 1.25, 96, 0.0234375, 6], np.float64)
    rng = np.random.default_rng(21)
    x = np.empty((R, T, H), np.float32)
    for s in range(R):
        for t in range(T):
            for b in range(H // 32):
                c = mults[rng.integers(len(mults))]
                blk = c * rng.choice(mids, size=32) * rng.choice([-1.0, 1.0], size=32)
                blk[rng.integers(32)] = 6.0 * c * rng.choice([-1.0, 1.0])
                x[s, t, b * 32:(b + 1) * 32] = blk
    xb = torch.from_numpy(x).to(torch.bfloat16)
    nudge = rng.random(xb.shape) < 0.2
    xi = xb.view(torch.int16)
    xi[torch.from_numpy(nudge)] += torch.from_numpy(rng.choice([-1, 1], size=int(nudge.sum()))
                                                    ).to(torch.int16)
    inp = Inputs(wl, 0)
    inp.x = xb.to(DEV)
    op = EpDispatchCombineOp(make_config(wl))
    d_x, d_w, d_sc, _, recv_d = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)
    op.sync()
    recv, src_pos, slot = check_route(inp, recv_d, op.get_dispatch_src_token_pos())
    q, sc = oracle.quant_tokens_fp4(bits16(xb))
    x_ref, sc_ref = oracle.place_rows(q, inp.ntok, slot), oracle.place_rows(sc, inp.ntok, slot)
    gx, gsc = host(d_x), host(d_sc)
    for r in range(R):
        n = recv[r]
        assert np.array_equal(gsc[r, :n].view(np.uint32), sc_ref[r, :n].view(np.uint32))
        assert np.array_equal(gx[r, :n], x_ref[r, :n]), f"codes rank {r}"
    op.reset()


def test_cuda_graph_replay_bulk_paths():
    """Graph capture and replay with the bulk-copy dispatch and combine (chosen
    automatically from 8192 tokens on), compared with the oracle."""
    wl = WORKLOADS["mid_masked"].with_(tokens_per_rank=1024, hidden=1024)
    R, T = wl.world_size, wl.tokens_per_rank
    inp = Inputs(wl, 2)
    op = EpDispatchCombineOp(make_config(wl))
    y = make_expert_outputs(wl, R * T, 2, device=DEV)
    out = torch.empty((R, T, wl.hidden), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, None)
        op.combine(y, d[1], None, out=out, call_reset=True)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        d = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, None)
        op.combine(y, d[1], None, out=out, call_reset=True)
    out.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    op.sync()
    recv, src_pos, slot = oracle.route(inp.idx, inp.ntok, wl.experts_per_rank)
    ref, _ = oracle.combine(host(y), inp.idx, inp.ntok, slot, wl.experts_per_rank, out_dtype="bf16")
    assert np.array_equal(host(out), ref)


# ----------------------------------------------------------- more dtypes

def test_fp32_input_copy_dispatch():
    """f32 tokens pass through dispatch bit for bit (copy mode), vector and bulk kernels."""
    wl = WORKLOADS["tiny"].with_(tokens_per_rank=300, hidden=520)
    R, T, H = wl.world_size, wl.tokens_per_rank, wl.hidden
    inp = Inputs(wl, 3, ragged=True)
    x = torch.randn((R, T, H), device=DEV, dtype=torch.float32)
    for impl in ("vector", "bulk"):
        op = EpDispatchCombineOp(make_config(wl, data_type=torch.float32, dispatch_impl=impl))
        d_x, d_w, _, d_idx, recv_d = op.dispatch(x, inp.w_d, None, inp.idx_d, inp.ntok)
        op.sync()
        recv, src_pos, slot = check_route(inp, recv_d, op.get_dispatch_src_token_pos())
        ref = oracle.place_rows(host(x), inp.ntok, slot)
        gx = host(d_x)
        for r in range(R):
            assert np.array_equal(gx[r, :recv[r]].view(np.uint32), ref[r, :recv[r]].view(np.uint32))
        op.reset()


def test_fp4_passthrough_with_scales():
    """Pre-quantised FP4 payloads (two E2M1 codes per byte) and their scales
    pass through dispatch unchanged."""
    fp4 = getattr(torch, "float4_e2m1fn_x2", None)
    if fp4 is None:
        pytest.skip("torch has no packed FP4 dtype")
    wl = WORKLOADS["ds_v3_latency"].with_(tokens_per_rank=70, hidden=1024)
    R, T, H = wl.world_size, wl.tokens_per_rank, wl.hidden
    inp = Inputs(wl, 8, ragged=True)
    packed = torch.randint(0, 256, (R, T, H // 2), dtype=torch.uint8, device=DEV)
    scales = torch.rand((R, T, H // 32), device=DEV, dtype=torch.float32)
    op = EpDispatchCombineOp(make_config(wl, data_type=fp4, quant_type="none",
                                         scale_dim=H // 32, scale_type_size=4))
    d_x, d_w, d_sc, d_idx, recv_d = op.dispatch(packed.view(fp4), inp.w_d, scales, inp.idx_d,
                                                inp.ntok)
    op.sync()
    recv, src_pos, slot = check_route(inp, recv_d, op.get_dispatch_src_token_pos())
    x_ref = oracle.place_rows(host(packed), inp.ntok, slot)
    sc_ref = oracle.place_rows(host(scales), inp.ntok, slot)
    gx = d_x.contiguous().view(torch.uint8).cpu().numpy()
    gs = host(d_sc).view(np.float32)
    for r in range(R):
        n = recv[r]
        assert np.array_equal(gx[r, :n], x_ref[r, :n])
        assert np.array_equal(gs[r, :n].reshape(n, -1).view(np.uint32), sc_ref[r, :n].view(np.uint32))
    op.reset()


@pytest.mark.parametrize("quant", ["fp8", "fp4"])
def test_convert_dispatch_output_carries_quantised_rows(quant):
    """convert_dispatch_output after a quantising dispatch carries codes and
    block scales into the packed layout, equal to the fused packed dispatch."""
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(tokens_per_rank=140, hidden=1024, mask_prob=0.1,
                                               dispatch_dtype=quant)
    R, T, Er = wl.world_size, wl.tokens_per_rank, wl.experts_per_rank
    inp = Inputs(wl, 5, ragged=True)
    cfg = make_config(wl, standard_moe=2)
    op = EpDispatchCombineOp(cfg)
    d_x, d_w, d_sc, d_idx, recv_d = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)
    o = E.ep_convert_dispatch_output(op._handle, d_x.data_ptr(), d_idx.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    v = op._std_views(o)
    op.sync()
    q, sc = oracle_quant(cfg, inp.x_bits())
    pcap = std_pcap(wl)
    ref = oracle.std_layout(inp.idx, inp.ntok, Er, pcap)
    px_ref = oracle.std_place_rows(q, inp.ntok, ref["row_map"], pcap)
    ps_ref = oracle.std_place_rows(sc, inp.ntok, ref["row_map"], pcap)
    base, rows = host(v["rank_base"]).astype(np.int64), ref["rank_rows"]
    gx = pool_to_ranks(host(v["packed_recv_x"]), base, rows, pcap)
    gs = pool_to_ranks(host(v["packed_recv_scales"]), base, rows, pcap)
    gsi = pool_to_ranks(host(v["packed_recv_src_info"]), base, rows, pcap, fill=-2)
    for r in range(R):
        n = ref["rank_rows"][r]
        used = ref["src_info"][r, :n] >= 0
        assert np.array_equal(gsi[r, :n], ref["src_info"][r, :n])
        assert np.array_equal(gx[r, :n][used], px_ref[r, :n][used])
        assert np.array_equal(gs[r, :n][used].view(np.uint32), ps_ref[r, :n][used].view(np.uint32))
    op.reset()


# ------------------------------------------ small batches: summed chunk counts

@pytest.mark.parametrize("name,over,seed", [
    ("ds_v3_latency", dict(tokens_per_rank=512, hidden=1024), 4),    # 16 chunks: summed counts
    ("ds_v3_latency", dict(tokens_per_rank=513, hidden=1024), 5),    # 24 chunks: scanned offsets
    ("ds_v3_latency", dict(tokens_per_rank=257, hidden=1024, dispatch_dtype="fp4"), 6),
    ("ds_v3_latency", dict(dispatch_dtype="bf16", hidden=1032), 7),
    ("tiny", dict(world_size=1, experts_per_rank=8, topk=4, tokens_per_rank=4096), 8),
    ("tiny", dict(world_size=16, experts_per_rank=2, topk=8, tokens_per_rank=256), 9),
    ("mid_masked", dict(tokens_per_rank=200, mask_prob=0.5, hidden=1024), 10),
])
def test_small_batch_chunk_offsets(name, over, seed):
    """Up to 16 routing chunks the dispatch kernel adds up the earlier chunks'
    counts itself (the layout skips its offset scan) and writes
    recv_num_token; beyond that the layout's scanned offsets are used. Both
    against the oracle, ragged token counts included."""
    run_2d(WORKLOADS[name].with_(**over), seed=seed, ragged=True)


# ------------------------------- quantisation with arbitrary (inexact) scales

def _quant_sweep(fmt, amax_bits, impl="auto"):
    """Every finite bf16 value with |x| <= amax in blocks whose amax is fixed,
    for each amax in amax_bits: codes and scales from dispatch against the
    oracle's encoder, bit for bit."""
    blk = 128 if fmt == "fp8" else 32
    per = blk - 1
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = (allb.astype(np.uint32) << 16).view(np.float32)
    rows = []
    for ab in amax_bits:
        amax = float((np.uint32(ab) << np.uint32(16)).view(np.float32))
        keep = np.isfinite(vals) & (np.abs(vals) <= amax)
        bits = allb[keep]
        nblk = -(-len(bits) // per)
        b = np.zeros((nblk, blk), np.uint16)
        b[:, per] = ab
        flat = b[:, :per].reshape(-1)
        flat[:len(bits)] = bits
        b[:, :per] = flat.reshape(nblk, per)
        rows.append(b)
    x = np.concatenate(rows).reshape(-1)
    H = 1024
    T = -(-x.size // H)
    xx = np.zeros(T * H, np.uint16)
    xx[:x.size] = x
    x = xx.reshape(1, T, H)
    wl = WORKLOADS["tiny"].with_(world_size=1, experts_per_rank=1, topk=1, tokens_per_rank=T,
                                 hidden=H, dispatch_dtype=fmt, expert_output="random")
    op = EpDispatchCombineOp(make_config(wl, dispatch_impl=impl))
    xd = torch.from_numpy(x.view(np.int16)).to(DEV).view(torch.bfloat16)
    w = torch.ones((1, T, 1), dtype=torch.float32, device=DEV)
    idx = torch.zeros((1, T, 1), dtype=torch.int32, device=DEV)
    d_x, _, d_sc, _, _ = op.dispatch(xd, w, None, idx, [T])
    op.sync()
    q_ref, sc_ref = (oracle.quant_tokens if fmt == "fp8" else oracle.quant_tokens_fp4)(x)
    assert np.array_equal(host(d_sc)[0, :T].view(np.uint32), sc_ref[0].view(np.uint32))
    assert np.array_equal(host(d_x)[0, :T], q_ref[0])
    op.reset()


def _bf16_bits(v):
    return int((np.array([v], np.float32).view(np.uint32)[0] + 0x8000) >> 16)


@pytest.mark.parametrize("impl", ["auto", "vector"])
@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
def test_quant_codes_every_bf16_value_inexact_scales(fmt, impl):
    """Codes of the correctly rounded quotient for every input: all finite
    bf16 values under amax values whose scale amax/448 (or amax/6) is inexact,
    exact, a power of two, below 2^-90 or above 2^125, or subnormal."""
    rng = np.random.default_rng(31 if fmt == "fp8" else 32)
    amax = [_bf16_bits(v) for v in (1.0, 3.0, 7.0, 100.0, 0.3, 1e-3, 5e4, 1e-20, 1e30)]
    amax += [_bf16_bits(v) for v in (448.0, 6.0, 448.0 * 2.0 ** -40, 6.0 * 2.0 ** 20, 1e-25)]
    amax += [int(b) for b in (rng.integers(0x0080, 0x7F7F, size=6))]     # random finite positives
    amax += [0x0001, 0x0050, 0x0100, 0x7F7F, 0x7F00]                      # tiny scales, huge amax
    _quant_sweep(fmt, amax, impl)


def _blocks_every_amax(a_lo: int, a_hi: int, blk: int, binades: int = 24) -> np.ndarray:
    """bf16 bits of blocks of `blk` elements: for every positive finite bf16
    block maximum a in [a_lo, a_hi) (bit patterns), every bf16 x of either sign
    with |x| <= a and |x| in the `binades` binades below a, plus zeros; the
    last element of each block is a itself. Values per maximum are padded
    with +0 to whole blocks."""
    per = blk - 1
    a = np.arange(a_lo, a_hi, dtype=np.int64)
    lo = np.maximum(1, a - 128 * binades)
    n = 2 * (a - lo + 1) + 2                     # +/- each magnitude, and +/-0
    nblk = -(-n // per)
    out = np.zeros((int(nblk.sum()), blk), np.uint16)
    out[:, per] = np.repeat(a, nblk).astype(np.uint16)
    vals = np.zeros(int((nblk * per).sum()), np.uint16)
    start = np.concatenate([[0], np.cumsum(nblk * per)[:-1]])
    for j in range(len(a)):                       # (a_hi - a_lo) is small per chunk
        mags = np.arange(lo[j], a[j] + 1, dtype=np.uint16)
        v = np.concatenate([mags, mags | np.uint16(0x8000), np.array([0, 0x8000], np.uint16)])
        vals[start[j]:start[j] + len(v)] = v
    out[:, :per] = vals.reshape(-1, per)
    return out.reshape(-1)


@pytest.mark.slow
@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
def test_quant_codes_every_block_maximum(fmt):
    """A code depends only on the element and its block's maximum (the scale
    is amax / 448 or amax / 6). For every positive finite bf16 block maximum
    and every bf16 element of either sign in the 24 binades below it (smaller
    elements quote far below half the smallest nonzero code), dispatch's
    codes and scales equal the oracle's, which divides with IEEE rounding:
    the kernel's reciprocal-and-residual quotient (taken below 8192 source
    tokens for FP8, always for FP4) is checked on every input pair whose code
    it can decide."""
    blk = 128 if fmt == "fp8" else 32
    H = 1024
    T = 4096   # below 8192 tokens FP8 dispatch takes the reciprocal-and-residual quotients
    wl = WORKLOADS["tiny"].with_(world_size=1, experts_per_rank=1, topk=1, tokens_per_rank=T,
                                 hidden=H, dispatch_dtype=fmt, expert_output="random")
    op = EpDispatchCombineOp(make_config(wl))
    w = torch.ones((1, T, 1), dtype=torch.float32, device=DEV)
    idx = torch.zeros((1, T, 1), dtype=torch.int32, device=DEV)
    quant = oracle.quant_tokens if fmt == "fp8" else oracle.quant_tokens_fp4
    pending = np.zeros(0, np.uint16)
    a_next, a_end = 1, 0x7F80                     # every positive finite bf16
    checked = 0
    while a_next < a_end or pending.size:
        while pending.size < T * H and a_next < a_end:
            hi = min(a_end, a_next + 256)
            pending = np.concatenate([pending, _blocks_every_amax(a_next, hi, blk)])
            a_next = hi
        x = np.zeros(T * H, np.uint16)
        m = min(pending.size, T * H)
        x[:m] = pending[:m]
        pending = pending[m:]
        ntok = -(-m // H)
        xd = torch.from_numpy(x.view(np.int16)).to(DEV).view(torch.bfloat16).view(1, T, H)
        d_x, _, d_sc, _, _ = op.dispatch(xd, w, None, idx, [ntok])
        op.sync()
        xs = x.reshape(1, T, H)[:, :ntok]
        q_ref, sc_ref = quant(np.ascontiguousarray(xs))
        assert np.array_equal(host(d_sc)[0, :ntok].view(np.uint32), sc_ref[0].view(np.uint32))
        assert np.array_equal(host(d_x)[0, :ntok], q_ref[0]), "codes"
        op.reset()
        checked += m
    assert checked > 150_000_000


# ---------------------------------------- launch configuration and tuning files

def test_launch_config_per_call_and_auto_mode(tmp_path, monkeypatch):
    """Per-call block_num / warp_per_block (User Guide, section 6) and auto
    mode reading per-shape rules from a tuning file (section 10): the handle
    takes the chosen launch configuration per phase, and results stay bit
    for bit those of the default configuration."""
    from combine_route_layout_gb300 import tuning
    wl = WORKLOADS["ds_v3_latency"].with_(tokens_per_rank=300, hidden=1024)
    inp = Inputs(wl, 5, ragged=True)
    y = make_expert_outputs(wl, wl.world_size * wl.tokens_per_rank, 5, device=DEV)
    ref_op = EpDispatchCombineOp(make_config(wl))
    rd = ref_op.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)
    ref_x, ref_sc = rd[0].clone(), rd[2].clone()
    ref_out, _ = ref_op.combine(y, rd[1], None, call_reset=True)

    d = str(tmp_path)
    monkeypatch.setenv("EP_TUNING_CONFIG_DIR", d)
    tuning.save_rule("2d", 8, "dispatch", {"dtype": "fp8", "num_tokens": 512, "hidden_dim": 1024,
                                           "impl": "vector", "block_num": 152,
                                           "warp_per_block": 4}, d)
    tuning.save_rule("2d", 8, "combine", {"dtype": "bf16", "num_tokens": 512, "hidden_dim": 1024,
                                          "impl": "bulk", "block_num": 304,
                                          "warp_per_block": 8}, d)
    op = EpDispatchCombineOp(make_config(wl, launch_config_mode="auto"))
    dd = op.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)
    assert op.get_launch_config(E.EP_PHASE_DISPATCH) == ("vector", 152, 4)
    out, _ = op.combine(y, dd[1], None, call_reset=True)
    assert op.get_launch_config(E.EP_PHASE_COMBINE) == ("bulk", 304, 8)
    op.sync()
    recv = host(rd[4])
    for r in range(wl.world_size):
        n = recv[r]
        assert np.array_equal(host(dd[0])[r, :n], host(ref_x)[r, :n])
        assert np.array_equal(host(dd[2])[r, :n].view(np.uint32), host(ref_sc)[r, :n].view(np.uint32))
    def same_valid(a, b):   # rows past a rank's token count are never written
        ga, gb = host(a), host(b)
        return all(np.array_equal(ga[s, :n], gb[s, :n]) for s, n in enumerate(inp.ntok))

    assert same_valid(out, ref_out)

    man = EpDispatchCombineOp(make_config(wl))
    md = man.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp.ntok, block_num=456, warp_per_block=2)
    assert man.get_launch_config(E.EP_PHASE_DISPATCH) == ("auto", 456, 2)
    mout, _ = man.combine(y, md[1], None, call_reset=True, block_num=76, warp_per_block=4)
    assert man.get_launch_config(E.EP_PHASE_COMBINE) == ("auto", 76, 4)
    assert same_valid(mout, ref_out)
    md = man.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)   # back to the config's
    assert man.get_launch_config(E.EP_PHASE_DISPATCH) == ("auto", -1, 8)
    man.reset()
    man.set_launch_config(E.EP_PHASE_DISPATCH, "vector", 304, 4)     # a new base setting
    md = man.dispatch(inp.x, inp.w_d, None, inp.idx_d, inp.ntok)
    assert man.get_launch_config(E.EP_PHASE_DISPATCH) == ("vector", 304, 4)
    man.reset()


@pytest.mark.parametrize("std", [False, True])
def test_tuner_sweeps_and_writes_rules(tmp_path, monkeypatch, std):
    """The tuner times its candidates on a small shape and saves the fastest."""
    from combine_route_layout_gb300 import tuning
    monkeypatch.setitem(tuning.SCOPES, "tiny", {"grids": [-1, 152], "warps": [8],
                                                "bulk_grids": [-1]})
    wl = WORKLOADS["skewed_zipf_std_moe" if std else "ds_v3_latency"].with_(
        tokens_per_rank=64, hidden=512)
    cfg = make_config(wl)
    for phase in ("dispatch", "combine"):
        rule = tuning.tune_shape(cfg, phase, "tiny", iters=3)
        assert rule["num_tokens"] == 64 and rule["hidden_dim"] == 512
        assert rule["impl"] in ("vector", "bulk") and rule["latency_us"] > 0
        assert rule["candidates"] == len(tuning._candidates(phase, cfg, "tiny")) >= 2
        p = tuning.save_rule("stdmoe" if std else "2d", 8, phase, rule, str(tmp_path))
        assert tuning.lookup(tuning.load_rules("stdmoe" if std else "2d", 8, phase,
                                               str(tmp_path)),
                             rule["dtype"], 512, 64) == json.load(open(p))["rules"][0]
