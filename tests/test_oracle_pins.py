"""Pins the CPU oracle to facts other than itself (runs without a GPU).

Each check is chosen so that a plausible mistake in the oracle (a dropped
term, a wrong sign, a wrong index or stride, a transposed operand, an
off-by-one in the order) fails at least one of them:
  * codecs against brute-force nearest-code search and against torch's casts;
  * quantisation against a torch composition and the format's error bound;
  * routing against an independent per-destination enumerator and invariants;
  * combine against the identity-expert invariant (MORI-EP User Guide,
    section 7; "Choosing an EP API and backend", bench_ep identity check)
    and against an exact f64 sum within a rounding bound;
  * standard-MoE layout against histograms, alignment and a second
    construction from the 2D receive buffers.
"""
import os

import numpy as np
import pytest
import torch

from gen import WORKLOADS, make_indices, make_num_tokens, make_tokens, make_weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split("|")])
    return rows


# ------------------------------------------------------------------ codecs

def _e4m3_brute(v: np.ndarray, oracle) -> np.ndarray:
    """Nearest same-signed finite code by exhaustive search; ties to even code."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.int64)
    vals = np.abs(oracle.e4m3_to_f32(codes).astype(np.float64))
    out = np.empty(v.shape, np.uint8)
    for i, x in enumerate(v.astype(np.float64)):
        neg = np.signbit(x)
        cand = codes[(codes >= 0x80) == neg]
        mags = vals[(codes >= 0x80) == neg]
        d = np.abs(mags - abs(x))
        best = d.min()
        tied = cand[d == best]
        even = tied[(tied & 1) == 0]
        out[i] = (even if len(even) else tied)[0]
    return out


def test_e4m3_golden_special_values(oracle_lib):
    for expr, code in _read_golden("e4m3_ocp_special_values.txt"):
        v = np.float32(eval(expr, {"__builtins__": {}}))
        got = int(oracle_lib.e4m3_from_f32(np.array([v]))[0])
        assert got == int(code, 16), (expr, hex(got), code)
    assert int(oracle_lib.e4m3_from_f32(np.array([np.nan], np.float32))[0]) == 0x7F


def test_e4m3_decode_matches_torch(oracle_lib):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle_lib.e4m3_to_f32(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_encode_vs_brute_force(oracle_lib):
    rng = np.random.default_rng(7)
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    vals = oracle_lib.e4m3_to_f32(codes).astype(np.float64)
    mags = np.unique(np.abs(vals))
    mids = (mags[1:] + mags[:-1]) / 2
    pts = [mags, mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
           np.nextafter(mids.astype(np.float32), np.float32(-np.inf)),
           np.array([448.0, 460.0, 464.0, 470.0, 1e6, 2.0**-10, 2.0**-11, 1e-30])]
    v = np.concatenate([p.astype(np.float32) for p in pts])
    v = np.concatenate([v, -v, rng.standard_normal(3000).astype(np.float32) * 30,
                        (rng.random(1000) * 2.0**-6).astype(np.float32)])
    assert np.array_equal(oracle_lib.e4m3_from_f32(v), _e4m3_brute(v, oracle_lib))


def test_e4m3_encode_vs_torch_in_range(oracle_lib):
    rng = np.random.default_rng(8)
    u = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    v = u.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) <= 448.0)]
    v = np.concatenate([v, rng.standard_normal(100000).astype(np.float32) * 100])
    v = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle_lib.e4m3_from_f32(v), ref)


def test_bf16_round_vs_torch(oracle_lib):
    rng = np.random.default_rng(9)
    u = rng.integers(0, 2**32, size=500000, dtype=np.uint64).astype(np.uint32)
    # plus every tie pattern and the values next to it
    ties = (rng.integers(0, 2**16, size=20000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    u = np.concatenate([u, ties, ties + 1, ties - 1,
                        np.array([0x7F7F8000, 0x7F7FFFFF, 0xFF7F8000, 0x00008000, 0x00018000],
                                 np.uint32)])
    v = u.view(np.float32)
    fin = ~np.isnan(v)
    ref = _bits(torch.from_numpy(v[fin]).to(torch.bfloat16))
    assert np.array_equal(oracle_lib.bf16_from_f32(v[fin]), ref)
    nanb = oracle_lib.bf16_from_f32(v[~fin])
    assert np.all(np.isnan(oracle_lib.bf16_to_f32(nanb)))


# ---------------------------------------------------------- quantisation

def _quant_torch(xb: torch.Tensor):
    """Per-128 block quantisation composed from torch library ops."""
    x = xb.float().reshape(-1, 128)
    amax = x.abs().amax(dim=1, keepdim=True)
    scale = amax / 448.0
    v = torch.where(amax == 0, x, x / torch.where(amax == 0, torch.ones_like(scale), scale))
    v = v.clamp(-448.0, 448.0)
    q = v.to(torch.float8_e4m3fn).view(torch.uint8)
    return q.reshape(xb.shape).numpy(), scale.reshape(*xb.shape[:-1], -1).numpy()


@pytest.mark.parametrize("dist", ["normal", "normal_outliers", "uniform"])
def test_quant_matches_torch_composition(oracle_lib, dist):
    wl = WORKLOADS["ds_v3_latency"].with_(tokens_per_rank=4, world_size=2, token_dist=dist,
                                          outlier_frac=0.01, outlier_scale=50.0)
    xb = make_tokens(wl, seed=3)
    xb[0, 0, :128] = 0.0                                  # an all-zero block
    xb[0, 1, 128:256] = -0.0                              # negative zeros
    xb[1, 2, :128] = torch.tensor(1e-38).to(torch.bfloat16)  # tiny block (subnormal scale)
    q, sc = oracle_lib.quant_tokens(_bits(xb))
    q_ref, sc_ref = _quant_torch(xb)
    assert np.array_equal(sc.view(np.uint32), sc_ref.view(np.uint32))
    assert np.array_equal(q, q_ref)
    assert np.all(q[0, 1, 128:256] == 0x80)


def test_quant_invariants(oracle_lib):
    wl = WORKLOADS["ds_v3_throughput"].with_(tokens_per_rank=8, world_size=2)
    xb = make_tokens(wl, seed=11)
    q, sc = oracle_lib.quant_tokens(_bits(xb))
    x = xb.float().numpy().reshape(-1, 128)
    qb = q.reshape(-1, 128)
    s = sc.reshape(-1, 1).astype(np.float64)
    # the element of largest magnitude encodes to +-448
    am = np.abs(x).argmax(axis=1)
    top = qb[np.arange(len(qb)), am]
    assert np.all((top & 0x7F) == 0x7E)
    # E4M3 error bound: relative 2^-4 in the normal range, absolute 2^-10 * scale below it
    dec = oracle_lib.e4m3_to_f32(qb).astype(np.float64) * s
    err = np.abs(dec - x)
    normal = np.abs(x) / s >= 2.0**-6
    assert np.all(err[normal] <= 2.0**-4 * np.abs(x[normal]) * (1 + 1e-6))
    assert np.all(err[~normal] <= 2.0**-10 * np.broadcast_to(s, x.shape)[~normal] * (1 + 1e-6))


# ----------------------------------------------------------------- routing

def _route_brute(idx, ntok, Er):
    """Per destination: scan all (s, t) in order and keep those with an owned expert."""
    R, T, k = idx.shape
    rows = {r: [] for r in range(R)}
    for r in range(R):
        for s in range(R):
            for t in range(int(ntok[s])):
                if any(e >= 0 and e // Er == r for e in idx[s, t]):
                    rows[r].append((s, t))
    return rows


def _check_route(idx, ntok, Er, recv, src_pos, slot):
    R, T, k = idx.shape
    brute = _route_brute(idx, ntok, Er)
    for r in range(R):
        assert recv[r] == len(brute[r])
        enc = [s * (R * T) + t for s, t in brute[r]]
        assert list(src_pos[r, :recv[r]]) == enc
        assert np.all(src_pos[r, recv[r]:] == -1)
        for i, (s, t) in enumerate(brute[r]):
            assert slot[s, t, r] == i
    # tokens not routed to a rank have slot -1; sum of counts = sum of |D|
    nD = 0
    for s in range(R):
        for t in range(int(ntok[s])):
            D = {int(e) // Er for e in idx[s, t] if e >= 0}
            nD += len(D)
            for r in range(R):
                assert (slot[s, t, r] >= 0) == (r in D)
    assert recv.sum() == nD


@pytest.mark.parametrize("name,ragged,seed", [("tiny", False, 0), ("tiny", True, 1),
                                              ("mid_masked", True, 2)])
def test_route_vs_brute_force(oracle_lib, name, ragged, seed):
    wl = WORKLOADS[name].with_(tokens_per_rank=min(WORKLOADS[name].tokens_per_rank, 12))
    if name == "mid_masked":
        wl = wl.with_(mask_prob=0.3)
    idx = make_indices(wl, seed=seed)
    ntok = make_num_tokens(wl, ragged=ragged, seed=seed)
    recv, src_pos, slot = oracle_lib.route(idx, ntok, wl.experts_per_rank)
    _check_route(idx, ntok, wl.experts_per_rank, recv, src_pos, slot)


def test_src_token_pos_golden(oracle_lib):
    for R, Tm, s, t, pos in _read_golden("src_token_pos_examples.txt"):
        R, Tm, s, t, pos = map(int, (R, Tm, s, t, pos))
        idx = np.full((R, Tm, 1), -1, np.int32)
        idx[s, t, 0] = 0                              # expert 0 lives on rank 0
        ntok = np.full(R, Tm, np.int32)
        recv, src_pos, slot = oracle_lib.route(idx, ntok, 1)
        assert recv[0] == 1 and src_pos[0, 0] == pos
        assert divmod(int(src_pos[0, 0]), R * Tm) == (s, t)


def test_route_rejects_bad_index(oracle_lib):
    idx = np.zeros((2, 3, 2), np.int32)
    idx[1, 2, 1] = 8                                  # E = 2 * 4
    with pytest.raises(oracle_lib.OracleError) as ei:
        oracle_lib.route(idx, np.array([3, 3], np.int32), 4)
    assert ei.value.code == oracle_lib.ORC_ERR_INDEX


def test_dispatch_payload_is_identity_copy(oracle_lib):
    wl = WORKLOADS["tiny"]
    idx, w = make_indices(wl), make_weights(wl)
    x = _bits(make_tokens(wl))
    ntok = make_num_tokens(wl, ragged=True, seed=4)
    d = oracle_lib.dispatch(x, w, idx, ntok, wl.experts_per_rank)
    R, T = wl.world_size, wl.tokens_per_rank
    for r in range(R):
        for i in range(d["recv_num_token"][r]):
            s, t = divmod(int(d["src_pos"][r, i]), R * T)
            assert np.array_equal(d["x"][r, i], x[s, t])
            assert np.array_equal(d["w"][r, i].view(np.uint32), w[s, t].view(np.uint32))
            assert np.array_equal(d["idx"][r, i], idx[s, t])


# ----------------------------------------------------------------- combine

def _identity_setup(name="tiny", seed=0, **kw):
    wl = WORKLOADS[name].with_(**kw)
    idx, w = make_indices(wl, seed=seed), make_weights(wl, seed=seed)
    xb = make_tokens(wl, seed=seed)
    ntok = make_num_tokens(wl, ragged=(seed % 2 == 1), seed=seed)
    return wl, idx, w, xb, _bits(xb), ntok


def _ndest(idx, Er):
    R, T, k = idx.shape
    out = np.zeros((R, T), np.int64)
    for s in range(R):
        for t in range(T):
            out[s, t] = len({int(e) // Er for e in idx[s, t] if e >= 0})
    return out


@pytest.mark.parametrize("seed", [0, 1])
def test_combine_identity_expert_f32(oracle_lib, seed):
    wl, idx, w, xb, x, ntok = _identity_setup(seed=seed, mask_prob=0.25)
    d = oracle_lib.dispatch(x, w, idx, ntok, wl.experts_per_rank)
    out, out_w = oracle_lib.combine(d["x"], idx, ntok, d["slot"], wl.experts_per_rank,
                                    w_recv=d["w"], out_dtype="fp32")
    nD = _ndest(idx, wl.experts_per_rank)
    exp = xb.float().numpy() * nD[..., None]              # exact: |D| <= 8, 8-bit significand
    for s in range(wl.world_size):
        n = ntok[s]
        assert np.array_equal(out[s, :n], exp[s, :n])
        has = nD[s, :n] > 0
        assert np.array_equal(out_w[s, :n][has].view(np.uint32), w[s, :n][has].view(np.uint32))
        assert np.all(out_w[s, :n][~has] == 0)


def test_combine_identity_expert_bf16(oracle_lib):
    wl, idx, w, xb, x, ntok = _identity_setup("mid_masked", tokens_per_rank=16, hidden=512)
    d = oracle_lib.dispatch(x, w, idx, ntok, wl.experts_per_rank)
    out, _ = oracle_lib.combine(d["x"], idx, ntok, d["slot"], wl.experts_per_rank, out_dtype="bf16")
    nD = _ndest(idx, wl.experts_per_rank)
    exp = _bits((xb.float() * torch.from_numpy(nD[..., None]).float()).to(torch.bfloat16))
    assert np.array_equal(out, exp)


def test_combine_weighted_identity(oracle_lib):
    wl, idx, w, xb, x, ntok = _identity_setup(mask_prob=0.2)
    d = oracle_lib.dispatch(x, w, idx, ntok, wl.experts_per_rank)
    out, _ = oracle_lib.combine(d["x"], idx, ntok, d["slot"], wl.experts_per_rank,
                                w_recv=d["w"], weighted=True, out_dtype="fp32")
    wsum = np.where(idx >= 0, w.astype(np.float64), 0.0).sum(-1)
    exp = xb.double().numpy() * wsum[..., None]
    err = np.abs(out - exp)
    bound = 8 * 2.0**-24 * np.abs(xb.double().numpy()) * 2 + 1e-45
    assert np.all(err <= bound)


def test_combine_random_y_vs_exact_sum(oracle_lib):
    wl, idx, w, xb, x, ntok = _identity_setup(mask_prob=0.1)
    R, T, H = wl.world_size, wl.tokens_per_rank, wl.hidden
    d = oracle_lib.dispatch(x, w, idx, ntok, wl.experts_per_rank)
    rng = np.random.default_rng(5)
    y = rng.standard_normal((R, R * T, H)).astype(np.float32)
    for weighted in (False, True):
        out, _ = oracle_lib.combine(y, idx, ntok, d["slot"], wl.experts_per_rank,
                                    w_recv=d["w"], weighted=weighted, out_dtype="fp32")
        for s in range(R):
            for t in range(ntok[s]):
                exact = np.zeros(H)
                mag = np.zeros(H)
                for r in range(R):
                    i = d["slot"][s, t, r]
                    if i < 0:
                        continue
                    wr = sum(float(w[s, t, j]) for j in range(wl.topk)
                             if idx[s, t, j] >= 0 and idx[s, t, j] // wl.experts_per_rank == r)
                    c = wr if weighted else 1.0
                    exact += c * y[r, i].astype(np.float64)
                    mag += abs(c) * np.abs(y[r, i].astype(np.float64))
                assert np.all(np.abs(out[s, t] - exact) <= 2 * R * 2.0**-24 * mag + 1e-40)


# ---------------------------------------------------------- standard MoE

def _check_std_layout(res, idx, ntok, Er, pcap):
    R, T, k = idx.shape
    E = R * Er
    hist = np.zeros(E, np.int64)
    for s in range(R):
        for e in idx[s, :ntok[s]].ravel():
            if e >= 0:
                hist[e] += 1
    assert np.array_equal(res["count"].ravel(), hist)
    for r in range(R):
        off = 0
        for el in range(Er):
            assert res["seg_off"][r, el] == off and off % 128 == 0
            off += -(-int(res["count"][r, el]) // 128) * 128
        assert res["rank_rows"][r] == off
    seen = set()
    for s in range(R):
        for t in range(ntok[s]):
            for j in range(k):
                e = int(idx[s, t, j])
                m = int(res["row_map"][s, t, j])
                if e < 0:
                    assert m == -1
                    continue
                r, el = divmod(e, Er)
                assert m // pcap == r
                row = m % pcap
                lo = res["seg_off"][r, el]
                assert lo <= row < lo + res["count"][r, el]
                assert res["src_info"][r, row] == s * R * T + t
                assert m not in seen
                seen.add(m)
    for r in range(R):
        for el in range(Er):
            lo, c = res["seg_off"][r, el], res["count"][r, el]
            seg = res["src_info"][r, lo:lo + c]
            assert np.all(np.diff(seg) > 0)                  # canonical (s, t) order
            pad_end = lo + (-(-int(c) // 128) * 128)
            assert np.all(res["src_info"][r, lo + c:pad_end] == -1)
            for s in range(R):
                lr = int(res["layout_range"][r, el, s])
                b, n = lr >> 32, lr & 0xFFFFFFFF
                assert n == int(np.sum(seg // (R * T) == s))
                assert b == int(np.sum(seg // (R * T) < s))


@pytest.mark.parametrize("router,seed", [("uniform", 0), ("zipf", 1), ("zipf", 2)])
def test_std_layout_invariants(oracle_lib, router, seed):
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(tokens_per_rank=40, hidden=128, world_size=4,
                                               experts_per_rank=3, topk=4, router=router,
                                               mask_prob=0.1)
    idx = make_indices(wl, seed=seed)
    ntok = make_num_tokens(wl, ragged=True, seed=seed)
    pcap = wl.world_size * wl.tokens_per_rank * wl.topk + 127 * wl.experts_per_rank
    res = oracle_lib.std_layout(idx, ntok, wl.experts_per_rank, pcap)
    _check_std_layout(res, idx, ntok, wl.experts_per_rank, pcap)


def test_std_layout_capacity_and_duplicates(oracle_lib):
    idx = np.array([[[0, 1]], [[0, 2]]], np.int32)       # R=2, Tmax=1, k=2, E_r=2
    ntok = np.array([1, 1], np.int32)
    with pytest.raises(oracle_lib.OracleError) as ei:
        oracle_lib.std_layout(idx, ntok, 2, 200)          # needs 256 rows on rank 0
    assert ei.value.code == oracle_lib.ORC_ERR_CAPACITY
    dup = np.array([[[1, 1]], [[0, 2]]], np.int32)
    with pytest.raises(oracle_lib.OracleError):
        oracle_lib.std_layout(dup, ntok, 2, 512)


def test_convert_dispatch_output_equals_fused(oracle_lib):
    """Two constructions of the packed layout: from the source tokens and from
    the 2D receive buffers (MORI-EP User Guide, section 4)."""
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(tokens_per_rank=24, hidden=128, mask_prob=0.1)
    idx, w = make_indices(wl, seed=3), make_weights(wl, seed=3)
    x = _bits(make_tokens(wl, seed=3))
    ntok = make_num_tokens(wl, ragged=True, seed=3)
    pcap = wl.world_size * wl.tokens_per_rank * wl.topk + 127 * wl.experts_per_rank
    fused = oracle_lib.std_dispatch(x, idx, ntok, wl.experts_per_rank, pcap)
    d = oracle_lib.dispatch(x, w, idx, ntok, wl.experts_per_rank)
    conv = oracle_lib.convert_dispatch_output(d["recv_num_token"], d["x"], d["idx"], d["src_pos"],
                                              wl.tokens_per_rank, wl.experts_per_rank, pcap)
    for key in ("count", "seg_off", "rank_rows", "row_map", "src_info", "layout_range"):
        assert np.array_equal(fused[key], conv[key]), key
    used = fused["src_info"] >= 0
    assert np.array_equal(fused["x"][used], conv["x"][used])


def test_std_combine_identity(oracle_lib):
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(tokens_per_rank=20, hidden=256, mask_prob=0.1)
    idx, w = make_indices(wl, seed=1), make_weights(wl, seed=1)
    xb = make_tokens(wl, seed=1)
    x = _bits(xb)
    ntok = make_num_tokens(wl, ragged=True, seed=1)
    pcap = wl.world_size * wl.tokens_per_rank * wl.topk + 127 * wl.experts_per_rank
    p = oracle_lib.std_dispatch(x, idx, ntok, wl.experts_per_rank, pcap)
    nvalid = (idx >= 0).sum(-1)
    out = oracle_lib.std_combine(p["x"], idx, ntok, p["row_map"], wl.experts_per_rank,
                                 weighted=False, out_dtype="fp32")
    exp = xb.float().numpy() * nvalid[..., None]
    outw = oracle_lib.std_combine(p["x"], idx, ntok, p["row_map"], wl.experts_per_rank,
                                  w=w, weighted=True, out_dtype="fp32")
    wsum = np.where(idx >= 0, w.astype(np.float64), 0.0).sum(-1)
    expw = xb.double().numpy() * wsum[..., None]
    for s in range(wl.world_size):
        n = ntok[s]
        assert np.array_equal(out[s, :n], exp[s, :n])
        bound = 8 * 2.0**-24 * np.abs(xb[s, :n].double().numpy()) * 2 + 1e-45
        assert np.all(np.abs(outw[s, :n] - expw[s, :n]) <= bound)


def test_convert_combine_input_round_trip(oracle_lib):
    """Identity experts through packed -> 2D conversion -> 2D combine equal
    identity experts through the standard-MoE combine (unweighted)."""
    wl = WORKLOADS["skewed_zipf_std_moe"].with_(tokens_per_rank=20, hidden=128, mask_prob=0.1,
                                               router="uniform")
    idx, w = make_indices(wl, seed=2), make_weights(wl, seed=2)
    xb = make_tokens(wl, seed=2)
    x = _bits(xb)
    ntok = make_num_tokens(wl, ragged=False)
    Er = wl.experts_per_rank
    pcap = wl.world_size * wl.tokens_per_rank * wl.topk + 127 * Er
    d = oracle_lib.dispatch(x, w, idx, ntok, Er)
    conv = oracle_lib.convert_dispatch_output(d["recv_num_token"], d["x"], d["idx"], d["src_pos"],
                                              wl.tokens_per_rank, Er, pcap)
    y2d = oracle_lib.convert_combine_input(conv["x"], d["recv_num_token"], d["src_pos"], idx,
                                           conv["row_map"], Er, out_dtype="fp32")
    out2d, _ = oracle_lib.combine(y2d, idx, ntok, d["slot"], Er, out_dtype="fp32")
    out_std = oracle_lib.std_combine(conv["x"], idx, ntok, conv["row_map"], Er, weighted=False,
                                     out_dtype="fp32")
    assert np.array_equal(out2d, out_std)
    exp = xb.float().numpy() * (idx >= 0).sum(-1)[..., None]
    assert np.array_equal(out2d, exp)


# -------------------------------------------- pins catch planted mistakes

def test_pins_detect_planted_mistakes(oracle_lib):
    """Corrupt oracle outputs the way a plausible bug would and check that the
    pins above reject each one."""
    wl = WORKLOADS["tiny"].with_(tokens_per_rank=6)
    idx = make_indices(wl, seed=5)
    ntok = make_num_tokens(wl)
    recv, src_pos, slot = oracle_lib.route(idx, ntok, wl.experts_per_rank)
    _check_route(idx, ntok, wl.experts_per_rank, recv, src_pos, slot)
    bad_pos = src_pos.copy()
    r = int(np.argmax(recv))
    bad_pos[r, [0, 1]] = bad_pos[r, [1, 0]]             # order swapped
    with pytest.raises(AssertionError):
        _check_route(idx, ntok, wl.experts_per_rank, recv, bad_pos, slot)
    bad_pos = src_pos.copy()
    bad_pos[r, 0] = (bad_pos[r, 0] % (wl.world_size * wl.tokens_per_rank)) * wl.tokens_per_rank
    with pytest.raises(AssertionError):                 # wrong stride in the encoding
        _check_route(idx, ntok, wl.experts_per_rank, recv, bad_pos, slot)
    bad_slot = slot.copy()
    bad_slot[0, 0] = np.where(bad_slot[0, 0] >= 0, -1, bad_slot[0, 0])  # dropped destination
    with pytest.raises(AssertionError):
        _check_route(idx, ntok, wl.experts_per_rank, recv, src_pos, bad_slot)
    # wrong sign in the quantiser: codes no longer satisfy the error bound
    xb = make_tokens(WORKLOADS["ds_v3_latency"].with_(tokens_per_rank=1, world_size=1), seed=1)
    q, sc = oracle_lib.quant_tokens(_bits(xb))
    x = xb.float().numpy().reshape(-1)
    dec = oracle_lib.e4m3_to_f32(q.reshape(-1) ^ 0x80).astype(np.float64) * np.repeat(sc.ravel(), 128)
    assert np.any(np.abs(dec - x) > 2.0**-4 * np.abs(x) + 2.0**-10 * np.repeat(sc.ravel(), 128))


# ------------------------------------------------------------------- FP4

def test_e2m1_golden_values(oracle_lib):
    for expr, code in _read_golden("e2m1_ocp_values.txt"):
        v = np.float32(eval(expr, {"__builtins__": {}}))
        assert int(oracle_lib.e2m1_from_f32(np.array([v]))[0]) == int(code, 16), expr
    mags = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(oracle_lib.e2m1_to_f32(np.arange(8))) == mags
    assert list(oracle_lib.e2m1_to_f32(np.arange(8, 16))) == [-m for m in mags]


def test_e2m1_encode_vs_brute_force(oracle_lib):
    rng = np.random.default_rng(12)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    mids = (mags[1:] + mags[:-1]) / 2
    v = np.concatenate([mags, mids, np.nextafter(mids.astype(np.float32), np.float32(9)),
                        np.nextafter(mids.astype(np.float32), np.float32(-1)),
                        rng.random(20000) * 8]).astype(np.float32)
    v = np.concatenate([v, -v])
    got = oracle_lib.e2m1_from_f32(v)
    for x, c in zip(v.astype(np.float64), got):
        d = np.abs(mags - abs(x))
        tied = np.nonzero(d == d.min())[0]
        m = tied[(tied & 1) == 0][0] if len(tied) > 1 else tied[0]
        assert c == (m | (8 if np.signbit(x) else 0)), (x, c)


def test_fp4_quant_invariants(oracle_lib):
    wl = WORKLOADS["ds_v3_throughput"].with_(tokens_per_rank=6, world_size=2, hidden=1024)
    xb = make_tokens(wl, seed=13)
    xb[0, 0, :32] = 0.0
    xb[0, 1, 32:64] = -0.0
    q, sc = oracle_lib.quant_tokens_fp4(_bits(xb))
    assert q.shape[-1] == 512 and sc.shape[-1] == 32
    x = xb.float().numpy().reshape(-1)
    codes = np.stack([q & 0xF, q >> 4], axis=-1).reshape(-1)   # even element in the low nibble
    s = np.repeat(sc.reshape(-1).astype(np.float64), 32)
    # every code is the encoder's code of x / scale (or of x when the block is all zero)
    v = np.where(s == 0, x, x / np.where(s == 0, 1, s).astype(np.float32))
    assert np.array_equal(codes, oracle_lib.e2m1_from_f32(v.astype(np.float32)))
    # the element of largest magnitude in each block encodes to +-6
    xb32 = x.reshape(-1, 32)
    top = codes.reshape(-1, 32)[np.arange(len(xb32)), np.abs(xb32).argmax(1)]
    nz = np.abs(xb32).max(1) > 0
    assert np.all((top[nz] & 7) == 7)
    nblk = 1024 // 32                                    # blocks per token
    assert np.all(codes.reshape(-1, 32)[0] == 0) and np.all(codes.reshape(-1, 32)[nblk + 1] == 8)
    # E2M1 error bound: half a code step in units of the scale
    dec = oracle_lib.e2m1_to_f32(codes).astype(np.float64) * s
    a = np.abs(x) / np.where(s == 0, 1, s)
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    assert np.all(np.abs(dec - x) <= 0.5 * step * s * (1 + 1e-6) + 1e-30)


# ------------------------------------- placement and token-sampled variants

def test_place_rows_against_direct_placement(oracle_lib):
    """place_rows puts row (s, t) at slot[s, t, r] of every destination r and
    nothing else (a direct Python placement from the route's slot map);
    std_place_rows does the same with the packed row map."""
    wl = WORKLOADS["tiny"].with_(mask_prob=0.2)
    idx, ntok = make_indices(wl, 3), make_num_tokens(wl, ragged=True, seed=3)
    R, T, k = idx.shape
    rows = np.arange(R * T * 3, dtype=np.int32).reshape(R, T, 3) + 1
    recv, src_pos, slot = oracle_lib.route(idx, ntok, wl.experts_per_rank)
    got = oracle_lib.place_rows(rows, ntok, slot)
    want = np.zeros((R, R * T, 3), np.int32)
    for s in range(R):
        for t in range(int(ntok[s])):
            for r in range(R):
                if slot[s, t, r] >= 0:
                    want[r, slot[s, t, r]] = rows[s, t]
    assert np.array_equal(got, want)
    pcap = R * T * k + 127 * wl.experts_per_rank
    lay = oracle_lib.std_layout(idx, ntok, wl.experts_per_rank, pcap)
    got = oracle_lib.std_place_rows(rows, ntok, lay["row_map"], pcap)
    want = np.zeros((R, pcap, 3), np.int32)
    for s in range(R):
        for t in range(int(ntok[s])):
            for j in range(k):
                g = lay["row_map"][s, t, j]
                if g >= 0:
                    want.reshape(R * pcap, 3)[g] = rows[s, t]
    assert np.array_equal(got, want)


@pytest.mark.parametrize("weighted,od", [(False, "bf16"), (True, "fp32")])
def test_combine_tokens_equals_combine_rows(oracle_lib, weighted, od):
    """The token-sampled combines give exactly the rows of the full ones (which
    the identity invariants and exact sums above pin), in the order asked."""
    wl = WORKLOADS["tiny"].with_(mask_prob=0.1)
    idx, ntok = make_indices(wl, 4), make_num_tokens(wl, ragged=True, seed=4)
    R, T, k = idx.shape
    w = make_weights(wl, 4)
    rng = np.random.default_rng(4)
    recv, src_pos, slot = oracle_lib.route(idx, ntok, wl.experts_per_rank)
    y = rng.standard_normal((R, R * T, wl.hidden)).astype(np.float32)
    w_recv = oracle_lib.place_rows(w, ntok, slot)
    full, full_w = oracle_lib.combine(y, idx, ntok, slot, wl.experts_per_rank, w_recv=w_recv,
                                      weighted=weighted, out_dtype=od)
    toks = np.array([s * T + t for s in range(R) for t in range(int(ntok[s]))], np.int64)
    toks = toks[rng.permutation(len(toks))]
    part, part_w = oracle_lib.combine_tokens(toks, y, idx, slot, wl.experts_per_rank,
                                             w_recv=w_recv, weighted=weighted, out_dtype=od)
    assert np.array_equal(part, full[toks // T, toks % T])
    assert np.array_equal(part_w, full_w[toks // T, toks % T])
    pcap = R * T * k + 127 * wl.experts_per_rank
    lay = oracle_lib.std_layout(idx, ntok, wl.experts_per_rank, pcap)
    Y = rng.standard_normal((R, pcap, wl.hidden)).astype(np.float32)
    sfull = oracle_lib.std_combine(Y, idx, ntok, lay["row_map"], wl.experts_per_rank, w=w,
                                   weighted=weighted, out_dtype=od)
    spart = oracle_lib.std_combine_tokens(toks, Y, idx, lay["row_map"], wl.experts_per_rank,
                                          w=w, weighted=weighted, out_dtype=od)
    assert np.array_equal(spart, sfull[toks // T, toks % T])
