"""Shared helpers for the GPU parity tests: run a workload through libep and
through the CPU oracle on the same seeded inputs and compare.

Comparisons are bit-exact: routing metadata, payload bytes, FP8 codes and
scales are integers or bit copies, and both combines reduce in the same
fixed order with one final rounding, so the f32/bf16 outputs must agree bit
for bit (stricter than the 1 bf16 ulp / 1e-6 relative bound the method allows).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from combine_route_layout_gb300 import EpDispatchCombineConfig, EpDispatchCombineOp
from gen import make_expert_outputs, make_indices, make_num_tokens, make_tokens, make_weights

DEV = "cuda"


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def make_config(wl, **over) -> EpDispatchCombineConfig:
    kw = dict(
        data_type=torch.bfloat16, world_size=wl.world_size, hidden_dim=wl.hidden, scale_dim=0,
        scale_type_size=4, max_token_type_size=4, max_num_inp_token_per_rank=wl.tokens_per_rank,
        num_experts_per_rank=wl.experts_per_rank, num_experts_per_token=wl.topk,
        quant_type={"fp8": "fp8_e4m3_block128", "fp4": "fp4_e2m1_block32"}.get(wl.dispatch_dtype,
                                                                            "none"),
        combine_dtype=torch.bfloat16,
        combine_out_dtype=torch.float32 if wl.combine_out_dtype == "fp32" else torch.bfloat16,
        weighted_combine=wl.weighted, standard_moe=wl.standard_moe)
    kw.update(over)
    return EpDispatchCombineConfig(**kw)


class Inputs:
    def __init__(self, wl, seed=None, ragged=False, device_payload=None):
        seed = wl.seed if seed is None else seed
        self.wl = wl
        self.idx = make_indices(wl, seed)
        self.w = make_weights(wl, seed)
        self.ntok = make_num_tokens(wl, ragged=ragged, seed=seed)
        big = wl.world_size * wl.tokens_per_rank * wl.hidden > 64 * 1024 * 1024
        on_dev = big if device_payload is None else device_payload
        self.x = make_tokens(wl, seed, device=DEV if on_dev else "cpu").to(DEV)
        self.idx_d = torch.from_numpy(self.idx).to(DEV)
        self.w_d = torch.from_numpy(self.w).to(DEV)

    def x_bits(self, rows=None) -> np.ndarray:
        """bf16 bits of the payload on the host ([R, T, H] or selected [n, H] rows)."""
        if rows is None:
            return bits16(self.x)
        s, t = rows
        return bits16(self.x[torch.as_tensor(s, device=DEV), torch.as_tensor(t, device=DEV)])


def oracle_quant(cfg, xb: np.ndarray):
    """The oracle's codes and block scales for the config's quantisation."""
    if cfg.quant_type == "fp8_e4m3_block128":
        return oracle.quant_tokens(xb)
    return oracle.quant_tokens_fp4(xb)


def check_route(inp: Inputs, recv_d, src_pos_d):
    wl = inp.wl
    recv, src_pos, slot = oracle.route(inp.idx, inp.ntok, wl.experts_per_rank)
    assert np.array_equal(host(recv_d), recv), "recv_num_token"
    sp = host(src_pos_d)
    for r in range(wl.world_size):
        assert np.array_equal(sp[r, :recv[r]], src_pos[r, :recv[r]]), f"src_token_pos rank {r}"
    return recv, src_pos, slot


def sample_rows(recv, n_per_rank, seed=0):
    rng = np.random.default_rng(seed)
    out = []
    for r, n in enumerate(recv):
        if n == 0:
            continue
        m = min(int(n), n_per_rank)
        rows = np.sort(rng.choice(int(n), size=m, replace=False))
        rows[-1] = n - 1                 # always include the last (tail) row
        rows[0] = 0
        out += [(r, int(i)) for i in np.unique(rows)]
    return out


def sample_tokens(wl, ntok, n, seed=0):
    rng = np.random.default_rng(seed + 17)
    g = [s * wl.tokens_per_rank + t for s in range(wl.world_size) for t in range(int(ntok[s]))]
    g = np.array(g, np.int64)
    if len(g) <= n:
        return g
    pick = np.sort(rng.choice(len(g), size=n, replace=False))
    return np.unique(np.concatenate([g[pick], g[:1], g[-1:]]))


# ----------------------------------------------------- standard-MoE packed pool

def std_pcap(wl) -> int:
    """Per-rank capacity of the oracle's [R][pcap] packed arrays: the worst
    case of one rank (every token of every rank on all of its experts)."""
    return wl.world_size * wl.tokens_per_rank * min(wl.topk, wl.experts_per_rank) + \
        127 * wl.experts_per_rank


def std_pool_rows(wl) -> int:
    """Rows of the library's packed pool by default: one per (token, slot)
    plus 127 padding rows per expert."""
    return wl.world_size * wl.tokens_per_rank * wl.topk + 127 * wl.num_experts


def pool_to_ranks(pool: np.ndarray, base, rows, pcap: int, fill=0) -> np.ndarray:
    """A host copy of a packed-pool array [pool rows, ...] rearranged as the
    oracle's [R][pcap, ...]: rank r's rows base[r] .. base[r] + rows[r] - 1 at
    the start of its slot, `fill` after them."""
    R = len(base)
    out = np.full((R, pcap) + pool.shape[1:], fill, dtype=pool.dtype)
    for r in range(R):
        out[r, :rows[r]] = pool[base[r]:base[r] + rows[r]]
    return out


def oracle_rows_to_pool(orow: np.ndarray, base, pcap: int) -> np.ndarray:
    """The oracle's packed row numbers (r * pcap + row) as pool rows
    (base[r] + row); -1 stays -1."""
    orow = np.asarray(orow, np.int64)
    r, i = orow // pcap, orow % pcap
    return np.where(orow >= 0, np.asarray(base, np.int64)[np.maximum(r, 0)] + i, -1)
