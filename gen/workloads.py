"""Workload definitions and seeded generators.

Shapes follow the DeepSeek-V3 example of the MORI-EP User Guide (section 2,
"DeepSeek V3 example": hidden 7168, 256 experts over 8 ranks, top-8) and its
benchmark table (section 9, 4096 tokens; README "Latency" table, 128 tokens).
Random top-k selection follows the guide's complete example (section 7),
which draws each token's experts as a prefix of a random permutation.

Every generator takes an explicit seed and a stream id so the token payload,
router ids, router weights and expert outputs are independent streams.
Large payloads can be drawn directly on a CUDA device with torch's generator;
the values then differ from the CPU stream but are still a pure function of
(seed, device type), and both sides of a parity check read the same tensor.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np
import torch

_STREAM_IDX = 1
_STREAM_W = 2
_STREAM_X = 3
_STREAM_Y = 4
_STREAM_MASK = 5
_STREAM_OUTLIER = 6


@dataclass(frozen=True)
class Workload:
    name: str
    world_size: int          # simulated EP ranks (R)
    experts_per_rank: int    # E_r
    tokens_per_rank: int     # max_num_inp_token_per_rank (Tmax)
    hidden: int              # H
    topk: int                # k
    dispatch_dtype: str      # "bf16" (copy), "fp8" (OCP E4M3 per-128) or "fp4" (E2M1 per-32)
    combine_out_dtype: str   # "bf16" or "fp32"
    router: str = "uniform"  # "uniform" or "zipf"
    zipf_s: float = 1.2
    mask_prob: float = 0.0   # probability that a top-k slot is dropped (-1)
    token_dist: str = "normal"   # "normal", "normal_outliers", "uniform"
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    expert_output: str = "random"  # "identity" (y = dispatched x) or "random" N(0,1)
    weighted: bool = False
    standard_moe: bool = False
    seed: int = 0

    @property
    def num_experts(self) -> int:
        return self.world_size * self.experts_per_rank

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    # 8 ranks x 4 experts, 16 tokens/rank, hidden 256, top-4, fp32 identity combine
    "tiny": Workload("tiny", 8, 4, 16, 256, 4, "bf16", "fp32",
                     expert_output="identity"),
    # DeepSeek-V3 decode-size batch: 128 tokens/rank, FP8 dispatch, bf16 combine
    "ds_v3_latency": Workload("ds_v3_latency", 8, 32, 128, 7168, 8, "fp8", "bf16"),
    # DeepSeek-V3 prefill-size batch: 4096 tokens/rank, 1% outliers x50
    "ds_v3_throughput": Workload("ds_v3_throughput", 8, 32, 4096, 7168, 8, "fp8", "bf16",
                                 token_dist="normal_outliers", outlier_frac=0.01,
                                 outlier_scale=50.0),
    # Zipf(1.2) expert popularity, bf16 dispatch + per-expert repack, weighted fp32 combine
    "skewed_zipf_std_moe": Workload("skewed_zipf_std_moe", 8, 32, 4096, 7168, 8, "bf16", "fp32",
                                    router="zipf", zipf_s=1.2, weighted=True,
                                    standard_moe=True),
    # the prefill shape with FP4 E2M1 block-32 quantisation in dispatch
    "ds_v3_throughput_fp4": Workload("ds_v3_throughput_fp4", 8, 32, 4096, 7168, 8, "fp4", "bf16",
                                     token_dist="normal_outliers", outlier_frac=0.01,
                                     outlier_scale=50.0),
    # mid-size MoE, 5% of top-k slots dropped, inputs U(-1,1)
    "mid_masked": Workload("mid_masked", 8, 16, 2048, 4096, 8, "bf16", "bf16",
                           mask_prob=0.05, token_dist="uniform"),
}


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream]))


def make_num_tokens(wl: Workload, ragged: bool = False, seed: int | None = None) -> np.ndarray:
    """Tokens held by each source rank: all full, or a seeded ragged mix in [0, Tmax]."""
    if not ragged:
        return np.full(wl.world_size, wl.tokens_per_rank, dtype=np.int32)
    rng = _rng(wl.seed if seed is None else seed, 99)
    n = rng.integers(0, wl.tokens_per_rank + 1, size=wl.world_size).astype(np.int32)
    n[0] = wl.tokens_per_rank          # keep one full rank and one empty rank
    if wl.world_size > 1:
        n[-1] = 0
    return n


def make_indices(wl: Workload, seed: int | None = None) -> np.ndarray:
    """Top-k expert ids, int32 [R, Tmax, k]; distinct within a row; -1 = dropped slot.

    uniform: a uniformly random ordered k-subset of the E experts (the prefix of
    a random permutation). zipf: Plackett-Luce sampling without replacement with
    popularity p_e proportional to (e+1)^-s (expert 0 hottest), drawn with the
    Gumbel-top-k construction.
    """
    seed = wl.seed if seed is None else seed
    rng = _rng(seed, _STREAM_IDX)
    R, T, k, E = wl.world_size, wl.tokens_per_rank, wl.topk, wl.num_experts
    n = R * T
    if wl.router == "uniform":
        keys = rng.random((n, E))
    elif wl.router == "zipf":
        logp = -wl.zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
        keys = logp[None, :] + rng.gumbel(size=(n, E))
    else:
        raise ValueError(wl.router)
    top = np.argpartition(-keys, k - 1, axis=1)[:, :k]
    order = np.argsort(-np.take_along_axis(keys, top, axis=1), axis=1, kind="stable")
    ids = np.take_along_axis(top, order, axis=1).astype(np.int32)
    if wl.mask_prob > 0:
        drop = _rng(seed, _STREAM_MASK).random((n, k)) < wl.mask_prob
        ids[drop] = -1
    return np.ascontiguousarray(ids.reshape(R, T, k))


def make_weights(wl: Workload, seed: int | None = None) -> np.ndarray:
    """Router weights, f32 [R, Tmax, k]: softmax (in f64) of k iid N(0,1) logits."""
    seed = wl.seed if seed is None else seed
    rng = _rng(seed, _STREAM_W)
    R, T, k = wl.world_size, wl.tokens_per_rank, wl.topk
    z = rng.standard_normal((R, T, k))
    z = np.exp(z - z.max(axis=-1, keepdims=True))
    return (z / z.sum(axis=-1, keepdims=True)).astype(np.float32)


def _to_bf16(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.bfloat16)


def make_tokens(wl: Workload, seed: int | None = None, device: str | torch.device = "cpu") -> torch.Tensor:
    """Token payload, bf16 [R, Tmax, H] = round-to-nearest-even of an f32 sample."""
    seed = wl.seed if seed is None else seed
    R, T, H = wl.world_size, wl.tokens_per_rank, wl.hidden
    dev = torch.device(device)
    if dev.type == "cpu":
        rng = _rng(seed, _STREAM_X)
        if wl.token_dist == "uniform":
            x = rng.uniform(-1.0, 1.0, size=(R, T, H)).astype(np.float32)
        else:
            x = rng.standard_normal((R, T, H), dtype=np.float32)
            if wl.token_dist == "normal_outliers":
                hit = _rng(seed, _STREAM_OUTLIER).random((R, T, H)) < wl.outlier_frac
                x[hit] *= np.float32(wl.outlier_scale)
        return _to_bf16(torch.from_numpy(x))
    g = torch.Generator(device=dev)
    g.manual_seed(seed * 1000 + _STREAM_X)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device=dev)
    for r in range(R):  # per rank to bound the f32 temporary
        if wl.token_dist == "uniform":
            xr = torch.rand((T, H), generator=g, device=dev, dtype=torch.float32) * 2.0 - 1.0
        else:
            xr = torch.randn((T, H), generator=g, device=dev, dtype=torch.float32)
            if wl.token_dist == "normal_outliers":
                hit = torch.rand((T, H), generator=g, device=dev) < wl.outlier_frac
                xr = torch.where(hit, xr * wl.outlier_scale, xr)
        out[r] = _to_bf16(xr)
    return out


def make_expert_outputs(wl: Workload, rows_per_rank: int, seed: int | None = None,
                        device: str | torch.device = "cpu",
                        dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """Stand-in expert outputs, [R, rows_per_rank, H] ~ N(0,1) rounded to `dtype`.

    Drawn for every row of the receive capacity, independent of the routing,
    so the same tensor serves any recv layout.
    """
    seed = wl.seed if seed is None else seed
    R, H = wl.world_size, wl.hidden
    dev = torch.device(device)
    if dev.type == "cpu":
        rng = _rng(seed, _STREAM_Y)
        y = rng.standard_normal((R, rows_per_rank, H), dtype=np.float32)
        return torch.from_numpy(y).to(dtype)
    g = torch.Generator(device=dev)
    g.manual_seed(seed * 1000 + _STREAM_Y)
    out = torch.empty((R, rows_per_rank, H), dtype=dtype, device=dev)
    for r in range(R):
        out[r] = torch.randn((rows_per_rank, H), generator=g, device=dev,
                             dtype=torch.float32).to(dtype)
    return out
