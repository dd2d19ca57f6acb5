"""Launch-parameter tuning files and the tuner that writes them.

The MORI-EP User Guide, section 10 (Tuning), describes a tuner that sweeps
block_num / warp_per_block for each (kernel, dtype, num_tokens, hidden_dim),
keeps the fastest, and saves rules to JSON files that auto mode (section 6,
Launch Configuration) reads at run time. This module does the same for the
kernels of this library on one GPU:

* files: ``<dir>/sm103_gb300_<kernel>_ep<R>_<phase>.json`` with ``kernel``
  "2d" (receive layout) or "stdmoe" (packed layout) and ``phase`` "dispatch"
  or "combine"; ``<dir>`` is ``tuning_configs/`` beside this module, or the
  directory named by ``EP_TUNING_CONFIG_DIR``;
* rules: one per (dtype, hidden_dim, num_tokens), sorted by that key, with
  ``impl`` ("vector" or "bulk"), ``block_num`` (<= 0: one occupancy-sized
  wave), ``warp_per_block``, and the measured ``latency_us`` and
  ``bandwidth_gbps`` (recorded for readers; only the launch fields are used);
* lookup: among the rules of the same dtype and hidden_dim, the one with the
  smallest num_tokens >= the batch's tokens per rank, else the largest;
* saving replaces the rule with the same key and prints the old and new one.

The tuner times each candidate with CUDA events on the current stream, with
the L2 evicted (a 256 MB read) before every timed launch, and keeps the
lowest median. Launch parameters never change results, only speed.

Usage: ``python -m combine_route_layout_gb300.tuning --ep 8 --experts-per-rank 32
--topk 8 --hidden 7168 --dtype fp8 --tokens 128,1024,4096 [--scope full]``.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics

GPU_TAG = "sm103_gb300"
_HERE = os.path.dirname(os.path.abspath(__file__))

# candidate launch parameters (block_num <= 0: one occupancy-sized wave)
SCOPES = {
    "quick": {"grids": [-1, 304, 608, 1216], "warps": [4, 8], "bulk_grids": [-1, 456, 912]},
    "full": {"grids": [-1, 152, 304, 456, 608, 912, 1216, 2432], "warps": [2, 4, 8],
             "bulk_grids": [-1, 152, 304, 456, 608, 912, 1216]},
}


def config_dir() -> str:
    return os.environ.get("EP_TUNING_CONFIG_DIR") or os.path.join(_HERE, "tuning_configs")


def rules_path(kernel: str, ep_size: int, phase: str, directory: str | None = None) -> str:
    d = directory or config_dir()
    return os.path.join(d, f"{GPU_TAG}_{kernel}_ep{ep_size}_{phase}.json")


def dispatch_dtype_name(cfg) -> str:
    """Dtype key of the dispatch phase: the payload format it writes."""
    import torch
    if cfg.quant_type == "fp8_e4m3_block128":
        return "fp8"
    if cfg.quant_type == "fp4_e2m1_block32":
        return "fp4"
    return {torch.bfloat16: "bf16", torch.float32: "fp32",
            torch.float8_e4m3fn: "fp8_passthrough"}.get(cfg.data_type, "fp4_passthrough")


def combine_dtype_name(cfg) -> str:
    """Dtype key of the combine phase: the expert-output dtype it reads."""
    import torch
    return "fp32" if cfg.combine_dtype == torch.float32 else "bf16"


def load_rules(kernel: str, ep_size: int, phase: str, directory: str | None = None) -> list:
    p = rules_path(kernel, ep_size, phase, directory)
    if not os.path.exists(p):
        return []
    with open(p) as f:
        return json.load(f).get("rules", [])


def lookup(rules: list, dtype: str, hidden_dim: int, num_tokens: int):
    """The rule for a batch of num_tokens tokens per rank, or None."""
    cand = [r for r in rules if r["dtype"] == dtype and r["hidden_dim"] == hidden_dim]
    if not cand:
        return None
    above = [r for r in cand if r["num_tokens"] >= num_tokens]
    if above:
        return min(above, key=lambda r: r["num_tokens"])
    return max(cand, key=lambda r: r["num_tokens"])


def save_rule(kernel: str, ep_size: int, phase: str, rule: dict,
              directory: str | None = None) -> str:
    """Insert or replace `rule` (keyed by dtype, hidden_dim, num_tokens)."""
    p = rules_path(kernel, ep_size, phase, directory)
    doc = {"version": "1.0", "gpu": GPU_TAG, "kernel_type": kernel, "ep_size": ep_size,
           "phase": phase, "rules": []}
    if os.path.exists(p):
        with open(p) as f:
            doc = json.load(f)
    key = (rule["dtype"], rule["hidden_dim"], rule["num_tokens"])
    old = [r for r in doc["rules"] if (r["dtype"], r["hidden_dim"], r["num_tokens"]) == key]
    if old:
        print(f"replace {key}: {old[0]} -> {rule}")
    doc["rules"] = [r for r in doc["rules"]
                    if (r["dtype"], r["hidden_dim"], r["num_tokens"]) != key] + [rule]
    doc["rules"].sort(key=lambda r: (r["dtype"], r["hidden_dim"], r["num_tokens"]))
    os.makedirs(os.path.dirname(p), exist_ok=True)
    with open(p, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")
    return p


# ---------------------------------------------------------------- the tuner

def _candidates(phase: str, cfg, scope: str):
    sc = SCOPES[scope]
    out = [("vector", g, w) for g in sc["grids"] for w in sc["warps"]]
    bulk_ok = (phase == "combine" and
               (cfg.num_experts_per_token if cfg.standard_moe else cfg.world_size) <= 8) or \
              (phase == "dispatch" and cfg.quant_type == "none")
    if bulk_ok:
        out += [("bulk", g, 8) for g in sc["bulk_grids"]]
    return out


def tune_shape(cfg, phase: str, scope: str = "quick", iters: int = 20, seed: int = 0):
    """Sweep one (config, phase) on the current GPU; returns the best rule."""
    import torch
    from .ep import EP_PHASE_COMBINE, EP_PHASE_DISPATCH, EpDispatchCombineOp

    dev = torch.device("cuda")
    R, T, H = cfg.world_size, cfg.max_num_inp_token_per_rank, cfg.hidden_dim
    k, E = cfg.num_experts_per_token, cfg.world_size * cfg.num_experts_per_rank
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    # uniformly random distinct top-k ids, softmax weights, N(0,1) payloads
    idx = torch.rand((R * T, E), generator=g, device=dev).argsort(dim=1)[:, :k]
    idx = idx.to(torch.int32).reshape(R, T, k).contiguous()
    w = torch.softmax(torch.randn((R, T, k), generator=g, device=dev), dim=-1)
    x = torch.randn((R, T, H), generator=g, device=dev).to(cfg.data_type)
    op = EpDispatchCombineOp(cfg, use_tuning_files=False)  # the candidates set the launch
    ph = EP_PHASE_DISPATCH if phase == "dispatch" else EP_PHASE_COMBINE
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    st = torch.cuda.current_stream()

    def run_dispatch():
        if cfg.standard_moe:
            return op.dispatch_standard_moe(x, w, None, idx)
        return op.dispatch(x, w, None, idx)

    # expert outputs: the dispatched rows (any values serve for timing)
    d = run_dispatch()
    if cfg.standard_moe:
        y = torch.randn((d["packed_recv_x"].shape[0], H), generator=g, device=dev,
                        dtype=cfg.combine_dtype)   # every row of the packed pool
        n_rows = int((idx >= 0).sum())   # valid (token, slot) pairs; padding rows excluded
    else:
        y = torch.randn((R, op.cap, H), generator=g, device=dev, dtype=cfg.combine_dtype)
        n_rows = int(d[4].sum())
    op.reset()
    # algorithmic bytes of the phase (the same formulas as bench.py)
    row = {"fp8": H + 4 * (H // 128), "fp4": H // 2 + 4 * (H // 32)}.get(
        dispatch_dtype_name(cfg), H * x.element_size())
    yb = y.element_size()
    bo = 4 if cfg.combine_out_dtype == torch.float32 else 2
    if phase == "dispatch":
        nbytes = R * T * (H * x.element_size() + 8 * k) + n_rows * (
            (row + 4) if cfg.standard_moe else (row + 8 * k + 4))
    else:
        nbytes = (n_rows * (H * yb + 4) + R * T * (8 * k + bo * H) if cfg.standard_moe
                  else n_rows * (H * yb + 4 * k + 4) + R * T * (H * bo + 4 * k))

    def one(timed: bool):
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        torch.sum(flush, dim=0, out=sink)
        if phase == "dispatch" and timed:
            ev[0].record(st)
        dd = run_dispatch()
        if phase == "dispatch" and timed:
            ev[1].record(st)
        if phase == "combine":
            torch.sum(flush, dim=0, out=sink)
            if timed:
                ev[0].record(st)
        if cfg.standard_moe:
            op.combine_standard_moe(y, w, idx, call_reset=True)
        else:
            op.combine(y, dd[1], idx, call_reset=True, want_weights=False)
        if phase == "combine" and timed:
            ev[1].record(st)
        return ev

    results = []
    for impl, grid, warps in _candidates(phase, cfg, scope):
        op.set_launch_config(ph, impl, grid, warps)
        for _ in range(3):
            one(False)
        evs = [one(True) for _ in range(iters)]
        torch.cuda.synchronize()
        us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs)
        results.append((us, impl, grid, warps))
    us, impl, grid, warps = min(results)
    dt = dispatch_dtype_name(cfg) if phase == "dispatch" else combine_dtype_name(cfg)
    return {"dtype": dt, "num_tokens": T, "hidden_dim": H, "impl": impl, "block_num": grid,
            "warp_per_block": warps, "latency_us": round(us, 2),
            "bandwidth_gbps": round(nbytes / (us * 1e-6) / 1e9, 1),
            "candidates": len(results)}


def main(argv=None):
    import torch
    from .ep import EpDispatchCombineConfig
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--ep", type=int, default=8, help="simulated ranks (world_size)")
    ap.add_argument("--experts-per-rank", type=int, default=32)
    ap.add_argument("--topk", type=int, default=8)
    ap.add_argument("--hidden", type=int, default=7168)
    ap.add_argument("--dtype", default="fp8", choices=["bf16", "fp8", "fp4"],
                    help="dispatch payload (bf16 = copy)")
    ap.add_argument("--combine-dtype", default="bf16", choices=["bf16", "fp32"])
    ap.add_argument("--standard-moe", action="store_true")
    ap.add_argument("--tokens", default="128,1024,4096", help="tokens per rank, comma-separated")
    ap.add_argument("--phase", default="both", choices=["dispatch", "combine", "both"])
    ap.add_argument("--scope", default=os.environ.get("EP_TUNING_SCOPE", "quick"),
                    choices=list(SCOPES))
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--out", default=None, help="directory for the rule files")
    a = ap.parse_args(argv)
    kernel = "stdmoe" if a.standard_moe else "2d"
    phases = ["dispatch", "combine"] if a.phase == "both" else [a.phase]
    for t in [int(v) for v in a.tokens.split(",")]:
        cfg = EpDispatchCombineConfig(
            data_type=torch.bfloat16, world_size=a.ep, hidden_dim=a.hidden, scale_dim=0,
            scale_type_size=4, max_token_type_size=4, max_num_inp_token_per_rank=t,
            num_experts_per_rank=a.experts_per_rank, num_experts_per_token=a.topk,
            quant_type={"fp8": "fp8_e4m3_block128", "fp4": "fp4_e2m1_block32"}.get(a.dtype,
                                                                                "none"),
            combine_dtype=torch.float32 if a.combine_dtype == "fp32" else torch.bfloat16,
            weighted_combine=a.standard_moe, standard_moe=a.standard_moe,
            # uniform routing puts about T*k rows on a rank: room for 1.5x that
            max_packed_rows_per_rank=(3 * t * a.topk // 2 + 128 * a.experts_per_rank
                                      if a.standard_moe else 0))
        for phase in phases:
            rule = tune_shape(cfg, phase, a.scope, a.iters)
            path = save_rule(kernel, a.ep, phase, rule, a.out)
            print(json.dumps({"phase": phase, "file": os.path.basename(path), **rule}),
                  flush=True)
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
