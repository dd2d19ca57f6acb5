"""Benchmark: MoE expert-parallel dispatch + combine on simulated EP ranks.

One step = ep_dispatch (routing layout + payload kernel) followed by
ep_combine with call_reset (combine kernel), on inputs resident in HBM.
Default workload: DeepSeek-V3 prefill shape from the MORI-EP User Guide's
benchmark table (8 ranks x 32 experts, 4096 tokens/rank, hidden 7168, top-8,
FP8 E4M3 dispatch with per-128 scales, bf16 combine); its inputs are larger
than L2. The 128-token decode shape is also timed (with an L2 flush between
iterations) and reported under "latency_shape".

Prints one JSON line. `--impl reference` times the CPU oracle (plain
single-threaded C) on a bounded sample of the same workload instead.
Multi-GPU (torchrun): every rank runs an independent replica of the
workload on its own GPU (the simulated EP group fits one GPU); value is the
sum over ranks, time the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gen import WORKLOADS, make_expert_outputs, make_indices, make_num_tokens, make_tokens, \
    make_weights  # noqa: E402

METRIC = "dispatch/combine µs and effective GB/s at 128 & 4096 tok/rank; % of HBM peak"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------ byte model

def algorithmic_bytes(wl, C: int, P: int, Ttot: int) -> dict:
    """Bytes each step must move (reads + writes), counted from the routing.

    2D dispatch reads every token once (payload + weights + ids) and writes
    one received row per (token, destination rank): payload, FP8 scales,
    weights, ids and its src_token_pos. 2D combine reads one expert-output row
    plus its weights and slot per copy and writes the token's output row and
    weights. Standard MoE moves one row per valid (token, slot).
    """
    H, k = wl.hidden, wl.topk
    row = {"fp8": H + 4 * (H // 128), "fp4": H // 2 + 4 * (H // 32)}.get(wl.dispatch_dtype, 2 * H)
    bo = 4 if wl.combine_out_dtype == "fp32" else 2
    if not wl.standard_moe:
        d_read = Ttot * (2 * H + 8 * k)
        d_write = C * (row + 8 * k + 4)
        c_read = C * (2 * H + 4 * k + 4)
        c_write = Ttot * (H * bo + 4 * k)
    else:
        d_read = Ttot * (2 * H + 8 * k)
        d_write = P * (row + 4)
        c_read = P * (2 * H + 4) + Ttot * 8 * k
        c_write = Ttot * bo * H
    return {"dispatch": d_read + d_write, "combine": c_read + c_write,
            "dispatch_read": d_read, "dispatch_write": d_write,
            "combine_read": c_read, "combine_write": c_write}


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(kernel_key: str, workload: str):
    """Per-launch DRAM bytes from a committed one-pass ncu capture of this
    phase's kernel on this workload (profiles/traffic.json), if none of the
    kernel's source files has changed since it was captured."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)[f"{kernel_key}:{workload}"]
        m = hashlib.sha256()
        for src in rec["sources"]:
            m.update(open(os.path.join(ROOT, src), "rb").read())
        if m.hexdigest()[:16] != rec["sources_sha256_16"]:
            return None
        return rec
    except Exception:
        return None


# ----------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.result = None
        if not self.proc:
            return
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if sm:
            self.result = {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax,
                           "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------- our arm

COMBINE_IMPL = "auto"
DISPATCH_IMPL = "auto"
E2E_STREAMS = 2


LAUNCH = {"block_num": -1, "warp_num_per_block": 8}
LAUNCH_MODE = "manual"   # "auto": per-shape rules from the library's tuning files


def make_op(wl, device):
    from combine_route_layout_gb300 import EpDispatchCombineConfig, EpDispatchCombineOp
    cfg = EpDispatchCombineConfig(
        data_type=torch.bfloat16, world_size=wl.world_size, hidden_dim=wl.hidden, scale_dim=0,
        scale_type_size=4, max_token_type_size=4,
        max_num_inp_token_per_rank=wl.tokens_per_rank,
        num_experts_per_rank=wl.experts_per_rank, num_experts_per_token=wl.topk,
        quant_type={"fp8": "fp8_e4m3_block128", "fp4": "fp4_e2m1_block32"}.get(wl.dispatch_dtype,
                                                                            "none"),
        combine_dtype=torch.bfloat16,
        combine_out_dtype=torch.float32 if wl.combine_out_dtype == "fp32" else torch.bfloat16,
        weighted_combine=wl.weighted, standard_moe=wl.standard_moe, combine_impl=COMBINE_IMPL,
        dispatch_impl=DISPATCH_IMPL, block_num=LAUNCH["block_num"],
        warp_num_per_block=LAUNCH["warp_num_per_block"], launch_config_mode=LAUNCH_MODE)
    return EpDispatchCombineOp(cfg, device)


def chosen_kernels(step) -> dict:
    """The dispatch and combine kernels the library ran for this step, from
    the handle's launch configuration and the library's automatic rules (bulk
    copies from 8192 source tokens: 2D combine with up to 8 ranks, copy-mode
    dispatch)."""
    from combine_route_layout_gb300 import ep as E
    wl = step.wl
    dimpl = step.op.get_launch_config(E.EP_PHASE_DISPATCH)[0]
    cimpl = step.op.get_launch_config(E.EP_PHASE_COMBINE)[0]
    many = step.Ttot >= 8192
    cb_ok = (wl.topk if wl.standard_moe else wl.world_size) <= 8
    cbulk = cb_ok and cimpl != "vector" and (cimpl == "bulk" or (many and not wl.standard_moe))
    quant = wl.dispatch_dtype in ("fp8", "fp4")
    dbulk = not quant and dimpl != "vector" and (dimpl == "bulk" or many)
    return {"combine": "combine_bulk_kernel" if cbulk else
            ("combine_std_kernel" if wl.standard_moe else "combine_2d_kernel"),
            "dispatch": "dispatch_quant_kernel" if quant else
            ("dispatch_bulk_copy_kernel" if dbulk else "dispatch_copy_kernel")}


class Step:
    """Device-resident inputs and one dispatch + combine step."""

    def __init__(self, wl, device, seed=0):
        self.wl = wl
        self.dev = device
        self.op = make_op(wl, device)
        self.x = make_tokens(wl, seed, device=device)
        self.idx = torch.from_numpy(make_indices(wl, seed)).to(device)
        self.w = torch.from_numpy(make_weights(wl, seed)).to(device)
        from combine_route_layout_gb300 import ep as _ep
        self.ntok = make_num_tokens(wl)
        self.ntok_c = _ep._i32_array(self.ntok)
        R, T = wl.world_size, wl.tokens_per_rank
        if wl.standard_moe:
            v = self.op.dispatch_standard_moe(self.x, self.w, None, self.idx, self.ntok)
            torch.cuda.synchronize()
            self.counts = v["packed_recv_count"].sum().item()
            self.rank_rows = v["rank_rows"].cpu().numpy()
            rows = self.op.pcap
        else:
            d = self.op.dispatch(self.x, self.w, None, self.idx, self.ntok)
            torch.cuda.synchronize()
            self.recv = d[4].cpu().numpy()
            rows = R * T
        self.op.reset()
        self.op.sync()
        if wl.standard_moe:   # expert outputs for every row of the packed pool, [pool, H]
            self.y = make_expert_outputs(wl.with_(world_size=1), rows, seed, device=device)[0]
        else:
            self.y = make_expert_outputs(wl, rows, seed, device=device)
        self.out = torch.empty((R, T, wl.hidden),
                               dtype=torch.float32 if wl.combine_out_dtype == "fp32"
                               else torch.bfloat16, device=device)
        self.out_w = torch.empty((R, T, wl.topk), dtype=torch.float32, device=device)
        Ttot = int(self.ntok.sum())
        C = 0 if wl.standard_moe else int(self.recv.sum())
        P = int(self.counts) if wl.standard_moe else 0
        self.bytes = algorithmic_bytes(wl, C, P, Ttot)
        self.C, self.P, self.Ttot = C, P, Ttot

    def dispatch(self, x=None, w=None, idx=None):
        x = self.x if x is None else x
        w = self.w if w is None else w
        idx = self.idx if idx is None else idx
        if self.wl.standard_moe:
            return self.op.dispatch_standard_moe(x, w, None, idx, self.ntok_c)
        return self.op.dispatch(x, w, None, idx, self.ntok_c)

    def combine(self, d, y=None, w=None):
        y = self.y if y is None else y
        if self.wl.standard_moe:
            self.op.combine_standard_moe(y, self.w if w is None else w, None, out=self.out,
                                         call_reset=True)
        else:
            self.op.combine(y, d[1], None, out=self.out, out_weights=self.out_w, call_reset=True)


def time_steps(step: Step, K: int, W: int, flush: torch.Tensor | None, dist_barrier):
    st = torch.cuda.current_stream()
    for _ in range(W):
        d = step.dispatch()
        step.combine(d)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    flush_sink = torch.empty((), dtype=torch.float32, device=step.dev) if flush is not None else None
    dist_barrier()
    torch.cuda.synchronize()
    t0.record(st)
    for i in range(K):
        if flush is not None:
            # evict L2 between iterations (outside the kernel events) by reading a
            # buffer twice its size: a read leaves clean lines, so the timed kernels
            # pay no write-back for it
            torch.sum(flush, dim=0, out=flush_sink)
        ev[i][0].record(st)
        d = step.dispatch()
        ev[i][1].record(st)
        step.combine(d)
        ev[i][2].record(st)
    t1.record(st)
    torch.cuda.synchronize()
    dist_barrier()
    total_ms = t0.elapsed_time(t1)
    disp = [e[0].elapsed_time(e[1]) for e in ev]
    comb = [e[1].elapsed_time(e[2]) for e in ev]
    return total_ms, disp, comb


def event_floor_us(dev, iters: int, flush: torch.Tensor) -> dict:
    """What CUDA events read around one and around two back-to-back
    one-element kernels, after the same L2-evicting read as the decode-shape
    steps: the fixed launch and event cost inside every such measurement."""
    a = torch.zeros(1, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    st = torch.cuda.current_stream()
    out = {}
    for n in (1, 2):
        ts = []
        for i in range(iters + 5):
            torch.sum(flush, dim=0, out=sink)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(n):
                a.add_(1.0)
            e1.record(st)
            torch.cuda.synchronize()
            if i >= 5:
                ts.append(e0.elapsed_time(e1) * 1e3)
        out[f"{n}_kernel{'s' if n > 1 else ''}_us_median"] = round(statistics.median(ts), 2)
    return out


def graph_step_times(step: Step, iters: int, flush: torch.Tensor):
    """Dispatch + combine captured once into a CUDA graph and replayed, with an
    L2-evicting read before each replay; returns per-replay device times (µs)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            step.combine(step.dispatch())
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step.combine(step.dispatch())
    sink = torch.empty((), dtype=torch.float32, device=step.dev)
    st = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(iters)]
    for i in range(iters):
        torch.sum(flush, dim=0, out=sink)
        ev[i][0].record(st)
        g.replay()
        ev[i][1].record(st)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e3 for a, b in ev]


def time_e2e(step: Step, K: int, W: int, dist_barrier):
    """Same step through the public API with pinned host inputs: H2D of the
    step's inputs (tokens, weights, ids, the expert-output rows that will be
    read) and D2H of the combined output, all inside the timed region."""
    wl = step.wl
    st = torch.cuda.current_stream()
    xh = step.x.cpu().pin_memory()
    wh = step.w.cpu().pin_memory()
    ih = step.idx.cpu().pin_memory()
    # only the expert-output rows the combine reads travel (the packed pool's
    # ranks are consecutive from row 0)
    yh, ybytes = [], 0
    if wl.standard_moe:
        n = int(step.rank_rows.sum())
        h = step.y[:n].cpu().pin_memory()
        yh.append((None, n, h))
        ybytes += h.numel() * h.element_size()
    for r in range(wl.world_size if not wl.standard_moe else 0):
        n = int(step.recv[r])
        if n == 0:
            continue
        h = step.y[r, :n].cpu().pin_memory()
        yh.append((r, n, h))
        ybytes += h.numel() * h.element_size()
    oh = torch.empty(step.out.shape, dtype=step.out.dtype, pin_memory=True)
    # two device copies of every input: step i uploads into set i % 2 while
    # step i - 1 still computes on the other
    bufs = [{"x": torch.empty_like(step.x), "w": torch.empty_like(step.w),
             "idx": torch.empty_like(step.idx), "y": torch.empty_like(step.y)}
            for _ in range(2)]
    h2d = xh.numel() * xh.element_size() + wh.numel() * 4 + ih.numel() * 4 + ybytes
    d2h = oh.numel() * oh.element_size()

    # Uploads run on their own streams (copy engines) and overlap the
    # previous step's dispatch and combine; the output's device->host copy
    # runs on another and overlaps the next uploads (the link is full
    # duplex). Each step still moves all of its inputs up and its result down.
    up = [torch.cuda.Stream() for _ in range(E2E_STREAMS)]
    down = torch.cuda.Stream()
    done = [None, None]      # combine of the last step that used each input set
    state = {"read": None, "i": 0}

    def one():
        b = state["i"] % 2
        state["i"] += 1
        B = bufs[b]
        for us in up:
            if done[b] is not None:
                us.wait_event(done[b])
        with torch.cuda.stream(up[0]):
            B["x"].copy_(xh, non_blocking=True)
            B["w"].copy_(wh, non_blocking=True)
            B["idx"].copy_(ih, non_blocking=True)
        for j, (r, n, h) in enumerate(yh):
            with torch.cuda.stream(up[(j + 1) % len(up)]):
                (B["y"][:n] if r is None else B["y"][r, :n]).copy_(h, non_blocking=True)
        st.wait_stream(up[0])
        d = step.dispatch(B["x"], B["w"], B["idx"])
        for us in up[1:]:
            st.wait_stream(us)
        if state["read"] is not None:             # the previous output has been read
            st.wait_event(state["read"])
        step.combine(d, y=B["y"], w=B["w"])
        done[b] = torch.cuda.Event()
        done[b].record(st)
        down.wait_event(done[b])
        with torch.cuda.stream(down):
            oh.copy_(step.out, non_blocking=True)
        state["read"] = torch.cuda.Event()
        state["read"].record(down)

    for _ in range(max(2, W)):
        one()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    dist_barrier()
    t0.record(st)
    for us in up + [down]:                        # nothing timed starts before t0
        us.wait_event(t0)
    for _ in range(K):
        one()
    for us in up:
        st.wait_stream(us)
    st.wait_stream(down)                          # the last output is on the host
    t1.record(st)
    torch.cuda.synchronize()
    dist_barrier()
    return t0.elapsed_time(t1), h2d, d2h


def cpu_oracle_step(wl, tokens_per_rank: int, seed: int = 0, y=None):
    """One dispatch + combine of the workload restricted to `tokens_per_rank`
    tokens per source rank, on the CPU oracle. Returns (seconds, bytes)."""
    import oracle
    sw = wl.with_(tokens_per_rank=tokens_per_rank)
    idx = make_indices(sw, seed)
    w = make_weights(sw, seed)
    x = make_tokens(sw, seed).view(torch.int16).numpy().view(np.uint16)
    ntok = make_num_tokens(sw)
    R, T = sw.world_size, sw.tokens_per_rank
    Er = sw.experts_per_rank
    od = "fp32" if sw.combine_out_dtype == "fp32" else "bf16"
    if sw.standard_moe:
        pcap = R * T * min(sw.topk, Er) + 127 * Er
        if y is None:
            y = make_expert_outputs(sw, pcap, seed).view(torch.int16).numpy().view(np.uint16)
        t = time.perf_counter()
        res = oracle.std_dispatch(x, idx, ntok, Er, pcap, quant_fp8=sw.dispatch_dtype == "fp8")
        # (the packed-layout oracle quantises FP8 only; FP4 workloads use the 2D layout)
        oracle.std_combine(y, idx, ntok, res["row_map"], Er, w=w, weighted=sw.weighted,
                           out_dtype=od)
        dt = time.perf_counter() - t
        P = int(res["count"].sum())
        b = algorithmic_bytes(sw, 0, P, int(ntok.sum()))
    else:
        if y is None:
            y = make_expert_outputs(sw, R * T, seed).view(torch.int16).numpy().view(np.uint16)
        t = time.perf_counter()
        d = oracle.dispatch(x, w, idx, ntok, Er, quant_fp8=sw.dispatch_dtype == "fp8",
                            quant_fp4=sw.dispatch_dtype == "fp4")
        oracle.combine(y, idx, ntok, d["slot"], Er, w_recv=d["w"], weighted=sw.weighted,
                       out_dtype=od)
        dt = time.perf_counter() - t
        b = algorithmic_bytes(sw, int(d["recv_num_token"].sum()), 0, int(ntok.sum()))
    return dt, b["dispatch"] + b["combine"], y


def host_cpu():
    """CPU model, logical CPU count and architecture of the host."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                v = line.split(":", 1)[1].strip()
                if v and not v.isdigit():
                    model = v
                    break
    except Exception:
        pass
    return {"model": model or platform.processor() or platform.machine(),
            "nproc": os.cpu_count(), "arch": platform.machine()}


class pinned_core:
    """Run the enclosed CPU work on one core (the first this process may use)."""

    def __enter__(self):
        self.before = os.sched_getaffinity(0)
        self.core = min(self.before)
        os.sched_setaffinity(0, {self.core})
        return self

    def __exit__(self, *a):
        os.sched_setaffinity(0, self.before)


def pctl(xs, q):
    return float(np.percentile(np.asarray(xs, dtype=np.float64), q))


def cpu_baseline(wl, sample_tokens: int, reps: int):
    """The oracle (single-threaded C) on `reps` dispatch + combine passes of the
    workload restricted to `sample_tokens` tokens per rank, pinned to one core."""
    dts, bys, y = [], [], None
    with pinned_core() as pc:
        for _ in range(reps):
            dt, by, y = cpu_oracle_step(wl, sample_tokens, y=y)
            dts.append(dt)
            bys.append(by)
    gbs = sum(bys) / sum(dts) / 1e9
    per = [b / t / 1e9 for b, t in zip(bys, dts)]
    cpu = host_cpu()
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "pinned_core": pc.core, "cpu_model": cpu["model"], "nproc": cpu["nproc"],
            "arch": cpu["arch"], "pass_GBps_p10": round(pctl(per, 10), 4),
            "pass_GBps_p90": round(pctl(per, 90), 4),
            "sample": f"{wl.name} restricted to {sample_tokens} tokens/rank "
                      f"({wl.world_size * sample_tokens} tokens), {reps} dispatch+combine "
                      f"passes, single-threaded C on one pinned core, {sum(dts):.1f} s"}


# tokens/rank of each workload's CPU-oracle sample (about a second or two of C)
CPU_SAMPLE_TOKENS = {"tiny": 16, "ds_v3_latency": 128, "ds_v3_throughput": 128,
                     "skewed_zipf_std_moe": 96, "mid_masked": 256, "ds_v3_throughput_fp4": 128}
ALL_WORKLOADS = ("tiny", "ds_v3_latency", "ds_v3_throughput", "skewed_zipf_std_moe", "mid_masked")


def path_dtype(wl) -> str:
    d = {"fp8": "fp8_e4m3 dispatch (f32 quantisation)",
         "fp4": "fp4_e2m1 dispatch (f32 quantisation)"}.get(wl.dispatch_dtype, "bf16 dispatch")
    comb = "weighted " if wl.weighted else ""
    return f"{d}, bf16 {comb}combine, f32 accumulate, {wl.combine_out_dtype} out"


def time_workload(wl, dev, K: int, W: int, cpu_reps: int, with_cpu: bool):
    """One workload: dispatch and combine µs (median, p10, p90) with CUDA
    events, GB/s and fraction of the measured HBM peak, plus the oracle's
    baseline on a sample of the same workload. Inputs of the small workloads
    fit in L2, so a 256 MB read evicts it before each step (outside the
    events); the large ones exceed L2."""
    step = Step(wl, dev)
    small = step.Ttot * wl.hidden * 2 < 128 * 1024 * 1024
    flush = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev) if small else None
    _, disp, comb = time_steps(step, K, W, flush, lambda: None)
    peak, _ = hbm_peak()
    b = step.bytes
    rec = {"tokens_per_rank": wl.tokens_per_rank, "world_size": wl.world_size,
           "hidden": wl.hidden, "topk": wl.topk, "dtype": path_dtype(wl),
           "standard_moe": wl.standard_moe, "copies_C": step.C, "packed_rows_P": step.P,
           "kernels": chosen_kernels(step), "iters": K,
           "l2": "flushed (256 MB read) before each step" if small else "inputs larger than L2"}
    kern = chosen_kernels(step)
    for name, ts in (("dispatch", disp), ("combine", comb)):
        us = [t * 1e3 for t in ts]
        med = statistics.median(us)
        gbs = b[name] / (med * 1e-6) / 1e9
        rec[name] = {"us_median": round(med, 2), "us_p10": round(pctl(us, 10), 2),
                     "us_p90": round(pctl(us, 90), 2), "bytes": b[name], "GBps": round(gbs, 1),
                     "frac_of_peak": round(gbs / peak, 4)}
        tr = profiled_traffic(f"{name}_{'std' if wl.standard_moe else '2d'}", wl.name)
        rec[name]["traffic"] = (tr["dram_bytes_per_launch"]
                                if tr and tr["kernel"].startswith(kern[name]) else None)
    del step, flush
    torch.cuda.empty_cache()
    if with_cpu:
        rec["cpu_baseline"] = cpu_baseline(wl, CPU_SAMPLE_TOKENS.get(wl.name, 64), cpu_reps)
    return rec


# ----------------------------------------------------------- main

def sweep(wl, dev, K: int, W: int):
    """Launch-configuration sweep (the local counterpart of a launch tuner):
    dispatch and combine times over block_num x warp_num_per_block for the
    vector kernels, plus the library's automatic choice. One JSON line."""
    global COMBINE_IMPL, DISPATCH_IMPL
    results = []
    grids = [-1, 152, 304, 456, 608, 912, 1216]
    warps = [4, 8]
    for impl in ("vector", "auto"):
        COMBINE_IMPL = DISPATCH_IMPL = impl
        for bn in (grids if impl == "vector" else [-1]):
            for wp in (warps if impl == "vector" else [8]):
                LAUNCH["block_num"], LAUNCH["warp_num_per_block"] = bn, wp
                step = Step(wl, dev)
                _, disp, comb = time_steps(step, K, W, None, lambda: None)
                results.append({"impl": impl, "block_num": bn, "warp_num_per_block": wp,
                                "dispatch_us": round(statistics.median(disp) * 1e3, 2),
                                "combine_us": round(statistics.median(comb) * 1e3, 2)})
                del step
                torch.cuda.empty_cache()
    LAUNCH["block_num"], LAUNCH["warp_num_per_block"] = -1, 8
    best_d = min(results, key=lambda r: r["dispatch_us"])
    best_c = min(results, key=lambda r: r["combine_us"])
    return {"sweep": wl.name, "results": results, "best_dispatch": best_d,
            "best_combine": best_c}


def convert_leg(wl, dev, K: int, W: int):
    """The standard-MoE layout reached through the 2D path and the two
    conversions (User Guide, section 4): dispatch, convert_dispatch_output,
    convert_combine_input, combine, each timed with CUDA events (inputs
    larger than L2). Algorithmic bytes: convert_dispatch_output reads each
    receive row once and writes one packed row plus its src_info per valid
    (token, slot); convert_combine_input reads every packed row and writes
    one receive row per (token, destination)."""
    from combine_route_layout_gb300 import EpDispatchCombineConfig, EpDispatchCombineOp
    from gen import make_indices, make_num_tokens, make_tokens, make_weights
    R, T, H, k = wl.world_size, wl.tokens_per_rank, wl.hidden, wl.topk
    cfg = EpDispatchCombineConfig(
        data_type=torch.bfloat16, world_size=R, hidden_dim=H, scale_dim=0, scale_type_size=4,
        max_token_type_size=4, max_num_inp_token_per_rank=T,
        num_experts_per_rank=wl.experts_per_rank, num_experts_per_token=k,
        combine_dtype=torch.bfloat16, combine_out_dtype=torch.float32, standard_moe=2)
    op = EpDispatchCombineOp(cfg, dev)
    x = make_tokens(wl, device=dev)
    w = torch.from_numpy(make_weights(wl)).to(dev)
    idx = torch.from_numpy(make_indices(wl)).to(dev)
    ntok = make_num_tokens(wl)
    st = torch.cuda.current_stream()
    d = op.dispatch(x, w, None, idx, ntok)
    px, pcount, psrc, prange = op.convert_dispatch_output(d[0], d[3])
    torch.cuda.synchronize()
    C = int(d[4].sum())
    P = int((idx >= 0).sum())
    y = torch.randn(px.shape, device=dev, dtype=torch.float32).to(torch.bfloat16)
    y2d = op.convert_combine_input(y, psrc, prange)
    op.combine(y2d, d[1], None, call_reset=True)
    torch.cuda.synchronize()
    times = {"dispatch": [], "convert_dispatch_output": [], "convert_combine_input": [],
             "combine": []}
    for it in range(W + K):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        ev[0].record(st)
        d = op.dispatch(x, w, None, idx, ntok)
        ev[1].record(st)
        op.convert_dispatch_output(d[0], d[3])
        ev[2].record(st)
        op.convert_combine_input(y, psrc, prange, out=y2d)
        ev[3].record(st)
        op.combine(y2d, d[1], None, call_reset=True)
        ev[4].record(st)
        torch.cuda.synchronize()
        if it >= W:
            for j, name in enumerate(times):
                times[name].append(ev[j].elapsed_time(ev[j + 1]) * 1e3)
    peak, _ = hbm_peak()
    nbytes = {"convert_dispatch_output": C * 2 * H + P * (2 * H + 4),
              "convert_combine_input": P * 2 * H + C * 2 * H}
    out = {"workload": wl.name, "copies_C": C, "slots_P": P, "steps": K}
    for name, ts in times.items():
        us = statistics.median(ts)
        rec = {"us_median": round(us, 2)}
        if name in nbytes:
            gbs = nbytes[name] / (us * 1e-6) / 1e9
            rec.update(bytes=nbytes[name], GBps=round(gbs, 1), frac_of_peak=round(gbs / peak, 4))
        out[name] = rec
    return out


def split_leg(wl, dev, K: int, W: int):
    """The split send / receive phases with every rank a handle on this GPU
    (User Guide, section 3, split dispatch/combine): dispatch = every rank's
    dispatch_send, then every rank's dispatch_recv; combine = every rank's
    combine_send (zero-copy: the expert outputs are in the registered
    buffers), then every rank's combine_recv. Every rank runs on a stream of
    its own, as ranks on separate GPUs would run side by side; a phase ends
    when all ranks' streams have finished it (events), and no kernel waits
    on another rank's. Bytes as for the single-workspace path (the same
    receive rows and outputs), so GB/s compare directly; the staging and the
    pull's second copy of each row are extra. Eager timing includes the
    host's per-rank launches; the graph timings replay each phase captured
    once."""
    from combine_route_layout_gb300 import EpDispatchCombineConfig
    from combine_route_layout_gb300.ranks import EpRankOp
    R, T = wl.world_size, wl.tokens_per_rank
    cfg = EpDispatchCombineConfig(
        data_type=torch.bfloat16, world_size=R, hidden_dim=wl.hidden, scale_dim=0,
        scale_type_size=4, max_token_type_size=4, max_num_inp_token_per_rank=T,
        num_experts_per_rank=wl.experts_per_rank, num_experts_per_token=wl.topk,
        quant_type={"fp8": "fp8_e4m3_block128", "fp4": "fp4_e2m1_block32"}.get(wl.dispatch_dtype,
                                                                            "none"),
        combine_dtype=torch.bfloat16,
        combine_out_dtype=torch.float32 if wl.combine_out_dtype == "fp32" else torch.bfloat16,
        weighted_combine=wl.weighted)
    ops = [EpRankOp(cfg, r, dev) for r in range(R)]
    ptrs = [op.workspace.data_ptr() for op in ops]
    for op in ops:
        op.set_peers(ptrs)
    x = make_tokens(wl, 0, device=dev)
    idx = torch.from_numpy(make_indices(wl, 0)).to(dev)
    w = torch.from_numpy(make_weights(wl, 0)).to(dev)
    ntok = make_num_tokens(wl)
    y = make_expert_outputs(wl, R * T, 0, device=dev)
    outs = [torch.empty((T, wl.hidden), dtype=cfg.combine_out_dtype, device=dev) for _ in range(R)]

    lanes = [torch.cuda.Stream(device=dev) for _ in range(R)]

    def phase(fn):
        """fn(r, op) on every rank's stream, after all work so far on the
        current stream; the current stream then waits for every rank."""
        cur = torch.cuda.current_stream()
        out = []
        for r, op in enumerate(ops):
            lanes[r].wait_stream(cur)
            with torch.cuda.stream(lanes[r]):
                out.append(fn(r, op))
        for ln in lanes:
            cur.wait_stream(ln)
        return out

    def dispatch():
        views = phase(lambda r, op: op.dispatch_send(x[r], w[r], None, idx[r], int(ntok[r])))
        phase(lambda r, op: op.dispatch_recv())
        return views

    def combine(views):
        # zero-copy: the experts' outputs are already in each rank's registered
        # combine input (written once below, outside the timed region)
        phase(lambda r, op: op.combine_send(None, views[r][1] if wl.weighted else None,
                                            out=outs[r], want_weights=False))
        phase(lambda r, op: op.combine_recv(call_reset=True))

    views = dispatch()
    torch.cuda.synchronize()
    recv = torch.cat([v[4] for v in views]).cpu().numpy()
    for r, op in enumerate(ops):
        op.get_registered_combine_input_buffer()[:int(recv[r])].copy_(y[r, :int(recv[r])])
    combine(views)
    b = algorithmic_bytes(wl, int(recv.sum()), 0, int(ntok.sum()))
    small = int(ntok.sum()) * wl.hidden * 2 < 128 * 1024 * 1024
    flush = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev) if small else None
    sink = torch.empty((), dtype=torch.float32, device=dev)
    st = torch.cuda.current_stream()
    d_us, c_us = [], []
    for it in range(W + K):
        if flush is not None:
            torch.sum(flush, dim=0, out=sink)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(st)
        views = dispatch()
        e[1].record(st)
        combine(views)
        e[2].record(st)
        torch.cuda.synchronize()
        if it >= W:
            d_us.append(e[0].elapsed_time(e[1]) * 1e3)
            c_us.append(e[1].elapsed_time(e[2]) * 1e3)
    # the same phases captured once into CUDA graphs and replayed: device time
    # without the host's per-rank launch overhead
    gd, gc = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(st)
    with torch.cuda.stream(side):
        combine(dispatch())
    st.wait_stream(side)
    torch.cuda.synchronize()
    holder = {}
    with torch.cuda.graph(gd):
        holder["v"] = dispatch()
    with torch.cuda.graph(gc):
        combine(holder["v"])
    gd_us, gc_us = [], []
    for it in range(W + K):
        if flush is not None:
            torch.sum(flush, dim=0, out=sink)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(st)
        gd.replay()
        e[1].record(st)
        gc.replay()
        e[2].record(st)
        torch.cuda.synchronize()
        if it >= W:
            gd_us.append(e[0].elapsed_time(e[1]) * 1e3)
            gc_us.append(e[1].elapsed_time(e[2]) * 1e3)
    peak, _ = hbm_peak()
    rec = {"workload": wl.name, "ranks": R, "iters": K,
           "l2": "flushed (256 MB read) before each step" if small else "inputs larger than L2",
           "graph_dispatch_us_median": round(statistics.median(gd_us), 2),
           "graph_combine_us_median": round(statistics.median(gc_us), 2)}
    # eager: each phase issued rank by rank from Python (16 library calls and
    # their stream forks per step), so at small sizes the host sets the pace;
    # graph: the device time of the same phases
    for name, us, gus in (("dispatch", d_us, gd_us), ("combine", c_us, gc_us)):
        med = statistics.median(us)
        gbs = b[name] / (med * 1e-6) / 1e9
        gmed = statistics.median(gus)
        ggbs = b[name] / (gmed * 1e-6) / 1e9
        rec[name] = {"us_median": round(med, 2), "us_p10": round(pctl(us, 10), 2),
                     "us_p90": round(pctl(us, 90), 2), "GBps": round(gbs, 1),
                     "frac_of_peak": round(gbs / peak, 4),
                     "graph_us_median": round(gmed, 2), "graph_us_p10": round(pctl(gus, 10), 2),
                     "graph_us_p90": round(pctl(gus, 90), 2), "graph_GBps": round(ggbs, 1),
                     "graph_frac_of_peak": round(ggbs / peak, 4)}
    return rec


def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier_fn(world):
    if world <= 1:
        return lambda: None
    import torch.distributed as dist

    def b():
        dist.barrier()
    return b


def reduce_max(v: float, world: int) -> float:
    if world <= 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, wl, rank, world):
    if rank != 0:
        return None
    steps, warm = args.steps, args.warmup
    # per-step sample: --ref-tokens tokens/rank, shrunk so that all steps take
    # about two minutes of oracle time at most (~3.5 ms per token/rank per step)
    T = max(8, min(args.ref_tokens, int(120.0 / (0.0035 * (steps + warm)))))
    y = None
    tot, by = 0.0, 0
    with pinned_core() as pc:
        for _ in range(warm):
            _, _, y = cpu_oracle_step(wl, T, y=y)
        for _ in range(steps):
            dt, b, y = cpu_oracle_step(wl, T, y=y)
            tot += dt
            by += b
    gbs = by / tot / 1e9
    cpu = host_cpu()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": warm,
        "ms_per_step": round(tot / steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": path_dtype(wl), "data": "synthetic",
        "config": {"workload": wl.name, "sample_tokens_per_rank": T, "world_size": wl.world_size,
                   "experts_per_rank": wl.experts_per_rank, "hidden": wl.hidden, "topk": wl.topk},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "pinned_core": pc.core, "cpu_model": cpu["model"],
                         "nproc": cpu["nproc"], "arch": cpu["arch"],
                         "sample": f"{wl.name} restricted to {T} tokens/rank per step, "
                                   f"single-threaded C oracle on one pinned core, "
                                   f"{tot:.1f} s over {steps} steps"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="ds_v3_throughput", choices=sorted(WORKLOADS))
    ap.add_argument("--latency-workload", default="ds_v3_latency")
    ap.add_argument("--combine-impl", default="auto", choices=["auto", "vector", "bulk"])
    ap.add_argument("--convert", action="store_true",
                    help="time the 2D path plus the standard-MoE conversions instead")
    ap.add_argument("--launch-mode", default="manual", choices=["manual", "auto"],
                    help="auto: launch parameters from the library's tuning files")
    ap.add_argument("--dispatch-impl", default="auto", choices=["auto", "vector", "bulk"])
    ap.add_argument("--sweep", action="store_true",
                    help="time dispatch/combine over launch configurations instead")
    ap.add_argument("--split", action="store_true",
                    help="time the split send/receive phases (every rank a handle) instead")
    ap.add_argument("--e2e-streams", type=int, default=2,
                    help="side streams carrying the expert-output H2D copies in the e2e leg")
    ap.add_argument("--tokens-per-rank", type=int, default=0,
                    help="override the workload's tokens per rank (small profiling cases)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-latency", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload lines of the other configs")
    ap.add_argument("--cpu-tokens", type=int, default=256,
                    help="tokens/rank of the headline workload's CPU-oracle sample")
    ap.add_argument("--cpu-reps", type=int, default=3)
    ap.add_argument("--ref-tokens", type=int, default=128,
                    help="tokens/rank per step of the reference (oracle) arm")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    global COMBINE_IMPL, DISPATCH_IMPL, E2E_STREAMS, LAUNCH_MODE
    COMBINE_IMPL = args.combine_impl
    DISPATCH_IMPL = args.dispatch_impl
    LAUNCH_MODE = args.launch_mode
    E2E_STREAMS = max(1, args.e2e_streams)
    rank, world, local = dist_setup(args.gpus)
    wl = WORKLOADS[args.workload]
    if args.tokens_per_rank > 0:
        wl = wl.with_(tokens_per_rank=args.tokens_per_rank)
    if args.impl == "reference":
        line = run_reference(args, wl, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.sweep:
        if rank == 0:
            print(json.dumps(sweep(wl, dev, args.steps, args.warmup)), flush=True)
        return
    if args.split:
        if rank == 0:
            print(json.dumps({"split_path": split_leg(wl, dev, args.steps, args.warmup)}),
                  flush=True)
        return
    if args.convert:
        if rank == 0:
            print(json.dumps({"convert_path": convert_leg(wl, dev, args.steps, args.warmup)}),
                  flush=True)
        return
    barrier = barrier_fn(world)
    step = Step(wl, dev)
    peak, peak_src = hbm_peak()
    with ClockSampler(local) as clk:
        total_ms, disp, comb = time_steps(step, args.steps, args.warmup, None, barrier)
    total_ms = reduce_max(total_ms, world)
    K = args.steps
    per_step = total_ms / K
    b = step.bytes
    step_bytes = b["dispatch"] + b["combine"]
    value = step_bytes * world / (per_step * 1e-3) / 1e9
    d_us = statistics.median(disp) * 1e3
    c_us = statistics.median(comb) * 1e3
    d_mean = statistics.mean(disp) * 1e3
    c_mean = statistics.mean(comb) * 1e3
    d_gbs = b["dispatch"] / (d_mean * 1e-6) / 1e9
    c_gbs = b["combine"] / (c_mean * 1e-6) / 1e9
    dom = "combine" if c_mean >= d_mean else "dispatch"
    dom_key = {"combine": "combine_2d" if not wl.standard_moe else "combine_std",
               "dispatch": "dispatch_2d" if not wl.standard_moe else "dispatch_std"}[dom]
    dom_kernel = chosen_kernels(step)[dom]
    ach = c_gbs if dom == "combine" else d_gbs
    tr = profiled_traffic(dom_key, wl.name)
    if tr and not tr["kernel"].startswith(dom_kernel):
        tr = None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": path_dtype(wl), "data": "synthetic",
        "config": {"workload": wl.name, "world_size": wl.world_size,
                   "experts_per_rank": wl.experts_per_rank, "tokens_per_rank": wl.tokens_per_rank,
                   "hidden": wl.hidden, "topk": wl.topk, "dispatch_payload": wl.dispatch_dtype,
                   "combine_out": wl.combine_out_dtype, "standard_moe": wl.standard_moe,
                   "l2": "inputs larger than L2 (129 MB); no flush",
                   "copies_C": step.C, "packed_rows_P": step.P,
                   "launch_mode": LAUNCH_MODE, "kernels": chosen_kernels(step),
                   "parallelism": f"replicas x{world}, 8 simulated EP ranks each"},
        "dispatch": {"us_median": round(d_us, 2), "us_mean": round(d_mean, 2),
                     "us_p10": round(pctl(disp, 10) * 1e3, 2),
                     "us_p90": round(pctl(disp, 90) * 1e3, 2),
                     "bytes": b["dispatch"], "GBps": round(d_gbs, 1),
                     "frac_of_peak": round(d_gbs / peak, 4)},
        "combine": {"us_median": round(c_us, 2), "us_mean": round(c_mean, 2),
                    "us_p10": round(pctl(comb, 10) * 1e3, 2),
                    "us_p90": round(pctl(comb, 90) * 1e3, 2),
                    "bytes": b["combine"], "GBps": round(c_gbs, 1),
                    "frac_of_peak": round(c_gbs / peak, 4)},
        "roofline": {"bound": "hbm", "kernel": dom_kernel, "achieved": round(ach, 1),
                     "peak": peak, "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "unit": "GB/s", "frac": round(ach / peak, 4),
                     "traffic": tr["dram_bytes_per_launch"] if tr else None},
        "clocks": clk.result,
        "gpu_launches": 3 * K,
    }

    if not args.no_latency and rank == 0:
        lw = WORKLOADS[args.latency_workload]
        ls = Step(lw, dev)
        flush = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
        lk = max(50, K)
        _, ld, lc = time_steps(ls, lk, max(args.warmup, 5), flush, lambda: None)
        lb = ls.bytes
        graph_us = graph_step_times(ls, lk, flush)
        line["latency_shape"] = {
            "workload": lw.name, "iters": lk, "l2": "flushed (256 MB read) before each step",
            "dispatch_us_median": round(statistics.median(ld) * 1e3, 2),
            "combine_us_median": round(statistics.median(lc) * 1e3, 2),
            "dispatch_GBps": round(lb["dispatch"] / (statistics.median(ld) * 1e-3) / 1e9, 1),
            "combine_GBps": round(lb["combine"] / (statistics.median(lc) * 1e-3) / 1e9, 1),
            "graph_step_us": round(statistics.median(graph_us), 2),
            "graph_step_GBps": round((lb["dispatch"] + lb["combine"])
                                     / (statistics.median(graph_us) * 1e-6) / 1e9, 1),
            # events around near-empty kernels under the same protocol (dispatch
            # launches two kernels, combine one)
            "event_floor": event_floor_us(dev, lk, flush),
        }
        del ls, flush

    if not args.no_e2e:
        ke = min(K, 20)  # host-link bound (~18 ms a step): a few steps suffice
        e_ms, h2d, d2h = time_e2e(step, ke, args.warmup, barrier)
        e_ms = reduce_max(e_ms, world)
        line["e2e"] = {"value": round(step_bytes * world / (e_ms / ke * 1e-3) / 1e9, 2),
                       "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                       "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e_ms / ke, 3),
                       "steps": ke}
    if not args.no_workloads and rank == 0:
        # every workload of the method's configs, each with its own CPU-oracle
        # baseline (rank 0 of a single-GPU run only)
        wk = {}
        for name in ALL_WORKLOADS:
            if name == wl.name:
                continue
            wk[name] = time_workload(WORKLOADS[name], dev, max(50, min(K, 100)), args.warmup,
                                     args.cpu_reps, not args.no_cpu_baseline and world == 1)
        line["workloads"] = wk
        # the packed layout reached through the 2D path: both conversions on
        # the Zipf-skewed shape
        line["convert_path"] = convert_leg(WORKLOADS["skewed_zipf_std_moe"], dev, 20, 3)
        # the split send / receive phases, every rank a workspace of its own
        line["split_path"] = [split_leg(WORKLOADS[n], dev, 20, 3)
                              for n in ("ds_v3_latency", "ds_v3_throughput")]
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_tokens, args.cpu_reps)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
