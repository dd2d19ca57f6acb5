"""CPU oracle for MoE expert-parallel dispatch / combine (test infrastructure).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package. It wraps the plain single-threaded C in ep_oracle.c with
numpy arrays; Python here only allocates and composes calls, every value is
computed in the C code. Nothing here is shared with the CUDA library.

Array conventions (R ranks, Tmax tokens per rank, k slots, H hidden):
  x      uint16 [R, Tmax, H]   bf16 bit patterns
  w      float32 [R, Tmax, k]
  idx    int32 [R, Tmax, k]    global expert id, -1 = dropped slot
  ntok   int32 [R]             tokens held by each source rank
Receive buffers have cap = R * Tmax rows per destination rank.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB, build

ORC_OK = 0
ORC_ERR_ARG = -1
ORC_ERR_CAPACITY = -3
ORC_ERR_INDEX = -4
DT_BF16 = 0
DT_F32 = 1

_lib = None


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what} failed with code {code}")
        self.code = code


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            build()
        _lib = ctypes.CDLL(LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        L = ctypes.c_int64
        _lib.oracle_bf16_from_f32.restype = ctypes.c_uint16
        _lib.oracle_bf16_from_f32.argtypes = [ctypes.c_float]
        _lib.oracle_bf16_to_f32.restype = ctypes.c_float
        _lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        _lib.oracle_e4m3_from_f32.restype = ctypes.c_uint8
        _lib.oracle_e4m3_from_f32.argtypes = [ctypes.c_float]
        _lib.oracle_e4m3_to_f32.restype = ctypes.c_float
        _lib.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
        _lib.oracle_e4m3_from_f32_array.argtypes = [P, L, P]
        _lib.oracle_bf16_from_f32_array.argtypes = [P, L, P]
        _lib.oracle_quant_tokens.argtypes = [L, I, P, P, P]
        _lib.oracle_quant_tokens_fp4.argtypes = [L, I, P, P, P]
        _lib.oracle_e2m1_from_f32_array.argtypes = [P, L, P]
        _lib.oracle_e2m1_to_f32.restype = ctypes.c_float
        _lib.oracle_e2m1_to_f32.argtypes = [ctypes.c_uint8]
        _lib.oracle_route.argtypes = [I, I, I, I, P, P, P, P, P]
        _lib.oracle_place_rows.argtypes = [I, I, L, P, P, P, P]
        _lib.oracle_combine.argtypes = [I, I, I, I, I, P, P, P, I, P, P, I, I, P, P]
        _lib.oracle_combine_tokens.argtypes = [I, I, I, I, I, P, L, P, P, I, P, P, I, I, P, P]
        _lib.oracle_std_combine_tokens.argtypes = [I, I, I, I, P, L, P, P, I, P, P, I, I, P]
        _lib.oracle_std_layout.argtypes = [I, I, I, I, L, P, P, P, P, P, P, P, P]
        _lib.oracle_std_place_rows.argtypes = [I, I, I, L, P, P, P, P]
        _lib.oracle_std_combine.argtypes = [I, I, I, I, I, P, P, P, I, P, P, I, I, P]
        _lib.oracle_convert_dispatch_output.argtypes = [I, I, I, I, L, L, P, P, P, P, P, P, P,
                                                        P, P, P, P]
        _lib.oracle_convert_combine_input.argtypes = [I, I, I, I, I, P, P, P, P, I, P, I, P]
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags.c_contiguous, "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(code: int, what: str) -> None:
    if code != ORC_OK:
        raise OracleError(code, what)


def _dt(name_or_dtype) -> int:
    if name_or_dtype in ("bf16", np.uint16):
        return DT_BF16
    if name_or_dtype in ("fp32", np.float32):
        return DT_F32
    raise ValueError(name_or_dtype)


# ------------------------------------------------------------------ codecs

def bf16_from_f32(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint16)
    lib().oracle_bf16_from_f32_array(_p(v), v.size, _p(out))
    return out


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening (the low 16 bits become zero)."""
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def e4m3_from_f32(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().oracle_e4m3_from_f32_array(_p(v), v.size, _p(out))
    return out


def e4m3_to_f32(c: np.ndarray) -> np.ndarray:
    c = np.asarray(c, np.uint8)
    table = np.array([lib().oracle_e4m3_to_f32(i) for i in range(256)], np.float32)
    return table[c]


def e2m1_from_f32(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().oracle_e2m1_from_f32_array(_p(v), v.size, _p(out))
    return out


def e2m1_to_f32(c: np.ndarray) -> np.ndarray:
    c = np.asarray(c, np.uint8)
    table = np.array([lib().oracle_e2m1_to_f32(i) for i in range(16)], np.float32)
    return table[c & 0xF]


def quant_tokens_fp4(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """x uint16 [..., H] -> (packed E2M1 uint8 [..., H/2], scales f32 [..., H/32])."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    H = x.shape[-1]
    assert H % 32 == 0
    n = x.size // H
    q = np.empty(x.shape[:-1] + (H // 2,), np.uint8)
    sc = np.empty(x.shape[:-1] + (H // 32,), np.float32)
    lib().oracle_quant_tokens_fp4(n, H, _p(x), _p(q), _p(sc))
    return q, sc


def quant_tokens(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """x uint16 [..., H] -> (codes uint8 [..., H], scales f32 [..., H/128])."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    H = x.shape[-1]
    assert H % 128 == 0
    n = x.size // H
    q = np.empty(x.shape, np.uint8)
    sc = np.empty(x.shape[:-1] + (H // 128,), np.float32)
    lib().oracle_quant_tokens(n, H, _p(x), _p(q), _p(sc))
    return q, sc


# --------------------------------------------------------- 2D dispatch

def route(idx: np.ndarray, ntok: np.ndarray, experts_per_rank: int):
    idx = np.ascontiguousarray(idx, np.int32)
    ntok = np.ascontiguousarray(ntok, np.int32)
    R, T, k = idx.shape
    cap = R * T
    recv = np.empty(R, np.int32)
    src_pos = np.empty((R, cap), np.int32)
    slot = np.empty((R, T, R), np.int32)
    _check(lib().oracle_route(R, T, k, experts_per_rank, _p(ntok), _p(idx), _p(recv),
                              _p(src_pos), _p(slot)), "route")
    return recv, src_pos, slot


def place_rows(rows: np.ndarray, ntok: np.ndarray, slot: np.ndarray) -> np.ndarray:
    """rows [R, Tmax, ...] (any dtype) -> [R, R*Tmax, ...]; unrouted rows are zero."""
    rows = np.ascontiguousarray(rows)
    R, T = rows.shape[:2]
    row_bytes = rows.itemsize * int(np.prod(rows.shape[2:], dtype=np.int64))
    out = np.zeros((R, R * T) + rows.shape[2:], rows.dtype)
    lib().oracle_place_rows(R, T, row_bytes, _p(np.ascontiguousarray(ntok, np.int32)),
                            _p(np.ascontiguousarray(slot, np.int32)), _p(rows), _p(out))
    return out


def dispatch(x: np.ndarray, w: np.ndarray, idx: np.ndarray, ntok: np.ndarray,
             experts_per_rank: int, quant_fp8: bool = False, scales: np.ndarray | None = None,
             quant_fp4: bool = False):
    """Full 2D dispatch. x: uint16 bf16 bits or uint8 fp8 codes [R, Tmax, H].

    Returns a dict with recv_num_token, src_pos, slot, x, w, idx, scales
    (scales: computed f32 block scales when quant_fp8, else the pass-through
    rows or None). Receive rows past recv_num_token are zero-filled.
    """
    recv, src_pos, slot = route(idx, ntok, experts_per_rank)
    out = {"recv_num_token": recv, "src_pos": src_pos, "slot": slot}
    if quant_fp8 or quant_fp4:
        q, sc = quant_tokens(x) if quant_fp8 else quant_tokens_fp4(x)
        out["x"] = place_rows(q, ntok, slot)
        out["scales"] = place_rows(sc, ntok, slot)
    else:
        out["x"] = place_rows(x, ntok, slot)
        out["scales"] = None if scales is None else place_rows(scales, ntok, slot)
    out["w"] = place_rows(w, ntok, slot)
    out["idx"] = place_rows(idx, ntok, slot)
    return out


def combine(y: np.ndarray, idx: np.ndarray, ntok: np.ndarray, slot: np.ndarray,
            experts_per_rank: int, w_recv: np.ndarray | None = None, weighted: bool = False,
            out_dtype: str = "bf16"):
    """y [R, R*Tmax, H] (uint16 bf16 bits or float32) -> (out [R, Tmax, H], out_w or None)."""
    y = np.ascontiguousarray(y)
    R, cap, H = y.shape
    T = cap // R
    k = idx.shape[-1]
    od = _dt(out_dtype)
    out = np.zeros((R, T, H), np.uint16 if od == DT_BF16 else np.float32)
    out_w = np.zeros((R, T, k), np.float32) if w_recv is not None else None
    wr = None if w_recv is None else np.ascontiguousarray(w_recv, np.float32)
    _check(lib().oracle_combine(R, T, k, experts_per_rank, H,
                                _p(np.ascontiguousarray(ntok, np.int32)),
                                _p(np.ascontiguousarray(idx, np.int32)),
                                _p(np.ascontiguousarray(slot, np.int32)), _dt(y.dtype.type), _p(y),
                                _p(wr), int(weighted), od, _p(out), _p(out_w)), "combine")
    return out, out_w


def combine_tokens(tokens: np.ndarray, y: np.ndarray, idx: np.ndarray, slot: np.ndarray,
                   experts_per_rank: int, w_recv: np.ndarray | None = None,
                   weighted: bool = False, out_dtype: str = "bf16"):
    """Combine for the listed global source tokens g = s*Tmax + t only:
    returns (out [n, H], out_w [n, k] or None)."""
    tokens = np.ascontiguousarray(tokens, np.int64)
    y = np.ascontiguousarray(y)
    R, cap, H = y.shape
    T = cap // R
    k = idx.shape[-1]
    od = _dt(out_dtype)
    out = np.zeros((len(tokens), H), np.uint16 if od == DT_BF16 else np.float32)
    out_w = np.zeros((len(tokens), k), np.float32) if w_recv is not None else None
    wr = None if w_recv is None else np.ascontiguousarray(w_recv, np.float32)
    _check(lib().oracle_combine_tokens(R, T, k, experts_per_rank, H, _p(tokens), len(tokens),
                                       _p(np.ascontiguousarray(idx, np.int32)),
                                       _p(np.ascontiguousarray(slot, np.int32)), _dt(y.dtype.type),
                                       _p(y), _p(wr), int(weighted), od, _p(out), _p(out_w)),
           "combine_tokens")
    return out, out_w


# --------------------------------------------------------- standard MoE

def std_layout(idx: np.ndarray, ntok: np.ndarray, experts_per_rank: int, pcap: int):
    idx = np.ascontiguousarray(idx, np.int32)
    R, T, k = idx.shape
    Er = experts_per_rank
    res = {
        "count": np.empty((R, Er), np.int32),
        "seg_off": np.empty((R, Er), np.int32),
        "rank_rows": np.empty(R, np.int32),
        "row_map": np.empty((R, T, k), np.int32),
        "src_info": np.empty((R, pcap), np.int32),
        "layout_range": np.empty((R, Er, R), np.int64),
    }
    _check(lib().oracle_std_layout(R, T, k, Er, pcap, _p(np.ascontiguousarray(ntok, np.int32)),
                                   _p(idx), _p(res["count"]), _p(res["seg_off"]),
                                   _p(res["rank_rows"]), _p(res["row_map"]), _p(res["src_info"]),
                                   _p(res["layout_range"])), "std_layout")
    return res


def std_place_rows(rows: np.ndarray, ntok: np.ndarray, row_map: np.ndarray, pcap: int) -> np.ndarray:
    rows = np.ascontiguousarray(rows)
    R, T = rows.shape[:2]
    k = row_map.shape[-1]
    row_bytes = rows.itemsize * int(np.prod(rows.shape[2:], dtype=np.int64))
    out = np.zeros((R, pcap) + rows.shape[2:], rows.dtype)
    lib().oracle_std_place_rows(R, T, k, row_bytes, _p(np.ascontiguousarray(ntok, np.int32)),
                                _p(np.ascontiguousarray(row_map, np.int32)), _p(rows), _p(out))
    return out


def std_dispatch(x: np.ndarray, idx: np.ndarray, ntok: np.ndarray, experts_per_rank: int,
                 pcap: int, quant_fp8: bool = False):
    res = std_layout(idx, ntok, experts_per_rank, pcap)
    if quant_fp8:
        q, sc = quant_tokens(x)
        res["x"] = std_place_rows(q, ntok, res["row_map"], pcap)
        res["scales"] = std_place_rows(sc, ntok, res["row_map"], pcap)
    else:
        res["x"] = std_place_rows(x, ntok, res["row_map"], pcap)
        res["scales"] = None
    return res


def std_combine(Y: np.ndarray, idx: np.ndarray, ntok: np.ndarray, row_map: np.ndarray,
                experts_per_rank: int, w: np.ndarray | None = None, weighted: bool = True,
                out_dtype: str = "fp32") -> np.ndarray:
    Y = np.ascontiguousarray(Y)
    R, pcap, H = Y.shape
    T, k = idx.shape[1], idx.shape[2]
    od = _dt(out_dtype)
    out = np.zeros((R, T, H), np.uint16 if od == DT_BF16 else np.float32)
    wp = None if w is None else np.ascontiguousarray(w, np.float32)
    _check(lib().oracle_std_combine(R, T, k, experts_per_rank, H,
                                    _p(np.ascontiguousarray(ntok, np.int32)),
                                    _p(np.ascontiguousarray(idx, np.int32)),
                                    _p(np.ascontiguousarray(row_map, np.int32)),
                                    _dt(Y.dtype.type), _p(Y), _p(wp), int(weighted), od, _p(out)),
           "std_combine")
    return out


def std_combine_tokens(tokens: np.ndarray, Y: np.ndarray, idx: np.ndarray, row_map: np.ndarray,
                       experts_per_rank: int, w: np.ndarray | None = None,
                       weighted: bool = True, out_dtype: str = "fp32") -> np.ndarray:
    tokens = np.ascontiguousarray(tokens, np.int64)
    Y = np.ascontiguousarray(Y)
    R = idx.shape[0]
    k = idx.shape[-1]
    H = Y.shape[-1]
    od = _dt(out_dtype)
    out = np.zeros((len(tokens), H), np.uint16 if od == DT_BF16 else np.float32)
    wp = None if w is None else np.ascontiguousarray(w, np.float32)
    _check(lib().oracle_std_combine_tokens(R, k, experts_per_rank, H, _p(tokens), len(tokens),
                                           _p(np.ascontiguousarray(idx, np.int32)),
                                           _p(np.ascontiguousarray(row_map, np.int32)),
                                           _dt(Y.dtype.type), _p(Y), _p(wp), int(weighted), od,
                                           _p(out)), "std_combine_tokens")
    return out


def convert_dispatch_output(recv_num_token: np.ndarray, recv_x: np.ndarray, recv_idx: np.ndarray,
                            recv_src_pos: np.ndarray, Tmax: int, experts_per_rank: int, pcap: int):
    recv_x = np.ascontiguousarray(recv_x)
    R, cap = recv_x.shape[:2]
    k = recv_idx.shape[-1]
    Er = experts_per_rank
    row_bytes = recv_x.itemsize * int(np.prod(recv_x.shape[2:], dtype=np.int64))
    res = {
        "count": np.empty((R, Er), np.int32),
        "seg_off": np.empty((R, Er), np.int32),
        "rank_rows": np.empty(R, np.int32),
        "row_map": np.empty((R, Tmax, k), np.int32),
        "x": np.zeros((R, pcap) + recv_x.shape[2:], recv_x.dtype),
        "src_info": np.empty((R, pcap), np.int32),
        "layout_range": np.empty((R, Er, R), np.int64),
    }
    _check(lib().oracle_convert_dispatch_output(
        R, Tmax, k, Er, pcap, row_bytes, _p(np.ascontiguousarray(recv_num_token, np.int32)),
        _p(recv_x), _p(np.ascontiguousarray(recv_idx, np.int32)),
        _p(np.ascontiguousarray(recv_src_pos, np.int32)), _p(res["count"]), _p(res["seg_off"]),
        _p(res["rank_rows"]), _p(res["row_map"]), _p(res["x"]), _p(res["src_info"]),
        _p(res["layout_range"])), "convert_dispatch_output")
    return res


def convert_combine_input(Y: np.ndarray, recv_num_token: np.ndarray, recv_src_pos: np.ndarray,
                          idx: np.ndarray, row_map: np.ndarray, experts_per_rank: int,
                          out_dtype: str = "bf16") -> np.ndarray:
    Y = np.ascontiguousarray(Y)
    R, T, k = idx.shape
    H = Y.shape[-1]
    od = _dt(out_dtype)
    out = np.zeros((R, R * T, H), np.uint16 if od == DT_BF16 else np.float32)
    _check(lib().oracle_convert_combine_input(
        R, T, k, experts_per_rank, H, _p(np.ascontiguousarray(recv_num_token, np.int32)),
        _p(np.ascontiguousarray(recv_src_pos, np.int32)), _p(np.ascontiguousarray(idx, np.int32)),
        _p(np.ascontiguousarray(row_map, np.int32)), _dt(Y.dtype.type), _p(Y), od, _p(out)),
        "convert_combine_input")
    return out
