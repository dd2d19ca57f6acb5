"""Thin Python binding of libep (include/ep.h).

Argument marshalling only: every step of dispatch and combine runs in the
CUDA kernels of libep.so. Functions named ep_* wrap the C entry points one
to one (pointers as ints); EpDispatchCombineOp mirrors the operator API of
the MORI-EP User Guide (section 3 "Operator API", section 4 "Standard MoE
Compatibility") on torch tensors, with PyTorch used only for device memory
and streams. There is no CPU fallback: importing this module fails if the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, fields

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libep.so")

EP_OK = 0
EP_ERR_INVALID_ARG = -1
EP_ERR_STATE = -2
EP_ERR_CAPACITY = -3
EP_ERR_INVALID_INDEX = -4
EP_ERR_CUDA = -5
EP_ERR_TIMEOUT = -6
EP_ERR_WORKSPACE = -7
EP_ERR_UNSUPPORTED = -8

EP_DTYPE_BF16 = 0
EP_DTYPE_FP32 = 1
EP_DTYPE_FP8_E4M3 = 2
EP_DTYPE_FP4_E2M1X2 = 3
EP_QUANT_NONE = 0
EP_QUANT_FP8_E4M3_BLOCK128 = 1
EP_QUANT_FP4_E2M1_BLOCK32 = 2
EP_COMBINE_AUTO = 0
EP_COMBINE_VECTOR = 1
EP_COMBINE_BULK = 2
EP_DISPATCH_AUTO = 0
EP_DISPATCH_VECTOR = 1
EP_DISPATCH_BULK = 2
EP_PHASE_DISPATCH = 0
EP_PHASE_COMBINE = 1
IMPL_OF = {"auto": 0, "vector": 1, "bulk": 2}        # same codes for both phases
IMPL_NAME = {v: k for k, v in IMPL_OF.items()}

_FP4X2 = getattr(torch, "float4_e2m1fn_x2", None)   # packed pairs of E2M1 codes
_TORCH_OF = {EP_DTYPE_BF16: torch.bfloat16, EP_DTYPE_FP32: torch.float32,
             EP_DTYPE_FP8_E4M3: torch.float8_e4m3fn}
if _FP4X2 is not None:
    _TORCH_OF[EP_DTYPE_FP4_E2M1X2] = _FP4X2
_EP_OF = {v: k for k, v in _TORCH_OF.items()}
_QUANT_OF = {"none": EP_QUANT_NONE, "fp8_e4m3_block128": EP_QUANT_FP8_E4M3_BLOCK128,
             "fp4_e2m1_block32": EP_QUANT_FP4_E2M1_BLOCK32}


class EpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libep status {status}: {message}")
        self.status = status


class ep_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "world_size", "hidden_dim", "scale_dim", "scale_type_size", "max_token_type_size",
        "max_num_inp_token_per_rank", "num_experts_per_rank", "num_experts_per_token",
        "data_type", "quant_type", "combine_dtype", "combine_out_dtype", "weighted_combine",
        "standard_moe", "max_packed_rows_per_rank", "block_num", "warp_num_per_block",
        "combine_impl", "dispatch_impl", "use_external_inp_buf")]


class ep_dispatch_out(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("weights", ctypes.c_void_p), ("indices", ctypes.c_void_p),
                ("recv_num_token", ctypes.c_void_p), ("src_token_pos", ctypes.c_void_p),
                ("cap", ctypes.c_int64), ("x_row_bytes", ctypes.c_int64),
                ("scale_row_bytes", ctypes.c_int64)]


class ep_std_moe_out(ctypes.Structure):
    _fields_ = [("packed_x", ctypes.c_void_p), ("packed_scales", ctypes.c_void_p),
                ("packed_count", ctypes.c_void_p), ("packed_src_info", ctypes.c_void_p),
                ("packed_layout_range", ctypes.c_void_p), ("expert_offset", ctypes.c_void_p),
                ("rank_rows", ctypes.c_void_p), ("rank_base", ctypes.c_void_p),
                ("pcap", ctypes.c_int64), ("x_row_bytes", ctypes.c_int64)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(there is no fallback path)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    S = ctypes.c_int
    sig = {
        "ep_workspace_size": (Z, [P]),
        "ep_config_create": (S, [P, P, Z, P]),
        "ep_destroy": (None, [P]),
        "ep_dispatch": (S, [P, P, P, P, P, P, P, P]),
        "ep_combine": (S, [P, P, P, P, P, P, I, P]),
        "ep_get_dispatch_src_token_pos": (S, [P, P]),
        "ep_reset": (S, [P, P]),
        "ep_dispatch_standard_moe": (S, [P, P, P, P, P, P, P, P]),
        "ep_combine_standard_moe": (S, [P, P, P, P, P, I, P]),
        "ep_convert_dispatch_output": (S, [P, P, P, P, P]),
        "ep_convert_combine_input": (S, [P, P, P, P]),
        "ep_sync": (S, [P, P]),
        "ep_last_error": (ctypes.c_char_p, []),
        "ep_routing_layout_noalloc": (S, [I, I, I, I, P, P, P, P, P, P, P]),
        "ep_get_registered_combine_input_buffer": (S, [P, P]),
        "ep_set_launch_config": (S, [P, I, I, I, I]),
        "ep_get_launch_config": (S, [P, I, P, P, P]),
        "ep_selftest_bounded_wait": (S, [P, P]),
        "ep_rank_workspace_size": (Z, [P]),
        "ep_rank_create": (S, [P, I, P, Z, P]),
        "ep_rank_destroy": (None, [P]),
        "ep_rank_set_peers": (S, [P, P]),
        "ep_dispatch_send": (S, [P, P, P, P, P, I, P, P]),
        "ep_dispatch_recv": (S, [P, P]),
        "ep_combine_send": (S, [P, P, P, P, P, P]),
        "ep_combine_recv": (S, [P, I, P]),
        "ep_rank_reset": (S, [P]),
        "ep_rank_get_registered_combine_input_buffer": (S, [P, P]),
        "ep_rank_get_dispatch_src_token_pos": (S, [P, P]),
        "ep_rank_sync": (S, [P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def _check(status: int) -> None:
    if status != EP_OK:
        raise EpError(status, _lib.ep_last_error().decode())


def _ref(obj):
    return ctypes.byref(obj) if obj is not None else None


# ------------------------------------------------------- C entry points

def ep_workspace_size(cfg: ep_config) -> int:
    return int(_lib.ep_workspace_size(ctypes.byref(cfg)))


def ep_config_create(cfg: ep_config, d_workspace: int, workspace_bytes: int) -> int:
    h = ctypes.c_void_p()
    _check(_lib.ep_config_create(ctypes.byref(cfg), d_workspace, workspace_bytes, ctypes.byref(h)))
    return h.value


def ep_destroy(handle: int) -> None:
    _lib.ep_destroy(handle)


def _i32_array(values):
    if isinstance(values, ctypes.Array):
        return values
    return (ctypes.c_int32 * len(values))(*[int(n) for n in values])


def ep_dispatch(handle, x, weights, scales, indices, num_tokens, stream) -> ep_dispatch_out:
    out = ep_dispatch_out()
    _check(_lib.ep_dispatch(handle, x, weights, scales, indices, _i32_array(num_tokens), stream,
                            ctypes.byref(out)))
    return out


def ep_combine(handle, expert_out, weights, indices, out, out_weights, call_reset, stream) -> None:
    _check(_lib.ep_combine(handle, expert_out, weights, indices, out, out_weights,
                           int(call_reset), stream))


def ep_get_dispatch_src_token_pos(handle) -> int:
    p = ctypes.c_void_p()
    _check(_lib.ep_get_dispatch_src_token_pos(handle, ctypes.byref(p)))
    return p.value


def ep_get_registered_combine_input_buffer(handle) -> int:
    p = ctypes.c_void_p()
    _check(_lib.ep_get_registered_combine_input_buffer(handle, ctypes.byref(p)))
    return p.value


def ep_reset(handle, stream=None) -> None:
    _check(_lib.ep_reset(handle, stream))


def ep_dispatch_standard_moe(handle, x, weights, scales, indices, num_tokens,
                             stream) -> ep_std_moe_out:
    out = ep_std_moe_out()
    _check(_lib.ep_dispatch_standard_moe(handle, x, weights, scales, indices,
                                         _i32_array(num_tokens), stream, ctypes.byref(out)))
    return out


def ep_combine_standard_moe(handle, expert_out, weights, indices, out, call_reset, stream) -> None:
    _check(_lib.ep_combine_standard_moe(handle, expert_out, weights, indices, out,
                                        int(call_reset), stream))


def ep_convert_dispatch_output(handle, dispatch_x, dispatch_indices, stream) -> ep_std_moe_out:
    out = ep_std_moe_out()
    _check(_lib.ep_convert_dispatch_output(handle, dispatch_x, dispatch_indices, stream,
                                           ctypes.byref(out)))
    return out


def ep_convert_combine_input(handle, packed_y, combine_in, stream) -> None:
    _check(_lib.ep_convert_combine_input(handle, packed_y, combine_in, stream))


def ep_selftest_bounded_wait(handle, stream) -> None:
    _check(_lib.ep_selftest_bounded_wait(handle, stream))


def ep_sync(handle, stream) -> None:
    _check(_lib.ep_sync(handle, stream))


def ep_last_error() -> str:
    return _lib.ep_last_error().decode()


def ep_set_launch_config(handle, phase: int, impl: int, block_num: int,
                         warp_num_per_block: int) -> None:
    _check(_lib.ep_set_launch_config(handle, phase, impl, block_num, warp_num_per_block))


def ep_get_launch_config(handle, phase: int) -> tuple[int, int, int]:
    impl, bn, wp = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(_lib.ep_get_launch_config(handle, phase, ctypes.byref(impl), ctypes.byref(bn),
                                     ctypes.byref(wp)))
    return impl.value, bn.value, wp.value


def ep_routing_layout_noalloc(world_size, max_num_inp_token_per_rank, num_experts_per_rank,
                              num_experts_per_token, indices, num_tokens, recv_num_token,
                              src_token_pos, slot_map, error_flags, stream) -> None:
    """Routing layout with the library's static scratch (no device allocation)."""
    nt = (ctypes.c_int32 * len(num_tokens))(*[int(n) for n in num_tokens])
    _check(_lib.ep_routing_layout_noalloc(world_size, max_num_inp_token_per_rank,
                                          num_experts_per_rank, num_experts_per_token, indices,
                                          nt, recv_num_token, src_token_pos, slot_map,
                                          error_flags, stream))


# ------------------------------------------- one rank per workspace (split phases)

def ep_rank_workspace_size(cfg: ep_config) -> int:
    return int(_lib.ep_rank_workspace_size(ctypes.byref(cfg)))


def ep_rank_create(cfg: ep_config, rank: int, d_workspace: int, workspace_bytes: int) -> int:
    h = ctypes.c_void_p()
    _check(_lib.ep_rank_create(ctypes.byref(cfg), int(rank), d_workspace, workspace_bytes,
                               ctypes.byref(h)))
    return h.value


def ep_rank_destroy(handle: int) -> None:
    _lib.ep_rank_destroy(handle)


def ep_rank_set_peers(handle, peer_workspaces) -> None:
    arr = (ctypes.c_void_p * len(peer_workspaces))(*[int(p) for p in peer_workspaces])
    _check(_lib.ep_rank_set_peers(handle, arr))


def ep_dispatch_send(handle, x, weights, scales, indices, num_tokens: int, stream) -> ep_dispatch_out:
    out = ep_dispatch_out()
    _check(_lib.ep_dispatch_send(handle, x, weights, scales, indices, int(num_tokens), stream,
                                 ctypes.byref(out)))
    return out


def ep_dispatch_recv(handle, stream) -> None:
    _check(_lib.ep_dispatch_recv(handle, stream))


def ep_combine_send(handle, expert_out, weights, out, out_weights, stream) -> None:
    _check(_lib.ep_combine_send(handle, expert_out, weights, out, out_weights, stream))


def ep_combine_recv(handle, call_reset, stream) -> None:
    _check(_lib.ep_combine_recv(handle, int(call_reset), stream))


def ep_rank_reset(handle) -> None:
    _check(_lib.ep_rank_reset(handle))


def ep_rank_get_registered_combine_input_buffer(handle) -> int:
    p = ctypes.c_void_p()
    _check(_lib.ep_rank_get_registered_combine_input_buffer(handle, ctypes.byref(p)))
    return p.value


def ep_rank_get_dispatch_src_token_pos(handle) -> int:
    p = ctypes.c_void_p()
    _check(_lib.ep_rank_get_dispatch_src_token_pos(handle, ctypes.byref(p)))
    return p.value


def ep_rank_sync(handle, stream) -> None:
    _check(_lib.ep_rank_sync(handle, stream))


# ------------------------------------------------------- operator class

@dataclass
class EpDispatchCombineConfig:
    """EpDispatchCombineConfig (MORI-EP User Guide, section 2) for simulated
    ranks: all world_size ranks live in this process, so `rank` is absent."""
    data_type: torch.dtype
    world_size: int
    hidden_dim: int
    scale_dim: int
    scale_type_size: int
    max_token_type_size: int
    max_num_inp_token_per_rank: int
    num_experts_per_rank: int
    num_experts_per_token: int
    warp_num_per_block: int = 8
    block_num: int = -1
    quant_type: str = "none"            # "none" | "fp8_e4m3_block128" | "fp4_e2m1_block32"
    combine_dtype: torch.dtype = torch.bfloat16
    combine_out_dtype: torch.dtype = torch.bfloat16
    weighted_combine: bool = False
    standard_moe: bool | int = False    # 0/False: 2D layout; 1/True: packed only; 2: both
    max_packed_rows_per_rank: int = 0
    combine_impl: str = "auto"          # "auto" | "vector" | "bulk"
    dispatch_impl: str = "auto"         # "auto" | "vector" | "bulk" (copy mode)
    use_external_inp_buf: bool = True   # False: reserve a registered combine input buffer
    # "manual": block_num / warp_num_per_block above, or per-call overrides;
    # "auto": per-shape rules from the tuning files (User Guide, sections 6
    # and 10); the environment variable EP_LAUNCH_CONFIG_MODE=AUTO selects it too
    launch_config_mode: str = "manual"

    def to_c(self) -> ep_config:
        c = ep_config()
        c_fields = {n for n, _ in ep_config._fields_}
        for f in fields(self):
            if f.name not in c_fields:
                continue
            v = getattr(self, f.name)
            if f.name in ("data_type", "combine_dtype", "combine_out_dtype"):
                v = _EP_OF[v]
            elif f.name == "quant_type":
                v = _QUANT_OF[v]
            elif f.name in ("combine_impl", "dispatch_impl"):
                v = IMPL_OF[v]
            setattr(c, f.name, int(v))
        return c

    def auto_launch(self) -> bool:
        env = os.environ.get("EP_LAUNCH_CONFIG_MODE", "")
        return self.launch_config_mode == "auto" or env.upper() == "AUTO"


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def _stream():
    return torch.cuda.current_stream().cuda_stream


class EpDispatchCombineOp:
    """Operator over one workspace (User Guide, section 3). Inputs carry all
    ranks: x [R, Tmax, H], weights [R, Tmax, k], indices [R, Tmax, k] int32;
    num_tokens gives each source rank's token count (default Tmax)."""

    def __init__(self, config: EpDispatchCombineConfig, device: torch.device | str = "cuda",
                 use_tuning_files: bool | None = None):
        """use_tuning_files: None follows config.launch_config_mode and the
        EP_LAUNCH_CONFIG_MODE environment variable; False or True overrides both."""
        self.config = config
        self.c = config.to_c()
        nbytes = ep_workspace_size(self.c)
        if nbytes == 0:
            raise EpError(EP_ERR_INVALID_ARG, ep_last_error())
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self._handle = ep_config_create(self.c, self.workspace.data_ptr(), nbytes)
        R, T = config.world_size, config.max_num_inp_token_per_rank
        self.cap = R * T
        self._default_launch = {
            EP_PHASE_DISPATCH: (self.c.dispatch_impl, self.c.block_num, self.c.warp_num_per_block),
            EP_PHASE_COMBINE: (self.c.combine_impl, self.c.block_num, self.c.warp_num_per_block)}
        self._applied_launch = dict(self._default_launch)
        self._auto = config.auto_launch() if use_tuning_files is None else bool(use_tuning_files)
        self._rules = {}
        self._rule_choice = {}

    def __del__(self):
        h = getattr(self, "_handle", None)
        if h:
            ep_destroy(h)
            self._handle = None

    # views into the workspace ------------------------------------------------
    def _view(self, ptr: int, dtype: torch.dtype, shape) -> torch.Tensor:
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        off = ptr - self.workspace.data_ptr()
        assert 0 <= off and off + nbytes <= self.workspace.numel()
        return self.workspace[off:off + nbytes].view(dtype).view(*shape)

    _last_num_tokens = None  # token counts of the last dispatch (combine's tuning key)

    def _num_tokens(self, num_tokens):
        if num_tokens is None:
            R, T = self.config.world_size, self.config.max_num_inp_token_per_rank
            num_tokens = [T] * R
        self._last_num_tokens = num_tokens
        return num_tokens

    def _payload(self):
        """(dtype, columns) of a received payload row and the number of f32
        block scales per row (None without quantisation)."""
        cfg = self.config
        H = cfg.hidden_dim
        if cfg.quant_type == "fp8_e4m3_block128":
            return torch.float8_e4m3fn, H, H // 128
        if cfg.quant_type == "fp4_e2m1_block32":
            return torch.uint8, H // 2, H // 32
        if _FP4X2 is not None and cfg.data_type == _FP4X2:
            return cfg.data_type, H // 2, None
        return cfg.data_type, H, None

    # launch configuration (User Guide, sections 6 and 10) ---------------------
    def set_launch_config(self, phase: int, impl: str | int = "auto", block_num: int = -1,
                          warp_per_block: int = 8) -> None:
        """Base launch configuration of one phase for the calls that follow
        (per-call block_num / warp_per_block still override it for one call;
        auto mode still replaces it where a tuning rule matches)."""
        code = IMPL_OF[impl] if isinstance(impl, str) else int(impl)
        ep_set_launch_config(self._handle, phase, code, int(block_num), int(warp_per_block))
        self._default_launch[phase] = (code, int(block_num), int(warp_per_block))
        self._applied_launch[phase] = self._default_launch[phase]

    def get_launch_config(self, phase: int) -> tuple[str, int, int]:
        impl, bn, wp = ep_get_launch_config(self._handle, phase)
        return IMPL_NAME[impl], bn, wp

    def _tuning_key(self, phase: int) -> tuple[str, str]:
        """(kernel family, dtype) of a phase as the tuning files name them."""
        from .tuning import dispatch_dtype_name, combine_dtype_name
        kernel = "stdmoe" if self.config.standard_moe else "2d"
        if phase == EP_PHASE_DISPATCH:
            return kernel, dispatch_dtype_name(self.config)
        return kernel, combine_dtype_name(self.config)

    def _launch_for(self, phase: int, num_tokens, block_num, warp_per_block) -> None:
        want = self._default_launch[phase]
        if self._auto:  # per-call arguments are ignored in auto mode
            from . import tuning
            kernel, dt = self._tuning_key(phase)
            key = (phase, kernel)
            if key not in self._rules:
                self._rules[key] = tuning.load_rules(kernel, self.config.world_size,
                                                     "dispatch" if phase == EP_PHASE_DISPATCH
                                                     else "combine")
            n = int(max(num_tokens)) if num_tokens is not None else \
                self.config.max_num_inp_token_per_rank
            if (phase, n) not in self._rule_choice:
                rule = tuning.lookup(self._rules[key], dt, self.config.hidden_dim, n)
                self._rule_choice[(phase, n)] = None if rule is None else (
                    IMPL_OF[rule["impl"]], rule["block_num"], rule["warp_per_block"])
            if self._rule_choice[(phase, n)] is not None:
                want = self._rule_choice[(phase, n)]
        elif block_num is not None or warp_per_block is not None:
            want = (want[0], want[1] if block_num is None else int(block_num),
                    want[2] if warp_per_block is None else int(warp_per_block))
        if self._applied_launch[phase] != want:
            ep_set_launch_config(self._handle, phase, *want)
            self._applied_launch[phase] = want

    @staticmethod
    def decode_send_flat_idx(pos: int, world_size: int, max_tokens: int) -> tuple[int, int]:
        return divmod(int(pos), world_size * max_tokens)

    # section 3 ----------------------------------------------------------------
    def dispatch(self, input, weights, scales, indices, num_tokens=None, block_num=None,
                 warp_per_block=None):
        self._launch_for(EP_PHASE_DISPATCH, num_tokens, block_num, warp_per_block)
        o = ep_dispatch(self._handle, _ptr(input), _ptr(weights), _ptr(scales), _ptr(indices),
                        self._num_tokens(num_tokens), _stream())
        # the outputs always live at the same workspace offsets: build the views once
        key = (o.x, o.scales, o.weights, o.indices, o.recv_num_token)
        if getattr(self, "_dispatch_key", None) != key:
            self._dispatch_views = self._make_dispatch_views(o)
            self._dispatch_key = key
        return self._dispatch_views

    def _make_dispatch_views(self, o):
        cfg = self.config
        R, k = cfg.world_size, cfg.num_experts_per_token
        dt, cols, nsc = self._payload()
        x = self._view(o.x, dt, (R, self.cap, cols))
        if o.scales:
            if nsc is not None:
                sc = self._view(o.scales, torch.float32, (R, self.cap, nsc))
            else:
                sc = self._view(o.scales, torch.uint8, (R, self.cap, o.scale_row_bytes))
        else:
            sc = None
        w = self._view(o.weights, torch.float32, (R, self.cap, k))
        idx = self._view(o.indices, torch.int32, (R, self.cap, k))
        recv = self._view(o.recv_num_token, torch.int32, (R,))
        return x, w, sc, idx, recv

    def combine(self, input, weights, indices, out=None, out_weights=None, call_reset=False,
                want_weights=True, block_num=None, warp_per_block=None):
        cfg = self.config
        self._launch_for(EP_PHASE_COMBINE, self._last_num_tokens, block_num, warp_per_block)
        R, T, H, k = (cfg.world_size, cfg.max_num_inp_token_per_rank, cfg.hidden_dim,
                      cfg.num_experts_per_token)
        dev = self.workspace.device
        if out is None:
            out = torch.empty((R, T, H), dtype=cfg.combine_out_dtype, device=dev)
        if out_weights is None and want_weights and weights is not None:
            out_weights = torch.empty((R, T, k), dtype=torch.float32, device=dev)
        ep_combine(self._handle, _ptr(input), _ptr(weights), _ptr(indices), _ptr(out),
                   _ptr(out_weights), call_reset, _stream())
        return out, out_weights

    def reset(self):
        ep_reset(self._handle, _stream())

    def get_registered_combine_input_buffer(self, dtype=None):
        """Zero-copy combine input (User Guide, section 3): [R, cap, H] view of the
        workspace buffer that combine(input=None) reads in place."""
        cfg = self.config
        dtype = cfg.combine_dtype if dtype is None else dtype
        if dtype != cfg.combine_dtype:
            raise EpError(EP_ERR_INVALID_ARG, "registered buffer holds combine_dtype")
        p = ep_get_registered_combine_input_buffer(self._handle)
        return self._view(p, dtype, (cfg.world_size, self.cap, cfg.hidden_dim))

    def get_dispatch_src_token_pos(self):
        p = ep_get_dispatch_src_token_pos(self._handle)
        return self._view(p, torch.int32, (self.config.world_size, self.cap))

    def sync(self):
        ep_sync(self._handle, _stream())

    # section 4 ----------------------------------------------------------------
    def _std_views(self, o: ep_std_moe_out):
        """Packed layout views. The ranks share one pool of pcap rows: rank r's
        rows are packed_recv_x[rank_base[r] : rank_base[r] + rank_rows[r]]
        (device values; `packed_rank_rows` slices them on the host)."""
        cfg = self.config
        R, Er, H = cfg.world_size, cfg.num_experts_per_rank, cfg.hidden_dim
        dt, cols, nsc = self._payload()
        return {
            "packed_recv_x": self._view(o.packed_x, dt, (o.pcap, cols)),
            "packed_recv_scales": (self._view(o.packed_scales, torch.float32, (o.pcap, nsc))
                                   if o.packed_scales and nsc is not None else None),
            "packed_recv_count": self._view(o.packed_count, torch.int32, (R, Er)),
            "packed_recv_src_info": self._view(o.packed_src_info, torch.int32, (o.pcap,)),
            "packed_recv_layout_range": self._view(o.packed_layout_range, torch.int64, (R, Er, R)),
            "expert_offset": self._view(o.expert_offset, torch.int32, (R, Er)),
            "rank_rows": self._view(o.rank_rows, torch.int32, (R,)),
            "rank_base": self._view(o.rank_base, torch.int32, (R,)),
        }

    @staticmethod
    def packed_rank_rows(pool: torch.Tensor, rank_base, rank_rows, r: int) -> torch.Tensor:
        """Rank r's rows of a packed-pool tensor (host-side bounds: reads the
        base and row count, so it synchronises with the device)."""
        b = int(rank_base[r])
        return pool[b:b + int(rank_rows[r])]

    def dispatch_standard_moe(self, input, weights, scales, indices, num_tokens=None,
                              block_num=None, warp_per_block=None):
        self._launch_for(EP_PHASE_DISPATCH, num_tokens, block_num, warp_per_block)
        o = ep_dispatch_standard_moe(self._handle, _ptr(input), _ptr(weights), _ptr(scales),
                                     _ptr(indices), self._num_tokens(num_tokens), _stream())
        self.pcap = o.pcap
        return self._std_views(o)

    def combine_standard_moe(self, input, weights, indices, out=None, call_reset=False,
                             block_num=None, warp_per_block=None):
        cfg = self.config
        self._launch_for(EP_PHASE_COMBINE, self._last_num_tokens, block_num, warp_per_block)
        R, T, H = cfg.world_size, cfg.max_num_inp_token_per_rank, cfg.hidden_dim
        if out is None:
            out = torch.empty((R, T, H), dtype=cfg.combine_out_dtype, device=input.device)
        ep_combine_standard_moe(self._handle, _ptr(input), _ptr(weights), _ptr(indices),
                                _ptr(out), call_reset, _stream())
        return out

    def convert_dispatch_output(self, dispatch_out_x, dispatch_out_topk_idx):
        o = ep_convert_dispatch_output(self._handle, _ptr(dispatch_out_x),
                                       _ptr(dispatch_out_topk_idx), _stream())
        self.pcap = o.pcap
        v = self._std_views(o)
        return (v["packed_recv_x"], v["packed_recv_count"], v["packed_recv_src_info"],
                v["packed_recv_layout_range"])

    def convert_combine_input(self, packed_recv_x, packed_recv_src_info=None,
                              packed_recv_layout_range=None, out=None):
        """The src_info / layout_range arguments are accepted for API parity;
        the handle's packed layout defines where each row goes."""
        cfg = self.config
        if out is None:
            out = torch.empty((cfg.world_size, self.cap, cfg.hidden_dim), dtype=cfg.combine_dtype,
                              device=packed_recv_x.device)
        ep_convert_combine_input(self._handle, _ptr(packed_recv_x), _ptr(out), _stream())
        return out
