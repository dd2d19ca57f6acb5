"""The C ABI library without a GPU: every symbol declared in include/ep.h is
exported, and the host-side validation, workspace sizing and state machine
answer without touching a device (no kernel is launched here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ep.h")


@pytest.fixture(scope="module")
def ep():
    from combine_route_layout_gb300.build import build
    build()
    from combine_route_layout_gb300 import ep as mod
    return mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ep_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(ep):
    names = declared_functions()
    assert len(names) >= 13
    lib = ctypes.CDLL(ep.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_no_multicast_anywhere():
    """No TMA multicast form is used in any source of the product."""
    for d, _, files in os.walk(os.path.join(ROOT, "combine_route_layout_gb300")):
        for f in files:
            if f.endswith((".cu", ".cuh", ".h", ".cpp")):
                assert "multicast" not in open(os.path.join(d, f)).read(), f


def cfg(ep, **kw):
    base = dict(world_size=8, hidden_dim=7168, scale_dim=0, scale_type_size=4,
                max_token_type_size=4, max_num_inp_token_per_rank=4096, num_experts_per_rank=32,
                num_experts_per_token=8, data_type=ep.EP_DTYPE_BF16,
                quant_type=ep.EP_QUANT_FP8_E4M3_BLOCK128, combine_dtype=ep.EP_DTYPE_BF16,
                combine_out_dtype=ep.EP_DTYPE_BF16, weighted_combine=0, standard_moe=0,
                max_packed_rows_per_rank=0, block_num=0, warp_num_per_block=0, combine_impl=0,
                dispatch_impl=0, use_external_inp_buf=1)
    base.update(kw)
    c = ep.ep_config()
    for k, v in base.items():
        setattr(c, k, v)
    return c


def test_workspace_size_grows_with_layouts(ep):
    """standard_moe 0 reserves the 2D receive layout, 1 only the packed pool,
    2 both (and the conversion scratch)."""
    a = ep.ep_workspace_size(cfg(ep))
    b1 = ep.ep_workspace_size(cfg(ep, standard_moe=1))
    b2 = ep.ep_workspace_size(cfg(ep, standard_moe=2))
    # 2D receive payload alone: 8 ranks x 32768 rows x 7168 FP8 bytes
    assert a >= 8 * 32768 * 7168
    # the packed pool shared by the ranks: one row per (token, slot) plus 127
    # padding rows per expert, whatever the routing (not 8 per-rank worst cases)
    pool = 8 * 4096 * 8 + 127 * 256
    assert pool * 7168 <= b1 < 1.1 * pool * (7168 + 4 * 56 + 4) + 64 * 2**20
    assert a + pool * 7168 <= b2 < a + b1 + 64 * 2**20


@pytest.mark.parametrize("bad", [dict(world_size=0), dict(world_size=33), dict(hidden_dim=100),
                                 dict(num_experts_per_token=0), dict(num_experts_per_token=33),
                                 dict(num_experts_per_rank=0), dict(num_experts_per_rank=200),
                                 dict(max_num_inp_token_per_rank=0), dict(data_type=9),
                                 dict(hidden_dim=200), dict(quant_type=5),
                                 dict(combine_out_dtype=2), dict(scale_dim=3),
                                 dict(data_type=1, quant_type=1), dict(warp_num_per_block=16),
                                 dict(standard_moe=3), dict(standard_moe=-1),
                                 dict(standard_moe=1, use_external_inp_buf=0)])
def test_invalid_configs_rejected(ep, bad):
    c = cfg(ep, **bad)
    assert ep.ep_workspace_size(c) == 0
    with pytest.raises(ep.EpError) as ei:
        ep.ep_config_create(c, 1 << 20, 1 << 40)
    assert ei.value.status == ep.EP_ERR_INVALID_ARG


FAKE = 1 << 40   # an aligned address that is never dereferenced by these tests


def small(ep, **kw):
    return cfg(ep, hidden_dim=256, max_num_inp_token_per_rank=16, num_experts_per_rank=4,
               num_experts_per_token=4, quant_type=0, **kw)


def test_registered_buffer_is_reserved_in_the_workspace(ep):
    a = ep.ep_workspace_size(small(ep))
    b = ep.ep_workspace_size(small(ep, use_external_inp_buf=0))
    assert b - a >= 8 * (8 * 16) * 256 * 2          # [R][cap][H] bf16
    c = small(ep, use_external_inp_buf=0)
    h = ep.ep_config_create(c, FAKE, b)
    try:
        p = ep.ep_get_registered_combine_input_buffer(h)
        assert FAKE <= p < FAKE + b and p % 256 == 0
    finally:
        ep.ep_destroy(h)


def test_workspace_checks(ep):
    c = small(ep)
    n = ep.ep_workspace_size(c)
    with pytest.raises(ep.EpError) as ei:
        ep.ep_config_create(c, FAKE, n - 1)
    assert ei.value.status == ep.EP_ERR_WORKSPACE
    with pytest.raises(ep.EpError) as ei:
        ep.ep_config_create(c, FAKE + 16, n)
    assert ei.value.status == ep.EP_ERR_WORKSPACE
    with pytest.raises(ep.EpError):
        ep.ep_config_create(c, 0, n)
    h = ep.ep_config_create(c, FAKE, n)
    ep.ep_destroy(h)


def test_state_machine_without_device(ep):
    c = small(ep)
    h = ep.ep_config_create(c, FAKE, ep.ep_workspace_size(c))
    try:
        with pytest.raises(ep.EpError) as ei:
            ep.ep_combine(h, FAKE, FAKE, None, FAKE, None, 0, None)
        assert ei.value.status == ep.EP_ERR_STATE
        with pytest.raises(ep.EpError) as ei:
            ep.ep_get_dispatch_src_token_pos(h)
        assert ei.value.status == ep.EP_ERR_STATE
        with pytest.raises(ep.EpError) as ei:
            ep.ep_combine_standard_moe(h, FAKE, FAKE, None, FAKE, 0, None)
        assert ei.value.status == ep.EP_ERR_STATE
        with pytest.raises(ep.EpError) as ei:
            ep.ep_convert_combine_input(h, FAKE, FAKE, None)
        assert ei.value.status == ep.EP_ERR_STATE
        # bad dispatch arguments are refused before any launch
        with pytest.raises(ep.EpError) as ei:
            ep.ep_dispatch(h, FAKE, FAKE, None, FAKE, [17] + [0] * 7, None)
        assert ei.value.status == ep.EP_ERR_INVALID_ARG
        with pytest.raises(ep.EpError) as ei:
            ep.ep_dispatch(h, FAKE + 8, FAKE, None, FAKE, [1] * 8, None)
        assert ei.value.status == ep.EP_ERR_INVALID_ARG
        with pytest.raises(ep.EpError) as ei:
            ep.ep_dispatch(h, None, FAKE, None, FAKE, [1] * 8, None)
        assert ei.value.status == ep.EP_ERR_INVALID_ARG
        with pytest.raises(ep.EpError) as ei:        # standard_moe = 0
            ep.ep_dispatch_standard_moe(h, FAKE, FAKE, None, FAKE, [1] * 8, None)
        assert ei.value.status == ep.EP_ERR_INVALID_ARG
        with pytest.raises(ep.EpError) as ei:        # no packed layout: no conversion
            ep.ep_convert_dispatch_output(h, FAKE, FAKE, None)
        assert ei.value.status == ep.EP_ERR_INVALID_ARG
        with pytest.raises(ep.EpError) as ei:        # no registered buffer reserved
            ep.ep_get_registered_combine_input_buffer(h)
        assert ei.value.status == ep.EP_ERR_STATE
        ep.ep_reset(h)
        assert "registered" in ep.ep_last_error()
    finally:
        ep.ep_destroy(h)


def test_launch_config_per_phase(ep):
    """ep_set_launch_config / ep_get_launch_config: per phase, validated,
    starting from the config's block_num / warp_num_per_block."""
    c = small(ep, block_num=300, warp_num_per_block=4)
    h = ep.ep_config_create(c, FAKE, ep.ep_workspace_size(c))
    try:
        assert ep.ep_get_launch_config(h, ep.EP_PHASE_DISPATCH) == (0, 300, 4)
        assert ep.ep_get_launch_config(h, ep.EP_PHASE_COMBINE) == (0, 300, 4)
        ep.ep_set_launch_config(h, ep.EP_PHASE_COMBINE, ep.EP_COMBINE_BULK, 456, 8)
        assert ep.ep_get_launch_config(h, ep.EP_PHASE_COMBINE) == (2, 456, 8)
        assert ep.ep_get_launch_config(h, ep.EP_PHASE_DISPATCH) == (0, 300, 4)
        ep.ep_set_launch_config(h, ep.EP_PHASE_DISPATCH, ep.EP_DISPATCH_VECTOR, -1, 2)
        assert ep.ep_get_launch_config(h, ep.EP_PHASE_DISPATCH) == (1, -1, 2)
        for bad in [(2, 0, -1, 8), (0, 3, -1, 8), (1, -1, -1, 8), (0, 0, -1, 9)]:
            with pytest.raises(ep.EpError) as ei:
                ep.ep_set_launch_config(h, *bad)
            assert ei.value.status == ep.EP_ERR_INVALID_ARG
        assert ep.ep_get_launch_config(h, ep.EP_PHASE_DISPATCH) == (1, -1, 2)
    finally:
        ep.ep_destroy(h)


# ------------------------------------------------- one rank per workspace (split phases)

def test_rank_workspace_size(ep):
    """A rank's workspace holds its own tokens' send buffers and one rank's
    receive buffers (cap = world_size * Tmax rows), the registered combine
    input included; the packed layout is not available per rank."""
    c = small(ep)
    n = ep.ep_rank_workspace_size(c)
    assert n >= 8 * 16 * 256 * 2 * 2           # receive payload + registered combine input
    assert n < ep.ep_workspace_size(c)          # one rank, not the whole group
    assert ep.ep_rank_workspace_size(small(ep, standard_moe=1)) == 0
    with pytest.raises(ep.EpError) as ei:
        ep.ep_rank_create(small(ep, standard_moe=1), 0, FAKE, 1 << 30)
    assert ei.value.status == ep.EP_ERR_UNSUPPORTED


def test_rank_create_and_peer_checks(ep):
    c = small(ep)
    n = ep.ep_rank_workspace_size(c)
    for bad in (-1, 8):
        with pytest.raises(ep.EpError) as ei:
            ep.ep_rank_create(c, bad, FAKE, n)
        assert ei.value.status == ep.EP_ERR_INVALID_ARG
    with pytest.raises(ep.EpError) as ei:
        ep.ep_rank_create(c, 0, FAKE + 64, n)
    assert ei.value.status == ep.EP_ERR_WORKSPACE
    with pytest.raises(ep.EpError) as ei:
        ep.ep_rank_create(c, 0, FAKE, n - 1)
    assert ei.value.status == ep.EP_ERR_WORKSPACE
    me = FAKE + 3 * (1 << 32)
    h = ep.ep_rank_create(c, 3, me, n)
    try:
        peers = [FAKE + r * (1 << 32) for r in range(8)]
        ep.ep_rank_set_peers(h, peers)
        for broken in ([p + 16 if r == 5 else p for r, p in enumerate(peers)],
                       [0 if r == 1 else p for r, p in enumerate(peers)],
                       [p + 256 if r == 3 else p for r, p in enumerate(peers)]):
            with pytest.raises(ep.EpError) as ei:   # misaligned, NULL, not this rank's own
                ep.ep_rank_set_peers(h, broken)
            assert ei.value.status == ep.EP_ERR_INVALID_ARG
    finally:
        ep.ep_rank_destroy(h)


def test_rank_phase_state_machine_without_device(ep):
    """READY -send-> SENT -recv-> DISPATCHED -combine_send-> COMBINE_SENT
    -combine_recv-> COMBINED: every out-of-order call is refused before any
    launch, and the receive phases need the peer table."""
    c = small(ep)
    n = ep.ep_rank_workspace_size(c)
    h = ep.ep_rank_create(c, 0, FAKE, n)
    try:
        for call in (lambda: ep.ep_dispatch_recv(h, None),
                     lambda: ep.ep_combine_send(h, FAKE, FAKE, FAKE, None, None),
                     lambda: ep.ep_combine_recv(h, 0, None),
                     lambda: ep.ep_rank_get_dispatch_src_token_pos(h)):
            with pytest.raises(ep.EpError) as ei:
                call()
            assert ei.value.status == ep.EP_ERR_STATE
        for args in ((FAKE, FAKE, None, FAKE, 17), (FAKE, FAKE, None, FAKE, -1),
                     (FAKE + 8, FAKE, None, FAKE, 1), (None, FAKE, None, FAKE, 1)):
            with pytest.raises(ep.EpError) as ei:
                ep.ep_dispatch_send(h, *args, None)
            assert ei.value.status == ep.EP_ERR_INVALID_ARG
        p = ep.ep_rank_get_registered_combine_input_buffer(h)
        assert FAKE <= p < FAKE + n and p % 256 == 0
        ep.ep_rank_reset(h)
    finally:
        ep.ep_rank_destroy(h)


def test_packed_only_config_refuses_the_2d_calls(ep):
    """A standard_moe = 1 workspace holds only the packed pool: the 2D
    dispatch and the conversions are refused before any launch."""
    c = small(ep, standard_moe=1)
    h = ep.ep_config_create(c, FAKE, ep.ep_workspace_size(c))
    try:
        with pytest.raises(ep.EpError) as ei:
            ep.ep_dispatch(h, FAKE, FAKE, None, FAKE, [1] * 8, None)
        assert ei.value.status == ep.EP_ERR_INVALID_ARG
        assert "packed layout" in ep.ep_last_error()
        with pytest.raises(ep.EpError) as ei:
            ep.ep_convert_dispatch_output(h, FAKE, FAKE, None)
        assert ei.value.status == ep.EP_ERR_INVALID_ARG
    finally:
        ep.ep_destroy(h)
