"""GB300-native MoE expert-parallel dispatch / combine (simulated EP ranks on one GPU).

The compute lives in libep.so (hand-written sm_103a CUDA kernels behind the C
ABI of include/ep.h); `ep` is its thin Python binding. The binding is loaded
on first use, so `combine_route_layout_gb300.build` can run before the
library exists; any other use fails loudly if the library is missing.
"""

_EXPORTS = ("EpDispatchCombineConfig", "EpDispatchCombineOp", "EpError")
_RANK_EXPORTS = ("EpRankOp", "exchange_workspaces", "phase_barrier")


def __getattr__(name):
    import importlib
    if name == "ep" or name in _EXPORTS:
        ep = importlib.import_module(".ep", __name__)
        return ep if name == "ep" else getattr(ep, name)
    if name == "ranks" or name in _RANK_EXPORTS:
        ranks = importlib.import_module(".ranks", __name__)
        return ranks if name == "ranks" else getattr(ranks, name)
    raise AttributeError(name)
