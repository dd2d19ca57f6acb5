"""Tuning files (MORI-EP User Guide, section 10 Tuning, read by section 6's
auto mode): rule lookup, replacement and ordering, on the CPU."""
import json

import pytest
import torch

from combine_route_layout_gb300 import tuning


def rule(dtype, hidden, tokens, grid=608, warps=8, impl="vector"):
    return {"dtype": dtype, "num_tokens": tokens, "hidden_dim": hidden, "impl": impl,
            "block_num": grid, "warp_per_block": warps, "latency_us": 1.0,
            "bandwidth_gbps": 1.0}


def test_lookup_smallest_at_or_above_else_largest():
    rules = [rule("fp8", 7168, 128, 304), rule("fp8", 7168, 1024, 608),
             rule("fp8", 7168, 4096, 1216), rule("bf16", 7168, 128, 152),
             rule("fp8", 4096, 128, 76)]
    assert tuning.lookup(rules, "fp8", 7168, 1)["block_num"] == 304
    assert tuning.lookup(rules, "fp8", 7168, 128)["block_num"] == 304
    assert tuning.lookup(rules, "fp8", 7168, 129)["block_num"] == 608
    assert tuning.lookup(rules, "fp8", 7168, 4096)["block_num"] == 1216
    assert tuning.lookup(rules, "fp8", 7168, 9000)["block_num"] == 1216
    assert tuning.lookup(rules, "bf16", 7168, 4096)["block_num"] == 152
    assert tuning.lookup(rules, "fp8", 4096, 64)["block_num"] == 76
    assert tuning.lookup(rules, "fp4", 7168, 128) is None
    assert tuning.lookup([], "fp8", 7168, 128) is None


def test_save_replaces_and_sorts(tmp_path, capsys):
    d = str(tmp_path)
    tuning.save_rule("2d", 8, "dispatch", rule("fp8", 7168, 4096, 1216), d)
    tuning.save_rule("2d", 8, "dispatch", rule("bf16", 4096, 2048, 608), d)
    tuning.save_rule("2d", 8, "dispatch", rule("fp8", 7168, 128, 304), d)
    p = tuning.save_rule("2d", 8, "dispatch", rule("fp8", 7168, 4096, 912, 4), d)
    assert "replace" in capsys.readouterr().out
    assert p.endswith("sm103_gb300_2d_ep8_dispatch.json")
    doc = json.load(open(p))
    assert doc["ep_size"] == 8 and doc["phase"] == "dispatch" and doc["kernel_type"] == "2d"
    keys = [(r["dtype"], r["hidden_dim"], r["num_tokens"]) for r in doc["rules"]]
    assert keys == [("bf16", 4096, 2048), ("fp8", 7168, 128), ("fp8", 7168, 4096)]
    assert doc["rules"][-1]["block_num"] == 912 and doc["rules"][-1]["warp_per_block"] == 4
    assert tuning.load_rules("2d", 8, "dispatch", d) == doc["rules"]
    assert tuning.load_rules("2d", 8, "combine", d) == []


def test_config_dir_from_environment(tmp_path, monkeypatch):
    monkeypatch.setenv("EP_TUNING_CONFIG_DIR", str(tmp_path))
    assert tuning.rules_path("stdmoe", 4, "combine").startswith(str(tmp_path))


def test_committed_rule_files_are_well_formed():
    import glob
    import os
    files = glob.glob(os.path.join(os.path.dirname(tuning.__file__), "tuning_configs", "*.json"))
    for p in files:
        doc = json.load(open(p))
        assert doc["phase"] in ("dispatch", "combine")
        keys = [(r["dtype"], r["hidden_dim"], r["num_tokens"]) for r in doc["rules"]]
        assert keys == sorted(keys) and len(set(keys)) == len(keys)
        for r in doc["rules"]:
            assert r["impl"] in ("vector", "bulk") and r["warp_per_block"] <= 8


def test_dtype_names():
    from combine_route_layout_gb300.ep import EpDispatchCombineConfig
    base = dict(data_type=torch.bfloat16, world_size=8, hidden_dim=7168, scale_dim=0,
                scale_type_size=4, max_token_type_size=4, max_num_inp_token_per_rank=128,
                num_experts_per_rank=32, num_experts_per_token=8)
    assert tuning.dispatch_dtype_name(EpDispatchCombineConfig(**base)) == "bf16"
    assert tuning.dispatch_dtype_name(
        EpDispatchCombineConfig(**base, quant_type="fp8_e4m3_block128")) == "fp8"
    assert tuning.dispatch_dtype_name(
        EpDispatchCombineConfig(**base, quant_type="fp4_e2m1_block32")) == "fp4"
    assert tuning.combine_dtype_name(
        EpDispatchCombineConfig(**base, combine_dtype=torch.float32)) == "fp32"
    c = EpDispatchCombineConfig(**base, launch_config_mode="auto")
    assert c.auto_launch()
    assert not hasattr(c.to_c(), "launch_config_mode")
