"""Parameter, byte and block counts against the numbers the pages print
(tests/golden/page_counts.json names the page and section of each)."""

import json
import os

import oracle

COUNTS = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_counts.json")))


def test_lora_params_match_pages():
    for e in COUNTS["lora_params"]:
        assert oracle.lora_params(e["d"], e["k"], e["r"]) == e["params"], e["source"]
        if "full_params" in e:
            assert e["d"] * e["k"] == e["full_params"]
            assert e["full_params"] // e["params"] == e["ratio"]
            assert oracle.adapter_bytes(e["k"], e["d"], e["r"], 2) == e["bytes_16bit"]
            assert e["full_params"] * 2 == e["full_bytes_16bit"]


def test_model_totals_match_pages():
    q_v, qkv = COUNTS["model_totals"]
    per_layer = sum(oracle.lora_params(d, k, q_v["r"]) for d, k in q_v["modules"])
    assert round(per_layer / 1e6, 2) == q_v["per_layer_millions_2dp"]
    total = per_layer * q_v["layers"]
    assert round(total / 1e6, 1) == q_v["total_millions_1dp"]
    # the page doubles its rounded 32.8M; the exact figure is 65,536,000 bytes
    assert round(2 * round(total / 1e6, 1), 1) == q_v["fp16_MB_1dp"]
    assert 2 * total == 65_536_000

    per_layer = sum(oracle.lora_params(d, k, qkv["r"]) for d, k in qkv["modules"])
    assert round(per_layer / 1e6, 2) == qkv["per_layer_millions_2dp"]
    assert per_layer * qkv["layers"] == qkv["exact_total"]
    # the page multiplies the rounded per-layer figure
    rounded = round(per_layer / 1e6, 2)
    assert round(rounded * qkv["layers"], 1) == qkv["total_millions_1dp_from_rounded_layer"]
    assert round(2 * rounded * qkv["layers"], 1) == qkv["fp16_MB_1dp_from_rounded_layer"]


def test_slot_memory_matches_go_demo():
    e = COUNTS["slot_memory"]
    base_bytes = e["layers"] * e["modules"] * e["d"] * e["d"] * 2
    assert base_bytes / 2**30 == e["base_GiB"]
    for r, mib in e["per_adapter_MiB"].items():
        one = oracle.slot_memory_numbers(1, e["layers"], e["modules"], e["d"], int(r)) * 2
        assert one / 2**20 == mib
        slots = oracle.slot_memory_numbers(e["max_loras"], e["layers"], e["modules"], e["d"], int(r)) * 2
        assert slots / 2**30 == e["slots_GiB"][r]
        # the slot formula is the adapter_bytes sum over square d x d modules
        per_module = oracle.adapter_bytes(e["d"], e["d"], int(r), 2)
        assert per_module * e["layers"] * e["modules"] == one


def test_paged_block_count():
    e = COUNTS["paged_blocks"]
    assert oracle.blocks_for(e["adapter_MiB"] * 2**20, e["block_KiB"] * 2**10) == e["blocks"]
    # a block of 16 rank-rows of a K = 8192 bf16 arena is exactly that 256 KiB
    assert 16 * 8192 * 2 == e["block_KiB"] * 2**10
