"""The byte model reproduces the pages' worked speed-of-light example and the
shapes of the full-scale model."""
import json
import os

from persistent_moe_decode_02_gb300.roofline import sol_tokens_per_s, step_bytes
from synth import FULL, Dims

HERE = os.path.dirname(os.path.abspath(__file__))


def test_pages_worked_example():
    g = json.load(open(os.path.join(HERE, "golden", "pages_sol_example.json")))
    sol = sol_tokens_per_s(g["weight_bytes"] + g["kv_bytes"], 1, g["hbm_bytes_per_s"])
    assert round(sol, -1) == g["ceiling_tok_s_printed"]          # 471.8 -> "about 470"
    assert round(100 * g["megakernel_tok_s"] / sol) == g["megakernel_pct_printed"]
    assert round(100 * g["vllm_tok_s"] / sol) == g["vllm_pct_printed"]
    assert round(g["megakernel_tok_s"] / g["vllm_tok_s"], 2) == g["speedup_printed"]


def test_full_shape_bs1_8k_bytes():
    b = step_bytes(FULL, [8192])
    # 3.3B-class active parameters: 6.08 GB of bf16 weights (the LM head and
    # the 8 selected experts per layer included, the embedding as one row).
    assert round(b["weights"] / 1e9, 3) == 6.084
    assert round(b["kv_read"] / 1e9, 3) == 0.805
    assert round(b["total"] / 1e9, 2) == 6.89


def test_union_counts_each_expert_once():
    D = Dims(1, 64, 2, 1, 32, 8, 2, 16, 100)
    one = step_bytes(D, [10, 20], union_per_layer=[2])["weights"]
    two = step_bytes(D, [10, 20], union_per_layer=[4])["weights"]
    assert two - one == 2 * 2 * 3 * 64 * 16
    assert step_bytes(D, [5], logits=True)["logits"] == 4 * 100
