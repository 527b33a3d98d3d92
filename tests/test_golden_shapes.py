"""The synthetic workloads carry the shapes the pages print (tests/golden/page_shapes.json)."""
import json
import os

from moe_synth import spec

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_shapes.json")))


def test_mixtral_decode_matches_page_shapes():
    m = GOLD["mixtral_8x7b"]
    sp = spec("mixtral_decode")
    assert (sp.E, sp.k, sp.H, sp.I) == (m["experts"], m["topk"], m["hidden"], m["ffn"])


def test_fp8_decode_is_the_swap_ab_example():
    ex = GOLD["swap_ab_example"]
    sp = spec("fp8_decode", T=ex["A_rows_M"])
    # one token row of hidden size K against an expert block whose N is the
    # example's 8192 (the FP8 workload's intermediate size), at top-k = 8
    assert (sp.T, sp.H, sp.I, sp.k) == (ex["A_rows_M"], ex["A_cols_K"], ex["B_cols_N"],
                                        GOLD["fused_topk_example"]["topk"])
