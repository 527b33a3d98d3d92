"""Writes tests/golden/oracle_small.npz from the CPU oracle only (regression fixture).

Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from moe_synth import make_layer, spec  # noqa: E402


def main():
    sp = spec("tiny_f32", T=16, H=64, I=96, E=8, k=2)
    L = make_layer(sp)
    r = oracle.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm)
    s, ex, npp, counts = oracle.align(r["ids"], sp.E, 4)
    np.savez(os.path.join(os.path.dirname(__file__), "oracle_small.npz"), out=r["out"], ids=r["ids"], w=r["w"],
             sorted_ids=s, expert_ids=ex, num_post_pad=np.int32(npp), counts=counts)


if __name__ == "__main__":
    main()
