"""The oracle still reproduces the fixture tests/golden/make_golden.py wrote from it."""
import os

import numpy as np

import oracle
from moe_synth import make_layer, spec


def test_oracle_small_regression():
    g = np.load(os.path.join(os.path.dirname(__file__), "golden", "oracle_small.npz"))
    sp = spec("tiny_f32", T=16, H=64, I=96, E=8, k=2)
    L = make_layer(sp)
    r = oracle.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm)
    assert np.array_equal(r["ids"], g["ids"])
    np.testing.assert_allclose(r["out"], g["out"], rtol=1e-12, atol=1e-18)
    s, ex, npp, counts = oracle.align(r["ids"], sp.E, 4)
    assert np.array_equal(s, g["sorted_ids"]) and np.array_equal(ex, g["expert_ids"]) and npp == int(g["num_post_pad"])
