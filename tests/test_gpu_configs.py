"""GPU parity at the full sizes of the five workloads, in the launch configuration the
benchmark times (automatic orientation and splits).

Decode workloads are checked on every output token; prefill (T = 8192) on a
seeded sample of tokens the oracle computes one by one.  Weights are drawn on
the device by torch's seeded generator (an input, not a result of this
library) and copied to the host for the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_parity, make_tie_free
from moe_synth import make_layer, spec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_layer_scan_gb300 as m

    assert torch.cuda.is_available()
    return m


def _check(moe, name, T, n_sample=None, seed=None):
    sp = spec(name, T=T) if seed is None else spec(name, T=T, seed=seed)
    L = make_layer(sp, device="cuda")
    make_tie_free(L)
    out = moe.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm, L["w13_scale"], L["w2_scale"])
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    tokens = None
    if n_sample is not None:
        g = np.random.default_rng(sp.seed)
        tokens = np.sort(g.choice(T, size=n_sample, replace=False)).astype(np.int32)
    cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}
    ref = oracle.moe_forward(cpu["X"], cpu["Wr"], cpu["W13"], cpu["W2"], sp.k, sp.renorm, cpu["w13_scale"],
                             cpu["w2_scale"], tokens=tokens)["out"]
    got = out.float().cpu().numpy()
    if tokens is not None:
        got = got[tokens]
    kind = "e4m3" if sp.w == "e4m3" else sp.act
    return assert_parity(got, ref, kind, f"{name} T={T} seed={sp.seed}")


def test_tiny_f32_full(moe):
    _check(moe, "tiny_f32", 64)


@pytest.mark.parametrize("M", [1, 4, 16, 64])
def test_mixtral_decode_full(moe, M):
    _check(moe, "mixtral_decode", M)


@pytest.mark.parametrize("M", [1, 8, 32, 64])
def test_fine_decode_full(moe, M):
    _check(moe, "fine_decode", M)


@pytest.mark.parametrize("M", [1, 16, 64])
def test_fp8_decode_full(moe, M):
    _check(moe, "fp8_decode", M)


@pytest.mark.parametrize("name", ["prefill", "prefill_hot"])
@pytest.mark.parametrize("draw", range(8))
def test_prefill_full_sampled(moe, name, draw):
    """Eight independent draws of each prefill workload (the benchmark's draw first), 192 sampled
    tokens each."""
    base = spec(name, T=8192).seed
    _check(moe, name, 8192, n_sample=192, seed=base + 1000 * draw)
