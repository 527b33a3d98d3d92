"""moe_forward_noalloc: the layer for callers that cannot allocate device memory.

It must give the same results as moe_forward (which takes a caller-allocated
workspace), call after call, using only the library's fixed device array.
This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from helpers import TOL, make_tie_free, rel_err
from moe_synth import make_layer, spec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_layer_scan_gb300 as m

    assert torch.cuda.is_available()
    return m


def _layer(name, **kw):
    L = make_layer(spec(name, **kw))
    make_tie_free(L)
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}


CASES = [("tiny_f32", {"T": 64}, "f32"),
         ("fine_decode", {"T": 64}, "bf16"),
         ("mixtral_decode", {"T": 5, "I": 2048}, "bf16"),
         ("fp8_decode", {"T": 16, "H": 1024, "I": 1024}, "e4m3")]


@pytest.mark.parametrize("name,kw,tol", CASES)
def test_noalloc_matches_moe_forward_twice(moe, name, kw, tol):
    L = _layer(name, **kw)
    sp = L["spec"]
    args = (L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm, L["w13_scale"], L["w2_scale"])
    ref = moe.moe_forward(*args)
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    ref = ref.float().cpu().numpy()
    for call in range(2):
        out = torch.full_like(L["X"], float("nan"))
        before = torch.cuda.memory_allocated()
        moe.moe_forward_noalloc(*args, out=out)
        torch.cuda.synchronize()
        assert moe.moe_get_status() == 0
        assert torch.cuda.memory_allocated() == before
        got = out.float().cpu().numpy()
        assert np.isfinite(got).all()
        assert rel_err(got, ref, f"noalloc {name} call {call}") <= TOL[tol]


def test_noalloc_rejects_shapes_beyond_its_array(moe):
    sp = spec("prefill", T=8192)
    need = moe.moe_workspace_size(sp.T, sp.H, sp.I, sp.E, sp.k, moe.MOE_BF16, moe.MOE_BF16)
    assert need > moe.NOALLOC_MAX_WORKSPACE
    X = torch.zeros(sp.T, sp.H, dtype=torch.bfloat16, device="cuda")
    Wr = torch.zeros(sp.E, sp.H, dtype=torch.bfloat16, device="cuda")
    W13 = torch.zeros(sp.E, 2 * 128, sp.H, dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros(sp.E, sp.H, 128, dtype=torch.bfloat16, device="cuda")
    need_small = moe.moe_workspace_size(sp.T, sp.H, 128, sp.E, sp.k, moe.MOE_BF16, moe.MOE_BF16)
    assert need_small > moe.NOALLOC_MAX_WORKSPACE
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward_noalloc(X, Wr, W13, W2, sp.k, True)
    assert e.value.code == moe.MOE_ERR_WORKSPACE
