"""moe_forward_noalloc: the layer for callers that cannot allocate device memory.

It must give the same results as moe_forward (which takes a caller-allocated
workspace), call after call, using only the library's fixed device array.
Both entry points build the same plan and run the same deterministic kernels,
so their outputs are compared bit for bit (which is also within every
tolerance of the parity tests).  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from helpers import assert_parity, make_tie_free
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


CASES = [("tiny_f32", {"T": 64}, "f32", None),
         ("fine_decode", {"T": 64}, "bf16", None),
         ("mixtral_decode", {"T": 5, "I": 2048}, "bf16", None),
         ("mixtral_decode", {"T": 5, "I": 2048}, "bf16", {"single_launch": 1}),
         ("fp8_decode", {"T": 16, "H": 1024, "I": 1024}, "e4m3", None),
         ("int4_decode", {"T": 9, "H": 1024, "I": 1024}, "bf16", None)]


def _args(L):
    sp = L["spec"]
    return (L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm, L["w13_scale"], L["w2_scale"])


def _wfmt(L):
    return "int4" if L["spec"].w == "int4" else None


def _noalloc_equals_forward(moe, L, kind, options, label):
    ref = moe.moe_forward(*_args(L), options=options, w_format=_wfmt(L))
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    out = torch.full_like(L["X"], float("nan"))
    before = torch.cuda.memory_allocated()
    moe.moe_forward_noalloc(*_args(L), out=out, options=options, w_format=_wfmt(L))
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    assert torch.cuda.memory_allocated() == before
    assert torch.equal(out, ref), f"{label}: differs from moe_forward"
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert_parity(got, ref.float().cpu().numpy(), kind, label)


@pytest.mark.parametrize("name,kw,kind,options", CASES)
def test_noalloc_matches_moe_forward_twice(moe, name, kw, kind, options):
    L = _layer(name, **kw)
    for call in range(2):
        _noalloc_equals_forward(moe, L, kind, options, f"noalloc {name} {options} call {call}")


def test_noalloc_single_launch_after_other_shapes(moe):
    """The single-launch kernel keeps a launch tag and counters in the workspace: a single-launch
    call, a multi-kernel call of another shape that overwrites the shared array, then the
    single-launch call again, all equal to moe_forward on fresh workspaces."""
    fused = {"single_launch": 1}
    a = _layer("mixtral_decode", T=5, I=2048)
    b = _layer("fine_decode", T=48)
    c = _layer("fine_decode", T=7, H=512, I=256, E=32)
    _noalloc_equals_forward(moe, a, "bf16", fused, "fused A")
    _noalloc_equals_forward(moe, b, "bf16", None, "multi-kernel B")
    _noalloc_equals_forward(moe, a, "bf16", fused, "fused A again")
    _noalloc_equals_forward(moe, c, "bf16", fused, "fused C")
    _noalloc_equals_forward(moe, a, "bf16", fused, "fused A third")


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
