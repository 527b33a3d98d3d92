"""Sentinel checks (compute-sanitizer is closed on this machine; these stand in for its
initialisation and out-of-bounds checks on the layer's own buffers).

* The workspace is filled with NaN / garbage bit patterns before a call: the output must
  be bit-identical to a call on a zero-filled workspace, so no word the kernels read is
  left over from an earlier call or uninitialised (padding rows included).
* `out` is pre-filled with a sentinel: every element must be overwritten, and nothing is
  written past its end (a guard region after `out` keeps its sentinel).
Both orientations, single CTAs and CTA pairs, K splits, the FP8 and INT4 paths, and the
single-launch kernel.
"""
import pytest
import torch

from helpers import make_tie_free
from moe_synth import make_layer, spec

pytestmark = pytest.mark.gpu

CASES = [("mixtral_decode", dict(T=7, H=512, I=384, E=8, k=2), {}),
         ("fine_decode", dict(T=33, H=512, I=256, E=64, k=8), {"split_k": 3}),
         ("fine_decode", dict(T=6, H=512, I=256, E=64, k=8), {"split_k": 3}),  # splits summed in GEMM1
         ("prefill", dict(T=300, H=512, I=256, E=8, k=2), {"orientation": 2, "cta_pair": 1}),
         ("prefill", dict(T=300, H=512, I=256, E=8, k=2), {"orientation": 2, "cta_pair": 2}),
         ("fp8_decode", dict(T=20, H=512, I=256, E=16, k=4), {}),
         ("fp8_decode", dict(T=260, H=512, I=256, E=8, k=2), {"orientation": 2}),
         ("int4_decode", dict(T=9, H=512, I=512, E=8, k=2), {}),
         ("mixtral_decode", dict(T=5, H=512, I=384, E=8, k=2), {"single_launch": 1}),
         ("tiny_f32", dict(T=40, H=128, I=96, E=8, k=2), {})]


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_layer_scan_gb300 as m

    assert torch.cuda.is_available()
    return m


@pytest.mark.parametrize("name,kw,options", CASES)
def test_stale_workspace_and_sentinel_output(moe, name, kw, options):
    L = make_layer(spec(name, **kw))
    make_tie_free(L)
    sp = L["spec"]
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}
    wfmt = "int4" if sp.w == "int4" else None
    act = moe.MOE_F32 if sp.act == "f32" else moe.MOE_BF16
    wdt = {"f32": moe.MOE_F32, "bf16": moe.MOE_BF16, "e4m3": moe.MOE_E4M3, "int4": moe.MOE_INT4}[sp.w]
    need = moe.moe_workspace_size(sp.T, sp.H, sp.I, sp.E, sp.k, act, wdt, options)
    outs = []
    for fill in (0x00, 0xFF, 0x7F, 0xA5):  # zeros, NaN patterns, large values, garbage
        ws = torch.full((need,), fill, dtype=torch.uint8, device="cuda")
        guard = 4096
        buf = torch.empty(d["X"].numel() + guard, dtype=d["X"].dtype, device="cuda")
        buf.fill_(float("nan"))
        out = buf[: d["X"].numel()].view_as(d["X"])
        moe.moe_forward(d["X"], d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm, d["w13_scale"], d["w2_scale"], out=out,
                        workspace=ws, options=options, w_format=wfmt)
        torch.cuda.synchronize()
        assert moe.moe_get_status() == 0
        assert torch.isfinite(out).all(), f"fill {fill:#x}: an output element was not written"
        assert torch.isnan(buf[d["X"].numel():]).all(), f"fill {fill:#x}: a write past the end of out"
        outs.append(out.clone())
    for o in outs[1:]:
        assert torch.equal(o, outs[0]), "the result depends on the workspace's previous contents"
