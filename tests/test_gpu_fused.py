"""GPU parity of the single-launch decode kernel (the whole layer as one cooperative
kernel): against the CPU oracle within the bf16 tolerance, and bit for bit against
the multi-kernel sequence, which performs the same arithmetic in the same order.

Covers activation tiles gathered inside GEMM1 (<= 32 tokens) and gathered into
expert order first (33-64 tokens), K-split GEMM1 (partials summed by the CTA that
finishes the last split) and unsplit GEMM1, a hidden size with a half last GEMM2
tile, full-softmax weights (no renorm), 256 experts, the 512-pair limit, repeated
launches on one workspace, and CUDA-graph replay.

Parity against the oracle uses the bf16 reading of the tolerance: the error
beyond the final rounding of out to bf16 within 2e-2 of RMS(out), and the plain
max|err|/RMS within 2e-2 wherever that rounding can cost at most half of it.
Several shapes (fine-grained routing with small H) put outputs at 6-9 RMS.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, assert_parity, make_tie_free, rel_err
from moe_synth import make_layer, spec

pytestmark = pytest.mark.gpu

FUSED = {"single_launch": 1}
MULTI = {"single_launch": 2}


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_layer_scan_gb300 as m

    assert torch.cuda.is_available()
    return m


def _layer(name, **kw):
    L = make_layer(spec(name, **kw))
    make_tie_free(L)
    return L


def _dev(L):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}


def _run(moe, d, options):
    sp = d["spec"]
    out = moe.moe_forward(d["X"], d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm, options=options)
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    return out


def _ref(L):
    sp = L["spec"]
    return oracle.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm)["out"]


SHAPES = [  # name, T, H, I, E, k
    ("mixtral_decode", 1, 256, 384, 8, 2),
    ("mixtral_decode", 7, 384, 256, 16, 4),
    ("mixtral_decode", 33, 256, 256, 8, 2),
    ("fine_decode", 64, 512, 256, 64, 8),
    ("fine_decode", 5, 512, 384, 128, 8),
    ("fine_decode", 16, 640, 256, 64, 8),
    ("fine_decode", 3, 256, 256, 256, 8),
    ("fine_decode", 64, 256, 256, 128, 8),
    ("fine_decode", 40, 256, 128, 64, 8),
    ("fine_decode", 24, 256, 256, 32, 4),
]



@pytest.mark.parametrize("name,T,H,I,E,k,renorm", [s + (True,) for s in SHAPES] + [("fine_decode", 9, 256, 256, 32, 8,
                                                                                           False)])
def test_single_launch_matches_oracle_and_multi_kernel(moe, name, T, H, I, E, k, renorm):
    L = _layer(name, T=T, H=H, I=I, E=E, k=k, renorm=renorm)
    d = _dev(L)
    plan = moe.moe_plan_info(T, H, I, E, k, moe.MOE_BF16, moe.MOE_BF16, FUSED)
    assert plan["single_launch"] == 1 and plan["kernel_launches"] == 1
    fused = _run(moe, d, FUSED)
    multi = _run(moe, d, MULTI)
    assert_parity(fused.float().cpu().numpy(), _ref(L), "bf16", f"single launch {name} T={T} E={E}")
    assert torch.equal(fused, multi)


@pytest.mark.parametrize("split_k", [1, 2, 3])
def test_single_launch_k_splits(moe, split_k):
    """GEMM1 unsplit (SiLU in the epilogue) and split (partials summed by the last CTA of a tile)."""
    L = _layer("fine_decode", T=6, H=768, I=256, E=16, k=4)
    d = _dev(L)
    f = _run(moe, d, {"single_launch": 1, "split_k": split_k})
    m = _run(moe, d, {"single_launch": 2, "split_k": split_k})
    assert_parity(f.float().cpu().numpy(), _ref(L), "bf16", f"split_k={split_k}")
    assert torch.equal(f, m)


@pytest.mark.parametrize("act_split", [1, 2])
def test_single_launch_intermediate_single_or_hi_lo(moe, act_split):
    L = _layer("mixtral_decode", T=12, H=384, I=256, E=8, k=2)
    d = _dev(L)
    f = _run(moe, d, {"single_launch": 1, "act_split": act_split})
    m = _run(moe, d, {"single_launch": 2, "act_split": act_split})
    assert_parity(f.float().cpu().numpy(), _ref(L), "bf16", f"act_split={act_split}")
    assert torch.equal(f, m)


def test_single_launch_repeated_on_one_workspace(moe):
    """Back-to-back launches reuse the workspace counters: each launch zeroes and tags its own."""
    L = _layer("fine_decode", T=4, H=512, I=256, E=32, k=8)
    d = _dev(L)
    sp = d["spec"]
    ws = torch.empty(moe.moe_workspace_size(4, 512, 256, 32, 8, moe.MOE_BF16, moe.MOE_BF16, FUSED),
                     dtype=torch.uint8, device="cuda")
    outs = []
    Xs = [d["X"], torch.flip(d["X"], dims=[0]).contiguous(), d["X"] * 0.5]
    for r in range(6):
        outs.append(moe.moe_forward(Xs[r % 3], d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm, workspace=ws,
                                    options=FUSED))
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    for r in range(6):
        ref = moe.moe_forward(Xs[r % 3], d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm, options=MULTI)
        assert torch.equal(outs[r], ref)


def test_single_launch_graph_replay(moe):
    """A captured launch replayed with new inputs: every replay zeroes its counters again."""
    L = _layer("mixtral_decode", T=3, H=512, I=384, E=8, k=2)
    d = _dev(L)
    sp = d["spec"]
    X = d["X"].clone()
    ws = torch.empty(moe.moe_workspace_size(3, 512, 384, 8, 2, moe.MOE_BF16, moe.MOE_BF16, FUSED),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty(3, 512, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        moe.moe_forward(X, d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm, out=out, workspace=ws, options=FUSED,
                        stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.moe_forward(X, d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm, out=out, workspace=ws, options=FUSED,
                        stream=torch.cuda.current_stream())
    gen = torch.Generator(device="cpu").manual_seed(7)
    for r in range(4):
        newx = torch.randn(3, 512, generator=gen).to(torch.bfloat16).cuda()
        X.copy_(newx)
        g.replay()
        torch.cuda.synchronize()
        assert moe.moe_get_status() == 0
        ref = moe.moe_forward(newx, d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm, options=MULTI)
        assert torch.equal(out, ref), f"replay {r}"


def test_single_launch_refuses_unsupported_shapes(moe):
    with pytest.raises(moe.MoeError) as e:
        moe.moe_plan_info(65, 256, 256, 8, 2, moe.MOE_BF16, moe.MOE_BF16, {"single_launch": 1, "orientation": 1})
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoeError) as e:
        moe.moe_plan_info(8, 256, 256, 8, 2, moe.MOE_BF16, moe.MOE_E4M3, FUSED)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoeError) as e:
        moe.moe_plan_info(8, 256, 256, 300, 2, moe.MOE_BF16, moe.MOE_BF16, FUSED)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("name,M", [("mixtral_decode", 1), ("mixtral_decode", 16), ("mixtral_decode", 64),
                                    ("fine_decode", 1), ("fine_decode", 8), ("fine_decode", 64)])
def test_single_launch_full_size(moe, name, M):
    """The workloads at full size: every output token against the oracle, and bit for bit against the
    multi-kernel sequence whenever both plans use the same K splits (the single launch runs GEMM1
    unsplit above 8 tokens)."""
    sp = spec(name, T=M)
    L = make_layer(sp, device="cuda")
    make_tie_free(L)
    f = moe.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm, options=FUSED)
    m = moe.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm, options=MULTI)
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    pf = moe.moe_plan_info(M, sp.H, sp.I, sp.E, sp.k, moe.MOE_BF16, moe.MOE_BF16, FUSED)
    pm = moe.moe_plan_info(M, sp.H, sp.I, sp.E, sp.k, moe.MOE_BF16, moe.MOE_BF16, MULTI)
    if (pf["splits_gemm1"], pf["splits_gemm2"]) == (pm["splits_gemm1"], pm["splits_gemm2"]):
        assert torch.equal(f, m)
    cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}
    ref = oracle.moe_forward(cpu["X"], cpu["Wr"], cpu["W13"], cpu["W2"], sp.k, sp.renorm)["out"]
    assert_parity(f.float().cpu().numpy(), ref, "bf16", f"single launch {name} M={M}")


@pytest.mark.parametrize("M", [16, 64])
def test_single_launch_unsplit_gemm1_matches_forced_plan(moe, M):
    """Above 8 tokens the single launch runs GEMM1 unsplit: the same as both paths forced to one split."""
    sp = spec("fine_decode", T=M, H=1024, I=512, E=64)
    L = make_layer(sp, device="cuda")
    pf = moe.moe_plan_info(M, sp.H, sp.I, sp.E, sp.k, moe.MOE_BF16, moe.MOE_BF16, FUSED)
    assert pf["splits_gemm1"] == 1
    opts = {"split_k": 1}
    f = moe.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm, options={**FUSED, **opts})
    m = moe.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm, options={**MULTI, **opts})
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    assert torch.equal(f, m)
