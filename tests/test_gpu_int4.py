"""GPU parity of the INT4 weight-only layer (codes dequantised to bf16 inside the GEMM main
loop) against the oracle, and bit for bit against the bf16 layer run on the same weights
decoded outside (same tiles and one K split, so the same MMA inputs in the same order).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, assert_parity, make_tie_free, rel_err
from moe_synth import INT4_NIBBLE_OF, make_layer, spec

pytestmark = pytest.mark.gpu
INT4 = {"w_format": "int4"}


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_layer_scan_gb300 as m

    assert torch.cuda.is_available()
    return m


def _decoded(packed, scales):
    """bf16 weights [.., rows, K] from packed codes [.., rows, K/2] and group-major scales [.., K/128, rows]."""
    b = packed.to(torch.int32)
    *lead, rows, kh = b.shape
    words = (b.reshape(*lead, rows, kh // 4, 4) << torch.tensor([0, 8, 16, 24], dtype=torch.int32)).sum(-1)
    q = torch.stack([(words >> (4 * INT4_NIBBLE_OF[e])) & 0xF for e in range(8)], dim=-1).reshape(*lead, rows, kh * 2)
    q = torch.where(q >= 8, q - 16, q).float()
    return (q * scales.transpose(-1, -2).float().repeat_interleave(128, dim=-1)).to(torch.bfloat16)


def _layer(T, H, I, E, k, name="int4_decode"):
    L = make_layer(spec(name, T=T, H=H, I=I, E=E, k=k))
    make_tie_free(L)
    return L


def _run(moe, L, options=None, dev_weights=None):
    sp = L["spec"]
    d = {kk: (v.cuda() if isinstance(v, torch.Tensor) else v) for kk, v in L.items()}
    out = moe.moe_forward(d["X"], d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm, d["w13_scale"], d["w2_scale"],
                          options=options, **INT4)
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    return out


@pytest.mark.parametrize("T,H,I,E,k", [(1, 256, 256, 8, 2), (5, 512, 256, 16, 4), (33, 256, 512, 8, 2),
                                       (64, 512, 512, 32, 8), (100, 256, 256, 8, 2)])
def test_int4_layer_matches_oracle(moe, T, H, I, E, k):
    L = _layer(T, H, I, E, k)
    out = _run(moe, L)
    sp = L["spec"]
    ref = oracle.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm, L["w13_scale"], L["w2_scale"],
                             w_format="int4")["out"]
    assert_parity(out.float().cpu().numpy(), ref, "bf16", f"int4 T={T}")


@pytest.mark.parametrize("T,splits,act_split", [(3, 1, 2), (3, 2, 2), (20, 1, 2), (48, 1, 2), (20, 1, 1), (3, 2, 1)])
def test_int4_layer_equals_bf16_layer_on_decoded_weights(moe, T, splits, act_split):
    """Same plan on both: K splits and the intermediate's form (hi + lo, or one bf16; the INT4 default
    is one bf16, the bf16 path's default hi + lo)."""
    L = _layer(T, 512, 512, 16, 4)
    sp = L["spec"]
    opts = {"split_k": splits, "act_split": act_split}
    a = _run(moe, L, opts)
    W13 = _decoded(L["W13"], L["w13_scale"]).cuda()
    W2 = _decoded(L["W2"], L["w2_scale"]).cuda()
    b = moe.moe_forward(L["X"].cuda(), L["Wr"].cuda(), W13, W2, sp.k, sp.renorm, options=opts)
    torch.cuda.synchronize()
    # same MMA inputs in the same order: INT4 splits K in 128-element raw stages and bf16 in
    # 64-element blocks, and at H = I = 512 both put a two-way split at element 256
    assert torch.equal(a, b)


def test_int4_refuses_token_major(moe):
    with pytest.raises(moe.MoeError) as e:
        moe.moe_plan_info(512, 512, 512, 8, 2, moe.MOE_BF16, moe.MOE_INT4, {"orientation": 2})
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("T,H,I", [(129, 512, 512), (8, 384, 512), (8, 512, 640)])
def test_int4_refuses_unsupported_shapes(moe, T, H, I):
    """More than 128 tokens, or H / I not a multiple of the 256-row weight tile."""
    with pytest.raises(moe.MoeError) as e:
        moe.moe_plan_info(T, H, I, 8, 2, moe.MOE_BF16, moe.MOE_INT4)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED


def test_int4_empty_batch(moe):
    L = _layer(4, 256, 256, 8, 2)
    sp = L["spec"]
    d = {kk: (v.cuda() if isinstance(v, torch.Tensor) else v) for kk, v in L.items()}
    out = moe.moe_forward(d["X"][:0], d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm, d["w13_scale"], d["w2_scale"],
                          **INT4)
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0 and out.shape == (0, 256)


def test_int4_graph_replay_and_determinism(moe):
    """A captured INT4 layer replayed on new inputs equals eager calls bit for bit."""
    L = _layer(6, 512, 256, 16, 4)
    sp = L["spec"]
    d = {kk: (v.cuda() if isinstance(v, torch.Tensor) else v) for kk, v in L.items()}
    X = d["X"].clone()
    ws = torch.empty(moe.moe_workspace_size(6, 512, 256, 16, 4, moe.MOE_BF16, moe.MOE_INT4), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(6, 512, dtype=torch.bfloat16, device="cuda")
    args = (d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm, d["w13_scale"], d["w2_scale"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        moe.moe_forward(X, *args, out=out, workspace=ws, stream=s, **INT4)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.moe_forward(X, *args, out=out, workspace=ws, stream=torch.cuda.current_stream(), **INT4)
    gen = torch.Generator(device="cpu").manual_seed(11)
    for r in range(3):
        newx = torch.randn(6, 512, generator=gen).to(torch.bfloat16).cuda()
        X.copy_(newx)
        g.replay()
        torch.cuda.synchronize()
        assert moe.moe_get_status() == 0
        ref = moe.moe_forward(newx, *args, **INT4)
        assert torch.equal(out, ref), f"replay {r}"


@pytest.mark.parametrize("M", [1, 16, 64])
def test_int4_decode_full_size(moe, M):
    sp = spec("int4_decode", T=M)
    L = make_layer(sp, device="cuda")
    make_tie_free(L)
    out = moe.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm, L["w13_scale"], L["w2_scale"], **INT4)
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    tokens = np.arange(M) if M <= 16 else np.sort(np.random.default_rng(5).choice(M, 16, replace=False))
    cpu = {kk: (v.cpu() if isinstance(v, torch.Tensor) else v) for kk, v in L.items()}
    ref = oracle.moe_forward(cpu["X"], cpu["Wr"], cpu["W13"], cpu["W2"], sp.k, sp.renorm, cpu["w13_scale"],
                             cpu["w2_scale"], tokens=tokens.astype(np.int32), w_format="int4")["out"]
    assert_parity(out.float().cpu().numpy()[tokens], ref, "bf16", f"int4 full M={M}")
