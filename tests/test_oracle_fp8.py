"""Pins of the oracle's FP8 quantisation points against independent derivations.

The FP8 layer ("Mixture-of-Experts kernel engineering on Amazon SageMaker AI",
section "Routage backend pour la quantisation des tenseurs FP8": per-tensor
FP8) quantises the layer input with one dynamic scale s_a1 = amax(X)/448, the
SiLU(gate)*up intermediate with one dynamic scale s_a2 = amax/448 over every
routed (token, expert) pair of the call, and dequantises with the per-expert
weight scales in the GEMM epilogues.  Each test below builds inputs on which
the answer follows from that definition without the oracle:

* inputs on a scaled e4m3 grid (x = code * s_a1 exactly), so that the input
  quantisation is exact and the layer differs from the fp64 layer on the
  dequantised weights only by the e4m3 rounding of the intermediate, whose
  bound is computed element by element from an fp64 intermediate formed in
  torch;
* a two-token layer whose expected output is derived in the test from the
  definition, with torch's e4m3 cast as the rounding routine.

Together they fail if the oracle drops or inverts s_a1, ignores or misindexes
the per-expert w13 scale, takes s_a2 per token, or takes it over a requested
subset of tokens instead of every token of the call.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

E4M3_MAX = 448.0


def _e4(codes) -> np.ndarray:
    return oracle.e4m3_to_f64(np.asarray(codes, np.uint8).ravel()).reshape(np.shape(codes))


def _codes(rng, shape, lo=0x20, hi=0x60):
    """Random normal-range e4m3 codes with random signs."""
    mag = rng.integers(lo, hi, size=shape).astype(np.uint8)
    return mag | (rng.integers(0, 2, size=shape).astype(np.uint8) << 7)


def _e4m3_rne_satfinite(v: np.ndarray) -> np.ndarray:
    """Values of e4m3 codes of fp32 values: saturate to +-448, then torch's round-to-nearest-even cast."""
    c = np.clip(np.asarray(v, np.float32), -E4M3_MAX, E4M3_MAX)
    return torch.from_numpy(c).to(torch.float8_e4m3fn).double().numpy()


def _exact_input_layer(s_a1: float, seed: int, T=7, H=32, I=24, E=4, k=2, s13=None, s2=None):
    """A layer whose input is e4m3 codes times s_a1 (exact in bf16), with one element at 448 * s_a1."""
    rng = np.random.default_rng(seed)
    xc = _codes(rng, (T, H), 0x08, 0x78)
    xc[0, 3] = 0x7E  # 448: the input amax is 448 * s_a1, so the dynamic input scale is s_a1 exactly
    x = (_e4(xc) * s_a1).astype(np.float32)
    X = torch.from_numpy(x).to(torch.bfloat16)
    assert torch.equal(X.float(), torch.from_numpy(x)), "inputs must be exact in bf16"
    Wr = torch.from_numpy(rng.standard_normal((E, H)).astype(np.float32) * (0.05 / max(s_a1, 1.0))).to(torch.bfloat16)
    w13c, w2c = _codes(rng, (E, 2 * I, H)), _codes(rng, (E, H, I))
    s13 = np.array([2.0 ** -9, 3 * 2.0 ** -11, 2.0 ** -10, 5 * 2.0 ** -12][:E] if s13 is None else s13, np.float32)
    s2 = np.array([2.0 ** -7, 2.0 ** -9, 3 * 2.0 ** -10, 2.0 ** -8][:E] if s2 is None else s2, np.float32)
    return dict(X=X, Wr=Wr, w13c=w13c, w2c=w2c, s13=s13, s2=s2, T=T, H=H, I=I, E=E, k=k)


def _dequantised(L):
    w13 = _e4(L["w13c"]) * L["s13"][:, None, None].astype(np.float64)
    w2 = _e4(L["w2c"]) * L["s2"][:, None, None].astype(np.float64)
    return w13, w2


def _check_against_f64(L, renorm=False):
    """FP8 oracle layer vs the fp64 oracle layer on dequantised weights, within the intermediate's
    e4m3 rounding bound computed element by element from an fp64 intermediate formed in torch."""
    k, I = L["k"], L["I"]
    r8 = oracle.moe_forward(L["X"], L["Wr"], L["w13c"], L["w2c"], k, renorm, w13_scale=L["s13"], w2_scale=L["s2"])
    w13, w2 = _dequantised(L)
    # dequantised weights are e4m3 values times the scale: exact in fp32
    assert np.array_equal(w13.astype(np.float32).astype(np.float64), w13)
    r64 = oracle.moe_forward(L["X"].float(), L["Wr"].float(), torch.from_numpy(w13.astype(np.float32)),
                             torch.from_numpy(w2.astype(np.float32)), k, renorm)
    assert np.array_equal(r8["ids"], r64["ids"])
    x = L["X"].double()
    W13, W2 = torch.from_numpy(w13), torch.from_numpy(w2)
    a = torch.empty(L["T"], k, I, dtype=torch.float64)
    for t in range(L["T"]):
        for j in range(k):
            e = int(r64["ids"][t, j])
            g = W13[e, :I] @ x[t]
            u = W13[e, I:] @ x[t]
            a[t, j] = torch.nn.functional.silu(g) * u
    s_a2 = float(r8["act_scales"][1])
    # the intermediate scale is the amax of every routed pair over 448, in fp32
    assert s_a2 == pytest.approx(float(np.float32(np.float32(a.abs().max().item()) / np.float32(448.0))), rel=1e-6)
    # per element of the intermediate: half an e4m3 step, relative 2^-4 among normals and
    # 2^-10 * s_a2 among subnormals (plus the fp32 rounding of a and of a / s_a2)
    da = a.abs() * (2.0 ** -4) * (1 + 2.0 ** -20) + s_a2 * 2.0 ** -10
    bound = np.zeros((L["T"], L["H"]))
    for t in range(L["T"]):
        for j in range(k):
            e = int(r64["ids"][t, j])
            bound[t] += r64["w"][t, j] * (W2[e].abs() @ da[t, j]).numpy()
    err = np.abs(r8["out"] - r64["out"])
    assert np.all(err <= bound * (1 + 1e-9) + 1e-300), float((err / np.maximum(bound, 1e-300)).max())
    return r8, r64, bound


@pytest.mark.parametrize("s_a1", [24.0, 3 * 2.0 ** -6, 1.0])
def test_fp8_input_scale_is_applied(s_a1):
    """With x = e4m3 code * s_a1, quantisation by s_a1 is exact and s_a1 is multiplied back in the
    GEMM1 epilogue: the layer equals the fp64 layer up to the intermediate's rounding.  Inputs up to
    448 * 24 saturate without the scale; 3 * 2^-6 leaves them in e4m3's subnormal range."""
    L = _exact_input_layer(s_a1, seed=21)
    r8, r64, bound = _check_against_f64(L)
    assert float(r8["act_scales"][0]) == s_a1
    rms = np.sqrt(np.mean(r64["out"] ** 2))
    # the bound (a sum of absolute values) stays below the output's RMS, so a scale error of
    # a factor 2 or more anywhere in GEMM1 shows
    assert bound.max() < rms


def test_fp8_w13_scale_alone():
    """Per-expert w13 scales changed alone (by a different factor per expert): the FP8 layer follows
    the fp64 layer on the rescaled weights, and moves by more than the rounding bound."""
    base = _exact_input_layer(2.0, seed=33)
    r_a, _, bound_a = _check_against_f64(base)
    moved = dict(base)
    moved["s13"] = base["s13"] * np.array([2.0, 0.5, 4.0, 0.25], np.float32)
    r_b, _, bound_b = _check_against_f64(moved)
    assert np.array_equal(r_a["ids"], r_b["ids"])
    diff = np.abs(r_b["out"] - r_a["out"])
    assert np.all(diff.max(axis=1) > (bound_a + bound_b).max(axis=1)), "w13 scale change not visible"


def _two_token_layer(seed=12, H=16):
    """E = k = 1, I = 1: every token has one intermediate value, routed with weight 1."""
    rng = np.random.default_rng(seed)
    xc = _codes(rng, (2, H))
    xc[0, 0] = 0x7E  # input amax 448: input scale 1, x exact
    x = _e4(xc).astype(np.float32)
    X = torch.from_numpy(x).to(torch.bfloat16)
    assert torch.equal(X.float(), torch.from_numpy(x))
    w13c = _codes(rng, (1, 2, H), 0x20, 0x58)
    w2c = _codes(rng, (1, H, 1), 0x20, 0x58)
    s13 = np.array([2.0 ** -9], np.float32)
    s2 = np.array([3 * 2.0 ** -8], np.float32)
    Wr = torch.zeros(1, H, dtype=torch.bfloat16)
    return X, Wr, w13c, w2c, s13, s2


def _two_token_expected(X, w13c, w2c, s13, s2):
    """The FP8 definition written out for I = 1: s_a2 = amax over both tokens / 448 (fp32); each
    token's code = e4m3(a / s_a2) (fp32 division, RNE, saturating); y = code * s_a2 * w2."""
    x = X.double().numpy()
    w = _e4(w13c[0]) * np.float64(s13[0])
    g, u = x @ w[0], x @ w[1]
    a = g / (1.0 + np.exp(-g)) * u
    s = np.float32(np.float32(np.abs(a).max()) / np.float32(448.0))
    q = _e4m3_rne_satfinite(a.astype(np.float32) / s)
    w2 = _e4(w2c[0, :, 0]) * np.float64(s2[0])
    return a, float(s), q[:, None] * float(s) * w2[None, :]


def test_fp8_intermediate_scale_is_layer_wide():
    X, Wr, w13c, w2c, s13, s2 = _two_token_layer()
    a, s, expected = _two_token_expected(X, w13c, w2c, s13, s2)
    # the draw discriminates: token 1's code under the layer-wide scale is off its exact value by
    # more than 2 %, while a per-token scale would code it (as that token's amax) nearly exactly
    assert abs(a[0]) > abs(a[1])
    q1 = abs(float(a[1]) / s)
    assert abs(_e4m3_rne_satfinite(np.array([q1]))[0] - q1) > 0.02 * q1
    r = oracle.moe_forward(X, Wr, w13c, w2c, 1, True, w13_scale=s13, w2_scale=s2)
    assert float(r["act_scales"][1]) == s
    np.testing.assert_allclose(r["out"], expected, rtol=1e-12, atol=0)
    per_token = a[1] * (_e4(w2c[0, :, 0]) * np.float64(s2[0]))
    assert np.abs(r["out"][1] - per_token).max() > 0.02 * np.abs(per_token).max()


def test_fp8_intermediate_scale_covers_all_tokens_of_the_call():
    """Asking for a subset of output rows does not change the scales: s_a2 is still the amax over
    every token of the call (here set by token 0, which is not requested)."""
    X, Wr, w13c, w2c, s13, s2 = _two_token_layer()
    _, s, expected = _two_token_expected(X, w13c, w2c, s13, s2)
    sub = oracle.moe_forward(X, Wr, w13c, w2c, 1, True, w13_scale=s13, w2_scale=s2, tokens=[1])
    assert float(sub["act_scales"][1]) == s
    assert float(sub["act_scales"][0]) == 1.0
    np.testing.assert_allclose(sub["out"][0], expected[1], rtol=1e-12, atol=0)
