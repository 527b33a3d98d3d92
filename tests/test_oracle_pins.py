"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks one step of the layer against a brute-force alternative, a
closed form, a special case that reduces to a library routine, or an
invariant the method must satisfy, so that a dropped term, wrong sign, wrong
index or transposed operand in the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from moe_synth import make_layer, spec

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

def test_bf16_encode_matches_torch_rne():
    g = torch.Generator().manual_seed(1)
    x = torch.cat([
        torch.randn(20000, generator=g) * torch.logspace(-30, 30, 20000),
        torch.tensor([0.0, -0.0, 1.0, -1.0, 65504.0, 3.4e38, -3.4e38, 1e-40, 1.00390625, 1.01171875]),
    ])
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f32_to_bf16(x.numpy())
    assert np.array_equal(got, ref)


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = oracle.bf16_to_f64(bits)
    fin = np.isfinite(t)
    assert np.array_equal(got[fin], t[fin])
    assert np.all(np.isnan(got[np.isnan(t)]))


def test_e4m3_decode_spec_values():
    # Values stated by the OCP 8-bit floating point specification for E4M3.
    table = {0x00: 0.0, 0x38: 1.0, 0xC0: -2.0, 0x7E: 448.0, 0xFE: -448.0, 0x08: 2.0 ** -6,
             0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x30: 0.5, 0x3C: 1.5}
    for code, v in table.items():
        assert oracle.e4m3_to_f64([code])[0] == v, hex(code)
    assert np.isnan(oracle.e4m3_to_f64([0x7F])[0]) and np.isnan(oracle.e4m3_to_f64([0xFF])[0])
    assert math.copysign(1.0, oracle.e4m3_to_f64([0x80])[0]) == -1.0


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_to_f64(codes)
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.all(np.isnan(got[~fin]))


def test_e4m3_encode_matches_torch_in_range():
    g = torch.Generator().manual_seed(2)
    x = torch.cat([torch.randn(30000, generator=g) * torch.logspace(-4, 2.6, 30000),
                   torch.linspace(-448, 448, 20001)]).clamp(-448, 448)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.f32_to_e4m3(x.numpy())
    assert np.array_equal(got, ref)


def test_e4m3_encode_ties_even_and_saturates():
    vals = oracle.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    codes = oracle.f32_to_e4m3(mids)
    lo = np.arange(0, 0x7E)
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(codes.astype(np.int64), expect)
    sat = oracle.f32_to_e4m3(np.array([449.0, 464.0, 1e9, np.inf, -500.0, -np.inf], dtype=np.float32))
    assert list(sat) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    rt = oracle.f32_to_e4m3(vals.astype(np.float32))
    assert np.array_equal(rt.astype(np.int64), np.arange(0, 0x7F))


def test_silu_matches_torch():
    z = np.concatenate([np.linspace(-40, 40, 4001), [0.0, 1e-8, -700.0, 700.0]])
    ref = torch.nn.functional.silu(torch.from_numpy(z)).numpy()
    got = np.array([oracle.silu(v) for v in z])
    np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-300)


# --------------------------------------------------------------------------
# Router (step 1) and top-k (step 2)
# --------------------------------------------------------------------------

def test_router_logits_match_numpy_matmul():
    sp = spec("tiny_f32", T=13, H=40, E=7)
    L = make_layer(sp, weights=False)
    got = oracle.router_logits(L["X"], L["Wr"])
    ref = L["X"].double().numpy() @ L["Wr"].double().numpy().T
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)
    Lb = make_layer(spec("mixtral_decode", T=5, H=64, E=8), weights=False)
    got = oracle.router_logits(Lb["X"], Lb["Wr"])
    ref = Lb["X"].double().numpy() @ Lb["Wr"].double().numpy().T
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def _brute_topk(logits, k, renorm):
    p = scipy.special.softmax(logits, axis=1)
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k))
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-p[t, e], e))[:k]
        ids[t] = order
        w[t] = p[t, order]
        if renorm:
            w[t] /= w[t].sum()
    return ids, w


@pytest.mark.parametrize("E,k", [(2, 1), (8, 2), (16, 8), (5, 5), (13, 3)])
@pytest.mark.parametrize("renorm", [False, True])
def test_topk_matches_full_sort(E, k, renorm):
    rng = np.random.default_rng(E * 100 + k)
    lg = rng.standard_normal((64, E))
    # force exact ties on some rows: lower index must win
    lg[::5, : E // 2] = lg[::5, [0]]
    lg[1::7, -1] = lg[1::7, 0]
    ids, w = oracle.topk(lg, k, renorm)
    bids, bw = _brute_topk(lg, k, renorm)
    assert np.array_equal(ids, bids)
    np.testing.assert_allclose(w, bw, rtol=1e-13, atol=0)


def test_topk_weight_closed_forms():
    # E=2, k=1: the winner's weight is the logistic function of the logit gap.
    lg = np.array([[0.3, -1.2], [2.0, 2.5], [0.0, 0.0]])
    ids, w = oracle.topk(lg, 1, False)
    assert list(ids[:, 0]) == [0, 1, 0]
    gaps = np.array([1.5, 0.5, 0.0])
    np.testing.assert_allclose(w[:, 0], 1 / (1 + np.exp(-gaps)), rtol=1e-15)
    # equal logits: every expert weighs 1/E; renormalised k of them weigh 1/k
    flat = np.full((3, 6), 0.7)
    ids, w = oracle.topk(flat, 4, False)
    assert np.array_equal(ids, np.tile(np.arange(4), (3, 1)))
    np.testing.assert_allclose(w, 1 / 6, rtol=1e-15)
    ids, w = oracle.topk(flat, 4, True)
    np.testing.assert_allclose(w, 1 / 4, rtol=1e-15)


def test_topk_weight_invariants():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((200, 32)) * 3
    _, w = oracle.topk(lg, 8, True)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=8 * 2.0 ** -52)
    ids, w = oracle.topk(lg, 8, False)
    assert np.all(w.sum(1) <= 1.0 + 1e-15)
    assert np.all(np.diff(w, axis=1) <= 0)  # descending weights
    # ratio of two weights is exp of the logit difference
    r = w[:, 0] / w[:, 1]
    d = lg[np.arange(200), ids[:, 0]] - lg[np.arange(200), ids[:, 1]]
    np.testing.assert_allclose(r, np.exp(d), rtol=1e-12)
    _, wall = oracle.topk(lg, 32, False)
    np.testing.assert_allclose(wall.sum(1), 1.0, rtol=1e-14)


# --------------------------------------------------------------------------
# Permutation (step 3)
# --------------------------------------------------------------------------

def _brute_align(ids, E, B):
    T, k = ids.shape
    flat = ids.ravel()
    order = sorted(range(T * k), key=lambda f: (flat[f], f))
    sorted_ids, expert_ids = [], []
    for e in range(E):
        mine = [f for f in order if flat[f] == e]
        if not mine:
            continue
        pad = -len(mine) % B
        sorted_ids += mine + [T * k] * pad
        expert_ids += [e] * ((len(mine) + pad) // B)
    return np.array(sorted_ids, np.int32), np.array(expert_ids, np.int32)


@pytest.mark.parametrize("T,k,E,B", [(1, 1, 1, 1), (1, 2, 8, 16), (37, 2, 8, 16), (64, 8, 128, 16),
                                     (100, 3, 5, 4), (257, 8, 64, 128), (0, 2, 4, 8)])
def test_align_matches_brute_force_and_invariants(T, k, E, B):
    rng = np.random.default_rng(T * 31 + E)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if T else np.zeros((0, k), np.int32)
    s, ex, npp, counts = oracle.align(ids, E, B)
    bs, bex = _brute_align(ids, E, B)
    assert np.array_equal(s, bs) and np.array_equal(ex, bex)
    n = T * k
    # bijection over the flat pair indices, the rest is the sentinel
    real = s[s < n]
    assert np.array_equal(np.sort(real), np.arange(n))
    assert np.all(s[s >= n] == n)
    # each block belongs to one expert, and every real entry in it routes there
    assert npp % B == 0 and len(ex) == npp // B
    for b in range(npp // B):
        blk = s[b * B:(b + 1) * B]
        assert np.all(ids.ravel()[blk[blk < n]] == ex[b])
    assert np.array_equal(counts, np.bincount(ids.ravel(), minlength=E))
    assert npp == sum(-(-c // B) * B for c in counts)
    # within an expert, ascending flat index (stable)
    for e in range(E):
        seg = s[np.repeat(ex, B) == e]
        seg = seg[seg < n]
        assert np.all(np.diff(seg) > 0)


# --------------------------------------------------------------------------
# Whole-layer forward
# --------------------------------------------------------------------------

def _dense_ffn(x, w13, w2):
    """Dense SiLU FFN (gate rows first) with torch float64 matmuls."""
    x = torch.as_tensor(x, dtype=torch.float64)
    w13 = torch.as_tensor(w13, dtype=torch.float64)
    w2 = torch.as_tensor(w2, dtype=torch.float64)
    I = w13.shape[0] // 2
    g = x @ w13[:I].T
    u = x @ w13[I:].T
    return (torch.nn.functional.silu(g) * u) @ w2.T


def _small(T=9, H=48, I=40, E=6, k=2, renorm=True, dt="f32"):
    sp = spec("tiny_f32", T=T, H=H, I=I, E=E, k=k, renorm=renorm, act=dt, w=dt, x_std=1.0, w_std=0.2,
              wr_std=0.5)
    return make_layer(sp)


def test_forward_identical_experts_is_dense_ffn():
    L = _small(E=5, k=3, renorm=True)
    L["W13"][:] = L["W13"][2]
    L["W2"][:] = L["W2"][2]
    r = oracle.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], 3, True)
    ref = _dense_ffn(L["X"], L["W13"][0], L["W2"][0]).numpy()
    np.testing.assert_allclose(r["out"], ref, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("renorm", [False, True])
def test_forward_single_expert_is_dense_ffn(renorm):
    L = _small(E=1, k=1, renorm=renorm)
    r = oracle.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], 1, renorm)
    ref = _dense_ffn(L["X"], L["W13"][0], L["W2"][0]).numpy()
    np.testing.assert_allclose(r["out"], ref, rtol=1e-11, atol=1e-12)


def test_forward_all_experts_is_softmax_mixture():
    L = _small(E=4, k=4, renorm=True)
    r = oracle.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], 4, True)
    p = torch.softmax(L["X"].double() @ L["Wr"].double().T, dim=1)
    ref = sum(p[:, e:e + 1] * _dense_ffn(L["X"], L["W13"][e], L["W2"][e]) for e in range(4)).numpy()
    np.testing.assert_allclose(r["out"], ref, rtol=1e-10, atol=1e-12)


def test_forward_topk_mixture_uses_routing_weights():
    L = _small(E=6, k=2, renorm=False)
    r = oracle.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], 2, False)
    p = torch.softmax(L["X"].double() @ L["Wr"].double().T, dim=1).numpy()
    for t in range(L["X"].shape[0]):
        top = sorted(range(6), key=lambda e: (-p[t, e], e))[:2]
        ref = sum(p[t, e] * _dense_ffn(L["X"][t:t + 1], L["W13"][e], L["W2"][e]).numpy()[0] for e in top)
        np.testing.assert_allclose(r["out"][t], ref, rtol=1e-10, atol=1e-12)


def test_forward_expert_relabelling_invariance():
    L = _small(E=7, k=3, renorm=True)
    r0 = oracle.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], 3, True)
    perm = torch.tensor([3, 6, 0, 5, 1, 4, 2])
    r1 = oracle.moe_forward(L["X"], L["Wr"][perm], L["W13"][perm], L["W2"][perm], 3, True)
    np.testing.assert_allclose(r1["out"], r0["out"], rtol=1e-12, atol=1e-14)
    assert np.array_equal(perm.numpy()[r1["ids"]], r0["ids"])


def test_forward_token_subset_and_bf16_inputs():
    L = _small(T=11, E=5, k=2, dt="bf16")
    full = oracle.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], 2, True)
    sub = oracle.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], 2, True, tokens=[7, 0, 3])
    np.testing.assert_array_equal(sub["out"], full["out"][[7, 0, 3]])
    # bf16 storage is read exactly: the same values held in fp32 give the same layer
    f32 = oracle.moe_forward(L["X"].float(), L["Wr"].float(), L["W13"].float(), L["W2"].float(), 2, True)
    np.testing.assert_array_equal(f32["out"], full["out"])


def test_forward_gate_and_up_halves_are_distinct():
    L = _small(E=3, k=1, renorm=True)
    I = L["W13"].shape[1] // 2
    a = oracle.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], 1, True)
    swapped = torch.cat([L["W13"][:, I:], L["W13"][:, :I]], dim=1).contiguous()
    b = oracle.moe_forward(L["X"], L["Wr"], swapped, L["W2"], 1, True)
    assert np.abs(a["out"] - b["out"]).max() > 1e-3 * np.abs(a["out"]).max()


def test_forward_fp8_exact_inputs_against_dequantised_f64():
    """FP8 mode on inputs the e4m3 grid holds exactly (input amax 448 -> input scale 1).

    The FP8 output then differs from the fp64 layer on dequantised weights only by
    the e4m3 rounding of the intermediate (relative half-ulp 2^-4 per element).
    """
    rng = np.random.default_rng(5)
    T, H, I, E, k = 6, 32, 24, 4, 2
    codes = lambda shape: rng.integers(0x08, 0x60, size=shape).astype(np.uint8) | (
        rng.integers(0, 2, size=shape).astype(np.uint8) << 7)
    xc = codes((T, H))
    xc[0, 0] = 0x7E  # 448 -> dynamic input scale is exactly 1
    x = oracle.e4m3_to_f64(xc.ravel()).reshape(T, H).astype(np.float32)
    X = torch.from_numpy(x).to(torch.bfloat16)
    assert torch.equal(X.float(), torch.from_numpy(x))
    Wr = torch.from_numpy(rng.standard_normal((E, H)).astype(np.float32) * 0.01).to(torch.bfloat16)
    w13c, w2c = codes((E, 2 * I, H)), codes((E, H, I))
    s13 = np.array([2.0 ** -9, 2.0 ** -8, 2.0 ** -10, 2.0 ** -9], np.float32)
    s2 = np.array([2.0 ** -7, 2.0 ** -9, 2.0 ** -8, 2.0 ** -8], np.float32)
    r8 = oracle.moe_forward(X, Wr, w13c, w2c, k, False, w13_scale=s13, w2_scale=s2)
    assert r8["act_scales"][0] == 1.0
    w13 = (oracle.e4m3_to_f64(w13c.ravel()).reshape(E, 2 * I, H) * s13[:, None, None]).astype(np.float32)
    w2 = (oracle.e4m3_to_f64(w2c.ravel()).reshape(E, H, I) * s2[:, None, None]).astype(np.float32)
    r64 = oracle.moe_forward(X.float(), Wr.float(), w13, w2, k, False)
    assert np.array_equal(r8["ids"], r64["ids"])
    err = np.abs(r8["out"] - r64["out"]).max() / np.sqrt(np.mean(r64["out"] ** 2))
    assert 0 < err < 0.1
    # the intermediate scale is its amax over 448: 448 * s_a2 reproduces an amax of the fp64 intermediate
    assert r8["act_scales"][1] > 0


def test_forward_fp8_scale_is_applied():
    """Doubling every weight scale doubles gate/up pre-activations and the down projection."""
    rng = np.random.default_rng(6)
    T, H, I, E, k = 5, 32, 16, 3, 2
    X = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    Wr = torch.from_numpy(rng.standard_normal((E, H)).astype(np.float32) * 0.2).to(torch.bfloat16)
    w13c = rng.integers(0, 0x7E, size=(E, 2 * I, H)).astype(np.uint8)
    w2c = rng.integers(0, 0x7E, size=(E, H, I)).astype(np.uint8)
    s = np.full(E, 2.0 ** -8, np.float32)
    a = oracle.moe_forward(X, Wr, w13c, w2c, k, True, w13_scale=s, w2_scale=s)
    b = oracle.moe_forward(X, Wr, w13c, w2c, k, True, w13_scale=s, w2_scale=2 * s)
    np.testing.assert_allclose(b["out"], 2 * a["out"], rtol=1e-14, atol=1e-300)
