"""GPU parity of the router (steps 1-2) and the permutation (step 3) against the CPU oracle.

Routing ids, the sorted pair list, the block-to-expert map, the padded length
and the per-expert counts must match bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import make_tie_free
from moe_synth import make_layer, spec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_layer_scan_gb300 as m

    assert torch.cuda.is_available()
    return m


def _logits_with_ties(T, E, seed):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[::3, : max(1, E // 3)] = lg[::3, :1]  # exact ties: lower index must rank first
    lg[1::5, -1] = lg[1::5, 0]
    return lg


@pytest.mark.parametrize("T,E,k,renorm", [(1, 8, 2, True), (37, 8, 2, True), (64, 128, 8, True), (300, 64, 8, False),
                                          (5, 1024, 32, True), (16, 3, 3, False), (129, 33, 1, False)])
def test_topk_from_logits_bit_exact(moe, T, E, k, renorm):
    lg = _logits_with_ties(T, E, T * 7 + E)
    w, ids = moe.moe_topk_from_logits(torch.from_numpy(lg).cuda(), k, renorm)
    rid, rw = oracle.topk(lg.astype(np.float64), k, renorm)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=1e-5, atol=1e-7)


def test_topk_special_values(moe):
    """Ranking by value, lower expert index on equal values: -0 and +0 are equal, -inf
    logits rank (last), NaN logits never rank; when fewer than k experts rank, the
    remaining picks are expert 0 with weight 0 (renormalised weights)."""
    E, k = 64, 8
    lg = np.random.default_rng(5).standard_normal((3, E)).astype(np.float32)
    lg[0] = -(np.abs(lg[0]) + 1.0)          # every other value below -1
    lg[0, [3, 9, 40]] = 9.0                 # equal top values
    lg[0, 17], lg[0, 5] = 8.0, 8.0
    lg[0, 20], lg[0, 12] = np.float32(-0.0), np.float32(0.0)  # -0 and +0 tie: picks 6 and 7
    lg[1, :] = -np.inf
    lg[1, [7, 33]] = [1.0, 2.0]
    lg[2, :] = np.nan
    lg[2, [4, 44, 60, 2, 31]] = [0.5, 0.25, 0.5, -1.0, 3.0]
    w, ids = moe.moe_topk_from_logits(torch.from_numpy(lg).cuda(), k, True)
    ids, w = ids.cpu().numpy(), w.cpu().numpy()
    for t in range(3):
        v = lg[t].astype(np.float64)
        ranked = sorted([e for e in range(E) if not np.isnan(v[e])], key=lambda e: (-v[e], e))[:k]
        want = ranked + [0] * (k - len(ranked))
        assert list(ids[t]) == want, (t, list(ids[t]), want)
        vals = np.array([v[e] for e in ranked] + [-np.inf] * (k - len(ranked)))
        ex = np.exp(vals - vals[0])
        np.testing.assert_allclose(w[t], ex / ex.sum(), rtol=1e-5, atol=1e-7)
    # -0 and +0 tie: the lower index (12) comes first
    assert list(ids[0]).index(12) < list(ids[0]).index(20)


@pytest.mark.parametrize("name,T", [("tiny_f32", 64), ("mixtral_decode", 64), ("fine_decode", 64),
                                    ("fp8_decode", 64), ("prefill", 8192), ("prefill_hot", 8192)])
def test_route_matches_oracle(moe, name, T):
    sp = spec(name, T=T)
    L = make_layer(sp, weights=False)
    make_tie_free(L)
    logits, w, ids = moe.moe_route(L["X"].cuda(), L["Wr"].cuda(), sp.k, sp.renorm)
    ref_lg = oracle.router_logits(L["X"], L["Wr"])
    rid, rw = oracle.topk(ref_lg, sp.k, sp.renorm)
    assert np.array_equal(ids.cpu().numpy(), rid)
    # fp32 summation of H products: |err| <= H * 2^-24 * sum_h |x_h w_h| (plus the product roundings)
    bound = (sp.H + 2) * 2.0 ** -24 * (np.abs(L["X"].double().numpy()) @ np.abs(L["Wr"].double().numpy()).T)
    assert np.all(np.abs(logits.cpu().numpy() - ref_lg) <= bound)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=1e-4, atol=1e-6)


@pytest.mark.parametrize("T,H,E,k", [(256, 256, 40, 6), (300, 384, 256, 8), (1000, 128, 8, 2), (255, 256, 64, 8),
                                     (257, 512, 16, 4), (512, 256, 64, 8), (2000, 256, 96, 8), (4864, 256, 64, 8),
                                     (40, 256, 33, 4), (77, 384, 9, 2), (200, 256, 130, 8), (32, 256, 5, 2),
                                     (31, 256, 7, 2)])
def test_route_tensor_core_and_cuda_core_paths(moe, T, H, E, k):
    """T >= 256 bf16 batches take the tcgen05 logits GEMM (E in the N slot, masked to E; split into 2 or 4
    column tiles when the 128-token tiles would leave SMs idle: 512 x 64, 4864 x 64 and 300 x 256 take 4,
    2000 x 96 and the 8192-token prefill layers take 2); shorter ones the CUDA cores, from 32 tokens with
    four experts per CTA (expert counts that are not a multiple of 4 included), below with one."""
    sp = spec("prefill", T=T, H=H, E=E, k=k)
    L = make_layer(sp, weights=False)
    make_tie_free(L)
    logits, w, ids = moe.moe_route(L["X"].cuda(), L["Wr"].cuda(), k, True)
    ref_lg = oracle.router_logits(L["X"], L["Wr"])
    rid, rw = oracle.topk(ref_lg, k, True)
    assert np.array_equal(ids.cpu().numpy(), rid)
    bound = (H + 2) * 2.0 ** -24 * (np.abs(L["X"].double().numpy()) @ np.abs(L["Wr"].double().numpy()).T)
    assert np.all(np.abs(logits.cpu().numpy() - ref_lg) <= bound)


def _random_ids(T, k, E, seed, skew=False):
    rng = np.random.default_rng(seed)
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        p /= p.sum()
        return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


# (up to 32 pairs go to a single-warp kernel, up to 1024 to a one-pair-per-thread kernel,
# more to the block-wide kernel: the list covers all three and their boundaries)
@pytest.mark.parametrize("T,k,E,B", [(1, 1, 1, 1), (1, 2, 8, 16), (1, 8, 128, 16), (4, 8, 128, 16), (3, 8, 1024, 16),
                                     (16, 2, 8, 16), (2, 3, 7, 1), (5, 6, 40, 128), (4, 8, 64, 1000), (3, 10, 33, 16),
                                     (37, 2, 8, 16), (64, 8, 128, 16), (100, 3, 5, 4), (128, 8, 128, 16),
                                     (33, 1, 1024, 16), (40, 8, 1024, 1), (17, 3, 7, 1000), (129, 8, 64, 16),
                                     (257, 8, 64, 128), (1000, 6, 1024, 16), (8192, 8, 64, 128), (333, 7, 9, 1024)])
def test_align_bit_exact(moe, T, k, E, B):
    ids = _random_ids(T, k, E, T + 31 * E, skew=(T % 2 == 0))
    s, ex, npp, counts = moe.moe_align(torch.from_numpy(ids).cuda(), E, B)
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    rs, rex, rnpp, rcounts = oracle.align(ids, E, B)
    n = int(npp.item())
    assert n == rnpp
    assert np.array_equal(s.cpu().numpy()[:n], rs)
    assert np.array_equal(ex.cpu().numpy()[: n // B], rex)
    assert np.array_equal(counts.cpu().numpy(), rcounts)


@pytest.mark.parametrize("T,k", [(3, 8), (64, 8), (512, 8)])
def test_align_drops_and_flags_bad_ids(moe, T, k):
    ids = _random_ids(T, k, 64, 11)
    bad = ids.copy()
    bad[1, 2] = 64
    bad[2, 0] = -2
    s, ex, npp, counts = moe.moe_align(torch.from_numpy(bad).cuda(), 64, 16)
    assert moe.moe_get_status() == moe.MOE_ERR_DEVICE_INDEX
    assert moe.moe_get_status() == 0
    keep = (bad >= 0) & (bad < 64)
    rcounts = np.bincount(bad[keep], minlength=64)
    assert np.array_equal(counts.cpu().numpy(), rcounts)
    n = int(npp.item())
    rows = s.cpu().numpy()[:n]
    flat = np.flatnonzero(keep.reshape(-1))
    assert np.array_equal(np.sort(rows[rows < T * k]), flat)  # every kept pair once, no dropped one


def test_align_is_deterministic_and_flags_bad_ids(moe):
    ids = _random_ids(512, 8, 64, 5)
    a = moe.moe_align(torch.from_numpy(ids).cuda(), 64, 16)
    b = moe.moe_align(torch.from_numpy(ids).cuda(), 64, 16)
    n = int(a[2].item())
    assert torch.equal(a[0][:n], b[0][:n]) and torch.equal(a[1][: n // 16], b[1][: n // 16])
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    bad = ids.copy()
    bad[3, 1] = 64
    bad[7, 0] = -2
    moe.moe_align(torch.from_numpy(bad).cuda(), 64, 16)
    assert moe.moe_get_status() == moe.MOE_ERR_DEVICE_INDEX
    assert moe.moe_get_status() == 0  # cleared by the read
