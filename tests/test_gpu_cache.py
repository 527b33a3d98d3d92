"""GPU checks of the layer on a given routing and of the expert cache.

moe_forward_routed on moe_route's routing reproduces moe_forward bit for bit.  The
cached layer (host-resident experts, a smaller pool of device slots, misses copied in,
least recently used evicted) is checked

* against the CPU oracle over sequences of batches whose experts do not all fit, in
  bf16 and FP8, including calls with more distinct experts than slots (run in passes)
  and the full-size fine-grained decode batch of 64 tokens through 48 slots;
* bit for bit against the resident layer when both plans coincide (one K split), in
  every copy mode: copies overlapped with the expert kernels (per-slot readiness
  words), copies before the kernels, and a copy kernel reading host memory;
* for its counters (hits + misses = distinct experts per pass, bytes copied).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_parity, make_tie_free
from moe_synth import make_layer, resample_tokens, spec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_layer_scan_gb300 as m

    assert torch.cuda.is_available()
    return m


def _cache(moe, L, slots, max_tokens, mode=0):
    sp = L["spec"]
    c = moe.ExpertCache(L["W13"].pin_memory(), L["W2"].pin_memory(), n_slots=slots, max_tokens=max_tokens, topk=sp.k,
                        w13_scale=L["w13_scale"], w2_scale=L["w2_scale"])
    c.set_copy_mode(mode)
    return c


def _oracle(L):
    sp = L["spec"]
    return oracle.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm, L["w13_scale"], L["w2_scale"])


def test_forward_routed_matches_forward(moe):
    sp = spec("fine_decode", T=12, H=512, I=256, E=32, k=8)
    L = make_layer(sp, device="cuda")
    ref = moe.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm)
    _, w, ids = moe.moe_route(L["X"], L["Wr"], sp.k, sp.renorm)
    got = moe.moe_forward_routed(L["X"], w, ids, L["W13"], L["W2"])
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    assert torch.equal(got, ref)


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("name,slots,T", [("fine_decode", 12, 3), ("fp8_decode", 13, 3), ("fine_decode", 12, 8)])
def test_cached_layer_matches_resident(moe, mode, name, slots, T):
    """Both runs with one K split, so their plans coincide; T = 8 with top-4 of 32 experts needs
    more than 12 experts in most calls (passes)."""
    sp = spec(name, T=T, H=256, I=256, E=32, k=4)
    L = make_layer(sp, device="cpu")
    cache = _cache(moe, L, slots, max_tokens=8, mode=mode)
    W13, W2, Wr = L["W13"].cuda(), L["W2"].cuda(), L["Wr"].cuda()
    s13 = None if L["w13_scale"] is None else L["w13_scale"].cuda()
    s2 = None if L["w2_scale"] is None else L["w2_scale"].cuda()
    opts = {"split_k": 1}
    distinct = 0
    for step in range(8):
        resample_tokens(L, torch.arange(sp.T), 100 + step)
        X = L["X"].cuda()
        got = cache.forward(X, Wr, sp.renorm, options=opts)
        ref = moe.moe_forward(X, Wr, W13, W2, sp.k, sp.renorm, s13, s2, options=opts)
        torch.cuda.synchronize()
        assert moe.moe_get_status() == 0
        assert torch.equal(got, ref), f"step {step}"
        _, _, ids = moe.moe_route(X, Wr, sp.k, sp.renorm)
        distinct += int(torch.unique(ids).numel())
    st = cache.stats()
    assert st["calls"] == 8 and st["hits"] + st["misses"] == distinct
    assert st["misses"] >= slots  # the pool was filled, so later misses evicted
    per_expert = (2 * sp.I * sp.H + sp.H * sp.I) * (1 if sp.w == "e4m3" else 2)
    assert st["bytes_h2d"] == st["misses"] * per_expert
    if T == 8:
        assert st["passes"] > st["calls"]
    cache.close()


@pytest.mark.parametrize("name,slots,T,E,k", [("fine_decode", 20, 6, 64, 8), ("fine_decode", 10, 6, 64, 8),
                                              ("fp8_decode", 24, 2, 32, 8), ("mixtral_decode", 3, 5, 8, 2),
                                              ("prefill", 12, 96, 16, 2),  # 96 tokens: token-major GEMMs
                                              ("prefill", 12, 4200, 16, 2)])  # 4200: token-order row gather
def test_cached_layer_matches_oracle(moe, name, slots, T, E, k):
    """A sequence of batches with evictions (and, where slots < distinct experts, passes)
    against the CPU oracle."""
    sp = spec(name, T=T, H=512, I=256, E=E, k=k)
    L = make_layer(sp, device="cpu")
    make_tie_free(L)
    cache = _cache(moe, L, slots, max_tokens=T)
    Wr = L["Wr"].cuda()
    kind = "e4m3" if sp.w == "e4m3" else "bf16"
    for step in range(6):
        if step:
            resample_tokens(L, torch.arange(sp.T), 300 + step)
            make_tie_free(L)
        got = cache.forward(L["X"].cuda(), Wr, sp.renorm)
        torch.cuda.synchronize()
        assert moe.moe_get_status() == 0
        assert_parity(got.float().cpu().numpy(), _oracle(L)["out"], kind, f"cached {name} slots={slots} step {step}")
    st = cache.stats()
    assert st["evictions"] > 0
    cache.close()


@pytest.mark.parametrize("slots", [48, 24])
def test_cached_fine_decode_full_size(moe, slots):
    """The fine-grained decode layer at 64 tokens (about fifty distinct experts per call under
    its Zipf-skewed routing) through a pool of 48 or 24 slots: passes, against the oracle and the
    resident layer."""
    sp = spec("fine_decode", T=64)
    L = make_layer(sp, device="cpu")
    make_tie_free(L)
    cache = _cache(moe, L, slots, max_tokens=64)
    X, Wr = L["X"].cuda(), L["Wr"].cuda()
    got = cache.forward(X, Wr, sp.renorm)
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    st = cache.stats()
    r = _oracle(L)
    distinct = len(np.unique(r["ids"]))
    assert st["passes"] == -(-distinct // slots) and st["misses"] == distinct
    ref = r["out"]
    assert_parity(got.float().cpu().numpy(), ref, "bf16", "cached fine_decode M=64, 48 slots")
    resident = moe.moe_forward(X, Wr, L["W13"].cuda(), L["W2"].cuda(), sp.k, sp.renorm)
    torch.cuda.synchronize()
    assert_parity(got.float().cpu().numpy(), resident.float().cpu().numpy(), "bf16", "cached vs resident")
    cache.close()


def test_cache_refusals(moe):
    sp = spec("prefill", T=4, H=256, I=256, E=32, k=8)
    L = make_layer(sp, device="cpu")
    with pytest.raises(moe.MoeError) as e:
        moe.ExpertCache(L["W13"], L["W2"], n_slots=6, max_tokens=4, topk=sp.k)  # fewer slots than top-k
    assert e.value.code == moe.MOE_ERR_ARG
    # FP8: the intermediate scale spans every pair of the call, so a call must fit in one pass
    sp8 = spec("fp8_decode", T=4, H=256, I=256, E=32, k=8)
    L8 = make_layer(sp8, device="cpu")
    cache = moe.ExpertCache(L8["W13"], L8["W2"], n_slots=12, max_tokens=4, topk=sp8.k, w13_scale=L8["w13_scale"],
                            w2_scale=L8["w2_scale"])  # pageable: registered
    _, _, ids = moe.moe_route(L8["X"].cuda(), L8["Wr"].cuda(), sp8.k, sp8.renorm)
    assert torch.unique(ids).numel() > 12
    with pytest.raises(moe.MoeError) as e:
        cache.forward(L8["X"].cuda(), L8["Wr"].cuda(), sp8.renorm)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoeError) as e:
        cache.set_copy_mode(7)
    assert e.value.code == moe.MOE_ERR_ARG
    cache.close()
