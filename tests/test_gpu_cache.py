"""GPU checks of the layer on a given routing and of the expert cache.

moe_forward_routed on moe_route's routing reproduces moe_forward bit for bit.  The
cached layer (host-resident experts, a smaller pool of device slots, misses copied in,
least recently used evicted) reproduces the resident layer bit for bit over a sequence
of batches whose experts do not all fit (both runs with one K split, so their plans
coincide), in bf16 and FP8; its counters agree with the distinct experts per call.
"""
import numpy as np
import pytest
import torch

from moe_synth import make_layer, resample_tokens, spec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_layer_scan_gb300 as m

    assert torch.cuda.is_available()
    return m


def test_forward_routed_matches_forward(moe):
    sp = spec("fine_decode", T=12, H=512, I=256, E=32, k=8)
    L = make_layer(sp, device="cuda")
    ref = moe.moe_forward(L["X"], L["Wr"], L["W13"], L["W2"], sp.k, sp.renorm)
    _, w, ids = moe.moe_route(L["X"], L["Wr"], sp.k, sp.renorm)
    got = moe.moe_forward_routed(L["X"], w, ids, L["W13"], L["W2"])
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    assert torch.equal(got, ref)


@pytest.mark.parametrize("name,slots", [("fine_decode", 12), ("fp8_decode", 13)])  # >= T*k distinct
def test_cached_layer_matches_resident(moe, name, slots):
    sp = spec(name, T=3, H=256, I=256, E=32, k=4)
    L = make_layer(sp, device="cpu")
    w13h = L["W13"].pin_memory()
    w2h = L["W2"].pin_memory()
    cache = moe.ExpertCache(w13h, w2h, n_slots=slots, max_tokens=8, topk=sp.k, w13_scale=L["w13_scale"],
                            w2_scale=L["w2_scale"])
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
    cache.close()


def test_cache_refuses_more_experts_than_slots(moe):
    sp = spec("prefill", T=4, H=256, I=256, E=32, k=8)
    L = make_layer(sp, device="cpu")
    with pytest.raises(moe.MoeError) as e:
        moe.ExpertCache(L["W13"], L["W2"], n_slots=6, max_tokens=4, topk=sp.k)  # fewer slots than top-k
    assert e.value.code == moe.MOE_ERR_ARG
    cache = moe.ExpertCache(L["W13"], L["W2"], n_slots=12, max_tokens=4, topk=sp.k)  # pageable: registered
    _, _, ids = moe.moe_route(L["X"].cuda(), L["Wr"].cuda(), sp.k, sp.renorm)
    assert torch.unique(ids).numel() > 12
    with pytest.raises(moe.MoeError) as e:
        cache.forward(L["X"].cuda(), L["Wr"].cuda(), sp.renorm)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED
    cache.close()
