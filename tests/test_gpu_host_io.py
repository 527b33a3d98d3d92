"""moe_forward_host: the layer from pinned host memory to pinned host memory through the
C ABI (a copy kernel reading the host batch, the layer storing its output into host memory,
one stream) gives bit for bit what moe_forward gives on device buffers, over several
batches that reuse the staging buffer, and refuses pageable host buffers."""
import pytest
import torch

from moe_synth import make_layer, resample_tokens, spec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_layer_scan_gb300 as m

    assert torch.cuda.is_available()
    return m


@pytest.mark.parametrize("name,kw", [("mixtral_decode", dict(T=5, H=512, I=256, E=8, k=2)),
                                     ("fp8_decode", dict(T=16, H=512, I=256, E=16, k=4)),
                                     ("prefill", dict(T=300, H=512, I=256, E=8, k=2)),
                                     ("tiny_f32", dict(T=33, H=64, I=96, E=8, k=2))])
def test_host_io_matches_device_forward(moe, name, kw):
    sp = spec(name, **kw)
    L = make_layer(sp, device="cpu")
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}
    s = torch.cuda.Stream()
    hidden_dev = torch.empty(L["X"].shape, dtype=L["X"].dtype, device="cuda")
    out_host = torch.empty(L["X"].shape, dtype=L["X"].dtype).pin_memory()
    for step in range(3):
        if step:
            resample_tokens(L, torch.arange(sp.T), 50 + step)
        xh = L["X"].pin_memory()
        got = moe.moe_forward_host(xh, d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm, d["w13_scale"], d["w2_scale"],
                                   hidden_dev=hidden_dev, out_host=out_host, stream=s)
        s.synchronize()
        assert moe.moe_get_status() == 0
        ref = moe.moe_forward(xh.cuda(), d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm, d["w13_scale"], d["w2_scale"])
        torch.cuda.synchronize()
        assert torch.equal(got, ref.cpu()), f"step {step}"


def test_host_io_refuses_pageable_buffers(moe):
    sp = spec("mixtral_decode", T=4, H=256, I=256, E=8, k=2)
    L = make_layer(sp, device="cpu")
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward_host(L["X"], d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm)  # pageable input
    assert e.value.code == moe.MOE_ERR_ARG
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward_host(L["X"].pin_memory(), d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm,
                             out_host=torch.empty(L["X"].shape, dtype=L["X"].dtype))  # pageable output
    assert e.value.code == moe.MOE_ERR_ARG


def test_host_io_unaligned_input(moe):
    """A host batch that does not start on a 16-byte boundary goes through the copy engine
    instead of the copy kernel, with the same result."""
    sp = spec("mixtral_decode", T=6, H=256, I=256, E=8, k=2)
    L = make_layer(sp, device="cpu")
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}
    flat = torch.empty(sp.T * sp.H + 1, dtype=L["X"].dtype).pin_memory()
    xh = flat[1:].view(sp.T, sp.H)  # two bytes past a 16-byte boundary
    xh.copy_(L["X"])
    assert xh.data_ptr() % 16 != 0
    s = torch.cuda.Stream()
    got = moe.moe_forward_host(xh, d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm, stream=s)
    s.synchronize()
    ref = moe.moe_forward(L["X"].cuda(), d["Wr"], d["W13"], d["W2"], sp.k, sp.renorm)
    torch.cuda.synchronize()
    assert torch.equal(got, ref.cpu())
