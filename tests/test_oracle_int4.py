"""Pins of the oracle's INT4 weight decoding (the stored format: 8 consecutive K
elements per 32-bit word, element e in nibble (e even ? e/2 : 4 + e/2), two's
complement codes, one bf16 scale per (row, 128 K elements) stored group-major per
expert [E][K/128][rows], weight = q * s rounded once to bf16).  The INT4 layer must equal the bf16 layer of the same oracle on
weights decoded independently here (torch arithmetic from the codes); with E = k = 1
it is the dense SiLU FFN of those weights.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_synth import make_layer, spec


def _pack(q):
    """codes int [rows, K] in [-8, 7] -> uint8 [rows, K/2] in the stored format (written from the definition)."""
    rows, K = q.shape
    out = np.zeros((rows, K // 2), dtype=np.uint8)
    for w in range(K // 8):
        for e in range(8):
            nib = e // 2 if e % 2 == 0 else 4 + e // 2
            code = q[:, 8 * w + e].astype(np.int64) & 0xF
            byte = 4 * w + nib // 2
            out[:, byte] |= (code << (4 * (nib % 2))).astype(np.uint8)
    return out


def _decode_torch(q, s):
    """weights bf16 [rows, K] = bf16(q * s) with s [rows, K/128] bf16."""
    sf = torch.from_numpy(s.view(np.int16)).view(torch.bfloat16).float().repeat_interleave(128, dim=1)
    return (torch.from_numpy(q.astype(np.float32)) * sf).to(torch.bfloat16)


def _rand_int4(rows, K, seed):
    g = np.random.default_rng(seed)
    q = g.integers(-8, 8, size=(rows, K))
    s = torch.from_numpy(g.uniform(1e-3, 4e-3, size=(rows, K // 128)).astype(np.float32)).to(torch.bfloat16)
    return q, s.view(torch.uint16).numpy()


@pytest.mark.parametrize("T,H,I,E,k", [(3, 256, 128, 4, 2), (2, 128, 256, 1, 1)])
def test_int4_layer_equals_bf16_layer_on_decoded_weights(T, H, I, E, k):
    L = make_layer(spec("mixtral_decode", T=T, H=H, I=I, E=E, k=k), weights=False)
    q13 = [_rand_int4(2 * I, H, 10 + e) for e in range(E)]
    q2 = [_rand_int4(H, I, 50 + e) for e in range(E)]
    W13q = np.stack([_pack(q) for q, _ in q13])
    W2q = np.stack([_pack(q) for q, _ in q2])
    S13 = torch.from_numpy(np.stack([s.T for _, s in q13]).copy().view(np.int16)).view(torch.bfloat16)
    S2 = torch.from_numpy(np.stack([s.T for _, s in q2]).copy().view(np.int16)).view(torch.bfloat16)
    W13 = torch.stack([_decode_torch(q, s) for q, s in q13])
    W2 = torch.stack([_decode_torch(q, s) for q, s in q2])
    a = oracle.moe_forward(L["X"], L["Wr"], torch.from_numpy(W13q), torch.from_numpy(W2q), k, True, S13, S2,
                           w_format="int4")["out"]
    b = oracle.moe_forward(L["X"], L["Wr"], W13, W2, k, True)["out"]
    assert np.array_equal(a, b)
    if E == 1:
        x = L["X"].double()
        g = x @ W13[0, :I].double().T
        u = x @ W13[0, I:].double().T
        dense = (g / (1 + torch.exp(-g)) * u) @ W2[0].double().T
        np.testing.assert_allclose(a, dense.numpy(), rtol=1e-10, atol=1e-12)


def test_synthetic_int4_weights_decode_near_the_drawn_weights():
    """The input generator's codes and scales (an offline quantiser stand-in) reproduce its bf16 weights
    within half a code step; the oracle reads them in the same format."""
    from moe_synth import _int4_encode_groupwise

    g = torch.Generator().manual_seed(3)
    w = torch.randn(64, 256, generator=g) * 0.02
    packed, s = _int4_encode_groupwise(w)
    q = np.zeros((64, 256), dtype=np.int64)
    pk = packed.numpy()
    for col in range(256):
        word, e = divmod(col, 8)
        nib = e // 2 if e % 2 == 0 else 4 + e // 2
        byte = pk[:, 4 * word + nib // 2].astype(np.int64)
        v = (byte >> (4 * (nib % 2))) & 0xF
        q[:, col] = np.where(v >= 8, v - 16, v)
    sf = s.float().repeat_interleave(128, dim=1).numpy()
    assert np.all(np.abs(q * sf - w.numpy()) <= 0.5 * sf + 1e-9)
