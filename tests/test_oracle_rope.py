"""Pins of the oracle's inverse rotary embedding + per-head e4m3 quantisation against
properties the definition fixes: rotation by a zero angle is the identity, by a right
angle a signed swap of the two halves; the inverse undoes a forward rotation computed
independently in float64; pair norms are preserved; unrotated elements pass through;
the largest element of every vector encodes to +-448; dequantised codes reproduce the
rotated values within e4m3's rounding; a zero vector gets scale 1 and (signed) zero codes.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def _bf16_bits(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.uint16).numpy()


def _bf16_vals(bits):
    return torch.from_numpy(np.asarray(bits, dtype=np.uint16).astype(np.int16)).view(torch.bfloat16).float().numpy()


def _table(angles):
    a = np.asarray(angles, dtype=np.float64)
    return np.concatenate([np.cos(a), np.sin(a)], axis=1).astype(np.float32)


def _x(T, heads, D, seed):
    g = np.random.default_rng(seed)
    return _bf16_bits(g.standard_normal((T, heads, D)))


def test_zero_angle_is_identity_and_max_encodes_to_448():
    T, heads, D, R = 5, 3, 64, 64
    x = _x(T, heads, D, 1)
    cs = np.concatenate([np.ones((4, R // 2)), np.zeros((4, R // 2))], axis=1).astype(np.float32)
    q, sc, y = oracle.inv_rope_fp8_quant(x, np.arange(T, dtype=np.int32) % 4, cs, R, return_rotated=True)
    xv = _bf16_vals(x)
    assert np.array_equal(y, xv)
    for t in range(T):
        for h in range(heads):
            j = int(np.argmax(np.abs(xv[t, h])))
            assert q[t, h, j] == (0x7E if xv[t, h, j] > 0 else 0xFE)


def test_right_angle_is_signed_half_swap():
    T, heads, D, R = 4, 2, 32, 32
    x = _x(T, heads, D, 2)
    half = R // 2
    cs = np.concatenate([np.zeros((1, half)), np.ones((1, half))], axis=1).astype(np.float32)
    pos = np.zeros(T, dtype=np.int32)
    _, _, y = oracle.inv_rope_fp8_quant(x, pos, cs, R, return_rotated=True)
    xv = _bf16_vals(x)
    assert np.array_equal(y[..., :half], xv[..., half:])
    assert np.array_equal(y[..., half:], -xv[..., :half])


def test_inverse_undoes_an_independent_forward_rotation():
    T, heads, D, R = 6, 4, 128, 96
    g = np.random.default_rng(3)
    x0 = g.standard_normal((T, heads, D))
    half = R // 2
    ang = g.uniform(-np.pi, np.pi, size=(T, half))
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    fwd = x0.copy()  # forward rotation by +angle, float64
    fwd[..., :half] = x0[..., :half] * c - x0[..., half:R] * s
    fwd[..., half:R] = x0[..., half:R] * c + x0[..., :half] * s
    _, _, y = oracle.inv_rope_fp8_quant(_bf16_bits(fwd), np.arange(T, dtype=np.int32), _table(ang), R,
                                        return_rotated=True)
    err = np.abs(y - x0).max(axis=-1) / np.abs(x0).max(axis=-1)
    assert err.max() < 2.0 ** -7  # bf16 rounding of the rotated input, fp32 table and arithmetic


def test_pair_norms_preserved_and_tail_passes_through():
    T, heads, D, R = 3, 5, 80, 48
    x = _x(T, heads, D, 4)
    g = np.random.default_rng(5)
    ang = g.uniform(0, 100, size=(3, R // 2))
    _, _, y = oracle.inv_rope_fp8_quant(x, np.array([2, 0, 1], dtype=np.int32), _table(ang), R, return_rotated=True)
    xv = _bf16_vals(x).astype(np.float64)
    h = R // 2
    n_in = xv[..., :h] ** 2 + xv[..., h:R] ** 2
    n_out = y[..., :h].astype(np.float64) ** 2 + y[..., h:R].astype(np.float64) ** 2
    assert np.all(np.abs(n_out - n_in) <= 1e-5 * (n_in + 1e-30) + 1e-12)
    assert np.array_equal(y[..., R:], xv[..., R:].astype(np.float32))


def test_dequantised_codes_within_e4m3_rounding_and_zero_vector():
    T, heads, D, R = 4, 3, 64, 32
    x = _x(T, heads, D, 6)
    x[1, 2, :] = 0  # a zero vector
    g = np.random.default_rng(7)
    ang = g.uniform(0, 10, size=(T, R // 2))
    q, sc, y = oracle.inv_rope_fp8_quant(x, np.arange(T, dtype=np.int32), _table(ang), R, return_rotated=True)
    assert sc[1, 2] == 1.0 and not (q[1, 2] & 0x7F).any()  # +-0 (the sign of a zero product is kept)
    deq = oracle.e4m3_to_f64(q.ravel()).reshape(q.shape) * sc[..., None].astype(np.float64)
    y64 = y.astype(np.float64)
    # e4m3: 3 mantissa bits (half-ulp 2^-4 relative), subnormal step 2^-9 (half 2^-10) in scaled units
    bound = 2.0 ** -4 * np.abs(y64) + 2.0 ** -10 * sc[..., None]
    assert np.all(np.abs(deq - y64) <= bound * (1 + 1e-6))


def test_rot_dim_zero_is_plain_per_head_quantisation():
    T, heads, D = 2, 2, 16
    x = _x(T, heads, D, 8)
    q, sc, y = oracle.inv_rope_fp8_quant(x, np.zeros(T, dtype=np.int32), np.zeros((1, 0), np.float32), 0,
                                         return_rotated=True)
    assert np.array_equal(y, _bf16_vals(x))
    assert np.allclose(sc, np.abs(_bf16_vals(x)).max(axis=-1) / 448.0, rtol=1e-7)


def test_position_out_of_range_is_rejected():
    with pytest.raises(ValueError):
        oracle.inv_rope_fp8_quant(_x(1, 1, 8, 9), np.array([5], dtype=np.int32), np.zeros((2, 8), np.float32), 8)
