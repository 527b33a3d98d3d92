"""GPU parity of the inverse rotary embedding + per-head e4m3 quantisation kernel against
the oracle: codes and scales bit for bit (both sides decide every code in the same fp32
arithmetic), over rotated / partly rotated / unrotated heads, head sizes up to 1024,
zero vectors, the first and last table positions, the persistent and shared-memory staged
forms of the kernel on odd large layouts, and the full-size prefill layout.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_synth import make_rope_inputs, rope_spec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_layer_scan_gb300 as m

    assert torch.cuda.is_available()
    return m


def _check(moe, d):
    rs = d["spec"]
    x, pos, cs = d["x"], d["pos"], d["cos_sin"]
    q, sc = moe.moe_inv_rope_fp8_quant(x.cuda(), pos.cuda(), cs.cuda(), rs.rot_dim)
    torch.cuda.synchronize()
    assert moe.moe_get_status() == 0
    rq, rsc = oracle.inv_rope_fp8_quant(x, pos, cs, rs.rot_dim)
    gq, gsc = q.cpu().numpy(), sc.cpu().numpy()
    assert np.array_equal(gsc.view(np.uint32), rsc.view(np.uint32))
    assert np.array_equal(gq, rq), f"{int((gq != rq).sum())} codes differ"


@pytest.mark.parametrize("T,heads,D,R", [(1, 1, 64, 64), (37, 8, 128, 64), (300, 32, 128, 128), (5, 16, 576, 64),
                                         (7, 3, 256, 0), (3, 2, 1024, 1024), (2, 3, 1024, 512), (9, 5, 36, 4)])
def test_inv_rope_fp8_bit_exact(moe, T, heads, D, R):
    d = make_rope_inputs(rope_spec("gqa_decode", T=T, heads=heads, head_dim=D, rot_dim=R, max_pos=512))
    _check(moe, d)


def test_zero_vectors_and_table_edges(moe):
    d = make_rope_inputs(rope_spec("gqa_decode", T=6, heads=4, max_pos=300))
    d["x"][2, 1] = 0
    d["x"][4] = 0
    d["pos"][0] = 0
    d["pos"][5] = 299
    _check(moe, d)


# Large inputs: long vectors (32 lanes each) from 4 MB go through the kernel that stages
# chunks of consecutive vectors and their tokens' table rows in shared memory (head counts
# that do not divide a chunk, partly rotated heads, a ragged last chunk); short vectors
# through the persistent register kernel (odd head counts, one head per token).
@pytest.mark.parametrize("T,heads,D,R", [(5000, 7, 128, 128), (300, 40, 200, 64), (20000, 1, 128, 96),
                                         (1100, 9, 576, 64)])
def test_inv_rope_fp8_large_bit_exact(moe, T, heads, D, R):
    d = make_rope_inputs(rope_spec("gqa_decode", T=T, heads=heads, head_dim=D, rot_dim=R, max_pos=4096))
    assert T * heads * D * 2 >= 4 << 20
    _check(moe, d)


@pytest.mark.parametrize("T,heads,D,R", [(5000, 7, 128, 128), (1100, 9, 576, 64)])
def test_large_position_outside_table_is_flagged(moe, T, heads, D, R):
    d = make_rope_inputs(rope_spec("gqa_decode", T=T, heads=heads, head_dim=D, rot_dim=R, max_pos=4096))
    pos = d["pos"].clone()
    pos[T - 679] = -1
    moe.moe_inv_rope_fp8_quant(d["x"].cuda(), pos.cuda(), d["cos_sin"].cuda(), R)
    assert moe.moe_get_status() == moe.MOE_ERR_DEVICE_INDEX
    assert moe.moe_get_status() == 0


@pytest.mark.parametrize("name", ["gqa_prefill", "mla_decode"])
def test_inv_rope_fp8_full_size(moe, name):
    _check(moe, make_rope_inputs(rope_spec(name)))


def test_position_outside_table_is_flagged(moe):
    d = make_rope_inputs(rope_spec("gqa_decode", T=4, max_pos=64))
    pos = d["pos"].clone()
    pos[2] = 64
    moe.moe_inv_rope_fp8_quant(d["x"].cuda(), pos.cuda(), d["cos_sin"].cuda(), 128)
    assert moe.moe_get_status() == moe.MOE_ERR_DEVICE_INDEX
    assert moe.moe_get_status() == 0
