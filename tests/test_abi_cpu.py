"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
entry point include/moe_api.h declares, sizes its workspace, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__

    __graft_entry__._builder().build()
    import mixture_experts_layer_scan_gb300 as m

    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "moe_api.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(moe):
    names = _declared()
    assert len(names) >= 10
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(moe.EXPORTS) == names


def test_exports_nothing_else(moe):
    import subprocess

    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True, text=True).stdout
    syms = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert syms == set(_declared())


def test_strerror_and_version(moe):
    assert moe.strerror(0) == "ok"
    assert "workspace" in moe.strerror(moe.MOE_ERR_WORKSPACE)
    assert moe.version() >= 100


def test_workspace_size_rules(moe):
    f32 = moe.moe_workspace_size(64, 256, 512, 8, 2, moe.MOE_F32, moe.MOE_F32)
    assert f32 > 0 and f32 % 256 == 0
    dec = moe.moe_workspace_size(64, 4096, 14336, 8, 2, moe.MOE_BF16, moe.MOE_BF16)
    pre = moe.moe_workspace_size(8192, 4096, 2048, 64, 8, moe.MOE_BF16, moe.MOE_BF16)
    fp8 = moe.moe_workspace_size(64, 4096, 8192, 64, 8, moe.MOE_BF16, moe.MOE_E4M3)
    assert 0 < dec < pre and fp8 > 0
    # the prefill workspace holds at least the sorted rows, the intermediate and the fp32 expert outputs Y
    cap = 8192 * 8 + 64 * 127
    assert pre >= cap * 4096 * 2 + cap * 2048 * 2 + 8192 * 8 * 4096 * 4
    with pytest.raises(moe.MoeError) as e:
        moe.moe_workspace_size(64, 4000, 14336, 8, 2, moe.MOE_BF16, moe.MOE_BF16)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoeError) as e:
        moe.moe_workspace_size(64, 4096, 1024, 8, 9, moe.MOE_BF16, moe.MOE_BF16)
    assert e.value.code == moe.MOE_ERR_ARG
    with pytest.raises(moe.MoeError) as e:
        moe.moe_workspace_size(64, 4096, 1024, 8, 2, moe.MOE_F32, moe.MOE_BF16)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED


def test_plan_info(moe):
    d = moe.moe_plan_info(1, 2048, 768, 128, 8, moe.MOE_BF16, moe.MOE_BF16)
    assert d["orientation"] == moe.ORIENT_SWAP_AB and d["block"] == 16 and d["act_split"] == 1
    # router, top-k, permutation, GEMM1 (its last-arriving CTA per tile sums the K splits), GEMM2, combine
    assert d["splits_gemm1"] > 1 and d["kernel_launches"] == 6
    assert d["workspace_bytes"] == moe.moe_workspace_size(1, 2048, 768, 128, 8, moe.MOE_BF16, moe.MOE_BF16)
    p = moe.moe_plan_info(8192, 4096, 2048, 64, 8, moe.MOE_BF16, moe.MOE_BF16)
    assert p["orientation"] == moe.ORIENT_TOKEN_MAJOR and p["block"] == 128 and p["kernel_launches"] == 7
    assert p["cta_pair"] == 1
    single = moe.moe_plan_info(8192, 4096, 2048, 64, 8, moe.MOE_BF16, moe.MOE_BF16, {"cta_pair": 2})
    assert single["block"] == 128 and single["cta_pair"] == 0
    # pairs need 256-row GEMM2 weight tiles (H % 256 == 0)
    assert moe.moe_plan_info(8192, 4224, 2048, 64, 8, moe.MOE_BF16, moe.MOE_BF16)["cta_pair"] == 0
    with pytest.raises(moe.MoeError) as e:
        moe.moe_plan_info(8192, 4224, 2048, 64, 8, moe.MOE_BF16, moe.MOE_BF16, {"cta_pair": 1})
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED
    f = moe.moe_plan_info(64, 4096, 8192, 64, 8, moe.MOE_BF16, moe.MOE_E4M3)
    assert f["act_split"] == 0 and f["kernel_launches"] >= 9
    assert moe.moe_plan_info(64, 256, 512, 8, 2, moe.MOE_F32, moe.MOE_F32)["orientation"] == 0


@pytest.mark.parametrize("T,H,I,E,k,w,s2", [
    (1, 4096, 14336, 8, 2, "bf16", 4),     # exactly k experts: 32 whole tiles want about 4 splits
    (16, 4096, 14336, 8, 2, "bf16", 1),    # every expert active: one 128-tile wave of whole rows
    (64, 4096, 14336, 8, 2, "bf16", 1),
    (4, 4096, 14336, 8, 2, "bf16", 7),     # about 5.5 of 8 experts active: wave counts alone
    (1, 4096, 8192, 64, 8, "e4m3", 1),     # exactly 8 experts x 16 tiles
    (8, 2048, 768, 128, 8, "bf16", 2),     # few active experts of many: wave counts alone
    (16, 4096, 14336, 8, 2, "int4", 7),    # INT4 is bound by the MMA rate: wave counts alone
])
def test_gemm2_split_plans(moe, T, H, I, E, k, w, s2):
    """GEMM2's K splits: the shared-bandwidth model where the active-expert count is known
    (one token, or at least 4E pairs), the wave count elsewhere and for INT4."""
    wdt = {"bf16": moe.MOE_BF16, "e4m3": moe.MOE_E4M3, "int4": moe.MOE_INT4}[w]
    assert moe.moe_plan_info(T, H, I, E, k, moe.MOE_BF16, wdt)["splits_gemm2"] == s2


def test_align_capacity(moe):
    assert moe.moe_align_capacity(64, 8, 128, 16) == (512 + 128 * 15, (512 + 128 * 15) // 16)
    assert moe.moe_align_capacity(1, 2, 8, 16) == (2 + 2 * 15, 32 // 16)
    assert moe.moe_align_capacity(0, 2, 8, 16) == (0, 0)


def test_forward_argument_errors_before_launch(moe):
    lib = moe.lib()
    v = ctypes.c_void_p
    fake = v(0x1000)  # never dereferenced: every call below fails validation first
    odd = v(0x1008)
    ws = v(0x100000)
    # T = 0 is a successful no-op
    assert lib.moe_forward(None, None, None, None, 0, 256, 256, 8, 2, 1, 1, 1, None, None, None, None, 0, None,
                           None) == 0
    # null pointers
    assert lib.moe_forward(None, fake, fake, fake, 4, 256, 256, 8, 2, 1, 1, 1, None, None, fake, ws, 1 << 30, None,
                           None) == moe.MOE_ERR_ARG
    # misaligned
    assert lib.moe_forward(odd, fake, fake, fake, 4, 256, 256, 8, 2, 1, 1, 1, None, None, fake, ws, 1 << 30, None,
                           None) == moe.MOE_ERR_ALIGNMENT
    # workspace too small
    assert lib.moe_forward(fake, fake, fake, fake, 4, 256, 256, 8, 2, 1, 1, 1, None, None, fake, ws, 1024, None,
                           None) == moe.MOE_ERR_WORKSPACE
    # FP8 without scales
    assert lib.moe_forward(fake, fake, fake, fake, 4, 256, 256, 8, 2, 1, 1, 2, None, None, fake, ws, 1 << 30, None,
                           None) == moe.MOE_ERR_ARG
    # bad sizes
    assert lib.moe_forward(fake, fake, fake, fake, 4, 256, 256, 2000, 2, 1, 1, 1, None, None, fake, ws, 1 << 30,
                           None, None) == moe.MOE_ERR_ARG
    assert lib.moe_route(fake, fake, 4, 256, 8, 0, 1, 1, fake, fake, fake, None) == moe.MOE_ERR_ARG
    # logits_out is required: the router writes the logits there before ranking them (no scratch of its own)
    assert lib.moe_route(fake, fake, 4, 256, 8, 2, 1, 1, None, fake, fake, None) == moe.MOE_ERR_ARG
    assert lib.moe_align(fake, 4, 2, 8, 0, fake, fake, fake, None, None) == moe.MOE_ERR_ARG
    assert lib.moe_topk_from_logits(fake, 4, 8, 9, 1, fake, fake, None) == moe.MOE_ERR_ARG
    # host-to-host forward: a no-op at T = 0; null buffers and bad sizes before any copy
    assert lib.moe_forward_host(None, None, None, None, None, 0, 256, 256, 8, 2, 1, 1, 1, None, None, None, None, 0,
                                None, None) == 0
    for hh, hd, oh in ((None, fake, fake), (fake, None, fake), (fake, fake, None)):
        assert lib.moe_forward_host(hh, hd, fake, fake, fake, 4, 256, 256, 8, 2, 1, 1, 1, None, None, oh, ws, 1 << 30,
                                    None, None) == moe.MOE_ERR_ARG
    assert lib.moe_forward_host(fake, fake, fake, fake, fake, 4, 256, 256, 2000, 2, 1, 1, 1, None, None, fake, ws,
                                1 << 30, None, None) == moe.MOE_ERR_ARG


def test_int4_plans_and_argument_errors(moe):
    """INT4 weights (host logic only): swap-AB up to 128 tokens with H and I multiples of 256, one bf16
    intermediate by default, the hi/lo pair on request; scales are required."""
    p = moe.moe_plan_info(64, 4096, 14336, 8, 2, moe.MOE_BF16, moe.MOE_INT4)
    assert p["orientation"] == moe.ORIENT_SWAP_AB and p["act_split"] == 0
    assert moe.moe_plan_info(64, 4096, 14336, 8, 2, moe.MOE_BF16, moe.MOE_INT4, {"act_split": 2})["act_split"] == 1
    assert moe.moe_plan_info(100, 512, 512, 8, 2, moe.MOE_BF16, moe.MOE_INT4)["orientation"] == moe.ORIENT_SWAP_AB
    for T, H, I, opts in [(129, 512, 512, None), (8, 384, 512, None), (8, 512, 640, None),
                          (64, 512, 512, {"orientation": 2})]:
        with pytest.raises(moe.MoeError) as e:
            moe.moe_plan_info(T, H, I, 8, 2, moe.MOE_BF16, moe.MOE_INT4, opts)
        assert e.value.code == moe.MOE_ERR_UNSUPPORTED, (T, H, I, opts)
    with pytest.raises(moe.MoeError):  # fp32 activations with INT4 weights
        moe.moe_plan_info(8, 512, 512, 8, 2, moe.MOE_F32, moe.MOE_INT4)
    lib = moe.lib()
    fake, ws = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x100000)
    # INT4 without group scales: rejected before anything is launched
    assert lib.moe_forward(fake, fake, fake, fake, 4, 512, 512, 8, 2, 1, 1, moe.MOE_INT4, None, None, fake, ws,
                           1 << 30, None, None) == moe.MOE_ERR_ARG
    # the INT4 workspace is sized from the same plan
    assert moe.moe_workspace_size(64, 4096, 14336, 8, 2, moe.MOE_BF16, moe.MOE_INT4) == p["workspace_bytes"]
