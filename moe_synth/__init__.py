"""Seeded synthetic inputs for the fused MoE layer forward.

This module serves both the CUDA library's tests/benchmark and the CPU oracle.
It holds none of the layer's arithmetic: it only draws inputs with the shapes,
value distributions and routing structure of the workloads the pages discuss
(Mixtral-style 8 experts top-2 with hidden 4096 and FFN 14336; fine-grained
top-8 decode; FP8 per-tensor weights; long prefill batches).

Layouts (row-major, contiguous):
  X    [T, H]       activations (float32 or bfloat16)
  Wr   [E, H]       router weight, same dtype as X
  W13  [E, 2I, H]   gate rows [0, I) above up rows [I, 2I); bf16/fp32, or e4m3 codes
  W2   [E, H, I]    down projection
  w13_scale, w2_scale [E] float32 per-expert FP8 scales (None unless e4m3)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}


@dataclass
class LayerSpec:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    renorm: bool
    act: str = "bf16"
    w: str = "bf16"
    seed: int = 1234
    x_std: float = 1.0
    w_std: float = 0.02
    wr_std: Optional[float] = None  # None -> 1/sqrt(H): router logits ~ N(0, 1)
    router: str = "gauss"  # "gauss" | "zipf" | "hot"
    zipf_s: float = 1.1
    hot_experts: int = 4
    hot_frac: float = 0.5
    hot_boost: float = 10.0
    extra: dict = field(default_factory=dict)


# The five workloads (decode ones take their token count M at build time).
def spec(name: str, T: Optional[int] = None, **over) -> LayerSpec:
    base = {
        "tiny_f32": dict(T=64, H=256, E=8, I=512, k=2, renorm=True, act="f32", w="f32", seed=1234,
                         x_std=0.02, w_std=0.02, wr_std=0.02),
        "mixtral_decode": dict(T=64, H=4096, E=8, I=14336, k=2, renorm=True, seed=1235),
        "fine_decode": dict(T=64, H=2048, E=128, I=768, k=8, renorm=True, seed=1236, router="zipf"),
        "fp8_decode": dict(T=64, H=4096, E=64, I=8192, k=8, renorm=False, w="e4m3", seed=1237),
        "int4_decode": dict(T=64, H=4096, E=8, I=14336, k=2, renorm=True, w="int4", seed=1239),
        "prefill": dict(T=8192, H=4096, E=64, I=2048, k=8, renorm=True, seed=1238),
        "prefill_hot": dict(T=8192, H=4096, E=64, I=2048, k=8, renorm=True, seed=1238, router="hot"),
    }[name]
    base = dict(base)
    if T is not None:
        base["T"] = T
    base.update(over)
    return LayerSpec(name=name, **base)


DECODE_M = {"mixtral_decode": (1, 4, 16, 64), "fine_decode": (1, 8, 32, 64), "fp8_decode": (1, 16, 64),
            "int4_decode": (1, 16, 64)}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _zipf_bias(E: int, s: float, g: torch.Generator) -> torch.Tensor:
    """log of a Zipf(s) pmf over ranks 1..E, ranks assigned to experts by a seeded permutation."""
    ranks = torch.arange(1, E + 1, dtype=torch.float64)
    pmf = ranks.pow(-s)
    pmf = pmf / pmf.sum()
    perm = torch.randperm(E, generator=g)
    bias = torch.empty(E, dtype=torch.float64)
    bias[perm] = pmf.log()
    return bias.float()


def _fp8_encode_expertwise(w: torch.Tensor):
    """Per-expert-tensor FP8 weights: scale = amax / 448, codes via torch's e4m3 cast (inputs only)."""
    amax = w.abs().amax().float()
    s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (w / s).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return codes, s


def _structure_columns(sp: LayerSpec, X: torch.Tensor, rows: Optional[torch.Tensor], hot_tokens: Optional[torch.Tensor]):
    """Re-apply the routing-structure input features to the given rows (all rows if None)."""
    H = sp.H
    if sp.router == "zipf":
        if rows is None:
            X[:, H - 1] = 1.0
        else:
            X[rows, H - 1] = 1.0
    elif sp.router == "hot":
        col = torch.zeros(X.shape[0], dtype=X.dtype, device=X.device)
        col[hot_tokens] = 1.0
        if rows is None:
            X[:, H - 2] = col
        else:
            X[rows, H - 2] = col[rows]


# Nibble of element e (0..7) inside a 32-bit word of 8 consecutive K elements (the INT4 storage format).
INT4_NIBBLE_OF = (0, 4, 1, 5, 2, 6, 3, 7)


def _int4_encode_groupwise(w: torch.Tensor):
    """Stand-in for an offline INT4 weight quantiser (the kind AWQ / GPTQ produce, here without
    calibration): a bf16 scale per (row, 128 K elements) = max |w| / 7, codes round(w / s) clamped to
    [-8, 7]; returns (packed codes uint8 [rows, K/2], scales bf16 [rows, K/128])."""
    rows, K = w.shape
    wg = w.float().reshape(rows, K // 128, 128)
    s = (wg.abs().amax(dim=2) / 7.0).clamp_min(1e-8).to(torch.bfloat16)
    q = torch.round(wg / s.float()[:, :, None]).clamp_(-8, 7).to(torch.int32).reshape(rows, K // 8, 8)
    nib = torch.tensor(INT4_NIBBLE_OF, dtype=torch.int32, device=w.device)
    word = torch.zeros(rows, K // 8, dtype=torch.int64, device=w.device)
    for el in range(8):
        word |= ((q[:, :, el] & 0xF).to(torch.int64) << (4 * int(nib[el])))
    b = torch.stack([(word >> (8 * i)) & 0xFF for i in range(4)], dim=2).to(torch.uint8)
    return b.reshape(rows, K // 2), s


def make_layer(sp: LayerSpec, device="cpu", weights: bool = True) -> dict:
    """Draw one synthetic layer + token batch.  Deterministic in (spec, device)."""
    dev = torch.device(device)
    g = _gen(sp.seed, dev)
    gcpu = _gen(sp.seed + 7919, "cpu")  # small host-side draws (permutations, hot-token choice)
    adt = DTYPES[sp.act]
    T, H, I, E = sp.T, sp.H, sp.I, sp.E
    wr_std = sp.wr_std if sp.wr_std is not None else 1.0 / math.sqrt(H)

    X = (torch.randn(T, H, generator=g, device=dev) * sp.x_std)
    Wr = (torch.randn(E, H, generator=g, device=dev) * wr_std)
    hot_tokens = None
    hot = None
    if sp.router == "zipf":
        Wr[:, H - 1] = _zipf_bias(E, sp.zipf_s, gcpu).to(dev)
    elif sp.router == "hot":
        perm = torch.randperm(E, generator=gcpu)
        hot = perm[: sp.hot_experts].sort().values
        n_hot = int(round(sp.hot_frac * T))
        hot_tokens = torch.randperm(T, generator=gcpu)[:n_hot].sort().values.to(dev)
        Wr[:, H - 2] = 0.0
        Wr[hot.to(dev), H - 2] = sp.hot_boost
    _structure_columns(sp, X, None, hot_tokens)

    out = {
        "spec": sp,
        "X": X.to(adt).contiguous(),
        "Wr": Wr.to(adt).contiguous(),
        "hot_experts": hot,
        "hot_tokens": None if hot_tokens is None else hot_tokens.cpu(),
        "W13": None, "W2": None, "w13_scale": None, "w2_scale": None,
    }
    if not weights:
        return out
    if sp.w == "int4":
        W13 = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=dev)
        W2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=dev)
        # scales group-major per expert: [E][K/128][rows]
        s13 = torch.empty(E, H // 128, 2 * I, dtype=torch.bfloat16, device=dev)
        s2 = torch.empty(E, I // 128, H, dtype=torch.bfloat16, device=dev)
        for e in range(E):
            W13[e], s = _int4_encode_groupwise(torch.randn(2 * I, H, generator=g, device=dev) * sp.w_std)
            s13[e] = s.t()
            W2[e], s = _int4_encode_groupwise(torch.randn(H, I, generator=g, device=dev) * sp.w_std)
            s2[e] = s.t()
        out.update(W13=W13, W2=W2, w13_scale=s13, w2_scale=s2)
    elif sp.w == "e4m3":
        W13 = torch.empty(E, 2 * I, H, dtype=torch.float8_e4m3fn, device=dev)
        W2 = torch.empty(E, H, I, dtype=torch.float8_e4m3fn, device=dev)
        s13 = torch.empty(E, dtype=torch.float32, device=dev)
        s2 = torch.empty(E, dtype=torch.float32, device=dev)
        for e in range(E):
            W13[e], s13[e] = _fp8_encode_expertwise(torch.randn(2 * I, H, generator=g, device=dev) * sp.w_std)
            W2[e], s2[e] = _fp8_encode_expertwise(torch.randn(H, I, generator=g, device=dev) * sp.w_std)
        out.update(W13=W13, W2=W2, w13_scale=s13, w2_scale=s2)
    else:
        wdt = DTYPES[sp.w]
        W13 = torch.empty(E, 2 * I, H, dtype=wdt, device=dev)
        W2 = torch.empty(E, H, I, dtype=wdt, device=dev)
        for e in range(E):
            W13[e] = (torch.randn(2 * I, H, generator=g, device=dev) * sp.w_std).to(wdt)
            W2[e] = (torch.randn(H, I, generator=g, device=dev) * sp.w_std).to(wdt)
        out.update(W13=W13, W2=W2)
    return out


def resample_tokens(layer: dict, rows, attempt: int) -> None:
    """Redraw the activation rows ``rows`` (in place, seeded by attempt), keeping the routing structure."""
    sp: LayerSpec = layer["spec"]
    X = layer["X"]
    rows = torch.as_tensor(rows, dtype=torch.long)
    if rows.numel() == 0:
        return
    g = _gen(sp.seed * 1000003 + 17 * attempt + 1, "cpu")
    fresh = torch.randn(rows.numel(), sp.H, generator=g) * sp.x_std
    Xf = X.float().cpu()
    Xf[rows] = fresh
    hot = layer.get("hot_tokens")
    _structure_columns(sp, Xf, rows, hot)
    layer["X"] = Xf.to(X.dtype).to(X.device).contiguous()


def to_device(layer: dict, device) -> dict:
    out = dict(layer)
    for key in ("X", "Wr", "W13", "W2", "w13_scale", "w2_scale"):
        if out.get(key) is not None:
            out[key] = out[key].to(device)
    return out


# -- inverse rotary embedding + per-head FP8 quantisation inputs -------------------

@dataclass
class RopeSpec:
    name: str
    T: int
    heads: int
    head_dim: int
    rot_dim: int
    max_pos: int = 8192
    theta: float = 10000.0
    seed: int = 4321


def rope_spec(name: str, **over) -> RopeSpec:
    """Head layouts of attention blocks around MoE layers: a Llama-style query (32 heads of 128,
    fully rotated) and an MLA-style query (128 heads of 576: 64 rotated, 512 not)."""
    base = {
        "gqa_prefill": dict(T=8192, heads=32, head_dim=128, rot_dim=128),
        "gqa_decode": dict(T=64, heads=32, head_dim=128, rot_dim=128),
        "mla_decode": dict(T=64, heads=128, head_dim=576, rot_dim=64),
    }[name]
    base = dict(base)
    base.update(over)
    return RopeSpec(name=name, **base)


def make_rope_inputs(rs: RopeSpec, device="cpu") -> dict:
    """x [T, heads, head_dim] bf16 ~ N(0,1) with a few large outliers per vector, positions [T] int32
    uniform in [0, max_pos), and the cos/sin table [max_pos, rot_dim] fp32 of the standard rotary
    frequencies theta^(-2i/rot_dim) (the table a serving stack precomputes: an input here)."""
    g = _gen(rs.seed, "cpu")
    x = torch.randn(rs.T, rs.heads, rs.head_dim, generator=g, dtype=torch.float32)
    spikes = torch.rand(rs.T, rs.heads, rs.head_dim, generator=g) < 0.01
    x = torch.where(spikes, x * 8.0, x)
    pos = torch.randint(0, rs.max_pos, (rs.T,), generator=g, dtype=torch.int32)
    half = rs.rot_dim // 2
    if half > 0:
        inv = rs.theta ** (-torch.arange(half, dtype=torch.float64) * 2.0 / rs.rot_dim)
        ang = torch.arange(rs.max_pos, dtype=torch.float64)[:, None] * inv[None, :]
        cos_sin = torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).to(torch.float32)
    else:
        cos_sin = torch.zeros(rs.max_pos, 0, dtype=torch.float32)
    d = {"spec": rs, "x": x.to(torch.bfloat16), "pos": pos, "cos_sin": cos_sin.contiguous()}
    if device != "cpu":
        d = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    return d
