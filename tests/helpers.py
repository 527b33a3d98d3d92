"""Shared test helpers: tie-free routing inputs and error metrics.

Tests may use the oracle; the product library never does.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from moe_synth import resample_tokens


def routing_gap(logits: np.ndarray, k: int) -> np.ndarray:
    """Per token, the gap between the k-th and (k+1)-th largest logit (inf when k == E)."""
    E = logits.shape[1]
    if k >= E:
        return np.full(logits.shape[0], np.inf)
    srt = -np.sort(-logits, axis=1)
    return srt[:, k - 1] - srt[:, k]


def make_tie_free(layer: dict, min_gap_rel: float = 1e-3, max_rounds: int = 30) -> None:
    """Redraw tokens whose k-th/(k+1)-th router logits are closer than min_gap_rel * rms(logits).

    A fp32 router on the GPU sums in another order than the fp64 oracle; with
    this gap both pick the same experts, so routing can be compared exactly.
    """
    sp = layer["spec"]
    for attempt in range(max_rounds):
        lg = oracle.router_logits(layer["X"].cpu(), layer["Wr"].cpu())
        scale = float(np.sqrt(np.mean(lg * lg))) or 1.0
        bad = np.nonzero(routing_gap(lg, sp.k) < min_gap_rel * scale)[0]
        if bad.size == 0:
            return
        resample_tokens(layer, torch.from_numpy(bad), attempt)
    raise RuntimeError("could not make routing tie-free")


def rel_err(got, ref, label: str = "") -> float:
    """max |got - ref| / RMS(ref), the layer-output error measure (printed for the log)."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(r * r)))
    err = float(np.max(np.abs(g - r))) / (rms if rms > 0 else 1.0)
    print(f"[parity] {label} max|err|/rms = {err:.3e}")
    return err


TOL = {"f32": 1e-5, "bf16": 2e-2, "e4m3": 6e-2}


def bf16_half_ulp(v) -> np.ndarray:
    """Half the spacing of bf16 numbers at |v| (8 significant bits): the largest error of a
    round-to-nearest cast of v to bf16, 2^(floor(log2 |v|) - 8) in the normal range."""
    a = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 8.0)


def parity_metrics(got, ref) -> dict:
    """The error measures of a layer output against the oracle's fp64 output, all relative to RMS(ref):
      err    max |got - ref|
      floor  max half-ulp of bf16 at ref: what rounding the exact result to bf16 alone can cost
      excess max (|got - ref| - half-ulp of bf16 at max(|got|, |ref|)), clipped at 0: the error
             beyond the final rounding of the output to bf16, i.e. of the arithmetic before it"""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(r * r))) or 1.0
    d = np.abs(g - r)
    hu = bf16_half_ulp(np.maximum(np.abs(g), np.abs(r)))
    return {"err": float(d.max()) / rms, "floor": float(bf16_half_ulp(r).max()) / rms,
            "excess": float(np.maximum(d - hu, 0.0).max()) / rms, "max_over_rms": float(np.abs(r).max()) / rms}


def assert_parity(got, ref, kind: str, label: str = "") -> dict:
    """Layer-output parity at the tolerance of `kind` ("f32", "bf16", "e4m3": 1e-5, 2e-2, 6e-2 of
    max|err| / RMS(out)).

    fp32 outputs: max|err| / RMS <= 1e-5.
    bf16 outputs (the bf16 and FP8 layers): the bar bounds the layer's arithmetic; the one rounding
    of the output to bf16, which the fp64 oracle does not have and no bf16 result avoids, comes on
    top of it (half an ulp of the output element).  So every element must satisfy
        |got - ref| <= tol * RMS(ref) + half-ulp_bf16(max(|got|, |ref|)),
    and where that rounding can cost at most half the bar (floor <= tol / 2) the plain
    max|err| / RMS <= tol is asserted as well.  At an output of 6 RMS or more the rounding alone
    reaches 1.6e-2 to 3.1e-2 of RMS, so the plain measure cannot meet 2e-2 on every draw."""
    tol = TOL[kind]
    m = parity_metrics(got, ref)
    print(f"[parity] {label} err={m['err']:.3e} excess={m['excess']:.3e} floor={m['floor']:.3e} "
          f"max/rms={m['max_over_rms']:.2f}")
    if kind == "f32":
        assert m["err"] <= tol, f"{label}: max|err|/rms {m['err']:.3g} > {tol}"
        return m
    assert m["excess"] <= tol, f"{label}: error beyond the output rounding {m['excess']:.3g} > {tol}"
    if m["floor"] <= tol / 2:
        assert m["err"] <= tol, f"{label}: max|err|/rms {m['err']:.3g} > {tol} (floor {m['floor']:.3g})"
    return m
