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
