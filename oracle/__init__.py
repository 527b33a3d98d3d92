"""Plain CPU oracle of the fused MoE layer forward (ctypes wrapper over moe_oracle.c).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product library and
its Python binding never do.  It shares no code with the CUDA path.

Every function takes numpy arrays (or CPU torch tensors, converted with
``.numpy()``) in the storage formats of the layer: float32, bfloat16 as raw
uint16 bit patterns, e4m3 as raw uint8 codes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, BF16, E4M3, INT4 = 0, 1, 2, 3

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/libmoe_oracle.so (plain C, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp", "-o", tmp,
                               _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_f32_to_e4m3_satfinite.restype = ctypes.c_uint8
        lib.oracle_f32_to_e4m3_satfinite.argtypes = [ctypes.c_float]
        lib.oracle_silu.restype = ctypes.c_double
        lib.oracle_silu.argtypes = [ctypes.c_double]
        lib.oracle_e4m3_scale.restype = ctypes.c_float
        lib.oracle_e4m3_scale.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_quant.restype = ctypes.c_uint8
        lib.oracle_e4m3_quant.argtypes = [ctypes.c_float, ctypes.c_float]
        lib.oracle_router_logits.restype = None
        lib.oracle_router_logits.argtypes = [P, P, i, i, i, i, P]
        lib.oracle_topk.restype = i
        lib.oracle_topk.argtypes = [P, i, i, i, i, P, P]
        lib.oracle_align.restype = i
        lib.oracle_align.argtypes = [P, i, i, i, i, P, P, P, P]
        lib.oracle_moe_forward.restype = i
        lib.oracle_moe_forward.argtypes = [P, P, P, P, i, i, i, i, i, i, i, i, P, P, P, i, P, P, P, P]
        lib.oracle_inv_rope_fp8.restype = i
        lib.oracle_inv_rope_fp8.argtypes = [P, i, i, i, i, P, P, i, P, P, P]
        lib.oracle_set_threads.restype = None
        lib.oracle_set_threads.argtypes = [i]
        lib.oracle_get_threads.restype = i
        lib.oracle_get_threads.argtypes = []
        _lib = lib
        return lib


def _np(a):
    """numpy view of a numpy array or CPU torch tensor, bit patterns for bf16/fp8."""
    if isinstance(a, np.ndarray):
        return np.ascontiguousarray(a)
    import torch

    t = a.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def _dtype_code(a) -> int:
    if isinstance(a, np.ndarray):
        return {np.dtype(np.float32): F32, np.dtype(np.uint16): BF16, np.dtype(np.uint8): E4M3}[a.dtype]
    import torch

    return {torch.float32: F32, torch.bfloat16: BF16, torch.float8_e4m3fn: E4M3, torch.uint8: E4M3}[a.dtype]


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


# -- number formats ----------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_bf16_to_f64(int(v)) for v in b], dtype=np.float64)


def f32_to_bf16(x) -> np.ndarray:
    lib = _load()
    v = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.oracle_f32_to_bf16(float(f)) for f in v], dtype=np.uint16)


def e4m3_to_f64(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.oracle_e4m3_to_f64(int(v)) for v in c], dtype=np.float64)


def f32_to_e4m3(x) -> np.ndarray:
    lib = _load()
    v = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.oracle_f32_to_e4m3_satfinite(float(f)) for f in v], dtype=np.uint8)


def e4m3_scale(amax: float) -> float:
    return float(_load().oracle_e4m3_scale(float(amax)))


def silu(z: float) -> float:
    return float(_load().oracle_silu(float(z)))


# -- layer steps -------------------------------------------------------------

def router_logits(X, Wr) -> np.ndarray:
    """logits[T,E] (float64) of the router gate GEMM on the stored inputs."""
    x, wr = _np(X), _np(Wr)
    dt = _dtype_code(X)
    T, H = x.shape
    E = wr.shape[0]
    out = np.empty((T, E), dtype=np.float64)
    _load().oracle_router_logits(_ptr(x), _ptr(wr), dt, T, H, E, _ptr(out))
    return out


def topk(logits, k: int, renorm: bool):
    """(ids int32 [T,k], weights float64 [T,k]) of softmax -> top-k (-> renorm)."""
    lg = np.ascontiguousarray(np.asarray(logits, dtype=np.float64))
    T, E = lg.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    rc = _load().oracle_topk(_ptr(lg), T, E, int(k), int(bool(renorm)), _ptr(ids), _ptr(w))
    if rc != 0:
        raise ValueError(f"oracle_topk failed ({rc})")
    return ids, w


def align_capacity(T: int, k: int, E: int, B: int) -> int:
    n = T * k
    return n + min(E, n) * (B - 1)


def align(ids, E: int, B: int):
    """(sorted_ids, expert_ids, num_post_pad, counts) of the block-padded expert sort."""
    a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    T, k = a.shape
    cap = max(align_capacity(T, k, E, B), 1)
    sorted_ids = np.full(cap, -1, dtype=np.int32)
    expert_ids = np.full(max(cap // B, 1), -1, dtype=np.int32)
    npp = np.zeros(1, dtype=np.int32)
    counts = np.zeros(E, dtype=np.int32)
    rc = _load().oracle_align(_ptr(a), T, k, E, B, _ptr(sorted_ids), _ptr(expert_ids), _ptr(npp), _ptr(counts))
    if rc != 0:
        raise ValueError(f"oracle_align failed ({rc})")
    n = int(npp[0])
    return sorted_ids[:n].copy(), expert_ids[: n // B].copy(), n, counts


def moe_forward(X, Wr, W13, W2, topk_k: int, renorm: bool, w13_scale=None, w2_scale=None, tokens=None,
                w_format=None):
    """Layer output (float64 [n,H]) plus the routing of all T tokens and the FP8 activation scales.

    Returns dict(out, ids, w, act_scales).  ``tokens`` selects a subset of output rows.
    ``w_format="int4"``: W13 [E,2I,H/2] and W2 [E,H,I/2] are packed INT4 codes (uint8) and the scales
    bf16 group scales, group-major per expert: [E,H/128,2I] and [E,I/128,H].
    """
    x, wr, w13, w2 = _np(X), _np(Wr), _np(W13), _np(W2)
    adt, wdt = _dtype_code(X), _dtype_code(W13)
    T, H = x.shape
    E = wr.shape[0]
    I = w13.shape[1] // 2
    if w_format == "int4":
        wdt = INT4
        s13 = np.ascontiguousarray(_np(w13_scale), dtype=np.uint16)
        s2 = np.ascontiguousarray(_np(w2_scale), dtype=np.uint16)
        w13_scale = w2_scale = None
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    n = T if tok is None else tok.shape[0]
    out = np.empty((n, H), dtype=np.float64)
    ids = np.empty((T, topk_k), dtype=np.int32)
    w = np.empty((T, topk_k), dtype=np.float64)
    scales = np.zeros(2, dtype=np.float32)
    if w_format != "int4":
        s13 = None if w13_scale is None else np.ascontiguousarray(_np(w13_scale), dtype=np.float32)
        s2 = None if w2_scale is None else np.ascontiguousarray(_np(w2_scale), dtype=np.float32)
    rc = _load().oracle_moe_forward(
        _ptr(x), _ptr(wr), _ptr(w13), _ptr(w2), adt, wdt, T, H, I, E, int(topk_k), int(bool(renorm)),
        None if s13 is None else _ptr(s13), None if s2 is None else _ptr(s2),
        None if tok is None else _ptr(tok), n, _ptr(out), _ptr(ids), _ptr(w), _ptr(scales))
    if rc != 0:
        raise ValueError(f"oracle_moe_forward failed ({rc})")
    return {"out": out, "ids": ids, "w": w, "act_scales": scales}


def inv_rope_fp8_quant(X, positions, cos_sin, rot_dim: int, return_rotated: bool = False):
    """(codes uint8 [T,heads,D], scales float32 [T,heads][, rotated float32 [T,heads,D]]) of the inverse
    rotary embedding + per-head e4m3 quantisation; X is bf16 [T,heads,D] (bit patterns or a torch tensor)."""
    x = np.ascontiguousarray(_np(X), dtype=np.uint16)
    T, heads, D = x.shape
    pos = np.ascontiguousarray(_np(positions), dtype=np.int32)
    cs = np.ascontiguousarray(_np(cos_sin), dtype=np.float32)
    max_pos = cs.shape[0]
    q = np.empty((T, heads, D), dtype=np.uint8)
    sc = np.empty((T, heads), dtype=np.float32)
    y = np.empty((T, heads, D), dtype=np.float32) if return_rotated else None
    rc = _load().oracle_inv_rope_fp8(_ptr(x), T, heads, D, int(rot_dim), _ptr(pos), _ptr(cs), max_pos,
                                     None if y is None else _ptr(y), _ptr(q), _ptr(sc))
    if rc != 0:
        raise ValueError(f"oracle_inv_rope_fp8 failed ({rc})")
    return (q, sc, y) if return_rotated else (q, sc)
