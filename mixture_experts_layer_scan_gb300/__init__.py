"""Python binding of the GB300 fused MoE layer library (ctypes over include/moe_api.h).

Argument marshalling only: every step of the layer runs in the CUDA kernels of
libmoe_gb300.so.  PyTorch supplies device memory and streams.  The names
mirror the C entry points; each raises MoeError on a nonzero return code.
If the shared library is missing this module fails at import, loudly: there is
no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_F32, MOE_BF16, MOE_E4M3, MOE_INT4 = 0, 1, 2, 3
MOE_OK, MOE_ERR_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, -1, -2, -3
MOE_ERR_CUDA, MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_DEVICE_INDEX, MOE_ERR_ALIGNMENT = -4, -5, -6, -7
ORIENT_AUTO, ORIENT_SWAP_AB, ORIENT_TOKEN_MAJOR = 0, 1, 2
STAGES = ("route", "align", "gather", "gemm1", "act", "gemm2", "combine")
NUM_STAGES = len(STAGES)
# phase stamps of the single-launch kernel (moe_options.trace), in the order of moe_trace_event
TRACE_EVENTS = ("start", "router", "barrier0", "topk", "barrier1", "tables", "gathered", "g1_issued", "g2_ready",
                "issued", "mma_done", "g1_done", "epi_done", "comb_first", "comb_done", "end")
TRACE_WORDS = len(TRACE_EVENTS)

# every entry point include/moe_api.h declares
EXPORTS = ("moe_strerror", "moe_workspace_size", "moe_plan_info", "moe_align_capacity", "moe_route",
           "moe_topk_from_logits", "moe_align", "moe_forward", "moe_forward_noalloc", "moe_get_status",
           "moe_version", "moe_inv_rope_fp8_quant", "moe_forward_routed", "moe_cache_create", "moe_cache_destroy",
           "moe_cache_workspace_size", "moe_forward_cached", "moe_cache_stats", "moe_cache_lru_plan",
           "moe_cache_set_copy_mode", "moe_copy_from_host", "moe_forward_host")
NOALLOC_MAX_WORKSPACE = 32 << 20


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} ({code})")


class moe_options(ctypes.Structure):
    _fields_ = [("orientation", ctypes.c_int), ("split_k", ctypes.c_int), ("inject_timeout", ctypes.c_int),
                ("act_split", ctypes.c_int), ("trace", ctypes.c_void_p), ("single_launch", ctypes.c_int),
                ("stage_begin", ctypes.c_void_p * NUM_STAGES),
                ("stage_end", ctypes.c_void_p * NUM_STAGES), ("cta_pair", ctypes.c_int)]


class moe_plan(ctypes.Structure):
    _fields_ = [("orientation", ctypes.c_int), ("block", ctypes.c_int), ("splits_gemm1", ctypes.c_int),
                ("splits_gemm2", ctypes.c_int), ("act_split", ctypes.c_int), ("kernel_launches", ctypes.c_int),
                ("single_launch", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t), ("cta_pair", ctypes.c_int)]


class moe_cache_stats_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_ulonglong) for n in ("calls", "hits", "misses", "evictions", "bytes_h2d", "passes")]


CACHE_COPY_OVERLAP, CACHE_COPY_SERIAL, CACHE_COPY_KERNEL = 0, 1, 2


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    P, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.moe_strerror.restype = ctypes.c_char_p
    lib.moe_strerror.argtypes = [i]
    lib.moe_version.restype = i
    lib.moe_version.argtypes = []
    lib.moe_workspace_size.restype = i
    lib.moe_workspace_size.argtypes = [i, i, i, i, i, i, i, P, ctypes.POINTER(sz)]
    lib.moe_plan_info.restype = i
    lib.moe_plan_info.argtypes = [i, i, i, i, i, i, i, P, ctypes.POINTER(moe_plan)]
    lib.moe_align_capacity.restype = i
    lib.moe_align_capacity.argtypes = [i, i, i, i, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    lib.moe_route.restype = i
    lib.moe_route.argtypes = [P, P, i, i, i, i, i, i, P, P, P, P]
    lib.moe_topk_from_logits.restype = i
    lib.moe_topk_from_logits.argtypes = [P, i, i, i, i, P, P, P]
    lib.moe_align.restype = i
    lib.moe_align.argtypes = [P, i, i, i, i, P, P, P, P, P]
    lib.moe_forward.restype = i
    lib.moe_forward.argtypes = [P, P, P, P, i, i, i, i, i, i, i, i, P, P, P, P, sz, P, P]
    lib.moe_forward_noalloc.restype = i
    lib.moe_forward_noalloc.argtypes = [P, P, P, P, i, i, i, i, i, i, i, i, P, P, P, P, P]
    lib.moe_forward_host.restype = i
    lib.moe_forward_host.argtypes = [P, P, P, P, P, i, i, i, i, i, i, i, i, P, P, P, P, sz, P, P]
    lib.moe_get_status.restype = i
    lib.moe_get_status.argtypes = [P]
    lib.moe_forward_routed.restype = i
    lib.moe_forward_routed.argtypes = [P, P, P, P, P, i, i, i, i, i, i, i, P, P, P, P, sz, P, P]
    lib.moe_cache_create.restype = i
    lib.moe_cache_create.argtypes = [P, P, P, P, i, i, i, i, i, i, i, ctypes.POINTER(P)]
    lib.moe_cache_destroy.restype = i
    lib.moe_cache_destroy.argtypes = [P]
    lib.moe_cache_set_copy_mode.restype = i
    lib.moe_cache_set_copy_mode.argtypes = [P, i]
    lib.moe_copy_from_host.restype = i
    lib.moe_copy_from_host.argtypes = [P, P, sz, P]
    lib.moe_cache_workspace_size.restype = i
    lib.moe_cache_workspace_size.argtypes = [P, i, i, P, ctypes.POINTER(sz)]
    lib.moe_forward_cached.restype = i
    lib.moe_forward_cached.argtypes = [P, P, P, i, i, i, P, P, sz, P, P]
    lib.moe_cache_stats.restype = i
    lib.moe_cache_stats.argtypes = [P, ctypes.POINTER(moe_cache_stats_t)]
    lib.moe_cache_lru_plan.restype = i
    lib.moe_cache_lru_plan.argtypes = [i, i, i, i, P, P, P, ctypes.POINTER(ctypes.c_ulonglong),
                                       ctypes.POINTER(ctypes.c_ulonglong)]
    lib.moe_inv_rope_fp8_quant.restype = i
    lib.moe_inv_rope_fp8_quant.argtypes = [P, i, i, i, i, P, P, i, P, P, P]
    return lib


_lib = _load()


def lib():
    return _lib


def strerror(code: int) -> str:
    return _lib.moe_strerror(int(code)).decode()


def version() -> int:
    return int(_lib.moe_version())


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise MoeError(rc, where)


def _dt(t: torch.Tensor) -> int:
    return {torch.float32: MOE_F32, torch.bfloat16: MOE_BF16, torch.float8_e4m3fn: MOE_E4M3,
            torch.uint8: MOE_E4M3}[t.dtype]


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _opts(options) -> Optional[ctypes.POINTER(moe_options)]:
    if options is None:
        return None
    if isinstance(options, moe_options):
        return ctypes.byref(options)
    o = moe_options()
    o.orientation = int(options.get("orientation", 0))
    o.split_k = int(options.get("split_k", 0))
    o.inject_timeout = int(options.get("inject_timeout", 0))
    o.act_split = int(options.get("act_split", 0))
    o.single_launch = int(options.get("single_launch", 0))
    o.cta_pair = int(options.get("cta_pair", 0))
    if options.get("trace") is not None:
        o.trace = ctypes.c_void_p(options["trace"].data_ptr())
    for name, ev in (options.get("stage_begin") or {}).items():
        o.stage_begin[STAGES.index(name)] = ctypes.c_void_p(ev.cuda_event)
    for name, ev in (options.get("stage_end") or {}).items():
        o.stage_end[STAGES.index(name)] = ctypes.c_void_p(ev.cuda_event)
    return ctypes.byref(o)


def moe_workspace_size(T: int, H: int, I: int, E: int, topk: int, act_dtype: int, w_dtype: int, options=None) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.moe_workspace_size(T, H, I, E, topk, act_dtype, w_dtype, _opts(options), ctypes.byref(n)),
           "moe_workspace_size")
    return int(n.value)


def moe_plan_info(T: int, H: int, I: int, E: int, topk: int, act_dtype: int, w_dtype: int, options=None) -> dict:
    info = moe_plan()
    _check(_lib.moe_plan_info(T, H, I, E, topk, act_dtype, w_dtype, _opts(options), ctypes.byref(info)),
           "moe_plan_info")
    return {name: getattr(info, name) for name, _ in moe_plan._fields_}


def moe_align_capacity(T: int, topk: int, E: int, block: int):
    a, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(_lib.moe_align_capacity(T, topk, E, block, ctypes.byref(a), ctypes.byref(b)), "moe_align_capacity")
    return int(a.value), int(b.value)


def moe_route(hidden: torch.Tensor, router_w: torch.Tensor, topk: int, renorm: bool, logits=None, topk_w=None,
              topk_ids=None, stream=None):
    """Router logits [T,E] fp32, top-k weights [T,k] fp32 and ids [T,k] int32."""
    T, H = hidden.shape
    E = router_w.shape[0]
    dev = hidden.device
    logits = torch.empty(T, E, dtype=torch.float32, device=dev) if logits is None else logits
    topk_w = torch.empty(T, topk, dtype=torch.float32, device=dev) if topk_w is None else topk_w
    topk_ids = torch.empty(T, topk, dtype=torch.int32, device=dev) if topk_ids is None else topk_ids
    _check(_lib.moe_route(_p(hidden), _p(router_w), T, H, E, topk, int(bool(renorm)), _dt(hidden), _p(logits),
                          _p(topk_w), _p(topk_ids), _stream(stream)), "moe_route")
    return logits, topk_w, topk_ids


def moe_topk_from_logits(logits: torch.Tensor, topk: int, renorm: bool, topk_w=None, topk_ids=None, stream=None):
    T, E = logits.shape
    dev = logits.device
    topk_w = torch.empty(T, topk, dtype=torch.float32, device=dev) if topk_w is None else topk_w
    topk_ids = torch.empty(T, topk, dtype=torch.int32, device=dev) if topk_ids is None else topk_ids
    _check(_lib.moe_topk_from_logits(_p(logits), T, E, topk, int(bool(renorm)), _p(topk_w), _p(topk_ids),
                                     _stream(stream)), "moe_topk_from_logits")
    return topk_w, topk_ids


def moe_align(topk_ids: torch.Tensor, E: int, block: int, stream=None, with_counts: bool = True):
    """(sorted_ids, expert_ids, num_post_pad[1], expert_counts) as full-capacity int32 device tensors."""
    T, k = topk_ids.shape
    cap, bcap = moe_align_capacity(T, k, E, block)
    dev = topk_ids.device
    sorted_ids = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    expert_ids = torch.empty(max(bcap, 1), dtype=torch.int32, device=dev)
    npp = torch.zeros(4, dtype=torch.int32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev) if with_counts else None
    _check(_lib.moe_align(_p(topk_ids), T, k, E, block, _p(sorted_ids), _p(expert_ids), _p(npp), _p(counts),
                          _stream(stream)), "moe_align")
    return sorted_ids, expert_ids, npp[:1], counts


def moe_forward(hidden: torch.Tensor, router_w: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor, topk: int,
                renorm: bool, w13_scale=None, w2_scale=None, out=None, workspace=None, options=None, stream=None,
                w_format=None):
    """One fused MoE layer forward; returns out [T,H] in the activation dtype.

    w_format="int4": w13 [E,2I,H/2] and w2 [E,H,I/2] are packed INT4 codes (uint8) with bf16 group
    scales, group-major per expert: w13_scale [E,H/128,2I] and w2_scale [E,I/128,H]."""
    T, H = hidden.shape
    E, twoI, H2 = w13.shape
    I = twoI // 2
    div = 2 if w_format == "int4" else 1
    if H2 * div != H or w2.shape != (E, H, I // div) or router_w.shape != (E, H):
        raise ValueError("inconsistent shapes")
    act, wdt = _dt(hidden), (MOE_INT4 if w_format == "int4" else _dt(w13))
    opts = _opts(options)
    need = moe_workspace_size(T, H, I, E, topk, act, wdt, options)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=hidden.device)
    out = torch.empty_like(hidden) if out is None else out
    _check(_lib.moe_forward(_p(hidden), _p(router_w), _p(w13), _p(w2), T, H, I, E, topk, int(bool(renorm)), act, wdt,
                            _p(w13_scale), _p(w2_scale), _p(out), _p(workspace), workspace.numel(), opts,
                            _stream(stream)), "moe_forward")
    return out


def moe_forward_host(hidden_host: torch.Tensor, router_w: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor, topk: int,
                     renorm: bool, w13_scale=None, w2_scale=None, hidden_dev=None, out_host=None, workspace=None,
                     options=None, stream=None, w_format=None):
    """The layer from pinned host memory to pinned host memory (moe_forward_host): a copy kernel
    brings hidden_host into the device staging buffer hidden_dev, and the layer stores its output
    straight into out_host, all on `stream`.  Returns out_host, complete once the stream's work is.
    hidden_host and out_host must be page-locked (Tensor.pin_memory())."""
    T, H = hidden_host.shape
    E, twoI, H2 = w13.shape
    I = twoI // 2
    div = 2 if w_format == "int4" else 1
    if H2 * div != H or w2.shape != (E, H, I // div) or router_w.shape != (E, H):
        raise ValueError("inconsistent shapes")
    dev = router_w.device
    act, wdt = _dt(hidden_host), (MOE_INT4 if w_format == "int4" else _dt(w13))
    need = moe_workspace_size(T, H, I, E, topk, act, wdt, options)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    hidden_dev = torch.empty(hidden_host.shape, dtype=hidden_host.dtype, device=dev) if hidden_dev is None else hidden_dev
    out_host = torch.empty(hidden_host.shape, dtype=hidden_host.dtype).pin_memory() if out_host is None else out_host
    _check(_lib.moe_forward_host(_p(hidden_host), _p(hidden_dev), _p(router_w), _p(w13), _p(w2), T, H, I, E, topk,
                                 int(bool(renorm)), act, wdt, _p(w13_scale), _p(w2_scale), _p(out_host),
                                 _p(workspace), workspace.numel(), _opts(options), _stream(stream)),
           "moe_forward_host")
    return out_host


def moe_forward_noalloc(hidden: torch.Tensor, router_w: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor, topk: int,
                        renorm: bool, w13_scale=None, w2_scale=None, out=None, options=None, stream=None,
                        w_format=None):
    """moe_forward without a workspace argument, for callers that cannot allocate device memory.

    The library keeps the workspace in its own fixed device array (NOALLOC_MAX_WORKSPACE bytes per
    device); larger shapes raise MoeError(MOE_ERR_WORKSPACE).  Pass `out` to allocate nothing here either.
    w_format="int4" takes packed INT4 weights as moe_forward does.
    """
    T, H = hidden.shape
    E, twoI, H2 = w13.shape
    I = twoI // 2
    div = 2 if w_format == "int4" else 1
    if H2 * div != H or w2.shape != (E, H, I // div) or router_w.shape != (E, H):
        raise ValueError("inconsistent shapes")
    wdt = MOE_INT4 if w_format == "int4" else _dt(w13)
    out = torch.empty_like(hidden) if out is None else out
    _check(_lib.moe_forward_noalloc(_p(hidden), _p(router_w), _p(w13), _p(w2), T, H, I, E, topk, int(bool(renorm)),
                                    _dt(hidden), wdt, _p(w13_scale), _p(w2_scale), _p(out), _opts(options),
                                    _stream(stream)), "moe_forward_noalloc")
    return out


def moe_get_status(stream=None) -> int:
    return int(_lib.moe_get_status(_stream(stream)))


def moe_inv_rope_fp8_quant(x: torch.Tensor, positions: torch.Tensor, cos_sin: torch.Tensor, rot_dim: int,
                           q_out=None, scale_out=None, stream=None):
    """Inverse rotary embedding + per-head e4m3 quantisation of x [T, heads, head_dim] (bf16):
    (codes uint8 [T, heads, head_dim], scales float32 [T, heads])."""
    T, heads, D = x.shape
    assert x.dtype == torch.bfloat16 and x.is_contiguous()
    dev = x.device
    q_out = torch.empty(T, heads, D, dtype=torch.uint8, device=dev) if q_out is None else q_out
    scale_out = torch.empty(T, heads, dtype=torch.float32, device=dev) if scale_out is None else scale_out
    _check(_lib.moe_inv_rope_fp8_quant(_p(x), T, heads, D, int(rot_dim), _p(positions), _p(cos_sin),
                                       cos_sin.shape[0], _p(q_out), _p(scale_out), _stream(stream)),
           "moe_inv_rope_fp8_quant")
    return q_out, scale_out


def moe_forward_routed(hidden: torch.Tensor, topk_w: torch.Tensor, topk_ids: torch.Tensor, w13: torch.Tensor,
                       w2: torch.Tensor, w13_scale=None, w2_scale=None, out=None, workspace=None, options=None,
                       stream=None):
    """Steps 3-7 of the layer on a given routing (topk_w fp32 [T,k], topk_ids int32 [T,k])."""
    T, H = hidden.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    k = topk_ids.shape[1]
    act, wdt = _dt(hidden), _dt(w13)
    o = dict(options or {})
    o["single_launch"] = 2
    need = moe_workspace_size(T, H, I, E, k, act, wdt, o)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=hidden.device)
    out = torch.empty_like(hidden) if out is None else out
    _check(_lib.moe_forward_routed(_p(hidden), _p(topk_w), _p(topk_ids), _p(w13), _p(w2), T, H, I, E, k, act, wdt,
                                   _p(w13_scale), _p(w2_scale), _p(out), _p(workspace), workspace.numel(), _opts(o),
                                   _stream(stream)), "moe_forward_routed")
    return out


class ExpertCache:
    """Host-resident expert weights with a pool of `n_slots` device slots (moe_cache_* in the C ABI).

    w13 [E,2I,H] and w2 [E,H,I] are CPU tensors (pinned ones avoid a registration); the cache keeps
    references to them for its lifetime.
    """

    def __init__(self, w13: torch.Tensor, w2: torch.Tensor, n_slots: int, max_tokens: int, topk: int, w13_scale=None,
                 w2_scale=None):
        if w13.is_cuda or w2.is_cuda:
            raise ValueError("expert weights must be host tensors")
        E, twoI, H = w13.shape
        self.E, self.H, self.I, self.topk, self.n_slots = E, H, twoI // 2, topk, n_slots
        self._keep = (w13.contiguous(), w2.contiguous(),
                      None if w13_scale is None else w13_scale.float().contiguous(),
                      None if w2_scale is None else w2_scale.float().contiguous())
        h = ctypes.c_void_p(0)
        _check(_lib.moe_cache_create(_p(self._keep[0]), _p(self._keep[1]), _p(self._keep[2]), _p(self._keep[3]), E, H,
                                     self.I, _dt(w13), n_slots, max_tokens, topk, ctypes.byref(h)), "moe_cache_create")
        self._h = h

    def set_copy_mode(self, mode: int) -> None:
        """CACHE_COPY_OVERLAP (default), CACHE_COPY_SERIAL or CACHE_COPY_KERNEL."""
        _check(_lib.moe_cache_set_copy_mode(self._h, int(mode)), "moe_cache_set_copy_mode")

    def close(self):
        if self._h is not None and self._h.value:
            _lib.moe_cache_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace_size(self, T: int, act_dtype: int = MOE_BF16, options=None) -> int:
        n = ctypes.c_size_t(0)
        _check(_lib.moe_cache_workspace_size(self._h, T, act_dtype, _opts(options), ctypes.byref(n)),
               "moe_cache_workspace_size")
        return int(n.value)

    def forward(self, hidden: torch.Tensor, router_w: torch.Tensor, renorm: bool, out=None, workspace=None,
                options=None, stream=None) -> torch.Tensor:
        T = hidden.shape[0]
        if workspace is None:
            workspace = torch.empty(self.workspace_size(T, _dt(hidden), options), dtype=torch.uint8,
                                    device=hidden.device)
        out = torch.empty_like(hidden) if out is None else out
        _check(_lib.moe_forward_cached(self._h, _p(hidden), _p(router_w), T, int(bool(renorm)), _dt(hidden), _p(out),
                                       _p(workspace), workspace.numel(), _opts(options), _stream(stream)),
               "moe_forward_cached")
        return out

    def stats(self) -> dict:
        st = moe_cache_stats_t()
        _check(_lib.moe_cache_stats(self._h, ctypes.byref(st)), "moe_cache_stats")
        return {n: int(getattr(st, n)) for n, _ in moe_cache_stats_t._fields_}


def moe_copy_from_host(src: torch.Tensor, dst: torch.Tensor, stream=None) -> torch.Tensor:
    """The expert cache's copy kernel: src (pinned host tensor) -> dst (device tensor, same bytes)."""
    n = src.numel() * src.element_size()
    if src.is_cuda or not dst.is_cuda or dst.numel() * dst.element_size() != n:
        raise ValueError("src must be a host tensor and dst a device tensor of the same size")
    _check(_lib.moe_copy_from_host(_p(src), _p(dst), n, _stream(stream)), "moe_copy_from_host")
    return dst


def moe_cache_lru_plan(E: int, n_slots: int, ids):
    """The cache's slot policy on a sequence of calls (ids int32 [n_calls, pairs]), host only:
    (slot_ids [n_calls, pairs], loaded_expert [n_calls, n_slots], hits, misses)."""
    import numpy as np

    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    n_calls, pairs = ids.shape
    slot_ids = np.empty_like(ids)
    loaded = np.empty((n_calls, n_slots), dtype=np.int32)
    hits, misses = ctypes.c_ulonglong(0), ctypes.c_ulonglong(0)
    _check(_lib.moe_cache_lru_plan(E, n_slots, n_calls, pairs, ids.ctypes.data_as(ctypes.c_void_p),
                                   slot_ids.ctypes.data_as(ctypes.c_void_p), loaded.ctypes.data_as(ctypes.c_void_p),
                                   ctypes.byref(hits), ctypes.byref(misses)), "moe_cache_lru_plan")
    return slot_ids, loaded, int(hits.value), int(misses.value)
