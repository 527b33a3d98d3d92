"""Benchmark of the fused MoE layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME] [--no-sweep]

One step is one moe_forward call (router, permutation, gather, GEMM1 with the
SiLU(gate)*up epilogue, GEMM2, combine) on one synthetic token batch with the
weights resident in HBM.  The headline workload is the Mixtral-shaped decode
layer (hidden 4096, 8 experts, FFN 14336, top-2) at M = 64 tokens; a sweep over
the other decode batch sizes, the fine-grained and FP8 decode layers and the
8192-token prefill layer follows in "sweep" (fewer steps each).

Prints ONE JSON line (rank 0).  Under torchrun every rank runs its own replica
on its own GPU (tokens are independent: weak scaling, no collective on the data
path); the timed region is bracketed by a barrier and the max over ranks is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from moe_synth import make_layer, resample_tokens, spec  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
METRIC = "MoE-layer tokens/s; decode weight-stream HBM GB/s, prefill TFLOP/s vs peak"

WORKLOADS = {
    "mixtral_decode_M64": ("mixtral_decode", 64), "mixtral_decode_M16": ("mixtral_decode", 16),
    "mixtral_decode_M4": ("mixtral_decode", 4), "mixtral_decode_M1": ("mixtral_decode", 1),
    "fine_decode_M64": ("fine_decode", 64), "fine_decode_M32": ("fine_decode", 32),
    "fine_decode_M8": ("fine_decode", 8), "fine_decode_M1": ("fine_decode", 1),
    "fp8_decode_M64": ("fp8_decode", 64), "fp8_decode_M16": ("fp8_decode", 16), "fp8_decode_M1": ("fp8_decode", 1),
    "int4_decode_M64": ("int4_decode", 64), "int4_decode_M16": ("int4_decode", 16), "int4_decode_M1": ("int4_decode", 1),
    "prefill_T8192": ("prefill", 8192), "prefill_hot_T8192": ("prefill_hot", 8192),
    "tiny_f32_T64": ("tiny_f32", 64),
}
SWEEP_SKIP = {"tiny_f32_T64"}  # correctness-size fp32 layer: not a throughput workload
HEADLINE = "mixtral_decode_M64"
SINGLE_LAUNCH = {"auto": 0, "on": 1, "off": 2}  # moe_options.single_launch


def max_over_ranks(x: float, world: int, device) -> float:
    """Max of a per-rank number over all ranks (the timing rule: the slowest rank sets the job time)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own batch of tokens_per_rank per step."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------
# algorithmic work of one layer call (from the realised routing)
# ----------------------------------------------------------------------------
def work(sp, n_active: int, act_split: bool):
    # weight bytes per element: e4m3 1, fp32 4, bf16 2, INT4 half a byte plus a 2-byte scale per 128
    wb = {"e4m3": 1.0, "f32": 4.0, "bf16": 2.0, "int4": 0.5 + 2.0 / 128}[sp.w]
    ab = 4 if sp.act == "f32" else 2
    n = sp.T * sp.k
    I, H = sp.I, sp.H
    w13 = int(n_active * 2 * I * H * wb)
    w2 = int(n_active * H * I * wb)
    a_bytes = n * I * (1 if sp.w == "e4m3" else ab * (2 if act_split else 1))
    g1_bytes = w13 + n * H * (1 if sp.w == "e4m3" else ab) + a_bytes
    g2_bytes = w2 + a_bytes + n * H * 4
    layer_bytes = w13 + w2 + sp.E * H * ab + 2 * sp.T * H * ab
    flops1 = 2.0 * n * 2 * I * H
    flops2 = 2.0 * n * H * I
    return {"w13_bytes": w13, "w2_bytes": w2, "gemm1_bytes": g1_bytes, "gemm2_bytes": g2_bytes,
            "layer_bytes": layer_bytes, "gemm1_flops": flops1, "gemm2_flops": flops2,
            "layer_flops": flops1 + flops2 + 2.0 * sp.T * sp.E * H, "bytes_per_active_expert": int(3 * I * H * wb)}


def _sha(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def traffic_from_profiles(kernel: str, workload: str):
    """dram bytes per launch from a committed ncu summary, if the kernel source has not changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    e = d.get(f"{kernel}:{workload}")
    if not e:
        return None
    src = os.path.join(ROOT, "mixture_experts_layer_scan_gb300", "csrc", "moe_gemm_tc.cu")
    if e.get("source_sha") != _sha(src):
        return None
    return e.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                s, m = float(f[1]), float(f[2])
            except ValueError:
                continue
            sm.append(s)
            mx = m
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        loaded = [s for s in sm if s > 0.5 * (mx or max(sm))] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# our implementation
# ----------------------------------------------------------------------------
class L2Flush:
    """Evicts the previous step's data from L2 between timed steps: a 256 MB write (twice L2), then a
    256 MB read of another buffer, so that the write's dirty lines are written back here rather than
    by the timed step that would otherwise evict them."""

    def __init__(self, dev):
        self.wr = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        self.rd = torch.zeros(64 * 1024 * 1024, dtype=torch.int32, device=dev)
        self.sink = torch.zeros((), dtype=torch.int32, device=dev)

    def __call__(self):
        self.wr.zero_()
        torch.amax(self.rd, dim=0, out=self.sink)


def run_ours(args, rank, world, dev):
    import mixture_experts_layer_scan_gb300 as moe

    pk = peaks()
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)  # graph capture needs a non-default stream
    torch.cuda.set_stream(stream)
    flush_buf = L2Flush(dev)
    names = [args.workload] + ([] if args.no_sweep else
                               [w for w in WORKLOADS if w != args.workload and w not in SWEEP_SKIP])
    results = {}
    head = None
    for wi, wname in enumerate(names):
        base, T = WORKLOADS[wname]
        sp = spec(base, T=T)
        L = make_layer(sp, device=dev)
        X, Wr, W13, W2 = L["X"], L["Wr"], L["W13"], L["W2"]
        s13, s2 = L["w13_scale"], L["w2_scale"]
        act = moe.MOE_F32 if sp.act == "f32" else moe.MOE_BF16
        wdt = {"f32": moe.MOE_F32, "bf16": moe.MOE_BF16, "e4m3": moe.MOE_E4M3, "int4": moe.MOE_INT4}[sp.w]
        wfmt = "int4" if sp.w == "int4" else None
        base_opts = {"single_launch": SINGLE_LAUNCH[args.single_launch]}
        plan = moe.moe_plan_info(T, sp.H, sp.I, sp.E, sp.k, act, wdt, base_opts)
        # the two decode paths (one cooperative kernel / the multi-kernel sequence) where both apply
        paths = {}
        for pname, code in (("single_launch", 1), ("multi_kernel", 2)):
            try:
                paths[pname] = moe.moe_plan_info(T, sp.H, sp.I, sp.E, sp.k, act, wdt, {"single_launch": code})
            except moe.MoeError:
                pass
        ws_bytes = max([plan["workspace_bytes"]] + [q["workspace_bytes"] for q in paths.values()])
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        out = torch.empty_like(X)
        # realised routing (the library's own router on the same batch)
        _, _, ids = moe.moe_route(X, Wr, sp.k, sp.renorm)
        n_active = int(torch.unique(ids).numel())
        wk = work(sp, n_active, bool(plan["act_split"]))
        weights_active = wk["w13_bytes"] + wk["w2_bytes"]
        flush = weights_active < 2 * L2_BYTES  # else the step's own inputs exceed L2

        def step(options=None):
            o = dict(base_opts)
            o.update(options or {})
            moe.moe_forward(X, Wr, W13, W2, sp.k, sp.renorm, s13, s2, out=out, workspace=ws, options=o, w_format=wfmt,
                            stream=stream)

        is_head = wi == 0
        K = args.steps if is_head else min(args.steps, args.sweep_steps)
        W = max(3, args.warmup)
        for _ in range(W):
            step()
        torch.cuda.synchronize()
        assert moe.moe_get_status() == 0
        # CUDA graph of one layer call (replayed: no host launch gaps between steps)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            step()
        for _ in range(W):
            graph.replay()
        torch.cuda.synchronize()

        def timed(fn, k, flush_between):
            if not flush_between:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(k):
                    fn()
                e1.record(stream)
                e1.synchronize()
                return e0.elapsed_time(e1)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
            for a, b in evs:
                flush_buf()
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize()
            return sum(a.elapsed_time(b) for a, b in evs)

        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        sampler = ClockSampler(torch.cuda.current_device()) if is_head and rank == 0 else None
        if sampler:
            sampler.__enter__()
        total_ms = timed(graph.replay, K, flush)
        if sampler:
            sampler.__exit__()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        total_ms = max_over_ranks(total_ms, world, dev)
        ms = total_ms / K
        eager_ms = timed(step, min(K, 200), flush) / min(K, 200)
        paths_ms = {}
        if len(paths) == 2:
            for pname, code in (("single_launch", 1), ("multi_kernel", 2)):
                g_alt = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g_alt, stream=stream, capture_error_mode="thread_local"):
                    step({"single_launch": code})
                for _ in range(W):
                    g_alt.replay()
                ka = min(K, 500)
                paths_ms[pname] = timed(g_alt.replay, ka, flush) / ka
                del g_alt
            assert moe.moe_get_status() == 0

        # per-stage durations (CUDA events recorded by the library on this stream)
        kk = min(K, 100)
        stage_ev = []
        for _ in range(kk):
            b = {n: torch.cuda.Event(enable_timing=True) for n in moe.STAGES}
            e = {n: torch.cuda.Event(enable_timing=True) for n in moe.STAGES}
            for ev in list(b.values()) + list(e.values()):
                ev.record(stream)  # torch creates the CUDA event on first record; the library re-records it
            stage_ev.append((b, e))
        for b, e in stage_ev:
            if flush:
                flush_buf()
            step({"stage_begin": b, "stage_end": e})
        torch.cuda.synchronize()
        stage_ms = {n: sum(b[n].elapsed_time(e[n]) for b, e in stage_ev) / kk for n in moe.STAGES}
        assert moe.moe_get_status() == 0

        tok_s = job_tokens_per_s(T, world, ms)
        decode = sp.T <= 64
        g1_ms, g2_ms = stage_ms["gemm1"], stage_ms["gemm2"]
        r = {"tokens_per_s": tok_s, "ms_per_step": ms, "eager_ms_per_step": eager_ms, "active_experts": n_active,
             "plan": plan, "stage_ms": stage_ms, "l2": "flushed between steps (256 MB write + 256 MB read)" if flush else "inputs larger than L2"}
        if paths_ms:
            r["paths_ms_per_step"] = paths_ms
        if decode:
            r["layer_hbm_gbs"] = wk["layer_bytes"] / (ms / 1e3) / 1e9
            r["layer_hbm_frac"] = r["layer_hbm_gbs"] / pk["hbm_gbs"]
            r["gemm1_hbm_gbs"] = wk["gemm1_bytes"] / (g1_ms / 1e3) / 1e9
            r["gemm2_hbm_gbs"] = wk["gemm2_bytes"] / (g2_ms / 1e3) / 1e9
            r["gemm1_frac"] = r["gemm1_hbm_gbs"] / pk["hbm_gbs"]
            r["gemm2_frac"] = r["gemm2_hbm_gbs"] / pk["hbm_gbs"]
        else:
            # steps run back to back for K steps (about half a second at this size), long
            # enough for the part to reach its power cap: fractions of the sustained peak,
            # and of the burst peak alongside
            peak_t = pk["bf16_tflops_sustained"] * (2 if sp.w == "e4m3" else 1)
            peak_b = pk["bf16_tflops"] * (2 if sp.w == "e4m3" else 1)
            r["layer_tflops"] = wk["layer_flops"] / (ms / 1e3) / 1e12
            r["layer_tensor_frac"] = r["layer_tflops"] / peak_t
            r["layer_tensor_frac_burst"] = r["layer_tflops"] / peak_b
            r["gemm1_tflops"] = wk["gemm1_flops"] / (g1_ms / 1e3) / 1e12
            r["gemm2_tflops"] = wk["gemm2_flops"] / (g2_ms / 1e3) / 1e12
            r["gemm1_frac"] = r["gemm1_tflops"] / peak_t
            r["gemm2_frac"] = r["gemm2_tflops"] / peak_t
            r["gemm1_frac_burst"] = r["gemm1_tflops"] / peak_b
            r["gemm2_frac_burst"] = r["gemm2_tflops"] / peak_b
        r["work"] = wk
        results[wname] = r

        if is_head:
            head = dict(r)
            head["spec"] = sp
            head["clocks"] = sampler.summary() if sampler else None
            head["K"], head["W"] = K, W
            # end to end through the C ABI with host buffers (moe_forward_host): the batch
            # read from pinned host memory into the device, the layer, its output stored into
            # pinned host memory, every step, on the timed stream
            Xh = X.cpu().pin_memory()
            outh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
            Xd = torch.empty_like(X)

            def e2e_step():
                moe.moe_forward_host(Xh, Wr, W13, W2, sp.k, sp.renorm, s13, s2, hidden_dev=Xd, out_host=outh,
                                     workspace=ws, options=base_opts, stream=stream, w_format=wfmt)

            for _ in range(W):
                e2e_step()
            torch.cuda.synchronize()
            ke = min(K, 500)
            e2e_ms = timed(e2e_step, ke, False) / ke
            e2e_ms = max_over_ranks(e2e_ms, world, dev)
            head["e2e"] = {"value": job_tokens_per_s(T, world, e2e_ms), "unit": "tokens/s",
                           "api": "moe_forward_host (pinned host batch read by a copy kernel, output stored "
                                  "into pinned host memory by the layer, one stream)",
                           "h2d_bytes_per_step": X.numel() * X.element_size(),
                           "d2h_bytes_per_step": out.numel() * out.element_size()}
            head["cpu_layer"] = (L, sp)
        del L, X, Wr, W13, W2, ws, out, graph
        torch.cuda.empty_cache()
    return head, results, pk


def run_rope(dev, pk, steps=200):
    """The inverse rotary embedding + per-head FP8 quantisation kernel on two head layouts: device time
    per call (CUDA events, L2 flushed before each call: its footprint is below L2) against HBM peak."""
    import mixture_experts_layer_scan_gb300 as moe
    from moe_synth import make_rope_inputs, rope_spec

    stream = torch.cuda.current_stream(dev)
    flush_buf = L2Flush(dev)
    out = {}
    for name in ("gqa_prefill", "mla_decode"):
        d = make_rope_inputs(rope_spec(name), device=dev)
        rs = d["spec"]
        q = torch.empty(rs.T, rs.heads, rs.head_dim, dtype=torch.uint8, device=dev)
        sc = torch.empty(rs.T, rs.heads, dtype=torch.float32, device=dev)

        def call():
            moe.moe_inv_rope_fp8_quant(d["x"], d["pos"], d["cos_sin"], rs.rot_dim, q, sc, stream=stream)

        for _ in range(5):
            call()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            flush_buf()
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize()
        assert moe.moe_get_status() == 0
        us = sum(a.elapsed_time(b) for a, b in evs) / steps * 1e3
        n = rs.T * rs.heads * rs.head_dim
        nbytes = n * 2 + n + rs.T * rs.heads * 4 + rs.T * 4 + rs.T * rs.rot_dim * 4
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {"us_per_call": us, "algorithmic_bytes": nbytes, "hbm_gbs": gbs, "frac": gbs / pk["hbm_gbs"],
                     "shape": {"T": rs.T, "heads": rs.heads, "head_dim": rs.head_dim, "rot_dim": rs.rot_dim},
                     "l2": "flushed before each call (256 MB write + 256 MB read)"}
    return out


def run_offload(dev, steps=48, warm=8, slots=48, M=8, M_big=64, steps_big=12):
    """The expert cache on the fine-grained decode layer (128 experts of 9.4 MB, all in pinned host
    memory; `slots` of them in HBM): a sequence of Zipf-routed batches, each call timed end to end
    (routing, the host read-back and slot plan, the copies of missing experts, the expert steps), in
    each copy mode, against the same batches with every expert resident; then M_big-token batches,
    which need more experts than slots (passes).  Also the host -> device copy bandwidth of one
    expert's weights by the copy engine (pinned cudaMemcpyAsync) and by the cache's copy kernel."""
    import mixture_experts_layer_scan_gb300 as moe

    sp = spec("fine_decode", T=M_big)
    L = make_layer(sp, device="cpu")
    w13h, w2h = L["W13"].pin_memory(), L["W2"].pin_memory()
    W13, W2, Wr = L["W13"].to(dev), L["W2"].to(dev), L["Wr"].to(dev)

    def batches(T, n, seed0):
        out = []
        for b in range(n):
            resample_tokens(L, torch.arange(M_big), seed0 + b)
            out.append(L["X"][:T].contiguous().to(dev))
        return out

    small = batches(M, warm + steps, 7000)
    big = batches(M_big, 2 + steps_big, 9000)
    res = {"workload": f"fine_decode_M{M}", "experts": sp.E, "expert_mb": round((3 * sp.H * sp.I * 2) / 2 ** 20, 2),
           "slots": slots, "steps": steps,
           "timing": "host wall clock per call, eager (the cached call synchronises on its routing)"}

    def run_cached(mode, xs, n_warm, T):
        cache = moe.ExpertCache(w13h, w2h, n_slots=slots, max_tokens=M_big, topk=sp.k)
        cache.set_copy_mode(mode)
        ws = torch.empty(cache.workspace_size(T), dtype=torch.uint8, device=dev)
        out = torch.empty(T, sp.H, dtype=torch.bfloat16, device=dev)
        for X in xs[:n_warm]:
            cache.forward(X, Wr, sp.renorm, out=out, workspace=ws)
        torch.cuda.synchronize()
        st0 = cache.stats()
        t0 = time.perf_counter()
        for X in xs[n_warm:]:
            cache.forward(X, Wr, sp.renorm, out=out, workspace=ws)
        torch.cuda.synchronize()
        ms = (time.perf_counter() - t0) / (len(xs) - n_warm) * 1e3
        st1 = cache.stats()
        assert moe.moe_get_status() == 0
        cache.close()
        d = {k: st1[k] - st0[k] for k in st1}
        return ms, d

    def run_resident(xs, n_warm, T):
        wsr = torch.empty(moe.moe_workspace_size(T, sp.H, sp.I, sp.E, sp.k, moe.MOE_BF16, moe.MOE_BF16),
                          dtype=torch.uint8, device=dev)
        out = torch.empty(T, sp.H, dtype=torch.bfloat16, device=dev)
        for X in xs[:n_warm]:
            moe.moe_forward(X, Wr, W13, W2, sp.k, sp.renorm, out=out, workspace=wsr)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for X in xs[n_warm:]:
            moe.moe_forward(X, Wr, W13, W2, sp.k, sp.renorm, out=out, workspace=wsr)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / (len(xs) - n_warm) * 1e3

    def median_of_3(fn):
        # host-clock timings wander with the host (the cached call waits on its routing):
        # three repetitions, the median reported
        runs = sorted((fn() for _ in range(3)), key=lambda r: r[0] if isinstance(r, tuple) else r)
        return runs[1]

    modes = {"overlap": moe.CACHE_COPY_OVERLAP, "serial": moe.CACHE_COPY_SERIAL, "copy_kernel": moe.CACHE_COPY_KERNEL}
    res["timing"] += ", median of 3 repetitions"
    res["resident_ms_per_call"] = median_of_3(lambda: run_resident(small, warm, M))
    res["resident_tokens_per_s"] = M / (res["resident_ms_per_call"] * 1e-3)
    for name, mode in modes.items():
        try:
            ms, d = median_of_3(lambda: run_cached(mode, small, warm, M))
        except moe.MoeError as e:
            res[f"cached_{name}"] = {"unavailable": str(e)}
            continue
        distinct = d["hits"] + d["misses"]
        res[f"cached_{name}"] = {"ms_per_call": ms, "tokens_per_s": M / (ms * 1e-3),
                                 "hit_rate": d["hits"] / max(1, distinct), "misses_per_call": d["misses"] / steps,
                                 "h2d_bytes_per_call": d["bytes_h2d"] / steps}
    ms, d = median_of_3(lambda: run_cached(moe.CACHE_COPY_OVERLAP, big, 2, M_big))
    rb = median_of_3(lambda: run_resident(big, 2, M_big))
    res[f"fine_decode_M{M_big}"] = {"cached_ms_per_call": ms, "resident_ms_per_call": rb,
                                    "cached_tokens_per_s": M_big / (ms * 1e-3), "passes_per_call": d["passes"] / steps_big,
                                    "misses_per_call": d["misses"] / steps_big,
                                    "h2d_bytes_per_call": d["bytes_h2d"] / steps_big, "copy_mode": "overlap"}
    # host -> device copy bandwidth of one expert's weights, both methods
    src = torch.cat([w13h[0].flatten(), w2h[0].flatten()]).pin_memory()
    dst = torch.empty_like(src, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        dst.copy_(src, non_blocking=True)
    e0.record()
    for _ in range(20):
        dst.copy_(src, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    res["h2d_gbs_copy_engine"] = 20 * src.numel() * 2 / (e0.elapsed_time(e1) * 1e-3) / 1e9
    for _ in range(3):
        moe.moe_copy_from_host(src, dst)
    e0.record()
    for _ in range(20):
        moe.moe_copy_from_host(src, dst)
    e1.record()
    torch.cuda.synchronize()
    res["h2d_gbs_copy_kernel"] = 20 * src.numel() * 2 / (e0.elapsed_time(e1) * 1e-3) / 1e9
    return res


def cpu_baseline(L, sp, budget_s=20.0):
    """The CPU oracle, as it stands, on a bounded token sample of the workload: on all host cores, and
    single-threaded on a smaller sample."""
    import oracle

    all_cores = len(os.sched_getaffinity(0))
    cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}

    def timed(threads, n):
        oracle.set_threads(threads)
        t0 = time.perf_counter()
        oracle.moe_forward(cpu["X"], cpu["Wr"], cpu["W13"], cpu["W2"], sp.k, sp.renorm, cpu["w13_scale"],
                           cpu["w2_scale"], tokens=list(range(n)))
        return time.perf_counter() - t0

    oracle.set_threads(all_cores)
    cores = oracle.get_threads()
    n = min(sp.T, max(1, 2 * cores))
    dt = timed(cores, n)
    n1 = min(sp.T, 2)
    dt1 = timed(1, n1)
    oracle.set_threads(all_cores)
    return {"value": n / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of the {sp.T} tokens of the batch (full layer weights, routing of all {sp.T} tokens), "
                      f"{dt:.1f} s on {cores} threads",
            "single_thread": {"value": n1 / dt1, "unit": "tokens/s", "cores": 1,
                              "sample": f"{n1} of the {sp.T} tokens, {dt1:.1f} s on 1 thread"}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--sweep-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--single-launch", default="auto", choices=sorted(SINGLE_LAUNCH),
                    help="decode batches: the whole layer as one cooperative kernel (on), the multi-kernel "
                         "sequence (off), or the library's choice (auto)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count (smaller cases for profiling)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.tokens:
        WORKLOADS[args.workload] = (WORKLOADS[args.workload][0], args.tokens)
    base, T = WORKLOADS[args.workload]
    sp = spec(base, T=T)
    config = {"workload": args.workload, "tokens": T, "hidden": sp.H, "experts": sp.E, "intermediate": sp.I,
              "topk": sp.k, "renorm": sp.renorm, "weights": sp.w, "activations": sp.act}

    if args.impl == "reference":
        if world > 1 and rank != 0:
            return
        import oracle

        oracle.build()
        L = make_layer(sp, device="cuda" if torch.cuda.is_available() else "cpu")
        oracle.set_threads(len(os.sched_getaffinity(0)))
        cores = oracle.get_threads()
        cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}
        n = min(T, max(1, cores))
        tokens = list(range(n))

        def ref_step():
            oracle.moe_forward(cpu["X"], cpu["Wr"], cpu["W13"], cpu["W2"], sp.k, sp.renorm, cpu["w13_scale"],
                               cpu["w2_scale"], tokens=tokens)

        steps, warm = min(args.steps, 5), min(max(args.warmup, 0), 1)
        for _ in range(warm):
            ref_step()
        t0 = time.perf_counter()
        for _ in range(steps):
            ref_step()
        dt = (time.perf_counter() - t0) / steps
        v = n / dt
        sample = f"{n} of the {T} tokens per step, {steps} timed steps (full weights), {cores} threads"
        print(json.dumps({"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1,
                          "steps": steps, "warmup": warm, "ms_per_step": dt * 1e3, "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                          "config": config,
                          "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                           "sample": sample},
                          "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}))
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local)
    head, results, pk = run_ours(args, rank, world, dev)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    hsp = head["spec"]
    decode = hsp.T <= 64
    wk = head["work"]
    if decode:
        roof = {"kernel": "k_gemm_tc (GEMM1, w13 + SiLU(gate)*up)", "bound": "hbm",
                "achieved": head["gemm1_hbm_gbs"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": head["gemm1_frac"], "peak_source": pk["source"] + " (hbm_gbs)",
                "algorithmic_bytes_per_launch": wk["gemm1_bytes"],
                "per_unit": f"{2 * hsp.I * hsp.H * 2} B of w13 per active expert x {head['active_experts']} active"}
    else:
        roof = {"kernel": "k_gemm_pair (GEMM1, CTA pairs)" if head["plan"].get("cta_pair") else "k_gemm_tc (GEMM1)",
                "bound": "tensor", "achieved": head["gemm1_tflops"],
                "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s", "frac": head["gemm1_frac"],
                "frac_of_burst": head["gemm1_frac_burst"],
                "peak_source": pk["source"] + " (bf16_tflops_sustained: back-to-back steps reach the power cap; "
                                              "frac_of_burst against bf16_tflops)"}
    roof["traffic"] = traffic_from_profiles("gemm1", args.workload)
    line = {"metric": METRIC, "value": head["tokens_per_s"], "unit": "tokens/s", "n_gpus": world, "steps": head["K"],
            "warmup": head["W"], "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if hsp.act == "bf16" and hsp.w == "bf16" else hsp.w,
            "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights, random-init Mixtral-shaped experts)",
            "config": dict(config, l2=head["l2"], launch="CUDA graph of one moe_forward call",
                           eager_ms_per_step=head["eager_ms_per_step"], plan=head["plan"],
                           active_experts=head["active_experts"]),
            "roofline": roof,
            "layer": {"hbm_gbs": head.get("layer_hbm_gbs"), "frac": head.get("layer_hbm_frac"),
                      "algorithmic_bytes": wk["layer_bytes"]} if decode else
                     {"tflops": head.get("layer_tflops"), "frac": head.get("layer_tensor_frac"),
                      "frac_of_burst": head.get("layer_tensor_frac_burst")},
            "stage_ms": head["stage_ms"], "clocks": head["clocks"], "e2e": head["e2e"],
            "gpu_launches": head["plan"]["kernel_launches"] * head["K"]}
    if not args.no_cpu_baseline:
        L, csp = head["cpu_layer"]
        line["cpu_baseline"] = cpu_baseline(L, csp)
    sweep = {}
    for name, r in results.items():
        if name == args.workload:
            continue
        keep = {k: v for k, v in r.items() if k not in ("work", "plan")}
        keep["stage_ms"] = {k: round(v, 4) for k, v in r["stage_ms"].items()}
        sweep[name] = keep
    if sweep:
        line["sweep"] = sweep
    if not args.no_sweep:
        line["inv_rope_fp8"] = run_rope(dev, pk)
        line["expert_offload"] = run_offload(dev)
    print(json.dumps(line, default=float))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
