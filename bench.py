#!/usr/bin/env python3
"""Benchmark of the MXFP4 MoE expert layer at DFlash verification token counts.

Metric: MoE-layer tokens/s at T = 256 (32 sequences x a DFlash block of 8) on the full-shape
layer (H=6144, I=2048, E=384, top-8), plus achieved HBM GB/s as a fraction of the measured
B300 peak.  One JSON line on stdout (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--layer NAME]
                  [--act mxfp8|bf16] [--path auto|multi|persistent]

ours       K forward calls through the C ABI with all inputs resident in HBM (the 7.7 GB of
           packed weights exceed L2, so no L2 flush is needed), timed with CUDA events on the
           launching stream; then the same K calls again with an event before each kernel
           (the per-kernel split and the dominant kernel's duration for the roofline); then
           K end-to-end calls with host buffers (pinned x and logits copied in, y copied out,
           inside the timed region); then µs per layer of every config, hot and with L2
           flushed (rank 0, N = 1); then the CPU oracle on a bounded sample (rank 0, N = 1).
reference  the fp64 CPU oracle on the host cores, each step a bounded sample of the workload.
N > 1      one process per GPU (torchrun); each rank runs an independent replica of the layer
           (the layer needs no exchange on one GPU), value = all ranks' tokens / max time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s at T=256; achieved HBM GB/s as fraction of B300 peak"
UNIT = "tokens/s"
PEAK_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_traffic.txt")
# the sources the GEMM kernels compile from (the DRAM traffic figures stay valid while
# these are unchanged; host-side code does not change a kernel's traffic)
KERNEL_SOURCES = [os.path.join(ROOT, "mxfp4_expert_layer_dflash_b300", "csrc", f)
                  for f in ("combine.cuh", "common.cuh", "fmt.cuh", "gemm_tc.cuh", "grid_sync.cuh",
                            "ptx.cuh", "quant.cuh", "route.cuh", "route_layer.cuh",
                            "route_small.cuh")]
# kernels of one forward in launch order, per execution path
STEP_NAMES = {1: ["route_topk", "route_permute", "act_quant", "gemm1", "gemm2", "combine"],
              2: ["route_topk", "route_permute", "act_quant", "gemm1+gemm2+combine"],
              3: ["route_topk", "route_permute", "act_quant", "gemm1+gemm2", "combine"]}
PATHS = {"auto": 0, "multi": 1, "persistent": 2, "gemms": 3}
PATH_NAMES = {1: "multi", 2: "persistent", 3: "gemms"}
SMALL_ROUTE_TOKENS = 32  # up to this T the first three steps are one kernel, route_act


def step_names(path: int, T: int):
    """Kernels of one forward in launch order: with the whole-layer launch (path 2) a block
    of at most 32 tokens is one kernel; otherwise the first three steps are one kernel for
    such a block."""
    names = STEP_NAMES[path]
    if T <= SMALL_ROUTE_TOKENS:
        return ["layer"] if path == 2 else ["route_act"] + names[3:]
    return names


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(PEAK_FALLBACK), "fallback"


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def read_traffic(kernel: str, layer: str):
    """DRAM bytes per launch of `kernel` on `layer` from the committed ncu summary, or None
    when there is none or the kernel sources changed since it was captured."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    kv = {}
    for line in open(TRAFFIC_FILE):
        line = line.split("#", 1)[0].strip()
        if ":" in line:
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_sha") != kernel_source_sha() or kv.get("layer") != layer:
        return None
    v = kv.get(f"{kernel}_dram_bytes_per_launch")
    return float(v) if v else None


def layer_bytes(L, cnt):
    """Algorithmic bytes: touched experts' packed weights + scales, x, logits and y."""
    touched = int((cnt > 0).sum())
    w13 = 2 * L.I * L.H // 2 + 2 * L.I * L.H // 32
    w2 = L.H * L.I // 2 + L.H * L.I // 32
    act = L.T * L.H * 2 + L.T * L.E * 4 + L.T * L.H * 2
    return touched, touched * w13, touched * w2, touched * (w13 + w2) + act


# ------------------------------------------------------------------------- clocks

class ClockSampler:
    """SM clocks, power and clock-event (throttle) reasons of one GPU, read through NVML by a
    background thread every `period_s` while active, each sample time-stamped, so that the
    samples inside a timed region of a few tens of milliseconds can be picked out
    (`mark_start` / `mark_stop` around it).  Reads only; changes no setting.  Falls back to
    `nvidia-smi -lms 50` when NVML is unavailable."""
    REASONS = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
               "sw_power_cap": 0x4, "hw_power_brake_slowdown": 0x80}
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index: int, period_s: float = 0.002):
        self.cuda_index = cuda_index
        self.period = period_s
        self.samples = []          # (time, sm_mhz, max_mhz, reasons bitmask)
        self.window = None
        self.source = None

    def _nvml(self):
        """NVML through the driver's own library (ctypes; read-only queries), and a handle for
        this process's CUDA device (matched by UUID, else by index)."""
        import torch
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        uuid = str(torch.cuda.get_device_properties(self.cuda_index).uuid)
        for u in (uuid, "GPU-" + uuid):
            if nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0:
                return nv, h
        if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.cuda_index), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        return nv, h

    def _run_nvml(self, nv, h):
        sm_clock = ctypes.c_uint(1)  # NVML_CLOCK_SM
        mx, sm, rs = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
        nv.nvmlDeviceGetMaxClockInfo(h, sm_clock, ctypes.byref(mx))
        reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, sm_clock, ctypes.byref(sm)) == 0 and \
                    reasons(h, ctypes.byref(rs)) == 0:
                self.samples.append((time.perf_counter(), float(sm.value), float(mx.value),
                                     int(rs.value)))
            self._stop.wait(self.period)

    def __enter__(self):
        import threading
        self._stop = threading.Event()
        self.proc = None
        try:
            nv, h = self._nvml()
            self.thread = threading.Thread(target=self._run_nvml, args=(nv, h), daemon=True)
            self.thread.start()
            self.source = f"NVML every {self.period * 1e3:.0f} ms"
        except Exception:  # noqa: BLE001 - no NVML: nvidia-smi at its fastest period
            self.thread = None
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                     "-i", str(self.cuda_index), "-lms", "50"], stdout=subprocess.PIPE,
                    stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi every 50 ms"
            except OSError:
                self.proc = None
        self.t_enter = time.perf_counter()
        return self

    def mark_start(self):
        self.window = [time.perf_counter(), None]

    def mark_stop(self):
        if self.window:
            self.window[1] = time.perf_counter()

    def __exit__(self, *exc):
        self._stop.set()
        if self.thread is not None:
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for l in out.splitlines():
                f = [x.strip() for x in l.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm, mx = float(f[1]), float(f[2])
                except ValueError:
                    continue
                rs = 0
                for n, v in zip(names, f[5:9]):
                    if v.lower() == "active":
                        rs |= self.REASONS[n]
                self.samples.append((None, sm, mx, rs))

    def summary(self):
        """Samples inside the marked timed region (all samples since warm-up began when no
        sample fell inside it, e.g. with the coarse nvidia-smi fallback)."""
        inside = [s for s in self.samples if s[0] is not None and self.window and
                  self.window[0] <= s[0] <= (self.window[1] or s[0])]
        use = inside or self.samples
        sm = [s[1] for s in use]
        mx = max((s[2] for s in use), default=0.0)
        reasons = sorted({n for s in use for n, b in self.REASONS.items() if s[3] & b})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": reasons, "samples": len(sm),
                "window": "timed region" if inside else "warm-up and timed region",
                "source": self.source}


# ------------------------------------------------------------------------- events

class Events:
    """Raw cudaEvent_t handles (the library records step markers into them)."""

    def __init__(self):
        self.rt = ctypes.CDLL("libcudart.so.13")
        self.rt.cudaEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
        self.rt.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p,
                                                 ctypes.c_void_p]
        self.rt.cudaEventDestroy.argtypes = [ctypes.c_void_p]

    def create(self, n):
        arr = (ctypes.c_void_p * n)()
        for i in range(n):
            h = ctypes.c_void_p()
            assert self.rt.cudaEventCreate(ctypes.byref(h)) == 0
            arr[i] = h
        return arr

    def elapsed_ms(self, a, b) -> float:
        ms = ctypes.c_float()
        assert self.rt.cudaEventElapsedTime(ctypes.byref(ms), a, b) == 0
        return float(ms.value)

    def destroy(self, arr):
        for h in arr:
            self.rt.cudaEventDestroy(h)


# ------------------------------------------------------------------------- oracle leg

def _host_packed_weights_parallel(L, quantize, experts):
    """LY.host_packed_weights for `experts`, one host thread per expert at a time (the
    generator and the packing are C calls that release the GIL); same arrays."""
    from concurrent.futures import ThreadPoolExecutor
    from synth import synth as S
    E, H, I = L.E, L.H, L.I
    w13 = np.zeros((E, 2 * I, H // 2), np.uint8)
    s13 = np.zeros((E, 2 * I, H // 32), np.uint8)
    w2 = np.zeros((E, H, I // 2), np.uint8)
    s2 = np.zeros((E, H, I // 32), np.uint8)

    def one(e):
        a = S.normal_f32(L.seed, S.ID_W13, e * 2 * I * H, 2 * I * H, S.W_SIGMA).reshape(2 * I, H)
        w13[e], s13[e] = quantize(a)
        b = S.normal_f32(L.seed, S.ID_W2, e * H * I, H * I, S.W_SIGMA).reshape(H, I)
        w2[e], s2[e] = quantize(b)
    with ThreadPoolExecutor(max_workers=min(16, cpu_cores())) as ex:
        list(ex.map(one, sorted(set(int(v) for v in experts))))
    return w13, s13, w2, s2


def oracle_sample(L, n_tokens: int, act: str = "mxfp8"):
    """Prepare the oracle's inputs for the first n_tokens tokens (packing excluded from any
    timing): returns a closure that runs the oracle on a list of token indices (MXFP8
    emulation for the mxfp8 mode, the exact fp64 layer for the bf16 mode)."""
    from oracle import oracle as O
    from synth import layers as LY
    x, lg = LY.host_x(L), LY.host_logits(L)
    toks = np.arange(min(n_tokens, L.T))
    ridx, _ = O.route(lg[toks], L.k)
    w = _host_packed_weights_parallel(L, O.mxfp4_quantize, np.unique(ridx))

    mode = O.ACT_MXFP8 if act == "mxfp8" else O.ACT_EXACT

    def run(tokens):
        O.moe_forward(x, lg, *w, L.k, mode, tokens=np.asarray(tokens, dtype=np.int64))
    return run, int(np.unique(ridx).size)


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_layer_sample(L, act, n_tokens):
    """(run, description): the oracle over the first n_tokens tokens of layer L, one call per
    step — the same sample in both arms (the whole layer by default)."""
    n = min(n_tokens, L.T)
    run, n_exp = oracle_sample(L, n, act)
    toks = list(range(n))
    mode = "MXFP8-emulation" if act == "mxfp8" else "exact"
    what = "the whole layer" if n == L.T else f"the first {n} of {L.T} tokens"
    return (lambda: run(toks)), n, (f"{what} ({n} tokens, {n_exp} experts) per step, fp64 "
                                    f"oracle in {mode} mode; MXFP4 packing excluded")


def run_reference(args, L, rank):
    if rank != 0:
        return
    log(f"[reference] preparing oracle inputs for {L.name}")
    run, n_tok, sample = oracle_layer_sample(L, args.act, args.cpu_tokens)
    for i in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for i in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = args.steps * n_tok / dt
    cores = cpu_cores()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{L.name}: {L.desc}", "parallelism": "host threads",
                   "act_mode": args.act},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------------- our path

CONFIG_LAYERS = [("c0", "tiny"), ("c1", "mid_t8"), ("c2", "full_t8"), ("c3", "full_t256"),
                 ("c4", "full_t1024_zipf")]


def measure_config(L, steps, flush, flush_dirty):
    """µs per layer of one config: hot (back-to-back forwards, L2 warm) and cold (L2
    emptied before each forward by `flush`; the forward alone is timed with events around
    it; also with the dirty-line flush, for comparison), plus the routing's touched experts.
    The forward is replayed from a CUDA graph so that small layers are not timed by the
    host's enqueue."""
    import torch
    import mxfp4_expert_layer_dflash_b300 as moe
    from synth import layers as LY
    x = torch.from_numpy(LY.host_x(L).view(np.int16)).view(torch.bfloat16).cuda()
    lg = torch.from_numpy(LY.host_logits(L)).cuda()
    w = LY.device_packed_weights(L, moe.mxfp4_quantize)
    y = torch.empty((L.T, L.H), dtype=torch.bfloat16, device="cuda")
    cnt = torch.empty(L.E, dtype=torch.int32, device="cuda")
    aux = [torch.empty(n, dtype=dt, device="cuda") for n, dt in
           ((L.T * L.k, torch.int32), (L.T * L.k, torch.float32), (L.E + 1, torch.int32),
            (L.T * L.k, torch.int32), (L.T * L.k, torch.int32))]
    moe.moe_mxfp4_route(lg, L.T, L.E, L.k, aux[0], aux[1], cnt, *aux[2:])
    touched, _, _, b_layer = layer_bytes(L, cnt.cpu().numpy())

    def fwd():
        moe.moe_mxfp4_forward(x, lg, *w, L.T, L.H, L.I, L.E, L.k, y)

    def fwd_bf16():
        moe.moe_mxfp4_forward_ex(x, lg, *w, L.T, L.H, L.I, L.E, L.k, y,
                                 act_mode=moe.MOE_ACT_BF16)
    run, how = _replayable(fwd)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        run()
    b.record()
    torch.cuda.synchronize()
    hot_us = a.elapsed_time(b) / steps * 1e3
    cold_us, _ = _time_cold(fwd, min(steps, 50), flush)
    dirty_us, _ = _time_cold(fwd, min(steps, 50), flush_dirty)
    bf16_us, _ = _time_cold(fwd_bf16, min(steps, 50), flush)
    if moe.moe_mxfp4_get_status() != 0:
        raise RuntimeError(f"device status error in config {L.name}")
    del w
    torch.cuda.empty_cache()
    return {"layer": L.desc, "touched_experts": touched, "alg_bytes": b_layer,
            "path": PATH_NAMES[moe.moe_mxfp4_select_path(L.T, L.H, L.I, L.E,
                                                                             L.k)],
            "us_hot": hot_us, "us_cold_l2_flushed": cold_us, "flush": flush.desc,
            "us_cold_l2_dirty": dirty_us, "issued_as": how,
            "tokens_per_s_cold": L.T / (cold_us * 1e-6),
            "hbm_gbs_cold": b_layer / (cold_us * 1e-6) / 1e9,
            "bf16_mode_us_cold": bf16_us, "bf16_mode_hbm_gbs_cold": b_layer / (bf16_us * 1e-6) / 1e9}


def _replayable(fn):
    """fn captured once in a CUDA graph (after warm-up calls: scratch grown, one-time set-up
    done), so that timing sees the device work and not the host's enqueue cost of a call of a
    few microseconds; returns (callable, "graph"), or (fn, "eager") if capture fails."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g.replay, "graph"
    except Exception as e:  # noqa: BLE001 - fall back to plain calls, and say so
        log(f"[bench] graph capture failed ({e}); timing plain calls")
        torch.cuda.synchronize()
        return fn, "eager"


class L2Flush:
    """Empties the L2 before a cold-cache call: writes a buffer of twice the L2's size
    (126 MB), then (unless `dirty`) reads another of the same size, so that the call starts
    with none of its data in L2 and with no dirty lines of the flush left, whose write-back it
    would otherwise pay (11-18 µs at the full layer shape: 126 MB of write-back)."""

    def __init__(self, dirty=False):
        import torch
        n = 2 * 126 * 2**20 // 4
        self.w = torch.empty(n, dtype=torch.float32, device="cuda")
        self.r = None if dirty else torch.ones(n, dtype=torch.float32, device="cuda")
        self.acc = torch.zeros(1, dtype=torch.float32, device="cuda")

    def __call__(self):
        import torch
        self.w.add_(1)
        if self.r is not None:
            torch.sum(self.r, dim=0, keepdim=True, out=self.acc)

    @property
    def desc(self):
        return ("252 MB written, then 252 MB read" if self.r is not None
                else "252 MB written (L2 left full of dirty lines)")


def _time_cold(fn, steps, flush):
    """median µs of one call with L2 flushed before each (events around the call only),
    and how the call was issued ("graph" replay or "eager")"""
    import torch
    run, how = _replayable(fn)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for e0, e1 in ev:
        flush()
        e0.record()
        run()
        e1.record()
    torch.cuda.synchronize()
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in ev) * 1e3, how


def measure_next_rows(pk, flush):
    """The steps beside the layer: the router (split-K bf16 GEMM + top-k), the layer with the
    router in front, a dense MXFP8 projection (K = N = 6144), the rejection-sampling
    verification of the drafted block, each against its roofline, and a chain of 4 layers in
    one call against 4 successive calls."""
    import torch
    import mxfp4_expert_layer_dflash_b300 as moe
    from synth import layers as LY
    from synth import synth as S
    hbm = float(pk["hbm_gbs"])
    bf16_tf = float(pk["bf16_tflops"])
    rep = {}
    for T in (8, 256):
        H, E, k = 6144, 384, 8
        x = torch.from_numpy(S.x_bf16(100 + T, T, H).view(np.int16)).view(torch.bfloat16).cuda()
        w = torch.from_numpy(S.router_bf16(100 + T, E, H).view(np.int16)).view(
            torch.bfloat16).cuda()
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
        us, how = _time_cold(lambda: moe.moe_router_topk(x, w, T, H, E, k, idx, gate), 50,
                             flush)
        byt = E * H * 2 + T * H * 2 + T * k * 8
        fl = 2.0 * T * H * E
        rep[f"router_t{T}"] = {
            "shape": f"T={T} H={H} E={E} top-{k}, bf16 router weights", "us_cold": us,
            "issued_as": how,
            "alg_bytes": byt, "hbm_frac": byt / (us * 1e-6) / 1e9 / hbm,
            "tflops": fl / (us * 1e-6) / 1e12, "tensor_frac_bf16": fl / (us * 1e-6) / 1e12 / bf16_tf}
    for T in (8, 256):
        K = N = 6144
        x = torch.from_numpy(S.x_bf16(200 + T, T, K).view(np.int16)).view(torch.bfloat16).cuda()
        wf = torch.empty((N, K), dtype=torch.float32, device="cuda")
        S.dev_fill_normal_f32(200 + T, S.ID_WDENSE, 0, N * K, S.W_SIGMA, wf.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
        codes = torch.empty((N, K), dtype=torch.uint8, device="cuda")
        sc = torch.empty((N, K // 32), dtype=torch.uint8, device="cuda")
        moe.mxfp8_quantize(wf, N, K, codes, sc)
        del wf
        y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
        us, how = _time_cold(lambda: moe.moe_fp8_dense_forward(x, codes, sc, T, K, N, y), 50,
                             flush)
        byt = N * K + N * K // 32 + T * K * 2 + T * N * 2
        fl = 2.0 * T * K * N
        rep[f"dense_fp8_t{T}"] = {
            "shape": f"T={T} K={K} N={N}, MXFP8 weights and activations", "us_cold": us,
            "issued_as": how,
            "alg_bytes": byt, "hbm_frac": byt / (us * 1e-6) / 1e9 / hbm,
            "tflops": fl / (us * 1e-6) / 1e12,
            "tensor_frac_fp8": fl / (us * 1e-6) / 1e12 / (2.0 * bf16_tf)}
    # rejection-sampling verification: 32 sequences (T = 256 verify tokens) x 7 drafts + 1
    Sq, g, V = 32, 7, 152064
    pv, qv, dv, uv, Uv = S.verify_inputs(1, Sq, g, V)
    tens = [torch.from_numpy(a).cuda() for a in (pv, qv, dv, uv)]
    Ut = torch.from_numpy(Uv.view(np.int64)).cuda()
    n_acc = torch.empty(Sq, dtype=torch.int32, device="cuda")
    tok = torch.empty((Sq, g + 1), dtype=torch.int32, device="cuda")
    us, how = _time_cold(lambda: moe.moe_verify_block(*tens, Ut, Sq, g, V, n_acc, tok), 50,
                         flush)
    rows = int(sum(2 if a < g else 1 for a in n_acc.cpu().numpy()))
    byt = rows * V * 4 + Sq * g * 16 + Sq * (g + 2) * 4
    rep["verify_s32_g7"] = {
        "shape": f"S={Sq} sequences x {g} drafted tokens (+1), V={V}; drafter accepting "
                 f"{float(n_acc.float().mean()):.2f} of {g}",
        "us_cold": us, "issued_as": how, "alg_bytes": byt,
        "hbm_frac": byt / (us * 1e-6) / 1e9 / hbm,
        "note": "bytes: the row(s) each sequence's outcome reads (2 after a rejection, else 1)"}
    del tens, pv, qv
    L = LY.LAYERS["full_t256"]
    x = torch.from_numpy(LY.host_x(L).view(np.int16)).view(torch.bfloat16).cuda()
    lg = torch.from_numpy(LY.host_logits(L)).cuda()
    wts = LY.device_packed_weights(L, moe.mxfp4_quantize)
    w_r = torch.from_numpy(S.router_bf16(L.seed, L.E, L.H).view(np.int16)).view(
        torch.bfloat16).cuda()
    y = torch.empty((L.T, L.H), dtype=torch.bfloat16, device="cuda")
    us_r, how = _time_cold(lambda: moe.moe_mxfp4_forward_routed(x, w_r, *wts, L.T, L.H, L.I,
                                                                L.E, L.k, y), 20, flush)
    us_l, _ = _time_cold(lambda: moe.moe_mxfp4_forward(x, lg, *wts, L.T, L.H, L.I, L.E, L.k, y),
                         20, flush)
    rep["routed_layer_t256"] = {"shape": L.desc + ", router in front", "us_cold": us_r,
                                "us_cold_layer_on_given_logits": us_l, "issued_as": how}
    del wts
    torch.cuda.empty_cache()
    # a chain of 4 layers (distinct weights and logits) against 4 successive calls
    for name in ("mid_t8", "full_t8"):
        chain, succ, n, L = _chain_calls(LY.LAYERS[name], 4)
        us_c, how = _time_cold(chain, 20, flush)
        us_s, _ = _time_cold(succ, 20, flush)
        rep[f"chain_{name}_x{n}"] = {
            "shape": f"{n} layers of {L.desc.replace(f' seed={L.seed}', '')}, no residual",
            "us_cold_per_layer_chain": us_c / n, "us_cold_per_layer_successive": us_s / n,
            "speedup": us_s / us_c, "issued_as": how}
        del chain, succ
        torch.cuda.empty_cache()
    if moe.moe_mxfp4_get_status() != 0:
        raise RuntimeError("device status error in the next-rows report")
    return rep


def _chain_calls(L0, n, residual=False):
    """(chain call, n successive calls, n, layer) for n layers shaped like L0 (seeds L0.seed,
    L0.seed + 1, ...), all inputs on the device"""
    import torch
    import mxfp4_expert_layer_dflash_b300 as moe
    from synth import layers as LY
    Ls = [LY.Layer(f"{L0.name}_l{l}", L0.H, L0.I, L0.E, L0.k, L0.T, L0.seed + l)
          for l in range(n)]
    x = torch.from_numpy(LY.host_x(Ls[0]).view(np.int16)).view(torch.bfloat16).cuda()
    lgs = [torch.from_numpy(LY.host_logits(L)).cuda() for L in Ls]
    ws = [LY.device_packed_weights(L, moe.mxfp4_quantize) for L in Ls]
    y = torch.empty((L0.T, L0.H), dtype=torch.bfloat16, device="cuda")
    tmp = [torch.empty_like(y) for _ in range(2)]
    T, H, I, E, k = L0.T, L0.H, L0.I, L0.E, L0.k

    def chain():
        moe.moe_mxfp4_forward_chain(x, lgs, [w[0] for w in ws], [w[1] for w in ws],
                                    [w[2] for w in ws], [w[3] for w in ws], T, H, I, E, k, y,
                                    residual=residual)

    def succ():
        cur = x
        for l in range(n):
            out = y if l == n - 1 else tmp[l & 1]
            moe.moe_mxfp4_forward(cur, lgs[l], *ws[l], T, H, I, E, k, out)
            cur = out
    return chain, succ, n, L0


ROWS = ("router_t8", "router_t256", "dense_fp8_t8", "dense_fp8_t256", "verify_s32_g7",
        "chain_mid_t8_x4")


def run_row(args):
    """One call beside the layer, --warmup then --steps times back to back (a small, fixed
    command for profilers); prints its mean µs.  Not the benchmark's contract line."""
    import torch
    import mxfp4_expert_layer_dflash_b300 as moe
    from synth import synth as S
    name = args.row
    if name.startswith("router"):
        T, H, E, k = int(name[len("router_t"):]), 6144, 384, 8
        x = torch.from_numpy(S.x_bf16(100 + T, T, H).view(np.int16)).view(torch.bfloat16).cuda()
        w = torch.from_numpy(S.router_bf16(100 + T, E, H).view(np.int16)).view(
            torch.bfloat16).cuda()
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
        fn = lambda: moe.moe_router_topk(x, w, T, H, E, k, idx, gate)  # noqa: E731
    elif name.startswith("dense"):
        T, K, N = int(name[len("dense_fp8_t"):]), 6144, 6144
        x = torch.from_numpy(S.x_bf16(200 + T, T, K).view(np.int16)).view(torch.bfloat16).cuda()
        wf = torch.empty((N, K), dtype=torch.float32, device="cuda")
        S.dev_fill_normal_f32(200 + T, S.ID_WDENSE, 0, N * K, S.W_SIGMA, wf.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
        codes = torch.empty((N, K), dtype=torch.uint8, device="cuda")
        sc = torch.empty((N, K // 32), dtype=torch.uint8, device="cuda")
        moe.mxfp8_quantize(wf, N, K, codes, sc)
        del wf
        y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
        fn = lambda: moe.moe_fp8_dense_forward(x, codes, sc, T, K, N, y)  # noqa: E731
    elif name.startswith("chain"):
        from synth import layers as LY
        fn = _chain_calls(LY.LAYERS["mid_t8"], 4)[0]
    else:
        Sq, g, V = 32, 7, 152064
        pv, qv, dv, uv, Uv = S.verify_inputs(1, Sq, g, V)
        tens = [torch.from_numpy(a).cuda() for a in (pv, qv, dv, uv)]
        Ut = torch.from_numpy(Uv.view(np.int64)).cuda()
        n_acc = torch.empty(Sq, dtype=torch.int32, device="cuda")
        tok = torch.empty((Sq, g + 1), dtype=torch.int32, device="cuda")
        fn = lambda: moe.moe_verify_block(*tens, Ut, Sq, g, V, n_acc, tok)  # noqa: E731
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    if moe.moe_mxfp4_get_status() != 0:
        raise RuntimeError(f"device status error in row {name}")
    print(json.dumps({"row": name, "us_per_call_back_to_back": a.elapsed_time(b) / args.steps * 1e3}))


def max_over_ranks(values, dist, device):
    """Element-wise max of per-rank timings over the process group (every rank gets it)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tokens_per_s(world: int, T: int, ms: float) -> float:
    """Whole-job throughput of `world` replicas of a T-token layer finishing in ms (the slowest
    rank's time): every rank's tokens over that time."""
    return world * T / (ms * 1e-3)


def run_ours(args, L, rank, world, local_rank):
    import torch
    import mxfp4_expert_layer_dflash_b300 as moe
    from synth import layers as LY

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    log(f"[rank {rank}] building {L.name} on cuda:{local_rank}")
    x_h, lg_h = LY.host_x(L), LY.host_logits(L)
    x = torch.from_numpy(x_h.view(np.int16)).view(torch.bfloat16).cuda()
    lg = torch.from_numpy(lg_h).cuda()
    w13, s13, w2, s2 = LY.device_packed_weights(L, moe.mxfp4_quantize)
    y = torch.empty((L.T, L.H), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    # routing counts for the byte model (the library's own routing)
    cnt = torch.empty(L.E, dtype=torch.int32, device="cuda")
    tk = [torch.empty(L.T * L.k, dtype=dt, device="cuda")
          for dt in (torch.int32, torch.float32)]
    aux = [torch.empty(n, dtype=torch.int32, device="cuda") for n in (L.E + 1, L.T * L.k,
                                                                       L.T * L.k)]
    moe.moe_mxfp4_route(lg, L.T, L.E, L.k, tk[0], tk[1], cnt, *aux)
    touched, b_gemm1, b_gemm2, b_layer = layer_bytes(L, cnt.cpu().numpy())

    act = moe.MOE_ACT_BF16 if args.act == "bf16" else moe.MOE_ACT_MXFP8
    path = PATHS[args.path] or moe.moe_mxfp4_select_path(L.T, L.H, L.I, L.E, L.k, act)
    names = step_names(path, L.T)
    ev = Events()
    nsteps = len(names) + 1
    marks = [ev.create(nsteps) for _ in range(args.steps)]

    def fwd(step_events=None):
        moe.moe_mxfp4_forward_ex(x, lg, w13, s13, w2, s2, L.T, L.H, L.I, L.E, L.k, y, stream,
                                 act_mode=act, path=path, step_events=step_events)

    clk = ClockSampler(local_rank)
    with clk:       # clocks sampled from the warm-up on; the summary keeps the timed region
        for _ in range(args.warmup):
            fwd()
        if moe.moe_mxfp4_get_status() != 0:
            raise RuntimeError("device status error during warm-up")
        if dist:
            dist.barrier()
        torch.cuda.synchronize()

        # timed region: plain forward calls (event records between kernels cost about a
        # microsecond each, so the per-kernel split comes from a second, marked pass)
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        launches0 = moe.moe_mxfp4_launch_count()
        clk.mark_start()
        start.record(stream)
        for i in range(args.steps):
            fwd()
        stop.record(stream)
        torch.cuda.synchronize()
        clk.mark_stop()
    launches = moe.moe_mxfp4_launch_count() - launches0
    if dist:
        dist.barrier()
    ms = start.elapsed_time(stop) / args.steps
    status = moe.moe_mxfp4_get_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    # marked pass: the same K forwards with an event before each kernel and after the last
    m_start, m_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    m_start.record(stream)
    for i in range(args.steps):
        fwd(marks[i])
    m_stop.record(stream)
    torch.cuda.synchronize()
    marked_ms = m_start.elapsed_time(m_stop) / args.steps
    if moe.moe_mxfp4_get_status() != 0:
        raise RuntimeError("device status error in the marked pass")

    per_step = {n: [] for n in names}
    for m in marks:
        for j, n in enumerate(names):
            per_step[n].append(ev.elapsed_ms(m[j], m[j + 1]))
    step_ms = {n: statistics.mean(v) for n, v in per_step.items()}
    for m in marks:
        ev.destroy(m)

    # end-to-end through the public API with host buffers
    x_pin = torch.from_numpy(x_h.view(np.int16)).view(torch.bfloat16).pin_memory()
    lg_pin = torch.from_numpy(lg_h).pin_memory()
    y_pin = torch.empty((L.T, L.H), dtype=torch.bfloat16).pin_memory()
    h2d = x_pin.numel() * 2 + lg_pin.numel() * 4
    d2h = y_pin.numel() * 2
    for _ in range(args.warmup):
        x.copy_(x_pin, non_blocking=True)
        lg.copy_(lg_pin, non_blocking=True)
        fwd()
        y_pin.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for _ in range(args.steps):
        x.copy_(x_pin, non_blocking=True)
        lg.copy_(lg_pin, non_blocking=True)
        fwd()
        y_pin.copy_(y, non_blocking=True)
    e_stop.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e_start.elapsed_time(e_stop) / args.steps

    # the same steps with the copies on a second stream (independent batches served back to
    # back): each step's inputs go into one of two device buffers while the previous step
    # computes, and its result comes back while the next one computes
    cs = torch.cuda.Stream()
    xb, lgb, yb = [x, torch.empty_like(x)], [lg, torch.empty_like(lg)], [y, torch.empty_like(y)]
    h2d_ev = [torch.cuda.Event(), torch.cuda.Event()]
    done_ev = [torch.cuda.Event(), torch.cuda.Event()]

    def overlapped(n):
        with torch.cuda.stream(cs):
            xb[0].copy_(x_pin, non_blocking=True)
            lgb[0].copy_(lg_pin, non_blocking=True)
            h2d_ev[0].record(cs)
        for i in range(n):
            b = i & 1
            stream.wait_event(h2d_ev[b])
            moe.moe_mxfp4_forward_ex(xb[b], lgb[b], w13, s13, w2, s2, L.T, L.H, L.I, L.E, L.k,
                                     yb[b], stream, act_mode=act, path=path)
            done_ev[b].record(stream)
            with torch.cuda.stream(cs):
                if i + 1 < n:
                    if i >= 1:
                        cs.wait_event(done_ev[1 - b])  # step i-1 no longer reads that buffer
                    xb[1 - b].copy_(x_pin, non_blocking=True)
                    lgb[1 - b].copy_(lg_pin, non_blocking=True)
                    h2d_ev[1 - b].record(cs)
                cs.wait_event(done_ev[b])
                y_pin.copy_(yb[b], non_blocking=True)
        stream.wait_stream(cs)

    overlapped(args.warmup)
    torch.cuda.synchronize()
    o_start, o_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    o_start.record(stream)
    overlapped(args.steps)
    o_stop.record(stream)
    torch.cuda.synchronize()
    e2e_ov_ms = o_start.elapsed_time(o_stop) / args.steps
    if moe.moe_mxfp4_get_status() != 0:
        raise RuntimeError("device status error in the end-to-end passes")

    # max over ranks
    if dist:
        ms, e2e_ms, e2e_ov_ms = max_over_ranks([ms, e2e_ms, e2e_ov_ms], dist, "cuda")
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    pk, pk_src = peaks()
    hbm = float(pk["hbm_gbs"])
    gemm_bytes = {"gemm1": b_gemm1, "gemm2": b_gemm2, "gemm1+gemm2": b_gemm1 + b_gemm2,
                  "gemm1+gemm2+combine": b_gemm1 + b_gemm2, "layer": b_layer}
    dominant = max((n for n in names if n in gemm_bytes), key=lambda n: step_ms[n])
    dom_bytes = gemm_bytes[dominant]
    achieved = dom_bytes / (step_ms[dominant] * 1e-3) / 1e9
    # the committed DRAM figures are those of the MXFP8-mode GEMM kernels
    traffic = read_traffic(dominant, L.name) if args.act == "mxfp8" else None
    layer_gbs = b_layer / (ms * 1e-3) / 1e9

    out = {
        "metric": METRIC, "value": job_tokens_per_s(world, L.T, ms), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e2m1xe4m3->f32" if args.act == "mxfp8" else "e2m1->bf16 x bf16->f32",
        "data": "synthetic",
        "config": {"workload": f"{L.name}: {L.desc}", "global_batch": world * L.T,
                   "seq_len": 8, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (packed weights %.2f GB)" % (b_layer / 1e9),
                   "touched_experts": touched, "act_mode": args.act,
                   "path": PATH_NAMES[path]},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                     "peak_source": f"{pk_src} hbm_gbs", "algorithmic_bytes": dom_bytes},
        "layer_roofline": {"achieved": layer_gbs, "peak": hbm, "unit": "GB/s",
                           "frac": layer_gbs / hbm, "algorithmic_bytes": b_layer,
                           "us_per_layer": ms * 1e3},
        "step_ms": step_ms,
        "marked_pass_ms_per_step": marked_ms,
        "gpu_launches": int(launches),
        "e2e": {"value": job_tokens_per_s(world, L.T, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "e2e_overlapped": {"value": job_tokens_per_s(world, L.T, e2e_ov_ms), "unit": UNIT,
                           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                           "ms_per_step": e2e_ov_ms,
                           "how": "the same copies on a second stream into two device buffers, "
                                  "overlapped with the neighbouring steps' compute"},
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_config_sweep:
        log("[rank 0] measuring every config (hot and L2-flushed)")
        flush, flush_dirty = L2Flush(), L2Flush(dirty=True)
        rep = {}
        for tag, name in CONFIG_LAYERS:
            r = measure_config(LY.LAYERS[name], 200 if LY.LAYERS[name].T < 256 else 50, flush,
                               flush_dirty)
            r["hbm_frac_cold"] = r["hbm_gbs_cold"] / hbm
            Lc = LY.LAYERS[name]
            flops = 2.0 * Lc.T * Lc.k * 3 * Lc.H * Lc.I
            r["tflops_cold"] = flops / (r["us_cold_l2_flushed"] * 1e-6) / 1e12
            # the block-scaled FP4 x FP8 MMA runs at the FP8 rate: 2 x the bf16 peak
            r["tensor_frac_cold"] = r["tflops_cold"] / (2.0 * float(pk["bf16_tflops"]))
            if not args.no_cpu_baseline:  # the oracle on the first 4 tokens (packing untimed)
                n_tok = min(4, Lc.T)
                run, _ = oracle_sample(Lc, n_tok)
                t0 = time.perf_counter()
                run(list(range(n_tok)))
                r["cpu_oracle_tokens_per_s"] = n_tok / (time.perf_counter() - t0)
                r["cpu_oracle_sample"] = f"first {n_tok} tokens, fp64, MXFP8 emulation, {cpu_cores()} cores"
            rep[tag] = r
        out["configs_report_peaks"] = {
            "hbm_gbs": hbm, "fp8_tflops": 2.0 * float(pk["bf16_tflops"]),
            "source": f"{pk_src}: hbm_gbs; bf16_tflops (burst) x 2, the nominal FP8/bf16 ratio"}
        out["configs_report"] = rep
        log("[rank 0] measuring the router, the routed layer and the dense projection")
        out["next_rows"] = measure_next_rows(pk, flush)
        del flush, flush_dirty
    if world == 1 and not args.no_cpu_baseline:
        log("[rank 0] timing the CPU oracle over the layer")
        run, n_tok, sample = oracle_layer_sample(L, args.act, args.cpu_tokens)
        t0 = time.perf_counter()
        run()                     # one step: the same sample the reference arm times per step
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {
            "value": n_tok / dt, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{sample}; one step, {dt:.1f} s"}
    print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layer", default="full_t256")
    ap.add_argument("--path", choices=sorted(PATHS), default="auto")
    ap.add_argument("--act", choices=["mxfp8", "bf16"], default="mxfp8",
                    help="activation mode of the layer (the headline is mxfp8)")
    ap.add_argument("--row", choices=ROWS, default=None,
                    help="only run one call beside the layer (a profiling command)")
    ap.add_argument("--cpu-tokens", type=int, default=1 << 30,
                    help="tokens of the layer the CPU oracle runs per step (default: all)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-config-sweep", action="store_true",
                    help="skip the per-config µs/layer report")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from synth import layers as LY
    L = LY.LAYERS[args.layer]
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.row:
        run_row(args)
    elif args.impl == "reference":
        run_reference(args, L, rank)
    else:
        run_ours(args, L, rank, world, local_rank)


if __name__ == "__main__":
    main()
