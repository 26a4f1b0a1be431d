"""Benchmark of the KDA layer core on GB300.

One JSON line on rank 0.  A step is one ``kda_prefill`` call on the
K3-shaped layer workload (B=1, H=96, T=4096, d_k=d_v=128, bf16 q/k/v/beta/
gate, fp32 log alpha and states, gated RMSNorm output): every prefill row of
the hot path (prologue, decay rescale, Gram, UT solve, W/U, state chain,
output, epilogue).  ``value`` is prefill tokens/s over all ranks with inputs
resident in HBM; the one-token decode step (64 sequences x 96 heads, state in
place) is measured in the same run and reported under ``decode``, and so are
the varlen prefill (8 packed sequences of 1,024..16,384 tokens) and the
decay-extreme prefill (T = 262,144), under ``prefill_varlen`` and
``prefill_extreme``.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--legs prefill,e2e,decode,varlen,extreme]

Multi-GPU runs are independent replicas (the path has no exchange step): each
rank runs the same workload, ``value`` = total tokens / max-over-ranks time.
``--impl reference`` times the CPU oracle on a bounded sample of the same
workload on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA tokens/s (prefill, decode) on 1 GB300; % tensor-core / % HBM roofline"
WORKLOAD = "k3-prefill: B=1, H=96, T=4096, d_k=d_v=128, bf16 q/k/v/beta/gate, fp32 log-alpha " \
           "and state, gated per-head RMSNorm output"
H, T, D = 96, 4096, 128
# algorithmic bytes per (token, head): q, k, v, gate, y (bf16, 256 B each),
# log alpha (fp32, 512 B), beta (bf16, 2 B); plus the state read and written once
BYTES_PER_TOKEN_HEAD = 5 * 2 * D + 4 * D + 2
STATE_BYTES = 4 * D * D
DEC_N, DEC_STEPS = 64, 256
WS_BLOCK_BYTES = 74240  # tensor-core path: workspace block per (64-token chunk, head)
# decode: state read + write per (sequence, head) and the token's inputs/outputs
DEC_BYTES_PER_UNIT = 2 * STATE_BYTES + 4 * 2 * D + 4 * D + 2


def prefill_bytes(T_=T, H_=H, N_=1, s0=True):
    """Method bytes of one call: 1,794 B per (token, head), and per (sequence,
    head) the state written once, and read once when an initial state is given."""
    return BYTES_PER_TOKEN_HEAD * T_ * H_ + (2 if s0 else 1) * STATE_BYTES * H_ * N_


def prefill_flops(chunk: int, T_=T, H_=H, d=D):
    """Algorithmic flops of the chunked form per call: 6 d^2 + 4 C d + C^2/3
    per (token, head) (triangle-aware count of the chunk algebra)."""
    return (6 * d * d + 4 * chunk * d + chunk * chunk / 3.0) * T_ * H_


def code_sha16(path: str) -> str:
    """Hash of a source file's code: comments and whitespace stripped, so that
    an edit of a comment does not count as a change of the kernel."""
    with open(path) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    src = re.sub(r"\s+", "", src)
    return hashlib.sha256(src.encode()).hexdigest()[:16]


def measured_traffic() -> dict:
    """DRAM bytes (read + write) per launch of each kernel, from the ncu
    summaries under profiles/: lines of the form

        traffic: kernel=<name> bytes_per_launch=<B> source=<file> code_sha16=<h>

    An entry counts only while the kernel's source file still has the code it
    had when the counters were taken (same code_sha16); otherwise the kernel
    has changed since, and its traffic is unknown (None)."""
    out = {}
    for fn in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(fn) as f:
            for line in f:
                if not line.startswith("traffic:"):
                    continue
                kv = dict(t.split("=", 1) for t in line.split()[1:] if "=" in t)
                src = os.path.join(ROOT, kv.get("source", ""))
                if os.path.isfile(src) and code_sha16(src) == kv.get("code_sha16"):
                    out[kv["kernel"]] = float(kv["bytes_per_launch"])
    return out


def kernel_plan(path: str, chunk: int, T_=T, H_=H, N_=1, chunks=None):
    """(kernel, roofline bound, method bytes, algorithmic flops, workspace bytes)
    per launch of one prefill call, in launch order.  Method bytes are the
    method's own inputs and outputs that the kernel reads or writes (the
    1,794 B per token and head of the call, and the states); the workspace the
    tensor-core path passes from its second kernel to its third is counted
    apart."""
    if path == "simt":
        return [("prefill_simt_kernel<128,bf16>", "hbm", prefill_bytes(T_, H_, N_),
                 prefill_flops(16, T_, H_), 0)]
    if path == "tc":
        nck = chunks if chunks is not None else (T_ // chunk) * H_
        ws = WS_BLOCK_BYTES * nck
        # prep reads q, k, v, log alpha and beta; chain reads the gate, writes y
        # and reads S0 / writes S_T
        prep_b = (3 * 2 * D + 4 * D + 2) * T_ * H_
        chain_b = 2 * 2 * D * T_ * H_ + 2 * STATE_BYTES * H_ * N_
        # tensor-core flops issued per (chunk, head): Gram 3 x 4 x (128x16x128);
        # U~ 2 x (128x64x64) (T as a bf16 hi/lo pair); W 128x128x64.  Chain:
        # [D | O] 128x128x128, S += U K^ 128x128x64, O += U P^T 128x64x64
        prep_f = (3 * 4 * 2 * 128 * 16 * 128 + 2 * 2 * 128 * 64 * 64
                  + 2 * 128 * 128 * 64) * nck
        chain_f = (2 * 128 * 128 * 128 + 2 * 128 * 128 * 64 + 2 * 128 * 64 * 64) * nck
        return [("chunk_base_kernel", "hbm", 4 * 2 * N_, 0.0, 0),
                ("prep_kernel", "hbm", prep_b, prep_f, ws),
                ("chain_kernel", "hbm", chain_b, chain_f, ws)]
    raise ValueError(f"no kernel plan for path {path}")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "src": "fallback"}


# ------------------------------------------------------------------ dist
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world):
    if world <= 1:
        return None
    import torch.distributed as dist
    backend = "nccl" if __import__("torch").cuda.is_available() else "gloo"
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch
    dev = torch.device("cuda") if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # the raw samples: KDA_CLOCK_LOG_DIR if set (to keep them), else a temp dir
        log_dir = os.environ.get("KDA_CLOCK_LOG_DIR") or tempfile.gettempdir()
        self.path = os.path.join(log_dir, f"clocks_gpu{index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(nm)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["no samples"]}
        loaded = [s for s in sms if s > 0.5 * max(sms)]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sms)}


class NvmlSampler:
    """SM clock and clock-event reasons read through NVML (the driver's
    libnvidia-ml, by ctypes) every ~1 ms from a thread, so that even a
    millisecond-long timed region is sampled; nvidia-smi cannot sample faster
    than its loop interval.  Reads only."""

    # NVML clock-event reason bits (nvml.h): the ones a measurement is checked for
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, index: int):
        import ctypes
        import threading
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._lib = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            self._h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self._h)) != 0:
                return
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(self._h, ctypes.c_int(1), ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self._lib = lib
        except (OSError, AttributeError):
            self._lib = None

    def _run(self):
        import ctypes
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self._lib.nvmlDeviceGetClockInfo(self._h, ctypes.c_int(1), ctypes.byref(clk)) == 0 \
                    and self._reasons_fn(self._h, ctypes.byref(rs)) == 0:
                self.samples.append((float(clk.value), int(rs.value)))
            time.sleep(0.001)

    def __enter__(self):
        import threading
        if self._lib is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return None
        loaded = [c for c, _ in self.samples if c > 0.5 * max(c for c, _ in self.samples)]
        reasons = sorted({nm for _, r in self.samples for bit, nm in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples), "source": "nvml, ~1 ms"}


# ------------------------------------------------------------------ our arm
N_UP = 4  # host->device copy streams of the end-to-end leg
LEGS = ("prefill", "e2e", "decode", "varlen", "extreme")


def time_prefill(inp, args, stream, dist, *, steps, warmup, max_seqlen=0, clocks=False):
    """Device time of one kda_prefill call on `inp` (inputs resident in HBM):
    `warmup` untimed calls, then `steps` calls between CUDA events on the
    launching stream, a barrier and a synchronise on both sides; then the
    per-kernel times from events the library records around each of its
    kernels, over a second pass of the same calls."""
    import torch

    from linear_attention_recurrence_prefill_gb300 import kda

    dev = inp.q.device
    N = inp.N
    o = torch.empty_like(inp.q)
    S_T = torch.empty((N, inp.H, D, D), dtype=torch.float32, device=dev)
    o_opts = kda.kda_options_init(impl=kda.IMPLS[args.path], max_seqlen=max_seqlen)
    ws_bytes = kda.kda_prefill_workspace_size(inp.T, N, inp.H, D, D, o_opts)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    path, launches, chunk = kda.kda_prefill_path(inp.T, N, inp.H, D, D, kda.KDA_BF16, o_opts)

    def call(events=None):
        kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0, inp.cu_seqlens, N,
                        o, S_T, gate=inp.gate, impl=args.path, max_seqlen=max_seqlen,
                        workspace=ws if ws_bytes else None, phase_events=events)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    if kda.kda_get_last_error() != kda.KDA_OK:
        raise RuntimeError(f"device status word set during the {inp.name} warm-up")
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(torch.cuda.current_device()) if clocks else None
    nv = NvmlSampler(torch.cuda.current_device()) if clocks else None
    if clk:
        clk.__enter__()
    try:
        barrier(dist)
        torch.cuda.synchronize()
        if nv:
            nv.__enter__()
        ev0.record(stream)
        for _ in range(steps):
            call()
        ev1.record(stream)
        torch.cuda.synchronize()
        if nv:
            nv.__exit__(None, None, None)
        barrier(dist)
    finally:
        if nv:
            nv.__exit__(None, None, None)
        if clk:
            clk.__exit__(None, None, None)
    ms = max_over_ranks(dist, ev0.elapsed_time(ev1) / steps)
    per = [[torch.cuda.Event(enable_timing=True) for _ in range(launches + 1)]
           for _ in range(steps)]
    for evs in per:        # torch creates the CUDA event on first record
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    for evs in per:
        call(evs)
    torch.cuda.synchronize()
    if kda.kda_get_last_error() != kda.KDA_OK:
        raise RuntimeError(f"device status word set during the {inp.name} calls")
    kern = []
    for i in range(launches):
        kern.append(statistics.mean(evs[i].elapsed_time(evs[i + 1]) for evs in per))
    del ws, o, S_T
    # the tensor-core path skips its first kernel (chunk bases) for equal lengths
    launched = launches - (1 if path == "tc" and inp.cu_seqlens is None else 0)
    return dict(ms=ms, path=path, chunk=chunk, launches=launches, launched=launched,
                kernel_ms=kern, ws_bytes=ws_bytes,
                clocks=((nv.summary() if nv else None) or clk.summary()) if clk else None)


def prefill_leg(inp, args, stream, dist, peaks, *, steps, warmup, max_seqlen=0):
    """Tokens/s and the HBM fraction on the method's bytes for one workload."""
    lens = inp.meta.get("lengths") or [inp.T // inp.N] * inp.N
    r = time_prefill(inp, args, stream, dist, steps=steps, warmup=warmup, max_seqlen=max_seqlen)
    tokens = inp.T
    nbytes = prefill_bytes(tokens, inp.H, inp.N, s0=inp.S0 is not None)
    chunks = sum((L + r["chunk"] - 1) // r["chunk"] for L in lens) * inp.H \
        if r["path"] == "tc" else None
    plan = kernel_plan(r["path"], r["chunk"], tokens, inp.H, inp.N, chunks)
    return {"workload": inp.name, "tokens": tokens, "sequences": inp.N, "steps": steps,
            "warmup": warmup, "ms_per_step": r["ms"],
            "value": tokens * int(os.environ.get("WORLD_SIZE", "1")) / (r["ms"] / 1e3),
            "unit": "tokens/s", "method_bytes": nbytes,
            "hbm_frac": nbytes / (r["ms"] / 1e3) / 1e9 / peaks["hbm_gbs"],
            "kernel_ms": {plan[i][0]: r["kernel_ms"][i] for i in range(r["launches"])},
            "path": r["path"], "chunk": r["chunk"]}


def run_ours(args, rank, world, local, dist):
    import torch

    from linear_attention_recurrence_prefill_gb300 import inputs, kda

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    traffic = measured_traffic()
    kda.load()
    legs = set(args.legs.split(","))
    stream = torch.cuda.current_stream()
    line = {}

    # --- the K3-shaped prefill: the headline number (inputs resident; 688 MB
    # of token inputs per step, larger than L2) ---
    inp = inputs.k3(dev)
    r = time_prefill(inp, args, stream, dist, steps=args.steps, warmup=args.warmup, clocks=True)
    ms_max, path, chunk, launches = r["ms"], r["path"], r["chunk"], r["launches"]
    kernels = kernel_plan(path, chunk)
    assert len(kernels) == launches, (kernels, launches)
    kern_ms = {kernels[i][0]: r["kernel_ms"][i] for i in range(launches)}
    dom_i = max(range(launches), key=lambda i: r["kernel_ms"][i])
    dom, dom_bound, dom_method_bytes, dom_flops, dom_ws = kernels[dom_i]
    dom_ms = r["kernel_ms"][dom_i]
    call_bytes = prefill_bytes()
    # the roofline of the dominant kernel on the method's bytes of the whole
    # call: every kernel of the call exists to move those bytes, so this is
    # the fraction of HBM the call would reach if it took the dominant
    # kernel's time
    achieved = call_bytes / (dom_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": traffic.get(dom), "kernel": dom,
            "kernel_ms": dom_ms, "algorithmic_bytes": call_bytes,
            "kernel_method_bytes": dom_method_bytes,
            "kernel_method_frac": dom_method_bytes / (dom_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
            "workspace_bytes": dom_ws,
            "workspace_note": "operand blocks the tensor-core path writes in its second kernel "
                              "and reads in its third (not method bytes)",
            "tensor_tflops": dom_flops / (dom_ms / 1e3) / 1e12,
            "tensor_frac": dom_flops / (dom_ms / 1e3) / 1e12 / peaks["bf16_tflops"],
            "peak_src": "of measured (MEASURED_PEAKS.json, burst)"
            if peaks["src"] == "measured" else "of fallback"}
    tokens = T * world
    line.update({
        "metric": METRIC, "value": tokens / (ms_max / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": world, "seq_len": T, "heads": H,
                   "head_dim": D, "parallelism": f"replicas x{world}" if world > 1 else "single",
                   "path": path, "chunk": chunk,
                   "l2": "inputs larger than L2 (688 MB of token inputs per step)"},
        "prefill": {"hbm_gbs_algorithmic": call_bytes / (ms_max / 1e3) / 1e9,
                    "hbm_frac": call_bytes / (ms_max / 1e3) / 1e9 / peaks["hbm_gbs"],
                    "tflops_algorithmic": prefill_flops(chunk) / (ms_max / 1e3) / 1e12,
                    "kernel_ms": kern_ms,
                    "traffic_per_launch": {k[0]: traffic.get(k[0]) for k in kernels}},
        "roofline": roof,
        "clocks": r["clocks"],
        "gpu_launches": r["launched"] * args.steps,
    })

    if "e2e" in legs:
        line["e2e"] = run_e2e(args, inp, stream, dist, tokens, world)
    del inp
    torch.cuda.empty_cache()

    if "decode" in legs:
        line["decode"] = run_decode(args, dev, stream, dist, peaks, traffic)
        torch.cuda.empty_cache()
    for name in ("varlen", "extreme"):
        if name not in legs:
            continue
        w = inputs.varlen(dev) if name == "varlen" else inputs.extreme(dev)
        ms_len = max(w.meta["lengths"]) if name == "varlen" else 0
        line[f"prefill_{name}"] = prefill_leg(w, args, stream, dist, peaks,
                                              steps=max(3, min(args.steps, 10)), warmup=3,
                                              max_seqlen=ms_len)
        del w
        torch.cuda.empty_cache()

    # --- CPU baseline (oracle) on rank 0 at N=1 ---
    cpu = cpu_baseline(args) if (rank == 0 and world == 1 and not args.no_cpu) else None
    line["cpu_baseline"] = cpu
    return line if rank == 0 else None


def run_e2e(args, inp, stream, dist, tokens, world):
    """The same metric end to end through the public API, host buffers in and
    out.  A serving loop pipelines steps: step i+1's inputs go up (several copy
    streams, double-buffered device inputs and outputs) while step i runs, and
    step i's results come back on another stream.  Every step's own
    host->device and device->host copies are inside the timed region."""
    import torch

    from linear_attention_recurrence_prefill_gb300 import kda

    o = torch.empty_like(inp.q)
    S_T = torch.empty((1, H, D, D), dtype=torch.float32, device=inp.q.device)
    o_opts = kda.kda_options_init(impl=kda.IMPLS[args.path])
    ws_bytes = kda.kda_prefill_workspace_size(T, 1, H, D, D, o_opts)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=inp.q.device)
    host = {n: getattr(inp, n).cpu().pin_memory() for n in
            ("q", "k", "v", "log_alpha", "beta", "gate", "S0")}
    devb = [{n: torch.empty_like(getattr(inp, n)) for n in host} for _ in range(2)]
    outs = [(torch.empty_like(o), torch.empty_like(S_T)) for _ in range(2)]
    y_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    st_host = torch.empty(S_T.shape, dtype=S_T.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = y_host.numel() * y_host.element_size() + st_host.numel() * st_host.element_size()
    # copies in flight on four streams: each tensor in two halves, the pieces
    # dealt out largest first
    up = [torch.cuda.Stream() for _ in range(N_UP)]
    down = torch.cuda.Stream()
    pieces = []
    for n, t in host.items():
        half = (t.shape[0] + 1) // 2
        pieces += [(n, 0, half), (n, half, t.shape[0])]
    pieces.sort(key=lambda p: -(p[2] - p[1]) * host[p[0]][0].numel() * host[p[0]].element_size())
    groups = [[] for _ in up]
    load = [0] * len(up)
    for pc in pieces:
        g = load.index(min(load))
        groups[g].append(pc)
        load[g] += (pc[2] - pc[1]) * host[pc[0]][0].numel() * host[pc[0]].element_size()
    done_in = [[torch.cuda.Event() for _ in up] for _ in range(2)]
    done_run = [torch.cuda.Event() for _ in range(2)]
    done_out = [torch.cuda.Event() for _ in range(2)]
    started = [False, False]

    def e2e_step(i):
        b = i % 2
        for g, grp in enumerate(groups):
            if started[b]:                      # the buffer's previous step has run
                up[g].wait_event(done_run[b])
            with torch.cuda.stream(up[g]):
                for n, r0, r1 in grp:
                    devb[b][n][r0:r1].copy_(host[n][r0:r1], non_blocking=True)
            done_in[b][g].record(up[g])
        for ev in done_in[b]:
            stream.wait_event(ev)
        if started[b]:                          # its outputs have been read back
            stream.wait_event(done_out[b])
        ob, sb = outs[b]
        d = devb[b]
        kda.kda_prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["S0"], None, 1,
                        ob, sb, gate=d["gate"], impl=args.path,
                        workspace=ws if ws_bytes else None, stream=stream)
        done_run[b].record(stream)
        down.wait_event(done_run[b])
        with torch.cuda.stream(down):
            y_host.copy_(ob, non_blocking=True)
            st_host.copy_(sb, non_blocking=True)
        done_out[b].record(down)
        started[b] = True

    e2e_steps = max(4, min(args.steps, 10))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(dist)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for st in up + [down]:
        st.wait_stream(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(down)
    ev1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, ev0.elapsed_time(ev1) / e2e_steps)
    del host, devb, outs, ws
    return {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}


def run_decode(args, dev, stream, dist, peaks, traffic):
    import torch

    from linear_attention_recurrence_prefill_gb300 import inputs, kda

    di = inputs.decode(dev)
    S = di.S.clone()
    o = torch.empty((DEC_N, H, D), dtype=torch.bfloat16, device=dev)

    def steps(n):
        for t in range(n):
            kda.kda_decode_step(di.q[t], di.k[t], di.v[t], di.log_alpha[t], di.beta[t], S, o)

    # The 256-step loop runs as one captured CUDA graph, as a serving loop
    # would: the launches are recorded once, so the timed region is the GPU's
    # work, not the per-call Python marshalling.
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        steps(8)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        steps(DEC_STEPS)
    graph.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(1, min(args.steps, 3))
    times = []
    for _ in range(reps):
        barrier(dist)
        torch.cuda.synchronize()
        ev0.record()
        graph.replay()
        ev1.record()
        torch.cuda.synchronize()
        times.append(ev0.elapsed_time(ev1))
    ms = max_over_ranks(dist, statistics.median(times))
    per_step_ms = ms / DEC_STEPS
    del graph
    bytes_step = DEC_BYTES_PER_UNIT * DEC_N * H
    gbs = bytes_step / (per_step_ms / 1e3) / 1e9
    world = int(os.environ.get("WORLD_SIZE", "1"))
    del di, S
    return {"metric": "KDA decode tokens/s (64 sequences x 96 heads, 256 steps, state in place)",
            "value": DEC_N * DEC_STEPS * world / (ms / 1e3), "unit": "tokens/s",
            "ms_per_step": per_step_ms,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "bytes_per_launch": bytes_step,
                         "kernel": "decode_kernel<128,bf16>",
                         "traffic": traffic.get("decode_kernel<128,bf16>")},
            "gpu_launches": DEC_STEPS * reps}


# ------------------------------------------------------------------ CPU oracle
def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _oracle_step(inp, heads):
    import oracle
    sl = lambda t: t[:, :heads].contiguous()  # noqa: E731
    t0 = time.perf_counter()
    o, _ = oracle.prefill(sl(inp.q), sl(inp.k), sl(inp.v), sl(inp.log_alpha), sl(inp.beta),
                          inp.S0[:, :heads].contiguous())
    oracle.gated_rmsnorm(o, sl(inp.gate))
    return time.perf_counter() - t0


def _calibrated_heads(inp, target_s: float) -> int:
    """Heads per oracle step so that one step takes about target_s seconds."""
    probe = min(H, max(4, cpu_cores()))
    dt = _oracle_step(inp, probe)
    return max(1, min(H, int(probe * target_s / max(dt, 1e-3))))


def cpu_baseline(args):
    """The oracle, as it stands, on the prefill workload (all OpenMP threads):
    every token of the first `heads` heads, `heads` chosen so that the sample
    is about 10 s of CPU work (all 96 heads when that fits).  Beside it the
    per-core figure: head 0 alone, which the oracle's loop over (sequence,
    head) gives to one thread."""
    from linear_attention_recurrence_prefill_gb300 import inputs

    inp = inputs.k3("cpu")
    heads = _calibrated_heads(inp, args.cpu_seconds)
    dt = _oracle_step(inp, heads)
    dt1 = min(_oracle_step(inp, 1) for _ in range(2))
    return {"value": heads * T / H / dt, "unit": "tokens/s", "cores": cpu_cores(),
            "kind": "oracle",
            "sample": f"k3 workload, all {T} tokens of the first {heads} of {H} heads "
                      f"({heads * T} head-tokens, {dt:.1f} s); tokens/s = head-tokens/s / {H}",
            "seconds": dt,
            "single_core": {"value": T / dt1, "unit": "head-tokens/s",
                            "sample": f"head 0, all {T} tokens, one thread ({dt1:.2f} s)"}}


def run_reference(args, rank, world):
    """Reference arm: the oracle timed on the host cores, W warm-up and K timed
    steps, each step the same bounded sample of the workload."""
    if rank != 0:
        return None
    from linear_attention_recurrence_prefill_gb300 import inputs

    inp = inputs.k3("cpu")
    per_step = max(1.0, min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup)))
    heads = _calibrated_heads(inp, per_step)
    for _ in range(args.warmup):
        _oracle_step(inp, heads)
    times = [_oracle_step(inp, heads) for _ in range(args.steps)]
    dt = statistics.mean(times)
    value = heads * T / H / dt
    sample = (f"k3 workload, all {T} tokens of the first {heads} of {H} heads per step "
              f"({heads * T} head-tokens); tokens/s = head-tokens/s / {H}")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": T / value * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": 1, "seq_len": T, "heads": H,
                   "head_dim": D, "parallelism": "host cores (OpenMP)",
                   "note": "CPU oracle (token-by-token fp64 recurrence)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--path", choices=["auto", "simt", "tc"], default="auto",
                    help="prefill implementation inside libkda (default: auto)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target seconds of CPU work for the oracle sample")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU baseline leg")
    ap.add_argument("--legs", default=",".join(LEGS),
                    help="comma list of what to measure besides the K3-shaped prefill: "
                         + ", ".join(LEGS[1:]) + " (default: all)")
    args = ap.parse_args(argv)
    bad = set(args.legs.split(",")) - set(LEGS)
    if bad:
        ap.error(f"unknown legs: {sorted(bad)}")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank, world, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    dist = init_dist(world)
    line = run_ours(args, rank, world, local, dist)
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
