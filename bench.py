"""Benchmark of the attention forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--cta-pair]
    python bench.py --impl reference ...     # the fp64 CPU oracle, timed on host cores
    python bench.py --microbench             # ex2 and tcgen05 throughput per SM clock

Prints ONE JSON line (rank 0).  A step is one forward pass over the whole
workload (default: bf16, causal, B=2 H=32 S=8192 D=128, inputs 2*N(0,1)):
`value` is TFLOP/s with inputs resident in HBM, counted as 4*B*H*Sq*Sk*D
(halved for causal), timed per step with CUDA events on the launching stream
and the L2 flushed between timed steps (a 256 MiB write, then a 256 MiB read so no
dirty lines are left to write back during the timed step); `e2e` is the same
metric through the public API with pinned host inputs copied in and O/LSE
copied out inside the timed region (steps pipelined over copy-in, compute and
copy-out streams with two buffer sets, as a serving loop runs them).  Under torchrun each rank runs the same
workload on its own GPU (the pass shards over independent (batch, head)
problems; no collective on the data path): value = all ranks' FLOPs / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOPS (bf16, causal, 8K, d=128) and % of GB300 tensor peak"
DEFAULT_WORKLOAD = "bf16_causal_8k"
L2_FLUSH_BYTES = 256 << 20


def _cache_used(w, x):
    """Cache workloads: keys each sequence attends over (filled length + new rows)."""
    return [int(n) + w.cache_new for n in x["cache_seqlens"].tolist()]


def _flops(w, x) -> float:
    """Algorithmic FLOPs of one pass: 4 * Sq * Sk * D per (batch, head), halved when causal
    (cache workloads: 4 * D per visible (query row, key) pair, bottom-right causal)."""
    if w.cache_new:
        tot = 0.0
        for used in _cache_used(w, x):
            for i in range(w.seqlen_q):
                vis = min(used, used - w.seqlen_q + i + 1) if w.causal else used
                tot += 4.0 * w.heads * w.head_dim * max(vis, 0)
        return tot
    if w.varlen:
        sq, sk = x["seqlens"]
        tot = sum(4.0 * w.heads * a * b * w.head_dim for a, b in zip(sq, sk))
    else:
        tot = 4.0 * w.batch * w.heads * w.seqlen_q * w.seqlen_k * w.head_dim
    return tot / 2 if w.causal else tot


def exp2_bound(flops: float, head_dim: int, tensor_peak_tflops: float, sms: int,
               sm_mhz: float, exp2_per_clk_per_sm: float) -> dict:
    """The two ceilings of a pass through the forward kernel: the tensor pipe (the
    algorithmic FLOPs at the tensor peak) and the MUFU (one exp2 per visible (query row,
    key) pair, i.e. FLOPs / (4 D), at the ex2 rate measured by the throughput probe).
    The larger time is attainable."""
    exps = flops / (4.0 * head_dim)
    exp2_ms = exps / (exp2_per_clk_per_sm * sms * sm_mhz * 1e6) * 1e3
    tensor_ms = flops / (tensor_peak_tflops * 1e12) * 1e3
    return {"exp2_per_launch": exps, "exp2_per_clk_per_sm": exp2_per_clk_per_sm,
            "sms": sms, "sm_mhz": sm_mhz, "exp2_ms": exp2_ms, "tensor_ms": tensor_ms,
            "attainable_ms": max(exp2_ms, tensor_ms),
            "limit": "tensor" if tensor_ms >= exp2_ms else "exp2"}


# ------------------------------------------------------------------ throughput probes
def _microbench_lib():
    import ctypes
    from exact_attention_forward_gb300 import _build
    lib = ctypes.CDLL(_build.build_microbench())
    vp, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_ulonglong
    lib.fa_mb_ex2.restype = i32
    lib.fa_mb_ex2.argtypes = [i32, i32, vp, vp, vp]
    lib.fa_mb_ex2_per_cta.restype = i64
    lib.fa_mb_ex2_per_cta.argtypes = [i32]
    lib.fa_mb_mma.restype = i32
    lib.fa_mb_mma.argtypes = [i32, i32, i32, i32, vp, vp, u64, vp]
    lib.fa_mb_mma_flops_per_cta.restype = i64
    lib.fa_mb_mma_flops_per_cta.argtypes = [i32, i32, i32]
    return lib


def _per_sm_rates(units_per_cta: float, cycles) -> dict:
    rates = sorted(units_per_cta / float(c) for c in cycles if c > 0)
    return {"median": statistics.median(rates), "min": rates[0], "max": rates[-1]}


def measure_ex2_rate(dev, iters: int = 2048, packed: bool = False) -> dict:
    """ex2.approx.ftz.f32 per SM clock (one 1024-thread CTA per SM, clock64-timed);
    packed: ex2.approx.f16x2, counting both halves."""
    import torch
    lib = _microbench_lib()
    lib.fa_mb_ex2_f16x2.restype = ctypes.c_int
    lib.fa_mb_ex2_f16x2.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cyc = torch.zeros(sms, dtype=torch.int64, device=dev)
    sink = torch.zeros(1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    fn = lib.fa_mb_ex2_f16x2 if packed else lib.fa_mb_ex2
    for _ in range(2):  # the first launch also loads the module
        rc = fn(sms, iters, cyc.data_ptr(), sink.data_ptr(), stream)
        if rc != 0:
            raise RuntimeError(f"ex2 probe launch failed ({rc})")
    torch.cuda.synchronize(dev)
    return _per_sm_rates(lib.fa_mb_ex2_per_cta(iters) * (2 if packed else 1), cyc.cpu().tolist())


def measure_mma_rate(dev, n: int, fp8: bool, iters: int = 2048) -> dict:
    """tcgen05.mma FLOP per SM clock, M = 128, N = n, one issuing thread per SM (n = -128:
    N = 128 in the PV form, A from Tensor Memory and B MN-major)."""
    import torch
    lib = _microbench_lib()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cyc = torch.zeros(sms, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    for _ in range(2):
        rc = lib.fa_mb_mma(sms, n, int(fp8), iters, cyc.data_ptr(), err.data_ptr(),
                           2_000_000_000, stream)
        if rc != 0:
            raise RuntimeError(f"fa_mb_mma launch failed ({rc})")
    torch.cuda.synchronize(dev)
    if int(err.item()) != 0:
        raise RuntimeError("fa_mb_mma: a bounded wait ran out")
    return _per_sm_rates(lib.fa_mb_mma_flops_per_cta(n, int(fp8), iters), cyc.cpu().tolist())


def measure_load_rate(dev, window: int, iters: int = 4096) -> dict:
    """cp.async.bulk bytes per SM clock into shared memory, each CTA (one per SM) reading its
    own `window` bytes cyclically (after a first untimed pass)."""
    import torch
    lib = _microbench_lib()
    lib.fa_mb_load.restype = ctypes.c_int
    lib.fa_mb_load.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_int,
                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_void_p]
    lib.fa_mb_load_bytes_per_cta.restype = ctypes.c_longlong
    lib.fa_mb_load_bytes_per_cta.argtypes = [ctypes.c_int]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    src = torch.ones(sms * window, dtype=torch.uint8, device=dev)
    cyc = torch.zeros(sms, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    for _ in range(2):
        rc = lib.fa_mb_load(sms, src.data_ptr(), window, iters, cyc.data_ptr(), err.data_ptr(),
                            2_000_000_000, stream)
        if rc != 0:
            raise RuntimeError(f"fa_mb_load launch failed ({rc})")
    torch.cuda.synchronize(dev)
    if int(err.item()) != 0:
        raise RuntimeError("fa_mb_load: a bounded wait ran out")
    return _per_sm_rates(lib.fa_mb_load_bytes_per_cta(iters), cyc.cpu().tolist())


def measure_mma_with_load(dev, window: int = 256 << 10, iters: int = 4096) -> dict:
    """bf16 SS-form MMA FLOP per SM clock while bulk copies stream into the same shared
    memory, and the copies' bytes per SM clock over the same cycles."""
    import torch
    lib = _microbench_lib()
    lib.fa_mb_mma_with_load.restype = ctypes.c_int
    lib.fa_mb_mma_with_load.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_ulonglong,
                                        ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_void_p]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    src = torch.ones(sms * window, dtype=torch.uint8, device=dev)
    cyc = torch.zeros(sms, dtype=torch.int64, device=dev)
    nb = torch.zeros(sms, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    for _ in range(2):
        rc = lib.fa_mb_mma_with_load(sms, src.data_ptr(), window, iters, cyc.data_ptr(),
                                     nb.data_ptr(), err.data_ptr(), 2_000_000_000, stream)
        if rc != 0:
            raise RuntimeError(f"fa_mb_mma_with_load launch failed ({rc})")
    torch.cuda.synchronize(dev)
    if int(err.item()) != 0:
        raise RuntimeError("fa_mb_mma_with_load: a bounded wait ran out")
    c, b = cyc.cpu().tolist(), nb.cpu().tolist()
    flops = lib.fa_mb_mma_flops_per_cta(128, 0, iters)
    return {"mma_flop_per_clk_per_sm": _per_sm_rates(flops, c),
            "copy_bytes_per_clk_per_sm": statistics.median(x / y for x, y in zip(b, c) if y > 0)}


def run_microbench(args):
    """One JSON line: ex2 and tcgen05 rates per SM clock, and what they give at the SM
    clock sampled while they ran."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    ex2 = measure_ex2_rate(dev)
    ex2_f16x2 = measure_ex2_rate(dev, packed=True)
    mma = {}
    for n, fp8 in ((64, False), (128, False), (256, False), (128, True), (256, True)):
        mma[f"{'e4m3' if fp8 else 'bf16'}_m128_n{n}"] = measure_mma_rate(dev, n, fp8)
    for fp8 in (False, True):  # the PV form: A from Tensor Memory, B MN-major
        mma[f"{'e4m3' if fp8 else 'bf16'}_m128_n128_a_tmem_b_mn_major"] = measure_mma_rate(dev, -128, fp8)
    mma["bf16_m128_n128_with_copies"] = measure_mma_with_load(dev)
    loads = {"l2_window_256KiB": measure_load_rate(dev, 256 << 10),
             "hbm_window_32MiB": measure_load_rate(dev, 32 << 20, iters=2048)}
    clocks = sampler.stop()
    mhz = clocks.get("sm_mhz") or 2070.0
    line = {"microbench": "ex2 / tcgen05 / bulk-copy throughput", "sms": sms, "clocks": clocks,
            "load_bytes_per_clk_per_sm": loads,
            "load_gbs_chip_at_sm_mhz": {k: v["median"] * sms * mhz * 1e6 / 1e9 for k, v in loads.items()},
            "ex2_per_clk_per_sm": ex2, "ex2_f16x2_per_clk_per_sm": ex2_f16x2,
            "ex2_per_s_chip_at_sm_mhz": ex2["median"] * sms * mhz * 1e6,
            "mma_flop_per_clk_per_sm": mma,
            "mma_tflops_chip_at_sm_mhz": {k: v["median"] * sms * mhz * 1e6 / 1e12
                                          for k, v in mma.items() if "median" in v}}
    print(json.dumps(line), flush=True)
    return 0


def _bytes(w, x) -> float:
    """Compulsory HBM bytes of one pass: Q, K, V read once; O (bf16) and LSE (fp32) written.
    Cache workloads: the filled cache rows each sequence uses are read once, the new rows
    are read once and written into the cache once."""
    q, k, v = x["q"], x["k"], x["v"]
    rows = q.numel() // q.shape[-1]  # query rows x heads = LSE entries
    out = rows * v.shape[-1] * 2 + rows * 4 + q.numel() * q.element_size()
    if w.cache_new:
        row_kv = k.shape[2] * k.shape[3] * k.element_size()  # one cache row of one tensor
        used = sum(_cache_used(w, x))
        new = x["k_new"].numel() * x["k_new"].element_size()
        return out + 2 * used * row_kv + 2 * 2 * new
    return out + (k.numel() + v.numel()) * q.element_size()


def _source_sha() -> str:
    """Hash of the kernel sources with comments and blank lines removed (the sources hold
    no comment markers inside strings), to tell whether recorded ncu counters still apply:
    a change of code changes it, a change of comments does not."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_forward_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if not os.path.isfile(os.path.join(csrc, f)):  # (the throughput probes' folder)
            continue
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(f.encode() + code.encode())
    return h.hexdigest()[:16]


def _recorded_traffic(workload: str):
    """DRAM bytes per launch of the forward kernel from a committed ncu summary, or None
    if none was recorded for this workload or the kernel sources changed since."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_sha") != _source_sha():
        return None
    return rec.get("bytes_per_launch")


def max_over_ranks(x: float, device=None) -> float:
    """The slowest rank's value (all_reduce MAX); identity when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, steps: int, max_ms: float) -> float:
    """Whole-job rate: every rank processed `units_per_rank` per step (weak scaling),
    over the slowest rank's time."""
    return world * units_per_rank * steps / (max_ms * 1e-3)


def measure_fp8_gemm_peak(device, n: int = 8192, iters: int = 10) -> float:
    """Dense e4m3 GEMM throughput of the library GEMM (torch._scaled_mm, n^3, best of
    `iters`, CUDA events): the denominator for e4m3 runs, measured on this GPU."""
    import torch
    a = torch.randn(n, n, device=device).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=device).to(torch.float8_e4m3fn).t()  # column-major B
    one = torch.ones((), device=device, dtype=torch.float32)
    for _ in range(3):
        torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(iters):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    return 2.0 * n ** 3 / (best * 1e-3) / 1e12


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def start(self):
        import torch
        args = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                "-lms", "100"]
        try:
            prop = torch.cuda.get_device_properties(self.dev)
            bus = f"{prop.pci_domain_id:08X}:{prop.pci_bus_id:02X}:{prop.pci_device_id:02X}.0"
            args += ["-i", bus]
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(args, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle (baseline)
def _oracle_rows_flops(w, rows, used=None):
    sq, sk = w.seqlen_q, w.seqlen_k
    tot = 0.0
    for b, _, i in rows:
        if used is not None:
            sk = used[b]
        n = sk if not w.causal else max(0, min(sk, i + sk - sq + 1))
        tot += 4.0 * n * w.head_dim
    return tot


def _oracle_inputs(w, x):
    """What the oracle attends over: for cache workloads, the caches with the new rows
    appended (by the oracle's own append) and the per-sequence lengths."""
    if not w.cache_new:
        return dict(q=x["q"], k=x["k"], v=x["v"], descale=x["descale"], seqused_k=None)
    import oracle
    lens = x["cache_seqlens"].tolist()
    return dict(q=x["q"], k=oracle.append_kv(x["k"], x["k_new"], lens),
                v=oracle.append_kv(x["v"], x["v_new"], lens), descale=x["descale"],
                seqused_k=_cache_used(w, x))


def _oracle_sample(w, xo, budget_s: float, seed: int = 0):
    """Time the oracle on seeded random rows of the workload until ~budget_s of CPU work."""
    import numpy as np
    import oracle

    rng = np.random.default_rng(seed)
    n = 16
    while True:
        rows = np.stack([rng.integers(0, w.batch, n), rng.integers(0, w.heads, n),
                         rng.integers(0, w.seqlen_q, n)], axis=1).astype(np.int64)
        t0 = time.perf_counter()
        oracle.attention_rows(xo["q"], xo["k"], xo["v"], rows, softmax_scale=w.softmax_scale,
                              causal=w.causal, descale=xo["descale"], seqused_k=xo["seqused_k"])
        dt = time.perf_counter() - t0
        if dt >= budget_s or n >= w.batch * w.heads * w.seqlen_q:
            return _oracle_rows_flops(w, rows, xo["seqused_k"]), dt, n
        grow = max(2.0, min(16.0, budget_s / max(dt, 1e-3)))
        n = int(n * grow)


def _oracle_threads():
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return int(os.environ.get("OMP_NUM_THREADS", n))


def run_reference(args, w):
    """The reference arm: the fp64 oracle, as it stands, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    os.environ.setdefault("OMP_NUM_THREADS", str(_oracle_threads()))
    from exact_attention_forward_gb300 import inputs
    x = inputs.make_inputs(w)
    xo = _oracle_inputs(w, x)
    per_step = max(2.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        _oracle_sample(w, xo, per_step / 4, seed=1)
    flops = secs = 0.0
    rows_total = 0
    for s in range(args.steps):
        f, dt, n = _oracle_sample(w, xo, per_step, seed=100 + s)
        flops += f
        secs += dt
        rows_total += n
    value = flops / secs / 1e12
    full = _flops(w, x)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        # one step = the whole workload; the oracle computes a sample of its rows per step,
        # so the time of a whole step follows from the sampled rate
        "ms_per_step": full / (value * 1e12) * 1e3,
        "sample_ms_per_step": 1e3 * secs / max(1, args.steps),
        "sample_fraction_per_step": flops / max(1, args.steps) / full,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": _oracle_threads(),
                         "kind": "oracle",
                         "sample": f"{rows_total} seeded random query rows of {w.name} "
                                   f"over {args.steps} steps"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


L2_NOTE = ("GPU arm: L2 flushed between timed steps (256 MiB write + 256 MiB read, untimed); "
           "CPU oracle arm: not applicable")


def _config(w):
    """The workload, identical in both arms' lines."""
    c = {"workload": w.name, "batch": w.batch, "heads": w.heads, "heads_k": w.kv_heads,
         "seqlen_q": w.seqlen_q,
         "seqlen_k": w.seqlen_k, "head_dim": w.head_dim, "causal": w.causal,
         "input_dtype": w.dtype, "values": f"{w.amp:g}*N(0,1) seed {w.seed}", "l2": L2_NOTE}
    if w.varlen:
        c["varlen"] = f"{w.n_seqs} seqs U{{1..{w.seqlen_q}}} + {len(w.empty_k_at)} with Sk=0"
    if w.cache_new:
        c["kv_cache"] = (f"capacity {w.seqlen_k}, filled U{{{w.seqlen_k // 2}.."
                         f"{w.seqlen_k - w.cache_new}}}, {w.cache_new} new row(s) appended per step")
    if w.v_dtype:
        c["v_dtype"] = w.v_dtype
    if w.descale != "tensor":
        c["descale"] = "per (batch, K/V head)"
    return c


# ------------------------------------------------------------------ GPU arm
def run_gpu(args, w):
    import torch
    import torch.distributed as dist

    import exact_attention_forward_gb300 as fa
    from exact_attention_forward_gb300 import inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    fa.load_library()

    x = inputs.make_inputs(w)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    cu_q = x["cu_seqlens_q"].to(dev) if w.varlen else None
    cu_k = x["cu_seqlens_k"].to(dev) if w.varlen else None
    fp8 = w.dtype == "e4m3"
    descale = ([torch.as_tensor(d, dtype=torch.float32).to(dev) for d in x["descale"]]
               if fp8 else None)
    cache = None
    if w.cache_new:
        cache = {n: x[n].to(dev) for n in ("k_new", "v_new", "cache_seqlens")}
    o_shape = (q.shape[0], q.shape[1], q.shape[2], v.shape[-1]) if not w.varlen else \
        (q.shape[0], q.shape[1], v.shape[-1])
    o = torch.empty(o_shape, dtype=torch.bfloat16, device=dev)
    lse_shape = (w.batch, w.heads, w.seqlen_q) if not w.varlen else (w.heads, q.shape[0])
    lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    ws = None
    pair = bool(getattr(args, "cta_pair", False))
    if pair and (fp8 or w.head_dim != 128 or w.cache_new):
        raise SystemExit("--cta-pair runs the bf16 head-dim-128 attention workloads only")
    if not w.varlen and not pair:
        if w.cache_new:
            need = fa.kvcache_workspace_size(w.batch, w.heads, w.kv_heads, w.seqlen_q, w.seqlen_k,
                                             w.head_dim, w.causal)
        else:
            need = fa.workspace_size(w.batch, w.heads, w.seqlen_q, w.seqlen_k, w.head_dim, w.causal,
                                     heads_k=w.kv_heads)
        if need:
            ws = torch.empty(need, dtype=torch.uint8, device=dev)
    if ws is None:
        splits = 1
    elif w.cache_new:
        splits = fa.kvcache_num_splits(w.batch, w.heads, w.kv_heads, w.seqlen_q, w.seqlen_k, w.causal)
    else:
        splits = fa.num_splits(w.batch, w.heads, w.seqlen_q, w.seqlen_k, w.causal, heads_k=w.kv_heads)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2():
        # evict the previous step's working set: write 256 MiB, then read another 256 MiB
        # so the dirty lines are written back before (not during) the timed step
        flush.zero_()
        flush_rd.max()

    def step():
        if cache is not None:  # append the new rows (same rows, same place: idempotent), attend
            fa.fwd_kvcache(q, k, v, cache["cache_seqlens"], cache["k_new"], cache["v_new"],
                           causal=w.causal, softmax_scale=w.softmax_scale, descale=descale,
                           workspace=ws, out=o, lse=lse, stream=stream)
            return
        fa.fwd(q, k, v, causal=w.causal, softmax_scale=w.softmax_scale, cu_seqlens_q=cu_q,
               cu_seqlens_k=cu_k, max_seqlen_q=x["max_seqlen_q"], max_seqlen_k=x["max_seqlen_k"],
               descale=descale, workspace=ws, out=o, lse=lse, stream=stream, cta_pair=pair)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    st, flags = fa.device_error(clear=True)
    if st != 0:
        raise RuntimeError(f"device error word {flags:#x} after warm-up")

    sampler = ClockSampler(dev.index)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush_l2()  # not timed
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(sum(times_ms), dev)
    flops = _flops(w, x)
    value = job_throughput(flops, world, args.steps, total_ms) / 1e12
    ms_per_step = total_ms / args.steps

    # ---------------- end to end through the public API, host buffers
    e2e = None
    if not args.skip_e2e:
        # Per step, the inputs come from pinned host memory -- Q, K, V, or for a cache
        # workload Q, the new K/V rows and the cache lengths (the cache itself is state that
        # lives on the device) -- and O and LSE go back to pinned host memory.  Steps are
        # pipelined the way a serving loop would run them: copies in on one stream, the
        # forward pass on another, copies out on a third, two buffer sets in rotation, so
        # step i+1's inputs travel while step i computes.
        names = ("q", "k_new", "v_new", "cache_seqlens") if cache is not None else ("q", "k", "v")
        nbuf = 2
        host = {n: x[n].cpu().contiguous().pin_memory() for n in names}
        devb = [{n: torch.empty_like(host[n], device=dev) for n in names} for _ in range(nbuf)]
        outs = [(torch.empty_like(o), torch.empty_like(lse)) for _ in range(nbuf)]
        hres = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                 torch.empty(lse.shape, dtype=lse.dtype).pin_memory()) for _ in range(nbuf)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(nbuf)]
        ev_comp = [torch.cuda.Event() for _ in range(nbuf)]
        ev_out = [torch.cuda.Event() for _ in range(nbuf)]

        def e2e_step(i):
            bi = i % nbuf
            d, (oo, ll), (ho, hl) = devb[bi], outs[bi], hres[bi]
            with torch.cuda.stream(s_in):
                if i >= nbuf:
                    s_in.wait_event(ev_comp[bi])  # step i-nbuf's pass has read these inputs
                for n in names:
                    d[n].copy_(host[n], non_blocking=True)
                ev_in[bi].record(s_in)
            stream.wait_event(ev_in[bi])
            if i >= nbuf:
                stream.wait_event(ev_out[bi])  # step i-nbuf's results have left these buffers
            if cache is not None:
                fa.fwd_kvcache(d["q"], k, v, d["cache_seqlens"], d["k_new"], d["v_new"],
                               causal=w.causal, softmax_scale=w.softmax_scale, descale=descale,
                               workspace=ws, out=oo, lse=ll, stream=stream)
            else:
                fa.fwd(d["q"], d["k"], d["v"], causal=w.causal, softmax_scale=w.softmax_scale,
                       cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=x["max_seqlen_q"],
                       max_seqlen_k=x["max_seqlen_k"], descale=descale, workspace=ws, out=oo,
                       lse=ll, stream=stream, cta_pair=pair)
            ev_comp[bi].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[bi])
                ho.copy_(oo, non_blocking=True)
                hl.copy_(ll, non_blocking=True)
                ev_out[bi].record(s_out)

        for i in range(2 * nbuf):
            e2e_step(i)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        n_e2e = max(3, min(args.steps, 20))
        if world > 1:
            dist.barrier()
        e0.record(s_in)
        for i in range(n_e2e):
            e2e_step(i)
        s_out.wait_stream(stream)
        s_out.wait_stream(s_in)
        e1.record(s_out)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = sum(t.numel() * t.element_size() for t in hres[0])
        e2e = {"value": job_throughput(flops, world, n_e2e, e2e_ms) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms / n_e2e}

    st, flags = fa.device_error(clear=True)
    if st != 0:
        raise RuntimeError(f"device error word {flags:#x} after timing")

    peaks, peak_src = _peaks()
    fp8_peak = None
    if fp8:
        try:
            fp8_peak = measure_fp8_gemm_peak(dev)
        except Exception as exc:  # keep the line; fall back to the nominal ratio
            print(f"fp8 GEMM peak not measured: {exc}", file=sys.stderr)
    kernel_ms = ms_per_step
    if w.cache_new or (w.seqlen_q <= 256 and not w.varlen and not w.causal and splits > 1):
        bound, unit = "hbm", "GB/s"
        achieved = _bytes(w, x) / (kernel_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
    else:
        bound, unit = "tensor", "TFLOP/s"
        achieved = flops / (kernel_ms * 1e-3) / 1e12
        peak = fp8_peak if fp8_peak else peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)
    if fp8 and fp8_peak:
        src = "torch._scaled_mm e4m3 8192^3 measured in this run (best of 10)"
    else:
        src = f"{peak_src} MEASURED_PEAKS.json burst" + (
            " x2 (fp8/bf16 nominal ratio)" if fp8 and bound == "tensor" else "")
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak,
                "traffic": _recorded_traffic(w.name + ("/cta_pair" if pair else "")),
                "peak_source": src,
                "frac_of_sustained": (achieved / peaks.get("bf16_tflops_sustained", peak)
                                      if bound == "tensor" and not fp8 else None)}
    if bound == "tensor":
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        sm_mhz = clocks.get("sm_mhz") or peaks.get("sm_max_mhz") or 2070.0
        try:  # the ex2 rate, measured now by the throughput probe (a few ms)
            ex2 = measure_ex2_rate(dev)
            roofline["exp2_bound"] = exp2_bound(flops, w.head_dim, peak, sms, sm_mhz,
                                                ex2["median"])
            roofline["exp2_bound"]["exp2_rate_source"] = (
                "measured in this run: ex2.approx.ftz.f32 throughput probe, one 1024-thread "
                "CTA per SM, clock64-timed (median over SMs)")
        except Exception as exc:  # keep the line; say why the second ceiling is missing
            roofline["exp2_bound"] = {"unavailable": f"ex2 probe failed: {exc}"}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if not fp8 else "e4m3", "data": "synthetic",
        "config": _config(w),
        "kernel": "cta_pair (clusters of 2, cta_group::2)" if pair else "one CTA per SM",
        "clocks": clocks, "e2e": e2e,
        # per step: the forward kernel, the split merge when the key range is split, and the
        # cache-append copy kernel when a call appends more than 4 rows per sequence (fewer
        # are written by the forward kernel itself)
        "gpu_launches": args.steps * ((2 if splits > 1 else 1) +
                                      (1 if cache is not None and w.cache_new > 4 else 0)),
        "roofline": roofline,
        "step_ms": {"min": min(times_ms), "median": statistics.median(times_ms),
                    "max": max(times_ms)},
        "key_splits": splits,
    }
    if rank == 0 and not args.skip_cpu_baseline and world == 1:
        os.environ.setdefault("OMP_NUM_THREADS", str(_oracle_threads()))
        f, dt, n = _oracle_sample(w, _oracle_inputs(w, x), args.cpu_seconds)
        line["cpu_baseline"] = {"value": f / dt / 1e12, "unit": "TFLOP/s",
                                "cores": _oracle_threads(), "kind": "oracle",
                                "sample": f"{n} seeded random query rows of {w.name} "
                                          f"({dt:.1f} s, fp64)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cta-pair", action="store_true",
                    help="time the CTA-pair kernel (fa_fwd_2cta) instead of the one-CTA kernel")
    ap.add_argument("--microbench", action="store_true",
                    help="measure the ex2 and tcgen05 throughput per SM clock and exit")
    args = ap.parse_args(argv)
    if args.microbench:
        return run_microbench(args)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    from exact_attention_forward_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
