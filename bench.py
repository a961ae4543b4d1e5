"""Benchmark of the quantized attention prefill path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
K channel mean, Q/K int8 quantization, V e4m3 quantization (qattn_prepare,
one or two launches; the three separate calls for tensor/head granules) and
the fused attention kernel (qattn_fwd).  Default workload: LLM prefill, B=1,
32 query heads / 8 KV heads, 8192 tokens, d=128, causal (the 8K causal
prefill shape the throughput target is stated on).  Other workloads: tiny,
vit, swin, chunk32k (prefill on an int8 KV cache) and decode32k (a step
appends one token to the int8 cache, quantizes its Q and decodes); modes
--exact24 (the 24-bit exact split mode on the int8 cache) and --intsoftmax
(QFlash's integer-only attention on per-tensor int8 codes).

The line's value is device-resident throughput; "e2e" is the same step
through the public path with host buffers, the copies in and out overlapped
across consecutive steps (pipeline.OverlappedSteps; decode: serial).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--exact24 | --intsoftmax] [--no-cpu-baseline]
    python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention effective TOPS and % of measured GB300 dense int8/fp8 tensor peak"
UNIT = "TOPS"
# Seconds of oracle work the reference arm spends on its warm-up and timed
# steps together, whatever --steps and --warmup are.
REF_BUDGET_S = 100.0
# Seconds of oracle work (one warm-up and one timed step) behind the GPU
# line's cpu_baseline.
CPU_BASELINE_S = 16.0


def _peaks():
    """Measured GB300 peaks (generated file), else the documented fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16": float(p["bf16_tflops"]),
                "bf16_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def mixed_peak(peaks, sustained=True):
    """Peak of the attention contraction from the cuBLAS bf16 figure: half the
    algorithmic ops (QK^T) run at the fp16 rate (= the measured bf16 rate),
    half (PV) at the e4m3 rate (= the fp16 rate times the nominal 4.5/2.25
    ratio); harmonic combination."""
    p16 = peaks["bf16_sustained"] if sustained else peaks["bf16"]
    p8 = 2.0 * p16
    return 1.0 / (0.5 / p16 + 0.5 / p8)


def tensor_roofline(achieved, peaks, unit_peaks):
    """The attention kernel's tensor roofline against the stricter of two
    measured peaks: the tcgen05 kind::f16 and kind::f8f6f4 loops run in this
    process on this GPU (quantized_attention_gb300.peaks), and the cuBLAS
    bf16 burst figure with the nominal e4m3/f16 ratio.  Both are reported."""
    cub_burst = mixed_peak(peaks, sustained=False)
    cub_sus = mixed_peak(peaks, sustained=True)
    r = {"bound": "tensor", "achieved": achieved, "unit": "TFLOP/s",
         "peak_cublas_burst": cub_burst, "frac_cublas_burst": achieved / cub_burst,
         "peak_cublas_sustained": cub_sus, "frac_cublas_sustained": achieved / cub_sus}
    if unit_peaks is not None:
        m = unit_peaks["mixed"]
        r.update({"peak_tcgen05_loops": m, "frac_tcgen05_loops": achieved / m,
                  "tcgen05_f16": unit_peaks["f16"], "tcgen05_f8": unit_peaks["f8"]})
    if unit_peaks is not None and unit_peaks["mixed"] >= cub_burst:
        r["peak"] = unit_peaks["mixed"]
        r["peak_basis"] = (f"measured in this run: tcgen05 kind::f16 {unit_peaks['f16']:.1f} and "
                           f"kind::f8f6f4 {unit_peaks['f8']:.1f} TFLOP/s loops (QK^T half, PV half, "
                           f"harmonic), the stricter of it and the cuBLAS bf16 burst figure "
                           f"({peaks['source']}) with the nominal e4m3/f16 ratio")
    else:
        r["peak"] = cub_burst
        r["peak_basis"] = (f"{peaks['source']} cuBLAS bf16 burst {peaks['bf16']:.1f} for QK^T, "
                           f"2x that (nominal e4m3/f16 ratio) for PV, harmonic; the stricter of "
                           f"it and the tcgen05 loops measured in this run")
    r["frac"] = achieved / r["peak"]
    return r


def _attn_traffic(wl_name):
    """DRAM bytes per attention-kernel launch from the committed ncu capture
    (profiles/attn_fwd_<workload>_traffic.txt), or None when there is none for
    this workload or the kernel source has changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"attn_fwd_{wl_name}_traffic.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#") and "=" in line:
                k, v = line.split("=", 1)
                kv[k] = v
    h = hashlib.sha256()
    for name in ("attn_fwd.cu", "sm103_ptx.cuh", "qattn_check.cuh"):
        with open(os.path.join(ROOT, "quantized_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    if kv.get("workload") != wl_name or kv.get("kernel_source_sha256") != h.hexdigest():
        return None
    return int(kv["dram_bytes_read"]) + int(kv["dram_bytes_write"])


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------

# Active clock-event reason bits of NVML (nvml.h), by the names nvidia-smi
# prints for them.
_NVML_REASONS = ((0x4, "sw_power_cap"), (0x8, "hw_slowdown"), (0x20, "sw_thermal_slowdown"),
                 (0x40, "hw_thermal_slowdown"), (0x80, "hw_power_brake_slowdown"))


class _NvmlClocks:
    """Read-only NVML queries through ctypes (the library ships with the
    driver): the SM clock, its maximum and the active clock-event reasons of
    one device.  Raises OSError when NVML or the device is unavailable."""
    SM = 1  # NVML_CLOCK_SM

    def __init__(self, index: int):
        import ctypes
        self.ct = ctypes
        L = ctypes.CDLL("libnvidia-ml.so.1")
        if L.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.L = L
        self.h = ctypes.c_void_p()
        if L.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            L.nvmlShutdown()
            raise OSError("no NVML device handle")
        try:
            self.reasons_fn = L.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self.reasons_fn = L.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        if L.nvmlDeviceGetMaxClockInfo(self.h, ctypes.c_int(self.SM), ctypes.byref(mx)) != 0:
            L.nvmlShutdown()
            raise OSError("no maximum SM clock")
        self.max_mhz = float(mx.value)

    def sample(self):
        """(SM MHz, reason bits), or None if a query failed."""
        ct = self.ct
        c, r = ct.c_uint(0), ct.c_ulonglong(0)
        if self.L.nvmlDeviceGetClockInfo(self.h, ct.c_int(self.SM), ct.byref(c)) != 0:
            return None
        if self.reasons_fn(self.h, ct.byref(r)) != 0:
            return None
        return float(c.value), int(r.value)

    def close(self):
        self.L.nvmlShutdown()


class ClockSampler:
    """Samples the SM clock and the clock-event reasons while the timed steps
    run: NVML polled every 2 ms from a thread (so even a timed region of a few
    milliseconds is sampled), else nvidia-smi every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_s: float = 0.002):
        self.gpu = gpu_index
        self.period = period_s
        self.proc = None
        self.nvml = None
        self.samples = []
        self.lines = []

    def _poll(self):
        while not self._stop.is_set():
            v = self.nvml.sample()
            if v is not None:
                self.samples.append(v)
            self._stop.wait(self.period)

    def __enter__(self):
        import threading
        try:
            self.nvml = _NvmlClocks(self.gpu)
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            self._stop = threading.Event()
            v = self.nvml.sample()  # one sample as the region opens
            if v is not None:
                self.samples.append(v)
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.nvml is not None:
            v = self.nvml.sample()  # one sample as the region closes
            if v is not None:
                self.samples.append(v)
            self._stop.set()
            self._thread.join(timeout=5)
            self.nvml.close()
            return
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if self.samples:
            return summarize_nvml_samples(self.samples, self.nvml.max_mhz if self.nvml else None)
        return summarize_smi_lines(self.lines)


def summarize_nvml_samples(samples, max_mhz):
    """Median SM clock, maximum and the union of the active slowdown reasons
    of (MHz, NVML reason bits) samples."""
    reasons = sorted({name for _, bits in samples for bit, name in _NVML_REASONS if bits & bit})
    return {"sm_mhz": statistics.median(m for m, _ in samples), "sm_max_mhz": max_mhz,
            "reasons": reasons, "samples": len(samples), "source": "nvml, every 2 ms"}


def summarize_smi_lines(lines):
    """The same summary from nvidia-smi's CSV lines (FIELDS order)."""
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            mx.append(float(f[2]))
        except ValueError:
            continue
        for n, v in zip(names, f[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
            "samples": len(sm), "source": "nvidia-smi, every 200 ms"}


# ----------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline): bounded sample, all host cores
# ----------------------------------------------------------------------------

_SAMPLE = None


def _init_worker(sample):
    global _SAMPLE
    _SAMPLE = sample


def _oracle_sample_worker(args):
    head, rows_lo, rows_hi = args
    from oracle import qattn_oracle as O
    wl, inp, prep = _SAMPLE
    rows = np.arange(rows_lo, rows_hi)
    O.run_workload(inp, prep, heads=[(0, head)], rows=rows)
    return 4 * wl.d * int(O.visible_mask(rows, wl.Nk, wl.causal, wl.pos0).sum())


def sample_problem(wl_name):
    """The bounded sample: batch 0, the first KV head and the query heads that
    read it, with every token (the quantization sees the same data as in the
    full workload, so the codes are identical)."""
    from oracle import qattn_oracle as O
    from quantized_attention_gb300 import inputs as I
    wl = I.WORKLOADS[wl_name]
    full = I.make_inputs(wl)
    g = wl.Hq // wl.Hkv
    sub = wl.replace(B=1, Hq=g, Hkv=1)
    kw = {"Q": full.Q[:1, :g].copy(), "bias": full.bias}
    if wl.kv_codes:
        kw.update(K_codes=full.K_codes[:1, :1].copy(), K_scale=full.K_scale[:1, :1].copy(),
                  V_codes=full.V_codes[:1, :1].copy(), V_scale=full.V_scale[:1, :1].copy())
    else:
        kw.update(K=full.K[:1, :1].copy(), V=full.V[:1, :1].copy())
    inp = I.Inputs(sub, **kw)
    return sub, inp, O.prepare(inp)


def oracle_items(wl, rows, n_items):
    """Up to n_items (query head, row_lo, row_hi) spans covering `rows` query
    rows of the sample, heaviest first: under a causal mask the last rows of
    each query head see the most keys.  Spans never repeat a row."""
    rows = max(1, min(rows, wl.Hq * wl.Nq))
    n_items = max(1, min(n_items, rows))
    per = -(-rows // n_items)
    items, left = [], rows
    for t in range(n_items):
        h, k = t % wl.Hq, t // wl.Hq
        hi = wl.Nq - k * per
        lo = max(0, hi - min(per, left))
        if hi <= 0 or lo >= hi:
            break
        items.append((h, lo, hi))
        left -= hi - lo
        if left <= 0:
            break
    return items


def run_oracle_items(pool, items):
    """Times the oracle on the items in the pool; returns (ops, seconds)."""
    t0 = time.perf_counter()
    ops = sum(pool.map(_oracle_sample_worker, items))
    return ops, time.perf_counter() - t0


def time_cpu_budgeted(wl_name, warmup, steps, budget_s):
    """The reference arm: warmup + steps oracle steps in about budget_s
    seconds whatever their number.  Two calibration passes (the heaviest 1 and
    8 rows on each core) give the per-call cost and the per-row cost; every
    step then runs the same sample of heaviest rows, sized so that all steps
    fit the budget (at least one row per core), at most every row of the
    sample."""
    sample = sample_problem(wl_name)
    wl = sample[0]
    pool, cores = make_pool(sample)
    try:
        run_oracle_items(pool, oracle_items(wl, cores, cores))  # workers' first call
        # time per pass with r rows per core: a + b r (a: per-call cost)
        _, t1 = run_oracle_items(pool, oracle_items(wl, cores, cores))
        _, t8 = run_oracle_items(pool, oracle_items(wl, 8 * cores, cores))
        b = max((t8 - t1) / 7.0, 1e-6)
        a = max(t1 - b, 0.0)
        n = max(1, warmup + steps)
        r = int((budget_s / n - a) / b)
        rows = max(1, min(r * cores, wl.Hq * wl.Nq))
        # one span per core while spans are short; more, dealt out dynamically,
        # once long spans would differ in weight under a causal mask
        items = oracle_items(wl, rows, cores if r < 64 else 4 * cores)
        for _ in range(warmup):
            run_oracle_items(pool, items)
        ops, secs = 0, 0.0
        for _ in range(steps):
            o, s = run_oracle_items(pool, items)
            ops += o
            secs += s
    finally:
        pool.close()
    n_rows = sum(hi - lo for _, lo, hi in items)
    desc = (f"{n_rows} query rows per step of {wl_name} (batch 0, KV head 0: "
            f"{len(items)} spans, heaviest rows first), sized so {warmup}+{steps} steps "
            f"fit about {budget_s:.0f} s")
    return ops, secs, cores, desc


def make_pool(sample):
    """A spawn-started pool over every host core, each worker holding the
    sample and running its NumPy/BLAS on one thread (so `cores` is the number
    of threads in use, with no oversubscription)."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0))
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    os.environ.update({k: "1" for k in keys})
    try:
        pool = mp.get_context("spawn").Pool(cores, initializer=_init_worker, initargs=(sample,))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return pool, cores


def time_cpu_mode_baseline(mode, wl_name, budget_s=10.0):
    """The oracle of an extra mode, as it stands, on whole items of the
    workload (one process) until about budget_s seconds of CPU time; returns
    (ops, seconds, cores, description).  ops counts 4 d per visible (query,
    key) pair, as the GPU line does."""
    from oracle import qattn_oracle as O
    from quantized_attention_gb300 import inputs as I
    wl = I.WORKLOADS[wl_name]
    inp = I.make_inputs(wl)
    ops, n, t0 = 0, 0, time.perf_counter()
    if mode == "intsoftmax":  # per-tensor codes of Q, K, V, then the integer attention
        qc, sq = O.quantize_sym(inp.Q, O.GRAN_TENSOR)
        kc, sk = O.quantize_sym(inp.K, O.GRAN_TENSOR)
        vc, _ = O.quantize_sym(inp.V, O.GRAN_TENSOR)
        sq, sk = F32(np.asarray(sq).reshape(-1)[0]), F32(np.asarray(sk).reshape(-1)[0])
        heads = [(b, h) for b in range(wl.B) for h in range(wl.Hq)]
        while n < len(heads) and time.perf_counter() - t0 < budget_s:
            O.attn_intsoftmax(qc, sq, kc, sk, vc, heads=[heads[n]])
            ops += 4 * wl.d * wl.Nq * wl.Nk
            n += 1
        desc = (f"per-tensor codes of the whole tensors, then {n} whole (image, head) attentions "
                f"of {wl_name}, int64 NumPy, one process")
    else:  # exact24: 128-row query blocks of head 0 against the whole cache
        nblk = (wl.Nq + 127) // 128
        while n < nblk and time.perf_counter() - t0 < budget_s:
            rows = np.arange(n * 128, min(wl.Nq, n * 128 + 128))
            O.attn_exact24(inp.Q, inp.K_codes, inp.K_scale, inp.V_codes, inp.V_scale,
                           causal=wl.causal, q_pos0=wl.q_pos0, heads=[(0, 0)], rows=rows)
            ops += 4 * wl.d * int(O.visible_mask(rows, wl.Nk, wl.causal, wl.pos0).sum())
            n += 1
        desc = f"{n} blocks of 128 query rows of head 0 of {wl_name} over the whole cache, one process"
    return ops, time.perf_counter() - t0, 1, desc


F32 = np.float32


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    ops, secs, cores, desc = time_cpu_budgeted(args.workload, args.warmup, args.steps,
                                               REF_BUDGET_S)
    value = ops / secs / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8+e4m3",
            "data": "synthetic", "config": _config(args.workload),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _config(wl_name):
    from quantized_attention_gb300 import inputs as I
    wl = I.WORKLOADS[wl_name]
    return {"workload": f"{wl_name}: B={wl.B} Hq={wl.Hq} Hkv={wl.Hkv} Nq={wl.Nq} Nk={wl.Nk} "
                        f"d={wl.d} causal={int(wl.causal)} q_pos0={wl.pos0}",
            "granularity": {0: "tensor", 1: "head", 2: "block128"}[wl.q_gran],
            "kv_input": "int8 codes" if wl.kv_codes else "bf16",
            "output": "bf16", "l2": "flushed (256 MB write) before every timed step",
            **({"step": "append the new token's K/V to the int8 cache (running K mean), "
                        "quantize its Q, decode over all Nk cached keys"} if wl.kv_codes and
               wl_name.startswith("decode") else {})}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def prefill_roofline(wl, attn_ms, ops, has_bias, peaks, unit_peaks, v_ld):
    """Roofline of qattn_fwd's kernel on a prefill workload: tensor-bound for
    long rows; for ViT / Swin (197 / 49 keys) the operands' bytes bound it
    (HBM), with the tensor fraction beside."""
    achieved = ops / (attn_ms * 1e-3) / 1e12
    tr = tensor_roofline(achieved, peaks, unit_peaks)
    tr["kernel"] = "attn_fwd_kernel (the one launch of qattn_fwd)"
    if wl.name.split("@")[0] not in ("vit", "swin"):
        return tr
    alg_bytes = (wl.B * wl.Hq * wl.Nq * wl.d + wl.B * wl.Hkv * wl.Nk * wl.d  # Q, K codes
                 + wl.B * wl.Hkv * wl.d * v_ld                              # V8^T
                 + wl.B * wl.Hq * wl.Nq * wl.d * 2                          # bf16 O
                 + (wl.Nq * wl.Nk * 4 if has_bias else 0))                 # fp32 bias
    gbs = alg_bytes / (attn_ms * 1e-3) / 1e9
    return {"bound": "hbm",
            "kernel": ("attn_window_kernel (qattn_fwd's warp-level kernel for short windows)"
                       if wl.name.startswith("swin") else tr["kernel"]),
            "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": gbs / peaks["hbm_gbs"],
            "peak_basis": f"{peaks['source']} HBM copy rate",
            "algorithmic_bytes": alg_bytes,
            "tensor_frac": tr["frac"], "traffic": None}


def measure_unit_peaks():
    """tcgen05 / mma.sync / MUFU loop rates on this GPU, or (error, None)."""
    try:
        from quantized_attention_gb300 import peaks as PK
        rates = PK.measure()
        return rates, PK.attention_peak(rates)
    except Exception as e:  # reported in the line; the cuBLAS figure then stands alone
        return {"error": f"{type(e).__name__}: {e}"}, None


def time_prefill_workload(name, steps, warmup, flush, stream, local, peaks, unit_peaks):
    """Device time of the prefill step (pre-pass + qattn_fwd) on one more
    workload, with the same L2 flush and clock sampling as the main line."""
    import torch
    from quantized_attention_gb300 import binding as qb
    from quantized_attention_gb300 import inputs as I
    from quantized_attention_gb300.pipeline import device_inputs, problem_for

    wl = I.WORKLOADS[name]
    inp = I.make_inputs(wl)
    dev = device_inputs(inp)
    bias = dev.pop("bias", None)
    P = problem_for(wl, out_dtype=qb.DT_BF16, k_carrier=True)
    for _ in range(warmup):
        P.quantize(**dev, stream=stream)
        P.attend(bias, stream)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    with ClockSampler(local) as clk:
        for i in range(steps):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            P.quantize(**dev, stream=stream)
            ev[i][1].record(stream)
            P.attend(bias, stream)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
    if qb.get_error() != 0:
        raise RuntimeError(f"device error word set during the {name} steps")
    step_ms = sum(a.elapsed_time(c) for a, _, c in ev) / steps
    attn_ms = sum(b.elapsed_time(c) for _, b, c in ev) / steps
    ops = 4 * wl.d * wl.unmasked_pairs()
    return {"config": _config(name)["workload"], "steps": steps, "warmup": warmup,
            "ms_per_step": step_ms, "value": ops / (step_ms * 1e-3) / 1e12, "unit": UNIT,
            "attn_kernel_ms": attn_ms,
            "roofline": prefill_roofline(wl, attn_ms, ops, bias is not None, peaks, unit_peaks,
                                         qb.v_ld(wl.Nk)),
            "gpu_launches": P.kernel_launches() * steps, "clocks": clk.summary()}


def max_over_ranks(ms: float, world: int) -> float:
    """The slowest rank's time (every rank gets it), then a barrier; the
    identity for one process."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def whole_job_value(ops_per_rank: float, world: int, ms_per_step: float) -> float:
    """TOPS of the whole job: every rank runs its own copy of the workload
    (weak scaling), over the slowest rank's time per step."""
    return world * ops_per_rank / (ms_per_step * 1e-3) / 1e12


def gpu_arm(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)

    from quantized_attention_gb300 import binding as qb
    from quantized_attention_gb300 import inputs as I
    from quantized_attention_gb300.pipeline import device_inputs, problem_for

    unit_rates, unit_peaks = (measure_unit_peaks() if not args.no_unit_peaks
                              else ({"skipped": "--no-unit-peaks"}, None))
    wl = I.WORKLOADS[args.workload]
    inp = I.make_inputs(wl)
    dev = device_inputs(inp)
    bias = dev.pop("bias", None)
    decode = wl.name.startswith("decode")
    P = problem_for(wl, out_dtype=qb.DT_BF16, k_carrier=not decode)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device="cuda")

    ops = 4 * wl.d * wl.unmasked_pairs()
    if decode:  # the int8 cache is device state; a step appends the new token, quantizes its Q, decodes
        hdr = torch.from_numpy(inp.K_header_mean).to("cuda")
        P.set_cache(dev["K_codes"], dev["V_codes"], dev["V_scale"], K_scale=dev["K_scale"], K_mean=hdr)
        k_new, v_new = I.make_append_tokens(inp, 1)
        dev["K_new"] = torch.from_numpy(k_new).to(device="cuda", dtype=torch.bfloat16)
        dev["V_new"] = torch.from_numpy(v_new).to(device="cuda", dtype=torch.bfloat16)
        cache_bytes = 2 * wl.B * wl.Hkv * wl.Nk * wl.d  # K and V codes, read once

    if args.exact24:  # the 24-bit exact split mode on the int8 cache
        if not wl.kv_codes:
            raise SystemExit("--exact24 needs an int8-cache workload (chunk32k, decode32k)")
        e24_shape = qb.make_shape(wl.B, wl.Hq, wl.Hkv, wl.Nq, wl.Nk, wl.d)
        e24_params = qb.make_params(causal=wl.causal, q_pos0=wl.q_pos0, out_dtype=qb.DT_BF16)
        e24_ws = torch.empty(max(qb.workspace_size(e24_shape, e24_params), 256), dtype=torch.uint8,
                             device="cuda")

    if args.intsoftmax:  # QFlash: per-tensor int8 codes of bf16 Q, K, V, integer-only attention
        if wl.kv_codes or wl.causal:
            raise SystemExit("--intsoftmax needs an unmasked bf16 workload (vit, tiny)")
        from quantized_attention_gb300.pipeline import QFlashProblem
        ism = QFlashProblem(wl.B, wl.Hq, wl.Hkv, wl.Nq, wl.Nk, wl.d)

    def run_exact24():
        qb.fwd_exact24(dev["Q"], dev["K_codes"], dev["K_scale"], dev["V_codes"], dev["V_scale"],
                       e24_shape, e24_params, P.O, P.lse, e24_ws, stream)

    def step():
        if args.intsoftmax:
            ism.quantize(dev["Q"], dev["K"], dev["V"], stream)
            ev_a.record(stream)
            ism.attend(stream)
            ev_b.record(stream)
            return
        if args.exact24:
            ev_a.record(stream)
            run_exact24()
            ev_b.record(stream)
            return
        if decode:
            P.append(dev["K_new"], dev["V_new"], wl.Nk - 1, stream)  # the token at row Nk-1
            P.quantize_q(dev["Q"], dev["K_scale"], stream)
            ev_a.record(stream)
            P.decode(stream)
            ev_b.record(stream)
            return
        P.quantize(**dev, stream=stream)
        ev_a.record(stream)
        P.attend(bias, stream)
        ev_b.record(stream)

    for _ in range(args.warmup):
        ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        step()
    torch.cuda.synchronize()
    if qb.get_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    attn_a = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    attn_b = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)  # evict L2 (outside the timed interval)
            starts[i].record(stream)
            ev_a, ev_b = attn_a[i], attn_b[i]
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    if qb.get_error() != 0:
        raise RuntimeError("device error word set during the timed steps")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    attn_ms = [a.elapsed_time(b) for a, b in zip(attn_a, attn_b)]
    total_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    value = whole_job_value(ops, world, ms_per_step)

    # ---- end to end through the public API, host buffers, copies timed
    if args.intsoftmax:  # bf16 Q, K, V in, the int8 output codes back
        host = {k: v.cpu().pin_memory() for k, v in dev.items() if k in ("Q", "K", "V")}
        out_dev = ism.O
    else:
        host = {k: v.cpu().pin_memory() for k, v in dev.items()
                if (not decode and not args.exact24) or k in ("Q", "K_new", "V_new")}
        out_dev = P.O
    out_host = torch.empty(out_dev.shape, dtype=out_dev.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step():
        for k, v in host.items():
            dev[k].copy_(v, non_blocking=True)
        if args.intsoftmax:
            ism.run(dev["Q"], dev["K"], dev["V"], stream)
        elif args.exact24:
            run_exact24()
        elif decode:
            P.append(dev["K_new"], dev["V_new"], wl.Nk - 1, stream)
            P.quantize_q(dev["Q"], dev["K_scale"], stream)
            P.decode(stream)
        else:
            P.run(**dev, bias=bias, stream=stream)
        out_host.copy_(out_dev, non_blocking=True)

    # decode steps are sequential (each appends the token the next one reads);
    # the other modes' steps are independent and run overlapped
    overlapped = not decode
    copy_ms = None
    e_s = torch.cuda.Event(enable_timing=True)
    e_e = torch.cuda.Event(enable_timing=True)
    e_ms = 0.0
    if overlapped:
        # prefill as a stream of independent steps: step i's host-to-device
        # copies, step i-1's kernels and step i-2's device-to-host copy overlap
        # (two buffer sets, three streams); the L2 flush runs on the compute
        # stream before each step's kernels, inside the timed interval
        from quantized_attention_gb300.pipeline import OverlappedSteps

        if args.intsoftmax:
            def compute(d_in, d_out, s):
                ism.run(d_in["Q"], d_in["K"], d_in["V"], s, out=d_out)
        elif args.exact24:  # the cache is resident; each step brings its queries
            def compute(d_in, d_out, s):
                qb.fwd_exact24(d_in["Q"], dev["K_codes"], dev["K_scale"], dev["V_codes"],
                               dev["V_scale"], e24_shape, e24_params, d_out, P.lse, e24_ws, s)
        else:
            def compute(d_in, d_out, s):
                P.run(**d_in, bias=bias, stream=s, out=d_out)

        runner = OverlappedSteps(host, out_dev, compute)
        flush_i = [0]

        def before(s):
            with torch.cuda.stream(s):
                flush.fill_(flush_i[0] & 0xFF)
            flush_i[0] += 1

        for _ in range(max(1, args.warmup)):
            runner.step(before)
        runner.sync()
        if world > 1:
            dist.barrier()
        e_s.record(runner.s_in)
        for _ in range(args.steps):
            runner.step(before)
        e_e.record(runner.s_out)
        runner.sync()
        e_ms = e_s.elapsed_time(e_e)
        # the host link alone: the same copies and schedule with no kernels
        copies = OverlappedSteps(host, out_dev, lambda d_in, d_out, s: None)
        for _ in range(max(1, args.warmup)):
            copies.step()
        copies.sync()
        c_s, c_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c_s.record(copies.s_in)
        for _ in range(args.steps):
            copies.step()
        c_e.record(copies.s_out)
        copies.sync()
        copy_ms = c_s.elapsed_time(c_e) / args.steps
    else:
        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            e_s.record(stream)
            e2e_step()
            e_e.record(stream)
            torch.cuda.synchronize()
            e_ms += e_s.elapsed_time(e_e)
    e_ms = max_over_ranks(e_ms, world)
    e2e_value = whole_job_value(ops, world, e_ms / args.steps)

    if rank != 0:
        return 0
    peaks = _peaks()
    attn_avg_ms = sum(attn_ms) / len(attn_ms)
    roofline = prefill_roofline(wl, attn_avg_ms, ops, bias is not None, peaks, unit_peaks,
                                qb.v_ld(wl.Nk))
    if roofline["bound"] == "tensor":
        roofline["traffic"] = _attn_traffic(args.workload)
        roofline["traffic_unit"] = "bytes per launch (ncu dram read + write)"
    if args.intsoftmax:  # the integer softmax dominates: an ALU roofline
        # algorithmic integer operations per score: S - m, ShiftExp2's five
        # (quotient, remainder, halving, + X0, shift), requantization's three
        # (multiply, shift, clamp), the row-sum add and the max compare
        int_ops = INTSM_OPS_PER_SCORE * wl.unmasked_pairs()
        alu_tops = int_ops / (attn_avg_ms * 1e-3) / 1e12
        alu_peak = NUM_SMS * INT32_LANES_PER_SM * SM_MAX_GHZ / 1e3
        roofline = {"bound": "alu", "kernel": "intsm_attn_kernel (qattn_fwd_intsoftmax)",
                    "achieved": alu_tops, "peak": alu_peak, "unit": "TOP/s (int32)",
                    "frac": alu_tops / alu_peak,
                    "peak_basis": (f"{NUM_SMS} SMs x {INT32_LANES_PER_SM} int32 lanes per clock "
                                   f"(64 ALU-pipe + 64 FMA-pipe, from ncu pipe counters) x "
                                   f"{SM_MAX_GHZ} GHz"),
                    "algorithmic_ops": int_ops, "ops_per_score": INTSM_OPS_PER_SCORE,
                    "tensor_tops": ops / (attn_avg_ms * 1e-3) / 1e12,
                    "traffic": None}
    if args.exact24:  # three exact fp16 tensor-core products per attention product
        mma_tflops = 3 * ops / (attn_avg_ms * 1e-3) / 1e12
        pb = peaks["bf16"]
        if unit_peaks is not None:
            pb = max(pb, unit_peaks["f16"])
        roofline = {"bound": "tensor",
                    "kernel": "exact24_tc_kernel + q_split/k_rows_f16/v_t_f16 (qattn_fwd_exact24)",
                    "achieved": mma_tflops, "peak": pb, "unit": "TFLOP/s", "frac": mma_tflops / pb,
                    "peak_basis": "the stricter of the cuBLAS bf16 burst figure and the tcgen05 "
                                  "kind::f16 loop (fp16 MMA runs at the bf16 rate); achieved counts "
                                  "the 3 fp16 products per attention product",
                    "traffic": None}
    if decode and not args.exact24:  # memory-bound: the cache's bytes over the decode call's time
        gbs = cache_bytes / (attn_avg_ms * 1e-3) / 1e9
        ref_us = _stream_ref_us(dev["K_codes"], dev["V_codes"], flush, stream)
        roofline = {"bound": "hbm", "kernel": "qattn_decode (2 launches: fused scores + PV over key chunks, chunk combine)",
                    "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": gbs / peaks["hbm_gbs"],
                    "peak_basis": f"{peaks['source']} HBM copy rate",
                    "algorithmic_bytes": cache_bytes, "traffic": None,
                    "stream_ref": {"op": "torch.sum over one buffer holding the cache's bytes (as fp32), "
                                         "same L2 flush before each launch",
                                   "us": ref_us, "GB/s": cache_bytes / (ref_us * 1e-6) / 1e9}}
    cpu = None
    if not args.no_cpu_baseline:
        if args.exact24 or args.intsoftmax:
            c_ops, c_s, cores, desc = time_cpu_mode_baseline(
                "intsoftmax" if args.intsoftmax else "exact24", args.workload)
        else:
            c_ops, c_s, cores, desc = time_cpu_budgeted(args.workload, 1, 1, CPU_BASELINE_S)
        cpu = {"value": c_ops / c_s / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{desc}; {c_s:.1f} s"}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": ("int8 codes, int32 integer softmax" if args.intsoftmax
                      else "int8 cache codes, fp16 exact parts, fp32" if args.exact24 else "int8+e4m3"),
            "data": "synthetic",
            "config": {**_config(args.workload),
                       **({"mode": "24-bit exact split (qattn_fwd_exact24)",
                           "step": "split Q, attention with exact fp16 products"} if args.exact24 else {}),
                       **({"mode": "integer-only softmax (qattn_fwd_intsoftmax)",
                           "step": "per-tensor int8 codes of bf16 Q, K, V (qattn_quantize_qk), "
                                   "integer-only attention",
                           "granularity": "tensor", "kv_input": "bf16",
                           "output": "int8 codes"} if args.intsoftmax else {})},
            "attn_kernel_ms": attn_avg_ms,
            "roofline": roofline, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "schedule": ("overlapped: step i's host-to-device copies, step i-1's kernels "
                                 "and step i-2's device-to-host copy in flight together "
                                 "(pipeline.OverlappedSteps); L2 flush inside the timed interval"
                                 if overlapped else "serial: copies in, kernels, copy out"),
                    **({"copy_only_ms_per_step": copy_ms,
                        "copy_bound_value": world * ops / (copy_ms * 1e-3) / 1e12}
                       if copy_ms else {})},
            "gpu_launches": (ism.kernel_launches() if args.intsoftmax else 2 if args.exact24
                             else P.decode_launches(append=True) if decode
                             else P.kernel_launches()) * args.steps,
            "clocks": clk.summary(),
            "unit_peaks": {k: ({"rate": v["rate"], "unit": v["unit"], "sm_mhz": v["sm_mhz"],
                                "per_sm_per_clk": v["per_sm_per_clk"]} if isinstance(v, dict) else v)
                           for k, v in unit_rates.items()}}
    if not (args.exact24 or args.intsoftmax or decode or args.no_workloads):
        # the other prefill workloads, device-timed with fewer steps each
        subs = {}
        for name in SUB_WORKLOADS:
            if name == args.workload:
                continue
            subs[name] = time_prefill_workload(name, min(args.steps, 20), args.warmup, flush,
                                               stream, local, peaks, unit_peaks)
        line["workloads"] = subs
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# prefill workloads timed beside the main one (sub-records of the line)
SUB_WORKLOADS = ("llm8k", "chunk32k", "vit", "swin", "tiny")

# GB300 unit counts for the ALU roofline of the integer-only mode
NUM_SMS = 152
INT32_LANES_PER_SM = 128
SM_MAX_GHZ = 2.07
INTSM_OPS_PER_SCORE = 11


def _stream_ref_us(k_codes, v_codes, flush, stream, reps=20):
    """Device time of one library streaming read (torch.sum over the bytes
    viewed as fp32, its vectorized reduction) of a buffer with the cache's
    bytes, after the same L2 flush as the timed steps: what a plain read of
    these bytes costs at this size, launch and ramp included."""
    import torch
    buf = torch.cat([k_codes.reshape(-1), v_codes.reshape(-1)])
    evs = []
    for i in range(reps + 3):
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        buf.view(torch.float32).sum()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs[3:]]
    return sum(ms) / len(ms) * 1e3


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="llm8k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other prefill workloads' sub-records")
    ap.add_argument("--no-unit-peaks", action="store_true",
                    help="skip the tcgen05 / mma.sync / MUFU rate loops (profiling runs)")
    ap.add_argument("--intsoftmax", action="store_true",
                    help="time QFlash's integer-only attention (qattn_fwd_intsoftmax) with "
                         "per-tensor int8 codes of bf16 Q, K, V")
    ap.add_argument("--exact24", action="store_true",
                    help="time the 24-bit exact split mode (qattn_fwd_exact24) on an int8-cache workload")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return reference_arm(args)
    return gpu_arm(args)


if __name__ == "__main__":
    sys.exit(main())
