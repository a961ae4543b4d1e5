"""Measured execution rates of the units the attention kernels use
(``qattn_peak_loop`` in libqattn.so, declared in include/qattn_peaks.h).

``measure()`` runs each loop on every SM of the current device for about
``target_ms`` and returns its rate, the SM clock it ran at (cycles counted in
the kernel over the event-timed duration) and the rate per SM per clock.  The
roofline of the fused attention combines the two tcgen05 rates: half of its
algorithmic operations (QK^T) run as kind::f16 and half (PV) as kind::f8f6f4,
so its peak is the harmonic combination ``mixed_peak``.
"""
from __future__ import annotations

import torch

from . import binding as qb

TC_F16, TC_F8, MMA_S8, MMA_F16, MMA_E4M3, EX2, TC_ATTN_MIX = range(7)

# name: (kind, n, operations per loop round and CTA, CTAs per SM, unit); the
# light loops first, so that the power-limited clock of the tcgen05 loops
# does not carry over into them
LOOPS = {
    "mufu_ex2": (EX2, 0, 256 * 8, 4, "Tex2/s"),
    "mma_sync_s8": (MMA_S8, 0, 8 * 8 * 2 * 16 * 8 * 32, 4, "TOP/s"),
    "mma_sync_f16": (MMA_F16, 0, 8 * 8 * 2 * 16 * 8 * 16, 4, "TFLOP/s"),
    "mma_sync_e4m3": (MMA_E4M3, 0, 8 * 8 * 2 * 16 * 8 * 32, 4, "TFLOP/s"),
    "tcgen05_f16_n128": (TC_F16, 128, 4 * 2 * 128 * 128 * 16, 1, "TFLOP/s"),
    "tcgen05_f16_n256": (TC_F16, 256, 4 * 2 * 128 * 256 * 16, 1, "TFLOP/s"),
    "tcgen05_f8_n128": (TC_F8, 128, 4 * 2 * 128 * 128 * 32, 1, "TFLOP/s"),
    "tcgen05_f8_n256": (TC_F8, 256, 4 * 2 * 128 * 256 * 32, 1, "TFLOP/s"),
    # the fused attention's per-block sequence: 8 f16 (QK^T) + 4 f8 (PV) MMAs
    "tcgen05_attn_mix": (TC_ATTN_MIX, 128, 8 * 2 * 128 * 128 * 16 + 4 * 2 * 128 * 128 * 32, 1,
                         "TFLOP/s"),
}


def _run(kind, n, iters, blocks, clocks, err, sink, stream):
    st = qb.lib().qattn_peak_loop(kind, n, iters, blocks, qb._p(clocks), qb._p(err), qb._p(sink),
                                  qb._stream(stream))
    if st != 0:
        raise RuntimeError(f"qattn_peak_loop(kind={kind}) returned {st}")


def measure(target_ms: float = 5.0, names=None) -> dict:
    """Rates of the loops in LOOPS (all by default) on the current device."""
    dev = torch.cuda.current_device()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    stream = torch.cuda.current_stream()
    out = {}
    for name in (names or LOOPS):
        kind, n, ops_round, per_sm, unit = LOOPS[name]
        blocks = sms * per_sm
        clocks = torch.zeros(4 * blocks, dtype=torch.int64, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        sink = torch.zeros(1, dtype=torch.int32, device="cuda")
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def timed(iters):
            a.record(stream)
            _run(kind, n, iters, blocks, clocks, err, sink, stream)
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b)

        iters = 256
        ms = timed(iters)  # first launch: calibration and warm-up
        iters = max(256, int(iters * target_ms / max(ms, 1e-3)))
        timed(iters)
        ms = timed(iters)
        if int(err.item()) != 0:
            raise RuntimeError(f"{name}: a completion wait ran out")
        c = clocks.view(blocks, 4).cpu()
        cyc = (c[:, 1] - c[:, 0]).double()
        ns = (c[:, 3] - c[:, 2]).double().clamp(min=1.0)
        mhz = float((cyc / ns).median()) * 1e3  # the clock the loops ran at
        ops = float(ops_round) * iters * blocks
        rate = ops / (ms * 1e-3)
        out[name] = {"rate": rate / 1e12, "unit": unit, "ms": ms, "sm_mhz": mhz,
                     "per_sm_per_clk": rate / sms / (mhz * 1e6),
                     "cta_span_of_elapsed": float(ns.median()) / (ms * 1e6)}
    return out


def mixed_peak(p_qk: float, p_pv: float) -> float:
    """Peak of a kernel whose algorithmic operations are half QK^T at rate
    p_qk and half PV at rate p_pv: 1 / (0.5 / p_qk + 0.5 / p_pv)."""
    return 1.0 / (0.5 / p_qk + 0.5 / p_pv)


def attention_peak(rates: dict) -> dict:
    """The fused attention's measured mixed peak from ``measure()``'s tcgen05
    rates (the best N of each kind)."""
    f16 = max(rates[k]["rate"] for k in rates if k.startswith("tcgen05_f16"))
    f8 = max(rates[k]["rate"] for k in rates if k.startswith("tcgen05_f8"))
    return {"f16": f16, "f8": f8, "mixed": mixed_peak(f16, f8)}
