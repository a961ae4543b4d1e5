"""Comparison helpers shared by the GPU parity tests (test code only)."""
import numpy as np
import torch

#: output gate: max relative error over |ref| > 1e-2 and max absolute error
REL_TOL = 2e-3
ABS_TOL = 2e-3
REL_FLOOR = 1e-2


def e4m3_bytes_to_values(t: torch.Tensor) -> np.ndarray:
    """uint8 e4m3 bytes -> float64 values (via torch's float8_e4m3fn view)."""
    return t.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()


def check_output(gpu: np.ndarray, ref: np.ndarray, bound: np.ndarray, what: str = ""):
    """Gate of the recipe's output: max relative error <= 2e-3 over
    |ref| > 1e-2 and max absolute error <= 2e-3, element by element.

    ``bound`` is the oracle's per-element flip allowance: the largest change
    that rounding the other way the e4m3 codes of 448 P that lie within the
    exp2 accuracy window of a rounding midpoint can cause (either rounding is
    a correct result of the recipe; the GPU's ex2.approx and NumPy's exp2
    may land on opposite sides).  The gate applies to the error beyond that
    allowance.  In addition, an element whose raw error breaks the gate must
    carry a positive allowance (a row with an ambiguous code): no raw excess
    is left unexplained.  Returns a dict of the observed errors.
    """
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    excess = np.maximum(err - bound, 0.0)
    big = np.abs(ref) > REL_FLOOR
    rel = float((excess[big] / np.abs(ref[big])).max(initial=0.0))
    absx = float(excess.max(initial=0.0))
    raw_over = (err > ABS_TOL) | (big & (err > REL_TOL * np.abs(ref)))
    stats = {"max_rel_beyond_flip_bound": rel, "max_abs_beyond_flip_bound": absx,
             "max_rel_raw": float((err[big] / np.abs(ref[big])).max(initial=0.0)),
             "max_abs_raw": float(err.max(initial=0.0)),
             "n_raw_over_gate": int(raw_over.sum()),
             "n_elems_with_flip_allowance": int((bound > 0).sum()), "n": int(err.size)}
    assert np.isfinite(gpu).all(), f"{what}: non-finite output"
    assert rel <= REL_TOL, f"{what}: relative error {rel:.3e} > {REL_TOL} ({stats})"
    assert absx <= ABS_TOL, f"{what}: absolute error {absx:.3e} > {ABS_TOL} ({stats})"
    unexplained = int((raw_over & (bound <= 0)).sum())
    assert unexplained == 0, f"{what}: {unexplained} raw errors over the gate without a flip ({stats})"
    return stats


def rel_err_vs_fp64(gpu: np.ndarray, ref64: np.ndarray) -> float:
    """max |gpu - ref| / max |ref| (reported, not gated)."""
    return float(np.abs(np.asarray(gpu, np.float64) - ref64).max() / max(np.abs(ref64).max(), 1e-30))
