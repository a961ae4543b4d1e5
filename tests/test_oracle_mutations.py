"""Planted mistakes in the oracle must be caught by its pins.

Each case copies the oracle's source, applies one plausible slip (a wrong
rounding rule, a dropped rescale, an off-by-one mask, a transposed head
mapping...), loads the copy as a separate module on the CPU and runs the pin
that is meant to catch it against the copy.  The real oracle is untouched.
"""
import importlib.util
import os
import types

import pytest

import tests.test_oracle_pins as P

SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "qattn_oracle.py")

MUTATIONS = [
    ("rint(a / step) * step", "floor(a / step + 0.5) * step", "test_e4m3_worked_cases"),
    ("q = np.minimum(q, P_SCALE)", "q = q", "test_e4m3_worked_cases"),
    ("F32(QMAX) / amax, F32(0)", "F32(128) / amax, F32(0)", "test_quantizer_hand_cases"),
    ("scale = (amax / F32(QMAX))", "scale = (amax / F32(128))", "test_quantizer_hand_cases"),
    ("/ F64(Nk)", "/ F64(Nk - 1)", "test_mean_exact_on_dyadic_values"),
    ("np.arange(Hq) // (Hq // Hkv)", "np.arange(Hq) % Hkv", "test_scores_match_python_loops"),
    ("O = alpha.astype(F64)[:, None] * O + Pq", "O = O + Pq", "test_blockwise_loop_equals_dense_softmax"),
    ("l = alpha.astype(F64) * l +", "l = l +", "test_blockwise_loop_equals_dense_softmax"),
    ("x = (t - m_new[:, None])", "x = (t - m_new[:, None] - 1)", "test_p_bounded_by_one_and_p8_by_448"),
    ("return k <= (q_pos0", "return k < (q_pos0", "test_blockwise_loop_equals_dense_softmax"),
    ("t = (t + bias2[:, k0:k1]", "t = (t - bias2[:, k0:k1]", "test_blockwise_loop_equals_dense_softmax"),
    ("(Kx - np.asarray(k_mean, dtype=F32)", "(Kx + np.asarray(k_mean, dtype=F32)", "test_smoothing_shrinks_outlier_channels_via_prepare"),
    ("F32(P_SCALE) / amax, F32(0)).astype(F32)\n    s_v", "F32(240) / amax, F32(0)).astype(F32)\n    s_v", "test_v_bf16_path"),
    # the static P scale: 240, or 127 with e4m3 rounding, instead of 448
    ("P448 = (P * ftype(P_SCALE)).astype(ftype)\n            Pq = e4m3_round(P448) / P_SCALE",
     "P448 = (P * ftype(240.0)).astype(ftype)\n            Pq = e4m3_round(P448) / 240.0",
     "test_static_p_scale_worked_cases"),
    ("P448 = (P * ftype(P_SCALE)).astype(ftype)\n            Pq = e4m3_round(P448) / P_SCALE",
     "P448 = (P * ftype(127.0)).astype(ftype)\n            Pq = e4m3_round(P448) / 127.0",
     "test_static_p_scale_worked_cases"),
    # flip allowance: a window too narrow to see the midpoints, half a step
    # per flip instead of a whole one, no rescale of the allowance by alpha
    ("window = 2.0 ** -20 * (4.0 + span) * Ps", "window = 2.0 ** -40 * (4.0 + span) * Ps",
     "test_flip_bound_covers_every_flip"),
    ("(amb * step / scale) @ absV", "(amb * step / scale / 2) @ absV", "test_flip_bound_covers_every_flip"),
    ("Bacc = alpha.astype(F64)[:, None] * Bacc +", "Bacc = Bacc +", "test_flip_bound_covers_every_flip"),
]


def _load_mutant(old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    src = src.replace(old, new, 1)
    spec = importlib.util.spec_from_loader("qattn_oracle_mutant", loader=None)
    mod = types.ModuleType(spec.name)
    exec(compile(src, SRC + " (mutant)", "exec"), mod.__dict__)
    return mod


def test_smoothing_shrinks_outlier_channels_via_prepare(O=None):
    """Smoothing as the recipe applies it (quantize_qk's K - mu) must shrink
    the outlier channels of the llm8k structure to <= 4.1x the median."""
    import numpy as np
    from quantized_attention_gb300 import inputs as I

    O = O or P.O
    wl = I.small("llm8k", Hq=1, Hkv=1, Nq=128, Nk=2048)
    inp = I.make_inputs(wl)
    mu = O.smooth_k(inp.K)
    _, _, kc, ks = O.quantize_qk(inp.Q, inp.K, k_mean=mu, q_gran=O.GRAN_TENSOR,
                                 k_gran=O.GRAN_TENSOR)
    amax = np.abs(kc[0, 0].astype(np.float64)).max(axis=0)
    assert amax.max() / np.median(amax) <= 4.1


@pytest.mark.parametrize("old,new,pin", MUTATIONS, ids=[f"{i}-{m[2]}" for i, m in enumerate(MUTATIONS)])
def test_planted_mistake_is_caught(old, new, pin):
    mutant = _load_mutant(old, new)
    if pin == "test_smoothing_shrinks_outlier_channels_via_prepare":
        with pytest.raises(AssertionError):
            test_smoothing_shrinks_outlier_channels_via_prepare(mutant)
        return
    fn = getattr(P, pin)
    saved = P.O
    P.O = mutant
    try:
        with pytest.raises(AssertionError):
            if pin == "test_blockwise_loop_equals_dense_softmax":
                for case in P.test_blockwise_loop_equals_dense_softmax.pytestmark[0].args[1]:
                    fn(case)
            elif pin == "test_flip_bound_covers_every_flip":
                mp = pytest.MonkeyPatch()
                try:
                    fn(mp)
                finally:
                    mp.undo()
            else:
                fn()
    finally:
        P.O = saved
