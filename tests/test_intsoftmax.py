"""Pins of the oracle's QFlash integer-only attention ("QFlash", sections
4.2-4.6 and Algorithm 1).  ScaleRelease's definition (its Appendix B.1) is not
in the pages, so the multi-tile rescaling is a reading and stays unpinned;
these pins fix everything else.  CPU only."""
import os
import types

import numpy as np
import pytest

from oracle import qattn_oracle as O

SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "qattn_oracle.py")


def _case(seed, B=1, H=3, N=197, d=64, sig=2.0):
    rng = np.random.default_rng(seed)
    Q = rng.normal(size=(B, H, N, d)) * sig
    K = rng.normal(size=(B, H, N, d)) * sig
    V = rng.normal(size=(B, H, N, d))
    sq, sk, sv = (np.float32(np.abs(x).max() / 127) for x in (Q, K, V))
    code = lambda x, s: np.clip(np.rint(x / s), -127, 127).astype(np.int8)
    return code(Q, sq), sq, code(K, sk), sk, code(V, sv), sv


def test_constants():
    for sq, sk, d in ((0.02, 0.02, 64), (3 / 127, 5 / 127, 32), (1e-3, 2e-3, 128)):
        st, x0, M, r = O.intsm_constants(sq, sk, O.default_sm_scale(d))
        assert abs(x0 * float(st) - 1) <= float(st) / 2 + 1e-7      # X0 = rint(1 / s~)
        assert 128 < M <= 256                                         # n = ceil(log2(127 s~))
        assert abs(M / 2.0 ** r - 127 * float(st)) <= 2.0 ** -r / 2   # M = rint(127 s~ 2^r)


def test_shift_exp2_at_powers_of_two_and_error_bound():
    st, x0, _, _ = O.intsm_constants(0.02, 0.02, O.default_sm_scale(64))
    k = np.arange(0, 20)
    assert np.array_equal(O.shift_exp2(-k * x0, x0), x0 >> k)       # R = 0: exact shifts
    X = -np.arange(0, 6 * x0)
    approx = O.shift_exp2(X, x0).astype(np.float64) * float(st)
    exact = 2.0 ** (float(st) * X)
    # 2^r ~ r/2 + 1 on (-1, 0] is off by at most 6.15%; the integer floors add 2^-Q / X0
    bound = 0.0615 + 2.0 ** (np.ceil(X / -x0)) / x0
    assert np.all(np.abs(approx - exact) <= exact * bound + 1e-12)
    assert np.all(np.diff(O.shift_exp2(X, x0)[::-1]) >= 0)             # monotonic in X


def test_requant_maps_one_to_the_top_code():
    for sq, sk in ((0.02, 0.02), (0.05, 0.01)):
        _, x0, M, r = O.intsm_constants(sq, sk, O.default_sm_scale(64))
        top = int(O.requant_p(np.array([x0]), M, r)[0])
        assert top in (126, 127)
        P = np.arange(0, x0 + 1)
        Y = O.requant_p(P, M, r)
        assert np.all(np.diff(Y) >= 0) and np.abs(Y - P * 127.0 / x0).max() <= 1.5


def test_requant_with_a_negative_shift_saturates():
    """s~ > 2 (coarse scales): ratio = 127 s~ > 256, so n > 8 and r < 0; every
    P >= 1 is worth more than 127 codes and saturates, P = 0 stays 0."""
    st, x0, M, r = O.intsm_constants(4.0, 4.0, 0.125)
    assert float(st) > 2 and r < 0 and x0 == 1
    assert O.requant_p(np.array([0, 1, 2, 5]), M, r).tolist() == [0, 127, 127, 127]
    assert np.floor(1 * 127 * float(st)) > 127


def test_single_tile_against_python_integers():
    """One key tile: no rescale happens; Python-integer loops give the same
    codes (exp by the page's decomposition, requantization, floor division)."""
    qc, sq, kc, sk, vc, sv = _case(3, H=1, N=40, d=32)
    out = O.attn_intsoftmax(qc, sq, kc, sk, vc)
    _, x0, M, r = O.intsm_constants(sq, sk, O.default_sm_scale(32))
    for i in range(0, 40, 7):
        S = [int(sum(int(a) * int(b) for a, b in zip(qc[0, 0, i], kc[0, 0, j]))) for j in range(40)]
        m = max(S)
        Y = []
        for s in S:
            X = s - m
            q = -((-X) // x0)
            R = X - q * x0
            p = ((R >> 1) + x0) >> min(-q, 62)
            Y.append(min((p * M) >> r, 127))
        l = sum(Y)
        for c in range(0, 32, 5):
            o = sum(y * int(vc[0, 0, j, c]) for j, y in enumerate(Y))
            assert out[0, i, c] == max(-127, min(127, o // l))


def _err(out, vc, sv, qc, sq, kc, sk):
    ref = O.attn_fp64(qc.astype(float) * sq, kc.astype(float) * sk, vc.astype(float) * sv, causal=False)
    o = out.reshape(ref.shape) * float(sv)
    return np.abs(o - ref).max() / float(sv), 10 * np.log10((ref ** 2).sum() / ((o - ref) ** 2).sum())


@pytest.mark.parametrize("d,N", [(64, 197), (32, 49)])
def test_matches_fp64_softmax_within_the_approximation(d, N):
    """Against dense fp64 attention on the dequantized codes: each weight is
    off by at most the ShiftExp2 bound (6.15%) and the requantization step, so
    the output code is within 0.15 * max|v| + 2 of the exact one."""
    qc, sq, kc, sk, vc, sv = _case(4, N=N, d=d)
    out = O.attn_intsoftmax(qc, sq, kc, sk, vc)
    maxcode, sqnr = _err(out, vc, sv, qc, sq, kc, sk)
    assert maxcode <= 0.15 * np.abs(vc).max() + 2
    assert sqnr >= 20.0


MUTATIONS = [
    ("q = -((-X) // x0)                  # truncation toward zero for X <= 0",
     "q = X // x0"),                                                      # floor, R in [0, X0)
    ("O = scale_release(O, alpha[:, None], x0) + Y @ v[k0:k0 + INTSM_TILE]",
     "O = O + Y @ v[k0:k0 + INTSM_TILE]"),                               # no rescale of O
]


@pytest.mark.parametrize("old,new", MUTATIONS, ids=["floor-div", "no-rescale"])
def test_planted_mistakes_fail(old, new):
    src = open(SRC).read()
    assert old in src
    mod = types.ModuleType("qattn_oracle_intsm_mutant")
    exec(compile(src.replace(old, new, 1), SRC, "exec"), mod.__dict__)
    # a key block late in the row with the row's largest scores: the running
    # max rises in the last tile, so a missing rescale shows
    qc, sq, kc, sk, vc, sv = _case(5, N=197, d=64)
    kc = kc.copy()
    kc[:, :, 180:] = np.clip(qc[:, :, :17] * 3, -127, 127)
    try:
        out = mod.attn_intsoftmax(qc, sq, kc, sk, vc)
    except Exception:
        return  # a crash also counts as caught
    good = O.attn_intsoftmax(qc, sq, kc, sk, vc)
    maxcode, sqnr = _err(out, vc, sv, qc, sq, kc, sk)
    maxcode_g, sqnr_g = _err(good, vc, sv, qc, sq, kc, sk)
    assert sqnr < sqnr_g - 3 or maxcode > 0.15 * np.abs(vc).max() + 2
