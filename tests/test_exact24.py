"""Pins of the oracle's 24-bit exact split mode (Strata PR, "What it does":
both operands of QK^T and PV split into three exact 8-bit parts, X = h*65536 +
l*256 + m; "Measured": ~2e-6 max relative error against FP64).  CPU only."""
import os
import types

import numpy as np
import pytest

from oracle import qattn_oracle as O

SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "qattn_oracle.py")
TOL = 5e-6  # max |O - O_fp64| / max |O_fp64|; the page reports ~2e-6


def _case(seed, B=1, Hq=4, Hkv=2, Nq=12, Nk=300, d=128):
    rng = np.random.default_rng(seed)
    Q = rng.normal(size=(B, Hq, Nq, d)).astype(np.float32)
    Q = (Q.view(np.uint32) & 0xFFFF0000).view(np.float32)  # bf16 values
    kc = np.clip(np.rint(rng.normal(size=(B, Hkv, Nk, d)) * 28), -127, 127).astype(np.int8)
    vc = np.clip(np.rint(rng.normal(size=(B, Hkv, Nk, d)) * 28), -127, 127).astype(np.int8)
    sk = rng.uniform(0.02, 0.06, size=(B, Hkv, d)).astype(np.float32)
    sv = rng.uniform(0.02, 0.06, size=(B, Hkv, d)).astype(np.float32)
    return Q, kc, sk, vc, sv


def _fp64(Q, kc, sk, vc, sv, causal):
    K = kc.astype(np.float64) * sk[:, :, None, :]
    V = vc.astype(np.float64) * sv[:, :, None, :]
    return O.attn_fp64(Q, K, V, causal=causal)


def test_split24_reconstructs_exactly_and_parts_are_bytes():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-127, 127, 20000), [127.0, -127.0, 0.0, 1e-6, -1e-6,
                                                         0.5 / 65536, 126.99999]]).astype(np.float32)
    h, l, m = O.split24(x)
    X = np.rint((x * np.float32(65536)).astype(np.float32)).astype(np.int64)
    assert np.array_equal(h * 65536 + l * 256 + m, X)
    assert h.min() >= -127 and h.max() <= 127
    assert l.min() >= -128 and l.max() <= 127
    assert m.min() >= 0 and m.max() <= 255


@pytest.mark.parametrize("causal", [False, True])
def test_exact24_matches_fp64_attention(causal):
    """Against dense fp64 attention on the dequantized cache (codes x channel
    scales): the page's accuracy class (~2e-6), both mask modes, GQA."""
    Q, kc, sk, vc, sv = _case(1)
    out, lse = O.attn_exact24(Q, kc, sk, vc, sv, causal=causal)
    ref = _fp64(Q, kc, sk, vc, sv, causal)
    assert np.abs(out - ref).max() / np.abs(ref).max() <= TOL


def test_exact24_lse_matches_fp64():
    Q, kc, sk, vc, sv = _case(2, Nk=200)
    _, lse = O.attn_exact24(Q, kc, sk, vc, sv, causal=False)
    K = kc.astype(np.float64) * sk[:, :, None, :]
    s = np.einsum("bhqd,bhkd->bhqk", Q.astype(np.float64),
                  np.repeat(K, Q.shape[1] // K.shape[1], axis=1)) / np.sqrt(Q.shape[3])
    want = np.log(np.exp(s - s.max(-1, keepdims=True)).sum(-1)) + s.max(-1)
    np.testing.assert_allclose(lse, want.reshape(lse.shape), rtol=0, atol=2e-5)


def test_fully_masked_rows_give_zero():
    """Causal rows that see no key (q_pos0 < 0) output 0 with lse -inf."""
    Q, kc, sk, vc, sv = _case(3, Nq=4, Nk=70)
    out, lse = O.attn_exact24(Q, kc, sk, vc, sv, causal=True, q_pos0=-2)
    assert np.all(out[:, :2] == 0) and np.all(np.isneginf(lse[:, :2]))
    assert np.all(np.isfinite(lse[:, 2:]))


def _mutant(old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"anchor not found: {old!r}"
    mod = types.ModuleType("qattn_oracle_exact24_mutant")
    exec(compile(src.replace(old, new, 1), SRC, "exec"), mod.__dict__)
    return mod


MUTATIONS = [
    ("Oc = (ph @ vcb) + (pl @ vcb) / 256.0 + (pm @ vcb) / 65536.0",
     "Oc = (ph @ vcb) + (pl @ vcb) / 256.0"),                                  # a part dropped
    ("np.float32(sg / 256) * Sl", "np.float32(sg / 65536) * Sl"),            # wrong part weight
    ("O = alpha[:, None] * O + sp.astype(np.float64)[:, None] * Oc",
     "O = O + sp.astype(np.float64)[:, None] * Oc"),                          # no rescale
    ("cfac = np.float32(np.float32(sm_scale) * LOG2E_F32)\n    if q_pos0 is None:\n        q_pos0 = Nk - Nq\n    heads = heads",
     "cfac = np.float32(sm_scale)\n    if q_pos0 is None:\n        q_pos0 = Nk - Nq\n    heads = heads"),  # log2 e dropped
]


@pytest.mark.parametrize("old,new", MUTATIONS, ids=[m[1][:30] for m in MUTATIONS])
def test_planted_mistakes_fail_the_fp64_pin(old, new):
    mod = _mutant(old, new)
    Q, kc, sk, vc, sv = _case(1)
    out, _ = mod.attn_exact24(Q, kc, sk, vc, sv, causal=True)
    ref = _fp64(Q, kc, sk, vc, sv, True)
    assert np.abs(out - ref).max() / np.abs(ref).max() > TOL
