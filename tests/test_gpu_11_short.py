"""The warp-level kernel for short non-causal key sequences (qattn_fwd with
QATTN_FWD_SHORT; the automatic choice for the ViT/DeiT and Swin shapes)
against the oracle, and against the persistent tensor-core kernel on the same
quantized operands: the two compute the same recipe and differ only in the
order of fp32 accumulations."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import qattn_oracle as O
from quantized_attention_gb300 import binding as qb
from quantized_attention_gb300 import inputs as I
from quantized_attention_gb300.pipeline import device_inputs, problem_for
from tests.gpu_common import ensure_library, gpu_lse_rows, gpu_out_rows
from tests.parity import check_output

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


CASES = [
    I.small("vit", B=2, Hq=3, Hkv=3),                           # N 197: two key blocks
    I.small("swin", B=8, Hq=3, Hkv=3),                          # N 49, d 32, bias
    I.small("tiny"),                                            # N 256, block scales
    I.small("vit", B=1, Hq=4, Hkv=2, Nq=100, Nk=250, q_gran=2, k_gran=2),  # GQA, ragged
    I.small("vit", B=1, Hq=2, Hkv=2, Nq=30, Nk=129, d=32),      # one key in the 2nd block
    I.small("swin", B=2, Hq=2, Hkv=1, Nq=200, Nk=17),           # Nq > Nk, bias, 1 step of keys
    I.small("swin", B=3, Hq=2, Hkv=1, Nq=33, Nk=50),            # window kernel: GQA, Nq != Nk
    I.small("vit", B=4, Hq=2, Hkv=2, Nq=64, Nk=64),             # window kernel: d 64, full window
    I.small("vit", B=1, Hq=2, Hkv=1, Nq=255, Nk=255, d=32),     # one key short of the longest head
]


def _ids(w):
    return f"{w.name}-B{w.B}-H{w.Hq}/{w.Hkv}-q{w.Nq}-k{w.Nk}-d{w.d}"


def _run(wl, inp, kernel):
    P = problem_for(wl, out_dtype=qb.DT_F32, want_lse=True, fwd_kernel=kernel)
    dev = device_inputs(inp)
    bias = dev.pop("bias", None)
    P.run(**dev, bias=bias)
    torch.cuda.synchronize()
    assert qb.get_error() == 0
    return P


@pytest.mark.parametrize("wl", CASES, ids=[_ids(w) for w in CASES])
def test_short_kernel_parity(wl):
    inp = I.make_inputs(wl)
    prep = O.prepare(inp)
    heads = [(b, h) for b in range(wl.B) for h in range(wl.Hq)][:6]
    rows = np.arange(wl.Nq)
    ref = O.run_workload(inp, prep, heads=heads, rows=rows, want_bound=True)
    Ps = _run(wl, inp, qb.FWD_SHORT)
    got = gpu_out_rows(Ps, heads, rows)
    check_output(got, ref["O"], ref["bound"], _ids(wl))
    Pt = _run(wl, inp, qb.FWD_TC)
    tc = gpu_out_rows(Pt, heads, rows)
    scale = max(np.abs(tc).max(), 1e-30)
    assert np.abs(got - tc).max() <= 2e-6 * scale, _ids(wl)
    ls, lt = gpu_lse_rows(Ps, heads, rows), gpu_lse_rows(Pt, heads, rows)
    np.testing.assert_allclose(ls, lt, rtol=0, atol=2e-5)


BIAS_CASES = [
    I.small("swin", B=3, Hq=3, Hkv=3),                                  # N 49, d 32: the window kernel
    I.small("tiny", B=2, Hq=2, Hkv=1, Nq=130, Nk=200, has_bias=True),   # d 64, ragged blocks, GQA
]


@pytest.mark.parametrize("wl", BIAS_CASES, ids=[_ids(w) for w in BIAS_CASES])
@pytest.mark.parametrize("kernel", [qb.FWD_AUTO, qb.FWD_SHORT, qb.FWD_TC], ids=["auto", "short", "tc"])
def test_per_head_bias(wl, kernel):
    """A bias per head ([Hq][Nq][Nk], bias_head_stride = Nq Nk; the window
    kernel keeps a head index's bias fragments and refills them when the index
    changes): every head against the oracle run with that head's bias."""
    inp = I.make_inputs(wl)
    prep = O.prepare(inp)
    rng = np.random.default_rng(20241)
    bias3 = rng.standard_normal((wl.Hq, wl.Nq, wl.Nk)).astype(np.float32)
    P = problem_for(wl, out_dtype=qb.DT_F32, want_lse=True, fwd_kernel=kernel,
                    bias_head_stride=wl.Nq * wl.Nk)
    dev = device_inputs(inp)
    dev.pop("bias", None)
    P.run(**dev, bias=torch.from_numpy(bias3).to("cuda"))
    torch.cuda.synchronize()
    assert qb.get_error() == 0
    rows = np.arange(wl.Nq)
    for h in range(wl.Hq):
        heads = [(b, h) for b in range(wl.B)]
        ref = O.run_workload(dataclasses.replace(inp, bias=bias3[h]), prep, heads=heads, rows=rows,
                             want_bound=True)
        check_output(gpu_out_rows(P, heads, rows), ref["O"], ref["bound"], f"head {h}")


def test_short_kernel_is_the_automatic_choice():
    wl = CASES[1]
    inp = I.make_inputs(wl)
    a = _run(wl, inp, qb.FWD_AUTO)
    s = _run(wl, inp, qb.FWD_SHORT)
    assert torch.equal(a.O, s.O)


@pytest.mark.parametrize("kw", [dict(causal=True), dict(d=128)], ids=["causal", "d128"])
def test_short_kernel_rejects_other_shapes(kw):
    wl = I.small("tiny", **kw)
    P = problem_for(wl, fwd_kernel=qb.FWD_SHORT)
    dev = device_inputs(I.make_inputs(wl))
    with pytest.raises(qb.QattnError) as e:
        P.run(**dev)
    assert e.value.status == qb.ERR_UNSUPPORTED
