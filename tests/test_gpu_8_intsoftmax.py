"""qattn_fwd_intsoftmax (QFlash's integer-only attention) against the oracle's
attn_intsoftmax: every step is integer arithmetic, so the int8 output codes
must match bit for bit, on the ViT/DeiT and Swin-window shapes."""
import numpy as np
import pytest
import torch

from oracle import qattn_oracle as O
from quantized_attention_gb300 import binding as qb
from quantized_attention_gb300 import inputs as I
from tests.gpu_common import ensure_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


CASES = [
    I.small("vit", B=2, Hq=3, Hkv=3),                       # DeiT-Tiny heads, N 197, d 64
    I.small("vit", B=1, Hq=12, Hkv=12),                     # ViT-Base heads
    I.small("swin", B=16, Hq=3, Hkv=3, has_bias=False),     # Swin stage-1 windows, N 49, d 32
    I.small("vit", B=1, Hq=4, Hkv=2, Nq=100, Nk=300),       # GQA, ragged tiles
    I.small("vit", B=1, Hq=2, Hkv=2, Nq=70, Nk=150, d=128),
    I.small("vit", B=1, Hq=2, Hkv=1, Nq=300, Nk=129),       # 3 CTAs per head; a 1-key tail tile
    I.small("vit", B=1, Hq=1, Hkv=1, Nq=1, Nk=1, d=32),      # one row, one key
]


def _ids(w):
    return f"B{w.B}-H{w.Hq}/{w.Hkv}-q{w.Nq}-k{w.Nk}-d{w.d}"


def _tensor_codes(x):
    s = np.float32(np.abs(x).max() / np.float32(127.0))
    return np.clip(np.rint(x / s), -127, 127).astype(np.int8), s


def _run(wl, qc, sq, kc, sk, vc, fill=0):
    dev = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x)).to(device="cuda", dtype=dt)
    out = torch.full((wl.B, wl.Hq, wl.Nq, wl.d), fill, dtype=torch.int8, device="cuda")
    qb.fwd_intsoftmax(dev(qc, torch.int8), dev(np.array([sq], np.float32), torch.float32),
                      dev(kc, torch.int8), dev(np.array([sk], np.float32), torch.float32),
                      dev(vc, torch.int8), qb.make_shape(wl.B, wl.Hq, wl.Hkv, wl.Nq, wl.Nk, wl.d),
                      qb.make_params(), out)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.int64)


def _check(got, want):
    got = got.reshape(want.shape)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:3].tolist()}"


@pytest.mark.parametrize("wl", CASES, ids=[_ids(w) for w in CASES])
def test_intsoftmax_bit_exact(wl):
    inp = I.make_inputs(wl)
    qc, sq = _tensor_codes(inp.Q * 2.0)   # sharper rows than N(0, 1) scores give
    kc, sk = _tensor_codes(inp.K * 2.0)
    vc, _ = _tensor_codes(inp.V)
    want = O.attn_intsoftmax(qc, sq, kc, sk, vc)
    got = _run(wl, qc, sq, kc, sk, vc)
    assert qb.get_error() == 0
    _check(got, want)


@pytest.mark.parametrize("wl", [CASES[0], CASES[2], CASES[3]], ids=["deit", "swin", "gqa"])
def test_library_codes_then_intsoftmax_bit_exact(wl):
    """The whole QFlash path from bf16 activations: the library's per-tensor
    int8 codes of Q, K and V (QFlash, section 4, eq. (1)-(2)) equal the
    oracle's quantizer bit for bit, and the integer-only attention on them
    equals the oracle's on the oracle's codes."""
    from quantized_attention_gb300.pipeline import QFlashProblem, device_inputs
    inp = I.make_inputs(wl)
    dev = device_inputs(inp)
    P = QFlashProblem(wl.B, wl.Hq, wl.Hkv, wl.Nq, wl.Nk, wl.d)
    P.run(dev["Q"], dev["K"], dev["V"])
    torch.cuda.synchronize()
    assert qb.get_error() == 0
    want = {}
    for name, x, codes, scale in (("Q", inp.Q, P.q_codes, P.q_scale), ("K", inp.K, P.k_codes, P.k_scale),
                                  ("V", inp.V, P.v_codes, P.v_scale)):
        c, s = O.quantize_sym(x, O.GRAN_TENSOR)
        assert np.array_equal(codes.cpu().numpy(), c), name
        assert np.float32(scale.item()) == np.float32(np.asarray(s).reshape(-1)[0]), name
        want[name] = (c, np.float32(np.asarray(s).reshape(-1)[0]))
    ref = O.attn_intsoftmax(want["Q"][0], want["Q"][1], want["K"][0], want["K"][1], want["V"][0])
    _check(P.O.cpu().numpy().astype(np.int64), ref)


def test_intsoftmax_coarse_scales_bit_exact():
    """s~ > 2: X0 = 1 and the requantization shift is negative (every P >= 1
    saturates); the rescale runs with alpha in {0, 1}."""
    wl = CASES[0]
    inp = I.make_inputs(wl)
    qc, _ = _tensor_codes(inp.Q)
    kc, _ = _tensor_codes(inp.K)
    vc, _ = _tensor_codes(inp.V)
    want = O.attn_intsoftmax(qc, np.float32(4.0), kc, np.float32(4.0), vc)
    got = _run(wl, qc, np.float32(4.0), kc, np.float32(4.0), vc)
    assert qb.get_error() == 0
    _check(got, want)


def test_intsoftmax_fine_scales_bit_exact():
    """Fine scales: X0 ~ 2.2e7 > 2^23, so P * M needs 64 bits (the kernel's
    wide requantization path)."""
    wl = CASES[3]
    inp = I.make_inputs(wl)
    qc, _ = _tensor_codes(inp.Q)
    kc, _ = _tensor_codes(inp.K)
    vc, _ = _tensor_codes(inp.V)
    sq = sk = np.float32(5e-4)
    _, x0, _, _ = O.intsm_constants(sq, sk, O.default_sm_scale(wl.d))
    assert x0 > 2 ** 23
    want = O.attn_intsoftmax(qc, sq, kc, sk, vc)
    got = _run(wl, qc, sq, kc, sk, vc)
    assert qb.get_error() == 0
    _check(got, want)


def test_intsoftmax_scales_outside_the_domain_flagged():
    """1/s~ above 2^30: the kernel writes nothing and the error word reports
    an invalid argument (the scales live on the device)."""
    wl = CASES[0]
    inp = I.make_inputs(wl)
    qc, _ = _tensor_codes(inp.Q)
    kc, _ = _tensor_codes(inp.K)
    vc, _ = _tensor_codes(inp.V)
    got = _run(wl, qc, np.float32(1e-6), kc, np.float32(1e-6), vc, fill=55)
    assert qb.get_error() == qb.ERR_INVALID_ARG
    assert np.all(got == 55)
    assert qb.get_error() == 0  # read and cleared


def test_intsoftmax_rejects_causal():
    p = qb.make_params(causal=True)
    z = torch.zeros(64 * 64, dtype=torch.int8, device="cuda")
    f = torch.ones(1, dtype=torch.float32, device="cuda")
    with pytest.raises(qb.QattnError):
        qb.fwd_intsoftmax(z, f, z, f, z, qb.make_shape(1, 1, 1, 64, 64, 64), p, z)
