"""qattn_prepare (the pre-pass in one or two launches) writes, byte for byte,
what qattn_smooth_k + qattn_quantize_qk + qattn_quantize_v write: the K mean,
Q/K codes and scales, K's fp16 carriers, V's transposed e4m3 codes and scales
-- with block granules, and with tensor granules for heads of at most 256
keys (d 32 or 64)."""
import pytest
import torch

from quantized_attention_gb300 import binding as qb
from quantized_attention_gb300 import inputs as I
from quantized_attention_gb300.pipeline import device_inputs, problem_for
from tests.gpu_common import ensure_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


CASES = [
    I.small("llm8k", Hq=8, Hkv=2, Nq=1000, Nk=1000),      # GQA, d 128, ragged blocks
    I.small("llm8k", Hq=4, Hkv=4, Nq=130, Nk=2100, d=64),  # Nq != Nk, many mean chunks
    I.small("swin", B=3, Hq=3, Hkv=3, has_bias=False),     # d 32, N 49: short heads
    I.small("vit", B=2, Hq=2, Hkv=1, Nq=197, Nk=197),      # tensor-granule workload at block granules
    I.small("swin", B=5, Hq=4, Hkv=2, Nq=128, Nk=100, d=64),  # short heads (one warp each), GQA, d 64
    I.small("swin", B=2, Hq=2, Hkv=2, Nq=7, Nk=1),         # short heads: one key
]


def _ids(w):
    return f"B{w.B}-H{w.Hq}/{w.Hkv}-q{w.Nq}-k{w.Nk}-d{w.d}"


OUTS = ("q_codes", "q_scales", "k_codes", "k_scales", "k_mean", "v8t", "v_scales", "k_carrier")


TENSOR_CASES = [
    I.small("vit", B=2, Hq=3, Hkv=3, Nq=197, Nk=197),          # the ViT head shape
    I.small("vit", B=3, Hq=4, Hkv=2, Nq=300, Nk=256, d=32),    # GQA, the longest keys, Nq > 256
    I.small("vit", B=2, Hq=2, Hkv=2, Nq=5, Nk=1),              # one key
    I.small("vit", B=1, Hq=2, Hkv=1, Nq=129, Nk=129, d=64),    # ragged past one 128-row block
]


def _check_prepare(wl, carrier):
    dev = device_inputs(I.make_inputs(wl))
    dev.pop("bias", None)
    res = []
    for fused in (False, True):
        P = problem_for(wl, k_carrier=carrier, fused_prepass=fused)
        assert P.fused_prepass == fused
        for name in OUTS:  # poison every output first
            t = getattr(P, name)
            if t is not None:
                t.view(torch.uint8).fill_(0xA5)
        P.quantize(**dev)
        torch.cuda.synchronize()
        assert qb.get_error() == 0
        res.append({n: getattr(P, n).clone() for n in OUTS if getattr(P, n) is not None})
    for n in res[0]:
        a, b = res[0][n].view(torch.uint8), res[1][n].view(torch.uint8)
        assert torch.equal(a, b), f"{n}: {int((a != b).sum())} bytes differ"


@pytest.mark.parametrize("wl", CASES, ids=[_ids(w) for w in CASES])
@pytest.mark.parametrize("carrier", [True, False])
def test_prepare_equals_three_calls(wl, carrier):
    _check_prepare(wl.replace(q_gran=qb.GRAN_BLOCK, k_gran=qb.GRAN_BLOCK), carrier)


@pytest.mark.parametrize("wl", TENSOR_CASES, ids=[_ids(w) for w in TENSOR_CASES])
@pytest.mark.parametrize("carrier", [True, False])
def test_prepare_tensor_granules_equals_three_calls(wl, carrier):
    wl = wl.replace(q_gran=qb.GRAN_TENSOR, k_gran=qb.GRAN_TENSOR)
    assert qb.prepare_launches(qb.make_shape(wl.B, wl.Hq, wl.Hkv, wl.Nq, wl.Nk, wl.d),
                               qb.make_params(q_gran=qb.GRAN_TENSOR, k_gran=qb.GRAN_TENSOR)) == 2
    _check_prepare(wl, carrier)


def test_prepare_rejects_other_granules():
    wl = CASES[0].replace(q_gran=qb.GRAN_HEAD)
    P = problem_for(wl, fused_prepass=False)
    dev = device_inputs(I.make_inputs(wl))
    with pytest.raises(qb.QattnError) as e:
        qb.prepare(dev["Q"], dev["K"], dev["V"], P.shape, P.params, P.q_codes, P.q_scales,
                   P.k_codes, P.k_scales, P.k_mean, P.v8t, P.ldv, P.v_scales, P.workspace)
    assert e.value.status == qb.ERR_UNSUPPORTED
