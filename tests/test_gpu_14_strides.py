"""The pre-pass reads its inputs at any strides: Q, K and V taken in place from
a packed projection output [B, N, 3, H, d] (a non-contiguous view per tensor)
give, byte for byte, the codes, scales, means and e4m3 V of the same tensors
made dense -- through qattn_prepare (two-launch, short-head and tensor-granule
paths) and through the three separate calls (per-tensor granules)."""
import numpy as np
import pytest
import torch

from quantized_attention_gb300 import binding as qb
from quantized_attention_gb300.pipeline import Problem
from tests.gpu_common import ensure_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


CASES = [  # B, H, N, d, granularity, fused pre-pass
    (2, 4, 300, 128, qb.GRAN_BLOCK, True),    # qattn_prepare, two launches
    (3, 2, 49, 32, qb.GRAN_BLOCK, True),      # qattn_prepare, one warp per head
    (2, 3, 197, 64, qb.GRAN_TENSOR, False),   # smooth_k, quantize_qk (two passes), quantize_v
    (1, 2, 260, 64, qb.GRAN_BLOCK, False),    # the three calls with block granules
    (2, 3, 197, 64, qb.GRAN_TENSOR, True),    # qattn_prepare, tensor granules
]


def _outputs(P):
    out = {"q_codes": P.q_codes, "q_scales": P.q_scales, "k_codes": P.k_codes,
           "k_scales": P.k_scales, "k_mean": P.k_mean, "v8t": P.v8t, "v_scales": P.v_scales}
    if P.k_carrier is not None:
        out["k_carrier"] = P.k_carrier
    return {k: v.clone() for k, v in out.items()}


@pytest.mark.parametrize("B,H,N,d,gran,fused", CASES,
                         ids=[f"B{c[0]}-H{c[1]}-N{c[2]}-d{c[3]}-g{c[4]}-{'prep' if c[5] else 'calls'}"
                              for c in CASES])
def test_packed_qkv_views_equal_dense_inputs(B, H, N, d, gran, fused):
    g = torch.Generator().manual_seed(B * 1000 + N + d)
    qkv = torch.randn((B, N, 3, H, d), generator=g).to(device="cuda", dtype=torch.bfloat16)
    qkv[:, :, 1, :, 5] += 6.0  # a K channel offset for the mean to remove
    views = [qkv[:, :, i].permute(0, 2, 1, 3) for i in range(3)]  # [B, H, N, d], strided
    assert not views[0].is_contiguous()
    res = []
    for inputs in (views, [v.contiguous() for v in views]):
        P = Problem(B, H, H, N, N, d, q_gran=gran, k_gran=gran, fused_prepass=fused)
        for t in (P.q_codes, P.k_codes, P.v8t):
            t.fill_(0x5A)  # stale bytes that must all be overwritten
        P.quantize(*inputs)
        torch.cuda.synchronize()
        assert qb.get_error() == 0
        res.append(_outputs(P))
    strided, dense = res
    for k in dense:
        assert torch.equal(strided[k].view(torch.uint8), dense[k].view(torch.uint8)), k
