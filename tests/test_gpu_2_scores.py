"""The int32 score tiles from the tensor-core path (int8 codes carried
exactly in fp16, fp32 accumulation) equal the exact integer products."""
import numpy as np
import pytest
import torch

from oracle import qattn_oracle as O
from quantized_attention_gb300 import binding as qb
from tests.gpu_common import ensure_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def _gpu_scores(q, k):
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    shape = qb.make_shape(B, Hq, Hkv, Nq, Nk, d)
    ws = torch.empty(max(qb.workspace_size(shape, qb.make_params()), 256), dtype=torch.uint8,
                     device="cuda")
    S = torch.full((B, Hq, Nq, Nk), -7, dtype=torch.int32, device="cuda")
    qb.debug_qk_scores(torch.from_numpy(q).cuda(), torch.from_numpy(k).cuda(), shape, S, ws)
    torch.cuda.synchronize()
    assert qb.get_error() == 0
    return S.cpu().numpy()


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d", [
    (1, 1, 1, 128, 128, 64), (1, 1, 1, 256, 384, 128), (1, 2, 1, 197, 300, 128),
    (2, 4, 2, 49, 49, 32), (1, 3, 3, 1, 1, 64), (1, 2, 2, 130, 129, 32), (3, 8, 2, 64, 200, 128),
])
def test_random_codes(B, Hq, Hkv, Nq, Nk, d):
    rng = np.random.default_rng(B * 1000 + Nq + Nk + d)
    q = rng.integers(-127, 128, size=(B, Hq, Nq, d)).astype(np.int8)
    k = rng.integers(-127, 128, size=(B, Hkv, Nk, d)).astype(np.int8)
    assert np.array_equal(_gpu_scores(q, k), O.qk_scores(q, k))


@pytest.mark.parametrize("d", [32, 64, 128])
def test_extreme_magnitudes(d):
    """|S| up to d * 127^2 = 2,064,512 (d = 128) and partial sums that grow to
    half of that before cancelling: exact only if the accumulator keeps every
    integer below 2^21 exactly."""
    q = np.full((1, 1, 128, d), 127, np.int8)
    k = np.full((1, 1, 128, d), 127, np.int8)
    q[0, 0, 1::2] = -127
    k[0, 0, 2::3, : d // 2] = -127
    q[0, 0, 5, : d // 2] = 127
    q[0, 0, 5, d // 2:] = -127
    k[0, 0, 7] = np.arange(d) % 255 - 127
    q[0, 0, 9] = 1
    S = _gpu_scores(q, k)
    ref = O.qk_scores(q, k)
    assert np.abs(ref).max() == d * 127 * 127
    assert np.array_equal(S, ref)
