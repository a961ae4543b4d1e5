"""Pre-passes on the GPU are bit-identical to the oracle: channel mean,
int8 codes and scales of Q and K (every granularity, bf16 K and int8-cache
K), e4m3 V bytes (transposed, zero-padded) and V scales."""
import numpy as np
import pytest
import torch

from oracle import qattn_oracle as O
from quantized_attention_gb300 import inputs as I
from tests.gpu_common import ensure_library, run_gpu
from tests.parity import e4m3_bytes_to_values

pytestmark = pytest.mark.gpu

CASES = [
    I.WORKLOADS["tiny"],
    I.small("vit", B=3),
    I.small("vit", B=2, q_gran=I.GRAN_HEAD, k_gran=I.GRAN_HEAD),
    I.small("swin", B=5),
    I.small("llm8k", Hq=4, Hkv=2, Nq=640, Nk=640),
    I.small("llm8k", Hq=2, Hkv=1, Nq=333, Nk=333, d=64),
    I.small("chunk32k", Hq=4, Hkv=2, Nq=256, Nk=1024, q_pos0=768),
    I.small("chunk32k", Hq=2, Hkv=2, Nq=100, Nk=301, q_pos0=201, d=32),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


@pytest.mark.parametrize("wl", CASES, ids=[w.name + f"-N{w.Nk}-d{w.d}-g{w.q_gran}" for w in CASES])
def test_prepasses_bit_exact(wl):
    inp = I.make_inputs(wl)
    prep = O.prepare(inp)
    P = run_gpu(wl, inp)
    if not wl.kv_codes:
        assert np.array_equal(P.k_mean.cpu().numpy().view(np.uint32), prep["mu"].view(np.uint32))
        assert np.array_equal(P.k_codes.cpu().numpy(), prep["k_codes"])
    assert np.array_equal(P.q_codes.cpu().numpy(), prep["q_codes"])
    assert np.array_equal(P.q_scales.cpu().numpy().view(np.uint32),
                          np.ascontiguousarray(prep["q_scales"]).ravel().view(np.uint32))
    assert np.array_equal(P.k_scales.cpu().numpy().view(np.uint32),
                          np.ascontiguousarray(prep["k_scales"]).ravel().view(np.uint32))
    v8t = P.v8t.cpu()
    vals = e4m3_bytes_to_values(v8t)
    assert np.array_equal(vals[..., : wl.Nk].transpose(0, 1, 3, 2), prep["v8"])
    assert not v8t[..., wl.Nk:].any(), "V padding must be zero"
    assert np.array_equal(P.v_scales.cpu().numpy().view(np.uint32), prep["s_v"].view(np.uint32))


def test_channel_mean_edge_values():
    """Channel mean on bf16 patterns that exercise the fixed-point rounding:
    values below 2^-17 (rounded to the 2^-24 grid, ties to even), subnormals,
    zeros of both signs, and magnitudes up to 2^18."""
    from quantized_attention_gb300 import binding as qb

    rng = np.random.default_rng(21)
    B, H, N, d = 1, 2, 300, 32
    sign = rng.integers(0, 2, size=(B, H, N, d)).astype(np.uint32) << 15
    exp = rng.integers(0, 146, size=(B, H, N, d)).astype(np.uint32)
    exp[..., :4] = rng.integers(95, 112, size=(B, H, N, 4))  # the rounding region
    mant = rng.integers(0, 128, size=(B, H, N, d)).astype(np.uint32)
    bits = (sign | (exp << 7) | mant).astype(np.uint32)
    K = (bits << 16).view(np.float32).reshape(B, H, N, d)
    mu_ref = O.smooth_k(K)
    shape = qb.make_shape(B, H, H, 8, N, d)
    ws = torch.empty(max(qb.workspace_size(shape, qb.make_params()), 256), dtype=torch.uint8,
                     device="cuda")
    Kd = torch.from_numpy(K.copy()).to("cuda").to(torch.bfloat16)
    mu = torch.empty((B, H, d), dtype=torch.float32, device="cuda")
    for _ in range(2):  # the workspace accumulators must be cleared on every call
        qb.smooth_k(Kd, shape, mu, ws)
        torch.cuda.synchronize()
        assert np.array_equal(mu.cpu().numpy().view(np.uint32), mu_ref.view(np.uint32))
