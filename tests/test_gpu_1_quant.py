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


MEAN_SHAPES = [(49, 32), (300, 32), (1000, 32), (30, 64), (197, 64), (700, 64), (16, 128),
               (128, 128), (640, 128)]


@pytest.mark.parametrize("N,d", MEAN_SHAPES, ids=[f"N{n}-d{d}" for n, d in MEAN_SHAPES])
def test_channel_mean_edge_values(N, d):
    """Channel mean on bf16 patterns that exercise the fixed-point rounding:
    values below 2^-17 (rounded to the 2^-24 grid, ties to even), subnormals,
    zeros of both signs, magnitudes up to 2^18, and a sparse sprinkling of
    magnitudes in [2^20, 2^24) (the kernels' wide-range decode).  The shapes
    cover one warp per head, one CTA per head and several CTAs per head."""
    from quantized_attention_gb300 import binding as qb

    rng = np.random.default_rng(21 + N + d)
    B, H = 1, 2
    sign = rng.integers(0, 2, size=(B, H, N, d)).astype(np.uint32) << 15
    exp = rng.integers(0, 146, size=(B, H, N, d)).astype(np.uint32)
    exp[..., :4] = rng.integers(95, 112, size=(B, H, N, 4))  # the rounding region
    wide = rng.random(size=(B, H, N, d)) < 0.01
    exp[wide] = rng.integers(147, 151, size=int(wide.sum()))
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


def _bf16_pieces(S: int) -> list:
    """Split the integer S (in units of 2^-24) into bf16 values whose
    round(x * 2^24) are exact and sum to S: each piece keeps the top 8 bits."""
    out, r = [], S
    while r != 0:
        a = abs(r)
        L = a.bit_length()
        p = a if L <= 8 else (a >> (L - 8)) << (L - 8)
        p = p if r > 0 else -p
        out.append(p)
        r -= p
    return out


@pytest.mark.parametrize("N", [7, 49, 300, 1000])
def test_channel_mean_rounding_midpoints(N):
    """Channel means whose exact value S / Nk lies at or next to an fp32
    rounding midpoint (ties to even, and one or two units either side), in
    magnitudes from 2^-20 to 2^25: the kernels' integer division must round
    exactly as the definition's fp64 route does."""
    from quantized_attention_gb300 import binding as qb

    rng = np.random.default_rng(1234 + N)
    B, H, d = 1, 8, 32
    K = np.zeros((B, H, N, d), dtype=np.float32)
    for h in range(H):
        for c in range(d):
            e = int(rng.integers(-20, 26))
            k = int(rng.integers(2 ** 23, 2 ** 24))
            num = N * (2 * k + 1)  # N * b * 2^(24 - e), b the midpoint
            A = (num << e) if e >= 0 else round(num / 2 ** (-e))
            A += int(rng.integers(-2, 3))
            A = min(max(A, 1), 2 ** 53 - 1)
            S = A if rng.random() < 0.5 else -A
            pieces = _bf16_pieces(S)
            rows = rng.choice(N, size=len(pieces), replace=False)
            for r, p in zip(rows, pieces):
                K[0, h, r, c] = np.float32(p) * np.float32(2.0 ** -24)
    bits = K.view(np.uint32)
    assert not (bits & 0xFFFF).any(), "every piece must be a bf16 value"
    mu_ref = O.smooth_k(K)
    shape = qb.make_shape(B, H, H, 8, N, d)
    ws = torch.empty(max(qb.workspace_size(shape, qb.make_params()), 256), dtype=torch.uint8,
                     device="cuda")
    Kd = torch.from_numpy(K.copy()).to("cuda").to(torch.bfloat16)
    mu = torch.empty((B, H, d), dtype=torch.float32, device="cuda")
    qb.smooth_k(Kd, shape, mu, ws)
    torch.cuda.synchronize()
    assert np.array_equal(mu.cpu().numpy().view(np.uint32), mu_ref.view(np.uint32))
