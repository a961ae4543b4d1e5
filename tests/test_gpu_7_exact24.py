"""qattn_fwd_exact24 (24-bit exact split attention on an int8 KV cache) against
the oracle's attn_exact24, and against dense fp64 attention on the dequantized
cache (the mode's accuracy class, ~2e-6 on the Strata PR's measurements)."""
import numpy as np
import pytest
import torch

from oracle import qattn_oracle as O
from quantized_attention_gb300 import binding as qb
from quantized_attention_gb300 import inputs as I
from tests.gpu_common import ensure_library

pytestmark = pytest.mark.gpu
TOL = 5e-6  # max |gpu - ref| / max |ref|: the oracle differs only by exp2 (fp64 vs ex2.approx)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


CASES = [
    I.small("chunk32k", Hq=8, Hkv=2, Nq=100, Nk=700, q_pos0=None),
    I.small("chunk32k", B=2, Hq=4, Hkv=4, Nq=70, Nk=333, q_pos0=None, d=64, causal=False),
    I.small("chunk32k", Hq=4, Hkv=1, Nq=128, Nk=1000, q_pos0=500),   # tokens mid-cache
]


def _ids(w):
    return f"B{w.B}-H{w.Hq}/{w.Hkv}-q{w.Nq}-k{w.Nk}-d{w.d}-c{int(w.causal)}"


def _run(wl, inp):
    dev = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x)).to(device="cuda", dtype=dt)
    shape = qb.make_shape(wl.B, wl.Hq, wl.Hkv, wl.Nq, wl.Nk, wl.d)
    params = qb.make_params(causal=wl.causal, q_pos0=wl.q_pos0)
    O_ = torch.empty((wl.B, wl.Hq, wl.Nq, wl.d), dtype=torch.float32, device="cuda")
    lse = torch.empty((wl.B, wl.Hq, wl.Nq), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(qb.workspace_size(shape, params), 256), dtype=torch.uint8, device="cuda")
    qb.fwd_exact24(dev(inp.Q, torch.bfloat16), dev(inp.K_codes, torch.int8),
                   dev(inp.K_scale, torch.float32), dev(inp.V_codes, torch.int8),
                   dev(inp.V_scale, torch.float32), shape, params, O_, lse, ws)
    torch.cuda.synchronize()
    assert qb.get_error() == 0
    return O_.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("wl", CASES, ids=[_ids(w) for w in CASES])
def test_exact24_matches_oracle(wl):
    inp = I.make_inputs(wl)
    got, lse = _run(wl, inp)
    want, want_lse = O.attn_exact24(inp.Q, inp.K_codes, inp.K_scale, inp.V_codes, inp.V_scale,
                                    causal=wl.causal, q_pos0=wl.q_pos0)
    got = got.reshape(want.shape)
    assert np.abs(got - want).max() <= TOL * np.abs(want).max(), _ids(wl)
    lse = lse.reshape(want_lse.shape)
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], want_lse[fin], rtol=0, atol=1e-5)


def test_exact24_against_fp64_attention():
    wl = CASES[0]
    inp = I.make_inputs(wl)
    got, _ = _run(wl, inp)
    K = inp.K_codes.astype(np.float64) * inp.K_scale[:, :, None, :]
    V = inp.V_codes.astype(np.float64) * inp.V_scale[:, :, None, :]
    ref = O.attn_fp64(inp.Q, K, V, causal=wl.causal, q_pos0=wl.q_pos0)
    got = got.reshape(ref.shape)
    assert np.abs(got - ref).max() <= TOL * np.abs(ref).max()


def test_exact24_full_chunk_shape_sampled():
    """The Strata PR's shape: 2048 queries against 32768 cached keys (32/8
    heads, d 128, causal from position 30720); sampled heads and rows."""
    wl = I.WORKLOADS["chunk32k"]
    inp = I.make_inputs(wl)
    got, _ = _run(wl, inp)
    heads = [(0, 0), (0, 13), (0, 31)]
    rows = np.array([0, 1, 777, 2047])
    want, _ = O.attn_exact24(inp.Q, inp.K_codes, inp.K_scale, inp.V_codes, inp.V_scale,
                             causal=wl.causal, q_pos0=wl.q_pos0, heads=heads, rows=rows)
    sub = np.stack([got[0, h][rows] for (_, h) in heads])
    assert np.abs(sub - want).max() <= TOL * np.abs(want).max()


def test_exact24_no_keys():
    """An empty cache (Nk = 0): the oracle gives out = 0 and lse = -inf for
    every row; the call writes exactly that over poisoned outputs."""
    wl = I.small("chunk32k", Hq=4, Hkv=2, Nq=70, Nk=0, q_pos0=0)
    inp = I.make_inputs(wl)
    want, want_lse = O.attn_exact24(inp.Q, inp.K_codes, inp.K_scale, inp.V_codes, inp.V_scale,
                                    causal=wl.causal, q_pos0=wl.q_pos0)
    dev = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x)).to(device="cuda", dtype=dt)
    shape = qb.make_shape(wl.B, wl.Hq, wl.Hkv, wl.Nq, 0, wl.d)
    params = qb.make_params(causal=wl.causal, q_pos0=wl.q_pos0)
    O_ = torch.full((wl.B, wl.Hq, wl.Nq, wl.d), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((wl.B, wl.Hq, wl.Nq), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(qb.workspace_size(shape, params), 256), dtype=torch.uint8, device="cuda")
    qb.fwd_exact24(dev(inp.Q, torch.bfloat16), dev(inp.K_codes, torch.int8),
                   dev(inp.K_scale, torch.float32), dev(inp.V_codes, torch.int8),
                   dev(inp.V_scale, torch.float32), shape, params, O_, lse, ws)
    torch.cuda.synchronize()
    assert qb.get_error() == 0
    assert np.array_equal(O_.cpu().numpy().reshape(want.shape), want)
    assert np.array_equal(lse.cpu().numpy().reshape(want_lse.shape), want_lse)


def test_exact24_cache_capacity_and_bf16_out():
    """The cache holds capacity > Nk rows (qattn_params.kv_capacity), the rows past Nk
    filled with extreme codes the call must not read; the fp32 output matches the
    oracle on the first Nk rows, and the bf16 output is the fp32 one rounded."""
    wl = I.small("chunk32k", Hq=4, Hkv=2, Nq=130, Nk=300, q_pos0=170)
    inp = I.make_inputs(wl)
    cap = 448
    dev = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x)).to(device="cuda", dtype=dt)
    Kc = np.full((wl.B, wl.Hkv, cap, wl.d), 127, dtype=np.int8)
    Vc = np.full((wl.B, wl.Hkv, cap, wl.d), -128, dtype=np.int8)
    Kc[:, :, :wl.Nk] = inp.K_codes
    Vc[:, :, :wl.Nk] = inp.V_codes
    shape = qb.make_shape(wl.B, wl.Hq, wl.Hkv, wl.Nq, wl.Nk, wl.d)
    outs = {}
    for out_dt, tdt in ((qb.DT_F32, torch.float32), (qb.DT_BF16, torch.bfloat16)):
        params = qb.make_params(causal=wl.causal, q_pos0=wl.q_pos0, kv_capacity=cap, out_dtype=out_dt)
        O_ = torch.full((wl.B, wl.Hq, wl.Nq, wl.d), float("nan"), dtype=tdt, device="cuda")
        ws = torch.empty(max(qb.workspace_size(shape, params), 256), dtype=torch.uint8, device="cuda")
        qb.fwd_exact24(dev(inp.Q, torch.bfloat16), dev(Kc, torch.int8), dev(inp.K_scale, torch.float32),
                       dev(Vc, torch.int8), dev(inp.V_scale, torch.float32), shape, params, O_, None, ws)
        torch.cuda.synchronize()
        assert qb.get_error() == 0
        outs[out_dt] = O_
    want, _ = O.attn_exact24(inp.Q, inp.K_codes, inp.K_scale, inp.V_codes, inp.V_scale,
                             causal=wl.causal, q_pos0=wl.q_pos0)
    got = outs[qb.DT_F32].cpu().numpy().astype(np.float64).reshape(want.shape)
    assert np.abs(got - want).max() <= TOL * np.abs(want).max()
    assert torch.equal(outs[qb.DT_BF16], outs[qb.DT_F32].to(torch.bfloat16))
