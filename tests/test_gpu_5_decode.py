"""Decode on an int8 KV cache (qattn_decode) against the oracle's recipe on the
same codes: a few query tokens per head, long caches with a ragged last
block, GQA groups, both head dims, and the full 32K-key decode shape on
sampled heads."""
import numpy as np
import pytest
import torch

from oracle import qattn_oracle as O
from quantized_attention_gb300 import binding as qb
from quantized_attention_gb300 import inputs as I
from quantized_attention_gb300.pipeline import device_inputs, problem_for
from tests.gpu_common import ensure_library
from tests.parity import check_output

pytestmark = pytest.mark.gpu

CASES = [
    I.small("chunk32k", Hq=8, Hkv=2, Nq=1, Nk=4173, q_pos0=None),
    I.small("chunk32k", Hq=8, Hkv=2, Nq=2, Nk=1500, q_pos0=None),
    I.small("chunk32k", Hq=4, Hkv=1, Nq=4, Nk=700, q_pos0=None, d=64),
    I.small("chunk32k", Hq=2, Hkv=2, Nq=1, Nk=100, q_pos0=None),
    I.small("chunk32k", Hq=8, Hkv=4, Nq=3, Nk=2048, q_pos0=1000),  # tokens mid-cache
    I.small("chunk32k", Hq=16, Hkv=2, Nq=2, Nk=1100, q_pos0=None),  # 16 rows per KV head
]

# Enough key blocks that pass 2 gives each CTA a chunk of several blocks, so the
# accumulators are rescaled as the running max grows inside a chunk.
LONG_CASES = [
    I.small("chunk32k", Hq=32, Hkv=16, Nq=8, Nk=8192, q_pos0=None),          # 16 rows, d 128
    I.small("chunk32k", Hq=16, Hkv=16, Nq=1, Nk=16384, q_pos0=None, d=64),   # 1 row, d 64
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def _ids(w):
    return f"H{w.Hq}/{w.Hkv}-q{w.Nq}-k{w.Nk}-d{w.d}-p{w.pos0}"


def run_decode(wl, inp, out_dtype=qb.DT_F32):
    P = problem_for(wl, out_dtype=out_dtype, want_lse=True)
    dev = device_inputs(inp)
    P.quantize(**dev)
    amax = torch.empty(dev["V_scale"].shape, dtype=torch.float32, device="cuda")
    qb.kv_header_init(dev["V_codes"], wl.Nk, amax)
    ws = torch.empty(max(qb.workspace_size(P.shape, P.params), 256), dtype=torch.uint8,
                     device="cuda")
    qb.decode(P.q_codes, P.q_scales, dev["K_codes"], P.k_scales, dev["V_codes"],
              dev["V_scale"], amax, P.shape, P.params, P.O, P.lse, ws)
    torch.cuda.synchronize()
    assert qb.get_error() == 0
    return P


@pytest.mark.parametrize("wl", CASES, ids=[_ids(w) for w in CASES])
def test_decode_matches_oracle(wl):
    inp = I.make_inputs(wl)
    prep = O.prepare(inp)
    P = run_decode(wl, inp)
    heads = [(b, h) for b in range(wl.B) for h in range(wl.Hq)]
    rows = np.arange(wl.Nq)
    ref = O.run_workload(inp, prep, heads=heads, rows=rows, want_bound=True)
    gpu = P.O.cpu().numpy().reshape(len(heads), wl.Nq, wl.d).astype(np.float64)
    check_output(gpu, ref["O"], ref["bound"], _ids(wl))
    lse = P.lse.cpu().numpy().reshape(len(heads), wl.Nq).astype(np.float64)
    fin = np.isfinite(ref["lse"])
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], ref["lse"][fin], rtol=0, atol=1e-4)


@pytest.mark.parametrize("wl", LONG_CASES, ids=[_ids(w) for w in LONG_CASES])
def test_decode_multi_block_chunks_sampled_heads(wl):
    inp = I.make_inputs(wl)
    prep = O.prepare(inp)
    P = run_decode(wl, inp)
    G = wl.Hq // wl.Hkv
    picked = [0, 1, wl.Hq - G, wl.Hq - 1]  # both ends of the first and last KV groups
    heads = [(0, h) for h in picked]
    ref = O.run_workload(inp, prep, heads=heads, rows=np.arange(wl.Nq), want_bound=True)
    gpu = P.O.cpu().numpy().reshape(wl.Hq, wl.Nq, wl.d)[picked].astype(np.float64)
    check_output(gpu, ref["O"], ref["bound"], _ids(wl))


def test_decode_32k_full_shape_sampled_heads():
    """The decode32k shape: 32 query heads / 8 KV heads, one token against
    32768 cached int8 keys; every head checked against the oracle."""
    wl = I.WORKLOADS["decode32k"]
    inp = I.make_inputs(wl)
    prep = O.prepare(inp)
    P = run_decode(wl, inp)
    heads = [(0, h) for h in range(wl.Hq)]
    ref = O.run_workload(inp, prep, heads=heads, rows=np.arange(wl.Nq), want_bound=True)
    gpu = P.O.cpu().numpy().reshape(len(heads), wl.Nq, wl.d).astype(np.float64)
    check_output(gpu, ref["O"], ref["bound"], "decode32k")
    # the bf16 output the bench times is the fp32 output rounded to bf16
    P16 = run_decode(wl, inp, out_dtype=qb.DT_BF16)
    got16 = P16.O.float().cpu().numpy().reshape(gpu.shape).astype(np.float64)
    want16 = torch.from_numpy(gpu.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got16, want16)


def test_decode_same_as_prefill_kernel():
    """qattn_decode and qattn_fwd (after qattn_quantize_v) on the same codes."""
    wl = I.small("chunk32k", Hq=8, Hkv=2, Nq=2, Nk=3000, q_pos0=None)
    inp = I.make_inputs(wl)
    Pd = run_decode(wl, inp)
    P = problem_for(wl, want_lse=True)
    dev = device_inputs(inp)
    P.run(**dev)
    torch.cuda.synchronize()
    a, b = Pd.O.cpu().numpy(), P.O.cpu().numpy()
    assert np.abs(a - b).max() <= 2e-3 * np.abs(b).max()


def test_decode_ignores_workspace_contents():
    """The chunk records and the unit counter carry a per-call tag, so the
    workspace needs no clearing: zeros, 0xFF bytes, random bytes or a previous
    call's records for another shape give bit-identical outputs."""
    wl = I.small("chunk32k", Hq=8, Hkv=2, Nq=2, Nk=5000, q_pos0=None)
    inp = I.make_inputs(wl)
    P = problem_for(wl, want_lse=True)
    dev = device_inputs(inp)
    P.quantize(**dev)
    amax = torch.empty(dev["V_scale"].shape, dtype=torch.float32, device="cuda")
    qb.kv_header_init(dev["V_codes"], wl.Nk, amax)
    n = max(qb.workspace_size(P.shape, P.params), 256)

    def run(ws):
        qb.decode(P.q_codes, P.q_scales, dev["K_codes"], P.k_scales, dev["V_codes"],
                  dev["V_scale"], amax, P.shape, P.params, P.O, P.lse, ws)
        torch.cuda.synchronize()
        assert qb.get_error() == 0
        return P.O.clone(), P.lse.clone()

    gen = torch.Generator(device="cuda").manual_seed(5)
    fills = [torch.zeros(n, dtype=torch.uint8, device="cuda"),
             torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda"),
             torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=gen)]
    o0, l0 = run(fills[0])
    for ws in fills[1:]:
        o, l = run(ws)
        assert torch.equal(o, o0) and torch.equal(l, l0)
    # the same workspace after a decode of another shape, then twice in a row
    other = I.small("chunk32k", Hq=4, Hkv=1, Nq=4, Nk=3000, q_pos0=None)
    run_decode(other, I.make_inputs(other))  # its own workspace; then reuse ours below
    ws = fills[2]
    for _ in range(2):
        o, l = run(ws)
        assert torch.equal(o, o0) and torch.equal(l, l0)
