"""Fused attention output on the GPU against the oracle, element by element,
at sizes the oracle finishes in seconds: several tiles, ragged tails, GQA,
causal alignment, bias, every head dim, and the degenerate cases."""
import numpy as np
import pytest

from oracle import qattn_oracle as O
from quantized_attention_gb300 import binding as qb
from quantized_attention_gb300 import inputs as I
from tests.gpu_common import ensure_library, gpu_lse_rows, gpu_out_rows, run_gpu
from tests.parity import check_output, rel_err_vs_fp64

pytestmark = pytest.mark.gpu

CASES = [
    I.WORKLOADS["tiny"],
    I.small("vit", B=3),
    I.small("vit", B=2, q_gran=I.GRAN_HEAD, k_gran=I.GRAN_HEAD),
    I.small("swin", B=6),
    I.small("llm8k", Hq=4, Hkv=2, Nq=640, Nk=640),
    I.small("llm8k", Hq=2, Hkv=1, Nq=333, Nk=333, d=64),
    I.small("llm8k", Hq=2, Hkv=2, Nq=300, Nk=300, d=32),
    I.small("llm8k", Hq=2, Hkv=1, Nq=200, Nk=400, q_pos0=100),      # pos0 not on a block edge
    I.small("llm8k", Hq=2, Hkv=1, Nq=300, Nk=100),                  # Nq > Nk: early rows see nothing
    I.small("llm8k", Hq=1, Hkv=1, Nq=1, Nk=1, d=64),                # single token
    I.small("llm8k", Hq=2, Hkv=1, Nq=1, Nk=777),                    # one query (decode-shaped row)
    I.small("llm8k", Hq=2, Hkv=1, Nq=255, Nk=255),                  # one row short of two tiles
    I.small("llm8k", B=2, Hq=8, Hkv=1, Nq=200, Nk=200),             # eight query heads per KV head
    I.small("tiny", causal=False, Nq=3, Nk=1000),                   # few rows, many keys
    I.small("chunk32k", Hq=4, Hkv=2, Nq=256, Nk=1024, q_pos0=768),
    I.small("chunk32k", Hq=2, Hkv=2, Nq=100, Nk=301, q_pos0=201, d=32),
    # bias read from global memory: several key blocks with a ragged last one,
    # every head dim, causal and not (the shared-memory copy covers Swin)
    I.small("tiny", has_bias=True, Nq=300, Nk=300),
    I.small("swin", B=2, Nq=200, Nk=200),
    I.small("tiny", has_bias=True, d=128, Nq=130, Nk=257, causal=True),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def _ids(w):
    return f"{w.name}-B{w.B}-H{w.Hq}/{w.Hkv}-{w.Nq}x{w.Nk}-d{w.d}-c{int(w.causal)}"


@pytest.mark.parametrize("wl", CASES, ids=[_ids(w) for w in CASES])
def test_output_matches_oracle(wl):
    inp = I.make_inputs(wl)
    prep = O.prepare(inp)
    P = run_gpu(wl, inp)
    heads = [(b, h) for b in range(wl.B) for h in range(wl.Hq)][:16]
    rows = np.arange(wl.Nq)
    ref = O.run_workload(inp, prep, heads=heads, rows=rows, want_bound=True)
    gpu = gpu_out_rows(P, heads, rows)
    stats = check_output(gpu, ref["O"], ref["bound"], _ids(wl))
    lse = gpu_lse_rows(P, heads, rows)
    fin = np.isfinite(ref["lse"])
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], ref["lse"][fin], rtol=0, atol=1e-4)
    K, V = O.real_kv(inp)
    ref64 = O.attn_fp64(inp.Q, K, V, causal=wl.causal, q_pos0=wl.q_pos0, bias=inp.bias,
                        heads=heads, rows=rows)
    print(f"{_ids(wl)}: {stats}; rel err vs fp64 {rel_err_vs_fp64(gpu, ref64):.3e}")


def test_bf16_output():
    wl = I.small("llm8k", Hq=2, Hkv=1, Nq=384, Nk=384)
    inp = I.make_inputs(wl)
    prep = O.prepare(inp)
    P32 = run_gpu(wl, inp)
    P16 = run_gpu(wl, inp, out_dtype=qb.DT_BF16)
    heads = [(0, 0), (0, 1)]
    rows = np.arange(wl.Nq)
    o32 = gpu_out_rows(P32, heads, rows)
    o16 = gpu_out_rows(P16, heads, rows)
    # the bf16 output is the fp32 output rounded to nearest even
    import torch
    want = torch.from_numpy(o32.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(o16, want)


def test_repeat_calls_identical():
    wl = I.small("llm8k", Hq=2, Hkv=1, Nq=256, Nk=256)
    inp = I.make_inputs(wl)
    a = run_gpu(wl, inp).O.cpu().numpy()
    b = run_gpu(wl, inp).O.cpu().numpy()
    assert np.array_equal(a, b)


@pytest.mark.parametrize("wl", [I.small("llm8k", Hq=4, Hkv=2, Nq=384, Nk=384),
                                I.small("chunk32k", Hq=2, Hkv=1, Nq=128, Nk=512, q_pos0=384),
                                I.small("swin", B=3)],
                         ids=["llm8k", "chunk32k", "swin"])
def test_without_k_carrier_identical(wl):
    """qattn_fwd converting the K codes itself (no carrier from
    qattn_quantize_qk) gives bit-identical outputs, and the carriers
    qattn_quantize_qk writes are the K codes as fp16."""
    import torch
    inp = I.make_inputs(wl)
    a = run_gpu(wl, inp, k_carrier=True)
    b = run_gpu(wl, inp, k_carrier=False)
    assert np.array_equal(a.O.cpu().numpy(), b.O.cpu().numpy())
    assert np.array_equal(a.lse.cpu().numpy(), b.lse.cpu().numpy())
    codes = a._k_codes.to(torch.float16)
    assert torch.equal(a.k_carrier.view(torch.int16), codes.view(torch.int16))


INT8_PV_CASES = [
    I.small("llm8k", Hq=4, Hkv=2, Nq=640, Nk=640),
    I.small("llm8k", Hq=2, Hkv=1, Nq=333, Nk=333, d=64),
    I.small("llm8k", Hq=2, Hkv=2, Nq=300, Nk=300, d=32),
    I.small("vit", B=2),
    I.small("chunk32k", Hq=4, Hkv=2, Nq=256, Nk=1024, q_pos0=768),
]


@pytest.mark.parametrize("wl", INT8_PV_CASES, ids=[_ids(w) for w in INT8_PV_CASES])
def test_int8_pv_ablation_matches_oracle(wl):
    """pv_mode = QATTN_PV_INT8: P quantized as rint(127 P) (the int8 PV the ZINC
    post rejects), against the oracle's int8 mode, with the same 2e-3 gate and
    its flip allowance for codes next to a rounding midpoint."""
    inp = I.make_inputs(wl)
    prep = O.prepare(inp)
    P = run_gpu(wl, inp, pv_mode=qb.PV_INT8)
    heads = [(b, h) for b in range(wl.B) for h in range(wl.Hq)][:8]
    rows = np.arange(wl.Nq)
    ref = O.run_workload(inp, prep, heads=heads, rows=rows, want_bound=True, p_quant="int8")
    check_output(gpu_out_rows(P, heads, rows), ref["O"], ref["bound"], _ids(wl))
    lse = gpu_lse_rows(P, heads, rows)
    fin = np.isfinite(ref["lse"])
    np.testing.assert_allclose(lse[fin], ref["lse"][fin], rtol=0, atol=1e-4)
    # and it is not the e4m3 recipe
    e4 = O.run_workload(inp, prep, heads=heads, rows=rows)["O"]
    assert np.abs(gpu_out_rows(P, heads, rows) - e4).max() > 1e-3


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("out_dtype", [qb.DT_F32, qb.DT_BF16])
def test_no_keys(causal, out_dtype):
    """Nk = 0: every row is fully masked.  The oracle gives out = 0 and
    lse = -inf; the call writes exactly that over poisoned outputs and reads
    no K, V or workspace buffer."""
    import torch
    wl = I.small("tiny", Hq=2, Hkv=1, Nq=100, Nk=0, causal=causal)
    inp = I.make_inputs(wl)
    prep = O.prepare(inp)
    ref = O.run_workload(inp, prep)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    odt = torch.bfloat16 if out_dtype == qb.DT_BF16 else torch.float32
    out = torch.full((wl.B, wl.Hq, wl.Nq, wl.d), float("nan"), dtype=odt, device="cuda")
    lse = torch.full((wl.B, wl.Hq, wl.Nq), 7.0, dtype=torch.float32, device="cuda")
    qb.fwd(dev(prep["q_codes"]), dev(prep["q_scales"]), None, None, None, qb.v_ld(0), None, None,
           qb.make_shape(wl.B, wl.Hq, wl.Hkv, wl.Nq, 0, wl.d),
           qb.make_params(causal=causal, q_gran=wl.q_gran, k_gran=wl.k_gran, out_dtype=out_dtype),
           out, lse, None)
    torch.cuda.synchronize()
    assert qb.get_error() == 0
    assert np.array_equal(out.float().cpu().numpy().reshape(ref["O"].shape), ref["O"])
    assert np.array_equal(lse.cpu().numpy().reshape(ref["lse"].shape), ref["lse"])


NO_KEY_CASES = [
    I.small("tiny", Nq=77, Nk=0),                                 # bf16 K/V, block granules
    I.small("vit", B=2, Nq=50, Nk=0),                             # per-tensor granules
    I.small("chunk32k", Hq=4, Hkv=2, Nq=64, Nk=0, q_pos0=0),      # an empty int8 cache
]


@pytest.mark.parametrize("wl", NO_KEY_CASES, ids=[_ids(w) for w in NO_KEY_CASES])
def test_no_keys_through_the_pipeline(wl):
    """Nk = 0 through the public path (quantize, then attend): Q's codes and
    scales as the oracle's, every row fully masked (out = 0, lse = -inf)."""
    import torch
    from quantized_attention_gb300.pipeline import device_inputs, problem_for
    inp = I.make_inputs(wl)
    prep = O.prepare(inp)
    ref = O.run_workload(inp, prep)
    P = problem_for(wl, want_lse=True)
    P.O.fill_(float("nan"))
    P.lse.fill_(7.0)
    dev = device_inputs(inp)
    bias = dev.pop("bias", None)
    P.run(**dev, bias=bias)
    torch.cuda.synchronize()
    assert qb.get_error() == 0
    assert np.array_equal(P.q_codes.cpu().numpy().reshape(prep["q_codes"].shape), prep["q_codes"])
    assert np.array_equal(P.q_scales.cpu().numpy().ravel(), prep["q_scales"].ravel())
    assert np.array_equal(P.O.float().cpu().numpy().reshape(ref["O"].shape), ref["O"])
    assert np.array_equal(P.lse.cpu().numpy().reshape(ref["lse"].shape), ref["lse"])
