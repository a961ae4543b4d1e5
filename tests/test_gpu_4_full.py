"""Every workload at its full size, in the launch configuration bench.py
times (same kernels, same grid; fp32 output for the 2e-3 gate, and the bf16
output checked to be the rounded fp32 output): quantized operands compared
in full, attention outputs on sampled heads and query tiles that the oracle
computes one by one."""
import numpy as np
import pytest
import torch

from oracle import qattn_oracle as O
from quantized_attention_gb300 import binding as qb
from quantized_attention_gb300 import inputs as I
from tests.gpu_common import ensure_library, gpu_out_rows, run_gpu
from tests.parity import check_output, e4m3_bytes_to_values, rel_err_vs_fp64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def _samples(wl):
    rng = np.random.default_rng(99)
    if wl.name == "tiny":
        return [(0, 0)], np.arange(wl.Nq)
    if wl.name in ("vit", "swin"):
        hs = sorted({(int(rng.integers(wl.B)), int(rng.integers(wl.Hq))) for _ in range(6)})
        return hs, np.arange(wl.Nq)
    last = (wl.Nq - 1) // 128
    tiles = sorted({0, last // 2, last})
    rows = np.concatenate([np.arange(t * 128, min(wl.Nq, t * 128 + 128)) for t in tiles])
    return [(0, 0), (0, 5), (0, wl.Hq - 1)], rows


@pytest.mark.parametrize("name", ["tiny", "vit", "swin", "llm8k", "chunk32k"])
def test_full_size_workload(name):
    wl = I.WORKLOADS[name]
    inp = I.make_inputs(wl)
    prep = O.prepare(inp)
    P = run_gpu(wl, inp, want_lse=False)
    assert np.array_equal(P.q_codes.cpu().numpy(), prep["q_codes"])
    if not wl.kv_codes:
        assert np.array_equal(P.k_codes.cpu().numpy(), prep["k_codes"])
    v8 = e4m3_bytes_to_values(P.v8t)[..., : wl.Nk].transpose(0, 1, 3, 2)
    assert np.array_equal(v8, prep["v8"])
    heads, rows = _samples(wl)
    ref = O.run_workload(inp, prep, heads=heads, rows=rows, want_bound=True)
    gpu = gpu_out_rows(P, heads, rows)
    stats = check_output(gpu, ref["O"], ref["bound"], name)
    P16 = run_gpu(wl, inp, out_dtype=qb.DT_BF16, want_lse=False)
    o16 = gpu_out_rows(P16, heads, rows)
    want16 = torch.from_numpy(gpu.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(o16, want16)
    K, V = O.real_kv(inp)
    ref64 = O.attn_fp64(inp.Q, K, V, causal=wl.causal, q_pos0=wl.q_pos0, bias=inp.bias,
                        heads=heads, rows=rows)
    print(f"{name}: {stats}; rel err vs fp64 {rel_err_vs_fp64(gpu, ref64):.3e}")
