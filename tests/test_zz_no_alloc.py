"""qattn_quantize_v_noalloc (for callers that cannot allocate device memory)
gives exactly what qattn_quantize_v gives with a caller workspace.

Two calls in a row, the second on smaller-magnitude inputs: if the shared
static scratch were not cleared between calls, the second call would keep the
first call's larger channel maxima and its output would differ.  Collected last
so a stop-at-first-failure run has already run every other test."""
import numpy as np
import pytest
import torch

from quantized_attention_gb300 import binding as qb
from quantized_attention_gb300 import inputs as I
from tests.gpu_common import ensure_library

pytestmark = pytest.mark.gpu


def _v_inputs(wl, scale):
    inp = I.make_inputs(wl)
    if wl.kv_codes:
        return (torch.from_numpy(inp.V_codes).cuda(), qb.DT_I8,
                torch.from_numpy(inp.V_scale).cuda())
    return (torch.from_numpy(inp.V * np.float32(scale)).to("cuda", torch.bfloat16), qb.DT_BF16,
            None)


@pytest.mark.parametrize("wl", [I.small("llm8k", Hq=4, Hkv=2, Nq=300, Nk=300),
                                I.small("chunk32k", Hq=4, Hkv=2, Nq=128, Nk=640, q_pos0=512),
                                I.small("swin", B=7)],
                         ids=["bf16-V", "int8-V-codes", "swin-d32"])
def test_noalloc_matches_workspace_entry_point(wl):
    ensure_library()
    shape = qb.make_shape(wl.B, wl.Hq, wl.Hkv, wl.Nq, wl.Nk, wl.d)
    ldv = qb.v_ld(wl.Nk)
    ws = torch.empty(max(qb.workspace_size(shape, qb.make_params()), 256), dtype=torch.uint8,
                     device="cuda")
    for call, scale in enumerate((8.0, 0.25)):
        V, dt, chan = _v_inputs(wl, scale)
        if chan is not None and call == 1:
            V = (V // 3).contiguous()  # smaller codes on the second call
        ref_v8 = torch.full((wl.B, wl.Hkv, wl.d, ldv), 0x55, dtype=torch.uint8, device="cuda")
        ref_s = torch.full((wl.B, wl.Hkv, wl.d), -1.0, dtype=torch.float32, device="cuda")
        qb.quantize_v(V, dt, chan, shape, ref_v8, ldv, ref_s, ws)
        got_v8 = torch.full_like(ref_v8, 0xAA)
        got_s = torch.full_like(ref_s, -2.0)
        qb.quantize_v_noalloc(V, dt, chan, shape, got_v8, ldv, got_s)
        torch.cuda.synchronize()
        assert qb.get_error() == 0
        assert torch.equal(got_v8, ref_v8), f"call {call}: e4m3 V differs"
        assert torch.equal(got_s.view(torch.int32), ref_s.view(torch.int32)), f"call {call}: scales differ"


def test_noalloc_rejects_oversized_problem():
    ensure_library()
    shape = qb.make_shape(4097, 4, 4, 49, 49, 32)  # B*Hkv*d = 524416 > 524288
    fake = torch.empty(16, dtype=torch.uint8, device="cuda")
    st = qb.lib().qattn_quantize_v_noalloc(qb._p(fake), qb.DT_BF16, None, __import__("ctypes").byref(shape),
                                           qb._p(fake), qb.v_ld(49), qb._p(fake), qb._stream())
    assert st == 2  # QATTN_ERR_UNSUPPORTED, nothing launched
