"""Shared set-up of the GPU tests: build/load the library once, run the
library path and the oracle on the same seeded inputs."""
import os

import numpy as np
import torch

from quantized_attention_gb300 import binding as qb
from quantized_attention_gb300.pipeline import device_inputs, problem_for


def ensure_library():
    from quantized_attention_gb300 import build
    if not os.path.exists(qb.library_path()):
        build.build(checked=os.path.abspath(qb.library_path()) == build.CHECK_LIB)
    qb.lib()


def run_gpu(wl, inp, out_dtype=qb.DT_F32, want_lse=True, k_carrier=True, pv_mode=qb.PV_E4M3):
    P = problem_for(wl, out_dtype=out_dtype, want_lse=want_lse, k_carrier=k_carrier,
                    pv_mode=pv_mode)
    dev = device_inputs(inp)
    bias = dev.pop("bias", None)
    P.run(**dev, bias=bias)
    torch.cuda.synchronize()
    assert qb.get_error() == 0, "device error word set"
    return P


def gpu_out_rows(P, heads, rows):
    """GPU output [len(heads), len(rows), d] as float64 numpy."""
    o = P.O.float().cpu().numpy()
    return np.stack([o[b, h][rows] for (b, h) in heads]).astype(np.float64)


def gpu_lse_rows(P, heads, rows):
    l = P.lse.cpu().numpy()
    return np.stack([l[b, h][rows] for (b, h) in heads]).astype(np.float64)
