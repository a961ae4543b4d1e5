"""qattn: quantized flash-attention prefill for GB300 (sm_103a).

int8 Q/K codes with an exact integer QK^T (after K's channel mean is
subtracted), an fp32 online softmax, and e4m3 P (static scale 448) times
per-channel e4m3 V, in hand-written tcgen05/TMA kernels behind a C ABI
(include/qattn.h).  This package is the Python binding of that library.
"""
from . import binding  # noqa: F401
from .binding import (DT_BF16, DT_F32, DT_I8, GRAN_BLOCK, GRAN_HEAD, GRAN_TENSOR,  # noqa: F401
                      QattnError)

__all__ = ["binding", "pipeline", "inputs", "QattnError"]
