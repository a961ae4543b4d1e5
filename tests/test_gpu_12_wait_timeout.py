"""The kernels' bounded wait gives up instead of hanging: qattn_debug_wait_timeout
runs it on an mbarrier that nothing arrives at.  The wait must report failure
after its time limit with the abort flag raised, qattn_get_error must return
QATTN_ERR_TIMEOUT once and then OK, and the context must stay usable (the next
kernel of the library gives exact results)."""
import time

import numpy as np
import pytest
import torch

from oracle import qattn_oracle as O
from quantized_attention_gb300 import binding as qb
from tests.gpu_common import ensure_library

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    ensure_library()
    torch.cuda.synchronize()
    assert qb.get_error() == qb.OK  # nothing left over from earlier calls

    result = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    qb.debug_wait_timeout(result)
    st = qb.get_error()  # synchronises the stream
    waited = time.perf_counter() - t0
    assert st == qb.ERR_TIMEOUT
    assert result.cpu().tolist() == [0, 1]  # wait failed, abort flag raised
    # the limit is 4e9 SM cycles: at least ~1.9 s at the 2070 MHz maximum clock
    assert 1.0 <= waited <= 60.0, waited
    assert qb.get_error() == qb.OK  # the word was cleared

    # the context still runs the library's kernels correctly
    rng = np.random.default_rng(12)
    q = rng.integers(-127, 128, size=(1, 2, 130, 64)).astype(np.int8)
    k = rng.integers(-127, 128, size=(1, 1, 200, 64)).astype(np.int8)
    shape = qb.make_shape(1, 2, 1, 130, 200, 64)
    ws = torch.empty(max(qb.workspace_size(shape, qb.make_params()), 256), dtype=torch.uint8,
                     device="cuda")
    S = torch.full((1, 2, 130, 200), -7, dtype=torch.int32, device="cuda")
    qb.debug_qk_scores(torch.from_numpy(q).cuda(), torch.from_numpy(k).cuda(), shape, S, ws)
    torch.cuda.synchronize()
    assert qb.get_error() == qb.OK
    assert np.array_equal(S.cpu().numpy(), O.qk_scores(q, k))
