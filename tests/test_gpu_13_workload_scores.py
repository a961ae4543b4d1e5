"""The int32 score tiles of the five workloads' own codes, bit-exact.

Each workload at full size runs its pre-pass through the public path (the
codes the attention kernel reads: llm8k's smoothed outlier channels,
chunk32k's Q with the cache's K channel scales folded in, ViT's per-tensor
codes); qattn_debug_qk_scores, which issues the same tensor-core product as
qattn_fwd, then computes the score tiles of sampled heads and query tiles
against every key, and they must equal the oracle's exact integer products of
the oracle's codes (QFlash, section 4.2, eq. (3): int8 codes, int32 results).
"""
import numpy as np
import pytest
import torch

from oracle import qattn_oracle as O
from quantized_attention_gb300 import binding as qb
from quantized_attention_gb300 import inputs as I
from quantized_attention_gb300.pipeline import device_inputs, problem_for
from tests.gpu_common import ensure_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def _slices(wl):
    """(b, h, first row, rows) of the sampled score tiles."""
    if wl.name == "tiny":
        return [(0, 0, 0, wl.Nq)]
    rng = np.random.default_rng(7)
    if wl.name in ("vit", "swin"):
        hs = sorted({(int(rng.integers(wl.B)), int(rng.integers(wl.Hq))) for _ in range(8)})
        return [(b, h, 0, wl.Nq) for b, h in hs]
    last = (wl.Nq - 1) // 128
    tiles = sorted({0, last // 2, last})
    return [(0, h, t * 128, min(128, wl.Nq - t * 128)) for h in (0, 13, wl.Hq - 1) for t in tiles]


@pytest.mark.parametrize("name", ["tiny", "vit", "swin", "llm8k", "chunk32k"])
def test_workload_score_tiles_bit_exact(name):
    wl = I.WORKLOADS[name]
    inp = I.make_inputs(wl)
    prep = O.prepare(inp)
    P = problem_for(wl)
    dev = device_inputs(inp)
    dev.pop("bias", None)
    P.quantize(**dev)
    torch.cuda.synchronize()
    g = wl.Hq // wl.Hkv
    shape = qb.make_shape(1, 1, 1, 1, wl.Nk, wl.d)
    ws = torch.empty(max(qb.workspace_size(qb.make_shape(1, 1, 1, 128, wl.Nk, wl.d),
                                           qb.make_params()), 256), dtype=torch.uint8,
                     device="cuda")
    for b, h, r0, nr in _slices(wl):
        shape.Nq = nr
        q = P.q_codes[b, h, r0:r0 + nr].reshape(1, 1, nr, wl.d)
        k = P._k_codes[b, h // g].reshape(1, 1, wl.Nk, wl.d)
        S = torch.full((1, 1, nr, wl.Nk), -7, dtype=torch.int32, device="cuda")
        qb.debug_qk_scores(q, k, shape, S, ws)
        torch.cuda.synchronize()
        assert qb.get_error() == 0
        want = O.qk_scores(prep["q_codes"][b:b + 1, h:h + 1, r0:r0 + nr],
                           prep["k_codes"][b:b + 1, h // g:h // g + 1])
        got = S.cpu().numpy()
        assert np.array_equal(got, want), f"{name} (b={b}, h={h}, rows {r0}..{r0 + nr - 1})"
