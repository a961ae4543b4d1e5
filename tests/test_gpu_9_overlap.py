"""pipeline.OverlappedSteps (host copies in, kernels, host copy out, with
consecutive steps in flight together on three streams) gives, step by step,
exactly the outputs of the serial path on the same inputs, with several input
sets used in turn so that a step reading another step's buffers would show."""
import pytest
import torch

from quantized_attention_gb300 import binding as qb
from quantized_attention_gb300 import inputs as I
from quantized_attention_gb300.pipeline import OverlappedSteps, device_inputs, problem_for
from tests.gpu_common import ensure_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


@pytest.mark.parametrize("name,kw", [
    ("llm8k", dict(Hq=4, Hkv=2, Nq=640, Nk=640)),                 # bf16 K/V, causal, GQA
    ("chunk32k", dict(Hq=4, Hkv=1, Nq=256, Nk=900, q_pos0=None)),  # int8 cache codes
])
def test_overlapped_steps_match_serial(name, kw):
    wl = I.small(name, **kw)
    P = problem_for(wl, out_dtype=qb.DT_BF16)
    sets = []
    for seed in (11, 12, 13):
        dev = device_inputs(I.make_inputs(wl.replace(seed=seed)))
        dev.pop("bias", None)
        P.run(**dev)
        torch.cuda.synchronize()
        sets.append(({k: v.cpu().pin_memory() for k, v in dev.items()}, P.O.clone()))
    assert qb.get_error() == 0
    assert not torch.equal(sets[0][1], sets[1][1])  # the sets differ

    runner = OverlappedSteps([h for h, _ in sets], P.O,
                             lambda d_in, d_out, s: P.run(**d_in, stream=s, out=d_out))
    pending = []
    for i in range(8):
        pending.append((i, runner.step()))
        if i % 2 == 1:  # a host output is reused two steps later: read it before then
            runner.sync()
            for j, host in pending:
                want = sets[j % 3][1].cpu()
                assert torch.equal(host, want), f"step {j}"
            pending = []
    assert qb.get_error() == 0
