"""qattn_kv_append (the int8 cache's append with a running channel mean of K in
its header) against the oracle, bit for bit, and decode steps on a cache grown
by appends (capacity larger than the rows in use)."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import qattn_oracle as O
from quantized_attention_gb300 import binding as qb
from quantized_attention_gb300 import inputs as I
from quantized_attention_gb300.pipeline import problem_for
from tests.gpu_common import ensure_library
from tests.parity import check_output

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def _dev(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x)).to(device="cuda", dtype=dtype)


def _cache(inp, n0, cap):
    """The workload's first n0 cache rows in arrays of capacity cap (rest 0),
    its header mean, and the V max of the rows in use."""
    B, H, _, d = inp.K_codes.shape
    kc = np.zeros((B, H, cap, d), np.int8)
    vc = np.zeros((B, H, cap, d), np.int8)
    kc[:, :, :n0] = inp.K_codes[:, :, :n0]
    vc[:, :, :n0] = inp.V_codes[:, :, :n0]
    amax = np.abs(vc[:, :, :n0].astype(np.int32)).max(axis=2).astype(np.float32)
    return kc, vc, inp.K_header_mean.astype(np.float32).copy(), amax


@pytest.mark.parametrize("d,chunks", [(128, [1, 5, 1, 30, 1, 12]), (64, [7, 1, 1, 40])])
def test_kv_append_bit_exact(d, chunks):
    wl = I.small("decode32k", Hkv=4, Hq=8, Nk=200, d=d)
    inp = I.make_inputs(wl)
    T = sum(chunks)
    cap = wl.Nk + T
    kc, vc, mu, amax = _cache(inp, wl.Nk, cap)
    Kn, Vn = I.make_append_tokens(inp, T, seed=1)
    ref = (mu, amax, kc, vc)
    g_kc, g_vc = _dev(kc, torch.int8), _dev(vc, torch.int8)
    g_mu, g_am = _dev(mu, torch.float32), _dev(amax, torch.float32)
    g_ks, g_vs = _dev(inp.K_scale, torch.float32), _dev(inp.V_scale, torch.float32)
    pos = wl.Nk
    for c in chunks:
        ref = O.kv_append(Kn[:, :, pos - wl.Nk:pos - wl.Nk + c], Vn[:, :, pos - wl.Nk:pos - wl.Nk + c],
                          pos, inp.K_scale, inp.V_scale, *ref)
        qb.kv_append(_dev(Kn[:, :, pos - wl.Nk:pos - wl.Nk + c], torch.bfloat16),
                     _dev(Vn[:, :, pos - wl.Nk:pos - wl.Nk + c], torch.bfloat16), pos, g_ks, g_vs,
                     g_mu, g_am, g_kc, g_vc)
        pos += c
    torch.cuda.synchronize()
    assert qb.get_error() == 0
    r_mu, r_am, r_kc, r_vc = ref
    assert np.array_equal(g_kc.cpu().numpy(), r_kc)
    assert np.array_equal(g_vc.cpu().numpy(), r_vc)
    assert np.array_equal(g_mu.cpu().numpy().view(np.uint32), r_mu.view(np.uint32))
    assert np.array_equal(g_am.cpu().numpy(), r_am)


def test_kv_append_rejects_bad_arguments():
    B, H, T, d, cap = 1, 2, 3, 64, 8
    Kn = torch.zeros((B, H, T, d), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((B, H, cap, d), dtype=torch.int8, device="cuda")
    f = torch.zeros((B, H, d), dtype=torch.float32, device="cuda")
    with pytest.raises(qb.QattnError):
        qb.kv_append(Kn, Kn, cap - 2, f, f, f, f, kc, kc)  # pos + T > capacity
    with pytest.raises(qb.QattnError):
        qb.kv_append(Kn, Kn, -1, f, f, f, f, kc, kc)


def test_decode_steps_on_an_appended_cache():
    """A decode loop: append the new token (running mean), quantize its Q,
    decode over the rows in use of a larger cache; each step against the
    oracle on the oracle's own appended cache."""
    base = I.small("decode32k", Hq=8, Hkv=2, Nq=1, Nk=1500, d=128)
    inp0 = I.make_inputs(base)
    steps, cap = 3, 1600
    kc, vc, mu, amax = _cache(inp0, base.Nk, cap)
    Kn, Vn = I.make_append_tokens(inp0, steps, seed=2)
    ref = (mu, amax, kc, vc)
    g_kc, g_vc = _dev(kc, torch.int8), _dev(vc, torch.int8)
    g_ks, g_vs = _dev(inp0.K_scale, torch.float32), _dev(inp0.V_scale, torch.float32)
    g_mu = _dev(mu, torch.float32)
    rng = np.random.default_rng(9)
    for s in range(steps):
        n = base.Nk + s  # rows before this token
        ref = O.kv_append(Kn[:, :, s:s + 1], Vn[:, :, s:s + 1], n, inp0.K_scale, inp0.V_scale, *ref)
        wl = dataclasses.replace(base, Nk=n + 1)
        Q = I.to_bf16(rng.normal(size=(wl.B, wl.Hq, 1, wl.d)).astype(np.float32))
        r_mu, r_am, r_kc, r_vc = ref
        inp = I.Inputs(wl, Q, K_codes=r_kc[:, :, :n + 1], K_scale=inp0.K_scale,
                       K_header_mean=inp0.K_header_mean, V_codes=r_vc[:, :, :n + 1],
                       V_scale=inp0.V_scale)
        P = problem_for(wl, want_lse=True)
        P.set_cache(g_kc, g_vc, g_vs, K_scale=g_ks, K_mean=g_mu)
        if s > 0:
            P._cache_vamax = g_am  # the header carried from the last step
        P.append(_dev(Kn[:, :, s:s + 1], torch.bfloat16), _dev(Vn[:, :, s:s + 1], torch.bfloat16), n)
        g_mu, g_am = P._cache_kmean, P._cache_vamax
        P.quantize_q(_dev(Q, torch.bfloat16), g_ks)
        P.decode()
        torch.cuda.synchronize()
        assert qb.get_error() == 0
        assert np.array_equal(g_kc.cpu().numpy()[:, :, :n + 1], r_kc[:, :, :n + 1])
        assert np.array_equal(g_am.cpu().numpy(), r_am)
        prep = O.prepare(inp)
        heads = [(0, h) for h in range(wl.Hq)]
        want = O.run_workload(inp, prep, heads=heads, rows=np.arange(1), want_bound=True)
        got = P.O.cpu().numpy().reshape(wl.Hq, 1, wl.d).astype(np.float64)
        check_output(got, want["O"], want["bound"], f"step {s}")


@pytest.mark.parametrize("d,cap,Nk", [(128, 300, 300), (128, 300, 129), (64, 70, 1), (32, 257, 200),
                                      (64, 16, 0)])
def test_header_init_matches_oracle(d, cap, Nk):
    """qattn_kv_header_init: the max |V code| per channel over the rows in use of
    a cache filled outside the library, bit-exact with the oracle's definition
    (rows beyond Nk hold larger codes that must not count)."""
    rng = np.random.default_rng(d + cap + Nk)
    B, H = 2, 3
    codes = rng.integers(-100, 101, size=(B, H, cap, d)).astype(np.int8)
    codes[:, :, Nk:, :] = 127          # unused rows: never read
    codes[0, 1, :, 5] = 0              # an all-zero channel
    if Nk > 3:
        codes[1, 2, Nk - 1, 7] = -127  # the extreme code in the last row in use
    dev = torch.from_numpy(codes).cuda()
    out = torch.full((B, H, d), -1.0, dtype=torch.float32, device="cuda")
    qb.kv_header_init(dev, Nk, out)
    torch.cuda.synchronize()
    assert qb.get_error() == 0
    assert np.array_equal(out.cpu().numpy(), O.kv_header(codes, Nk))
