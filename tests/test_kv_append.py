"""Pins of the oracle's KV-cache append with a running channel mean of K in the
cache header (ZINC post, "K's outliers, and the subtraction softmax does not
notice": during decode K arrives one token at a time and the header keeps a
running mean that lags by one token).  CPU only."""
import numpy as np
import pytest

from oracle import qattn_oracle as O


def _empty(B, H, cap, d):
    z = np.zeros((B, H, d), np.float32)
    return z.copy(), z.copy(), np.zeros((B, H, cap, d), np.int8), np.zeros((B, H, cap, d), np.int8)


def _tokens(rng, B, H, T, d, loc=0.0, scale=1.0):
    x = rng.normal(loc, scale, size=(B, H, T, d)).astype(np.float32)
    # bf16 inputs: keep 8 mantissa bits
    return (x.view(np.uint32) & 0xFFFF0000).view(np.float32)


def test_first_two_tokens_closed_form():
    """Token 0 is quantized against the empty header's zero mean, token 1
    against token 0 exactly (the mean of one token), then the mean moves."""
    rng = np.random.default_rng(0)
    B, H, d, cap = 1, 2, 8, 4
    sk = np.full((B, H, d), 0.02, np.float32)
    sv = np.full((B, H, d), 0.03, np.float32)
    K = _tokens(rng, B, H, 2, d)
    V = _tokens(rng, B, H, 2, d)
    mu, amax, kc, vc = O.kv_append(K, V, 0, sk, sv, *_empty(B, H, cap, d))
    want0 = np.clip(np.rint(K[:, :, 0] / sk), -127, 127)
    want1 = np.clip(np.rint((K[:, :, 1] - K[:, :, 0]) / sk), -127, 127)
    assert np.array_equal(kc[:, :, 0].astype(np.float32), want0)
    assert np.array_equal(kc[:, :, 1].astype(np.float32), want1)
    # mean of two tokens: K0 + (K1 - K0) / 2, exact in fp32 here up to one rounding
    np.testing.assert_allclose(mu, (K[:, :, 0] + K[:, :, 1]) / 2, rtol=0, atol=1e-6)
    assert np.array_equal(kc[:, :, 2:], np.zeros_like(kc[:, :, 2:]))
    assert np.array_equal(amax, np.maximum(np.abs(vc[:, :, 0]), np.abs(vc[:, :, 1])).astype(np.float32))


def test_running_mean_tracks_the_dense_mean():
    """After N appends from an empty header the fp32 recurrence equals the
    mean of the N rows to within its accumulated rounding."""
    rng = np.random.default_rng(1)
    B, H, d, N = 2, 2, 16, 300
    K = _tokens(rng, B, H, N, d, loc=0.7, scale=1.5)
    V = _tokens(rng, B, H, N, d)
    sk = np.full((B, H, d), 0.05, np.float32)
    mu, _, _, _ = O.kv_append(K, V, 0, sk, sk, *_empty(B, H, N, d))
    dense = K.astype(np.float64).mean(axis=2)
    assert np.abs(mu - dense).max() <= 1e-5 * np.abs(K).max()


def test_lag_by_one_against_earlier_mean():
    """Token n's code is its K minus the mean of tokens 0..n-1 (fp64 here),
    rounded; fp32 rounding of that mean can move a code by at most one."""
    rng = np.random.default_rng(2)
    B, H, d, N = 1, 1, 32, 200
    K = _tokens(rng, B, H, N, d, loc=2.0)
    V = _tokens(rng, B, H, N, d)
    sk = np.full((B, H, d), 0.04, np.float32)
    _, _, kc, _ = O.kv_append(K, V, 0, sk, sk, *_empty(B, H, N, d))
    Kd = K.astype(np.float64)
    prev = np.concatenate([np.zeros((B, H, 1, d)), np.cumsum(Kd, axis=2)[:, :, :-1]], axis=2)
    mean_before = prev / np.maximum(np.arange(N), 1)[None, None, :, None]
    want = np.clip(np.rint((Kd - mean_before) / 0.04), -127, 127)
    diff = np.abs(kc.astype(np.float64) - want)
    assert diff.max() <= 1 and (diff == 0).mean() > 0.99


def test_updating_the_mean_first_is_caught():
    """A plausible mistake -- including the new token in the mean before
    quantizing it -- changes token 1's code (pins the lag)."""
    rng = np.random.default_rng(3)
    B, H, d = 1, 1, 64
    K = _tokens(rng, B, H, 2, d, scale=3.0)
    sk = np.full((B, H, d), 0.02, np.float32)
    _, _, kc, _ = O.kv_append(K, K, 0, sk, sk, *_empty(B, H, 2, d))
    wrong = np.clip(np.rint((K[:, :, 1] - (K[:, :, 0] + K[:, :, 1]) / 2) / sk), -127, 127)
    assert not np.array_equal(kc[:, :, 1].astype(np.float32), wrong)


def test_saturation_and_amax():
    B, H, d = 1, 1, 4
    K = np.array([[[[1000.0, -1000.0, 0.5, -0.5]]]], np.float32)
    V = np.array([[[[9.0, -9.0, 0.01, 0.0]]]], np.float32)
    s = np.full((B, H, d), 0.01, np.float32)
    mu, amax, kc, vc = O.kv_append(K, V, 0, s, s, *_empty(B, H, 1, d))
    assert kc[0, 0, 0].tolist() == [127, -127, 50, -50]
    assert vc[0, 0, 0].tolist() == [127, -127, 1, 0]
    assert amax[0, 0].tolist() == [127.0, 127.0, 1.0, 0.0]


@pytest.mark.parametrize("chunks", [[1] * 12, [5, 7], [12]])
def test_chunked_appends_equal_single_steps(chunks):
    rng = np.random.default_rng(4)
    B, H, d, N = 2, 3, 8, 12
    K = _tokens(rng, B, H, N, d, loc=1.0)
    V = _tokens(rng, B, H, N, d)
    sk = rng.uniform(0.01, 0.05, size=(B, H, d)).astype(np.float32)
    sv = rng.uniform(0.01, 0.05, size=(B, H, d)).astype(np.float32)
    ref = O.kv_append(K, V, 0, sk, sv, *_empty(B, H, N, d))
    state = _empty(B, H, N, d)
    pos = 0
    for T in chunks:
        state = O.kv_append(K[:, :, pos:pos + T], V[:, :, pos:pos + T], pos, sk, sv, *state)
        pos += T
    for a, b in zip(ref, state):
        assert np.array_equal(a, b)


def test_header_of_codes_equals_the_appended_header():
    """kv_header (the V max |code| of a cache filled elsewhere) equals the header
    kv_append builds while it writes those codes one token at a time, for any
    number of rows in use; an empty cache has a zero header."""
    rng = np.random.default_rng(9)
    B, H, d, cap, T = 2, 3, 16, 40, 29
    sk = np.full((B, H, d), 0.05, np.float32)
    sv = rng.uniform(0.01, 0.05, size=(B, H, d)).astype(np.float32)
    K = _tokens(rng, B, H, T, d)
    V = _tokens(rng, B, H, T, d, scale=2.0)
    state = _empty(B, H, cap, d)
    for t in range(T):
        state = O.kv_append(K[:, :, t:t + 1], V[:, :, t:t + 1], t, sk, sv, *state)
        assert np.array_equal(O.kv_header(state[3], t + 1), state[1])
    assert not O.kv_header(state[3], 0).any()
