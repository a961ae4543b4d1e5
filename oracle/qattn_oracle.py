"""CPU oracle for quantized flash-attention prefill (int8 QK^T, fp8 e4m3 PV).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the package's
``smoke()`` check and the CPU-baseline leg of ``bench.py`` may import it.  It
shares no code with the CUDA path: plain NumPy, written step by step from the
pages, slow on purpose and easy to check by eye.

Sources (page title, section):

* [ZINC-ATTN]  "int8 Flash Attention on RDNA4: QK Wants Integers, PV Wants
  FP8" -- sections "The scale P needs is already sitting in a register",
  "K's outliers, and the subtraction softmax does not notice",
  "fp8 is not faster, it is shaped correctly".
* [QFLASH]     "QFlash: Bridging Quantization and Memory Efficiency in Vision
  Transformer Attention" -- section 4, eq. (1)-(3), Algorithm 1, section 2.1;
  sections 4.3-4.6 for the integer-only attention (attn_intsoftmax).
* [STRATA]     "prompt_attn_i8v3_kernel" pull request -- the 24-bit exact split
  mode (attn_exact24).
* The ZINC post's decode section -- the int8 KV cache and its running-mean
  header (kv_append).

Precision: the pages fix fp32 for the online softmax statistics and for every
value that decides a quantized code (K - mu, x * 127/amax, P * 448); those are
computed in np.float32.  Sums that decide nothing (the row sum l, the output
accumulator O) are kept in float64.

Readings where the pages are silent (each one is listed in the design notes):

* The channel mean is taken per (batch, KV head) over all Nk keys, as an
  int64 fixed-point sum of round(K * 2^24), so that any summation order gives
  the same bits; with no keys it is 0 (every row is then fully masked).
* The int8 quantizer multiplies by the fp32 reciprocal 127/amax instead of
  dividing by amax/127; ties round to even; codes lie in [-127, 127].
* Q/K scale granules: one per tensor, per (batch, head), or per (batch, head,
  128-token block); the key block of the online softmax is also 128 tokens.
* V gets one scale per (batch, KV head, channel): amax over all keys / 448.
* The row sum l accumulates the unquantized fp32 P, not the e4m3 P.
* The running max is exact and O is rescaled whenever it grows, so P <= 1
  always holds and P * 448 never exceeds the e4m3 range.
* Causal masks are bottom-right aligned: key k is visible to query i iff
  k <= q_pos0 + i, with q_pos0 = Nk - Nq unless given.
* GQA: query head h reads KV head h // (Hq / Hkv).
* An additive bias [Nq, Nk] in natural-log units is added after scaling.

Functions whose result has no independent pin are marked "parity unpinned"
(scale_release: QFlash's ScaleRelease, whose definition is not in the pages);
every other function is pinned by the CPU tests tests/test_oracle_pins.py,
tests/test_oracle_mutations.py, tests/test_mean_rounding_claim.py,
tests/test_prob_mass.py, tests/test_kv_append.py, tests/test_exact24.py and
tests/test_intsoftmax.py.
"""
from __future__ import annotations

import math

import numpy as np

F32 = np.float32
F64 = np.float64

#: fp32(log2 e): the exponent base change used by the softmax (QFLASH eq. (5))
LOG2E_F32 = F32(1.4426950408889634)
#: static P scale: the largest finite e4m3 value (ZINC-ATTN, "fp8 is not faster")
P_SCALE = 448.0
#: 2^(b-1) - 1 for b = 8 (QFLASH eq. (1)-(2))
QMAX = 127
#: tokens per scale granule in block granularity, and keys per softmax block
BLOCK = 128
#: fixed-point fraction bits of the channel-mean sum
FIX_BITS = 24

GRAN_TENSOR = 0
GRAN_HEAD = 1
GRAN_BLOCK = 2


# ---------------------------------------------------------------------------
# fp8 e4m3 (ZINC-ATTN "fp8 is not faster": four exponent bits, three mantissa
# bits, largest value 448).  Written from the format definition: exponent bias
# 7, subnormal step 2^-9, no infinities, 0x7F/0xFF are NaN.
# ---------------------------------------------------------------------------

def e4m3_round(x) -> np.ndarray:
    """Round to the nearest e4m3 value, ties to even, saturating at +-448.

    Returns float64 values.  For |x| in binade [2^e, 2^(e+1)) the grid step is
    2^(e-3); below 2^-6 the subnormal step 2^-9 applies.  Every step is a
    power of two, so a/step and the rounding are exact in float64.
    """
    x64 = np.asarray(x, dtype=F64)
    a = np.abs(x64)
    _, E = np.frexp(a)               # a = f * 2^E, f in [0.5, 1)
    e = np.maximum(E - 1, -6)        # binade exponent, clamped at the subnormal range
    step = np.ldexp(1.0, e - 3)
    q = np.rint(a / step) * step     # np.rint: round half to even
    q = np.minimum(q, P_SCALE)       # satfinite
    return np.copysign(q, x64)


def e4m3_midpoint_distance(a) -> tuple[np.ndarray, np.ndarray]:
    """For a >= 0: (distance to the nearest e4m3 rounding midpoint, grid step)."""
    a = np.asarray(a, dtype=F64)
    _, E = np.frexp(a)
    e = np.maximum(E - 1, -6)
    step = np.ldexp(1.0, e - 3)
    frac = a / step - np.floor(a / step)
    return np.abs(frac - 0.5) * step, step


# ---------------------------------------------------------------------------
# a1: K channel mean (ZINC-ATTN "K's outliers": subtracting the per-channel
# mean of K shifts every score in a row by the same q.mu, which softmax
# ignores; the mean is one reduction over the K block).
# ---------------------------------------------------------------------------

def smooth_k(K: np.ndarray) -> np.ndarray:
    """mu[b, h, c] = mean over keys of K[b, h, :, c], as fp32.

    Fixed point: fix(x) = round_half_even(x * 2^24) as int64, summed exactly,
    then mu = fp32(fp64(sum) * 2^-24 / Nk).  With no keys (Nk = 0) the mean
    has no value and nothing is subtracted from anything: mu = 0 (a reading).
    """
    K = np.asarray(K, dtype=F32)
    Nk = K.shape[2]
    if Nk == 0:
        return np.zeros((K.shape[0], K.shape[1], K.shape[3]), dtype=F32)
    fix = np.rint(K.astype(F64) * 2.0 ** FIX_BITS).astype(np.int64)
    s = fix.sum(axis=2, dtype=np.int64)
    assert np.abs(s).max(initial=0) < 2 ** 53, "channel sum leaves the exact range"
    mu = (s.astype(F64) * 2.0 ** -FIX_BITS) / F64(Nk)
    return mu.astype(F32)


# ---------------------------------------------------------------------------
# a2: symmetric int8 quantizer (QFLASH eq. (1)-(2): s_X = ||X||_inf / (2^(b-1)-1),
# X_hat = round(X / s_X)).
# ---------------------------------------------------------------------------

def granule_amax(x: np.ndarray, gran: int) -> np.ndarray:
    """max |x| per scale granule.  x: [B, H, N, d].

    tensor -> shape (1,), head -> [B, H], block -> [B, H, ceil(N/128)].
    """
    a = np.abs(np.asarray(x, dtype=F32))
    B, H, N, d = a.shape
    if gran == GRAN_TENSOR:
        return np.array([a.max(initial=0.0)], dtype=F32)
    if gran == GRAN_HEAD:
        return a.reshape(B, H, N * d).max(axis=2, initial=0.0).astype(F32)
    if gran == GRAN_BLOCK:
        nb = -(-N // BLOCK)
        pad = np.zeros((B, H, nb * BLOCK, d), dtype=F32)
        pad[:, :, :N] = a
        return pad.reshape(B, H, nb, BLOCK * d).max(axis=3).astype(F32)
    raise ValueError(f"unknown granularity {gran}")


def expand_per_token(g: np.ndarray, gran: int, B: int, H: int, N: int) -> np.ndarray:
    """Per-granule values -> [B, H, N] (the granule of each token)."""
    if gran == GRAN_TENSOR:
        return np.broadcast_to(g.reshape(1, 1, 1), (B, H, N))
    if gran == GRAN_HEAD:
        return np.broadcast_to(g[:, :, None], (B, H, N))
    return g[:, :, np.arange(N) // BLOCK]


def quantize_sym(x: np.ndarray, gran: int) -> tuple[np.ndarray, np.ndarray]:
    """codes = clip(rint(x * (127 / amax)), -127, 127); scale = amax / 127.

    All in fp32; inv = 0 (and so every code 0) where amax == 0.
    """
    x = np.asarray(x, dtype=F32)
    B, H, N, _ = x.shape
    amax = granule_amax(x, gran)
    with np.errstate(divide="ignore"):
        inv = np.where(amax > 0, F32(QMAX) / amax, F32(0)).astype(F32)
    scale = (amax / F32(QMAX)).astype(F32)
    inv_tok = expand_per_token(inv, gran, B, H, N)[..., None]
    prod = (x * inv_tok).astype(F32)
    codes = np.clip(np.rint(prod), -QMAX, QMAX).astype(np.int8)
    return codes, scale


def kv_head_of(Hq: int, Hkv: int) -> np.ndarray:
    """GQA: KV head read by each query head (contiguous groups)."""
    assert Hq % Hkv == 0
    return np.arange(Hq) // (Hq // Hkv)


def quantize_qk(Q, K=None, *, k_mean=None, K_codes=None, k_chan_scale=None,
                q_gran=GRAN_BLOCK, k_gran=GRAN_BLOCK):
    """Q (and K) -> int8 codes and fp32 scales.

    bf16 K: K' = fp32(K) - mu, then quantize_sym (ZINC-ATTN "K's outliers").
    int8 K codes with per-(b, KV head, channel) scale s_c: the codes are used
    as they are; s_c is folded into Q (Q' = fp32(Q) * s_c) so that the integer
    dot product stays exact, and every K scale is 1.
    Returns (q_codes, q_scales, k_codes, k_scales).
    """
    Qx = np.asarray(Q, dtype=F32)
    B, Hq = Qx.shape[:2]
    if K_codes is not None:
        Hkv = K_codes.shape[1]
        s = np.asarray(k_chan_scale, dtype=F32)[:, kv_head_of(Hq, Hkv)]  # [B, Hq, d]
        Qx = (Qx * s[:, :, None, :]).astype(F32)
        q_codes, q_scales = quantize_sym(Qx, q_gran)
        k_amax = granule_amax(np.zeros_like(K_codes[..., :1], dtype=F32), k_gran)
        return q_codes, q_scales, np.asarray(K_codes, dtype=np.int8), np.ones_like(k_amax)
    Kx = np.asarray(K, dtype=F32)
    if k_mean is not None:
        Kx = (Kx - np.asarray(k_mean, dtype=F32)[:, :, None, :]).astype(F32)
    q_codes, q_scales = quantize_sym(Qx, q_gran)
    k_codes, k_scales = quantize_sym(Kx, k_gran)
    return q_codes, q_scales, k_codes, k_scales


# ---------------------------------------------------------------------------
# a3: V -> e4m3 with per-channel scales.
# ---------------------------------------------------------------------------

def quantize_v(V: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """bf16 V -> (V8 values [B, H, N, d] float64, s_v [B, H, d] fp32).

    amax_c over all keys; V8 = e4m3(fp32(V * fp32(448 / amax_c))); s_v = amax_c / 448.
    """
    V = np.asarray(V, dtype=F32)
    amax = np.abs(V).max(axis=2, initial=0.0).astype(F32)
    with np.errstate(divide="ignore"):
        inv = np.where(amax > 0, F32(P_SCALE) / amax, F32(0)).astype(F32)
    s_v = (amax / F32(P_SCALE)).astype(F32)
    v8 = e4m3_round((V * inv[:, :, None, :]).astype(F32))
    return v8, s_v


def quantize_v_codes(V_codes: np.ndarray, v_chan_scale: np.ndarray):
    """int8 V codes with per-channel scale s_c -> (V8 values, s_v).

    amax_c = max |code|; V8 = e4m3(fp32(code * fp32(448 / amax_c)));
    s_v = fp32(fp32(s_c * amax_c) / 448).
    """
    Vc = np.asarray(V_codes, dtype=np.int8)
    amax = np.abs(Vc.astype(np.int32)).max(axis=2, initial=0).astype(F32)
    with np.errstate(divide="ignore"):
        inv = np.where(amax > 0, F32(P_SCALE) / amax, F32(0)).astype(F32)
    v8 = e4m3_round((Vc.astype(F32) * inv[:, :, None, :]).astype(F32))
    s_v = ((np.asarray(v_chan_scale, dtype=F32) * amax).astype(F32) / F32(P_SCALE)).astype(F32)
    return v8, s_v


# ---------------------------------------------------------------------------
# a4: integer scores (QFLASH eq. (3): C_hat = A_hat . B_hat in int32).
# ---------------------------------------------------------------------------

def qk_scores(q_codes: np.ndarray, k_codes: np.ndarray) -> np.ndarray:
    """S[b, h, i, k] = sum_c q[b, h, i, c] * k[b, h_kv, k, c] as int32.

    Computed with a float64 matmul of the integer codes, exact because
    |S| <= d * 127^2 < 2^53.
    """
    B, Hq, Nq, d = q_codes.shape
    Hkv = k_codes.shape[1]
    assert d * QMAX * QMAX < 2 ** 31
    kh = kv_head_of(Hq, Hkv)
    qf = q_codes.astype(F64)
    kf = k_codes.astype(F64)[:, kh]
    S = np.matmul(qf, np.swapaxes(kf, 2, 3))
    return S.astype(np.int64).astype(np.int32)


# ---------------------------------------------------------------------------
# a5-a10: blockwise online softmax and PV (ZINC-ATTN "The scale P needs is
# already sitting in a register": P = exp(s - m) <= 1, static scale; QFLASH
# section 2.1 and Algorithm 1: running row max, rescale, row sum, normalize).
# ---------------------------------------------------------------------------

def visible_mask(rows: np.ndarray, Nk: int, causal: bool, q_pos0: int) -> np.ndarray:
    """[R, Nk] bool: key k visible to query row i."""
    k = np.arange(Nk)[None, :]
    if not causal:
        return np.ones((len(rows), Nk), dtype=bool)
    return k <= (q_pos0 + np.asarray(rows))[:, None]


def online_softmax_pv(S, c, V8, s_v, *, visible, bias2=None, p_quant="e4m3",
                      ftype=F32, want_bound=False, check_p=True):
    """One head, a set of query rows.

    S        [R, Nk]   scores in code units (integers, or reals in the
                       unquantized pin)
    c        [R, nb]   per (row, key block) factor sq * sk * sm_scale * log2e
    V8       [Nk, d]   V values (e4m3 values, or reals)
    s_v      [d]       per-channel V scale
    visible  [R, Nk]   mask
    bias2    [R, Nk]   bias * log2e in log2 units, or None
    p_quant  "e4m3" (P8 = e4m3(P * 448) / 448), "int8" (static 127, the
             rejected int8 PV of ZINC-ATTN), or None (P used as is)
    ftype    precision of t, m, alpha, P (np.float32 for the recipe)

    Key blocks of 128 are visited in ascending order.  Per block and row:
      t = S * c (+ bias2);  masked -> -inf
      m_new = max(m, max_k t);  alpha = exp2(m - m_new)
      P = exp2(t - m_new) <= 1
      l = alpha * l + sum P            (unquantized P)
      O = alpha * O + quant(P) @ V
    Finally O * s_v / l (0 where l == 0).

    With want_bound, also returns a per-element bound on how far the output
    can move if any code of P (e4m3 of P * 448, or the int8 rint(P * 127))
    whose value lies within the exp2-accuracy window of a rounding midpoint
    is rounded the other way.
    """
    S = np.asarray(S)
    R, Nk = S.shape
    d = V8.shape[1]
    nb = -(-Nk // BLOCK)
    m = np.full(R, -np.inf, dtype=ftype)
    l = np.zeros(R, dtype=F64)
    O = np.zeros((R, d), dtype=F64)
    Bacc = np.zeros((R, d), dtype=F64) if want_bound else None
    absV = np.abs(np.asarray(V8, dtype=F64))
    p_max = 0.0
    n_amb = 0
    for j in range(nb):
        k0, k1 = j * BLOCK, min(Nk, (j + 1) * BLOCK)
        t = (S[:, k0:k1].astype(ftype) * c[:, j : j + 1].astype(ftype)).astype(ftype)
        if bias2 is not None:
            t = (t + bias2[:, k0:k1].astype(ftype)).astype(ftype)
        vis = visible[:, k0:k1]
        t = np.where(vis, t, ftype(-np.inf)).astype(ftype)
        m_new = np.maximum(m, t.max(axis=1)).astype(ftype)
        with np.errstate(invalid="ignore"):
            alpha = np.where(np.isneginf(m_new), ftype(1),
                             np.exp2((m - m_new).astype(ftype))).astype(ftype)
            x = (t - m_new[:, None]).astype(ftype)
            P = np.where(vis & ~np.isneginf(t), np.exp2(x), ftype(0)).astype(ftype)
        if check_p:
            assert not (P > 1).any(), "P <= 1 violated"
        p_max = max(p_max, float(P.max(initial=0.0)))
        l = alpha.astype(F64) * l + P.astype(F64).sum(axis=1)
        if p_quant == "e4m3":
            P448 = (P * ftype(P_SCALE)).astype(ftype)
            Pq = e4m3_round(P448) / P_SCALE
        elif p_quant == "int8":
            Pq = np.rint((P * ftype(QMAX)).astype(ftype)).astype(F64) / QMAX
        else:
            Pq = P.astype(F64)
        O = alpha.astype(F64)[:, None] * O + Pq @ np.asarray(V8[k0:k1], dtype=F64)
        if want_bound:
            assert p_quant in ("e4m3", "int8")
            span = np.abs(t.astype(F64)) + np.abs(m_new.astype(F64))[:, None]
            span = np.where(np.isfinite(span), span, 0.0)
            if p_quant == "e4m3":
                dist, step = e4m3_midpoint_distance(P448)
                Ps, scale = P448.astype(F64), P_SCALE
            else:  # int8: midpoints at k + 1/2, a flip moves the code by 1
                Ps = (P * ftype(QMAX)).astype(F64)
                dist = np.abs(Ps - (np.floor(Ps) + 0.5))
                step, scale = np.ones_like(Ps), float(QMAX)
            window = 2.0 ** -20 * (4.0 + span) * Ps
            amb = (dist <= window) & (Ps > 0)
            n_amb += int(amb.sum())
            Bacc = alpha.astype(F64)[:, None] * Bacc + (amb * step / scale) @ absV[k0:k1]
        m = m_new
    with np.errstate(divide="ignore", invalid="ignore"):
        inv_l = np.where(l > 0, 1.0 / l, 0.0)
    out = O * np.asarray(s_v, dtype=F64)[None, :] * inv_l[:, None]
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0, (m.astype(F64) + np.log2(np.where(l > 0, l, 1.0))) * math.log(2.0),
                       -np.inf)
    res = {"O": out, "l": l, "m": m, "lse": lse, "p_max": p_max}
    if want_bound:
        res["bound"] = Bacc * np.asarray(s_v, dtype=F64)[None, :] * inv_l[:, None]
        res["n_ambiguous"] = n_amb
    return res


def default_sm_scale(d: int) -> np.float32:
    """1/sqrt(d) rounded to fp32 (QFLASH Algorithm 1, s = s_Q s_K d^(-1/2) log2 e)."""
    return F32(1.0 / math.sqrt(d))


def block_factor(sq: np.ndarray, sk: np.ndarray, sm_scale) -> np.ndarray:
    """c = fp32(fp32(fp32(sq * sk) * sm_scale) * log2e); sq [R, 1], sk [1, nb]."""
    c = (np.asarray(sq, F32) * np.asarray(sk, F32)).astype(F32)
    c = (c * F32(sm_scale)).astype(F32)
    return (c * LOG2E_F32).astype(F32)


def attn_fwd(q_codes, q_scales, k_codes, k_scales, v8, s_v, *, q_gran, k_gran,
             causal, q_pos0=None, sm_scale=None, bias=None, heads=None, rows=None,
             p_quant="e4m3", want_bound=False):
    """The recipe's attention output on given (b, h) heads and query rows.

    q_codes [B, Hq, Nq, d] int8, k_codes [B, Hkv, Nk, d] int8, v8 [B, Hkv, Nk, d]
    e4m3 values, s_v [B, Hkv, d].  heads: list of (b, h) (default all);
    rows: query indices (default all).  Returns dict with O [len(heads), R, d]
    float64 and, with want_bound, the flip bound of the same shape.
    """
    B, Hq, Nq, d = q_codes.shape
    Hkv, Nk = k_codes.shape[1], k_codes.shape[2]
    kh = kv_head_of(Hq, Hkv)
    pos0 = Nk - Nq if q_pos0 is None else q_pos0
    sm = default_sm_scale(d) if sm_scale is None else F32(sm_scale)
    rows = np.arange(Nq) if rows is None else np.asarray(rows)
    heads = [(b, h) for b in range(B) for h in range(Hq)] if heads is None else heads
    sq_tok = expand_per_token(np.asarray(q_scales, F32), q_gran, B, Hq, Nq)
    nb = -(-Nk // BLOCK)
    sk_blk = expand_per_token(np.asarray(k_scales, F32), k_gran, B, Hkv, nb * BLOCK)[:, :, ::BLOCK]
    vis = visible_mask(rows, Nk, causal, pos0)
    bias2 = None
    if bias is not None:
        bias2 = (np.asarray(bias, F32)[rows] * LOG2E_F32).astype(F32)
    outs, bounds, lses = [], [], []
    for (b, h) in heads:
        g = kh[h]
        S = np.matmul(q_codes[b, h, rows].astype(F64), k_codes[b, g].astype(F64).T)
        c = block_factor(sq_tok[b, h, rows][:, None], sk_blk[b, g][None, :], sm)
        r = online_softmax_pv(S, c, v8[b, g], s_v[b, g], visible=vis, bias2=bias2,
                              p_quant=p_quant, want_bound=want_bound)
        outs.append(r["O"])
        lses.append(r["lse"])
        if want_bound:
            bounds.append(r["bound"])
    res = {"O": np.stack(outs), "lse": np.stack(lses)}
    if want_bound:
        res["bound"] = np.stack(bounds)
    return res


def attn_blockwise_real(Q, K, V, *, causal, q_pos0=None, sm_scale=None, bias=None,
                        ftype=F64, p_quant=None):
    """The same blockwise loop on real (unquantized) Q, K, V, for pinning the
    loop against dense softmax attention.  Returns [B, Hq, Nq, d] float64."""
    Q = np.asarray(Q, F64)
    K = np.asarray(K, F64)
    V = np.asarray(V, F64)
    B, Hq, Nq, d = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    kh = kv_head_of(Hq, Hkv)
    pos0 = Nk - Nq if q_pos0 is None else q_pos0
    sm = (1.0 / math.sqrt(d)) if sm_scale is None else sm_scale
    nb = -(-Nk // BLOCK)
    rows = np.arange(Nq)
    vis = visible_mask(rows, Nk, causal, pos0)
    bias2 = None if bias is None else np.asarray(bias, F64) * math.log2(math.e)
    out = np.zeros((B, Hq, Nq, d))
    c = np.full((Nq, nb), sm * math.log2(math.e), dtype=F64)
    for b in range(B):
        for h in range(Hq):
            S = Q[b, h] @ K[b, kh[h]].T
            r = online_softmax_pv(S, c, V[b, kh[h]], np.ones(d), visible=vis,
                                  bias2=bias2, p_quant=p_quant, ftype=ftype)
            out[b, h] = r["O"]
    return out


# ---------------------------------------------------------------------------
# Unquantized reference (reported beside parity, not gated).
# ---------------------------------------------------------------------------

def attn_fp64(Q, K, V, *, causal, q_pos0=None, sm_scale=None, bias=None,
              heads=None, rows=None):
    """softmax(Q K^T * sm_scale + bias, masked) V, dense, in float64."""
    Q = np.asarray(Q)
    K = np.asarray(K)
    V = np.asarray(V)
    B, Hq, Nq, d = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    group = Hq // Hkv
    pos0 = Nk - Nq if q_pos0 is None else q_pos0
    sm = (1.0 / math.sqrt(d)) if sm_scale is None else float(sm_scale)
    rows = np.arange(Nq) if rows is None else np.asarray(rows)
    heads = [(b, h) for b in range(B) for h in range(Hq)] if heads is None else heads
    # written out here rather than shared with the recipe, so that the dense
    # reference checks the recipe's mask and head mapping
    keys = np.arange(Nk)
    if causal:
        vis = keys[None, :] - rows[:, None] <= pos0
    else:
        vis = np.ones((len(rows), Nk), dtype=bool)
    outs = []
    for (b, h) in heads:
        s = (Q[b, h, rows].astype(F64) @ K[b, h // group].astype(F64).T) * sm
        if bias is not None:
            s = s + np.asarray(bias, F64)[rows]
        s = np.where(vis, s, -np.inf)
        mx = s.max(axis=1, keepdims=True)
        mx = np.where(np.isfinite(mx), mx, 0.0)
        p = np.exp(s - mx)
        den = p.sum(axis=1, keepdims=True)
        o = (p @ V[b, h // group].astype(F64)) / np.where(den > 0, den, 1.0)
        outs.append(o)
    return np.stack(outs)


# ---------------------------------------------------------------------------
# The whole recipe from inputs (a1-a10), used by tests and the CPU baseline.
# ---------------------------------------------------------------------------

def prepare(inp) -> dict:
    """Quantize one workload's inputs: returns codes, scales, V8 and s_v."""
    wl = inp.wl
    if wl.kv_codes:
        qc, qs, kc, ks = quantize_qk(inp.Q, K_codes=inp.K_codes, k_chan_scale=inp.K_scale,
                                     q_gran=wl.q_gran, k_gran=wl.k_gran)
        v8, s_v = quantize_v_codes(inp.V_codes, inp.V_scale)
        mu = None
    else:
        mu = smooth_k(inp.K)
        qc, qs, kc, ks = quantize_qk(inp.Q, inp.K, k_mean=mu, q_gran=wl.q_gran, k_gran=wl.k_gran)
        v8, s_v = quantize_v(inp.V)
    return {"mu": mu, "q_codes": qc, "q_scales": qs, "k_codes": kc, "k_scales": ks,
            "v8": v8, "s_v": s_v}


def run_workload(inp, prep=None, *, heads=None, rows=None, want_bound=False, p_quant="e4m3"):
    """Recipe output for chosen heads/rows of a workload (parity target).
    p_quant="int8" gives the static-127 int8 PV ablation instead."""
    wl = inp.wl
    prep = prepare(inp) if prep is None else prep
    return attn_fwd(prep["q_codes"], prep["q_scales"], prep["k_codes"], prep["k_scales"],
                    prep["v8"], prep["s_v"], q_gran=wl.q_gran, k_gran=wl.k_gran,
                    causal=wl.causal, q_pos0=wl.q_pos0, bias=inp.bias, heads=heads,
                    rows=rows, want_bound=want_bound, p_quant=p_quant)


def real_kv(inp):
    """The real-valued K and V a workload stands for (fp64 reference input)."""
    if inp.wl.kv_codes:
        K = inp.K_codes.astype(F64) * inp.K_scale[:, :, None, :].astype(F64)
        if inp.K_header_mean is not None:
            K = K + inp.K_header_mean[:, :, None, :].astype(F64)
        V = inp.V_codes.astype(F64) * inp.V_scale[:, :, None, :].astype(F64)
        return K, V
    return inp.K, inp.V


# ---------------------------------------------------------------------------
# Probability-mass diagnostic (ZINC-ATTN, "Then the easy matmul turns out to be
# the hard one" and its figure): how much of an attention row's probability
# mass lies below what a static-127 int8 grid can hold.  Round to nearest sends
# every probability below half a step, 0.5 / 127 ~ 0.0039, to zero.
# ---------------------------------------------------------------------------

INT8_ZERO_THRESHOLD = 0.5 / QMAX

# The figure's magnitude decades: < 1e-4, [1e-4, 1e-3), [1e-3, 1e-2),
# [1e-2, 1e-1), >= 1e-1.
MASS_DECADE_EDGES = (1e-4, 1e-3, 1e-2, 1e-1)


def kv_append(K_new, V_new, pos, k_chan_scale, v_chan_scale, k_mean, v_code_amax,
              k_codes, v_codes):
    """Append T tokens to an int8 KV cache whose header keeps a running channel
    mean of K ([ZINC-ATTN] "K's outliers, and the subtraction softmax does not
    notice": during decode K arrives one token at a time, the cache header
    keeps a running channel mean, and the mean lags by one token).

    For token t at cache position n = pos + t, per (batch, KV head, channel):
        k_code = clip(rint(fp32(fp32(K - mu) / s_k)), -127, 127)  (mu of the n earlier tokens)
        mu     = fp32(mu + fp32(fp32(K - mu) / (n + 1)))          (then the header moves on)
        v_code = clip(rint(fp32(V / s_v)), -127, 127);  amax = max(amax, |v_code|)
    Readings (the page gives none of these): the cache's codes use fixed
    per-channel scales s_k, s_v from its header; codes are x / s rounded half
    to even; the running mean is the plain fp32 recurrence above.

    K_new, V_new: [B, Hkv, T, d] values (bf16 inputs as float32).  k_mean,
    v_code_amax, k_chan_scale, v_chan_scale: [B, Hkv, d] float32.  k_codes,
    v_codes: [B, Hkv, capacity, d] int8.  Returns updated copies
    (k_mean, v_code_amax, k_codes, v_codes).
    """
    K_new = np.asarray(K_new, dtype=np.float32)
    V_new = np.asarray(V_new, dtype=np.float32)
    mu = np.array(k_mean, dtype=np.float32, copy=True)
    amax = np.array(v_code_amax, dtype=np.float32, copy=True)
    kc = np.array(k_codes, dtype=np.int8, copy=True)
    vc = np.array(v_codes, dtype=np.int8, copy=True)
    sk = np.asarray(k_chan_scale, dtype=np.float32)
    sv = np.asarray(v_chan_scale, dtype=np.float32)
    T = K_new.shape[2]
    for t in range(T):
        n = pos + t
        diff = (K_new[:, :, t, :] - mu).astype(np.float32)
        kc[:, :, n, :] = np.clip(np.rint((diff / sk).astype(np.float32)), -127, 127).astype(np.int8)
        mu = (mu + (diff / np.float32(n + 1)).astype(np.float32)).astype(np.float32)
        code_v = np.clip(np.rint((V_new[:, :, t, :] / sv).astype(np.float32)), -127, 127)
        vc[:, :, n, :] = code_v.astype(np.int8)
        amax = np.maximum(amax, np.abs(code_v).astype(np.float32))
    return mu, amax, kc, vc


def kv_header(v_codes, Nk):
    """The cache header's V part for a cache filled elsewhere: per (batch, KV
    head, channel) the largest |code| over rows 0..Nk-1 (0 for Nk = 0) -- the
    quantity kv_append keeps as tokens arrive."""
    v = np.asarray(v_codes)[:, :, :Nk, :].astype(np.int64)
    if Nk == 0:
        return np.zeros((v.shape[0], v.shape[1], v.shape[3]), np.float32)
    return np.abs(v).max(axis=2).astype(np.float32)


EXACT24_GROUP = 64   # q scaled per (head, 64-channel group)
EXACT24_CHUNK = 64   # P scaled per (row, 64-key chunk); also the online-softmax block


def split24(x):
    """x (fp32, |x| <= 127) -> int64 parts (h, l, m) with
    X = rint(fp32(x * 65536)) = h * 65536 + l * 256 + m, h and l signed bytes and
    m an unsigned byte (Strata PR, "What it does", "Operands": 24 bits, each
    part's product sum exact in int32)."""
    X = np.rint((np.asarray(x, np.float32) * np.float32(65536.0)).astype(np.float32)).astype(np.int64)
    m = X & 255
    r = (X - m) >> 8
    l = ((r + 128) & 255) - 128
    h = (r - l) >> 8
    return h, l, m


def attn_exact24(Q, k_codes, k_chan_scale, v_codes, v_chan_scale, *, causal, q_pos0=None,
                 sm_scale=None, heads=None, rows=None):
    """High-accuracy attention on an int8 KV cache with operands split exact to
    24 bits (Strata PR, "What it does", "Operands"; parity "Measured": max
    relative error ~2e-6 against FP64).  Steps, per (batch, query head):

    1. q' = fp32(q * s_k[c]) (the cache's K channel scales folded into q);
       per 64-channel group g over all the head's query rows,
       s_g = fp32(max|q'| / 127), x = fp32(q' / s_g), split24(x) -> (h, l, m).
    2. Per group, three exact integer dots with the K codes; S = sum over
       groups of fp32(s_g * Sh) + fp32(s_g/256 * Sl) + fp32(s_g/65536 * Sm),
       accumulated in fp32 in group order; t = fp32(S * fp32(sm_scale * log2 e)).
    3. Online softmax over 64-key chunks in order (running max m, P = 2^(t - m)
       in float64 here); per (row, chunk) s_p = fp32(max P / 127),
       x = fp32(P / s_p), split24(x) -> (h, l, m); three exact integer dots
       with the V codes give O_chunk = s_p * (Oh + Ol/256 + Om/65536).
    4. O = alpha * O + O_chunk, l = alpha * l + sum P (float64); out = O * s_v / l.

    Readings (not on the page): the K and V channel scales of the int8 cache
    are factored out of the dots (K's folded into q, V's applied at the end, so
    "p . v_scale" reduces to p); the chunk is 64 keys; P's chunk maximum is
    taken over the visible keys.  Q: [B, Hq, Nq, d] values; k_codes, v_codes:
    [B, Hkv, Nk, d] int8; scales [B, Hkv, d].  Returns out [len(heads), R, d]
    and lse (natural log of the softmax denominator of the scaled scores).
    """
    Q = np.asarray(Q, np.float32)
    B, Hq, Nq, d = Q.shape
    Hkv, Nk = k_codes.shape[1], k_codes.shape[2]
    G = Hq // Hkv
    if sm_scale is None:
        sm_scale = default_sm_scale(d)
    cfac = np.float32(np.float32(sm_scale) * LOG2E_F32)
    if q_pos0 is None:
        q_pos0 = Nk - Nq
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    rows = np.arange(Nq) if rows is None else np.asarray(rows)
    out = np.zeros((len(heads), len(rows), d))
    lse = np.zeros((len(heads), len(rows)))
    ng = d // EXACT24_GROUP
    for hi, (b, h) in enumerate(heads):
        kv = h // G
        qp = (Q[b, h] * k_chan_scale[b, kv][None, :]).astype(np.float32)          # [Nq, d]
        kc = k_codes[b, kv].astype(np.int64)                                       # [Nk, d]
        vc = v_codes[b, kv].astype(np.int64)
        S = np.zeros((len(rows), Nk), np.float32)
        for g in range(ng):
            cs = slice(g * EXACT24_GROUP, (g + 1) * EXACT24_GROUP)
            sg = np.float32(np.abs(qp[:, cs]).max() / np.float32(127.0))
            if sg == 0:
                continue
            x = (qp[rows][:, cs] / sg).astype(np.float32)
            ph, pl, pm = split24(x)
            Sh, Sl, Sm = ph @ kc[:, cs].T, pl @ kc[:, cs].T, pm @ kc[:, cs].T        # exact int64
            S = (S + (sg * Sh.astype(np.float32)).astype(np.float32)).astype(np.float32)
            S = (S + (np.float32(sg / 256) * Sl.astype(np.float32)).astype(np.float32)).astype(np.float32)
            S = (S + (np.float32(sg / 65536) * Sm.astype(np.float32)).astype(np.float32)).astype(np.float32)
        t = (S * cfac).astype(np.float32).astype(np.float64)
        vis = visible_mask(rows, Nk, causal, q_pos0)
        t[~vis] = -np.inf
        m = np.full(len(rows), -np.inf)
        l = np.zeros(len(rows))
        O = np.zeros((len(rows), d))
        for k0 in range(0, Nk, EXACT24_CHUNK):
            tk = t[:, k0:k0 + EXACT24_CHUNK]
            m_new = np.maximum(m, tk.max(axis=1))
            live = np.isfinite(m_new)
            prev = live & np.isfinite(m)
            alpha = np.where(prev, np.exp2(np.where(prev, m, 0.0) - np.where(prev, m_new, 0.0)), 0.0)
            P = np.where(live[:, None], np.exp2(tk - np.where(live, m_new, 0.0)[:, None]), 0.0)
            pmax = P.max(axis=1)
            sp = (pmax.astype(np.float32) / np.float32(127.0)).astype(np.float32)
            safe = np.where(sp > 0, sp, np.float32(1.0))
            x = (P.astype(np.float32) / safe[:, None]).astype(np.float32)
            x[sp == 0] = 0
            ph, pl, pm = split24(x)
            vcb = vc[k0:k0 + EXACT24_CHUNK]
            Oc = (ph @ vcb) + (pl @ vcb) / 256.0 + (pm @ vcb) / 65536.0
            O = alpha[:, None] * O + sp.astype(np.float64)[:, None] * Oc
            l = alpha * l + P.sum(axis=1)
            m = m_new
        sv = v_chan_scale[b, kv].astype(np.float64)
        ok = l > 0
        out[hi] = np.where(ok[:, None], O * sv[None, :] / np.where(ok, l, 1.0)[:, None], 0.0)
        lse[hi] = np.where(ok, (m + np.log2(np.where(ok, l, 1.0))) * np.log(2.0), -np.inf)
    return out, lse


INTSM_TILE = 64          # key tile of the integer online softmax (Bc)
INTSM_M0 = -(1 << 21)    # initial running max (QFlash Algorithm 1)


def intsm_constants(sq, sk, sm_scale):
    """Integer constants of QFlash's integer softmax, from the per-tensor
    scales ("QFlash", section 4.3 eq. (5)-(8), section 4.4 eq. (9)-(10)):
    s~ = fp32(fp32(fp32(sq * sk) * sm_scale) * log2 e) (the scale of an
    exponent in base 2); X0 = rint(fp32(1 / s~)) (the integer that stands for
    -1 in the exponent); the requantization of P (scale s~) to int8 codes of
    scale 1/127: ratio = fp32(127 * s~), n = ceil(log2 ratio), r = 8 - n,
    M = rint(ratio * 2^r).  Returns (s~, X0, M, r)."""
    st = np.float32(np.float32(np.float32(np.float32(sq) * np.float32(sk)) * np.float32(sm_scale)) * LOG2E_F32)
    x0 = int(np.rint(np.float32(np.float32(1.0) / st)))
    ratio = np.float32(np.float32(127.0) * st)
    f, e = np.frexp(np.float64(ratio))          # ratio = f * 2^e, f in [0.5, 1): exact
    n = int(e) - 1 if f == 0.5 else int(e)      # ceil(log2 ratio)
    r = 8 - n
    M = int(np.rint(np.float64(ratio) * 2.0 ** r))
    return st, max(x0, 1), M, r


def shift_exp2(X, x0):
    """QFlash's ShiftExp2 ("QFlash", section 4.3): for integer X <= 0,
    2^(s~ X) ~= s~ ((R >> 1) + X0) >> -Q with X = Q X0 + R, Q = X / X0
    truncated toward zero and R in (-X0, 0] (eq. (6)); 2^(s~ R) ~= s~ R / 2 + 1
    (eq. (7)).  Integer in, integer out (scale s~); int64 arrays."""
    X = np.asarray(X, dtype=np.int64)
    q = -((-X) // x0)                  # truncation toward zero for X <= 0
    R = X - q * x0                     # in (-x0, 0]
    base = (R >> 1) + x0               # arithmetic shift: floor(R / 2)
    sh = np.minimum(-q, 62)
    return np.where(-q >= 62, 0, base >> sh)


def requant_p(P, M, r):
    """QFlash's requantization (section 4.4, eq. (10)): Y = (X * M) >> r,
    clamped to the int8 codes [0, 127] of P's scale 1/127.  The shift is a
    multiplication by 2^-r, so a negative r (s~ > 2) shifts left."""
    PM = np.asarray(P, np.int64) * M
    return np.minimum(PM >> r if r >= 0 else PM << -r, 127)


def scale_release(x, alpha, x0):
    """ScaleRelease (named in "QFlash" section 4.6; its definition, Appendix
    B.1, is not in the pages -- PARITY UNPINNED): the reading taken here
    multiplies by the max-offset factor alpha (scale s~) and divides by the
    integer X0 ~= 1/s~ that stands for the inverse scale, floor division in
    int64: floor(x * alpha / X0)."""
    return (np.asarray(x, np.int64) * np.asarray(alpha, np.int64)) // x0


def attn_intsoftmax(q_codes, sq, k_codes, sk, v_codes, *, sm_scale=None, heads=None, rows=None):
    """QFlash's integer-only attention ("QFlash", Algorithm 1, sections 4.2-4.6):
    per query row, over key tiles of 64 in order: S = q.k (int32),
    m' = max(m, rowmax S) (m starts at -2^21), alpha = ShiftExp2(m - m'),
    P = ShiftExp2(S - m'), Y = requant(P), l = ScaleRelease(l, alpha) + sum Y,
    O = ScaleRelease(O, alpha) + Y.v (int32 dots); out = floor(O / l), int8
    codes of V's scale (s_O = s_V).  Per-tensor scales sq, sk (floats);
    q_codes [B, Hq, N, d], k/v codes [B, Hkv, N, d] int8.  No mask (the
    workloads are ViT/DeiT/Swin windows).  Returns int64 [len(heads), R, d]."""
    B, Hq, N, d = q_codes.shape
    Hkv = k_codes.shape[1]
    G = Hq // Hkv
    if sm_scale is None:
        sm_scale = default_sm_scale(d)
    _, x0, M, r = intsm_constants(sq, sk, sm_scale)
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    rows = np.arange(N) if rows is None else np.asarray(rows)
    Nk = k_codes.shape[2]
    out = np.zeros((len(heads), len(rows), d), np.int64)
    for hi, (b, h) in enumerate(heads):
        q = q_codes[b, h][rows].astype(np.int64)
        k = k_codes[b, h // G].astype(np.int64)
        v = v_codes[b, h // G].astype(np.int64)
        m = np.full(len(rows), INTSM_M0, np.int64)
        l = np.zeros(len(rows), np.int64)
        O = np.zeros((len(rows), d), np.int64)
        for k0 in range(0, Nk, INTSM_TILE):
            S = q @ k[k0:k0 + INTSM_TILE].T                   # exact int32 values
            m_new = np.maximum(m, S.max(axis=1))
            alpha = shift_exp2(m - m_new, x0)
            Y = requant_p(shift_exp2(S - m_new[:, None], x0), M, r)
            l = scale_release(l, alpha, x0) + Y.sum(axis=1)
            O = scale_release(O, alpha[:, None], x0) + Y @ v[k0:k0 + INTSM_TILE]
            m = m_new
        out[hi] = np.clip(O // np.maximum(l, 1)[:, None], -127, 127)
    return out


def attn_probs_fp64(Q, K, *, causal, q_pos0=None, sm_scale=None, bias=None, heads=None,
                    rows=None):
    """softmax(Q K^T * sm_scale + bias) of the chosen rows, dense, float64.
    Returns [len(heads), len(rows), Nk] (masked keys have probability 0)."""
    Q = np.asarray(Q, dtype=F64)
    K = np.asarray(K, dtype=F64)
    B, Hq, Nq, d = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    g = Hq // Hkv
    if sm_scale is None:
        sm_scale = float(default_sm_scale(d))
    q0 = (Nk - Nq) if q_pos0 is None else q_pos0
    heads = [(b, h) for b in range(B) for h in range(Hq)] if heads is None else heads
    rows = np.arange(Nq) if rows is None else np.asarray(rows)
    vis = visible_mask(rows, Nk, causal, q0)
    out = np.zeros((len(heads), len(rows), Nk), dtype=F64)
    for i, (b, h) in enumerate(heads):
        s = Q[b, h][rows] @ K[b, h // g].T * float(sm_scale)
        if bias is not None:
            s = s + np.asarray(bias, F64)[rows]
        s = np.where(vis, s, -np.inf)
        mx = s.max(axis=1, keepdims=True)
        e = np.where(vis, np.exp(s - np.where(np.isfinite(mx), mx, 0.0)), 0.0)
        tot = e.sum(axis=1, keepdims=True)
        out[i] = np.where(tot > 0, e / np.where(tot > 0, tot, 1.0), 0.0)
    return out


def mass_profile(probs, edges=MASS_DECADE_EDGES, threshold=INT8_ZERO_THRESHOLD):
    """Per row: the fraction of the row's probability mass in each magnitude
    bin (len(edges) + 1 bins) and below `threshold`.  probs [..., N] rows of
    probabilities (each row sums to 1, or to 0 for a fully masked row)."""
    p = np.asarray(probs, dtype=F64)
    tot = p.sum(axis=-1)
    safe = np.where(tot > 0, tot, 1.0)
    bounds = (0.0,) + tuple(edges) + (np.inf,)
    bins = np.stack([np.where((p >= lo) & (p < hi), p, 0.0).sum(axis=-1) / safe
                     for lo, hi in zip(bounds[:-1], bounds[1:])], axis=-1)
    # zeroed by the static-127 grid: rint(127 p) == 0, i.e. 127 p <= 1/2 (the
    # tie rounds to the even code 0)
    below = np.where(p * QMAX <= threshold * QMAX, p, 0.0).sum(axis=-1) / safe
    # the same threshold applied to p / max p: the flash-attention P = exp(s - m)
    # <= 1 is quantized relative to the row max, not after normalization
    pmax = p.max(axis=-1, keepdims=True)
    rel = p / np.where(pmax > 0, pmax, 1.0)
    below_rel = np.where(rel * QMAX <= threshold * QMAX, p, 0.0).sum(axis=-1) / safe
    return {"bins": bins, "below": below, "below_rel_max": below_rel}
