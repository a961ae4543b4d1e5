"""Seeded synthetic workloads for quantized attention prefill.

This module only draws random inputs; it holds none of the quantization
recipe's arithmetic (no channel mean, no scale search, no rounding to codes
with a data-derived scale).  Both the CUDA path and the CPU oracle receive the
arrays it returns.

Shapes follow the pages' workloads:

* ``tiny``      1 head, 256 tokens, d=64, three K channels offset by +8.
* ``vit``       ViT-B/16 attention (QFlash, Table 1, workload A3: 12 heads x
                197 tokens x d=64), 64 images.  K has per-channel offsets and
                three channels scaled x20.  Per-tensor Q/K scales.
* ``swin``      Swin window attention (QFlash, Table 1, A4-A7: 49-token
                windows, d=32), 4096 windows x 4 heads, one 49x49 bias.
* ``llm8k``     LLM prefill, 32 query heads / 8 KV heads, 8192 tokens, d=128,
                causal.  K carries a per-channel mean and five outlier
                channels at 12, 18.5, 26, 37 and 44 times the median channel
                magnitude ("int8 Flash Attention on RDNA4", the K-outlier
                figure).
* ``chunk32k``  chunked long-context prefill: 2048 queries at positions
                30720..32767 against 32768 cached keys held as int8 codes with
                per-(head, channel) fp32 scales (the int8 KV cache of the same
                post, "What actually changed for decode").

Inputs are generated in fp32 with ``numpy.random.Generator(PCG64(seed))`` and
rounded to bf16 (round to nearest even) where the workload is bf16.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

GRAN_TENSOR = 0
GRAN_HEAD = 1
GRAN_BLOCK = 2

#: channels of K that carry the outliers in the ``llm8k`` structure
LLM_OUTLIER_CHANNELS = (7, 35, 62, 91, 118)
#: outlier magnitudes relative to the median channel (K-outlier figure, raw K)
LLM_OUTLIER_RATIOS = (12.0, 18.5, 26.0, 37.0, 44.0)
#: outlier magnitudes relative to the median channel after mean subtraction
#: (the same figure: every channel lands between 0.5x and 4.1x)
CACHE_OUTLIER_RATIOS = (2.2, 2.6, 3.1, 3.6, 4.1)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    q_gran: int
    k_gran: int
    seed: int
    q_pos0: Optional[int] = None  # None: Nk - Nq (bottom-right alignment)
    has_bias: bool = False
    kv_codes: bool = False  # K/V arrive as int8 codes with per-channel scales

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def pos0(self) -> int:
        return self.Nk - self.Nq if self.q_pos0 is None else self.q_pos0

    def unmasked_pairs(self) -> int:
        """(query, key) pairs that are not masked, over all batches and heads."""
        if not self.causal:
            per_head = self.Nq * self.Nk
        else:
            i = np.arange(self.Nq, dtype=np.int64)
            per_head = int(np.clip(self.pos0 + i + 1, 0, self.Nk).sum())
        return per_head * self.B * self.Hq


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 1, 256, 256, 64, False, GRAN_BLOCK, GRAN_BLOCK, 1),
    "vit": Workload("vit", 64, 12, 12, 197, 197, 64, False, GRAN_TENSOR, GRAN_TENSOR, 2),
    "swin": Workload("swin", 4096, 4, 4, 49, 49, 32, False, GRAN_BLOCK, GRAN_BLOCK, 3,
                     has_bias=True),
    "llm8k": Workload("llm8k", 1, 32, 8, 8192, 8192, 128, True, GRAN_BLOCK, GRAN_BLOCK, 4),
    "chunk32k": Workload("chunk32k", 1, 32, 8, 2048, 32768, 128, True, GRAN_BLOCK, GRAN_BLOCK,
                         5, q_pos0=30720, kv_codes=True),
    # one decode token at position 32767 against the chunk32k-shaped int8 cache
    "decode32k": Workload("decode32k", 1, 32, 8, 1, 32768, 128, True, GRAN_BLOCK, GRAN_BLOCK,
                          6, kv_codes=True),
}


def to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest even); returned as exact fp32 values."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def _llm_keys(rng: np.random.Generator, B: int, H: int, N: int, d: int) -> np.ndarray:
    """K = Z * sigma_c + mu_c with five outlier channels (fp32, before bf16)."""
    K = np.empty((B, H, N, d), dtype=np.float32)
    out = np.array([c for c in LLM_OUTLIER_CHANNELS if c < d], dtype=np.int64)
    ratios = np.array(LLM_OUTLIER_RATIOS[: len(out)], dtype=np.float32)
    for b in range(B):
        for h in range(H):
            mu = (0.5 * _normal(rng, (d,))).astype(np.float32)
            sigma = np.ones(d, dtype=np.float32)
            z = _normal(rng, (N, d))
            typical = z * sigma + mu
            a_med = float(np.median(np.abs(typical).max(axis=0)))
            signs = np.where(rng.random(len(out)) < 0.5, -1.0, 1.0).astype(np.float32)
            mu[out] = signs * ratios * a_med
            sigma[out] = 2.0
            K[b, h] = z * sigma + mu
    return K


@dataclasses.dataclass
class Inputs:
    """One workload's inputs (numpy, host).  bf16 tensors are fp32 arrays of
    bf16-exact values; int8 codes are int8 arrays."""
    wl: Workload
    Q: np.ndarray
    K: Optional[np.ndarray] = None          # bf16 path
    V: Optional[np.ndarray] = None
    K_codes: Optional[np.ndarray] = None    # int8-cache path
    K_scale: Optional[np.ndarray] = None    # [B, Hkv, d] fp32
    K_header_mean: Optional[np.ndarray] = None  # [B, Hkv, d] fp32 (cache header)
    V_codes: Optional[np.ndarray] = None
    V_scale: Optional[np.ndarray] = None
    bias: Optional[np.ndarray] = None       # [Nq, Nk] fp32, natural-log units


def make_inputs(wl: Workload) -> Inputs:
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    B, Hq, Hkv, Nq, Nk, d = wl.B, wl.Hq, wl.Hkv, wl.Nq, wl.Nk, wl.d
    name = wl.name.split("@")[0]
    Q = to_bf16(_normal(rng, (B, Hq, Nq, d)))
    if wl.kv_codes:
        return _make_cache_inputs(rng, wl, Q)
    if name == "vit":
        K = _normal(rng, (B, Hkv, Nk, d))
        off = (np.sqrt(2.0) * _normal(rng, (Hkv, d))).astype(np.float32)
        gain = np.ones(d, dtype=np.float32)
        gain[[c for c in (5, 29, 51) if c < d]] = 20.0
        K = to_bf16((K + off[None, :, None, :]) * gain)
    elif name == "llm8k":
        K = to_bf16(_llm_keys(rng, B, Hkv, Nk, d))
    else:
        K = _normal(rng, (B, Hkv, Nk, d))
        if name == "tiny":
            K[..., [c for c in (3, 17, 42) if c < d]] += 8.0
        K = to_bf16(K)
    V = to_bf16(_normal(rng, (B, Hkv, Nk, d)))
    bias = _normal(rng, (Nq, Nk)) if wl.has_bias else None
    return Inputs(wl, Q, K=K, V=V, bias=bias)


def _make_cache_inputs(rng: np.random.Generator, wl: Workload, Q: np.ndarray) -> Inputs:
    """int8 K/V cache: codes shaped by N(0,1) over +-4.5 sigma, per-channel scales.

    K's five outlier channels keep their post-mean-subtraction magnitude
    (2.2-4.1x the median) in the per-channel scales; the raw channel means,
    which carry the 12-44x outliers, sit in the cache header and matter only
    to the unquantized fp64 reference (softmax ignores them exactly)."""
    B, Hkv, Nk, d = wl.B, wl.Hkv, wl.Nk, wl.d
    span = np.float32(127.0 / 4.5)
    kz = _normal(rng, (B, Hkv, Nk, d))
    K_codes = np.clip(np.rint(kz * span), -127, 127).astype(np.int8)
    sig = rng.uniform(0.5, 1.5, size=(B, Hkv, d)).astype(np.float32)
    out = [c for c in LLM_OUTLIER_CHANNELS if c < d]
    sig[:, :, out] = np.array(CACHE_OUTLIER_RATIOS[: len(out)], dtype=np.float32)
    K_scale = (sig / span).astype(np.float32)
    hdr = (0.5 * _normal(rng, (B, Hkv, d))).astype(np.float32)
    signs = np.where(rng.random((B, Hkv, len(out))) < 0.5, -1.0, 1.0).astype(np.float32)
    hdr[:, :, out] = signs * np.array(LLM_OUTLIER_RATIOS[: len(out)], dtype=np.float32) * 4.5
    vz = _normal(rng, (B, Hkv, Nk, d))
    V_codes = np.clip(np.rint(vz * span), -127, 127).astype(np.int8)
    V_scale = (rng.uniform(0.8, 1.2, size=(B, Hkv, d)) / span).astype(np.float32)
    return Inputs(wl, Q, K_codes=K_codes, K_scale=K_scale, K_header_mean=hdr,
                  V_codes=V_codes, V_scale=V_scale)


def make_append_tokens(inp: Inputs, T: int, seed: int = 0):
    """T new tokens for an int8-cache workload, shaped like its cache: raw K =
    the header's channel mean + N(0, sigma_c) with the cache's channel spread,
    V = N(0, 1) at the V codes' scale; bf16 values as fp32, [B, Hkv, T, d]."""
    wl = inp.wl
    rng = np.random.Generator(np.random.PCG64(10007 * wl.seed + seed))
    span = np.float32(127.0 / 4.5)
    sig = (inp.K_scale * span)[:, :, None, :]
    K = inp.K_header_mean[:, :, None, :] + _normal(rng, (wl.B, wl.Hkv, T, wl.d)) * sig
    V = _normal(rng, (wl.B, wl.Hkv, T, wl.d)) * (inp.V_scale * span)[:, :, None, :]
    return to_bf16(K.astype(np.float32)), to_bf16(V.astype(np.float32))


def small(name: str, **kw) -> Workload:
    """A reduced-size copy of a named workload (same structure, new sizes)."""
    return WORKLOADS[name].replace(name=name + "@small", **kw)
