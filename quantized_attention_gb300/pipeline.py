"""The whole prefill path for one problem shape, with its device buffers.

``Problem.run`` issues, on the current stream, the library calls of the
recipe in order: K channel mean, Q/K int8 codes, per-channel e4m3 V, fused
attention.  Buffers are allocated once (PyTorch supplies the memory) and
reused across calls.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as qb


class Problem:
    def __init__(self, B, Hq, Hkv, Nq, Nk, d, *, causal=False, q_gran=qb.GRAN_BLOCK,
                 k_gran=qb.GRAN_BLOCK, q_pos0=None, kv_codes=False, out_dtype=qb.DT_F32,
                 bias_head_stride=0, want_lse=False, k_carrier=True, pv_mode=qb.PV_E4M3,
                 fused_prepass=True, fwd_kernel=qb.FWD_AUTO, device="cuda"):
        self.B, self.Hq, self.Hkv, self.Nq, self.Nk, self.d = B, Hq, Hkv, Nq, Nk, d
        self.kv_codes = kv_codes
        self.shape = qb.make_shape(B, Hq, Hkv, Nq, Nk, d)
        self.params = qb.make_params(causal=causal, q_gran=q_gran, k_gran=k_gran,
                                     out_dtype=out_dtype, q_pos0=q_pos0,
                                     bias_head_stride=bias_head_stride, pv_mode=pv_mode,
                                     fwd_kernel=fwd_kernel)
        self.ldv = qb.v_ld(Nk)
        dev = torch.device(device)
        i8, f32 = torch.int8, torch.float32
        self.q_codes = torch.empty((B, Hq, Nq, d), dtype=i8, device=dev)
        self.q_scales = torch.empty((qb.n_scales(q_gran, B, Hq, Nq),), dtype=f32, device=dev)
        self.k_codes = None if kv_codes else torch.empty((B, Hkv, Nk, d), dtype=i8, device=dev)
        self.k_scales = torch.empty((qb.n_scales(k_gran, B, Hkv, Nk),), dtype=f32, device=dev)
        self.k_mean = None if kv_codes else torch.empty((B, Hkv, d), dtype=f32, device=dev)
        # fp16 carriers of the K codes, written by quantize_qk and read by fwd
        # (None: fwd converts the codes itself, in the workspace)
        self.k_carrier = (torch.empty((B, Hkv, Nk, d), dtype=torch.float16, device=dev)
                          if k_carrier else None)
        self.v8t = torch.empty((B, Hkv, d, self.ldv), dtype=torch.uint8, device=dev)
        self.v_scales = torch.empty((B, Hkv, d), dtype=f32, device=dev)
        odt = torch.bfloat16 if out_dtype == qb.DT_BF16 else f32
        self.O = torch.empty((B, Hq, Nq, d), dtype=odt, device=dev)
        self.lse = torch.empty((B, Hq, Nq), dtype=f32, device=dev) if want_lse else None
        ws = max(qb.workspace_size(self.shape, self.params), 256)
        self.workspace = torch.empty((ws,), dtype=torch.uint8, device=dev)
        # qattn_prepare covers bf16 K/V with block granules (one or two
        # launches instead of four) and with tensor granules for heads of at
        # most 256 keys (two instead of five); other cases take the three calls
        self.fused_prepass = (fused_prepass and not kv_codes and Nk > 0 and
                              qb.prepare_launches(self.shape, self.params) > 0)

    def quantize(self, Q, K=None, V=None, *, K_codes=None, K_scale=None, V_codes=None,
                 V_scale=None, stream=None):
        """a1-a3: codes and scales for Q, K and V."""
        if self.kv_codes:
            qb.quantize_qk(Q, K_codes, qb.DT_I8, None, K_scale, self.shape, self.params,
                           self.q_codes, self.q_scales, None, self.k_scales, self.workspace, stream,
                           k_carrier=self.k_carrier)
            qb.quantize_v(V_codes, qb.DT_I8, V_scale, self.shape, self.v8t, self.ldv,
                          self.v_scales, self.workspace, stream)
            self._k_codes = K_codes
        elif self.fused_prepass:  # the same outputs in two launches
            qb.prepare(Q, K, V, self.shape, self.params, self.q_codes, self.q_scales,
                       self.k_codes, self.k_scales, self.k_mean, self.v8t, self.ldv,
                       self.v_scales, self.workspace, stream, k_carrier=self.k_carrier)
            self._k_codes = self.k_codes
        else:
            qb.smooth_k(K, self.shape, self.k_mean, self.workspace, stream)
            qb.quantize_qk(Q, K, qb.DT_BF16, self.k_mean, None, self.shape, self.params,
                           self.q_codes, self.q_scales, self.k_codes, self.k_scales,
                           self.workspace, stream, k_carrier=self.k_carrier)
            qb.quantize_v(V, qb.DT_BF16, None, self.shape, self.v8t, self.ldv, self.v_scales,
                          self.workspace, stream)
            self._k_codes = self.k_codes

    def quantize_q(self, Q, K_scale, stream=None):
        """Decode on an int8 cache: only the new tokens' Q codes (K's channel
        scales folded in) and the K scales; the cache itself stays as stored."""
        qb.quantize_qk(Q, self._cache_k, qb.DT_I8, None, K_scale, self.shape, self.params,
                       self.q_codes, self.q_scales, None, self.k_scales, self.workspace, stream)

    def set_cache(self, K_codes, V_codes, V_scale, K_scale=None, K_mean=None):
        """The int8 KV cache qattn_decode reads ([B, Hkv, capacity, d], rows
        0..Nk-1 in use) and its header: the per-channel max |V code| of the
        rows in use, and for qattn_kv_append the channel scales and the
        running channel mean of K (zeros if not given)."""
        self._cache_k, self._cache_v, self._cache_vs = K_codes, V_codes, V_scale
        self._cache_vamax = torch.empty(V_scale.shape, dtype=torch.float32, device=V_codes.device)
        qb.kv_header_init(V_codes, self.shape.Nk, self._cache_vamax)
        self._cache_ks = K_scale
        self._cache_kmean = (K_mean.clone().contiguous() if K_mean is not None
                             else torch.zeros_like(V_scale))
        self.params.kv_capacity = K_codes.shape[2]

    def append(self, K_new, V_new, pos: int, stream=None):
        """qattn_kv_append: tokens K_new, V_new (bf16 [B, Hkv, T, d]) into the
        cache at rows pos.., updating the header (running K mean, V max)."""
        qb.kv_append(K_new, V_new, pos, self._cache_ks, self._cache_vs, self._cache_kmean,
                     self._cache_vamax, self._cache_k, self._cache_v, stream)

    def decode(self, stream=None):
        """qattn_decode on the cache given to set_cache."""
        qb.decode(self.q_codes, self.q_scales, self._cache_k, self.k_scales, self._cache_v,
                  self._cache_vs, self._cache_vamax, self.shape, self.params, self.O, self.lse,
                  self.workspace, stream)
        return self.O

    def attend(self, bias: Optional[torch.Tensor] = None, stream=None,
               out: Optional[torch.Tensor] = None):
        """a4-a10: the fused attention kernel on the quantized operands, into
        ``out`` (shaped and typed like ``self.O``) or ``self.O``."""
        O = self.O if out is None else out
        if O.shape != self.O.shape or O.dtype != self.O.dtype or not O.is_contiguous():
            raise ValueError("out must be a contiguous tensor like Problem.O")
        qb.fwd(self.q_codes, self.q_scales, self._k_codes, self.k_scales, self.v8t, self.ldv,
               self.v_scales, bias, self.shape, self.params, O, self.lse, self.workspace,
               stream, k_carrier=self.k_carrier)
        return O

    def short_fwd(self) -> bool:
        """Whether qattn_fwd runs a warp-level short-sequence kernel (the
        library's own choice, asked of it)."""
        return qb.fwd_kernel_choice(self.shape, self.params) == qb.FWD_SHORT

    def kernel_launches(self) -> int:
        """Kernels of this library that one ``run`` launches (memsets excluded)."""
        # [K carriers converted in qattn_fwd's workspace,] the attention kernel
        fwd = 1 + int(self.k_carrier is None and not self.short_fwd())
        if self.fused_prepass:
            return qb.prepare_launches(self.shape, self.params) + fwd
        two_pass = (self.params.q_gran != qb.GRAN_BLOCK or
                    (not self.kv_codes and self.params.k_gran != qb.GRAN_BLOCK))
        n = 1 + int(two_pass)                        # Q and K codes (one grid)
        if self.kv_codes:
            n += int(self.k_carrier is not None)     # K carriers (K scales: the Q launch)
        else:
            n += 1                                   # channel mean
        n += 2                                       # V amax, V e4m3 transpose
        return n + fwd

    def decode_launches(self, append: bool = False) -> int:
        """Kernels one [append +] quantize_q + decode launches: [the cache
        append,] Q codes with the K scales set to 1 (two passes for a
        tensor/head granule), then the decode's two."""
        return int(append) + 1 + int(self.params.q_gran != qb.GRAN_BLOCK) + 2

    def run(self, Q, K=None, V=None, *, K_codes=None, K_scale=None, V_codes=None,
            V_scale=None, bias=None, stream=None, out=None):
        self.quantize(Q, K, V, K_codes=K_codes, K_scale=K_scale, V_codes=V_codes,
                      V_scale=V_scale, stream=stream)
        return self.attend(bias, stream, out)


class OverlappedSteps:
    """Steps whose inputs come from pinned host memory and whose result goes
    back to pinned host memory, with step i's host-to-device copies, step
    i-1's kernels and step i-2's device-to-host copy in flight together.

    Two device sets of inputs and outputs and two pinned host outputs
    alternate; three streams (copy in, compute, copy out) are ordered by
    events: a set's inputs are overwritten only after the compute that read
    them, its output only after the copy that read it.  ``compute(dev_in,
    dev_out, stream)`` issues one step's kernels on ``stream``.  Device
    buffers are allocated once, like those of ``Problem``.
    """

    def __init__(self, host_inputs, out_like: torch.Tensor, compute, device="cuda"):
        # host_inputs: one dict of pinned tensors, or a list of them used in turn
        self.host_inputs = host_inputs if isinstance(host_inputs, list) else [host_inputs]
        for h in self.host_inputs:
            for t in h.values():
                if not t.is_pinned():
                    raise ValueError("host inputs must be pinned")
        first = self.host_inputs[0]
        dev = torch.device(device)
        self.dev_in = [{k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in first.items()}
                       for _ in range(2)]
        self.dev_out = [torch.empty_like(out_like, device=dev) for _ in range(2)]
        self.host_out = [torch.empty(out_like.shape, dtype=out_like.dtype).pin_memory()
                         for _ in range(2)]
        self.compute = compute
        self.s_in, self.s_comp, self.s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_comp = [torch.cuda.Event() for _ in range(2)]
        self.ev_out = [torch.cuda.Event() for _ in range(2)]
        self.steps = 0

    def step(self, before=None):
        """Issue one step (asynchronously); ``before(stream)`` runs on the
        compute stream ahead of the step's kernels.  Returns the pinned host
        tensor that receives the step's result once ``sync()`` returns (it is
        reused two steps later)."""
        b = self.steps & 1
        host = self.host_inputs[self.steps % len(self.host_inputs)]
        if self.steps >= 2:
            self.s_in.wait_event(self.ev_comp[b])    # the compute two steps back read dev_in[b]
        with torch.cuda.stream(self.s_in):
            for k, v in host.items():
                self.dev_in[b][k].copy_(v, non_blocking=True)
        self.ev_in[b].record(self.s_in)
        self.s_comp.wait_event(self.ev_in[b])
        if self.steps >= 2:
            self.s_comp.wait_event(self.ev_out[b])   # dev_out[b]'s copy two steps back is done
        if before is not None:
            before(self.s_comp)
        self.compute(self.dev_in[b], self.dev_out[b], self.s_comp)
        self.ev_comp[b].record(self.s_comp)
        self.s_out.wait_event(self.ev_comp[b])
        with torch.cuda.stream(self.s_out):
            self.host_out[b].copy_(self.dev_out[b], non_blocking=True)
        self.ev_out[b].record(self.s_out)
        self.steps += 1
        return self.host_out[b]

    def sync(self):
        """Wait for every step issued so far."""
        for s in (self.s_in, self.s_comp, self.s_out):
            s.synchronize()


class QFlashProblem:
    """QFlash's integer-only attention for one shape: per-tensor int8 codes of
    bf16 Q, K and V ("QFlash", section 4, eq. (1)-(2), made by
    qattn_quantize_qk's per-tensor Q path: V as a query tensor with no keys),
    then qattn_fwd_intsoftmax.  The output is int8 codes of V's scale."""

    def __init__(self, B, Hq, Hkv, Nq, Nk, d, *, sm_scale=0.0, device="cuda"):
        dev = torch.device(device)
        self.shape = qb.make_shape(B, Hq, Hkv, Nq, Nk, d)
        self.params = qb.make_params(sm_scale=sm_scale)
        tensor = qb.make_params(q_gran=qb.GRAN_TENSOR, k_gran=qb.GRAN_TENSOR)
        self._qk = (qb.make_shape(B, Hq, Hkv, Nq, Nk, d), tensor)
        self._v = (qb.make_shape(B, Hkv, Hkv, Nk, 0, d), tensor)
        i8, f32 = torch.int8, torch.float32
        self.q_codes = torch.empty((B, Hq, Nq, d), dtype=i8, device=dev)
        self.k_codes = torch.empty((B, Hkv, Nk, d), dtype=i8, device=dev)
        self.v_codes = torch.empty((B, Hkv, Nk, d), dtype=i8, device=dev)
        self.q_scale = torch.empty(1, dtype=f32, device=dev)
        self.k_scale = torch.empty(1, dtype=f32, device=dev)
        self.v_scale = torch.empty(1, dtype=f32, device=dev)
        self.O = torch.empty((B, Hq, Nq, d), dtype=i8, device=dev)
        ws = max(qb.workspace_size(*self._qk), qb.workspace_size(*self._v), 256)
        self.workspace = torch.empty((ws,), dtype=torch.uint8, device=dev)

    def quantize(self, Q, K, V, stream=None):
        qb.quantize_qk(Q, K, qb.DT_BF16, None, None, *self._qk, self.q_codes, self.q_scale,
                       self.k_codes, self.k_scale, self.workspace, stream)
        qb.quantize_qk(V, None, qb.DT_BF16, None, None, *self._v, self.v_codes, self.v_scale,
                       None, None, self.workspace, stream)

    def attend(self, stream=None, out=None):
        O = self.O if out is None else out
        qb.fwd_intsoftmax(self.q_codes, self.q_scale, self.k_codes, self.k_scale, self.v_codes,
                          self.shape, self.params, O, stream)
        return O

    def run(self, Q, K, V, stream=None, out=None):
        self.quantize(Q, K, V, stream)
        return self.attend(stream, out)

    @staticmethod
    def kernel_launches() -> int:
        """Kernels one run launches: two passes per per-tensor quantize call
        (amax, codes), then the attention kernel."""
        return 2 + 2 + 1


def problem_for(wl, **kw) -> Problem:
    """A Problem sized for a workload from quantized_attention_gb300.inputs."""
    return Problem(wl.B, wl.Hq, wl.Hkv, wl.Nq, wl.Nk, wl.d, causal=wl.causal, q_gran=wl.q_gran,
                   k_gran=wl.k_gran, q_pos0=wl.q_pos0, kv_codes=wl.kv_codes, **kw)


def device_inputs(inp, device="cuda") -> dict:
    """Host inputs (numpy) -> device tensors with the library's dtypes."""
    def bf16(x):
        return torch.from_numpy(x).to(device=device, dtype=torch.bfloat16)

    d = {"Q": bf16(inp.Q)}
    if inp.wl.kv_codes:
        d["K_codes"] = torch.from_numpy(inp.K_codes).to(device)
        d["K_scale"] = torch.from_numpy(inp.K_scale).to(device)
        d["V_codes"] = torch.from_numpy(inp.V_codes).to(device)
        d["V_scale"] = torch.from_numpy(inp.V_scale).to(device)
    else:
        d["K"] = bf16(inp.K)
        d["V"] = bf16(inp.V)
    if inp.bias is not None:
        d["bias"] = torch.from_numpy(inp.bias).to(device)
    return d
