"""ctypes binding of libqattn.so (the C ABI in include/qattn.h).

Argument marshalling only: every step of the recipe runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  The
functions raise if the library is missing -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

# QATTN_LIBRARY: the path of another build of the library to load instead
# (e.g. the checked build, _lib/check/libqattn.so)
_LIB_PATH = os.environ.get("QATTN_LIBRARY") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), "_lib", "libqattn.so")
_lib = None

OK = 0
FWD_AUTO, FWD_TC, FWD_SHORT = 0, 1, 2
ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE, ERR_BOUNDS = 1, 2, 3, 4, 5, 6
GRAN_TENSOR, GRAN_HEAD, GRAN_BLOCK = 0, 1, 2
DT_BF16, DT_F32, DT_I8, DT_E4M3 = 0, 1, 2, 3
POS0_BOTTOM_RIGHT = -(2 ** 63)
PV_E4M3, PV_INT8 = 0, 1

EXPORTED = (
    "qattn_version", "qattn_status_string", "qattn_workspace_size", "qattn_v_ld",
    "qattn_smooth_k", "qattn_quantize_qk", "qattn_quantize_v", "qattn_fwd",
    "qattn_debug_qk_scores", "qattn_get_error", "qattn_quantize_v_noalloc", "qattn_decode",
    "qattn_kv_append", "qattn_fwd_exact24", "qattn_fwd_intsoftmax", "qattn_prepare",
    "qattn_fwd_kernel_choice", "qattn_prepare_launches", "qattn_debug_wait_timeout",
    "qattn_peak_loop", "qattn_kv_header_init", "qattn_checked", "qattn_debug_bounds_probe",
)


class QattnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("Hq", ctypes.c_int64), ("Hkv", ctypes.c_int64),
                ("Nq", ctypes.c_int64), ("Nk", ctypes.c_int64), ("d", ctypes.c_int64)]


class Params(ctypes.Structure):
    _fields_ = [("causal", ctypes.c_int32), ("q_gran", ctypes.c_int32),
                ("k_gran", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("q_pos0", ctypes.c_int64), ("sm_scale", ctypes.c_float),
                ("pv_mode", ctypes.c_int32), ("bias_head_stride", ctypes.c_int64),
                ("kv_capacity", ctypes.c_int64), ("fwd_kernel", ctypes.c_int32)]


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Loads libqattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with quantized_attention_gb300.build.build()")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    PS, PP = ctypes.POINTER(Shape), ctypes.POINTER(Params)
    L.qattn_version.restype = ctypes.c_int
    L.qattn_status_string.restype = ctypes.c_char_p
    L.qattn_status_string.argtypes = [ctypes.c_int]
    L.qattn_workspace_size.restype = sz
    L.qattn_workspace_size.argtypes = [PS, PP]
    L.qattn_v_ld.restype = i64
    L.qattn_v_ld.argtypes = [i64]
    L.qattn_smooth_k.argtypes = [vp, vp, PS, vp, vp, sz, vp]
    L.qattn_quantize_qk.argtypes = [vp, vp, vp, vp, ctypes.c_int, vp, vp, PS, PP, vp, vp, vp, vp,
                                    vp, vp, sz, vp]
    L.qattn_quantize_v.argtypes = [vp, vp, ctypes.c_int, vp, PS, vp, i64, vp, vp, sz, vp]
    L.qattn_prepare.argtypes = [vp, vp, vp, vp, vp, vp, PS, PP, vp, vp, vp, vp, vp, vp, vp, i64, vp,
                                vp, sz, vp]
    L.qattn_quantize_v_noalloc.argtypes = [vp, ctypes.c_int, vp, PS, vp, i64, vp, vp]
    L.qattn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, vp, vp, PS, PP, vp, vp, vp, sz, vp]
    L.qattn_debug_qk_scores.argtypes = [vp, vp, PS, vp, vp, sz, vp]
    L.qattn_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, PS, PP, vp, vp, vp, sz, vp]
    L.qattn_kv_append.argtypes = [vp, vp, i64, i64, i64, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp]
    L.qattn_kv_header_init.argtypes = [vp, i64, i64, i64, i64, i64, vp, vp]
    L.qattn_fwd_exact24.argtypes = [vp, vp, vp, vp, vp, PS, PP, vp, vp, vp, sz, vp]
    L.qattn_fwd_intsoftmax.argtypes = [vp, vp, vp, vp, vp, PS, PP, vp, vp]
    L.qattn_get_error.argtypes = [vp]
    L.qattn_debug_wait_timeout.argtypes = [vp, vp]
    L.qattn_fwd_kernel_choice.argtypes = [PS, PP]
    L.qattn_fwd_kernel_choice.restype = ctypes.c_int
    L.qattn_prepare_launches.argtypes = [PS, PP]
    L.qattn_prepare_launches.restype = ctypes.c_int
    L.qattn_checked.argtypes = []
    L.qattn_checked.restype = ctypes.c_int
    L.qattn_debug_bounds_probe.argtypes = [vp]
    ci = ctypes.c_int
    L.qattn_peak_loop.argtypes = [ci, ci, ci, ci, vp, vp, vp, vp]
    L.qattn_peak_loop.restype = ci
    for name in ("qattn_smooth_k", "qattn_quantize_qk", "qattn_quantize_v", "qattn_fwd",
                 "qattn_decode", "qattn_kv_append", "qattn_fwd_exact24", "qattn_fwd_intsoftmax",
                 "qattn_debug_qk_scores", "qattn_get_error", "qattn_quantize_v_noalloc",
                 "qattn_prepare", "qattn_debug_wait_timeout", "qattn_kv_header_init",
                 "qattn_debug_bounds_probe"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def checked() -> bool:
    """Whether the loaded library is the checked build (QATTN_CHECK=1)."""
    return bool(lib().qattn_checked())


def debug_bounds_probe(stream=None):
    """One guard that fails for half a warp, touching no memory: the checked
    build then reports ERR_BOUNDS from get_error(), the normal build OK."""
    _check(lib().qattn_debug_bounds_probe(_stream(stream)), "qattn_debug_bounds_probe")


def status_string(st: int) -> str:
    return lib().qattn_status_string(st).decode()


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _nbytes(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def _stream(stream: Optional[torch.cuda.Stream] = None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(st: int, where: str):
    if st != OK:
        raise QattnError(st, where)


def _dense(t: torch.Tensor, dtype, name: str):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _input(t: Optional[torch.Tensor], dtype, name: str):
    """An input the pre-pass reads at any strides: returns its strides as a
    ctypes int64[4] (None when dense).  The last stride must be 1 and the
    others multiples of 16 bytes (the library checks and rejects otherwise)."""
    if t is None:
        return None
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != 4:
        raise ValueError(f"{name} must be 4-D [B, H, N, d]")
    if t.is_contiguous():
        return None
    return (ctypes.c_int64 * 4)(*t.stride())


def make_shape(B, Hq, Hkv, Nq, Nk, d) -> Shape:
    return Shape(B, Hq, Hkv, Nq, Nk, d)


def make_params(causal=False, q_gran=GRAN_BLOCK, k_gran=GRAN_BLOCK, out_dtype=DT_F32,
                q_pos0=None, sm_scale=0.0, bias_head_stride=0, pv_mode=PV_E4M3,
                kv_capacity=0, fwd_kernel=0) -> Params:
    return Params(int(bool(causal)), q_gran, k_gran, out_dtype,
                  POS0_BOTTOM_RIGHT if q_pos0 is None else int(q_pos0), float(sm_scale),
                  int(pv_mode), int(bias_head_stride), int(kv_capacity), int(fwd_kernel))


def version() -> int:
    return lib().qattn_version()


def workspace_size(shape: Shape, params: Params) -> int:
    return lib().qattn_workspace_size(ctypes.byref(shape), ctypes.byref(params))


def v_ld(Nk: int) -> int:
    return lib().qattn_v_ld(Nk)


def n_scales(gran: int, B: int, H: int, N: int) -> int:
    return {GRAN_TENSOR: 1, GRAN_HEAD: B * H}.get(gran, B * H * ((N + 127) // 128))


def smooth_k(K, shape, k_mean, workspace, stream=None):
    ks = _input(K, torch.bfloat16, "K")
    _dense(k_mean, torch.float32, "k_mean")
    _check(lib().qattn_smooth_k(_p(K), ks, ctypes.byref(shape), _p(k_mean), _p(workspace),
                                _nbytes(workspace), _stream(stream)),
           "qattn_smooth_k")


def quantize_qk(Q, K, k_dtype, k_mean, k_chan_scale, shape, params, q_codes, q_scales,
                k_codes, k_scales, workspace, stream=None, k_carrier=None):
    qs = _input(Q, torch.bfloat16, "Q")
    ks = _input(K, torch.int8 if k_dtype == DT_I8 else torch.bfloat16, "K")  # None: no keys
    if k_carrier is not None:
        _dense(k_carrier, torch.float16, "k_carrier")
    _check(lib().qattn_quantize_qk(_p(Q), qs, _p(K), ks, k_dtype, _p(k_mean), _p(k_chan_scale),
                                   ctypes.byref(shape), ctypes.byref(params), _p(q_codes),
                                   _p(q_scales), _p(k_codes), _p(k_scales), _p(k_carrier),
                                   _p(workspace), _nbytes(workspace),
                                   _stream(stream)),
           "qattn_quantize_qk")


def prepare(Q, K, V, shape, params, q_codes, q_scales, k_codes, k_scales, k_mean, v8t, ldv,
            v_scales, workspace, stream=None, k_carrier=None):
    """qattn_prepare: K mean, Q/K codes and V's e4m3 codes in two launches."""
    st = [_input(t, torch.bfloat16, name) for t, name in ((Q, "Q"), (K, "K"), (V, "V"))]
    if k_carrier is not None:
        _dense(k_carrier, torch.float16, "k_carrier")
    _check(lib().qattn_prepare(_p(Q), st[0], _p(K), st[1], _p(V), st[2], ctypes.byref(shape),
                               ctypes.byref(params),
                               _p(q_codes), _p(q_scales), _p(k_codes), _p(k_scales),
                               _p(k_carrier), _p(k_mean), _p(v8t), ldv, _p(v_scales),
                               _p(workspace), _nbytes(workspace),
                               _stream(stream)),
           "qattn_prepare")


def quantize_v(V, v_dtype, v_chan_scale, shape, v8t, ldv, v_scales, workspace, stream=None):
    vs = _input(V, torch.int8 if v_dtype == DT_I8 else torch.bfloat16, "V")
    _check(lib().qattn_quantize_v(_p(V), vs, v_dtype, _p(v_chan_scale), ctypes.byref(shape), _p(v8t),
                                  ldv, _p(v_scales), _p(workspace),
                                  _nbytes(workspace), _stream(stream)),
           "qattn_quantize_v")


def quantize_v_noalloc(V, v_dtype, v_chan_scale, shape, v8t, ldv, v_scales, stream=None):
    """qattn_quantize_v for callers that cannot allocate: the library keeps the
    scratch in its own static device array (see include/qattn.h)."""
    _dense(V, torch.int8 if v_dtype == DT_I8 else torch.bfloat16, "V")
    _check(lib().qattn_quantize_v_noalloc(_p(V), v_dtype, _p(v_chan_scale), ctypes.byref(shape),
                                          _p(v8t), ldv, _p(v_scales), _stream(stream)),
           "qattn_quantize_v_noalloc")


def fwd(q_codes, q_scales, k_codes, k_scales, v8t, ldv, v_scales, bias, shape, params, O, lse,
        workspace, stream=None, k_carrier=None):
    if k_carrier is not None:
        _dense(k_carrier, torch.float16, "k_carrier")
    ws_bytes = _nbytes(workspace)
    _check(lib().qattn_fwd(_p(q_codes), _p(q_scales), _p(k_codes), _p(k_carrier), _p(k_scales),
                           _p(v8t), ldv, _p(v_scales), _p(bias), ctypes.byref(shape),
                           ctypes.byref(params), _p(O), _p(lse), _p(workspace), ws_bytes,
                           _stream(stream)),
           "qattn_fwd")


def decode(q_codes, q_scales, k_codes, k_scales, v_codes, v_chan_scale, v_code_amax, shape,
           params, O, lse, workspace, stream=None):
    """Decode step on an int8 KV cache (see qattn_decode in include/qattn.h)."""
    _dense(k_codes, torch.int8, "k_codes")
    _dense(v_codes, torch.int8, "v_codes")
    _check(lib().qattn_decode(_p(q_codes), _p(q_scales), _p(k_codes), _p(k_scales), _p(v_codes),
                              _p(v_chan_scale), _p(v_code_amax), ctypes.byref(shape),
                              ctypes.byref(params), _p(O), _p(lse), _p(workspace),
                              _nbytes(workspace), _stream(stream)),
           "qattn_decode")


def fwd_exact24(Q, k_codes, k_chan_scale, v_codes, v_chan_scale, shape, params, O, lse,
                workspace, stream=None):
    """24-bit exact split attention on an int8 KV cache (see qattn_fwd_exact24)."""
    _dense(Q, torch.bfloat16, "Q")
    _dense(k_codes, torch.int8, "k_codes")
    _dense(v_codes, torch.int8, "v_codes")
    _check(lib().qattn_fwd_exact24(_p(Q), _p(k_codes), _p(k_chan_scale), _p(v_codes),
                                   _p(v_chan_scale), ctypes.byref(shape), ctypes.byref(params),
                                   _p(O), _p(lse), _p(workspace),
                                   _nbytes(workspace), _stream(stream)),
           "qattn_fwd_exact24")


def fwd_intsoftmax(q_codes, q_scale, k_codes, k_scale, v_codes, shape, params, O_codes,
                   stream=None):
    """QFlash integer-only attention on per-tensor int8 codes (see
    qattn_fwd_intsoftmax); O_codes: int8 codes of V's scale."""
    for t, nm in ((q_codes, "q_codes"), (k_codes, "k_codes"), (v_codes, "v_codes"),
                  (O_codes, "O_codes")):
        _dense(t, torch.int8, nm)
    _check(lib().qattn_fwd_intsoftmax(_p(q_codes), _p(q_scale), _p(k_codes), _p(k_scale),
                                      _p(v_codes), ctypes.byref(shape), ctypes.byref(params),
                                      _p(O_codes), _stream(stream)),
           "qattn_fwd_intsoftmax")


def kv_append(K_new, V_new, pos, k_chan_scale, v_chan_scale, k_mean, v_code_amax, k_codes,
              v_codes, stream=None):
    """Append tokens to an int8 KV cache with a running-mean header (see
    qattn_kv_append in include/qattn.h).  K_new, V_new: bf16 [B, Hkv, T, d];
    k_codes, v_codes: int8 [B, Hkv, capacity, d]; scales and header fp32 [B, Hkv, d]."""
    _dense(K_new, torch.bfloat16, "K_new")
    _dense(V_new, torch.bfloat16, "V_new")
    _dense(k_codes, torch.int8, "k_codes")
    _dense(v_codes, torch.int8, "v_codes")
    for t, nm in ((k_chan_scale, "k_chan_scale"), (v_chan_scale, "v_chan_scale"),
                  (k_mean, "k_mean"), (v_code_amax, "v_code_amax")):
        _dense(t, torch.float32, nm)
    B, H, T, d = K_new.shape
    _check(lib().qattn_kv_append(_p(K_new), _p(V_new), B, H, T, d, int(pos), k_codes.shape[2],
                                 _p(k_chan_scale), _p(v_chan_scale), _p(k_mean), _p(v_code_amax),
                                 _p(k_codes), _p(v_codes), _stream(stream)),
           "qattn_kv_append")


def kv_header_init(v_codes, Nk, v_code_amax, stream=None):
    """The cache header's per-channel max |V code| over rows 0..Nk-1 (see
    qattn_kv_header_init in include/qattn.h).  v_codes: int8 [B, Hkv,
    capacity, d]; v_code_amax: fp32 [B, Hkv, d] (written)."""
    _dense(v_codes, torch.int8, "v_codes")
    _dense(v_code_amax, torch.float32, "v_code_amax")
    B, H, cap, d = v_codes.shape
    _check(lib().qattn_kv_header_init(_p(v_codes), B, H, int(Nk), d, cap, _p(v_code_amax),
                                      _stream(stream)),
           "qattn_kv_header_init")


def debug_qk_scores(q_codes, k_codes, shape, S, workspace, stream=None):
    _dense(q_codes, torch.int8, "q_codes")
    _dense(k_codes, torch.int8, "k_codes")
    _dense(S, torch.int32, "S")
    _check(lib().qattn_debug_qk_scores(_p(q_codes), _p(k_codes), ctypes.byref(shape), _p(S),
                                       _p(workspace), _nbytes(workspace),
                                       _stream(stream)),
           "qattn_debug_qk_scores")


def fwd_kernel_choice(shape: Shape, params: Params) -> int:
    """The kernel qattn_fwd runs (FWD_TC or FWD_SHORT), or -1 if it would reject the call."""
    return lib().qattn_fwd_kernel_choice(ctypes.byref(shape), ctypes.byref(params))


def prepare_launches(shape: Shape, params: Params) -> int:
    """Kernels qattn_prepare launches (1 or 2), or -1 if it would reject the call."""
    return lib().qattn_prepare_launches(ctypes.byref(shape), ctypes.byref(params))


def debug_wait_timeout(result, stream=None):
    """Runs the kernels' bounded wait on a barrier nothing completes; result is
    a device int32[2] that receives {wait succeeded, abort flag}."""
    _dense(result, torch.int32, "result")
    if result.numel() < 2:
        raise ValueError("result: needs 2 int32 elements")
    _check(lib().qattn_debug_wait_timeout(_p(result), _stream(stream)), "qattn_debug_wait_timeout")


def get_error(stream=None) -> int:
    return lib().qattn_get_error(_stream(stream))
