"""The C-ABI library builds, loads without a GPU, exports every function
include/qattn.h declares, and rejects bad arguments on the host (no kernel
launch, no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from quantized_attention_gb300 import binding, build
    if not os.path.exists(binding.library_path()):
        build.build()
    return binding.lib()


def _declared():
    """Every function declared by the headers under include/."""
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(qattn_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_every_declared_function_is_exported(L):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    from quantized_attention_gb300 import binding
    assert sorted(binding.EXPORTED) == names


def test_checked_build_exports_the_same_and_says_so(L):
    """The bounds-checked build (QATTN_CHECK=1) is the same ABI; only
    qattn_checked() tells the two apart."""
    from quantized_attention_gb300 import binding, build
    if not os.path.exists(build.CHECK_LIB):
        build.build(checked=True)
    C = ctypes.CDLL(build.CHECK_LIB)
    for n in _declared():
        assert hasattr(C, n), n
    assert C.qattn_checked() == 1
    assert L.qattn_checked() == (1 if os.path.abspath(binding.library_path()) == build.CHECK_LIB else 0)
    C.qattn_status_string.restype = ctypes.c_char_p
    assert b"checked build" in C.qattn_status_string(binding.ERR_BOUNDS)


def test_library_override_loads_the_checked_build(L):
    """QATTN_LIBRARY points the binding at another build of the library."""
    import subprocess
    import sys
    from quantized_attention_gb300 import build
    if not os.path.exists(build.CHECK_LIB):
        build.build(checked=True)
    code = ("from quantized_attention_gb300 import binding as qb; import os; "
            "assert os.path.samefile(qb.library_path(), os.environ['QATTN_LIBRARY']); "
            "assert qb.checked(); print('ok')")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       env=dict(os.environ, QATTN_LIBRARY=build.CHECK_LIB), timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr


def test_host_only_queries(L):
    from quantized_attention_gb300 import binding as qb
    assert qb.version() == 100
    assert qb.status_string(0) == "ok" and "workspace" in qb.status_string(5)
    assert qb.v_ld(49) == 64 and qb.v_ld(128) == 128 and qb.v_ld(1) == 16
    s = qb.make_shape(1, 32, 8, 8192, 8192, 128)
    p = qb.make_params(causal=True)
    # at least the fp16 carriers of the K codes (Q codes are widened in-kernel)
    assert qb.workspace_size(s, p) >= 2 * 8 * 8192 * 128
    assert qb.workspace_size(qb.make_shape(0, 32, 8, 8192, 8192, 128), p) == 0


def test_invalid_arguments_rejected_on_host(L):
    from quantized_attention_gb300 import binding as qb
    vp = ctypes.c_void_p
    s = qb.make_shape(1, 4, 2, 256, 256, 64)
    p = qb.make_params()
    fake = vp(1 << 20)  # aligned, never dereferenced: validation fails first
    # the failure-path check wants an 8-byte aligned result
    assert L.qattn_debug_wait_timeout(None, None) == 1
    assert L.qattn_debug_wait_timeout(vp((1 << 20) + 4), None) == 1
    # null outputs
    assert L.qattn_fwd(None, fake, fake, None, fake, fake, 256, fake, None, ctypes.byref(s),
                       ctypes.byref(p), fake, None, fake, 1 << 30, None) == 1
    # misaligned pointers
    assert L.qattn_fwd(vp((1 << 20) + 4), fake, fake, None, fake, fake, 256, fake, None,
                       ctypes.byref(s), ctypes.byref(p), fake, None, fake, 1 << 30, None) == 1
    assert L.qattn_fwd(fake, fake, fake, vp((1 << 20) + 2), fake, fake, 256, fake, None,
                       ctypes.byref(s), ctypes.byref(p), fake, None, fake, 1 << 30, None) == 1
    # the persistent kernel without a K carrier needs a workspace
    p_tc = qb.make_params(fwd_kernel=qb.FWD_TC)
    assert L.qattn_fwd(fake, fake, fake, None, fake, fake, 256, fake, None, ctypes.byref(s),
                       ctypes.byref(p_tc), fake, None, None, 0, None) == 5
    # the short-sequence kernel on a shape it does not cover, and an unknown kernel choice
    s_c = qb.make_shape(1, 4, 2, 256, 256, 128)
    p_short = qb.make_params(fwd_kernel=qb.FWD_SHORT)
    assert L.qattn_fwd(fake, fake, fake, None, fake, fake, 256, fake, None, ctypes.byref(s_c),
                       ctypes.byref(p_short), fake, None, None, 0, None) == 2
    p_causal = qb.make_params(causal=True, fwd_kernel=qb.FWD_SHORT)
    assert L.qattn_fwd(fake, fake, fake, None, fake, fake, 256, fake, None, ctypes.byref(s),
                       ctypes.byref(p_causal), fake, None, None, 0, None) == 2
    p_bad = qb.make_params(fwd_kernel=7)
    assert L.qattn_fwd(fake, fake, fake, None, fake, fake, 256, fake, None, ctypes.byref(s),
                       ctypes.byref(p_bad), fake, None, None, 0, None) == 1
    # unsupported head dim
    s96 = qb.make_shape(1, 4, 2, 256, 256, 96)
    assert L.qattn_smooth_k(fake, None, ctypes.byref(s96), fake, fake, 1 << 30, None) == 2
    # Hq not a multiple of Hkv
    s_bad = qb.make_shape(1, 5, 2, 256, 256, 64)
    assert L.qattn_smooth_k(fake, None, ctypes.byref(s_bad), fake, fake, 1 << 30, None) == 1
    # ldv too small
    assert L.qattn_quantize_v(fake, None, 0, None, ctypes.byref(s), fake, 128, fake, fake, 1 << 30,
                              None) == 1
    # int8 P ablation with a bias: unsupported
    p_i8 = qb.make_params(pv_mode=qb.PV_INT8)
    assert L.qattn_fwd(fake, fake, fake, None, fake, fake, 256, fake, fake, ctypes.byref(s),
                       ctypes.byref(p_i8), fake, None, fake, 1 << 30, None) == 2
    # bad P mode
    p_pv = qb.make_params(pv_mode=3)
    assert L.qattn_fwd(fake, fake, fake, None, fake, fake, 256, fake, None, ctypes.byref(s),
                       ctypes.byref(p_pv), fake, None, fake, 1 << 30, None) == 1
    # bad enum
    p_bad = qb.make_params(q_gran=7)
    assert L.qattn_quantize_qk(fake, None, fake, None, 0, None, None, ctypes.byref(s),
                               ctypes.byref(p_bad), fake, fake, fake, fake, None, fake, 1 << 30,
                               None) == 1
    # misaligned K carrier
    assert L.qattn_quantize_qk(fake, None, fake, None, 0, None, None, ctypes.byref(s),
                               ctypes.byref(p), fake, fake, fake, fake, vp((1 << 20) + 8), fake,
                               1 << 30, None) == 1
    # workspace too small
    assert L.qattn_smooth_k(fake, None, ctypes.byref(s), fake, fake, 16, None) == 5
    # input strides: the last must be 1, the others multiples of 16 bytes;
    # int8 cache K codes are dense only
    i64x4 = ctypes.c_int64 * 4
    for bad in (i64x4(256 * 64, 256 * 64, 64, 2), i64x4(256 * 64, 256 * 64, 60, 1),
                i64x4(-64, 256 * 64, 64, 1)):
        assert L.qattn_smooth_k(fake, bad, ctypes.byref(s), fake, fake, 1 << 30, None) == 1
        assert L.qattn_quantize_v(fake, bad, 0, None, ctypes.byref(s), fake, 256, fake, fake,
                                  1 << 30, None) == 1
    packed = i64x4(256 * 3 * 2 * 64, 64, 3 * 2 * 64, 1)  # [B][N][3][H][d] viewed as [B][H][N][d]
    assert L.qattn_quantize_qk(fake, packed, fake, packed, 2, None, fake, ctypes.byref(s),
                               ctypes.byref(p), fake, fake, None, fake, None, fake, 1 << 30,
                               None) == 2
    # empty problem: ok, nothing launched
    s0 = qb.make_shape(0, 4, 2, 256, 256, 64)
    assert L.qattn_fwd(None, None, None, None, None, None, 0, None, None, ctypes.byref(s0),
                       ctypes.byref(p), None, None, None, 0, None) == 0
    for empty in (qb.make_shape(1, 0, 2, 256, 256, 64), qb.make_shape(1, 4, 2, 0, 256, 64)):
        assert L.qattn_fwd(None, None, None, None, None, None, 0, None, None, ctypes.byref(empty),
                           ctypes.byref(p), None, None, None, 0, None) == 0
    # no keys: the outputs are still required; the short kernel does not take it
    s_nk0 = qb.make_shape(1, 4, 2, 32, 0, 64)
    assert L.qattn_fwd(fake, fake, None, None, None, None, 16, None, None, ctypes.byref(s_nk0),
                       ctypes.byref(p), None, None, None, 0, None) == 1
    assert L.qattn_fwd(fake, fake, None, None, None, None, 16, None, None, ctypes.byref(s_nk0),
                       ctypes.byref(p_short), fake, None, None, 0, None) == 2
    assert qb.fwd_kernel_choice(s_nk0, p) == qb.FWD_TC


def test_decode_and_append_arguments_rejected_on_host(L):
    from quantized_attention_gb300 import binding as qb
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    # qattn_kv_append: pos + T beyond the capacity, negative pos, d out of range,
    # misaligned bf16 / fp32 pointers, null codes; T = 0 is a no-op (no launch)
    assert L.qattn_kv_append(fake, fake, 1, 2, 3, 64, 6, 8, fake, fake, fake, fake, fake, fake, None) == 1
    assert L.qattn_kv_append(fake, fake, 1, 2, 3, 64, -1, 8, fake, fake, fake, fake, fake, fake, None) == 1
    assert L.qattn_kv_append(fake, fake, 1, 2, 3, 2048, 0, 8, fake, fake, fake, fake, fake, fake, None) == 1
    assert L.qattn_kv_append(vp((1 << 20) + 1), fake, 1, 2, 3, 64, 0, 8, fake, fake, fake, fake,
                             fake, fake, None) == 1
    assert L.qattn_kv_append(fake, fake, 1, 2, 3, 64, 0, 8, fake, fake, vp((1 << 20) + 2), fake,
                             fake, fake, None) == 1
    assert L.qattn_kv_append(fake, fake, 1, 2, 3, 64, 0, 8, fake, fake, fake, fake, None, fake, None) == 1
    assert L.qattn_kv_append(fake, fake, 1, 2, 0, 64, 8, 8, fake, fake, fake, fake, fake, fake, None) == 0
    # qattn_decode: a capacity below the rows in use, a negative capacity
    s = qb.make_shape(1, 8, 2, 1, 1000, 128)
    for cap, st in ((999, 1), (-5, 1)):
        p = qb.make_params(causal=True, kv_capacity=cap)
        assert L.qattn_decode(fake, fake, fake, fake, fake, fake, fake, ctypes.byref(s),
                              ctypes.byref(p), fake, None, fake, 1 << 30, None) == st
    # an empty cache, the int8-P ablation, more than 16 rows per KV head, d = 32
    p = qb.make_params(causal=True)
    for shp, pp in ((qb.make_shape(1, 8, 2, 1, 0, 128), p),
                    (s, qb.make_params(causal=True, pv_mode=qb.PV_INT8)),
                    (qb.make_shape(1, 8, 2, 5, 1000, 128), p),
                    (qb.make_shape(1, 8, 2, 1, 1000, 32), p)):
        assert L.qattn_decode(fake, fake, fake, fake, fake, fake, fake, ctypes.byref(shp),
                              ctypes.byref(pp), fake, None, fake, 1 << 30, None) == 2


def test_kernel_choices_follow_the_documented_rules(L):
    """qattn_fwd_kernel_choice / qattn_prepare_launches (host only) against the
    rules include/qattn.h states for qattn_fwd_kernel and qattn_prepare."""
    from quantized_attention_gb300 import binding as qb
    shapes = [(49, 49), (64, 64), (65, 64), (64, 65), (1, 1), (197, 197), (128, 128),
              (129, 100), (256, 256), (300, 300)]
    for d in (32, 64, 128):
        for nq, nk in shapes:
            s = qb.make_shape(2, 4, 2, nq, nk, d)
            for causal in (False, True):
                for pv in (qb.PV_E4M3, qb.PV_INT8):
                    short_ok = d in (32, 64) and not causal and pv == qb.PV_E4M3 and 1 <= nk <= 256
                    window = short_ok and nq <= 64 and nk <= 64
                    for kern in (qb.FWD_AUTO, qb.FWD_TC, qb.FWD_SHORT):
                        p = qb.make_params(causal=causal, pv_mode=pv, fwd_kernel=kern)
                        if kern == qb.FWD_SHORT:
                            want = qb.FWD_SHORT if short_ok else -1
                        elif kern == qb.FWD_AUTO and window:
                            want = qb.FWD_SHORT
                        else:
                            want = qb.FWD_TC
                        assert qb.fwd_kernel_choice(s, p) == want, (d, nq, nk, causal, pv, kern)
            p = qb.make_params()
            assert qb.prepare_launches(s, p) == (1 if d <= 64 and nq <= 128 and nk <= 128 else 2)
            assert qb.prepare_launches(s, qb.make_params(q_gran=qb.GRAN_TENSOR)) == -1
            tens = qb.make_params(q_gran=qb.GRAN_TENSOR, k_gran=qb.GRAN_TENSOR)
            assert qb.prepare_launches(s, tens) == (2 if d <= 64 and nk <= 256 else -1)
            assert qb.prepare_launches(s, qb.make_params(q_gran=qb.GRAN_HEAD, k_gran=qb.GRAN_HEAD)) == -1
    assert qb.fwd_kernel_choice(qb.make_shape(1, 4, 2, 64, 64, 96), qb.make_params()) == -1
    assert qb.prepare_launches(qb.make_shape(1, 4, 2, 64, 0, 64), qb.make_params()) == -1


def test_extra_modes_arguments_rejected_on_host(L):
    """qattn_fwd_intsoftmax and qattn_fwd_exact24 reject what their header
    limits exclude before any device work."""
    from quantized_attention_gb300 import binding as qb
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    p = qb.make_params()

    def ism(shape, params=p, O=fake, k_scale=fake):
        return L.qattn_fwd_intsoftmax(fake, fake, fake, k_scale, fake, ctypes.byref(shape),
                                      ctypes.byref(params), O, None)

    ok = qb.make_shape(1, 3, 3, 197, 197, 64)
    assert ism(ok, params=qb.make_params(causal=True)) == 2            # no mask
    assert ism(qb.make_shape(1, 3, 3, 197, 0, 64)) == 2                # no keys
    assert ism(qb.make_shape(1, 3, 3, 197, (1 << 17) + 1, 64)) == 2    # int32 O bound
    assert ism(qb.make_shape(1, 3, 3, 197, 197, 96)) == 2              # head dim
    assert ism(ok, O=vp((1 << 20) + 8)) == 1                           # O alignment
    assert ism(ok, k_scale=None) == 1
    assert ism(qb.make_shape(0, 3, 3, 197, 197, 64), O=None) == 0      # empty: nothing to do

    def e24(shape, params=p, Q=fake, ws=fake, ws_bytes=1 << 30):
        return L.qattn_fwd_exact24(Q, fake, fake, fake, fake, ctypes.byref(shape),
                                   ctypes.byref(params), fake, None, ws, ws_bytes, None)

    cache = qb.make_shape(1, 4, 2, 64, 1000, 128)
    assert e24(qb.make_shape(1, 4, 2, 64, 1000, 32)) == 2              # d in {64, 128}
    assert e24(cache, params=qb.make_params(kv_capacity=999)) == 1     # capacity below Nk
    assert e24(cache, Q=vp((1 << 20) + 2)) == 1                        # Q alignment
    assert e24(cache, ws=None, ws_bytes=0) == 5                        # workspace
    assert e24(cache, ws_bytes=16) == 5


_LOG_PROBE = """
from quantized_attention_gb300 import binding as qb
s = qb.make_shape(2, 4, 2, 300, 300, 128)
print(qb.fwd_kernel_choice(s, qb.make_params(causal=True)))
print(qb.fwd_kernel_choice(qb.make_shape(1, 4, 2, 49, 49, 64), qb.make_params()))
"""


@pytest.mark.parametrize("value", ["1", "", "0", None])
def test_launch_log_follows_the_environment(L, value):
    """QATTN_LOG set: one "[qattn]" line on stderr per call naming the entry
    point, the shape and the kernel; unset, "" or "0": nothing on stderr."""
    import subprocess
    import sys
    env = dict(os.environ)
    env.pop("QATTN_LOG", None)
    if value is not None:
        env["QATTN_LOG"] = value
    r = subprocess.run([sys.executable, "-c", _LOG_PROBE], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.split() == ["1", "2"]
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("[qattn]")]
    if value == "1":
        assert len(lines) == 2, r.stderr
        assert "qattn_fwd_kernel_choice B=2 Hq=4 Hkv=2 Nq=300 Nk=300 d=128 causal=1" in lines[0]
        assert lines[0].endswith("persistent tcgen05")
        assert lines[1].endswith("warp-level")
    else:
        assert lines == [], r.stderr
