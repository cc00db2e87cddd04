"""The C ABI on the CPU: the library loads, exports every symbol the header
declares, and rejects bad arguments on the host before any CUDA call.
No compute is launched here (no GPU in this environment)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from quantized_swiglu_mlp_gb300 import build as qbuild
from quantized_swiglu_mlp_gb300 import ops

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "qswiglu.h")
OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return ops.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"QSW_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(names) == set(ops.EXPORTED), names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


FAKE = 0x10000          # aligned, never dereferenced: validation fails or M == 0 first


def fwd(lib, M=4, H=256, I=64, gs_g=64, bits_g=4, gs_u=64, bits_u=4, variant=0,
        x=FAKE, wg=FAKE, sg=FAKE, bg=FAKE, wu=FAKE, su=FAKE, bu=FAKE, out=FAKE):
    return lib.qswiglu_forward(x, M, H, I, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u,
                               variant, out, None)


def test_m_zero_is_a_noop(lib):
    assert fwd(lib, M=0) == OK
    assert lib.affine_qmm(FAKE, 0, 256, 64, FAKE, FAKE, FAKE, 64, 4, FAKE, None) == OK
    assert lib.qsw_silu_mul(FAKE, FAKE, 0, 0, FAKE, None) == OK


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), INVALID),
    (dict(H=0), INVALID),
    (dict(I=0), INVALID),
    (dict(H=48), UNSUPPORTED),                 # H % 32 != 0
    (dict(gs_g=48), UNSUPPORTED),              # group size not a multiple of 32
    (dict(gs_u=96), UNSUPPORTED),              # does not divide H=256
    (dict(bits_g=3), UNSUPPORTED),
    (dict(bits_u=16), UNSUPPORTED),
    (dict(bits_g=2, H=96, gs_g=32, gs_u=32), UNSUPPORTED),   # 2-bit needs H % 64 == 0
    (dict(variant=7), INVALID),
    (dict(x=0), INVALID),
    (dict(wg=0), INVALID),
    (dict(su=0), INVALID),
    (dict(out=0), INVALID),
    (dict(x=FAKE + 8), UNSUPPORTED),           # 16-byte alignment
    (dict(wu=FAKE + 4), UNSUPPORTED),
    (dict(out=FAKE + 2), UNSUPPORTED),
    (dict(sg=FAKE + 1), UNSUPPORTED),
])
def test_forward_rejects(lib, kw, code):
    assert fwd(lib, **kw) == code


def test_affine_qmm_rejects(lib):
    assert lib.affine_qmm(FAKE, 4, 100, 64, FAKE, FAKE, FAKE, 32, 4, FAKE, None) == UNSUPPORTED
    assert lib.affine_qmm(FAKE, 4, 256, -1, FAKE, FAKE, FAKE, 64, 4, FAKE, None) == INVALID
    assert lib.affine_qmm(0, 4, 256, 64, FAKE, FAKE, FAKE, 64, 4, FAKE, None) == INVALID
    assert lib.affine_qmm(FAKE, 4, 256, 64, FAKE, FAKE, FAKE, 64, 5, FAKE, None) == UNSUPPORTED


def test_silu_mul_rejects(lib):
    assert lib.qsw_silu_mul(FAKE, FAKE, -1, 0, FAKE, None) == INVALID
    assert lib.qsw_silu_mul(FAKE, FAKE, 8, 2, FAKE, None) == INVALID     # debug variants only fuse
    assert lib.qsw_silu_mul(0, FAKE, 8, 0, FAKE, None) == INVALID
    assert lib.qsw_silu_mul(FAKE + 2, FAKE, 8, 0, FAKE, None) == UNSUPPORTED


def test_gemv_limit_is_clamped(lib):
    saved = ops.qsw_get_gemv_max_m()
    try:
        ops.qsw_set_gemv_max_m(1000)
        assert ops.qsw_get_gemv_max_m() == 32
        ops.qsw_set_gemv_max_m(-5)
        assert ops.qsw_get_gemv_max_m() == 0
        ops.qsw_set_gemv_max_m(8)
        assert ops.qsw_get_gemv_max_m() == 8
    finally:
        ops.qsw_set_gemv_max_m(saved)


def test_counters_and_strings(lib):
    ops.qsw_reset_counters()
    assert ops.qsw_get_counters() == [0] * ops.NUM_COUNTERS
    assert fwd(lib, M=0) == OK                       # a no-op launches nothing
    assert ops.qsw_get_counters() == [0] * ops.NUM_COUNTERS
    assert ops.qsw_status_string(0) == "ok"
    assert "unsupported" in ops.qsw_status_string(2)
    assert ops.qsw_status_string(99) == "unknown status"
    assert ops.qsw_version() >= 100


def test_python_binding_rejects_host_tensors(lib):
    import torch
    x = torch.zeros(2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ops.qswiglu_forward(x, x, x, x, 64, 4, x, x, x, 64, 4)


def test_early_weight_stream_switch():
    """The early weight stream is off by default and toggles process-wide."""
    from quantized_swiglu_mlp_gb300 import ops
    ops.load_library()
    saved = ops.qsw_get_early_weight_stream()
    try:
        ops.qsw_set_early_weight_stream(True)
        assert ops.qsw_get_early_weight_stream() is True
        ops.qsw_set_early_weight_stream(False)
        assert ops.qsw_get_early_weight_stream() is False
    finally:
        ops.qsw_set_early_weight_stream(saved)



def fwd_ws(lib, ws, ws_bytes, M=4):
    return lib.qswiglu_forward_ws(FAKE, M, 256, 64, FAKE, FAKE, FAKE, 64, 4, FAKE, FAKE, FAKE, 64, 4,
                                  0, FAKE, ws, ws_bytes, None)


def test_workspace_entry_points_validate_on_the_host(lib):
    """The *_ws entry points check the workspace before anything is launched:
    a misaligned one is unsupported, a null one means whole tiles only, and
    argument errors are reported as for the plain entry points."""
    assert fwd_ws(lib, FAKE + 64, 1 << 30) == UNSUPPORTED          # 256-byte alignment
    assert fwd_ws(lib, None, 0, M=0) == OK
    assert fwd_ws(lib, FAKE, 1 << 30, M=0) == OK
    assert fwd_ws(lib, FAKE, 1 << 30, M=-1) == INVALID
    assert lib.affine_qmm_ws(FAKE, 4, 256, 64, FAKE, FAKE, FAKE, 64, 4, FAKE, FAKE + 16, 1 << 30,
                             None) == UNSUPPORTED
    assert lib.affine_qmm_ws(FAKE, 0, 256, 64, FAKE, FAKE, FAKE, 64, 4, FAKE, FAKE, 1 << 30, None) == OK
    # no device is current here: the size query answers 0
    assert lib.qsw_workspace_bytes() == 0


def test_stream_k_mode_switch(lib):
    """Stream-K scheduling defaults to auto; out-of-range modes are ignored."""
    saved = ops.qsw_get_stream_k()
    try:
        assert saved == ops.STREAM_K_AUTO
        for mode in (ops.STREAM_K_OFF, ops.STREAM_K_ALWAYS, ops.STREAM_K_AUTO):
            ops.qsw_set_stream_k(mode)
            assert ops.qsw_get_stream_k() == mode
        ops.qsw_set_stream_k(7)
        assert ops.qsw_get_stream_k() == ops.STREAM_K_AUTO
    finally:
        ops.qsw_set_stream_k(saved)


def test_noalloc_entry_point_validates_on_the_host(lib):
    """The static-scratch entry point checks its arguments before anything
    (including its first-use set-up) touches the device."""
    call = lambda M, variant, x=FAKE: lib.qswiglu_forward_noalloc(x, M, 256, 64, FAKE, FAKE, FAKE, 64, 4, FAKE,
                                                                    FAKE, FAKE, 64, 4, variant, FAKE, None)
    assert call(0, 0) == OK
    assert call(-1, 0) == INVALID
    assert call(4, 7) == INVALID
    assert call(4, 0, x=FAKE + 8) == UNSUPPORTED


def test_mlp_entry_point_validates_on_the_host(lib):
    """The whole-MLP entry point checks both stages' arguments first."""
    def mlp(M=4, variant=0, act=0, h=None, hidden=FAKE, I=64, gs_d=32, bits_d=4):
        return lib.qsw_mlp_forward_ex(FAKE, h, M, 256, I, 96, FAKE, FAKE, FAKE, 64, 4, FAKE, FAKE, FAKE, 64, 4,
                                      FAKE, FAKE, FAKE, gs_d, bits_d, variant, act, hidden, FAKE, None, 0, None)
    assert mlp(M=0) == OK
    assert mlp(variant=2) == INVALID            # debug variants have no whole-block meaning
    assert mlp(act=3) == INVALID
    assert mlp(hidden=None) == INVALID
    assert mlp(h=FAKE + 2) == UNSUPPORTED        # residual alignment
    assert mlp(gs_d=48) == UNSUPPORTED           # down group size
    assert mlp(I=48) == UNSUPPORTED              # I is the down projection's K
    assert mlp(bits_d=3) == UNSUPPORTED


def test_debug_build_is_built_and_exports_the_same_abi(lib):
    """The debug build (QSW_DEBUG_BOUNDS) is built beside the regular one,
    exports every declared symbol and says which build it is."""
    dbg = ctypes.CDLL(qbuild.DEBUG_LIB_PATH)
    for name in declared_functions():
        assert hasattr(dbg, name), name
    dbg.qsw_debug_build.restype = ctypes.c_int
    lib.qsw_debug_build.restype = ctypes.c_int
    assert dbg.qsw_debug_build() == 1 and lib.qsw_debug_build() == 0
    dbg.qsw_status_string.restype = ctypes.c_char_p
    assert b"debug" in dbg.qsw_status_string(5)
