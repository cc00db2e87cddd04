"""Python binding of libqswiglu.so (the C ABI in include/qswiglu.h).

Argument marshalling only: tensors are checked for device, dtype and
contiguity, and their data pointers, sizes and the current CUDA stream are
passed to the C entry points, which enqueue the CUDA kernels.  There is no
fallback: if the library is missing or a call fails, these functions raise.

Tensor conventions (torch, all on one CUDA device, contiguous):
  x            bfloat16 or float16 [M, H]   (leading dims are flattened into M)
  w            int32 or uint32 [rows, H*bits/32]  packed codes, little-endian
  scales/biases x's dtype [rows, H/gs]
  result       x's dtype [M, rows]
The activation dtype (bf16 or f16) is taken from x; the calls go to the
library's *_ex entry points with that dtype.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libqswiglu.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "lib", "libqswiglu_debug.so")   # built with QSW_DEBUG_BOUNDS

MATCH, F32, DEBUG_GATE, DEBUG_UP = 0, 1, 2, 3
VARIANTS = {"match": MATCH, "f32": F32, "debug_gate": DEBUG_GATE, "debug_up": DEBUG_UP}
CNT_FUSED_TC, CNT_FUSED_GEMV, CNT_QMM_TC, CNT_QMM_GEMV, CNT_SILU_MUL, CNT_GEMV_STREAM = range(6)
NUM_COUNTERS = 6
STATUS = {0: "QSW_OK", 1: "QSW_ERR_INVALID_ARG", 2: "QSW_ERR_UNSUPPORTED", 3: "QSW_ERR_CUDA",
          4: "QSW_ERR_TIMEOUT", 5: "QSW_ERR_BOUNDS"}
STREAM_K_OFF, STREAM_K_AUTO, STREAM_K_ALWAYS = 0, 1, 2
ACT_BF16, ACT_F16 = 0, 1
SMALL_M_AUTO, SMALL_M_RING, SMALL_M_STREAM = 0, 1, 2
EXPORTED = ("qswiglu_forward", "affine_qmm", "qswiglu_forward_ws", "affine_qmm_ws", "qswiglu_forward_noalloc",
            "qswiglu_forward_ex", "affine_qmm_ex", "qsw_silu_mul_ex", "qsw_mlp_forward_ex", "qsw_workspace_bytes",
            "qsw_set_stream_k", "qsw_get_stream_k", "qsw_silu_mul", "qsw_check_device_errors",
            "qsw_set_gemv_max_m", "qsw_get_gemv_max_m", "qsw_set_early_weight_stream",
            "qsw_get_early_weight_stream", "qsw_set_small_m_kernel", "qsw_get_small_m_kernel", "qsw_set_wait_timeout_ns", "qsw_debug_withhold_next_fill", "qsw_debug_build",
            "qsw_get_counters", "qsw_reset_counters", "qsw_status_string", "qsw_version")

_lock = threading.Lock()
_lib = None


class QswError(RuntimeError):
    def __init__(self, fn: str, code: int, message: str):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({message})")
        self.code = code


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libqswiglu.so and declare its signatures.  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built; run quantized_swiglu_mlp_gb300.build.build() "
                               "(or __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        p, i64, i32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64
        lib.qswiglu_forward.argtypes = [p, i64, i64, i64, p, p, p, i32, i32, p, p, p, i32, i32, i32, p, p]
        lib.qswiglu_forward.restype = i32
        lib.affine_qmm.argtypes = [p, i64, i64, i64, p, p, p, i32, i32, p, p]
        lib.affine_qmm.restype = i32
        sz = ctypes.c_size_t
        lib.qswiglu_forward_ws.argtypes = [p, i64, i64, i64, p, p, p, i32, i32, p, p, p, i32, i32, i32, p, p, sz, p]
        lib.qswiglu_forward_ws.restype = i32
        lib.affine_qmm_ws.argtypes = [p, i64, i64, i64, p, p, p, i32, i32, p, p, sz, p]
        lib.affine_qmm_ws.restype = i32
        lib.qsw_workspace_bytes.restype = sz
        lib.qswiglu_forward_noalloc.argtypes = [p, i64, i64, i64, p, p, p, i32, i32, p, p, p, i32, i32, i32, p, p]
        lib.qswiglu_forward_noalloc.restype = i32
        lib.qswiglu_forward_ex.argtypes = [p, i64, i64, i64, p, p, p, i32, i32, p, p, p, i32, i32, i32, i32, p,
                                           p, sz, p]
        lib.qswiglu_forward_ex.restype = i32
        lib.affine_qmm_ex.argtypes = [p, i64, i64, i64, p, p, p, i32, i32, i32, p, p, p, sz, p]
        lib.affine_qmm_ex.restype = i32
        lib.qsw_mlp_forward_ex.argtypes = [p, p, i64, i64, i64, i64, p, p, p, i32, i32, p, p, p, i32, i32,
                                           p, p, p, i32, i32, i32, i32, p, p, p, sz, p]
        lib.qsw_mlp_forward_ex.restype = i32
        lib.qsw_silu_mul_ex.argtypes = [p, p, i64, i32, i32, p, p]
        lib.qsw_silu_mul_ex.restype = i32
        lib.qsw_set_stream_k.argtypes = [i32]
        lib.qsw_get_stream_k.restype = i32
        lib.qsw_silu_mul.argtypes = [p, p, i64, i32, p, p]
        lib.qsw_silu_mul.restype = i32
        lib.qsw_check_device_errors.argtypes = [p]
        lib.qsw_check_device_errors.restype = i32
        lib.qsw_set_gemv_max_m.argtypes = [i32]
        lib.qsw_get_gemv_max_m.restype = i32
        lib.qsw_set_early_weight_stream.argtypes = [i32]
        lib.qsw_get_early_weight_stream.restype = i32
        lib.qsw_set_wait_timeout_ns.argtypes = [u64]
        lib.qsw_set_small_m_kernel.argtypes = [i32]
        lib.qsw_get_small_m_kernel.restype = i32
        lib.qsw_get_counters.argtypes = [ctypes.POINTER(u64), i32]
        lib.qsw_status_string.argtypes = [i32]
        lib.qsw_status_string.restype = ctypes.c_char_p
        lib.qsw_version.restype = i32
        _lib = lib
        return lib


def _check(fn: str, code: int) -> None:
    if code != 0:
        msg = load_library().qsw_status_string(code).decode()
        raise QswError(fn, code, msg)


def _stream_ptr(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _need(t: torch.Tensor, name: str, dtypes, device=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


_PACKED = (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,)
_BF16 = (torch.bfloat16,)
_ACT = {torch.bfloat16: ACT_BF16, torch.float16: ACT_F16}


def _operand(w, s, b, name, device, K, bits, gs, dtype=torch.bfloat16):
    _need(w, f"{name} packed weights", _PACKED, device)
    _need(s, f"{name} scales", (dtype,), device)
    _need(b, f"{name} biases", (dtype,), device)
    rows = w.shape[0]
    if w.dim() != 2 or w.shape[1] * 32 != K * bits:
        raise ValueError(f"{name} packed weights must be [rows, K*bits/32], got {tuple(w.shape)}")
    if s.shape != (rows, K // gs) or b.shape != s.shape:
        raise ValueError(f"{name} scales/biases must be [rows, K/gs] = {(rows, K // gs)}")
    return rows


_workspaces: dict = {}


def workspace_bytes(device=None) -> int:
    """Bytes of stream-K workspace the tensor-core kernel needs on `device`."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(load_library().qsw_workspace_bytes())


def workspace(device=None, stream=None) -> torch.Tensor | None:
    """The stream-K workspace used by calls on (device, stream) with workspace="auto".

    Created zero-filled (and the fill completed) on first use, then kept for
    the life of the process: one per stream, since a workspace may not be
    shared by calls that can run concurrently.  Returns None while the current
    stream is being captured into a CUDA graph and none exists yet (the call
    then runs whole tiles only); make one call before capturing.
    """
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    key = (dev.index, _stream_ptr(stream))
    ws = _workspaces.get(key)
    if ws is None:
        if torch.cuda.is_current_stream_capturing():
            return None
        with torch.cuda.device(dev):
            ws = torch.zeros(workspace_bytes(dev), dtype=torch.uint8, device=dev)
            torch.cuda.current_stream(dev).synchronize()
        _workspaces[key] = ws
    return ws


def _workspace_arg(ws, device, stream):
    if isinstance(ws, str):
        if ws != "auto":
            raise ValueError('workspace must be "auto", None or a uint8 CUDA tensor')
        ws = workspace(device, stream)
    if ws is None:
        return None, 0
    _need(ws, "workspace", (torch.uint8,), device)
    return ws.data_ptr(), ws.numel()


def qsw_set_stream_k(mode: int) -> None:
    load_library().qsw_set_stream_k(int(mode))


def qsw_get_stream_k() -> int:
    return int(load_library().qsw_get_stream_k())


def qswiglu_forward(x, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u, variant=MATCH,
                    out=None, stream=None, workspace="auto") -> torch.Tensor:
    """hidden = silu(x . Wg^T) * (x . Wu^T) on the GPU; returns bf16 [..., I].

    workspace: "auto" (the per-stream workspace of workspace()), None (whole
    tiles only) or a zero-initialised uint8 tensor of at least
    workspace_bytes() bytes owned by the caller.  x may be bfloat16 or float16;
    scales, biases and the result share its dtype.
    """
    lib = load_library()
    _need(x, "x", tuple(_ACT))
    dt = x.dtype
    H = x.shape[-1]
    x2 = x.reshape(-1, H)
    M = x2.shape[0]
    I = _operand(wg, sg, bg, "gate", x.device, H, bits_g, gs_g, dt)
    if _operand(wu, su, bu, "up", x.device, H, bits_u, gs_u, dt) != I:
        raise ValueError("gate and up must have the same number of rows")
    if out is None:
        out = torch.empty((M, I), dtype=dt, device=x.device)
    else:
        _need(out, "out", (dt,), x.device)
        if out.numel() != M * I:
            raise ValueError("out has the wrong size")
    ws_ptr, ws_bytes = _workspace_arg(workspace, x.device, stream)
    code = lib.qswiglu_forward_ex(x2.data_ptr(), M, H, I, wg.data_ptr(), sg.data_ptr(), bg.data_ptr(),
                                  int(gs_g), int(bits_g), wu.data_ptr(), su.data_ptr(), bu.data_ptr(),
                                  int(gs_u), int(bits_u), int(variant), _ACT[dt], out.data_ptr(), ws_ptr,
                                  ws_bytes, _stream_ptr(stream))
    _check("qswiglu_forward_ex", code)
    return out.view(*x.shape[:-1], I)


def qswiglu_forward_noalloc(x, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u, variant=MATCH,
                            out=None, stream=None) -> torch.Tensor:
    """qswiglu_forward (bf16) with stream-K scheduling on the library's static
    scratch array (no workspace); calls through it must not run concurrently."""
    lib = load_library()
    _need(x, "x", _BF16)
    H = x.shape[-1]
    x2 = x.reshape(-1, H)
    M = x2.shape[0]
    I = _operand(wg, sg, bg, "gate", x.device, H, bits_g, gs_g)
    if _operand(wu, su, bu, "up", x.device, H, bits_u, gs_u) != I:
        raise ValueError("gate and up must have the same number of rows")
    if out is None:
        out = torch.empty((M, I), dtype=torch.bfloat16, device=x.device)
    else:
        _need(out, "out", _BF16, x.device)
        if out.numel() != M * I:
            raise ValueError("out has the wrong size")
    code = lib.qswiglu_forward_noalloc(x2.data_ptr(), M, H, I, wg.data_ptr(), sg.data_ptr(), bg.data_ptr(),
                                       int(gs_g), int(bits_g), wu.data_ptr(), su.data_ptr(), bu.data_ptr(),
                                       int(gs_u), int(bits_u), int(variant), out.data_ptr(), _stream_ptr(stream))
    _check("qswiglu_forward_noalloc", code)
    return out.view(*x.shape[:-1], I)


def affine_qmm(x, w, s, b, gs, bits, y=None, stream=None, workspace="auto", residual=None) -> torch.Tensor:
    """y = T(x . W^T + residual) with W affine-quantised, T = x's dtype; returns [..., N].

    workspace: as for qswiglu_forward; x may be bfloat16 or float16.  residual:
    None, or an [..., N] tensor of x's dtype added before the one rounding (it
    may be y itself).
    """
    lib = load_library()
    _need(x, "x", tuple(_ACT))
    dt = x.dtype
    K = x.shape[-1]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    N = _operand(w, s, b, "w", x.device, K, bits, gs, dt)
    if y is None:
        y = torch.empty((M, N), dtype=dt, device=x.device)
    else:
        _need(y, "y", (dt,), x.device)
        if y.numel() != M * N:
            raise ValueError("y has the wrong size")
    r_ptr = None
    if residual is not None:
        _need(residual, "residual", (dt,), x.device)
        if residual.numel() != M * N:
            raise ValueError("residual has the wrong size")
        r_ptr = residual.data_ptr()
    ws_ptr, ws_bytes = _workspace_arg(workspace, x.device, stream)
    code = lib.affine_qmm_ex(x2.data_ptr(), M, K, N, w.data_ptr(), s.data_ptr(), b.data_ptr(),
                             int(gs), int(bits), _ACT[dt], r_ptr, y.data_ptr(), ws_ptr, ws_bytes,
                             _stream_ptr(stream))
    _check("affine_qmm_ex", code)
    return y.view(*x.shape[:-1], N)


def mlp_forward(x, h, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u, wd, sd, bd, gs_d, bits_d,
                variant=MATCH, out=None, hidden=None, stream=None, workspace="auto") -> torch.Tensor:
    """The whole MLP block: y = T(h + (silu(x . Wg^T) * (x . Wu^T)) . Wd^T).

    h: the residual [..., Ho] (x's dtype) or None; it may be `out`.  hidden: an
    [M, I] buffer for the intermediate (allocated when None).  Returns y [..., Ho].
    """
    lib = load_library()
    _need(x, "x", tuple(_ACT))
    dt = x.dtype
    H = x.shape[-1]
    x2 = x.reshape(-1, H)
    M = x2.shape[0]
    I = _operand(wg, sg, bg, "gate", x.device, H, bits_g, gs_g, dt)
    if _operand(wu, su, bu, "up", x.device, H, bits_u, gs_u, dt) != I:
        raise ValueError("gate and up must have the same number of rows")
    Ho = _operand(wd, sd, bd, "down", x.device, I, bits_d, gs_d, dt)
    if hidden is None:
        hidden = torch.empty((M, I), dtype=dt, device=x.device)
    else:
        _need(hidden, "hidden", (dt,), x.device)
        if hidden.numel() != M * I:
            raise ValueError("hidden has the wrong size")
    if out is None:
        out = torch.empty((M, Ho), dtype=dt, device=x.device)
    else:
        _need(out, "out", (dt,), x.device)
        if out.numel() != M * Ho:
            raise ValueError("out has the wrong size")
    h_ptr = None
    if h is not None:
        _need(h, "h", (dt,), x.device)
        if h.numel() != M * Ho:
            raise ValueError("h has the wrong size")
        h_ptr = h.data_ptr()
    ws_ptr, ws_bytes = _workspace_arg(workspace, x.device, stream)
    code = lib.qsw_mlp_forward_ex(x2.data_ptr(), h_ptr, M, H, I, Ho, wg.data_ptr(), sg.data_ptr(), bg.data_ptr(),
                                  int(gs_g), int(bits_g), wu.data_ptr(), su.data_ptr(), bu.data_ptr(), int(gs_u),
                                  int(bits_u), wd.data_ptr(), sd.data_ptr(), bd.data_ptr(), int(gs_d), int(bits_d),
                                  int(variant), _ACT[dt], hidden.data_ptr(), out.data_ptr(), ws_ptr, ws_bytes,
                                  _stream_ptr(stream))
    _check("qsw_mlp_forward_ex", code)
    return out.view(*x.shape[:-1], Ho)


def qsw_silu_mul(g, u, variant=MATCH, out=None, stream=None) -> torch.Tensor:
    """out = silu(g) * u elementwise over bf16 (or float16) tensors of equal shape."""
    lib = load_library()
    _need(g, "g", tuple(_ACT))
    _need(u, "u", (g.dtype,), g.device)
    if g.shape != u.shape:
        raise ValueError("g and u must have the same shape")
    if out is None:
        out = torch.empty_like(g)
    else:
        _need(out, "out", (g.dtype,), g.device)
        if out.numel() != g.numel():
            raise ValueError("out has the wrong size")
    _check("qsw_silu_mul_ex", lib.qsw_silu_mul_ex(g.data_ptr(), u.data_ptr(), g.numel(), int(variant),
                                                  _ACT[g.dtype], out.data_ptr(), _stream_ptr(stream)))
    return out


def unfused_swiglu(x, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u, variant=MATCH,
                   stream=None, workspace="auto") -> torch.Tensor:
    """The unfused comparison path: two affine_qmm calls, then silu*mul."""
    g = affine_qmm(x, wg, sg, bg, gs_g, bits_g, stream=stream, workspace=workspace)
    u = affine_qmm(x, wu, su, bu, gs_u, bits_u, stream=stream, workspace=workspace)
    return qsw_silu_mul(g, u, variant, out=g, stream=stream)


def qsw_check_device_errors(stream=None) -> None:
    _check("qsw_check_device_errors", load_library().qsw_check_device_errors(_stream_ptr(stream)))


def qsw_set_gemv_max_m(m: int) -> None:
    load_library().qsw_set_gemv_max_m(int(m))


def qsw_get_gemv_max_m() -> int:
    return int(load_library().qsw_get_gemv_max_m())


def qsw_set_wait_timeout_ns(ns: int) -> None:
    load_library().qsw_set_wait_timeout_ns(int(ns))


def qsw_debug_withhold_next_fill() -> None:
    """Test hook: the next small-M call leaves its first units unrequested, so
    its waits run out (see include/qswiglu.h)."""
    load_library().qsw_debug_withhold_next_fill()


def qsw_debug_build() -> bool:
    """Whether the loaded library is the debug build (QSW_DEBUG_BOUNDS)."""
    lib = load_library()
    lib.qsw_debug_build.restype = ctypes.c_int
    return bool(lib.qsw_debug_build())


def qsw_get_counters() -> list[int]:
    arr = (ctypes.c_uint64 * NUM_COUNTERS)()
    load_library().qsw_get_counters(arr, NUM_COUNTERS)
    return list(arr)


def qsw_reset_counters() -> None:
    load_library().qsw_reset_counters()


def qsw_status_string(code: int) -> str:
    return load_library().qsw_status_string(int(code)).decode()


def qsw_set_early_weight_stream(on: bool) -> None:
    load_library().qsw_set_early_weight_stream(1 if on else 0)


def qsw_get_early_weight_stream() -> bool:
    return bool(load_library().qsw_get_early_weight_stream())


def qsw_set_small_m_kernel(kernel: int) -> None:
    """SMALL_M_AUTO (default), SMALL_M_RING or SMALL_M_STREAM (include/qswiglu.h)."""
    load_library().qsw_set_small_m_kernel(int(kernel))


def qsw_get_small_m_kernel() -> int:
    return int(load_library().qsw_get_small_m_kernel())


def qsw_version() -> int:
    return int(load_library().qsw_version())
