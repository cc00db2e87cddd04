"""CPU oracle for the fused weight-quantized SwiGLU expansion.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product library
(``quantized_swiglu_mlp_gb300``) never imports this package.

The arithmetic lives in ``qsw_oracle.c`` (plain C, f64, explicit bf16
round-to-nearest-even at each point the method rounds); this module only builds
it with gcc and marshals numpy arrays through ctypes.  Every array is host
memory: bf16 values travel as uint16 bit patterns.

Every function that takes activations has a ``dtype`` argument: "bf16" (the
default) or "f16", the two activation dtypes the pages' kernels accept; x,
scales, biases and results are then that dtype's bit patterns.

Parity status of each function (what pins it is in tests/test_oracle_pins.py):
  bf16_round    pinned (library cast on binary32 inputs, exact rational rounding)
  f16_round     pinned (numpy's IEEE binary16 conversion, exhaustive decode of
                all 65536 patterns, hand-worked boundary values)
  unpack        pinned (hand-packed words, round trip)
  dequant       pinned (hand-worked rows, exact rational brute force)
  qswiglu       pinned (hand-worked 2x8 example, x=0, integer special case,
                brute force on tiny shapes, K-permutation invariance)
  qmm           pinned (integer special case, brute force, residual brute force)
  mlp           pinned (x=0 gives y=h, brute force of the whole block, composition)
  silu_mul      pinned (hand-worked values, silu(0)=0, MATCH == fused MATCH)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsw_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()

MATCH, F32, DEBUG_GATE, DEBUG_UP = 0, 1, 2, 3
DTYPES = {"bf16": 0, "f16": 1}


def _dt(dtype) -> int:
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {sorted(DTYPES)}, got {dtype!r}")
    return DTYPES[dtype]


def build(force: bool = False) -> str:
    """Compile qsw_oracle.c with gcc (OpenMP, no fp contraction) into liboracle.so."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _declare(lib):
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.orc_f64_to_bf16.argtypes = [ctypes.c_double]
    lib.orc_f64_to_bf16.restype = ctypes.c_uint16
    lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_f64.restype = ctypes.c_double
    lib.orc_f64_to_f16.argtypes = [ctypes.c_double]
    lib.orc_f64_to_f16.restype = ctypes.c_uint16
    lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.orc_f16_to_f64.restype = ctypes.c_double
    lib.orc_unpack.argtypes = [p, i64, i32, p]
    lib.orc_dequant.argtypes = [p, p, p, i64, i64, i32, i32, i32, p]
    q_args = [p, i64, i64, i64, p, p, p, i32, i32, p, p, p, i32, i32, i32, i32]
    lib.orc_qswiglu.argtypes = q_args + [p]
    lib.orc_qswiglu.restype = i32
    lib.orc_qswiglu_rows.argtypes = q_args + [p, i64, p, p, p]
    lib.orc_qswiglu_rows.restype = i32
    lib.orc_qswiglu_pairs.argtypes = q_args + [p, i64, p]
    lib.orc_qswiglu_pairs.restype = i32
    lib.orc_qmm.argtypes = [p, i64, i64, i64, p, p, p, i32, i32, i32, p, p]
    lib.orc_qmm.restype = i32
    lib.orc_mlp.argtypes = [p, p, i64, i64, i64, i64, p, p, p, i32, i32, p, p, p, i32, i32,
                            p, p, p, i32, i32, i32, i32, p, p]
    lib.orc_mlp.restype = i32
    lib.orc_silu_mul.argtypes = [p, p, i64, i32, i32, p]
    lib.orc_num_threads.restype = i32
    lib.orc_set_num_threads.argtypes = [i32]
    return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def bf16_bits_to_f64(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (a bit shift into binary32)."""
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class OracleLib:
    """The oracle's entry points bound to one compiled copy of qsw_oracle.c."""

    def __init__(self, path: str):
        self.path = path
        self.lib = _declare(ctypes.CDLL(path))

    def num_threads(self) -> int:
        return self.lib.orc_num_threads()

    def set_num_threads(self, n: int) -> None:
        self.lib.orc_set_num_threads(int(n))

    def f64_to_bf16(self, v: float) -> int:
        """One round-to-nearest-even of an exact double to a bf16 bit pattern."""
        return int(self.lib.orc_f64_to_bf16(float(v)))

    def bf16_to_f64(self, h: int) -> float:
        return float(self.lib.orc_bf16_to_f64(int(h) & 0xFFFF))

    def bf16_round_array(self, v) -> np.ndarray:
        f = self.lib.orc_f64_to_bf16
        flat = np.asarray(v, dtype=np.float64).ravel()
        return np.array([f(float(t)) for t in flat], dtype=np.uint16).reshape(np.shape(v))

    def f64_to_f16(self, v: float) -> int:
        """One round-to-nearest-even of an exact double to a binary16 bit pattern."""
        return int(self.lib.orc_f64_to_f16(float(v)))

    def f16_to_f64(self, h: int) -> float:
        return float(self.lib.orc_f16_to_f64(int(h) & 0xFFFF))

    def round_array(self, v, dtype="bf16") -> np.ndarray:
        """Doubles -> bit patterns of `dtype`, one rounding each."""
        f = self.lib.orc_f64_to_f16 if _dt(dtype) else self.lib.orc_f64_to_bf16
        flat = np.asarray(v, dtype=np.float64).ravel()
        return np.array([f(float(t)) for t in flat], dtype=np.uint16).reshape(np.shape(v))

    def unpack(self, words: np.ndarray, n_codes: int, bits: int) -> np.ndarray:
        words = _c(words, np.uint32)
        if words.size * (32 // bits) < n_codes:
            raise ValueError("not enough words")
        out = np.empty(n_codes, dtype=np.uint8)
        self.lib.orc_unpack(_ptr(words), n_codes, bits, _ptr(out))
        return out

    def dequant(self, w, s, b, K: int, gs: int, bits: int, dtype="bf16") -> np.ndarray:
        """Dequantised operand (rounded to `dtype`) as exact doubles, [rows, K]."""
        w, s, b = _c(w, np.uint32), _c(s, np.uint16), _c(b, np.uint16)
        rows = w.shape[0]
        out = np.empty((rows, K), dtype=np.float64)
        self.lib.orc_dequant(_ptr(w), _ptr(s), _ptr(b), rows, K, gs, bits, _dt(dtype), _ptr(out))
        return out

    @staticmethod
    def _qargs(x, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u):
        x = _c(x, np.uint16)
        M, H = x.shape
        wg, sg, bg = _c(wg, np.uint32), _c(sg, np.uint16), _c(bg, np.uint16)
        wu, su, bu = _c(wu, np.uint32), _c(su, np.uint16), _c(bu, np.uint16)
        I = wg.shape[0]
        if wg.shape != (I, H * bits_g // 32) or wu.shape != (I, H * bits_u // 32):
            raise ValueError("packed weight shape mismatch")
        if sg.shape != (I, H // gs_g) or bg.shape != sg.shape:
            raise ValueError("gate scale/bias shape mismatch")
        if su.shape != (I, H // gs_u) or bu.shape != su.shape:
            raise ValueError("up scale/bias shape mismatch")
        keep = (x, wg, sg, bg, wu, su, bu)
        args = [_ptr(x), M, H, I, _ptr(wg), _ptr(sg), _ptr(bg), gs_g, bits_g,
                _ptr(wu), _ptr(su), _ptr(bu), gs_u, bits_u]
        return keep, args, M, H, I

    def qswiglu(self, x, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u,
                variant=MATCH, rows=None, return_acc=False, dtype="bf16"):
        """hidden [len(rows) or M, I] as bit patterns (uint16) of `dtype`.

        With return_acc, also returns the unrounded f64 gate and up projections."""
        keep, args, M, H, I = self._qargs(x, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u)
        if rows is None:
            n_rows, rows_p, rows_arr = M, None, None
        else:
            rows_arr = _c(np.asarray(rows, dtype=np.int64), np.int64)
            if rows_arr.size and (rows_arr.min() < 0 or rows_arr.max() >= M):
                raise IndexError("row out of range")
            n_rows, rows_p = rows_arr.size, _ptr(rows_arr)
        out = np.empty((n_rows, I), dtype=np.uint16)
        g = np.empty((n_rows, I), dtype=np.float64) if return_acc else None
        u = np.empty((n_rows, I), dtype=np.float64) if return_acc else None
        rc = self.lib.orc_qswiglu_rows(*args, int(variant), _dt(dtype), rows_p, n_rows, _ptr(out),
                                       _ptr(g) if return_acc else None,
                                       _ptr(u) if return_acc else None)
        del keep, rows_arr
        if rc != 0:
            raise MemoryError("oracle allocation failed")
        return (out, g, u) if return_acc else out

    def qswiglu_pairs(self, x, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u, variant, pairs,
                      dtype="bf16"):
        """hidden[m, i] for each (m, i) in pairs ([n, 2] int64), as uint16 bits of `dtype`."""
        keep, args, M, H, I = self._qargs(x, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u)
        pairs = _c(np.asarray(pairs, dtype=np.int64).reshape(-1, 2), np.int64)
        if pairs.size and (pairs[:, 0].min() < 0 or pairs[:, 0].max() >= M
                           or pairs[:, 1].min() < 0 or pairs[:, 1].max() >= I):
            raise IndexError("pair out of range")
        out = np.empty(pairs.shape[0], dtype=np.uint16)
        rc = self.lib.orc_qswiglu_pairs(*args, int(variant), _dt(dtype), _ptr(pairs), pairs.shape[0],
                                        _ptr(out))
        del keep
        if rc != 0:
            raise MemoryError("oracle allocation failed")
        return out

    def qmm(self, x, w, s, b, gs, bits, dtype="bf16", residual=None):
        """Quantised linear y = T(x . W^T + residual) as uint16 [M, N] bits of T = `dtype`."""
        x, w, s, b = _c(x, np.uint16), _c(w, np.uint32), _c(s, np.uint16), _c(b, np.uint16)
        M, K = x.shape
        N = w.shape[0]
        if w.shape != (N, K * bits // 32) or s.shape != (N, K // gs) or b.shape != s.shape:
            raise ValueError("shape mismatch")
        r = None if residual is None else _c(residual, np.uint16)
        if r is not None and r.shape != (M, N):
            raise ValueError("residual shape mismatch")
        y = np.empty((M, N), dtype=np.uint16)
        if self.lib.orc_qmm(_ptr(x), M, K, N, _ptr(w), _ptr(s), _ptr(b), gs, bits, _dt(dtype),
                            None if r is None else _ptr(r), _ptr(y)) != 0:
            raise MemoryError("oracle allocation failed")
        return y

    def mlp(self, x, h, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u, wd, sd, bd, gs_d, bits_d,
            variant=MATCH, dtype="bf16"):
        """Whole MLP block y = T(h + hidden . Wd^T); returns (y [M, Ho], hidden [M, I])."""
        keep, args, M, H, I = self._qargs(x, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u)
        wd, sd, bd = _c(wd, np.uint32), _c(sd, np.uint16), _c(bd, np.uint16)
        Ho = wd.shape[0]
        if wd.shape != (Ho, I * bits_d // 32) or sd.shape != (Ho, I // gs_d) or bd.shape != sd.shape:
            raise ValueError("down weight shape mismatch")
        hh = None if h is None else _c(h, np.uint16)
        if hh is not None and hh.shape != (M, Ho):
            raise ValueError("residual shape mismatch")
        hidden = np.empty((M, I), dtype=np.uint16)
        y = np.empty((M, Ho), dtype=np.uint16)
        rc = self.lib.orc_mlp(args[0], None if hh is None else _ptr(hh), M, H, I, Ho, *args[4:],
                              _ptr(wd), _ptr(sd), _ptr(bd), gs_d, bits_d, int(variant), _dt(dtype),
                              _ptr(hidden), _ptr(y))
        del keep
        if rc != 0:
            raise MemoryError("oracle allocation failed")
        return y, hidden

    def silu_mul(self, g, u, variant=MATCH, dtype="bf16"):
        g, u = _c(g, np.uint16), _c(u, np.uint16)
        if g.shape != u.shape:
            raise ValueError("shape mismatch")
        out = np.empty_like(g)
        self.lib.orc_silu_mul(_ptr(g), _ptr(u), g.size, int(variant), _dt(dtype), _ptr(out))
        return out


_default: OracleLib | None = None


def default() -> OracleLib:
    """The oracle built from qsw_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
        return _default


def build_variant(src_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (used to check that the pins
    reject planted mistakes).  Same flags as build()."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", "-fno-fast-math", src, "-o", out_path, "-lm"],
                   check=True, capture_output=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def __getattr__(name):
    # module-level shortcuts: oracle.qswiglu(...), oracle.qmm(...), ...
    if name in ("num_threads", "set_num_threads", "f64_to_bf16", "bf16_to_f64",
                "bf16_round_array", "f64_to_f16", "f16_to_f64", "round_array", "unpack", "dequant",
                "qswiglu", "qswiglu_pairs", "qmm", "mlp", "silu_mul"):
        return getattr(default(), name)
    raise AttributeError(name)
