"""Seeded synthetic inputs for the quantized SwiGLU expansion.

This module is shared by the tests, the benchmark and the oracle checks.  It
holds no arithmetic of the method itself: it draws random numbers, casts them
to bf16 with the library cast, and packs integer codes into uint32 words in the
storage layout the kernels read (code k of a row at bits (k mod pf)*bits of
word k/pf, pf = 32/bits, least significant code first).

Recipe (one CPU ``torch.Generator`` seeded once, drawn in this order):
  x      ~ N(0, x_std^2) in f32, cast to T                          [M, H]
  q_g    ~ uniform integers 0 .. 2^bits_g - 1                       [I, H]
  s_g    ~ U(lo, hi) in f32, cast to T                              [I, H/gs_g]
  b_g    = -2^(bits_g-1) * s_g, exact in T (power-of-two multiple)
  q_u, s_u, b_u likewise with bits_u, gs_u.
T is the activation dtype: bf16 (default) or f16; values travel as uint16 bits.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass
class QuantMatrix:
    """One [rows, K] affine-quantised matrix in the kernels' storage layout."""
    packed: np.ndarray          # uint32 [rows, K*bits/32]
    scales: np.ndarray          # uint16 (bits of the activation dtype) [rows, K/gs]
    biases: np.ndarray          # uint16 (bits of the activation dtype) [rows, K/gs]
    gs: int
    bits: int
    codes: np.ndarray | None = None   # uint8 [rows, K], kept only on request


@dataclass
class Case:
    """A full set of inputs for one call: x plus gate and up weights."""
    x: np.ndarray               # uint16 (bits of the activation dtype) [M, H]
    gate: QuantMatrix
    up: QuantMatrix
    meta: dict = field(default_factory=dict)
    dtype: str = "bf16"         # activation dtype: "bf16" or "f16"

    @property
    def M(self) -> int:
        return self.x.shape[0]

    @property
    def H(self) -> int:
        return self.x.shape[1]

    @property
    def I(self) -> int:
        return self.gate.packed.shape[0]

    def oracle_args(self):
        """Positional arguments in (x, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u) order."""
        g, u = self.gate, self.up
        return (self.x, g.packed, g.scales, g.biases, g.gs, g.bits,
                u.packed, u.scales, u.biases, u.gs, u.bits)

    def digest(self) -> str:
        h = hashlib.sha256()
        for a in (self.x, self.gate.packed, self.gate.scales, self.gate.biases,
                  self.up.packed, self.up.scales, self.up.biases):
            h.update(np.ascontiguousarray(a).tobytes())
        return h.hexdigest()[:16]


def f32_to_bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Library float32 -> bf16 cast, returned as raw uint16 bit patterns."""
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


TORCH_DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16}


def f32_to_bits(t: torch.Tensor, dtype: str = "bf16") -> np.ndarray:
    """Library float32 -> `dtype` cast, returned as raw uint16 bit patterns."""
    return t.to(TORCH_DTYPES[dtype]).view(torch.int16).numpy().view(np.uint16).copy()


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack uint8 codes [rows, K] into uint32 words [rows, K*bits/32], LSB first."""
    if bits not in (2, 4, 8):
        raise ValueError("bits must be 2, 4 or 8")
    pf = 32 // bits
    rows, K = codes.shape
    if K % pf:
        raise ValueError("K must be a multiple of the pack factor")
    out = np.zeros((rows, K // pf), dtype=np.uint32)
    step = max(1, (1 << 22) // max(K, 1))      # bound the temporaries
    for r0 in range(0, rows, step):
        c = codes[r0:r0 + step].reshape(-1, K // pf, pf).astype(np.uint32)
        acc = np.zeros(c.shape[:2], dtype=np.uint32)
        for j in range(pf):
            acc |= c[:, :, j] << np.uint32(bits * j)
        out[r0:r0 + step] = acc
    return out


def _quant_matrix(gen: torch.Generator, rows: int, K: int, bits: int, gs: int,
                  scale_range, keep_codes: bool, dtype: str = "bf16") -> QuantMatrix:
    codes = torch.randint(0, 1 << bits, (rows, K), generator=gen, dtype=torch.uint8).numpy()
    lo, hi = scale_range
    s32 = torch.rand((rows, K // gs), generator=gen, dtype=torch.float32) * (hi - lo) + lo
    td = TORCH_DTYPES[dtype]
    s_t = s32.to(td)
    b_t = (s_t.to(torch.float32) * -float(1 << (bits - 1))).to(td)   # exact: power-of-two multiple
    return QuantMatrix(
        packed=pack_codes(codes, bits),
        scales=s_t.view(torch.int16).numpy().view(np.uint16).copy(),
        biases=b_t.view(torch.int16).numpy().view(np.uint16).copy(),
        gs=gs, bits=bits, codes=codes if keep_codes else None)


def make_case(M: int, H: int, I: int, *, bits_g: int = 4, gs_g: int = 64,
              bits_u: int | None = None, gs_u: int | None = None,
              x_std: float = 1.0, scale_range=(0.005, 0.02), seed: int = 0,
              keep_codes: bool = False, dtype: str = "bf16") -> Case:
    bits_u = bits_g if bits_u is None else bits_u
    gs_u = gs_g if gs_u is None else gs_u
    if H % gs_g or H % gs_u:
        raise ValueError("group sizes must divide H")
    if dtype not in TORCH_DTYPES:
        raise ValueError(f"dtype must be one of {sorted(TORCH_DTYPES)}")
    gen = torch.Generator(device="cpu").manual_seed(seed)
    x = f32_to_bits(torch.randn((M, H), generator=gen, dtype=torch.float32) * x_std, dtype)
    gate = _quant_matrix(gen, I, H, bits_g, gs_g, scale_range, keep_codes, dtype)
    up = _quant_matrix(gen, I, H, bits_u, gs_u, scale_range, keep_codes, dtype)
    return Case(x=x, gate=gate, up=up, dtype=dtype,
                meta=dict(M=M, H=H, I=I, bits_g=bits_g, gs_g=gs_g, bits_u=bits_u,
                          gs_u=gs_u, x_std=x_std, scale_range=tuple(scale_range), seed=seed,
                          dtype=dtype))


def bits_to_device(a: np.ndarray, dev, dtype: str = "bf16") -> torch.Tensor:
    """uint16 bit patterns -> a tensor of the activation dtype on `dev`."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(TORCH_DTYPES[dtype])


def _bits_to_bf16(a: np.ndarray, dev) -> torch.Tensor:
    return bits_to_device(a, dev, "bf16")


def _words_to_dev(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(dev)


def operand_to_device(qm: QuantMatrix, dev, dtype: str = "bf16"):
    """(packed int32, scales, biases, gs, bits) on `dev`; scales/biases in `dtype`."""
    return (_words_to_dev(qm.packed, dev), bits_to_device(qm.scales, dev, dtype),
            bits_to_device(qm.biases, dev, dtype), qm.gs, qm.bits)


def device_args(case: Case, dev):
    """(x, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u) as torch tensors on `dev`."""
    return (bits_to_device(case.x, dev, case.dtype), *operand_to_device(case.gate, dev, case.dtype),
            *operand_to_device(case.up, dev, case.dtype))


def make_x(M: int, H: int, *, x_std: float = 1.0, seed: int = 0, dtype: str = "bf16") -> np.ndarray:
    gen = torch.Generator(device="cpu").manual_seed(seed)
    return f32_to_bits(torch.randn((M, H), generator=gen, dtype=torch.float32) * x_std, dtype)


# The five synthetic workloads: sizes, code widths, group sizes and value ranges.
WORKLOADS = {
    "tiny_prefill": dict(M=6, H=512, I=1536, bits_g=4, gs_g=64, x_std=1.0,
                         scale_range=(0.005, 0.02)),
    "decode": dict(M=1, H=2048, I=8192, bits_g=4, gs_g=64, x_std=1.0,
                   scale_range=(0.005, 0.02)),
    "mid_prefill": dict(M=512, H=2048, I=8192, bits_g=4, gs_g=64, x_std=1.0,
                        scale_range=(0.005, 0.02)),
    "large_prefill": dict(M=4096, H=4096, I=14336, bits_g=4, gs_g=64, x_std=0.5,
                          scale_range=(0.002, 0.01)),
    "mixed": dict(M=2048, H=2560, I=10240, bits_g=4, gs_g=64, bits_u=8, gs_u=32,
                  x_std=1.0, scale_range=(0.005, 0.02)),
}
MIXED_M_SWEEP = (1, 2, 3, 4, 8, 64, 2048)


def workload_case(name: str, *, M: int | None = None, seed: int = 0,
                  keep_codes: bool = False) -> Case:
    kw = dict(WORKLOADS[name])
    if M is not None:
        kw["M"] = M
    return make_case(seed=seed, keep_codes=keep_codes, **kw)
