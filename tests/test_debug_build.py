"""The debug build (libqswiglu_debug.so, QSW_DEBUG_BOUNDS) on small cases of
the three kernels: every kernel fills its shared-memory staging (and the
tensor-core kernel its TMEM accumulators) with NaN patterns first, so a read
of staging data that was never written would surface as NaN and fail the
oracle comparison, and its address and copy checks would report
QSW_ERR_BOUNDS.  Run in a fresh process, which loads only the debug build."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_SCRIPT = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, {root!r})
import oracle
from quantized_swiglu_mlp_gb300 import build, inputs, ops
from tests.exact_sums import projection_context
from tests.gpu_util import device_args, to_bits
from tests.tolerances import check_f32, check_match_with_projections, check_projection

ops.load_library(build.DEBUG_LIB_PATH)
assert ops.qsw_debug_build()
torch.cuda.set_device(0)
dev = torch.device("cuda:0")

def fused(case, kernel):
    a = device_args(case, dev)
    outs = {{v: to_bits(ops.qswiglu_forward(*a, variant=v)) for v in range(4)}}
    ops.qsw_check_device_errors()      # raises on QSW_ERR_BOUNDS or a timeout
    dt = case.dtype
    h, g64, u64 = oracle.qswiglu(*case.oracle_args(), variant=oracle.MATCH, return_acc=True, dtype=dt)
    _, _, bg, bu = projection_context(case, kernel)
    ok, info = check_match_with_projections(
        outs[0], outs[2], outs[3], h, oracle.round_array(g64, dt), oracle.round_array(u64, dt),
        lambda g, u: oracle.silu_mul(np.ascontiguousarray(g), np.ascontiguousarray(u), oracle.MATCH, dtype=dt),
        dt, exact=(g64, u64), bounds=(bg, bu))
    assert ok, (case.M, case.H, case.I, kernel, info)
    ok, info = check_f32(outs[1], oracle.qswiglu(*case.oracle_args(), variant=oracle.F32, dtype=dt), dt)
    assert ok, (case.M, case.H, case.I, kernel, "f32", info)

shapes = [(1, 64, 8, 4, 64, 4, 64), (130, 512, 200, 4, 64, 4, 64), (257, 2080, 384, 4, 32, 8, 32),
          (64, 256, 203, 8, 64, 4, 128), (200, 640, 136, 2, 64, 8, 64)]
for mode in (ops.STREAM_K_OFF, ops.STREAM_K_ALWAYS):
    ops.qsw_set_stream_k(mode)
    ops.qsw_set_gemv_max_m(0)
    for M, H, I, bg_, gg, bu_, gu in shapes:
        fused(inputs.make_case(M, H, I, bits_g=bg_, gs_g=gg, bits_u=bu_, gs_u=gu, seed=M + H), "tensor_core")
ops.qsw_set_gemv_max_m(32)
for kernel in (ops.SMALL_M_RING, ops.SMALL_M_STREAM):
    ops.qsw_set_small_m_kernel(kernel)
    for M, H, I, bg_, gg, bu_, gu in [(1, 512, 8, 4, 64, 4, 64), (3, 512, 203, 4, 64, 4, 64),
                                      (8, 512, 64, 2, 64, 4, 32), (17, 1024, 100, 4, 64, 4, 64),
                                      (6, 2048, 20000, 4, 64, 4, 64), (2, 2080, 64, 4, 32, 8, 32),
                                      (12, 1024, 100, 4, 64, 8, 32), (20, 512, 64, 4, 64, 4, 64)]:
        fused(inputs.make_case(M, H, I, bits_g=bg_, gs_g=gg, bits_u=bu_, gs_u=gu, seed=M * 3 + H), "small_m")
    fused(inputs.make_case(5, 512, 136, seed=9, dtype="f16"), "small_m")
ops.qsw_set_gemv_max_m(0)
fused(inputs.make_case(150, 512, 136, seed=9, dtype="f16"), "tensor_core")
# the single-operand form on the three kernels
for limit, M, kernel in ((0, 70, ops.SMALL_M_AUTO), (32, 3, ops.SMALL_M_RING), (32, 3, ops.SMALL_M_STREAM)):
    ops.qsw_set_small_m_kernel(kernel)
    ops.qsw_set_gemv_max_m(limit)
    case = inputs.make_case(M, 1024, 300, bits_g=4, gs_g=64, seed=M)
    x, w, s, b, gs, bits = device_args(case, dev)[:6]
    y = to_bits(ops.affine_qmm(x, w, s, b, gs, bits))
    ops.qsw_check_device_errors()
    ok, info = check_projection(y, oracle.qmm(case.x, case.gate.packed, case.gate.scales, case.gate.biases, gs, bits))
    assert ok, ("qmm", limit, kernel, info)
print("OK")
"""


def test_debug_build_matches_the_oracle():
    r = subprocess.run([sys.executable, "-c", _SCRIPT.format(root=ROOT)], capture_output=True, text=True,
                       timeout=900, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout[-3000:] + r.stderr[-3000:]
