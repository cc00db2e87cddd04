"""The no-alloc fused entry point: stream-K scheduling on the library's static
scratch array instead of a caller workspace.  Parity with the oracle, repeated
calls and CUDA-graph replays (the scratch's launch counter carries over), and
no device memory taken by the calls."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from quantized_swiglu_mlp_gb300 import inputs, ops
from tests.exact_sums import projection_context
from tests.gpu_util import device_args, to_bits
from tests.tolerances import check_f32, check_match_with_projections

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch.cuda.set_device(0)
    ops.load_library()
    return torch.device("cuda:0")


@pytest.fixture
def forced_split():
    saved_k, saved_m = ops.qsw_get_stream_k(), ops.qsw_get_gemv_max_m()
    ops.qsw_set_stream_k(ops.STREAM_K_ALWAYS)
    ops.qsw_set_gemv_max_m(0)
    yield
    ops.qsw_set_stream_k(saved_k)
    ops.qsw_set_gemv_max_m(saved_m)


def _match_ok(case, outs):
    h_ref, g64, u64 = oracle.qswiglu(*case.oracle_args(), variant=oracle.MATCH, return_acc=True)
    _, _, bnd_g, bnd_u = projection_context(case, "tensor_core")
    return check_match_with_projections(
        to_bits(outs[ops.MATCH]), to_bits(outs[ops.DEBUG_GATE]), to_bits(outs[ops.DEBUG_UP]), h_ref,
        oracle.bf16_round_array(g64), oracle.bf16_round_array(u64),
        lambda g, u: oracle.silu_mul(np.ascontiguousarray(g), np.ascontiguousarray(u), oracle.MATCH),
        exact=(g64, u64), bounds=(bnd_g, bnd_u))


@pytest.mark.parametrize("shape", [(300, 512, 1536, 4, 64, 4, 64), (257, 2080, 384, 4, 32, 8, 32)],
                         ids=["M300_H512_I1536", "M257_H2080_I384_mixed"])
def test_noalloc_matches_oracle(dev, forced_split, shape):
    M, H, I, bg, gg, bu, gu = shape
    case = inputs.make_case(M, H, I, bits_g=bg, gs_g=gg, bits_u=bu, gs_u=gu, seed=M + 3)
    a = device_args(case, dev)
    before = ops.qsw_get_counters()[ops.CNT_FUSED_TC]
    outs = {v: ops.qswiglu_forward_noalloc(*a, variant=v) for v in (ops.MATCH, ops.DEBUG_GATE, ops.DEBUG_UP)}
    f32 = ops.qswiglu_forward_noalloc(*a, variant=ops.F32)
    ops.qsw_check_device_errors()
    assert ops.qsw_get_counters()[ops.CNT_FUSED_TC] == before + 4
    ok, info = _match_ok(case, outs)
    assert ok, info
    ok, info = check_f32(to_bits(f32), oracle.qswiglu(*case.oracle_args(), variant=oracle.F32))
    assert ok, info


def test_noalloc_graph_replays_and_takes_no_memory(dev, forced_split):
    """Captured in a CUDA graph and replayed with new x: each replay matches
    the oracle for its x; eager calls and replays leave the device's free
    memory unchanged."""
    base = inputs.make_case(300, 512, 1536, seed=51)
    a = device_args(base, dev)
    x_static = a[0].clone()
    outs = {v: torch.empty((300, 1536), dtype=torch.bfloat16, device=dev)
            for v in (ops.MATCH, ops.DEBUG_GATE, ops.DEBUG_UP)}
    stream = torch.cuda.Stream(device=dev)

    def calls():
        for v, o in outs.items():
            ops.qswiglu_forward_noalloc(x_static, *a[1:], variant=v, out=o, stream=stream)

    with torch.cuda.stream(stream):
        calls()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info(dev)[0]
    with torch.cuda.stream(stream):
        for _ in range(5):
            calls()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(dev)[0] == free0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        calls()
    torch.cuda.synchronize()
    for seed in (61, 62):
        xb = inputs.make_x(300, 512, seed=seed)
        x_static.copy_(torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16))
        for o in outs.values():
            o.fill_(0)
        g.replay()
        ops.qsw_check_device_errors()
        ok, info = _match_ok(inputs.Case(x=xb, gate=base.gate, up=base.up), outs)
        assert ok, info


_FIRST_USE_IN_CAPTURE = r"""
import sys
import torch
sys.path.insert(0, {root!r})
import oracle
from quantized_swiglu_mlp_gb300 import inputs, ops
from tests.gpu_util import device_args, to_bits
from tests.tolerances import check_match
ops.load_library()
torch.cuda.set_device(0)
dev = torch.device("cuda:0")
ops.qsw_set_stream_k(ops.STREAM_K_ALWAYS)
ops.qsw_set_gemv_max_m(0)
case = inputs.make_case(300, 512, 1536, seed=11)
a = device_args(case, dev)
want = oracle.qswiglu(*case.oracle_args(), variant=oracle.MATCH)
out = torch.empty((300, 1536), dtype=torch.bfloat16, device=dev)
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):   # the process's first no-alloc call
    ops.qswiglu_forward_noalloc(*a, variant=ops.MATCH, out=out, stream=s)
for _ in range(2):
    out.fill_(0)
    with torch.cuda.stream(s):
        g.replay()
    torch.cuda.synchronize()
    ops.qsw_check_device_errors(s)
    assert check_match(to_bits(out), want)[0], "replay"
    e = ops.qswiglu_forward_noalloc(*a, variant=ops.MATCH, stream=s)
    torch.cuda.synchronize()
    ops.qsw_check_device_errors(s)
    assert check_match(to_bits(e), want)[0], "eager"
print("OK")
"""


def test_noalloc_first_use_inside_capture(dev):
    """In a fresh process the first no-alloc call is made inside a CUDA-graph
    capture (so the scratch header's zeroing is recorded into the graph); two
    replays interleaved with eager calls on the same stream all match the
    oracle."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_USE_IN_CAPTURE.format(root=root)], capture_output=True,
                       text=True, timeout=600, cwd=root)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout[-2000:] + r.stderr[-2000:]
