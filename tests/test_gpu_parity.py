"""CUDA path vs the oracle, element by element, through the C ABI.

Small shapes span several tiles and ragged tails on both kernels; the five
workload shapes are checked on sampled rows/elements at full size in the
launch configuration the benchmark times.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from quantized_swiglu_mlp_gb300 import inputs, ops
from tests.exact_sums import projection_context
from tests.gpu_util import device_args, to_bits
from tests.tolerances import TO_F64, check_f32, check_match, check_match_with_projections, check_projection

pytestmark = pytest.mark.gpu

VARIANTS = [ops.MATCH, ops.F32, ops.DEBUG_GATE, ops.DEBUG_UP]
VNAMES = {ops.MATCH: "match", ops.F32: "f32", ops.DEBUG_GATE: "gate", ops.DEBUG_UP: "up"}


@pytest.fixture(scope="module")
def dev():
    torch.cuda.set_device(0)
    ops.load_library()
    return torch.device("cuda:0")


@pytest.fixture
def gemv_limit():
    saved = ops.qsw_get_gemv_max_m()
    yield ops.qsw_set_gemv_max_m
    ops.qsw_set_gemv_max_m(saved)


@pytest.fixture
def small_m_kernel():
    saved = ops.qsw_get_small_m_kernel()
    yield ops.qsw_set_small_m_kernel
    ops.qsw_set_small_m_kernel(saved)


# the two small-M kernels: slot ring (bulk copies into CTA-shared slots) and
# warp-streamed (M <= 16)
SMALL_M_KERNELS = [ops.SMALL_M_RING, ops.SMALL_M_STREAM]
KNAMES = {ops.SMALL_M_RING: "ring", ops.SMALL_M_STREAM: "stream"}


def expect_small_m(before, kernel, M, counter=None):
    """The call(s) since `before` ran on the small-M path, on the selected
    kernel (the warp-streamed one serves M <= 32 at these shapes, in launches of up to 16 rows)."""
    after = ops.qsw_get_counters()
    if counter is not None:
        assert after[counter] > before[counter]
    reg = after[ops.CNT_GEMV_STREAM] > before[ops.CNT_GEMV_STREAM]
    assert reg == (kernel == ops.SMALL_M_STREAM and M <= 32), (kernel, M)


def check(variant, got, want, dtype="bf16"):
    """F32 and the stored projections against the oracle (MATCH goes through
    check_fused, which also needs the projections)."""
    if variant == ops.MATCH:
        ok, info = check_match(got, want, dtype)
    elif variant == ops.F32:
        ok, info = check_f32(got, want, dtype)
    else:
        ok, info = check_projection(got, want, dtype)
    assert ok, info


def run_fused(case, dev, variant, args=None):
    out = ops.qswiglu_forward(*(args or device_args(case, dev)), variant=variant)
    ops.qsw_check_device_errors()
    return to_bits(out)


def match_epilogue(g, u, dtype="bf16"):
    return oracle.silu_mul(np.ascontiguousarray(g), np.ascontiguousarray(u), oracle.MATCH, dtype=dtype)


def check_fused(case, dev, variant, rows=None, pairs=None):
    """Run `variant` on the GPU and compare with the oracle on all rows, the
    listed rows, or the listed (m, i) pairs.  Returns the GPU result.  MATCH
    is checked with the stored projections, the exact f64 sums and the
    accumulation bound of the kernel that ran."""
    a = device_args(case, dev)
    before = ops.qsw_get_counters()[ops.CNT_FUSED_TC]
    got = run_fused(case, dev, variant, a)
    kernel = "tensor_core" if ops.qsw_get_counters()[ops.CNT_FUSED_TC] > before else "small_m"
    if rows is not None:
        sel = (np.asarray(rows),)
    elif pairs is not None:
        sel = (pairs[:, 0], pairs[:, 1])
    else:
        sel = (slice(None),)
    dt = case.dtype
    if pairs is not None:
        want = {v: oracle.qswiglu_pairs(*case.oracle_args(), v, pairs, dtype=dt)
                for v in (variant, ops.DEBUG_GATE, ops.DEBUG_UP)}
        h_ref, g_ref, u_ref = want[variant], want[ops.DEBUG_GATE], want[ops.DEBUG_UP]
        if variant == ops.MATCH:
            g64, u64, bnd_g, bnd_u = projection_context(case, kernel, pairs=pairs)
    elif variant == ops.MATCH:
        h_ref, g64, u64 = oracle.qswiglu(*case.oracle_args(), variant=variant, rows=rows, return_acc=True,
                                         dtype=dt)
        g_ref, u_ref = oracle.round_array(g64, dt), oracle.round_array(u64, dt)
        _, _, bnd_g, bnd_u = projection_context(case, kernel, rows=rows)
    else:
        h_ref = oracle.qswiglu(*case.oracle_args(), variant=variant, rows=rows, dtype=dt)
    if variant == ops.MATCH:
        g_gpu = run_fused(case, dev, ops.DEBUG_GATE, a)[sel]
        u_gpu = run_fused(case, dev, ops.DEBUG_UP, a)[sel]
        ok, info = check_match_with_projections(got[sel], g_gpu, u_gpu, h_ref, g_ref, u_ref,
                                                lambda g, u: match_epilogue(g, u, dt), dt,
                                                exact=(g64, u64), bounds=(bnd_g, bnd_u))
        assert ok, info
    else:
        check(variant, got[sel], h_ref, dt)
    return got


# (M, H, I, bits_g, gs_g, bits_u, gs_u): tiles of 128 rows x 128 columns x 64 K
TC_SHAPES = [
    (1, 64, 8, 4, 64, 4, 64),          # one partial tile everywhere
    (3, 96, 40, 4, 32, 4, 32),         # K tail of 32, M in {2,3} territory
    (130, 512, 200, 4, 64, 4, 64),     # 2 M tiles, 2 N tiles, ragged both
    (257, 2080, 384, 4, 32, 8, 32),    # 3 M tiles, 3 N tiles, K tail, mixed specs
    (64, 256, 203, 8, 64, 4, 128),     # I % 8 != 0 (scalar stores)
    (200, 640, 136, 2, 64, 8, 64),     # 2-bit gate
    (128, 1024, 256, 8, 32, 8, 32),    # exact tiles, 8-bit both
]

# The slot-ring small-M kernel stages a unit's scale rows with 16-byte copies,
# so it takes shapes with (H / gs) % 8 == 0; with it selected the others run on
# the tensor-core kernel (test_small_m_routes_unstageable_shapes).
GEMV_SHAPES = [
    (1, 512, 8, 4, 64, 4, 64),         # one partial unit
    (2, 256, 40, 4, 32, 8, 32),        # mixed specs, 5 units
    (3, 512, 203, 4, 64, 4, 64),       # ragged last unit
    (4, 2304, 136, 8, 32, 4, 32),      # 8-bit gate
    (8, 512, 64, 2, 64, 4, 32),        # 2-bit gate
    (9, 1024, 48, 4, 128, 8, 32),      # two x row groups
    (17, 1024, 100, 4, 64, 4, 64),     # four x row groups
    (6, 2048, 20000, 4, 64, 4, 64),    # more units than staging slots: slot refills
]


def _ids(shapes):
    return ["M{}_H{}_I{}_g{}x{}_u{}x{}".format(*s) for s in shapes]


@pytest.mark.parametrize("shape", TC_SHAPES, ids=_ids(TC_SHAPES))
@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: VNAMES[v])
def test_tensor_core_kernel(dev, gemv_limit, shape, variant):
    M, H, I, bg, gg, bu, gu = shape
    case = inputs.make_case(M, H, I, bits_g=bg, gs_g=gg, bits_u=bu, gs_u=gu, seed=M * 7 + H)
    gemv_limit(0)
    before = ops.qsw_get_counters()[ops.CNT_FUSED_TC]
    check_fused(case, dev, variant)
    assert ops.qsw_get_counters()[ops.CNT_FUSED_TC] > before


@pytest.mark.parametrize("kernel", SMALL_M_KERNELS, ids=lambda k: KNAMES[k])
@pytest.mark.parametrize("shape", GEMV_SHAPES, ids=_ids(GEMV_SHAPES))
@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: VNAMES[v])
def test_small_m_kernel(dev, gemv_limit, small_m_kernel, kernel, shape, variant):
    M, H, I, bg, gg, bu, gu = shape
    case = inputs.make_case(M, H, I, bits_g=bg, gs_g=gg, bits_u=bu, gs_u=gu, seed=M * 11 + H)
    gemv_limit(32)
    small_m_kernel(kernel)
    before = ops.qsw_get_counters()
    check_fused(case, dev, variant)
    expect_small_m(before, kernel, M, ops.CNT_FUSED_GEMV)


# More small-M shapes: many slot refills per CTA, odd M, 2- and 8-bit
# operands, K blocks fewer than warps, the mixed-spec workload's specs.
MORE_SMALL_M_SHAPES = [
    (1, 2048, 30000, 4, 64, 4, 64),    # 30000 rows: each CTA's slots are refilled many times
    (7, 1024, 1203, 4, 64, 8, 32),     # M odd, ragged last unit
    (2, 4096, 3000, 2, 64, 4, 128),    # 2-bit gate, 32 K blocks per unit
    (5, 256, 17, 8, 32, 8, 32),        # 3 units, 2 K blocks: most warps idle
    (3, 2560, 10240, 4, 64, 8, 32),    # the mixed-spec workload's specs
    (16, 1024, 2000, 4, 64, 8, 32),    # two x row groups, mixed specs
    (13, 2048, 1203, 2, 64, 4, 64),    # two x row groups, odd M, 2-bit gate, ragged last unit
    (27, 1024, 520, 4, 64, 8, 32),     # M > 16: launches over row chunks of 16 and 11
]


@pytest.mark.parametrize("kernel", SMALL_M_KERNELS, ids=lambda k: KNAMES[k])
@pytest.mark.parametrize("shape", MORE_SMALL_M_SHAPES, ids=_ids(MORE_SMALL_M_SHAPES))
@pytest.mark.parametrize("variant", [ops.MATCH, ops.F32], ids=["match", "f32"])
def test_small_m_kernel_more_shapes(dev, gemv_limit, small_m_kernel, kernel, shape, variant):
    M, H, I, bg, gg, bu, gu = shape
    case = inputs.make_case(M, H, I, bits_g=bg, gs_g=gg, bits_u=bu, gs_u=gu, seed=M * 13 + I)
    gemv_limit(32)
    small_m_kernel(kernel)
    before = ops.qsw_get_counters()
    check_fused(case, dev, variant, rows=list(range(M)))
    if not (kernel == ops.SMALL_M_RING and M > 16):   # (where the slot-ring kernel may not fit)
        expect_small_m(before, kernel, M, ops.CNT_FUSED_GEMV)


@pytest.mark.parametrize("kernel", SMALL_M_KERNELS, ids=lambda k: KNAMES[k])
@pytest.mark.parametrize("M,K,N", [(1, 2048, 1000), (3, 1024, 203), (8, 512, 40), (2, 8192, 2048), (12, 2048, 520),
                                   (19, 1024, 300)])
@pytest.mark.parametrize("with_residual", [False, True], ids=["plain", "residual"])
def test_small_m_single_operand(dev, gemv_limit, small_m_kernel, kernel, M, K, N, with_residual):
    """affine_qmm on the small-M kernels (ragged units), with and without a
    residual."""
    case = inputs.make_case(M, K, N, bits_g=4, gs_g=64, seed=M + K + N)
    gemv_limit(32)
    small_m_kernel(kernel)
    x, w, s, b, gs, bits = device_args(case, dev)[:6]
    h = inputs.make_x(M, N, seed=K) if with_residual else None
    before = ops.qsw_get_counters()
    y = ops.affine_qmm(x, w, s, b, gs, bits, residual=None if h is None else inputs.bits_to_device(h, dev))
    got = to_bits(y)
    ops.qsw_check_device_errors()
    if not (kernel == ops.SMALL_M_RING and M > 16):   # (where the slot-ring kernel may not fit)
        assert ops.qsw_get_counters()[ops.CNT_QMM_GEMV] == before[ops.CNT_QMM_GEMV] + 1
        expect_small_m(before, kernel, M)
    want = oracle.qmm(case.x, case.gate.packed, case.gate.scales, case.gate.biases, gs, bits, residual=h)
    ok, info = check_projection(got, want)
    assert ok, info


@pytest.mark.parametrize("early", [False, True], ids=["plain", "early_weights"])
def test_small_m_wait_runs_out(dev, gemv_limit, small_m_kernel, early_weights, early):
    """A fill that never comes: with the test hook, the next call on the
    slot-ring small-M kernel never requests its CTAs' first units.  Every wait on them gives up after the
    (short) limit, the kernel returns without trapping, the error word reports
    QSW_ERR_TIMEOUT, and the next call on the same stream is correct again."""
    case = inputs.workload_case("decode")
    gemv_limit(16)
    small_m_kernel(ops.SMALL_M_RING)
    early_weights(early)
    a = device_args(case, dev)
    want = oracle.qswiglu(*case.oracle_args(), variant=ops.MATCH)
    ops.qsw_set_wait_timeout_ns(20_000_000)
    try:
        ops.qsw_debug_withhold_next_fill()
        ops.qswiglu_forward(*a, variant=ops.MATCH)
        with pytest.raises(ops.QswError) as e:
            ops.qsw_check_device_errors()
        assert e.value.code == 4   # QSW_ERR_TIMEOUT
        got = to_bits(ops.qswiglu_forward(*a, variant=ops.MATCH))
        ops.qsw_check_device_errors()
    finally:
        ops.qsw_set_wait_timeout_ns(4_000_000_000)
    ok, info = check_match(got, want)
    assert ok, info


@pytest.mark.parametrize("shape", [(2, 96, 40, 4, 32, 4, 32), (3, 2080, 64, 4, 32, 8, 32)],
                         ids=["groups_per_row_12", "k_tail"])
def test_small_m_routes_unstageable_shapes(dev, gemv_limit, small_m_kernel, shape):
    """Shapes the slot-ring kernel cannot stage go to the tensor-core kernel
    when it is selected; the warp-streamed kernel takes them."""
    M, H, I, bg, gg, bu, gu = shape
    case = inputs.make_case(M, H, I, bits_g=bg, gs_g=gg, bits_u=bu, gs_u=gu, seed=5)
    gemv_limit(32)
    small_m_kernel(ops.SMALL_M_RING)
    before = ops.qsw_get_counters()
    check_fused(case, dev, ops.MATCH)
    after = ops.qsw_get_counters()
    assert after[ops.CNT_FUSED_TC] > before[ops.CNT_FUSED_TC]
    assert after[ops.CNT_FUSED_GEMV] == before[ops.CNT_FUSED_GEMV]
    small_m_kernel(ops.SMALL_M_STREAM)
    before = ops.qsw_get_counters()
    for v in VARIANTS:
        check_fused(case, dev, v)
    expect_small_m(before, ops.SMALL_M_STREAM, M, ops.CNT_FUSED_GEMV)


@pytest.mark.parametrize("kernel", SMALL_M_KERNELS, ids=lambda k: KNAMES[k])
@pytest.mark.parametrize("M", [1, 4, 8])
def test_small_m_projection_rate(dev, gemv_limit, small_m_kernel, kernel, M):
    """The exact-projection rate of the small-M kernels on a large sample
    (mixed specs, H=2560, all 10240 outputs)."""
    case = inputs.workload_case("mixed", M=M, seed=7)
    gemv_limit(32)
    small_m_kernel(kernel)
    a = device_args(case, dev)
    _, g64, u64 = oracle.qswiglu(*case.oracle_args(), variant=ops.MATCH, return_acc=True)
    before = ops.qsw_get_counters()[ops.CNT_FUSED_GEMV]
    for v, ref in ((ops.DEBUG_GATE, g64), (ops.DEBUG_UP, u64)):
        got = run_fused(case, dev, v, a)
        ok, info = check_projection(got, oracle.bf16_round_array(ref))
        assert ok and got.size >= 10_000, info
    assert ops.qsw_get_counters()[ops.CNT_FUSED_GEMV] == before + 2


@pytest.mark.parametrize("limit,M,kernel", [(0, 24, ops.SMALL_M_AUTO), (32, 24, ops.SMALL_M_RING),
                                            (32, 6, ops.SMALL_M_RING), (32, 6, ops.SMALL_M_STREAM),
                                            (32, 12, ops.SMALL_M_STREAM), (32, 24, ops.SMALL_M_STREAM)],
                         ids=["tensor_core", "small_m_ring_M24", "small_m_ring_M6", "small_m_stream_M6",
                              "small_m_stream_M12", "small_m_stream_M24_chunks"])
def test_fused_match_equals_unfused(dev, gemv_limit, small_m_kernel, limit, M, kernel):
    """MATCH is the unfused composition op for op, and both kernels compute it
    bit for bit: each kernel folds every K block into the f32 accumulator the
    same way in its fused and single-operand forms (same K split; an MMA's
    result for one A row does not depend on the other rows -- measured: the
    fused gate/up projections equal affine_qmm's bit for bit), and the MATCH
    epilogue rounds at the same points as the elementwise kernel."""
    case = inputs.make_case(M, 1024, 264, bits_g=4, gs_g=64, bits_u=8, gs_u=32, seed=3)
    gemv_limit(limit)
    small_m_kernel(kernel)
    before = ops.qsw_get_counters()
    a = device_args(case, dev)
    # whole tiles: the fused and single-operand launches split K differently
    # under stream-K scheduling, which changes the f32 summation order
    fused = to_bits(ops.qswiglu_forward(*a, variant=ops.MATCH, workspace=None))
    unfused = to_bits(ops.unfused_swiglu(*a, variant=ops.MATCH, workspace=None))
    x, wg, sg, bg, gsg, btg, wu, su, bu, gsu, btu = a
    pg = to_bits(ops.qswiglu_forward(*a, variant=ops.DEBUG_GATE, workspace=None))
    pu = to_bits(ops.qswiglu_forward(*a, variant=ops.DEBUG_UP, workspace=None))
    sg_ = to_bits(ops.affine_qmm(x, wg, sg, bg, gsg, btg, workspace=None))
    su_ = to_bits(ops.affine_qmm(x, wu, su, bu, gsu, btu, workspace=None))
    ops.qsw_check_device_errors()
    if limit:
        expect_small_m(before, kernel, M, ops.CNT_FUSED_GEMV)
    assert np.array_equal(pg, sg_) and np.array_equal(pu, su_)
    assert np.array_equal(fused, unfused)


@pytest.mark.parametrize("limit,kernel", [(0, ops.SMALL_M_AUTO), (32, ops.SMALL_M_RING), (32, ops.SMALL_M_STREAM)],
                         ids=["tensor_core", "small_m_ring", "small_m_stream"])
@pytest.mark.parametrize("bits,gs", [(4, 64), (8, 32), (2, 64)])
def test_affine_qmm(dev, gemv_limit, small_m_kernel, limit, kernel, bits, gs):
    M, K, N = (5, 1024, 300) if limit else (140, 640, 300)
    case = inputs.make_case(M, K, N, bits_g=bits, gs_g=gs, seed=bits + gs)
    gemv_limit(limit)
    small_m_kernel(kernel)
    x, w, s, b, _, _ = device_args(case, dev)[:6]
    got = to_bits(ops.affine_qmm(x, w, s, b, gs, bits))
    ops.qsw_check_device_errors()
    want = oracle.qmm(case.x, case.gate.packed, case.gate.scales, case.gate.biases, gs, bits)
    ok, info = check_projection(got, want)
    assert ok, info


@pytest.mark.parametrize("variant", [ops.MATCH, ops.F32], ids=["match", "f32"])
@pytest.mark.parametrize("n", [0, 7, 8, 1000, 65539])
def test_silu_mul(dev, variant, n):
    rng = np.random.default_rng(n)
    g = inputs.f32_to_bf16_bits(torch.from_numpy(rng.normal(0, 4, n).astype(np.float32)))
    u = inputs.f32_to_bf16_bits(torch.from_numpy(rng.normal(0, 2, n).astype(np.float32)))
    gd = torch.from_numpy(g.view(np.int16)).to(dev).view(torch.bfloat16)
    ud = torch.from_numpy(u.view(np.int16)).to(dev).view(torch.bfloat16)
    got = to_bits(ops.qsw_silu_mul(gd, ud, variant))
    want = oracle.silu_mul(g, u, variant)
    if variant == ops.MATCH:
        ok, info = check_match(got, want)
    else:
        ok, info = check_f32(got, want)
    assert ok, info


def test_all_bf16_gate_values(dev):
    """Every finite bf16 gate value through the elementwise MATCH step."""
    h = np.arange(0, 0x10000, dtype=np.uint32)
    keep = np.isfinite((h << 16).view(np.float32))
    g = h[keep].astype(np.uint16)
    u = inputs.f32_to_bf16_bits(torch.full((g.size,), 1.5))
    gd = torch.from_numpy(g.view(np.int16)).to(dev).view(torch.bfloat16)
    ud = torch.from_numpy(u.view(np.int16)).to(dev).view(torch.bfloat16)
    got = to_bits(ops.qsw_silu_mul(gd, ud, ops.MATCH))
    ok, info = check_match(got, oracle.silu_mul(g, u, ops.MATCH))
    assert ok, info


def test_paired_and_scalar_match_epilogues_agree(dev):
    """The MATCH epilogue has a paired form (two elements per bf16x2
    instruction: tensor-core epilogue, vector silu*mul) and a scalar form
    (small-M kernel, silu*mul tail); over every finite bf16 gate value and a
    spread of up values the two give the same bits.  The scalar form is reached
    through 7-element silu*mul calls (all tail), at two offsets so that every
    element lands in one of them."""
    h = np.arange(0, 0x10000, dtype=np.uint32)
    g = h[np.isfinite((h << 16).view(np.float32))].astype(np.uint16)
    n = (g.size // 8) * 8
    g = g[:n]
    rng = np.random.default_rng(7)
    u = inputs.f32_to_bf16_bits(torch.from_numpy(rng.normal(0, 2, n).astype(np.float32)))
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    paired = to_bits(ops.qsw_silu_mul(to_dev(g), to_dev(u), ops.MATCH))
    scalar = np.zeros(n, dtype=np.uint16)
    seen = np.zeros(n, dtype=bool)
    for shift in (0, 1):
        gd, ud = to_dev(np.roll(g, -shift)), to_dev(np.roll(u, -shift))
        out = torch.zeros_like(gd)
        for k in range(0, n - 7, 8):
            ops.qsw_silu_mul(gd[k:k + 7], ud[k:k + 7], ops.MATCH, out=out[k:k + 7])
        got = np.roll(to_bits(out), shift)
        idx = (np.arange(n) + shift) % n   # rolled position -> original position
        covered = np.zeros(n, dtype=bool)
        for k in range(0, n - 7, 8):
            covered[idx[k:k + 7]] = True
        scalar[covered & ~seen] = got[covered & ~seen]
        seen |= covered
    ops.qsw_check_device_errors()
    assert seen.all()
    assert np.array_equal(paired, scalar), np.flatnonzero(paired != scalar)[:10]


@pytest.mark.parametrize("limit", [0, 32], ids=["tensor_core", "small_m"])
def test_zero_input_gives_zero(dev, gemv_limit, limit):
    case = inputs.make_case(5, 256, 130, seed=1)
    case.x[:] = 0
    gemv_limit(limit)
    for v in VARIANTS:
        assert np.all(run_fused(case, dev, v) == 0)


def test_empty_m_is_noop(dev):
    case = inputs.make_case(1, 64, 16, seed=0)
    a = list(device_args(case, dev))
    a[0] = a[0][:0]
    out = ops.qswiglu_forward(*a)
    assert out.shape == (0, 16)


def test_leading_dims_are_flattened(dev, gemv_limit):
    case = inputs.make_case(6, 512, 96, seed=5)
    gemv_limit(0)
    a = list(device_args(case, dev))
    flat = to_bits(ops.qswiglu_forward(*a))
    a[0] = a[0].view(2, 3, 512)
    out = ops.qswiglu_forward(*a)
    assert out.shape == (2, 3, 96)
    assert np.array_equal(to_bits(out.reshape(6, 96)), flat)


# ------------------------------------------------------------ full sizes ----

def _sampled(case, dev, variant, rows, limit, gemv_limit):
    gemv_limit(limit)
    got = check_fused(case, dev, variant, rows=rows)
    rng = np.random.default_rng(123)
    pairs = np.stack([rng.integers(0, case.M, 64), rng.integers(0, case.I, 64)], axis=1)
    check_fused(case, dev, variant, pairs=pairs)
    return got


@pytest.mark.parametrize("kernel", SMALL_M_KERNELS, ids=lambda k: KNAMES[k])
@pytest.mark.parametrize("variant", [ops.MATCH, ops.F32], ids=["match", "f32"])
def test_full_decode(dev, gemv_limit, small_m_kernel, kernel, variant):
    case = inputs.workload_case("decode")
    small_m_kernel(kernel)
    before = ops.qsw_get_counters()
    _sampled(case, dev, variant, [0], 16, gemv_limit)
    expect_small_m(before, kernel, 1, ops.CNT_FUSED_GEMV)


@pytest.mark.parametrize("kernel", SMALL_M_KERNELS, ids=lambda k: KNAMES[k])
def test_decode_projection_rate(dev, gemv_limit, small_m_kernel, kernel):
    """The exact-projection rate at the decode workload, in the benchmark's
    launch configuration: every output of three x seeds (24,576 elements per
    projection), so the 99.9 % bar is enforced, not only reported."""
    gemv_limit(16)
    small_m_kernel(kernel)
    got = {ops.DEBUG_GATE: [], ops.DEBUG_UP: []}
    want = {ops.DEBUG_GATE: [], ops.DEBUG_UP: []}
    for seed in (0, 1, 2):
        case = inputs.workload_case("decode", seed=seed)
        a = device_args(case, dev)
        _, g64, u64 = oracle.qswiglu(*case.oracle_args(), variant=ops.MATCH, return_acc=True)
        for v, ref in ((ops.DEBUG_GATE, g64), (ops.DEBUG_UP, u64)):
            got[v].append(run_fused(case, dev, v, a))
            want[v].append(oracle.bf16_round_array(ref))
    for v in (ops.DEBUG_GATE, ops.DEBUG_UP):
        g, w = np.concatenate(got[v], axis=None), np.concatenate(want[v], axis=None)
        ok, info = check_projection(g, w)
        assert ok and g.size >= 20_000, info


def test_full_tiny_prefill(dev, gemv_limit):
    case = inputs.workload_case("tiny_prefill")
    for limit in (16, 0):
        _sampled(case, dev, ops.MATCH, list(range(6)), limit, gemv_limit)


def test_full_mid_prefill(dev, gemv_limit):
    case = inputs.workload_case("mid_prefill")
    _sampled(case, dev, ops.MATCH, [0, 1, 127, 128, 300, 511], 16, gemv_limit)


@pytest.mark.parametrize("variant", [ops.MATCH, ops.F32], ids=["match", "f32"])
def test_full_large_prefill(dev, gemv_limit, variant):
    case = inputs.workload_case("large_prefill")
    _sampled(case, dev, variant, [0, 1, 2047, 4095], 16, gemv_limit)


@pytest.mark.parametrize("M", inputs.MIXED_M_SWEEP)
def test_full_mixed_sweep(dev, gemv_limit, M):
    case = inputs.workload_case("mixed", M=M)
    rows = list(range(M)) if M <= 8 else [0, M // 2, M - 1]
    got = _sampled(case, dev, ops.MATCH, rows, 16, gemv_limit)
    if M <= 32:
        # the other kernel at the same M meets the same bound
        gemv_limit(0 if M <= 16 else 32)
        check_fused(case, dev, ops.MATCH, rows=rows)


@pytest.mark.parametrize("mode", [ops.STREAM_K_ALWAYS, ops.STREAM_K_AUTO], ids=["always", "auto"])
@pytest.mark.parametrize("seed", [0, 1])
def test_large_prefill_projection_rate(dev, gemv_limit, stream_k, mode, seed):
    """The exact-projection rate at H = 4096 (three accumulation chains per
    tile) on 8 rows that include the last row tile, whose tiles the ragged
    wave splits between SMs (stream-K): 114,688 values per projection."""
    case = inputs.workload_case("large_prefill", seed=seed)
    gemv_limit(0)
    stream_k(mode)
    rows = [0, 1, 2047, 2048, 3839, 3840, 4094, 4095]
    a = device_args(case, dev)
    _, g64, u64 = oracle.qswiglu(*case.oracle_args(), variant=ops.MATCH, rows=rows, return_acc=True)
    _, _, bnd_g, bnd_u = projection_context(case, "tensor_core", rows=rows)
    for v, ref, bnd in ((ops.DEBUG_GATE, g64, bnd_g), (ops.DEBUG_UP, u64, bnd_u)):
        got = run_fused(case, dev, v, a)[np.asarray(rows)]
        ok, info = check_projection(got, oracle.bf16_round_array(ref), exact=ref, bound=bnd)
        assert ok and got.size >= 100_000, info


@pytest.mark.parametrize("M", [16, 24, 32, 48, 128, 256])
def test_mixed_sweep_more_m(dev, gemv_limit, M):
    """The mixed-spec workload at the M values the benchmark adds around the
    small-M / tensor-core cut-over: both kernels where both apply (M <= 32)."""
    case = inputs.workload_case("mixed", M=M)
    rows = [0, M // 2, M - 1]
    _sampled(case, dev, ops.MATCH, rows, 32 if M <= 32 else 16, gemv_limit)
    if M <= 32:
        gemv_limit(0)
        check_fused(case, dev, ops.MATCH, rows=rows)


@pytest.fixture
def early_weights():
    saved = ops.qsw_get_early_weight_stream()
    yield ops.qsw_set_early_weight_stream
    ops.qsw_set_early_weight_stream(saved)


@pytest.mark.parametrize("kernel", SMALL_M_KERNELS, ids=lambda k: KNAMES[k])
@pytest.mark.parametrize("graph", [False, True], ids=["stream", "graph"])
def test_early_weight_stream_reads_previous_output(dev, gemv_limit, small_m_kernel, early_weights, kernel, graph):
    """With the early weight stream on, a small-M call may start while the call
    before it runs; it must still read x only after that call wrote it.  Three
    fused calls are chained (I == H, each call's hidden is the next call's x),
    on a stream and captured in a CUDA graph, and every output is checked
    against the oracle fed the GPU's own previous output."""
    gemv_limit(16)
    small_m_kernel(kernel)
    early_weights(True)
    cases = [inputs.make_case(2, 1024, 1024, seed=s, scale_range=(0.01, 0.03)) for s in (11, 12, 13)]
    args = [device_args(c, dev) for c in cases]
    x0 = args[0][0]
    outs = [torch.empty((2, 1024), dtype=torch.bfloat16, device=dev) for _ in cases]
    stream = torch.cuda.Stream(device=dev)

    def chain():
        x = x0
        for a, o in zip(args, outs):
            ops.qswiglu_forward(x, *a[1:], variant=ops.MATCH, out=o, stream=stream)
            x = o

    torch.cuda.synchronize()
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            chain()
        for o in outs:
            o.fill_(0)
        torch.cuda.synchronize()
        g.replay()
    else:
        with torch.cuda.stream(stream):
            chain()
    ops.qsw_check_device_errors(stream)
    x_bits = to_bits(x0)
    for c, o in zip(cases, outs):
        step = inputs.Case(x=x_bits, gate=c.gate, up=c.up)
        want = oracle.qswiglu(*step.oracle_args(), variant=oracle.MATCH)
        got = to_bits(o)
        ok, info = check_match(got, want)
        assert ok, info
        x_bits = got


# ------------------------------------------------------------- stream-K ----

@pytest.fixture
def stream_k():
    saved = ops.qsw_get_stream_k()
    yield ops.qsw_set_stream_k
    ops.qsw_set_stream_k(saved)


def _epoch(ws: torch.Tensor) -> int:
    """The launch counter the tensor-core kernel keeps at the start of the workspace."""
    torch.cuda.synchronize()
    return int(ws[:4].view(torch.int32).item())


# (M, H, I, bits_g, gs_g, bits_u, gs_u, rows): rows=None checks every row
SK_SHAPES = [
    # 48 tiles of 8 K steps; always-split spreads them over every SM, 2-4 CTAs
    # per tile, most ranges starting inside a scale entry
    (300, 512, 1536, 4, 64, 4, 64, None),
    # mixed specs, K tail of 32, ragged N
    (257, 2080, 384, 4, 32, 8, 32, None),
    # 2-bit gate, 8-bit up
    (64, 640, 136, 2, 64, 8, 64, None),
    # 158 tiles of 64 K steps on 152 SMs: 6 + 152 tiles split over 152 ranges of
    # ~66 K steps (three accumulation chains per range), one finisher per tile
    (300, 4096, 5000, 4, 64, 4, 64, [0, 1, 127, 128, 255, 256, 299]),
]


@pytest.mark.parametrize("shape", SK_SHAPES, ids=lambda s: "M{}_H{}_I{}_g{}x{}_u{}x{}".format(*s[:7]))
@pytest.mark.parametrize("mode", [ops.STREAM_K_OFF, ops.STREAM_K_ALWAYS], ids=["whole_tiles", "split"])
@pytest.mark.parametrize("variant", [ops.MATCH, ops.F32], ids=["match", "f32"])
def test_stream_k(dev, gemv_limit, stream_k, shape, mode, variant):
    """Split and whole-tile schedules of the tensor-core kernel both match the
    oracle; the workspace's launch counter shows which one ran."""
    M, H, I, bg, gg, bu, gu, rows = shape
    case = inputs.make_case(M, H, I, bits_g=bg, gs_g=gg, bits_u=bu, gs_u=gu, seed=M + I)
    gemv_limit(0)
    stream_k(mode)
    ws = ops.workspace(dev)
    e0 = _epoch(ws)
    check_fused(case, dev, variant, rows=rows)
    launches = 3 if variant == ops.MATCH else 1
    assert _epoch(ws) == e0 + (launches if mode == ops.STREAM_K_ALWAYS else 0)


@pytest.mark.parametrize("mode", [ops.STREAM_K_OFF, ops.STREAM_K_ALWAYS], ids=["whole_tiles", "split"])
def test_stream_k_affine_qmm(dev, gemv_limit, stream_k, mode):
    """The single-operand form (128 output columns per tile) under both schedules."""
    case = inputs.make_case(200, 1024, 1000, bits_g=4, gs_g=64, seed=5)
    gemv_limit(0)
    stream_k(mode)
    x, w, s, b, gs, bits = device_args(case, dev)[:6]
    got = to_bits(ops.affine_qmm(x, w, s, b, gs, bits))
    ops.qsw_check_device_errors()
    want = oracle.qmm(case.x, case.gate.packed, case.gate.scales, case.gate.biases, gs, bits)
    ok, info = check_projection(got, want)
    assert ok, info


def test_stream_k_graph_replays(dev, gemv_limit, stream_k):
    """Split calls captured in a CUDA graph: every replay launches them anew
    (the workspace's counter advances by one per call), and each replay's
    results match the oracle for the x it was given, so no replay reads
    partials a previous one left behind."""
    gemv_limit(0)
    stream_k(ops.STREAM_K_ALWAYS)
    base = inputs.make_case(300, 512, 1536, seed=31)
    a = device_args(base, dev)
    x_static = a[0].clone()
    outs = {v: torch.empty((300, 1536), dtype=torch.bfloat16, device=dev)
            for v in (ops.MATCH, ops.DEBUG_GATE, ops.DEBUG_UP)}
    stream = torch.cuda.Stream(device=dev)
    ws = ops.workspace(dev, stream)

    def calls():
        for v, o in outs.items():
            ops.qswiglu_forward(x_static, *a[1:], variant=v, out=o, stream=stream)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        calls()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        calls()
    torch.cuda.synchronize()
    for seed in (41, 42, 43):
        xb = inputs.make_x(300, 512, seed=seed)
        x_static.copy_(torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16))
        for o in outs.values():
            o.fill_(0)
        e0 = _epoch(ws)
        g.replay()
        ops.qsw_check_device_errors()
        assert _epoch(ws) == e0 + len(outs)
        step = inputs.Case(x=xb, gate=base.gate, up=base.up)
        h_ref, g64, u64 = oracle.qswiglu(*step.oracle_args(), variant=oracle.MATCH, return_acc=True)
        _, _, bnd_g, bnd_u = projection_context(step, "tensor_core")
        ok, info = check_match_with_projections(
            to_bits(outs[ops.MATCH]), to_bits(outs[ops.DEBUG_GATE]), to_bits(outs[ops.DEBUG_UP]), h_ref,
            oracle.bf16_round_array(g64), oracle.bf16_round_array(u64), match_epilogue,
            exact=(g64, u64), bounds=(bnd_g, bnd_u))
        assert ok, info


def test_workspace_size_is_checked(dev, gemv_limit):
    """A caller-owned workspace smaller than qsw_workspace_bytes() is refused."""
    case = inputs.make_case(130, 512, 200, seed=2)
    a = device_args(case, dev)
    need = ops.workspace_bytes(dev)
    assert need >= 128 * 1024 * torch.cuda.get_device_properties(dev).multi_processor_count
    small = torch.zeros(need - 1024, dtype=torch.uint8, device=dev)
    with pytest.raises(ops.QswError):
        ops.qswiglu_forward(*a, workspace=small)
    mine = torch.zeros(need, dtype=torch.uint8, device=dev)
    gemv_limit(0)
    got = to_bits(ops.qswiglu_forward(*a, variant=ops.F32, workspace=mine))
    ops.qsw_check_device_errors()
    ok, info = check_f32(got, oracle.qswiglu(*case.oracle_args(), variant=oracle.F32))
    assert ok, info


# ------------------------------------------------------ f16 activations ----

F16_TC_SHAPES = [
    (130, 512, 200, 4, 64, 4, 64),     # 2 M tiles, ragged N
    (257, 2080, 384, 4, 32, 8, 32),    # K tail, mixed specs
    (200, 640, 136, 2, 64, 8, 64),     # 2-bit gate, 8-bit up
]
F16_GEMV_SHAPES = [
    (1, 512, 8, 4, 64, 4, 64),
    (3, 512, 203, 4, 64, 4, 64),       # ragged last unit
    (4, 2304, 136, 8, 32, 4, 32),      # 8-bit gate
    (9, 1024, 48, 4, 128, 8, 32),      # two x row groups
]


@pytest.mark.parametrize("shape", F16_TC_SHAPES, ids=_ids(F16_TC_SHAPES))
@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: VNAMES[v])
def test_f16_tensor_core_kernel(dev, gemv_limit, shape, variant):
    """f16 activations (x, scales, biases, hidden) on the tensor-core kernel."""
    M, H, I, bg, gg, bu, gu = shape
    case = inputs.make_case(M, H, I, bits_g=bg, gs_g=gg, bits_u=bu, gs_u=gu, seed=M * 5 + H, dtype="f16")
    gemv_limit(0)
    before = ops.qsw_get_counters()[ops.CNT_FUSED_TC]
    got = check_fused(case, dev, variant)
    assert ops.qsw_get_counters()[ops.CNT_FUSED_TC] > before
    assert got.dtype == np.uint16


@pytest.mark.parametrize("kernel", SMALL_M_KERNELS, ids=lambda k: KNAMES[k])
@pytest.mark.parametrize("shape", F16_GEMV_SHAPES, ids=_ids(F16_GEMV_SHAPES))
@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: VNAMES[v])
def test_f16_small_m_kernel(dev, gemv_limit, small_m_kernel, kernel, shape, variant):
    M, H, I, bg, gg, bu, gu = shape
    case = inputs.make_case(M, H, I, bits_g=bg, gs_g=gg, bits_u=bu, gs_u=gu, seed=M * 3 + H, dtype="f16")
    gemv_limit(32)
    small_m_kernel(kernel)
    before = ops.qsw_get_counters()
    check_fused(case, dev, variant)
    expect_small_m(before, kernel, M, ops.CNT_FUSED_GEMV)


@pytest.mark.parametrize("limit", [0, 32], ids=["tensor_core", "small_m"])
@pytest.mark.parametrize("bits,gs", [(4, 64), (8, 32), (2, 64)])
def test_f16_affine_qmm(dev, gemv_limit, limit, bits, gs):
    M, K, N = (5, 1024, 300) if limit else (140, 640, 300)
    case = inputs.make_case(M, K, N, bits_g=bits, gs_g=gs, seed=bits + gs + 1, dtype="f16")
    gemv_limit(limit)
    x, w, s, b, _, _ = device_args(case, dev)[:6]
    y = ops.affine_qmm(x, w, s, b, gs, bits)
    assert y.dtype == torch.float16
    got = to_bits(y)
    ops.qsw_check_device_errors()
    want = oracle.qmm(case.x, case.gate.packed, case.gate.scales, case.gate.biases, gs, bits, dtype="f16")
    ok, info = check_projection(got, want, "f16")
    assert ok, info


def test_f16_all_gate_values(dev):
    """Every finite f16 gate value through the elementwise MATCH and F32 steps,
    and the paired (vector) and scalar (tail) forms bit for bit."""
    h = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    g = h[np.isfinite(h.view(np.float16))]
    n = (g.size // 8) * 8
    g = g[:n]
    u = inputs.f32_to_bits(torch.full((n,), 1.5), "f16")
    gd = inputs.bits_to_device(g, dev, "f16")
    ud = inputs.bits_to_device(u, dev, "f16")
    for variant, chk in ((ops.MATCH, check_match), (ops.F32, check_f32)):
        got = to_bits(ops.qsw_silu_mul(gd, ud, variant))
        ok, info = chk(got, oracle.silu_mul(g, u, variant, dtype="f16"), "f16")
        assert ok, info
    paired = to_bits(ops.qsw_silu_mul(gd, ud, ops.MATCH))
    scalar = np.zeros(n, dtype=np.uint16)
    out = torch.zeros_like(gd)
    for k in range(0, n - 7, 8):
        ops.qsw_silu_mul(gd[k:k + 7], ud[k:k + 7], ops.MATCH, out=out[k:k + 7])
    ops.qsw_check_device_errors()
    got7 = to_bits(out)
    mask = (np.arange(n) % 8) != 7
    assert np.array_equal(paired[mask], got7[mask])


@pytest.mark.parametrize("limit", [0, 32], ids=["tensor_core", "small_m"])
def test_f16_fused_match_equals_unfused(dev, gemv_limit, limit):
    case = inputs.make_case(24, 1024, 264, bits_g=4, gs_g=64, bits_u=8, gs_u=32, seed=4, dtype="f16")
    gemv_limit(limit)
    a = device_args(case, dev)
    fused = to_bits(ops.qswiglu_forward(*a, variant=ops.MATCH, workspace=None))
    unfused = to_bits(ops.unfused_swiglu(*a, variant=ops.MATCH, workspace=None))
    ops.qsw_check_device_errors()
    if limit == 0:
        assert np.array_equal(fused, unfused)
    else:
        ok, info = check_match(fused, unfused, "f16")
        assert ok, info


@pytest.mark.parametrize("mode", [ops.STREAM_K_OFF, ops.STREAM_K_ALWAYS], ids=["whole_tiles", "split"])
def test_f16_stream_k(dev, gemv_limit, stream_k, mode):
    case = inputs.make_case(300, 512, 1536, seed=77, dtype="f16")
    gemv_limit(0)
    stream_k(mode)
    check_fused(case, dev, ops.MATCH)


def test_f16_full_mid_prefill(dev, gemv_limit):
    """The mid-prefill shape with f16 activations, sampled rows, in the
    benchmark's launch configuration."""
    kw = dict(inputs.WORKLOADS["mid_prefill"])
    case = inputs.make_case(dtype="f16", seed=0, **kw)
    _sampled(case, dev, ops.MATCH, [0, 1, 127, 128, 300, 511], 16, gemv_limit)


def test_f16_full_decode(dev, gemv_limit):
    kw = dict(inputs.WORKLOADS["decode"])
    case = inputs.make_case(dtype="f16", seed=0, **kw)
    _sampled(case, dev, ops.MATCH, [0], 16, gemv_limit)


def test_plain_bf16_entry_points(dev, gemv_limit):
    """The fixed-signature entry points (bf16, no workspace) called directly
    through the C ABI."""
    lib = ops.load_library()
    case = inputs.make_case(40, 512, 136, seed=19)
    x, wg, sg, bg, gsg, btg, wu, su, bu, gsu, btu = device_args(case, dev)
    s = torch.cuda.current_stream().cuda_stream
    for limit in (0, 32):
        gemv_limit(limit)
        out = torch.empty((40, 136), dtype=torch.bfloat16, device=dev)
        assert lib.qswiglu_forward(x.data_ptr(), 40, 512, 136, wg.data_ptr(), sg.data_ptr(), bg.data_ptr(), gsg, btg,
                                   wu.data_ptr(), su.data_ptr(), bu.data_ptr(), gsu, btu, ops.F32, out.data_ptr(),
                                   s) == 0
        y = torch.empty((40, 136), dtype=torch.bfloat16, device=dev)
        assert lib.affine_qmm(x.data_ptr(), 40, 512, 136, wg.data_ptr(), sg.data_ptr(), bg.data_ptr(), gsg, btg,
                              y.data_ptr(), s) == 0
        ops.qsw_check_device_errors()
        ok, info = check_f32(to_bits(out), oracle.qswiglu(*case.oracle_args(), variant=oracle.F32))
        assert ok, info
        want = oracle.qmm(case.x, case.gate.packed, case.gate.scales, case.gate.biases, gsg, btg)
        ok, info = check_projection(to_bits(y), want)
        assert ok, info


# ---------------------------------------------- residual and whole MLP ----

def _mlp_inputs(M, H, I, Ho, dtype, seed):
    case = inputs.make_case(M, H, I, bits_g=4, gs_g=64, bits_u=8, gs_u=32, seed=seed, dtype=dtype)
    down = inputs.make_case(1, I, Ho, bits_g=4, gs_g=64, seed=seed + 1, dtype=dtype).gate
    h = inputs.make_x(M, Ho, seed=seed + 2, dtype=dtype)
    return case, down, h


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("limit", [0, 32], ids=["tensor_core", "small_m"])
def test_affine_qmm_residual(dev, gemv_limit, dtype, limit):
    """y = T(x . W^T + r): the residual joins the f32 accumulator before the
    one rounding, also when y is r itself."""
    M, K, N = (5, 1024, 300) if limit else (140, 640, 300)
    case = inputs.make_case(M, K, N, bits_g=4, gs_g=64, seed=71, dtype=dtype)
    r = inputs.make_x(M, N, seed=72, x_std=3.0, dtype=dtype)
    gemv_limit(limit)
    x, w, s, b, gs, bits = device_args(case, dev)[:6]
    rd = inputs.bits_to_device(r, dev, dtype)
    got = to_bits(ops.affine_qmm(x, w, s, b, gs, bits, residual=rd))
    inplace = rd.clone()
    ops.affine_qmm(x, w, s, b, gs, bits, y=inplace, residual=inplace)
    ops.qsw_check_device_errors()
    want = oracle.qmm(case.x, case.gate.packed, case.gate.scales, case.gate.biases, gs, bits, dtype=dtype,
                      residual=r)
    ok, info = check_projection(got, want, dtype)
    assert ok, info
    assert np.array_equal(to_bits(inplace), got)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("limit", [0, 32], ids=["tensor_core", "small_m"])
@pytest.mark.parametrize("variant", [ops.MATCH, ops.F32], ids=["match", "f32"])
def test_mlp_forward(dev, gemv_limit, dtype, limit, variant):
    """The whole block: hidden is exactly the fused expansion's output, and y
    is the down projection of that hidden plus the residual (checked against
    the oracle fed the GPU's hidden, and end to end against the oracle's block)."""
    M = 5 if limit else 130
    case, down, h = _mlp_inputs(M, 512, 256, 200, dtype, 31)
    gemv_limit(limit)
    a = device_args(case, dev)
    d = inputs.operand_to_device(down, dev, dtype)
    hd = inputs.bits_to_device(h, dev, dtype)
    hidden = torch.empty((M, 256), dtype=inputs.TORCH_DTYPES[dtype], device=dev)
    y = to_bits(ops.mlp_forward(a[0], hd, *a[1:], *d, variant=variant, hidden=hidden))
    fused = to_bits(ops.qswiglu_forward(*a, variant=variant))
    ops.qsw_check_device_errors()
    hid = to_bits(hidden)
    assert np.array_equal(hid, fused)
    want = oracle.qmm(hid, down.packed, down.scales, down.biases, down.gs, down.bits, dtype=dtype, residual=h)
    ok, info = check_projection(y, want, dtype)
    assert ok, info
    y_ref, _ = oracle.mlp(case.x, h, *case.oracle_args()[1:], down.packed, down.scales, down.biases, down.gs,
                          down.bits, variant=variant, dtype=dtype)
    yg, yr = TO_F64[dtype](y), TO_F64[dtype](y_ref)
    assert np.linalg.norm(yg - yr) <= 1e-2 * np.linalg.norm(yr)


def test_mlp_forward_in_place_and_no_residual(dev, gemv_limit):
    case, down, h = _mlp_inputs(40, 512, 128, 96, "bf16", 41)
    gemv_limit(0)
    a = device_args(case, dev)
    d = inputs.operand_to_device(down, dev)
    hd = inputs.bits_to_device(h, dev)
    ref = to_bits(ops.mlp_forward(a[0], hd, *a[1:], *d))
    inplace = hd.clone()
    ops.mlp_forward(a[0], inplace, *a[1:], *d, out=inplace)
    none = to_bits(ops.mlp_forward(a[0], None, *a[1:], *d))
    ops.qsw_check_device_errors()
    assert np.array_equal(to_bits(inplace), ref)
    hid = to_bits(ops.qswiglu_forward(*a))
    want = oracle.qmm(hid, down.packed, down.scales, down.biases, down.gs, down.bits)
    ok, info = check_projection(none, want)
    assert ok, info


def test_full_mlp_decode(dev, gemv_limit):
    """The decode shape as a whole block: H = Ho = 2048, I = 8192, 4-bit gs 64."""
    case = inputs.workload_case("decode")
    down = inputs.make_case(1, 8192, 2048, bits_g=4, gs_g=64, seed=5).gate
    h = inputs.make_x(1, 2048, seed=6)
    gemv_limit(16)
    a = device_args(case, dev)
    d = inputs.operand_to_device(down, dev)
    hidden = torch.empty((1, 8192), dtype=torch.bfloat16, device=dev)
    y = to_bits(ops.mlp_forward(a[0], inputs.bits_to_device(h, dev), *a[1:], *d, hidden=hidden))
    ops.qsw_check_device_errors()
    want = oracle.qmm(to_bits(hidden), down.packed, down.scales, down.biases, 64, 4, residual=h)
    ok, info = check_projection(y, want)
    assert ok, info


@pytest.mark.parametrize("M", [1, 2])
def test_small_m_large_k_single_operand(dev, gemv_limit, M):
    """The decode-size down projection (K = 8192, N = 2048) runs on the small-M
    kernel: x is staged with its real rows only and units are 8 rows."""
    case = inputs.make_case(M, 8192, 2048, bits_g=4, gs_g=64, seed=90 + M)
    gemv_limit(16)
    x, w, s, b, gs, bits = device_args(case, dev)[:6]
    before = ops.qsw_get_counters()[ops.CNT_QMM_GEMV]
    got = to_bits(ops.affine_qmm(x, w, s, b, gs, bits))
    ops.qsw_check_device_errors()
    assert ops.qsw_get_counters()[ops.CNT_QMM_GEMV] == before + 1
    want = oracle.qmm(case.x, case.gate.packed, case.gate.scales, case.gate.biases, gs, bits)
    ok, info = check_projection(got, want)
    assert ok, info
