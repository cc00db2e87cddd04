// Small-M kernel for the quantised SwiGLU expansion (decode, M <= 32) and for
// the single quantised linear at small M.
//
// Method: mlx-bun pages, src/model/fused-swiglu-kernel.ts -- at decode the two
// projections are memory-bound GEMVs and "reading Wg/Wu dominates".  The design
// streams the packed rows from HBM exactly once, as early and as deep as
// possible, and keeps everything but the dequantisation off the critical path:
//
//  * unit of work: 8 output rows (fused: rows r..r+7 of Wg AND of Wu; single
//    linear: rows r..r+7 of W, A rows 8..15 of the MMA left zero, so that a
//    unit stays small at large K).  One persistent CTA per SM takes units
//    round-robin.
//  * a unit's rows are contiguous in HBM: ONE 1-D bulk (TMA) copy per array
//    (codes of each operand, each scale and bias array) lands it in a
//    shared-memory ring slot, completing on the slot's mbarrier.  At kernel
//    start every slot is in flight, so each SM requests its share at once.
//  * the 16 warps form 4 groups of 4; group q takes the CTA's units q, q+4, ...
//    and its 4 warps split K in 128-code blocks, so every warp does several
//    blocks per unit and the per-unit bookkeeping stays small.  Where every
//    unit of a CTA fits in its slots at once (decode: 7 units per CTA), the
//    warps form 8 groups of 2 instead: one unit per group, so no group works
//    through two units in turn.  One warp of the
//    group adds the 4 partial sums in a fixed order and applies the epilogue.
//  * x is the same for every unit: it is staged once per CTA in shared memory,
//    already permuted into MMA B-fragment order (bank-conflict-free reads);
//    only its M real rows are stored (the padding rows of the 8-row fragment
//    are zeros made at the read), so K = 8192 fits at small M.
//  * a lane (g = lane/4, c = lane%4) dequantises 32 codes of gate row g and of
//    up row g to the activation dtype T (bf16 or f16) in registers
//    (w = T(s*q + b), one rounding) and feeds
//    them as A rows g and g+8 of mma.sync m16n8k16 with x (8 rows, zero padded)
//    as B: one MMA yields gate and up of the same outputs.  The K order inside
//    each 8-code group is interleaved (codes j, j+4); x is permuted the same way.
//  * each 128-code block accumulates in a fresh fragment that is then added to
//    the warp's running f32 sum (short tensor-core accumulation chains).
//
// Every wait is bounded; on a timeout the CTA raises an abort flag, lets its
// own copies land and returns, and the host reads the device error word.
#include <atomic>

#include "qsw_internal.h"
#include "qsw_smallm.cuh"

namespace qsw {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kWideGroup = 4;                   // warps sharing one unit (default)
constexpr int kNarrowGroup = 2;                 // ... when every unit of a CTA fits in its slots at once
constexpr int kBlockK = kSmallBlockK;           // codes per K block
constexpr int kChunk = kSmallChunk;             // codes per lane per block
constexpr int kSmemBudget = 200 * 1024;
constexpr int kMaxSlots = 16;
constexpr int kXBlockBytes = 4 * 32 * 16;       // B fragments of one block, one full x row group (2 KB)
constexpr int kXPre = 4;                        // x pieces per thread requested ahead of the weights

__device__ unsigned int g_gemv_error;

struct GemvParams {
  const uint16_t *x;
  int M, K, N;
  const uint32_t *w0, *w1;
  const uint16_t *s0, *b0, *s1, *b1;
  GroupDiv gd0, gd1;
  uint32_t ng0, ng1;      // groups per row (K / gs)
  int x_rows;             // x rows staged per row group: min(8, M) (the others are zero fragments)
  int variant;
  uint16_t *out;
  const uint16_t *res;    // single-operand form: [M, N] added before the rounding (or null)
  int units, slots;
  int pitch0, pitch1;     // packed bytes per row of operand 0 / 1
  int sb_off;             // byte offset of the scale/bias rows inside a slot
  int slot_bytes;
  int x_off;              // byte offset of the staged x fragments
  int red_off;            // byte offset of the partial sums
  int bar_off;            // byte offset of the barriers
  int early;              // launched as a programmatic dependent (early weight stream)
  int withhold;           // test only: the first fill of slot 0 is never issued (1) or as usual (0)
  uint64_t timeout_ns;
};

// Issue the bulk copies of unit u into a slot (lanes 0..5 of the calling warp).
template <int BITS0, int BB, bool DUAL>
__device__ __forceinline__ void issue_unit(const GemvParams &p, uint8_t *base, uint64_t *bar, unsigned int *issued,
                                           int u, int lane) {
  constexpr int R = 8;
  const uint32_t r0 = static_cast<uint32_t>(u) * R;
  const uint32_t rows = static_cast<uint32_t>(p.N) - r0 < static_cast<uint32_t>(R) ? static_cast<uint32_t>(p.N) - r0
                                                                                     : static_cast<uint32_t>(R);
  const uint32_t sb0 = R * p.ng0 * 2, sb1 = DUAL ? R * p.ng1 * 2 : 0;   // bytes of one s/b array region
  if (lane == 0) {
    debug_check(r0 + rows <= static_cast<uint32_t>(p.N) && rows >= 1, &g_gemv_error);
    debug_check(p.sb_off + 2 * sb0 + 2 * sb1 <= static_cast<uint32_t>(p.slot_bytes), &g_gemv_error);
    const uint32_t bytes = rows * (p.pitch0 + (DUAL ? p.pitch1 : 0)) + rows * 4 * (p.ng0 + (DUAL ? p.ng1 : 0));
    mbar_arrive_expect_tx(bar, bytes);
    *issued += 1;   // fills of this slot so far (for draining after an abort)
  }
  __syncwarp();
  if (lane == 0)
    bulk_copy_g2s(base, p.w0 + static_cast<int64_t>(r0) * (p.pitch0 / 4), rows * p.pitch0, bar);
  if (DUAL && lane == 1)
    bulk_copy_g2s(base + R * p.pitch0, p.w1 + static_cast<int64_t>(r0) * (p.pitch1 / 4), rows * p.pitch1, bar);
  if (lane >= 2 && lane < (DUAL ? 6 : 4)) {
    const int arr = lane - 2;   // s0, b0, s1, b1
    const uint16_t *src = arr == 0 ? p.s0 : arr == 1 ? p.b0 : arr == 2 ? p.s1 : p.b1;
    const uint32_t ng = arr < 2 ? p.ng0 : p.ng1;
    const uint32_t region = arr < 2 ? arr * sb0 : 2 * sb0 + (arr - 2) * sb1;
    bulk_copy_g2s(base + p.sb_off + region, src + static_cast<int64_t>(r0) * ng, rows * ng * 2, bar);
  }
}

template <int BITS0, int BITS1, bool DUAL, int NG, int GW, class A>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const GemvParams p) {
  constexpr int kGroupWarps = GW;                 // warps sharing one unit
  constexpr int kGroups = kWarps / kGroupWarps;   // units in progress per CTA
  constexpr int R = 8;                      // output rows per unit
  constexpr int BB = DUAL ? BITS1 : BITS0;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.bar_off);               // [kMaxSlots]
  uint64_t *red_full = full + kMaxSlots;                                          // [kGroups][2]
  uint64_t *red_free = red_full + 2 * kGroups;                                    // [kGroups][2]
  uint64_t *x_ready = red_free + 2 * kGroups;                                     // x staged
  uint64_t *x_requested = x_ready + 1;                                            // x loads issued
  unsigned int *done_cnt = reinterpret_cast<unsigned int *>(x_requested + 1);     // [kMaxSlots]
  unsigned int *issued_cnt = done_cnt + kMaxSlots;                                     // [kMaxSlots]
  volatile int *abort_flag = reinterpret_cast<volatile int *>(issued_cnt + kMaxSlots);
  float *red = reinterpret_cast<float *>(smem + p.red_off);   // [kGroups][2][kGroupWarps][NG][32][4]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned int *err = &g_gemv_error;
  const uint32_t K = static_cast<uint32_t>(p.K);
  const uint32_t nkb = (K + kBlockK - 1) / kBlockK;
  const int my_units = (p.units - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                       static_cast<int>(gridDim.x);
  auto unit_of = [&](int i) { return static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x); };

  if constexpr (kDebugBounds) {
    debug_poison_smem(smem, static_cast<uint32_t>(p.bar_off));   // slots, x, partial sums
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.slots; ++s) {
      mbar_init(&full[s], 1);
      done_cnt[s] = 0;
      issued_cnt[s] = 0;
    }
    for (int b = 0; b < 2 * kGroups; ++b) {
      mbar_init(&red_full[b], kGroupWarps);
      mbar_init(&red_free[b], 1);
    }
    mbar_init(x_ready, kWarps - 1);
    mbar_init(x_requested, kWarps - 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // x -> shared memory in B-fragment order, once per CTA: for block kb, x row
  // group G, fragment word q (0..15) of lane L = 4n + c sits at
  // ((kb*NG + G)*4 + q/4)*512 + L*16 + (q%4)*4 bytes.  Every staging thread
  // requests its first pieces of x BEFORE the weight copies are issued: behind
  // the weight stream of all SMs, x would only arrive microseconds later.  The
  // last warp issues the copies and stages no x: issuing stalls while the copy
  // engine is saturated, and no other warp should wait for that.
  // Only the lanes of real x rows are staged: lane L = 4n + c carries row n
  // of a group, so rows n >= x_rows (padding when M < 8) are zero fragments
  // synthesised at the read, and a block of one group takes x_rows * 64 bytes.
  const int x_lanes = 4 * p.x_rows;                        // staged lanes per (block, group)
  const uint32_t x_piece = static_cast<uint32_t>(p.x_rows) * 64;   // bytes per (block, group, j)
  const int x_total = static_cast<int>(nkb) * NG * x_lanes;   // (kb, G, lane) triples
  auto load_x = [&](int e, uint4 (&xv)[4]) {
    const int L = e % x_lanes, G = (e / x_lanes) % NG, kb = (e / x_lanes) / NG;
    const int m = 8 * G + (L >> 2);
    const uint32_t k = static_cast<uint32_t>(kb) * kBlockK + (L & 3) * kChunk;
    if (k < K && m < p.M) {
      const uint4 *xp = reinterpret_cast<const uint4 *>(p.x + static_cast<int64_t>(m) * p.K + k);
#pragma unroll
      for (int q = 0; q < 4; ++q) xv[q] = __ldg(xp + q);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) xv[q] = make_uint4(0, 0, 0, 0);
    }
  };
  auto store_x = [&](int e, const uint4 (&xv)[4]) {
    const int L = e % x_lanes, G = (e / x_lanes) % NG, kb = (e / x_lanes) / NG;
    uint8_t *dst = smem + p.x_off + static_cast<size_t>(kb * NG + G) * 4 * x_piece + L * 16;
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // x values 8j..8j+7: (x0,x1) (x2,x3) (x4,x5) (x6,x7)
      *reinterpret_cast<uint4 *>(dst + j * x_piece) = x_fragment(xv[j]);
    }
  };
  constexpr int kStageThreads = kThreads - 32;
  const bool stager = static_cast<int>(threadIdx.x) < kStageThreads;
  // Each group owns `spg` slots and uses them in turn, so a slot only ever
  // holds the units of one group, in order (a waiter is never more than one
  // fill ahead of its slot).  The last warp puts the first units of every slot
  // in flight, every group's first unit first; later fills are issued by the
  // group's warp that finishes last.
  const int spg = p.slots / kGroups;
  auto issue_round = [&](int s) {
    for (int q = 0; q < kGroups; ++q) {
      const int i = q + s * kGroups;
      // (the test hook leaves slot 0 without its first fill: waits on it run out)
      if (i < my_units && !(p.withhold && i == 0))
        issue_unit<BITS0, BB, DUAL>(p, smem + (q * spg + s) * p.slot_bytes, &full[q * spg + s],
                                    &issued_cnt[q * spg + s], unit_of(i), lane);
    }
  };
  uint4 x_pre[kXPre][4];
  auto preload_x = [&]() {
#pragma unroll
    for (int r = 0; r < kXPre; ++r)
      if (stager && static_cast<int>(threadIdx.x) + r * kStageThreads < x_total)
        load_x(threadIdx.x + r * kStageThreads, x_pre[r]);
  };
  int first_round = 0;
  if (p.early) {
    // Programmatic dependent launch: the next call may be scheduled as soon as
    // every CTA of this one has got here.  Weights are not written by earlier
    // work on the stream (caller's guarantee), so the first unit of every group
    // is requested before waiting for that work; x is read only after it.
    if (threadIdx.x == 0) griddep_launch_dependents();
    __syncthreads();
    if (!stager) issue_round(0);
    first_round = 1;
    // Start x's way into L2 while that work finishes (a cold x would otherwise
    // be read from HBM behind the weight stream, after the wait).  A prefetch
    // changes no value: if that work is still writing x, its writes land in
    // L2 all the same, and x is read only after the wait.
    if (warp == 0 && lane < p.M) prefetch_l2_bulk(p.x + static_cast<int64_t>(lane) * p.K, static_cast<uint32_t>(p.K) * 2);
    griddep_wait();
    preload_x();
    if (stager) {
      __syncwarp();
      if (lane == 0) mbar_arrive(x_requested);   // this warp's x loads are in flight
    } else if (!warp_wait(x_requested, 0, abort_flag, p.timeout_ns, err)) {
      first_round = spg;   // give up issuing; the waits below time out the same way
    }
  } else {
    preload_x();
    __syncthreads();
  }
  if (!stager) {
    for (int s = first_round; s < spg; ++s) issue_round(s);
  } else {
#pragma unroll
    for (int r = 0; r < kXPre; ++r)
      if (static_cast<int>(threadIdx.x) + r * kStageThreads < x_total)
        store_x(threadIdx.x + r * kStageThreads, x_pre[r]);
    for (int e = threadIdx.x + kXPre * kStageThreads; e < x_total; e += kStageThreads) {
      uint4 xv[4];
      load_x(e, xv);
      store_x(e, xv);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(x_ready);
  }
  const bool x_ok = warp_wait_lazy(x_ready, 0, abort_flag, p.timeout_ns, err, 2000);

  const int grp = warp / kGroupWarps, gw = warp % kGroupWarps;
  const int g = lane >> 2, c = lane & 3;
  const uint32_t sb0 = R * p.ng0 * 2, sb1 = DUAL ? R * p.ng1 * 2 : 0;
  // lanes past the staged rows read lane 0's piece and zero it (rows >= M)
  const bool x_live = lane < x_lanes;
  const uint32_t xbase = smem_u32(smem + p.x_off) + (x_live ? lane : 0) * 16;
  for (int ig = 0; x_ok; ++ig) {
    const int i = grp + ig * kGroups;
    if (i >= my_units) break;
    const int slot = grp * spg + ig % spg, round = ig / spg;
    if (!warp_wait_lazy(&full[slot], round & 1, abort_flag, p.timeout_ns, err, 2000)) break;
    const uint32_t base = smem_u32(smem + slot * p.slot_bytes);
    // A rows g (gate, or the single operand) and g+8 (up; zero in the
    // single-operand form, whose units are 8 rows of one matrix)
    const int ga = g, gb = g;
    const uint32_t rowa = base + ga * p.pitch0 + c * (kChunk * BITS0 / 8);
    const uint32_t rowb = base + R * p.pitch0 + gb * p.pitch1 + c * (kChunk * BB / 8);
    const uint32_t sbase = base + p.sb_off;
    const uint32_t s_a = sbase + ga * p.ng0 * 2, b_a = s_a + sb0;
    const uint32_t s_b = sbase + 2 * sb0 + gb * p.ng1 * 2;
    const uint32_t b_b = s_b + sb1;
    float sum[NG][4];
#pragma unroll
    for (int G = 0; G < NG; ++G)
#pragma unroll
      for (int q = 0; q < 4; ++q) sum[G][q] = 0.0f;

#pragma unroll 1
    for (uint32_t kb = gw; kb < nkb; kb += kGroupWarps) {
      // kb is warp-uniform; past K (only in the last block) the codes are
      // replaced by zeros, and every lane runs the MMAs
      const uint32_t k = kb * kBlockK + c * kChunk;
      const bool kval = k < K;
      Chunk<BITS0, A> ca;
      Chunk<BB, A> cb;
      uint32_t sa = 0, ba = 0, sb = 0, bb = 0;
      if (kval) {
        debug_check((kb * kBlockK + (c + 1) * kChunk) * BITS0 / 8 <= static_cast<uint32_t>(p.pitch0) &&
                        (!DUAL || (kb * kBlockK + (c + 1) * kChunk) * BB / 8 <= static_cast<uint32_t>(p.pitch1)) &&
                        p.gd0(k) < p.ng0 && (!DUAL || p.gd1(k) < p.ng1),
                    err);
        ca.load(rowa + kb * (kBlockK * BITS0 / 8));
        const uint32_t ia = p.gd0(k) * 2;
        sa = lds_u16(s_a + ia);
        ba = lds_u16(b_a + ia);
        if (DUAL) {
          cb.load(rowb + kb * (kBlockK * BB / 8));
          const uint32_t ib = p.gd1(k) * 2;
          sb = lds_u16(s_b + ib);
          bb = lds_u16(b_b + ib);
        } else {
#pragma unroll
          for (int q = 0; q < Chunk<BB, A>::kWords; ++q) cb.w[q] = 0;
        }
      } else {
#pragma unroll
        for (int q = 0; q < Chunk<BITS0, A>::kWords; ++q) ca.w[q] = 0;
#pragma unroll
        for (int q = 0; q < Chunk<BB, A>::kWords; ++q) cb.w[q] = 0;
      }
      __syncwarp();
      const uint32_t sa2 = splat_bf16(static_cast<uint16_t>(sa)), ba2 = splat_bf16(static_cast<uint16_t>(ba));
      const uint32_t sb2 = splat_bf16(static_cast<uint16_t>(sb)), bb2 = splat_bf16(static_cast<uint16_t>(bb));
      float acc[NG][4];
#pragma unroll
      for (int G = 0; G < NG; ++G)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[G][q] = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t pa[4], pb[4] = {0u, 0u, 0u, 0u};
        ca.dequant(j, sa2, ba2, pa);
        if (DUAL) cb.dequant(j, sb2, bb2, pb);
#pragma unroll
        for (int G = 0; G < NG; ++G) {
          uint4 xf = lds128(xbase + ((kb * NG + G) * 4 + j) * x_piece);
          if (!x_live) xf = make_uint4(0u, 0u, 0u, 0u);
          // A rows g (operand a) and g+8 (operand b); k_local 2c,2c+1 <- pair 2h,
          // k_local 2c+8,2c+9 <- pair 2h+1
          const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
          const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
          mma_16816<A>(acc[G], a0, xf.x, xf.y);
          mma_16816<A>(acc[G], a1, xf.z, xf.w);
        }
      }
#pragma unroll
      for (int G = 0; G < NG; ++G)
#pragma unroll
        for (int q = 0; q < 4; ++q) sum[G][q] += acc[G][q];
    }

    // Done with the slot: the last of all warps of the group to get here
    // refills it with the unit `slots` further on.  Every read of the slot is
    // ordered before that warp's counter increment; its copies after it, behind
    // a proxy fence (generic reads before async-proxy writes).
    __syncwarp();
    unsigned int prev = 0;
    if (lane == 0) {
      __threadfence_block();
      prev = atomicAdd(&done_cnt[slot], 1u);
      __threadfence_block();
    }
    prev = __shfl_sync(0xffffffffu, prev, 0);
    if (prev == kGroupWarps - 1) {
      if (lane == 0) done_cnt[slot] = 0;
      fence_proxy_async_smem();
      const int i_next = i + spg * kGroups;   // this group's next unit for the slot
      if (i_next < my_units)
        issue_unit<BITS0, BB, DUAL>(p, smem + slot * p.slot_bytes, &full[slot], &issued_cnt[slot],
                                    unit_of(i_next), lane);
    }

    // partial sums of the group -> one warp reduces them in a fixed order
    const int buf = ig & 1;
    const uint32_t use = static_cast<uint32_t>(ig >> 1);
    uint64_t *rf = &red_full[grp * 2 + buf], *rfree = &red_free[grp * 2 + buf];
    if (use > 0 && !warp_wait_lazy(rfree, (use - 1) & 1, abort_flag, p.timeout_ns, err, 2000)) break;
    float *rb = red + ((grp * 2 + buf) * kGroupWarps) * NG * 128;
#pragma unroll
    for (int G = 0; G < NG; ++G)
      *reinterpret_cast<float4 *>(rb + ((gw * NG + G) * 32 + lane) * 4) =
          make_float4(sum[G][0], sum[G][1], sum[G][2], sum[G][3]);
    __syncwarp();
    if (lane == 0) mbar_arrive(rf);
    if (gw == 0) {
      if (!warp_wait_lazy(rf, use & 1, abort_flag, p.timeout_ns, err, 2000)) break;
      const int64_t r0 = static_cast<int64_t>(unit_of(i)) * R;
      for (int e = lane; e < R * NG * 8; e += 32) {
        const int G = e / (R * 8), rem = e % (R * 8);
        const int row = rem / 8, n = rem % 8;
        const int m = 8 * G + n;
        const int64_t i_out = r0 + row;
        if (m >= p.M || i_out >= p.N) continue;
        // accumulator element of (A row a, x col n): lane 4*(a % 8) + n/2,
        // register (n & 1) + 2*(a >= 8).  Gate (or the single operand) is A
        // row `row`; in the fused form up is A row row+8.
        const int l = 4 * (row & 7) + (n >> 1);
        const int qa = (n & 1) + ((row >= 8) ? 2 : 0);
        float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
        for (int w = 0; w < kGroupWarps; ++w) {
          const float *rw = rb + ((w * NG + G) * 32 + l) * 4;
          s0 += rw[qa];
          if (DUAL) s1 += rw[(n & 1) + 2];
        }
        const int64_t o = static_cast<int64_t>(m) * p.N + i_out;
        const float v = DUAL ? swiglu_epilogue<A>(p.variant, s0, s1) : (p.res ? s0 + A::lo(p.res[o]) : s0);
        p.out[o] = A::store(v);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(rfree);
    }
  }

  // After an abort, let every copy this CTA issued land before it exits.
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    for (int s = 0; s < p.slots; ++s)
      if (issued_cnt[s] > 0) mbar_wait_drain(&full[s], (issued_cnt[s] - 1) & 1, 100000000ull);
  }
}

struct Layout {
  int slot_bytes, sb_off, x_off, red_off, bar_off, total, slots;
  int group_warps;   // warps sharing one unit
};

// Shared-memory layout for the given shape; slots == 0 when it does not fit.
Layout plan(int64_t K, int64_t N, int M, int gs0, int gs1, int bits0, int bits1, bool dual, int num_sms,
            int group_warps = kWideGroup) {
  const int64_t R = 8;
  const int64_t kGroupWarps = group_warps, kGroups = kWarps / group_warps;
  const int NG = M <= 8 ? 1 : M <= 16 ? 2 : 4;
  const int64_t pitch0 = K * bits0 / 8, pitch1 = dual ? K * bits1 / 8 : 0;
  const int64_t ng = K / gs0 + (dual ? K / gs1 : 0);
  Layout l{};
  l.sb_off = static_cast<int>(R * (pitch0 + pitch1));
  l.slot_bytes = static_cast<int>((l.sb_off + R * 4 * ng + 127) / 128 * 128);
  const int64_t nkb = (K + kBlockK - 1) / kBlockK;
  const int64_t x_rows = M < 8 ? M : 8;
  const int64_t x_bytes = nkb * NG * kXBlockBytes * x_rows / 8;
  const int64_t red_bytes = static_cast<int64_t>(kGroups) * 2 * kGroupWarps * NG * 128 * 4;
  const int64_t bar_bytes = (kMaxSlots + 4 * kGroups + 2) * 8 + 2 * kMaxSlots * 4 + 16;
  const int64_t fixed = x_bytes + red_bytes + bar_bytes;
  const int64_t units = (N + R - 1) / R;
  const int64_t grid = units < num_sms ? units : num_sms;
  const int64_t per_cta = (units + grid - 1) / grid;
  // slots per group: what fits, at most what one group can use
  int64_t spg = (kSmemBudget - fixed) / l.slot_bytes / kGroups;
  const int64_t per_group = (per_cta + kGroups - 1) / kGroups;
  if (spg > kMaxSlots / kGroups) spg = kMaxSlots / kGroups;
  if (spg > per_group) spg = per_group;
  if (spg < 1) return Layout{};
  const int64_t slots = spg * kGroups;
  l.slots = static_cast<int>(slots);
  l.group_warps = group_warps;
  l.x_off = static_cast<int>(slots * l.slot_bytes);
  l.red_off = static_cast<int>(l.x_off + x_bytes);
  l.bar_off = static_cast<int>(l.red_off + red_bytes);
  l.total = static_cast<int>(l.bar_off + bar_bytes);
  return l;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <int BITS0, int BITS1, bool DUAL, int NG, int GW, class A>
cudaError_t launch_cfg(GemvParams p, const Layout &l, cudaStream_t stream, int num_sms) {
  constexpr int R = 8;
  p.pitch0 = p.K * BITS0 / 8;
  p.pitch1 = DUAL ? p.K * BITS1 / 8 : 0;
  p.units = (p.N + R - 1) / R;
  p.slots = l.slots;
  p.slot_bytes = l.slot_bytes;
  p.sb_off = l.sb_off;
  p.x_off = l.x_off;
  p.red_off = l.red_off;
  p.bar_off = l.bar_off;
  const int grid = p.units < num_sms ? p.units : num_sms;
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(attr_done.load() & (uint64_t(1) << dev))) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<BITS0, BITS1, DUAL, NG, GW, A>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(uint64_t(1) << dev);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = l.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.early ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_kernel<BITS0, BITS1, DUAL, NG, GW, A>, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int BITS0, int BITS1, bool DUAL, class A>
cudaError_t launch_ng(const GemvParams &p, const Layout &l, cudaStream_t stream, int num_sms) {
  if (p.M <= 8) {
    if (l.group_warps == kNarrowGroup) return launch_cfg<BITS0, BITS1, DUAL, 1, kNarrowGroup, A>(p, l, stream, num_sms);
    return launch_cfg<BITS0, BITS1, DUAL, 1, kWideGroup, A>(p, l, stream, num_sms);
  }
  if (p.M <= 16) return launch_cfg<BITS0, BITS1, DUAL, 2, kWideGroup, A>(p, l, stream, num_sms);
  return launch_cfg<BITS0, BITS1, DUAL, 4, kWideGroup, A>(p, l, stream, num_sms);
}

template <int BITS0, class A>
cudaError_t launch_dual_bits1(const GemvParams &p, const Layout &l, int bits1, cudaStream_t stream, int num_sms) {
  switch (bits1) {
    case 2: return launch_ng<BITS0, 2, true, A>(p, l, stream, num_sms);
    case 4: return launch_ng<BITS0, 4, true, A>(p, l, stream, num_sms);
    case 8: return launch_ng<BITS0, 8, true, A>(p, l, stream, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

template <class A>
cudaError_t launch_act(const GemvParams &p, const Layout &l, int bits0, int bits1, bool dual, cudaStream_t stream,
                       int num_sms) {
  if (dual) {
    switch (bits0) {
      case 2: return launch_dual_bits1<2, A>(p, l, bits1, stream, num_sms);
      case 4: return launch_dual_bits1<4, A>(p, l, bits1, stream, num_sms);
      case 8: return launch_dual_bits1<8, A>(p, l, bits1, stream, num_sms);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (bits0) {
    case 2: return launch_ng<2, 2, false, A>(p, l, stream, num_sms);
    case 4: return launch_ng<4, 4, false, A>(p, l, stream, num_sms);
    case 8: return launch_ng<8, 8, false, A>(p, l, stream, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

std::atomic<int> g_withhold{0};

}  // namespace

void gemv_withhold_next() { g_withhold.store(1); }

bool gemv_fits(int64_t M, int64_t K, int64_t N, const QuantOperand &op0, const QuantOperand *op1, int num_sms) {
  const bool dual = op1 != nullptr;
  const QuantOperand &o1 = dual ? *op1 : op0;
  // scale/bias rows of a unit are staged by 16-byte bulk copies
  if ((K / op0.gs) % 8 != 0 || (dual && (K / o1.gs) % 8 != 0)) return false;
  if (!aligned16(op0.s) || !aligned16(op0.b) || (dual && (!aligned16(o1.s) || !aligned16(o1.b)))) return false;
  if (M < 1 || M > kGemvMaxM || num_sms < 1) return false;
  return plan(K, N, static_cast<int>(M), op0.gs, o1.gs, op0.bits, o1.bits, dual, num_sms).slots > 0;
}

cudaError_t launch_gemv(const void *x, int64_t M, int64_t K, int64_t N, const QuantOperand &op0,
                        const QuantOperand *op1, int variant, int act, void *out, const void *residual,
                        cudaStream_t stream, uint64_t timeout_ns, int num_sms, bool early_weights) {
  if (!gemv_fits(M, K, N, op0, op1, num_sms)) return cudaErrorInvalidValue;
  const QuantOperand &o1 = op1 ? *op1 : op0;
  Layout l = plan(K, N, static_cast<int>(M), op0.gs, o1.gs, op0.bits, o1.bits, op1 != nullptr, num_sms);
  // Units of 2 warps where every unit of a CTA fits in its slots at once (M <= 8):
  // one unit per group, so no group takes two units in turn (decode: 9.70 vs
  // 10.00 us per call).
  if (M <= 8) {
    const Layout narrow =
        plan(K, N, static_cast<int>(M), op0.gs, o1.gs, op0.bits, o1.bits, op1 != nullptr, num_sms, kNarrowGroup);
    const int64_t units = (N + 7) / 8, grid = units < num_sms ? units : num_sms;
    if (narrow.slots > 0 && narrow.slots >= (units + grid - 1) / grid) l = narrow;
  }
  GemvParams p{};
  p.x = static_cast<const uint16_t *>(x);
  p.M = static_cast<int>(M);
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.w0 = op0.w;
  p.s0 = op0.s;
  p.b0 = op0.b;
  p.gd0 = GroupDiv::make(op0.gs);
  p.w1 = o1.w;
  p.s1 = o1.s;
  p.b1 = o1.b;
  p.gd1 = GroupDiv::make(o1.gs);
  p.ng0 = static_cast<uint32_t>(K / op0.gs);
  p.ng1 = static_cast<uint32_t>(K / o1.gs);
  p.x_rows = M < 8 ? static_cast<int>(M) : 8;
  p.variant = variant;
  p.out = static_cast<uint16_t *>(out);
  p.res = op1 ? nullptr : static_cast<const uint16_t *>(residual);
  p.timeout_ns = timeout_ns;
  p.early = early_weights ? 1 : 0;
  p.withhold = g_withhold.exchange(0);
  if (act == ActF16::kId) return launch_act<ActF16>(p, l, op0.bits, o1.bits, op1 != nullptr, stream, num_sms);
  if (act == ActBf16::kId) return launch_act<ActBf16>(p, l, op0.bits, o1.bits, op1 != nullptr, stream, num_sms);
  return cudaErrorInvalidValue;
}

// Read and clear the device error word of this translation unit's kernels.
cudaError_t gemv_take_errors(unsigned int *out) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof v);
  if (e != cudaSuccess) return e;
  if (v) {
    e = cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof zero);
    if (e != cudaSuccess) return e;
  }
  *out = v;
  return cudaSuccess;
}

}  // namespace qsw
