// Warp-streamed small-M kernel (M <= 16 per launch; up to 32 rows as launches
// over row chunks of 16): the fused SwiGLU expansion and the single quantised
// linear, for decode-sized batches.
//
// Method: mlx-bun pages, src/model/fused-swiglu-kernel.ts -- at decode the two
// projections are weight-streaming GEMVs.  Measured on this GPU, such a call
// spends as much time in per-call fixed costs (launch, staging x, the final
// reduction) as in its weight stream or its dequantisation, so the design
// keeps every step outside the block loop short and division-free:
//
//  * unit of work: 8 output features.  Fused: A rows 0..7 of mma.sync
//    m16n8k16 are gate rows, rows 8..15 the up rows of the same features, so
//    one MMA yields both projections; single linear: rows 8..15 are zero.
//    With M > 8, x has two row groups of 8 and every dequantised A fragment
//    feeds one MMA per group.  CTA b takes a contiguous range of units (sizes
//    differ by at most one);
//    the CTA's (unit, 128-code K block) items, unit-major, are cut into one
//    contiguous range per warp, so a warp runs many consecutive blocks between
//    synchronisations and the only CTA barriers are "x staged" and "partials
//    written";
//  * every warp streams its own blocks: each lane copies its 32 codes of A
//    rows g and g+8 (g = lane/4) per block with 16-byte cp.async copies into
//    a private ring of kDepth stages in shared memory, kDepth blocks ahead of
//    the block it computes, and waits only for its own copies
//    (cp.async.wait_group) -- no barrier, no copy engine, no slot bookkeeping;
//  * the lane dequantises its codes to the activation dtype T (w = T(s*q + b),
//    one rounding) with the K order inside each 8-code group interleaved
//    (codes j, j+4 paired); x is staged once per CTA in shared memory in the
//    matching B-fragment order (all 8 fragment rows for short x, its real
//    rows only for long x);
//  * scales and biases are read per block through L1; each warp requests the
//    scale rows of its units into L1 when it starts;
//  * each block accumulates in a fresh fragment that is added to the warp's
//    running f32 sum; at a unit boundary the sum goes to a shared-memory
//    partial, and after one barrier the warp holding a unit's last block adds
//    the unit's partials in warp order (deterministic), every lane its own
//    accumulator registers, and applies the epilogue.
//
// With one row group two CTAs fit on an SM (at most 64 registers per thread,
// about 100 KB of shared memory at decode sizes), so with the early weight
// stream the next call's CTAs start and request their first blocks while this
// call computes.
// The kernel has no spin waits: cp.async.wait_group waits for the thread's own
// copies, which always complete.
#include <atomic>

#include "qsw_internal.h"
#include "qsw_smallm.cuh"

namespace qsw {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kDepth = 3;                     // ring stages per warp
constexpr int kBlockK = kSmallBlockK;         // codes per K block
constexpr int kChunk = kSmallChunk;           // codes per lane per block
constexpr int kSmemBudget = 200 * 1024;
constexpr int64_t kMaxK = 16384;              // the group-index multiply below is exact up to here

__device__ unsigned int g_gemv_stream_error;

struct StreamParams {
  const uint16_t *x;
  int M, K, N;
  const uint32_t *w0, *w1;
  const uint16_t *s0, *b0, *s1, *b1;
  uint32_t gm0, gm1;      // group index of code k: umulhi(k >> 4, gm) (gm = ceil(2^31 / (gs / 32)))
  uint32_t ng0, ng1;      // groups per row (K / gs)
  int variant;
  uint16_t *out;
  const uint16_t *res;    // single-operand form: [M, N] added before the rounding (or null)
  int nkb;                // K blocks per row
  int x_rows;             // rows of x staged per block: 8 (rows >= M as zeros) or min(M, 8)
  int uq, ur;             // CTA b has uq + (b < ur) units, starting at b * uq + min(b, ur)
  int slots;              // partial-sum slots per warp
  int red_off, ring_off, tab_off;   // byte offsets of the partial sums, the rings, the warp tables
  int early;
};

// 16- or 8-byte asynchronous copy global -> shared, tracked per thread.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// One bf16/f16 value, zero-extended into 32 bits (through L1).
__device__ __forceinline__ uint32_t ldg_u16(const uint16_t *p) {
  uint32_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void prefetch_l1(const void *p) { asm volatile("prefetch.global.L1 [%0];" ::"l"(p)); }

// Layout of one operand's codes in a ring stage: piece q (16 bytes) of lane L
// at q * 512 + L * 16 (2-bit: the lane's 8 bytes at L * 8), so that a warp's
// copies and reads of one piece are 512 consecutive bytes.
template <int BITS>
__host__ __device__ constexpr int chunk_bytes() {
  return BITS == 2 ? 256 : BITS / 4 * 512;
}
template <int BITS>
__host__ __device__ constexpr int lane_bytes() {
  return BITS == 2 ? 8 : 16;
}
template <int BITS0, int BITS1, bool DUAL>
__host__ __device__ constexpr int stage_bytes() {
  return chunk_bytes<BITS0>() + (DUAL ? chunk_bytes<BITS1>() : 0);
}

template <int BITS>
__device__ __forceinline__ void copy_chunk(uint32_t dst, const uint32_t *src) {
  if constexpr (BITS == 2) {
    cp_async8(dst, src);
  } else {
#pragma unroll
    for (int q = 0; q < BITS / 4; ++q) cp_async16(dst + q * 512, src + 4 * q);
  }
}
template <int BITS>
__device__ __forceinline__ void read_chunk(uint32_t (&w)[BITS], uint32_t src) {
  if constexpr (BITS == 2) {
    const uint2 v = lds64(src);
    w[0] = v.x;
    w[1] = v.y;
  } else {
#pragma unroll
    for (int q = 0; q < BITS / 4; ++q) {
      const uint4 v = lds128(src + q * 512);
      w[4 * q + 0] = v.x;
      w[4 * q + 1] = v.y;
      w[4 * q + 2] = v.z;
      w[4 * q + 3] = v.w;
    }
  }
}

// XF: all 8 fragment rows of each x row group are staged (p.x_rows == 8 * NG),
// so the staging layout is a compile-time constant.  NG: x row groups of 8
// (M <= 8: 1; M <= 16: 2, which share every dequantised A fragment).
// MB: CTAs meant to share an SM (2 caps the registers at 64 a thread; used
// where the shared memory of two CTAs fits).
template <int BITS0, int BITS1, bool DUAL, bool XF, int NG, int MB, class A>
__global__ void __launch_bounds__(kThreads, MB) gemv_stream_kernel(const StreamParams p) {
  constexpr int BB = DUAL ? BITS1 : BITS0;
  constexpr int SB = stage_bytes<BITS0, BITS1, DUAL>();
  extern __shared__ __align__(128) uint8_t smem[];
  float *red = reinterpret_cast<float *>(smem + p.red_off);   // [kWarps][slots][32][4]
  int *ufirst_tab = reinterpret_cast<int *>(smem + p.tab_off);  // [kWarps]: CTA-local unit of a warp's first item
  int *wfirst_tab = ufirst_tab + kWarps;                         // [units of the CTA]: first warp of a unit
  unsigned int *err = &g_gemv_stream_error;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const uint32_t K = static_cast<uint32_t>(p.K);
  const int nkb = p.nkb;
  const int b = static_cast<int>(blockIdx.x);
  const int u_begin = b * p.uq + (b < p.ur ? b : p.ur);
  const int ucount = p.uq + (b < p.ur ? 1 : 0);
  const int items = ucount * nkb;
  const int i_begin = static_cast<int>(static_cast<int64_t>(warp) * items / kWarps);
  const int i_end = static_cast<int>(static_cast<int64_t>(warp + 1) * items / kWarps);
  const int u_first = i_begin / nkb;
  const uint32_t ring = smem_u32(smem + p.ring_off) + warp * (kDepth * SB);

  if constexpr (kDebugBounds) {   // x, partial sums, rings, warp tables
    debug_poison_smem(smem, static_cast<uint32_t>(p.tab_off + (kWarps + p.uq + 1) * 4));
    __syncthreads();
  }

  // x of a non-dependent launch is requested first: behind the weight stream
  // it would arrive microseconds later.  Lane L = 4n + c carries row n of x.
  // Where x is short all 8 fragment rows are staged (rows >= M as zeros: the
  // fastest reads); for long x only its min(M, 8) real rows are, and a lane of
  // a row n >= M reads the fragment of lane L mod (4 min(M, 8)) instead: B
  // column n of the MMA then holds another row's values, which only affects
  // output column n, and columns n >= M are never stored.
  const int x_lanes = XF ? 32 : 4 * p.x_rows;
  const uint32_t x_piece = static_cast<uint32_t>(x_lanes) * 16;   // bytes of one (block, group, j) piece
  const int x_total = nkb * NG * 32;   // (block, group, lane) entries of 64 bytes; lanes >= x_lanes are not staged
  auto load_x = [&](int e, uint4 (&xv)[4]) {
    const int L = e & 31, kb = (e >> 5) / NG;
    const int m = 8 * ((e >> 5) % NG) + (L >> 2);
    const uint32_t k = static_cast<uint32_t>(kb) * kBlockK + (L & 3) * kChunk;
    if (k < K && m < p.M) {
      const uint4 *xp = reinterpret_cast<const uint4 *>(p.x + static_cast<int64_t>(m) * p.K + k);
#pragma unroll
      for (int q = 0; q < 4; ++q) xv[q] = __ldg(xp + q);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) xv[q] = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  // For block kb, row group G and fragment piece j (x values 8j..8j+7 of each
  // lane's chunk), lane L = 4n + c's 16 bytes sit at ((kb*NG + G)*4 + j)*x_piece
  // + L*16: row 8G + n of x, codes kb*128 + 32c + 8j ... + 7 permuted into
  // (x0,x4) (x1,x5) (x2,x6) (x3,x7) pairs.
  auto store_x = [&](int e, const uint4 (&xv)[4]) {
    uint8_t *dst = smem + static_cast<size_t>(e >> 5) * 4 * x_piece + (e & 31) * 16;
#pragma unroll
    for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4 *>(dst + j * x_piece) = x_fragment(xv[j]);
  };
  uint4 x_first[4];
  const bool has_x = static_cast<int>(threadIdx.x) < x_total && static_cast<int>(threadIdx.x & 31) < x_lanes;
  if (!p.early && has_x) load_x(threadIdx.x, x_first);

  // --- warp tables for the final reduction, and the scale rows into L1 ---
  // A warp with no items (fewer items than warps) is marked -1: it may sit
  // between a unit's first and last warp, and holds no partial sum.
  if (lane == 0) ufirst_tab[warp] = i_begin < i_end ? u_first : -1;
  if (i_begin < i_end) {
    const int u_last = (i_end - 1) / nkb;
    for (int u = u_first + lane; u <= u_last; u += 32) {
      debug_check(u < ucount, err);
      if (u * nkb >= i_begin) wfirst_tab[u] = warp;             // the unit's first item is the warp's
    }
    // 8 rows x ng groups x 2 bytes per array, contiguous: 128-byte lines
    const int arrays = DUAL ? 4 : 2;
    for (int a = 0; a < arrays; ++a) {
      const uint16_t *base = a == 0 ? p.s0 : a == 1 ? p.b0 : a == 2 ? p.s1 : p.b1;
      const uint32_t ng = a < 2 ? p.ng0 : p.ng1;
      const int64_t r_end = static_cast<int64_t>(8) * (u_begin + u_last + 1) < p.N
                                ? static_cast<int64_t>(8) * (u_begin + u_last + 1)
                                : static_cast<int64_t>(p.N);
      const int64_t last = r_end * ng;
      for (int64_t e = static_cast<int64_t>(8) * (u_begin + u_first) * ng + lane * 64; e < last; e += 32 * 64)
        prefetch_l1(base + e);
    }
  }

  // --- the weight stream: item i (CTA-local) = (unit i / nkb, block i % nkb) ---
  // The lane's copy cursor advances by constant strides and jumps to the next
  // unit's rows after a unit's last block.
  constexpr uint32_t kStep0 = kBlockK * BITS0 / 32, kStep1 = kBlockK * BB / 32;   // words per block of a row
  const uint32_t wpr0 = K * BITS0 / 32, wpr1 = K * BB / 32;                       // words per packed row
  const bool k_full = (K % kBlockK) == 0;
  // every lane of every item of this CTA in range (no ragged unit or block):
  // the per-lane guards below are skipped (warp-uniform)
  const bool all_in = k_full && 8 * (u_begin + ucount) <= p.N;
  int ld_left = i_end - i_begin;
  int ld_kb = i_begin - u_first * nkb;
  int ld_row0 = 8 * (u_begin + u_first);   // first A row of the unit being requested
  uint32_t ld_k = static_cast<uint32_t>(ld_kb) * kBlockK + c * kChunk;
  const uint32_t *pa = p.w0 + static_cast<int64_t>(ld_row0 + g) * wpr0 + ld_k * BITS0 / 32;
  const uint32_t *pb = p.w1 + static_cast<int64_t>(ld_row0 + g) * wpr1 + ld_k * BB / 32;
  const uint32_t lane0 = lane * lane_bytes<BITS0>(), lane1 = chunk_bytes<BITS0>() + lane * lane_bytes<BB>();
  uint32_t ld_stage = 0;
  auto issue_next = [&]() {
    if (ld_left > 0) {   // warp-uniform
      // lanes past N or K copy nothing: their scale and bias read as 0 below, so w = 0
      if (all_in || (ld_row0 + g < p.N && ld_k < K)) {
        debug_check(ld_k + kChunk <= K && ld_row0 + g < p.N, err);
        copy_chunk<BITS0>(ring + ld_stage + lane0, pa);
        if constexpr (DUAL) copy_chunk<BITS1>(ring + ld_stage + lane1, pb);
      }
      --ld_left;
      pa += kStep0;
      pb += kStep1;
      ld_k += kBlockK;
      if (++ld_kb == nkb) {
        ld_kb = 0;
        ld_k = c * kChunk;
        ld_row0 += 8;
        pa += 8 * static_cast<int64_t>(wpr0) - static_cast<int64_t>(nkb) * kStep0;
        pb += 8 * static_cast<int64_t>(wpr1) - static_cast<int64_t>(nkb) * kStep1;
      }
    }
    cp_async_commit();   // one group per item (empty past the range), so the waits count items
    ld_stage = ld_stage + SB == kDepth * SB ? 0 : ld_stage + SB;
  };

  if (p.early && threadIdx.x == 0) griddep_launch_dependents();
#pragma unroll
  for (int s = 0; s < kDepth; ++s) issue_next();

  // --- x -> shared memory, once per CTA ---
  if (p.early) {
    // programmatic dependent: x is read only after the preceding work is done
    if (warp == 0 && lane < p.M)
      prefetch_l2_bulk(p.x + static_cast<int64_t>(lane) * p.K, static_cast<uint32_t>(p.K) * 2);
    griddep_wait();
    if (has_x) load_x(threadIdx.x, x_first);
  }
  if (has_x) store_x(threadIdx.x, x_first);
  for (int e = threadIdx.x + kThreads; e < x_total; e += kThreads) {
    if ((e & 31) >= x_lanes) continue;
    uint4 xv[4];
    load_x(e, xv);
    store_x(e, xv);
  }
  __syncthreads();

  // --- the warp's blocks ---
  const uint32_t xstep = x_piece;
  const uint32_t xbase = smem_u32(smem) + (XF ? lane : lane % x_lanes) * 16;
  float sum[NG][4];
#pragma unroll
  for (int G = 0; G < NG; ++G)
#pragma unroll
    for (int q = 0; q < 4; ++q) sum[G][q] = 0.0f;
  int cu = u_first, ckb = i_begin - u_first * nkb;
  uint32_t xb = xbase + static_cast<uint32_t>(ckb) * NG * 4 * xstep;
  int c_row = 8 * (u_begin + u_first) + g;
  uint32_t ck = static_cast<uint32_t>(ckb) * kBlockK + c * kChunk;
  int64_t so0 = static_cast<int64_t>(c_row) * p.ng0, so1 = static_cast<int64_t>(c_row) * p.ng1;
  uint32_t cs = 0;   // offset of the stage being computed
  auto flush = [&]() {
    const int t = cu - u_first;
    debug_check(t >= 0 && t < p.slots, err);
#pragma unroll
    for (int G = 0; G < NG; ++G)
      *reinterpret_cast<float4 *>(red + (((warp * p.slots + t) * NG + G) * 32 + lane) * 4) =
          make_float4(sum[G][0], sum[G][1], sum[G][2], sum[G][3]);
  };
  // the next block's scales and biases (through L1, one block ahead of their
  // use), zero past N or K
  uint32_t sa = 0u, ba = 0u, sb = 0u, bb = 0u;
  auto load_scales = [&]() {
    sa = ba = sb = bb = 0u;
    if (all_in || (c_row < p.N && ck < K)) {
      const uint32_t gi0 = __umulhi(ck >> 4, p.gm0);
      debug_check(gi0 < p.ng0, err);
      sa = ldg_u16(p.s0 + so0 + gi0);
      ba = ldg_u16(p.b0 + so0 + gi0);
      if constexpr (DUAL) {
        const uint32_t gi1 = __umulhi(ck >> 4, p.gm1);
        debug_check(gi1 < p.ng1, err);
        sb = ldg_u16(p.s1 + so1 + gi1);
        bb = ldg_u16(p.b1 + so1 + gi1);
      }
    }
  };
  const int n_items = i_end - i_begin;
  if (n_items > 0) load_scales();
#pragma unroll 1
  for (int i = 0; i < n_items; ++i) {
    cp_async_wait<kDepth - 1>();   // this lane's copies of the block have landed
    Chunk<BITS0, A> ca;
    Chunk<BB, A> cb;
    read_chunk<BITS0>(ca.w, ring + cs + lane0);
    if constexpr (DUAL) read_chunk<BITS1>(cb.w, ring + cs + lane1);
    // (a lane past N or K reads stale stage bytes: with scale and bias 0 they dequantise to 0)
    const uint32_t sa2 = sa * 0x00010001u, ba2 = ba * 0x00010001u;
    const uint32_t sb2 = sb * 0x00010001u, bb2 = bb * 0x00010001u;
    float acc[NG][4];
#pragma unroll
    for (int G = 0; G < NG; ++G)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[G][q] = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t pa4[4], pb4[4] = {0u, 0u, 0u, 0u};
      ca.dequant(j, sa2, ba2, pa4);
      if constexpr (DUAL) cb.dequant(j, sb2, bb2, pb4);
      // A rows g and g+8; k_local 2c,2c+1 <- pair 2h, k_local 2c+8,2c+9 <- pair 2h+1
      const uint32_t a0[4] = {pa4[0], pb4[0], pa4[1], pb4[1]};
      const uint32_t a1[4] = {pa4[2], pb4[2], pa4[3], pb4[3]};
#pragma unroll
      for (int G = 0; G < NG; ++G) {
        const uint4 xf = lds128(xb + (G * 4 + j) * xstep);
        mma_16816<A>(acc[G], a0, xf.x, xf.y);
        mma_16816<A>(acc[G], a1, xf.z, xf.w);
      }
    }
#pragma unroll
    for (int G = 0; G < NG; ++G)
#pragma unroll
      for (int q = 0; q < 4; ++q) sum[G][q] += acc[G][q];
    // the stage is read: refill it with the block kDepth items on
    cs = cs + SB == kDepth * SB ? 0 : cs + SB;
    issue_next();
    xb += NG * 4 * xstep;
    ck += kBlockK;
    if (++ckb == nkb) {   // the unit's last block: its partial sum is complete
      flush();
#pragma unroll
      for (int G = 0; G < NG; ++G)
#pragma unroll
        for (int q = 0; q < 4; ++q) sum[G][q] = 0.0f;
      ckb = 0;
      ++cu;
      xb = xbase;
      ck = c * kChunk;
      c_row += 8;
      so0 += 8 * static_cast<int64_t>(p.ng0);
      so1 += 8 * static_cast<int64_t>(p.ng1);
    }
    if (i + 1 < n_items) load_scales();
  }
  if (ckb != 0 && n_items > 0) flush();   // the range ended inside a unit
  cp_async_wait<0>();                     // (only empty groups remain)
  __syncthreads();

  // --- partial sums of each unit, in warp order, then the epilogue ---
  // The warp that holds a unit's last block finishes it: lane (g, c) adds the
  // partials of its own accumulator registers (A rows g and g+8, x columns 2c
  // and 2c+1 of each row group G) over the unit's warps in warp order and
  // applies the epilogue to its outputs (i = 8u + g, m = 8G + 2c and 8G + 2c + 1).
  if (i_begin < i_end) {
    const int u_last = (i_end - 1) / nkb;
    for (int u = u_first; u <= u_last; ++u) {
      if ((u + 1) * nkb - 1 >= i_end) continue;   // the unit ends in a later warp's range
      float4 s4[NG];
#pragma unroll
      for (int G = 0; G < NG; ++G) s4[G] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      for (int w = wfirst_tab[u]; w <= warp; ++w) {
        const int uf = ufirst_tab[w];
        if (uf < 0) continue;   // no items
        const int t = u - uf;
        debug_check(t >= 0 && t < p.slots, err);
#pragma unroll
        for (int G = 0; G < NG; ++G) {
          const float4 v = *reinterpret_cast<const float4 *>(red + (((w * p.slots + t) * NG + G) * 32 + lane) * 4);
          s4[G].x += v.x;
          s4[G].y += v.y;
          s4[G].z += v.z;
          s4[G].w += v.w;
        }
      }
      const int64_t i_out = static_cast<int64_t>(u_begin + u) * 8 + g;
      if (i_out >= p.N) continue;
#pragma unroll
      for (int G = 0; G < NG; ++G) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int m = 8 * G + 2 * c + q;
          if (m >= p.M) break;
          const float gv = q ? s4[G].y : s4[G].x, uv = q ? s4[G].w : s4[G].z;
          const int64_t o = static_cast<int64_t>(m) * p.N + i_out;
          const float v = DUAL ? swiglu_epilogue<A>(p.variant, gv, uv) : (p.res ? gv + A::lo(p.res[o]) : gv);
          p.out[o] = A::store(v);
        }
      }
    }
  }
}

// x row groups of 8: one for M <= 8, two for M <= 16.
int stream_groups(int64_t M) { return M > 8 ? 2 : 1; }

// Rows of x staged per block: with one row group, all 8 fragment rows while
// they take at most 48 KB (K <= 3072), else only the real ones (so that two
// CTAs, e.g. of a decode block's expansion and down projection, still fit on
// an SM); with two row groups, all 16.
int64_t stream_x_rows(int64_t M, int64_t K) {
  if (stream_groups(M) == 2) return 16;
  const int64_t nkb = (K + kBlockK - 1) / kBlockK;
  return nkb * 4 * 8 * 64 <= 48 * 1024 ? 8 : (M < 8 ? M : 8);
}

struct StreamLayout {
  int red_off, ring_off, tab_off, slots, total;
};

// Shared-memory layout; total == 0 when the shape does not fit.
StreamLayout stream_plan(int64_t M, int64_t K, int64_t N, int num_sms, int stage) {
  StreamLayout l{};
  if (M < 1 || M > 16 || K > kMaxK || num_sms < 1) return l;
  const int64_t ng = stream_groups(M);
  const int64_t nkb = (K + kBlockK - 1) / kBlockK;
  const int64_t units = (N + 7) / 8;
  const int64_t grid = units < num_sms ? units : num_sms;
  const int64_t ucta = (units + grid - 1) / grid;              // most units of a CTA
  const int64_t ipw = (ucta * nkb + kWarps - 1) / kWarps;      // most items of a warp
  int64_t slots = (ipw + nkb - 1) / nkb + 1;                  // units a contiguous item range can touch
  if (slots > ucta) slots = ucta;
  const int64_t x_bytes = (nkb * 4 * stream_x_rows(M, K) * 64 + 127) / 128 * 128;
  const int64_t red_bytes = kWarps * slots * 512 * ng;
  const int64_t ring_bytes = static_cast<int64_t>(kWarps) * kDepth * stage;
  const int64_t tab_bytes = (kWarps + ucta + 1) * 4;
  const int64_t total = x_bytes + red_bytes + ring_bytes + tab_bytes;
  if (total > kSmemBudget) return l;
  l.red_off = static_cast<int>(x_bytes);
  l.ring_off = static_cast<int>(x_bytes + red_bytes);
  l.tab_off = static_cast<int>(x_bytes + red_bytes + ring_bytes);
  l.slots = static_cast<int>(slots);
  l.total = static_cast<int>(total);
  return l;
}

int stage_of(int bits0, int bits1, bool dual) {
  auto chunk = [](int bits) { return bits == 2 ? 256 : bits / 4 * 512; };
  return chunk(bits0) + (dual ? chunk(bits1) : 0);
}

template <int BITS0, int BITS1, bool DUAL, bool XF, int NG, int MB, class A>
cudaError_t launch_x(const StreamParams &p, const StreamLayout &l, int grid, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(attr_done.load() & (uint64_t(1) << dev))) {
    cudaError_t e = cudaFuncSetAttribute(gemv_stream_kernel<BITS0, BITS1, DUAL, XF, NG, MB, A>,
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
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_stream_kernel<BITS0, BITS1, DUAL, XF, NG, MB, A>, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int BITS0, int BITS1, bool DUAL, class A>
cudaError_t launch_cfg(StreamParams p, const StreamLayout &l, cudaStream_t stream, int num_sms) {
  const int units = (p.N + 7) / 8;
  const int grid = units < num_sms ? units : num_sms;
  p.nkb = (p.K + kBlockK - 1) / kBlockK;
  p.x_rows = static_cast<int>(stream_x_rows(p.M, p.K));
  p.uq = units / grid;
  p.ur = units % grid;
  p.slots = l.slots;
  p.red_off = l.red_off;
  p.ring_off = l.ring_off;
  p.tab_off = l.tab_off;
  if (p.x_rows == 16) return launch_x<BITS0, BITS1, DUAL, true, 2, 1, A>(p, l, grid, stream);
  if (p.x_rows != 8) return launch_x<BITS0, BITS1, DUAL, false, 1, 2, A>(p, l, grid, stream);
  // two CTAs per SM where their shared memory fits (228 KB per SM, 1 KB reserved
  // per CTA), else one with twice the registers (measured: mixed specs, M <= 8,
  // 4 % faster)
  return 2 * (l.total + 1024) <= 228 * 1024 ? launch_x<BITS0, BITS1, DUAL, true, 1, 2, A>(p, l, grid, stream)
                                            : launch_x<BITS0, BITS1, DUAL, true, 1, 1, A>(p, l, grid, stream);
}

template <int BITS0, class A>
cudaError_t launch_bits1(const StreamParams &p, const StreamLayout &l, int bits1, cudaStream_t stream, int num_sms) {
  switch (bits1) {
    case 2: return launch_cfg<BITS0, 2, true, A>(p, l, stream, num_sms);
    case 4: return launch_cfg<BITS0, 4, true, A>(p, l, stream, num_sms);
    case 8: return launch_cfg<BITS0, 8, true, A>(p, l, stream, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

template <class A>
cudaError_t launch_act(const StreamParams &p, const StreamLayout &l, int bits0, int bits1, bool dual,
                       cudaStream_t stream, int num_sms) {
  if (dual) {
    switch (bits0) {
      case 2: return launch_bits1<2, A>(p, l, bits1, stream, num_sms);
      case 4: return launch_bits1<4, A>(p, l, bits1, stream, num_sms);
      case 8: return launch_bits1<8, A>(p, l, bits1, stream, num_sms);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (bits0) {
    case 2: return launch_cfg<2, 2, false, A>(p, l, stream, num_sms);
    case 4: return launch_cfg<4, 4, false, A>(p, l, stream, num_sms);
    case 8: return launch_cfg<8, 8, false, A>(p, l, stream, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

uint32_t group_magic(int gs) {
  const uint64_t d = static_cast<uint64_t>(gs / 32);
  return static_cast<uint32_t>(((uint64_t(1) << 31) + d - 1) / d);
}

}  // namespace

// Rows of x one launch takes; more rows run as consecutive launches over
// row chunks of this size, each streaming the weights once.
constexpr int64_t kStreamChunk = 16;

bool gemv_stream_fits(int64_t M, int64_t K, int64_t N, const QuantOperand &op0, const QuantOperand *op1,
                      int num_sms) {
  const QuantOperand &o1 = op1 ? *op1 : op0;
  if (M < 1 || M > kGemvMaxM) return false;
  const int64_t mc = M < kStreamChunk ? M : kStreamChunk;
  return stream_plan(mc, K, N, num_sms, stage_of(op0.bits, o1.bits, op1 != nullptr)).total > 0 &&
         stream_plan(1, K, N, num_sms, stage_of(op0.bits, o1.bits, op1 != nullptr)).total > 0;
}

namespace {

cudaError_t launch_chunk(const void *x, int64_t M, int64_t K, int64_t N, const QuantOperand &op0,
                         const QuantOperand *op1, int variant, int act, void *out, const void *residual,
                         cudaStream_t stream, int num_sms, bool early_weights) {
  const QuantOperand &o1 = op1 ? *op1 : op0;
  const StreamLayout l = stream_plan(M, K, N, num_sms, stage_of(op0.bits, o1.bits, op1 != nullptr));
  if (l.total == 0) return cudaErrorInvalidValue;
  StreamParams p{};
  p.x = static_cast<const uint16_t *>(x);
  p.M = static_cast<int>(M);
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.w0 = op0.w;
  p.s0 = op0.s;
  p.b0 = op0.b;
  p.gm0 = group_magic(op0.gs);
  p.w1 = o1.w;
  p.s1 = o1.s;
  p.b1 = o1.b;
  p.gm1 = group_magic(o1.gs);
  p.ng0 = static_cast<uint32_t>(K / op0.gs);
  p.ng1 = static_cast<uint32_t>(K / o1.gs);
  p.variant = variant;
  p.out = static_cast<uint16_t *>(out);
  p.res = op1 ? nullptr : static_cast<const uint16_t *>(residual);
  p.early = early_weights ? 1 : 0;
  if (act == ActF16::kId) return launch_act<ActF16>(p, l, op0.bits, o1.bits, op1 != nullptr, stream, num_sms);
  if (act == ActBf16::kId) return launch_act<ActBf16>(p, l, op0.bits, o1.bits, op1 != nullptr, stream, num_sms);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemv_stream(const void *x, int64_t M, int64_t K, int64_t N, const QuantOperand &op0,
                               const QuantOperand *op1, int variant, int act, void *out, const void *residual,
                               cudaStream_t stream, int num_sms, bool early_weights) {
  if (!gemv_stream_fits(M, K, N, op0, op1, num_sms)) return cudaErrorInvalidValue;
  // rows [m0, m0 + mc) of x, of the output and of the residual (row-major, 2-byte elements)
  for (int64_t m0 = 0; m0 < M; m0 += kStreamChunk) {
    const int64_t mc = M - m0 < kStreamChunk ? M - m0 : kStreamChunk;
    const cudaError_t e = launch_chunk(static_cast<const uint16_t *>(x) + m0 * K, mc, K, N, op0, op1, variant, act,
                                       static_cast<uint16_t *>(out) + m0 * N,
                                       residual ? static_cast<const uint16_t *>(residual) + m0 * N : nullptr,
                                       stream, num_sms, early_weights);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Read and clear the device error word of this translation unit's kernel.
cudaError_t gemv_stream_take_errors(unsigned int *out) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemv_stream_error, sizeof v);
  if (e != cudaSuccess) return e;
  if (v) {
    e = cudaMemcpyToSymbol(g_gemv_stream_error, &zero, sizeof zero);
    if (e != cudaSuccess) return e;
  }
  *out = v;
  return cudaSuccess;
}

}  // namespace qsw
