// Small-M kernel for the quantised SwiGLU expansion (decode, M <= 32) and for
// the single quantised linear at small M.
//
// Method: mlx-bun pages, src/model/fused-swiglu-kernel.ts -- at decode the two
// projections are memory-bound GEMVs and "reading Wg/Wu dominates".  Here the
// packed rows are streamed once with 128-bit loads, dequantised in registers to
// bf16 (w = bf16(s*q + b), one rounding) and reduced over K on the tensor
// cores with mma.sync m16n8k16 (a cheap reduction engine for this HBM-bound
// path; the contraction is not what bounds it).
//
// Work split: one CTA owns 16 output rows (i); its 8 warps split K in blocks
// of 128 codes.  Inside a block, lane (g = lane/4, c = lane%4) owns the
// 32-code chunk c of rows g and g+8.  The order of K inside an 8-code group
// is free as long as A (weights) and B (x) agree, so each lane dequantises
// with the interleaved pairing (codes j, j+4) and permutes its own x values
// the same way.  Partial sums meet in shared memory in a fixed order.
#include "qsw_device.cuh"
#include "qsw_internal.h"

namespace qsw {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kBlockK = 128;   // codes per K block
constexpr int kChunk = 32;     // codes per lane per block

struct GemvParams {
  const uint16_t *x;
  int64_t M, K, N;
  QuantOperand op[2];
  int variant;
  uint16_t *out;
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Packed words covering one lane's 32 codes of one row.
template <int BITS>
struct RowChunk {
  static constexpr int kWords = kChunk * BITS / 32;   // 4, 8 or 2
  uint32_t w[kWords];
  uint32_t s2, b2;   // group scale/bias splatted to bf16x2

  __device__ __forceinline__ void load(const QuantOperand &op, int64_t row, int64_t k, int64_t K, bool valid) {
    if (!valid) {
#pragma unroll
      for (int i = 0; i < kWords; ++i) w[i] = 0;
      s2 = 0;
      b2 = 0;
      return;
    }
    const uint32_t *p = op.w + row * (K * BITS / 32) + k * BITS / 32;
    if constexpr (BITS == 2) {
      const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
      w[0] = v.x;
      w[1] = v.y;
    } else {
#pragma unroll
      for (int i = 0; i < kWords / 4; ++i) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p) + i);
        w[4 * i + 0] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
      }
    }
    const int64_t gidx = row * (K / op.gs) + k / op.gs;
    s2 = splat_bf16(__ldg(op.s + gidx));
    b2 = splat_bf16(__ldg(op.b + gidx));
  }

  // Eight dequantised codes (sub-chunk j), interleaved pairing.
  __device__ __forceinline__ void dequant(int j, uint32_t (&o)[4]) const {
    if constexpr (BITS == 4) {
      Dequant8<4>::interleaved(w[j], s2, b2, o);
    } else if constexpr (BITS == 8) {
      Dequant8<8>::interleaved(w[2 * j], w[2 * j + 1], s2, b2, o);
    } else {
      Dequant8<2>::interleaved(w[j >> 1] >> (16 * (j & 1)), s2, b2, o);
    }
  }
};

template <int BITS0, int BITS1, bool DUAL, int NG>
struct BlockData {
  RowChunk<BITS0> a0[2];             // operand 0, rows g and g+8
  RowChunk<BITS1> a1[DUAL ? 2 : 1];  // operand 1 (unused when single)
  uint4 xv[NG][4];                   // x rows 8G+g, 32 values
};

template <int BITS0, int BITS1, bool DUAL, int NG>
__device__ __forceinline__ void load_block(const GemvParams &p, int64_t kb, int64_t r0, int g, int c,
                                           BlockData<BITS0, BITS1, DUAL, NG> &bd) {
  const int64_t k = kb * kBlockK + c * kChunk;
  const bool kvalid = k < p.K;
  bd.a0[0].load(p.op[0], r0, k, p.K, kvalid && r0 < p.N);
  bd.a0[1].load(p.op[0], r0 + 8, k, p.K, kvalid && r0 + 8 < p.N);
  if constexpr (DUAL) {
    bd.a1[0].load(p.op[1], r0, k, p.K, kvalid && r0 < p.N);
    bd.a1[1].load(p.op[1], r0 + 8, k, p.K, kvalid && r0 + 8 < p.N);
  }
#pragma unroll
  for (int G = 0; G < NG; ++G) {
    const int64_t m = 8 * G + g;
    if (kvalid && m < p.M) {
      const uint4 *xp = reinterpret_cast<const uint4 *>(p.x + m * p.K + k);
#pragma unroll
      for (int i = 0; i < 4; ++i) bd.xv[G][i] = __ldg(xp + i);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) bd.xv[G][i] = make_uint4(0, 0, 0, 0);
    }
  }
}

template <int BITS0, int BITS1, bool DUAL, int NG>
__device__ __forceinline__ void compute_block(const BlockData<BITS0, BITS1, DUAL, NG> &bd,
                                              float (&acc0)[NG][4], float (&acc1)[NG][4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t p0r0[4], p0r1[4];
    bd.a0[0].dequant(j, p0r0);
    bd.a0[1].dequant(j, p0r1);
    uint32_t p1r0[4], p1r1[4];
    if constexpr (DUAL) {
      bd.a1[0].dequant(j, p1r0);
      bd.a1[1].dequant(j, p1r1);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t a0[4] = {p0r0[2 * h], p0r1[2 * h], p0r0[2 * h + 1], p0r1[2 * h + 1]};
      uint32_t a1[4] = {0, 0, 0, 0};
      if constexpr (DUAL) {
        a1[0] = p1r0[2 * h];
        a1[1] = p1r1[2 * h];
        a1[2] = p1r0[2 * h + 1];
        a1[3] = p1r1[2 * h + 1];
      }
#pragma unroll
      for (int G = 0; G < NG; ++G) {
        // x values of sub-chunk j: q0=(x0,x1) q1=(x2,x3) q2=(x4,x5) q3=(x6,x7);
        // the weights pair codes (p, p+4), so x is paired the same way.
        const uint4 xs = bd.xv[G][j];
        uint32_t b0, b1;
        if (h == 0) {
          b0 = prmt(xs.x, xs.z, 0x5410u);   // (x0, x4)
          b1 = prmt(xs.x, xs.z, 0x7632u);   // (x1, x5)
        } else {
          b0 = prmt(xs.y, xs.w, 0x5410u);   // (x2, x6)
          b1 = prmt(xs.y, xs.w, 0x7632u);   // (x3, x7)
        }
        mma_bf16_16816(acc0[G], a0, b0, b1);
        if constexpr (DUAL) mma_bf16_16816(acc1[G], a1, b0, b1);
      }
    }
  }
}

template <int BITS0, int BITS1, bool DUAL, int NG>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const GemvParams p) {
  constexpr int NMAT = DUAL ? 2 : 1;
  __shared__ float red[kWarps][NMAT][NG][32][4];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 16 + g;
  const int64_t nkb = (p.K + kBlockK - 1) / kBlockK;

  float acc0[NG][4], acc1[NG][4];
#pragma unroll
  for (int G = 0; G < NG; ++G)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc0[G][i] = acc1[G][i] = 0.0f;

  // Two blocks in flight per warp: the loads of both are issued before either
  // is consumed.
  int64_t kb = warp;
  for (; kb + kWarps < nkb; kb += 2 * kWarps) {
    BlockData<BITS0, BITS1, DUAL, NG> d0, d1;
    load_block(p, kb, r0, g, c, d0);
    load_block(p, kb + kWarps, r0, g, c, d1);
    compute_block(d0, acc0, acc1);
    compute_block(d1, acc0, acc1);
  }
  if (kb < nkb) {
    BlockData<BITS0, BITS1, DUAL, NG> d0;
    load_block(p, kb, r0, g, c, d0);
    compute_block(d0, acc0, acc1);
  }

#pragma unroll
  for (int G = 0; G < NG; ++G)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      red[warp][0][G][lane][i] = acc0[G][i];
      if constexpr (DUAL) red[warp][NMAT - 1][G][lane][i] = acc1[G][i];
    }
  __syncthreads();

  // Each element of the 16 x (8*NG) tile: fixed-order sum over the warps.
  for (int e = threadIdx.x; e < NG * 128; e += kThreads) {
    const int G = e >> 7, l = (e >> 2) & 31, q = e & 3;
    const int row = (l >> 2) + ((q & 2) ? 8 : 0);
    const int n = 2 * (l & 3) + (q & 1);
    const int64_t m = 8 * G + n;
    const int64_t i = static_cast<int64_t>(blockIdx.x) * 16 + row;
    if (m >= p.M || i >= p.N) continue;
    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      s0 += red[w][0][G][l][q];
      if constexpr (DUAL) s1 += red[w][NMAT - 1][G][l][q];
    }
    const float v = DUAL ? swiglu_epilogue(p.variant, s0, s1) : s0;
    p.out[m * p.N + i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

template <int BITS0, int BITS1, bool DUAL>
cudaError_t launch_ng(const GemvParams &p, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((p.N + 15) / 16));
  if (p.M <= 8) {
    gemv_kernel<BITS0, BITS1, DUAL, 1><<<grid, kThreads, 0, stream>>>(p);
  } else if (p.M <= 16) {
    gemv_kernel<BITS0, BITS1, DUAL, 2><<<grid, kThreads, 0, stream>>>(p);
  } else {
    gemv_kernel<BITS0, BITS1, DUAL, 4><<<grid, kThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

template <int BITS0>
cudaError_t launch_dual_bits1(const GemvParams &p, int bits1, cudaStream_t stream) {
  switch (bits1) {
    case 2: return launch_ng<BITS0, 2, true>(p, stream);
    case 4: return launch_ng<BITS0, 4, true>(p, stream);
    case 8: return launch_ng<BITS0, 8, true>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gemv(const void *x, int64_t M, int64_t K, int64_t N, const QuantOperand &op0,
                        const QuantOperand *op1, int variant, void *out, cudaStream_t stream) {
  if (M < 1 || M > kGemvMaxM) return cudaErrorInvalidValue;
  GemvParams p{};
  p.x = static_cast<const uint16_t *>(x);
  p.M = M;
  p.K = K;
  p.N = N;
  p.op[0] = op0;
  p.op[1] = op1 ? *op1 : op0;
  p.variant = variant;
  p.out = static_cast<uint16_t *>(out);
  if (op1) {
    switch (op0.bits) {
      case 2: return launch_dual_bits1<2>(p, op1->bits, stream);
      case 4: return launch_dual_bits1<4>(p, op1->bits, stream);
      case 8: return launch_dual_bits1<8>(p, op1->bits, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (op0.bits) {
    case 2: return launch_ng<2, 2, false>(p, stream);
    case 4: return launch_ng<4, 4, false>(p, stream);
    case 8: return launch_ng<8, 8, false>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qsw
