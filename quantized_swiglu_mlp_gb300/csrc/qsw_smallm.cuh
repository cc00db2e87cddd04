// Device helpers of the small-M kernel (qsw_gemv.cu): the legacy-MMA step,
// 1-D bulk copies and shared-memory loads, and the per-lane chunk of 32 codes
// with its dequantisation.
//
// The kernel feeds dequantised weights as the A operand of
// mma.sync.m16n8k16 and x as B.  A lane (g = lane/4, c = lane%4) owns 32
// consecutive codes (one "chunk") of each of its two A rows per 128-code K
// block; inside every 8-code group the K order is interleaved (codes j and
// j+4 form a pair), and x is staged with the same permutation, which leaves
// the dot products unchanged.
#pragma once

#include "qsw_device.cuh"

namespace qsw {

constexpr int kSmallBlockK = 128;   // codes per K block
constexpr int kSmallChunk = 32;     // codes per lane per block

// D += A . B, m16n8k16, f32 accumulators, A and B in the activation dtype.
// A pure function of its register operands (not volatile), so the compiler
// may schedule it freely around the loads that feed it.
template <class A>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (A::kId == ActF16::kId) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// One 1-D bulk copy global -> shared, completing on `bar` (bytes and both
// addresses multiples of 16).
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bring [src, src + bytes) into L2; no data returns to the SM.  Both the
// address and the size are multiples of 16 bytes.
__device__ __forceinline__ void prefetch_l2_bulk(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Shared-memory loads at a 32-bit shared address, written as ordinary C++
// loads (through the generic window of the shared address space) so that the
// compiler can schedule them early; every barrier wait that guards the data
// carries a memory clobber, which keeps them after it.
__device__ __forceinline__ const void *smem_ptr(uint32_t addr) {
  return __cvta_shared_to_generic(static_cast<size_t>(addr));
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) { return *static_cast<const uint4 *>(smem_ptr(addr)); }
__device__ __forceinline__ uint2 lds64(uint32_t addr) { return *static_cast<const uint2 *>(smem_ptr(addr)); }
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) { return *static_cast<const uint16_t *>(smem_ptr(addr)); }

// 32 codes of one row (the lane's chunk of a 128-code block), from shared memory.
template <int BITS, class A>
struct Chunk {
  static constexpr int kWords = kSmallChunk * BITS / 32;   // 4, 8 or 2
  uint32_t w[kWords];
  __device__ __forceinline__ void load(uint32_t addr) {
    if constexpr (BITS == 2) {
      const uint2 v = lds64(addr);
      w[0] = v.x;
      w[1] = v.y;
    } else {
#pragma unroll
      for (int i = 0; i < kWords / 4; ++i) {
        const uint4 v = lds128(addr + 16 * i);
        w[4 * i + 0] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
      }
    }
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < kWords; ++i) w[i] = 0u;
  }
  // eight codes (sub-chunk j), interleaved pairing (codes p, p+4 in word p)
  __device__ __forceinline__ void dequant(int j, uint32_t s2, uint32_t b2, uint32_t (&o)[4]) const {
    if constexpr (BITS == 4) {
      Dequant8<4, A>::interleaved(w[j], s2, b2, o);
    } else if constexpr (BITS == 8) {
      Dequant8<8, A>::interleaved(w[2 * j], w[2 * j + 1], s2, b2, o);
    } else {
      Dequant8<2, A>::interleaved(w[j >> 1] >> (16 * (j & 1)), s2, b2, o);
    }
  }
};

// x (rows of the activation dtype) -> the B fragments of one 128-code block:
// the 32 values x[8j .. 8j+7] (j = 0..3) of a lane's chunk, loaded as four
// 16-byte words, become four 16-byte fragments, one per j, each holding the
// pairs (x0,x4) (x1,x5) (x2,x6) (x3,x7) that match Dequant8's interleaved
// pairs of the A rows.
__device__ __forceinline__ uint4 x_fragment(const uint4 &v) {
  return make_uint4(prmt(v.x, v.z, 0x5410u),    // (x0, x4)
                    prmt(v.x, v.z, 0x7632u),    // (x1, x5)
                    prmt(v.y, v.w, 0x5410u),    // (x2, x6)
                    prmt(v.y, v.w, 0x7632u));   // (x3, x7)
}

}  // namespace qsw
