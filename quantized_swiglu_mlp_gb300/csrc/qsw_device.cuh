// Device-side building blocks shared by the qswiglu kernels (sm_103a):
// inline-PTX wrappers for mbarrier / TMA / tcgen05, bounded waits, the
// packed-code -> bf16 dequantisation and the SwiGLU epilogues.
//
// Method source: mlx-bun pages, src/model/fused-swiglu-kernel.ts
//   - dequantised weights are staged as the activation dtype (bf16) before the
//     block MMA (the Wgs/Wus threadgroup tiles), i.e. w = bf16(scale*q + bias);
//   - MATCH epilogue: gate and up rounded to bf16 out of the float accumulator,
//     then sigma = bf16(1/(1+exp(-g))), silu = bf16(g*sigma), h = bf16(silu*u);
//   - F32 epilogue: no rounding before the final store.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qsw {

// ------------------------------------------------------------------ errors --

// Device error word bits: a kernel gave up on a wait; a debug-build check of
// an address or a copy coordinate failed.
enum : unsigned { DEVERR_TIMEOUT = 1u, DEVERR_BOUNDS = 2u };

// ------------------------------------------------------------ debug build --
// Built with QSW_DEBUG_BOUNDS, the kernels (1) fill their shared-memory
// staging areas (and the tensor-core kernel its TMEM accumulators) with 0xFF
// bytes at start -- a NaN in bf16, f16 and f32 -- so that a read of staging
// data that was never written shows up as NaN in the results, and (2) check
// copy coordinates and address ranges, recording a failure in the device
// error word (DEVERR_BOUNDS) and going on: nothing traps.  Both compile to
// nothing in the regular build.
#ifdef QSW_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif

__device__ __forceinline__ void debug_check(bool ok, unsigned int *err) {
  if (kDebugBounds && !ok) atomicOr(err, DEVERR_BOUNDS);
}

// Every thread of the CTA: [p, p + bytes) of shared memory (16-byte aligned;
// a partial last 16 bytes is left) := 0xFF.  The caller synchronises.
__device__ __forceinline__ void debug_poison_smem(uint8_t *p, uint32_t bytes) {
  if (kDebugBounds)
    for (uint32_t i = threadIdx.x * 16; i + 16 <= bytes; i += blockDim.x * 16)
      *reinterpret_cast<uint4 *>(p + i) = make_uint4(~0u, ~0u, ~0u, ~0u);
}

// ----------------------------------------------------------------- helpers --

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// ---------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may be suspended by the hardware for up to
// `hint_ns` until the phase completes, instead of returning at once.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait until the barrier's phase with the given parity has completed.  Never
// spins forever: gives up after `timeout_ns`, or as soon as another role of the
// CTA has raised `abort`.  Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          uint64_t timeout_ns, unsigned int *err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort = 1;
        atomicOr(err, DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Warp-collective wait for waits that may be long: lane 0 waits with the
// hardware suspend hint (the thread sleeps until the phase completes, so an
// idle warp takes no issue slots from the warps doing work), then every lane
// observes the completed phase itself (immediate).  The result is
// warp-uniform; false means "give up".
__device__ __forceinline__ bool warp_wait_lazy(uint64_t *bar, uint32_t parity, volatile int *abort,
                                               uint64_t timeout_ns, unsigned int *err, uint32_t suspend_ns) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0 && !mbar_try_wait(bar, parity)) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
      if (mbar_try_wait_suspend(bar, parity, suspend_ns)) break;
      if (*abort) {
        ok = 0;
        break;
      }
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort = 1;
        atomicOr(err, DEVERR_TIMEOUT);
        ok = 0;
        break;
      }
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok) return false;
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, timeout_ns, err));
}

// Wait executed by a whole warp for waits that are usually short: lane 0
// polls, then every lane observes the completed phase itself; the outcome is
// warp-uniform (false: give up).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort, uint64_t timeout_ns,
                                          unsigned int *err) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort, timeout_ns, err) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok) return false;
  return __all_sync(0xffffffffu, mbar_try_wait(bar, parity));
}

// Wait used while tearing down after an abort: ignores the abort flag (it is
// already raised) and gives up silently after `timeout_ns`.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
  return true;
}

// ------------------------------------------------ programmatic dependents --

// Let the next grid on the stream (launched as a programmatic dependent) be
// scheduled; wait until every grid this one depends on has completed and its
// memory is visible.  Both are no-ops without a programmatic dependency.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// --------------------------------------------------------------------- TMA --

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// Make generic-proxy writes to shared memory visible to the async proxy
// (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- tcgen05 --

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] . B[smem]^T, bf16 inputs, f32 accumulator, one CTA.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread t of the warp receives the
// 16 columns of TMEM lane (lane_base + t).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Inverse of tmem_ld16: thread t writes 16 consecutive columns of TMEM lane
// (lane_base + t).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major bf16 tile stored in the
// 128-byte-swizzled canonical layout: rows of 64 bf16 (128 B), 8-row groups
// 1024 B apart, tile base 1024-byte aligned.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);   // start address
  d |= static_cast<uint64_t>(1) << 16;                       // leading byte offset (unused when swizzled)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;               // stride byte offset: 8 rows x 128 B
  d |= static_cast<uint64_t>(1) << 46;                       // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                       // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16 with A and B both of `fmt` (0 f16,
// 1 bf16: the two operands always share their type), f32 D, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_f16kind(int m, int n, uint32_t fmt) {
  return (1u << 4)                                   // D format f32
         | (fmt << 7)                                // A format
         | (fmt << 10)                               // B format
         | (static_cast<uint32_t>(n >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24);    // M / 16
}

// ----------------------------------------------------------- bf16 helpers ---

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// d = a*b + c with a single rounding to bf16 per lane.
__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// (a & mask) | c
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(c));
  return d;
}
// Two f32 -> bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ uint32_t splat_bf16(uint16_t v) { return static_cast<uint32_t>(v) * 0x00010001u; }
// Lane-wise bf16 product, correctly rounded (nearest even).
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float bf16x2_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16x2_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// ------------------------------------------------------ activation dtype ----
// The activation dtype T of x, the scales and biases, the dequantised weights
// (the tensor-core operands) and hidden: bf16 or f16.  Each trait supplies
// the paired (two values per 32-bit register) arithmetic the kernels use.

struct ActBf16 {
  static constexpr int kId = 0;
  static constexpr uint32_t kUmmaFormat = 1;   // instruction-descriptor A/B format
  // 128 in both halves: (0x4300 | q) is the bf16 value 128 + q for q < 128
  static constexpr uint32_t kMagic2 = 0x43004300u;
  __device__ __forceinline__ static uint32_t sub2(uint32_t a, uint32_t b) { return bf16x2_sub(a, b); }
  __device__ __forceinline__ static uint32_t fma2(uint32_t a, uint32_t b, uint32_t c) { return bf16x2_fma(a, b, c); }
  __device__ __forceinline__ static uint32_t mul2(uint32_t a, uint32_t b) { return bf16x2_mul(a, b); }
  __device__ __forceinline__ static uint32_t pack2(float lo, float hi) { return pack_bf16x2(lo, hi); }
  __device__ __forceinline__ static float lo(uint32_t v) { return bf16x2_lo(v); }
  __device__ __forceinline__ static float hi(uint32_t v) { return bf16x2_hi(v); }
  __device__ __forceinline__ static uint16_t store(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
};

struct ActF16 {
  static constexpr int kId = 1;
  static constexpr uint32_t kUmmaFormat = 0;
  // 1024 in both halves: (0x6400 | q) is the f16 value 1024 + q for q < 1024
  static constexpr uint32_t kMagic2 = 0x64006400u;
  __device__ __forceinline__ static uint32_t sub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  __device__ __forceinline__ static uint32_t fma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
  }
  __device__ __forceinline__ static uint32_t mul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
  }
  __device__ __forceinline__ static float lo(uint32_t v) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xffffu)));
  }
  __device__ __forceinline__ static float hi(uint32_t v) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)));
  }
  __device__ __forceinline__ static uint16_t store(float v) { return __half_as_ushort(__float2half_rn(v)); }
};

// Exact integer code -> bf16 value for 8-bit codes: the byte is placed in the
// mantissa of the f32 2^23 and 2^23 is subtracted (exact), then narrowed
// (exact: every integer 0..255 is a bf16).
__device__ __forceinline__ float code8_to_f32(uint32_t word, uint32_t byte_sel) {
  const uint32_t bits = prmt(word, 0x4B000000u, 0x7650u | byte_sel);
  return __uint_as_float(bits) - 8388608.0f;
}

// ----------------------------------------------------- dequantisation -------
// Eight consecutive codes of one row -> eight weights w = T(s*q + b) (one
// rounding, fma.rn on the pair), returned as four T x2 words.  `s2`/`b2` hold
// the group's scale and bias in both halves.  The natural order puts code 2j
// in the low half of word j and code 2j+1 in the high half (k order, as the
// tensor-core tile needs).  Codes of 2 and 4 bits become exact T values by
// placing them in the mantissa of a power of two (A::kMagic2) and subtracting
// it; 8-bit codes go through f32 for bf16 (128 + q overflows its 7-bit
// mantissa), and the same way for f16.

template <int BITS, class A>
struct Dequant8;

template <class A>
struct Dequant8<4, A> {
  // `w` holds the eight codes (code j at bits 4j).
  __device__ __forceinline__ static void natural(uint32_t w, uint32_t s2, uint32_t b2, uint32_t (&o)[4]) {
    const uint32_t v = w >> 4;   // low nibble of byte j of v = code 2j+1
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // byte j of w -> byte 0, byte j of v -> byte 2; keep the low nibbles
      const uint32_t t = prmt(w, v, static_cast<uint32_t>(j) | (static_cast<uint32_t>(4 + j) << 8));
      const uint32_t q = A::sub2(and_or(t, 0x000F000Fu, A::kMagic2), A::kMagic2);
      o[j] = A::fma2(q, s2, b2);
    }
  }
  // Interleaved order (codes j and j+4 in word j): cheaper, used where the K
  // order inside an 8-code group is free.
  __device__ __forceinline__ static void interleaved(uint32_t w, uint32_t s2, uint32_t b2, uint32_t (&o)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t q = A::sub2(and_or(w >> (4 * j), 0x000F000Fu, A::kMagic2), A::kMagic2);
      o[j] = A::fma2(q, s2, b2);
    }
  }
};

template <class A>
struct Dequant8<8, A> {
  // `w0` holds codes 0..3, `w1` codes 4..7 (one byte each).
  __device__ __forceinline__ static void natural(uint32_t w0, uint32_t w1, uint32_t s2, uint32_t b2,
                                                 uint32_t (&o)[4]) {
    o[0] = A::fma2(A::pack2(code8_to_f32(w0, 0), code8_to_f32(w0, 1)), s2, b2);
    o[1] = A::fma2(A::pack2(code8_to_f32(w0, 2), code8_to_f32(w0, 3)), s2, b2);
    o[2] = A::fma2(A::pack2(code8_to_f32(w1, 0), code8_to_f32(w1, 1)), s2, b2);
    o[3] = A::fma2(A::pack2(code8_to_f32(w1, 2), code8_to_f32(w1, 3)), s2, b2);
  }
  __device__ __forceinline__ static void interleaved(uint32_t w0, uint32_t w1, uint32_t s2, uint32_t b2,
                                                     uint32_t (&o)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = A::fma2(A::pack2(code8_to_f32(w0, j), code8_to_f32(w1, j)), s2, b2);
  }
};

template <class A>
struct Dequant8<2, A> {
  // `h` holds the eight codes in its low 16 bits (code j at bits 2j).
  __device__ __forceinline__ static void natural(uint32_t h, uint32_t s2, uint32_t b2, uint32_t (&o)[4]) {
    const uint32_t v2 = h >> 2, v4 = h >> 4, v6 = h >> 6;
    // byte B of h carries codes 4B..4B+3; the low 2 bits of byte B of h, v2,
    // v4, v6 are codes 4B, 4B+1, 4B+2, 4B+3.
    const uint32_t t0 = prmt(h, v2, 0x0400u);    // codes 0, 1
    const uint32_t t1 = prmt(v4, v6, 0x0400u);   // codes 2, 3
    const uint32_t t2 = prmt(h, v2, 0x0501u);    // codes 4, 5
    const uint32_t t3 = prmt(v4, v6, 0x0501u);   // codes 6, 7
    const uint32_t t[4] = {t0, t1, t2, t3};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t q = A::sub2(and_or(t[j], 0x00030003u, A::kMagic2), A::kMagic2);
      o[j] = A::fma2(q, s2, b2);
    }
  }
  __device__ __forceinline__ static void interleaved(uint32_t h, uint32_t s2, uint32_t b2, uint32_t (&o)[4]) {
    // codes j and j+4 sit in bytes 0 and 1 at bit 2j
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t t = prmt(h >> (2 * j), 0u, 0x0100u);
      const uint32_t q = A::sub2(and_or(t, 0x00030003u, A::kMagic2), A::kMagic2);
      o[j] = A::fma2(q, s2, b2);
    }
  }
};

// ------------------------------------------------------------- group index --

// k / gs for the scale/bias group of code k without a runtime division when gs
// is a power of two (shift >= 0); otherwise a 32-bit division.
struct GroupDiv {
  int gs;
  int shift;   // log2(gs) when gs is a power of two, else -1
  __host__ __device__ static GroupDiv make(int g) {
    int s = -1;
    if (g > 0 && (g & (g - 1)) == 0) {
      s = 0;
      while ((1 << s) < g) ++s;
    }
    return GroupDiv{g, s};
  }
  __device__ __forceinline__ uint32_t operator()(uint32_t k) const {
    return shift >= 0 ? (k >> shift) : k / static_cast<uint32_t>(gs);
  }
};

// ---------------------------------------------------------------- epilogue --

enum : int { VAR_MATCH = 0, VAR_F32 = 1, VAR_DEBUG_GATE = 2, VAR_DEBUG_UP = 3 };

// sigma(v) = 1 / (1 + e^-v) with the hardware exponential and reciprocal
// approximations: branch-free, so an epilogue thread overlaps the 16 elements
// it holds.  Their few-ulp f32 error is far below the rounding to the
// activation dtype that follows; for v < -88 the denominator overflows and
// sigma is 0 (the true value is below 2^-126).
__device__ __forceinline__ float sigmoid_fast(float v) { return __fdividef(1.0f, 1.0f + __expf(-v)); }

// v rounded to the activation dtype and back (exact widening).
template <class A>
__device__ __forceinline__ float round_act(float v) {
  const uint32_t p = A::pack2(v, 0.0f);
  return A::lo(p);
}

// hidden = silu(g) * u for one element, from the f32 projections; the caller
// rounds the result to the activation dtype at the store.
template <class A>
__device__ __forceinline__ float swiglu_epilogue(int variant, float g, float u) {
  if (variant == VAR_MATCH) {
    const float gb = round_act<A>(g), ub = round_act<A>(u);
    const float sig = round_act<A>(sigmoid_fast(gb));
    const float silu = round_act<A>(gb * sig);
    return silu * ub;   // exact product of two T values; rounded once by the caller's store
  }
  if (variant == VAR_F32) return (g * sigmoid_fast(g)) * u;
  return variant == VAR_DEBUG_GATE ? g : u;
}

// The MATCH epilogue of two elements at once, (g0, u0) in the low half of the
// result and (g1, u1) in the high half: the same roundings as
// swiglu_epilogue(VAR_MATCH) followed by the store's rounding, since a product
// of two bf16 (or two f16) values is exact in f32 and mul.rn on the pair
// rounds that exact product to nearest even.  Bit-identical to the scalar
// form, in about half the instructions.
template <class A>
__device__ __forceinline__ uint32_t swiglu_match2(float g0, float g1, float u0, float u1) {
  const uint32_t gb = A::pack2(g0, g1), ub = A::pack2(u0, u1);
  const uint32_t sig = A::pack2(sigmoid_fast(A::lo(gb)), sigmoid_fast(A::hi(gb)));
  return A::mul2(A::mul2(gb, sig), ub);
}

}  // namespace qsw
