// Tensor-core kernel for the quantised SwiGLU expansion (prefill, any M) and
// for the single quantised linear.
//
// Method: mlx-bun pages, src/model/fused-swiglu-kernel.ts -- one output tile
// per work unit, the K=H reduction looped inside, the x tile loaded ONCE and
// fed to both the gate and the up product; dequantised weights staged as bf16
// before the MMA; gate/up rounded out of the f32 accumulator for MATCH.  The
// single-operand form follows src/model/steel-linear-kernel.ts (float
// accumulator cast to bf16 at the store).
//
// GB300 design (sm_103a), one persistent CTA per SM, warp-specialised:
//   warp 0      TMA producer: x tile [128 x 64] (128-byte swizzle) and the
//               packed-code tiles of this stage, one mbarrier per stage;
//   warp 1      TMEM owner and MMA issuer: per 64-wide K step, four
//               tcgen05.mma kind::f16 M=128 N=256 K=16 into a TMEM accumulator
//               (two accumulators of 256 columns, double-buffered);
//   warps 2-9   dequantisers: packed codes (smem) + scale/bias (global) ->
//               bf16 weights written straight into the 128-byte-swizzled
//               K-major operand layout the tensor core reads;
//   warps 10-13 epilogue: tcgen05.ld of the accumulator, the SwiGLU epilogue,
//               128-bit stores of bf16 hidden.
// The B operand of one MMA stacks 128 gate rows over 128 up rows (N = 256),
// so a single MMA stream computes both projections from one staged x tile.
//
// Every mbarrier wait is bounded; a CTA that gives up raises a shared abort
// flag so its other roles exit too, waits (bounded) for its own copies and
// MMAs in flight, frees its TMEM and returns.  The host reads the error word.
#include <atomic>
#include <mutex>

#include "qsw_device.cuh"
#include "qsw_internal.h"

namespace qsw {
namespace {

constexpr int BM = 128;   // rows of x per tile = UMMA M
constexpr int BK = 64;    // K per stage: one 128-byte swizzle atom of bf16
constexpr int BN = 256;   // UMMA N (B-tile rows)
constexpr int kDeqWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpDeq0 = 2, kWarpEpi0 = kWarpDeq0 + kDeqWarps;
constexpr int kThreads = 32 * (kWarpEpi0 + kEpiWarps);   // 448
constexpr uint32_t kTmemCols = 512;                       // two 256-column accumulators
constexpr int kMaxSmem = 232448;                          // opt-in limit per block

__device__ unsigned int g_prefill_error;

template <int BITS0, int BITS1, bool DUAL>
struct Cfg {
  static constexpr int kRows0 = DUAL ? 128 : 256;   // B rows from operand 0
  static constexpr int kRows1 = DUAL ? 128 : 0;     // B rows from operand 1
  static constexpr int kOutCols = DUAL ? 128 : 256; // output columns per tile
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kP0Pitch = BK * BITS0 / 8;   // bytes per packed row per stage
  static constexpr int kP1Pitch = BK * BITS1 / 8;
  static constexpr int kP0Bytes = kRows0 * kP0Pitch;
  static constexpr int kP1Bytes = kRows1 * kP1Pitch;
  static constexpr int kStageBytes = kABytes + kBBytes + kP0Bytes + kP1Bytes;
  static constexpr int kTxBytes = kABytes + kP0Bytes + kP1Bytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kStages = (4 * kStageBytes + 1024 + kBarBytes <= kMaxSmem) ? 4 : 3;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + kBarBytes;
  static_assert(kStageBytes % 1024 == 0, "stage must keep 1024-byte alignment");
  static_assert(kSmemBytes <= kMaxSmem, "shared memory budget");
  static_assert((3 * kStages + 5) * 8 + 8 <= kBarBytes, "barrier area");
};

struct PrefillParams {
  int64_t M, K, N;
  const uint16_t *s0, *b0;
  const uint16_t *s1, *b1;
  int gs0, gs1;
  GroupDiv gd0, gd1;
  int variant;
  uint16_t *out;
  int m_tiles, num_tiles, k_steps;
  uint64_t timeout_ns;
};

// Eight codes of one packed row (chunk c of a 64-code stage) -> 16 bytes of bf16.
template <int BITS>
__device__ __forceinline__ uint4 dequant_chunk(const uint8_t *prow, int c, uint32_t s2, uint32_t b2) {
  uint32_t o[4];
  if constexpr (BITS == 4) {
    Dequant8<4>::natural(*reinterpret_cast<const uint32_t *>(prow + 4 * c), s2, b2, o);
  } else if constexpr (BITS == 8) {
    const uint2 v = *reinterpret_cast<const uint2 *>(prow + 8 * c);
    Dequant8<8>::natural(v.x, v.y, s2, b2, o);
  } else {
    Dequant8<2>::natural(*reinterpret_cast<const uint16_t *>(prow + 2 * c), s2, b2, o);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_global_v4(void *p, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Wait executed by every lane of a warp; the outcome is made warp-uniform so
// that the whole warp either proceeds (converged) or leaves together.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort, uint64_t timeout_ns,
                                          unsigned int *err) {
  const bool ok = mbar_wait(bar, parity, abort, timeout_ns, err);
  return __all_sync(0xffffffffu, ok);
}

// Scale and bias of one (row, group), packed as (bias << 16) | scale.
__device__ __forceinline__ uint32_t load_sb(const uint16_t *s, const uint16_t *b, int64_t idx) {
  return static_cast<uint32_t>(__ldg(s + idx)) | (static_cast<uint32_t>(__ldg(b + idx)) << 16);
}

template <int BITS0, int BITS1, bool DUAL>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w0,
                   const __grid_constant__ CUtensorMap tm_w1, const PrefillParams p) {
  using C = Cfg<BITS0, BITS1, DUAL>;
  constexpr int S = C::kStages;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S * C::kStageBytes);
  uint64_t *full = bars;             // TMA bytes landed (x + packed codes)
  uint64_t *deq = bars + S;          // bf16 weights written by the dequantisers
  uint64_t *empty = bars + 2 * S;    // MMAs of the stage completed
  // Accumulation: each tile's K range is split in two halves that accumulate
  // in the two TMEM buffers X (first half) and Y (second half); the epilogue
  // adds Y into X with f32 adds.  Shorter tensor-core accumulation chains keep
  // the rounding of the stored projections close to a correctly rounded sum.
  // X of tile t is buffer t%2, Y the other one, so roles swap every tile.
  uint64_t *acc_full = bars + 3 * S; // both chains of the tile are complete
  uint64_t *y_free = acc_full + 1;   // Y has been added into X (Y reusable)
  uint64_t *x_free = acc_full + 2;   // X has been read out (X reusable)
  uint64_t *mma_done = acc_full + 3;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  auto stage_a = [&](int s) { return smem + s * C::kStageBytes; };
  auto stage_b = [&](int s) { return smem + s * C::kStageBytes + C::kABytes; };
  auto stage_p0 = [&](int s) { return smem + s * C::kStageBytes + C::kABytes + C::kBBytes; };
  auto stage_p1 = [&](int s) { return smem + s * C::kStageBytes + C::kABytes + C::kBBytes + C::kP0Bytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned int *err = &g_prefill_error;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&deq[s], kDeqWarps);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(y_free, kEpiWarps);
    mbar_init(x_free, kEpiWarps);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpTma && lane == 0) {
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_w0);
    if (DUAL) prefetch_tensormap(&tm_w1);
  }
  if (warp == kWarpMma) {
    __syncwarp();
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int last_parity[4] = {-1, -1, -1, -1};
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        const int m0 = (t % p.m_tiles) * BM;
        const int n0 = (t / p.m_tiles) * C::kOutCols;
        for (int kb = 0; kb < p.k_steps; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.timeout_ns, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], C::kTxBytes);
          tma_load_2d(stage_a(stage), &tm_x, &full[stage], kb * BK, m0);
          tma_load_2d(stage_p0(stage), &tm_w0, &full[stage], kb * BK * BITS0 / 32, n0);
          if (DUAL) tma_load_2d(stage_p1(stage), &tm_w1, &full[stage], kb * BK * BITS1 / 32, n0);
          last_parity[stage] = static_cast<int>(phase);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA's memory goes away
        for (int s = 0; s < S; ++s)
          if (last_parity[s] >= 0) mbar_wait_drain(&full[s], static_cast<uint32_t>(last_parity[s]), 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issue --
    if (lane == 0) {
      constexpr uint32_t kIdesc = umma_idesc_bf16(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const int k_half = (p.k_steps + 1) / 2;   // first chain: K steps [0, k_half)
      int lt = 0;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++lt) {
        const uint32_t x_tmem = tmem_base + static_cast<uint32_t>((lt & 1) * BN);
        const uint32_t y_tmem = tmem_base + static_cast<uint32_t>(((lt + 1) & 1) * BN);
        const uint32_t prev_parity = static_cast<uint32_t>((lt - 1) & 1);
        for (int kb = 0; kb < p.k_steps; ++kb) {
          // X of this tile was Y of the previous one, and Y was its X
          if (lt > 0 && (kb == 0 || kb == k_half)) {
            if (!mbar_wait(kb == 0 ? y_free : x_free, prev_parity, abort_flag, p.timeout_ns, err)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const uint32_t d_tmem = kb < k_half ? x_tmem : y_tmem;
          const bool chain_start = (kb == 0 || kb == k_half);
          if (!mbar_wait(&full[stage], phase, abort_flag, p.timeout_ns, err) ||
              !mbar_wait(&deq[stage], phase, abort_flag, p.timeout_ns, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = umma_desc_sw128(smem_u32(stage_a(stage)));
          const uint64_t bdesc = umma_desc_sw128(smem_u32(stage_b(stage)));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // +32 bytes of K per step inside the 128-byte swizzle atom
            umma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, kIdesc, (chain_start && kk == 0) ? 0u : 1u);
          }
          umma_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(acc_full);
      }
      if (!ok) {
        umma_commit(mma_done);
        mbar_wait_drain(mma_done, 0, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp < kWarpEpi0) {
    // ---------------------------------------------------------- dequantise --
    const int dt = threadIdx.x - kWarpDeq0 * 32;   // 0..255
    const int c = dt & 7;                          // 8-code chunk within the stage
    const int r0 = dt >> 3;                        // rows r0 + 32 j, j = 0..7
    const int64_t ng0 = p.K / p.gs0, ng1 = DUAL ? p.K / p.gs1 : 1;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      const int64_t n0 = static_cast<int64_t>(t / p.m_tiles) * C::kOutCols;
      // offset of the scale row of each of this thread's 8 B rows (row clamped
      // into range); 32-bit: rows * groups < 2^31 is checked on the host
      uint32_t srow[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int n = r0 + 32 * j;
        const int64_t r = n0 + (DUAL ? (n & 127) : n);
        const uint32_t rc = static_cast<uint32_t>(r < p.N ? r : p.N - 1);
        srow[j] = rc * static_cast<uint32_t>((!DUAL || j < 4) ? ng0 : ng1);
      }
      auto fetch_sb = [&](int kb, uint32_t (&sb)[8]) {
        const uint32_t k = static_cast<uint32_t>(kb) * BK + 8 * c;
        const uint32_t kc = k < static_cast<uint32_t>(p.K) ? k : static_cast<uint32_t>(p.K) - 1;
        const uint32_t grp0 = p.gd0(kc), grp1 = p.gd1(kc);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const bool first = !DUAL || j < 4;
          sb[j] = first ? load_sb(p.s0, p.b0, srow[j] + grp0) : load_sb(p.s1, p.b1, srow[j] + grp1);
        }
      };
      // scale/bias registers for steps kb, kb+1, kb+2: the global loads are
      // issued two K steps before they are used, hiding their latency
      uint32_t sb_cur[8], sb_next[8], sb_next2[8];
      fetch_sb(0, sb_cur);
      if (1 < p.k_steps) fetch_sb(1, sb_next);
      for (int kb = 0; kb < p.k_steps; ++kb) {
        if (kb + 2 < p.k_steps) fetch_sb(kb + 2, sb_next2);
        if (!warp_wait_lazy(&full[stage], phase, abort_flag, p.timeout_ns, err, 1000)) {
          ok = false;
          break;
        }
        const bool kvalid = static_cast<int64_t>(kb) * BK + 8 * c < p.K;
        const uint32_t bbase = smem_u32(stage_b(stage));
        const uint8_t *p0 = stage_p0(stage);
        const uint8_t *p1 = stage_p1(stage);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int n = r0 + 32 * j;
          const uint32_t s2 = prmt(sb_cur[j], 0, 0x1010u);   // scale in both halves
          const uint32_t b2 = prmt(sb_cur[j], 0, 0x3232u);   // bias in both halves
          uint4 v = make_uint4(0, 0, 0, 0);
          if (kvalid) {
            if (!DUAL || j < 4) {
              v = dequant_chunk<BITS0>(p0 + (DUAL ? (n & 127) : n) * C::kP0Pitch, c, s2, b2);
            } else {
              v = dequant_chunk<BITS1>(p1 + (n & 127) * C::kP1Pitch, c, s2, b2);
            }
          }
          // 128-byte swizzle: 16-byte chunk c of row n lands at chunk c ^ (n mod 8)
          st_shared_v4(bbase + n * 128 + ((c ^ (n & 7)) << 4), v);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&deq[stage]);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          sb_cur[j] = sb_next[j];
          sb_next[j] = sb_next2[j];
        }
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int quarter = warp & 3;   // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;
    const bool vec_ok = (p.N % 8) == 0;
    const bool two_chains = p.k_steps > 1;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    int lt = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++lt) {
      // the epilogue idles for a whole tile's main loop: wait without spinning
      if (!warp_wait_lazy(acc_full, static_cast<uint32_t>(lt & 1), abort_flag, p.timeout_ns, err, 10000)) break;
      tc_fence_after();
      const uint32_t tbase = lane_base + static_cast<uint32_t>((lt & 1) * BN);          // X
      const uint32_t ybase = lane_base + static_cast<uint32_t>(((lt + 1) & 1) * BN);    // Y
      if (two_chains) {
        // X += Y over all columns, f32 adds rounded to nearest
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 16) {
          uint32_t ra[16], rb[16];
          __syncwarp();
          tmem_ld16(tbase + c0, ra);
          tmem_ld16(ybase + c0, rb);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) ra[e] = __float_as_uint(__uint_as_float(ra[e]) + __uint_as_float(rb[e]));
          tmem_st16(tbase + c0, ra);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(y_free);   // Y may take the next tile's first chain
      const int64_t m = static_cast<int64_t>(t % p.m_tiles) * BM + row;
      const int64_t n0 = static_cast<int64_t>(t / p.m_tiles) * C::kOutCols;
      uint16_t *orow = p.out + m * p.N;
#pragma unroll 1
      for (int c0 = 0; c0 < C::kOutCols; c0 += 16) {
        uint32_t ra[16], rb[16];
        __syncwarp();   // tcgen05.ld is warp-collective
        tmem_ld16(tbase + c0, ra);
        if (DUAL) tmem_ld16(tbase + 128 + c0, rb);
        tmem_ld_wait();
        if (m < p.M) {
          uint32_t packed[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float v0, v1;
            if (DUAL) {
              v0 = swiglu_epilogue(p.variant, __uint_as_float(ra[e]), __uint_as_float(rb[e]));
              v1 = swiglu_epilogue(p.variant, __uint_as_float(ra[e + 1]), __uint_as_float(rb[e + 1]));
            } else {
              v0 = __uint_as_float(ra[e]);
              v1 = __uint_as_float(ra[e + 1]);
            }
            packed[e / 2] = pack_bf16x2(v0, v1);
          }
          const int64_t col = n0 + c0;
          if (vec_ok && col + 16 <= p.N) {
            st_global_v4(orow + col, make_uint4(packed[0], packed[1], packed[2], packed[3]));
            st_global_v4(orow + col + 8, make_uint4(packed[4], packed[5], packed[6], packed[7]));
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (col + e < p.N) orow[col + e] = static_cast<uint16_t>(packed[e / 2] >> (16 * (e & 1)));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(x_free);   // X may take the next tile's second chain
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ host ----

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

bool encode_2d(CUtensorMap *map, CUtensorMapDataType dtype, int elem_bytes, const void *base, uint64_t inner,
               uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem_bytes)};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BITS0, int BITS1, bool DUAL>
cudaError_t launch_impl(const void *x, int64_t M, int64_t K, int64_t N, const QuantOperand &op0,
                        const QuantOperand *op1, int variant, void *out, cudaStream_t stream, uint64_t timeout_ns,
                        int num_sms) {
  using C = Cfg<BITS0, BITS1, DUAL>;
  CUtensorMap tm_x, tm_w0, tm_w1;
  if (!encode_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, K, M, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_2d(&tm_w0, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, op0.w, K * BITS0 / 32, N, BK * BITS0 / 32, C::kRows0,
                 CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (DUAL) {
    if (!encode_2d(&tm_w1, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, op1->w, K * BITS1 / 32, N, BK * BITS1 / 32, C::kRows1,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    tm_w1 = tm_w0;
  }

  PrefillParams p{};
  p.M = M;
  p.K = K;
  p.N = N;
  p.s0 = op0.s;
  p.b0 = op0.b;
  p.gs0 = op0.gs;
  p.s1 = DUAL ? op1->s : op0.s;
  p.b1 = DUAL ? op1->b : op0.b;
  p.gs1 = DUAL ? op1->gs : op0.gs;
  p.gd0 = GroupDiv::make(p.gs0);
  p.gd1 = GroupDiv::make(p.gs1);
  if (N * (K / (p.gs0 < p.gs1 ? p.gs0 : p.gs1)) >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  p.variant = variant;
  p.out = static_cast<uint16_t *>(out);
  p.m_tiles = static_cast<int>((M + BM - 1) / BM);
  const int64_t n_tiles = (N + C::kOutCols - 1) / C::kOutCols;
  const int64_t tiles = static_cast<int64_t>(p.m_tiles) * n_tiles;
  if (tiles > (int64_t(1) << 30)) return cudaErrorInvalidValue;
  p.num_tiles = static_cast<int>(tiles);
  p.k_steps = static_cast<int>((K + BK - 1) / BK);
  p.timeout_ns = timeout_ns;

  // opt in to the large shared-memory carve-out once per device and instantiation
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(attr_done.load() & (uint64_t(1) << dev))) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<BITS0, BITS1, DUAL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(uint64_t(1) << dev);
  }
  const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
  prefill_kernel<BITS0, BITS1, DUAL><<<grid, kThreads, C::kSmemBytes, stream>>>(tm_x, tm_w0, tm_w1, p);
  return cudaGetLastError();
}

template <int BITS0>
cudaError_t dual_bits1(int bits1, const void *x, int64_t M, int64_t K, int64_t N, const QuantOperand &op0,
                       const QuantOperand *op1, int variant, void *out, cudaStream_t stream, uint64_t timeout_ns,
                       int num_sms) {
  switch (bits1) {
    case 2: return launch_impl<BITS0, 2, true>(x, M, K, N, op0, op1, variant, out, stream, timeout_ns, num_sms);
    case 4: return launch_impl<BITS0, 4, true>(x, M, K, N, op0, op1, variant, out, stream, timeout_ns, num_sms);
    case 8: return launch_impl<BITS0, 8, true>(x, M, K, N, op0, op1, variant, out, stream, timeout_ns, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill(const void *x, int64_t M, int64_t K, int64_t N, const QuantOperand &op0,
                           const QuantOperand *op1, int variant, void *out, cudaStream_t stream,
                           uint64_t timeout_ns, int num_sms) {
  if (op1) {
    switch (op0.bits) {
      case 2: return dual_bits1<2>(op1->bits, x, M, K, N, op0, op1, variant, out, stream, timeout_ns, num_sms);
      case 4: return dual_bits1<4>(op1->bits, x, M, K, N, op0, op1, variant, out, stream, timeout_ns, num_sms);
      case 8: return dual_bits1<8>(op1->bits, x, M, K, N, op0, op1, variant, out, stream, timeout_ns, num_sms);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (op0.bits) {
    case 2: return launch_impl<2, 2, false>(x, M, K, N, op0, nullptr, variant, out, stream, timeout_ns, num_sms);
    case 4: return launch_impl<4, 4, false>(x, M, K, N, op0, nullptr, variant, out, stream, timeout_ns, num_sms);
    case 8: return launch_impl<8, 8, false>(x, M, K, N, op0, nullptr, variant, out, stream, timeout_ns, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

// Read and clear the device error word of this translation unit's kernels.
cudaError_t prefill_take_errors(unsigned int *out) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_prefill_error, sizeof v);
  if (e != cudaSuccess) return e;
  if (v) {
    e = cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof zero);
    if (e != cudaSuccess) return e;
  }
  *out = v;
  return cudaSuccess;
}

}  // namespace qsw
