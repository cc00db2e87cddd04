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
// GB300 design (sm_103a), one persistent CTA per SM, warp-specialised, three
// shared-memory rings filled by TMA and one filled by the dequantisers:
//   x ring      stages of 2 x tiles [256 x 64], 128-byte swizzle   TMA -> MMA
//   codes ring  packed codes of the tile's 128 B rows, per K step  TMA -> dequant
//   scale ring  per operand: scales and biases of 8 groups         TMA -> dequant
//   B ring      stages of 2 dequantised B tiles [128 x 64]         dequant -> MMA
// (a stage is two 64-wide K steps: the MMA issuer pays one barrier wait and
// one commit per 16 UMMAs instead of per 8, and those shared-memory round
// trips are what its loop spends beyond the tensor core's own time).
// Roles:
//   warp 0      producer of the codes and scale rings;
//   warp 1      TMEM owner and MMA issuer: per 64-wide K step, 2 x 4
//               tcgen05.mma kind::f16 M=128 N=128 K=16, one per 128-row half of
//               the x tile, both against the same B tile (every dequantised
//               weight serves 256 rows of x), two K steps per ring stage;
//   warp 2      producer of the x ring (two producers, so that neither stream
//               waits behind the other's ring);
//   warps 3-18  dequantisers: each thread turns 16 codes of one B row into bf16
//               per K step and writes them into the swizzled K-major layout the
//               tensor core reads;
//   warps 19-22 epilogue: tcgen05.ld of the accumulator, the SwiGLU epilogue,
//               16-byte stores of bf16 hidden.
// The B operand stacks 64 gate rows over 64 up rows (N = 128), so one MMA
// stream computes both projections from one staged x tile.
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

constexpr int BM = 256;   // rows of x per tile: two UMMAs (M = 128 each) share every B tile
constexpr int UM = 128;   // UMMA M
constexpr int BK = 64;    // K per step: one 128-byte swizzle atom of bf16
constexpr int BN = 128;   // UMMA N (B-tile rows)
constexpr int kDeqWarps = 16;
constexpr int kEpiWarps = 4;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpX = 2, kWarpDeq0 = 3, kWarpEpi0 = kWarpDeq0 + kDeqWarps;
constexpr int kThreads = 32 * (kWarpEpi0 + kEpiWarps);   // 736
constexpr uint32_t kTmemCols = 512;                       // X and Y, each two 128-column accumulators
constexpr int kMaxSmem = 232448;                          // opt-in limit per block
constexpr int kAccCols = 2 * BN;                          // TMEM columns of X (or Y): one accumulator per x half
constexpr int kXBytes = BM * BK * 2;                      // 32 KB
constexpr int kBBytes = BN * BK * 2;                      // 16 KB
constexpr int kGroupsPerEntry = 8;                        // scale groups per ring entry (16 bytes)
constexpr int kBarBytes = 512;
constexpr int kSub = 2;                                   // K steps (64 wide) per x/B ring stage
constexpr int kChainStages = 11;                          // ring stages per accumulation chain, at most (22 K steps)
constexpr int kPartFloats = 2 * UM * BN;                  // f32 partial accumulator of one split tile (128 KB)

__device__ unsigned int g_prefill_error;

// Static stream-K workspace for the entry point that allocates nothing: sized
// for up to kStaticScratchSms SMs (header + one partial slot per SM), zero at
// module load and zeroed again (header) on first use per device.
constexpr int kStaticScratchSms = 192;
constexpr size_t kStaticScratchBytes =
    4096 + static_cast<size_t>(kStaticScratchSms) * 2 * 128 * 128 * sizeof(float);
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

template <int BITS0, int BITS1, bool DUAL>
struct Cfg {
  static constexpr int kRows0 = DUAL ? 64 : 128;    // B rows from operand 0
  static constexpr int kRows1 = DUAL ? 64 : 0;      // B rows from operand 1
  static constexpr int kOutCols = DUAL ? 64 : 128;  // output columns per tile
  static constexpr int kC0Pitch = BK * BITS0 / 8;   // packed bytes per row per K step
  static constexpr int kC1Pitch = BK * BITS1 / 8;
  static constexpr int kC0Bytes = kRows0 * kC0Pitch;
  static constexpr int kCodesBytes = kC0Bytes + kRows1 * kC1Pitch;
  // one scale-ring entry: [rows][8] scales then [rows][8] biases, per operand
  static constexpr int kS0Bytes = kRows0 * 2 * kGroupsPerEntry;
  static constexpr int kS1Bytes = kRows1 * 2 * kGroupsPerEntry;
  static constexpr int kEntryBytes = 2 * kS0Bytes + 2 * kS1Bytes;
  // The x and B rings hold stages of kSub consecutive K steps (one barrier
  // wait and one commit per stage for the MMA issuer); codes and scales keep
  // rings of single K steps.
  static constexpr int kSb = 2;   // B ring, stages
  static constexpr int kSx = 2;   // x ring, stages (advances with the B ring: same depth)
  static constexpr int kXStage = kSub * kXBytes;
  static constexpr int kBStage = kSub * kBBytes;
  static constexpr int kBudget = kMaxSmem - 1024 - kBarBytes;
  static constexpr int kFixed = kSx * kXStage + kSb * kBStage + 2 * kEntryBytes;
  static constexpr int kScFit = (kBudget - kFixed) / kCodesBytes;
  static constexpr int kSc = kScFit > 4 ? 4 : kScFit;   // codes ring, K steps
  static constexpr int kXOff = 0;
  static constexpr int kBOff = kXOff + kSx * kXStage;
  static constexpr int kCOff = kBOff + kSb * kBStage;
  static constexpr int kSOff = kCOff + kSc * kCodesBytes;
  static constexpr int kBarOff = kSOff + 2 * kEntryBytes;
  static constexpr int kSmemBytes = kBarOff + kBarBytes + 1024;
  static_assert(kSc >= 2, "codes ring too small");
  static_assert(kSx == kSb, "the x and B rings share their barriers' slot index");
  static_assert(kSc >= kSub, "the codes ring must hold a stage");
  static_assert(kCodesBytes % 1024 == 0 && kC0Bytes % 128 == 0, "codes ring alignment");
  static_assert(kEntryBytes % 128 == 0 && kS0Bytes % 128 == 0, "scale ring alignment");
  static_assert(kSmemBytes <= kMaxSmem, "shared memory budget");
};

struct PrefillParams {
  int64_t M, K, N;
  const uint16_t *s0, *b0;   // scales/biases (read directly only where they cannot be TMA-staged)
  const uint16_t *s1, *b1;
  int ng0, ng1;              // groups per row
  GroupDiv gd0, gd1;
  int sb_tma0, sb_tma1;      // scale ring filled by TMA (else by plain loads)
  int variant;
  uint16_t *out;
  const uint16_t *res;       // single-operand form: [M, N] added to the accumulator before the rounding (or null)
  int m_tiles, num_tiles, k_steps;
  int sk_tiles;              // tiles [0, sk_tiles) are shared out stream-K style (0: none)
  float *ws_part;            // [grid][kPartFloats] partial accumulators of split tiles
  unsigned int *ws_ctrl;     // [0] launch epoch, [1] CTAs done in this launch
  unsigned int *ws_flags;    // [grid][4] epoch tag per epilogue warp: that warp's partial rows are written
  uint64_t timeout_ns;
};

// Work list of one CTA: segments, each a K range [kb0, kb1) of one output tile.
// Tiles [0, sk_tiles) are shared out stream-K style: their (tile, K step)
// units are cut into one contiguous, equal range per CTA, so a tile can be
// split between CTAs with neighbouring ranges; the other tiles go round-robin,
// whole, after them.  Ranges are handed out in reverse block order: the CTA
// that finishes a split tile (the one holding its K steps from 0, which it
// reaches last) waits only for CTAs with lower block indices, which start
// first.  A CTA's first segment may start inside a tile (it then contributes a
// partial accumulator); only its last stream-K segment may end inside one (it
// then finishes the tile).
struct Seg {
  int tile, kb0, kb1;
};

struct Sched {
  int64_t u1;        // end of this CTA's stream-K units
  int tile0, kbf;    // tile and K step of its first unit
  int n_sk, n_seg;   // stream-K segments, all segments
  __device__ __forceinline__ void init(const PrefillParams &p) {
    const int64_t G = gridDim.x, rev = G - 1 - blockIdx.x;
    const int64_t U = static_cast<int64_t>(p.sk_tiles) * p.k_steps;
    const int64_t u0 = U * rev / G;
    u1 = U * (rev + 1) / G;
    tile0 = static_cast<int>(u0 / p.k_steps);
    kbf = static_cast<int>(u0 - static_cast<int64_t>(tile0) * p.k_steps);
    n_sk = u1 > u0 ? static_cast<int>((u1 - 1) / p.k_steps) - tile0 + 1 : 0;
    const int dp = p.num_tiles - p.sk_tiles;   // whole tiles, round-robin
    n_seg = n_sk + (dp - static_cast<int>(blockIdx.x) + static_cast<int>(G) - 1) / static_cast<int>(G);
  }
  __device__ __forceinline__ Seg seg(int ls, const PrefillParams &p) const {
    if (ls < n_sk) {
      const int t = tile0 + ls;
      const int64_t hi = u1 - static_cast<int64_t>(t) * p.k_steps;
      return {t, ls == 0 ? kbf : 0, hi < p.k_steps ? static_cast<int>(hi) : p.k_steps};
    }
    return {p.sk_tiles + static_cast<int>(blockIdx.x) + (ls - n_sk) * static_cast<int>(gridDim.x), 0, p.k_steps};
  }
};

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned int *p, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int atom_add_acq_rel_gpu(unsigned int *p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ uint4 ld_global_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// Wait (every lane of the warp) until another CTA has published `tag` in
// `flag`.  Bounded like the mbarrier waits; the result is warp-uniform.
__device__ __forceinline__ bool flag_wait(const unsigned int *flag, unsigned int tag, volatile int *abort,
                                          uint64_t timeout_ns, unsigned int *err) {
  bool ok = true;
  if (ld_acquire_gpu(flag) != tag) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
      __nanosleep(128);
      if (ld_acquire_gpu(flag) == tag) break;
      if ((it & 15u) == 0) {
        if (*abort) {
          ok = false;
          break;
        }
        if (globaltimer_ns() - t0 > timeout_ns) {
          *abort = 1;
          atomicOr(err, DEVERR_TIMEOUT);
          ok = false;
          break;
        }
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void st_global_v4(void *p, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// 16 consecutive codes of one row (quarter q of a K step) -> two 16-byte
// chunks of bf16 weights, stored at the swizzled positions of chunks 2q and
// 2q+1 of B-tile row `row`.
template <int BITS, class A>
__device__ __forceinline__ void dequant16(uint32_t codes_addr, uint32_t s2, uint32_t b2, uint32_t brow_addr, int row,
                                          int q) {
  uint32_t w[BITS / 2 > 0 ? BITS / 2 : 1];   // 16 codes = BITS/2 words
  if constexpr (BITS == 2) {
    w[0] = ld_shared_u32(codes_addr);
  } else if constexpr (BITS == 4) {
    const uint2 v = ld_shared_v2(codes_addr);
    w[0] = v.x;
    w[1] = v.y;
  } else {
    const uint4 v = ld_shared_v4(codes_addr);
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {   // chunk i: codes 8i .. 8i+7 of the 16
    uint32_t o[4];
    if constexpr (BITS == 4) {
      Dequant8<4, A>::natural(w[i], s2, b2, o);
    } else if constexpr (BITS == 8) {
      Dequant8<8, A>::natural(w[2 * i], w[2 * i + 1], s2, b2, o);
    } else {
      Dequant8<2, A>::natural(w[0] >> (16 * i), s2, b2, o);
    }
    // 128-byte swizzle: 16-byte chunk c of row n lands at chunk c ^ (n mod 8)
    const int c = 2 * q + i;
    st_shared_v4(brow_addr + static_cast<uint32_t>((c ^ (row & 7)) << 4), make_uint4(o[0], o[1], o[2], o[3]));
  }
}

// SwiGLU epilogue of 16 (gate, up) accumulator pairs -> 8 packed pairs of T.
template <int VARIANT, class A>
__device__ __forceinline__ void epilogue16(const uint32_t (&g)[16], const uint32_t (&u)[16], uint32_t (&out)[8]) {
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    if (VARIANT == VAR_MATCH)
      out[e / 2] = swiglu_match2<A>(__uint_as_float(g[e]), __uint_as_float(g[e + 1]), __uint_as_float(u[e]),
                                    __uint_as_float(u[e + 1]));
    else
      out[e / 2] = A::pack2(swiglu_epilogue<A>(VARIANT, __uint_as_float(g[e]), __uint_as_float(u[e])),
                            swiglu_epilogue<A>(VARIANT, __uint_as_float(g[e + 1]), __uint_as_float(u[e + 1])));
  }
}

template <int BITS0, int BITS1, bool DUAL, class A>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_c0,
                   const __grid_constant__ CUtensorMap tm_c1, const __grid_constant__ CUtensorMap tm_s0,
                   const __grid_constant__ CUtensorMap tm_b0, const __grid_constant__ CUtensorMap tm_s1,
                   const __grid_constant__ CUtensorMap tm_b1, const PrefillParams p) {
  using C = Cfg<BITS0, BITS1, DUAL>;
  constexpr int Sx = C::kSx, Sb = C::kSb, Sc = C::kSc;
  constexpr int kOps = DUAL ? 2 : 1;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
  // The x and B rings advance together (slot k of both holds stage k mod 2):
  // one commit to b_empty releases both slots (the x producer waits on it
  // too).  Every barrier wait in the issuer's loop is shared-memory latency on
  // the tensor core's critical path, hence stages of two K steps.
  uint64_t *x_full = bars;              // x tiles of a stage landed (TMA bytes)
  uint64_t *b_full = x_full + Sx;       // B tiles of a stage written by all dequantisers
  uint64_t *b_empty = b_full + Sb;      // MMAs reading the x and B tiles completed
  uint64_t *c_full = b_empty + Sb;      // codes landed
  uint64_t *c_empty = c_full + Sc;      // codes consumed by all dequantisers
  uint64_t *s_full = c_empty + Sc;      // [op][2] scale entry landed
  uint64_t *s_empty = s_full + 4;       // [op][2] scale entry consumed
  // Accumulation: each segment's K range is split into chains of at most
  // kChainStages ring stages.  Chain 0 accumulates in TMEM buffer X, every later
  // chain in buffer Y, and the epilogue adds Y into X with f32 adds after each
  // of them.  Short tensor-core accumulation chains keep the rounding of the
  // stored projections close to a correctly rounded sum.  X of tile t is
  // buffer t%2, Y the other one, so roles swap every tile.
  uint64_t *acc_full = s_empty + 4;     // a chain that ends in Y (or a single-chain tile) is complete
  uint64_t *y_free = acc_full + 1;      // Y has been added into X (Y reusable)
  uint64_t *xacc_free = acc_full + 2;   // X has been read out (X reusable)
  uint64_t *mma_done = acc_full + 3;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  unsigned int *sk_tag_slot = reinterpret_cast<unsigned int *>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned int *err = &g_prefill_error;
  Sched S;
  S.init(p);
  // K steps per scale-ring entry of each operand (8 groups of gs codes)
  const int kpe0 = kGroupsPerEntry * p.gd0.gs / BK;
  const int kpe1 = kGroupsPerEntry * p.gd1.gs / BK;

  if constexpr (kDebugBounds) {
    debug_poison_smem(smem, C::kBarOff);   // every staging ring, before any copy lands
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < Sx; ++s) mbar_init(&x_full[s], 1);
    for (int s = 0; s < Sb; ++s) {
      mbar_init(&b_full[s], kDeqWarps);
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < Sc; ++s) {
      mbar_init(&c_full[s], 1);
      mbar_init(&c_empty[s], kDeqWarps);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], kDeqWarps / kOps);   // the warps that dequantise that operand
    }
    mbar_init(acc_full, 1);
    mbar_init(y_free, kEpiWarps);
    mbar_init(xacc_free, kEpiWarps);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    // this launch's tag for the split-tile flags: one more than the last
    // launch's (set by that launch's last CTA; never 0, the zero-filled state)
    unsigned int tag = 0;
    if (p.sk_tiles > 0) {
      tag = ld_acquire_gpu(p.ws_ctrl) + 1u;
      if (tag == 0) tag = 1;
    }
    *sk_tag_slot = tag;
    fence_mbar_init();
  }
  if (warp == kWarpTma && lane == 0) {
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_c0);
    if (p.sb_tma0) {
      prefetch_tensormap(&tm_s0);
      prefetch_tensormap(&tm_b0);
    }
    if (DUAL) {
      prefetch_tensormap(&tm_c1);
      if (p.sb_tma1) {
        prefetch_tensormap(&tm_s1);
        prefetch_tensormap(&tm_b1);
      }
    }
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
  const unsigned int sk_tag = *sk_tag_slot;
  if constexpr (kDebugBounds) {
    // every accumulator column := NaN before the first MMA (each epilogue warp
    // writes the 32 TMEM lanes of its quarter)
    if (warp >= kWarpEpi0) {
      const uint32_t q = static_cast<uint32_t>(warp & 3) * 32u;
      uint32_t nan16[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) nan16[e] = ~0u;
      for (uint32_t col = 0; col < kTmemCols; col += 16) tmem_st16(tmem_base + (q << 16) + col, nan16);
      tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  if (warp == kWarpTma) {
    // ------------------------------------------- codes and scale producer --
    // Warp-wide loop over this CTA's segments and their K steps; lane 0 issues
    // the TMA copies: the codes of every K step, and a scale entry (8 groups
    // per operand) wherever one starts -- at an entry boundary or at the
    // first K step of a segment.  Every step of this loop is on the critical
    // path of the whole CTA, so it keeps running positions instead of
    // dividing per K step.
    int n_c = 0;               // codes fills issued so far
    int n_e[2] = {0, 0};       // scale entries issued per operand
    bool ok = true;
    for (int ls = 0; ls < S.n_seg && ok; ++ls) {
      const Seg sg = S.seg(ls, p);
      const int n0_c = (sg.tile / p.m_tiles) * C::kOutCols;
      int epos[2], eidx[2];    // K step within the current entry, next entry index
      epos[0] = sg.kb0 % kpe0;
      eidx[0] = sg.kb0 / kpe0;
      epos[1] = DUAL ? sg.kb0 % kpe1 : 0;
      eidx[1] = DUAL ? sg.kb0 / kpe1 : 0;
      for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
        const int cs = n_c % Sc;
        if (!(ok = warp_wait(&c_empty[cs], ((n_c / Sc) & 1) ^ 1u, abort_flag, p.timeout_ns, err))) break;
        if (lane == 0) {
          uint8_t *dst = smem + C::kCOff + cs * C::kCodesBytes;
          mbar_arrive_expect_tx(&c_full[cs], C::kCodesBytes);
          debug_check((kb * BK * BITS0 / 32) % 4 == 0 && (kb * BK * BITS1 / 32) % 4 == 0, err);   // 16-byte x
          tma_load_2d(dst, &tm_c0, &c_full[cs], kb * BK * BITS0 / 32, n0_c);
          if (DUAL) tma_load_2d(dst + C::kC0Bytes, &tm_c1, &c_full[cs], kb * BK * BITS1 / 32, n0_c);
        }
        ++n_c;
#pragma unroll
        for (int op = 0; op < kOps; ++op) {
          const int kpe = op ? kpe1 : kpe0;
          const bool start = epos[op] == 0 || kb == sg.kb0;
          if (++epos[op] == kpe) epos[op] = 0;
          if (!start) continue;
          const int es = n_e[op] & 1;
          if (!(ok = warp_wait(&s_empty[op * 2 + es], ((n_e[op] >> 1) & 1) ^ 1u, abort_flag, p.timeout_ns,
                               err)))
            break;
          const int rows = op ? C::kRows1 : C::kRows0;
          uint8_t *sdst = smem + C::kSOff + es * C::kEntryBytes + (op ? 2 * C::kS0Bytes : 0);
          uint8_t *bdst = sdst + (op ? C::kS1Bytes : C::kS0Bytes);
          const int g0 = eidx[op]++ * kGroupsPerEntry;   // first group of the entry
          if (op ? p.sb_tma1 : p.sb_tma0) {
            if (lane == 0) {
              mbar_arrive_expect_tx(&s_full[op * 2 + es], 2 * rows * 2 * kGroupsPerEntry);
              debug_check(g0 % 8 == 0, err);   // 16-byte x (8 scales)
              tma_load_2d(sdst, op ? &tm_s1 : &tm_s0, &s_full[op * 2 + es], g0, n0_c);
              tma_load_2d(bdst, op ? &tm_b1 : &tm_b0, &s_full[op * 2 + es], g0, n0_c);
            }
          } else {
            // rows whose scale rows cannot be TMA-staged: plain loads
            const uint16_t *sgp = op ? p.s1 : p.s0;
            const uint16_t *bgp = op ? p.b1 : p.b0;
            const int ng = op ? p.ng1 : p.ng0;
            for (int idx = lane; idx < rows * kGroupsPerEntry; idx += 32) {
              const int r = idx / kGroupsPerEntry, gi = idx % kGroupsPerEntry;
              const int64_t row = static_cast<int64_t>(n0_c) + r;
              const int g = g0 + gi;
              uint16_t sv = 0, bv = 0;
              if (row < p.N && g < ng) {
                sv = __ldg(sgp + row * ng + g);
                bv = __ldg(bgp + row * ng + g);
              }
              st_shared_u16(smem_u32(sdst) + idx * 2, sv);
              st_shared_u16(smem_u32(bdst) + idx * 2, bv);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_full[op * 2 + es]);
          }
          ++n_e[op];
        }
        if (!ok) break;
      }
    }
    if (!ok && lane == 0) {
      // let the copies already issued land before the CTA's memory goes away
      for (int s = 0; s < Sc && s < n_c; ++s) {
        const int last = s + ((n_c - 1 - s) / Sc) * Sc;
        mbar_wait_drain(&c_full[s], (last / Sc) & 1, 100000000ull);
      }
      for (int op = 0; op < kOps; ++op)
        for (int e = n_e[op] - 2 < 0 ? 0 : n_e[op] - 2; e < n_e[op]; ++e)
          mbar_wait_drain(&s_full[op * 2 + (e & 1)], (e >> 1) & 1, 100000000ull);
    }
    __syncwarp();
  } else if (warp == kWarpX) {
    // ------------------------------------------------------- x producer ----
    if (lane == 0) {
      int n_x = 0;
      bool ok = true;
      for (int ls = 0; ls < S.n_seg && ok; ++ls) {
        const Seg sg = S.seg(ls, p);
        const int m0 = (sg.tile % p.m_tiles) * BM;
        for (int kb = sg.kb0; kb < sg.kb1; kb += kSub) {   // one stage: kSub K steps (fewer at the end)
          const int xs = n_x % Sx;
          const int nsub = sg.kb1 - kb < kSub ? sg.kb1 - kb : kSub;
          if (!mbar_wait(&b_empty[xs], ((n_x / Sx) & 1) ^ 1u, abort_flag, p.timeout_ns, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&x_full[xs], nsub * kXBytes);
          for (int j = 0; j < nsub; ++j) {
            debug_check(((kb + j) * BK) % 8 == 0, err);   // 16-byte x (8 activations)
            tma_load_2d(smem + C::kXOff + xs * C::kXStage + j * kXBytes, &tm_x, &x_full[xs], (kb + j) * BK, m0);
          }
          ++n_x;
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA's memory goes away
        for (int s = 0; s < Sx && s < n_x; ++s) {
          const int last = s + ((n_x - 1 - s) / Sx) * Sx;
          mbar_wait_drain(&x_full[s], (last / Sx) & 1, 100000000ull);
        }
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issue --
    if (lane == 0) {
      constexpr uint32_t kIdesc = umma_idesc_f16kind(UM, BN, A::kUmmaFormat);
      int n_x = 0, n_b = 0;
      bool ok = true;
      // Chains of at most kChainStages ring stages (see the accumulation note at
      // the barriers): chain 0 accumulates in X, chains 1.. in Y, and the
      // epilogue adds Y into X after each of them.  Completions per segment:
      // y_free and acc_full P each, xacc_free 1; y_base counts the y_free
      // completions of the earlier segments.
      int y_base = 0;
      for (int ls = 0; ls < S.n_seg && ok; ++ls) {
        const Seg sg = S.seg(ls, p);
        const int nst = (sg.kb1 - sg.kb0 + kSub - 1) / kSub;   // ring stages of this segment
        const int nc = (nst + kChainStages - 1) / kChainStages;
        const int clen = (nst + nc - 1) / nc;   // stages per chain (the last may be shorter)
        const int P = nc > 1 ? nc - 1 : 1;
        const uint32_t x_tmem = tmem_base + static_cast<uint32_t>((ls & 1) * kAccCols);
        const uint32_t y_tmem = tmem_base + static_cast<uint32_t>(((ls + 1) & 1) * kAccCols);
        int c = 0, cpos = 0;   // chain and stage within it
        for (int st = 0; st < nst; ++st) {
          const int kb = sg.kb0 + st * kSub;
          const int nsub = sg.kb1 - kb < kSub ? sg.kb1 - kb : kSub;
          if (cpos == 0) {
            // X of this segment was Y of the previous one, and Y was its X:
            // chain 0 needs the previous segment's last X += Y done, chain 1
            // the previous segment's X read out, chain c >= 2 the X += Y of
            // chain c-1
            uint64_t *bar = nullptr;
            int n = 0;
            if (c == 0 && ls > 0) {
              bar = y_free;
              n = y_base - 1;
            } else if (c == 1 && ls > 0) {
              bar = xacc_free;
              n = ls - 1;
            } else if (c >= 2) {
              bar = y_free;
              n = y_base + c - 2;
            }
            if (bar != nullptr) {
              if (!mbar_wait(bar, static_cast<uint32_t>(n & 1), abort_flag, p.timeout_ns, err)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
          }
          const uint32_t d_tmem = c == 0 ? x_tmem : y_tmem;
          const bool chain_start = cpos == 0;
          const int bs = n_b % Sb;
          if (!mbar_wait(&x_full[bs], (n_b / Sb) & 1, abort_flag, p.timeout_ns, err) ||
              !mbar_wait(&b_full[bs], (n_b / Sb) & 1, abort_flag, p.timeout_ns, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int j = 0; j < nsub; ++j) {
            // K step j of the stage: the x tile's two 128-row halves (16 KB
            // apart) against the same B tile
            const uint32_t xa = smem_u32(smem + C::kXOff + bs * C::kXStage + j * kXBytes);
            const uint64_t adesc0 = umma_desc_sw128(xa);
            const uint64_t adesc1 = umma_desc_sw128(xa + UM * 128);
            const uint64_t bdesc = umma_desc_sw128(smem_u32(smem + C::kBOff + bs * C::kBStage + j * kBBytes));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              // +32 bytes of K per step inside the 128-byte swizzle atom
              const uint32_t acc = (chain_start && j == 0 && kk == 0) ? 0u : 1u;
              umma_bf16(d_tmem, adesc0 + 2 * kk, bdesc + 2 * kk, kIdesc, acc);
              umma_bf16(d_tmem + BN, adesc1 + 2 * kk, bdesc + 2 * kk, kIdesc, acc);
            }
          }
          umma_commit(&b_empty[bs]);
          ++n_x;
          ++n_b;
          if (++cpos == clen || st + 1 == nst) {   // chain c complete
            if (c >= 1 || nc == 1) umma_commit(acc_full);
            ++c;
            cpos = 0;
          }
        }
        y_base += P;
      }
      if (!ok) {
        umma_commit(mma_done);
        mbar_wait_drain(mma_done, 0, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp < kWarpEpi0) {
    // ---------------------------------------------------------- dequantise --
    // Warp dw owns B rows 8 dw .. 8 dw + 7; lane = (row, quarter): lane / 4 is
    // the row, lane % 4 picks codes 16 q .. 16 q + 15 of the K step.  In the
    // fused form warps 0-7 hold the gate rows and warps 8-15 the up rows.
    const int dw = warp - kWarpDeq0;
    const int op = DUAL ? (dw >= kDeqWarps / 2) : 0;   // warp-uniform
    const int row = dw * 8 + (lane >> 2);                // B-tile row
    const int q = lane & 3;
    const int r_op = DUAL ? (row & (BN / 2 - 1)) : row;  // row within the operand's rows
    const int kpe = op ? kpe1 : kpe0;
    const GroupDiv gd = op ? p.gd1 : p.gd0;
    const int bits = op ? BITS1 : BITS0;
    const uint32_t c_row = static_cast<uint32_t>(C::kCOff + (op ? C::kC0Bytes : 0) +
                                                 r_op * (op ? C::kC1Pitch : C::kC0Pitch) + q * 2 * bits);
    const uint32_t s_row = static_cast<uint32_t>(C::kSOff + (op ? 2 * C::kS0Bytes : 0) + r_op * 16);
    const uint32_t b_row = s_row + static_cast<uint32_t>(op ? C::kS1Bytes : C::kS0Bytes);
    const uint32_t sbase = smem_u32(smem);
    int n_c = 0, n_b = 0, n_e = 0;
    bool ok = true;
    for (int ls = 0; ls < S.n_seg && ok; ++ls) {
      const Seg sg = S.seg(ls, p);
      int epos = sg.kb0 % kpe;   // K step within the current scale entry
      for (int kb = sg.kb0; kb < sg.kb1 && ok; kb += kSub) {   // one B stage
        const int nsub = sg.kb1 - kb < kSub ? sg.kb1 - kb : kSub;
        const int bs = n_b % Sb;
        for (int j = 0; j < nsub; ++j) {
          const int kbj = kb + j;
          const int es = n_e & 1;
          // a scale entry starts at an entry boundary or at the segment's first K step
          if ((epos == 0 || kbj == sg.kb0) &&
              !(ok = warp_wait(&s_full[op * 2 + es], (n_e >> 1) & 1, abort_flag, p.timeout_ns, err)))
            break;
          const int cs = n_c % Sc;
          if (!(ok = warp_wait(&c_full[cs], (n_c / Sc) & 1, abort_flag, p.timeout_ns, err))) break;
          if (j == 0 && !(ok = warp_wait(&b_empty[bs], ((n_b / Sb) & 1) ^ 1u, abort_flag, p.timeout_ns, err)))
            break;
          // scale and bias of this thread's 16 codes (one group: gs is a multiple of 32)
          const uint32_t gi = gd(static_cast<uint32_t>(epos * BK + 16 * q));
          const uint32_t eoff = static_cast<uint32_t>(es * C::kEntryBytes) + gi * 2;
          const uint32_t s2 = splat_bf16(static_cast<uint16_t>(ld_shared_u16(sbase + s_row + eoff)));
          const uint32_t b2 = splat_bf16(static_cast<uint16_t>(ld_shared_u16(sbase + b_row + eoff)));
          const uint32_t caddr = sbase + c_row + static_cast<uint32_t>(cs * C::kCodesBytes);
          const uint32_t baddr =
              sbase + static_cast<uint32_t>(C::kBOff + bs * C::kBStage + j * kBBytes + row * 128);
          if (op == 0)
            dequant16<BITS0, A>(caddr, s2, b2, baddr, row, q);
          else
            dequant16<BITS1, A>(caddr, s2, b2, baddr, row, q);
          // B stores visible to the tensor core, code reads done before the
          // codes slot is refilled (both proxies)
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&c_empty[cs]);
          ++n_c;
          if (++epos == kpe || kbj + 1 == sg.kb1) {
            if (lane == 0) mbar_arrive(&s_empty[op * 2 + es]);
            ++n_e;
            epos = 0;
          }
        }
        if (!ok) break;
        if (lane == 0) mbar_arrive(&b_full[bs]);
        ++n_b;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int quarter = warp & 3;   // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;
    const bool vec_ok = (p.N % 8) == 0;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    bool ok = true;
    int a_base = 0;   // acc_full completions of the earlier segments
    for (int ls = 0; ls < S.n_seg && ok; ++ls) {
      const Seg sg = S.seg(ls, p);
      const int t = sg.tile;
      const int nst = (sg.kb1 - sg.kb0 + kSub - 1) / kSub;   // ring stages of this segment
      const int nc = (nst + kChainStages - 1) / kChainStages;
      const int P = nc > 1 ? nc - 1 : 1;   // acc_full completions of this segment
      const uint32_t tbase = lane_base + static_cast<uint32_t>((ls & 1) * kAccCols);          // X
      const uint32_t ybase = lane_base + static_cast<uint32_t>(((ls + 1) & 1) * kAccCols);    // Y
      for (int q = 0; q < P; ++q) {
        // the epilogue idles for most of a chain: wait without spinning
        if (!(ok = warp_wait_lazy(acc_full, static_cast<uint32_t>((a_base + q) & 1), abort_flag, p.timeout_ns,
                                  err, 500)))
          break;
        tc_fence_after();
        if (nc > 1) {
          // X += Y over all columns, f32 adds rounded to nearest.  The next
          // chain waits for this pass, so it keeps four loads in flight per
          // wait (32 columns).
#pragma unroll 1
          for (int c0 = 0; c0 < kAccCols; c0 += 32) {   // both x halves' accumulators
            uint32_t ra[16], rb[16], rc[16], rd[16];
            __syncwarp();
            tmem_ld16(tbase + c0, ra);
            tmem_ld16(ybase + c0, rb);
            tmem_ld16(tbase + c0 + 16, rc);
            tmem_ld16(ybase + c0 + 16, rd);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              ra[e] = __float_as_uint(__uint_as_float(ra[e]) + __uint_as_float(rb[e]));
              rc[e] = __float_as_uint(__uint_as_float(rc[e]) + __uint_as_float(rd[e]));
            }
            tmem_st16(tbase + c0, ra);
            tmem_st16(tbase + c0 + 16, rc);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(y_free);   // Y may take the next chain
      }
      a_base += P;
      if (!ok) break;
      const int64_t m_tile0 = static_cast<int64_t>(t % p.m_tiles) * BM;
      if (sg.kb0 > 0) {
        // Contributor: this CTA holds K steps [kb0, kb1) of a tile another CTA
        // finishes.  Publish the f32 accumulator (rows below M) in this CTA's
        // partial slot, laid out [half][16-column chunk][4-column quad][row][4]
        // so that every 16-byte store (and load) of a warp covers 512
        // contiguous bytes, then flag this warp's rows.
        float *part = p.ws_part + static_cast<size_t>(blockIdx.x) * kPartFloats;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          const bool live = m_tile0 + h * UM + row < p.M;
#pragma unroll 1
          for (int j = 0; j < BN / 16; ++j) {
            uint32_t ra[16];
            __syncwarp();   // tcgen05.ld is warp-collective
            tmem_ld16(tbase + static_cast<uint32_t>(h * BN + 16 * j), ra);
            tmem_ld_wait();
            if (live) {
              float *dst = part + (static_cast<size_t>(h * (BN / 16) + j) * 4 * UM + row) * 4;
              debug_check(static_cast<size_t>(dst - part) + 3 * UM * 4 + 4 <= static_cast<size_t>(kPartFloats), err);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                st_global_v4(dst + i * UM * 4, make_uint4(ra[4 * i], ra[4 * i + 1], ra[4 * i + 2], ra[4 * i + 3]));
            }
          }
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(p.ws_flags + blockIdx.x * 4 + quarter, sk_tag);
      } else {
        // A tile that ends inside this segment's range is complete here; one
        // that continues past kb1 is finished here with the partials of the
        // CTAs holding its later K steps (lower block indices, in order).
        int n_parts = 0;
        if (sg.kb1 < p.k_steps) {
          const int64_t G = gridDim.x, rev = G - 1 - blockIdx.x;
          const int64_t U = static_cast<int64_t>(p.sk_tiles) * p.k_steps;
          const int64_t tile_end = static_cast<int64_t>(t + 1) * p.k_steps;
          for (int64_t rc = rev + 1; rc < G && U * rc / G < tile_end; ++rc) {
            const int c = static_cast<int>(G - 1 - rc);
            if (!(ok = flag_wait(p.ws_flags + c * 4 + quarter, sk_tag, abort_flag, p.timeout_ns, err))) break;
            ++n_parts;
          }
          if (!ok) break;
        }
        const int64_t n0 = static_cast<int64_t>(t / p.m_tiles) * C::kOutCols;
        // accumulator h holds x rows m0 + 128 h + (TMEM lane); in the fused form
        // columns 0-63 are gate, 64-127 up
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          const int64_t m = m_tile0 + h * UM + row;
          uint16_t *orow = p.out + m * p.N;
          const uint32_t hbase = tbase + static_cast<uint32_t>(h * BN);
#pragma unroll 1
          for (int c0 = 0; c0 < C::kOutCols; c0 += 16) {
            uint32_t ra[16], rb[16];
            __syncwarp();   // tcgen05.ld is warp-collective
            tmem_ld16(hbase + c0, ra);
            if (DUAL) tmem_ld16(hbase + BN / 2 + c0, rb);
            tmem_ld_wait();
            if (m < p.M) {
              for (int r = 1; r <= n_parts; ++r) {
                const float *src = p.ws_part + static_cast<size_t>(blockIdx.x - r) * kPartFloats +
                                   (static_cast<size_t>(h * (BN / 16) + c0 / 16) * 4 * UM + row) * 4;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const uint4 v = ld_global_v4(src + i * UM * 4);
                  ra[4 * i] = __float_as_uint(__uint_as_float(ra[4 * i]) + __uint_as_float(v.x));
                  ra[4 * i + 1] = __float_as_uint(__uint_as_float(ra[4 * i + 1]) + __uint_as_float(v.y));
                  ra[4 * i + 2] = __float_as_uint(__uint_as_float(ra[4 * i + 2]) + __uint_as_float(v.z));
                  ra[4 * i + 3] = __float_as_uint(__uint_as_float(ra[4 * i + 3]) + __uint_as_float(v.w));
                }
                if (DUAL) {
                  const float *usrc = src + static_cast<size_t>(BN / 2 / 16) * 4 * UM * 4;   // up chunk
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    const uint4 v = ld_global_v4(usrc + i * UM * 4);
                    rb[4 * i] = __float_as_uint(__uint_as_float(rb[4 * i]) + __uint_as_float(v.x));
                    rb[4 * i + 1] = __float_as_uint(__uint_as_float(rb[4 * i + 1]) + __uint_as_float(v.y));
                    rb[4 * i + 2] = __float_as_uint(__uint_as_float(rb[4 * i + 2]) + __uint_as_float(v.z));
                    rb[4 * i + 3] = __float_as_uint(__uint_as_float(rb[4 * i + 3]) + __uint_as_float(v.w));
                  }
                }
              }
              uint32_t packed[8];
              if (DUAL) {
                // one variant per launch: dispatch once, then 16 branch-free elements
                switch (p.variant) {
                  case VAR_MATCH: epilogue16<VAR_MATCH, A>(ra, rb, packed); break;
                  case VAR_F32: epilogue16<VAR_F32, A>(ra, rb, packed); break;
                  case VAR_DEBUG_GATE: epilogue16<VAR_DEBUG_GATE, A>(ra, rb, packed); break;
                  default: epilogue16<VAR_DEBUG_UP, A>(ra, rb, packed); break;
                }
              } else {
                // y = T(acc + r): the residual joins the f32 accumulator, one rounding
                uint32_t r2[8];
                const int64_t rcol = n0 + c0;
                if (p.res == nullptr) {
#pragma unroll
                  for (int e = 0; e < 8; ++e) r2[e] = 0u;   // +0 in both halves, bf16 and f16
                } else if (vec_ok && rcol + 16 <= p.N) {
                  const uint4 v0 = ld_global_v4(p.res + m * p.N + rcol);
                  const uint4 v1 = ld_global_v4(p.res + m * p.N + rcol + 8);
                  r2[0] = v0.x; r2[1] = v0.y; r2[2] = v0.z; r2[3] = v0.w;
                  r2[4] = v1.x; r2[5] = v1.y; r2[6] = v1.z; r2[7] = v1.w;
                } else {
#pragma unroll
                  for (int e = 0; e < 8; ++e) {
                    const uint32_t lo = rcol + 2 * e < p.N ? p.res[m * p.N + rcol + 2 * e] : 0u;
                    const uint32_t hi = rcol + 2 * e + 1 < p.N ? p.res[m * p.N + rcol + 2 * e + 1] : 0u;
                    r2[e] = lo | (hi << 16);
                  }
                }
#pragma unroll
                for (int e = 0; e < 16; e += 2)
                  packed[e / 2] = A::pack2(__uint_as_float(ra[e]) + A::lo(r2[e / 2]),
                                           __uint_as_float(ra[e + 1]) + A::hi(r2[e / 2]));
              }
              const int64_t col = n0 + c0;
              // columns past N (a ragged last tile) are skipped element by element below
              debug_check(m < p.M && col % 16 == 0, err);
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
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(xacc_free);   // X may take the next segment's chains 1..
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  if (p.sk_tiles > 0 && threadIdx.x == 0) {
    // the last CTA of the launch to get here publishes its tag as the epoch the
    // next launch counts on from (every CTA read the epoch before arriving)
    if (atom_add_acq_rel_gpu(p.ws_ctrl + 1, 1u) == gridDim.x - 1) {
      *reinterpret_cast<volatile unsigned int *>(p.ws_ctrl + 1) = 0u;
      st_release_gpu(p.ws_ctrl, sk_tag);
    }
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

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Scale/bias rows of an operand can be TMA-staged when their row stride and
// base are 16-byte aligned (K/gs a multiple of 8).
bool scales_tma_ok(const QuantOperand &op, int64_t K) {
  return (K / op.gs) % kGroupsPerEntry == 0 && aligned16(op.s) && aligned16(op.b);
}

bool encode_scales(CUtensorMap *s, CUtensorMap *b, const QuantOperand &op, int64_t K, int64_t N, int rows) {
  const uint64_t ng = static_cast<uint64_t>(K / op.gs);
  return encode_2d(s, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, op.s, ng, N, kGroupsPerEntry, rows,
                   CU_TENSOR_MAP_SWIZZLE_NONE) &&
         encode_2d(b, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, op.b, ng, N, kGroupsPerEntry, rows,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Workspace layout: [0] epoch, [1] CTAs done; flags from byte 256 (4 per CTA);
// partial accumulators from a 1 KB boundary, kPartFloats per CTA.
constexpr size_t kFlagsOff = 256;
size_t header_bytes(int num_sms) { return (kFlagsOff + 16 * static_cast<size_t>(num_sms) + 1023) & ~size_t(1023); }

// Stream-K split.  With at least as many tiles as SMs, the ragged last wave
// (rem = tiles mod SMs tiles) is shared out in equal K ranges first and the
// whole waves follow, so a finisher's partial reads and its epilogue overlap
// the MMAs of its next whole tile.  Where the ragged wave alone would give each
// CTA less than half a tile of K steps, one whole wave joins the split (ranges
// of at least one tile).  With fewer tiles than SMs all tiles are split, every
// CTA taking at least kSkMinUnits K steps.  Auto mode splits only where whole
// tiles would leave more than kSkMaxIdle of the SM time idle (more for fewer
// tiles than SMs, where the finisher's epilogue cannot be hidden), and not
// where a ragged wave of more than half the SMs is followed by fewer than
// kSkMinWaves whole waves: there a finisher's epilogue (partial reads, then
// the output) can hold up the second accumulation chain of its next tile by
// more than the split saves (measured: 256 tiles of 32 K steps on 152 SMs).
constexpr double kSkMaxIdle = 0.01;
constexpr double kSkMaxIdleFew = 0.25;
constexpr int64_t kSkMinUnits = 8;
constexpr int64_t kSkMinWaves = 3;

void plan_split(int64_t tiles, int64_t k_steps, int num_sms, int mode, bool have_ws, int *grid, int *sk_tiles) {
  const int64_t G = num_sms;
  *grid = static_cast<int>(tiles < G ? tiles : G);
  *sk_tiles = 0;
  if (!have_ws || mode == QSW_STREAM_K_OFF || G < 2) return;
  const double busy = static_cast<double>(tiles) / static_cast<double>(((tiles + G - 1) / G) * G);
  const bool auto_mode = mode == QSW_STREAM_K_AUTO;
  if (tiles >= G) {
    const int64_t rem = tiles % G;
    if (rem == 0 || (auto_mode && busy >= 1.0 - kSkMaxIdle)) return;
    if (auto_mode && 2 * rem >= G && tiles / G < kSkMinWaves) return;
    *grid = static_cast<int>(G);
    *sk_tiles = static_cast<int>(2 * rem >= G ? rem : rem + G);
    return;
  }
  if (auto_mode && busy >= 1.0 - kSkMaxIdleFew) return;
  const int64_t units = tiles * k_steps;
  int64_t g = mode == QSW_STREAM_K_ALWAYS ? units : units / kSkMinUnits;
  if (g > G) g = G;
  if (g <= tiles) return;
  *grid = static_cast<int>(g);
  *sk_tiles = static_cast<int>(tiles);
}

template <int BITS0, int BITS1, bool DUAL, class A>
cudaError_t launch_impl(const void *x, int64_t M, int64_t K, int64_t N, const QuantOperand &op0,
                        const QuantOperand *op1, int variant, void *out, const void *res, cudaStream_t stream,
                        uint64_t timeout_ns, int num_sms, const SplitWorkspace &ws) {
  using C = Cfg<BITS0, BITS1, DUAL>;
  CUtensorMap tm_x, tm_c0, tm_c1, tm_s0, tm_b0, tm_s1, tm_b1;
  const CUtensorMapDataType x_type = A::kId == ActF16::kId ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!encode_2d(&tm_x, x_type, 2, x, K, M, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_2d(&tm_c0, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, op0.w, K * BITS0 / 32, N, BK * BITS0 / 32, C::kRows0,
                 CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  tm_c1 = tm_c0;
  if (DUAL && !encode_2d(&tm_c1, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, op1->w, K * BITS1 / 32, N, BK * BITS1 / 32,
                         C::kRows1, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;

  PrefillParams p{};
  p.M = M;
  p.K = K;
  p.N = N;
  p.s0 = op0.s;
  p.b0 = op0.b;
  p.s1 = DUAL ? op1->s : op0.s;
  p.b1 = DUAL ? op1->b : op0.b;
  p.ng0 = static_cast<int>(K / op0.gs);
  p.ng1 = static_cast<int>(K / (DUAL ? op1->gs : op0.gs));
  p.gd0 = GroupDiv::make(op0.gs);
  p.gd1 = GroupDiv::make(DUAL ? op1->gs : op0.gs);
  if (N * (K / (op0.gs < p.gd1.gs ? op0.gs : p.gd1.gs)) >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  p.sb_tma0 = scales_tma_ok(op0, K) ? 1 : 0;
  p.sb_tma1 = DUAL ? (scales_tma_ok(*op1, K) ? 1 : 0) : 0;
  tm_s0 = tm_b0 = tm_s1 = tm_b1 = tm_c0;   // placeholders where no scale map is used
  if (p.sb_tma0 && !encode_scales(&tm_s0, &tm_b0, op0, K, N, C::kRows0)) return cudaErrorInvalidValue;
  if (p.sb_tma1 && !encode_scales(&tm_s1, &tm_b1, *op1, K, N, C::kRows1)) return cudaErrorInvalidValue;
  p.variant = variant;
  p.out = static_cast<uint16_t *>(out);
  p.res = DUAL ? nullptr : static_cast<const uint16_t *>(res);
  p.m_tiles = static_cast<int>((M + BM - 1) / BM);
  const int64_t n_tiles = (N + C::kOutCols - 1) / C::kOutCols;
  const int64_t tiles = static_cast<int64_t>(p.m_tiles) * n_tiles;
  if (tiles > (int64_t(1) << 30)) return cudaErrorInvalidValue;
  p.num_tiles = static_cast<int>(tiles);
  p.k_steps = static_cast<int>((K + BK - 1) / BK);
  p.timeout_ns = timeout_ns;
  int grid = 0;
  const bool have_ws = ws.ptr != nullptr && ws.bytes >= prefill_workspace_bytes(num_sms);
  plan_split(tiles, p.k_steps, num_sms, ws.mode, have_ws, &grid, &p.sk_tiles);
  if (p.sk_tiles > 0) {
    uint8_t *base = static_cast<uint8_t *>(ws.ptr);
    p.ws_ctrl = reinterpret_cast<unsigned int *>(base);
    p.ws_flags = reinterpret_cast<unsigned int *>(base + kFlagsOff);
    p.ws_part = reinterpret_cast<float *>(base + header_bytes(num_sms));
  }

  // opt in to the large shared-memory carve-out once per device and instantiation
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(attr_done.load() & (uint64_t(1) << dev))) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<BITS0, BITS1, DUAL, A>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(uint64_t(1) << dev);
  }
  prefill_kernel<BITS0, BITS1, DUAL, A><<<grid, kThreads, C::kSmemBytes, stream>>>(tm_x, tm_c0, tm_c1, tm_s0, tm_b0,
                                                                                 tm_s1, tm_b1, p);
  return cudaGetLastError();
}

template <int BITS0, class A>
cudaError_t dual_bits1(int bits1, const void *x, int64_t M, int64_t K, int64_t N, const QuantOperand &op0,
                       const QuantOperand *op1, int variant, void *out, const void *res, cudaStream_t stream,
                       uint64_t timeout_ns, int num_sms, const SplitWorkspace &ws) {
  switch (bits1) {
    case 2: return launch_impl<BITS0, 2, true, A>(x, M, K, N, op0, op1, variant, out, res, stream, timeout_ns, num_sms, ws);
    case 4: return launch_impl<BITS0, 4, true, A>(x, M, K, N, op0, op1, variant, out, res, stream, timeout_ns, num_sms, ws);
    case 8: return launch_impl<BITS0, 8, true, A>(x, M, K, N, op0, op1, variant, out, res, stream, timeout_ns, num_sms, ws);
    default: return cudaErrorInvalidValue;
  }
}

template <class A>
cudaError_t launch_act(const void *x, int64_t M, int64_t K, int64_t N, const QuantOperand &op0,
                       const QuantOperand *op1, int variant, void *out, const void *res, cudaStream_t stream,
                       uint64_t timeout_ns, int num_sms, const SplitWorkspace &ws) {
  if (op1) {
    switch (op0.bits) {
      case 2: return dual_bits1<2, A>(op1->bits, x, M, K, N, op0, op1, variant, out, res, stream, timeout_ns, num_sms, ws);
      case 4: return dual_bits1<4, A>(op1->bits, x, M, K, N, op0, op1, variant, out, res, stream, timeout_ns, num_sms, ws);
      case 8: return dual_bits1<8, A>(op1->bits, x, M, K, N, op0, op1, variant, out, res, stream, timeout_ns, num_sms, ws);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (op0.bits) {
    case 2: return launch_impl<2, 2, false, A>(x, M, K, N, op0, nullptr, variant, out, res, stream, timeout_ns, num_sms, ws);
    case 4: return launch_impl<4, 4, false, A>(x, M, K, N, op0, nullptr, variant, out, res, stream, timeout_ns, num_sms, ws);
    case 8: return launch_impl<8, 8, false, A>(x, M, K, N, op0, nullptr, variant, out, res, stream, timeout_ns, num_sms, ws);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t prefill_workspace_bytes(int num_sms) {
  return num_sms > 0 ? header_bytes(num_sms) + static_cast<size_t>(num_sms) * kPartFloats * sizeof(float) : 0;
}

cudaError_t prefill_static_workspace(int num_sms, cudaStream_t stream, void **ptr, size_t *bytes) {
  static_assert(kPartFloats == 2 * 128 * 128, "static scratch slot size");
  *ptr = nullptr;
  *bytes = 0;
  if (num_sms <= 0 || num_sms > kStaticScratchSms || prefill_workspace_bytes(num_sms) > kStaticScratchBytes)
    return cudaSuccess;   // whole tiles only
  static void *addr[64];
  static std::atomic<bool> ready[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!ready[dev].load(std::memory_order_acquire)) {
    // First use on this device: resolve the array's device address and zero
    // its header (epoch, done count, flags) on the caller's stream.  A failure
    // leaves the device unset, so the next call tries again.
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev].load(std::memory_order_relaxed)) {
      void *a = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&a, g_static_scratch);
      if (e != cudaSuccess) return e;
      e = cudaMemsetAsync(a, 0, header_bytes(num_sms), stream);
      if (e != cudaSuccess) return e;
      addr[dev] = a;
      ready[dev].store(true, std::memory_order_release);
    }
  }
  *ptr = addr[dev];
  *bytes = kStaticScratchBytes;
  return cudaSuccess;
}

cudaError_t launch_prefill(const void *x, int64_t M, int64_t K, int64_t N, const QuantOperand &op0,
                           const QuantOperand *op1, int variant, int act, void *out, const void *residual,
                           cudaStream_t stream, uint64_t timeout_ns, int num_sms, const SplitWorkspace &ws) {
  if (act == ActF16::kId)
    return launch_act<ActF16>(x, M, K, N, op0, op1, variant, out, residual, stream, timeout_ns, num_sms, ws);
  if (act == ActBf16::kId)
    return launch_act<ActBf16>(x, M, K, N, op0, op1, variant, out, residual, stream, timeout_ns, num_sms, ws);
  return cudaErrorInvalidValue;
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
