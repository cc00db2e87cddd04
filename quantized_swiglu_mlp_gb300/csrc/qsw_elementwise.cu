// Elementwise out = silu(g) * u over bf16 arrays: the last step of the unfused
// path (mlx-bun pages, src/model/qwen3.ts, Qwen3MLP.forward: sigmoid, then two
// multiplies, each producing a bf16 array).  HBM-bound: 16-byte loads and
// stores, grid sized to the SM count.
#include "qsw_device.cuh"
#include "qsw_internal.h"

namespace qsw {
namespace {

// Two elements; MATCH takes the paired form the tensor-core epilogue uses, the
// tail kernel below the scalar form (the two are bit-identical).
template <class A>
__device__ __forceinline__ uint32_t silu_mul_pair(int variant, uint32_t g, uint32_t u) {
  if (variant == VAR_MATCH) return swiglu_match2<A>(A::lo(g), A::hi(g), A::lo(u), A::hi(u));
  return A::pack2(swiglu_epilogue<A>(variant, A::lo(g), A::lo(u)), swiglu_epilogue<A>(variant, A::hi(g), A::hi(u)));
}

template <class A>
__global__ void silu_mul_vec_kernel(const uint4 *__restrict__ g, const uint4 *__restrict__ u, int64_t n8,
                                    int variant, uint4 *out) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 a = __ldg(g + i), b = __ldg(u + i);
    out[i] = make_uint4(silu_mul_pair<A>(variant, a.x, b.x), silu_mul_pair<A>(variant, a.y, b.y),
                        silu_mul_pair<A>(variant, a.z, b.z), silu_mul_pair<A>(variant, a.w, b.w));
  }
}

template <class A>
__global__ void silu_mul_tail_kernel(const uint16_t *g, const uint16_t *u, int64_t begin, int64_t n, int variant,
                                     uint16_t *out) {
  const int64_t i = begin + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (i < n) {
    const float gv = A::lo(g[i]), uv = A::lo(u[i]);
    out[i] = A::store(swiglu_epilogue<A>(variant, gv, uv));
  }
}

}  // namespace

template <class A>
cudaError_t launch_act(const void *g, const void *u, int64_t n, int variant, void *out, cudaStream_t stream) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t n8 = n / 8;
  if (n8 > 0) {
    const int threads = 256;
    int64_t blocks = (n8 + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    silu_mul_vec_kernel<A><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        static_cast<const uint4 *>(g), static_cast<const uint4 *>(u), n8, variant, static_cast<uint4 *>(out));
  }
  const int64_t rest = n - n8 * 8;
  if (rest > 0) {
    silu_mul_tail_kernel<A><<<1, 32, 0, stream>>>(static_cast<const uint16_t *>(g), static_cast<const uint16_t *>(u),
                                                  n8 * 8, n, variant, static_cast<uint16_t *>(out));
  }
  return cudaGetLastError();
}

cudaError_t launch_silu_mul(const void *g, const void *u, int64_t n, int variant, int act, void *out,
                            cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  if (act == ActF16::kId) return launch_act<ActF16>(g, u, n, variant, out, stream);
  if (act == ActBf16::kId) return launch_act<ActBf16>(g, u, n, variant, out, stream);
  return cudaErrorInvalidValue;
}

}  // namespace qsw
