// Host-side declarations shared by the qswiglu translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "qswiglu.h"

namespace qsw {

// One affine-quantised operand: packed codes [rows, K*bits/32], bf16
// scales/biases [rows, K/gs].
struct QuantOperand {
  const uint32_t *w;
  const uint16_t *s;
  const uint16_t *b;
  int gs;
  int bits;
};

// `act` (every launcher): the activation dtype, QSW_ACT_BF16 or QSW_ACT_F16 --
// x, scales, biases and the result share it.  `residual` (single-operand form
// only, else ignored): null, or [M, N] of that dtype added to the f32
// accumulator before the one rounding; it may be the output buffer itself.
//
// Small-M kernel: rows of x up to 32.  `dual` selects the fused SwiGLU
// (gate + up, epilogue `variant`) or a single quantised linear (y = bf16(x.W^T)).
// `early_weights`: launch as a programmatic dependent and stream weights
// before waiting for the preceding work (the caller guarantees that no earlier
// work on the stream writes the weight arrays).
cudaError_t launch_gemv(const void *x, int64_t M, int64_t K, int64_t N, const QuantOperand &op0,
                        const QuantOperand *op1, int variant, int act, void *out, const void *residual,
                        cudaStream_t stream, uint64_t timeout_ns, int num_sms, bool early_weights);

// Test hook: the next small-M launch never fills its CTAs' first slot, so
// that the waits on it run out.
void gemv_withhold_next();

// Warp-streamed small-M kernel (M <= 16): same arguments and result as
// launch_gemv; it has no spin waits.
cudaError_t launch_gemv_stream(const void *x, int64_t M, int64_t K, int64_t N, const QuantOperand &op0,
                               const QuantOperand *op1, int variant, int act, void *out, const void *residual,
                               cudaStream_t stream, int num_sms, bool early_weights);

// Whether the warp-streamed kernel applies (M <= 16, K <= 16384, x, the
// partial sums and the warps' rings fit in shared memory).
bool gemv_stream_fits(int64_t M, int64_t K, int64_t N, const QuantOperand &op0, const QuantOperand *op1,
                      int num_sms);

// Whether the slot-ring small-M kernel can stage rows of length K (else the
// tensor-core kernel serves every M).
bool gemv_fits(int64_t M, int64_t K, int64_t N, const QuantOperand &op0, const QuantOperand *op1, int num_sms);

// Stream-K workspace of the tensor-core kernel: null ptr (or fewer than
// prefill_workspace_bytes() bytes) means whole tiles only.
struct SplitWorkspace {
  void *ptr;
  size_t bytes;
  int mode;   // qsw_stream_k_mode
};

size_t prefill_workspace_bytes(int num_sms);

// The library's static stream-K workspace on the current device (a device
// array of the library, not an allocation); *ptr stays null where it is too
// small for the SM count.  Its header is zeroed on `stream` at first use.
cudaError_t prefill_static_workspace(int num_sms, cudaStream_t stream, void **ptr, size_t *bytes);

// Tensor-core kernel (tcgen05 + TMA), any M.
cudaError_t launch_prefill(const void *x, int64_t M, int64_t K, int64_t N, const QuantOperand &op0,
                           const QuantOperand *op1, int variant, int act, void *out, const void *residual,
                           cudaStream_t stream, uint64_t timeout_ns, int num_sms, const SplitWorkspace &ws);

cudaError_t launch_silu_mul(const void *g, const void *u, int64_t n, int variant, int act, void *out,
                            cudaStream_t stream);

// Largest M the small-M kernel accepts.
constexpr int64_t kGemvMaxM = 32;

}  // namespace qsw
