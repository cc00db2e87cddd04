// C ABI of libqswiglu.so (declared in include/qswiglu.h): argument checks,
// routing between the small-M and tensor-core kernels, dispatch counters and
// the device error word.
//
// Accepted specs follow fusedSwigluSupported() in the mlx-bun pages
// (src/model/fused-swiglu-kernel.ts): bits in {2,4,8}, group size a multiple of
// 32, H a multiple of 32, gate and up specs independent.
#include <atomic>
#include <cstdlib>
#include <mutex>

#include "qswiglu.h"
#include "qsw_device.cuh"
#include "qsw_internal.h"

namespace qsw {
cudaError_t prefill_take_errors(unsigned int *out);
cudaError_t gemv_take_errors(unsigned int *out);
cudaError_t gemv_stream_take_errors(unsigned int *out);
}

namespace {

std::atomic<uint64_t> g_counters[QSW_NUM_COUNTERS];
std::atomic<int> g_gemv_max_m{-1};   // -1: not yet initialised
std::atomic<uint64_t> g_timeout_ns{4000000000ull};
std::atomic<int> g_early_weights{0};
std::atomic<int> g_stream_k{QSW_STREAM_K_AUTO};
std::atomic<int> g_small_m_kernel{QSW_SMALL_M_AUTO};

int gemv_max_m() {
  int v = g_gemv_max_m.load(std::memory_order_relaxed);
  if (v < 0) {
    int init = 32;
    if (const char *env = std::getenv("QSW_GEMV_MAX_M")) init = std::atoi(env);
    if (init < 0) init = 0;
    if (init > qsw::kGemvMaxM) init = static_cast<int>(qsw::kGemvMaxM);
    int expected = -1;
    g_gemv_max_m.compare_exchange_strong(expected, init);
    v = g_gemv_max_m.load();
  }
  return v;
}

int sm_count() {
  static int counts[64];
  static std::once_flag flags[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::call_once(flags[dev], [dev] {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    counts[dev] = n;
  });
  return counts[dev];
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

enum Route { ROUTE_TC = 0, ROUTE_RING = 1, ROUTE_STREAM = 2 };

// Which kernel serves M rows: the small-M path up to the small-M limit (the
// warp-streamed kernel unless the slot-ring one is selected, where it
// applies), else -- or where neither small-M kernel applies -- the tensor-core
// kernel.
Route route(int64_t M, int64_t K, int64_t N, const qsw::QuantOperand &op0, const qsw::QuantOperand *op1) {
  if (M > gemv_max_m()) return ROUTE_TC;
  if (g_small_m_kernel.load(std::memory_order_relaxed) != QSW_SMALL_M_RING &&
      qsw::gemv_stream_fits(M, K, N, op0, op1, sm_count()))
    return ROUTE_STREAM;
  if (qsw::gemv_fits(M, K, N, op0, op1, sm_count())) return ROUTE_RING;
  return ROUTE_TC;
}

// The small-M kernel `r` (ROUTE_RING or ROUTE_STREAM).
cudaError_t launch_small_m(Route r, const void *x, int64_t M, int64_t K, int64_t N, const qsw::QuantOperand &op0,
                           const qsw::QuantOperand *op1, int variant, int act, void *out, const void *residual,
                           cudaStream_t s) {
  const bool early = g_early_weights.load(std::memory_order_relaxed) != 0;
  if (r == ROUTE_STREAM) {
    const cudaError_t e =
        qsw::launch_gemv_stream(x, M, K, N, op0, op1, variant, act, out, residual, s, sm_count(), early);
    if (e == cudaSuccess) g_counters[QSW_CNT_GEMV_STREAM].fetch_add(1, std::memory_order_relaxed);
    return e;
  }
  return qsw::launch_gemv(x, M, K, N, op0, op1, variant, act, out, residual, s, g_timeout_ns.load(), sm_count(), early);
}

qsw_status check_spec(int64_t K, int gs, int bits) {
  if (gs <= 0 || K <= 0) return QSW_ERR_INVALID_ARG;
  if (bits != 2 && bits != 4 && bits != 8) return QSW_ERR_UNSUPPORTED;
  if (gs % 32 != 0 || K % gs != 0) return QSW_ERR_UNSUPPORTED;
  if (bits == 2 && K % 64 != 0) return QSW_ERR_UNSUPPORTED;
  return QSW_OK;
}

qsw_status check_operand(const uint32_t *w, const void *s, const void *b, int64_t K, int gs, int bits) {
  if (!w || !s || !b) return QSW_ERR_INVALID_ARG;
  const qsw_status st = check_spec(K, gs, bits);
  if (st != QSW_OK) return st;
  if (!aligned(w, 16) || !aligned(s, 2) || !aligned(b, 2)) return QSW_ERR_UNSUPPORTED;
  return QSW_OK;
}

qsw_status check_shape(int64_t M, int64_t K, int64_t N) {
  if (M < 0 || K <= 0 || N <= 0) return QSW_ERR_INVALID_ARG;
  if (K % 32 != 0) return QSW_ERR_UNSUPPORTED;
  // TMA coordinates and tile counts are 32-bit
  if (K > (int64_t(1) << 30) || N > (int64_t(1) << 30) || M > (int64_t(1) << 30)) return QSW_ERR_UNSUPPORTED;
  return QSW_OK;
}

qsw_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QSW_OK : QSW_ERR_CUDA; }

// A workspace is optional; if given it must be aligned and large enough.
qsw_status check_workspace(const void *ws, size_t bytes, qsw::SplitWorkspace *out) {
  out->ptr = nullptr;
  out->bytes = 0;
  out->mode = g_stream_k.load(std::memory_order_relaxed);
  if (!ws) return QSW_OK;
  if (!aligned(ws, 256)) return QSW_ERR_UNSUPPORTED;
  if (bytes < qsw::prefill_workspace_bytes(sm_count())) return QSW_ERR_INVALID_ARG;
  out->ptr = const_cast<void *>(ws);
  out->bytes = bytes;
  return QSW_OK;
}

// The fused expansion behind every entry point: argument checks, then the
// small-M or tensor-core kernel.  `static_scratch`: the tensor-core kernel
// takes the library's static stream-K workspace (resolved only on that path).
qsw_status fused_forward(const void *x, int64_t M, int64_t H, int64_t I, const uint32_t *wg, const void *sg,
                         const void *bg, int gs_g, int bits_g, const uint32_t *wu, const void *su, const void *bu,
                         int gs_u, int bits_u, int variant, int act, void *out, void *workspace,
                         size_t workspace_bytes, bool static_scratch, void *stream) {
  qsw_status st = check_shape(M, H, I);
  if (st != QSW_OK) return st;
  qsw::SplitWorkspace ws;
  if ((st = check_workspace(workspace, workspace_bytes, &ws)) != QSW_OK) return st;
  if (variant < QSW_MATCH || variant > QSW_DEBUG_UP) return QSW_ERR_INVALID_ARG;
  if (act != QSW_ACT_BF16 && act != QSW_ACT_F16) return QSW_ERR_INVALID_ARG;
  if ((st = check_operand(wg, sg, bg, H, gs_g, bits_g)) != QSW_OK) return st;
  if ((st = check_operand(wu, su, bu, H, gs_u, bits_u)) != QSW_OK) return st;
  if (M == 0) return QSW_OK;   // nothing to read or write: x and out may be null
  if (!x || !out) return QSW_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16)) return QSW_ERR_UNSUPPORTED;

  const qsw::QuantOperand g{wg, static_cast<const uint16_t *>(sg), static_cast<const uint16_t *>(bg), gs_g, bits_g};
  const qsw::QuantOperand u{wu, static_cast<const uint16_t *>(su), static_cast<const uint16_t *>(bu), gs_u, bits_u};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Route r = route(M, H, I, g, &u);
  if (r != ROUTE_TC) {
    st = from_cuda(launch_small_m(r, x, M, H, I, g, &u, variant, act, out, nullptr, s));
    if (st == QSW_OK) g_counters[QSW_CNT_FUSED_GEMV].fetch_add(1, std::memory_order_relaxed);
  } else {
    if (static_scratch && qsw::prefill_static_workspace(sm_count(), s, &ws.ptr, &ws.bytes) != cudaSuccess)
      return QSW_ERR_CUDA;
    st = from_cuda(
        qsw::launch_prefill(x, M, H, I, g, &u, variant, act, out, nullptr, s, g_timeout_ns.load(), sm_count(), ws));
    if (st == QSW_OK) g_counters[QSW_CNT_FUSED_TC].fetch_add(1, std::memory_order_relaxed);
  }
  return st;
}

}  // namespace

extern "C" {

qsw_status qswiglu_forward_ex(const void *x, int64_t M, int64_t H, int64_t I, const uint32_t *wg, const void *sg,
                              const void *bg, int gs_g, int bits_g, const uint32_t *wu, const void *su,
                              const void *bu, int gs_u, int bits_u, int variant, int act_dtype, void *out,
                              void *workspace, size_t workspace_bytes, void *stream) {
  return fused_forward(x, M, H, I, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u, variant, act_dtype, out,
                       workspace, workspace_bytes, false, stream);
}

qsw_status qswiglu_forward_ws(const void *x, int64_t M, int64_t H, int64_t I, const uint32_t *wg, const void *sg,
                              const void *bg, int gs_g, int bits_g, const uint32_t *wu, const void *su,
                              const void *bu, int gs_u, int bits_u, int variant, void *out, void *workspace,
                              size_t workspace_bytes, void *stream) {
  return fused_forward(x, M, H, I, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u, variant, QSW_ACT_BF16, out,
                       workspace, workspace_bytes, false, stream);
}

qsw_status qswiglu_forward(const void *x, int64_t M, int64_t H, int64_t I, const uint32_t *wg, const void *sg,
                           const void *bg, int gs_g, int bits_g, const uint32_t *wu, const void *su, const void *bu,
                           int gs_u, int bits_u, int variant, void *out, void *stream) {
  return qswiglu_forward_ws(x, M, H, I, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u, variant, out, nullptr, 0,
                            stream);
}

qsw_status affine_qmm_ex(const void *x, int64_t M, int64_t K, int64_t N, const uint32_t *w, const void *s,
                         const void *b, int gs, int bits, int act_dtype, const void *residual, void *y,
                         void *workspace, size_t workspace_bytes, void *stream) {
  qsw_status st = check_shape(M, K, N);
  if (st != QSW_OK) return st;
  qsw::SplitWorkspace ws;
  if ((st = check_workspace(workspace, workspace_bytes, &ws)) != QSW_OK) return st;
  if (act_dtype != QSW_ACT_BF16 && act_dtype != QSW_ACT_F16) return QSW_ERR_INVALID_ARG;
  if ((st = check_operand(w, s, b, K, gs, bits)) != QSW_OK) return st;
  if (M == 0) return QSW_OK;   // nothing to read or write: x and y may be null
  if (!x || !y) return QSW_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(residual, 16)) return QSW_ERR_UNSUPPORTED;

  const qsw::QuantOperand op{w, static_cast<const uint16_t *>(s), static_cast<const uint16_t *>(b), gs, bits};
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const Route r = route(M, K, N, op, nullptr);
  if (r != ROUTE_TC) {
    st = from_cuda(launch_small_m(r, x, M, K, N, op, nullptr, QSW_DEBUG_GATE, act_dtype, y, residual, cs));
    if (st == QSW_OK) g_counters[QSW_CNT_QMM_GEMV].fetch_add(1, std::memory_order_relaxed);
  } else {
    st = from_cuda(qsw::launch_prefill(x, M, K, N, op, nullptr, QSW_DEBUG_GATE, act_dtype, y, residual, cs,
                                       g_timeout_ns.load(), sm_count(), ws));
    if (st == QSW_OK) g_counters[QSW_CNT_QMM_TC].fetch_add(1, std::memory_order_relaxed);
  }
  return st;
}

qsw_status affine_qmm_ws(const void *x, int64_t M, int64_t K, int64_t N, const uint32_t *w, const void *s,
                         const void *b, int gs, int bits, void *y, void *workspace, size_t workspace_bytes,
                         void *stream) {
  return affine_qmm_ex(x, M, K, N, w, s, b, gs, bits, QSW_ACT_BF16, nullptr, y, workspace, workspace_bytes, stream);
}

qsw_status affine_qmm(const void *x, int64_t M, int64_t K, int64_t N, const uint32_t *w, const void *s,
                      const void *b, int gs, int bits, void *y, void *stream) {
  return affine_qmm_ws(x, M, K, N, w, s, b, gs, bits, y, nullptr, 0, stream);
}

qsw_status qswiglu_forward_noalloc(const void *x, int64_t M, int64_t H, int64_t I, const uint32_t *wg,
                                   const void *sg, const void *bg, int gs_g, int bits_g, const uint32_t *wu,
                                   const void *su, const void *bu, int gs_u, int bits_u, int variant, void *out,
                                   void *stream) {
  return fused_forward(x, M, H, I, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u, variant, QSW_ACT_BF16, out,
                       nullptr, 0, true, stream);
}

qsw_status qsw_mlp_forward_ex(const void *x, const void *h, int64_t M, int64_t H, int64_t I, int64_t Ho,
                              const uint32_t *wg, const void *sg, const void *bg, int gs_g, int bits_g,
                              const uint32_t *wu, const void *su, const void *bu, int gs_u, int bits_u,
                              const uint32_t *wd, const void *sd, const void *bd, int gs_d, int bits_d,
                              int variant, int act_dtype, void *hidden, void *y, void *workspace,
                              size_t workspace_bytes, void *stream) {
  // every argument of both stages is checked before the first launch
  if (variant != QSW_MATCH && variant != QSW_F32) return QSW_ERR_INVALID_ARG;
  qsw_status st = check_shape(M, H, I);
  if (st != QSW_OK || (st = check_shape(M, I, Ho)) != QSW_OK) return st;
  if ((st = check_operand(wg, sg, bg, H, gs_g, bits_g)) != QSW_OK) return st;
  if ((st = check_operand(wu, su, bu, H, gs_u, bits_u)) != QSW_OK) return st;
  if ((st = check_operand(wd, sd, bd, I, gs_d, bits_d)) != QSW_OK) return st;
  if (act_dtype != QSW_ACT_BF16 && act_dtype != QSW_ACT_F16) return QSW_ERR_INVALID_ARG;
  qsw::SplitWorkspace ws;
  if ((st = check_workspace(workspace, workspace_bytes, &ws)) != QSW_OK) return st;
  if (M == 0) return QSW_OK;
  if (!x || !hidden || !y) return QSW_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(hidden, 16) || !aligned(y, 16) || !aligned(h, 16)) return QSW_ERR_UNSUPPORTED;
  st = fused_forward(x, M, H, I, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u, variant, act_dtype, hidden,
                     workspace, workspace_bytes, false, stream);
  if (st != QSW_OK) return st;
  return affine_qmm_ex(hidden, M, I, Ho, wd, sd, bd, gs_d, bits_d, act_dtype, h, y, workspace, workspace_bytes,
                       stream);
}

size_t qsw_workspace_bytes(void) { return qsw::prefill_workspace_bytes(sm_count()); }

void qsw_set_stream_k(int mode) {
  if (mode >= QSW_STREAM_K_OFF && mode <= QSW_STREAM_K_ALWAYS) g_stream_k.store(mode);
}

int qsw_get_stream_k(void) { return g_stream_k.load(); }

qsw_status qsw_silu_mul_ex(const void *g, const void *u, int64_t n, int variant, int act_dtype, void *out,
                           void *stream) {
  if (n < 0) return QSW_ERR_INVALID_ARG;
  if (variant != QSW_MATCH && variant != QSW_F32) return QSW_ERR_INVALID_ARG;
  if (act_dtype != QSW_ACT_BF16 && act_dtype != QSW_ACT_F16) return QSW_ERR_INVALID_ARG;
  if (n == 0) return QSW_OK;
  if (!g || !u || !out) return QSW_ERR_INVALID_ARG;
  if (!aligned(g, 16) || !aligned(u, 16) || !aligned(out, 16)) return QSW_ERR_UNSUPPORTED;
  const qsw_status st =
      from_cuda(qsw::launch_silu_mul(g, u, n, variant, act_dtype, out, static_cast<cudaStream_t>(stream)));
  if (st == QSW_OK) g_counters[QSW_CNT_SILU_MUL].fetch_add(1, std::memory_order_relaxed);
  return st;
}

qsw_status qsw_silu_mul(const void *g, const void *u, int64_t n, int variant, void *out, void *stream) {
  return qsw_silu_mul_ex(g, u, n, variant, QSW_ACT_BF16, out, stream);
}

qsw_status qsw_check_device_errors(void *stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return QSW_ERR_CUDA;
  unsigned int a = 0, b = 0, c = 0;
  if (qsw::prefill_take_errors(&a) != cudaSuccess) return QSW_ERR_CUDA;
  if (qsw::gemv_take_errors(&b) != cudaSuccess) return QSW_ERR_CUDA;
  if (qsw::gemv_stream_take_errors(&c) != cudaSuccess) return QSW_ERR_CUDA;
  if ((a | b | c) & qsw::DEVERR_BOUNDS) return QSW_ERR_BOUNDS;
  return (a | b | c) ? QSW_ERR_TIMEOUT : QSW_OK;
}

void qsw_set_gemv_max_m(int m) {
  if (m < 0) m = 0;
  if (m > qsw::kGemvMaxM) m = static_cast<int>(qsw::kGemvMaxM);
  g_gemv_max_m.store(m);
}

int qsw_get_gemv_max_m(void) { return gemv_max_m(); }

void qsw_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1); }

void qsw_debug_withhold_next_fill(void) { qsw::gemv_withhold_next(); }

int qsw_debug_build(void) {
#ifdef QSW_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

void qsw_set_small_m_kernel(int kernel) {
  if (kernel >= QSW_SMALL_M_AUTO && kernel <= QSW_SMALL_M_STREAM) g_small_m_kernel.store(kernel);
}

int qsw_get_small_m_kernel(void) { return g_small_m_kernel.load(); }

void qsw_set_early_weight_stream(int on) { g_early_weights.store(on ? 1 : 0); }

int qsw_get_early_weight_stream(void) { return g_early_weights.load(); }

void qsw_get_counters(uint64_t *out, int n) {
  if (!out) return;
  for (int i = 0; i < n && i < QSW_NUM_COUNTERS; ++i) out[i] = g_counters[i].load();
}

void qsw_reset_counters(void) {
  for (auto &c : g_counters) c.store(0);
}

const char *qsw_status_string(qsw_status s) {
  switch (s) {
    case QSW_OK: return "ok";
    case QSW_ERR_INVALID_ARG: return "invalid argument";
    case QSW_ERR_UNSUPPORTED: return "unsupported shape, spec or alignment";
    case QSW_ERR_CUDA: return "CUDA error";
    case QSW_ERR_TIMEOUT: return "device-side wait timed out";
    case QSW_ERR_BOUNDS: return "device-side address or copy check failed (debug build)";
    default: return "unknown status";
  }
}

int qsw_version(void) { return 105; }

}  // extern "C"
