// Host side of the C ABI declared in include/mq.h: argument validation,
// device checks, the device error word, and dispatch to the kernels.
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "mq_internal.cuh"

namespace mq {

mq_status quantize_act_launch(const void* x, mq_dtype xt, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                              uint16_t* xs, cudaStream_t stream);
size_t select_workspace_bytes(int64_t N, int64_t K);
mq_status select_blocks_launch(const uint16_t* w, int64_t N, int64_t K, const void* xcal, mq_dtype xct,
                               int64_t C, int64_t ksel, int32_t* row_ptr, int32_t* col_idx, double* h_out,
                               double* delta_out, void* ws, cudaStream_t stream);
mq_status pack_weights_launch(const uint16_t* w, int64_t N, int64_t K, const int32_t* row_ptr,
                              const int32_t* col_idx, int64_t nnzb, uint8_t* wpk, uint8_t* rpk, cudaStream_t stream);
size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
mq_status gemm_launch(const uint8_t* xq, const uint16_t* xs, int64_t M, const uint8_t* wpk, int64_t N, int64_t K,
                      const int32_t* row_ptr, const int32_t* col_idx, int64_t nnzb, const uint8_t* rpk, void* y,
                      int64_t ldy, mq_dtype yt, int32_t* dots_w, int32_t* dots_r, void* ws, size_t ws_bytes,
                      cudaStream_t stream);
size_t general_workspace_bytes(int64_t M, int64_t N, int64_t K);
size_t zipper_workspace_bytes(int64_t M, int64_t tiles, int64_t K);
mq_status zipper_launch(bool* handled, int nmat, const uint8_t* const* wpk, const int64_t* N,
                        const int32_t* const* row_ptr, const int32_t* const* col_idx, const int64_t* nnzb,
                        const uint8_t* const* rpk, void* const* y, const int64_t* ldy, mq_dtype yt, const uint8_t* xq,
                        const uint16_t* xs, const void* x, mq_dtype xt, int64_t ldx, uint8_t* xq_out,
                        uint16_t* xs_out, int64_t M, int64_t K, int32_t* dots_w, int32_t* dots_r, void* ws,
                        size_t ws_bytes, cudaStream_t stream);
mq_status gemm_plan_info(int64_t M, int64_t N, int64_t K, int32_t* info);
mq_status wait_timeout_probe_launch(cudaStream_t stream);
mq_status error_word_address(uint32_t** out);

static thread_local char g_last_error[512] = "";
static std::atomic<uint64_t> g_timeout_ns{1000000000ull};

mq_status set_error(mq_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

mq_status launch_status(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(MQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return MQ_OK;
}

uint64_t wait_timeout_ns() { return g_timeout_ns.load(); }

// Incremented each time mq_check_device_error reports a device-side timeout:
// after one, workspace counters may have been left nonzero.
static std::atomic<uint64_t> g_timeout_epoch{0};
uint64_t timeout_epoch() { return g_timeout_epoch.load(); }

constexpr int kMaxDevices = 64;
static int g_dev_ok[kMaxDevices];  // 0 unknown, 1 ok, -1 unsupported
static int g_dev_sms[kMaxDevices];
static uint32_t* g_err_word[kMaxDevices];
static std::mutex g_dev_mu;

// The first check of a device also resolves the device address of its error
// word (a module-scope __device__ variable, so nothing is allocated).
mq_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return launch_status("cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return set_error(MQ_ERR_UNSUPPORTED_DEVICE, "device index %d", dev);
  if (g_dev_ok[dev] == 1) return MQ_OK;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev_ok[dev] == 1) return MQ_OK;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return launch_status("device attributes");
  if (major != 10 || minor != 3) {
    g_dev_ok[dev] = -1;
    return set_error(MQ_ERR_UNSUPPORTED_DEVICE, "compute capability %d.%d; this library is built for 10.3 (sm_103a)",
                     major, minor);
  }
  uint32_t* word = nullptr;
  if (mq_status s = error_word_address(&word); s != MQ_OK) return s;
  g_err_word[dev] = word;
  g_dev_sms[dev] = sms;
  g_dev_ok[dev] = 1;
  return MQ_OK;
}

uint32_t* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return g_err_word[dev];
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return g_dev_sms[dev];
}

static bool sizes_ok(int64_t M, int64_t N, int64_t K) {
  const int64_t lim = int64_t(1) << 20;
  return M >= 1 && M <= lim && N >= kTileN && N <= lim && K >= kGroup && K <= lim && N % kTileN == 0 &&
         K % kGroup == 0;
}

}  // namespace mq

using namespace mq;

#define MQ_CHECK(cond, status, ...) \
  do {                              \
    if (!(cond)) return set_error(status, __VA_ARGS__); \
  } while (0)

extern "C" {

const char* mq_version(void) { return "mq-gb300 0.1 (sm_103a)"; }

const char* mq_status_string(mq_status s) {
  switch (s) {
    case MQ_OK: return "ok";
    case MQ_ERR_INVALID_ARG: return "invalid argument";
    case MQ_ERR_ALIGNMENT: return "misaligned buffer";
    case MQ_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case MQ_ERR_CUDA: return "CUDA error";
    case MQ_ERR_TIMEOUT: return "device-side wait timed out";
    case MQ_ERR_WORKSPACE: return "workspace too small or misaligned";
  }
  return "unknown status";
}

const char* mq_last_error(void) { return g_last_error; }

void mq_set_wait_timeout_ns(uint64_t ns) {
  if (ns < 1000ull) ns = 1000ull;
  if (ns > 60000000000ull) ns = 60000000000ull;
  g_timeout_ns.store(ns);
}

mq_status mq_quantize_act(const void* x, mq_dtype xt, int64_t M, int64_t K, int64_t ldx, uint8_t* xq, uint16_t* xs,
                          mq_stream_t stream) {
  MQ_CHECK(x && xq && xs, MQ_ERR_INVALID_ARG, "quantize_act: NULL pointer");
  MQ_CHECK(xt == MQ_F16 || xt == MQ_BF16, MQ_ERR_INVALID_ARG, "quantize_act: x must be fp16 or bf16");
  MQ_CHECK(M >= 1 && M <= (int64_t(1) << 20) && K >= kGroup && K % kGroup == 0 && K <= (int64_t(1) << 20) && ldx >= K,
           MQ_ERR_INVALID_ARG, "quantize_act: bad sizes M=%lld K=%lld ldx=%lld", (long long)M, (long long)K,
           (long long)ldx);
  MQ_CHECK(aligned(x, 8) && ldx % 4 == 0 && aligned(xq, 16) && aligned(xs, 16), MQ_ERR_ALIGNMENT,
           "quantize_act: x (and ldx*2 bytes) must be 8-byte aligned, xq and xs 16-byte aligned");
  if (mq_status s = check_device(); s != MQ_OK) return s;
  return quantize_act_launch(x, xt, M, K, ldx, xq, xs, reinterpret_cast<cudaStream_t>(stream));
}

int64_t mq_num_selected(int64_t N, int64_t K, double budget) {
  if (N < kBlockRows || K < kGroup || N % kBlockRows || K % kGroup) return 0;
  const int64_t nb = (N / kBlockRows) * (K / kGroup);
  if (!(budget > 0.0)) return 0;
  double t = floor(budget * static_cast<double>(nb) + 1e-9);
  if (t > static_cast<double>(nb)) t = static_cast<double>(nb);
  return static_cast<int64_t>(t);
}

size_t mq_select_workspace_bytes(int64_t N, int64_t K) {
  if (N < kBlockRows || K < kGroup) return 0;
  return select_workspace_bytes(N, K);
}

mq_status mq_select_blocks(const uint16_t* w, int64_t N, int64_t K, const void* xcal, mq_dtype xct, int64_t C,
                           double budget, int32_t* row_ptr, int32_t* col_idx, double* h_out, double* delta_out,
                           void* ws, size_t ws_bytes, mq_stream_t stream) {
  MQ_CHECK(w && xcal && row_ptr, MQ_ERR_INVALID_ARG, "select_blocks: NULL pointer");
  MQ_CHECK(sizes_ok(1, N, K) && C >= 1 && C <= (int64_t(1) << 24), MQ_ERR_INVALID_ARG,
           "select_blocks: bad sizes N=%lld K=%lld C=%lld", (long long)N, (long long)K, (long long)C);
  MQ_CHECK(budget >= 0.0 && budget <= 1.0, MQ_ERR_INVALID_ARG, "select_blocks: budget %g outside [0, 1]", budget);
  MQ_CHECK(xct == MQ_F16 || xct == MQ_BF16, MQ_ERR_INVALID_ARG, "select_blocks: xcal must be fp16 or bf16");
  const int64_t ksel = mq_num_selected(N, K, budget);
  MQ_CHECK(ksel == 0 || col_idx, MQ_ERR_INVALID_ARG, "select_blocks: col_idx is NULL but %lld blocks are selected",
           (long long)ksel);
  MQ_CHECK(aligned(w, 8) && aligned(row_ptr, 4) && aligned(col_idx, 4) && aligned(h_out, 8) && aligned(delta_out, 8),
           MQ_ERR_ALIGNMENT, "select_blocks: misaligned pointer");
  MQ_CHECK(ws && aligned(ws, 256) && ws_bytes >= select_workspace_bytes(N, K), MQ_ERR_WORKSPACE,
           "select_blocks: workspace of %zu bytes (256-aligned) needed", select_workspace_bytes(N, K));
  if (mq_status s = check_device(); s != MQ_OK) return s;
  return select_blocks_launch(w, N, K, xcal, xct, C, ksel, row_ptr, col_idx, h_out, delta_out, ws,
                              reinterpret_cast<cudaStream_t>(stream));
}

mq_status mq_pack_weights(const uint16_t* w, int64_t N, int64_t K, const int32_t* row_ptr, const int32_t* col_idx,
                          int64_t nnzb, uint8_t* wpk, uint8_t* rpk, mq_stream_t stream) {
  MQ_CHECK(w && wpk, MQ_ERR_INVALID_ARG, "pack_weights: NULL pointer");
  MQ_CHECK(sizes_ok(1, N, K), MQ_ERR_INVALID_ARG, "pack_weights: bad sizes N=%lld K=%lld", (long long)N,
           (long long)K);
  MQ_CHECK(nnzb >= 0 && nnzb <= (N / kBlockRows) * (K / kGroup), MQ_ERR_INVALID_ARG, "pack_weights: bad nnzb %lld",
           (long long)nnzb);
  MQ_CHECK(nnzb == 0 || (row_ptr && col_idx && rpk), MQ_ERR_INVALID_ARG,
           "pack_weights: residual pointers are NULL but nnzb = %lld", (long long)nnzb);
  MQ_CHECK(aligned(w, 8) && aligned(wpk, 16) && aligned(rpk, 16), MQ_ERR_ALIGNMENT,
           "pack_weights: w must be 8-byte aligned, outputs 16-byte aligned");
  if (mq_status s = check_device(); s != MQ_OK) return s;
  return pack_weights_launch(w, N, K, row_ptr, col_idx, nnzb, wpk, rpk, reinterpret_cast<cudaStream_t>(stream));
}

size_t mq_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (!sizes_ok(M, N, K)) return 0;
  return gemm_workspace_bytes(M, N, K);
}

mq_status mq_gemm_workspace_init(void* ws, size_t ws_bytes, mq_stream_t stream) {
  if (ws_bytes == 0) return MQ_OK;
  MQ_CHECK(ws, MQ_ERR_INVALID_ARG, "gemm_workspace_init: NULL workspace");
  if (cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return launch_status("gemm_workspace_init");
  return MQ_OK;
}

static mq_status gemm_common(const uint8_t* xq, const uint16_t* xs, int64_t M, const uint8_t* wpk, int64_t N,
                             int64_t K, const int32_t* row_ptr, const int32_t* col_idx, int64_t nnzb,
                             const uint8_t* rpk, void* ws, size_t ws_bytes) {
  MQ_CHECK(xq && xs && wpk, MQ_ERR_INVALID_ARG, "gemm: NULL pointer");
  MQ_CHECK(sizes_ok(M, N, K), MQ_ERR_INVALID_ARG, "gemm: bad sizes M=%lld N=%lld K=%lld", (long long)M,
           (long long)N, (long long)K);
  MQ_CHECK(nnzb >= 0 && nnzb <= (N / kBlockRows) * (K / kGroup), MQ_ERR_INVALID_ARG, "gemm: bad nnzb %lld",
           (long long)nnzb);
  MQ_CHECK(nnzb == 0 || (row_ptr && col_idx && rpk), MQ_ERR_INVALID_ARG,
           "gemm: residual pointers are NULL but nnzb = %lld", (long long)nnzb);
  MQ_CHECK(aligned(xq, 16) && aligned(xs, 16) && aligned(wpk, 16) && aligned(rpk, 16) && aligned(row_ptr, 4) &&
               aligned(col_idx, 4),
           MQ_ERR_ALIGNMENT, "gemm: xq, xs, wpk, rpk must be 16-byte aligned");
  const size_t need = gemm_workspace_bytes(M, N, K);
  MQ_CHECK(ws_bytes >= need && (need == 0 || (ws && aligned(ws, 256))), MQ_ERR_WORKSPACE,
           "gemm: workspace of %zu bytes (256-aligned) needed, %zu given", need, ws_bytes);
  return check_device();
}

mq_status mq_w4a4_residual_gemm(const uint8_t* xq, const uint16_t* xs, int64_t M, const uint8_t* wpk, int64_t N,
                                int64_t K, const int32_t* row_ptr, const int32_t* col_idx, int64_t nnzb,
                                const uint8_t* rpk, void* y, mq_dtype yt, void* ws, size_t ws_bytes,
                                mq_stream_t stream) {
  MQ_CHECK(y, MQ_ERR_INVALID_ARG, "gemm: y is NULL");
  MQ_CHECK(yt == MQ_BF16 || yt == MQ_F32, MQ_ERR_INVALID_ARG, "gemm: y must be bf16 or fp32");
  MQ_CHECK(aligned(y, yt == MQ_F32 ? 4 : 2), MQ_ERR_ALIGNMENT, "gemm: y misaligned");
  if (mq_status s = gemm_common(xq, xs, M, wpk, N, K, row_ptr, col_idx, nnzb, rpk, ws, ws_bytes); s != MQ_OK)
    return s;
  return gemm_launch(xq, xs, M, wpk, N, K, row_ptr, col_idx, nnzb, rpk, y, N, yt, nullptr, nullptr, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

mq_status mq_debug_group_dots(const uint8_t* xq, const uint16_t* xs, int64_t M, const uint8_t* wpk, int64_t N,
                              int64_t K, const int32_t* row_ptr, const int32_t* col_idx, int64_t nnzb,
                              const uint8_t* rpk, int32_t* dw, int32_t* dr, void* ws, size_t ws_bytes,
                              mq_stream_t stream) {
  MQ_CHECK(dw && (nnzb == 0 || dr), MQ_ERR_INVALID_ARG, "debug_group_dots: NULL output");
  if (mq_status s = gemm_common(xq, xs, M, wpk, N, K, row_ptr, col_idx, nnzb, rpk, ws, ws_bytes); s != MQ_OK)
    return s;
  return gemm_launch(xq, xs, M, wpk, N, K, row_ptr, col_idx, nnzb, rpk, nullptr, N, MQ_F32, dw, dr, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

// Workspace of the fused linear: the decode kernel's over all matrices' tiles
// when it covers the shape, else the quantized activations after the largest
// general-kernel workspace (whose zeroed prefix stays at the start).
static size_t linear_ws(int64_t M, int64_t K, int nmat, const int64_t* N, size_t* gen_bytes) {
  int64_t tiles = 0;
  size_t gen = 0;
  for (int i = 0; i < nmat; ++i) {
    tiles += N[i] / kTileN;
    gen = std::max(gen, general_workspace_bytes(M, N[i], K));
  }
  *gen_bytes = 0;
  if (const size_t z = zipper_workspace_bytes(M, tiles, K)) return z;
  const size_t Mp = static_cast<size_t>((M + 7) / 8 * 8), G = static_cast<size_t>(K / kGroup);
  gen = (gen + 255) / 256 * 256;
  *gen_bytes = gen;
  return gen + (G * Mp * 64 + 255) / 256 * 256 + (G * Mp * 2 + 255) / 256 * 256;
}

size_t mq_linear_workspace_bytes(int64_t M, int64_t K, int nmat, const int64_t* N) {
  if (nmat < 1 || nmat > 4 || !N) return 0;
  for (int i = 0; i < nmat; ++i)
    if (!sizes_ok(M, N[i], K)) return 0;
  size_t gen = 0;
  return linear_ws(M, K, nmat, N, &gen);
}

mq_status mq_w4a4_residual_linear(const void* x, mq_dtype xt, int64_t M, int64_t K, int64_t ldx, int nmat,
                                  const mq_matrix* mats, mq_dtype yt, uint8_t* xq, uint16_t* xs, void* ws,
                                  size_t ws_bytes, mq_stream_t stream) {
  MQ_CHECK(x && mats, MQ_ERR_INVALID_ARG, "linear: NULL pointer");
  MQ_CHECK(nmat >= 1 && nmat <= 4, MQ_ERR_INVALID_ARG, "linear: 1 to 4 matrices, %d given", nmat);
  MQ_CHECK(xt == MQ_F16 || xt == MQ_BF16, MQ_ERR_INVALID_ARG, "linear: x must be fp16 or bf16");
  MQ_CHECK(yt == MQ_BF16 || yt == MQ_F32, MQ_ERR_INVALID_ARG, "linear: y must be bf16 or fp32");
  MQ_CHECK(ldx >= K, MQ_ERR_INVALID_ARG, "linear: ldx %lld < K %lld", (long long)ldx, (long long)K);
  MQ_CHECK(aligned(x, 8) && ldx % 4 == 0 && aligned(xq, 16) && aligned(xs, 16), MQ_ERR_ALIGNMENT,
           "linear: x (and ldx*2 bytes) must be 8-byte aligned, xq and xs 16-byte aligned");
  const uint8_t* wpk[4];
  const int32_t* rp[4];
  const int32_t* ci[4];
  const uint8_t* rpk[4];
  void* y[4];
  int64_t N[4], nz[4], ldy[4];
  for (int i = 0; i < nmat; ++i) {
    const mq_matrix& m = mats[i];
    MQ_CHECK(m.wpk && m.y, MQ_ERR_INVALID_ARG, "linear: matrix %d: NULL pointer", i);
    MQ_CHECK(sizes_ok(M, m.N, K), MQ_ERR_INVALID_ARG, "linear: matrix %d: bad sizes M=%lld N=%lld K=%lld", i,
             (long long)M, (long long)m.N, (long long)K);
    MQ_CHECK(m.nnzb >= 0 && m.nnzb <= (m.N / kBlockRows) * (K / kGroup), MQ_ERR_INVALID_ARG,
             "linear: matrix %d: bad nnzb %lld", i, (long long)m.nnzb);
    MQ_CHECK(m.nnzb == 0 || (m.row_ptr && m.col_idx && m.rpk), MQ_ERR_INVALID_ARG,
             "linear: matrix %d: residual pointers are NULL but nnzb = %lld", i, (long long)m.nnzb);
    MQ_CHECK(m.ldy >= m.N, MQ_ERR_INVALID_ARG, "linear: matrix %d: ldy %lld < N %lld", i, (long long)m.ldy,
             (long long)m.N);
    MQ_CHECK(aligned(m.wpk, 16) && aligned(m.rpk, 16) && aligned(m.row_ptr, 4) && aligned(m.col_idx, 4) &&
                 aligned(m.y, yt == MQ_F32 ? 4 : 2),
             MQ_ERR_ALIGNMENT, "linear: matrix %d: wpk and rpk must be 16-byte aligned", i);
    wpk[i] = m.wpk;
    rp[i] = m.row_ptr;
    ci[i] = m.col_idx;
    rpk[i] = m.rpk;
    y[i] = m.y;
    N[i] = m.N;
    nz[i] = m.nnzb;
    ldy[i] = m.ldy;
  }
  if (mq_status s = check_device(); s != MQ_OK) return s;
  size_t gen = 0;
  const size_t need = linear_ws(M, K, nmat, N, &gen);
  MQ_CHECK(ws && aligned(ws, 256) && ws_bytes >= need, MQ_ERR_WORKSPACE,
           "linear: workspace of %zu bytes (256-aligned) needed, %zu given", need, ws_bytes);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  bool handled = false;
  if (gen == 0) {  // one launch: quantize in the prologue, every matrix's tiles in one sequence
    const mq_status zs = zipper_launch(&handled, nmat, wpk, N, rp, ci, nz, rpk, y, ldy, yt, nullptr, nullptr, x, xt,
                                       ldx, xq, xs, M, K, nullptr, nullptr, ws, ws_bytes, st);
    if (zs != MQ_OK || handled) return zs;
  }
  // the quantizer, then each matrix's GEMM
  const size_t Mp = static_cast<size_t>((M + 7) / 8 * 8), G = static_cast<size_t>(K / kGroup);
  uint8_t* qbuf = xq ? xq : static_cast<uint8_t*>(ws) + gen;
  uint16_t* sbuf = xs ? xs : reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + gen + (G * Mp * 64 + 255) / 256 * 256);
  if (mq_status s = quantize_act_launch(x, xt, M, K, ldx, qbuf, sbuf, st); s != MQ_OK) return s;
  for (int i = 0; i < nmat; ++i)
    if (mq_status s = gemm_launch(qbuf, sbuf, M, wpk[i], N[i], K, rp[i], ci[i], nz[i], rpk[i], y[i], ldy[i], yt,
                                  nullptr, nullptr, ws, gen, st);
        s != MQ_OK)
      return s;
  return MQ_OK;
}

mq_status mq_gemm_plan(int64_t M, int64_t N, int64_t K, int32_t* info) {
  MQ_CHECK(info, MQ_ERR_INVALID_ARG, "gemm_plan: info is NULL");
  MQ_CHECK(sizes_ok(M, N, K), MQ_ERR_INVALID_ARG, "gemm_plan: bad sizes M=%lld N=%lld K=%lld", (long long)M,
           (long long)N, (long long)K);
  if (mq_status s = check_device(); s != MQ_OK) return s;
  return gemm_plan_info(M, N, K, info);
}

mq_status mq_check_device_error(mq_stream_t stream) {
  if (mq_status s = check_device(); s != MQ_OK) return s;
  const cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return set_error(MQ_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
  uint32_t* word = device_error_word();
  uint32_t h = 0;
  if (cudaMemcpy(&h, word, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return launch_status("error word read");
  if (h != 0) {
    if (cudaMemset(word, 0, sizeof(uint32_t)) != cudaSuccess) return launch_status("error word reset");
    if (h & kDevErrTimeout) {
      g_timeout_epoch.fetch_add(1);
      return set_error(MQ_ERR_TIMEOUT, "a device-side wait ran out (error word 0x%x)", h);
    }
  }
  return MQ_OK;
}

mq_status mq_debug_wait_timeout(mq_stream_t stream) {
  if (mq_status s = check_device(); s != MQ_OK) return s;
  return wait_timeout_probe_launch(reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
