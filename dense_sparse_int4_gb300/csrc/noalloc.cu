// mq_w4a4_residual_gemm_noalloc: the fused GEMM for callers that cannot
// allocate device memory (a runtime whose allocator is owned by someone else,
// a process that must not call cudaMalloc while a graph or a latency-critical
// loop is live, an embedder that passes in only its own input and output
// buffers).  Instead of a caller-provided workspace, it uses the fixed scratch
// array below.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds kNoAllocScratchBytes of it until the process exits.  Host
// code cannot use the array's name as a device address, so on the first call
// on each device, with that device current, the entry point resolves the
// address with cudaGetSymbolAddress (checking the result) and caches it.
//
// The GEMM kernels read the first kWsZeroBytes of a workspace as counters and
// flags and leave them zero when they finish; the loader zero-fills the array,
// so nothing needs clearing per call.  Only after a device-side wait has run
// out (reported by mq_check_device_error) may those counters be left dirty:
// the next call on that device clears them, on the stream, first.
#include <atomic>
#include <mutex>

#include "mq_internal.cuh"

namespace mq {

size_t gemm_run_workspace_bytes(int64_t M, int64_t N, int64_t K);
uint64_t timeout_epoch();

// 8 MiB: decode batches (up to 32 tokens) need the zeroed counter prefix, one
// activation image per 128-input group (at most 4.3 KiB each) and two fp32
// pieces of a 128-row x 32-token tile per SM (32 KiB per SM): about 5.3 MB at
// K = 14336 on a 152-SM GPU.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
static void* g_noalloc_ptr[kNoAllocMaxDevices];
static uint64_t g_noalloc_epoch[kNoAllocMaxDevices];  // timeout epoch the counters were last cleared for
static std::mutex g_noalloc_mu;

static mq_status noalloc_scratch(void** out, bool* dirty) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return launch_status("noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kNoAllocMaxDevices) return set_error(MQ_ERR_UNSUPPORTED_DEVICE, "noalloc: device index %d", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return set_error(MQ_ERR_CUDA, "noalloc: scratch address on device %d: %s", dev, cudaGetErrorString(e));
    g_noalloc_ptr[dev] = p;
    g_noalloc_epoch[dev] = timeout_epoch();
  }
  const uint64_t ep = timeout_epoch();
  *dirty = g_noalloc_epoch[dev] != ep;
  g_noalloc_epoch[dev] = ep;
  *out = g_noalloc_ptr[dev];
  return MQ_OK;
}

}  // namespace mq

extern "C" mq_status mq_w4a4_residual_gemm_noalloc(const uint8_t* xq, const uint16_t* xs, int64_t M,
                                                   const uint8_t* wpk, int64_t N, int64_t K,
                                                   const int32_t* row_ptr, const int32_t* col_idx, int64_t nnzb,
                                                   const uint8_t* rpk, void* y, mq_dtype yt, mq_stream_t stream) {
  using namespace mq;
  if (mq_status s = check_device(); s != MQ_OK) return s;
  if (mq_gemm_workspace_bytes(M, N, K) == 0)
    return set_error(MQ_ERR_INVALID_ARG, "noalloc gemm: bad sizes M=%lld N=%lld K=%lld", (long long)M, (long long)N,
                     (long long)K);
  const size_t need = gemm_run_workspace_bytes(M, N, K);
  if (need > kNoAllocScratchBytes)
    return set_error(MQ_ERR_WORKSPACE,
                     "noalloc gemm: M=%lld N=%lld K=%lld needs %zu bytes of scratch, more than the fixed %zu",
                     (long long)M, (long long)N, (long long)K, need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  bool dirty = false;
  if (mq_status s = noalloc_scratch(&scratch, &dirty); s != MQ_OK) return s;
  if (dirty && cudaMemsetAsync(scratch, 0, kWsZeroBytes, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return launch_status("noalloc gemm: clearing the counters after a timeout");
  return mq_w4a4_residual_gemm(xq, xs, M, wpk, N, K, row_ptr, col_idx, nnzb, rpk, y, yt, scratch,
                               kNoAllocScratchBytes, stream);
}
