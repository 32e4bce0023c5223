// The device error word and the failure-detection probe.
//
// Every bounded device-side wait that runs out ORs kDevErrTimeout into the
// error word of its device; mq_check_device_error reads and clears it.  The
// word is a module-scope __device__ variable (one instance per device, no
// allocation); host code takes its device address once per device with
// cudaGetSymbolAddress and hands that pointer to the kernels.
#include "mq_internal.cuh"

namespace mq {

__device__ uint32_t g_device_error_word;

mq_status error_word_address(uint32_t** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_device_error_word);
  if (e != cudaSuccess) return set_error(MQ_ERR_CUDA, "error word address: %s", cudaGetErrorString(e));
  *out = static_cast<uint32_t*>(p);
  return MQ_OK;
}

// One CTA waits, bounded, on an mbarrier phase that nothing completes.
__global__ void wait_timeout_probe_kernel(uint64_t timeout_ns, uint32_t* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, timeout_ns, err);
  __syncthreads();
}

mq_status wait_timeout_probe_launch(cudaStream_t stream) {
  uint32_t* err = device_error_word();
  if (!err) return set_error(MQ_ERR_CUDA, "error word unavailable");
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(wait_timeout_ns(), err);
  return launch_status("wait_timeout_probe");
}

}  // namespace mq
