// Rate microbenchmarks: the measured peaks that roofline fractions are read
// against, kept in their own library (libmq_peaks.so), apart from the product.
//
//  * the dense 5th-generation tensor-core rate for E4M3 operands
//    (tcgen05.mma kind::f8f6f4, M = 128, N = 256, K = 32, fp32 accumulators in
//    tensor memory, both operands in shared memory): the roof of the prefill
//    shapes, whose int4 codes run as exact E4M3;
//  * the legacy warp-level mma.sync rates for E4M3 (m16n8k32, fp32
//    accumulators), s8 (m16n8k32) and s4 (m16n8k64, int32 accumulators): the
//    integer A/B context next to the E4M3 path the decode kernel takes;
//  * the E4M3 mma.sync rate at the decode kernel's occupancy and data flow
//    (16 warps per SM, four accumulator chains per warp, 32-token tiles):
//    operands loaded from shared memory and unpacked every K-step as the
//    kernel does, against the same MMAs fed from registers.
//
// The first two kernels keep many independent accumulators per issuing
// thread, so they measure issue throughput, not latency.  Waits are bounded.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint32_t s_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Shared-memory operand descriptor: 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}
// Instruction descriptor: fp32 D, E4M3 A and B, K-major both, N, M = 128.
__host__ __device__ constexpr uint32_t idesc_e4m3(int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
}

constexpr int kTcN = 256;            // one MMA: 128 x 256 x 32
constexpr int kTcSmem = 120 * 1024;  // keeps one CTA per SM, so the 512 tensor-memory columns are free

__global__ void __launch_bounds__(128, 1) tc_e4m3_rate(int iters, int* err, unsigned long long* cycles) {
  extern __shared__ uint8_t raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  uint8_t* sm = raw + ((1024u - (s_u32(raw) & 1023u)) & 1023u);
  // A: 128 rows x 128 bytes, B: 256 rows x 128 bytes of finite E4M3 bits
  for (int i = threadIdx.x; i < (128 + kTcN) * 128 / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(sm)[i] = (static_cast<uint32_t>(i) * 2654435761u) & 0x77777777u;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(s_u32(&tbase)) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s_u32(&bar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tb = tbase;
  if (threadIdx.x == 0) {
    const uint32_t a_s = s_u32(sm), b_s = s_u32(sm + 128 * 128);
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
      const uint32_t d = tb + (i & 1) * kTcN;  // two accumulators alternate
      const uint32_t ks = 32u * (i & 3);       // the four K-steps of a 128-byte row
      asm volatile(
          "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
          " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
          "l"(desc_sw128(a_s + ks)), "l"(desc_sw128(b_s + ks)), "r"(idesc_e4m3(kTcN)), "r"(i >= 2 ? 1 : 0)
          : "memory");
    }
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(s_u32(&bar))
                 : "memory");
    const uint64_t w0 = gtime();
    uint32_t done = 0;
    while (!done) {
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], 0;\n"
          " selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(done)
          : "r"(s_u32(&bar))
          : "memory");
      if (!done && gtime() - w0 > 2000000000ull) {  // bounded: report and leave
        atomicOr(err, 1);
        break;
      }
    }
    atomicMax(cycles, static_cast<unsigned long long>(clock64() - t0));
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tb) : "memory");
}

// Legacy warp MMAs.  kKind 0: E4M3 m16n8k32 (fp32 D), 1: s8 m16n8k32, 2: s4 m16n8k64 (int32 D).
constexpr int kChains = 8;

template <int kKind>
__device__ __forceinline__ void mma_one(uint32_t (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (kKind == 0) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else if constexpr (kKind == 1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k64.row.col.s32.s4.s4.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

template <int kKind>
__global__ void __launch_bounds__(512) mma_sync_rate(int iters, uint32_t magic, uint32_t* sink) {
  uint32_t a[4], d[kChains][4];
  const uint32_t seed = (threadIdx.x + 1u) * 2654435761u;
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = (seed >> i) & 0x37373737u;  // finite E4M3 / small integers
  const uint32_t b0 = seed & 0x35353535u, b1 = (seed >> 3) & 0x35353535u;
#pragma unroll
  for (int c = 0; c < kChains; ++c) d[c][0] = d[c][1] = d[c][2] = d[c][3] = 0u;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) mma_one<kKind>(d[c], a, b0, b1);
  }
  uint32_t x = 0;
#pragma unroll
  for (int c = 0; c < kChains; ++c) x ^= d[c][0] ^ d[c][1] ^ d[c][2] ^ d[c][3];
  if (x == magic) sink[0] = x;  // keeps the chains live; magic is never hit in practice
}

// The decode kernel's group product at 32 tokens (16 rows per warp, four
// 8-token blocks one at a time, weights unpacked from INT4 every block),
// repeated over two shared-memory units chosen pseudo-randomly per iteration
// (nothing is loop-invariant).  kFeed 0: operands from shared memory; 1: the
// same MMAs with register operands.
__device__ __forceinline__ void unpack_u4p(uint32_t p, uint32_t& ev, uint32_t& od) {
  const uint32_t u = p ^ 0x88888888u;
  ev = u & 0x0F0F0F0Fu;
  od = (u >> 4) & 0x0F0F0F0Fu;
}
__device__ __forceinline__ void mma_f32_e4m3(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, bool zero) {
  if (zero)
    asm volatile("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%10, %10, %10, %10};"
                 : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
  else
    asm volatile("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
constexpr int kFedUnit = 8448, kFedImg = 32 * 136, kFedSmem = 2 * kFedUnit + 2 * kFedImg;

template <int kFeed>
__global__ void __launch_bounds__(512, 1) mma_fed_rate(int iters, float* sink) {
  extern __shared__ __align__(16) uint8_t fs[];
  for (int i = threadIdx.x; i < kFedSmem / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(fs)[i] = (static_cast<uint32_t>(i) * 2654435761u) & 0x37373737u;  // finite E4M3
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int q = warp >> 3, rw = 16 * (warp & 7);
  float acc = 0.0f;
  for (int it = 0; it < iters; ++it) {
    const int sel = static_cast<int>((static_cast<uint32_t>(it) * 2654435761u) >> 31);
    const uint8_t* wr = fs + (q ^ sel) * kFedUnit + (rw + g) * 16 + t * 4;
    const uint8_t* img = fs + 2 * kFedUnit + (q ^ sel) * kFedImg;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      float d[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t a[4], b0, b1;
        if (kFeed == 0) {
          unpack_u4p(*reinterpret_cast<const uint32_t*>(wr + j * 2048), a[0], a[2]);
          unpack_u4p(*reinterpret_cast<const uint32_t*>(wr + j * 2048 + 128), a[1], a[3]);
          const uint2 b = *reinterpret_cast<const uint2*>(img + ((j * 4 + nb) * 32 + lane) * 8);
          b0 = b.x, b1 = b.y;
        } else {
          a[0] = 0x30303030u ^ static_cast<uint32_t>(sel), a[1] = 0x31313131u, a[2] = 0x32323232u, a[3] = 0x33333333u;
          b0 = 0x34343434u ^ static_cast<uint32_t>(nb), b1 = 0x35353535u ^ static_cast<uint32_t>(j);
        }
        mma_f32_e4m3(d, a, b0, b1, j == 0);
      }
      acc += d[0] + d[1] + d[2] + d[3];
    }
  }
  if (acc == 1234.5f) sink[0] = acc;  // keeps the MMAs live
}

}  // namespace

// ---------------------------------------------------------------------------
// host entry points (C ABI).  Each runs one untimed warm-up launch, then times
// one launch with CUDA events on the legacy default stream.  Return 0 on
// success, 1 on a CUDA error, 2 when a bounded wait gave up.
// ---------------------------------------------------------------------------

namespace {

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <typename Launch>
int timed(Launch launch, float* ms_out) {
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return 1;
  int rc = 0;
  if (!launch() || cudaDeviceSynchronize() != cudaSuccess) rc = 1;  // warm-up
  if (rc == 0) {
    cudaEventRecord(e0);
    if (!launch()) rc = 1;
    cudaEventRecord(e1);
    if (rc == 0 && cudaEventSynchronize(e1) != cudaSuccess) rc = 1;
    if (rc == 0 && cudaEventElapsedTime(ms_out, e0, e1) != cudaSuccess) rc = 1;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return rc;
}

}  // namespace

extern "C" {

// Dense tcgen05 E4M3 rate over all SMs (one CTA each): `iters` MMAs of
// 128 x 256 x 32 per SM.  *flops = 2 * 128 * 256 * 32 * iters * SMs / time;
// *sm_cycles = the slowest CTA's issue-to-completion clock cycles.
int mqp_tc_e4m3(int iters, double* flops, double* sm_cycles) {
  const int sms = sm_count();
  if (sms <= 0 || iters < 4 || !flops) return 1;
  if (cudaFuncSetAttribute(tc_e4m3_rate, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem) != cudaSuccess) return 1;
  int* err = nullptr;
  unsigned long long* cyc = nullptr;
  if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return 1;
  if (cudaMalloc(&cyc, sizeof(unsigned long long)) != cudaSuccess) {
    cudaFree(err);
    return 1;
  }
  cudaMemset(err, 0, sizeof(int));
  float ms = 0.f;
  int rc = timed(
      [&] {
        cudaMemset(cyc, 0, sizeof(unsigned long long));
        tc_e4m3_rate<<<sms, 128, kTcSmem>>>(iters, err, cyc);
        return cudaGetLastError() == cudaSuccess;
      },
      &ms);
  int herr = 0;
  unsigned long long hcyc = 0;
  if (rc == 0 && (cudaMemcpy(&herr, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
                  cudaMemcpy(&hcyc, cyc, sizeof(hcyc), cudaMemcpyDeviceToHost) != cudaSuccess))
    rc = 1;
  if (rc == 0 && herr) rc = 2;
  cudaFree(err);
  cudaFree(cyc);
  if (rc == 0) {
    *flops = 2.0 * 128 * kTcN * 32 * static_cast<double>(iters) * sms / (ms * 1e-3);
    if (sm_cycles) *sm_cycles = static_cast<double>(hcyc);
  }
  return rc;
}

// Warp-MMA rate (kind 0: E4M3 m16n8k32, 1: s8 m16n8k32, 2: s4 m16n8k64), 4
// CTAs of 16 warps per SM, 8 independent chains per warp.  *ops = multiply-adds
// x 2 per second.
int mqp_mma_sync(int kind, int iters, double* ops) {
  const int sms = sm_count();
  if (sms <= 0 || iters < 1 || !ops || kind < 0 || kind > 2) return 1;
  uint32_t* sink = nullptr;
  if (cudaMalloc(&sink, sizeof(uint32_t)) != cudaSuccess) return 1;
  const int grid = 4 * sms, threads = 512;
  float ms = 0.f;
  int rc = timed(
      [&] {
        if (kind == 0) mma_sync_rate<0><<<grid, threads>>>(iters, 0x9E3779B9u, sink);
        if (kind == 1) mma_sync_rate<1><<<grid, threads>>>(iters, 0x9E3779B9u, sink);
        if (kind == 2) mma_sync_rate<2><<<grid, threads>>>(iters, 0x9E3779B9u, sink);
        return cudaGetLastError() == cudaSuccess;
      },
      &ms);
  cudaFree(sink);
  if (rc == 0) {
    const double k = kind == 2 ? 64.0 : 32.0;
    const double per_mma = 2.0 * 16 * 8 * k;
    *ops = per_mma * kChains * static_cast<double>(iters) * (grid * threads / 32) / (ms * 1e-3);
  }
  return rc;
}

// The decode kernel's E4M3 group product over all SMs, one CTA of 16 warps
// each (feed 0: operands from shared memory, unpacked as the kernel does;
// feed 1: the same MMAs from registers).  *ops = multiply-adds x 2 per second.
int mqp_mma_fed(int feed, int iters, double* ops) {
  const int sms = sm_count();
  if (sms <= 0 || iters < 1 || !ops || feed < 0 || feed > 1) return 1;
  if (cudaFuncSetAttribute(mma_fed_rate<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFedSmem) != cudaSuccess ||
      cudaFuncSetAttribute(mma_fed_rate<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFedSmem) != cudaSuccess)
    return 1;
  float* sink = nullptr;
  if (cudaMalloc(&sink, sizeof(float)) != cudaSuccess) return 1;
  float ms = 0.f;
  int rc = timed(
      [&] {
        if (feed == 0) mma_fed_rate<0><<<sms, 512, kFedSmem>>>(iters, sink);
        if (feed == 1) mma_fed_rate<1><<<sms, 512, kFedSmem>>>(iters, sink);
        return cudaGetLastError() == cudaSuccess;
      },
      &ms);
  cudaFree(sink);
  if (rc == 0) *ops = 2.0 * 16 * 8 * 32 * 16 * static_cast<double>(iters) * (16.0 * sms) / (ms * 1e-3);
  return rc;
}

}  // extern "C"
