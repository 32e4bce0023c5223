// Activation quantizer (the ZipperEngine pipeline's quantization stage,
// MosaicQuant summary, Metodologia 3): per token m and per 128-input group g,
//   s = fp16_RNE(amax / 7) (saturated to 65504),  q = clamp(RNE(x / s), -7, 7),
// codes packed two per byte (even input in the low nibble).
//
// One warp per (m, g); lane l owns inputs 4l .. 4l+3 (one 8-byte load).
// Exactness: inputs are fp16/bf16, so amax is exact in fp32; amax/7 rounded
// to fp32 and then to fp16 lands on the same fp16 as the exact quotient (the
// quotient's expansion past fp16's rounding point is the period-3 pattern of
// k/7, never a run long enough to reach fp32's rounding point); x/s between
// an 11-bit and an 11-bit significand lies at least 2^-15 (relative) away from
// any half-integer unless it is one exactly, far above fp32's 2^-24, so rintf
// of the fp32 quotient is the exact round-half-even.
#include "mq_internal.cuh"

#include <cuda_bf16.h>

namespace mq {

__device__ __forceinline__ uint16_t scale_bits_from_amax(float amax) {
  __half h = __float2half_rn(__fdiv_rn(amax, 7.0f));
  uint16_t b = __half_as_ushort(h);
  if ((b & 0x7FFFu) == 0x7C00u) b = (b & 0x8000u) | 0x7BFFu;  // saturate
  return b;
}

__device__ __forceinline__ int code_of(float v, float s) {
  if (s == 0.0f) return 0;
  float t = rintf(__fdiv_rn(v, s));
  t = fminf(fmaxf(t, -7.0f), 7.0f);
  return static_cast<int>(t);
}

template <bool kBf16>
__device__ __forceinline__ void load4(const uint16_t* p, float (&v)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const uint32_t w[2] = {u.x, u.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint16_t lo = static_cast<uint16_t>(w[i] & 0xFFFFu), hi = static_cast<uint16_t>(w[i] >> 16);
    if (kBf16) {
      v[2 * i] = __uint_as_float(static_cast<uint32_t>(lo) << 16);
      v[2 * i + 1] = __uint_as_float(static_cast<uint32_t>(hi) << 16);
    } else {
      v[2 * i] = __half2float(__ushort_as_half(lo));
      v[2 * i + 1] = __half2float(__ushort_as_half(hi));
    }
  }
}

// Output layouts (group-major, so the GEMM fetches one group's activation
// tile with a single bulk copy): xq [K/128][Mp][64] bytes, xs [K/128][Mp]
// fp16, Mp = round_up(M, 8); the padding tokens m in [M, Mp) get zero codes
// and zero scales.
template <bool kBf16>
__global__ void __launch_bounds__(256) quantize_act_kernel(const uint16_t* __restrict__ x, int64_t M,
                                                           int64_t K, int64_t ldx, int64_t Mp,
                                                           uint8_t* __restrict__ xq,
                                                           uint16_t* __restrict__ xs) {
  // The next kernel (typically the GEMM, which starts by streaming weights)
  // may launch at once; x may be the preceding kernel's output, so wait for it.
  pdl_trigger();
  pdl_wait();
  const int64_t G = K / kGroup;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= Mp * G) return;
  const int64_t m = warp / G, g = warp % G;
  uint16_t* qdst = reinterpret_cast<uint16_t*>(xq + (g * Mp + m) * (kGroup / 2)) + lane;
  if (m >= M) {  // padding token
    *qdst = 0;
    if (lane == 0) xs[g * Mp + m] = 0;
    return;
  }
  float v[4];
  load4<kBf16>(x + m * ldx + g * kGroup + 4 * lane, v);
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const uint16_t sb = scale_bits_from_amax(amax);
  const float s = __half2float(__ushort_as_half(sb));
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) packed |= (static_cast<uint32_t>(code_of(v[i], s)) & 0xFu) << (4 * i);
  *qdst = static_cast<uint16_t>(packed);
  if (lane == 0) xs[g * Mp + m] = sb;
}

mq_status quantize_act_launch(const void* x, mq_dtype xt, int64_t M, int64_t K, int64_t ldx,
                              uint8_t* xq, uint16_t* xs, cudaStream_t stream) {
  const int64_t Mp = (M + 7) / 8 * 8;
  const int64_t warps = Mp * (K / kGroup);
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > 0x7FFFFFFF) return set_error(MQ_ERR_INVALID_ARG, "quantize_act: problem too large");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint16_t* xp = static_cast<const uint16_t*>(x);
  const cudaError_t e = (xt == MQ_BF16) ? cudaLaunchKernelEx(&cfg, quantize_act_kernel<true>, xp, M, K, ldx, Mp, xq, xs)
                                        : cudaLaunchKernelEx(&cfg, quantize_act_kernel<false>, xp, M, K, ldx, Mp, xq, xs);
  if (e != cudaSuccess) return launch_status("quantize_act launch");
  return launch_status("quantize_act");
}

}  // namespace mq
