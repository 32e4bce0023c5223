// Activation quantizer (the ZipperEngine pipeline's quantization stage,
// MosaicQuant summary, Metodologia 3): per token m and per 128-input group g,
//   s = fp16_RNE(amax / 7) (saturated to 65504),  q = clamp(RNE(x / s), -7, 7),
// codes packed two per byte (even input in the low nibble).
//
// Half a warp per (m, g); lane k of the half owns inputs 8k .. 8k+7.
// Exactness: inputs are fp16/bf16, so amax is exact in fp32; amax/7 rounded
// to fp32 and then to fp16 lands on the same fp16 as the exact quotient (the
// quotient's expansion past fp16's rounding point is the period-3 pattern of
// k/7, never a run long enough to reach fp32's rounding point).  The code is
// rint of a refined quotient, q1 = q0 + (x - q0 s) r with q0 = x r and
// r = 1/s rounded (the residual is exact in the fma): q1 lies within 2^-20 of
// x / s and equals it where x / s is a half-integer, while an input and a
// scale of at most 11 significant bits never put x / s closer than 2^-13 to a
// half-integer of magnitude 1/2 or more unless it is one; so rint(q1) is the
// exact round-half-even of x / s, without a division per input.
#include "mq_internal.cuh"

#include <cuda_bf16.h>

#include <algorithm>

namespace mq {

__device__ __forceinline__ uint16_t scale_bits_from_amax(float amax) {
  __half h = __float2half_rn(__fdiv_rn(amax, 7.0f));
  uint16_t b = __half_as_ushort(h);
  if ((b & 0x7FFFu) == 0x7C00u) b = (b & 0x8000u) | 0x7BFFu;  // saturate
  return b;
}

// clamp(RNE(v / s), -7, 7) for s != 0, with r = 1/s rounded (see the header).
__device__ __forceinline__ int code_of(float v, float s, float r) {
  const float q0 = v * r;
  const float q1 = fmaf(fmaf(q0, -s, v), r, q0);
  return static_cast<int>(fminf(fmaxf(rintf(q1), -7.0f), 7.0f));
}

// Eight consecutive inputs (two 8-byte loads: x and ldx need only 8-byte alignment).
template <bool kBf16>
__device__ __forceinline__ void load8(const uint16_t* p, float (&v)[8]) {
  const uint2 a = *reinterpret_cast<const uint2*>(p), b = *reinterpret_cast<const uint2*>(p + 4);
  const uint32_t w[4] = {a.x, a.y, b.x, b.y};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
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
  // The next kernel may launch at once; x may be the preceding kernel's
  // output, so wait for it.
  pdl_trigger();
  pdl_wait();
  const int64_t G = K / kGroup;
  // block (x, y): groups 16x .. 16x + 15 of tokens y, y + gridDim.y, ...
  const int64_t g = static_cast<int64_t>(blockIdx.x) * 16 + (threadIdx.x >> 4);
  const int k = threadIdx.x & 15;
  const unsigned half_mask = 0xFFFFu << (threadIdx.x & 16);  // this half-warp (the other may have left)
  if (g >= G) return;  // whole half-warps leave together
  for (int64_t m = blockIdx.y; m < Mp; m += gridDim.y) {
    uint32_t* qdst = reinterpret_cast<uint32_t*>(xq + (g * Mp + m) * (kGroup / 2)) + k;
    if (m >= M) {  // padding token
      *qdst = 0u;
      if (k == 0) xs[g * Mp + m] = 0;
      continue;
    }
    float v[8];
    load8<kBf16>(x + m * ldx + g * kGroup + 8 * k, v);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(half_mask, amax, o));
    const uint16_t sb = scale_bits_from_amax(amax);
    const float s = __half2float(__ushort_as_half(sb));
    uint32_t packed = 0;
    if (s != 0.0f) {
      const float r = __frcp_rn(s);
#pragma unroll
      for (int i = 0; i < 8; ++i) packed |= (static_cast<uint32_t>(code_of(v[i], s, r)) & 0xFu) << (4 * i);
    }
    *qdst = packed;
    if (k == 0) xs[g * Mp + m] = sb;
  }
}

mq_status quantize_act_launch(const void* x, mq_dtype xt, int64_t M, int64_t K, int64_t ldx,
                              uint8_t* xq, uint16_t* xs, cudaStream_t stream) {
  const int64_t Mp = (M + 7) / 8 * 8;
  const int64_t gx = (K / kGroup + 15) / 16;  // 16 groups per block
  if (gx > 0x7FFFFFFF || Mp <= 0) return set_error(MQ_ERR_INVALID_ARG, "quantize_act: problem too large");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(std::min<int64_t>(Mp, 65535)), 1);
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
