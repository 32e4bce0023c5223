// Offline packing of W^ = Q(W^) + R (MosaicQuant summary, Metodologia 1):
// the dense 4-bit base (per output row, per 128-input group) and the 4-bit
// residual of the selected 64x128 blocks (one scale per block row), written as
// the records the fused GEMM streams (codes and their scales side by side, so
// one bulk copy brings both; see mq_pack_weights in mq.h).
//
// Exactness: the base follows the same fp32 argument as the activation
// quantizer.  The residual R = w - s*q is exactly representable in fp32 (it
// is a multiple of min(ulp(w), ulp(s)) >= s*2^-12 and |R| <= s/2, so it
// carries at most 12 significant bits), hence amax_R, amax_R/7 -> fp16 and
// R/s_r -> rint are exact round-half-even decisions as well.
#include "mq_internal.cuh"

namespace mq {

__device__ __forceinline__ uint16_t pk_scale_bits(float amax) {
  uint16_t b = __half_as_ushort(__float2half_rn(__fdiv_rn(amax, 7.0f)));
  if ((b & 0x7FFFu) == 0x7C00u) b = (b & 0x8000u) | 0x7BFFu;
  return b;
}
__device__ __forceinline__ float pk_code(float v, float s) {
  if (s == 0.0f) return 0.0f;
  return fminf(fmaxf(rintf(__fdiv_rn(v, s)), -7.0f), 7.0f);
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
__device__ __forceinline__ uint16_t pack4(const float (&q)[4]) {
  uint32_t p = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) p |= (static_cast<uint32_t>(static_cast<int>(q[i])) & 0xFu) << (4 * i);
  return static_cast<uint16_t>(p);
}

// Base quantization of row n, group g by one warp: lane l holds inputs 4l..4l+3.
struct RowGroup {
  float v[4], q[4], s;
  uint16_t sbits;
};
__device__ __forceinline__ RowGroup quant_row_group(const uint16_t* __restrict__ w, int64_t K, int64_t n,
                                                    int64_t g, int lane) {
  RowGroup rg;
  const uint2 u = *reinterpret_cast<const uint2*>(w + n * K + g * kGroup + 4 * lane);
  rg.v[0] = __half2float(__ushort_as_half(static_cast<uint16_t>(u.x & 0xFFFFu)));
  rg.v[1] = __half2float(__ushort_as_half(static_cast<uint16_t>(u.x >> 16)));
  rg.v[2] = __half2float(__ushort_as_half(static_cast<uint16_t>(u.y & 0xFFFFu)));
  rg.v[3] = __half2float(__ushort_as_half(static_cast<uint16_t>(u.y >> 16)));
  float amax = fmaxf(fmaxf(fabsf(rg.v[0]), fabsf(rg.v[1])), fmaxf(fabsf(rg.v[2]), fabsf(rg.v[3])));
  amax = warp_max(amax);
  rg.sbits = pk_scale_bits(amax);
  rg.s = __half2float(__ushort_as_half(rg.sbits));
#pragma unroll
  for (int i = 0; i < 4; ++i) rg.q[i] = pk_code(rg.v[i], rg.s);
  return rg;
}

// One warp per (row n, group g).
__global__ void __launch_bounds__(256) pack_base_kernel(const uint16_t* __restrict__ w, int64_t N, int64_t K,
                                                        uint8_t* __restrict__ wpk) {
  const int64_t G = K / kGroup;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= N * G) return;
  const int64_t n = warp / G, g = warp % G;
  const RowGroup rg = quant_row_group(w, K, n, g, lane);
  const int64_t t = n / kTileN, r = n % kTileN;
  uint8_t* rec = wpk + (t * G + g) * kWRecBytes;
  // inputs 4l..4l+3 sit in K-step j = l/8, bytes 2*(l%8), 2*(l%8)+1 of the row's 16-byte chunk
  *reinterpret_cast<uint16_t*>(rec + (lane / 8) * 2048 + r * 16 + (lane % 8) * 2) = pack4(rg.q);
  if (lane == 0) *reinterpret_cast<uint16_t*>(rec + kWRecScales + 2 * r) = rg.sbits;
}

// One warp per (CSR entry i, block row r).
__global__ void __launch_bounds__(256) pack_residual_kernel(const uint16_t* __restrict__ w, int64_t N, int64_t K,
                                                            const int32_t* __restrict__ row_ptr,
                                                            const int32_t* __restrict__ col_idx, int64_t nnzb,
                                                            uint8_t* __restrict__ rpk) {
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= nnzb * kBlockRows) return;
  const int64_t i = warp / kBlockRows, r = warp % kBlockRows;
  // block row of entry i: last br with row_ptr[br] <= i
  int64_t lo = 0, hi = N / kBlockRows;  // invariant: row_ptr[lo] <= i < row_ptr[hi]
  while (hi - lo > 1) {
    const int64_t mid = (lo + hi) / 2;
    if (row_ptr[mid] <= i) lo = mid; else hi = mid;
  }
  const int64_t br = lo, g = col_idx[i];
  const int64_t n = br * kBlockRows + r;
  const RowGroup rg = quant_row_group(w, K, n, g, lane);
  float res[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) res[k] = rg.v[k] - rg.s * rg.q[k];  // exact in fp32
  float amax = fmaxf(fmaxf(fabsf(res[0]), fabsf(res[1])), fmaxf(fabsf(res[2]), fabsf(res[3])));
  amax = warp_max(amax);
  const uint16_t sb = pk_scale_bits(amax);
  const float s = __half2float(__ushort_as_half(sb));
  float q[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) q[k] = pk_code(res[k], s);
  uint8_t* rec = rpk + i * kRRecBytes;
  *reinterpret_cast<uint16_t*>(rec + (lane / 8) * 1024 + r * 16 + (lane % 8) * 2) = pack4(q);
  if (lane == 0) *reinterpret_cast<uint16_t*>(rec + kRRecScales + 2 * r) = sb;
}

mq_status pack_weights_launch(const uint16_t* w, int64_t N, int64_t K, const int32_t* row_ptr,
                              const int32_t* col_idx, int64_t nnzb, uint8_t* wpk, uint8_t* rpk,
                              cudaStream_t stream) {
  const int64_t warps = N * (K / kGroup);
  pack_base_kernel<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, stream>>>(w, N, K, wpk);
  if (mq_status s = launch_status("pack: base"); s != MQ_OK) return s;
  if (nnzb > 0) {
    const int64_t rw = nnzb * kBlockRows;
    pack_residual_kernel<<<static_cast<unsigned>((rw * 32 + 255) / 256), 256, 0, stream>>>(
        w, N, K, row_ptr, col_idx, nnzb, rpk);
    if (mq_status s = launch_status("pack: residual"); s != MQ_OK) return s;
  }
  return MQ_OK;
}

}  // namespace mq
