// Hessian-guided block selection (MosaicQuant summary, Metodologia 2):
//   h_k      = (sum_c xcal[c,k]^2) / C                     (diagonal Hessian)
//   R        = W^ - Q(W^)                                  (base residual)
//   Delta_b  = sum_{k in g} h_k * sum_{n in br} R[n,k]^2   (block b = (br, g))
// then the top floor(budget * #blocks) blocks by Delta (ties: lower b) as CSR.
//
// h and Delta are formed in float64 with explicitly rounded operations
// (__dmul_rn / __dadd_rn / __ddiv_rn: no fused multiply-add) in a fixed
// order - ascending c; ascending n within a column; ascending k - so both
// are reproducible bit for bit.  R is exact: w and s*q share a grid fine
// enough for their difference.
#include "mq_internal.cuh"

namespace mq {

__device__ __forceinline__ float half_bits_to_float(uint16_t b) { return __half2float(__ushort_as_half(b)); }
__device__ __forceinline__ double act_to_double(uint16_t b, bool bf16) {
  return bf16 ? static_cast<double>(__uint_as_float(static_cast<uint32_t>(b) << 16))
              : static_cast<double>(half_bits_to_float(b));
}

__device__ __forceinline__ uint16_t sel_scale_bits(float amax) {
  uint16_t b = __half_as_ushort(__float2half_rn(__fdiv_rn(amax, 7.0f)));
  if ((b & 0x7FFFu) == 0x7C00u) b = (b & 0x8000u) | 0x7BFFu;
  return b;
}

// One thread per input channel k.
__global__ void hessian_diag_kernel(const uint16_t* __restrict__ xcal, bool bf16, int64_t C, int64_t K,
                                    double* __restrict__ h) {
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (k >= K) return;
  double acc = 0.0;
  for (int64_t c = 0; c < C; ++c) {
    const double x = act_to_double(xcal[c * K + k], bf16);
    acc = __dadd_rn(acc, __dmul_rn(x, x));
  }
  h[k] = __ddiv_rn(acc, static_cast<double>(C));
}

// One CTA (128 threads) per block (br, g).
__global__ void __launch_bounds__(128) delta_kernel(const uint16_t* __restrict__ w, int64_t K,
                                                    const double* __restrict__ h,
                                                    double* __restrict__ delta) {
  const int64_t G = K / kGroup;
  const int64_t b = blockIdx.x;
  const int64_t br = b / G, g = b % G;
  __shared__ float wblk[kBlockRows][kGroup + 1];
  __shared__ float srow[kBlockRows];
  __shared__ double colsum[kGroup];
  const int tid = threadIdx.x;
  for (int i = tid; i < kBlockRows * kGroup; i += 128) {
    const int r = i / kGroup, k = i % kGroup;
    wblk[r][k] = half_bits_to_float(w[(br * kBlockRows + r) * K + g * kGroup + k]);
  }
  __syncthreads();
  if (tid < kBlockRows) {
    float amax = 0.0f;
    for (int k = 0; k < kGroup; ++k) amax = fmaxf(amax, fabsf(wblk[tid][k]));
    srow[tid] = half_bits_to_float(sel_scale_bits(amax));
  }
  __syncthreads();
  {
    const int k = tid;
    double col = 0.0;
    for (int r = 0; r < kBlockRows; ++r) {
      const float v = wblk[r][k], s = srow[r];
      float q = 0.0f;
      if (s != 0.0f) q = fminf(fmaxf(rintf(__fdiv_rn(v, s)), -7.0f), 7.0f);
      const double e = __dadd_rn(static_cast<double>(v), -__dmul_rn(static_cast<double>(s), static_cast<double>(q)));
      col = __dadd_rn(col, __dmul_rn(e, e));
    }
    colsum[k] = col;
  }
  __syncthreads();
  if (tid == 0) {
    double d = 0.0;
    for (int k = 0; k < kGroup; ++k) d = __dadd_rn(d, __dmul_rn(h[g * kGroup + k], colsum[k]));
    delta[b] = d;
  }
}

// rank_b = #{j : Delta_j > Delta_b or (Delta_j == Delta_b and j < b)}; the
// ranks are a permutation of 0..nb-1, so exactly ksel blocks get rank < ksel.
__global__ void __launch_bounds__(256) rank_select_kernel(const double* __restrict__ delta, int64_t nb,
                                                          int64_t ksel, uint8_t* __restrict__ chosen) {
  __shared__ double tile[2048];
  const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const double db = b < nb ? delta[b] : 0.0;
  int64_t rank = 0;
  for (int64_t base = 0; base < nb; base += 2048) {
    const int64_t n = min(static_cast<int64_t>(2048), nb - base);
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) tile[i] = delta[base + i];
    __syncthreads();
    if (b < nb)
      for (int64_t i = 0; i < n; ++i) {
        const double dj = tile[i];
        const int64_t j = base + i;
        rank += (dj > db) || (dj == db && j < b);
      }
  }
  if (b < nb) chosen[b] = rank < ksel ? 1 : 0;
}

// One CTA of 1024 threads builds the CSR (row_ptr over 64-row block rows,
// col_idx ascending within a row).
__global__ void __launch_bounds__(1024) build_csr_kernel(const uint8_t* __restrict__ chosen, int64_t NB,
                                                         int64_t G, int32_t* __restrict__ row_ptr,
                                                         int32_t* __restrict__ col_idx) {
  __shared__ int64_t part[1024];
  const int tid = threadIdx.x;
  const int64_t per = (NB + 1023) / 1024;
  const int64_t r0 = min(NB, tid * per), r1 = min(NB, r0 + per);
  int64_t cnt = 0;
  for (int64_t br = r0; br < r1; ++br)
    for (int64_t g = 0; g < G; ++g) cnt += chosen[br * G + g];
  part[tid] = cnt;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan (Hillis-Steele)
    const int64_t v = tid >= off ? part[tid - off] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int64_t pos = part[tid] - cnt;
  for (int64_t br = r0; br < r1; ++br) {
    row_ptr[br] = static_cast<int32_t>(pos);
    for (int64_t g = 0; g < G; ++g)
      if (chosen[br * G + g]) col_idx[pos++] = static_cast<int32_t>(g);
  }
  if (tid == 1023) row_ptr[NB] = static_cast<int32_t>(part[1023]);
}

static size_t align256(size_t b) { return (b + 255) / 256 * 256; }

size_t select_workspace_bytes(int64_t N, int64_t K) {
  const int64_t nb = (N / kBlockRows) * (K / kGroup);
  return align256(nb * 8) + align256(K * 8) + align256(nb);
}

mq_status select_blocks_launch(const uint16_t* w, int64_t N, int64_t K, const void* xcal, mq_dtype xct,
                               int64_t C, int64_t ksel, int32_t* row_ptr, int32_t* col_idx,
                               double* h_out, double* delta_out, void* ws, cudaStream_t stream) {
  const int64_t G = K / kGroup, NB = N / kBlockRows, nb = NB * G;
  uint8_t* base = static_cast<uint8_t*>(ws);
  double* delta = delta_out ? delta_out : reinterpret_cast<double*>(base);
  double* h = h_out ? h_out : reinterpret_cast<double*>(base + align256(nb * 8));
  uint8_t* chosen = base + align256(nb * 8) + align256(K * 8);
  hessian_diag_kernel<<<static_cast<unsigned>((K + 127) / 128), 128, 0, stream>>>(
      static_cast<const uint16_t*>(xcal), xct == MQ_BF16, C, K, h);
  if (mq_status s = launch_status("select: hessian"); s != MQ_OK) return s;
  delta_kernel<<<static_cast<unsigned>(nb), 128, 0, stream>>>(w, K, h, delta);
  if (mq_status s = launch_status("select: delta"); s != MQ_OK) return s;
  rank_select_kernel<<<static_cast<unsigned>((nb + 255) / 256), 256, 0, stream>>>(delta, nb, ksel, chosen);
  if (mq_status s = launch_status("select: rank"); s != MQ_OK) return s;
  build_csr_kernel<<<1, 1024, 0, stream>>>(chosen, NB, G, row_ptr, col_idx);
  return launch_status("select: csr");
}

}  // namespace mq
