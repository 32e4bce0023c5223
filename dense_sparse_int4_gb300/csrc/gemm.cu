// The fused W4A4 + block-sparse 4-bit residual GEMM (ZipperEngine, MosaicQuant
// summary, Metodologia 3): the residual product is computed inside the dense
// 4-bit GEMM, each activation tile is read once per output tile, and both
// partial products are reduce-added in the epilogue:
//
//   Y[m,n] = sum_g sx[m,g] * ( sw[n,g] * Dw[m,n,g] + sr[n,g] * Dr[m,n,g] )
//
// sm_103a design (one CTA = 128 weight rows x TN tokens x a K range):
//   * INT4 codes run on the 5th-generation tensor cores as E4M3 bytes holding
//     the same integers exactly (|q| <= 8 is exact in E4M3); products are at
//     most 49 and a group sum at most 6272 < 2^24, so the fp32 accumulator of
//     tcgen05.mma kind::f8f6f4 holds every group dot exactly.  (The
//     integer tensor-core kind is not available on sm_103a.)
//   * swap-AB: weight rows are the MMA M dimension (128), tokens the N
//     dimension (TN), so decode batches of 4..32 tokens fill one MMA.
//   * warp 0 (producer): 1-D bulk copies of the contiguous 8 KiB weight unit,
//     its 256 B of scales, the residual blocks of this tile and group, a 2-D
//     TMA box of packed activations (rows past M read as zeros) and the
//     activation scales, into a 4-deep shared-memory ring.
//   * warps 2-5 (converters, one per TMEM lane quarter): unpack weight codes
//     to E4M3 in registers and store them straight into tensor memory (the
//     MMA's A operand lives in TMEM: no shared-memory round trip), and unpack
//     the activations into a 128B-swizzled K-major shared-memory B tile.
//   * warp 1 (MMA issuer): 4 MMAs of K=32 per group into a double-buffered
//     TMEM accumulator, plus 4 more into a residual accumulator when the
//     group has a residual block in this tile (tiles and groups without one
//     issue nothing extra); tcgen05.commit releases the stages.
//   * warps 6-9 (drain): per group, tcgen05.ld the integer-valued dots and
//     reduce-add sx * (sw * Dw + sr * Dr) into fp32 registers (the scales
//     change every 128 inputs, so the accumulator is drained every group).
//   * split-K: CTAs of one output tile write fp32 partials to the workspace;
//     the last to arrive (atomic counter) sums them in split order and stores
//     Y, then resets the counter.  No floating-point atomics: deterministic.
// Every mbarrier wait is bounded (see mbar_wait).
#include "mq_internal.cuh"

#include <cuda_bf16.h>

#include <mutex>

namespace mq {

constexpr int kThreads = 320;  // 10 warps
constexpr int kWarpProducer = 0, kWarpMma = 1, kWarpConv0 = 2, kWarpDrain0 = 6;
constexpr int kMaxGroupsPerCta = 256;

template <int TN>
struct Cfg {
  // ring depth: enough weight bytes in flight per SM to cover HBM latency
  static constexpr int kStages = TN <= 32 ? 8 : (TN <= 64 ? 5 : 4);
  static constexpr int kB = TN * 128;      // E4M3 activations, SW128 K-major (1024-aligned)
  static constexpr int kA = 8192;          // packed base unit
  static constexpr int kR = 2 * 4096;      // packed residual blocks (top, bottom halves)
  static constexpr int kXQ = TN * 64;      // packed activations (TMA box)
  static constexpr int kWS = 256;          // base scales, 128 x fp16
  static constexpr int kRS = 256;          // residual scales, 2 x 64 x fp16
  static constexpr int kSX = TN * 2;       // activation scales, TN x fp16
  static constexpr int oB = 0;
  static constexpr int oA = oB + kB;
  static constexpr int oR = oA + kA;
  static constexpr int oXQ = oR + kR;
  static constexpr int oWS = oXQ + kXQ;
  static constexpr int oRS = oWS + kWS;
  static constexpr int oSX = oRS + kRS;
  static constexpr int oEnd = oSX + ((kSX + 15) / 16) * 16;
  static constexpr int kStageBytes = (oEnd + 1023) / 1024 * 1024;
  // TMEM columns: A ring 2 x (32 base + 32 residual), D_w x 2, D_r x 1
  static constexpr int tA = 0;
  static constexpr int tDw = 128;
  static constexpr int tDr = 128 + 2 * TN;
  static constexpr int kTmemNeed = 128 + 3 * TN;
  static constexpr int kTmemCols = kTmemNeed <= 256 ? 256 : 512;
  static_assert(kTmemNeed <= 512, "TMEM budget");
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align slack*/;
  static_assert(kSmemBytes + 4096 <= 227 * 1024, "shared memory budget");
  // instruction descriptor: D f32, A/B E4M3, both K-major, N = TN, M = 128
  static constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(TN >> 3) << 17) |
                                     (static_cast<uint32_t>(128 >> 4) << 24);
};

struct GemmParams {
  const uint8_t* wq;
  const uint16_t* wsc;
  const uint16_t* xs;  // [G][Mp]
  const int32_t* row_ptr;
  const int32_t* col_idx;
  const uint8_t* rq;
  const uint16_t* rsc;
  void* y;
  int y_f32;
  int32_t* dots_w;  // debug
  int32_t* dots_r;  // debug
  float* partials;
  int32_t* counters;
  int M, Mp, N, K, G, splits, nnzb;
  uint64_t timeout_ns;
  uint32_t* err;
};

// Shared-memory matrix descriptor: 128B-swizzled K-major tile, 8-row atoms of
// 1024 B (stride byte offset), descriptor version 1, start address >> 4.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

struct __align__(8) StageInfo {
  int32_t flags;    // bit 0: residual block for rows 0-63, bit 1: rows 64-127
  int32_t blk[2];   // CSR entry of each half
  int32_t pad;
};

template <int kStages>
struct __align__(8) Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t conv_full[2];
  uint64_t a_empty[2];
  uint64_t d_full[2];
  uint64_t d_empty[2];
  uint64_t dr_full;
  uint64_t dr_empty;
  StageInfo info[kStages];
  uint32_t tmem_base;
  int abort_flag;
  int is_last;
  int nres_total;  // drain-wide epilogue decision
};

template <int TN, bool kDebug>
__global__ void __launch_bounds__(kThreads, 1)
    w4a4_residual_gemm_kernel(const __grid_constant__ CUtensorMap xq_map, const GemmParams p) {
  using C = Cfg<TN>;
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Ctl<kStages> ctl;
  __shared__ int32_t res_flag_s[2][kMaxGroupsPerCta];  // per local group: CSR entry of top / bottom block or -1

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x;           // weight tile
  const int split = blockIdx.y;       // K split
  const int mt = blockIdx.z;          // token tile
  const int m0 = mt * TN;
  const int g_begin = static_cast<int>((static_cast<int64_t>(split) * p.G) / p.splits);
  const int g_end = static_cast<int>((static_cast<int64_t>(split + 1) * p.G) / p.splits);
  const int ngroups = g_end - g_begin;
  volatile int* abort_flag = &ctl.abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], 1 + 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.conv_full[i], 128);
      mbar_init(&ctl.a_empty[i], 1);
      mbar_init(&ctl.d_full[i], 1);
      mbar_init(&ctl.d_empty[i], 128);
    }
    mbar_init(&ctl.dr_full, 1);
    mbar_init(&ctl.dr_empty, 128);
    ctl.abort_flag = 0;
    ctl.is_last = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(&ctl.tmem_base, C::kTmemCols);
  if (warp == kWarpProducer) {
    // Residual blocks of this tile's two block rows inside [g_begin, g_end):
    // the CSR rows are ascending in g, so a scan of each row suffices.
    for (int i = lane; i < ngroups; i += 32) {
      res_flag_s[0][i] = -1;
      res_flag_s[1][i] = -1;
    }
    __syncwarp();
    for (int half = 0; half < 2; ++half) {
      const int br = 2 * t + half;
      // entries are clamped to [0, nnzb) so a malformed list cannot index out of bounds
      const int e0 = p.nnzb ? max(0, min(p.nnzb, p.row_ptr[br])) : 0;
      const int e1 = p.nnzb ? max(e0, min(p.nnzb, p.row_ptr[br + 1])) : 0;
      for (int e = e0 + lane; e < e1; e += 32) {
        const int g = p.col_idx[e];
        if (g >= g_begin && g < g_end) res_flag_s[half][g - g_begin] = e;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const uint64_t tmo = p.timeout_ns;

  if (warp == kWarpProducer) {
    if (lane == 0) {
      int it = 0;
      for (; it < ngroups; ++it) {
        const int st = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!mbar_wait(&ctl.empty[st], ph ^ 1, abort_flag, tmo, p.err)) break;
        const int g = g_begin + it;
        const int e_top = res_flag_s[0][it], e_bot = res_flag_s[1][it];
        StageInfo& si = ctl.info[st];
        si.flags = (e_top >= 0 ? 1 : 0) | (e_bot >= 0 ? 2 : 0);
        si.blk[0] = e_top;
        si.blk[1] = e_bot;
        uint8_t* sb = smem + st * C::kStageBytes;
        const int sx_rows = min(TN, p.Mp - m0);
        uint32_t bytes = C::kA + C::kWS + C::kXQ + sx_rows * 2;
        if (e_top >= 0) bytes += 4096 + 128;
        if (e_bot >= 0) bytes += 4096 + 128;
        mbar_arrive_expect_tx(&ctl.full[st], bytes);
        const int64_t unit = static_cast<int64_t>(t) * p.G + g;
        bulk_g2s(sb + C::oA, p.wq + unit * 8192, 8192, &ctl.full[st]);
        bulk_g2s(sb + C::oWS, p.wsc + unit * 128, 256, &ctl.full[st]);
        tma_2d_g2s(sb + C::oXQ, &xq_map, g * 64, m0, &ctl.full[st]);
        bulk_g2s(sb + C::oSX, p.xs + static_cast<int64_t>(g) * p.Mp + m0, sx_rows * 2, &ctl.full[st]);
        if (e_top >= 0) {
          bulk_g2s(sb + C::oR, p.rq + static_cast<int64_t>(e_top) * 4096, 4096, &ctl.full[st]);
          bulk_g2s(sb + C::oRS, p.rsc + static_cast<int64_t>(e_top) * 64, 128, &ctl.full[st]);
        }
        if (e_bot >= 0) {
          bulk_g2s(sb + C::oR + 4096, p.rq + static_cast<int64_t>(e_bot) * 4096, 4096, &ctl.full[st]);
          bulk_g2s(sb + C::oRS + 128, p.rsc + static_cast<int64_t>(e_bot) * 64, 128, &ctl.full[st]);
        }
      }
      // Before the CTA may exit, every copy issued must have landed (the
      // last kStages stages; earlier ones were consumed).  Bounded as well.
      volatile int never = 0;
      for (int j = max(0, it - kStages); j < it; ++j)
        mbar_wait(&ctl.full[j % kStages], (j / kStages) & 1, &never, tmo, p.err);
    }
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      int nres = 0;
      int issued = 0;
      for (int it = 0; it < ngroups; ++it) {
        const int st = it % kStages;
        const int a = it & 1, d = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait(&ctl.conv_full[a], aph, abort_flag, tmo, p.err)) break;
        if (!mbar_wait(&ctl.d_empty[d], aph ^ 1, abort_flag, tmo, p.err)) break;
        const bool has_res = ctl.info[st].flags != 0;
        if (has_res && !mbar_wait(&ctl.dr_empty, (nres & 1) ^ 1, abort_flag, tmo, p.err)) break;
        tc_fence_after();
        const uint32_t b_addr = smem_u32(smem + st * C::kStageBytes + C::oB);
        const uint32_t a_col = tmem + C::tA + a * 64;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          tc_mma_ts(tmem + C::tDw + d * TN, a_col + 8 * j, sw128_desc(b_addr + 32 * j), C::kIdesc, j > 0);
        if (has_res) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma_ts(tmem + C::tDr, a_col + 32 + 8 * j, sw128_desc(b_addr + 32 * j), C::kIdesc, j > 0);
        }
        tc_commit(&ctl.empty[st]);
        tc_commit(&ctl.a_empty[a]);
        tc_commit(&ctl.d_full[d]);
        if (has_res) {
          tc_commit(&ctl.dr_full);
          ++nres;
        }
        issued = it + 1;
      }
      // Let the last MMAs finish before TMEM can be released.
      if (issued > 0) {
        const int it = issued - 1;
        volatile int never = 0;
        mbar_wait(&ctl.d_full[it & 1], (it >> 1) & 1, &never, tmo, p.err);
      }
    }
  } else if (warp < kWarpDrain0) {
    // ---------------- converters ----------------
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;      // weight row of this thread (TMEM lane)
    const int ctid = (warp - kWarpConv0) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    for (int it = 0; it < ngroups; ++it) {
      const int st = it % kStages;
      const uint32_t ph = (it / kStages) & 1;
      const int a = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      if (!mbar_wait(&ctl.full[st], ph, abort_flag, tmo, p.err)) break;
      if (!mbar_wait(&ctl.a_empty[a], aph ^ 1, abort_flag, tmo, p.err)) break;
      tc_fence_after();
      uint8_t* sb = smem + st * C::kStageBytes;
      const uint32_t a_col = tmem + lane_base + C::tA + a * 64;
      // weights: K-step j of row r is the 16 bytes at j*2048 + r*16
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 pk = *reinterpret_cast<const uint4*>(sb + C::oA + j * 2048 + r * 16);
        uint32_t e[8];
        int4x8_to_e4m3(pk.x, e[0], e[1]);
        int4x8_to_e4m3(pk.y, e[2], e[3]);
        int4x8_to_e4m3(pk.z, e[4], e[5]);
        int4x8_to_e4m3(pk.w, e[6], e[7]);
        tmem_st8(a_col + 8 * j, e);
      }
      const int flags = ctl.info[st].flags;
      const int half = r >> 6;
      if (flags != 0) {  // whole warp takes this branch together (tcgen05.st is warp-wide)
        const bool mine = (flags >> half) & 1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t e[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          if (mine) {
            const uint4 pk = *reinterpret_cast<const uint4*>(sb + C::oR + half * 4096 + j * 1024 + (r & 63) * 16);
            int4x8_to_e4m3(pk.x, e[0], e[1]);
            int4x8_to_e4m3(pk.y, e[2], e[3]);
            int4x8_to_e4m3(pk.z, e[4], e[5]);
            int4x8_to_e4m3(pk.w, e[6], e[7]);
          }
          tmem_st8(a_col + 32 + 8 * j, e);
        }
      }
      // activations: row m, K-step j -> two 16-byte chunks 2j, 2j+1 of the
      // 128-byte swizzled row (chunk c of row m sits at chunk c ^ (m & 7))
      for (int idx = ctid; idx < TN * 4; idx += 128) {
        const int m = idx >> 2, j = idx & 3;
        const uint4 pk = *reinterpret_cast<const uint4*>(sb + C::oXQ + m * 64 + j * 16);
        uint4 lo, hi;
        int4x8_to_e4m3(pk.x, lo.x, lo.y);
        int4x8_to_e4m3(pk.y, lo.z, lo.w);
        int4x8_to_e4m3(pk.z, hi.x, hi.y);
        int4x8_to_e4m3(pk.w, hi.z, hi.w);
        uint8_t* row = sb + C::oB + (m >> 3) * 1024 + (m & 7) * 128;
        *reinterpret_cast<uint4*>(row + (((2 * j) ^ (m & 7)) * 16)) = lo;
        *reinterpret_cast<uint4*>(row + (((2 * j + 1) ^ (m & 7)) * 16)) = hi;
      }
      tc_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&ctl.conv_full[a]);
    }
  } else {
    // ---------------- drain ----------------
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int dtid = (warp - kWarpDrain0) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int n = t * kTileN + r;
    float acc[TN];
#pragma unroll
    for (int i = 0; i < TN; ++i) acc[i] = 0.0f;
    int nres = 0;
    bool ok = true;
    for (int it = 0; it < ngroups && ok; ++it) {
      const int st = it % kStages;
      const uint32_t ph = (it / kStages) & 1;
      const int d = it & 1;
      const uint32_t dph = (it >> 1) & 1;
      if (!mbar_wait(&ctl.full[st], ph, abort_flag, tmo, p.err)) { ok = false; break; }
      if (!mbar_wait(&ctl.d_full[d], dph, abort_flag, tmo, p.err)) { ok = false; break; }
      const uint8_t* sb = smem + st * C::kStageBytes;
      const StageInfo si = ctl.info[st];
      const bool any_res = si.flags != 0;
      const int half = r >> 6;
      const bool mine = (si.flags >> half) & 1;
      if (any_res && !mbar_wait(&ctl.dr_full, nres & 1, abort_flag, tmo, p.err)) { ok = false; break; }
      tc_fence_after();
      const float sw = __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(sb + C::oWS)[r]));
      const float sr = mine ? __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(sb + C::oRS)[r])) : 0.0f;
      const uint16_t* sxs = reinterpret_cast<const uint16_t*>(sb + C::oSX);
      const int g = g_begin + it;
#pragma unroll
      for (int c = 0; c < TN / 16; ++c) {
        uint32_t dw[16], dr[16];
        tmem_ld16(tmem + lane_base + C::tDw + d * TN + 16 * c, dw);
        if (any_res) tmem_ld16(tmem + lane_base + C::tDr + 16 * c, dr);
        tc_wait_ld();
        if (kDebug) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int m = m0 + 16 * c + i;
            if (m < p.M) {
              p.dots_w[(static_cast<int64_t>(m) * p.N + n) * p.G + g] = static_cast<int32_t>(__uint_as_float(dw[i]));
              if (mine)
                p.dots_r[(static_cast<int64_t>(m) * p.nnzb + si.blk[half]) * 64 + (r & 63)] =
                    static_cast<int32_t>(__uint_as_float(dr[i]));
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int mi = 16 * c + i;
            const float sx = (m0 + mi < p.Mp) ? __half2float(__ushort_as_half(sxs[mi])) : 0.0f;
            float tsum = sw * __uint_as_float(dw[i]);
            if (mine) tsum = fmaf(sr, __uint_as_float(dr[i]), tsum);
            acc[mi] = fmaf(sx, tsum, acc[mi]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&ctl.d_empty[d]);
      if (any_res) {
        mbar_arrive(&ctl.dr_empty);
        ++nres;
      }
      mbar_arrive(&ctl.empty[st]);
    }
    // ---------------- epilogue ----------------
    // All 128 drain threads agree on whether to run it (a thread that gave up
    // must not leave the others waiting at a named barrier).
    if (!ok) *abort_flag = 1;
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (dtid == 0) ctl.nres_total = (*abort_flag) ? 0 : 1;
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const bool run_epilogue = ctl.nres_total != 0;
    if (!kDebug && run_epilogue) {
      const int mvalid = min(TN, p.M - m0);
      const int tiles_n = p.N / kTileN;
      const int tile_id = mt * tiles_n + t;
      auto store = [&](int mi, float v) {
        const int64_t off = static_cast<int64_t>(m0 + mi) * p.N + n;
        if (p.y_f32)
          static_cast<float*>(p.y)[off] = v;
        else
          static_cast<__nv_bfloat16*>(p.y)[off] = __float2bfloat16_rn(v);
      };
      if (p.splits == 1) {
#pragma unroll
        for (int mi = 0; mi < TN; ++mi)
          if (mi < mvalid) store(mi, acc[mi]);
      } else {
        float* part = p.partials + (static_cast<int64_t>(tile_id) * p.splits) * (TN * kTileN);
        float* mine_part = part + static_cast<int64_t>(split) * (TN * kTileN);
#pragma unroll
        for (int mi = 0; mi < TN; ++mi) mine_part[mi * kTileN + r] = acc[mi];
        __threadfence();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (dtid == 0) {
          const int old = atomicAdd(&p.counters[tile_id], 1);
          ctl.is_last = (old == p.splits - 1) ? 1 : 0;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (ctl.is_last) {
          __threadfence();
#pragma unroll
          for (int mi = 0; mi < TN; ++mi) {
            if (mi < mvalid) {
              float sum = 0.0f;
              for (int s = 0; s < p.splits; ++s)
                sum += (s == split) ? acc[mi] : __ldcg(part + static_cast<int64_t>(s) * (TN * kTileN) + mi * kTileN + r);
              store(mi, sum);
            }
          }
          if (dtid == 0) p.counters[tile_id] = 0;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, C::kTmemCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

struct Plan {
  int tn;
  int tiles_m;
  int splits;
  size_t ws_partials;  // bytes
  size_t ws_counters;  // bytes
};

static int pick_tn(int64_t M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  return 128;
}

static size_t a256(size_t b) { return (b + 255) / 256 * 256; }

static Plan make_plan(int64_t M, int64_t N, int64_t K, int nsm) {
  Plan pl;
  pl.tn = pick_tn(M);
  pl.tiles_m = static_cast<int>((M + pl.tn - 1) / pl.tn);
  const int64_t G = K / kGroup;
  const int64_t base = (N / kTileN) * pl.tiles_m;
  const int64_t target = 2LL * nsm;
  int64_t s = (target + base - 1) / base;  // enough CTAs to cover the GPU twice
  const int64_t max_s = G >= 8 ? G / 4 : 1;  // keep >= 4 groups per split
  if (s > max_s) s = max_s;
  const int64_t min_s = (G + kMaxGroupsPerCta - 1) / kMaxGroupsPerCta;  // CTA-local residual map size
  if (s < min_s) s = min_s;
  if (s < 1) s = 1;
  pl.splits = static_cast<int>(s);
  if (pl.splits > 1) {
    pl.ws_partials = a256(static_cast<size_t>(base) * pl.splits * pl.tn * kTileN * sizeof(float));
    pl.ws_counters = a256(static_cast<size_t>(base) * sizeof(int32_t));
  } else {
    pl.ws_partials = 0;
    pl.ws_counters = 0;
  }
  return pl;
}

// The workspace size must not depend on the device, so the plan for sizing
// uses the largest SM count the library targets (152 on GB300).
constexpr int kPlanSms = 152;

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const Plan pl = make_plan(M, N, K, kPlanSms);
  return pl.ws_partials + pl.ws_counters;
}

template <int TN, bool kDebug>
static mq_status launch_tn(const CUtensorMap& map, const GemmParams& gp, const Plan& pl, cudaStream_t stream) {
  using C = Cfg<TN>;
  auto kern = w4a4_residual_gemm_kernel<TN, kDebug>;
  static bool attr_set = false;  // per template instance
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
      return launch_status("gemm: smem attribute");
    attr_set = true;
  }
  dim3 grid(gp.N / kTileN, pl.splits, pl.tiles_m);
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(map, gp);
  return launch_status("gemm");
}

mq_status gemm_launch(const uint8_t* xq, const uint16_t* xs, int64_t M, const uint8_t* wq, const uint16_t* wsc,
                      int64_t N, int64_t K, const int32_t* row_ptr, const int32_t* col_idx, int64_t nnzb,
                      const uint8_t* rq, const uint16_t* rsc, void* y, mq_dtype yt, int32_t* dots_w,
                      int32_t* dots_r, void* ws, size_t ws_bytes, cudaStream_t stream) {
  const Plan pl = make_plan(M, N, K, kPlanSms);
  if (ws_bytes < pl.ws_partials + pl.ws_counters || (pl.ws_partials && ws == nullptr))
    return set_error(MQ_ERR_WORKSPACE, "gemm: workspace of %zu bytes needed, %zu given",
                     pl.ws_partials + pl.ws_counters, ws_bytes);
  EncodeTiledFn enc = encode_fn();
  if (!enc) return set_error(MQ_ERR_CUDA, "gemm: cuTensorMapEncodeTiled unavailable");
  CUtensorMap map;
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(M)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(K / 2)};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(pl.tn)};
  const cuuint32_t estride[2] = {1, 1};
  CUresult cr = enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(xq), gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return set_error(MQ_ERR_CUDA, "gemm: tensor map encode failed (%d)", static_cast<int>(cr));
  GemmParams gp;
  gp.wq = wq;
  gp.wsc = wsc;
  gp.xs = xs;
  gp.row_ptr = row_ptr;
  gp.col_idx = col_idx;
  gp.rq = rq;
  gp.rsc = rsc;
  gp.y = y;
  gp.y_f32 = yt == MQ_F32;
  gp.dots_w = dots_w;
  gp.dots_r = dots_r;
  gp.partials = pl.ws_partials ? static_cast<float*>(ws) : nullptr;
  gp.counters = pl.ws_partials ? reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + pl.ws_partials) : nullptr;
  gp.M = static_cast<int>(M);
  gp.Mp = static_cast<int>((M + 7) / 8 * 8);
  gp.N = static_cast<int>(N);
  gp.K = static_cast<int>(K);
  gp.G = static_cast<int>(K / kGroup);
  gp.splits = pl.splits;
  gp.nnzb = static_cast<int>(nnzb);
  gp.timeout_ns = wait_timeout_ns();
  gp.err = device_error_word();
  if (!gp.err) return set_error(MQ_ERR_CUDA, "gemm: device error word unavailable");
  const bool dbg = dots_w != nullptr;
  switch (pl.tn) {
    case 16: return dbg ? launch_tn<16, true>(map, gp, pl, stream) : launch_tn<16, false>(map, gp, pl, stream);
    case 32: return dbg ? launch_tn<32, true>(map, gp, pl, stream) : launch_tn<32, false>(map, gp, pl, stream);
    case 64: return dbg ? launch_tn<64, true>(map, gp, pl, stream) : launch_tn<64, false>(map, gp, pl, stream);
    default: return dbg ? launch_tn<128, true>(map, gp, pl, stream) : launch_tn<128, false>(map, gp, pl, stream);
  }
}

}  // namespace mq
