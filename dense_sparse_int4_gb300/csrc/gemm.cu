// The fused W4A4 + block-sparse 4-bit residual GEMM (ZipperEngine, MosaicQuant
// summary, Metodologia 3): the residual product is computed inside the dense
// 4-bit GEMM, each activation tile is read once per output tile, and both
// partial products are reduce-added in the epilogue:
//
//   Y[m,n] = sum_g sx[m,g] * ( sw[n,g] * Dw[m,n,g] + sr[n,g] * Dr[m,n,g] )
//
// sm_103a design.
//   * Numbers: INT4 codes run on the 5th-generation tensor cores as E4M3 bytes
//     holding the same integers exactly (|q| <= 8 is exact in E4M3); products
//     are at most 49 and a group sum at most 6272, so the fp32 accumulator of
//     tcgen05.mma kind::f8f6f4 holds every group dot exactly.  (The integer
//     tensor-core kind is not available on sm_103a.)
//   * Shape: swap-AB.  128 weight rows are the MMA M dimension, TN tokens the
//     N dimension, so decode batches of 4..32 tokens fill one MMA.  A "unit"
//     is one 128-row weight tile x UG consecutive 128-input groups (UG = 2
//     for decode tiles: 16 KiB of codes in one bulk copy).
//   * Data movement: every operand is laid out so that a unit needs few, large
//     bulk copies (the bulk-copy engine's cost grows with the number of copies
//     as much as with bytes): the unit's weight codes and their scales are
//     contiguous, and so are the group-major packed activations and scales of
//     its groups.
//   * Schedule: persistent stream-K.  One CTA per SM takes an equal,
//     contiguous range of units (tile-major); tiles cut by a range boundary
//     are finished through the workspace by whichever CTA arrives last, which
//     sums the pieces in CTA order (deterministic; no floating-point atomics).
//   * Pipeline per CTA:
//       warps 0, 2 producers (alternating units, each unit's copies spread over
//               the warp's lanes): bulk copies into a ring of shared-memory stages
//               (weights, activations, scales) and, in block order, residual
//               blocks into a small ring of their own (so a stage does not
//               reserve room for residual blocks that are rarely there).
//               The first stages' weights are requested before anything else
//               (before the block list is read and before waiting on the
//               preceding kernel: programmatic dependent launch), so weight
//               streaming overlaps the kernel's start and its predecessor's end.
//       warp 1  reads the block list of the CTA's tiles into a residual map,
//               then issues the MMAs: 4 of K=32 per item into a ring of TMEM
//               accumulators.  An item is one group's base product or, only
//               where the block list has a block, its residual product, which
//               reuses the group's activation tile (residual-free groups issue
//               nothing extra).
//       converter groups of 4 warps (one per TMEM lane quarter), working on
//               alternating units: INT4 -> E4M3 in registers; weights go
//               straight into tensor memory (the MMA's A operand lives in
//               TMEM: no shared-memory round trip), activations into a
//               128B-swizzled K-major shared-memory tile.
//       4 drain warps: per item, tcgen05.ld the integer-valued dots and
//               reduce-add sx * (sw * Dw) or sx * (sr * Dr) into fp32 registers
//               (the scales change every 128 inputs); at tile ends, store Y
//               or a stream-K piece.
// Every mbarrier wait is bounded (see mbar_wait).
#include "mq_internal.cuh"

#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

// Timeline probes for profiling builds (compiled out unless MQ_GEMM_TRACE is
// defined, in which case the build supplies mq_trace_stamp).
#ifdef MQ_GEMM_TRACE
__device__ void mq_trace_stamp(int slot);
#define MQ_TRACE(slot) mq_trace_stamp(slot)
#else
#define MQ_TRACE(slot) ((void)0)
#endif

namespace mq {

constexpr int kGemmMaxDevices = 64;

// SMs of the current device, 0 when none is current.
static int current_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

// warps: 0 and 2 producers (alternating units), 1 block list + MMA, then converters, then drain
constexpr int kWarpProducer = 0, kWarpMma = 1, kWarpProducer2 = 2, kWarpConv0 = 3;
constexpr int kMaxGroupsPerCta = 1024;  // size of the CTA's residual map
constexpr int kPlanCtasNoDevice = 152;  // persistent CTAs when no device is current (workspace sizing): GB300's SMs
constexpr int kMinUnitsPerCta = 4;
constexpr int kRSlots = 6;              // residual-code ring: 6 x 4 KiB

template <int TN, int UG>
struct Cfg {
  static constexpr int kStages = TN <= 16 ? 7 : (TN <= 32 ? 5 : (TN <= 64 ? 3 : 4));  // shared-memory ring
  // Converter groups (4 warps each, one per TMEM lane quarter) take the
  // 128-input groups round-robin, so several groups are unpacked at once.
  static constexpr int kGroups = TN <= 16 ? 4 : (TN <= 32 ? 3 : (TN <= 64 ? 2 : 1));
  static constexpr int kSlotsPerGroup = kGroups >= 3 ? 2 : 8 / kGroups;
  static constexpr int kASlots = kGroups * kSlotsPerGroup;  // TMEM A ring (32 cols each), split per group
  static constexpr int kWarpDrain0 = kWarpConv0 + 4 * kGroups;  // 4 consecutive warps cover the 4 lane quarters
  static constexpr int kThreads = 32 * (kWarpDrain0 + 4);
  static constexpr int kDSlots = TN <= 16 ? 8 : (TN <= 32 ? 6 : (TN <= 64 ? 4 : 2));  // TMEM accumulators
  // stage layout, per group u of the unit
  static constexpr int kB = TN * 128;  // E4M3 activations, SW128 K-major (1024-aligned)
  static constexpr int kXQ = TN * 64;  // packed activations (group stride kXQ, or Mp*64 when merged)
  static constexpr int oB = 0;
  static constexpr int oA = oB + UG * kB;     // UG packed weight records (codes, then scales)
  static constexpr int oXQ = oA + UG * kWRecBytes;
  static constexpr int oEnd = oXQ + UG * kXQ;
  static constexpr int kStageBytes = (oEnd + 1023) / 1024 * 1024;
  static constexpr int kRingBytes = kStages * kStageBytes;
  // scale ring: the drain's inputs, so the big stages need not wait for it
  static constexpr int kScSlots = 16;
  static constexpr int sWS = 0;             // weight scales, UG x 128 fp16
  static constexpr int sRS = UG * 256;      // residual scales, UG x 2 x 64 fp16
  static constexpr int sSX = UG * 512;      // activation scales, UG x TN fp16
  static constexpr int kScBytes = ((sSX + UG * TN * 2) + 127) / 128 * 128;
  static constexpr int tA = 0;
  static constexpr int tD = kASlots * 32;
  static constexpr int kTmemNeed = tD + kDSlots * TN;
  static constexpr int kTmemCols = kTmemNeed <= 256 ? 256 : 512;
  static_assert(kTmemNeed <= 512, "TMEM budget");
  static constexpr int kSmemBytes = kRingBytes + kRSlots * 4096 + kScSlots * kScBytes + 1024 /*align slack*/;
  static_assert(kSmemBytes + 16 * 1024 <= 227 * 1024, "shared memory budget");
  // instruction descriptor: D f32, A/B E4M3, both K-major, N = TN, M = 128
  static constexpr uint32_t kIdesc =
      (1u << 4) | (static_cast<uint32_t>(TN >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
};

struct GemmParams {
  const uint8_t* xq;   // [G][Mp][64]
  const uint16_t* xs;  // [G][Mp]
  const uint8_t* wpk;  // base records
  const int32_t* row_ptr;
  const int32_t* col_idx;
  const uint8_t* rpk;  // residual records
  void* y;
  int y_f32;
  int32_t* dots_w;    // debug
  int32_t* dots_r;    // debug
  float* partials;    // [ctas][2 slots][128 rows][TN]
  int32_t* counters;  // [ctas]: pieces of the cut tile whose first unit is CTA c's
  int M, Mp, N, K, G, tiles_n, tiles_m, nnzb;
  int64_t ldy;  // elements between rows of Y
  int64_t units;  // tiles * G / UG
  int ctas;
  uint64_t timeout_ns;
  uint32_t* err;
};

// Shared-memory matrix descriptor: 128B-swizzled K-major tile, 8-row atoms of
// 1024 B (stride byte offset), descriptor version 1, start address >> 4.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// packed fp32 pairs (Blackwell f32x2 pipe)
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

template <int kStages, int kASlots, int kDSlots, int UG, int kScSlots>
struct __align__(8) Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t sc_full[kScSlots];
  uint64_t sc_empty[kScSlots];
  uint64_t r_full[kRSlots];
  uint64_t r_empty[kRSlots];
  uint64_t conv_full[kASlots];
  uint64_t a_empty[kASlots];
  uint64_t d_full[kDSlots];
  uint64_t d_empty[kDSlots];
  uint64_t drain_bar;  // bounded barrier of the 128 drain threads
  uint64_t red_bar;    // bulk loads of stream-K pieces
  uint64_t map_ready;  // residual map of the CTA's units is built
  int32_t blk[kStages][UG][2];    // CSR entry of each group's top / bottom residual block, or -1
  int32_t sblk[kScSlots][UG][2];  // the same, for the drain (lives as long as the scale slot)
  int64_t deferred[2];          // tiles this CTA completed last (at most its first and last)
  uint32_t tmem_base;
  int abort_flag;
  int ndeferred;
};

// first unit of CTA c, and the CTA that owns unit u (balanced contiguous ranges)
__device__ __forceinline__ int64_t cta_first_unit(int64_t c, int64_t U, int64_t P) { return c * U / P; }
__device__ __forceinline__ int64_t cta_of_unit(int64_t u, int64_t U, int64_t P) { return ((u + 1) * P - 1) / U; }

// Unpack one 64-byte row chunk (4 K-steps of 16 bytes, at `src + j*jstride`)
// of INT4 codes into E4M3 and store it to this thread's TMEM lane.
__device__ __forceinline__ void codes_to_tmem(const uint8_t* src, int jstride, uint32_t a_col) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 pk = *reinterpret_cast<const uint4*>(src + j * jstride);
    uint32_t ev[8];
    int4x8_to_e4m3(pk.x, ev[0], ev[1]);
    int4x8_to_e4m3(pk.y, ev[2], ev[3]);
    int4x8_to_e4m3(pk.z, ev[4], ev[5]);
    int4x8_to_e4m3(pk.w, ev[6], ev[7]);
    tmem_st8(a_col + 8 * j, ev);
  }
}

template <int TN, int UG, bool kDebug>
__global__ void __launch_bounds__(Cfg<TN, UG>::kThreads, 1) w4a4_residual_gemm_kernel(const GemmParams p) {
  using C = Cfg<TN, UG>;
  constexpr int NS = C::kStages, ND = C::kDSlots, NR = kRSlots;
  constexpr int NG = C::kGroups, SPG = C::kSlotsPerGroup, kWarpDrain0 = C::kWarpDrain0;
  extern __shared__ uint8_t smem_raw[];
  constexpr int NSC = C::kScSlots;
  __shared__ Ctl<NS, C::kASlots, ND, UG, NSC> ctl;
  __shared__ int32_t res_map[2][kMaxGroupsPerCta];   // per local group: CSR entry of top / bottom block or -1
  __shared__ int16_t res_slot[2][kMaxGroupsPerCta];  // its position in the CTA's residual-block order

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* rring = smem + C::kRingBytes;  // residual-code ring
  uint8_t* scring = rring + kRSlots * 4096;  // scale ring
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t U = p.units, P = p.ctas, c = blockIdx.x;
  const int64_t u0 = cta_first_unit(c, U, P), u1 = cta_first_unit(c + 1, U, P);
  const int nunits = static_cast<int>(u1 - u0);
  const int ngroups = nunits * UG;
  const int G = p.G, GU = p.G / UG;  // groups, units per tile
  volatile int* abort_flag = &ctl.abort_flag;
  const uint64_t tmo = p.timeout_ns;
  if (threadIdx.x == 0) MQ_TRACE(0);
  // Activations of a decode tile (one token tile, m0 = 0) are contiguous over
  // the unit's groups: one copy, group stride Mp rows; else one copy per group.
  const bool merged = (p.tiles_m == 1) && (p.Mp <= TN);
  const int xq_stride = merged ? p.Mp * 64 : C::kXQ;  // bytes between groups in the stage
  const int sx_stride = merged ? p.Mp : TN;           // fp16 entries between groups in the stage

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], 1);  // the MMA commit: codes converted, activation tile read
    }
    for (int s = 0; s < NSC; ++s) {
      mbar_init(&ctl.sc_full[s], 1);
      mbar_init(&ctl.sc_empty[s], 128);  // the drain threads
    }
    for (int s = 0; s < NR; ++s) {
      mbar_init(&ctl.r_full[s], 1);
      mbar_init(&ctl.r_empty[s], 64);  // the 64 converter threads of the block's half
    }
    for (int i = 0; i < C::kASlots; ++i) {
      mbar_init(&ctl.conv_full[i], 128);
      mbar_init(&ctl.a_empty[i], 1);
    }
    for (int i = 0; i < ND; ++i) {
      mbar_init(&ctl.d_full[i], 1);
      mbar_init(&ctl.d_empty[i], 128);
    }
    mbar_init(&ctl.drain_bar, 128);
    mbar_init(&ctl.red_bar, 1);
    mbar_init(&ctl.map_ready, 32);
    ctl.abort_flag = 0;
    ctl.ndeferred = 0;
    fence_mbar_init();
  }
  // The next kernel may launch now: before its own dependency wait it only
  // streams read-only weights, and everything else it touches waits for this
  // grid to complete.
  pdl_trigger();
  if (warp == kWarpMma) tmem_alloc(&ctl.tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  if (threadIdx.x == 0) MQ_TRACE(1);

  // unit -> tile (weight-tile major: consecutive tiles share a weight tile) -> (t, mt); first group g0
  auto unit_tile = [&](int64_t u) { return u / GU; };
  auto unit_g0 = [&](int64_t u) { return static_cast<int>(u % GU) * UG; };
  auto tile_t = [&](int64_t tile) { return static_cast<int>(tile / p.tiles_m); };
  auto tile_mt = [&](int64_t tile) { return static_cast<int>(tile % p.tiles_m); };

  if (warp == kWarpProducer || warp == kWarpProducer2) {
    const int pw = warp == kWarpProducer ? 0 : 1;  // producer warp pw fills units i = pw, pw + 2, ...
    // --- 1. weights (codes + scales) of the first stages, lane i of producer 0 arming stage i
    const int pre = min(NS, nunits);
    if (pw == 0 && lane < pre) {
      const int64_t u = u0 + lane;
      const int64_t wunit = static_cast<int64_t>(tile_t(unit_tile(u))) * G + unit_g0(u);
      uint8_t* sb = smem + lane * C::kStageBytes;
      mbar_expect_tx(&ctl.full[lane], UG * kWRecBytes);
      bulk_g2s(sb + C::oA, p.wpk + wunit * kWRecBytes, UG * kWRecBytes, &ctl.full[lane]);
      mbar_expect_tx(&ctl.sc_full[lane], UG * 256);
#pragma unroll
      for (int q = 0; q < UG; ++q)
        bulk_g2s(scring + lane * C::kScBytes + C::sWS + q * 256, p.wpk + (wunit + q) * kWRecBytes + kWRecScales, 256,
                 &ctl.sc_full[lane]);
    }
    __syncwarp();
    // --- 2. activations are the preceding kernel's output; the residual map
    // comes from the MMA warp
    pdl_wait();
    volatile int never0 = 0;
    mbar_wait(&ctl.map_ready, 0, &never0, tmo, p.err);
    // --- 3. one unit per iteration, its copies spread over the warp's lanes
    // (a bulk copy costs its issuing thread a fixed time, so one thread
    // issuing every copy would limit the stream)
    int i = pw;
    for (; i < nunits; i += 2) {
      const int st = i % NS;
      const int64_t u = u0 + i;
      const int64_t tile = unit_tile(u);
      const int g0 = unit_g0(u);
      const int m0 = tile_mt(tile) * TN;
      const int64_t wunit = static_cast<int64_t>(tile_t(tile)) * G + g0;
      uint8_t* sb = smem + st * C::kStageBytes;
      const int sc = i % NSC;
      uint8_t* scb = scring + sc * C::kScBytes;
      int wait_ok = 1;
      if (lane == 0 && i >= pre) wait_ok = mbar_wait(&ctl.empty[st], ((i / NS) & 1) ^ 1, abort_flag, tmo, p.err);
      if (lane == 0 && i >= NSC && wait_ok)
        wait_ok = mbar_wait(&ctl.sc_empty[sc], ((i / NSC) & 1) ^ 1, abort_flag, tmo, p.err);
      if (!__shfl_sync(0xFFFFFFFFu, wait_ok, 0)) break;
      const int rows = min(TN, p.Mp - m0);  // token rows present (multiple of 8)
      int e[UG][2];
      uint32_t rs_bytes = 0;
#pragma unroll
      for (int q = 0; q < UG; ++q)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          e[q][h] = res_map[h][i * UG + q];
          rs_bytes += e[q][h] >= 0 ? 128 : 0;
        }
      if (lane == 0) {
#pragma unroll
        for (int q = 0; q < UG; ++q) {
          ctl.blk[st][q][0] = ctl.sblk[sc][q][0] = e[q][0];
          ctl.blk[st][q][1] = ctl.sblk[sc][q][1] = e[q][1];
        }
        // weights of prefetched stages were already counted
        mbar_arrive_expect_tx(&ctl.full[st], (i >= pre ? UG * kWRecBytes : 0) + UG * rows * 64);
        mbar_arrive_expect_tx(&ctl.sc_full[sc], (i >= pre ? UG * 256 : 0) + UG * rows * 2 + rs_bytes);
        if (i < 12) MQ_TRACE(8 + i);
      }
      __syncwarp();
      if (i >= pre) {
        if (lane == 1) bulk_g2s(sb + C::oA, p.wpk + wunit * kWRecBytes, UG * kWRecBytes, &ctl.full[st]);
        if (lane >= 24 && lane < 24 + UG)
          bulk_g2s(scb + C::sWS + (lane - 24) * 256, p.wpk + (wunit + lane - 24) * kWRecBytes + kWRecScales, 256,
                   &ctl.sc_full[sc]);
      }
      if (merged) {
        if (lane == 3)
          bulk_g2s(sb + C::oXQ, p.xq + static_cast<int64_t>(g0) * p.Mp * 64, UG * p.Mp * 64, &ctl.full[st]);
        if (lane == 4) bulk_g2s(scb + C::sSX, p.xs + static_cast<int64_t>(g0) * p.Mp, UG * p.Mp * 2, &ctl.sc_full[sc]);
      } else if (lane >= 3 && lane < 3 + 2 * UG) {
        const int q = (lane - 3) >> 1;
        const int64_t row0 = static_cast<int64_t>(g0 + q) * p.Mp + m0;
        if (((lane - 3) & 1) == 0)
          bulk_g2s(sb + C::oXQ + q * C::kXQ, p.xq + row0 * 64, rows * 64, &ctl.full[st]);
        else
          bulk_g2s(scb + C::sSX + q * TN * 2, p.xs + row0, rows * 2, &ctl.sc_full[sc]);
      }
      // residual blocks: scales into the stage (lanes 8..), codes into the
      // residual ring in block order (lanes 16..)
      int rok = 1;
      if (lane >= 8 && lane < 8 + 2 * UG) {
        const int q = (lane - 8) >> 1, h = (lane - 8) & 1;
        if (e[q][h] >= 0)
          bulk_g2s(scb + C::sRS + (q * 2 + h) * 128, p.rpk + static_cast<int64_t>(e[q][h]) * kRRecBytes + kRRecScales, 128,
                   &ctl.sc_full[sc]);
      }
      if (lane >= 16 && lane < 16 + 2 * UG) {
        const int q = (lane - 16) >> 1, h = (lane - 16) & 1;
        if (e[q][h] >= 0) {
          const int ri = res_slot[h][i * UG + q];
          const int rs = ri % NR;
          if (mbar_wait(&ctl.r_empty[rs], ((ri / NR) & 1) ^ 1, abort_flag, tmo, p.err)) {
            mbar_arrive_expect_tx(&ctl.r_full[rs], 4096);
            bulk_g2s(rring + rs * 4096, p.rpk + static_cast<int64_t>(e[q][h]) * kRRecBytes, 4096, &ctl.r_full[rs]);
          } else {
            rok = 0;
          }
        }
      }
      if (!__all_sync(0xFFFFFFFFu, rok)) break;
    }
    // Every copy issued here is waited on by a consumer before the CTA ends;
    // after an abort, the end of the kernel gives copies in flight time to land.
  } else if (warp == kWarpMma) {
    // residual map of this CTA's groups, from the block-list rows of its tiles
    for (int i = lane; i < ngroups; i += 32) {
      res_map[0][i] = -1;
      res_map[1][i] = -1;
    }
    __syncwarp();
    if (p.nnzb > 0) {
      const int64_t gbase = u0 * UG;  // CTA-local group index = (tile*G + g) - gbase
      for (int64_t tile = unit_tile(u0); tile <= unit_tile(u1 - 1); ++tile) {
        const int t = tile_t(tile);
        for (int half = 0; half < 2; ++half) {
          const int br = 2 * t + half;
          // entries are clamped to [0, nnzb) so a malformed list cannot index out of bounds
          const int e0 = max(0, min(p.nnzb, p.row_ptr[br]));
          const int e1 = max(e0, min(p.nnzb, p.row_ptr[br + 1]));
          for (int e = e0 + lane; e < e1; e += 32) {
            const int g = p.col_idx[e];
            const int64_t lg = tile * G + g - gbase;
            if (g >= 0 && g < G && lg >= 0 && lg < ngroups) res_map[half][lg] = e;
          }
        }
      }
    }
    __syncwarp();
    // position of each residual block in the CTA's block order (groups
    // ascending, top half first): lane l scans a contiguous chunk of groups
    {
      const int chunk = (ngroups + 31) / 32;
      const int l0 = min(ngroups, lane * chunk), l1 = min(ngroups, l0 + chunk);
      int cnt = 0;
      for (int lg = l0; lg < l1; ++lg) cnt += (res_map[0][lg] >= 0) + (res_map[1][lg] >= 0);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      int pos = incl - cnt;
      for (int lg = l0; lg < l1; ++lg)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          if (res_map[h][lg] >= 0) res_slot[h][lg] = static_cast<int16_t>(pos++);
    }
    mbar_arrive(&ctl.map_ready);
    if (lane == 0) {
      int item = 0;   // global item order (accumulator ring)
      int gitem[NG];  // per converter group item counters (A rings)
#pragma unroll
      for (int gg = 0; gg < NG; ++gg) gitem[gg] = 0;
      bool ok = true;
      for (int i = 0; i < nunits && ok; ++i) {
        const int st = i % NS;
        const uint32_t b_base = smem_u32(smem + st * C::kStageBytes + C::oB);
        for (int q = 0; q < UG && ok; ++q) {
          const int grp = (i * UG + q) % NG;
          int nitems = 1;
          for (int k = 0; k < nitems; ++k, ++item) {
            int li = 0;
#pragma unroll
            for (int gg = 0; gg < NG; ++gg)
              if (gg == grp) li = gitem[gg]++;
            const int a = grp * SPG + li % SPG, d = item % ND;
            if (!mbar_wait(&ctl.conv_full[a], (li / SPG) & 1, abort_flag, tmo, p.err)) { ok = false; break; }
            if (k == 0) nitems = 1 + ((ctl.blk[st][q][0] >= 0) || (ctl.blk[st][q][1] >= 0));
            if (!mbar_wait(&ctl.d_empty[d], ((item / ND) & 1) ^ 1, abort_flag, tmo, p.err)) { ok = false; break; }
            tc_fence_after();
            if (q == 0 && k == 0 && i < 12) MQ_TRACE(44 + i);
            const uint32_t a_col = tmem + C::tA + a * 32;
            const uint32_t d_col = tmem + C::tD + d * TN;
            const uint32_t b_addr = b_base + q * C::kB;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tc_mma_ts(d_col, a_col + 8 * j, sw128_desc(b_addr + 32 * j), C::kIdesc, j > 0);
            tc_commit(&ctl.a_empty[a]);
            tc_commit(&ctl.d_full[d]);
          }
        }
        if (ok) tc_commit(&ctl.empty[st]);
      }
      // Let the issued MMAs finish before TMEM can be released.
      if (item > 0) {
        volatile int never = 0;
        const int last = item - 1;
        mbar_wait(&ctl.d_full[last % ND], (last / ND) & 1, &never, tmo, p.err);
      }
    }
  } else if (warp < kWarpDrain0) {
    // ---------------- converters ----------------
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // weight row of this thread (TMEM lane)
    const int grp = (warp - kWarpConv0) >> 2;
    const int ctid = (((warp - kWarpConv0) & 3) << 5) + lane;  // 0..127 within the group
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int half = r >> 6;
    volatile int never0 = 0;
    mbar_wait(&ctl.map_ready, 0, &never0, tmo, p.err);  // res_slot
    int item = 0;  // this converter group's items
    for (int k = grp; k < ngroups; k += NG) {
      const int i = k / UG, q = k % UG;
      const int st = i % NS;
      if (!mbar_wait(&ctl.full[st], (i / NS) & 1, abort_flag, tmo, p.err)) break;
      uint8_t* sb = smem + st * C::kStageBytes;
      const int e_top = ctl.blk[st][q][0], e_bot = ctl.blk[st][q][1];
      if (ctid == 0 && q == 0 && i < 12) MQ_TRACE(20 + i);
      {  // base item: weights of row r, K-step j = the 16 bytes at j*2048 + r*16
        const int a = grp * SPG + item % SPG;
        if (!mbar_wait(&ctl.a_empty[a], ((item / SPG) & 1) ^ 1, abort_flag, tmo, p.err)) break;
        tc_fence_after();
        codes_to_tmem(sb + C::oA + q * kWRecBytes + r * 16, 2048, tmem + lane_base + C::tA + a * 32);
        // activations: row m, K-step j -> two 16-byte chunks 2j, 2j+1 of the
        // 128-byte swizzled row (chunk c of row m sits at chunk c ^ (m & 7))
        const uint8_t* xsrc = sb + C::oXQ + q * xq_stride;
        uint8_t* btile = sb + C::oB + q * C::kB;
        for (int idx = ctid; idx < TN * 4; idx += 128) {
          const int m = idx >> 2, j = idx & 3;
          const uint4 pk = *reinterpret_cast<const uint4*>(xsrc + m * 64 + j * 16);
          uint4 lo, hi;
          int4x8_to_e4m3(pk.x, lo.x, lo.y);
          int4x8_to_e4m3(pk.y, lo.z, lo.w);
          int4x8_to_e4m3(pk.z, hi.x, hi.y);
          int4x8_to_e4m3(pk.w, hi.z, hi.w);
          uint8_t* row = btile + (m >> 3) * 1024 + (m & 7) * 128;
          *reinterpret_cast<uint4*>(row + (((2 * j) ^ (m & 7)) * 16)) = lo;
          *reinterpret_cast<uint4*>(row + (((2 * j + 1) ^ (m & 7)) * 16)) = hi;
        }
        tc_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        if (ctid == 0 && q == 0 && i < 12) MQ_TRACE(32 + i);
        mbar_arrive(&ctl.conv_full[a]);
        ++item;
      }
      if (e_top >= 0 || e_bot >= 0) {  // residual item (same activation tile)
        const int a = grp * SPG + item % SPG;
        if (!mbar_wait(&ctl.a_empty[a], ((item / SPG) & 1) ^ 1, abort_flag, tmo, p.err)) break;
        tc_fence_after();
        if ((half == 0 ? e_top : e_bot) >= 0) {  // warp-uniform: a warp's 32 rows sit in one half
          const int ri = res_slot[half][k];
          const int rs = ri % NR;
          if (!mbar_wait(&ctl.r_full[rs], (ri / NR) & 1, abort_flag, tmo, p.err)) break;
          codes_to_tmem(rring + rs * 4096 + (r & 63) * 16, 1024, tmem + lane_base + C::tA + a * 32);
          tc_wait_st();
          mbar_arrive(&ctl.r_empty[rs]);
        }
        tc_fence_before();
        mbar_arrive(&ctl.conv_full[a]);
        ++item;
      }
    }
  } else {
    // ---------------- drain + epilogue ----------------
    pdl_wait();  // the workspace and Y may still be in use by the preceding kernel
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int dtid = (warp - kWarpDrain0) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int half = r >> 6;
    uint64_t acc[TN / 2];  // packed fp32 pairs (tokens 2j, 2j+1)
#pragma unroll
    for (int i = 0; i < TN / 2; ++i) acc[i] = 0;
    int item = 0;
    int nbar = 0;  // phases of drain_bar used so far
    bool ok = true;
    // bounded barrier of the 128 drain threads (an mbarrier, so a broken pipeline cannot hang it)
    auto drain_sync = [&]() -> bool {
      mbar_arrive(&ctl.drain_bar);
      const bool passed = mbar_wait(&ctl.drain_bar, nbar & 1, abort_flag, tmo, p.err);
      ++nbar;
      return passed;
    };
    auto store_tile = [&](int m0, int n, int mvalid) {
#pragma unroll
      for (int j = 0; j < TN / 2; ++j) {
        float v[2];
        f2unpack(acc[j], v[0], v[1]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int mi = 2 * j + h;
          if (mi < mvalid) {
            const int64_t off = static_cast<int64_t>(m0 + mi) * p.ldy + n;
            if (p.y_f32)
              static_cast<float*>(p.y)[off] = v[h];
            else
              static_cast<__nv_bfloat16*>(p.y)[off] = __float2bfloat16_rn(v[h]);
          }
        }
      }
    };
    for (int i = 0; i < nunits && ok; ++i) {
      const int64_t u = u0 + i;
      const int sc = i % NSC;
      if (!mbar_wait(&ctl.sc_full[sc], (i / NSC) & 1, abort_flag, tmo, p.err)) { ok = false; break; }
      const uint8_t* scb = scring + sc * C::kScBytes;
      const int64_t tile = unit_tile(u);
      const int g0 = unit_g0(u);
      const int n = tile_t(tile) * kTileN + r;
      const int m0 = tile_mt(tile) * TN;
      for (int q = 0; q < UG && ok; ++q) {
        const int e_top = ctl.sblk[sc][q][0], e_bot = ctl.sblk[sc][q][1];
        const int nitems = 1 + (e_top >= 0 || e_bot >= 0);
        const int e_mine = half == 0 ? e_top : e_bot;
        const __half2* sx2 = reinterpret_cast<const __half2*>(reinterpret_cast<const uint16_t*>(scb + C::sSX) + q * sx_stride);
        for (int k = 0; k < nitems; ++k, ++item) {
          const int d = item % ND;
          if (!mbar_wait(&ctl.d_full[d], (item / ND) & 1, abort_flag, tmo, p.err)) { ok = false; break; }
          if (dtid == 0 && item >= 8 && item < 12) MQ_TRACE(68 + item - 8);
          tc_fence_after();
          const bool use = (k == 0) || (e_mine >= 0);
          const float s =
              (k == 0) ? __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(scb + C::sWS)[q * 128 + r]))
              : use    ? __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(scb + C::sRS)[q * 128 + r]))
                       : 0.0f;
          const uint64_t s2 = f2pack(s, s);
#pragma unroll
          for (int cc = 0; cc < TN / 16; ++cc) {
            uint32_t dv[16];
            tmem_ld16(tmem + lane_base + C::tD + d * TN + 16 * cc, dv);
            tc_wait_ld();
            if (dtid == 0 && cc == 0 && item >= 8 && item < 12) MQ_TRACE(72 + item - 8);
            if (kDebug) {
#pragma unroll
              for (int i2 = 0; i2 < 16; ++i2) {
                const int m = m0 + 16 * cc + i2;
                if (m < p.M && use) {
                  const int32_t v = static_cast<int32_t>(__uint_as_float(dv[i2]));
                  if (k == 0)
                    p.dots_w[(static_cast<int64_t>(m) * p.N + n) * G + g0 + q] = v;
                  else
                    p.dots_r[(static_cast<int64_t>(m) * p.nnzb + e_mine) * 64 + (r & 63)] = v;
                }
              }
            } else if (use) {
#pragma unroll
              for (int j2 = 0; j2 < 8; ++j2) {
                const int jp = 8 * cc + j2;  // token pair
                // tokens past the scale rows (m >= Mp) carry stale scales: zero them
                const float2 sxv = (m0 + 2 * jp < p.Mp) ? __half22float2(sx2[jp]) : make_float2(0.0f, 0.0f);
                const uint64_t t2 = f2mul(f2pack(__uint_as_float(dv[2 * j2]), __uint_as_float(dv[2 * j2 + 1])), s2);
                acc[jp] = f2fma(f2pack(sxv.x, sxv.y), t2, acc[jp]);
              }
            }
          }
          if (dtid == 0 && item >= 8 && item < 12) MQ_TRACE(76 + item - 8);
          tc_fence_before();
          mbar_arrive(&ctl.d_empty[d]);
        }
      }
      if (!ok) break;
      mbar_arrive(&ctl.sc_empty[sc]);  // scales read: the scale slot may be refilled
      if (dtid == 0 && i < 12) MQ_TRACE(56 + i);
      // ---- tile end: store Y, or hand a stream-K piece to the workspace ----
      const bool tile_end = (g0 + UG == G) || (i == nunits - 1);
      if (!kDebug && tile_end) {
        const int mvalid = min(TN, p.M - m0);
        const int64_t tu0 = tile * GU, tu1 = tu0 + GU;  // the tile's units
        if (tu0 >= u0 && tu1 <= u1) {  // whole tile in this CTA
          store_tile(m0, n, mvalid);
        } else {
          // A stream-K piece: write it (thread-contiguous rows), count it in;
          // the CTA that brings the count to the number of pieces finishes
          // the tile after its own range is done (deferred: no stall here).
          const int slot = (tile == unit_tile(u0)) ? 0 : 1;
          uint4* mypart = reinterpret_cast<uint4*>(p.partials + ((c * 2 + slot) * kTileN + r) * TN);
#pragma unroll
          for (int q4 = 0; q4 < TN / 4; ++q4)
            mypart[q4] = make_uint4(static_cast<uint32_t>(acc[2 * q4]), static_cast<uint32_t>(acc[2 * q4] >> 32),
                                    static_cast<uint32_t>(acc[2 * q4 + 1]), static_cast<uint32_t>(acc[2 * q4 + 1] >> 32));
          __threadfence();
          if (!drain_sync()) { ok = false; break; }
          if (dtid == 0) {
            const int64_t cf = cta_of_unit(tu0, U, P), cl = cta_of_unit(tu1 - 1, U, P);
            const int old = atomicAdd(&p.counters[cf], 1);  // CTA cf starts at most one cut tile
            if (old == static_cast<int>(cl - cf)) ctl.deferred[ctl.ndeferred++] = tile;
          }
        }
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc[j] = 0;
      }
    }
    if (dtid == 0) MQ_TRACE(2);
    // ---- finish the tiles this CTA completed last: bulk-copy every piece
    // into the (now idle) stage memory, sum in CTA order, store Y ----
    if (!kDebug && ok && drain_sync()) {
      const int nd = ctl.ndeferred;
      constexpr uint32_t kPieceBytes = TN * kTileN * 4;
      const int per_round = C::kRingBytes / kPieceBytes;
      int nred = 0;  // phases of red_bar used
      for (int di = 0; di < nd && ok; ++di) {
        const int64_t tile = ctl.deferred[di];
        const int64_t tu0 = tile * GU, tu1 = tu0 + GU;
        const int64_t cf = cta_of_unit(tu0, U, P), cl = cta_of_unit(tu1 - 1, U, P);
        const int m0 = tile_mt(tile) * TN;
        const int n = tile_t(tile) * kTileN + r;
        const int mvalid = min(TN, p.M - m0);
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc[j] = 0;
        for (int64_t cb = cf; cb <= cl && ok; cb += per_round) {
          const int npieces = static_cast<int>(min(static_cast<int64_t>(per_round), cl - cb + 1));
          if (dtid == 0) {
            __threadfence();
            fence_proxy_async_global();  // other CTAs' generic writes -> this bulk (async) read
            mbar_arrive_expect_tx(&ctl.red_bar, npieces * kPieceBytes);
            for (int k = 0; k < npieces; ++k) {
              const int64_t c2 = cb + k;
              const int slot2 = (tile == unit_tile(cta_first_unit(c2, U, P))) ? 0 : 1;
              bulk_g2s(smem + k * kPieceBytes, p.partials + (c2 * 2 + slot2) * (kTileN * TN), kPieceBytes,
                       &ctl.red_bar);
            }
          }
          if (!mbar_wait(&ctl.red_bar, nred & 1, abort_flag, tmo, p.err)) { ok = false; break; }
          ++nred;
          for (int k = 0; k < npieces; ++k) {
            const uint64_t* piece = reinterpret_cast<const uint64_t*>(smem + k * kPieceBytes) + r * (TN / 2);
#pragma unroll
            for (int j = 0; j < TN / 2; ++j) {
              float a0, a1, b0, b1;
              f2unpack(acc[j], a0, a1);
              f2unpack(piece[j], b0, b1);
              acc[j] = f2pack(a0 + b0, a1 + b1);  // ascending CTA order, one rounding per add
            }
          }
          if (!drain_sync()) { ok = false; break; }  // smem free for the next round
        }
        if (!ok) break;
        store_tile(m0, n, mvalid);
        if (dtid == 0) p.counters[cf] = 0;  // ready for the next launch
      }
    }
  }

  if (warp == kWarpDrain0 && lane == 0) MQ_TRACE(3);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*abort_flag) {
    // A wait gave up somewhere: bulk copies or MMAs may still be in flight
    // into this CTA's shared or tensor memory.  They finish within
    // microseconds on their own; give them 200 us (bounded) before release.
    if (threadIdx.x == 0) {
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 200000ull) {
      }
    }
    __syncthreads();
  }
  if (warp == kWarpMma) tmem_dealloc(tmem, C::kTmemCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

struct Plan {
  int tn, ug;
  int tiles_m, tiles_n, G;
  int64_t units;
  int ctas;
  size_t ws_partials;  // bytes
  size_t ws_counters;  // bytes
};

// Token-tile width.  Above 32 tokens, 64: two converter groups share a CTA's
// items (at 128 there is room for one), and the 2048-token prefill runs ~10 %
// faster than with 128-token tiles.
static int pick_tn(int64_t M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  return 64;
}

static size_t a256(size_t b) { return (b + 255) / 256 * 256; }

// The plan depends on (M, N, K) and the current device's SM count (the
// persistent grid; 152 when no device is current), so a workspace sized on a
// device serves that device.
static Plan make_plan(int64_t M, int64_t N, int64_t K) {
  Plan pl;
  pl.tn = pick_tn(M);
  pl.tiles_m = static_cast<int>((M + pl.tn - 1) / pl.tn);
  pl.tiles_n = static_cast<int>(N / kTileN);
  pl.G = static_cast<int>(K / kGroup);
  pl.ug = (pl.tn <= 64 && pl.G % 2 == 0) ? 2 : 1;
  pl.units = static_cast<int64_t>(pl.tiles_m) * pl.tiles_n * (pl.G / pl.ug);
  // at least kMinUnitsPerCta units per CTA bounds the pieces a tile is cut into
  const int sms = current_sms();  // one persistent CTA per SM of the current device
  int64_t ctas = std::min<int64_t>(sms > 0 ? sms : kPlanCtasNoDevice, std::max<int64_t>(1, pl.units / kMinUnitsPerCta));
  const int64_t min_ctas = (pl.units * pl.ug + kMaxGroupsPerCta - 1) / kMaxGroupsPerCta;
  if (ctas < min_ctas) ctas = min_ctas;
  pl.ctas = static_cast<int>(ctas);
  pl.ws_partials = a256(static_cast<size_t>(pl.ctas) * 2 * pl.tn * kTileN * sizeof(float));
  pl.ws_counters = kWsZeroBytes;  // counters [ctas] at the start, in the zeroed prefix
  return pl;
}

size_t zipper_workspace_bytes(int64_t M, int64_t tiles, int64_t K);
bool image_form_wanted(int64_t M);
size_t image_workspace_bytes(int64_t M, int64_t N, int64_t K);
mq_status image_gemm_launch(bool* handled, const uint8_t* xq, const uint16_t* xs, int64_t M, const uint8_t* wpk,
                            int64_t N, int64_t K, const int32_t* row_ptr, const int32_t* col_idx, int64_t nnzb,
                            const uint8_t* rpk, void* y, int64_t ldy, mq_dtype yt, int32_t* dots_w, int32_t* dots_r,
                            void* ws, size_t ws_bytes, cudaStream_t stream);

// Bytes of workspace of the general kernel: its pieces, or the image form's
// operand images where that form serves M (image_gemm.cu).
size_t general_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const Plan pl = make_plan(M, N, K);
  const size_t conv = pl.ws_partials + pl.ws_counters;
  return image_form_wanted(M) ? std::max(conv, image_workspace_bytes(M, N, K)) : conv;
}

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  return std::max(general_workspace_bytes(M, N, K), zipper_workspace_bytes(M, N / kTileN, K));
}

// Bytes of workspace the kernel that mq_w4a4_residual_gemm will run for
// (M, N, K) on the current device reads and writes.
size_t gemm_run_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (const size_t z = zipper_workspace_bytes(M, N / kTileN, K)) return z;
  const Plan pl = make_plan(M, N, K);
  return pl.ws_partials + pl.ws_counters;
}

template <int TN, int UG, bool kDebug>
static mq_status launch_cfg(const GemmParams& gp, const Plan& pl, cudaStream_t stream) {
  using C = Cfg<TN, UG>;
  auto kern = w4a4_residual_gemm_kernel<TN, UG, kDebug>;
  static std::mutex mu;
  static bool attr_set[kGemmMaxDevices] = {};  // per device, per template instance
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kGemmMaxDevices) return launch_status("gemm: device");
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
        return launch_status("gemm: smem attribute");
      attr_set[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.ctas), 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, gp) != cudaSuccess) return launch_status("gemm launch");
  return launch_status("gemm");
}

template <int TN, bool kDebug>
static mq_status launch_tn(const GemmParams& gp, const Plan& pl, cudaStream_t stream) {
  return pl.ug == 2 ? launch_cfg<TN, (TN <= 64 ? 2 : 1), kDebug>(gp, pl, stream) : launch_cfg<TN, 1, kDebug>(gp, pl, stream);
}

mq_status zipper_launch(bool* handled, int nmat, const uint8_t* const* wpk, const int64_t* N,
                        const int32_t* const* row_ptr, const int32_t* const* col_idx, const int64_t* nnzb,
                        const uint8_t* const* rpk, void* const* y, const int64_t* ldy, mq_dtype yt, const uint8_t* xq,
                        const uint16_t* xs, const void* x, mq_dtype xt, int64_t ldx, uint8_t* xq_out,
                        uint16_t* xs_out, int64_t M, int64_t K, int32_t* dots_w, int32_t* dots_r, void* ws,
                        size_t ws_bytes, cudaStream_t stream);

mq_status gemm_launch(const uint8_t* xq, const uint16_t* xs, int64_t M, const uint8_t* wpk, int64_t N, int64_t K,
                      const int32_t* row_ptr, const int32_t* col_idx, int64_t nnzb, const uint8_t* rpk, void* y,
                      int64_t ldy, mq_dtype yt, int32_t* dots_w, int32_t* dots_r, void* ws, size_t ws_bytes,
                      cudaStream_t stream) {
  bool handled = false;
  {
    // Decode batches: the stream-K kernel (zipper.cu), when it covers the shape.
    void* yy = y;
    const mq_status zs = zipper_launch(&handled, 1, &wpk, &N, &row_ptr, &col_idx, &nnzb, &rpk, &yy, &ldy, yt, xq, xs,
                                       nullptr, MQ_F16, 0, nullptr, nullptr, M, K, dots_w, dots_r, ws, ws_bytes,
                                       stream);
    if (handled || zs != MQ_OK) return zs;
  }
  {
    // Large batches: the image form, when the workspace holds its images.
    const mq_status is = image_gemm_launch(&handled, xq, xs, M, wpk, N, K, row_ptr, col_idx, nnzb, rpk, y, ldy, yt,
                                           dots_w, dots_r, ws, ws_bytes, stream);
    if (handled || is != MQ_OK) return is;
  }
  const Plan pl = make_plan(M, N, K);
  if (pl.ctas > kWsZeroBytes / 4)
    return set_error(MQ_ERR_INVALID_ARG, "gemm: M=%lld N=%lld K=%lld is too large for one launch", (long long)M,
                     (long long)N, (long long)K);
  if (ws_bytes < pl.ws_partials + pl.ws_counters || ws == nullptr)
    return set_error(MQ_ERR_WORKSPACE, "gemm: workspace of %zu bytes needed, %zu given",
                     pl.ws_partials + pl.ws_counters, ws_bytes);
  GemmParams gp;
  gp.xq = xq;
  gp.xs = xs;
  gp.wpk = wpk;
  gp.row_ptr = row_ptr;
  gp.col_idx = col_idx;
  gp.rpk = rpk;
  gp.y = y;
  gp.y_f32 = yt == MQ_F32;
  gp.dots_w = dots_w;
  gp.dots_r = dots_r;
  gp.counters = static_cast<int32_t*>(ws);
  gp.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + pl.ws_counters);
  gp.M = static_cast<int>(M);
  gp.Mp = static_cast<int>((M + 7) / 8 * 8);
  gp.N = static_cast<int>(N);
  gp.ldy = ldy;
  gp.K = static_cast<int>(K);
  gp.G = pl.G;
  gp.tiles_n = pl.tiles_n;
  gp.tiles_m = pl.tiles_m;
  gp.nnzb = static_cast<int>(nnzb);
  gp.units = pl.units;
  gp.ctas = pl.ctas;
  gp.timeout_ns = wait_timeout_ns();
  gp.err = device_error_word();
  if (!gp.err) return set_error(MQ_ERR_CUDA, "gemm: device error word unavailable");
  const bool dbg = dots_w != nullptr;
  switch (pl.tn) {
    case 16: return dbg ? launch_tn<16, true>(gp, pl, stream) : launch_tn<16, false>(gp, pl, stream);
    case 32: return dbg ? launch_tn<32, true>(gp, pl, stream) : launch_tn<32, false>(gp, pl, stream);
    default: return dbg ? launch_tn<64, true>(gp, pl, stream) : launch_tn<64, false>(gp, pl, stream);
  }
}

}  // namespace mq
