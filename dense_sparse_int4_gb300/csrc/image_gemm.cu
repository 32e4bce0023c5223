// Prefill form of the fused W4A4 + block-sparse 4-bit residual GEMM
// (ZipperEngine, MosaicQuant summary, Metodologia 3).  The same sum as the
// general kernel,
//
//   Y[m,n] = sum_g sx[m,g] * ( sw[n,g] * Dw[m,n,g] + sr[n,g] * Dr[m,n,g] ),
//
// for token counts at which the tensor pipe, not the weight stream, bounds
// the call.  The general kernel converts INT4 codes to E4M3 on the CUDA cores
// for every (token tile, weight tile) pair, so at thousands of tokens its
// converters, not the tensor cores, set the pace.  Here one pre-pass per call
// writes each operand once, as the exact shared-memory image the MMA reads:
//   * every base record's codes: 128 rows x 128 inputs of E4M3 (the same
//     integers), 128B-swizzled K-major, 16 KiB per (weight tile, group);
//   * every residual block's codes: 64 rows x 128 inputs, 8 KiB;
//   * the activations: per group, every token row (padded with zero codes to
//     whole token tiles), and their scales as fp32 (zero past M).
// The GEMM moves each operand with one 1-D bulk copy per stage and runs
// tcgen05.mma with both operands in shared memory; the CUDA cores only apply
// the per-group scales.
//
// A unit is two consecutive groups of one (weight tile, token tile) (one
// group at the end of a tile of odd G): every role pays its waits, arrivals
// and loop once per two groups.  Roles per CTA (one CTA per SM, persistent
// stream-K over units; tiles are token-tile major, so that the CTAs running at
// one time read the same few weight tiles and every image stays in L2):
//   warps 0, 2 producers, alternating units: one ring of 16 KiB slots takes
//              each unit's images in order (weight and activation image per
//              group, then one residual image (top block at 0, bottom block at
//              8 KiB) per group that has blocks); the drain's scales go to a
//              ring of their own.  Slots are released in unit order, so a
//              unit's slots are free once the unit that last held its last
//              slot is done.  The copies of a unit (up to 16) leave in one warp
//              instruction, their addresses worked out before the waits.
//   warp 1     builds the CTA's residual map and each unit's first slot,
//              then one thread issues per unit 4 MMAs (K = 32 each) per group
//              into a TMEM accumulator of 256 columns (the two groups side by
//              side), and, where a group has residual blocks, 4 more from its
//              residual image into the next accumulator (M = 128: a half
//              without a block gives rows nobody reads).
//   warps 3-10 drain, 2 warps per TMEM lane quarter, TN/2 tokens each (11
//              warps leave a thread 168 registers): load a group's dots (32
//              columns at a time), free the accumulator after
//              the last load, acc += sx * (s * D) in packed fp32 pairs; at tile
//              ends store Y or a stream-K piece.  Tiles cut by a CTA range are
//              finished by the CTA whose piece arrives last, summing the pieces
//              in CTA order (deterministic; no floating-point atomics).
// Every wait is bounded (mbar_wait): a broken pipeline reports a timeout in
// the device error word and the kernel returns.
#include "mq_internal.cuh"

#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace mq {

namespace {

constexpr int kImgMaxDevices = 64;
// the image form's default lower bound on M (measured: 64 tokens run faster on the
// converter form, 128 on this one)
constexpr int kImgMinTokens = 128;
constexpr int kImgMaxUnitsPerCta = 512;  // size of the CTA's residual map
constexpr int kImgPlanCtasNoDevice = 152;
constexpr int kImgMinUnitsPerCta = 4;
constexpr int kWImg = 16384;  // image of one (weight tile, group): 128 rows x 128 bytes
constexpr int kRImg = 8192;   // image of one residual block: 64 rows x 128 bytes
// warps 0 and 2 producers (alternating units), 1 block list + MMA, 3-10 drain
constexpr int kWarpProd = 0, kWarpMma = 1, kWarpProd2 = 2, kWarpDrain0 = 3, kDrainWarps = 8;

template <int TN>
struct ICfg {
  static constexpr int kUG = 2;         // groups per unit
  static constexpr int kA = kWImg;      // weight image of a group
  static constexpr int kB = TN * 128;   // activation image of a group
  // One ring of 16 KiB slots holds every image a unit needs, in order: the
  // weight and activation images of each group, then the residual image (top
  // block, bottom block) of each group that has one.  A unit takes 2 slots per
  // group and 1 per group with residual blocks, so the ring keeps three units
  // without residual in flight, and residual blocks take room only where the
  // block list has them.
  static constexpr int kSlot = 16384;
  static_assert(kA == kSlot && kB == kSlot && 2 * kRImg == kSlot, "one image per slot");
  static constexpr int kSlots = 12;
  static constexpr int kUnitBars = 8;   // full / done barriers, by unit (more than the units in flight)
  static constexpr int kScSlots = 8;
  // scale slot, per group: weight scales [128] fp16, residual scales [2][64] fp16, activation scales [TN] fp32
  static constexpr int sWS = 0, sRS = 256, sSX = 512;
  static constexpr int kScGroup = 512 + TN * 4;
  static constexpr int kScBytes = kUG * kScGroup;
  static constexpr int kDCols = kUG * TN;        // TMEM columns of one item (a unit's groups side by side)
  static constexpr int kDSlots = 512 / kDCols;   // TMEM accumulators (all 512 columns)
  static constexpr int kCols = TN * 4 / kDrainWarps;  // tokens per drain thread (4 lane quarters)
  static constexpr int kThreads = 32 * (kWarpDrain0 + kDrainWarps);
  static constexpr int kRingBytes = kSlots * kSlot;
  static constexpr int kSmemBytes = kRingBytes + kScSlots * kScBytes + 1024 /*align*/;
  static_assert(kSmemBytes + 12 * 1024 <= 227 * 1024, "shared memory budget");
  static_assert(kCols % 32 == 0, "a drain thread loads its dots in 32-column chunks");
  static_assert(kDSlots >= 2, "two accumulators at least");
  // instruction descriptor: D f32, A/B E4M3, both K-major, N = TN, M = 128
  static constexpr uint32_t kIdesc =
      (1u << 4) | (static_cast<uint32_t>(TN >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
};

struct PrepParams {
  const uint8_t* wpk;   // base records [tiles_n][G]
  const uint8_t* rpk;   // residual records [nnzb]
  const uint8_t* xq;    // [G][Mp][64]
  const uint16_t* xs;   // [G][Mp]
  uint8_t* wimg;        // [tiles_n * G][16384]
  uint8_t* rimg;        // [nnzb][8192]
  uint8_t* ximg;        // [G][Mt][128]
  float* sxf;           // [G][Mt]
  int M, Mp, Mt, G;
  int64_t n_w, n_r, n_x, n_s;  // weight, residual and activation images; activation scales
};

struct ImgParams {
  const uint8_t* wimg;
  const uint8_t* rimg;
  const uint8_t* ximg;
  const float* sxf;
  const uint8_t* wpk;  // records: the weight scales
  const uint8_t* rpk;  // residual records: their scales
  const int32_t* row_ptr;
  const int32_t* col_idx;
  void* y;
  int y_f32;
  int64_t ldy;
  int32_t* dots_w;    // debug: raw group dots
  int32_t* dots_r;
  float* partials;    // [ctas][2][128][TN]
  int32_t* counters;  // [ctas] (the workspace's zeroed prefix)
  int M, Mt, N, G, tiles_n, tiles_m, nnzb;
  int64_t units;
  int ctas;
  uint64_t timeout_ns;
  uint32_t* err;
};

template <int NU, int NSC, int ND>
struct __align__(8) ICtl {
  uint64_t full[NU];  // unit i (by i % NU): its images have landed
  uint64_t done[NU];  // unit i: its MMAs have completed (its slots are free)
  uint64_t sc_full[NSC];
  uint64_t sc_empty[NSC];
  uint64_t d_full[ND];
  uint64_t d_empty[ND];
  uint64_t drain_bar;  // bounded barrier of the drain threads
  uint64_t red_bar;    // bulk loads of stream-K pieces
  uint64_t map_ready;  // residual map built
  int32_t blk[NU][2][2];    // per group of unit i: CSR entries of its top / bottom residual block, or -1
  int32_t sblk[NSC][2][2];  // the same, for the drain (lives as long as the scale slot)
  int32_t ng[NU];           // groups of unit i (2, or 1 at the end of a tile of odd G)
  int32_t sng[NSC];
  int64_t deferred[2];      // cut tiles this CTA finishes (at most its first and last)
  uint32_t tmem_base;
  int abort_flag;
  int ndeferred;
};

__device__ __forceinline__ uint64_t img_desc(uint32_t saddr) {  // 128B-swizzled K-major, 8-row atoms of 1024 B
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}
// D[tmem] (+)= A[smem desc] * B[smem desc], E4M3 x E4M3 -> f32, one K = 32 step.
__device__ __forceinline__ void img_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ uint64_t p2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void u2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// One image of `rows` rows (128, or 64 for a residual block): the packed
// codes of row r, K-step j (16 bytes) at src + r*rs + j*js (a null source
// gives zero codes, rows at or past `valid` too) -> the 128B-swizzled K-major
// E4M3 image, row r at r*128, K-step j in chunks 2j (its codes 0..15) and
// 2j+1 (16..31), chunk c stored at c ^ (r & 7).  The block reads the codes
// into shared memory with 16-byte loads along the source's contiguous
// dimension, then writes the image in address order (one 16-byte chunk per
// thread and step): both sides coalesced.
__device__ __forceinline__ void image_tile(uint8_t (*sm)[64], const uint8_t* src, int64_t rs, int64_t js, int rows,
                                           int valid, uint8_t* img) {
  for (int it = threadIdx.x; it < rows * 4; it += blockDim.x) {
    // along r when rows are 16 bytes apart (records), else along j (activations)
    const int r = rs == 16 ? it % rows : it >> 2, j = rs == 16 ? it / rows : it & 3;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (src && r < valid) v = __ldg(reinterpret_cast<const uint4*>(src + r * rs + j * js));
    *reinterpret_cast<uint4*>(&sm[r][16 * j]) = v;
  }
  __syncthreads();
  for (int o = threadIdx.x; o < rows * 8; o += blockDim.x) {
    const int r = o >> 3, x = (o & 7) ^ (r & 7);  // chunk x of row r's codes: K-step x / 2, half x % 2
    const uint2 pk = *reinterpret_cast<const uint2*>(&sm[r][8 * x]);
    uint4 e;
    int4x8_to_e4m3(pk.x, e.x, e.y);
    int4x8_to_e4m3(pk.y, e.z, e.w);
    *reinterpret_cast<uint4*>(img + 16 * o) = e;
  }
  __syncthreads();
}

// The pre-pass: one block per image (a base record, a residual block, or 128
// token rows of one group's activations), then the activation scales.
__global__ void __launch_bounds__(256) image_prep_kernel(const PrepParams p) {
  __shared__ __align__(16) uint8_t sm[128][64];
  // The images overwrite the workspace a preceding GEMM may still read, and
  // the activations may be the preceding kernel's output.
  pdl_wait();
  pdl_trigger();
  const int64_t mtiles = p.Mt / 128;
  const int64_t n_w = p.n_w, n_r = p.n_r, n_x = static_cast<int64_t>(p.G) * mtiles;
  for (int64_t b = blockIdx.x; b < n_w + n_r + n_x; b += gridDim.x) {
    if (b < n_w) {
      image_tile(sm, p.wpk + b * kWRecBytes, 16, 2048, 128, 128, p.wimg + b * kWImg);
    } else if (b < n_w + n_r) {
      const int64_t e = b - n_w;
      image_tile(sm, p.rpk + e * kRRecBytes, 16, 1024, 64, 64, p.rimg + e * kRImg);
    } else {
      const int64_t x = b - n_w - n_r, g = x / mtiles;
      const int m0 = static_cast<int>(x - g * mtiles) * 128;
      image_tile(sm, p.xq + (g * p.Mp + m0) * 64, 64, 16, 128, p.M - m0, p.ximg + (g * p.Mt + m0) * 128);
    }
  }
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t k = tid; k < p.n_s; k += static_cast<int64_t>(gridDim.x) * blockDim.x) {  // scales as fp32, zero past M
    const int64_t g = k / p.Mt;
    const int m = static_cast<int>(k - g * p.Mt);
    p.sxf[k] = m < p.M ? __half2float(__ushort_as_half(p.xs[g * p.Mp + m])) : 0.0f;
  }
}

template <int TN, bool kDebug>
__global__ void __launch_bounds__(ICfg<TN>::kThreads, 1) image_gemm_kernel(const ImgParams p) {
  using C = ICfg<TN>;
  constexpr int NSL = C::kSlots, NU = C::kUnitBars, NSC = C::kScSlots, ND = C::kDSlots, UG = C::kUG;
  extern __shared__ uint8_t smem_raw[];
  __shared__ ICtl<NU, NSC, ND> ctl;
  // per local unit and group: CSR entry of the top / bottom block, or -1
  __shared__ int32_t res_map[UG][2][kImgMaxUnitsPerCta];
  // per local unit: its first slot, counted over the CTA's units (slot ubase[i] % NSL of the ring)
  __shared__ int32_t ubase[kImgMaxUnitsPerCta + 1];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* scring = smem + C::kRingBytes;
  auto slot = [&](int64_t k) { return smem + static_cast<int>(k % NSL) * C::kSlot; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t U = p.units, P = p.ctas, c = blockIdx.x;
  const int64_t u0 = c * U / P, u1 = (c + 1) * U / P;
  const int nunits = static_cast<int>(u1 - u0);
  const int G = p.G, UPT = (G + UG - 1) / UG;  // groups, units per tile
  volatile int* abort_flag = &ctl.abort_flag;
  const uint64_t tmo = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NU; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.done[s], 1);  // the MMA commit
    }
    for (int s = 0; s < NSC; ++s) {
      mbar_init(&ctl.sc_full[s], 1);
      mbar_init(&ctl.sc_empty[s], kDrainWarps);
    }
    for (int s = 0; s < ND; ++s) {
      mbar_init(&ctl.d_full[s], 1);
      mbar_init(&ctl.d_empty[s], kDrainWarps);
    }
    mbar_init(&ctl.drain_bar, kDrainWarps * 32);
    mbar_init(&ctl.red_bar, 1);
    mbar_init(&ctl.map_ready, 32);
    ctl.abort_flag = 0;
    ctl.ndeferred = 0;
    fence_mbar_init();
  }
  // The next kernel may launch now: it waits for this grid before it writes
  // anything this one reads.
  pdl_trigger();
  if (warp == kWarpMma) tmem_alloc(&ctl.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;

  // unit -> tile (token-tile major) and unit of the tile; tile -> weight tile t, token tile mt
  auto unit_tile = [&](int64_t u) { return u / UPT; };
  auto tile_t = [&](int64_t tile) { return static_cast<int>(tile % p.tiles_n); };
  auto tile_mt = [&](int64_t tile) { return static_cast<int>(tile / p.tiles_n); };
  auto owner = [&](int64_t u) { return ((u + 1) * P - 1) / U; };  // the CTA whose range holds unit u
  // A unit's position, advanced unit by unit: the per-unit loops do no
  // divisions (a 64-bit division is a software routine of hundreds of cycles,
  // and two roles would pay it every unit).
  struct Pos {
    int64_t tile;
    int j, t, mt;  // unit of the tile (groups UG*j, UG*j + 1), weight tile, token tile
  };
  const Pos pos0 = {unit_tile(u0), static_cast<int>(u0 % UPT), tile_t(unit_tile(u0)), tile_mt(unit_tile(u0))};
  auto advance = [&](Pos& q) {
    if (++q.j == UPT) {
      q.j = 0;
      ++q.tile;
      if (++q.t == p.tiles_n) q.t = 0, ++q.mt;
    }
  };

  if (warp == kWarpProd || warp == kWarpProd2) {
    const int pw = warp == kWarpProd ? 0 : 1;  // this producer fills units pw, pw + 2, ...
    pdl_wait();  // the images are the pre-pass's output
    volatile int never0 = 0;
    bool ok = mbar_wait(&ctl.map_ready, 0, &never0, tmo, p.err);
    Pos q = pos0;
    if (pw) advance(q);
    // lane L: group gq = L / 8 of the unit, copy kind k = L % 8 (0 weight image, 1 activation image,
    // 2 weight scales, 3 activation scales, 4 / 5 top / bottom residual scales, 6 / 7 their images)
    const int gq = (lane >> 3) & 1, kind = lane & 7, hh = kind & 1;
    for (int i = pw; ok && i < nunits; i += 2, advance(q), advance(q)) {
      const int ub = i % NU, sc = i % NSC;
      const int g0 = UG * q.j, t = q.t, m0 = q.mt * TN;
      const int ng = min(UG, G - g0);
      const int base = ubase[i], nsl = ubase[i + 1] - base;  // the unit's slots: [base, base + nsl) of the ring
      // Everything about the unit's copies is worked out before the waits: a
      // slot is refilled only after the MMAs that read it, so the time from
      // that release to the copies' issue is on the critical path.
      int e4[UG][2];  // residual entries of both groups (-1: none)
#pragma unroll
      for (int g2 = 0; g2 < UG; ++g2)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) e4[g2][h2] = g2 < ng ? res_map[g2][h2][i] : -1;
      const bool hr0 = e4[0][0] >= 0 || e4[0][1] >= 0;
      const int nblk = (e4[0][0] >= 0) + (e4[0][1] >= 0) + (e4[1][0] >= 0) + (e4[1][1] >= 0);
      // this lane's copy
      const bool mine = lane < 8 * ng;
      const int e = mine ? (gq ? e4[1][hh] : e4[0][hh]) : -1;
      const int nsr = __popc(__ballot_sync(0xFFFFFFFFu, (kind == 4 || kind == 5) && e >= 0));
      // The unit's copies, one per lane, leave in one warp instruction (a bulk
      // copy costs its issuing instruction a fixed time); selects, not a
      // switch: divergent lanes would resolve an indirect branch one after another.
      uint8_t* scb = scring + sc * C::kScBytes + gq * C::kScGroup;
      const int g = g0 + gq;
      const int64_t wrec = static_cast<int64_t>(t) * G + g;
      const int64_t ee = e >= 0 ? e : 0;
      const uint8_t* s_a = p.wimg + wrec * kWImg;
      const uint8_t* s_b = p.ximg + (static_cast<int64_t>(g) * p.Mt + m0) * 128;
      const uint8_t* s_ws = p.wpk + wrec * kWRecBytes + kWRecScales;
      const uint8_t* s_sx = reinterpret_cast<const uint8_t*>(p.sxf + static_cast<int64_t>(g) * p.Mt + m0);
      const uint8_t* s_rs = p.rpk + ee * kRRecBytes + kRRecScales;
      const uint8_t* s_ri = p.rimg + ee * kRImg;
      const uint8_t* src = kind == 0 ? s_a : kind == 1 ? s_b : kind == 2 ? s_ws : kind == 3 ? s_sx : kind < 6 ? s_rs : s_ri;
      // slots of the unit: weight, activation image per group, then one residual image per group with blocks
      const int ks = kind < 2 ? 2 * gq + kind : 2 * ng + (gq && hr0 ? 1 : 0);
      uint8_t* dst = kind < 2    ? slot(base + ks)
                     : kind == 2 ? scb + C::sWS
                     : kind == 3 ? scb + C::sSX
                     : kind < 6  ? scb + C::sRS + hh * 128
                                 : slot(base + ks) + hh * kRImg;
      const uint32_t bytes = kind < 2    ? static_cast<uint32_t>(C::kSlot)
                             : kind == 2 ? 256u
                             : kind == 3 ? static_cast<uint32_t>(TN * 4)
                             : kind < 6  ? 128u
                                         : static_cast<uint32_t>(kRImg);
      uint64_t* bar = (kind < 2 || kind >= 6) ? &ctl.full[ub] : &ctl.sc_full[sc];
      const bool issue = mine && (kind < 4 || e >= 0);
      int wait_ok = 1;
      if (lane == 0) {
        // The ring's slots are released in unit order (one MMA thread commits
        // them), so the slots are free once the unit that last held the
        // unit's last slot is done.
        const int prev = base + nsl - 1 - NSL;
        if (prev >= 0) {
          int o = i - 1;
          while (o > 0 && ubase[o] > prev) --o;
          wait_ok = mbar_wait(&ctl.done[o % NU], (o / NU) & 1, abort_flag, tmo, p.err);
        }
        if (wait_ok && i >= NSC) wait_ok = mbar_wait(&ctl.sc_empty[sc], ((i / NSC) & 1) ^ 1, abort_flag, tmo, p.err);
      }
      ok = __shfl_sync(0xFFFFFFFFu, wait_ok, 0);
      if (!ok) break;
      if (lane == 0) {  // one thread writes what the consumers read after its arrivals
#pragma unroll
        for (int g2 = 0; g2 < UG; ++g2)
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) ctl.blk[ub][g2][h2] = ctl.sblk[sc][g2][h2] = e4[g2][h2];
        ctl.ng[ub] = ctl.sng[sc] = ng;
        mbar_arrive_expect_tx(&ctl.full[ub], ng * 2 * C::kSlot + nblk * kRImg);
        mbar_arrive_expect_tx(&ctl.sc_full[sc], ng * (256 + TN * 4) + nsr * 128);
      }
      __syncwarp();
      if (issue) bulk_g2s(dst, src, bytes, bar);
      __syncwarp();
    }
    // Every copy issued here is waited on by a consumer before the CTA ends;
    // after an abort, the end of the kernel gives copies in flight time to land.
  } else if (warp == kWarpMma) {
    // residual map of this CTA's units, from the block-list rows of its tiles
    for (int i = lane; i < nunits; i += 32)
#pragma unroll
      for (int gq = 0; gq < UG; ++gq) res_map[gq][0][i] = res_map[gq][1][i] = -1;
    __syncwarp();
    if (p.nnzb > 0 && nunits > 0) {
      for (int64_t tile = unit_tile(u0); tile <= unit_tile(u1 - 1); ++tile) {
        const int t = tile_t(tile);
        for (int half = 0; half < 2; ++half) {
          const int br = 2 * t + half;
          // entries are clamped to [0, nnzb): a malformed list cannot index out of bounds
          const int e0 = max(0, min(p.nnzb, p.row_ptr[br]));
          const int e1 = max(e0, min(p.nnzb, p.row_ptr[br + 1]));
          for (int e = e0 + lane; e < e1; e += 32) {
            const int g = p.col_idx[e];
            const int64_t lu = tile * UPT + g / UG - u0;
            if (g >= 0 && g < G && lu >= 0 && lu < nunits) res_map[g % UG][half][lu] = e;
          }
        }
      }
    }
    __syncwarp();
    {  // each unit's first slot: 2 slots per group and 1 per group with residual blocks, summed in
       // unit order (lane l scans a contiguous chunk of units)
      const int chunk = (nunits + 31) / 32;
      const int l0 = min(nunits, lane * chunk), l1 = min(nunits, l0 + chunk);
      auto nsl = [&](int lu) {
        const int j = static_cast<int>((u0 + lu) % UPT);
        const int ng = min(UG, G - UG * j);
        int n = 2 * ng;
#pragma unroll
        for (int gq = 0; gq < UG; ++gq) n += (res_map[gq][0][lu] >= 0 || res_map[gq][1][lu] >= 0);
        return n;
      };
      int cnt = 0;
      for (int lu = l0; lu < l1; ++lu) cnt += nsl(lu);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      int pos = incl - cnt;
      for (int lu = l0; lu < l1; ++lu) {
        ubase[lu] = pos;
        pos += nsl(lu);
      }
      if (lane == 31) ubase[nunits] = incl;
    }
    __syncwarp();
    mbar_arrive(&ctl.map_ready);
    if (lane == 0) {
      int item = 0;
      bool ok = true;
      for (int i = 0; i < nunits && ok; ++i) {
        const int ub = i % NU;
        if (!mbar_wait(&ctl.full[ub], (i / NU) & 1, abort_flag, tmo, p.err)) break;
        const int ng = ctl.ng[ub];
        bool hr[UG];
#pragma unroll
        for (int gq = 0; gq < UG; ++gq) hr[gq] = gq < ng && (ctl.blk[ub][gq][0] >= 0 || ctl.blk[ub][gq][1] >= 0);
        const bool any_r = hr[0] || hr[1];
        const int base = ubase[i];
        for (int k = 0; k < 1 + any_r; ++k, ++item) {
          const int d = item % ND;
          if (!mbar_wait(&ctl.d_empty[d], ((item / ND) & 1) ^ 1, abort_flag, tmo, p.err)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int gq = 0; gq < UG; ++gq) {
            if (gq >= ng || (k == 1 && !hr[gq])) continue;
            const uint32_t b = smem_u32(slot(base + 2 * gq + 1));
            // the weight image, or the group's residual image (after the unit's weight and activation images)
            const uint32_t a = smem_u32(slot(k == 0 ? base + 2 * gq : base + 2 * ng + (gq && hr[0] ? 1 : 0)));
            const uint32_t d_col = tmem + d * C::kDCols + gq * TN;
#pragma unroll
            for (int j = 0; j < 4; ++j) img_mma(d_col, img_desc(a + 32 * j), img_desc(b + 32 * j), C::kIdesc, j > 0);
          }
          tc_commit(&ctl.d_full[d]);
        }
        if (ok) tc_commit(&ctl.done[ub]);  // the unit's slots are free once its MMAs complete
      }
      // the issued MMAs finish before TMEM can be released
      if (item > 0) {
        volatile int never = 0;
        const int last = item - 1;
        mbar_wait(&ctl.d_full[last % ND], (last / ND) & 1, &never, tmo, p.err);
      }
    }
  } else {
    // ---------------- drain + epilogue ----------------
    pdl_wait();  // Y and the workspace pieces may still be in use by the preceding kernel
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;              // weight row (TMEM lane)
    const int sub = (warp - kWarpDrain0) >> 2;      // token slice of the tile (kCols tokens)
    const int c0 = sub * C::kCols;                  // first token column of this thread
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int half = r >> 6;
    constexpr int NP = C::kCols / 2;  // token pairs per thread
    uint64_t acc[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) acc[j] = 0;
    int item = 0, nbar = 0;
    bool ok = true;
    auto drain_sync = [&]() -> bool {  // bounded barrier of the drain threads
      mbar_arrive(&ctl.drain_bar);
      const bool passed = mbar_wait(&ctl.drain_bar, nbar & 1, abort_flag, tmo, p.err);
      ++nbar;
      return passed;
    };
    auto store_tile = [&](int m0, int n) {
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        float v[2];
        u2(acc[j], v[0], v[1]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int m = m0 + c0 + 2 * j + h;
          if (m < p.M) {
            const int64_t off = static_cast<int64_t>(m) * p.ldy + n;
            if (p.y_f32)
              static_cast<float*>(p.y)[off] = v[h];
            else
              static_cast<__nv_bfloat16*>(p.y)[off] = __float2bfloat16_rn(v[h]);
          }
        }
      }
    };
    Pos q = pos0;
    for (int i = 0; i < nunits && ok; ++i, advance(q)) {
      const int64_t tile = q.tile;
      const int g0 = UG * q.j;
      const int n = q.t * kTileN + r, m0 = q.mt * TN;
      const int sc = i % NSC;
      if (!mbar_wait(&ctl.sc_full[sc], (i / NSC) & 1, abort_flag, tmo, p.err)) { ok = false; break; }
      const uint8_t* scb = scring + sc * C::kScBytes;
      const int ng = ctl.sng[sc];
      int e_mine[UG];
      bool any_r = false;
#pragma unroll
      for (int gq = 0; gq < UG; ++gq) {
        e_mine[gq] = gq < ng ? ctl.sblk[sc][gq][half] : -1;
        any_r = any_r || (gq < ng && (ctl.sblk[sc][gq][0] >= 0 || ctl.sblk[sc][gq][1] >= 0));
      }
      for (int k = 0; k < 1 + any_r; ++k, ++item) {
        const int d = item % ND;
        if (!mbar_wait(&ctl.d_full[d], (item / ND) & 1, abort_flag, tmo, p.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int gq = 0; gq < UG; ++gq) {
          const bool active = gq < ng && (k == 0 || e_mine[gq] >= 0);  // warp-uniform: a warp's rows sit in one half
          const uint8_t* scg = scb + gq * C::kScGroup;
          if constexpr (kDebug) {
#pragma unroll
           for (int dc = 0; dc < C::kCols / 32; ++dc) {
            uint32_t dv[32];
            if (active) {
              tmem_ld32(tmem + lane_base + d * C::kDCols + gq * TN + c0 + 32 * dc, dv);
              tc_wait_ld();
            }
            if (gq == UG - 1 && dc == C::kCols / 32 - 1) {  // every dot of the item this warp reads is in registers
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&ctl.d_empty[d]);
            }
            if (!active) continue;
            const int g = g0 + gq;
#pragma unroll
            for (int q2 = 0; q2 < 32; ++q2) {
              const int m = m0 + c0 + 32 * dc + q2;
              if (m < p.M) {
                const int32_t v = static_cast<int32_t>(__uint_as_float(dv[q2]));
                if (k == 0)
                  p.dots_w[(static_cast<int64_t>(m) * p.N + n) * G + g] = v;
                else
                  p.dots_r[(static_cast<int64_t>(m) * p.nnzb + e_mine[gq]) * 64 + (r & 63)] = v;
              }
            }
           }
          } else {
            // 32 columns at a time (with 18 warps' 96 registers a thread, 16 at a time measured faster;
            // with 11 warps and 168, 32)
            const uint32_t sxa = smem_u32(scg + C::sSX) + c0 * 4;
            uint64_t s2 = 0;
            if (active) {
              const uint16_t sbits = k == 0 ? reinterpret_cast<const uint16_t*>(scg + C::sWS)[r]
                                            : reinterpret_cast<const uint16_t*>(scg + C::sRS)[half * 64 + (r & 63)];
              const float s = __half2float(__ushort_as_half(sbits));
              s2 = p2(s, s);
            }
#pragma unroll
            for (int hx = 0; hx < C::kCols / 32; ++hx) {
              uint32_t dv[32];
              if (active) {
                tmem_ld32(tmem + lane_base + d * C::kDCols + gq * TN + c0 + 32 * hx, dv);
                tc_wait_ld();
              }
              if (gq == UG - 1 && hx == C::kCols / 32 - 1) {  // every dot of the item this warp reads is in registers
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl.d_empty[d]);
              }
              if (!active) continue;
#pragma unroll
              for (int j2 = 0; j2 < 8; ++j2) {
                uint64_t sx0, sx1;  // activation scales of token pairs 16 hx + 2 j2, + 1 of this thread's columns
                asm volatile("ld.shared.v2.u64 {%0, %1}, [%2];" : "=l"(sx0), "=l"(sx1) : "r"(sxa + 128 * hx + 16 * j2));
                const uint64_t t0 = mul2(p2(__uint_as_float(dv[4 * j2]), __uint_as_float(dv[4 * j2 + 1])), s2);
                const uint64_t t1 = mul2(p2(__uint_as_float(dv[4 * j2 + 2]), __uint_as_float(dv[4 * j2 + 3])), s2);
                acc[16 * hx + 2 * j2] = fma2(sx0, t0, acc[16 * hx + 2 * j2]);
                acc[16 * hx + 2 * j2 + 1] = fma2(sx1, t1, acc[16 * hx + 2 * j2 + 1]);
              }
            }
          }
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.sc_empty[sc]);  // scales read: the slot may be refilled
      // ---- tile end: store Y, or hand a stream-K piece to the workspace ----
      if (!kDebug && (q.j == UPT - 1 || i == nunits - 1)) {
        const int64_t tu0 = tile * UPT, tu1 = tu0 + UPT;  // the tile's units
        if (tu0 >= u0 && tu1 <= u1) {
          store_tile(m0, n);
        } else {
          // A piece: written by every drain thread, counted in by one; the CTA
          // that brings the count to the number of pieces finishes the tile
          // after its own range (no stall here).
          const int slot = (tile == pos0.tile) ? 0 : 1;
          uint4* part = reinterpret_cast<uint4*>(p.partials + ((c * 2 + slot) * kTileN + r) * TN + c0);
#pragma unroll
          for (int q4 = 0; q4 < NP / 2; ++q4)
            part[q4] = make_uint4(static_cast<uint32_t>(acc[2 * q4]), static_cast<uint32_t>(acc[2 * q4] >> 32),
                                  static_cast<uint32_t>(acc[2 * q4 + 1]), static_cast<uint32_t>(acc[2 * q4 + 1] >> 32));
          __threadfence();
          if (!drain_sync()) { ok = false; break; }
          if (warp == kWarpDrain0 && lane == 0) {
            const int64_t cf = owner(tu0), cl = owner(tu1 - 1);
            const int old = atomicAdd(&p.counters[cf], 1);  // CTA cf starts at most one cut tile
            if (old == static_cast<int>(cl - cf)) ctl.deferred[ctl.ndeferred++] = tile;
          }
        }
#pragma unroll
        for (int j = 0; j < NP; ++j) acc[j] = 0;
      }
    }
    // ---- finish the tiles this CTA completed last: bulk-copy every piece
    // into the (now idle) stage memory, sum in CTA order, store Y ----
    if (!kDebug && ok && drain_sync()) {
      const int nd = ctl.ndeferred;
      constexpr uint32_t kPieceBytes = TN * kTileN * 4;
      constexpr int kPerRound = C::kRingBytes / kPieceBytes;
      static_assert(kPerRound >= 1, "a piece fits the stage ring");
      int nred = 0;
      for (int di = 0; di < nd && ok; ++di) {
        const int64_t tile = ctl.deferred[di];
        const int64_t tu0 = tile * UPT, tu1 = tu0 + UPT;
        const int64_t cf = owner(tu0), cl = owner(tu1 - 1);
        const int m0 = tile_mt(tile) * TN, n = tile_t(tile) * kTileN + r;
#pragma unroll
        for (int j = 0; j < NP; ++j) acc[j] = 0;
        for (int64_t cb = cf; cb <= cl && ok; cb += kPerRound) {
          const int npieces = static_cast<int>(min(static_cast<int64_t>(kPerRound), cl - cb + 1));
          if (warp == kWarpDrain0 && lane == 0) {
            __threadfence();
            fence_proxy_async_global();  // other CTAs' generic writes -> this bulk (async) read
            mbar_arrive_expect_tx(&ctl.red_bar, npieces * kPieceBytes);
            for (int q = 0; q < npieces; ++q) {
              const int64_t c2 = cb + q;
              const int slot2 = (tile == unit_tile(c2 * U / P)) ? 0 : 1;
              bulk_g2s(smem + q * kPieceBytes, p.partials + (c2 * 2 + slot2) * (kTileN * TN), kPieceBytes,
                       &ctl.red_bar);
            }
          }
          if (!mbar_wait(&ctl.red_bar, nred & 1, abort_flag, tmo, p.err)) { ok = false; break; }
          ++nred;
          for (int q = 0; q < npieces; ++q) {
            const uint64_t* piece = reinterpret_cast<const uint64_t*>(smem + q * kPieceBytes) + (r * TN + c0) / 2;
#pragma unroll
            for (int j = 0; j < NP; ++j) {
              float a0, a1, b0, b1;
              u2(acc[j], a0, a1);
              u2(piece[j], b0, b1);
              acc[j] = p2(a0 + b0, a1 + b1);  // ascending CTA order, one rounding per add
            }
          }
          if (!drain_sync()) { ok = false; break; }  // stage memory free for the next round
        }
        if (!ok) break;
        store_tile(m0, n);
        if (warp == kWarpDrain0 && lane == 0) p.counters[cf] = 0;  // ready for the next launch
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*abort_flag) {
    // A wait gave up: bulk copies or MMAs may still be in flight into this
    // CTA's shared or tensor memory; give them 200 us (bounded) to land.
    if (threadIdx.x == 0) {
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 200000ull) {
      }
    }
    __syncthreads();
  }
  if (warp == kWarpMma) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

size_t a1k(size_t b) { return (b + 1023) / 1024 * 1024; }

struct IPlan {
  int tn, tiles_m, tiles_n, G, Mt;
  int64_t units;
  int ctas;
  size_t off_part, off_w, off_r, off_x, off_s, bytes;
};

int img_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

// "image" forces the image form for every M the general kernel takes, "conv"
// turns it off; otherwise it serves M >= kImgMinTokens.
int image_form_mode() {
  const char* v = std::getenv("MQ_GENERAL_FORM");
  if (v && std::strcmp(v, "image") == 0) return 1;
  if (v && std::strcmp(v, "conv") == 0) return -1;
  return 0;
}

// 128-token tiles: at 256 the drain's accumulators (64 registers a thread)
// do not fit the 96 registers 18 warps leave a thread.
int pick_img_tn(int64_t) { return 128; }

// The plan depends on (M, N, K, nnzb) and the current device's SM count (the
// persistent grid and its stream-K pieces; 152 when no device is current).
IPlan iplan(int64_t M, int64_t N, int64_t K, int64_t nnzb) {
  IPlan pl;
  pl.tn = pick_img_tn(M);
  pl.tiles_m = static_cast<int>((M + pl.tn - 1) / pl.tn);
  pl.tiles_n = static_cast<int>(N / kTileN);
  pl.G = static_cast<int>(K / kGroup);
  pl.Mt = pl.tiles_m * pl.tn;
  pl.units = static_cast<int64_t>(pl.tiles_m) * pl.tiles_n * ((pl.G + 1) / 2);  // units of two groups
  const int sms = img_sms();
  int64_t ctas = std::min<int64_t>(sms > 0 ? sms : kImgPlanCtasNoDevice,
                                   std::max<int64_t>(1, pl.units / kImgMinUnitsPerCta));
  const int64_t min_ctas = (pl.units + kImgMaxUnitsPerCta - 1) / kImgMaxUnitsPerCta;
  if (ctas < min_ctas) ctas = min_ctas;
  pl.ctas = static_cast<int>(ctas);
  pl.off_part = kWsZeroBytes;
  pl.off_w = pl.off_part + a1k(static_cast<size_t>(pl.ctas) * 2 * kTileN * pl.tn * sizeof(float));
  pl.off_r = pl.off_w + a1k(static_cast<size_t>(pl.tiles_n) * pl.G * kWImg);
  pl.off_x = pl.off_r + a1k(static_cast<size_t>(nnzb) * kRImg);
  pl.off_s = pl.off_x + a1k(static_cast<size_t>(pl.G) * pl.Mt * 128);
  pl.bytes = pl.off_s + a1k(static_cast<size_t>(pl.G) * pl.Mt * sizeof(float));
  return pl;
}

template <int TN, bool kDebug>
mq_status launch_img(const ImgParams& ip, const IPlan& pl, cudaStream_t stream) {
  using C = ICfg<TN>;
  auto kern = image_gemm_kernel<TN, kDebug>;
  static std::mutex mu;
  static bool attr_set[kImgMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kImgMaxDevices) return launch_status("image gemm: device");
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
        return launch_status("image gemm: smem attribute");
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
  if (cudaLaunchKernelEx(&cfg, kern, ip) != cudaSuccess) return launch_status("image gemm launch");
  return launch_status("image gemm");
}

}  // namespace

// Whether the image form serves (M, N, K) when its full workspace is given.
bool image_form_wanted(int64_t M) {
  const int mode = image_form_mode();
  if (mode < 0) return false;
  return mode > 0 || M >= kImgMinTokens;
}

// Workspace of the image form for (M, N, K) with the densest residual (every
// block), so that the size does not depend on the block list.
size_t image_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  return iplan(M, N, K, (N / kBlockRows) * (K / kGroup)).bytes;
}

// Tokens per tile and CTAs of the image form for (M, N, K).
void image_plan_info(int64_t M, int64_t N, int64_t K, int32_t* tn, int32_t* ctas) {
  const IPlan pl = iplan(M, N, K, 0);
  *tn = pl.tn;
  *ctas = pl.ctas;
}

// The pre-pass and the GEMM, when the image form is wanted for M and the
// workspace holds its images (`handled` false otherwise: the caller runs the
// general kernel).
mq_status image_gemm_launch(bool* handled, const uint8_t* xq, const uint16_t* xs, int64_t M, const uint8_t* wpk,
                            int64_t N, int64_t K, const int32_t* row_ptr, const int32_t* col_idx, int64_t nnzb,
                            const uint8_t* rpk, void* y, int64_t ldy, mq_dtype yt, int32_t* dots_w, int32_t* dots_r,
                            void* ws, size_t ws_bytes, cudaStream_t stream) {
  *handled = false;
  if (!image_form_wanted(M)) return MQ_OK;
  const IPlan pl = iplan(M, N, K, nnzb);
  if (ws == nullptr || ws_bytes < pl.bytes || !aligned(ws, 256)) return MQ_OK;
  if (pl.ctas > kWsZeroBytes / 4) return MQ_OK;
  *handled = true;
  uint8_t* base = static_cast<uint8_t*>(ws);
  const int Mp = static_cast<int>((M + 7) / 8 * 8);
  PrepParams pp;
  pp.wpk = wpk;
  pp.rpk = rpk;
  pp.xq = xq;
  pp.xs = xs;
  pp.wimg = base + pl.off_w;
  pp.rimg = base + pl.off_r;
  pp.ximg = base + pl.off_x;
  pp.sxf = reinterpret_cast<float*>(base + pl.off_s);
  pp.M = static_cast<int>(M);
  pp.Mp = Mp;
  pp.Mt = pl.Mt;
  pp.G = pl.G;
  pp.n_w = static_cast<int64_t>(pl.tiles_n) * pl.G;  // weight images
  pp.n_r = nnzb;                                      // residual images
  pp.n_x = static_cast<int64_t>(pl.G) * pl.Mt / 128;  // activation images of 128 token rows
  pp.n_s = static_cast<int64_t>(pl.G) * pl.Mt;
  {
    const int64_t images = pp.n_w + pp.n_r + pp.n_x;
    const int sms = img_sms();
    // one block per image, at most one wave (8 blocks of 256 threads per SM)
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(images, (sms > 0 ? sms : 152) * 8));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, image_prep_kernel, pp) != cudaSuccess) return launch_status("image prep launch");
  }
  ImgParams ip;
  ip.wimg = pp.wimg;
  ip.rimg = pp.rimg;
  ip.ximg = pp.ximg;
  ip.sxf = pp.sxf;
  ip.wpk = wpk;
  ip.rpk = rpk;
  ip.row_ptr = row_ptr;
  ip.col_idx = col_idx;
  ip.y = y;
  ip.y_f32 = yt == MQ_F32;
  ip.ldy = ldy;
  ip.dots_w = dots_w;
  ip.dots_r = dots_r;
  ip.partials = reinterpret_cast<float*>(base + pl.off_part);
  ip.counters = reinterpret_cast<int32_t*>(base);
  ip.M = static_cast<int>(M);
  ip.Mt = pl.Mt;
  ip.N = static_cast<int>(N);
  ip.G = pl.G;
  ip.tiles_n = pl.tiles_n;
  ip.tiles_m = pl.tiles_m;
  ip.nnzb = static_cast<int>(nnzb);
  ip.units = pl.units;
  ip.ctas = pl.ctas;
  ip.timeout_ns = wait_timeout_ns();
  ip.err = device_error_word();
  if (!ip.err) return set_error(MQ_ERR_CUDA, "image gemm: device error word unavailable");
  const bool dbg = dots_w != nullptr;
  return dbg ? launch_img<128, true>(ip, pl, stream) : launch_img<128, false>(ip, pl, stream);
}

}  // namespace mq
