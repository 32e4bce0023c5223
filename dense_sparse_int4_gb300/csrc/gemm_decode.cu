// The fused W4A4 + block-sparse 4-bit residual GEMM for decode batches (at
// most 32 tokens): the ZipperEngine of the MosaicQuant summary (Metodologia 3)
// laid out for sm_103a.  It computes
//
//   Y[m,n] = sum_g sx[m,g] * ( sw[n,g] * Dw[m,n,g] + sr[n,g] * Dr[m,n,g] )
//
// in one kernel: the residual product of a selected 64x128 block runs on the
// same activation tile as the dense product of its group, and both are
// reduce-added into the same fp32 accumulators.
//
// At decode sizes the work is streaming the 4-bit weights; the tensor cores
// have room to spare, but each 128x128 group needs four K=32 MMAs and 16384
// codes converted to E4M3, and both must keep up with HBM.  The design:
//   * Split-K over a thread-block cluster of CS CTAs.  A cluster owns whole
//     128-row weight tiles (one after another, persistently); CTA rank j
//     handles the same K slice [j*G/CS, (j+1)*G/CS) of every tile it visits,
//     so its activations are loaded and converted to E4M3 tensor-core tiles
//     once, at the start, and stay in shared memory.
//   * One bulk copy per stage: a stage is two consecutive base-weight records
//     of one tile (codes and scales side by side, 16.5 KiB); residual blocks
//     come as one record each into a small ring, only where the block list
//     has them.  The block list (CSR by 64-row block row) of every tile the
//     CTA visits is read once, up front, into a static map.
//   * Four converter warpgroups take the stages round-robin and convert each
//     group's codes in registers straight into their own double-buffered
//     tensor-memory A operand.  The weight codes are looked up as q + 8 (a
//     cheaper 16-entry table); the dot then exceeds the true one by exactly
//     8 * sum_k qx[m,k], which the drain subtracts (the group sums of the
//     resident activations are computed once).  All dots stay exact integers.
//   * One MMA warp serves the four warpgroups in whatever order their items
//     become ready, issuing each item's four MMAs back to back, so the
//     converters never wait on MMA issue.  Each warpgroup drains its own
//     results: acc[m] += sx[m] * (s * D[m]) in fp32.
//   * At the end of a tile the four warpgroup partials are added in a fixed
//     order into a row-major shared-memory buffer; each CTA then pushes the
//     rows owned by rank k into rank k's shared memory with one bulk copy
//     (distributed shared memory, counted on the owner's barrier), and each
//     rank sums its 128/CS rows over the CS partials in rank order and stores
//     Y.  No global workspace, no atomics: the result is deterministic.
// Every wait is bounded (mbar_wait): a wait that runs out records the error,
// raises the CTA's abort flag, and every role winds down.
#include "mq_internal.cuh"

#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

// Timeline probes for profiling builds (compiled out unless MQ_DEC_TRACE is
// defined, in which case the build supplies the two functions).
#ifdef MQ_DEC_TRACE
__device__ void mq_dec_trace_stamp(int slot);
__device__ void mq_dec_trace_prof(int w, const long long* acc, int n);
#define MQ_DTRACE(slot) mq_dec_trace_stamp(slot)
#define MQ_PT() (pt_ = clock64())
#define MQ_PA(k) (prof_[k] += clock64() - pt_)
#else
#define MQ_DTRACE(slot) ((void)0)
#define MQ_PT() ((void)0)
#define MQ_PA(k) ((void)0)
#endif

namespace mq {
namespace {

constexpr int kWG = 4;                  // converter warpgroups (warps 0..15)
constexpr int kWorkers = 32 * 16;
constexpr int kWarpMma = 16;           // MMA issue (kMmaWarps warps, each serving kWG / kMmaWarps warpgroups)
constexpr int kMmaWarps = 1;
constexpr int kWarpProducer = kWarpMma + kMmaWarps;
constexpr int kWarpEpi0 = kWarpProducer + 1;  // epilogue warps
// 20 warps: 5 per SM sub-partition, so each thread can have 96 registers
constexpr int kThreads = 32 * 20;
constexpr int kEpiThreads = kThreads - 32 * kWarpEpi0;
constexpr int kUG = 2;                  // groups per stage
constexpr int kStageBytes = kUG * kWRecBytes;
constexpr int kMaxStages = 16;
constexpr int kRSlots = 6;              // residual-record ring
constexpr int kMaxVisits = 16;          // tiles visited per CTA
constexpr int kMaxSlice = 32;           // groups in a CTA's K slice
constexpr int kMaxBBytes = 64 * 1024;   // resident activation tiles
constexpr int kSmemLimit = 227 * 1024;
constexpr int kTmemCols = 512;          // per warpgroup 128: A0, A1 (32 each), D0, D1 (TN each)
constexpr int kMaxCS = 8;

struct DecParams {
  const uint8_t* xq;   // [G][Mp][64]
  const uint16_t* xs;  // [G][Mp]
  const uint8_t* wpk;
  const int32_t* row_ptr;
  const int32_t* col_idx;
  const uint8_t* rpk;
  void* y;
  int y_f32;
  int32_t* dots_w;      // test hook: raw group dots instead of Y
  int32_t* dots_r;
  int M, Mp, N, G, nnzb, tiles;
  int cs, nclusters, nstages;
  uint32_t oSX, oRB, oRX, oR, oStage;  // shared-memory offsets; the activation tiles are at 0
  uint64_t timeout_ns;
  uint32_t* err;
};

struct __align__(8) DecCtl {
  uint64_t full[kMaxStages];     // producer arrival + record bytes
  uint64_t empty[kMaxStages];    // the 4 warps of the warpgroup that converted the stage
  uint64_t r_full[kRSlots];
  uint64_t r_empty[kRSlots];
  uint64_t a_ready[kWG][2];      // A buffer b of warpgroup w holds a converted item (4 warp arrivals)
  uint64_t d_ready[kWG][2];      // its MMAs are complete (tcgen05.commit)
  uint64_t work_bar;             // activation tiles converted (16 warp arrivals)
  uint64_t epi_bar;              // bounded barrier of the epilogue warps (one arrival each)
  uint64_t map_ready;            // residual map and ring positions are built
  uint64_t chain[kWG];           // warpgroup w may add its partial of the tile (w >= 1)
  uint64_t rb_done;              // the CTA's partial of the tile is complete
  uint64_t rx_full;              // every rank's rows for this CTA have landed (bytes)
  uint64_t rx_free;              // every owner has consumed this CTA's last push
  int32_t item_gl[kWG][2];       // slice group of the item in A buffer b (-1: warpgroup finished)
  int32_t map[kMaxVisits][kMaxSlice][2];   // CSR entry of the slice's residual blocks per tile, or -1
  int32_t rpos[kMaxVisits][kMaxSlice][2];  // position of that block in the residual-ring order
  int32_t sc_off[kMaxVisits + 1], sc_a0[kMaxVisits], sc_a1[kMaxVisits];
  uint32_t tmem_base;
  int abort_flag;
};

// --- cluster / misc PTX -------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster, together.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t mapa(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void remote_arrive(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Bulk copy of this CTA's shared memory into a cluster peer's; completion is
// counted in bytes on the peer's mbarrier.
__device__ __forceinline__ void bulk_s2peer(uint32_t dst_cluster, const void* src, uint32_t bytes,
                                            uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(smem_u32(src)), "r"(bytes), "r"(bar_cluster)
      : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait with cluster-scope acquire (for phases completed by other CTAs).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                  uint64_t timeout_ns, uint32_t* err_word) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > timeout_ns) {
      atomicOr(err_word, kDevErrTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint4 ld_global_16(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
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

// Eight INT4 codes q (two's complement nibbles, element i in bits 4i..4i+3)
// -> eight E4M3 bytes holding q + 8 exactly.  The nibble u = q + 8 is p ^ 8;
// two 8-entry prmt tables cover u in [0, 8) and [8, 16): a selector nibble
// with its top bit set makes prmt emit the sign of the table byte, 0 here
// (all entries are positive), so each table contributes only its own half
// and an OR merges them.  9 operations per 8 codes.
__device__ __forceinline__ void uint4x8_to_e4m3(uint32_t p, uint32_t& lo, uint32_t& hi) {
  constexpr uint32_t kLoA = 0x44403800u, kLoB = 0x4E4C4A48u;  // 0, 1, 2, 3 | 4, 5, 6, 7
  constexpr uint32_t kHiA = 0x53525150u, kHiB = 0x57565554u;  // 8, 9, 10, 11 | 12, 13, 14, 15
  const uint32_t u = p ^ 0x88888888u;
  lo = prmt(kLoA, kLoB, u) | prmt(kHiA, kHiB, p);
  hi = prmt(kLoA, kLoB, u >> 16) | prmt(kHiA, kHiB, p >> 16);
}

// Store 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// 64 bytes of one row's weight codes (4 K-steps of 16 bytes at src + j*jstride)
// -> E4M3 (q + 8) in this thread's TMEM lane, 32 columns in one store.
__device__ __forceinline__ void row_codes_to_tmem(const uint8_t* src, int jstride, uint32_t a_col) {
  uint4 pk[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) pk[j] = *reinterpret_cast<const uint4*>(src + j * jstride);
  uint32_t ev[32];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4x8_to_e4m3(pk[j].x, ev[8 * j + 0], ev[8 * j + 1]);
    uint4x8_to_e4m3(pk[j].y, ev[8 * j + 2], ev[8 * j + 3]);
    uint4x8_to_e4m3(pk[j].z, ev[8 * j + 4], ev[8 * j + 5]);
    uint4x8_to_e4m3(pk[j].w, ev[8 * j + 6], ev[8 * j + 7]);
  }
  tmem_st32(a_col, ev);
}

// Sum of the eight signed codes of a word of packed activations.
__device__ __forceinline__ int nibble_sum8(uint32_t p) {
  const uint32_t u = p ^ 0x88888888u;  // q + 8 in [1, 15]
  const uint32_t b = (u & 0x0F0F0F0Fu) + ((u >> 4) & 0x0F0F0F0Fu);
  return static_cast<int>((b * 0x01010101u) >> 24) - 64;
}

// One item of a converter warpgroup: a group's dense product (kind 0) or its
// residual product (kind 1).
struct Item {
  int i, q, kind;  // stage, group within the stage, kind
};

template <int TN, bool kDebug>
__global__ void __launch_bounds__(kThreads, 1) w4a4_decode_kernel(const DecParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ DecCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* btiles = smem;                                  // [ns][TN rows][128 B] E4M3, 128B-swizzled K-major
  float* sxs = reinterpret_cast<float*>(smem + p.oSX);     // [ns][TN] activation scales
  float* sums = sxs + kMaxSlice * TN;                      // [ns][TN] 8 * (sum of the group's activation codes)
  float* rb = reinterpret_cast<float*>(smem + p.oRB);      // [128 rows][TN] the CTA's partial of a tile
  float* rx = reinterpret_cast<float*>(smem + p.oRX);      // [CS sources][R rows][TN] the rows this CTA owns
  uint8_t* rring = smem + p.oR;                            // [kRSlots] residual records
  uint8_t* stages = smem + p.oStage;                       // [nstages] x two base records
  if (threadIdx.x == 0) MQ_DTRACE(0);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int CS = p.cs, NS = p.nstages, G = p.G;
  const int R = kTileN / CS;  // rows of a tile each rank finishes
  const int rank = static_cast<int>(cluster_rank());
  const int cid = static_cast<int>(cluster_index());
  const int gs = rank * G / CS, ge = (rank + 1) * G / CS, ns = ge - gs;  // this CTA's K slice
  const int spv = (ns + kUG - 1) / kUG;                                   // stages per visited tile
  const int nvis = (p.tiles - cid + p.nclusters - 1) / p.nclusters;       // tiles cid, cid + nclusters, ...
  const int total = nvis * spv;
  volatile int* abort_flag = &ctl.abort_flag;
  const uint64_t tmo = p.timeout_ns;
  auto tile_of = [&](int v) { return static_cast<int64_t>(cid) + static_cast<int64_t>(v) * p.nclusters; };
  auto stage_ng = [&](int i) { return min(kUG, ns - (i % spv) * kUG); };
  auto stage_rec = [&](int i) {  // first record of stage i
    return p.wpk + (tile_of(i / spv) * G + gs + (i % spv) * kUG) * kWRecBytes;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], 4);
    }
    for (int s = 0; s < kRSlots; ++s) {
      mbar_init(&ctl.r_full[s], 1);
      mbar_init(&ctl.r_empty[s], 4);
    }
    for (int w = 0; w < kWG; ++w) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&ctl.a_ready[w][b], 4);
        mbar_init(&ctl.d_ready[w][b], 1);
      }
      mbar_init(&ctl.chain[w], 4);
    }
    mbar_init(&ctl.work_bar, 16);
    mbar_init(&ctl.epi_bar, kEpiThreads / 32);
    mbar_init(&ctl.map_ready, 1);
    mbar_init(&ctl.rb_done, 4);
    mbar_init(&ctl.rx_full, 1);
    mbar_init(&ctl.rx_free, CS);
    ctl.abort_flag = 0;
    fence_mbar_init();
  }
  // The next kernel may start launching: everything it reads before its own
  // dependency wait is read-only here.
  pdl_trigger();
  // Every CTA of the cluster has its barriers initialised before any peer
  // pushes into them (also a barrier of this CTA's threads).
  cluster_sync_all();
  if (threadIdx.x == 0) MQ_DTRACE(1);

  if (warp == kWarpProducer) {
    // ---------------- producer: block list, then stages in order ----------------
    const int pre = min(NS, total);
    if (lane < pre) prefetch_l2(stage_rec(lane), stage_ng(lane) * kWRecBytes);  // no dependency: L2 only
    // Everything below may read buffers the preceding kernel wrote (weights
    // packed just before, the block list): wait for it.
    pdl_wait();
    if (lane == 0) MQ_DTRACE(2);
    if (lane < pre) {  // the first stages: weights in flight before the block list is read
      mbar_arrive_expect_tx(&ctl.full[lane], stage_ng(lane) * kWRecBytes);
      bulk_g2s(stages + lane * kStageBytes, stage_rec(lane), stage_ng(lane) * kWRecBytes, &ctl.full[lane]);
    }
    // Block list of every visited tile, restricted to this slice: lane v reads
    // the row pointers of tile v's two block rows, then all lanes read the
    // entries of all tiles at once.
    for (int idx = lane; idx < nvis * kMaxSlice * 2; idx += 32) (&ctl.map[0][0][0])[idx] = -1;
    if (p.nnzb > 0) {
      int a0 = 0, a1 = 0, a2 = 0;
      if (lane < nvis) {
        const int64_t br = 2 * tile_of(lane);
        a0 = max(0, min(p.nnzb, p.row_ptr[br]));
        a1 = max(a0, min(p.nnzb, p.row_ptr[br + 1]));
        a2 = max(a1, min(p.nnzb, p.row_ptr[br + 2]));
      }
      const int cnt = a2 - a0;
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane < nvis) {
        ctl.sc_off[lane] = incl - cnt;
        ctl.sc_a0[lane] = a0;
        ctl.sc_a1[lane] = a1;
      }
      const int nent = __shfl_sync(0xFFFFFFFFu, incl, 31);
      if (lane == 0) ctl.sc_off[nvis] = nent;
      __syncwarp();
      for (int base = 0; base < nent; base += 128) {
        int ev[4], gv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {  // loads first, so four are in flight per lane
          const int t = base + u * 32 + lane;
          ev[u] = -1;
          gv[u] = -1;
          if (t < nent) {
            int v = 0;
            while (v + 1 < nvis && ctl.sc_off[v + 1] <= t) ++v;
            ev[u] = ctl.sc_a0[v] + (t - ctl.sc_off[v]);
            gv[u] = p.col_idx[ev[u]];
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = base + u * 32 + lane;
          if (t < nent) {
            int v = 0;
            while (v + 1 < nvis && ctl.sc_off[v + 1] <= t) ++v;
            const int g = gv[u];
            if (g >= gs && g < ge) ctl.map[v][g - gs][ev[u] >= ctl.sc_a1[v] ? 1 : 0] = ev[u];
          }
        }
      }
    }
    __syncwarp();
    // Ring positions: the residual blocks in (tile, group, half) order; lane l
    // counts a contiguous chunk of that order.
    {
      const int nf = nvis * ns * 2;
      const int chunk = (nf + 31) / 32, f0 = min(nf, lane * chunk), f1 = min(nf, f0 + chunk);
      int cnt = 0;
      for (int f = f0; f < f1; ++f) cnt += ctl.map[f / (2 * ns)][(f / 2) % ns][f & 1] >= 0;
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      int pos = incl - cnt;
      for (int f = f0; f < f1; ++f)
        if (ctl.map[f / (2 * ns)][(f / 2) % ns][f & 1] >= 0) ctl.rpos[f / (2 * ns)][(f / 2) % ns][f & 1] = pos++;
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&ctl.map_ready);
      MQ_DTRACE(3);
    }
    for (int i = 0; i < total; ++i) {
      const int st = i % NS;
      const int v = i / spv, g0l = (i % spv) * kUG, ng = stage_ng(i);
      // lanes 0..3: the residual records of the stage's groups, into the ring
      int rok = 1;
      if (lane < kUG * 2 && (lane >> 1) < ng) {
        const int e = ctl.map[v][g0l + (lane >> 1)][lane & 1];
        if (e >= 0) {
          const int c = ctl.rpos[v][g0l + (lane >> 1)][lane & 1], slot = c % kRSlots;
          if (c >= kRSlots) rok = mbar_wait(&ctl.r_empty[slot], ((c / kRSlots) & 1) ^ 1, abort_flag, tmo, p.err);
          if (rok) {
            mbar_arrive_expect_tx(&ctl.r_full[slot], kRRecBytes);
            bulk_g2s(rring + slot * kRRecBytes, p.rpk + static_cast<int64_t>(e) * kRRecBytes, kRRecBytes,
                     &ctl.r_full[slot]);
          }
        }
      }
      if (!__all_sync(0xFFFFFFFFu, rok)) break;
      if (i >= pre) {  // the base records of stage i, once its slot is free
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait(&ctl.empty[st], ((i / NS) & 1) ^ 1, abort_flag, tmo, p.err);
          if (ok) {
            mbar_arrive_expect_tx(&ctl.full[st], ng * kWRecBytes);
            bulk_g2s(stages + st * kStageBytes, stage_rec(i), ng * kWRecBytes, &ctl.full[st]);
          }
        }
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
      }
      if (lane == 0 && i < 8) MQ_DTRACE(4 + i);
    }
  } else if (warp >= kWarpMma && warp < kWarpMma + kMmaWarps) {
    // ---------------- MMA issue: serve whichever of its warpgroups has an item ready ----------------
    const int w0 = (warp - kWarpMma) * (kWG / kMmaWarps);
    constexpr uint32_t kIdesc =
        (1u << 4) | (static_cast<uint32_t>(TN >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
    const bool ok0 = mbar_wait(&ctl.work_bar, 0, abort_flag, tmo, p.err);  // activation tiles and TMEM ready
    tc_fence_after();
    if (lane == 0 && ok0) {
      const uint32_t tmem = ctl.tmem_base;
      const uint32_t bt = smem_u32(btiles);
      int n[kWG / kMmaWarps] = {};
      int alive = kWG / kMmaWarps;
      uint64_t t_idle = 0;
#ifdef MQ_DEC_TRACE
      long long prof_[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0}, pt_ = 0, tl_ = clock64();
#endif
      while (alive > 0) {
        bool progressed = false;
#pragma unroll
        for (int x = 0; x < kWG / kMmaWarps; ++x) {
          const int w = w0 + x;
          if (n[x] < 0) continue;
          const int b = n[x] & 1;
          if (!mbar_test(&ctl.a_ready[w][b], (n[x] >> 1) & 1)) continue;
          const int gl = ctl.item_gl[w][b];
          if (gl < 0) {  // the warpgroup has no more items
            n[x] = -1;
            --alive;
            continue;
          }
          MQ_PT();
          tc_fence_after();
          const uint32_t a_col = tmem + w * 128 + 32 * b, d_col = tmem + w * 128 + 64 + TN * b;
          const uint32_t b_addr = bt + gl * (TN * 128);
#pragma unroll
          for (int j = 0; j < 4; ++j) tc_mma_ts(d_col, a_col + 8 * j, sw128_desc(b_addr + 32 * j), kIdesc, j > 0);
          tc_commit(&ctl.d_ready[w][b]);
          MQ_PA(0);
          ++n[x];
          progressed = true;
        }
        if (progressed) {
          t_idle = 0;
        } else {
          if (*abort_flag) break;
          const uint64_t now = globaltimer();
          if (t_idle == 0) {
            t_idle = now;
          } else if (now - t_idle > tmo) {
            atomicOr(p.err, kDevErrTimeout);
            *abort_flag = 1;
            break;
          }
        }
      }
#ifdef MQ_DEC_TRACE
      prof_[1] = clock64() - tl_;  // the whole issue loop
      if (w0 == 0) mq_dec_trace_prof(4, prof_, 9);
#endif
    }
  } else if (warp < kWarpMma) {
    // ---------------- converters + drain ----------------
    const int w = warp >> 2, quarter = warp & 3;
    const int r = quarter * 32 + lane;  // weight row of the tile = TMEM lane
    const int half = r >> 6;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    if (warp == 0) tmem_alloc(&ctl.tmem_base, kTmemCols);

    // --- this slice's activations, once: packed codes -> E4M3 tiles, their
    // group sums, and the scales -> fp32
    pdl_wait();
    {
      const int tid = threadIdx.x;  // 0..511
      for (int idx = tid; idx < ns * TN; idx += kWorkers) {
        const int gl = idx / TN, m = idx % TN;
        uint8_t* row = btiles + gl * (TN * 128) + (m >> 3) * 1024 + (m & 7) * 128;
        int sum = 0;
        float sx = 0.0f;
        if (m < p.Mp) {
          const uint8_t* src = p.xq + (static_cast<int64_t>(gs + gl) * p.Mp + m) * 64;
          uint4 pk[4];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) pk[jj] = ld_global_16(src + jj * 16);
          sx = __half2float(__ushort_as_half(p.xs[static_cast<int64_t>(gs + gl) * p.Mp + m]));
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            uint4 lo, hi;
            int4x8_to_e4m3(pk[jj].x, lo.x, lo.y);
            int4x8_to_e4m3(pk[jj].y, lo.z, lo.w);
            int4x8_to_e4m3(pk[jj].z, hi.x, hi.y);
            int4x8_to_e4m3(pk[jj].w, hi.z, hi.w);
            sum += nibble_sum8(pk[jj].x) + nibble_sum8(pk[jj].y) + nibble_sum8(pk[jj].z) + nibble_sum8(pk[jj].w);
            // 16-byte chunk c of row m is stored at chunk c ^ (m & 7) of its 128-byte row
            *reinterpret_cast<uint4*>(row + (((2 * jj) ^ (m & 7)) * 16)) = lo;
            *reinterpret_cast<uint4*>(row + (((2 * jj + 1) ^ (m & 7)) * 16)) = hi;
          }
        } else {
#pragma unroll
          for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(row + c * 16) = make_uint4(0, 0, 0, 0);
        }
        sxs[gl * TN + m] = sx;
        sums[gl * TN + m] = 8.0f * static_cast<float>(sum);
      }
      fence_proxy_async_smem();  // generic writes -> the tensor core's reads
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.work_bar);
      ok = mbar_wait(&ctl.work_bar, 0, abort_flag, tmo, p.err);
      tc_fence_after();
      if (threadIdx.x == 0) MQ_DTRACE(12);
    }
    const uint32_t tmem = ctl.tmem_base;
    const uint32_t colA = tmem + w * 128, colD = tmem + w * 128 + 64;  // buffer b: +32b, +TN*b

    uint64_t acc[TN / 2];
#pragma unroll
    for (int k = 0; k < TN / 2; ++k) acc[k] = 0;
#ifdef MQ_DEC_TRACE
    long long prof_[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0}, pt_ = 0;
#endif

    bool map_seen = false;
    // Items of this warpgroup: its stages in order; in a stage, the dense
    // items of its groups, then the residual items of the groups that have a
    // block.  Returns 1 (next item in `it`), 0 (no more items), -1 (gave up).
    auto advance = [&](Item& it) -> int {
      const int ng = stage_ng(it.i);
      if (it.kind == 0 && it.q + 1 < ng) {
        ++it.q;
        return 1;
      }
      // residual items of this stage, after its dense items
      if (!map_seen) {
        if (!mbar_wait(&ctl.map_ready, 0, abort_flag, tmo, p.err)) return -1;
        map_seen = true;
      }
      const int v = it.i / spv, g0l = (it.i % spv) * kUG;
      for (int q = it.kind == 0 ? 0 : it.q + 1; q < ng; ++q)
        if (ctl.map[v][g0l + q][0] >= 0 || ctl.map[v][g0l + q][1] >= 0) {
          it.kind = 1;
          it.q = q;
          return 1;
        }
      it.kind = 0;
      it.q = 0;
      it.i += kWG;
      return it.i < total ? 1 : 0;
    };
    // Per in-flight item, by buffer: the item, the row's scale and (residual)
    // the CSR entry of this thread's block (two named slots, so they stay in registers).
    struct InFlight {
      Item it;
      float s;
      int e;
    };
    InFlight fl0 = {{0, 0, 0}, 0.0f, -1}, fl1 = fl0;
    auto fl_get = [&](int b) -> InFlight { return b ? fl1 : fl0; };
    // Wait for the item's inputs and convert its codes into A buffer b (the
    // tensor-memory stores are issued, not awaited).
    auto convert = [&](const Item& it, int b, InFlight& f) -> bool {
      const int st = it.i % NS;
      const uint32_t a_col = colA + 32 * b + lane_base;
      const int v = it.i / spv, gl = (it.i % spv) * kUG + it.q;
      f.it = it;
      if (it.kind == 0) {
        MQ_PT();
        if (it.q == 0 && !mbar_wait(&ctl.full[st], (it.i / NS) & 1, abort_flag, tmo, p.err)) return false;
        MQ_PA(1);
        MQ_PT();
        const uint8_t* rec = stages + st * kStageBytes + it.q * kWRecBytes;
        f.s = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(rec + kWRecScales + 2 * r)));
        f.e = -1;
        row_codes_to_tmem(rec + r * 16, 2048, a_col);
        MQ_PA(2);
      } else {
        const int e = ctl.map[v][gl][half];
        f.e = e;
        f.s = 0.0f;
        if (e >= 0) {  // warp-uniform: a warp's 32 rows lie in one half
          const int c = ctl.rpos[v][gl][half], slot = c % kRSlots;
          MQ_PT();
          if (!mbar_wait(&ctl.r_full[slot], (c / kRSlots) & 1, abort_flag, tmo, p.err)) return false;
          MQ_PA(1);
          MQ_PT();
          const uint8_t* rec = rring + slot * kRRecBytes;
          f.s = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(rec + kRRecScales + 2 * (r & 63))));
          row_codes_to_tmem(rec + (r & 63) * 16, 1024, a_col);
          MQ_PA(2);
        }
      }
      return true;
    };
    // Hand the converted item in A buffer b to the MMA warp and release what
    // this warpgroup has read.
    auto handoff = [&](const Item& it, int b) {
      const int st = it.i % NS;
      const int v = it.i / spv, gl = (it.i % spv) * kUG + it.q;
      MQ_PT();
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (r == 0) ctl.item_gl[w][b] = gl;
        // the stage's codes and scales are read once its last dense item is converted
        if (it.kind == 0 && it.q == stage_ng(it.i) - 1) mbar_arrive(&ctl.empty[st]);
        if (it.kind == 1) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
            if (ctl.map[v][gl][h] >= 0) mbar_arrive(&ctl.r_empty[ctl.rpos[v][gl][h] % kRSlots]);
        }
        // item_gl is written by warp quarter 0 before its own arrival; the MMA
        // warp's wait needs all four arrivals, so it sees the value
        mbar_arrive(&ctl.a_ready[w][b]);
      }
      MQ_PA(6);
    };
    // acc[m] += sx[m] * (s * (D[m] - 8 * sum_m)) from D buffer b (or, as a test hook, store the dots)
    auto drain = [&](int b) {
      const InFlight f = fl_get(b);
      const Item it = f.it;
      const int gl = (it.i % spv) * kUG + it.q;
      const int e = f.e;
      const bool use = it.kind == 0 || e >= 0;
      const float4* sx4 = reinterpret_cast<const float4*>(sxs + gl * TN);
      const float4* su4 = reinterpret_cast<const float4*>(sums + gl * TN);
      const uint64_t s2 = f2pack(f.s, f.s), m1 = f2pack(-1.0f, -1.0f);
#pragma unroll
      for (int cc = 0; cc < TN / 16; ++cc) {
        uint32_t dv[16];
        tmem_ld16(colD + TN * b + 16 * cc + lane_base, dv);
        tc_wait_ld();
        if (kDebug) {
          if (use) {
            const int64_t n = tile_of(it.i / spv) * kTileN + r;
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) {
              const int m = 16 * cc + i2;
              if (m < p.M) {
                const int32_t d =
                    static_cast<int32_t>(__uint_as_float(dv[i2])) - static_cast<int32_t>(sums[gl * TN + m]);
                if (it.kind == 0)
                  p.dots_w[(static_cast<int64_t>(m) * p.N + n) * G + gs + gl] = d;
                else
                  p.dots_r[(static_cast<int64_t>(m) * p.nnzb + e) * 64 + (r & 63)] = d;
              }
            }
          }
        } else if (use) {
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const float4 sv = sx4[cc * 4 + j4], cv = su4[cc * 4 + j4];  // tokens 16cc + 4j4 .. +3
            const int jp = cc * 8 + j4 * 2;
            // the dot of q with x is the dot of q + 8 minus 8 * sum(x): exact integers
            const uint64_t d0 = f2fma(f2pack(cv.x, cv.y), m1,
                                      f2pack(__uint_as_float(dv[4 * j4]), __uint_as_float(dv[4 * j4 + 1])));
            const uint64_t d1 = f2fma(f2pack(cv.z, cv.w), m1,
                                      f2pack(__uint_as_float(dv[4 * j4 + 2]), __uint_as_float(dv[4 * j4 + 3])));
            acc[jp] = f2fma(f2pack(sv.x, sv.y), f2mul(d0, s2), acc[jp]);
            acc[jp + 1] = f2fma(f2pack(sv.z, sv.w), f2mul(d1, s2), acc[jp + 1]);
          }
        }
      }
      tc_fence_before();
    };
    // End of visit v: add this warpgroup's partial into the CTA's row-major
    // buffer, in warpgroup order.
    auto finish_visit = [&](int v) -> bool {
      bool passed;
      if (w == 0)  // every owner has consumed the previous tile's push out of this buffer
        passed = v == 0 || mbar_wait_cluster(&ctl.rx_free, (v - 1) & 1, abort_flag, tmo, p.err);
      else
        passed = mbar_wait(&ctl.chain[w], v & 1, abort_flag, tmo, p.err);
      if (!passed) return false;
      float4* row = reinterpret_cast<float4*>(rb + r * TN);
#pragma unroll
      for (int k = 0; k < TN / 4; ++k) {
        float4 a;
        f2unpack(acc[2 * k], a.x, a.y);
        f2unpack(acc[2 * k + 1], a.z, a.w);
        if (w != 0) {
          const float4 o = row[k];
          a.x = o.x + a.x;
          a.y = o.y + a.y;
          a.z = o.z + a.z;
          a.w = o.w + a.w;
        }
        row[k] = a;
        acc[2 * k] = 0;
        acc[2 * k + 1] = 0;
      }
      // the buffer is pushed by bulk copies (the async proxy): order these
      // generic writes before them
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(w + 1 < kWG ? &ctl.chain[w + 1] : &ctl.rb_done);
      if (r == 0 && v < 2) MQ_DTRACE(29 + w * 2 + v);
      return true;
    };

    // Pipeline: up to two items at the MMA warp; item k uses buffers k & 1.
    int cur_v = 0;  // visits before cur_v are finished
    int ndrained = 0;
    Item nxt;
    nxt.i = w;
    nxt.q = 0;
    nxt.kind = 0;
    bool have = ok && nxt.i < total;
    int k = 0;  // items submitted
    // Before the oldest in-flight item is drained: the visits before its own
    // are complete (items come in visit order), so they are finished first
    // (the accumulators then hold only this visit's items); then its MMAs.
    auto ready_to_drain = [&]() -> bool {
      const int b = ndrained & 1;
      MQ_PT();
      bool passed = true;
      const int vj = fl_get(b).it.i / spv;
      while (passed && cur_v < vj) passed = finish_visit(cur_v++);
      MQ_PA(5);
      if (!passed) return false;
      MQ_PT();
      passed = mbar_wait(&ctl.d_ready[w][b], (ndrained >> 1) & 1, abort_flag, tmo, p.err);
      MQ_PA(3);
      tc_fence_after();
      return passed;
    };
    auto drain_oldest = [&]() {
      MQ_PT();
      drain(ndrained & 1);
      MQ_PA(4);
      ++ndrained;
    };
    while (ok && have) {
      const int b = k & 1;
      // Item k-2 used buffers b: once its MMAs are done, A[b] is free; item k
      // is converted into it, and item k-2 is drained from D[b] while the
      // tensor-memory stores of the conversion complete.
      if (k >= 2 && !(ok = ready_to_drain())) break;
      InFlight f;
      if (!(ok = convert(nxt, b, f))) break;
      if (k >= 2) drain_oldest();
      if (b)
        fl1 = f;
      else
        fl0 = f;
      handoff(nxt, b);
      ++k;
      MQ_PT();
      const int adv = advance(nxt);
      MQ_PA(0);
      if (adv < 0) {
        ok = false;
        break;
      }
      have = adv > 0;
    }
    // the last in-flight items
    while (ok && ndrained < k) {
      if (!(ok = ready_to_drain())) break;
      drain_oldest();
    }
    if (ok) {  // tell the MMA warp this warpgroup is done (buffer k & 1 is free: item k-2 is drained)
      __syncwarp();
      if (lane == 0) {
        if (r == 0) ctl.item_gl[w][k & 1] = -1;
        mbar_arrive(&ctl.a_ready[w][k & 1]);
      }
    }
    while (ok && cur_v < nvis) ok = finish_visit(cur_v++);
#ifdef MQ_DEC_TRACE
    prof_[8] = k;
    if (r == 0) mq_dec_trace_prof(w, prof_, 9);
#endif
  } else {
    // ---------------- epilogue: push partial rows to their owners, sum the owned rows, store Y ----------------
    const int et = threadIdx.x - 32 * kWarpEpi0;  // 0 .. kEpiThreads-1
    const uint32_t chunk = static_cast<uint32_t>(R * TN * 4);  // one owner's rows of one partial
    pdl_wait();  // Y may still be in use by the preceding kernel
    int nsync = 0;
    bool ok = true;
    for (int v = 0; ok && v < nvis; ++v) {
      const int64_t tile = tile_of(v);
      if (et == 0 && CS > 1) mbar_arrive_expect_tx(&ctl.rx_full, CS * chunk);
      if (!mbar_wait(&ctl.rb_done, v & 1, abort_flag, tmo, p.err)) { ok = false; break; }
      if (et == 0 && v < 2) MQ_DTRACE(37 + v);
      const float* src;
      int nsrc;
      if (CS > 1) {
        if (et == 0) {  // one bulk copy per owner: rows [k*R, (k+1)*R) of this CTA's partial
          const uint32_t rx_dst = smem_u32(rx) + rank * chunk, bar = smem_u32(&ctl.rx_full);
          for (int k = 0; k < CS; ++k) bulk_s2peer(mapa(rx_dst, k), rb + k * (R * TN), chunk, mapa(bar, k));
        }
        if (!mbar_wait(&ctl.rx_full, v & 1, abort_flag, tmo, p.err)) { ok = false; break; }
        src = rx;
        nsrc = CS;
      } else {
        src = rb;
        nsrc = 1;
      }
      if (et == 0 && v < 2) MQ_DTRACE(39 + v);
      if (!kDebug) {
        // thread: one owned row, four tokens; sources summed in rank order
        for (int idx = et; idx < R * (TN / 4); idx += kEpiThreads) {
          const int row = idx % R, m4 = (idx / R) * 4;
          if (m4 >= p.M) continue;
          const float4* sp = reinterpret_cast<const float4*>(src + row * TN + m4);
          float4 s = sp[0];
          for (int j = 1; j < nsrc; ++j) {  // ascending rank = ascending K slice
            const float4 t = sp[j * (R * TN / 4)];
            s.x += t.x;
            s.y += t.y;
            s.z += t.z;
            s.w += t.w;
          }
          const int64_t n = tile * kTileN + rank * R + row;
          const float vals[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            if (m4 + t < p.M) {
              const int64_t o = static_cast<int64_t>(m4 + t) * p.N + n;
              if (p.y_f32)
                static_cast<float*>(p.y)[o] = vals[t];
              else
                static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(vals[t]);
            }
          }
        }
      }
      __syncwarp();
      if ((et & 31) == 0) mbar_arrive(&ctl.epi_bar);  // every epilogue warp has read the received rows
      if (!mbar_wait(&ctl.epi_bar, nsync & 1, abort_flag, tmo, p.err)) { ok = false; break; }
      ++nsync;
      if (et == 0 && v < 2) MQ_DTRACE(41 + v);
      // Tell every source its push has been consumed (it may reuse its buffer
      // and push again); not after the last tile: nobody waits for that.
      if (et == 0 && v + 1 < nvis) {
        if (CS > 1)
          for (int k = 0; k < CS; ++k) remote_arrive(mapa(smem_u32(&ctl.rx_free), k));
        else
          mbar_arrive(&ctl.rx_free);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) MQ_DTRACE(44);
  if (*abort_flag) {
    // A wait gave up: copies or MMAs may still be landing in this CTA's shared
    // or tensor memory.  They finish within microseconds; give them 200 us.
    if (threadIdx.x == 0) {
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 200000ull) {
      }
    }
    __syncthreads();
  }
  if (warp == 0) tmem_dealloc(ctl.tmem_base, kTmemCols);
  // Every CTA has received all its rows, so every push out of this CTA's
  // shared memory has been read.
  cluster_sync_all();
  if (threadIdx.x == 0) MQ_DTRACE(45);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

struct DecPlan {
  int tn, cs, nstages, nclusters;
  uint32_t oSX, oRB, oRX, oR, oStage, smem;
};

template <int TN, bool kDebug>
static const void* kernel_ptr() {
  return reinterpret_cast<const void*>(&w4a4_decode_kernel<TN, kDebug>);
}

// Co-resident clusters of `cs` CTAs of this kernel (one CTA per SM), per device.
static int max_clusters(int cs) {
  static std::mutex mu;
  static int cache[64][kMaxCS + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev][cs] != 0) return cache[dev][cs];
  const void* kern = kernel_ptr<32, false>();
  const int smem = kSmemLimit - static_cast<int>(sizeof(DecCtl));
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cs * 256), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[dev][cs] = n > 0 ? n : -1;
  return cache[dev][cs];
}

static uint32_t up1024(uint32_t b) { return (b + 1023u) / 1024u * 1024u; }

// Pick the cluster size: the makespan of a CTA is (visits x slice) groups
// plus a per-visit reduction; the slice's activation tiles must fit.
static bool decode_plan(int64_t M, int64_t N, int64_t K, DecPlan* out) {
  if (M > 32) return false;
  const int tn = M <= 16 ? 16 : 32;
  const int G = static_cast<int>(K / kGroup), tiles = static_cast<int>(N / kTileN);
  double best = 1e30;
  bool found = false;
  for (int cs = 1; cs <= kMaxCS; cs *= 2) {
    if (cs > G) break;
    const int ns = (G + cs - 1) / cs;
    const uint32_t bbytes = static_cast<uint32_t>(ns) * tn * 128;
    if (ns > kMaxSlice || bbytes > static_cast<uint32_t>(kMaxBBytes)) continue;
    DecPlan pl;
    pl.tn = tn;
    pl.cs = cs;
    pl.oSX = bbytes;
    pl.oRB = up1024(pl.oSX + 2 * kMaxSlice * tn * 4);  // scales, then group sums
    pl.oRX = pl.oRB + tn * kTileN * 4;
    pl.oR = pl.oRX + (cs > 1 ? tn * kTileN * 4 : 0);
    pl.oStage = up1024(pl.oR + kRSlots * kRRecBytes);
    const int avail = kSmemLimit - static_cast<int>(sizeof(DecCtl)) - 1024 - static_cast<int>(pl.oStage);
    pl.nstages = std::min(kMaxStages, avail / kStageBytes);
    if (pl.nstages < 3) continue;
    pl.smem = pl.oStage + pl.nstages * kStageBytes + 1024;
    const int ncl = max_clusters(cs);
    if (ncl <= 0) continue;
    pl.nclusters = std::min(tiles, ncl);
    const int rounds = (tiles + pl.nclusters - 1) / pl.nclusters;
    if (rounds > kMaxVisits) continue;
    const double cost = rounds * (ns + 1.0) + (cs > 1 ? 1.0 : 0.0);
    if (cost < best) {
      best = cost;
      *out = pl;
      found = true;
    }
  }
  return found;
}

template <int TN, bool kDebug>
static mq_status launch_decode(const DecParams& dp, const DecPlan& pl, cudaStream_t stream) {
  const void* kern = kernel_ptr<TN, kDebug>();
  static bool smem_set[64];  // per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return launch_status("decode gemm: device");
  if (!smem_set[dev]) {
    const int want = kSmemLimit - static_cast<int>(sizeof(DecCtl));
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, want) != cudaSuccess)
      return launch_status("decode gemm: smem attribute");
    smem_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.nclusters * pl.cs), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, w4a4_decode_kernel<TN, kDebug>, dp) != cudaSuccess)
    return launch_status("decode gemm launch");
  return launch_status("decode gemm");
}

}  // namespace

// Runs the decode kernel when it covers (M, N, K) on this device; *handled
// tells the caller whether it did (else the general kernel runs).
mq_status gemm_decode_launch(bool* handled, const uint8_t* xq, const uint16_t* xs, int64_t M, const uint8_t* wpk,
                             int64_t N, int64_t K, const int32_t* row_ptr, const int32_t* col_idx, int64_t nnzb,
                             const uint8_t* rpk, void* y, mq_dtype yt, int32_t* dots_w, int32_t* dots_r,
                             cudaStream_t stream) {
  *handled = false;
  DecPlan pl;
  if (!decode_plan(M, N, K, &pl)) return MQ_OK;
  *handled = true;
  DecParams dp;
  dp.xq = xq;
  dp.xs = xs;
  dp.wpk = wpk;
  dp.row_ptr = row_ptr;
  dp.col_idx = col_idx;
  dp.rpk = rpk;
  dp.y = y;
  dp.y_f32 = yt == MQ_F32;
  dp.dots_w = dots_w;
  dp.dots_r = dots_r;
  dp.M = static_cast<int>(M);
  dp.Mp = static_cast<int>((M + 7) / 8 * 8);
  dp.N = static_cast<int>(N);
  dp.G = static_cast<int>(K / kGroup);
  dp.nnzb = static_cast<int>(nnzb);
  dp.tiles = static_cast<int>(N / kTileN);
  dp.cs = pl.cs;
  dp.nclusters = pl.nclusters;
  dp.nstages = pl.nstages;
  dp.oSX = pl.oSX;
  dp.oRB = pl.oRB;
  dp.oRX = pl.oRX;
  dp.oR = pl.oR;
  dp.oStage = pl.oStage;
  dp.timeout_ns = wait_timeout_ns();
  dp.err = device_error_word();
  if (!dp.err) return set_error(MQ_ERR_CUDA, "decode gemm: device error word unavailable");
  const bool dbg = dots_w != nullptr;
  if (pl.tn == 16) return dbg ? launch_decode<16, true>(dp, pl, stream) : launch_decode<16, false>(dp, pl, stream);
  return dbg ? launch_decode<32, true>(dp, pl, stream) : launch_decode<32, false>(dp, pl, stream);
}

}  // namespace mq
