// The fused W4A4 + block-sparse 4-bit residual GEMM for decode batches (at
// most 32 tokens): the ZipperEngine of the MosaicQuant summary (Metodologia 3)
// laid out for sm_103a.  It computes
//
//   Y[m,n] = sum_g sx[m,g] * ( sw[n,g] * Dw[m,n,g] + sr[n,g] * Dr[m,n,g] )
//
// in one kernel: the residual product of a selected 64x128 block runs on the
// same activation operand as the dense product of its group, and both are
// reduce-added into the same fp32 accumulators.
//
// At decode sizes the work is streaming the 4-bit weights.  Every 128-input
// group has its own scales, so its integer dot must be finished, scaled and
// added before the next group's.  One kernel template, two ways to run the
// per-group products (the compute role), one frame around them:
//   * unpacking is a mask: a byte 0x00..0x0F read as E4M3 is exactly
//     b * 2^-9 (subnormals below 8, the lowest normal binade from 8), so the
//     nibble u = q + 8 (q XOR 8) moved into a byte is u * 2^-9 with no table
//     (4 operations per 8 codes).  The dot is then 2^-9 * (D + 8 * sum_k
//     qx[m,k]); the scaling step subtracts the activation term (the group
//     sums of the resident activations are computed once) and folds 2^9 into
//     the activation scale.  Every partial sum is a multiple of 2^-9 below
//     2^14 in magnitude, so the fp32 accumulation is exact;
//   * K is permuted inside each 8-code word: the even codes, then the odd
//     ones, which is the order the mask leaves them in.  The activations use
//     the same permutation, so the dot is unchanged;
//   * warp-MMA variant (the default up to 16 tokens): each of 12 warps owns
//     32 rows and every third group of the CTA's list; per group it unpacks
//     its rows' codes in registers, runs mma.sync m16n8k32 e4m3 against
//     resident activation fragments and scales the exact dots into register
//     accumulators.  No hand-offs between roles;
//   * tensor-memory variant (above 16 tokens): each of 4 warpgroups owns all
//     128 rows (thread = row = tensor-memory lane) and every fourth group; it
//     unpacks into double-buffered tensor-memory A operands, its first warp
//     issues the group's four tcgen05 MMAs (B = the 128-byte-swizzled
//     activation tile) once the warpgroup's four warps have stored theirs,
//     and the warpgroup drains the accumulators two items later.
// The frame:
//   * Split-K over a thread-block cluster of CS CTAs.  A cluster owns whole
//     128-row weight tiles (one after another, persistently); CTA rank j
//     handles the same K slice [j*G/CS, (j+1)*G/CS) of every tile it visits,
//     so its activations arrive by bulk copy, are converted once, and stay in
//     shared memory.
//   * A producer warp streams the base-weight records (codes and scales side
//     by side, 8.25 KiB, one bulk copy each) into a ring of stages; a second
//     one reads the block lists of every tile the CTA visits once, up front,
//     into a static map, and streams the residual block records of this slice
//     into a small ring.
//   * At the end of a tile the compute sets' partials are added in a fixed
//     order.  With one CTA per cluster the last set stores Y from registers;
//     otherwise each CTA pushes the rows owned by rank k into rank k's shared
//     memory with one bulk copy (distributed shared memory, counted on the
//     owner's barrier), and each rank sums its 128/CS rows over the CS
//     partials in rank order and stores Y.  No global workspace, no atomics:
//     the result is deterministic.
// Every wait is bounded (mbar_wait): a wait that runs out records the error,
// raises the CTA's abort flag, and every role winds down.
#include "mq_internal.cuh"

#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
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

constexpr int kEpiThreads = 64;
// Warp roles of the two variants of the kernel.  Compute warps come in sets
// of four; set q takes groups q, q + kSets, q + 2 kSets, .. of the CTA's list.
//   warp-MMA variant: 3 sets; warp w owns rows 32*(w%4) .. +31 of its set's
//     groups (16 warps in all: 4 per sub-partition, up to 128 registers);
//   tensor-memory variant: 4 sets (warpgroups); thread t of a warpgroup owns
//     row t (its tensor-memory lane) (20 warps: 5 per sub-partition, 96
//     registers).
// Then one producer warp, one residual-producer warp and two epilogue warps.
template <bool kTC>
struct Roles {
  static constexpr int kSets = kTC ? 4 : 3;
  static constexpr int kCompute = 4 * kSets;
  static constexpr int kProducer = kCompute;      // activations, then the base-weight stages
  static constexpr int kResidual = kCompute + 1;  // block list, then the residual records
  static constexpr int kEpi0 = kCompute + 2;      // epilogue warps
  static constexpr int kThreads = 32 * kEpi0 + kEpiThreads;
  static constexpr int kMaxReg = kTC ? 96 : 128;
};
constexpr int kTmemCols = 512;  // tensor-memory variant: per warpgroup A0, A1 (32 columns each), D0, D1 (TN each)
constexpr int kStageBytes = kWRecBytes;   // one group's base record per stage
constexpr int kMaxStages = 24;
constexpr int kRSlots = 6;                // residual-record ring
constexpr int kMaxVisits = 16;            // tiles visited per CTA
constexpr int kMaxSlice = 32;             // groups in a CTA's K slice
constexpr int kMaxBBytes = 112 * 1024;    // resident activation fragments
constexpr int kSmemLimit = 227 * 1024;
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
  uint32_t oSX, oRB, oRX, oR, oStage;  // shared-memory offsets; the activation fragments are at 0
  uint64_t timeout_ns;
  uint32_t* err;
};

struct __align__(8) DecCtl {
  uint64_t full[kMaxStages];     // producer arrival + record bytes
  uint64_t empty[kMaxStages];    // the 4 warps of the consuming set are done with the stage
  uint64_t r_full[kRSlots];
  uint64_t r_empty[kRSlots];     // the 2 warps that used the residual record
  uint64_t x_full;               // the slice's packed activations and scales have landed (bytes)
  uint64_t work_bar;             // activation fragments converted (one arrival per MMA warp)
  uint64_t epi_bar;              // bounded barrier of the 2 epilogue warps
  uint64_t map_ready;            // residual map and ring positions are built
  uint64_t chain[3];             // set q has added its partial of the tile (q < kSets - 1)
  uint64_t rb_done;              // the last set has added its partial: the CTA's partial is complete
  uint64_t rx_full;              // every rank's rows for this CTA have landed (bytes)
  uint64_t rx_free;              // every owner has consumed this CTA's last push
  uint64_t exit_bar;             // every warp of the CTA is done with its role
  uint64_t d_ready[4][2];        // tensor-memory variant: the MMAs of A/D buffer b of warpgroup w are complete
  uint32_t a_cnt[4][2];          // warps of warpgroup w that have stored A buffer b, over all its uses
  uint32_t tmem_base;
  int32_t map[kMaxVisits][kMaxSlice][2];   // CSR entry of the slice's residual blocks per tile, or -1
  int32_t rpos[kMaxVisits][kMaxSlice][2];  // position of that block in the residual-ring order
  int32_t sc_off[kMaxVisits + 1], sc_a0[kMaxVisits], sc_a1[kMaxVisits];
  int abort_flag;
};
// Static shared memory of the kernel: the control block, padded as the
// dynamic array that follows it is aligned.
constexpr int kCtlBytes = (static_cast<int>(sizeof(DecCtl)) + 127) / 128 * 128;

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
// Shared-memory counter increment with acquire-release ordering; returns the old value.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* ctr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_u32(ctr)), "r"(v)
               : "memory");
  return old;
}
// The same without ordering memory: only that every thread of the cluster got here.
__device__ __forceinline__ void cluster_sync_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;\n\tbarrier.cluster.wait;" ::: "memory");
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
// Bounded wait for the roles that wait long (producers for free slots, the
// epilogue for a finished tile): each try_wait may stay suspended up to
// `hint_ns` (it returns as soon as the phase completes), so the waiting warp
// takes few issue slots from the MMA warps.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_long(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                               uint64_t timeout_ns, uint32_t* err_word) {
  constexpr uint32_t kHintNs = 20000;
  if (mbar_try_wait_hint(bar, parity, kHintNs)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    __nanosleep(200);  // back off: a waiting warp issues nothing while asleep
    if (mbar_try_wait_hint(bar, parity, kHintNs)) return true;
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
// 16-byte shared-memory load by shared-window address.
__device__ __forceinline__ float4 lds_f4(uint32_t saddr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(saddr)
               : "memory");
  return v;
}

// D(16x8, fp32) += A(16x32, E4M3, row-major) * B(32x8, E4M3, column-major):
// the warp-level FP8 MMA.
__device__ __forceinline__ void mma_e4m3(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same with a zero accumulator in (the first K-step of a group).
__device__ __forceinline__ void mma_e4m3_zc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// Packed fp32 pairs (one instruction for two lanes' worth of fp32 math).
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

// Eight weight codes q (two's complement nibbles, element i in bits 4i..4i+3)
// -> two words of four E4M3 bytes holding (q + 8) * 2^-9 exactly: the even
// elements 0, 2, 4, 6 in `ev`, the odd ones in `od`.
__device__ __forceinline__ void unpack_u4(uint32_t p, uint32_t& ev, uint32_t& od) {
  const uint32_t u = p ^ 0x88888888u;
  ev = u & 0x0F0F0F0Fu;
  od = (u >> 4) & 0x0F0F0F0Fu;
}

// Store 16 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
// Shared-memory matrix descriptor of a K-major operand in 128-byte-swizzled
// rows (8-row atoms 1024 bytes apart).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// One output element (bf16 or fp32 Y, row-major [M][N]).
__device__ __forceinline__ void store_y(const DecParams& p, int m, int64_t n, float v) {
  const int64_t o = static_cast<int64_t>(m) * p.N + n;
  if (p.y_f32)
    static_cast<float*>(p.y)[o] = v;
  else
    static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(v);
}

// Sum of the eight signed codes of a word of packed activations.
__device__ __forceinline__ int nibble_sum8(uint32_t p) {
  const uint32_t u = p ^ 0x88888888u;  // q + 8 in [1, 15]
  const uint32_t b = (u & 0x0F0F0F0Fu) + ((u >> 4) & 0x0F0F0F0Fu);
  return static_cast<int>((b * 0x01010101u) >> 24) - 64;
}

template <int TN, bool kDebug, bool kTC>
__global__ void __maxnreg__(Roles<kTC>::kMaxReg) w4a4_decode_kernel(const DecParams p) {
  using RL = Roles<kTC>;
  constexpr int kSlots = RL::kSets, kMmaWarps = RL::kCompute, kWarpProducer = RL::kProducer;
  constexpr int kWarpResidual = RL::kResidual, kWarpEpi0 = RL::kEpi0, kThreads = RL::kThreads;
  static_assert(!kTC || TN % 16 == 0, "tensor-memory MMAs with M = 128 need N a multiple of 16");
  constexpr int NB = TN / 8;                 // 8-token blocks of one MMA
  constexpr int kGroupFrag = 4 * NB * 256;   // activation fragment bytes of one group
  constexpr int kChains = NB == 1 ? 2 : 1;   // accumulator sets per MMA tile, for independent MMAs
  extern __shared__ uint8_t smem_raw[];
  __shared__ DecCtl ctl;
  // 1024-aligned by offsetting the shared array itself (keeps accesses in the shared window)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  // Activation fragments: [ns][4 K-steps][NB][32 lanes] x 8 bytes (E4M3); lane
  // (g, t) of block nb holds token 8nb + g: the even codes 8t, 8t+2, .., 8t+6
  // of the K-step, then the odd ones.
  uint8_t* bfrag = smem;
  // [ns][TN/2] x {sx[2i], sx[2i+1], c[2i], c[2i+1]}: activation scales and the
  // offset term c = 2^-9 * 8 * (sum of the group's activation codes)
  float4* sxc = reinterpret_cast<float4*>(smem + p.oSX);
  float* rb = reinterpret_cast<float*>(smem + p.oRB);      // [128 rows][TN] the CTA's partial of a tile
  float* rx = reinterpret_cast<float*>(smem + p.oRX);      // [CS sources][R rows][TN] the rows this CTA owns
  uint8_t* rring = smem + p.oR;                            // [kRSlots] residual records
  uint8_t* stages = smem + p.oStage;                       // [nstages] base records
  if (threadIdx.x == 0) MQ_DTRACE(0);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int CS = p.cs, NS = p.nstages, G = p.G;
  const int R = kTileN / CS;  // rows of a tile each rank finishes
  const int rank = static_cast<int>(cluster_rank());
  const int cid = static_cast<int>(cluster_index());
  const int gs = rank * G / CS, ge = (rank + 1) * G / CS, ns = ge - gs;  // this CTA's K slice
  const int nvis = (p.tiles - cid + p.nclusters - 1) / p.nclusters;       // tiles cid, cid + nclusters, ...
  const int total = nvis * ns;                                            // stage i: group i % ns of visit i / ns
  volatile int* abort_flag = &ctl.abort_flag;
  const uint64_t tmo = p.timeout_ns;
  auto tile_of = [&](int v) { return static_cast<int64_t>(cid) + static_cast<int64_t>(v) * p.nclusters; };
  auto stage_rec = [&](int i) { return p.wpk + (tile_of(i / ns) * G + gs + i % ns) * kWRecBytes; };

  if (warp == 0) {  // barrier initialisation, spread over the lanes of warp 0
    for (int s = lane; s < NS; s += 32) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], 4);
    }
    if (lane < kRSlots) {
      mbar_init(&ctl.r_full[lane], 1);
      mbar_init(&ctl.r_empty[lane], kTC ? 4 : 2);
    }
    if (kTC && lane >= 8 && lane < 16) {
      ctl.a_cnt[(lane - 8) >> 1][lane & 1] = 0;
      mbar_init(&ctl.d_ready[(lane - 8) >> 1][lane & 1], 1);
    }
    if (lane + 1 < kSlots) mbar_init(&ctl.chain[lane], 4);
    if (lane == 16) mbar_init(&ctl.x_full, 1);
    if (lane == 17) mbar_init(&ctl.work_bar, kMmaWarps);
    if (lane == 18) mbar_init(&ctl.epi_bar, kEpiThreads / 32);
    if (lane == 19) mbar_init(&ctl.map_ready, 1);
    if (lane == 20) mbar_init(&ctl.rb_done, 4);
    if (lane == 21) mbar_init(&ctl.rx_full, 1);
    // With one CTA per cluster the last compute set stores Y itself and frees
    // the reduction buffer (one arrival per warp); else each owner frees it.
    if (lane == 22) mbar_init(&ctl.rx_free, CS == 1 && !kDebug ? 4 : CS);
    if (lane == 23) mbar_init(&ctl.exit_bar, kThreads / 32);
    if (lane == 24) ctl.abort_flag = 0;
    fence_mbar_init();
  }
  // The next kernel may start launching: everything it reads before its own
  // dependency wait is read-only here.
  pdl_trigger();
  // Every CTA of the cluster has its barriers initialised before any peer
  // pushes into them (also a barrier of this CTA's threads).
  cluster_sync_all();
  if (threadIdx.x == 0) MQ_DTRACE(1);

  // Sum the CS partials of this rank's R rows of tile `tile` (sources in rank
  // order) and store them to Y: item idx = (4-token block, row), items t0,
  // t0 + nthr, ..; four items' loads go ahead of their stores.
  auto store_owned = [&](const float* src, int nsrc, int64_t tile, int t0, int nthr) {
    const uint32_t src_s = smem_u32(src);
    const int rsh = __ffs(R) - 1;  // R = 128 / CS is a power of two
    constexpr int kU = 4;
    for (int base = t0; base < R * (TN / 4); base += kU * nthr) {
      float4 acc4[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int idx = base + u * nthr;
        const int row = idx & (R - 1), m4 = (idx >> rsh) * 4;
        if (idx < R * (TN / 4) && m4 < p.M) {
          const uint32_t a = src_s + static_cast<uint32_t>(row * TN + m4) * 4;
          float4 sv = lds_f4(a);
          for (int j = 1; j < nsrc; ++j) {  // ascending rank = ascending K slice
            const float4 t = lds_f4(a + static_cast<uint32_t>(j * R * TN) * 4);
            sv.x += t.x;
            sv.y += t.y;
            sv.z += t.z;
            sv.w += t.w;
          }
          acc4[u] = sv;
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int idx = base + u * nthr;
        const int row = idx & (R - 1), m4 = (idx >> rsh) * 4;
        if (idx < R * (TN / 4) && m4 < p.M) {
          const int64_t n = tile * kTileN + rank * R + row;
          const float vals[4] = {acc4[u].x, acc4[u].y, acc4[u].z, acc4[u].w};
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (m4 + t < p.M) store_y(p, m4 + t, n, vals[t]);
        }
      }
    }
  };
  // Threads that store the last tile's owned rows (several CTAs per cluster):
  // the epilogue warps and, having finished their last tile, the compute warps.
  constexpr int kLastStorers = kEpiThreads + 32 * kMmaWarps;

  if (warp == kWarpProducer) {
    // ---------------- producer: activations, then the base-weight stages in order ----------------
    const int pre = min(NS, total);
    if (lane < pre) prefetch_l2(stage_rec(lane), kWRecBytes);  // no dependency: L2 only
    // Everything below may read buffers the preceding kernel wrote (the
    // activations just quantized, weights just packed): wait for it.
    pdl_wait();
    if (lane == 0) MQ_DTRACE(2);
    {  // the slice's packed activations (group gl into the upper half of its
       // fragment block) and scales (into the reduction buffer, unused until
       // the first tile ends), ahead of every weight copy
      const uint32_t xbytes = static_cast<uint32_t>(p.Mp) * 64;
      if (lane == 0) mbar_arrive_expect_tx(&ctl.x_full, ns * xbytes + ns * p.Mp * 2);
      __syncwarp();
      for (int gl = lane; gl < ns; gl += 32)
        bulk_g2s(bfrag + gl * kGroupFrag + TN * 64, p.xq + static_cast<int64_t>(gs + gl) * xbytes, xbytes,
                 &ctl.x_full);
      if (lane == 0)
        bulk_g2s(rb, p.xs + static_cast<int64_t>(gs) * p.Mp, static_cast<uint32_t>(ns * p.Mp * 2), &ctl.x_full);
    }
    if (lane < pre) {  // the first stages, all at once
      mbar_arrive_expect_tx(&ctl.full[lane], kWRecBytes);
      bulk_g2s(stages + lane * kStageBytes, stage_rec(lane), kWRecBytes, &ctl.full[lane]);
    }
    // then each stage once its slot is free; (v, gl) = visit and group of
    // stage i, st its slot, ph the parity of the slot's previous use
    int v = pre / ns, gl = pre - (pre / ns) * ns, st = 0, ph = 0;
    for (int i = pre; i < total; ++i) {
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait_long(&ctl.empty[st], ph, abort_flag, tmo, p.err);
        if (ok) {
          mbar_arrive_expect_tx(&ctl.full[st], kWRecBytes);
          bulk_g2s(stages + st * kStageBytes, p.wpk + (tile_of(v) * G + gs + gl) * kWRecBytes, kWRecBytes,
                   &ctl.full[st]);
        }
      }
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
      if (lane == 0 && i < pre + 8) MQ_DTRACE(4 + i - pre);
      if (++gl == ns) gl = 0, ++v;
      if (++st == NS) st = 0, ph ^= 1;
    }
  } else if (warp == kWarpResidual) {
    // ---------------- residual producer: block list, then the residual records in order ----------------
    pdl_wait();  // the block list may have been written by the preceding kernel
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
    for (int i = 0, v = 0, gl = 0; i < total; ++i, gl = gl + 1 == ns ? 0 : gl + 1, v += gl == 0) {
      // lanes 0, 1: the residual records of stage i's two halves (group gl of visit v), into the ring
      int rok = 1;
      if (lane < 2) {
        const int e = ctl.map[v][gl][lane];
        if (e >= 0) {
          const int c = ctl.rpos[v][gl][lane], slot = c % kRSlots;
          if (c >= kRSlots) rok = mbar_wait_long(&ctl.r_empty[slot], ((c / kRSlots) & 1) ^ 1, abort_flag, tmo, p.err);
          if (rok) {
            mbar_arrive_expect_tx(&ctl.r_full[slot], kRRecBytes);
            bulk_g2s(rring + slot * kRRecBytes, p.rpk + static_cast<int64_t>(e) * kRRecBytes, kRRecBytes,
                     &ctl.r_full[slot]);
          }
        }
      }
      if (!__all_sync(0xFFFFFFFFu, rok)) break;
    }
  } else if (warp < kMmaWarps) {
   if constexpr (!kTC) {
    // ---------------- MMA warps ----------------
    const int gq = lane >> 2, tq = lane & 3;   // MMA fragment coordinates: row / token group, thread in group
    const int q = warp >> 2;                   // warp set: stages q, q + kSlots, ...
    const int rb0 = 32 * (warp & 3);           // first tile row of this warp
    const int half = rb0 >> 6;                 // residual block (64 rows) of its rows
    bool ok = true;

    // --- this slice's activations, once: packed codes -> E4M3 fragments,
    // their group sums, and the scales -> fp32.  Warp w converts groups w,
    // w + kMmaWarps, ..; each group's packed codes sit in the upper half of
    // its own fragment block, so the warp reads all of them before writing.
    pdl_wait();
    if (!(ok = mbar_wait(&ctl.x_full, 0, abort_flag, tmo, p.err))) {
      // fall through to the arrival below; the abort flag is up
    } else {
      const uint16_t* xs_raw = reinterpret_cast<const uint16_t*>(rb);  // [ns][Mp]
      float* sxcf = reinterpret_cast<float*>(sxc);
      for (int gl = warp; gl < ns; gl += kMmaWarps) {
        uint8_t* blk = bfrag + gl * kGroupFrag;
        const uint8_t* raw = blk + TN * 64;  // [Mp][64]
        uint32_t wv[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const int m = 8 * nb + gq;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            wv[nb][j] = m < p.Mp ? *reinterpret_cast<const uint32_t*>(raw + m * 64 + j * 16 + tq * 4) : 0u;
        }
        __syncwarp();
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          int sum = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t lo, hi;  // codes 0..3, 4..7 of the word
            int4x8_to_e4m3(wv[nb][j], lo, hi);
            *reinterpret_cast<uint2*>(blk + ((j * NB + nb) * 32 + lane) * 8) =
                make_uint2(prmt(lo, hi, 0x6420u), prmt(lo, hi, 0x7531u));  // even | odd codes
            sum += nibble_sum8(wv[nb][j]);
          }
          sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);  // the token's four quarters of each K-step
          sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
          const int m = 8 * nb + gq;
          if (tq == 0) {
            float* dst = sxcf + (gl * (TN / 2) + m / 2) * 4 + (m & 1);
            dst[0] = m < p.Mp ? 512.0f * __half2float(__ushort_as_half(xs_raw[gl * p.Mp + m])) : 0.0f;  // 2^9 sx
            dst[2] = static_cast<float>(sum) * (1.0f / 64.0f);  // 8 * sum * 2^-9, exact
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl.work_bar);
    ok = mbar_wait(&ctl.work_bar, 0, abort_flag, tmo, p.err) && ok;
    if (threadIdx.x == 0) MQ_DTRACE(12);

    // accumulators of row tile mt (rows rb0 + 16mt + gq, +8) and token block
    // nb, as fp32 pairs: [0] = row +0, tokens 8nb+2tq, +1; [1] = row +8, same tokens
    uint64_t acc[2][NB][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) acc[mt][nb][0] = acc[mt][nb][1] = 0ull;
#ifdef MQ_DEC_TRACE
    long long prof_[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0}, pt_ = 0;
#endif

    // One group's product for this warp's 32 rows, scaled into the
    // accumulators: dense (base record, K-steps 2048 bytes apart, first row
    // rb0) or residual (residual record, 1024 apart, first row rb0 - 64*half).
    // sc: the record's fp16 scales; e: the block's CSR entry (residual) or -1.
    auto group_product = [&](const uint8_t* codes, int jstride, int row0, const uint16_t* sc, int gl,
                             int64_t tile, int e) {
      float d[kChains][2][NB][4];
      const uint8_t* bg = bfrag + gl * kGroupFrag + lane * 8;
      const uint8_t* wr = codes + (row0 + gq) * 16 + tq * 4;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t a[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(wr + j * jstride + mt * 256);        // row +0
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(wr + j * jstride + mt * 256 + 128);  // row +8
          unpack_u4(w0, a[mt][0], a[mt][2]);
          unpack_u4(w1, a[mt][1], a[mt][3]);
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const uint2 b = *reinterpret_cast<const uint2*>(bg + (j * NB + nb) * 256);
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            if (j < kChains)
              mma_e4m3_zc(d[j % kChains][mt][nb], a[mt], b.x, b.y);
            else
              mma_e4m3(d[j % kChains][mt][nb], a[mt], b.x, b.y);
          }
        }
      }
      if (kChains > 1) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int r = 0; r < 4; ++r) d[0][mt][nb][r] += d[kChains - 1][mt][nb][r];
      }
      uint64_t s2[2][2];  // the rows' scales, paired
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float sv = __half2float(__ushort_as_half(sc[row0 + 16 * mt + 8 * h + gq]));
          s2[mt][h] = f2pack(sv, sv);
        }
      const float4* sg = sxc + gl * (TN / 2) + tq;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const float4 f = sg[4 * nb];  // tokens t0 = 8nb + 2tq, t0 + 1: 2^9 sx, 2^9 sx, c, c
        const uint64_t sx2 = f2pack(f.x, f.y), c2 = f2pack(f.z, f.w), m1 = f2pack(-1.0f, -1.0f);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          // 2^-9 times the dot of q with x: the measured dot minus the offset term, exact
          if (kDebug) {
            const float e00 = d[0][mt][nb][0] - f.z, e01 = d[0][mt][nb][1] - f.w;
            const float e10 = d[0][mt][nb][2] - f.z, e11 = d[0][mt][nb][3] - f.w;
            const float ev[2][2] = {{e00, e01}, {e10, e11}};
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                const int m = 8 * nb + 2 * tq + c, r = rb0 + 16 * mt + 8 * h + gq;
                if (m < p.M) {
                  const int32_t dv = static_cast<int32_t>(ev[h][c] * 512.0f);
                  if (e < 0)
                    p.dots_w[(static_cast<int64_t>(m) * p.N + tile * kTileN + r) * G + gs + gl] = dv;
                  else
                    p.dots_r[(static_cast<int64_t>(m) * p.nnzb + e) * 64 + (r & 63)] = dv;
                }
              }
          } else {
            const uint64_t e0 = f2fma(c2, m1, f2pack(d[0][mt][nb][0], d[0][mt][nb][1]));  // row +0
            const uint64_t e1 = f2fma(c2, m1, f2pack(d[0][mt][nb][2], d[0][mt][nb][3]));  // row +8
            acc[mt][nb][0] = f2fma(sx2, f2mul(s2[mt][0], e0), acc[mt][nb][0]);
            acc[mt][nb][1] = f2fma(sx2, f2mul(s2[mt][1], e1), acc[mt][nb][1]);
          }
        }
      }
    };
    // End of visit v: add this warp's partial into the CTA's row-major
    // buffer, set 0 first, then set 1, then set 2 (each over all 128 rows).
    auto finish_visit = [&](int v) -> bool {
      bool passed;
      if (q == 0)  // every owner has consumed the previous tile's push out of this buffer
        passed = v == 0 || mbar_wait_cluster(&ctl.rx_free, (v - 1) & 1, abort_flag, tmo, p.err);
      else
        passed = mbar_wait(&ctl.chain[q - 1], v & 1, abort_flag, tmo, p.err);
      if (!passed) return false;
      const bool direct = CS == 1 && !kDebug && q + 1 == kSlots;  // the last set stores Y
      const int64_t n0 = tile_of(v) * kTileN;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          float2* r0 = reinterpret_cast<float2*>(rb + (rb0 + 16 * mt + gq) * TN + 8 * nb + 2 * tq);
          float2* r1 = r0 + 4 * TN;  // row + 8
          float2 v0, v1;
          f2unpack(acc[mt][nb][0], v0.x, v0.y);
          f2unpack(acc[mt][nb][1], v1.x, v1.y);
          if (q != 0) {
            const float2 o0 = *r0, o1 = *r1;
            v0 = make_float2(o0.x + v0.x, o0.y + v0.y);
            v1 = make_float2(o1.x + v1.x, o1.y + v1.y);
          }
          if (direct) {
            const int m = 8 * nb + 2 * tq;
            const int64_t n = n0 + rb0 + 16 * mt + gq;
            if (m < p.M) store_y(p, m, n, v0.x), store_y(p, m, n + 8, v1.x);
            if (m + 1 < p.M) store_y(p, m + 1, n, v0.y), store_y(p, m + 1, n + 8, v1.y);
          } else {
            *r0 = v0;
            *r1 = v1;
          }
          acc[mt][nb][0] = acc[mt][nb][1] = 0ull;
        }
      // the buffer is pushed by bulk copies (the async proxy): order these
      // generic writes before them
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (q + 1 < kSlots)
          mbar_arrive(&ctl.chain[q]);
        else if (!direct)
          mbar_arrive(&ctl.rb_done);
        else if (v + 1 < nvis)
          mbar_arrive(&ctl.rx_free);  // this warp's rows of the buffer are read
      }
      if (lane == 0 && v == 0) MQ_DTRACE(13 + warp);
      return true;
    };

    bool map_seen = false;
    int cur_v = 0;
    // stage i = q, q + kSlots, ..: group gl of visit v, in slot st whose fill parity is ph
    int v = q / ns, gl = q - (q / ns) * ns, st = q, ph = 0;
    for (int i = q; ok && i < total; i += kSlots) {
      MQ_PT();
      while (ok && cur_v < v) ok = finish_visit(cur_v++);
      MQ_PA(5);
      if (!ok) break;
      MQ_PT();
      if (!(ok = mbar_wait(&ctl.full[st], ph, abort_flag, tmo, p.err))) break;
      MQ_PA(1);
      const int64_t tile = tile_of(v);
      const uint8_t* rec = stages + st * kStageBytes;
      MQ_PT();
      group_product(rec, 2048, rb0, reinterpret_cast<const uint16_t*>(rec + kWRecScales), gl, tile, -1);
      MQ_PA(2);
      // the residual block of this warp's rows, if the block list has one here
      if (!map_seen) {
        MQ_PT();
        if (!(ok = mbar_wait(&ctl.map_ready, 0, abort_flag, tmo, p.err))) break;
        MQ_PA(0);
        map_seen = true;
      }
      const int e = ctl.map[v][gl][half];
      if (e >= 0) {
        const int c = ctl.rpos[v][gl][half], slot = c % kRSlots;
        MQ_PT();
        if (!(ok = mbar_wait(&ctl.r_full[slot], (c / kRSlots) & 1, abort_flag, tmo, p.err))) break;
        MQ_PA(3);
        MQ_PT();
        const uint8_t* rrec = rring + slot * kRRecBytes;
        group_product(rrec, 1024, rb0 - 64 * half, reinterpret_cast<const uint16_t*>(rrec + kRRecScales), gl, tile,
                      e);
        MQ_PA(4);
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.r_empty[slot]);  // the 2 warps of this half release it
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.empty[st]);  // the set's 4 warps release the stage
      for (gl += kSlots; gl >= ns; gl -= ns) ++v;
      if ((st += kSlots) >= NS) st -= NS, ph ^= 1;
    }
    while (ok && cur_v < nvis) ok = finish_visit(cur_v++);
    // the last tile's owned rows, with the epilogue warps (several CTAs per cluster)
    if (ok && CS > 1 && !kDebug && mbar_wait(&ctl.rx_full, (nvis - 1) & 1, abort_flag, tmo, p.err))
      store_owned(rx, CS, tile_of(nvis - 1), kEpiThreads + threadIdx.x, kLastStorers);
#ifdef MQ_DEC_TRACE
    prof_[8] = (total - q + kSlots - 1) / kSlots;
    if (lane == 0 && warp < 4) mq_dec_trace_prof(warp, prof_, 9);
#endif
   } else {
    // ---------------- tensor-memory converters: warpgroup w owns all 128 rows (thread = row = TMEM lane) ----------------
    const int w = warp >> 2, quarter = warp & 3;
    const int r = quarter * 32 + lane;  // weight row of the tile
    const int half = r >> 6;            // residual block (64 rows) of the row; a warp's rows share it
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    float* sxf = reinterpret_cast<float*>(sxc);  // [ns][TN] 2^9 * activation scales
    float* cfv = sxf + kMaxSlice * TN;           // [ns][TN] offset terms 2^-9 * 8 * (sum of the codes)
    bool ok = true;
    if (warp == 0) tmem_alloc(&ctl.tmem_base, kTmemCols);

    // --- this slice's activations, once: packed codes -> E4M3 rows of the
    // 128-byte-swizzled, K-major B tile (token m = row m), with the same K
    // order as the A columns (per 8 codes: the even ones, then the odd ones);
    // group sums and scales.  Warp w converts groups w, w + 16, ..
    pdl_wait();
    if (mbar_wait(&ctl.x_full, 0, abort_flag, tmo, p.err)) {
      if (threadIdx.x == 0) MQ_DTRACE(55);
      const uint16_t* xs_raw = reinterpret_cast<const uint16_t*>(rb);  // [ns][Mp]
      constexpr int kLpt = 32 / TN, kWpl = 16 / kLpt;                   // lanes per token, words per lane
      const int m = lane / kLpt, t0 = (lane % kLpt) * kWpl;
      for (int gl = warp; gl < ns; gl += kMmaWarps) {
        uint8_t* blk = bfrag + gl * (TN * 128);
        const uint8_t* raw = blk + TN * 64;  // [Mp][64]
        uint32_t wv[kWpl];
#pragma unroll
        for (int u = 0; u < kWpl; ++u)
          wv[u] = m < p.Mp ? *reinterpret_cast<const uint32_t*>(raw + m * 64 + (t0 + u) * 4) : 0u;
        __syncwarp();
        uint8_t* row = blk + (m >> 3) * 1024 + (m & 7) * 128;
        int sum = 0;
#pragma unroll
        for (int u = 0; u < kWpl; ++u) {
          const int t = t0 + u;  // codes 8t .. 8t+7 -> bytes 8t .. 8t+7 of the row: 16-byte chunk t/2
          uint32_t lo, hi;
          int4x8_to_e4m3(wv[u], lo, hi);
          *reinterpret_cast<uint2*>(row + (((t >> 1) ^ (m & 7)) * 16) + (t & 1) * 8) =
              make_uint2(prmt(lo, hi, 0x6420u), prmt(lo, hi, 0x7531u));
          sum += nibble_sum8(wv[u]);
        }
        if (kLpt == 2) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
        if (lane % kLpt == 0) {
          sxf[gl * TN + m] = m < p.Mp ? 512.0f * __half2float(__ushort_as_half(xs_raw[gl * p.Mp + m])) : 0.0f;
          cfv[gl * TN + m] = static_cast<float>(sum) * (1.0f / 64.0f);
        }
      }
    } else {
      ok = false;
    }
    fence_proxy_async_smem();  // generic writes -> the tensor core's reads
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl.work_bar);
    ok = mbar_wait(&ctl.work_bar, 0, abort_flag, tmo, p.err) && ok;
    tc_fence_after();
    if (threadIdx.x == 0) MQ_DTRACE(12);

    const uint32_t tmem = ctl.tmem_base;
    // Per warpgroup 128 columns: A buffers b = 0, 1 (32 columns each), then D
    // buffers (kDCh accumulator chains of TN columns each: K-steps j and
    // j + kDCh accumulate into chain j; independent chains let the tensor
    // core overlap their MMAs, and their exact sums are added in the drain).
    constexpr int kDCh = TN == 16 ? 2 : 1;
    static_assert(64 + 2 * kDCh * TN <= 128, "tensor-memory columns per warpgroup");
    const uint32_t colA = tmem + w * 128, colD = tmem + w * 128 + 64;  // buffer b: +32b, +kDCh*TN*b
    const uint32_t bt = smem_u32(bfrag);
    // kind::f8f6f4, E4M3 x E4M3 -> f32, K-major A and B, N = TN, M = 128
    constexpr uint32_t kIdesc =
        (1u << 4) | (static_cast<uint32_t>(TN >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
    uint64_t acc[TN / 2];  // row r, tokens 2j, 2j+1
#pragma unroll
    for (int j = 0; j < TN / 2; ++j) acc[j] = 0ull;
#ifdef MQ_DEC_TRACE
    long long prof_[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0}, pt_ = 0;
#endif
    // Per A/D buffer: the item's group, visit, CSR entry (-1: dense; -2:
    // residual, none in this warp's half) and this row's scale.
    int fgl0 = 0, fv0 = 0, fe0 = -2, fgl1 = 0, fv1 = 0, fe1 = -2;
    float fs0 = 0.0f, fs1 = 0.0f;
    int kis = 0, kdr = 0;  // items issued, items drained by this warpgroup

    // 64 bytes of this row's codes (K-steps jstride apart) -> E4M3 (q + 8) * 2^-9
    // in A buffer columns a_col .. a_col + 31: word t -> columns 2t (even
    // codes), 2t + 1 (odd codes).
    auto convert_row = [&](const uint8_t* src, int jstride, uint32_t a_col) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint4 pk0 = *reinterpret_cast<const uint4*>(src + (2 * hh) * jstride);
        const uint4 pk1 = *reinterpret_cast<const uint4*>(src + (2 * hh + 1) * jstride);
        uint32_t ev[16];
        unpack_u4(pk0.x, ev[0], ev[1]);
        unpack_u4(pk0.y, ev[2], ev[3]);
        unpack_u4(pk0.z, ev[4], ev[5]);
        unpack_u4(pk0.w, ev[6], ev[7]);
        unpack_u4(pk1.x, ev[8], ev[9]);
        unpack_u4(pk1.y, ev[10], ev[11]);
        unpack_u4(pk1.z, ev[12], ev[13]);
        unpack_u4(pk1.w, ev[14], ev[15]);
        tmem_st16(a_col + 16 * hh, ev);
      }
    };
    // The converted A of item n is in tensor memory: the last of the
    // warpgroup's four warps to store its part issues the item's four K=32
    // MMAs (the counter of buffer b counts every use: the (n/2)-th use is
    // complete at 4 (n/2 + 1)), so no warp waits for another here.
    auto issue = [&](int n, int gl) -> bool {
      const int b = n & 1;
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && atom_add_acq_rel(&ctl.a_cnt[w][b], 1u) + 1u == 4u * static_cast<uint32_t>((n >> 1) + 1)) {
        tc_fence_after();
        const uint32_t b_addr = bt + gl * (TN * 128);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          tc_mma_ts(colD + kDCh * TN * b + TN * (j % kDCh), colA + 32 * b + 8 * j, sw128_desc(b_addr + 32 * j), kIdesc,
                    j >= kDCh);
        tc_commit(&ctl.d_ready[w][b]);
      }
      return true;
    };
    // Item n's MMAs are complete: acc += 2^9 sx * (s * (D - c)) for this row
    // (or, as a test hook, store the dots).
    auto retire = [&](int n) -> bool {
      const int b = n & 1;
      MQ_PT();
      if (!mbar_wait(&ctl.d_ready[w][b], (n >> 1) & 1, abort_flag, tmo, p.err)) return false;
      MQ_PA(5);
      MQ_PT();
      tc_fence_after();
      const int gl = b ? fgl1 : fgl0, e = b ? fe1 : fe0, vv = b ? fv1 : fv0;
      const float s = b ? fs1 : fs0;
      if (e != -2) {  // warp-uniform
        const float4* sx4 = reinterpret_cast<const float4*>(sxf + gl * TN);
        const float4* c4 = reinterpret_cast<const float4*>(cfv + gl * TN);
        const uint64_t s2 = f2pack(s, s), m1 = f2pack(-1.0f, -1.0f);
#pragma unroll
        for (int cc = 0; cc < TN / 16; ++cc) {
          uint32_t dv[16];
          tmem_ld16(colD + kDCh * TN * b + 16 * cc + lane_base, dv);
          if (kDCh == 2) {
            uint32_t dw[16];
            tmem_ld16(colD + kDCh * TN * b + TN + 16 * cc + lane_base, dw);
            tc_wait_ld();
#pragma unroll
            for (int t = 0; t < 16; ++t) dv[t] = __float_as_uint(__uint_as_float(dv[t]) + __uint_as_float(dw[t]));
          } else {
            tc_wait_ld();
          }
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const float4 sv = sx4[cc * 4 + j4], cv = c4[cc * 4 + j4];  // tokens 16cc + 4j4 .. +3
            if (kDebug) {
              const float cvv[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int m = 16 * cc + 4 * j4 + t;
                if (m < p.M) {
                  const int32_t dd = static_cast<int32_t>((__uint_as_float(dv[4 * j4 + t]) - cvv[t]) * 512.0f);
                  if (e < 0)
                    p.dots_w[(static_cast<int64_t>(m) * p.N + tile_of(vv) * kTileN + r) * G + gs + gl] = dd;
                  else
                    p.dots_r[(static_cast<int64_t>(m) * p.nnzb + e) * 64 + (r & 63)] = dd;
                }
              }
            } else {
              // 2^-9 times the dot of q with x: the measured dot minus the offset term, exact
              const uint64_t d0 = f2fma(f2pack(cv.x, cv.y), m1,
                                        f2pack(__uint_as_float(dv[4 * j4]), __uint_as_float(dv[4 * j4 + 1])));
              const uint64_t d1 = f2fma(f2pack(cv.z, cv.w), m1,
                                        f2pack(__uint_as_float(dv[4 * j4 + 2]), __uint_as_float(dv[4 * j4 + 3])));
              acc[cc * 8 + 2 * j4] = f2fma(f2pack(sv.x, sv.y), f2mul(s2, d0), acc[cc * 8 + 2 * j4]);
              acc[cc * 8 + 2 * j4 + 1] = f2fma(f2pack(sv.z, sv.w), f2mul(s2, d1), acc[cc * 8 + 2 * j4 + 1]);
            }
          }
        }
      }
      tc_fence_before();  // the loads precede the buffer's reuse
      MQ_PA(6);
      return true;
    };
    // End of visit vv: add this warpgroup's partial into the CTA's row-major
    // buffer, warpgroup 0 first, then 1, 2, 3.
    auto finish_visit = [&](int vv) -> bool {
      bool passed;
      if (w == 0)  // every owner has consumed the previous tile's push out of this buffer
        passed = vv == 0 || mbar_wait_cluster(&ctl.rx_free, (vv - 1) & 1, abort_flag, tmo, p.err);
      else
        passed = mbar_wait(&ctl.chain[w - 1], vv & 1, abort_flag, tmo, p.err);
      if (!passed) return false;
      const bool direct = CS == 1 && !kDebug && w + 1 == kSlots;  // the last warpgroup stores Y
      const int64_t n = tile_of(vv) * kTileN + r;
      float4* row = reinterpret_cast<float4*>(rb + r * TN);
#pragma unroll
      for (int k4 = 0; k4 < TN / 4; ++k4) {
        float4 a;
        f2unpack(acc[2 * k4], a.x, a.y);
        f2unpack(acc[2 * k4 + 1], a.z, a.w);
        if (w != 0) {
          const float4 o = row[k4];
          a = make_float4(o.x + a.x, o.y + a.y, o.z + a.z, o.w + a.w);
        }
        if (direct) {
          const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (4 * k4 + t < p.M) store_y(p, 4 * k4 + t, n, av[t]);
        } else {
          row[k4] = a;
        }
        acc[2 * k4] = acc[2 * k4 + 1] = 0ull;
      }
      // the buffer is pushed by bulk copies (the async proxy): order these
      // generic writes before them
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (w + 1 < kSlots)
          mbar_arrive(&ctl.chain[w]);
        else if (!direct)
          mbar_arrive(&ctl.rb_done);
        else if (vv + 1 < nvis)
          mbar_arrive(&ctl.rx_free);  // this warp's rows of the buffer are read
      }
      if (lane == 0 && vv == 0) MQ_DTRACE(13 + warp);
      return true;
    };

    bool map_seen = false;
    int cur_v = 0;
    // stage i = w, w + 4, ..: group gl of visit v, in slot st whose fill parity is ph
    int v = w / ns, gl = w - (w / ns) * ns, st = w, ph = 0;
    for (int i = w; ok && i < total; i += kSlots) {
      if (v != cur_v) {  // a new tile: drain what is in flight, then close the finished visits
        while (ok && kdr < kis) ok = retire(kdr++);
        while (ok && cur_v < v) ok = finish_visit(cur_v++);
        if (!ok) break;
      }
      // dense item
      if (kis - kdr >= 2 && !(ok = retire(kdr++))) break;
      MQ_PT();
      if (!(ok = mbar_wait(&ctl.full[st], ph, abort_flag, tmo, p.err))) break;
      MQ_PA(1);
      MQ_PT();
      {
        const uint8_t* rec = stages + st * kStageBytes;
        const float s = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(rec + kWRecScales + 2 * r)));
        convert_row(rec + r * 16, 2048, colA + 32 * (kis & 1) + lane_base);
        if (kis & 1) fgl1 = gl, fv1 = v, fe1 = -1, fs1 = s;
        else fgl0 = gl, fv0 = v, fe0 = -1, fs0 = s;
      }
      ok = issue(kis++, gl);
      if (lane == 0) mbar_arrive(&ctl.empty[st]);  // this warp's reads of the stage are done
      MQ_PA(2);
      if (!ok) break;
      // residual item, if the block list has a block in either half here
      if (!map_seen) {
        if (!(ok = mbar_wait(&ctl.map_ready, 0, abort_flag, tmo, p.err))) break;
        map_seen = true;
      }
      const int e0 = ctl.map[v][gl][0], e1 = ctl.map[v][gl][1];
      if (e0 >= 0 || e1 >= 0) {
        if (kis - kdr >= 2 && !(ok = retire(kdr++))) break;
        const int e = half ? e1 : e0;
        float sr = 0.0f;
        if (e >= 0) {
          const int c = ctl.rpos[v][gl][half], slot = c % kRSlots;
          MQ_PT();
          if (!(ok = mbar_wait(&ctl.r_full[slot], (c / kRSlots) & 1, abort_flag, tmo, p.err))) break;
          MQ_PA(3);
          MQ_PT();
          const uint8_t* rrec = rring + slot * kRRecBytes;
          sr = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(rrec + kRRecScales + 2 * (r & 63))));
          convert_row(rrec + (r & 63) * 16, 1024, colA + 32 * (kis & 1) + lane_base);
          MQ_PA(4);
        }
        if (kis & 1) fgl1 = gl, fv1 = v, fe1 = e >= 0 ? e : -2, fs1 = sr;
        else fgl0 = gl, fv0 = v, fe0 = e >= 0 ? e : -2, fs0 = sr;
        ok = issue(kis++, gl);
        if (lane == 0) {  // each warp releases every ring slot of this group once
          if (e0 >= 0) mbar_arrive(&ctl.r_empty[ctl.rpos[v][gl][0] % kRSlots]);
          if (e1 >= 0) mbar_arrive(&ctl.r_empty[ctl.rpos[v][gl][1] % kRSlots]);
        }
        if (!ok) break;
      }
      for (gl += kSlots; gl >= ns; gl -= ns) ++v;
      if ((st += kSlots) >= NS) st -= NS, ph ^= 1;
    }
    while (ok && kdr < kis) ok = retire(kdr++);
    while (ok && cur_v < nvis) ok = finish_visit(cur_v++);
    // the last tile's owned rows, with the epilogue warps (several CTAs per cluster)
    if (ok && CS > 1 && !kDebug && mbar_wait(&ctl.rx_full, (nvis - 1) & 1, abort_flag, tmo, p.err))
      store_owned(rx, CS, tile_of(nvis - 1), kEpiThreads + threadIdx.x, kLastStorers);
#ifdef MQ_DEC_TRACE
    prof_[8] = kis;
    if (lane == 0 && warp < 4) mq_dec_trace_prof(warp, prof_, 9);
#endif
   }

  } else {
    // ---------------- epilogue: push partial rows to their owners, sum the owned rows, store Y ----------------
    const int et = threadIdx.x - 32 * kWarpEpi0;  // 0 .. kEpiThreads-1
#ifdef MQ_DEC_TRACE
    long long prof_[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0}, pt_ = 0;
#endif
    const uint32_t chunk = static_cast<uint32_t>(R * TN * 4);  // one owner's rows of one partial
    pdl_wait();  // Y may still be in use by the preceding kernel
    int nsync = 0;
    bool ok = true;
    // (one CTA per cluster: the last compute set has stored Y)
    for (int v = 0; ok && v < nvis && !(CS == 1 && !kDebug); ++v) {
      const int64_t tile = tile_of(v);
      if (et == 0 && CS > 1) mbar_arrive_expect_tx(&ctl.rx_full, CS * chunk);
      if (!mbar_wait(&ctl.rb_done, v & 1, abort_flag, tmo, p.err)) { ok = false; break; }
      if (et == 0 && v < 2) MQ_DTRACE(45 + v);
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
      if (et == 0 && v < 2) MQ_DTRACE(47 + v);
      if (!kDebug) {
        MQ_PT();
        if (v + 1 == nvis && CS > 1)  // the compute warps are done and help
          store_owned(src, nsrc, tile, et, kLastStorers);
        else
          store_owned(src, nsrc, tile, et, kEpiThreads);
        MQ_PA(0);
      }
      if (et == 0 && v < 2) MQ_DTRACE(53 + v);
      __syncwarp();
      if ((et & 31) == 0) mbar_arrive(&ctl.epi_bar);  // every epilogue warp has read the received rows
      if (!mbar_wait(&ctl.epi_bar, nsync & 1, abort_flag, tmo, p.err)) { ok = false; break; }
      ++nsync;
      if (et == 0 && v < 2) MQ_DTRACE(49 + v);
#ifdef MQ_DEC_TRACE
      if (et == 0 && v == 0) mq_dec_trace_prof(5, prof_, 9);
#endif
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

  // Every role is done: warps that finish early wait suspended on a barrier
  // rather than in a hardware barrier, then all threads meet.
  __syncwarp();
  if (lane == 0) mbar_arrive(&ctl.exit_bar);
  mbar_wait(&ctl.exit_bar, 0, abort_flag, tmo, p.err);
  __syncthreads();
  if (threadIdx.x == 0) MQ_DTRACE(51);
  if (*abort_flag) {
    // A wait gave up: bulk copies may still be landing in this CTA's shared
    // memory.  They finish within microseconds; give them 200 us.
    if (threadIdx.x == 0) {
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 200000ull) {
      }
    }
    __syncthreads();
  }
  if (kTC && warp == 0) {  // every tensor-memory access of the CTA is complete
    tc_fence_after();
    tmem_dealloc(ctl.tmem_base, kTmemCols);
  }
  // Every CTA has received all its rows, so every push out of this CTA's
  // shared memory has been read (no data passes through this barrier).
  if (CS > 1) cluster_sync_relaxed();
  if (threadIdx.x == 0) MQ_DTRACE(52);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

struct DecPlan {
  bool tc;  // tensor-memory variant
  int tn, cs, nstages, nclusters;
  uint32_t oSX, oRB, oRX, oR, oStage, smem;
};

template <int TN, bool kDebug, bool kTC>
static const void* kernel_ptr() {
  return reinterpret_cast<const void*>(&w4a4_decode_kernel<TN, kDebug, kTC>);
}

// Co-resident clusters of `cs` CTAs of this kernel (one CTA per SM), per device.
static int max_clusters(int cs, bool tc) {
  static std::mutex mu;
  static int cache[64][2][kMaxCS + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  int& slot = cache[dev][tc ? 1 : 0][cs];
  if (slot != 0) return slot;
  const void* kern = tc ? kernel_ptr<32, false, true>() : kernel_ptr<32, false, false>();
  const int threads = tc ? Roles<true>::kThreads : Roles<false>::kThreads;
  const int smem = kSmemLimit - kCtlBytes;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cs * 256), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
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
  slot = n > 0 ? n : -1;
  return slot;
}

static uint32_t up1024(uint32_t b) { return (b + 1023u) / 1024u * 1024u; }

// Which variant runs: the tensor-memory one above 16 tokens (where the
// warp-level MMAs of a 32-token tile cost more than the tensor-memory round
// trips), the warp-MMA one up to 16 (measured on GB300: faster on every
// Llama-3-8B layer shape at 4 and 16 tokens, slower at 32).
// MQ_DECODE_VARIANT = "warp" or "tc" forces one (benchmarking and tests).
static bool decode_use_tc(int64_t M) {
  const char* v = getenv("MQ_DECODE_VARIANT");
  if (v && strcmp(v, "warp") == 0) return false;
  if (v && strcmp(v, "tc") == 0) return true;
  return M > 16;
}

// Pick the cluster size: the makespan of a CTA is (visits x slice) groups
// plus a per-visit reduction; the slice's activation tiles must fit.
static bool decode_plan(int64_t M, int64_t N, int64_t K, DecPlan* out) {
  if (M > 32) return false;
  const bool tc = decode_use_tc(M);
  const int tn = M <= 8 && !tc ? 8 : M <= 16 ? 16 : 32;
  const int sets = tc ? Roles<true>::kSets : Roles<false>::kSets;
  const int G = static_cast<int>(K / kGroup), tiles = static_cast<int>(N / kTileN);
  double best = 1e30;
  bool found = false;
  for (int cs = 1; cs <= kMaxCS; cs *= 2) {
    if (cs > G) break;
    const int ns = (G + cs - 1) / cs;
    const uint32_t bbytes = static_cast<uint32_t>(ns) * tn * 128;
    if (ns > kMaxSlice || bbytes > static_cast<uint32_t>(kMaxBBytes)) continue;
    DecPlan pl;
    pl.tc = tc;
    pl.tn = tn;
    pl.cs = cs;
    pl.oSX = bbytes;
    pl.oRB = up1024(pl.oSX + kMaxSlice * tn * 8);  // scales and offset terms
    pl.oRX = pl.oRB + tn * kTileN * 4;
    pl.oR = pl.oRX + (cs > 1 ? tn * kTileN * 4 : 0);
    pl.oStage = up1024(pl.oR + kRSlots * kRRecBytes);
    const int avail = kSmemLimit - kCtlBytes - 1024 - static_cast<int>(pl.oStage);
    pl.nstages = std::min(kMaxStages, avail / kStageBytes);
    if (pl.nstages < sets + 2) continue;  // every set busy, two more in flight
    pl.smem = pl.oStage + pl.nstages * kStageBytes + 1024;
    const int ncl = max_clusters(cs, tc);
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

template <int TN, bool kDebug, bool kTC>
static mq_status launch_decode(const DecParams& dp, const DecPlan& pl, cudaStream_t stream) {
  const void* kern = kernel_ptr<TN, kDebug, kTC>();
  static bool smem_set[64];  // per device, per instantiation
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return launch_status("decode gemm: device");
  if (!smem_set[dev]) {
    const int want = kSmemLimit - kCtlBytes;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, want) != cudaSuccess)
      return launch_status("decode gemm: smem attribute");
    smem_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.nclusters * pl.cs), 1, 1);
  cfg.blockDim = dim3(Roles<kTC>::kThreads, 1, 1);
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
  if (cudaLaunchKernelEx(&cfg, w4a4_decode_kernel<TN, kDebug, kTC>, dp) != cudaSuccess)
    return launch_status("decode gemm launch");
  return launch_status("decode gemm");
}

}  // namespace

// The kernel choice for (M, N, K) on the current device: {1 (warp-MMA
// variant) or 2 (tensor-memory variant), tokens per tile, cluster size,
// clusters, stages} for the decode kernel, else zeros.
bool zipper_plan_info(int64_t M, int64_t tiles, int64_t K, int32_t* form, int32_t* tn, int32_t* ctas, int32_t* stages);

mq_status gemm_plan_info(int64_t M, int64_t N, int64_t K, int32_t* info) {
  DecPlan pl;
  for (int i = 0; i < 5; ++i) info[i] = 0;
  const char* impl = getenv("MQ_DECODE_IMPL");
  if (!(impl && strcmp(impl, "cluster") == 0)) {
    if (zipper_plan_info(M, N / kTileN, K, &info[0], &info[1], &info[3], &info[4])) info[2] = 1;
    return MQ_OK;
  }
  if (decode_plan(M, N, K, &pl)) {
    info[0] = pl.tc ? 2 : 1;
    info[1] = pl.tn;
    info[2] = pl.cs;
    info[3] = pl.nclusters;
    info[4] = pl.nstages;
  }
  return MQ_OK;
}

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
  if (pl.tc) {
    if (pl.tn == 16)
      return dbg ? launch_decode<16, true, true>(dp, pl, stream) : launch_decode<16, false, true>(dp, pl, stream);
    return dbg ? launch_decode<32, true, true>(dp, pl, stream) : launch_decode<32, false, true>(dp, pl, stream);
  }
  if (pl.tn == 8)
    return dbg ? launch_decode<8, true, false>(dp, pl, stream) : launch_decode<8, false, false>(dp, pl, stream);
  if (pl.tn == 16)
    return dbg ? launch_decode<16, true, false>(dp, pl, stream) : launch_decode<16, false, false>(dp, pl, stream);
  return dbg ? launch_decode<32, true, false>(dp, pl, stream) : launch_decode<32, false, false>(dp, pl, stream);
}

}  // namespace mq
