// The fused W4A4 + block-sparse 4-bit residual GEMM for decode batches (up to
// 32 tokens): the ZipperEngine of the MosaicQuant summary (Metodologia 3) as a
// persistent, stream-K, tensor-memory kernel for sm_103a.  It computes
//
//   Y[m,n] = sum_g sx[m,g] * ( sw[n,g] * Dw[m,n,g] + sr[n,g] * Dr[m,n,g] )
//
// in one launch: the residual product of a selected 64x128 block runs on the
// same activation tile as the dense product of its group and both are
// reduce-added into the same fp32 accumulators.
//
// Work.  A "unit" is one 128-row weight tile x one 128-input group: one packed
// base record (8448 bytes) and, where the block list has a block in either
// 64-row half, one residual item more.  Units are ordered tile-major, over up to
// four weight matrices that share the activations (a grouped launch), and the
// CTAs (one per SM) take equal contiguous ranges of them (stream-K), so every SM
// streams the same number of weight bytes whatever the tile count.
//
// Numbers.  INT4 codes run on the tensor cores as E4M3 bytes (sm_103a has no
// integer tcgen05 kind):
//   * weights: a byte 0x00..0x0F read as E4M3 is exactly b * 2^-9, so the
//     nibble u = q + 8 (q XOR 8) moved into a byte is u * 2^-9: a mask and a
//     shift per 8 codes.  The MMA measures 2^-9 (D + 8 sum_k qx); the drain
//     subtracts the exact activation term and folds 2^9 into the activation
//     scale.  Every partial sum is a multiple of 2^-9 below 2^14: exact in fp32.
//   * activations: E4M3 bytes holding the integer codes exactly, in a
//     128-byte-swizzled K-major tile (the MMA's B operand), with K permuted
//     inside each 8-code word (even codes, then odd) as the weight unpack
//     leaves them.
//
// The launch, per CTA (16 warps):
//   prologue   every group's activation image (B tile, 2^9 sx, offset terms)
//              is built once per launch by one CTA (group g by CTA g mod P),
//              from the packed activations or, in the fused form, straight from
//              X (the quantizer runs here), written to the workspace and
//              published with a per-group flag;
//   warp 0     producer: bulk copies of each unit's base record and its
//              group's activation image into a ring of shared-memory stages;
//   warp 1     reads the block list of the CTA's tiles once into a residual map,
//              then streams the residual records into a ring of their own;
//   warp 2     issues each item's four K=32 tcgen05 MMAs (A = unpacked weights
//              in tensor memory, B = the stage's activation tile) into a ring
//              of 8 tensor-memory accumulators;
//   warps 4-11 unpack: lane quarter q (warp % 4) owns rows 32q..32q+31, the two
//              warpgroups split each item's four K-steps; codes go from the
//              stage to registers to tensor memory (no shared-memory round trip);
//   warps 12-15 drain: per item, load the exact dots from tensor memory and
//              reduce-add sx * (s * D) into fp32 registers; at a tile's end,
//              store Y, or hand the CTA's piece of a tile cut by a range
//              boundary to the workspace, where the last CTA to arrive sums the
//              pieces in CTA order (deterministic, no floating-point atomics).
// Every wait is bounded: a wait that runs out sets the device error word,
// raises the CTA's abort flag, and every role winds down.
#include "mq_internal.cuh"

#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

// Timeline probes for profiling builds: compiled out unless MQ_ZTRACE is
// defined, in which case stamps go to a buffer the host sets: ZT(slot) the
// global timer, ZC(slot) the SM cycle counter.
#ifdef MQ_ZTRACE
__device__ unsigned long long* g_zt_buf;
__device__ __forceinline__ void zt_put(int slot, unsigned long long v) {
  if (g_zt_buf && slot < 256) g_zt_buf[blockIdx.x * 256 + slot] = v;
}
__device__ __forceinline__ unsigned long long zt_gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define ZT_INIT unsigned long long* const zt_b = g_zt_buf ? g_zt_buf + blockIdx.x * 256 : nullptr
#define ZT(slot)                      \
  do {                                \
    if (zt_b) zt_b[slot] = zt_gtime(); \
  } while (0)
#define ZC(slot)                                                             \
  do {                                                                       \
    if (zt_b) zt_b[slot] = static_cast<unsigned long long>(clock64());       \
  } while (0)
extern "C" int mq_zt_set_buffer(void* p) {
  return cudaMemcpyToSymbol(g_zt_buf, &p, sizeof(p)) == cudaSuccess ? 0 : 1;
}
#else
#define ZT_INIT
#define ZT(slot) ((void)0)
#define ZC(slot) ((void)0)
#endif

namespace mq {
namespace {

constexpr int kNB = 8;             // items in flight: A/D buffer pairs in tensor memory
constexpr int kUS = 4;             // units per shared-memory stage (one bulk copy of their base records)
constexpr int kMinUnits = 8;       // units per CTA at least (bounds the pieces a tile is cut into)
constexpr int kRS = 8;             // residual-record ring slots
constexpr int kMaxUnits = 128;     // units per CTA (size of the residual map)
constexpr int kMaxStages = 8;
constexpr int kMaxMats = 4;
constexpr int kWarpProd = 0, kWarpRes = 1, kWarpMma = 2, kWarpConv0 = 4, kWarpDrain0 = 12;
constexpr int kConvWarps = 8, kDrainWarps = 4;
constexpr int kThreads = 32 * (kWarpDrain0 + kDrainWarps);
constexpr int kTmemCols = 512;
constexpr int kSmemLimit = 227 * 1024;

struct ZMat {
  const uint8_t* wpk;
  const int32_t* row_ptr;
  const int32_t* col_idx;
  const uint8_t* rpk;
  void* y;
  int64_t ldy;  // elements between rows of Y
  int tile0;    // first tile of this matrix in the launch's tile order
  int nnzb;
};

struct ZParams {
  ZMat mat[kMaxMats];
  int nmat;
  const uint8_t* xq;   // [G][Mp][64] packed activations (prologue from codes)
  const uint16_t* xs;  // [G][Mp] fp16
  const uint16_t* x;   // [M][ldx] fp16 / bf16 (prologue quantizes)
  int64_t ldx;
  int x_bf16;
  uint8_t* xq_out;     // optional: the quantized activations, as mq_quantize_act writes them
  uint16_t* xs_out;
  int M, Mp, G, tiles, ctas, nstages, stage_bytes;
  int64_t units;
  int y_f32;
  int raw;          // column form: the stages take X rows (else packed codes and scales)
  int cluster;      // warp-MMA form: CTAs per cluster (one tile per cluster, pieces through DSMEM), or 0
  int rx_off;       // its byte offset of the received pieces in dynamic shared memory
  int32_t* dots_w;  // test hook (one matrix): raw group dots instead of Y
  int32_t* dots_r;
  const uint8_t* act;  // workspace: [G] activation images (written by the image kernel)
  int32_t* tcount;     // [ctas] pieces that have arrived of the cut tile whose first unit is CTA c's
  float* part;         // [ctas][2][TN][128] stream-K pieces
  uint64_t timeout_ns;
  uint32_t* err;
};

struct __align__(8) ZCtl {
  uint64_t full[kMaxStages];   // stage landed: producer arrival + bytes
  uint64_t empty[kMaxStages];  // 8 unpack warps read the codes, 4 drain warps the scales
  uint64_t r_full[kRS];
  uint64_t r_empty[kRS];       // the 4 unpack and 2 drain warps of the record's half
  uint64_t a_full[kNB];        // 8 unpack warps stored item's A
  uint64_t d_full[kNB];        // the item's MMAs completed (commit)
  uint64_t d_empty[kNB];       // 4 drain warps loaded the item's D
  uint64_t map_ready;
  uint64_t exit_bar;
  uint64_t red_bar;            // stream-K pieces copied in for a deferred tile
  uint64_t drain_bar;          // bounded barrier of the 4 drain warps
  uint64_t tmem_ready;         // the tensor-memory allocation is published
  int32_t map[kMaxUnits][2];   // CSR entry of the residual block of (unit, half), or -1
  int32_t rpos[kMaxUnits][2];  // its position in the residual ring order
  uint32_t tmem_base;
  int abort_flag;
  int ndeferred;
  int deferred[2];             // cut tiles whose count this CTA completed
};

// Bytes of one activation image in the workspace and in a stage: the B tile
// (TN rows x 128 bytes), 2^9 sx and the offset terms (TN fp32 each), padded to
// a multiple of 1024 so every B tile keeps the 128-byte swizzle's alignment.
__host__ __device__ constexpr int act_rec_bytes(int tn) { return (tn * 128 + tn * 8 + 1023) / 1024 * 1024; }

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int32_t* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ float ld_shared_f32(const float* p) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
  return v;
}
__device__ __forceinline__ void st_shared_f32(float* p, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "f"(v)
               : "memory");
}
__device__ __forceinline__ void st_global_f32(float* p, float v) {
  asm volatile("st.global.cg.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void st_global_b16(void* p, unsigned short v) {
  asm volatile("st.global.b16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_gpu(int32_t* p, int v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Self-checks, compiled in with MQ_ZCHECK only: a failed bounds check records
// bit 8 + site in the device error word and skips the access; a wait that gave
// up records bit 24 + site.
#ifdef MQ_ZCHECK
__device__ __forceinline__ bool zcheck(bool ok, int bit, uint32_t* err) {
  if (!ok) atomicOr(err, 1u << bit);
  return ok;
}
#define ZOK(cond, site) zcheck((cond), 8 + (site), p.err)
#define ZW(ok, site) zcheck((ok), 24 + (site), p.err)
#else
#define ZOK(cond, site) true
#define ZW(ok, site) (ok)
#endif
// --- thread-block clusters -----------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster, with release / acquire ordering.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// This CTA's shared-memory address `saddr` as seen in cluster peer `rank`.
__device__ __forceinline__ uint32_t mapa_peer(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Bulk copy of this CTA's shared memory into a cluster peer's; completion is
// counted in bytes on the peer's mbarrier.  Addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_s2peer(uint32_t dst_cluster, const void* src, uint32_t bytes,
                                            uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(smem_u32(src)), "r"(bytes), "r"(bar_cluster)
      : "memory");
}
// This thread's bulk copies have read their sources.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}
// mbar_wait with cluster-scope acquire (for phases completed by cluster peers' copies).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                  uint64_t timeout_ns, uint32_t* err_word) {
  uint64_t t0 = 0;
  for (uint32_t n = 0;; ++n) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((n & 63u) == 63u) {
      if (*abort_flag) return false;
      const uint64_t now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > timeout_ns) {
        atomicOr(err_word, kDevErrTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// Bounded wait with back-off, for roles whose waits are long (producers).
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                uint64_t timeout_ns, uint32_t* err_word) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t n = 1;; ++n) {
    __nanosleep(32);
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63u) == 0) {
      if (*abort_flag) return false;
      const uint64_t now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > timeout_ns) {
        atomicOr(err_word, kDevErrTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}
// Bounded wait until a shared-memory counter (advanced by another warp of the CTA) exceeds `target`.
__device__ __forceinline__ bool count_wait(volatile int* v, int target, volatile int* abort_flag, uint64_t timeout_ns,
                                           uint32_t* err_word) {
  if (*v > target) return true;
  uint64_t t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if (*v > target) return true;
    if ((n & 63u) == 0) {
      if (*abort_flag) return false;
      const uint64_t now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > timeout_ns) {
        atomicOr(err_word, kDevErrTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}
// Bounded wait for a flag in global memory (written by another CTA) to become nonzero.
__device__ __forceinline__ bool flag_wait(const int32_t* f, volatile int* abort_flag, uint64_t timeout_ns,
                                          uint32_t* err_word) {
  if (ld_acquire_gpu(f) != 0) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    __nanosleep(100);
    if (ld_acquire_gpu(f) != 0) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > timeout_ns) {
      atomicOr(err_word, kDevErrTimeout);
      *abort_flag = 1;
      return false;
    }
  }
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

// Shared-memory matrix descriptor of a K-major operand in 128-byte-swizzled
// rows (8-row atoms 1024 bytes apart).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

// Load MLD consecutive 32-bit columns of this thread's tensor-memory lane.
template <int MLD>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&v)[MLD]) {
  if constexpr (MLD == 4) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                 : "r"(taddr)
                 : "memory");
  } else if constexpr (MLD == 8) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
  } else if constexpr (MLD == 16) {
    tmem_ld16(taddr, v);
  } else {
    tmem_ld32(taddr, v);
  }
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

// Eight weight codes (two's complement nibbles, element i in bits 4i..4i+3)
// -> two words of four E4M3 bytes holding (q + 8) * 2^-9 exactly: the even
// elements 0, 2, 4, 6 in `ev`, the odd ones in `od`.
__device__ __forceinline__ void unpack_u4(uint32_t p, uint32_t& ev, uint32_t& od) {
  const uint32_t u = p ^ 0x88888888u;
  ev = u & 0x0F0F0F0Fu;
  od = (u >> 4) & 0x0F0F0F0Fu;
}

// Sum of the eight signed codes of a word of packed activations.
__device__ __forceinline__ int nibble_sum8(uint32_t p) {
  const uint32_t u = p ^ 0x88888888u;  // q + 8 in [1, 15]
  const uint32_t b = (u & 0x0F0F0F0Fu) + ((u >> 4) & 0x0F0F0F0Fu);
  return static_cast<int>((b * 0x01010101u) >> 24) - 64;
}

// Byte offset of codes 8t..8t+7 (word t of 16) of token row m inside the
// activation image's 128-byte-swizzled K-major tile.
__device__ __forceinline__ int act_word_offset(int m, int t) {
  return (m >> 3) * 1024 + (m & 7) * 128 + (((t >> 1) ^ (m & 7)) << 4) + ((t & 1) << 3);
}

// Activation quantization (the quantizer's rule, bit-exact with mq_quantize_act):
// s = fp16_RNE(amax / 7) saturated, q = clamp(RNE(x / s), -7, 7) in IEEE fp32.
__device__ __forceinline__ uint16_t act_scale_bits(float amax) {
  const __half h = __float2half_rn(__fdiv_rn(amax, 7.0f));
  uint16_t b = __half_as_ushort(h);
  if ((b & 0x7FFFu) == 0x7C00u) b = (b & 0x8000u) | 0x7BFFu;
  return b;
}
__device__ __forceinline__ int act_code(float v, float s) {
  if (s == 0.0f) return 0;
  float t = rintf(__fdiv_rn(v, s));
  t = fminf(fmaxf(t, -7.0f), 7.0f);
  return static_cast<int>(t);
}
// E4M3 byte of an integer code |q| <= 7.
__device__ __forceinline__ uint32_t e4m3_of_code(int q) {
  const uint32_t a = static_cast<uint32_t>(q < 0 ? -q : q);
  const uint32_t mag = prmt(0x44403800u, 0x4E4C4A48u, a);  // bytes of 0,1,2,3 | 4,5,6,7
  return (mag & 0xFFu) | (q < 0 ? 0x80u : 0u);
}
__device__ __forceinline__ float act_value(const uint16_t* x, int64_t i, bool bf16) {
  const uint16_t b = x[i];
  return bf16 ? __uint_as_float(static_cast<uint32_t>(b) << 16) : __half2float(__ushort_as_half(b));
}

// first unit of CTA c, and the CTA that owns unit u (balanced contiguous ranges)
__device__ __forceinline__ int64_t first_unit(int64_t c, int64_t U, int64_t P) { return c * U / P; }
__device__ __forceinline__ int64_t owner_of(int64_t u, int64_t U, int64_t P) { return ((u + 1) * P - 1) / U; }
// The same in 32-bit arithmetic, for the warp-MMA form: its planner keeps units per CTA at most kMaxUnits
// and CTAs at most kWsZeroBytes / 4, so c * U and (u + 1) * P stay below 2^31.
__device__ __forceinline__ uint32_t first_unit32(uint32_t c, uint32_t U, uint32_t P) { return c * U / P; }
__device__ __forceinline__ uint32_t owner_of32(uint32_t u, uint32_t U, uint32_t P) { return ((u + 1) * P - 1) / U; }

__device__ __forceinline__ int mat_end_tile(const ZParams& p, int t);
__device__ __forceinline__ int mat_of_tile(const ZParams& p, int t) {
  int mi = 0;
#pragma unroll
  for (int i = 1; i < kMaxMats; ++i)
    if (i < p.nmat && t >= p.mat[i].tile0) mi = i;
  return mi;
}

__device__ __forceinline__ int mat_end_tile(const ZParams& p, int t) {  // one past the matrix's last tile
  const int mi = mat_of_tile(p, t);
  return mi + 1 < p.nmat ? p.mat[mi + 1].tile0 : p.tiles;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

// TN: tokens of the MMA tile (16 or 32); MLD: token columns the drain reads
// (4, 8, 16 or 32); kDebug: write raw group dots.
template <int TN, int MLD, bool kDebug>
__global__ void __launch_bounds__(kThreads, 1) zipper_decode_kernel(const ZParams p) {
  static_assert(MLD <= TN && TN % 16 == 0, "tile shape");
  constexpr int kArec = act_rec_bytes(TN);  // activation image: B tile, 2^9 sx, offset terms, padding
  constexpr int kAct = kUS * kArec;         // a stage: kUS activation images, then kUS base records
  constexpr uint32_t kIdesc =
      (1u << 4) | (static_cast<uint32_t>(TN >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
  extern __shared__ uint8_t smem_raw[];
  __shared__ ZCtl ctl;
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int S = p.nstages, SB = p.stage_bytes, G = p.G;
  uint8_t* stages = smem;                               // [S] stages, 1024-aligned
  uint8_t* rring = smem + static_cast<size_t>(S) * SB;  // [kRS] residual records
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t U = p.units, P = p.ctas, c = blockIdx.x;
  const int64_t u0 = first_unit(c, U, P), u1 = first_unit(c + 1, U, P);
  const int nu = static_cast<int>(u1 - u0);
  const int nstg = (nu + kUS - 1) / kUS;  // stages this CTA fills
  volatile int* abort_flag = &ctl.abort_flag;
  const uint64_t tmo = p.timeout_ns;
  ZT_INIT;

  if (threadIdx.x == 0) {
    ZT(0);
    ZC(6);
  }
  if (warp == 0) {
    for (int s = lane; s < S; s += 32) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], kConvWarps + kDrainWarps);
    }
    if (lane < kRS) {
      mbar_init(&ctl.r_full[lane], 1);
      mbar_init(&ctl.r_empty[lane], kConvWarps / 2 + kDrainWarps / 2);
    }
    if (lane < kNB) {
      mbar_init(&ctl.a_full[lane], kConvWarps);
      mbar_init(&ctl.d_full[lane], 1);
      mbar_init(&ctl.d_empty[lane], kDrainWarps);
    }
    if (lane == 8) mbar_init(&ctl.map_ready, 1);
    if (lane == 9) mbar_init(&ctl.exit_bar, kThreads / 32);
    if (lane == 10) mbar_init(&ctl.red_bar, 1);
    if (lane == 13) mbar_init(&ctl.drain_bar, kDrainWarps);
    if (lane == 14) mbar_init(&ctl.tmem_ready, 1);
    if (lane == 11) ctl.abort_flag = 0;
    if (lane == 12) ctl.ndeferred = 0;
    fence_mbar_init();
  }
  __syncthreads();  // barriers initialised
  if (threadIdx.x == 0) ZC(8);
  // The next kernel may start launching; it touches nothing this one uses
  // before its own dependency wait.
  pdl_trigger();
  // The tensor-memory allocation (by the MMA warp) is published through
  // tmem_ready, so the producers start streaming at once.
  auto tmem_wait = [&]() -> bool {
    const bool r = mbar_wait(&ctl.tmem_ready, 0, abort_flag, tmo, p.err);
    tc_fence_after();
    return r;
  };
  auto stage = [&](int s) { return stages + static_cast<size_t>(s) * SB; };
  auto wrec = [&](int64_t u) -> const uint8_t* {
    const int t = static_cast<int>(u / G), g = static_cast<int>(u - static_cast<int64_t>(t) * G);
    const ZMat& mt = p.mat[mat_of_tile(p, t)];
    return mt.wpk + (static_cast<int64_t>(t - mt.tile0) * G + g) * kWRecBytes;
  };
  // first unit after the matrix of unit u (records are contiguous inside one matrix)
  auto mat_end = [&](int64_t u) -> int64_t {
    const int mi = mat_of_tile(p, static_cast<int>(u / G));
    return static_cast<int64_t>(mi + 1 < p.nmat ? p.mat[mi + 1].tile0 : p.tiles) * G;
  };

  if (warp == kWarpProd) {
    // ---------------- producer: a stage = kUS units' base records and activation images ----------------
    // Bulk copies cost the copy engine a fixed time each, so a stage moves
    // its base records (contiguous within a matrix) in one copy and its
    // activation images (consecutive groups) in one more.
    auto stage_bytes = [&](int st) {
      const int n = min(kUS, nu - st * kUS);
      return static_cast<uint32_t>(n * (kWRecBytes + kArec));
    };
    auto issue_weights = [&](int st, int s) {
      int64_t ua = u0 + st * kUS;
      const int64_t ub = min(u1, ua + kUS), us = ua;
      while (ua < ub) {
        const int64_t e = min(ub, mat_end(ua));
        bulk_g2s(stage(s) + kAct + (ua - us) * kWRecBytes, wrec(ua), static_cast<uint32_t>((e - ua) * kWRecBytes),
                 &ctl.full[s]);
        ua = e;
      }
    };
    auto issue_act = [&](int st, int s) {
      int64_t ua = u0 + st * kUS;
      const int64_t ub = min(u1, ua + kUS), us = ua;
      while (ua < ub) {
        const int g = static_cast<int>(ua % G);
        const int64_t n = min(ub - ua, static_cast<int64_t>(G - g));
        bulk_g2s(stage(s) + (ua - us) * kArec, p.act + static_cast<int64_t>(g) * kArec,
                 static_cast<uint32_t>(n * kArec), &ctl.full[s]);
        ua += n;
      }
    };
    const int pre = min(S, nstg);
    // The first stages' base records are requested before the dependency wait:
    // the kernels that may run ahead of it (this library's, which ask for the
    // next launch early) never write packed weights.
    if (lane == 0) {
      for (int st = 0; st < pre; ++st) {
        mbar_arrive_expect_tx(&ctl.full[st], stage_bytes(st));
        issue_weights(st, st);
      }
    }
    pdl_wait();  // the activation images are the preceding kernel's output
    if (lane == 0) ZC(9);
    bool ok = true;
    if (lane == 0 && ok) {
      for (int st = 0; st < nstg; ++st) {
        const int s = st % S;
        if (st >= S) {
          if (!mbar_wait_sleep(&ctl.empty[s], ((st / S) - 1) & 1, abort_flag, tmo, p.err)) break;
          mbar_arrive_expect_tx(&ctl.full[s], stage_bytes(st));
          issue_weights(st, s);
        }
        issue_act(st, s);
        if (st < 16) ZC(16 + st);
      }
    }
  } else if (warp == kWarpRes) {
    // ---------------- residual map, then the residual records in order ----------------
    pdl_wait();
    for (int i = lane; i < nu * 2; i += 32) (&ctl.map[0][0])[i] = -1;
    __syncwarp();
    if (nu > 0) {
      const int t_lo = static_cast<int>(u0 / G), t_hi = static_cast<int>((u1 - 1) / G);
      for (int t = t_lo; t <= t_hi; ++t) {
        const ZMat& mt = p.mat[mat_of_tile(p, t)];
        if (mt.nnzb == 0) continue;
        const int64_t br = 2 * static_cast<int64_t>(t - mt.tile0);
        const int a0 = max(0, min(mt.nnzb, mt.row_ptr[br]));
        const int a1 = max(a0, min(mt.nnzb, mt.row_ptr[br + 1]));
        const int a2 = max(a1, min(mt.nnzb, mt.row_ptr[br + 2]));
        for (int e = a0 + lane; e < a2; e += 32) {
          const int g = mt.col_idx[e];
          if (g < 0 || g >= G) continue;
          const int64_t u = static_cast<int64_t>(t) * G + g;
          if (u >= u0 && u < u1) ctl.map[u - u0][e >= a1 ? 1 : 0] = e;
        }
      }
    }
    __syncwarp();
    {  // ring positions: residual records in (unit, half) order; lane l counts a chunk of it
      const int nf = nu * 2;
      const int chunk = (nf + 31) / 32, f0 = min(nf, lane * chunk), f1 = min(nf, f0 + chunk);
      int cnt = 0;
      for (int f = f0; f < f1; ++f) cnt += (&ctl.map[0][0])[f] >= 0;
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      int pos = incl - cnt;
      for (int f = f0; f < f1; ++f)
        if ((&ctl.map[0][0])[f] >= 0) (&ctl.rpos[0][0])[f] = pos++;
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&ctl.map_ready);
      ZC(11);
      for (int f = 0; f < nu * 2; ++f) {
        const int e = (&ctl.map[0][0])[f];
        if (e < 0) continue;
        const int cpos = (&ctl.rpos[0][0])[f], slot = cpos % kRS;
        if (cpos >= kRS && !mbar_wait_sleep(&ctl.r_empty[slot], ((cpos / kRS) - 1) & 1, abort_flag, tmo, p.err))
          break;
        const int t = static_cast<int>((u0 + f / 2) / G);
        const ZMat& mt = p.mat[mat_of_tile(p, t)];
        mbar_arrive_expect_tx(&ctl.r_full[slot], kRRecBytes);
        bulk_g2s(rring + slot * kRRecBytes, mt.rpk + static_cast<int64_t>(e) * kRRecBytes, kRRecBytes,
                 &ctl.r_full[slot]);
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------- MMA issue: four K=32 MMAs per item ----------------
    tmem_alloc(&ctl.tmem_base, kTmemCols);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl.tmem_ready);
    const uint32_t tmem = ctl.tmem_base;
    tc_fence_after();
    if (lane == 0 && mbar_wait(&ctl.map_ready, 0, abort_flag, tmo, p.err)) {
      int i = 0;
      bool ok = true;
      for (int ui = 0; ui < nu && ok; ++ui) {
        if (i < 16) ZC(64 + 8 * i + 7);
        const int st = ui / kUS, j = ui - st * kUS, s = st % S;
        const uint32_t bsm = smem_u32(stage(s) + j * kArec);
        const int nitems = (ctl.map[ui][0] >= 0 || ctl.map[ui][1] >= 0) ? 2 : 1;
        // the activation tile the MMAs read landed by bulk copy (long complete by now)
        if (j == 0 && !(ok = mbar_wait(&ctl.full[s], (st / S) & 1, abort_flag, tmo, p.err))) break;
        for (int it = 0; it < nitems; ++it, ++i) {
          const int b = i % kNB, k = i / kNB;
          if (i < 16) ZC(64 + 8 * i + 0);
          if (!(ok = mbar_wait(&ctl.a_full[b], k & 1, abort_flag, tmo, p.err))) break;
          if (i < 16) ZC(64 + 8 * i + 1);
          if (k > 0 && !(ok = mbar_wait(&ctl.d_empty[b], (k - 1) & 1, abort_flag, tmo, p.err))) break;
          if (i < 16) ZC(64 + 8 * i + 2);
          tc_fence_after();
          if (i < 16) ZC(64 + 8 * i + 3);
          const uint32_t a_col = tmem + 32 * b, d_col = tmem + 32 * kNB + TN * b;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
            tc_mma_ts(d_col, a_col + 8 * jj, sw128_desc(bsm + 32 * jj), kIdesc, jj > 0);
          if (i < 16) ZC(64 + 8 * i + 4);
          tc_commit(&ctl.d_full[b]);
          if (i < 16) ZC(64 + 8 * i + 5);
        }
      }
    }
    __syncwarp();
  } else if (warp >= kWarpConv0 && warp < kWarpDrain0) {
    // ---------------- unpack warps ----------------
    const int cw = warp - kWarpConv0, q = warp & 3, kh = cw >> 2;
    const int r = 32 * q + lane, half = q >> 1;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const int ct = cw * 32 + lane;  // 0..255
    bool ok = tmem_wait();
    const uint32_t tmem = ctl.tmem_base;
    // --- main loop: items in order ---
    ok = ok && mbar_wait(&ctl.map_ready, 0, abort_flag, tmo, p.err);
    int i = 0;
    for (int ui = 0; ui < nu && ok; ++ui) {
      const int st = ui / kUS, j = ui - st * kUS, s = st % S;
      {  // base item
        const int b = i % kNB, k = i / kNB;
        if (k > 0 && !(ok = mbar_wait(&ctl.d_full[b], (k - 1) & 1, abort_flag, tmo, p.err))) break;
        if (j == 0 && !(ok = mbar_wait(&ctl.full[s], (st / S) & 1, abort_flag, tmo, p.err))) break;
        if (ct == 0 && j == 0 && st < 16) ZC(32 + st);
        const uint8_t* src = stage(s) + kAct + j * kWRecBytes + (2 * kh) * 2048 + r * 16;
        const uint4 w0 = *reinterpret_cast<const uint4*>(src);
        const uint4 w1 = *reinterpret_cast<const uint4*>(src + 2048);
        if (j == kUS - 1 || ui == nu - 1) {  // this warp's reads of the stage are done
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.empty[s]);
        }
        uint32_t v[16];
        unpack_u4(w0.x, v[0], v[1]);
        unpack_u4(w0.y, v[2], v[3]);
        unpack_u4(w0.z, v[4], v[5]);
        unpack_u4(w0.w, v[6], v[7]);
        unpack_u4(w1.x, v[8], v[9]);
        unpack_u4(w1.y, v[10], v[11]);
        unpack_u4(w1.z, v[12], v[13]);
        unpack_u4(w1.w, v[14], v[15]);
        tmem_st16(tmem + 32 * b + 16 * kh + lane_base, v);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.a_full[b]);
        ++i;
      }
      const int e0 = ctl.map[ui][0], e1 = ctl.map[ui][1];
      if (e0 >= 0 || e1 >= 0) {  // residual item
        const int b = i % kNB, k = i / kNB;
        if (k > 0 && !(ok = mbar_wait(&ctl.d_full[b], (k - 1) & 1, abort_flag, tmo, p.err))) break;
        if ((half ? e1 : e0) >= 0) {
          const int cpos = ctl.rpos[ui][half], slot = cpos % kRS;
          if (!(ok = mbar_wait(&ctl.r_full[slot], (cpos / kRS) & 1, abort_flag, tmo, p.err))) break;
          const uint8_t* src = rring + slot * kRRecBytes + (2 * kh) * 1024 + (r & 63) * 16;
          const uint4 w0 = *reinterpret_cast<const uint4*>(src);
          const uint4 w1 = *reinterpret_cast<const uint4*>(src + 1024);
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.r_empty[slot]);
          uint32_t v[16];
          unpack_u4(w0.x, v[0], v[1]);
          unpack_u4(w0.y, v[2], v[3]);
          unpack_u4(w0.z, v[4], v[5]);
          unpack_u4(w0.w, v[6], v[7]);
          unpack_u4(w1.x, v[8], v[9]);
          unpack_u4(w1.y, v[10], v[11]);
          unpack_u4(w1.z, v[12], v[13]);
          unpack_u4(w1.w, v[14], v[15]);
          tmem_st16(tmem + 32 * b + 16 * kh + lane_base, v);
          tc_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.a_full[b]);
        ++i;
      }
    }
  } else if (warp >= kWarpDrain0) {
    // ---------------- drain warps: thread = weight row ----------------
    const int q = warp & 3, r = 32 * q + lane, half = q >> 1;
    const int dt = threadIdx.x - 32 * kWarpDrain0;  // 0..127
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    uint64_t acc[MLD / 2];
#pragma unroll
    for (int j = 0; j < MLD / 2; ++j) acc[j] = 0ull;
    bool ok = tmem_wait() && mbar_wait(&ctl.map_ready, 0, abort_flag, tmo, p.err);
    const uint32_t tmem = ctl.tmem_base;
    pdl_wait();  // Y and the workspace pieces may still be in use by the preceding kernel
    // Barrier of the 4 drain warps, bounded like every other wait (a warp that
    // gave up never leaves the others waiting).
    int nsync = 0;
    auto drain_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.drain_bar);
      return mbar_wait(&ctl.drain_bar, (nsync++) & 1, abort_flag, tmo, p.err);
    };

    // One item's dots of this row: acc += 2^9 sx * (s * (D - c)), or the test hook's raw dots.
    auto drain_item = [&](int i, const float* sx2, const float* cc, const uint16_t* sp, bool use, int ui,
                          int e) -> bool {
      const int b = i % kNB, k = i / kNB;
      if (!mbar_wait(&ctl.d_full[b], k & 1, abort_flag, tmo, p.err)) return false;
      tc_fence_after();
      const float s = use ? __half2float(__ushort_as_half(*sp)) : 0.0f;  // read only now: the copy has landed
      uint32_t d[MLD];
      tmem_ld_cols<MLD>(tmem + 32 * kNB + TN * b + lane_base, d);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.d_empty[b]);
      if (!use) return true;
      if constexpr (kDebug) {
        const int64_t u = u0 + ui;
        const int t = static_cast<int>(u / G), g = static_cast<int>(u % G);
#pragma unroll
        for (int m = 0; m < MLD; ++m) {
          if (m < p.M) {
            const int32_t dd = static_cast<int32_t>((__uint_as_float(d[m]) - cc[m]) * 512.0f);
            if (e < 0)
              p.dots_w[(static_cast<int64_t>(m) * (p.tiles * kTileN) + static_cast<int64_t>(t) * kTileN + r) * G + g] = dd;
            else
              p.dots_r[(static_cast<int64_t>(m) * p.mat[0].nnzb + e) * 64 + (r & 63)] = dd;
          }
        }
      } else {
        const uint64_t s2 = f2pack(s, s), m1 = f2pack(-1.0f, -1.0f);
        const float4* sx4 = reinterpret_cast<const float4*>(sx2);
        const float4* c4 = reinterpret_cast<const float4*>(cc);
#pragma unroll
        for (int j4 = 0; j4 < MLD / 4; ++j4) {
          const float4 sv = sx4[j4], cv = c4[j4];
          const uint64_t d0 = f2fma(f2pack(cv.x, cv.y), m1, f2pack(__uint_as_float(d[4 * j4]), __uint_as_float(d[4 * j4 + 1])));
          const uint64_t d1 =
              f2fma(f2pack(cv.z, cv.w), m1, f2pack(__uint_as_float(d[4 * j4 + 2]), __uint_as_float(d[4 * j4 + 3])));
          acc[2 * j4] = f2fma(f2pack(sv.x, sv.y), f2mul(s2, d0), acc[2 * j4]);
          acc[2 * j4 + 1] = f2fma(f2pack(sv.z, sv.w), f2mul(s2, d1), acc[2 * j4 + 1]);
        }
      }
      return true;
    };
    auto store_y = [&](const ZMat& mt, int64_t n, int m, float v) {
      const int64_t o = static_cast<int64_t>(m) * mt.ldy + n;
      if (p.y_f32)
        static_cast<float*>(mt.y)[o] = v;
      else
        static_cast<__nv_bfloat16*>(mt.y)[o] = __float2bfloat16_rn(v);
    };
    auto piece_of = [&](int64_t cc, int t) -> const float* {  // CTA cc's piece of tile t
      const int wc = (t == static_cast<int>(first_unit(cc, U, P) / G)) ? 0 : 1;
      return p.part + ((cc * 2 + wc) * TN) * static_cast<int64_t>(kTileN);
    };
    // Tile t is finished in this CTA's range: store it whole, or write this
    // CTA's piece and count it in; the CTA that completes the count sums the
    // pieces after its own range (deferred: no stall here).
    auto finish_tile = [&](int t) -> bool {
      const ZMat& mt = p.mat[mat_of_tile(p, t)];
      const int64_t n = static_cast<int64_t>(t - mt.tile0) * kTileN + r;
      const int64_t tu0 = static_cast<int64_t>(t) * G, tu1 = tu0 + G;
      if (tu0 >= u0 && tu1 <= u1) {  // the whole tile is this CTA's
#pragma unroll
        for (int j = 0; j < MLD / 2; ++j) {
          float lo, hi;
          f2unpack(acc[j], lo, hi);
          acc[j] = 0ull;
          if (2 * j < p.M) store_y(mt, n, 2 * j, lo);
          if (2 * j + 1 < p.M) store_y(mt, n, 2 * j + 1, hi);
        }
        return true;
      }
      float* mine = const_cast<float*>(piece_of(c, t));
#pragma unroll
      for (int j = 0; j < MLD / 2; ++j) {
        float lo, hi;
        f2unpack(acc[j], lo, hi);
        acc[j] = 0ull;
        if (2 * j < p.M) __stcg(mine + (2 * j) * kTileN + r, lo);
        if (2 * j + 1 < p.M) __stcg(mine + (2 * j + 1) * kTileN + r, hi);
      }
      __threadfence();
      if (!drain_sync()) return false;
      if (dt == 0) {  // a CTA is the first contributor of at most one cut tile: count it there
        const int64_t c_lo = owner_of(tu0, U, P), c_hi = owner_of(tu1 - 1, U, P);
        if (atomicAdd(p.tcount + c_lo, 1) == static_cast<int>(c_hi - c_lo)) ctl.deferred[ctl.ndeferred++] = t;
      }
      return true;
    };

    int i = 0;
    for (int ui = 0; ui < nu && ok; ++ui) {
      const int st = ui / kUS, j = ui - st * kUS, s = st % S;
      const int64_t u = u0 + ui;
      const int t = static_cast<int>(u / G), g = static_cast<int>(u - static_cast<int64_t>(t) * G);
      const uint8_t* sg = stage(s);
      const float* sx2 = reinterpret_cast<const float*>(sg + j * kArec + TN * 128);
      const float* cc = sx2 + TN;
      // the stage's bytes (activation scales, offset terms, row scales) were
      // written by the bulk copy: wait on its barrier too (long complete)
      if (j == 0 && !(ok = mbar_wait(&ctl.full[s], (st / S) & 1, abort_flag, tmo, p.err))) break;
      const uint16_t* swp = reinterpret_cast<const uint16_t*>(sg + kAct + j * kWRecBytes + kWRecScales + 2 * r);
      if (!(ok = drain_item(i++, sx2, cc, swp, true, ui, -1))) break;
      const int e0 = ctl.map[ui][0], e1 = ctl.map[ui][1];
      if (e0 >= 0 || e1 >= 0) {
        const int e = half ? e1 : e0;
        int slot = 0;
        const uint16_t* srp = nullptr;
        if (e >= 0) {
          const int cpos = ctl.rpos[ui][half];
          slot = cpos % kRS;
          if (!(ok = mbar_wait(&ctl.r_full[slot], (cpos / kRS) & 1, abort_flag, tmo, p.err))) break;
          srp = reinterpret_cast<const uint16_t*>(rring + slot * kRRecBytes + kRRecScales + 2 * (r & 63));
        }
        if (!(ok = drain_item(i++, sx2, cc, srp, e >= 0, ui, e))) break;
        __syncwarp();
        if (lane == 0 && e >= 0) mbar_arrive(&ctl.r_empty[slot]);
      }
      if (j == kUS - 1 || ui == nu - 1) {  // the stage's scales are read
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.empty[s]);
      }
      if (!kDebug && (g == G - 1 || ui == nu - 1) && !(ok = finish_tile(t))) break;
    }

    // Finish the tiles this CTA completed the count of: bring every piece
    // into the (now idle) stage memory with bulk copies, sum in CTA order,
    // store Y, and reset the tile's counter for the next launch.
    if (!kDebug && ok && (ok = drain_sync())) {
      const int nd = ctl.ndeferred;
      const uint32_t piece_bytes = static_cast<uint32_t>(p.M) * kTileN * 4;  // rows 0..M-1 of a piece
      const int per_round = max(1, static_cast<int>((static_cast<size_t>(S) * SB) / piece_bytes));
      int nred = 0;
      for (int di = 0; di < nd && ok; ++di) {
        const int t = ctl.deferred[di];
        const ZMat& mt = p.mat[mat_of_tile(p, t)];
        const int64_t n = static_cast<int64_t>(t - mt.tile0) * kTileN + r;
        const int64_t tu0 = static_cast<int64_t>(t) * G, tu1 = tu0 + G;
        const int64_t c_lo = owner_of(tu0, U, P), c_hi = owner_of(tu1 - 1, U, P);
        float sum[MLD];
        for (int64_t cb = c_lo; cb <= c_hi && ok; cb += per_round) {
          const int np = static_cast<int>(min(static_cast<int64_t>(per_round), c_hi - cb + 1));
          if (dt == 0) {
            __threadfence();
            fence_proxy_async_global();  // other CTAs' generic writes -> this bulk (async) read
            mbar_arrive_expect_tx(&ctl.red_bar, np * piece_bytes);
            for (int k = 0; k < np; ++k) bulk_g2s(stages + k * piece_bytes, piece_of(cb + k, t), piece_bytes, &ctl.red_bar);
          }
          if (!(ok = mbar_wait(&ctl.red_bar, nred & 1, abort_flag, tmo, p.err))) break;
          ++nred;
          for (int k = 0; k < np; ++k) {
            const float* pc = reinterpret_cast<const float*>(stages + k * piece_bytes) + r;
#pragma unroll
            for (int m = 0; m < MLD; ++m) {
              if (m < p.M) {
                const float v = pc[m * kTileN];
                sum[m] = (cb == c_lo && k == 0) ? v : sum[m] + v;  // ascending CTA order
              }
            }
          }
          if (!(ok = drain_sync())) break;  // the stage memory is free for the next round
        }
        if (!ok) break;
#pragma unroll
        for (int m = 0; m < MLD; ++m)
          if (m < p.M) store_y(mt, n, m, sum[m]);
        if (dt == 0) p.tcount[c_lo] = 0;
      }
    }
  }

  // Every role is done.
  __syncwarp();
  if (lane == 0) mbar_arrive(&ctl.exit_bar);
  mbar_wait(&ctl.exit_bar, 0, abort_flag, tmo, p.err);
  __syncthreads();
  if (threadIdx.x == 0) {
    ZT(5);
    ZC(7);
  }
  if (*abort_flag) {
    // A wait gave up: copies and MMAs may still be in flight; give them 200 us.
    if (threadIdx.x == 0) {
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 200000ull) {
      }
    }
    __syncthreads();
  }
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(ctl.tmem_base, kTmemCols);
  }
}


// ---------------------------------------------------------------------------
// The warp-MMA form (the default up to 32 tokens).
//
// Measured on GB300: a tcgen05.mma of M = 128, K = 32 costs the tensor pipe
// about 46 cycles at any N up to 64, and passing items between warps through
// mbarriers (unpack -> MMA issue -> drain) costs about 500 cycles per item even
// with no work in it -- more than the ~430 SM-cycles of HBM time a 128 x 128
// group of 4-bit weights is worth.  So here every warp carries its own rows
// through a whole group with no hand-off: unpack its codes into registers, run
// mma.sync m16n8k32 e4m3 against the activation fragments of the stage, and
// scale the exact dots into its own fp32 accumulators.  Warps meet only once
// per 4-unit stage (and at tile ends, to add their partials in a fixed order).
//
// Warps 0..15: four sets of four; set q takes unit q of every stage, warp w of
// a set owns rows 32w..32w+31 (two 16-row MMA tiles).  Warp 16: producer;
// warp 17: residual map and records.
// ---------------------------------------------------------------------------

// 16 compute warps in sets; a set takes one unit (128 rows) of every stage.
// Up to 16 tokens a warp owns 32 rows (two 16-row MMA tiles): sets of 4 warps,
// 4 units per stage.  At 32 tokens a warp owns 16 rows: its accumulators then
// fit the 96 registers a thread gets when 18 warps share the schedulers'
// register files, with sets of 8 warps and 2 units per stage.
__host__ __device__ constexpr int w_mt(int tn) { return tn == 32 ? 1 : 2; }  // 16-row MMA tiles per warp
__host__ __device__ constexpr int w_wps(int tn) { return 8 / w_mt(tn); }     // warps per set
__host__ __device__ constexpr int w_sets(int tn) { return 16 / w_wps(tn); }  // sets = units per stage
__host__ __device__ constexpr int w_threads(int tn) { return 32 * (16 + 2); }  // + producer, epilogue

// One bulk copy of the producer's schedule: source, offset in the stage, bytes.
struct __align__(16) CopyDesc {
  const uint8_t* src;
  uint32_t dst;
  uint32_t bytes;
};

constexpr int kCopiesPerStage = 8;          // weight runs + activation runs of a stage (4 units: at most 4 + 4)

template <int kMaxStg>  // stages per CTA at most: kMaxUnits / units per stage, + 1
struct __align__(16) WCtl {
  CopyDesc cp[kMaxStg][kCopiesPerStage];  // the stage's copies (bytes 0: none)
  uint32_t stage_tx[kMaxStg];             // bytes a stage's copies bring
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];  // the compute warps are done with the stage
  uint64_t r_full[kRS];
  uint64_t r_empty[kRS];       // the 2 warps of the record's half
  uint64_t tile_bar;           // bounded barrier of the compute warps (tile ends)
  uint64_t map_ready;
  uint64_t piece_written;      // every compute warp wrote its share of this CTA's stream-K piece
  uint64_t slot_free[kMaxStages];  // the producer handed the epilogue stage slot k (single use)
  uint64_t pieces_in;          // the other CTAs' pieces of the tile this CTA finishes are readable
  uint64_t exit_bar;
  int32_t map[kMaxUnits][2];
  int32_t rpos[kMaxUnits][2];
  const uint8_t* rsrc[kMaxUnits];  // residual records of the unit's matrix
  int abort_flag;
  volatile int r_issued;  // residual records issued so far (the producer issues them in ring order)
};

// D(16x8, fp32) += A(16x32, E4M3, row-major) * B(32x8, E4M3, column-major).
__device__ __forceinline__ void mma_e4m3(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// The same with a zero accumulator in (the first K-step of a group).
__device__ __forceinline__ void mma_e4m3_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// TN: tokens per tile (8, 16 or 32); kDebug: write raw group dots.
template <int TN, bool kDebug>
__global__ void __launch_bounds__(w_threads(TN), 1) zipper_warp_kernel(const ZParams p) {
  constexpr int NB = TN / 8;           // 8-token blocks of one MMA
  constexpr int kRedPasses = TN == 8 ? 1 : 2, kRedTok = TN / kRedPasses;  // tile sums: tokens per pass
  constexpr int kRedLd = kTileN + 4;  // token stride of a partial buffer: fragment writes hit distinct banks
  constexpr int MT = w_mt(TN), WPS = w_wps(TN);  // 16-row MMA tiles per warp, warps per set
  constexpr int US = w_sets(TN);       // units per stage = sets of compute warps
  constexpr int kWCompute = 16, kWProd = kWCompute, kWEpi = kWCompute + 1, kWThreads = w_threads(TN);
  constexpr int kMaxStg = kMaxUnits / US + 1;  // stages per CTA at most
  constexpr int kArec = TN * 136;      // activation image: B fragments, then {2^9 sx, c} pairs
  constexpr int kAct = US * kArec;     // a stage: US activation images, then US base records
  extern __shared__ uint8_t smem_raw[];
  __shared__ WCtl<kMaxStg> ctl;
  uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  const int S = p.nstages, SB = p.stage_bytes, G = p.G;
  uint8_t* stages = smem;
  uint8_t* rring = smem + static_cast<size_t>(S) * SB;
  float* red = reinterpret_cast<float*>(rring + kRS * kRRecBytes);  // [US sets][kRedTok][kRedLd] tile partials
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t U32 = static_cast<uint32_t>(p.units), P32 = static_cast<uint32_t>(p.ctas), c32 = blockIdx.x;
  const int64_t U = U32, P = P32, c = c32;
  const int64_t u0 = first_unit32(c32, U32, P32), u1 = first_unit32(c32 + 1, U32, P32);
  const int nu = static_cast<int>(u1 - u0);
  const int nstg = (nu + US - 1) / US;
  // Stream-K roles.  A cut tile is finished by the CTA holding its first
  // groups (its head); every other CTA on it publishes a piece (its share of
  // the tile's sums) and a flag.  A CTA publishes at most one piece (for its
  // first tile, when its range starts inside it) and finishes at most one
  // tile (its last, when its range holds that tile's head but not its end).
  // The pieces of the tile it finishes are the tails of later CTAs' ranges,
  // computed first there: usually in place long before they are needed.
  const int t_first = static_cast<int>(static_cast<uint32_t>(u0) / static_cast<uint32_t>(G));
  const int t_last = static_cast<int>(static_cast<uint32_t>(u1 - 1) / static_cast<uint32_t>(G));
  const bool publishes = !kDebug && u0 > static_cast<int64_t>(t_first) * G;
  const bool finishes =
      !kDebug && u0 <= static_cast<int64_t>(t_last) * G && u1 < static_cast<int64_t>(t_last + 1) * G;
  const int npc =
      finishes ? static_cast<int>(owner_of32(static_cast<uint32_t>((t_last + 1) * G - 1), U32, P32) - c32) : 0;
  const uint32_t piece_bytes = static_cast<uint32_t>(p.M) * kTileN * 4;  // tokens 0..M-1 of a [TN][128] piece
  // the pieces go into stage slots no stage needs any more, per_slot to a slot, if they fit in all slots
  const int per_slot = SB / static_cast<int>(piece_bytes);
  const int need_slots = per_slot > 0 ? (npc + per_slot - 1) / per_slot : S + 1;
  // (a partial last stage's slot is never released by the sets without a unit in it: not handed over)
  const bool pieces_in_smem = need_slots <= S - (nu % US != 0 ? 1 : 0);
  // the k-th handed-over slot is the one stage nstg + k would take
  auto piece_slot = [&](int k) -> uint32_t { return static_cast<uint32_t>((nstg + k) % S) * SB; };
  auto piece_of = [&](int64_t cc) -> float* { return p.part + cc * (TN * static_cast<int64_t>(kTileN)); };
  volatile int* abort_flag = &ctl.abort_flag;
  const uint64_t tmo = p.timeout_ns;
  ZT_INIT;
  if (threadIdx.x == 0) {
    ZT(0);
    ZC(6);
  }

  if (warp == 0) {
    for (int s = lane; s < S; s += 32) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], kWCompute);
    }
    if (lane < kRS) {
      mbar_init(&ctl.r_full[lane], 1);
      mbar_init(&ctl.r_empty[lane], WPS / 2);  // the warps of the record's 64-row half
    }
    if (lane == 10) mbar_init(&ctl.tile_bar, kWCompute);
    if (lane == 11) mbar_init(&ctl.map_ready, 1);
    if (lane == 12) mbar_init(&ctl.piece_written, kWCompute);
    if (lane < kMaxStages) mbar_init(&ctl.slot_free[lane], 1);
    if (lane == 17) mbar_init(&ctl.pieces_in, 1);
    if (lane == 14) mbar_init(&ctl.exit_bar, kWThreads / 32);
    if (lane == 15) ctl.abort_flag = 0;
    if (lane == 16) ctl.r_issued = 0;
    fence_mbar_init();
    if (lane == 0) ZC(11);
  }
  // Cluster mode: one tile per cluster; its CTAs' pieces go into the head
  // CTA's shared memory (rx) by bulk copy, counted on the head's pieces_in.
  // (read from the parameters where used: kept out of the compute warps' registers)
#define ZCK (kDebug ? 0 : p.cluster)
#define ZRX reinterpret_cast<float*>(smem + p.rx_off)
  if (ZCK > 0) {
    cluster_sync_all();  // every peer's barriers are initialised before any copy targets them
    if (finishes && threadIdx.x == 0) mbar_arrive_expect_tx(&ctl.pieces_in, static_cast<uint32_t>(npc) * piece_bytes);
  } else {
    __syncthreads();
  }
  if (threadIdx.x == 0) ZC(12);
  pdl_trigger();
  auto stage = [&](int s) { return stages + static_cast<size_t>(s) * SB; };
  auto copy_ok = [&](const CopyDesc& d) {  // a stage copy stays inside its slot, 16-byte aligned
    return ZOK(d.dst + d.bytes <= static_cast<uint32_t>(SB) && (d.bytes & 15u) == 0 && (d.dst & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(d.src) & 15u) == 0,
               1);
  };

  if (warp == kWProd) {
    // ---------------- producer: a stage = US units' base records and activation images, then the
    // residual records of those units ----------------
    // The lanes first lay out every stage's copies in a table, one lane per
    // unit (a pass of 32 - 32 % US units never splits a stage): a unit opens
    // a base-record run when it is its stage's first or the first of its
    // matrix, an activation run when it is its stage's first or group 0 of a
    // tile; a run ends where the next of its kind opens.  The base records of
    // a run are one copy, so are its activation images.
    constexpr int kUnitsPerPass = 32 - 32 % US;
    for (int j0 = 0; j0 < nu; j0 += kUnitsPerPass) {
      const int k = lane % US, first = lane - k;  // unit in stage, first lane of the stage
      const bool live = lane < kUnitsPerPass && j0 + lane < nu;
      int mi = 0, tt = 0, gg = 0;
      if (live) {
        const int u = static_cast<int>(u0) + j0 + lane;  // the planner keeps unit indexes below 2^31
        tt = u / G;
        gg = u - tt * G;
        mi = mat_of_tile(p, tt);
      }
      const int mi_prev = __shfl_up_sync(0xFFFFFFFFu, mi, 1);
      const unsigned wm = __ballot_sync(0xFFFFFFFFu, live && (k == 0 || mi != mi_prev));
      const unsigned am = __ballot_sync(0xFFFFFFFFu, live && (k == 0 || gg == 0));
      if (live) {
        const int st = j0 / US + lane / US;
        const int last = min(first + US, nu - j0);  // one past the stage's last lane
        const unsigned smask = ((1u << US) - 1u) << first, below = (1u << lane) - 1u, above = ~below & ~(1u << lane);
        const int nw = __popc(wm & smask);
        if ((wm >> lane) & 1u) {
          const unsigned nxt = wm & smask & above;
          const int end = nxt ? __ffs(nxt) - 1 : last;
          const ZMat& mt = p.mat[mi];
          const int ix = __popc(wm & smask & below);
          CopyDesc& d = ctl.cp[ZOK(st < kMaxStg && ix < kCopiesPerStage, 0) ? st : 0][ix & (kCopiesPerStage - 1)];
          d.src = mt.wpk + (static_cast<int64_t>(tt - mt.tile0) * G + gg) * kWRecBytes;
          d.dst = static_cast<uint32_t>(kAct + k * kWRecBytes);
          d.bytes = static_cast<uint32_t>((end - lane) * kWRecBytes);
          // the first stages' base records leave at once (their stage's count is posted
          // below: a transfer may complete before it, the phase cannot)
          if (st < S && copy_ok(d)) bulk_g2s(stage(st) + d.dst, d.src, d.bytes, &ctl.full[st]);
        }
        if ((am >> lane) & 1u) {
          const unsigned nxt = am & smask & above;
          const int end = nxt ? __ffs(nxt) - 1 : last;
          const int ix = nw + __popc(am & smask & below);
          CopyDesc& d = ctl.cp[ZOK(st < kMaxStg && ix < kCopiesPerStage, 0) ? st : 0][ix & (kCopiesPerStage - 1)];
          d.src = p.act + static_cast<int64_t>(gg) * kArec;
          d.dst = static_cast<uint32_t>(k * kArec);
          d.bytes = static_cast<uint32_t>((end - lane) * kArec);
        }
        if (k == 0) {
          for (int i = nw + __popc(am & smask); i < kCopiesPerStage; ++i) ctl.cp[st][i].bytes = 0;
          ctl.stage_tx[st] = static_cast<uint32_t>((last - first) * (kWRecBytes + kArec));
          if (st < S) mbar_arrive_expect_tx(&ctl.full[st], ctl.stage_tx[st]);
        }
      }
    }
    __syncwarp();
    const int pre = min(S, nstg);
    // The first stages' base records left during the table pass, before the
    // dependency wait: the kernels that may run ahead of it (this library's,
    // which ask for the next launch early) never write packed weights.  Then
    // the activation images of those stages, all in one instruction (lane:
    // stage, copy).
    if (lane == 0) ZC(13);
    if (lane == 0) ZC(8);
    pdl_wait();  // the activation images are the preceding kernel's output
    if (lane == 0) ZC(10);
    for (int i = lane; i < pre * kCopiesPerStage; i += 32) {
      const int st = i / kCopiesPerStage;
      const CopyDesc d = ctl.cp[st][i % kCopiesPerStage];
      if (d.bytes && d.dst < static_cast<uint32_t>(kAct) && copy_ok(d))
        bulk_g2s(stage(st) + d.dst, d.src, d.bytes, &ctl.full[st]);
    }
    __syncwarp();
    if (lane == 0) ZC(16);
    bool ok = ZW(mbar_wait(&ctl.map_ready, 0, abort_flag, tmo, p.err), 7);
    ok = __all_sync(0xFFFFFFFFu, ok);
    // Two cursors, neither waiting on the other: the residual records in ring
    // order (those of issued stages, each once its ring slot is free), and
    // the refills of stage slots as the compute warps free them.
    int bst = pre, bs = 0, bph = 1;  // next stage, its slot, the slot's fill parity
    int rf = 0;                       // next (unit, half) whose residual record is due
    const int nf = 2 * nu;
    uint64_t idle_since = 0;
    for (int idle = 0; ok && (bst < nstg || rf < nf);) {
      bool progress = false;
      const int rlim = min(nf, 2 * US * bst);
      if (rf < rlim) {
        const int f = rf + lane;
        bool ready = false;
        int e = -1, cpos = 0;
        if (f < rlim) {
          e = (&ctl.map[0][0])[f];
          cpos = e >= 0 ? (&ctl.rpos[0][0])[f] : 0;
          // the slot's previous record (cpos - kRS) has been issued, so the
          // slot's phase is one of two and the parity test is exact
          ready = e < 0 || cpos < kRS || mbar_test_wait(&ctl.r_empty[cpos % kRS], ((cpos / kRS) - 1) & 1);
        }
        const unsigned blocked = __ballot_sync(0xFFFFFFFFu, !ready);
        const int n = blocked ? __ffs(blocked) - 1 : 32;  // the ready prefix, in ring order
        if (lane < n && e >= 0) {
          const int slot = cpos % kRS;
          mbar_arrive_expect_tx(&ctl.r_full[slot], kRRecBytes);
          bulk_g2s(rring + slot * kRRecBytes, ctl.rsrc[f >> 1] + static_cast<int64_t>(e) * kRRecBytes, kRRecBytes,
                   &ctl.r_full[slot]);
        }
        const int nrec = __popc(__ballot_sync(0xFFFFFFFFu, lane < n && e >= 0));
        if (lane == 0 && nrec) ctl.r_issued = ctl.r_issued + nrec;
        rf += n;
        progress = n > 0;
      }
      if (bst < nstg) {
        int go = 0;
        if (lane == 0 && mbar_test_wait(&ctl.empty[bs], bph ^ 1)) {
          mbar_arrive_expect_tx(&ctl.full[bs], ctl.stage_tx[bst]);
          go = 1;
        }
        if (__shfl_sync(0xFFFFFFFFu, go, 0)) {
          if (lane < kCopiesPerStage) {
            const CopyDesc d = ctl.cp[bst][lane];
            if (d.bytes && copy_ok(d)) bulk_g2s(stage(bs) + d.dst, d.src, d.bytes, &ctl.full[bs]);
          }
          if (lane == 0 && bst < 16) ZC(16 + bst);
          ++bst;
          if (++bs == S) bs = 0, bph ^= 1;
          progress = true;
        }
      }
      if (progress) {
        idle = 0;
        continue;
      }
      // back off (32 ns doubling to 512 ns): the polls share a scheduler with compute warps
      __nanosleep(32u << min(idle >> 2, 4));
      if ((++idle & 15) == 0) {  // bounded: give up after the timeout without progress
        int give_up = 0;
        if (lane == 0) {
          const uint64_t now = globaltimer();
          if (*abort_flag) {
            give_up = 1;
          } else if (idle == 16) {
            idle_since = now;
          } else if (now - idle_since > tmo) {
            ZW(false, 7);
            atomicOr(p.err, kDevErrTimeout);
            *abort_flag = 1;
            give_up = 1;
          }
        }
        ok = !__shfl_sync(0xFFFFFFFFu, give_up, 0);
      }
    }
    // The slots stages nstg, nstg + 1, .. would take are free once the compute
    // warps are done with their last stages (at once if never filled): they
    // take the pieces of the tile this CTA finishes, handed over one by one.
    if (ok && ZCK == 0 && finishes && pieces_in_smem && lane == 0) {
      for (int k = 0; k < need_slots; ++k) {
        const int v = nstg + k, slot = v % S;  // the slot's last fill was stage v - S; its phases are waited in order
        if (v >= S && !ZW(mbar_wait_sleep(&ctl.empty[slot], ((v / S) - 1) & 1, abort_flag, tmo, p.err), 7)) break;
        mbar_arrive(&ctl.slot_free[k]);
      }
    }
    __syncwarp();
  } else if (warp == kWEpi) {
    // ---------------- epilogue: stream-K pieces off the compute warps' path ----------------
    pdl_wait();  // the flags and pieces in the workspace may still be in use by the preceding kernel
    bool ok = true;
    if (publishes && ZCK == 0) {  // release this CTA's piece once every compute warp has written its share
      if (lane == 0) {
        ok = ZW(mbar_wait_sleep(&ctl.piece_written, 0, abort_flag, tmo, p.err), 4);
        if (ok) {
          fence_acq_rel_gpu();
          st_relaxed_gpu(p.tcount + c, 1);
          ZC(88);
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    }
    if (finishes && ok && ZCK == 0) {
      // the flags of the other pieces (lane j: CTA c + 1 + j), then the pieces
      // into the free slot; each flag is cleared for the next launch once seen
      for (int j0 = 0; ok && j0 < npc; j0 += 32) {
        const int j = j0 + lane;
        bool seen = true;
        if (j < npc && ZOK(c + 1 + j < P, 4) && (seen = ZW(flag_wait(p.tcount + c + 1 + j, abort_flag, tmo, p.err), 5)))
          p.tcount[c + 1 + j] = 0;
        ok = __all_sync(0xFFFFFFFFu, seen);
      }
      if (lane == 0) ZC(89);
      if (ok && pieces_in_smem) {
        if (lane == 0) mbar_arrive_expect_tx(&ctl.pieces_in, npc * piece_bytes);
        for (int k = 0; ok && k < need_slots; ++k) {  // slot k: pieces k * per_slot ..
          if (lane == 0) ok = ZW(mbar_wait_sleep(&ctl.slot_free[k], 0, abort_flag, tmo, p.err), 6);
          if (!(ok = __shfl_sync(0xFFFFFFFFu, ok, 0))) break;
          const int j = k * per_slot + lane;
          if (lane < per_slot && j < npc && ZOK(piece_slot(k) + (lane + 1) * piece_bytes <= static_cast<uint32_t>(S) * SB, 5)) {
            fence_proxy_async_global();  // the pieces were written through the generic proxy
            bulk_g2s(stages + piece_slot(k) + lane * piece_bytes, piece_of(c + 1 + j), piece_bytes,
                     &ctl.pieces_in);
          }
        }
      } else if (ok && lane == 0) {
        mbar_arrive(&ctl.pieces_in);  // the compute warps read the pieces in place
      }
    }
  } else {
    // ---------------- compute warps ----------------
    const int q = warp / WPS, wq = warp % WPS;  // set, row block within the set
    const int g = lane >> 2, t = lane & 3;       // MMA fragment coordinates
    const int rw = 16 * MT * wq, half = rw >> 6;  // first row of this warp, its residual half
    if (warp == 0) {
      // Residual map of the CTA's units (CSR entry per unit and half) and the
      // records' ring positions.  The block lists are read before the
      // dependency wait, like the weights.
      for (int i = lane; i < nu * 2; i += 32) (&ctl.map[0][0])[i] = -1;
      __syncwarp();
      if (nu > 0) {
        for (int tt = t_first; tt <= t_last; ++tt) {
          const ZMat& mt = p.mat[mat_of_tile(p, tt)];
          if (mt.nnzb == 0) continue;
          const int64_t br = 2 * static_cast<int64_t>(tt - mt.tile0);
          const int a0 = max(0, min(mt.nnzb, mt.row_ptr[br]));
          const int a1 = max(a0, min(mt.nnzb, mt.row_ptr[br + 1]));
          const int a2 = max(a1, min(mt.nnzb, mt.row_ptr[br + 2]));
          for (int e = a0 + lane; e < a2; e += 32) {
            const int gg = mt.col_idx[e];
            if (gg < 0 || gg >= G) continue;
            const int64_t u = static_cast<int64_t>(tt) * G + gg;
            if (u >= u0 && u < u1) {
              ctl.map[u - u0][e >= a1 ? 1 : 0] = e;
              ctl.rsrc[u - u0] = mt.rpk;
            }
          }
        }
      }
      __syncwarp();
      const int nf = nu * 2;
      const int chunk = (nf + 31) / 32, f0 = min(nf, lane * chunk), f1 = min(nf, f0 + chunk);
      int cnt = 0;
      for (int fx = f0; fx < f1; ++fx) cnt += (&ctl.map[0][0])[fx] >= 0;
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      int pos = incl - cnt;
      for (int fx = f0; fx < f1; ++fx)
        if ((&ctl.map[0][0])[fx] >= 0) (&ctl.rpos[0][0])[fx] = pos++;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl.map_ready);
        ZC(9);
      }
    }
    bool ok = ZW(mbar_wait(&ctl.map_ready, 0, abort_flag, tmo, p.err), 0);
    pdl_wait();  // Y and the workspace pieces may still be in use by the preceding kernel
    // accumulators: [mt][nb] pairs {row r, tokens 8nb+2t, +1}, {row r+8, same tokens}
    uint64_t acc[MT][NB][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) acc[mt][nb][0] = acc[mt][nb][1] = 0ull;

    // One group's product for this warp's rows: codes (K-steps jstride apart,
    // 16 bytes per row, first row row0), fragments and scale pairs of the
    // group's activation image, row scales sc; into acc, or the test hook's dots.
    // The 8-token blocks are taken one at a time (the weight fragments are
    // unpacked again for each): the MMA results then never hold more than 8
    // registers next to the accumulators, and nothing spills.
    auto group_product = [&](const uint8_t* codes, int jstride, int row0, const uint16_t* sc, const uint8_t* img,
                             int64_t u, int e) {
      constexpr int NBH = 1;  // 8-token blocks per pass
      const uint8_t* wr = codes + (row0 + g) * 16 + t * 4;
      const float4* sg = reinterpret_cast<const float4*>(img + TN * 128) + t;  // token pairs 2t, 2t+1 of block nb
      float s[MT][2];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        s[mt][0] = __half2float(__ushort_as_half(sc[row0 + 16 * mt + g]));
        s[mt][1] = __half2float(__ushort_as_half(sc[row0 + 16 * mt + 8 + g]));
      }
#pragma unroll
      for (int nh = 0; nh < NB; nh += NBH) {
        float d[MT][NBH][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t a[MT][4];
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t w0 = *reinterpret_cast<const uint32_t*>(wr + j * jstride + mt * 256);        // row +0
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(wr + j * jstride + mt * 256 + 128);  // row +8
            unpack_u4(w0, a[mt][0], a[mt][2]);
            unpack_u4(w1, a[mt][1], a[mt][3]);
          }
#pragma unroll
          for (int i = 0; i < NBH; ++i) {
            const uint2 b = *reinterpret_cast<const uint2*>(img + ((j * NB + nh + i) * 32 + lane) * 8);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              if (j == 0)
                mma_e4m3_z(d[mt][i], a[mt], b.x, b.y);
              else
                mma_e4m3(d[mt][i], a[mt], b.x, b.y);
            }
          }
        }
        const uint64_t m1 = f2pack(-1.0f, -1.0f);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int i = 0; i < NBH; ++i) {
            const int nb = nh + i;
            const float4 f = sg[4 * nb];  // 2^9 sx (tokens 8nb+2t, +1), c (same tokens)
            if constexpr (kDebug) {
              const int tile = static_cast<int>(u / G), gg = static_cast<int>(u % G);
              const float ev[2][2] = {{d[mt][i][0] - f.z, d[mt][i][1] - f.w}, {d[mt][i][2] - f.z, d[mt][i][3] - f.w}};
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                  const int m = 8 * nb + 2 * t + cc, r = rw + 16 * mt + 8 * h + g;
                  if (m < p.M) {
                    const int32_t dv = static_cast<int32_t>(ev[h][cc] * 512.0f);
                    if (e < 0)
                      p.dots_w[(static_cast<int64_t>(m) * (p.tiles * kTileN) + static_cast<int64_t>(tile) * kTileN + r) *
                                   G +
                               gg] = dv;
                    else
                      p.dots_r[(static_cast<int64_t>(m) * p.mat[0].nnzb + e) * 64 + (r & 63)] = dv;
                  }
                }
            } else {
              const uint64_t sx2 = f2pack(f.x, f.y), c2 = f2pack(f.z, f.w);
              const uint64_t e0 = f2fma(c2, m1, f2pack(d[mt][i][0], d[mt][i][1]));  // row +0: exact 2^-9 D
              const uint64_t e1 = f2fma(c2, m1, f2pack(d[mt][i][2], d[mt][i][3]));  // row +8
              acc[mt][nb][0] = f2fma(sx2, f2mul(f2pack(s[mt][0], s[mt][0]), e0), acc[mt][nb][0]);
              acc[mt][nb][1] = f2fma(sx2, f2mul(f2pack(s[mt][1], s[mt][1]), e1), acc[mt][nb][1]);
            }
          }
        }
      }
    };
    // Explicit global stores and shared loads in the tile ends: a generic load
    // after a generic store that might alias it waits for the store to land.
    auto store_y = [&](const ZMat& mt, int64_t n, int m, float v) {
      const int64_t o = static_cast<int64_t>(m) * mt.ldy + n;
      if (p.y_f32)
        st_global_f32(static_cast<float*>(mt.y) + o, v);
      else
        st_global_b16(static_cast<__nv_bfloat16*>(mt.y) + o, __bfloat16_as_ushort(__float2bfloat16_rn(v)));
    };
    // End of tile `tile`: every warp writes its partial into its set's
    // buffer, then each warp adds the sets' partials of its slice of the rows
    // in set order (and, for the tile this CTA finishes, the other CTAs'
    // pieces in CTA order) and stores Y, or this CTA's piece.
    int nsync = 0;  // phases of tile_bar
    auto tile_sync = [&]() -> bool {  // all compute warps (bounded)
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.tile_bar);
      return ZW(mbar_wait(&ctl.tile_bar, (nsync++) & 1, abort_flag, tmo, p.err), 2);
    };
    auto flush = [&](int tile) -> bool {
      const ZMat& mt = p.mat[mat_of_tile(p, tile)];
      const int64_t nbase = static_cast<int64_t>(tile - mt.tile0) * kTileN;
      const bool pub = publishes && tile == t_first;  // write this CTA's piece
      const bool fin = finishes && tile == t_last;    // add the other CTAs' pieces
      float* piece = pub ? piece_of(c) : nullptr;
      float* mine = red + q * (kRedTok * kRedLd);
      const int slot0 = nstg % S;  // the first slot handed over for pieces
      if (fin) {
        const bool got = ZCK > 0 ? mbar_wait_cluster(&ctl.pieces_in, 0, abort_flag, tmo, p.err)
                                : mbar_wait(&ctl.pieces_in, 0, abort_flag, tmo, p.err);
        if (!ZW(got, 3)) return false;
        if (warp == 0 && lane == 0) ZC(92);
      }
#pragma unroll
      for (int pass = 0; pass < kRedPasses; ++pass) {  // tokens [pass * kRedTok, +kRedTok)
#pragma unroll
        for (int nb = pass * (NB / kRedPasses); nb < (pass + 1) * (NB / kRedPasses); ++nb)
#pragma unroll
          for (int mt2 = 0; mt2 < MT; ++mt2)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int r = rw + 16 * mt2 + 8 * h + g, m0 = 8 * nb + 2 * t - pass * kRedTok;
              float v0, v1;
              f2unpack(acc[mt2][nb][h], v0, v1);
              acc[mt2][nb][h] = 0ull;
              st_shared_f32(mine + m0 * kRedLd + r, v0);
              st_shared_f32(mine + (m0 + 1) * kRedLd + r, v1);
            }
        if (warp == kWCompute - WPS && lane == 0) ZC(170 + 4 * pass);
        if (!tile_sync()) return false;
        if (warp == kWCompute - WPS && lane == 0) ZC(171 + 4 * pass);
        // the pass's (row, token) entries of the tile, spread over the compute warps, row-major
        // within a token (consecutive lanes take consecutive rows: coalesced stores)
        for (int e = warp * 32 + lane; e < kTileN * kRedTok; e += 32 * kWCompute) {
          const int mr = e >> 7, m = pass * kRedTok + mr, r = e & (kTileN - 1);
          if (m >= p.M) continue;
          float v = ld_shared_f32(red + mr * kRedLd + r);
#pragma unroll
          for (int qq = 1; qq < US; ++qq) v += ld_shared_f32(red + (qq * kRedTok + mr) * kRedLd + r);  // set order
          if (fin && ZCK > 0) {
            for (int j = 0; j < npc; ++j)  // cluster rank order
              v += ld_shared_f32(ZRX + j * (piece_bytes / 4) + m * kTileN + r);
          } else if (fin && pieces_in_smem) {
            // piece j sits at slot (nstg + j / per_slot) % S, (j % per_slot) pieces in: walked, not divided
            uint32_t off = static_cast<uint32_t>(slot0) * SB;
            for (int j = 0, in = 0, sl = slot0; j < npc; ++j) {  // CTA order
              if (ZOK(off + (m * kTileN + r) * 4u < static_cast<uint32_t>(S) * SB, 6))
                v += ld_shared_f32(reinterpret_cast<const float*>(stages + off) + m * kTileN + r);
              if (++in == per_slot) {
                in = 0;
                sl = sl + 1 == S ? 0 : sl + 1;
                off = static_cast<uint32_t>(sl) * SB;
              } else {
                off += piece_bytes;
              }
            }
          } else if (fin) {
#pragma unroll 8
            for (int j = 0; j < npc; ++j) v += __ldcg(piece_of(c + 1 + j) + m * kTileN + r);  // CTA order
          }
          if (pub && ZCK > 0) {
            st_shared_f32(ZRX + m * kTileN + r, v);
          } else if (pub) {
            if (ZOK(c < P && m < TN, 9)) st_global_f32(piece + m * kTileN + r, v);
          } else if (ZOK(tile >= mt.tile0 && tile < mat_end_tile(p, tile) && m < p.M, 8)) {
            store_y(mt, nbase + r, m, v);
          }
        }
        if (warp == kWCompute - WPS && lane == 0) ZC(172 + 4 * pass);
        if (pass + 1 < kRedPasses && !tile_sync()) return false;  // the buffers are free again
        if (warp == kWCompute - WPS && lane == 0) ZC(173 + 4 * pass);
      }
      if (pub && ZCK > 0) {
        // the piece (this CTA's only tile) into the head CTA's shared memory, slot rank - 1
        fence_proxy_async_smem();  // this thread's writes of the piece, before the bulk copy reads them
        if (!tile_sync()) return false;
        if (warp == 0 && lane == 0) {
          const uint32_t rank = cluster_ctarank();
          if (ZOK(rank >= 1 && static_cast<int>(rank) < ZCK, 10)) {
            bulk_s2peer(mapa_peer(smem_u32(ZRX) + (rank - 1) * piece_bytes, 0), ZRX, piece_bytes,
                        mapa_peer(smem_u32(&ctl.pieces_in), 0));
            bulk_wait_read_all();  // the source stays valid until the copy has read it
          }
        }
        return true;
      }
      if (pub) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.piece_written);
      }
      return tile_sync();  // the buffers are free again
    };

    // set q takes units ui = q, q + US, ..: stage st = ui / US, one per step,
    // in slot s with fill parity ph (counters, not divisions)
    int f = 0, ui = q, st = 0, s = 0, ph = 0;
    int tile_end = static_cast<int>(min(u1, static_cast<int64_t>(t_first + 1) * G) - u0);  // first unit past the tile
    for (int tile = t_first; ok && tile <= t_last; ++tile, ++f, tile_end = min(nu, tile_end + G)) {
      for (; ok && ui < tile_end; ui += US) {
        if (!(ok = ZW(mbar_wait(&ctl.full[s], ph, abort_flag, tmo, p.err), 0))) break;
        if (warp == 0 && lane == 0 && st < 16) ZC(32 + st);
        if (warp == kWCompute - WPS && lane == 0 && st < 16) ZC(48 + st);
        const uint8_t* sg = stage(s);
        const uint8_t* img = sg + q * kArec;
        const uint8_t* rec = sg + kAct + q * kWRecBytes;
        group_product(rec, 2048, rw, reinterpret_cast<const uint16_t*>(rec + kWRecScales), img, u0 + ui, -1);
        if (warp == 0 && lane == 0 && st < 16) ZC(230 + st);
        const int e = ctl.map[ui][half];
        if (e >= 0) {  // the residual block of this warp's half
          const int cpos = ctl.rpos[ui][half], slot = cpos % kRS;
          // Sets run up to a few stages apart, so this slot may still hold (or await) a record two
          // laps older: its parity would alias.  Once record cpos is issued, every older record of
          // the slot has been consumed and the newer one waits for this warp: the parity is exact.
          if (!(ok = ZW(count_wait(&ctl.r_issued, cpos, abort_flag, tmo, p.err), 1))) break;
          if (!(ok = ZW(mbar_wait(&ctl.r_full[slot], (cpos / kRS) & 1, abort_flag, tmo, p.err), 1))) break;
          const uint8_t* rrec = rring + slot * kRRecBytes;
          group_product(rrec, 1024, rw - 64 * half, reinterpret_cast<const uint16_t*>(rrec + kRRecScales), img,
                        u0 + ui, e);
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.r_empty[slot]);
        }
        __syncwarp();
        if (warp == 0 && lane == 0 && st < 8) ZC(246 + st);
        if (lane == 0) mbar_arrive(&ctl.empty[s]);  // this warp is done with the stage
        ++st;
        if (++s == S) s = 0, ph ^= 1;
      }
      if (warp == 0 && lane == 0 && f < 8) ZC(64 + f);
      if (warp == kWCompute - WPS && lane == 0 && f < 8) ZC(72 + f);
      if (ok && !kDebug) ok = flush(tile);
      if (warp == kWCompute - WPS && lane == 0 && f < 8) ZC(80 + f);
    }

    // Finish the tiles whose count this CTA completed: after every compute
    // warp's last tile end the stage memory is idle; every piece is brought
    // into it with bulk copies (one per lane), summed in CTA order, stored.
  }

  // Every role is done.
  if (warp == kWCompute - WPS && lane == 0) ZC(90);
  __syncwarp();
  if (lane == 0) mbar_arrive(&ctl.exit_bar);
  mbar_wait(&ctl.exit_bar, 0, abort_flag, tmo, p.err);
  __syncthreads();
  if (threadIdx.x == 0) {
    ZT(5);
    ZC(7);
  }
  if (*abort_flag) {
    // A wait gave up: copies may still be in flight; give them 200 us.
    if (threadIdx.x == 0) {
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 200000ull) {
      }
    }
    __syncthreads();
  }
#undef ZCK
#undef ZRX
}

// ---------------------------------------------------------------------------
// Decode GEMM, column form (warp MMA, quantizer inside; the default for M <= 32)
// ---------------------------------------------------------------------------
// The launch's tiles are taken T at a time (T = the sets of compute warps: 4
// up to 16 tokens, 2 at 32), and a "column" is one 128-input group of such a
// tile-group.  One shared-memory stage holds one column: the T tiles' base
// records of the group and the group's activations (X rows as they are, or
// packed codes and scales).  Set q owns tile q of every tile-group, so its
// accumulators stay on one tile for the CTA's whole share of the tile-group,
// and the group's activation image (E4M3 codes in the MMA's B-fragment order,
// 2^9 sx, offset terms) is built once per stage in shared memory by all 16
// compute warps: the activation quantizer runs inside the GEMM, one stage
// ahead of the MMAs, on data the producer has already brought in.
//
// CTAs take equal contiguous ranges of columns (stream-K over every SM).  A
// tile-group cut by range boundaries is finished by the CTA holding its first
// group: every other CTA on it publishes a piece (its fp32 partial sums, in
// register-fragment order, so writes and reads are whole 256-byte rows per
// warp) and a flag; the finisher adds the pieces in CTA order (deterministic).

template <int TN>
struct ColGeo {
  static constexpr int T = w_sets(TN);                       // tiles per tile-group
  static constexpr int kImg = TN * 136;                      // B fragments, then {2^9 sx, c} per token pair
  static constexpr int kOffRec = (kImg + 127) / 128 * 128;   // T base records
  static constexpr int kOffRaw = kOffRec + T * kWRecBytes;   // X rows [TN][128] x 2 bytes, or codes [TN][64] + scales
  static constexpr int kRaw = TN * 256;
  static constexpr int kOffScales = TN * 64;                 // packed input: the scales after the codes
  static constexpr int kStage = (kOffRaw + kRaw + 127) / 128 * 128;
  static constexpr int kMaxCols = kMaxUnits / T;             // columns per CTA at most (residual map size)
  static constexpr int kPieceU64 = T * TN * 64;              // a piece: T tiles x 128 rows x TN tokens, fp32 pairs
};
static_assert(kWRecBytes % 128 == 0, "base records keep 128-byte alignment in a stage");

template <int kMaxCols, int T>
struct __align__(16) CCtl {
  uint64_t full[kMaxStages];    // the stage's base records landed
  uint64_t xfull[kMaxStages];   // the stage's activations landed
  uint64_t built[kMaxStages];   // every compute warp wrote its share of the stage's image
  uint64_t empty[kMaxStages];   // every compute warp is done with the stage
  uint64_t r_full[kRS];
  uint64_t r_empty[kRS];        // the warps of the record's 64-row half
  uint64_t map_ready;
  uint64_t piece_written;       // every compute warp wrote its share of this CTA's piece
  uint64_t pieces_in;           // the other CTAs' pieces of the tile-group this CTA finishes are readable
  uint64_t exit_bar;
  int32_t map[kMaxCols][T][2];  // CSR entry of the residual block of (column, tile, half), or -1
  int32_t rpos[kMaxCols][T][2]; // its position in the residual ring order
  const uint8_t* rsrc[kMaxCols][T];  // residual records of the tile's matrix
  int abort_flag;
  volatile int r_issued;        // residual records issued so far (in ring order)
};

__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t ld_global_cg_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.global.cg.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_global_cg_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.global.cg.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// Two floats holding integers |q| <= 7 -> their E4M3 bytes (exact), `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_of(float hi, float lo) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight inputs of one token (inputs 8k..8k+7 of a group) quantized with the
// token's scale s (an fp16 value, nonzero) and r = 1/s rounded to fp32:
// q = clamp(RNE(v / s), -7, 7), as the quantizer's IEEE division gives it.
// The quotient is refined once, q1 = q0 + (v - q0 s) r with q0 = v r (the
// residual exact in the fma), which puts q1 within 2^-20 of v / s and equal
// to it where v / s is a half-integer; an input and a scale of at most 11
// significant bits never put v / s closer than 2^-13 to a half-integer of
// magnitude 1/2 or more unless it is one, so rint(q1) is the exact
// round-half-even.  Out: the codes as floats.
__device__ __forceinline__ void quant8(const float (&v)[8], float s, float r, float (&q)[8]) {
  const uint64_t r2 = f2pack(r, r), ns2 = f2pack(-s, -s);
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const uint64_t v2 = f2pack(v[i], v[i + 1]);
    const uint64_t q0 = f2mul(v2, r2);
    const uint64_t e = f2fma(q0, ns2, v2);
    const uint64_t q1 = f2fma(e, r2, q0);
    float a, b;
    f2unpack(q1, a, b);
    q[i] = fminf(fmaxf(rintf(a), -7.0f), 7.0f);
    q[i + 1] = fminf(fmaxf(rintf(b), -7.0f), 7.0f);
  }
}

// TN: tokens per tile (8, 16 or 32); kDebug: write raw group dots.
template <int TN, bool kDebug>
__global__ void __launch_bounds__(w_threads(TN), 1) zipper_col_kernel(const ZParams p) {
  using Geo = ColGeo<TN>;
  constexpr int NB = TN / 8;                                // 8-token blocks of one MMA
  constexpr int MT = w_mt(TN), WPS = w_wps(TN), T = Geo::T;  // 16-row MMA tiles per warp, warps per set, sets
  constexpr int kWCompute = 16, kWProd = kWCompute, kWEpi = kWCompute + 1, kWThreads = w_threads(TN);
  extern __shared__ uint8_t smem_raw[];
  __shared__ CCtl<Geo::kMaxCols, T> ctl;
  uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  const int S = p.nstages, SB = p.stage_bytes, G = p.G;
  uint8_t* stages = smem;
  uint8_t* rring = smem + static_cast<size_t>(S) * SB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t C32 = static_cast<uint32_t>(p.units), P32 = static_cast<uint32_t>(p.ctas), c32 = blockIdx.x;
  const int64_t P = P32, c = c32;
  const int col0 = static_cast<int>(first_unit32(c32, C32, P32)), col1 = static_cast<int>(first_unit32(c32 + 1, C32, P32));
  const int nstg = col1 - col0;  // one stage per column
  // Stream-K roles (per tile-group): a CTA publishes at most one piece (its
  // first tile-group, when its range starts inside it) and finishes at most
  // one tile-group (its last, when its range holds that tile-group's first
  // group but not its last).
  const int t_first = col0 / G, t_last = (col1 - 1) / G;
  const bool publishes = !kDebug && col0 > t_first * G;
  const bool finishes = !kDebug && col0 <= t_last * G && col1 < (t_last + 1) * G;
  const int npc =
      finishes ? static_cast<int>(owner_of32(static_cast<uint32_t>((t_last + 1) * G - 1), C32, P32) - c32) : 0;
  auto piece_of = [&](int64_t cc) { return reinterpret_cast<uint64_t*>(p.part) + cc * Geo::kPieceU64; };
  volatile int* abort_flag = &ctl.abort_flag;
  const uint64_t tmo = p.timeout_ns;
  const uint32_t xbytes = p.raw ? static_cast<uint32_t>(p.M) * 256u : static_cast<uint32_t>(p.Mp) * 66u;

  if (warp == 0) {
    for (int s = lane; s < S; s += 32) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.xfull[s], 1);
      mbar_init(&ctl.built[s], kWCompute);
      mbar_init(&ctl.empty[s], kWCompute);
    }
    if (lane < kRS) {
      mbar_init(&ctl.r_full[lane], 1);
      mbar_init(&ctl.r_empty[lane], WPS / 2);  // the warps of the record's 64-row half
    }
    if (lane == 11) mbar_init(&ctl.map_ready, 1);
    if (lane == 12) mbar_init(&ctl.piece_written, kWCompute);
    if (lane == 13) mbar_init(&ctl.pieces_in, 1);
    if (lane == 14) mbar_init(&ctl.exit_bar, kWThreads / 32);
    if (lane == 15) ctl.abort_flag = 0;
    if (lane == 16) ctl.r_issued = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();
  auto stage = [&](int s) { return stages + static_cast<size_t>(s) * SB; };

  if (warp == kWProd) {
    // ---------------- producer: a stage = one column's T base records and its group's activations;
    // then the residual records, in ring order ----------------
    auto issue_w = [&](int st, int sl) {  // the stage's base records (lane q: tile q of the tile-group)
      const int cc = col0 + st, tg = cc / G, gg = cc - tg * G;
      const int nt = min(T, p.tiles - tg * T);
      if (lane < nt) {
        const int tt = tg * T + lane;
        const ZMat& mt = p.mat[mat_of_tile(p, tt)];
        const uint8_t* src = mt.wpk + (static_cast<int64_t>(tt - mt.tile0) * G + gg) * kWRecBytes;
        if (ZOK((reinterpret_cast<uintptr_t>(src) & 15u) == 0, 1))
          bulk_g2s(stage(sl) + Geo::kOffRec + lane * kWRecBytes, src, kWRecBytes, &ctl.full[sl]);
      }
      if (lane == 0) mbar_arrive_expect_tx(&ctl.full[sl], static_cast<uint32_t>(nt) * kWRecBytes);
    };
    auto issue_x = [&](int st, int sl) {  // the stage's activations: X rows (lane m), or codes + scales
      const int gg = (col0 + st) % G;
      uint8_t* raw = stage(sl) + Geo::kOffRaw;
      if (p.raw) {
        if (lane < p.M)
          bulk_g2s(raw + lane * 256, p.x + static_cast<int64_t>(lane) * p.ldx + static_cast<int64_t>(gg) * kGroup, 256u,
                   &ctl.xfull[sl]);
      } else {
        if (lane == 0)
          bulk_g2s(raw, p.xq + static_cast<int64_t>(gg) * p.Mp * 64, static_cast<uint32_t>(p.Mp) * 64u, &ctl.xfull[sl]);
        if (lane == 1)
          bulk_g2s(raw + Geo::kOffScales, p.xs + static_cast<int64_t>(gg) * p.Mp, static_cast<uint32_t>(p.Mp) * 2u,
                   &ctl.xfull[sl]);
      }
      if (lane == 0) mbar_arrive_expect_tx(&ctl.xfull[sl], xbytes);
    };
    const int pre = min(S, nstg);
    // The first stages' base records leave before the dependency wait (the
    // kernels that may run ahead of it never write packed weights); their
    // activations after it.
    for (int st = 0; st < pre; ++st) issue_w(st, st);
    pdl_wait();
    for (int st = 0; st < pre; ++st) issue_x(st, st);
    __syncwarp();
    bool ok = ZW(mbar_wait(&ctl.map_ready, 0, abort_flag, tmo, p.err), 7);
    ok = __all_sync(0xFFFFFFFFu, ok);
    int bst = pre, bs = 0, bph = 1;  // next stage, its slot, the slot's fill parity
    int rf = 0;                       // next (column, tile, half) whose residual record is due
    const int nf = 2 * T * nstg;
    uint64_t idle_since = 0;
    for (int idle = 0; ok && (bst < nstg || rf < nf);) {
      bool progress = false;
      const int rlim = min(nf, 2 * T * bst);
      if (rf < rlim) {
        const int f = rf + lane;
        bool ready = false;
        int e = -1, cpos = 0;
        if (f < rlim) {
          e = (&ctl.map[0][0][0])[f];
          cpos = e >= 0 ? (&ctl.rpos[0][0][0])[f] : 0;
          // the slot's previous record (cpos - kRS) has been issued, so the
          // slot's phase is one of two and the parity test is exact
          ready = e < 0 || cpos < kRS || mbar_test_wait(&ctl.r_empty[cpos % kRS], ((cpos / kRS) - 1) & 1);
        }
        const unsigned blocked = __ballot_sync(0xFFFFFFFFu, !ready);
        const int n = blocked ? __ffs(blocked) - 1 : 32;  // the ready prefix, in ring order
        if (lane < n && e >= 0) {
          const int slot = cpos % kRS;
          mbar_arrive_expect_tx(&ctl.r_full[slot], kRRecBytes);
          bulk_g2s(rring + slot * kRRecBytes, (&ctl.rsrc[0][0])[f >> 1] + static_cast<int64_t>(e) * kRRecBytes,
                   kRRecBytes, &ctl.r_full[slot]);
        }
        const int nrec = __popc(__ballot_sync(0xFFFFFFFFu, lane < n && e >= 0));
        if (lane == 0 && nrec) ctl.r_issued = ctl.r_issued + nrec;
        rf += n;
        progress = n > 0;
      }
      if (bst < nstg) {
        int go = 0;
        if (lane == 0 && mbar_test_wait(&ctl.empty[bs], bph ^ 1)) go = 1;
        if (__shfl_sync(0xFFFFFFFFu, go, 0)) {
          issue_w(bst, bs);
          issue_x(bst, bs);
          ++bst;
          if (++bs == S) bs = 0, bph ^= 1;
          progress = true;
        }
      }
      if (progress) {
        idle = 0;
        continue;
      }
      // back off (32 ns doubling to 512 ns): the polls share a scheduler with compute warps
      __nanosleep(32u << min(idle >> 2, 4));
      if ((++idle & 15) == 0) {  // bounded: give up after the timeout without progress
        int give_up = 0;
        if (lane == 0) {
          const uint64_t now = globaltimer();
          if (*abort_flag) {
            give_up = 1;
          } else if (idle == 16) {
            idle_since = now;
          } else if (now - idle_since > tmo) {
            ZW(false, 7);
            atomicOr(p.err, kDevErrTimeout);
            *abort_flag = 1;
            give_up = 1;
          }
        }
        ok = !__shfl_sync(0xFFFFFFFFu, give_up, 0);
      }
    }
    __syncwarp();
  } else if (warp == kWEpi) {
    // ---------------- epilogue: stream-K flags off the compute warps' path ----------------
    pdl_wait();  // the flags and pieces in the workspace may still be in use by the preceding kernel
    bool ok = true;
    if (publishes) {  // release this CTA's piece once every compute warp has written its share
      if (lane == 0) {
        ok = ZW(mbar_wait_sleep(&ctl.piece_written, 0, abort_flag, tmo, p.err), 4);
        if (ok) {
          fence_acq_rel_gpu();
          st_relaxed_gpu(p.tcount + c, 1);
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    }
    if (finishes && ok) {
      // the flags of the other pieces (lane j: CTA c + 1 + j), each cleared for
      // the next launch once seen; then the compute warps read the pieces
      for (int j0 = 0; ok && j0 < npc; j0 += 32) {
        const int j = j0 + lane;
        bool seen = true;
        if (j < npc && ZOK(c + 1 + j < P, 4) && (seen = ZW(flag_wait(p.tcount + c + 1 + j, abort_flag, tmo, p.err), 5)))
          p.tcount[c + 1 + j] = 0;
        ok = __all_sync(0xFFFFFFFFu, seen);
      }
      if (ok && lane == 0) mbar_arrive(&ctl.pieces_in);
    }
  } else {
    // ---------------- compute warps ----------------
    const int q = warp / WPS, wq = warp % WPS;    // set (= tile of the tile-group), row block within the set
    const int g = lane >> 2, t = lane & 3;         // MMA fragment coordinates
    const int rw = 16 * MT * wq, half = rw >> 6;   // first row of this warp, its residual half
    if (warp == 0) {
      // Residual map of the CTA's columns (CSR entry per column, tile and
      // half) and the records' ring positions.  The block lists are read
      // before the dependency wait, like the weights.
      int32_t* mp = &ctl.map[0][0][0];
      for (int i = lane; i < nstg * T * 2; i += 32) mp[i] = -1;
      __syncwarp();
      for (int tg = t_first; tg <= t_last; ++tg) {
        for (int qq = 0; qq < T; ++qq) {
          const int tt = tg * T + qq;
          if (tt >= p.tiles) break;
          const ZMat& mt = p.mat[mat_of_tile(p, tt)];
          if (mt.nnzb == 0) continue;
          const int64_t br = 2 * static_cast<int64_t>(tt - mt.tile0);
          const int a0 = max(0, min(mt.nnzb, mt.row_ptr[br]));
          const int a1 = max(a0, min(mt.nnzb, mt.row_ptr[br + 1]));
          const int a2 = max(a1, min(mt.nnzb, mt.row_ptr[br + 2]));
          for (int e = a0 + lane; e < a2; e += 32) {
            const int gg = mt.col_idx[e];
            if (gg < 0 || gg >= G) continue;
            const int cc = tg * G + gg;
            if (cc >= col0 && cc < col1) {
              ctl.map[cc - col0][qq][e >= a1 ? 1 : 0] = e;
              ctl.rsrc[cc - col0][qq] = mt.rpk;
            }
          }
        }
      }
      __syncwarp();
      const int nf = nstg * T * 2;
      const int chunk = (nf + 31) / 32, f0 = min(nf, lane * chunk), f1 = min(nf, f0 + chunk);
      int cnt = 0;
      for (int fx = f0; fx < f1; ++fx) cnt += mp[fx] >= 0;
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      int pos = incl - cnt;
      for (int fx = f0; fx < f1; ++fx)
        if (mp[fx] >= 0) (&ctl.rpos[0][0][0])[fx] = pos++;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.map_ready);
    }
    bool ok = ZW(mbar_wait(&ctl.map_ready, 0, abort_flag, tmo, p.err), 0);
    pdl_wait();  // X, Y and the workspace pieces may still be in use by the preceding kernel
    // accumulators: [mt][nb] pairs {row r, tokens 8nb+2t, +1}, {row r+8, same tokens}
    uint64_t acc[MT][NB][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) acc[mt][nb][0] = acc[mt][nb][1] = 0ull;

    // The image of a stage's group, built by every compute warp: lane
    // L = 32 warp + lane takes token m = L / 16 and its inputs 8k..8k+7,
    // k = L % 16 (one 8-code word of the image); a token's 16 lanes share a
    // half-warp.  Tokens M..TN-1 get zero codes, scales and offsets.
    int b_i = 0, b_s = 0, b_ph = 0;  // next stage to build, its slot, the slot's fill parity
    auto build_next = [&]() -> bool {
      if (!ZW(mbar_wait(&ctl.xfull[b_s], b_ph, abort_flag, tmo, p.err), 10)) return false;
      uint8_t* img = stage(b_s);
      const uint8_t* raw = img + Geo::kOffRaw;
      const int L = warp * 32 + lane;
      if (L < TN * 16) {  // whole warps
        const int m = L >> 4, k = L & 15;
        const bool real = m < p.M;
        const int gg = (col0 + b_i) % G;
        uint32_t ev, od;
        int sum;
        float sx;
        if (p.raw) {
          uint4 w = make_uint4(0u, 0u, 0u, 0u);
          if (real) w = *reinterpret_cast<const uint4*>(raw + m * 256 + k * 16);
          const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
          float v[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (p.x_bf16) {
              v[2 * i] = __uint_as_float(wv[i] << 16);
              v[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
            } else {
              v[2 * i] = __half2float(__ushort_as_half(static_cast<unsigned short>(wv[i] & 0xFFFFu)));
              v[2 * i + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(wv[i] >> 16)));
            }
          }
          float amax = 0.0f;
#pragma unroll
          for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
          const uint16_t sb = act_scale_bits(amax);
          const float sf = __half2float(__ushort_as_half(sb));
          float qf[8];
          if (sf != 0.0f) {
            quant8(v, sf, __frcp_rn(sf), qf);
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) qf[i] = 0.0f;
          }
          ev = e4m3x2_of(qf[2], qf[0]) | (e4m3x2_of(qf[6], qf[4]) << 16);
          od = e4m3x2_of(qf[3], qf[1]) | (e4m3x2_of(qf[7], qf[5]) << 16);
          const float fs = ((qf[0] + qf[1]) + (qf[2] + qf[3])) + ((qf[4] + qf[5]) + (qf[6] + qf[7]));
          sum = static_cast<int>(fs);
          sx = 512.0f * sf;
          // the quantized activations, as the quantizer writes them (once: the columns of tile-group 0)
          if (p.xq_out && col0 + b_i < G && m < p.Mp) {
            uint32_t pk = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) pk |= (static_cast<uint32_t>(static_cast<int>(qf[i])) & 0xFu) << (4 * i);
            *reinterpret_cast<uint32_t*>(p.xq_out + (static_cast<int64_t>(gg) * p.Mp + m) * 64 + k * 4) = pk;
            if (k == 0) p.xs_out[static_cast<int64_t>(gg) * p.Mp + m] = real ? sb : static_cast<uint16_t>(0);
          }
        } else {
          const uint32_t wv = real ? *reinterpret_cast<const uint32_t*>(raw + m * 64 + k * 4) : 0u;
          uint32_t lo, hi;
          int4x8_to_e4m3(wv, lo, hi);
          ev = prmt(lo, hi, 0x6420u);
          od = prmt(lo, hi, 0x7531u);
          sum = nibble_sum8(wv);
          sx = real ? 512.0f * __half2float(__ushort_as_half(
                                   *reinterpret_cast<const uint16_t*>(raw + Geo::kOffScales + m * 2)))
                    : 0.0f;
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        // codes 8k..8k+7 of token m: K-step k / 4, fragment lane 4 (m % 8) + k % 4 of block m / 8
        *reinterpret_cast<uint2*>(img + ((((k >> 2) * NB + (m >> 3)) * 32 + 4 * (m & 7) + (k & 3)) * 8)) =
            make_uint2(ev, od);
        if (k == 0) {
          float* sco = reinterpret_cast<float*>(img + TN * 128);  // {2^9 sx, 2^9 sx', c, c'} per token pair
          sco[(m >> 1) * 4 + (m & 1)] = sx;
          sco[(m >> 1) * 4 + 2 + (m & 1)] = static_cast<float>(sum) * (1.0f / 64.0f);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.built[b_s]);
      ++b_i;
      if (++b_s == S) b_s = 0, b_ph ^= 1;
      return true;
    };

    // One group's product for this warp's rows (the same arithmetic as the
    // warp-MMA form): codes (K-steps jstride apart, 16 bytes per row, first
    // row row0), the image's fragments and scale pairs, row scales sc; into
    // acc, or the test hook's dots.
    auto group_product = [&](const uint8_t* codes, int jstride, int row0, const uint16_t* sc, const uint8_t* img,
                             int tile, int gg, int e) {
      const uint8_t* wr = codes + (row0 + g) * 16 + t * 4;
      const float4* sg = reinterpret_cast<const float4*>(img + TN * 128) + t;  // token pairs 2t, 2t+1 of block nb
      float s[MT][2];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        s[mt][0] = __half2float(__ushort_as_half(sc[row0 + 16 * mt + g]));
        s[mt][1] = __half2float(__ushort_as_half(sc[row0 + 16 * mt + 8 + g]));
      }
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        float d[MT][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t a[MT][4];
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t w0 = *reinterpret_cast<const uint32_t*>(wr + j * jstride + mt * 256);        // row +0
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(wr + j * jstride + mt * 256 + 128);  // row +8
            unpack_u4(w0, a[mt][0], a[mt][2]);
            unpack_u4(w1, a[mt][1], a[mt][3]);
          }
          const uint2 b = *reinterpret_cast<const uint2*>(img + ((j * NB + nb) * 32 + lane) * 8);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            if (j == 0)
              mma_e4m3_z(d[mt], a[mt], b.x, b.y);
            else
              mma_e4m3(d[mt], a[mt], b.x, b.y);
          }
        }
        const uint64_t m1 = f2pack(-1.0f, -1.0f);
        const float4 f = sg[4 * nb];  // 2^9 sx (tokens 8nb+2t, +1), c (same tokens)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          if constexpr (kDebug) {
            const float ev[2][2] = {{d[mt][0] - f.z, d[mt][1] - f.w}, {d[mt][2] - f.z, d[mt][3] - f.w}};
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
                const int m = 8 * nb + 2 * t + cc, r = rw + 16 * mt + 8 * h + g;
                if (m < p.M) {
                  const int32_t dv = static_cast<int32_t>(ev[h][cc] * 512.0f);
                  if (e < 0)
                    p.dots_w[(static_cast<int64_t>(m) * (p.tiles * kTileN) + static_cast<int64_t>(tile) * kTileN + r) * G +
                             gg] = dv;
                  else
                    p.dots_r[(static_cast<int64_t>(m) * p.mat[0].nnzb + e) * 64 + (r & 63)] = dv;
                }
              }
          } else {
            const uint64_t sx2 = f2pack(f.x, f.y), c2 = f2pack(f.z, f.w);
            const uint64_t e0 = f2fma(c2, m1, f2pack(d[mt][0], d[mt][1]));  // row +0: exact 2^-9 D
            const uint64_t e1 = f2fma(c2, m1, f2pack(d[mt][2], d[mt][3]));  // row +8
            acc[mt][nb][0] = f2fma(sx2, f2mul(f2pack(s[mt][0], s[mt][0]), e0), acc[mt][nb][0]);
            acc[mt][nb][1] = f2fma(sx2, f2mul(f2pack(s[mt][1], s[mt][1]), e1), acc[mt][nb][1]);
          }
        }
      }
    };
    auto store_y = [&](const ZMat& mt, int64_t n, int m, float v) {
      const int64_t o = static_cast<int64_t>(m) * mt.ldy + n;
      if (p.y_f32)
        st_global_f32(static_cast<float*>(mt.y) + o, v);
      else
        st_global_b16(static_cast<__nv_bfloat16*>(mt.y) + o, __bfloat16_as_ushort(__float2bfloat16_rn(v)));
    };
    // End of this CTA's share of tile-group tg: the set's tile is complete
    // here (store Y), or is this CTA's piece (publish), or needs the later
    // CTAs' pieces first (finish: added in CTA order).  No cross-warp step.
    auto flush = [&](int tg) -> bool {
      const int tile = tg * T + q;
      const bool pub = publishes && tg == t_first;
      const bool fin = finishes && tg == t_last;
      const int64_t frag0 = static_cast<int64_t>((q * WPS + wq) * MT) * NB * 2 * 32 + lane;  // this lane's pairs
      if (fin) {
        if (!ZW(mbar_wait(&ctl.pieces_in, 0, abort_flag, tmo, p.err), 3)) return false;
        for (int j = 0; j < npc; ++j) {  // CTA order
          const uint64_t* pc = piece_of(c + 1 + j) + frag0;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
              for (int h = 0; h < 2; ++h)
                acc[mt][nb][h] = f2add(acc[mt][nb][h], ld_global_cg_u64(pc + ((mt * NB + nb) * 2 + h) * 32));
        }
      }
      if (pub) {
        uint64_t* pc = piece_of(c) + frag0;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int h = 0; h < 2; ++h) st_global_cg_u64(pc + ((mt * NB + nb) * 2 + h) * 32, acc[mt][nb][h]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.piece_written);
      } else if (tile < p.tiles) {
        const ZMat& mt = p.mat[mat_of_tile(p, tile)];
        const int64_t nbase = static_cast<int64_t>(tile - mt.tile0) * kTileN;
#pragma unroll
        for (int m2 = 0; m2 < MT; ++m2)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int r = rw + 16 * m2 + 8 * h + g, m0 = 8 * nb + 2 * t;
              float v0, v1;
              f2unpack(acc[m2][nb][h], v0, v1);
              if (m0 < p.M) store_y(mt, nbase + r, m0, v0);
              if (m0 + 1 < p.M) store_y(mt, nbase + r, m0 + 1, v1);
            }
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) acc[mt][nb][0] = acc[mt][nb][1] = 0ull;
      return true;
    };

    // Stages in order: build the image `ahead` stages in advance (every warp
    // its share), then wait for this stage's image and base records, run the
    // set's tile, release the stage.  Builds ahead let the warps drift apart
    // by that many stages (a residual block makes one set slower for a stage).
    const int ahead = min(2, S - 1);
    for (int i = 0; ok && i < min(ahead, nstg); ++i) ok = build_next();
    int s = 0, ph = 0;
    int tg = t_first, gg = col0 - t_first * G;
    for (int i = 0; ok && i < nstg; ++i) {
      if (b_i < nstg && !(ok = build_next())) break;
      if (!(ok = ZW(mbar_wait(&ctl.built[s], ph, abort_flag, tmo, p.err), 11))) break;
      if (!(ok = ZW(mbar_wait(&ctl.full[s], ph, abort_flag, tmo, p.err), 0))) break;
      const uint8_t* sg = stage(s);
      const int tile = tg * T + q;
      if (tile < p.tiles) {
        const uint8_t* rec = sg + Geo::kOffRec + q * kWRecBytes;
        group_product(rec, 2048, rw, reinterpret_cast<const uint16_t*>(rec + kWRecScales), sg, tile, gg, -1);
        const int e = ctl.map[i][q][half];
        if (e >= 0) {  // the residual block of this warp's half
          const int cpos = ctl.rpos[i][q][half], slot = cpos % kRS;
          // Sets run a few stages apart, so this slot may still hold (or await) a record two laps
          // older: its parity would alias.  Once record cpos is issued, every older record of the
          // slot has been consumed and the newer one waits for this warp: the parity is exact.
          if (!(ok = ZW(count_wait(&ctl.r_issued, cpos, abort_flag, tmo, p.err), 1))) break;
          if (!(ok = ZW(mbar_wait(&ctl.r_full[slot], (cpos / kRS) & 1, abort_flag, tmo, p.err), 1))) break;
          const uint8_t* rrec = rring + slot * kRRecBytes;
          group_product(rrec, 1024, rw - 64 * half, reinterpret_cast<const uint16_t*>(rrec + kRRecScales), sg, tile,
                        gg, e);
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.r_empty[slot]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.empty[s]);  // this warp is done with the stage
      if (++s == S) s = 0, ph ^= 1;
      if (++gg == G) {  // the tile-group's last group
        if (!kDebug && !(ok = flush(tg))) break;
        gg = 0;
        ++tg;
      }
    }
    if (ok && !kDebug && gg != 0) ok = flush(tg);  // a share ending inside a tile-group
  }

  // Every role is done.
  __syncwarp();
  if (lane == 0) mbar_arrive(&ctl.exit_bar);
  mbar_wait(&ctl.exit_bar, 0, abort_flag, tmo, p.err);
  __syncthreads();
  if (*abort_flag) {
    // A wait gave up: copies may still be in flight; give them 200 us.
    if (threadIdx.x == 0) {
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 200000ull) {
      }
    }
    __syncthreads();
  }
}

// The activation images of one launch, written to the workspace for the GEMM
// to bulk-copy: for group g, the MMA's B operand (the integer codes as E4M3
// bytes, K permuted inside each 8-code word like the weight unpack), 2^9 sx
// and the offset terms 2^-9 * 8 * sum_k qx.  From packed codes (xq, xs), or
// straight from X (kQuant: quantized here with mq_quantize_act's rule and
// bits; xq / xs written too when asked).  One CTA of 128 threads per (group,
// 8-token block): thread L takes token 8 blockIdx.y + L / 16 and the group's
// inputs 8k..8k+7, k = L % 16 (one 8-code word); a token's 16 threads share a
// half-warp.  Tokens M..TN-1 get zero codes, scales and offsets.
struct ImgParams {
  const uint8_t* xq;
  const uint16_t* xs;
  const uint16_t* x;
  int64_t ldx;
  int x_bf16;
  uint8_t* xq_out;
  uint16_t* xs_out;
  int M, Mp;
  uint8_t* act;
};

// kFrag: the warp-MMA form's layout (per K-step j and 8-token block nb, lane
// 4g + t holds token 8nb + g: the even codes 8t, 8t+2, .., 8t+6 of the K-step,
// then the odd ones; then {2^9 sx, 2^9 sx', c, c'} per token pair); else the
// tensor-memory form's swizzled tile (then 2^9 sx [TN], c [TN], padding).
template <int TN, bool kQuant, bool kFrag>
__global__ void __launch_bounds__(128) act_image_kernel(const ImgParams p) {
  constexpr int kArec = kFrag ? TN * 136 : act_rec_bytes(TN);
  constexpr int NB = TN / 8;
  const int64_t g = blockIdx.x;
  const int m = static_cast<int>(blockIdx.y) * 8 + static_cast<int>(threadIdx.x >> 4), k = threadIdx.x & 15;
  const bool real = m < p.M;
  pdl_trigger();
  // This CTA usually starts while the preceding kernel still runs: bring its
  // rows of X into L2 meanwhile (L2 is coherent with that kernel's writes, so
  // a line fetched early still reads the final values), one request per
  // 128-byte line.
  if constexpr (kQuant)
    if (real && (k & 7) == 0)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p.x + static_cast<int64_t>(m) * p.ldx + g * kGroup + 8 * k));
  // the inputs are the preceding kernel's output, and the previous GEMM may
  // still be reading the images this overwrites
  pdl_wait();
  uint8_t* rec = p.act + g * kArec;
  float* sco = reinterpret_cast<float*>(rec + TN * 128);
  uint32_t ev, od;
  int sum;
  float sx;
  if constexpr (kQuant) {
    uint32_t wv[4] = {0u, 0u, 0u, 0u};
    if (real) {  // x is 8-byte aligned and ldx a multiple of 4
      const uint2* src = reinterpret_cast<const uint2*>(p.x + static_cast<int64_t>(m) * p.ldx + g * kGroup + 8 * k);
      const uint2 a = src[0], b = src[1];
      wv[0] = a.x, wv[1] = a.y, wv[2] = b.x, wv[3] = b.y;
    }
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (p.x_bf16) {
        v[2 * i] = __uint_as_float(wv[i] << 16);
        v[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
      } else {
        v[2 * i] = __half2float(__ushort_as_half(static_cast<unsigned short>(wv[i] & 0xFFFFu)));
        v[2 * i + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(wv[i] >> 16)));
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const uint16_t sb = act_scale_bits(amax);
    const float sf = __half2float(__ushort_as_half(sb));
    float qf[8];
    if (sf != 0.0f) {
      quant8(v, sf, __frcp_rn(sf), qf);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) qf[i] = 0.0f;
    }
    ev = e4m3x2_of(qf[2], qf[0]) | (e4m3x2_of(qf[6], qf[4]) << 16);
    od = e4m3x2_of(qf[3], qf[1]) | (e4m3x2_of(qf[7], qf[5]) << 16);
    sum = static_cast<int>(((qf[0] + qf[1]) + (qf[2] + qf[3])) + ((qf[4] + qf[5]) + (qf[6] + qf[7])));
    sx = 512.0f * sf;
    if (p.xq_out && m < p.Mp) {
      uint32_t pk = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) pk |= (static_cast<uint32_t>(static_cast<int>(qf[i])) & 0xFu) << (4 * i);
      *reinterpret_cast<uint32_t*>(p.xq_out + (g * p.Mp + m) * 64 + k * 4) = pk;
      if (k == 0) p.xs_out[g * p.Mp + m] = real ? sb : static_cast<uint16_t>(0);
    }
  } else {
    const uint32_t wv = real ? *reinterpret_cast<const uint32_t*>(p.xq + (g * p.Mp + m) * 64 + k * 4) : 0u;
    uint32_t lo, hi;
    int4x8_to_e4m3(wv, lo, hi);
    ev = prmt(lo, hi, 0x6420u);
    od = prmt(lo, hi, 0x7531u);
    sum = nibble_sum8(wv);
    sx = real ? 512.0f * __half2float(__ushort_as_half(p.xs[g * p.Mp + m])) : 0.0f;
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  if (m >= TN) return;
  const int off = kFrag ? ((((k >> 2) * NB + (m >> 3)) * 32 + 4 * (m & 7) + (k & 3)) * 8) : act_word_offset(m, k);
  *reinterpret_cast<uint2*>(rec + off) = make_uint2(ev, od);
  if (k == 0) {
    sco[kFrag ? (m >> 1) * 4 + (m & 1) : m] = sx;
    sco[kFrag ? (m >> 1) * 4 + 2 + (m & 1) : TN + m] = static_cast<float>(sum) * (1.0f / 64.0f);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

size_t a256(size_t b) { return (b + 255) / 256 * 256; }

int sm_count_current() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

struct ZPlan {
  bool tc;   // the tensor-memory form
  bool col;  // the column form (else, without tc, the warp-MMA form)
  int tn, mld, ctas, nstages, stage_bytes, smem, arec;
  int64_t units;  // units, or columns in the column form
  size_t o_act, o_part, o_q, o_s, bytes;  // workspace layout after the zeroed prefix
  int cluster = 0;  // warp-MMA form: CTAs per cluster (one tile per cluster), or 0
  int rx_off = 0;   // its received pieces' offset in dynamic shared memory
};

// The decode kernel's form: 4 warp-MMA (the default), or as MQ_DECODE_VARIANT
// forces it (benchmarks and tests): 3 tensor-memory ("tc"), 5 column ("col").
int decode_form() {
  const char* v = getenv("MQ_DECODE_VARIANT");
  if (v && strcmp(v, "tc") == 0) return 3;
  if (v && strcmp(v, "col") == 0) return 5;
  return 4;
}

constexpr int kMinCols = 2;  // columns per CTA at least (bounds the pieces a tile-group is cut into)

// Static shared memory of the column form's control block (with its alignment slack).
template <int TN>
int c_ctl_bytes() {
  return (static_cast<int>(sizeof(CCtl<ColGeo<TN>::kMaxCols, ColGeo<TN>::T>)) + 127) / 128 * 128;
}

// Plan for M tokens over `tiles` 128-row tiles of K inputs; false if the
// decode kernel does not cover the shape.
// Static shared memory of the warp-MMA form's control block (with its alignment slack).
template <int TN>
int w_ctl_bytes() {
  return (static_cast<int>(sizeof(WCtl<kMaxUnits / w_sets(TN) + 1>)) + 127) / 128 * 128;
}

constexpr int kMaxClusterCtas = 8;           // portable cluster size
constexpr int kClusterRxBytes = 48 * 1024;   // the head CTA's room for its peers' pieces

// Clusters of k CTAs of the warp-MMA form (dynamic shared memory `smem`) that
// the current device holds at once, or 0; asked once per (device, size).
template <int TN>
int w_max_clusters(int dev, int k, int smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int>, int> cache;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_tuple(dev, k, smem);
  const auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  auto kern = zipper_warp_kernel<TN, false>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit - w_ctl_bytes<TN>()) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(k), 1, 1);
    cfg.blockDim = dim3(w_threads(TN), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(k);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();  // a refused query leaves no sticky error behind
  cache[key] = n;
  return n;
}

// Cluster mode is on unless MQ_DECODE_CLUSTER is "0" (benchmarks and tests).
bool cluster_mode_allowed() {
  const char* v = getenv("MQ_DECODE_CLUSTER");
  return !(v && strcmp(v, "0") == 0);
}

bool zplan(int64_t M, int64_t tiles, int64_t K, ZPlan* out) {
  if (M < 1 || M > 32) return false;
  ZPlan pl = {};
  const int form = decode_form();
  pl.tc = form == 3;
  pl.col = form == 5;
  pl.tn = pl.tc ? (M <= 16 ? 16 : 32) : (M <= 8 ? 8 : M <= 16 ? 16 : 32);
  pl.mld = M <= 4 ? 4 : M <= 8 ? 8 : M <= 16 ? 16 : 32;
  const int64_t G = K / kGroup;
  pl.units = tiles * G;
  const int sms = sm_count_current();
  if (sms <= 0 || sms > kWsZeroBytes / 4) return false;
  if (pl.col) {
    // columns: (tile-group of T tiles, group); one stage per column
    const int T = w_sets(pl.tn);
    const int64_t ncol = (tiles + T - 1) / T * G;
    pl.units = ncol;
    pl.ctas = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(sms, ncol / kMinCols)));
    if ((ncol + pl.ctas - 1) / pl.ctas > kMaxUnits / T || ncol >= (int64_t{1} << 31)) return false;
    int ctl_bytes;
    switch (pl.tn) {
      case 8: pl.stage_bytes = ColGeo<8>::kStage, ctl_bytes = c_ctl_bytes<8>(); break;
      case 16: pl.stage_bytes = ColGeo<16>::kStage, ctl_bytes = c_ctl_bytes<16>(); break;
      default: pl.stage_bytes = ColGeo<32>::kStage, ctl_bytes = c_ctl_bytes<32>(); break;
    }
    const int fixed = 128 + kRS * kRRecBytes;  // alignment, residual ring
    pl.nstages = std::min(kMaxStages, (kSmemLimit - ctl_bytes - fixed) / pl.stage_bytes);
    if (pl.nstages < 2) return false;
    pl.smem = pl.nstages * pl.stage_bytes + fixed;
    // workspace: the zeroed prefix (flags [ctas]), the stream-K pieces, and
    // the quantized activations for inputs the stages cannot copy directly
    const size_t Mp = static_cast<size_t>((M + 7) / 8 * 8);
    pl.o_part = kWsZeroBytes;
    pl.o_q = pl.o_part + a256(static_cast<size_t>(pl.ctas) * T * pl.tn * kTileN * sizeof(float));
    pl.o_s = pl.o_q + a256(static_cast<size_t>(G) * Mp * 64);
    pl.bytes = pl.o_s + a256(static_cast<size_t>(G) * Mp * 2);
    *out = pl;
    return true;
  }
  pl.ctas = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(sms, pl.units / kMinUnits)));
  if ((pl.units + pl.ctas - 1) / pl.ctas > kMaxUnits || pl.units >= (int64_t{1} << 31)) return false;
  int ctl_bytes, fixed;
  if (pl.tc) {
    pl.arec = act_rec_bytes(pl.tn);
    pl.stage_bytes = kUS * (pl.arec + kWRecBytes);  // a multiple of 1024
    ctl_bytes = (static_cast<int>(sizeof(ZCtl)) + 127) / 128 * 128;
    fixed = 1024 + kRS * kRRecBytes;
  } else {
    pl.arec = pl.tn * 136;
    pl.stage_bytes = (w_sets(pl.tn) * (pl.arec + kWRecBytes) + 127) / 128 * 128;
    ctl_bytes = pl.tn == 32 ? w_ctl_bytes<32>() : w_ctl_bytes<8>();
    // alignment, residual ring, tile partials (one pass over 8 tokens, two over 16 or 32)
    fixed = 128 + kRS * kRRecBytes + w_sets(pl.tn) * (kTileN + 4) * (pl.tn == 8 ? 8 : pl.tn / 2) * 4;
  }
  pl.nstages = std::min(kMaxStages, (kSmemLimit - ctl_bytes - fixed) / pl.stage_bytes);
  if (pl.nstages < 2) return false;
  pl.smem = pl.nstages * pl.stage_bytes + fixed;
  // Cluster mode (warp-MMA form): when k CTAs per tile over all tiles use
  // about as many SMs as stream-K would, each tile gets a cluster of k CTAs
  // (the stream-K partition over tiles x k CTAs then cuts tiles only inside
  // clusters) and the pieces travel by bulk copy into the head CTA's shared
  // memory instead of through the workspace and flags.
  if (!pl.tc && cluster_mode_allowed() && tiles > 0) {
    const int64_t kk = std::min<int64_t>(
        {kMaxClusterCtas, sms / tiles, G, kClusterRxBytes / (M * kTileN * 4) + 1});
    if (kk >= 2 && tiles * kk * 10 >= static_cast<int64_t>(pl.ctas) * 8 && (G + kk - 1) / kk <= kMaxUnits) {
      const int rx = static_cast<int>((kk - 1) * M * kTileN * 4 + 127) / 128 * 128;
      const int ns = std::min(kMaxStages, (kSmemLimit - ctl_bytes - fixed - rx) / pl.stage_bytes);
      const int smem = ns * pl.stage_bytes + fixed + rx;
      int dev = 0;
      const int fits = ns < 2 || cudaGetDevice(&dev) != cudaSuccess ? 0
                       : pl.tn == 8                                  ? w_max_clusters<8>(dev, static_cast<int>(kk), smem)
                       : pl.tn == 16                                 ? w_max_clusters<16>(dev, static_cast<int>(kk), smem)
                                                                     : w_max_clusters<32>(dev, static_cast<int>(kk), smem);
      if (fits >= tiles) {
        pl.cluster = static_cast<int>(kk);
        pl.ctas = static_cast<int>(tiles * kk);
        pl.nstages = ns;
        pl.smem = smem;
        pl.rx_off = ns * pl.stage_bytes + (fixed - 128);  // after the stages, the ring and the tile partials
      }
    }
  }
  // workspace: the zeroed prefix (tile counters [ctas]), the activation
  // images, the stream-K pieces
  pl.o_act = kWsZeroBytes;
  pl.o_part = pl.o_act + a256(static_cast<size_t>(G) * pl.arec);
  pl.bytes = pl.o_part + a256(static_cast<size_t>(pl.ctas) * 2 * pl.tn * kTileN * sizeof(float));
  *out = pl;
  return true;
}

template <int TN, int MLD, bool kDebug>
mq_status zlaunch(const ZParams& zp, const ZPlan& pl, cudaStream_t stream) {
  auto kern = zipper_decode_kernel<TN, MLD, kDebug>;
  static std::mutex mu;
  static bool attr_set[64];  // per device, per instantiation
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return launch_status("zipper: device");
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!attr_set[dev]) {
      // static shared memory (the control block) and dynamic together stay within the per-block limit
      const int ctl_bytes = (static_cast<int>(sizeof(ZCtl)) + 127) / 128 * 128;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit - ctl_bytes) != cudaSuccess)
        return launch_status("zipper: smem attribute");
      attr_set[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.ctas), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, zp) != cudaSuccess) return launch_status("zipper launch");
  return launch_status("zipper");
}

template <bool kDebug>
mq_status zdispatch(const ZParams& zp, const ZPlan& pl, cudaStream_t stream) {
  switch (pl.mld) {
    case 4: return zlaunch<16, 4, kDebug>(zp, pl, stream);
    case 8: return zlaunch<16, 8, kDebug>(zp, pl, stream);
    case 16: return zlaunch<16, 16, kDebug>(zp, pl, stream);
    default: return zlaunch<32, 32, kDebug>(zp, pl, stream);
  }
}

template <int TN, bool kDebug>
mq_status wlaunch(const ZParams& zp, const ZPlan& pl, cudaStream_t stream) {
  auto kern = zipper_warp_kernel<TN, kDebug>;
  // (the debug form ignores cluster mode: the same partition, no exchange)
  static std::mutex mu;
  static bool attr_set[64];  // per device, per instantiation
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return launch_status("zipper: device");
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!attr_set[dev]) {
      const int ctl_bytes = w_ctl_bytes<TN>();
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit - ctl_bytes) != cudaSuccess)
        return launch_status("zipper: smem attribute");
      attr_set[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.ctas), 1, 1);
  cfg.blockDim = dim3(w_threads(TN), 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!kDebug && pl.cluster > 0) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(pl.cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  if (cudaLaunchKernelEx(&cfg, kern, zp) != cudaSuccess) return launch_status("zipper launch");
  return launch_status("zipper");
}

template <int TN, bool kDebug>
mq_status claunch(const ZParams& zp, const ZPlan& pl, cudaStream_t stream) {
  auto kern = zipper_col_kernel<TN, kDebug>;
  static std::mutex mu;
  static bool attr_set[64];  // per device, per instantiation
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return launch_status("zipper: device");
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!attr_set[dev]) {
      const int ctl_bytes = c_ctl_bytes<TN>();
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit - ctl_bytes) != cudaSuccess)
        return launch_status("zipper: smem attribute");
      attr_set[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.ctas), 1, 1);
  cfg.blockDim = dim3(w_threads(TN), 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, zp) != cudaSuccess) return launch_status("zipper launch");
  return launch_status("zipper");
}

template <bool kDebug>
mq_status cdispatch(const ZParams& zp, const ZPlan& pl, cudaStream_t stream) {
  switch (pl.tn) {
    case 8: return claunch<8, kDebug>(zp, pl, stream);
    case 16: return claunch<16, kDebug>(zp, pl, stream);
    default: return claunch<32, kDebug>(zp, pl, stream);
  }
}

template <bool kDebug>
mq_status wdispatch(const ZParams& zp, const ZPlan& pl, cudaStream_t stream) {
  switch (pl.tn) {
    case 8: return wlaunch<8, kDebug>(zp, pl, stream);
    case 16: return wlaunch<16, kDebug>(zp, pl, stream);
    default: return wlaunch<32, kDebug>(zp, pl, stream);
  }
}

template <int TN, bool kQuant, bool kFrag>
mq_status image_launch(const ImgParams& ip, int G, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(G), TN / 8, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, act_image_kernel<TN, kQuant, kFrag>, ip) != cudaSuccess) return launch_status("image launch");
  return launch_status("image");
}

}  // namespace

mq_status quantize_act_launch(const void* x, mq_dtype xt, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                              uint16_t* xs, cudaStream_t stream);

// Workspace bytes of the decode kernel for M tokens over `tiles` tiles of K
// inputs on the current device, or 0 when it does not cover the shape.
size_t zipper_workspace_bytes(int64_t M, int64_t tiles, int64_t K) {
  ZPlan pl;
  return zplan(M, tiles, K, &pl) ? pl.bytes : 0;
}

// Plan summary for mq_gemm_plan: {form (3 tensor-memory, 4 warp-MMA, 5 column), tokens per tile, CTAs, stages,
// CTAs per cluster (1: no clusters)}.
bool zipper_plan_info(int64_t M, int64_t tiles, int64_t K, int32_t* form, int32_t* tn, int32_t* ctas, int32_t* stages,
                      int32_t* cluster) {
  ZPlan pl;
  if (!zplan(M, tiles, K, &pl)) return false;
  *form = pl.tc ? 3 : pl.col ? 5 : 4;
  *tn = pl.tn;
  *ctas = pl.ctas;
  *stages = pl.nstages;
  *cluster = pl.cluster > 0 ? pl.cluster : 1;
  return true;
}

// The kernel choice for (M, N, K) on the current device: {form (3: tensor
// memory, 4: warp MMA, 5: column), tokens per tile, CTAs per cluster, CTAs, stages} for the decode
// kernel, else zeros (the general kernel runs).
bool image_form_wanted(int64_t M);
void image_plan_info(int64_t M, int64_t N, int64_t K, int32_t* tn, int32_t* ctas);

mq_status gemm_plan_info(int64_t M, int64_t N, int64_t K, int32_t* info) {
  for (int i = 0; i < 5; ++i) info[i] = 0;
  zipper_plan_info(M, N / kTileN, K, &info[0], &info[1], &info[3], &info[4], &info[2]);
  if (info[0] == 0 && image_form_wanted(M)) {  // the general kernel's image form
    info[0] = 6;
    image_plan_info(M, N, K, &info[1], &info[3]);
  }
  return MQ_OK;
}

// One launch of the decode kernel over `nmat` matrices that share the
// activations: from packed activations (xq, xs) or, when x is given, from X
// (quantized in the prologue; xq_out / xs_out optional).  `handled` is false
// when the shape is not covered (the caller runs the general kernel).
mq_status zipper_launch(bool* handled, int nmat, const uint8_t* const* wpk, const int64_t* N,
                        const int32_t* const* row_ptr, const int32_t* const* col_idx, const int64_t* nnzb,
                        const uint8_t* const* rpk, void* const* y, const int64_t* ldy, mq_dtype yt, const uint8_t* xq,
                        const uint16_t* xs, const void* x, mq_dtype xt, int64_t ldx, uint8_t* xq_out,
                        uint16_t* xs_out, int64_t M, int64_t K, int32_t* dots_w, int32_t* dots_r, void* ws,
                        size_t ws_bytes, cudaStream_t stream) {
  *handled = false;
  if (nmat < 1 || nmat > kMaxMats) return set_error(MQ_ERR_INVALID_ARG, "zipper: 1 to %d matrices", kMaxMats);
  int64_t tiles = 0;
  for (int i = 0; i < nmat; ++i) tiles += N[i] / kTileN;
  ZPlan pl;
  if (!zplan(M, tiles, K, &pl)) return MQ_OK;
  *handled = true;
  if (ws == nullptr || ws_bytes < pl.bytes || !aligned(ws, 256))
    return set_error(MQ_ERR_WORKSPACE, "gemm: workspace of %zu bytes (256-aligned) needed, %zu given", pl.bytes,
                     ws_bytes);
  ZParams zp = {};
  int64_t t0 = 0;
  for (int i = 0; i < nmat; ++i) {
    zp.mat[i].wpk = wpk[i];
    zp.mat[i].row_ptr = row_ptr[i];
    zp.mat[i].col_idx = col_idx[i];
    zp.mat[i].rpk = rpk[i];
    zp.mat[i].y = y ? y[i] : nullptr;
    zp.mat[i].ldy = ldy ? ldy[i] : N[i];
    zp.mat[i].tile0 = static_cast<int>(t0);
    zp.mat[i].nnzb = static_cast<int>(nnzb[i]);
    t0 += N[i] / kTileN;
  }
  zp.nmat = nmat;
  zp.xq = xq;
  zp.xs = xs;
  zp.x = static_cast<const uint16_t*>(x);
  zp.ldx = ldx;
  zp.x_bf16 = xt == MQ_BF16;
  zp.xq_out = xq_out;
  zp.xs_out = xs_out;
  zp.M = static_cast<int>(M);
  zp.Mp = static_cast<int>((M + 7) / 8 * 8);
  zp.G = static_cast<int>(K / kGroup);
  zp.tiles = static_cast<int>(tiles);
  zp.ctas = pl.ctas;
  zp.nstages = pl.nstages;
  zp.stage_bytes = pl.stage_bytes;
  zp.units = pl.units;
  zp.y_f32 = yt == MQ_F32;
  zp.cluster = pl.cluster;
  zp.rx_off = pl.rx_off;
  zp.dots_w = dots_w;
  zp.dots_r = dots_r;
  uint8_t* w = static_cast<uint8_t*>(ws);
  zp.act = w + pl.o_act;
  zp.tcount = reinterpret_cast<int32_t*>(w);
  zp.part = reinterpret_cast<float*>(w + pl.o_part);
  ImgParams ip;
  ip.xq = xq;
  ip.xs = xs;
  ip.x = static_cast<const uint16_t*>(x);
  ip.ldx = ldx;
  ip.x_bf16 = xt == MQ_BF16;
  ip.xq_out = xq_out;
  ip.xs_out = xs_out;
  ip.M = zp.M;
  ip.Mp = zp.Mp;
  ip.act = w + pl.o_act;
  zp.timeout_ns = wait_timeout_ns();
  zp.err = device_error_word();
  if (!zp.err) return set_error(MQ_ERR_CUDA, "zipper: device error word unavailable");
  const bool quant = x != nullptr;
  mq_status st;
  if (pl.col) {
    // X rows go straight into the stages when every row starts on a 16-byte
    // boundary; otherwise the quantizer runs first and the stages take codes
    zp.raw = quant && aligned(x, 16) && ldx % 8 == 0;
    if (quant && !zp.raw) {
      uint8_t* qb = xq_out ? xq_out : w + pl.o_q;
      uint16_t* sbuf = xs_out ? xs_out : reinterpret_cast<uint16_t*>(w + pl.o_s);
      if ((st = quantize_act_launch(x, xt, M, K, ldx, qb, sbuf, stream)) != MQ_OK) return st;
      zp.xq = qb;
      zp.xs = sbuf;
      zp.xq_out = nullptr;
      zp.xs_out = nullptr;
    }
    return dots_w ? cdispatch<true>(zp, pl, stream) : cdispatch<false>(zp, pl, stream);
  }
  if (pl.tc)
    st = pl.tn == 16 ? (quant ? image_launch<16, true, false>(ip, zp.G, stream) : image_launch<16, false, false>(ip, zp.G, stream))
                     : (quant ? image_launch<32, true, false>(ip, zp.G, stream) : image_launch<32, false, false>(ip, zp.G, stream));
  else if (pl.tn == 8)
    st = quant ? image_launch<8, true, true>(ip, zp.G, stream) : image_launch<8, false, true>(ip, zp.G, stream);
  else if (pl.tn == 16)
    st = quant ? image_launch<16, true, true>(ip, zp.G, stream) : image_launch<16, false, true>(ip, zp.G, stream);
  else
    st = quant ? image_launch<32, true, true>(ip, zp.G, stream) : image_launch<32, false, true>(ip, zp.G, stream);
  if (st != MQ_OK) return st;
  if (pl.tc) return dots_w ? zdispatch<true>(zp, pl, stream) : zdispatch<false>(zp, pl, stream);
  return dots_w ? wdispatch<true>(zp, pl, stream) : wdispatch<false>(zp, pl, stream);
}

}  // namespace mq
