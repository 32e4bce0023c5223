// Internal helpers of the sm_103a library: PTX wrappers (mbarrier, bulk/TMA
// copies, tcgen05), bounded waits, the device error word, and host-side
// declarations shared by the translation units.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mq.h"

namespace mq {

constexpr int kGroup = 128;   // inputs per scale group
constexpr int kBlockRows = 64;  // output rows per residual block
constexpr int kTileN = 128;   // weight rows per GEMM tile (tensor-core M)
// packed records (mq_pack_weights): codes, then fp16 scales
constexpr int kWRecBytes = MQ_WREC_BYTES, kWRecScales = 8192;
constexpr int kRRecBytes = MQ_RREC_BYTES, kRRecScales = 4096;
static_assert(kWRecBytes == kWRecScales + 2 * kTileN && kRRecBytes == kRRecScales + 2 * kBlockRows, "records");

// device error word bits
constexpr uint32_t kDevErrTimeout = 1u;

// Every GEMM workspace starts with this many bytes that the kernels read as
// counters and flags: zero before the first use, and left zero by every
// launch that finishes normally.  Scratch (pieces, activation images) follows,
// so one workspace can serve GEMMs of any shape run one after another.
constexpr int kWsZeroBytes = 16384;

// ---------------------------------------------------------------------------
// host side (abi.cu)
// ---------------------------------------------------------------------------
mq_status set_error(mq_status s, const char* fmt, ...);
mq_status check_device();  // current device must be cc 10.3
mq_status launch_status(const char* what);  // cudaGetLastError -> status
uint64_t wait_timeout_ns();
uint32_t* device_error_word();  // address of the error word on the current device
int sm_count();
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------------------
// device side
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that may suspend the thread for up to `hint_ns` until the phase
// completes: a waiting warp sleeps instead of flooding the shared-memory pipe
// with polls that the warps still working have to queue behind.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Non-blocking test of an mbarrier phase (for a role that polls several).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Raise the expected transaction bytes of the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its writes are visible (no-op without PDL), and
// allow the next kernel in the stream to start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Bounded wait on an mbarrier phase.  Gives up after `timeout_ns` or when the
// CTA-wide abort flag is raised; on timeout it records the error in the
// device error word and raises the abort flag.  Returns false on give-up.
// The global timer and the abort flag are read once every 64 polls only: a
// waiting warp must notice a completed phase at once (the handoffs between
// roles sit on the critical path), and those reads are slow.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns, uint32_t* err_word) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait_sleep(bar, parity, 1000u)) return true;
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

// Acquire-release fence at GPU scope: with a barrier before it, it releases
// the CTA's earlier global writes to another CTA that acquires them (and
// acquires what a preceding atomic observed).  Lighter than __threadfence(),
// which is sequentially consistent.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// --- tcgen05 -----------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc], E4M3 x E4M3 -> f32, one K=32 step.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on `bar` when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Store 8 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}

// Load 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

// Load 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Eight INT4 codes (4-bit two's complement, element i in bits 4i..4i+3) to
// eight E4M3 bytes holding the same integers exactly: elements 0..3 in `lo`,
// 4..7 in `hi`, element order = byte order.  Two 8-entry byte tables (codes
// 0..7 and -8..-1) are looked up with prmt; prmt's sign-replicate mode (bit 3
// of a selector nibble) zeroes / saturates the entries of the other sign, and
// a third prmt builds the per-byte sign mask from the nibbles' top bits.
__device__ __forceinline__ void int4x8_to_e4m3(uint32_t p, uint32_t& lo, uint32_t& hi) {
  constexpr uint32_t kPosA = 0x44403800u, kPosB = 0x4E4C4A48u;  // 0, 1, 2, 3 | 4, 5, 6, 7
  constexpr uint32_t kNegA = 0xCACCCED0u, kNegB = 0xB8C0C4C8u;  // -8,-7,-6,-5 | -4,-3,-2,-1
  const uint32_t pn = p ^ 0x88888888u;
  const uint32_t p4 = p << 4;
  const uint32_t pos_lo = prmt(kPosA, kPosB, p);
  const uint32_t neg_lo = prmt(kNegA, kNegB, pn);
  const uint32_t msk_lo = prmt(p, p4, 0x9D8Cu);
  const uint32_t pos_hi = prmt(kPosA, kPosB, p >> 16);
  const uint32_t neg_hi = prmt(kNegA, kNegB, pn >> 16);
  const uint32_t msk_hi = prmt(p, p4, 0xBFAEu);
  lo = (neg_lo & msk_lo) | pos_lo;
  hi = (neg_hi & msk_hi) | pos_hi;
}

}  // namespace mq
