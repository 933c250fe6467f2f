// Blackwell (sm_103a) building blocks: mbarriers with bounded waits, TMA
// tensor copies, tensor-memory (TMEM) allocation / load / store, and the
// shared-memory and instruction descriptors of tcgen05.mma (kind::f16).
// Everything is inline PTX written for this library.
#pragma once

#include <cuda.h>

#include <atomic>

#include "common.cuh"

namespace tt {
namespace tc {

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Test whether the phase of `parity` has completed; the hardware may suspend
// the thread for a short while until it does (no busy spinning).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded waits. A wait gives up after kWaitNs nanoseconds of wall time
// (read from %globaltimer) or kWaitPolls polls, whichever comes first, or as
// soon as another role of the CTA has given up (*abort != 0); the first one
// to give up records where it stopped (g_wait_gave_up) and the caller sets
// TT_ERR_TIMEOUT.
// No wait in these kernels can spin forever.
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s
constexpr uint32_t kWaitPolls = 1u << 26;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Non-blocking test of the phase of `parity` (no suspension: cheap when the
// phase is already complete, the common case on a pipelined path).
__device__ __forceinline__ bool mbar_test_now(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Where the first wait of this module gave up: block, thread, site and
// parity packed into one word (0 = never), readable from a debugger. A store
// rather than a printf: a call on the cold path would hold registers in every
// kernel that waits.
static __device__ unsigned long long g_wait_gave_up;
__device__ __forceinline__ void record_timeout(int site, uint32_t parity) {
  const unsigned long long w = ((unsigned long long)blockIdx.x << 32) | ((unsigned long long)threadIdx.x << 16) |
                               ((unsigned long long)(site & 0xff) << 8) | (parity & 1u) | 0x80u;
  atomicCAS(&g_wait_gave_up, 0ull, w);
}

// Bounded wait for the phase of `parity` to complete. `site` identifies the
// wait in the timeout report; `limit_ns` shortens the wall-time limit (tests
// of the timeout path). Returns false on timeout or abort.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int site = 0,
                                          uint64_t limit_ns = kWaitNs) {
  if (mbar_test_now(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1; i < kWaitPolls; ++i) {
    if (mbar_test(bar, parity)) return true;
    if ((i & 255u) == 0u) {
      if (*abort) return false;
      if (global_ns() - t0 > limit_ns) break;
    }
  }
  if (atomicExch(const_cast<int*>(abort), 1) == 0) record_timeout(site, parity);
  return false;
}

// Bounded wait for the CTA's own asynchronous work (a TMA copy or the
// tcgen05 operations it committed) before the CTA leaves: unlike mbar_wait it
// ignores an abort, because shared or tensor memory must not be released
// while a copy or an MMA may still write it. Such work completes by itself,
// so the limit is only a guard: if it runs out, the CTA is marked as aborted
// (and so reports TT_ERR_TIMEOUT). Returns false then. The caller must pass
// the parity of a phase that has completed or is the current one: a barrier
// that completed another phase since names the current phase again with the
// same parity.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_test_now(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1; i < kWaitPolls; ++i) {
    if (mbar_test(bar, parity)) return true;
    if ((i & 255u) == 0u && global_ns() - t0 > kWaitNs) break;
  }
  if (atomicExch(const_cast<int*>(abort), 1) == 0) record_timeout(0xdd, parity);
  return false;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(smem_u32(dst)), "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
// Plain bulk copy (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ------------------------------------------------------------------ TMEM
// Allocation / deallocation: executed by one full warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

#define TT_R32(r)                                                                                              \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),    \
      "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),     \
      "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),    \
      "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define TT_RW32(r)                                                                                             \
  "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]),    \
      "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]),     \
      "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),    \
      "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
#define TT_IN32(r)                                                                                             \
  "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),  \
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), \
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), \
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])

// Warp-collective load of 32 consecutive 32-bit columns of this warp's 32
// TMEM lanes (thread t <- lane base+t). Asynchronous: call tmem_ld_wait()
// and tmem_pin() on the registers before using them.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : TT_R32(r)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Orders later uses of r after the preceding tmem_ld_wait().
__device__ __forceinline__ void tmem_pin(uint32_t (&r)[32]) { asm volatile("" : TT_RW32(r)); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      TT_IN32(r)
      : "memory");
}
// Warp-collective store of 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ UMMA
// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (16-byte units), fixed version field 1 at bit 46, and
// the swizzle mode in bits 61–63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// The descriptor of the operand `bytes` further on (a multiple of 16): only
// the start-address field changes, and shared-memory addresses stay below
// 2^18, so it never carries into the next field. Built once per buffer, a
// descriptor then costs one add per MMA.
__device__ __forceinline__ uint64_t desc_at(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B,
// A/B major-ness (0 = K-major, 1 = MN-major), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] · B[smem]
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] · B[smem]
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ------------------------------------------------------------------ thread-block clusters
// Whole-cluster barrier (every thread of every CTA of the cluster arrives;
// release/acquire: shared-memory writes before it are visible to peers'
// reads after it). Non-aligned forms: the threads of a warp may reach it
// one by one.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 dsmem_ld_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// Barrier over `nthreads` threads (a multiple of 32) on hardware barrier `id` (not 0: __syncthreads).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ softmax arithmetic
// max(a, b, c) in one instruction (the three-source form of max.f32, sm_100 and later).
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ------------------------------------------------------------------ host helpers
// Raise a kernel's dynamic shared-memory limit once per kernel and device
// (the attribute belongs to the current device's context, so each device
// gets its own call; the template parameter is the kernel itself, not its
// type). State per device: 0 not yet set, 1 set, -1 refused.
template <auto Kern>
inline bool smem_attr_set(int smem) {
  static std::atomic<int> state[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return false;
  int s = state[dev].load(std::memory_order_acquire);
  if (s == 0) {
    s = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess ? 1 : -1;
    state[dev].store(s, std::memory_order_release);
  }
  return s == 1;
}

// ------------------------------------------------------------------ host: tensor maps
// 2-D bf16 tensor map over a row-major [rows][cols] matrix (cols contiguous),
// box = 64 columns (128 bytes) x box_rows rows, 128-byte swizzle, zero fill
// out of bounds. Returns false if the driver rejects it.
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows);
// The same over rows `ld` elements apart (ld >= cols, ld·2 a multiple of 16 bytes).
bool make_tmap_bf16_ld(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t ld,
                       uint32_t box_rows);

}  // namespace tc
}  // namespace tt
