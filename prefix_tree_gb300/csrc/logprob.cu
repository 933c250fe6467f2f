// Weighted per-token log-probability, loss and dlogits.
//
// "Tree Training: Accelerating Agentic LLMs Training via Shared Prefix Reuse",
// Abstract: the mean of the per-branch losses can be rewritten as one sum over
// the tree's tokens, each token scaled by the share of branches that contain
// it, so each token's log-probability is computed exactly once:
//   lse_t = log Σ_v exp(z_tv),  logp_t = z_{t,y_t} − lse_t,
//   loss = −Σ_t w_t logp_t,     dlogits_tv = g·w_t·(softmax_tv − [v = y_t]).
//
// HBM-bound single pass. A row is split across a thread-block cluster of CL
// CTAs (≤ 8); each thread loads its share of the row into registers with
// 128-bit non-allocating loads one row ahead (the copy engine prefetches the
// slice into L2 kL2Ahead rows ahead), computes exp once per element
// against its own maximum and keeps the result in shared memory; the
// (max, sum) pairs are merged by warp shuffles, shared memory and then
// st.async into every CTA of the cluster; dlogits are formed from shared
// memory one row later and leave with 128-bit streaming stores, so HBM sees
// one read of the logits and one write of dlogits. The loss is a fixed-order
// fp64 reduction of the per-row terms (deterministic). Rows that do not fit
// the scheme (V > 163840, or ld / pointer not 16-byte aligned) take a generic
// two-pass kernel.
#include <cooperative_groups.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include <cuda_fp16.h>

#include "common.cuh"
#include "tc_common.cuh"

namespace cg = cooperative_groups;

namespace tt {
namespace {

constexpr int kLpThreads = 256;
// log2(e) split in two floats: hi = fp32 rounding of log2 e, lo = remainder.
constexpr float kL2eHi = 1.44269502162933349609375f;
constexpr float kL2eLo = 1.925963033500011079013347625732421875e-08f;
// 2^(x·log2 e + bias) on the hardware ex2 approximation (generic kernel only).
__device__ __forceinline__ float exp2_of_ln(float x, float bias) {
  return fast_exp2(fmaf(x, kL2eHi, fmaf(x, kL2eLo, bias)));
}

// exp(x)·2^K for a pair of values x in [-85, 0] and a constant integer K,
// accurate to ~2e-9 relative, for the few rescaling factors of a row (the
// per-element exponentials use exp_hw_scaled14 below). Cody–Waite reduction: n = rint(x·L_hi),
// f = x·L_hi − n + x·L_lo with L_hi + L_lo = log2 e (two FMAs, so f keeps the
// low part exactly), |f| <= 1/2 + 2^-20; 2^f by a degree-6 polynomial fitted
// to 2^f on [-1/2, 1/2] by least squares on Chebyshev nodes (this library's
// own fit, coefficients rounded to fp32); n + K is added to the
// exponent field. Adding 1.5·2^23 + K (an even integer) to x·L_hi in one FMA
// rounds it to the integer n + K held in the low mantissa bits, ties to even
// as rint would, so K costs no extra instruction. The result must stay a normal float
// (n + K >= -126), which x >= -85 guarantees (85·log2 e ≈ 122.6).
template <int K>
__device__ __forceinline__ float2 exp_scaled2_unclamped(float2 x) {
  constexpr float kMagic = 12582912.f + (float)K;
  // r = x·L_hi + magic with one rounding (to the integer n + K + magic)
  const float2 r = __ffma2_rn(x, make_float2(kL2eHi, kL2eHi), make_float2(kMagic, kMagic));
  const float2 nn = __ffma2_rn(r, make_float2(-1.f, -1.f), make_float2(kMagic, kMagic));  // −n, exact
  float2 f = __ffma2_rn(x, make_float2(kL2eHi, kL2eHi), nn);
  f = __ffma2_rn(x, make_float2(kL2eLo, kL2eLo), f);
  float2 p = make_float2(1.5337577497120947e-04f, 1.5337577497120947e-04f);
  p = __ffma2_rn(p, f, make_float2(1.3399859890341759e-03f, 1.3399859890341759e-03f));
  p = __ffma2_rn(p, f, make_float2(9.6185198053717613e-03f, 9.6185198053717613e-03f));
  p = __ffma2_rn(p, f, make_float2(5.5503290146589279e-02f, 5.5503290146589279e-02f));
  p = __ffma2_rn(p, f, make_float2(2.4022646248340607e-01f, 2.4022646248340607e-01f));
  p = __ffma2_rn(p, f, make_float2(6.9314718246459961e-01f, 6.9314718246459961e-01f));
  p = __ffma2_rn(p, f, make_float2(1.0f, 1.0f));
  // The low 9 bits of r's encoding are n + K in two's complement (the
  // constant's own low 9 bits are zero): shifted into the exponent field they
  // add n + K to the exponent of p (p is near 1).
  return make_float2(__int_as_float(__float_as_int(p.x) + (__float_as_int(r.x) << 23)),
                     __int_as_float(__float_as_int(p.y) + (__float_as_int(r.y) << 23)));
}
template <int K>
__device__ __forceinline__ float2 exp_scaled2(float2 x) {
  return exp_scaled2_unclamped<K>(make_float2(fmaxf(x.x, -85.f), fmaxf(x.y, -85.f)));
}

// exp(x) of every element, on the hardware ex2 approximation: the argument
// x·log2 e is formed as x·L_hi + x·L_lo (the split constant removes the
// systematic error of a rounded log2 e) with no offset inside it. Measured on
// the 12,669-row tree at V = 151936, the loss (~4.4e4) is within 2e-5 of the
// fp64 value and the mean logp error is ~4e-9: the approximation's errors do
// not accumulate into a bias there. The FMA-pipe polynomial above costs ~12
// FMA-pipe cycles per element and made the kernel compute-bound (0.54 of HBM
// bandwidth against 0.72).
__device__ __forceinline__ float2 exp_hw2(float2 x) {
  const float2 t = __ffma2_rn(x, make_float2(kL2eHi, kL2eHi), __fmul2_rn(x, make_float2(kL2eLo, kL2eLo)));
  return make_float2(fast_exp2(t.x), fast_exp2(t.y));
}

struct LpArgs {
  const __nv_bfloat16* logits;
  int64_t N, V, ld;
  const int32_t* targets;
  const float* weights;
  float g;
  float* logp;
  __nv_bfloat16* dlogits;
  int32_t* err;
};

// (m, s) represents s·exp(m); merge two such sums (generic kernel).
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;  // both empty
  s = s * exp2_of_ln(m - M, 0.f) + s2 * exp2_of_ln(m2 - M, 0.f);
  m = M;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_f16(uint32_t u) {
  return __half22float2(*reinterpret_cast<__half2*>(&u));
}

// Block-wide merge of (m, s); result valid in every thread.
__device__ __forceinline__ void block_merge(float& m, float& s) {
  __shared__ float sm[kLpThreads / 32], ss[kLpThreads / 32];
  for (int o = 16; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge(m, s, m2, s2);
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) { sm[w] = m; ss[w] = s; }
  __syncthreads();
  m = sm[0]; s = ss[0];
  for (int i = 1; i < kLpThreads / 32; ++i) lse_merge(m, s, sm[i], ss[i]);
  __syncthreads();  // sm/ss may be rewritten by the next call
}

// Distributed-shared-memory exchange of the per-CTA (max, sum) pairs: the
// sender stores into every peer's slot with st.async, which signals the
// peer's mbarrier with the bytes delivered; a receiver waits on its own
// mbarrier only (no cluster-wide barrier per row).
__device__ __forceinline__ uint32_t cluster_map(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_async_f2(uint32_t remote_addr, float2 v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
                   remote_addr),
               "f"(v.x), "f"(v.y), "r"(remote_bar)
               : "memory");
}
__device__ __forceinline__ bool xbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: 2 s of wall time, or until another thread of the CTA gave up
// (unless `drain`, used when the CTA is already giving up and only waits for
// its own copies in flight).
__device__ __forceinline__ bool xbar_wait(uint32_t bar, uint32_t parity, volatile int* abort, bool drain = false) {
  if (xbar_test(bar, parity)) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t0));
  for (uint32_t i = 1; i < (1u << 26); ++i) {
    if (xbar_test(bar, parity)) return true;
    if ((i & 255u) == 0u) {
      if (!drain && *abort) return false;
      uint64_t t;
      asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
      if (t - t0 > 2000000000ull) break;
    }
  }
  if (!drain && atomicExch(const_cast<int*>(abort), 1) == 0)
    tc::record_timeout(40, parity);
  return false;
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Geometry: a row is split over a cluster of CL <= 8 CTAs; each CTA owns a
// slice of at most kSliceVec 8-element vectors, kVecPerThread per thread.
constexpr int kVecPerThread = 10;
constexpr int kSliceVec = kVecPerThread * kLpThreads;  // 2560 vectors = 40 KB of bf16
constexpr int kXSlots = 4;                             // exchange slots (rows in the exchange)
constexpr int kL2Ahead = 2;                            // rows prefetched into L2 ahead of the current one
constexpr int kLpSmem = 2 * kSliceVec * 16;            // two rows of f16 exponentials: 81920 bytes

// One row per cluster at a time, persistent over the cluster's rows
// (row = cluster + it·nclusters), software-pipelined over two rows:
//   * row it (its logits already in registers): every thread takes its
//     maximum m_t and exp(z − m_t) of each of its elements (hardware ex2),
//     kept in shared-memory slot it & 1 as f16 (values >= 2^-14 are f16
//     normals, relative error 2^-11, below the bf16 rounding of dlogits;
//     smaller ones are f16 subnormals with absolute error <= 2^-25, so the
//     dlogit they give, g·w·e·exp(m_t − M)/S, is off by at most 3e-8·g·w)
//     and summed in fp32 (the sums carry 2^14 from the warp merge on, S14);
//     the loads of row it + 1 are issued; warps, then the
//     CTA, merge their (max, sum) pairs with one accurate rescaling each, and
//     the CTA's pair goes to every CTA of the cluster by st.async;
//   * row it − 1, whose exchange had the whole of row it's work to arrive:
//     combine the CL pairs (same order in every warp of every CTA, so all
//     agree on the row maximum M and sum S14), write logp, and turn the f16
//     values into bf16 dlogits with streaming stores.
// A thread reads and writes only its own vectors of a slot, so the slots
// need no barrier. The rescaling factors come from the accurate polynomial
// exponential, and no step needs fp64. HBM
// sees one read of the logits and one write of dlogits.
__global__ void __launch_bounds__(kLpThreads, 2) wlp_cluster_kernel(LpArgs a, int CL, int64_t nclusters) {
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(128) uint4 pbuf[];   // [2][kSliceVec] f16 exponentials
  __shared__ float2 wpart[2][kLpThreads / 32];      // per-warp pairs, double-buffered by row parity
  // cpart[x][r]: CTA r's pair of the row in exchange slot x = it % kXSlots. A
  // peer sends the pair of row it + kXSlots only after it has this CTA's pair
  // of row it + kXSlots − 1, sent after this CTA has read slot x for row it.
  __shared__ float2 cpart[kXSlots][8];
  __shared__ __align__(8) uint64_t xbar[kXSlots];
  __shared__ int abort_flag;
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = (int)a.V;
  const int nvec = (V + 7) / 8;
  const int v_lo = (int)((int64_t)rank * nvec / CL), v_hi = (int)((int64_t)(rank + 1) * nvec / CL);
  const int nv = v_hi - v_lo;  // vectors of this CTA's slice, <= kSliceVec
  const int64_t cid = blockIdx.x / CL;
  const int64_t nrows = (a.N - cid + nclusters - 1) / nclusters;
  const bool want_dl = a.dlogits != nullptr;
  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < kXSlots; ++i) tc::mbar_init(&xbar[i], 1);
    tc::fence_barrier_init();
  }
  cluster.sync();  // barriers initialised before any peer signals them

  // This thread's vectors are j = tid + c·kLpThreads (c < kVecPerThread), at
  // element offsets ebase + c·kLpThreads·8 of every row. Which of them exist
  // (bit c of vec_any) and which hold 8 elements (vec_full) does not depend
  // on the row, so the per-row loops only test a bit.
  const int ebase = (v_lo + tid) * 8;
  uint32_t vec_any = 0, vec_full = 0;
#pragma unroll
  for (int c = 0; c < kVecPerThread; ++c) {
    const int j = tid + c * kLpThreads;
    if (j < nv) vec_any |= 1u << c;
    if (j < nv && (v_lo + j) * 8 + 8 <= V) vec_full |= 1u << c;
  }
  uint4 raw[kVecPerThread];
  auto load_row = [&](int64_t row) {
    const __nv_bfloat16* z = a.logits + row * a.ld + ebase;
#pragma unroll
    for (int c = 0; c < kVecPerThread; ++c) {
      if (vec_full & (1u << c)) {
        raw[c] = ld_stream(z + c * kLpThreads * 8);
      } else {
        const int e = ebase + c * kLpThreads * 8;  // element offset in the row
        const bool any = (vec_any >> c) & 1u;
        uint32_t u[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t lo = (any && e + 2 * q < V) ? __bfloat16_as_ushort(z[c * kLpThreads * 8 + 2 * q]) : 0xff80u;
          const uint32_t hi =
              (any && e + 2 * q + 1 < V) ? __bfloat16_as_ushort(z[c * kLpThreads * 8 + 2 * q + 1]) : 0xff80u;
          u[q] = lo | (hi << 16);
        }
        raw[c] = make_uint4(u[0], u[1], u[2], u[3]);
      }
    }
  };
  // The slice's complete vectors, for the L2 prefetch kL2Ahead rows ahead.
  const int full_end = min(v_hi, V / 8);
  const uint32_t slice_bytes = full_end > v_lo ? (uint32_t)(full_end - v_lo) * 16u : 0u;
  auto prefetch_l2 = [&](int64_t row) {
    if (slice_bytes)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.logits + row * a.ld + (int64_t)v_lo * 8),
                   "r"(slice_bytes)
                   : "memory");
  };
  if (tid == 0)
    for (int64_t r = 1; r < kL2Ahead && r < nrows; ++r) prefetch_l2(cid + r * nclusters);
  load_row(cid);

  float mt_prev = -INFINITY, gw_prev = 0.f, zy_prev = 0.f;
  int y_prev = -1;
  bool ok = true;
  for (int64_t it = 0; it <= nrows; ++it) {
    float mt_cur = -INFINITY, gw_cur = 0.f, zy_cur = 0.f;
    int y_cur = -1;
    if (it < nrows) {
      const int64_t row = cid + it * nclusters;
      if (tid == 0 && it + kL2Ahead < nrows) prefetch_l2(row + kL2Ahead * nclusters);
      y_cur = a.targets[row];
      gw_cur = a.g * (a.weights ? a.weights[row] : 1.0f);
      if (rank == 0 && tid == 32 && y_cur >= 0 && y_cur < V) zy_cur = __bfloat162float(a.logits[row * a.ld + y_cur]);
      // thread maximum on packed bf16 pairs (exact)
      __nv_bfloat162 m2[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) m2[q] = __floats2bfloat162_rn(-INFINITY, -INFINITY);
#pragma unroll
      for (int c = 0; c < kVecPerThread; ++c) {
        const uint32_t u[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) m2[q] = __hmax2(m2[q], *reinterpret_cast<const __nv_bfloat162*>(&u[q]));
      }
      const __nv_bfloat162 mm = __hmax2(__hmax2(m2[0], m2[1]), __hmax2(m2[2], m2[3]));
      mt_cur = fmaxf(__low2float(mm), __high2float(mm));
      // z − m_t is exact in fp32; the hardware ex2 flushes arguments below
      // -126 to 0 (such terms are below 2^-126 of the thread's largest).
      const float mb = mt_cur == -INFINITY ? 0.f : mt_cur;
      const float2 nmb = make_float2(-mb, -mb);
      uint4* sl = pbuf + (it & 1) * kSliceVec;
      float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < kVecPerThread; ++c) {
        const int j = tid + c * kLpThreads;
        if (vec_any & (1u << c)) {
          const uint32_t u[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
          uint32_t pk[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const __nv_bfloat162 zc = *reinterpret_cast<const __nv_bfloat162*>(&u[q]);
            const float2 e = exp_hw2(__fadd2_rn(__bfloat1622float2(zc), nmb));
            s2 = __fadd2_rn(s2, e);
            pk[q] = pack_f16(e.x, e.y);
          }
          if (want_dl) sl[j] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      if (it + 1 < nrows) load_row(row + nclusters);  // in flight during the exchange and row it − 1's stores
      // warp pair: maximum M_w and Σ exp(z − M_w)·2^14 (lane 0's sum is used)
      float Mw = mt_cur;
#pragma unroll
      for (int o = 16; o; o >>= 1) Mw = fmaxf(Mw, __shfl_xor_sync(0xffffffffu, Mw, o));
      float Sw = mt_cur == -INFINITY ? 0.f : (s2.x + s2.y) * 16384.f * exp_scaled2<0>(make_float2(mb - Mw, 0.f)).x;
#pragma unroll
      for (int o = 16; o; o >>= 1) Sw += __shfl_xor_sync(0xffffffffu, Sw, o);
      if (lane == 0) wpart[it & 1][warp] = make_float2(Mw, Sw);
      // a failed exchange wait of the previous row leaves the loop here, for
      // every thread of the CTA together
      if (__syncthreads_or(!ok)) break;
      if (warp == 0) {
        // CTA pair from the warp pairs (one per lane), then lane r sends it to CTA r
        static_assert(kLpThreads / 32 <= 32, "one warp pair per lane");
        const float2 wp = lane < kLpThreads / 32 ? wpart[it & 1][lane] : make_float2(-INFINITY, 0.f);
        float Mc = wp.x;
#pragma unroll
        for (int o = 16; o; o >>= 1) Mc = fmaxf(Mc, __shfl_xor_sync(0xffffffffu, Mc, o));
        float Sc = wp.x == -INFINITY ? 0.f : wp.y * exp_scaled2<0>(make_float2(wp.x - Mc, 0.f)).x;
#pragma unroll
        for (int o = 16; o; o >>= 1) Sc += __shfl_xor_sync(0xffffffffu, Sc, o);
        Sc = __shfl_sync(0xffffffffu, Sc, 0);
        const int xs = (int)(it % kXSlots);
        if (lane == 0) tc::mbar_expect_tx(&xbar[xs], (uint32_t)(CL * 8));
        if (lane < CL)
          st_async_f2(cluster_map(smem_u32(&cpart[xs][rank]), lane), make_float2(Mc, Sc),
                      cluster_map(smem_u32(&xbar[xs]), lane));
      }
    }
    if (it >= 1) {
      // finish row it − 1
      const int64_t pit = it - 1, prow = cid + pit * nclusters;
      const int xs = (int)(pit % kXSlots);
      ok = __all_sync(0xffffffffu, xbar_wait(smem_u32(&xbar[xs]), (uint32_t)(pit / kXSlots) & 1u, &abort_flag));
      if (ok) {
        // row maximum M and Σ exp(z − M)·2^14, from lanes 0..CL-1 in a fixed tree
        const float2 pr = lane < CL ? cpart[xs][lane] : make_float2(-INFINITY, 0.f);
        float M = pr.x;
#pragma unroll
        for (int o = 4; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float t = pr.x == -INFINITY ? 0.f : pr.y * exp_scaled2<0>(make_float2(pr.x - M, 0.f)).x;
#pragma unroll
        for (int o = 4; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        const float S14 = __shfl_sync(0xffffffffu, t, 0);
        M = __shfl_sync(0xffffffffu, M, 0);
        const bool yok = y_prev >= 0 && y_prev < V;
        if (rank == 0 && tid == 32) {
          if (yok) {
            // logp = z_y − M − ln S with S = S14·2^-14 >= 1 (exact scaling). ln S
            // is logf's value L0 plus the correction S·e^-L0 − 1 (|·| ~ 1e-6, so
            // its square is negligible), taken with an FMA: accurate to ~6e-8.
            // z_y − M is exact; the sum with −L0 is an exact two-sum.
            const float S = S14 * 6.103515625e-05f;
            const float L0 = logf(S);
            const float tc = fmaf(S, exp_scaled2<0>(make_float2(-L0, 0.f)).x, -1.f);
            const float A = zy_prev - M;
            const float bh = A - L0;
            const float bv = bh - A;
            const float bl = (A - (bh - bv)) + (-L0 - bv);
            a.logp[prow] = bh + (bl - tc);
          } else {
            a.logp[prow] = __int_as_float(0x7fc00000);
            set_err(a.err, TT_ERR_INVALID_ARG);
          }
        }
        if (want_dl) {
          // softmax = exp(z − m_t) · 2^14·exp(m_t − M) / S14
          const float mb = mt_prev == -INFINITY ? 0.f : mt_prev;
          const float cfac = (mt_prev == -INFINITY || M == -INFINITY)
                                 ? 0.f
                                 : __fdividef(gw_prev * exp_scaled2<0>(make_float2(mb - M, 0.f)).x, S14);
          const float2 cf2 = make_float2(cfac * 16384.f, cfac * 16384.f);
          const uint4* sl = pbuf + (pit & 1) * kSliceVec;
          __nv_bfloat16* dz = a.dlogits + prow * a.ld + ebase;
          // the chunk of this thread that holds the target (its offset yd), or -1
          const int dv = yok ? (y_prev >> 3) - v_lo - tid : -1;
          const int cy = (dv >= 0 && dv % kLpThreads == 0) ? dv / kLpThreads : -1;
#pragma unroll
          for (int c = 0; c < kVecPerThread; ++c) {
            const int j = tid + c * kLpThreads;
            if (vec_any & (1u << c)) {
              const uint4 pv4 = sl[j];
              const uint32_t pq[4] = {pv4.x, pv4.y, pv4.z, pv4.w};
              uint32_t o[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float2 d = __fmul2_rn(unpack_f16(pq[q]), cf2);
                o[q] = pack_bf16(d.x, d.y);
              }
              if (c == cy) {
                const int yd = y_prev & 7;
                // the target's term −g·w, added to the element at offset yd
                float d[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const float2 f = __fmul2_rn(unpack_f16(pq[q]), cf2);
                  d[2 * q] = f.x;
                  d[2 * q + 1] = f.y;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) d[q] -= q == yd ? gw_prev : 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) o[q] = pack_bf16(d[2 * q], d[2 * q + 1]);
              }
              __nv_bfloat16* dzc = dz + c * kLpThreads * 8;
              if (vec_full & (1u << c)) {
                st_stream(dzc, make_uint4(o[0], o[1], o[2], o[3]));
              } else {
                const int e = ebase + c * kLpThreads * 8;  // element offset in the row
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  if (e + 2 * q < V) dzc[2 * q] = __ushort_as_bfloat16((unsigned short)(o[q] & 0xffffu));
                  if (e + 2 * q + 1 < V) dzc[2 * q + 1] = __ushort_as_bfloat16((unsigned short)(o[q] >> 16));
                }
              }
            }
          }
        }
      } else {
        set_err(a.err, TT_ERR_TIMEOUT);
      }
    }
    mt_prev = mt_cur;
    gw_prev = gw_cur;
    y_prev = y_cur;
    zy_prev = zy_cur;
  }
  cluster.sync();  // no CTA leaves while a peer may still deliver into its shared memory
}

// Generic row kernel: pass 1 online (max, sum) over the row, pass 2 writes
// dlogits re-reading the row (from L2 for rows that fit).
__global__ void __launch_bounds__(kLpThreads) wlp_generic_kernel(LpArgs a) {
  const int64_t row = blockIdx.x;
  const __nv_bfloat16* z = a.logits + row * a.ld;
  float m = -INFINITY, s = 0.f;
  for (int64_t v = threadIdx.x; v < a.V; v += kLpThreads) {
    const float x = __bfloat162float(z[v]);
    if (x > m) { s = s * exp2_of_ln(m - x, 0.f) + 1.f; m = x; }
    else s += exp2_of_ln(x - m, 0.f);
  }
  block_merge(m, s);
  const double lse = (double)m + log((double)s);
  const int y = a.targets[row];
  const bool yok = y >= 0 && y < a.V;
  const float w = a.weights ? a.weights[row] : 1.0f;
  if (threadIdx.x == 0) {
    if (yok) a.logp[row] = (float)((double)__bfloat162float(z[y]) - lse);
    else { a.logp[row] = __int_as_float(0x7fc00000); set_err(a.err, TT_ERR_INVALID_ARG); }
  }
  if (!a.dlogits) return;
  const float gw = a.g * w;
  const float lsef = (float)lse;
  __nv_bfloat16* dz = a.dlogits + row * a.ld;
  for (int64_t v = threadIdx.x; v < a.V; v += kLpThreads) {
    float d = gw * exp2_of_ln(__bfloat162float(z[v]) - lsef, 0.f);
    if (yok && v == y) d -= gw;
    dz[v] = __float2bfloat16_rn(d);
  }
}

// Rows of a long vocabulary on the SMs the clusters leave idle (the clusters
// of CL CTAs, two per SM, do not tile every GPC): two CTAs of 512 threads per
// SM, each on its own row, persistent over rows row0 + blockIdx.x +
// k·gridDim.x. Pass 1 streams the row in 16-byte vectors (eight loads in
// flight per thread) keeping each
// thread's (max, sum) with the accurate polynomial rescale; the block merges
// the pairs in a fixed tree; pass 2 reads the row again (from L2: it was read
// microseconds before) and writes dlogits = g·w·exp(z − lse), minus g·w at
// the target, rounded once to bf16. Its CTAs hold more registers than an SM
// running two cluster CTAs has free, so they only run on the idle SMs.
constexpr int kRowThreads = 512;
constexpr int kRowCtasPerSm = 2;
constexpr int kRowUnroll = 8;
#ifndef TT_ROW_SHARE
#define TT_ROW_SHARE 60
#endif
// Rows an idle SM takes per row of a cluster SM, in percent (a row kernel SM
// streams at about this fraction of a cluster SM's rate).
constexpr int kRowSharePct = TT_ROW_SHARE;
__device__ __forceinline__ void lse_merge_acc(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  const float2 f = exp_scaled2<0>(make_float2(m - M, m2 - M));
  s = s * f.x + s2 * f.y;
  m = M;
}
__global__ void __launch_bounds__(kRowThreads, kRowCtasPerSm) wlp_row_kernel(LpArgs a, int64_t row0, int64_t nrows) {
  __shared__ float2 wpair[kRowThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = (int)a.V;
  const int nfull = V / 8;  // complete 8-element vectors; the rest (V % 8 elements) is read element-wise
  for (int64_t row = row0 + blockIdx.x; row < row0 + nrows; row += gridDim.x) {
    const __nv_bfloat16* z = a.logits + row * a.ld;
    const uint4* zv = reinterpret_cast<const uint4*>(z);
    float m = -INFINITY, s = 0.f;
    auto add_vec = [&](const uint4 r) {
      const uint32_t u[4] = {r.x, r.y, r.z, r.w};
      float2 x[4];
      float mv = -INFINITY;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        x[q] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[q]));
        mv = tc::fmax3f(mv, x[q].x, x[q].y);
      }
      if (mv > m) {
        s = m == -INFINITY ? 0.f : s * exp_scaled2<0>(make_float2(m - mv, 0.f)).x;
        m = mv;
      }
      const float mb = m == -INFINITY ? 0.f : m;  // all -inf so far: exp(-inf − 0) = 0, not NaN
      const float2 nm = make_float2(-mb, -mb);
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 4; ++q) acc = __fadd2_rn(acc, exp_hw2(__fadd2_rn(x[q], nm)));
      s += acc.x + acc.y;
    };
    int j = tid;
    for (; j + (kRowUnroll - 1) * kRowThreads < nfull; j += kRowUnroll * kRowThreads) {
      uint4 r[kRowUnroll];
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) r[u] = ld_stream(zv + j + u * kRowThreads);
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) add_vec(r[u]);
    }
    for (; j < nfull; j += kRowThreads) add_vec(ld_stream(zv + j));
    if (tid < V - nfull * 8) {  // the last V % 8 elements, one per thread
      const float x = __bfloat162float(z[nfull * 8 + tid]);
      if (x > m) {
        s = m == -INFINITY ? 0.f : s * exp_scaled2<0>(make_float2(m - x, 0.f)).x;
        m = x;
      }
      s += exp_hw2(make_float2(x - (m == -INFINITY ? 0.f : m), -INFINITY)).x;
    }
    // fixed-tree block merge of (m, s): warps by shuffles, then warp 0 over the warps
#pragma unroll
    for (int o = 16; o; o >>= 1) lse_merge_acc(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
    if (lane == 0) wpair[warp] = make_float2(m, s);
    __syncthreads();
    {
      const float2 p = lane < kRowThreads / 32 ? wpair[lane] : make_float2(-INFINITY, 0.f);  // (-inf, 0): no term
      m = p.x;
      s = p.y;
#pragma unroll
      for (int o = 16; o; o >>= 1) lse_merge_acc(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
    }
    __syncthreads();  // wpair is rewritten by the next row
    // m, s: the row maximum M and Σ exp(z − M) >= 1, the same in every thread
    const int y = a.targets[row];
    const bool yok = y >= 0 && y < V;
    const float gw = a.g * (a.weights ? a.weights[row] : 1.0f);
    if (tid == 0) {
      if (yok) {
        // logp = z_y − M − ln S, ln S = logf's L0 plus the correction S·e^-L0 − 1, summed with an exact two-sum
        const float L0 = logf(s);
        const float tc = fmaf(s, exp_scaled2<0>(make_float2(-L0, 0.f)).x, -1.f);
        const float A = __bfloat162float(z[y]) - m;
        const float bh = A - L0;
        const float bv = bh - A;
        const float bl = (A - (bh - bv)) + (-L0 - bv);
        a.logp[row] = bh + (bl - tc);
      } else {
        a.logp[row] = __int_as_float(0x7fc00000);
        set_err(a.err, TT_ERR_INVALID_ARG);
      }
    }
    if (!a.dlogits) continue;
    const float cf = __fdividef(gw, s);
    const float mb = m == -INFINITY ? 0.f : m;
    const float2 cf2 = make_float2(cf, cf), nm = make_float2(-mb, -mb);
    __nv_bfloat16* dz = a.dlogits + row * a.ld;
    uint4* dzv = reinterpret_cast<uint4*>(dz);
    for (int jj = tid; jj < nfull; jj += kRowThreads) {
      const uint4 r = ld_stream(zv + jj);
      const uint32_t u[4] = {r.x, r.y, r.z, r.w};
      float d[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[q]));
        const float2 e = __fmul2_rn(exp_hw2(__fadd2_rn(x, nm)), cf2);
        d[2 * q] = e.x;
        d[2 * q + 1] = e.y;
      }
      const int yq = yok && (y >> 3) == jj ? (y & 7) : -1;  // the target's element in this vector, or -1
#pragma unroll
      for (int q = 0; q < 8; ++q) d[q] -= q == yq ? gw : 0.f;
      st_stream(dzv + jj, make_uint4(pack_bf16(d[0], d[1]), pack_bf16(d[2], d[3]), pack_bf16(d[4], d[5]),
                                     pack_bf16(d[6], d[7])));
    }
    if (tid < V - nfull * 8) {
      const int v = nfull * 8 + tid;
      float d = cf * exp_hw2(make_float2(__bfloat162float(z[v]) - mb, -INFINITY)).x;
      if (yok && y == v) d -= gw;
      dz[v] = __float2bfloat16_rn(d);
    }
  }
}

// loss = −Σ_t w_t logp_t in a fixed order (thread i takes rows i, i + 1024,
// ..., then a fixed tree over the threads), deterministic. The GPU's fp64
// pipe is narrow, so the sum is carried as an unevaluated pair of floats
// (hi + lo, ~48 significant bits): each product w·logp is split exactly with
// an FMA (hi = fl(w·l), lo = fma(w, l, −hi)), and pairs are added with
// Knuth's two-sum plus a renormalisation (the classic double-float addition).
// Only the final hi + lo is formed in fp64.
struct F2 {
  float hi, lo;
};
__device__ __forceinline__ F2 two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  return {s, (a - (s - bb)) + (b - bb)};
}
__device__ __forceinline__ F2 f2_add(F2 x, F2 y) {
  F2 s = two_sum(x.hi, y.hi);
  const F2 t = two_sum(x.lo, y.lo);
  s.lo += t.hi;
  s = two_sum(s.hi, s.lo);
  s.lo += t.lo;
  return two_sum(s.hi, s.lo);
}
// Launched as a programmatic dependent of the log-prob kernel: the launch is
// processed while that kernel runs, and griddepcontrol.wait holds the CTA
// until it has finished and its writes are visible. The rows of a thread are
// loaded eight at a time before they are summed (in the same order).
__global__ void __launch_bounds__(1024) loss_kernel(const float* logp, const float* weights, int64_t N, double* loss) {
  __shared__ float2 red[1024];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  F2 acc = {0.f, 0.f};
  constexpr int kU = 8;
  for (int64_t t0 = threadIdx.x; t0 < N; t0 += 1024 * kU) {
    float w[kU], l[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t t = t0 + (int64_t)u * 1024;
      w[u] = t < N ? (weights ? weights[t] : 1.0f) : 0.f;
      l[u] = t < N ? logp[t] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (t0 + (int64_t)u * 1024 >= N) break;
      const float p = -w[u] * l[u];
      acc = f2_add(acc, F2{p, fmaf(-w[u], l[u], -p)});
    }
  }
  red[threadIdx.x] = make_float2(acc.hi, acc.lo);
  __syncthreads();
  for (int o = 512; o; o >>= 1) {
    if (threadIdx.x < o) {
      const float2 a = red[threadIdx.x], b = red[threadIdx.x + o];
      const F2 s = f2_add(F2{a.x, a.y}, F2{b.x, b.y});
      red[threadIdx.x] = make_float2(s.hi, s.lo);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = (double)red[0].x + (double)red[0].y;
}

// Clusters of CL CTAs that can be resident at once (queried once per device and cluster size).
int cluster_capacity(int CL) {
  static std::atomic<int> max_clusters[kMaxDevices][9];
  const int dev = current_device();
  if (dev < 0 || CL < 1 || CL > 8) return 0;
  int mc = max_clusters[dev][CL].load(std::memory_order_relaxed);
  if (mc == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kLpThreads);
    cfg.dynamicSmemBytes = kLpSmem;
    cfg.gridDim = dim3((unsigned)(CL * 1024));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!tc::smem_attr_set<wlp_cluster_kernel>(kLpSmem) ||
        cudaOccupancyMaxActiveClusters(&mc, wlp_cluster_kernel, &cfg) != cudaSuccess || mc < 1)
      mc = 8;
    max_clusters[dev][CL].store(mc, std::memory_order_relaxed);
  }
  return mc;
}

cudaError_t launch_cluster(const LpArgs& a, int CL, cudaStream_t st) {
  if (!tc::smem_attr_set<wlp_cluster_kernel>(kLpSmem)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kLpThreads);
  cfg.dynamicSmemBytes = kLpSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // as many clusters as can be resident at once
  const int mc = cluster_capacity(CL);
  if (mc < 1) return cudaErrorInvalidDevice;
  const int64_t nclusters = std::min<int64_t>(a.N, mc);
  cfg.gridDim = dim3((unsigned)(nclusters * CL));
  KtScope kt(TT_KT_LOGPROB, st);
  return cudaLaunchKernelEx(&cfg, wlp_cluster_kernel, a, CL, nclusters);
}

// SMs the resident clusters leave idle (two cluster CTAs per SM), and the
// rows given to them: kRowSharePct rows per idle SM for every 100 rows per
// cluster SM; none for batches under four rows per SM.
struct RowSplit {
  int idle;
  int64_t rows;
};
RowSplit row_split(int64_t N, int CL) {
  const int nsm = sm_count(), mc = cluster_capacity(CL);
  RowSplit r{0, 0};
  if (nsm < 1 || mc < 1) return r;
  r.idle = nsm - (mc * CL + 1) / 2;
  if (r.idle < 1 || N < 4 * (int64_t)nsm) {
    r.idle = 0;
    return r;
  }
  const int64_t busy = nsm - r.idle;
  r.rows = N * r.idle * kRowSharePct / (busy * 100 + (int64_t)r.idle * kRowSharePct);
  return r;
}

// The side stream of a device for the idle-SM rows (created once).
cudaStream_t side_stream() {
  static std::atomic<cudaStream_t> streams[kMaxDevices];
  static std::mutex mu;
  const int dev = current_device();
  if (dev < 0) return nullptr;
  cudaStream_t q = streams[dev].load(std::memory_order_acquire);
  if (q) return q;
  std::lock_guard<std::mutex> lock(mu);
  q = streams[dev].load(std::memory_order_acquire);
  if (!q && cudaStreamCreateWithFlags(&q, cudaStreamNonBlocking) == cudaSuccess)
    streams[dev].store(q, std::memory_order_release);
  return streams[dev].load(std::memory_order_acquire);
}

// The cluster kernel on st for rows [0, N − R) and the row kernel on the idle
// SMs for the last R rows (a stream forked from st and joined back, so the
// loss kernel after it sees every row). Not while st is being captured (the
// side stream is shared by the device's calls): then the clusters take all rows.
cudaError_t launch_rows(const LpArgs& a, int CL, cudaStream_t st) {
  RowSplit sp = row_split(a.N, CL);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (sp.rows > 0 && (cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)) {
    (void)cudaGetLastError();
    sp.rows = 0;
  }
  cudaStream_t side = sp.rows > 0 ? side_stream() : nullptr;
  if (!side) return launch_cluster(a, CL, st);
  cudaEvent_t fork, join;
  if (cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess) return cudaErrorUnknown;
  if (cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) {
    cudaEventDestroy(fork);
    return cudaErrorUnknown;
  }
  cudaError_t e = cudaEventRecord(fork, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side, fork, 0);
  LpArgs head = a;
  head.N = a.N - sp.rows;
  if (e == cudaSuccess) e = launch_cluster(head, CL, st);  // the clusters first: they are placed before the rows
  if (e == cudaSuccess) {
    KtScope kt(TT_KT_LOGPROB, side);
    wlp_row_kernel<<<(unsigned)std::min<int64_t>((int64_t)sp.idle * kRowCtasPerSm, sp.rows), kRowThreads, 0, side>>>(
        a, a.N - sp.rows, sp.rows);
    e = cudaGetLastError();
  }
  // join even after an error, so that st never runs ahead of work on the side stream
  const cudaError_t e2 = cudaEventRecord(join, side);
  const cudaError_t e3 = cudaStreamWaitEvent(st, join, 0);
  cudaEventDestroy(fork);
  cudaEventDestroy(join);
  if (e == cudaSuccess) e = e2 != cudaSuccess ? e2 : e3;
  return e;
}

}  // namespace

// loss = −Σ_t w_t·logp_t in a fixed order (one CTA, double-float sums), as a
// programmatic dependent launch: it may be scheduled while the kernel that
// writes logp is still running and waits for it at its first instruction.
cudaError_t launch_weighted_loss(const float* logp, const float* weights, int64_t N, double* loss, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1024);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, loss_kernel, logp, weights, N, loss);
}

}  // namespace tt

using namespace tt;

TT_API int tt_weighted_logprob(const tt_bf16* logits, int64_t N, int64_t V, int64_t ld, const int32_t* targets,
                               const float* weights, float g, float* logp, double* loss, tt_bf16* dlogits,
                               int32_t* err, tt_stream_t stream) {
  if (!logits || !targets || !logp || !loss || !err || N < 0 || V < 1 || ld < V) return TT_ERR_INVALID_ARG;
  if (N > (int64_t)INT32_MAX / 8) return TT_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (N == 0) return cuda_status(launch_weighted_loss(logp, weights, 0, loss, st));
  LpArgs a;
  a.logits = reinterpret_cast<const __nv_bfloat16*>(logits);
  a.N = N; a.V = V; a.ld = ld; a.targets = targets; a.weights = weights; a.g = g; a.logp = logp;
  a.dlogits = reinterpret_cast<__nv_bfloat16*>(dlogits); a.err = err;
  const bool vec_ok = aligned16(logits) && (ld % 8 == 0) && (!dlogits || aligned16(dlogits));
  cudaError_t e = cudaSuccess;
  bool done = false;
  if (vec_ok) {
    const int64_t CL = ((V + 7) / 8 + kSliceVec - 1) / kSliceVec;  // slices of at most kSliceVec vectors
    if (CL <= 8) {
      e = launch_rows(a, (int)CL, st);
      done = true;
    }
  }
  if (!done) {
    KtScope kt(TT_KT_LOGPROB, st);
    wlp_generic_kernel<<<(unsigned)N, kLpThreads, 0, st>>>(a);
  }
  if (e != cudaSuccess) return TT_ERR_CUDA;
  TT_LAUNCH_CHECK();
  return cuda_status(launch_weighted_loss(logp, weights, N, loss, st));
}
