// Weighted per-token log-probability, loss and dlogits.
//
// "Tree Training: Accelerating Agentic LLMs Training via Shared Prefix Reuse",
// Abstract: averaging the loss over every branch equals a per-token weighted
// loss whose weight is the fraction of branches through the token, so each
// token's log-probability is computed exactly once:
//   lse_t = log Σ_v exp(z_tv),  logp_t = z_{t,y_t} − lse_t,
//   loss = −Σ_t w_t logp_t,     dlogits_tv = g·w_t·(softmax_tv − [v = y_t]).
//
// HBM-bound single pass. A row is split across a thread-block cluster of CL
// CTAs (≤ 8); each thread keeps its slice of the row in registers, loaded
// with 128-bit non-allocating loads, computes exp once per element against
// its own running maximum, and the (max, sum) pairs are merged by warp
// shuffles, shared memory and then distributed shared memory across the
// cluster. dlogits are written from the registers with 128-bit streaming
// stores, so HBM sees one read of the logits and one write of dlogits.
// The loss is a fixed-order fp64 reduction of the per-row terms
// (deterministic). Rows that do not fit the register scheme (V > 163840,
// or ld / pointer not 16-byte aligned) take a generic two-pass kernel.
#include <cooperative_groups.h>

#include <algorithm>

#include <cuda_fp16.h>

#include "common.cuh"

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

// exp(x)·2^k for a pair of values (x <= 0, integer k), accurate to ~2e-9
// relative and without bias, so that a row sum of 10^5 terms stays within
// ~1e-9 of the exact sum (both the hardware ex2 approximation and an
// argument x·log2 e rounded to fp32 near a large offset carry small
// systematic biases that, summed over a tree's rows, move the loss by more
// than 1e-4). Cody–Waite reduction: n = rint(x·L_hi), f = x·L_hi − n + x·L_lo
// with L_hi + L_lo = log2 e (two FMAs, so f keeps the low part exactly),
// |f| <= 1/2 + 2^-20; 2^f by a degree-6 polynomial fitted to 2^f on
// [-1/2, 1/2] by least squares on Chebyshev nodes (the fit is recorded in
// fit_exp2_poly.py next to this file); n + k added to the exponent field.
// Inputs are clamped to x >= -85 (e^-85 ~ 1e-37: such terms do not matter);
// the result must stay a normal float (n + k >= -126).
__device__ __forceinline__ float2 exp_scaled2(float2 x, int k) {
  constexpr float kMagic = 12582912.f;  // 1.5·2^23: adding it rounds to an integer in the low mantissa bits
  x = make_float2(fmaxf(x.x, -85.f), fmaxf(x.y, -85.f));  // 85·log2 e ≈ 122.6
  const float2 t0 = __fmul2_rn(x, make_float2(kL2eHi, kL2eHi));
  const float2 r = __fadd2_rn(t0, make_float2(kMagic, kMagic));
  const float2 n = __fadd2_rn(r, make_float2(-kMagic, -kMagic));
  float2 f = __ffma2_rn(x, make_float2(kL2eHi, kL2eHi), make_float2(-n.x, -n.y));
  f = __ffma2_rn(x, make_float2(kL2eLo, kL2eLo), f);
  float2 p = make_float2(1.5337577497120947e-04f, 1.5337577497120947e-04f);
  p = __ffma2_rn(p, f, make_float2(1.3399859890341759e-03f, 1.3399859890341759e-03f));
  p = __ffma2_rn(p, f, make_float2(9.6185198053717613e-03f, 9.6185198053717613e-03f));
  p = __ffma2_rn(p, f, make_float2(5.5503290146589279e-02f, 5.5503290146589279e-02f));
  p = __ffma2_rn(p, f, make_float2(2.4022646248340607e-01f, 2.4022646248340607e-01f));
  p = __ffma2_rn(p, f, make_float2(6.9314718246459961e-01f, 6.9314718246459961e-01f));
  p = __ffma2_rn(p, f, make_float2(1.0f, 1.0f));
  // the low mantissa bits of r hold n in two's complement: shifted into the
  // exponent field they add n (and k) to the exponent of p (p is near 1)
  return make_float2(__int_as_float(__float_as_int(p.x) + ((__float_as_int(r.x) + k) << 23)),
                     __int_as_float(__float_as_int(p.y) + ((__float_as_int(r.y) + k) << 23)));
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

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_f16(uint32_t u) {
  return __half22float2(*reinterpret_cast<__half2*>(&u));
}
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

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

// Warp-then-block reductions with a fixed combination order (deterministic).
__device__ __forceinline__ float block_max(float v, float* scratch) {
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  v = scratch[0];
  for (int i = 1; i < kLpThreads / 32; ++i) v = fmaxf(v, scratch[i]);
  __syncthreads();
  return v;
}
__device__ __forceinline__ float block_sum(float v, float* scratch) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  v = scratch[0];
  for (int i = 1; i < kLpThreads / 32; ++i) v += scratch[i];
  __syncthreads();
  return v;
}

// One row per cluster of CL CTAs at a time; persistent over rows. Per row:
// every thread takes exp(z − m_t)·2^14 of its elements against its own exact
// maximum m_t (kept as f16 for dlogits, summed in fp32); the CTA reduces its
// exact maximum M_c and the thread sums rescaled once by exp(m_t − M_c); the
// CTAs then exchange (M_c, S_c) through distributed shared memory with ONE
// cluster barrier and combine them in rank order. All rescaling factors come
// from the accurate exponential, so the row sum carries no systematic error.
// The next row's loads are issued right after the exponentials and land
// while this row is reduced and written.
template <int CH>
__global__ void __launch_bounds__(kLpThreads, 2) wlp_cluster_kernel(LpArgs a, int CL, int64_t nclusters) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ float scratch[kLpThreads / 32];
  // This CTA's (max, sum) of a row, read by the whole cluster after the row's
  // barrier. Slot it & 1 is rewritten two rows later, after the next row's
  // barrier, which every CTA reaches only once it has read this row's slots.
  __shared__ float2 part[2];
  const int rank = (int)cluster.block_rank();
  const int64_t nvec = (a.V + 7) / 8;
  const int64_t v_lo = rank * nvec / CL, v_hi = (rank + 1) * nvec / CL;
  const int tid = threadIdx.x;
  uint4 raw[CH];
  auto load_row = [&](int64_t row) {
    const __nv_bfloat16* z = a.logits + row * a.ld;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int64_t vi = v_lo + (int64_t)c * kLpThreads + tid;
      const int64_t e = vi * 8;
      if (vi < v_hi && e + 8 <= a.V) {
        raw[c] = ld_stream(z + e);
      } else {
        uint32_t u[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t lo = (vi < v_hi && e + 2 * j < a.V) ? __bfloat16_as_ushort(z[e + 2 * j]) : 0xff80u;
          const uint32_t hi = (vi < v_hi && e + 2 * j + 1 < a.V) ? __bfloat16_as_ushort(z[e + 2 * j + 1]) : 0xff80u;
          u[j] = lo | (hi << 16);
        }
        raw[c] = make_uint4(u[0], u[1], u[2], u[3]);
      }
    }
  };
  const int64_t row0 = blockIdx.x / CL;
  if (row0 < a.N) load_row(row0);
  int it = 0;
  for (int64_t row = row0; row < a.N; row += nclusters, ++it) {
    const int y = a.targets[row];
    const bool yok = y >= 0 && y < a.V;
    const float w = a.weights ? a.weights[row] : 1.0f;
    float zy = 0.f;
    if (rank == 0 && tid == 0 && yok) zy = __bfloat162float(a.logits[row * a.ld + y]);

    float mt = -INFINITY;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const uint32_t u[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) mt = fmaxf(mt, fmaxf(bf_lo(u[j]), bf_hi(u[j])));
    }
    // exp(z − m_t)·2^14 kept as f16 pairs (every value >= 2^-28 stays an f16
    // normal, relative error 2^-11 — below the bf16 rounding of dlogits); the
    // sum is taken in fp32 before packing. z − m_t is exact in fp32.
    const float mb = mt == -INFINITY ? 0.f : mt;
    uint32_t p[CH][4];
    float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const uint32_t u[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 e = exp_scaled2(make_float2(bf_lo(u[j]) - mb, bf_hi(u[j]) - mb), 14);
        s2 = __fadd2_rn(s2, e);
        p[c][j] = pack_f16(e.x, e.y);
      }
    }
    if (row + nclusters < a.N) load_row(row + nclusters);  // prefetch: in flight during reduction and stores
    const float Mc = block_max(mt, scratch);
    // this thread's sum relative to the CTA maximum (one accurate rescaling)
    const float st = mt == -INFINITY ? 0.f : (s2.x + s2.y) * exp_scaled2(make_float2(mb - Mc, 0.f), 0).x;
    const float Sc = block_sum(st, scratch);
    if (tid == 0) part[it & 1] = make_float2(Mc, Sc);
    cluster.sync();
    float2 pr[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) pr[r] = r < CL ? *cluster.map_shared_rank(&part[it & 1], r) : make_float2(-INFINITY, 0.f);
    float M = pr[0].x;
#pragma unroll
    for (int r = 1; r < 8; ++r) M = fmaxf(M, pr[r].x);
    float S14 = 0.f;  // Σ exp(z − M)·2^14, combined in rank order
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (pr[r].x != -INFINITY) S14 += pr[r].y * exp_scaled2(make_float2(pr[r].x - M, 0.f), 0).x;
    const double lse = (double)M + log((double)S14 * 6.103515625e-05);
    if (rank == 0 && tid == 0) {
      if (yok) a.logp[row] = (float)((double)zy - lse);
      else { a.logp[row] = __int_as_float(0x7fc00000); set_err(a.err, TT_ERR_INVALID_ARG); }
    }
    if (a.dlogits) {
      const float gw = a.g * w;
      // softmax = exp(z − m_t)·2^14 · 2^-14 · exp(m_t − lse)
      // (the exponent add of exp_scaled2 needs a normal result: scale by 2^-14 with a multiply)
      const float cfac =
          mt == -INFINITY ? 0.f : gw * exp_scaled2(make_float2((float)((double)mb - lse), 0.f), 0).x * 6.103515625e-05f;
      __nv_bfloat16* dz = a.dlogits + row * a.ld;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int64_t vi = v_lo + (int64_t)c * kLpThreads + tid;
        const int64_t e = vi * 8;
        if (vi >= v_hi) continue;
        float d[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = unpack_f16(p[c][j]);
          d[2 * j] = f.x * cfac;
          d[2 * j + 1] = f.y * cfac;
        }
        if (yok && y >= e && y < e + 8) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (e + j == y) d[j] -= gw;
        }
        if (e + 8 <= a.V) {
          st_stream(dz + e, make_uint4(pack_bf16(d[0], d[1]), pack_bf16(d[2], d[3]), pack_bf16(d[4], d[5]),
                                       pack_bf16(d[6], d[7])));
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (e + j < a.V) dz[e + j] = __float2bfloat16_rn(d[j]);
        }
      }
    }
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
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

// loss = −Σ_t w_t logp_t, fp64, fixed order (thread i takes rows i, i+1024, ...).
__global__ void __launch_bounds__(1024) loss_kernel(const float* logp, const float* weights, int64_t N, double* loss) {
  __shared__ double red[1024];
  double acc = 0.0;
  for (int64_t t = threadIdx.x; t < N; t += 1024) acc += -(double)(weights ? weights[t] : 1.0f) * (double)logp[t];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int o = 512; o; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = red[0];
}

template <int CH>
cudaError_t launch_cluster(const LpArgs& a, int CL, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kLpThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // as many clusters as can be resident at once (queried once per cluster size)
  static int max_clusters[9] = {0};
  if (max_clusters[CL] == 0) {
    cfg.gridDim = dim3((unsigned)(CL * 1024));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, wlp_cluster_kernel<CH>, &cfg) != cudaSuccess || n < 1) n = 16;
    max_clusters[CL] = n;
  }
  const int64_t nclusters = std::min<int64_t>(a.N, max_clusters[CL]);
  cfg.gridDim = dim3((unsigned)(nclusters * CL));
  return cudaLaunchKernelEx(&cfg, wlp_cluster_kernel<CH>, a, CL, nclusters);
}

}  // namespace
}  // namespace tt

using namespace tt;

TT_API int tt_weighted_logprob(const tt_bf16* logits, int64_t N, int64_t V, int64_t ld, const int32_t* targets,
                               const float* weights, float g, float* logp, double* loss, tt_bf16* dlogits,
                               int32_t* err, tt_stream_t stream) {
  if (!logits || !targets || !logp || !loss || !err || N < 0 || V < 1 || ld < V) return TT_ERR_INVALID_ARG;
  if (N > (int64_t)INT32_MAX / 8) return TT_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (N == 0) {
    loss_kernel<<<1, 1024, 0, st>>>(logp, weights, 0, loss);
    TT_LAUNCH_CHECK();
    return TT_OK;
  }
  LpArgs a;
  a.logits = reinterpret_cast<const __nv_bfloat16*>(logits);
  a.N = N; a.V = V; a.ld = ld; a.targets = targets; a.weights = weights; a.g = g; a.logp = logp;
  a.dlogits = reinterpret_cast<__nv_bfloat16*>(dlogits); a.err = err;
  const bool vec_ok = aligned16(logits) && (ld % 8 == 0) && (!dlogits || aligned16(dlogits));
  const int64_t per_cta = (int64_t)kLpThreads * 8;  // elements per CTA per chunk
  cudaError_t e = cudaSuccess;
  bool done = false;
  if (vec_ok) {
    const int chs[] = {1, 2, 4, 10};
    for (int ch : chs) {
      const int64_t CL = (V + per_cta * ch - 1) / (per_cta * ch);
      if (CL > 8) continue;
      const int cl = (int)CL;
      switch (ch) {
        case 1: e = launch_cluster<1>(a, cl, st); break;
        case 2: e = launch_cluster<2>(a, cl, st); break;
        case 4: e = launch_cluster<4>(a, cl, st); break;
        default: e = launch_cluster<10>(a, cl, st); break;
      }
      done = true;
      break;
    }
  }
  if (!done) wlp_generic_kernel<<<(unsigned)N, kLpThreads, 0, st>>>(a);
  if (e != cudaSuccess) return TT_ERR_CUDA;
  TT_LAUNCH_CHECK();
  loss_kernel<<<1, 1024, 0, st>>>(logp, weights, N, loss);
  TT_LAUNCH_CHECK();
  return TT_OK;
}
