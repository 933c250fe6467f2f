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

#include <cuda_fp16.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace tt {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kLpThreads = 256;

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

// (m, s) represents s·exp(m); merge two such sums.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;  // both empty
  s = s * fast_exp2((m - M) * kLog2e) + s2 * fast_exp2((m2 - M) * kLog2e);
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
}

template <int CH>
__global__ void __launch_bounds__(kLpThreads, 2) wlp_cluster_kernel(LpArgs a, int CL) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ float2 part;
  const int rank = (int)cluster.block_rank();
  const int64_t row = blockIdx.x / CL;
  const int64_t nvec = (a.V + 7) / 8;
  const int64_t v_lo = rank * nvec / CL, v_hi = (rank + 1) * nvec / CL;
  const __nv_bfloat16* z = a.logits + row * a.ld;
  const int tid = threadIdx.x;

  const int y = a.targets[row];
  const bool yok = y >= 0 && y < a.V;
  const float w = a.weights ? a.weights[row] : 1.0f;
  float zy = 0.f;
  if (rank == 0 && tid == 0 && yok) zy = __bfloat162float(z[y]);

  uint4 raw[CH];
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
  float m = -INFINITY;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const uint32_t u[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(bf_lo(u[j]), bf_hi(u[j])));
  }
  // Exponentials against the thread's own maximum, kept as f16 pairs scaled by
  // 2^14 (folded into the ex2 argument): every value >= 2^-28 stays an f16
  // normal (relative error 2^-11, below the bf16 rounding of dlogits); the
  // sum is taken in fp32 before packing.
  const float mb = (m == -INFINITY) ? 0.f : m;
  uint32_t p[CH][4];
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const uint32_t u[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float e0 = fast_exp2(fmaf(bf_lo(u[j]) - mb, kLog2e, 14.f));
      const float e1 = fast_exp2(fmaf(bf_hi(u[j]) - mb, kLog2e, 14.f));
      s += e0 + e1;
      p[c][j] = pack_f16(e0, e1);
    }
  }
  s *= 6.103515625e-05f;  // 2^-14, exact
  float bm = m, bs = s;
  block_merge(bm, bs);
  if (tid == 0) part = make_float2(bm, bs);
  cluster.sync();
  float M = -INFINITY, Ssum = 0.f;
  for (int r = 0; r < CL; ++r) {
    const float2 q = *cluster.map_shared_rank(&part, r);
    lse_merge(M, Ssum, q.x, q.y);
  }
  const double lse = (double)M + log((double)Ssum);
  if (rank == 0 && tid == 0) {
    if (yok) a.logp[row] = (float)((double)zy - lse);
    else { a.logp[row] = __int_as_float(0x7fc00000); set_err(a.err, TT_ERR_INVALID_ARG); }
  }
  if (a.dlogits) {
    const float gw = a.g * w;
    const float cfac = gw * fast_exp2((float)(((double)mb - lse) * 1.4426950408889634) - 14.f);
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
  cluster.sync();  // keep `part` alive until every CTA of the cluster has read it
}

// Generic row kernel: pass 1 online (max, sum) over the row, pass 2 writes
// dlogits re-reading the row (from L2 for rows that fit).
__global__ void __launch_bounds__(kLpThreads) wlp_generic_kernel(LpArgs a) {
  const int64_t row = blockIdx.x;
  const __nv_bfloat16* z = a.logits + row * a.ld;
  float m = -INFINITY, s = 0.f;
  for (int64_t v = threadIdx.x; v < a.V; v += kLpThreads) {
    const float x = __bfloat162float(z[v]);
    if (x > m) { s = s * fast_exp2((m - x) * kLog2e) + 1.f; m = x; }
    else s += fast_exp2((x - m) * kLog2e);
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
    float d = gw * fast_exp2((__bfloat162float(z[v]) - lsef) * kLog2e);
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
  cfg.gridDim = dim3((unsigned)(a.N * CL));
  cfg.blockDim = dim3(kLpThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, wlp_cluster_kernel<CH>, a, CL);
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
