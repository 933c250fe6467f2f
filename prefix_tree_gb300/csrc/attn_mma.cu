// Tree attention, forward and backward, on warp-level bf16 MMA (mma.sync
// m16n8k16, fp32 accumulation). Reference path of the library: every
// attention entry point can run on it, and the tensor-memory kernels are
// checked against the same oracle.
//
// "Tree Training", Abstract: each token attends only to its root-to-token
// path, so the DFS-serialised tree reproduces independent per-branch
// attention exactly. With the DFS layout, key k is an ancestor of query t iff
// k <= t < send[k] (send = end of the DFS span of k's segment subtree), a
// per-key column interval. AReaL-DTA, Key Contributions 1–2: chunk mode runs
// a query chunk at path offset s0 against a contiguous path K/V (query i sees
// keys 0..s0+i) and accumulates key/value gradients into the path.
//
// Tiles: 128 query rows x 64 keys per step (8 warps x 16 rows). Key blocks
// with no ancestor pair are skipped with the per-128-key max of send; the
// element mask is applied only on blocks not known to be fully visible.
// Backward: dQ kernel (query-tile-major, re-derives P) + dK/dV kernel
// (key-tile-major, loops over the descendant query range and the query heads
// of its group), so no atomics and deterministic results.
#include "common.cuh"

namespace tt {
namespace {

constexpr int kBM = 128;  // query rows per CTA (forward / dQ), keys per CTA (dK/dV)
constexpr int kBN = 64;   // keys per step (forward / dQ), queries per step (dK/dV)
constexpr int kThreads = 256;
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;

enum Mode { kTree = 0, kChunk = 1 };

struct AttnArgs {
  const __nv_bfloat16 *q, *k, *v;
  __nv_bfloat16* o;
  float* lse;        // [hq][lse_ld]
  const float* lse_in;
  const __nv_bfloat16* dO;
  const float* dsum;  // [hq][nq]
  __nv_bfloat16 *dq, *dk, *dv;
  float *dk_acc, *dv_acc;
  int64_t nq, nk, q_off, lse_ld;
  const int32_t* send;     // tree: per-key subtree end
  const int32_t* blk_min;  // tree: per-128-key-block min / max of send
  const int32_t* blk_max;
  const int32_t* order;    // tree: longest-first tile order
  const int64_t* hdr;      // tree: workspace header (valid flag)
  int hq, hkv;
  float scale, scale_log2;
  int32_t* err;
};

// ---------------------------------------------------------------- primitives
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void cp16(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(ok ? 16 : 0));
}
__device__ __forceinline__ void cp4(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(ok ? 4 : 0));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// Row r, column col of an R x D bf16 tile with 16-byte chunks XOR-swizzled by r % 8.
template <int D>
__device__ __forceinline__ uint32_t sw(const __nv_bfloat16* base, int r, int col) {
  return smem_u32(base + r * D + ((((col >> 3) ^ (r & 7))) << 3));
}

// Rows [row0, row0+R) of a token-major matrix (row stride ld elements,
// head column offset already applied), zero-filled outside [0, nrows).
template <int D>
__device__ __forceinline__ void load_rows(__nv_bfloat16* s, const __nv_bfloat16* g, int64_t row0, int64_t nrows,
                                          int64_t ld, int R) {
  constexpr int CPR = D / 8;
  for (int i = threadIdx.x; i < R * CPR; i += kThreads) {
    const int r = i / CPR, c = i % CPR;
    const int64_t gr = row0 + r;
    const bool ok = gr >= 0 && gr < nrows;
    cp16(smem_u32(s + r * D + ((c ^ (r & 7)) << 3)), g + (ok ? gr : 0) * ld + c * 8, ok);
  }
}
__device__ __forceinline__ void load_ints(int32_t* s, const int32_t* g, int64_t row0, int64_t nrows, int R) {
  for (int i = threadIdx.x; i < R; i += kThreads) {
    const int64_t gr = row0 + i;
    const bool ok = gr >= 0 && gr < nrows;
    cp4(smem_u32(s + i), g + (ok ? gr : 0), ok);
  }
}
__device__ __forceinline__ void load_floats(float* s, const float* g, int64_t row0, int64_t nrows, int R) {
  for (int i = threadIdx.x; i < R; i += kThreads) {
    const int64_t gr = row0 + i;
    const bool ok = gr >= 0 && gr < nrows;
    cp4(smem_u32(s + i), g + (ok ? gr : 0), ok);
  }
}

// Does the workspace describe a valid tree of N tokens? (tree mode)
__device__ __forceinline__ bool tree_ok(const AttnArgs& a) {
  if (a.hdr[0] != kTreeMagic || a.hdr[1] != a.nq) {
    if (threadIdx.x == 0) set_err(a.err, TT_ERR_INVALID_ARG);
    return false;
  }
  if (a.hdr[3] == 0) {
    if (threadIdx.x == 0) set_err(a.err, TT_ERR_INVALID_TREE);
    return false;
  }
  return true;
}

// S = A·Bᵀ for one warp: 16 rows of sA (row offset ra) x 64 rows of sB, over D.
template <int D>
__device__ __forceinline__ void warp_qkt(float (&s)[8][4], const __nv_bfloat16* sA, int ra,
                                         const __nv_bfloat16* sB, int lane) {
#pragma unroll
  for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    uint32_t af[4];
    ldsm4(af, sw<D>(sA, ra + (lane & 7) + ((lane >> 3) & 1) * 8, kk * 16 + (lane >> 4) * 8));
#pragma unroll
    for (int n2 = 0; n2 < 4; ++n2) {
      uint32_t bf[4];
      ldsm4(bf, sw<D>(sB, n2 * 16 + (lane & 7) + (lane >> 4) * 8, kk * 16 + ((lane >> 3) & 1) * 8));
      mma16816(s[2 * n2], af, bf[0], bf[1]);
      mma16816(s[2 * n2 + 1], af, bf[2], bf[3]);
    }
  }
}

// acc[D/8][4] += P·B where P (16 x 64) is held as C fragments and B is a
// 64 x D tile stored row-major (rows = the contraction index).
template <int D>
__device__ __forceinline__ void warp_pv(float (&acc)[D / 8][4], const float (&p)[8][4], const __nv_bfloat16* sB,
                                        int lane) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    uint32_t pa[4];
    pa[0] = pack_bf16(p[2 * kk][0], p[2 * kk][1]);
    pa[1] = pack_bf16(p[2 * kk][2], p[2 * kk][3]);
    pa[2] = pack_bf16(p[2 * kk + 1][0], p[2 * kk + 1][1]);
    pa[3] = pack_bf16(p[2 * kk + 1][2], p[2 * kk + 1][3]);
#pragma unroll
    for (int d2 = 0; d2 < D / 16; ++d2) {
      uint32_t bf[4];
      ldsm4t(bf, sw<D>(sB, kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, d2 * 16 + (lane >> 4) * 8));
      mma16816(acc[2 * d2], pa, bf[0], bf[1]);
      mma16816(acc[2 * d2 + 1], pa, bf[2], bf[3]);
    }
  }
}

__device__ __forceinline__ float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x + __shfl_xor_sync(0xffffffffu, x, 2);
}

// Query tile T of the forward / dQ grids.
__device__ __forceinline__ int query_tile(const AttnArgs& a, int mode, int ti) {
  const int nT = (int)((a.nq + kBM - 1) / kBM);
  return mode == kTree ? a.order[ti] : nT - 1 - ti;
}

// ---------------------------------------------------------------- forward
template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1) fwd_kernel(AttnArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* sK = sQ + kBM * D;
  __nv_bfloat16* sV = sK + 2 * kBN * D;
  int32_t* sSend = reinterpret_cast<int32_t*>(sV + 2 * kBN * D);
  if (MODE == kTree && !tree_ok(a)) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.x % a.hq;
  const int T = query_tile(a, MODE, blockIdx.x / a.hq);
  const int g = h / (a.hq / a.hkv);
  const int64_t q0 = (int64_t)T * kBM, q1 = min(q0 + kBM, a.nq);
  const int64_t ldq = (int64_t)a.hq * D, ldk = (int64_t)a.hkv * D;
  const int64_t kmax = MODE == kTree ? q1 : min(a.nk, a.q_off + q1);
  const int jend = (int)((kmax + kBN - 1) / kBN);
  auto next_block = [&](int j) {
    ++j;
    if (MODE == kTree)
      while (j < jend && a.blk_max[j >> 1] <= q0) ++j;
    return j;
  };
  auto issue = [&](int j, int buf) {
    load_rows<D>(sK + buf * kBN * D, a.k + g * D, (int64_t)j * kBN, a.nk, ldk, kBN);
    load_rows<D>(sV + buf * kBN * D, a.v + g * D, (int64_t)j * kBN, a.nk, ldk, kBN);
    if (MODE == kTree) load_ints(sSend + buf * kBN, a.send, (int64_t)j * kBN, a.nk, kBN);
  };

  load_rows<D>(sQ, a.q + h * D, q0, a.nq, ldq, kBM);
  int j = next_block(-1), buf = 0;
  if (j < jend) issue(j, 0);
  cp_commit();

  const int wr = warp * 16;
  const int64_t ra = q0 + wr + (lane >> 2), rb = ra + 8;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  float acc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  while (j < jend) {
    const int jn = next_block(j);
    if (jn < jend) issue(jn, buf ^ 1);
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    const __nv_bfloat16* cK = sK + buf * kBN * D;
    const __nv_bfloat16* cV = sV + buf * kBN * D;
    const int32_t* cS = sSend + buf * kBN;
    const int64_t kb = (int64_t)j * kBN;
    float s[8][4];
    warp_qkt<D>(s, sQ, wr, cK, lane);
    bool full;
    if (MODE == kTree) full = kb + kBN - 1 <= q0 && kb + kBN <= a.nk && a.blk_min[j >> 1] >= q1;
    else full = kb + kBN - 1 <= a.q_off + q0 && kb + kBN <= a.nk;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s[nt][e] * a.scale_log2;
        if (!full) {
          const int c = nt * 8 + (lane & 3) * 2 + (e & 1);
          const int64_t col = kb + c, row = e < 2 ? ra : rb;
          bool vis;
          if (MODE == kTree) vis = col <= row && row < cS[c];
          else vis = col <= a.q_off + row && col < a.nk;
          if (!vis) x = -INFINITY;
        }
        s[nt][e] = x;
      }
    }
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      mx_a = fmaxf(mx_a, fmaxf(s[nt][0], s[nt][1]));
      mx_b = fmaxf(mx_b, fmaxf(s[nt][2], s[nt][3]));
    }
    mx_a = quad_max(mx_a);
    mx_b = quad_max(mx_b);
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float mu_a = mn_a == -INFINITY ? 0.f : mn_a, mu_b = mn_b == -INFINITY ? 0.f : mn_b;
    const float c_a = fast_exp2(m_a - mu_a), c_b = fast_exp2(m_b - mu_b);
    float rs_a = 0.f, rs_b = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = fast_exp2(s[nt][0] - mu_a);
      s[nt][1] = fast_exp2(s[nt][1] - mu_a);
      s[nt][2] = fast_exp2(s[nt][2] - mu_b);
      s[nt][3] = fast_exp2(s[nt][3] - mu_b);
      rs_a += s[nt][0] + s[nt][1];
      rs_b += s[nt][2] + s[nt][3];
    }
    l_a = l_a * c_a + rs_a;
    l_b = l_b * c_b + rs_b;
    m_a = mn_a;
    m_b = mn_b;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      acc[i][0] *= c_a; acc[i][1] *= c_a; acc[i][2] *= c_b; acc[i][3] *= c_b;
    }
    warp_pv<D>(acc, s, cV, lane);
    __syncthreads();
    j = jn;
    buf ^= 1;
  }
  cp_wait<0>();
  l_a = quad_sum(l_a);
  l_b = quad_sum(l_b);
  const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f, inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
  const int64_t ldo = ldq;
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    const int col = i * 8 + (lane & 3) * 2;
    if (ra < a.nq)
      *reinterpret_cast<uint32_t*>(a.o + ra * ldo + h * D + col) = pack_bf16(acc[i][0] * inv_a, acc[i][1] * inv_a);
    if (rb < a.nq)
      *reinterpret_cast<uint32_t*>(a.o + rb * ldo + h * D + col) = pack_bf16(acc[i][2] * inv_b, acc[i][3] * inv_b);
  }
  if ((lane & 3) == 0) {
    if (ra < a.nq) a.lse[h * a.lse_ld + ra] = l_a > 0.f ? (m_a + __log2f(l_a)) * kLn2F : -INFINITY;
    if (rb < a.nq) a.lse[h * a.lse_ld + rb] = l_b > 0.f ? (m_b + __log2f(l_b)) * kLn2F : -INFINITY;
  }
}

// ---------------------------------------------------------------- backward
// dsum[h][t] = Σ_d dO[t,h,d]·O[t,h,d]
template <int D>
__global__ void dsum_kernel(AttnArgs a) {
  const int64_t wid = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= a.nq * a.hq) return;
  const int64_t t = wid / a.hq;
  const int h = (int)(wid % a.hq);
  const int64_t base = t * a.hq * D + (int64_t)h * D;
  float acc = 0.f;
#pragma unroll
  for (int c = lane * 2; c < D; c += 64) {
    const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(a.dO + base + c);
    const __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162*>(a.o + base + c);
    acc += __bfloat162float(x.x) * __bfloat162float(y.x) + __bfloat162float(x.y) * __bfloat162float(y.y);
  }
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) const_cast<float*>(a.dsum)[h * a.nq + t] = acc;
}

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1) dq_kernel(AttnArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* sdO = sQ + kBM * D;
  __nv_bfloat16* sK = sdO + kBM * D;
  __nv_bfloat16* sV = sK + 2 * kBN * D;
  int32_t* sSend = reinterpret_cast<int32_t*>(sV + 2 * kBN * D);
  if (MODE == kTree && !tree_ok(a)) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.x % a.hq;
  const int T = query_tile(a, MODE, blockIdx.x / a.hq);
  const int g = h / (a.hq / a.hkv);
  const int64_t q0 = (int64_t)T * kBM, q1 = min(q0 + kBM, a.nq);
  const int64_t ldq = (int64_t)a.hq * D, ldk = (int64_t)a.hkv * D;
  const int64_t kmax = MODE == kTree ? q1 : min(a.nk, a.q_off + q1);
  const int jend = (int)((kmax + kBN - 1) / kBN);
  auto next_block = [&](int j) {
    ++j;
    if (MODE == kTree)
      while (j < jend && a.blk_max[j >> 1] <= q0) ++j;
    return j;
  };
  auto issue = [&](int j, int buf) {
    load_rows<D>(sK + buf * kBN * D, a.k + g * D, (int64_t)j * kBN, a.nk, ldk, kBN);
    load_rows<D>(sV + buf * kBN * D, a.v + g * D, (int64_t)j * kBN, a.nk, ldk, kBN);
    if (MODE == kTree) load_ints(sSend + buf * kBN, a.send, (int64_t)j * kBN, a.nk, kBN);
  };
  load_rows<D>(sQ, a.q + h * D, q0, a.nq, ldq, kBM);
  load_rows<D>(sdO, a.dO + h * D, q0, a.nq, ldq, kBM);
  int j = next_block(-1), buf = 0;
  if (j < jend) issue(j, 0);
  cp_commit();

  const int wr = warp * 16;
  const int64_t ra = q0 + wr + (lane >> 2), rb = ra + 8;
  const float l2a = ra < a.nq ? a.lse_in[h * a.lse_ld + ra] * kLog2eF : 0.f;
  const float l2b = rb < a.nq ? a.lse_in[h * a.lse_ld + rb] * kLog2eF : 0.f;
  const float da = ra < a.nq ? a.dsum[h * a.nq + ra] : 0.f;
  const float db = rb < a.nq ? a.dsum[h * a.nq + rb] : 0.f;
  float acc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  while (j < jend) {
    const int jn = next_block(j);
    if (jn < jend) issue(jn, buf ^ 1);
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    const __nv_bfloat16* cK = sK + buf * kBN * D;
    const __nv_bfloat16* cV = sV + buf * kBN * D;
    const int32_t* cS = sSend + buf * kBN;
    const int64_t kb = (int64_t)j * kBN;
    float s[8][4], dp[8][4];
    warp_qkt<D>(s, sQ, wr, cK, lane);
    warp_qkt<D>(dp, sdO, wr, cV, lane);
    bool full;
    if (MODE == kTree) full = kb + kBN - 1 <= q0 && kb + kBN <= a.nk && a.blk_min[j >> 1] >= q1;
    else full = kb + kBN - 1 <= a.q_off + q0 && kb + kBN <= a.nk;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool top = e < 2;
        float p = fast_exp2(s[nt][e] * a.scale_log2 - (top ? l2a : l2b));
        if (!full) {
          const int c = nt * 8 + (lane & 3) * 2 + (e & 1);
          const int64_t col = kb + c, row = top ? ra : rb;
          bool vis;
          if (MODE == kTree) vis = col <= row && row < cS[c];
          else vis = col <= a.q_off + row && col < a.nk && row < a.nq;
          if (!vis) p = 0.f;
        }
        s[nt][e] = p * (dp[nt][e] - (top ? da : db));  // dS
      }
    }
    warp_pv<D>(acc, s, cK, lane);
    __syncthreads();
    j = jn;
    buf ^= 1;
  }
  cp_wait<0>();
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    const int col = i * 8 + (lane & 3) * 2;
    if (ra < a.nq)
      *reinterpret_cast<uint32_t*>(a.dq + ra * ldq + h * D + col) =
          pack_bf16(acc[i][0] * a.scale, acc[i][1] * a.scale);
    if (rb < a.nq)
      *reinterpret_cast<uint32_t*>(a.dq + rb * ldq + h * D + col) =
          pack_bf16(acc[i][2] * a.scale, acc[i][3] * a.scale);
  }
}

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1) dkdv_kernel(AttnArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* sV = sK + kBM * D;
  __nv_bfloat16* sQ = sV + kBM * D;
  __nv_bfloat16* sdO = sQ + 2 * kBN * D;
  float* sL = reinterpret_cast<float*>(sdO + 2 * kBN * D);  // [2][64] lse (natural)
  float* sDs = sL + 2 * kBN;                                // [2][64] dsum
  int32_t* sSendK = reinterpret_cast<int32_t*>(sDs + 2 * kBN);  // [128]
  if (MODE == kTree && !tree_ok(a)) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = blockIdx.x % a.hkv;
  const int bi = blockIdx.x / a.hkv;
  const int B = MODE == kTree ? a.order[bi] : bi;
  const int G = a.hq / a.hkv;
  const int64_t kb0 = (int64_t)B * kBM;
  const int64_t ldq = (int64_t)a.hq * D, ldk = (int64_t)a.hkv * D;
  // queries that see this key block: tree [kb0, max send); chunk i >= kb0 - s0
  int64_t qs, qe;
  if (MODE == kTree) { qs = kb0; qe = a.blk_max[B]; }
  else { qs = kb0 > a.q_off ? kb0 - a.q_off : 0; qe = a.nq; }
  qs = qs / kBN * kBN;
  const int nsub = qe > qs ? (int)((qe - qs + kBN - 1) / kBN) : 0;
  const int niter = nsub * G;
  auto issue = [&](int it, int buf) {
    const int h = g * G + it / nsub;
    const int64_t i0 = qs + (int64_t)(it % nsub) * kBN;
    load_rows<D>(sQ + buf * kBN * D, a.q + h * D, i0, a.nq, ldq, kBN);
    load_rows<D>(sdO + buf * kBN * D, a.dO + h * D, i0, a.nq, ldq, kBN);
    load_floats(sL + buf * kBN, a.lse_in + h * a.lse_ld, i0, a.nq, kBN);
    load_floats(sDs + buf * kBN, a.dsum + h * a.nq, i0, a.nq, kBN);
  };
  load_rows<D>(sK, a.k + g * D, kb0, a.nk, ldk, kBM);
  load_rows<D>(sV, a.v + g * D, kb0, a.nk, ldk, kBM);
  if (MODE == kTree) load_ints(sSendK, a.send, kb0, a.nk, kBM);
  if (niter > 0) issue(0, 0);
  cp_commit();

  const int wr = warp * 16;
  const int64_t ka = kb0 + wr + (lane >> 2), kbb = ka + 8;  // this thread's two key rows
  float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    dk[i][0] = dk[i][1] = dk[i][2] = dk[i][3] = 0.f;
    dv[i][0] = dv[i][1] = dv[i][2] = dv[i][3] = 0.f;
  }
  int buf = 0;
  for (int it = 0; it < niter; ++it) {
    if (it + 1 < niter) issue(it + 1, buf ^ 1);
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    const __nv_bfloat16* cQ = sQ + buf * kBN * D;
    const __nv_bfloat16* cdO = sdO + buf * kBN * D;
    const float* cL = sL + buf * kBN;
    const float* cD = sDs + buf * kBN;
    const int64_t i0 = qs + (int64_t)(it % nsub) * kBN;
    float st[8][4], dpt[8][4];
    warp_qkt<D>(st, sK, wr, cQ, lane);   // Sᵀ: keys x queries
    warp_qkt<D>(dpt, sV, wr, cdO, lane);  // dPᵀ
    bool full;
    if (MODE == kTree) full = i0 >= kb0 + kBM - 1 && i0 + kBN <= a.nq && kb0 + kBM <= a.nk && i0 + kBN <= a.blk_min[B];
    else full = a.q_off + i0 >= kb0 + kBM - 1 && i0 + kBN <= a.nq && kb0 + kBM <= a.nk;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = nt * 8 + (lane & 3) * 2 + (e & 1);
        const bool top = e < 2;
        float p = fast_exp2(st[nt][e] * a.scale_log2 - cL[c] * kLog2eF);
        if (!full) {
          const int64_t qi = i0 + c, kk = top ? ka : kbb;
          bool vis;
          if (MODE == kTree) vis = kk <= qi && qi < sSendK[kk - kb0] && qi < a.nq;
          else vis = kk <= a.q_off + qi && qi < a.nq && kk < a.nk;
          if (!vis) p = 0.f;
        }
        st[nt][e] = p;
        dpt[nt][e] = p * (dpt[nt][e] - cD[c]);
      }
    }
    warp_pv<D>(dv, st, cdO, lane);
    warp_pv<D>(dk, dpt, cQ, lane);
    __syncthreads();
    buf ^= 1;
  }
  cp_wait<0>();
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    const int col = i * 8 + (lane & 3) * 2;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int64_t kr = half ? kbb : ka;
      if (kr >= a.nk) continue;
      const float k0 = dk[i][2 * half] * a.scale, k1 = dk[i][2 * half + 1] * a.scale;
      const float v0 = dv[i][2 * half], v1 = dv[i][2 * half + 1];
      const int64_t off = kr * ldk + (int64_t)g * D + col;
      if (MODE == kTree) {
        *reinterpret_cast<uint32_t*>(a.dk + off) = pack_bf16(k0, k1);
        *reinterpret_cast<uint32_t*>(a.dv + off) = pack_bf16(v0, v1);
      } else {
        float2* pk = reinterpret_cast<float2*>(a.dk_acc + off);
        float2* pv = reinterpret_cast<float2*>(a.dv_acc + off);
        float2 x = *pk, y = *pv;
        x.x += k0; x.y += k1; y.x += v0; y.y += v1;
        *pk = x;
        *pv = y;
      }
    }
  }
}

// ---------------------------------------------------------------- launchers
template <int D>
constexpr size_t fwd_smem() { return (size_t)(kBM + 4 * kBN) * D * 2 + 2 * kBN * 4; }
template <int D>
constexpr size_t dq_smem() { return (size_t)(2 * kBM + 4 * kBN) * D * 2 + 2 * kBN * 4; }
template <int D>
constexpr size_t dkdv_smem() { return (size_t)(2 * kBM + 4 * kBN) * D * 2 + 4 * kBN * 4 + kBM * 4; }

template <typename K>
cudaError_t launch(K kern, size_t smem, unsigned grid, cudaStream_t st, const AttnArgs& a) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (grid == 0) return cudaSuccess;
  kern<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int D, int MODE>
cudaError_t run_fwd(const AttnArgs& a, cudaStream_t st) {
  const unsigned nT = (unsigned)((a.nq + kBM - 1) / kBM);
  return launch(fwd_kernel<D, MODE>, fwd_smem<D>(), nT * a.hq, st, a);
}

template <int D, int MODE>
cudaError_t run_bwd(const AttnArgs& a, cudaStream_t st) {
  const int64_t rows = a.nq * a.hq;
  dsum_kernel<D><<<(unsigned)((rows * 32 + kThreads - 1) / kThreads), kThreads, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned nT = (unsigned)((a.nq + kBM - 1) / kBM);
  e = launch(dq_kernel<D, MODE>, dq_smem<D>(), nT * a.hq, st, a);
  if (e != cudaSuccess) return e;
  const unsigned nB = (unsigned)((a.nk + kBM - 1) / kBM);
  return launch(dkdv_kernel<D, MODE>, dkdv_smem<D>(), nB * a.hkv, st, a);
}

int check_heads(int Hq, int Hkv, int d) {
  if (Hq < 1 || Hkv < 1) return TT_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return TT_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return TT_ERR_UNSUPPORTED;
  return TT_OK;
}

AttnArgs tree_args(const void* ws, int64_t N) {
  AttnArgs a = {};
  const TreeWs L = tree_ws_layout(0, N);
  a.hdr = ws_at<int64_t>(ws, L.hdr);
  a.send = ws_at<int32_t>(ws, L.send);
  a.blk_min = ws_at<int32_t>(ws, L.blk_min);
  a.blk_max = ws_at<int32_t>(ws, L.blk_max);
  return a;
}

}  // namespace

namespace tc {
int fwd_tree(const void* ws, const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t N, int Hq,
             int Hkv, int d, float scale, int32_t* err, cudaStream_t st);
int fwd_chunk(const void* q, int64_t C, int64_t s0, const void* k, const void* v, void* o, float* lse, int64_t lse_ld,
              int Hq, int Hkv, int d, float scale, int32_t* err, cudaStream_t st);
size_t bwd_ws_bytes(int64_t nq, int hq);
int bwd_tree(const void* ws, const void* Q, const void* K, const void* V, const void* O, const float* LSE,
             const void* dO, void* dQ, void* dK, void* dV, int64_t N, int Hq, int Hkv, int d, float scale,
             void* bws, int32_t* err, cudaStream_t st);
int bwd_chunk(const void* q, int64_t C, int64_t s0, const void* k, const void* v, const void* o, const float* lse,
              int64_t lse_ld, const void* dO, void* dq, float* dk_acc, float* dv_acc, int Hq, int Hkv, int d,
              float scale, void* bws, int32_t* err, cudaStream_t st);
}  // namespace tc
}  // namespace tt

using namespace tt;

#define TT_BF(p) reinterpret_cast<const __nv_bfloat16*>(p)
#define TT_BFW(p) reinterpret_cast<__nv_bfloat16*>(p)

TT_API int tt_tree_attn_fwd(const void* ws, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V, tt_bf16* O,
                            float* LSE, int64_t N, int Hq, int Hkv, int d, float scale, int32_t* err,
                            tt_stream_t stream) {
  int rc = check_heads(Hq, Hkv, d);
  if (rc) return rc;
  if (!ws || !Q || !K || !V || !O || !LSE || !err || N < 1 || N > INT32_MAX - kBM) return TT_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return TT_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!use_mma_kernels()) return tc::fwd_tree(ws, Q, K, V, O, LSE, N, Hq, Hkv, d, scale, err, st);
  AttnArgs a = tree_args(ws, N);
  a.order = ws_at<int32_t>(ws, tree_ws_layout(0, N).fwd_order);
  a.q = TT_BF(Q); a.k = TT_BF(K); a.v = TT_BF(V); a.o = TT_BFW(O); a.lse = LSE;
  a.nq = N; a.nk = N; a.q_off = 0; a.lse_ld = N; a.hq = Hq; a.hkv = Hkv;
  a.scale = scale; a.scale_log2 = scale * kLog2eF; a.err = err;
  cudaError_t e = d == 64 ? run_fwd<64, kTree>(a, st) : run_fwd<128, kTree>(a, st);
  return cuda_status(e);
}

TT_API size_t tt_tree_attn_bwd_workspace_bytes(int64_t N, int Hq) {
  if (N < 1 || Hq < 1) return 0;
  return align_up(tc::bwd_ws_bytes(N, Hq), 256);  // covers the warp-MMA kernels' [Hq][N] row sums too
}

TT_API int tt_tree_attn_bwd(const void* ws, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V, const tt_bf16* O,
                            const float* LSE, const tt_bf16* dO, tt_bf16* dQ, tt_bf16* dK, tt_bf16* dV, int64_t N,
                            int Hq, int Hkv, int d, float scale, void* bwd_ws, size_t bwd_ws_bytes, int32_t* err,
                            tt_stream_t stream) {
  int rc = check_heads(Hq, Hkv, d);
  if (rc) return rc;
  if (!ws || !Q || !K || !V || !O || !LSE || !dO || !dQ || !dK || !dV || !bwd_ws || !err || N < 1 ||
      N > INT32_MAX - kBM)
    return TT_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(dQ) ||
      !aligned16(dK) || !aligned16(dV))
    return TT_ERR_INVALID_ARG;
  if (bwd_ws_bytes < tt_tree_attn_bwd_workspace_bytes(N, Hq)) return TT_ERR_WORKSPACE;
  if (!aligned16(bwd_ws)) return TT_ERR_INVALID_ARG;
  if (!use_mma_kernels())
    return tc::bwd_tree(ws, Q, K, V, O, LSE, dO, dQ, dK, dV, N, Hq, Hkv, d, scale, bwd_ws, err,
                        reinterpret_cast<cudaStream_t>(stream));
  AttnArgs a = tree_args(ws, N);
  const TreeWs L = tree_ws_layout(0, N);
  a.q = TT_BF(Q); a.k = TT_BF(K); a.v = TT_BF(V); a.o = const_cast<__nv_bfloat16*>(TT_BF(O));
  a.lse_in = LSE; a.dO = TT_BF(dO); a.dsum = static_cast<float*>(bwd_ws);
  a.dq = TT_BFW(dQ); a.dk = TT_BFW(dK); a.dv = TT_BFW(dV);
  a.nq = N; a.nk = N; a.q_off = 0; a.lse_ld = N; a.hq = Hq; a.hkv = Hkv;
  a.scale = scale; a.scale_log2 = scale * kLog2eF; a.err = err;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // dQ grid uses the forward's query-tile order, dK/dV the key-block order.
  a.order = ws_at<int32_t>(ws, L.fwd_order);
  AttnArgs b = a;
  b.order = ws_at<int32_t>(ws, L.bwd_order);
  const int64_t rows = N * Hq;
  cudaError_t e;
  if (d == 64) {
    dsum_kernel<64><<<(unsigned)((rows * 32 + kThreads - 1) / kThreads), kThreads, 0, st>>>(a);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = launch(dq_kernel<64, kTree>, dq_smem<64>(), (unsigned)((N + kBM - 1) / kBM) * Hq, st, a);
    if (e == cudaSuccess)
      e = launch(dkdv_kernel<64, kTree>, dkdv_smem<64>(), (unsigned)((N + kBM - 1) / kBM) * Hkv, st, b);
  } else {
    dsum_kernel<128><<<(unsigned)((rows * 32 + kThreads - 1) / kThreads), kThreads, 0, st>>>(a);
    e = cudaGetLastError();
    if (e == cudaSuccess)
      e = launch(dq_kernel<128, kTree>, dq_smem<128>(), (unsigned)((N + kBM - 1) / kBM) * Hq, st, a);
    if (e == cudaSuccess)
      e = launch(dkdv_kernel<128, kTree>, dkdv_smem<128>(), (unsigned)((N + kBM - 1) / kBM) * Hkv, st, b);
  }
  return cuda_status(e);
}

TT_API int tt_tree_attn_chunk_fwd(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                  const tt_bf16* v_path, tt_bf16* o, float* lse, int64_t lse_ld, int Hq, int Hkv,
                                  int d, float scale, int32_t* err, tt_stream_t stream) {
  int rc = check_heads(Hq, Hkv, d);
  if (rc) return rc;
  if (!q || !k_path || !v_path || !o || !lse || !err || C < 1 || s0 < 0 || lse_ld < C ||
      s0 + C > (int64_t)INT32_MAX - kBM)
    return TT_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_path) || !aligned16(v_path) || !aligned16(o)) return TT_ERR_INVALID_ARG;
  if (!use_mma_kernels())
    return tc::fwd_chunk(q, C, s0, k_path, v_path, o, lse, lse_ld, Hq, Hkv, d, scale, err,
                         reinterpret_cast<cudaStream_t>(stream));
  AttnArgs a = {};
  a.q = TT_BF(q); a.k = TT_BF(k_path); a.v = TT_BF(v_path); a.o = TT_BFW(o); a.lse = lse;
  a.nq = C; a.nk = s0 + C; a.q_off = s0; a.lse_ld = lse_ld; a.hq = Hq; a.hkv = Hkv;
  a.scale = scale; a.scale_log2 = scale * kLog2eF; a.err = err;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = d == 64 ? run_fwd<64, kChunk>(a, st) : run_fwd<128, kChunk>(a, st);
  return cuda_status(e);
}

TT_API size_t tt_tree_attn_chunk_bwd_workspace_bytes(int64_t C, int Hq) {
  if (C < 1 || Hq < 1) return 0;
  return align_up(tc::bwd_ws_bytes(C, Hq), 256);
}

TT_API int tt_tree_attn_chunk_bwd(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                  const tt_bf16* v_path, const tt_bf16* o, const float* lse, int64_t lse_ld,
                                  const tt_bf16* dO, tt_bf16* dq, float* dk_acc, float* dv_acc, int Hq, int Hkv,
                                  int d, float scale, void* ws, size_t ws_bytes, int32_t* err, tt_stream_t stream) {
  int rc = check_heads(Hq, Hkv, d);
  if (rc) return rc;
  if (!q || !k_path || !v_path || !o || !lse || !dO || !dq || !dk_acc || !dv_acc || !ws || !err || C < 1 || s0 < 0 ||
      lse_ld < C || s0 + C > (int64_t)INT32_MAX - kBM)
    return TT_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_path) || !aligned16(v_path) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk_acc) || !aligned16(dv_acc))
    return TT_ERR_INVALID_ARG;
  if (ws_bytes < tt_tree_attn_chunk_bwd_workspace_bytes(C, Hq)) return TT_ERR_WORKSPACE;
  if (!aligned16(ws)) return TT_ERR_INVALID_ARG;
  if (!use_mma_kernels())
    return tc::bwd_chunk(q, C, s0, k_path, v_path, o, lse, lse_ld, dO, dq, dk_acc, dv_acc, Hq, Hkv, d, scale, ws, err,
                         reinterpret_cast<cudaStream_t>(stream));
  AttnArgs a = {};
  a.q = TT_BF(q); a.k = TT_BF(k_path); a.v = TT_BF(v_path); a.o = const_cast<__nv_bfloat16*>(TT_BF(o));
  a.lse_in = lse; a.dO = TT_BF(dO); a.dsum = static_cast<float*>(ws); a.dq = TT_BFW(dq);
  a.dk_acc = dk_acc; a.dv_acc = dv_acc;
  a.nq = C; a.nk = s0 + C; a.q_off = s0; a.lse_ld = lse_ld; a.hq = Hq; a.hkv = Hkv;
  a.scale = scale; a.scale_log2 = scale * kLog2eF; a.err = err;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = d == 64 ? run_bwd<64, kChunk>(a, st) : run_bwd<128, kChunk>(a, st);
  return cuda_status(e);
}
