// LM head fused with the weighted log-prob loss on the 5th-generation tensor
// cores: the logits z = H·Wᵀ are formed tile by tile in tensor memory and
// folded into per-row log-sum-exp partials there; they never reach global
// memory.
//
// "Tree Training", Abstract: averaging the per-branch losses equals one pass
// over the tree's tokens in which a token's term is scaled by the share of
// branches through it, so each token's log-probability is computed once:
//   lse_t = log Σ_v exp(z_tv),  logp_t = z_{t,y_t} − lse_t,
//   loss  = −Σ_t w_t·logp_t,    z_tv = <H_t, W_v>.
// The pages give no detail of the LM head itself; this is the plain product
// of the final hidden states H [N][Hd] with the vocabulary matrix W [V][Hd].
//
// lmhead_gemm_kernel<EPI_LSE> (the forward): persistent, one CTA per SM, 6 warps.
//   Tiles of 128 rows x 256 vocabulary entries, vocabulary-major (tile t =
//   v·nR + r): at any time the CTAs work on the row tiles of one or two
//   vocabulary tiles, so each 1 MB slice of W is read from DRAM once and
//   reused from L2 by every row tile, and H (N·Hd·2 bytes) stays in L2.
//   warp 0     TMA producer: per 64-wide K step one [128][64] box of H and
//              one [256][64] box of W into a 4-stage ring (48 KB a stage);
//   warp 1     MMA issuer (one thread): z_tile += A·Bᵀ, M = 128, N = 256,
//              K = 16 per instruction, into one of two TMEM accumulators
//              (256 columns each), so the epilogue of one tile overlaps the
//              MMAs of the next;
//   warps 2..5 epilogue, one thread per row (= TMEM lane): reads the tile's
//              256 fp32 logits in 32-column pieces, masks columns >= V, and
//              keeps an online maximum m of z and rescaled sum
//              s = Σ 2^((z − m)·log2 e); picks the target's raw logit when the
//              target column falls in the tile. Writes (m, s) per (vocab
//              tile, row) and z_{t,y_t} to the workspace. The maximum stays in
//              natural units, so the rounding of log2 e only scales the
//              exponents' offsets from it and does not shift lse.
// lmhead_combine_kernel: per row, merges the nV partials in a fixed order
//   (M = max m_j, S = Σ s_j·e^(m_j − M)), lse = M + ln S, logp.
// The fixed-order loss reduction of the log-prob call follows.
//
// Backward (gradients of g·loss): dz_tv = g·w_t·(e^(z_tv − lse_t) − [v == y_t]),
// dH = dz·W, dW = dzᵀ·H. The same persistent kernel, templated on its
// epilogue and on the major-ness of its operands, runs three GEMMs:
//   dz  = H·Wᵀ with the epilogue above turned into dz (bf16, stored: the
//         3.85 GB gradient of the logits is the one array the backward keeps);
//   dH  = dz·W   (A = dz K-major; B = W read MN-major: [64 vocab rows][64
//         hidden columns] boxes, no transpose);
//   dW  = dzᵀ·H  (A = dz and B = H both read MN-major), fp32 output.
// An MN-major operand is staged as [64 K rows][64 M-or-N columns] boxes with
// 128-byte swizzle: the UMMA descriptor's leading offset is one box (8 KB,
// the next 64 columns), its stride 1024 bytes (8 K rows), and each K = 16
// step advances 2048 bytes.
#include <algorithm>

#include "tc_common.cuh"

namespace tt {
namespace {

using namespace tc;

constexpr int kLhWarps = 6;
constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kBBytes = kBN * kBK * 2;  // 32 KB
constexpr uint32_t kBox = 64 * 64 * 2;       // one [64 K rows][64 columns] box of an MN-major operand
constexpr uint32_t kTmemCols = 512;          // two [128][256] fp32 accumulators
constexpr float kLog2e = 1.4426950408889634f;

// Epilogues: per-row log-sum-exp partials (forward), dz (bf16), plain bf16 / fp32 stores.
enum { EPI_LSE = 0, EPI_DZ = 1, EPI_BF16 = 2, EPI_F32 = 3 };

// mbarriers: FULL[s] (TMA bytes landed), EMPTY[s] (MMAs reading stage s done),
// ACC_FULL[a] (accumulator a holds a finished tile), ACC_EMPTY[a] (the 128
// epilogue threads have read it), FINAL (every MMA of the CTA done).
// TILE_FULL[r] / TILE_EMPTY[r]: the tile index in ring slot r published by
// the producer / read by the MMA thread and the 128 epilogue threads.
constexpr int kTileRing = 4;
constexpr int FULL = 0, EMPTY = FULL + kStages, ACC_FULL = EMPTY + kStages, ACC_EMPTY = ACC_FULL + 2,
              FINAL = ACC_EMPTY + 2, TILE_FULL = FINAL + 1, TILE_EMPTY = TILE_FULL + kTileRing,
              NBAR = TILE_EMPTY + kTileRing;

struct LhSmem {
  static constexpr uint32_t a0 = 0;
  static constexpr uint32_t b0 = a0 + kStages * kABytes;
  static constexpr uint32_t bars = b0 + kStages * kBBytes;
  static constexpr uint32_t ring = bars + NBAR * 8;  // [kTileRing] int64 tile indices
  static constexpr uint32_t misc = ring + kTileRing * 8;
  static constexpr uint32_t total = misc + 16 + 1024;  // + slack for 1024-byte alignment
};
static_assert(LhSmem::total <= 232448, "LM-head shared memory exceeds the per-CTA limit");

struct LhArgs {
  int64_t M, Ncols;  // output rows and columns
  int ksteps;        // ceil(K / 64)
  int nM, nN;        // tiles along M and N
  int64_t tiles;     // nM · nN
  int n_outer;       // tile order: 1 = t -> (n = t / nM, m = t % nM), 0 = (m = t / nN, n = t % nN)
  int* counter;      // tiles claimed so far (zero at launch): CTAs take tiles as they free up; NULL = fixed stride
  const int32_t* targets;  // EPI_LSE, EPI_DZ (M = tokens, N = vocabulary)
  const float* weights;    // EPI_DZ: NULL = ones
  float g;                 // EPI_DZ
  const float* lse;        // EPI_DZ: per row, natural log
  float* pm;               // EPI_LSE: [nN][M] max of z over the tile's columns
  float* ps;               // EPI_LSE: [nN][M] Σ 2^((z − m)·log2 e)
  float* pz;               // EPI_LSE: [M] z_{t, y_t}
  __nv_bfloat16* ob;       // EPI_DZ, EPI_BF16: [M][ldo]
  float* of;               // EPI_F32: [M][ldo]
  int64_t ldo;
  int32_t* err;
};

template <int EPI, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kLhWarps * 32, 1)
    lmhead_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const LhArgs a) {
  using L = LhSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::misc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar[FULL + i], 1);
      mbar_init(&bar[EMPTY + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[ACC_FULL + i], 1);
      mbar_init(&bar[ACC_EMPTY + i], 128);
    }
    mbar_init(&bar[FINAL], 1);
    for (int i = 0; i < kTileRing; ++i) {
      mbar_init(&bar[TILE_FULL + i], 1);
      mbar_init(&bar[TILE_EMPTY + i], 1 + 128);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const int64_t t_first = blockIdx.x, t_step = gridDim.x;
  volatile int64_t* ring = reinterpret_cast<volatile int64_t*>(sm + L::ring);
  // the tile of this CTA's it-th turn (a value >= tiles ends the loop): with
  // a counter, published by the producer through the ring; else fixed stride
  auto take_tile = [&](int it, int64_t& t, int site) -> bool {
    if (!a.counter) {
      t = t_first + (int64_t)it * t_step;
      return true;
    }
    const int r = it % kTileRing;
    if (!mbar_wait(&bar[TILE_FULL + r], (uint32_t)((it / kTileRing) & 1), abort_flag, site)) return false;
    t = ring[r];
    mbar_arrive(&bar[TILE_EMPTY + r]);
    return true;
  };
  auto tile_mn = [&](int64_t t, int& m, int& n) {
    if (a.n_outer) {
      n = (int)(t / a.nM);
      m = (int)(t % a.nM);
    } else {
      m = (int)(t / a.nN);
      n = (int)(t % a.nN);
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      int64_t kk = 0;  // K steps issued by this CTA (ring position)
      bool ok = true;
      for (int it = 0; ok; ++it) {
        int64_t t = t_first + (int64_t)it * t_step;
        if (a.counter) {
          // claim the next tile and publish it to the MMA thread and the epilogue
          const int r = it % kTileRing;
          if (it >= kTileRing &&
              !mbar_wait(&bar[TILE_EMPTY + r], (uint32_t)((it / kTileRing - 1) & 1), abort_flag, 5))
            break;
          t = (int64_t)atomicAdd(a.counter, 1);
          ring[r] = t;
          mbar_arrive(&bar[TILE_FULL + r]);
        }
        if (t >= a.tiles) break;
        int m, n;
        tile_mn(t, m, n);
        for (int ks = 0; ks < a.ksteps; ++ks, ++kk) {
          const int st = (int)(kk % kStages);
          if (kk >= kStages && !mbar_wait(&bar[EMPTY + st], (uint32_t)((kk / kStages - 1) & 1), abort_flag, 1)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&bar[FULL + st], kABytes + kBBytes);
          uint8_t* sa = sm + L::a0 + st * kABytes;
          uint8_t* sb = sm + L::b0 + st * kBBytes;
          if (A_MN) {  // A stored [K][M]: two [64 K][64 M] boxes
#pragma unroll
            for (int i = 0; i < kBM / 64; ++i) tma_load_2d(sa + i * kBox, &tmA, &bar[FULL + st], m * kBM + 64 * i, ks * kBK);
          } else {  // A stored [M][K]: one [128 M][64 K] box
            tma_load_2d(sa, &tmA, &bar[FULL + st], ks * kBK, m * kBM);
          }
          if (B_MN) {  // B stored [K][N]: four [64 K][64 N] boxes
#pragma unroll
            for (int i = 0; i < kBN / 64; ++i) tma_load_2d(sb + i * kBox, &tmB, &bar[FULL + st], n * kBN + 64 * i, ks * kBK);
          } else {  // B stored [N][K]: one [256 N][64 K] box
            tma_load_2d(sb, &tmB, &bar[FULL + st], ks * kBK, n * kBN);
          }
        }
      }
      // every copy issued has landed before the CTA may leave
      for (int64_t j = kk - 1; j >= 0 && j >= kk - kStages; --j)
        mbar_drain(&bar[FULL + (int)(j % kStages)], (uint32_t)((j / kStages) & 1), abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, kBN, A_MN ? 1 : 0, B_MN ? 1 : 0);
      // K-major: 128-byte rows of K, 8-row groups 1024 bytes apart, K = 16 is 32 bytes on.
      // MN-major: 64-column boxes kBox apart, 8 K rows 1024 bytes apart, K = 16 is 2048 bytes on.
      const uint64_t da = A_MN ? smem_desc(smem_u32(sm + L::a0), kBox, 1024) : smem_desc(smem_u32(sm + L::a0), 16, 1024);
      const uint64_t db = B_MN ? smem_desc(smem_u32(sm + L::b0), kBox, 1024) : smem_desc(smem_u32(sm + L::b0), 16, 1024);
      constexpr uint32_t ka = A_MN ? 2048 : 32, kb = B_MN ? 2048 : 32;
      int64_t kk = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        int64_t t;
        if (!take_tile(it, t, 6) || t >= a.tiles) break;
        const int acc = it & 1;
        // the epilogue has read this accumulator's previous tile (it − 2)
        if (it >= 2 && !mbar_wait(&bar[ACC_EMPTY + acc], (uint32_t)(((it - 2) >> 1) & 1), abort_flag, 2)) break;
        tc_fence_after();
        const uint32_t dcol = tbase + (uint32_t)acc * kBN;
        for (int ks = 0; ks < a.ksteps; ++ks, ++kk) {
          const int st = (int)(kk % kStages);
          if (!mbar_wait(&bar[FULL + st], (uint32_t)((kk / kStages) & 1), abort_flag, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            umma_ss(dcol, desc_at(da, st * kABytes + k * ka), desc_at(db, st * kBBytes + k * kb), idesc,
                    (ks > 0 || k > 0) ? 1u : 0u);
          umma_commit(&bar[EMPTY + st]);  // stage st free once these MMAs have read it
        }
        if (ok) umma_commit(&bar[ACC_FULL + acc]);
      }
      // completes after every MMA of this CTA (waited for even after an abort:
      // TMEM and shared memory must outlive the MMAs)
      umma_commit(&bar[FINAL]);
      mbar_drain(&bar[FINAL], 0, abort_flag);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;  // TMEM lane quarter this warp may read
    const int rl = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    for (int it = 0;; ++it) {
      int64_t t;
      if (!take_tile(it, t, 7) || t >= a.tiles) break;
      const int acc = it & 1;
      int m, n;
      tile_mn(t, m, n);
      const int64_t row = (int64_t)m * kBM + rl;
      const int64_t c0 = (int64_t)n * kBN;  // first column of the tile
      const bool row_ok = row < a.M;
      int y = -1;
      float gw = 0.f, lrow = 0.f;
      if (EPI == EPI_LSE || EPI == EPI_DZ) y = row_ok ? a.targets[row] : -1;
      if (EPI == EPI_DZ && row_ok) {
        gw = a.g * (a.weights ? a.weights[row] : 1.f);
        lrow = a.lse[row];
        if ((y < 0 || (int64_t)y >= a.Ncols) && n == 0) set_err(a.err, TT_ERR_INVALID_ARG);
      }
      const int64_t yc = (int64_t)y - c0;  // target column within the tile
      if (!mbar_wait(&bar[ACC_FULL + acc], (uint32_t)((it >> 1) & 1), abort_flag, 4)) break;
      tc_fence_after();
      float m_run = -INFINITY, s_run = 0.f, zt = 0.f;
      bool found = false;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tbase + lane_base + (uint32_t)acc * kBN + c * 32, u);
        tmem_ld_wait();
        tmem_pin(u);
        const int64_t col0 = c0 + c * 32;
        const int64_t nvalid = a.Ncols - col0;  // columns j < nvalid exist
        if (EPI == EPI_LSE) {
          float cm = -INFINITY;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float z = j < nvalid ? __uint_as_float(u[j]) : -INFINITY;
            u[j] = __float_as_uint(z);
            cm = fmaxf(cm, z);
          }
          if ((uint64_t)(yc - c * 32) < 32u) {
            // u[jc] by a tree of selects on the bits of jc (no indexed register access)
            const int jc = (int)(yc - c * 32);
            uint32_t sel[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) sel[j] = (jc & 16) ? u[j + 16] : u[j];
#pragma unroll
            for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
              for (int j = 0; j < w; ++j) sel[j] = (jc & w) ? sel[j + w] : sel[j];
            zt = __uint_as_float(sel[0]);
            found = true;
          }
          const float nm = fmaxf(m_run, cm);
          if (nm != -INFINITY) {
            s_run *= fast_exp2((m_run - nm) * kLog2e);  // 0 while m_run is still -inf (s_run is 0 then)
            const float2 l2 = make_float2(kLog2e, kLog2e), nn = make_float2(-nm, -nm);
            float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float2 x = __fmul2_rn(
                  __fadd2_rn(make_float2(__uint_as_float(u[2 * j]), __uint_as_float(u[2 * j + 1])), nn), l2);
              acc2 = __fadd2_rn(acc2, make_float2(fast_exp2(x.x), fast_exp2(x.y)));
            }
            s_run += acc2.x + acc2.y;
            m_run = nm;
          }
        } else if (EPI == EPI_F32) {
          if (row_ok) {
            float* dst = a.of + row * a.ldo + col0;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (4 * q < nvalid)
                *reinterpret_cast<float4*>(dst + 4 * q) =
                    make_float4(__uint_as_float(u[4 * q]), __uint_as_float(u[4 * q + 1]), __uint_as_float(u[4 * q + 2]),
                                __uint_as_float(u[4 * q + 3]));
          }
        } else {
          if (EPI == EPI_DZ) {
            // dz = g·w·(e^(z − lse) − [column == target])
            const float2 l2 = make_float2(kLog2e, kLog2e), nl = make_float2(-lrow, -lrow);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float2 x = __fmul2_rn(
                  __fadd2_rn(make_float2(__uint_as_float(u[2 * j]), __uint_as_float(u[2 * j + 1])), nl), l2);
              u[2 * j] = __float_as_uint(gw * fast_exp2(x.x));
              u[2 * j + 1] = __float_as_uint(gw * fast_exp2(x.y));
            }
            if ((uint64_t)(yc - c * 32) < 32u) {
              const int jc = (int)(yc - c * 32);
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j == jc) u[j] = __float_as_uint(__uint_as_float(u[j]) - gw);
            }
          }
          if (row_ok) {
            __nv_bfloat16* dst = a.ob + row * a.ldo + col0;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (8 * q < nvalid) {
                uint4 w4;
                w4.x = pack_bf16(__uint_as_float(u[8 * q + 0]), __uint_as_float(u[8 * q + 1]));
                w4.y = pack_bf16(__uint_as_float(u[8 * q + 2]), __uint_as_float(u[8 * q + 3]));
                w4.z = pack_bf16(__uint_as_float(u[8 * q + 4]), __uint_as_float(u[8 * q + 5]));
                w4.w = pack_bf16(__uint_as_float(u[8 * q + 6]), __uint_as_float(u[8 * q + 7]));
                *reinterpret_cast<uint4*>(dst + 8 * q) = w4;
              }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bar[ACC_EMPTY + acc]);
      if (EPI == EPI_LSE && row_ok) {
        a.pm[(int64_t)n * a.M + row] = m_run;
        a.ps[(int64_t)n * a.M + row] = s_run;
        if (found) a.pz[row] = zt;
      }
    }
  }
  if (*abort_flag && threadIdx.x == 0) set_err(a.err, TT_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// One persistent launch (one CTA per SM, at most one per tile).
template <int EPI, bool A_MN, bool B_MN>
int launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const LhArgs& a, cudaStream_t st) {
  const int smem = (int)LhSmem::total;
  if (!smem_attr_set<lmhead_gemm_kernel<EPI, A_MN, B_MN>>(smem)) return TT_ERR_CUDA;
  const int64_t grid = std::min<int64_t>(a.tiles, (int64_t)sm_count());
  {
    KtScope kt(TT_KT_LMHEAD, st);
    lmhead_gemm_kernel<EPI, A_MN, B_MN><<<(unsigned)grid, kLhWarps * 32, smem, st>>>(ta, tb, a);
  }
  return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

// Per row: M = max_j m_j, S = Σ_j s_j·e^(m_j − M) over the nV vocabulary
// tiles; lse = M + ln S, logp = z_{t,y_t} − lse. A target outside [0, V)
// sets err = TT_ERR_INVALID_ARG and that row's logp to NaN. A block takes 32
// rows (one per lane: consecutive rows, coalesced loads) and splits their
// tiles over kCombineWarps warps (warp w: tiles w, w + 8, ...); the warps'
// pairs are then merged in warp order, so the sums have a fixed order.
constexpr int kCombineWarps = 8;
__device__ __forceinline__ void lse_merge(float& M, float& S, float m, float s) {
  if (m > M) {
    S = S * expf(M - m) + s;
    M = m;
  } else if (m != -INFINITY) {
    S += s * expf(m - M);
  }
}
__global__ void __launch_bounds__(32 * kCombineWarps)
    lmhead_combine_kernel(const float* pm, const float* ps, const float* pz, int64_t N, int nV, int64_t V,
                          const int32_t* targets, float* logp, float* lse, int32_t* err) {
  __shared__ float2 part[kCombineWarps][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * 32 + lane;
  float M = -INFINITY, S = 0.f;
  if (row < N)
    for (int j = w; j < nV; j += kCombineWarps) lse_merge(M, S, pm[(int64_t)j * N + row], ps[(int64_t)j * N + row]);
  part[w][lane] = make_float2(M, S);
  __syncthreads();
  if (w != 0 || row >= N) return;
  M = -INFINITY;
  S = 0.f;
#pragma unroll
  for (int k = 0; k < kCombineWarps; ++k) lse_merge(M, S, part[k][lane].x, part[k][lane].y);
  const float l = M + logf(S);
  const int y = targets[row];
  float lp;
  if (y < 0 || (int64_t)y >= V) {
    set_err(err, TT_ERR_INVALID_ARG);
    lp = __int_as_float(0x7fc00000);
  } else {
    lp = pz[row] - l;
  }
  if (lse) lse[row] = l;
  logp[row] = lp;
}

struct LhWs {
  size_t pm, ps, pz, total;
};
LhWs lh_layout(int64_t N, int64_t V) {
  const int64_t nV = (V + kBN - 1) / kBN;
  LhWs w;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes, 256); return r; };
  w.pm = take(sizeof(float) * (size_t)nV * (size_t)N);
  w.ps = take(sizeof(float) * (size_t)nV * (size_t)N);
  w.pz = take(sizeof(float) * (size_t)N);
  w.total = o;
  return w;
}

}  // namespace
}  // namespace tt

using namespace tt;

TT_API size_t tt_lmhead_logprob_workspace_bytes(int64_t N, int64_t V) {
  if (N < 1 || V < 1) return 0;
  return lh_layout(N, V).total;
}

namespace {
LhArgs lh_args(int64_t M, int64_t Ncols, int64_t K, int n_outer, int32_t* err) {
  LhArgs a = {};
  a.M = M; a.Ncols = Ncols; a.ksteps = (int)((K + kBK - 1) / kBK);
  a.nM = (int)((M + kBM - 1) / kBM);
  a.nN = (int)((Ncols + kBN - 1) / kBN);
  a.tiles = (int64_t)a.nM * a.nN;
  a.n_outer = n_outer;
  a.err = err;
  return a;
}
int lh_check(const tt_bf16* hidden, const tt_bf16* w_vocab, int64_t N, int64_t V, int Hd, const int32_t* targets,
             const int32_t* err) {
  if (!hidden || !w_vocab || !targets || !err || N < 1 || V < 1 || Hd < 1) return TT_ERR_INVALID_ARG;
  if (Hd % kBK != 0) return TT_ERR_UNSUPPORTED;
  if (N > (int64_t)INT32_MAX - kBM || V > (int64_t)INT32_MAX - kBN) return TT_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(w_vocab)) return TT_ERR_INVALID_ARG;
  return TT_OK;
}
}  // namespace

TT_API int tt_lmhead_logprob(const tt_bf16* hidden, const tt_bf16* w_vocab, int64_t N, int64_t V, int Hd,
                             const int32_t* targets, const float* weights, float* logp, float* lse, double* loss,
                             void* ws, size_t ws_bytes, int32_t* err, tt_stream_t stream) {
  int rc = lh_check(hidden, w_vocab, N, V, Hd, targets, err);
  if (rc) return rc;
  if (!logp || !loss || !ws || !aligned16(ws)) return TT_ERR_INVALID_ARG;
  const LhWs Lw = lh_layout(N, V);
  if (ws_bytes < Lw.total) return TT_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  CUtensorMap mh, mw;
  if (!make_tmap_bf16(&mh, hidden, (uint64_t)Hd, (uint64_t)N, kBM) ||
      !make_tmap_bf16(&mw, w_vocab, (uint64_t)Hd, (uint64_t)V, kBN))
    return TT_ERR_CUDA;
  // z = H·Wᵀ: M = tokens, columns = vocabulary, K = Hd; vocabulary-major tiles
  LhArgs a = lh_args(N, V, Hd, 1, err);
  a.targets = targets;
  a.pm = ws_at<float>(ws, Lw.pm);
  a.ps = ws_at<float>(ws, Lw.ps);
  a.pz = ws_at<float>(ws, Lw.pz);
  // 58,806 equal tiles at the benchmarked shape: a fixed stride leaves no tail
  rc = launch_gemm<EPI_LSE, false, false>(mh, mw, a, st);
  if (rc) return rc;
  lmhead_combine_kernel<<<(unsigned)((N + 31) / 32), 32 * kCombineWarps, 0, st>>>(a.pm, a.ps, a.pz, N, a.nN, V,
                                                                                 targets, logp, lse, err);
  TT_LAUNCH_CHECK();
  return cuda_status(launch_weighted_loss(logp, weights, N, loss, st));
}

// dz [N][ldz] bf16 with ldz = V rounded up to 8 (16-byte rows for the tensor maps).
static inline int64_t dz_ld(int64_t V) { return (V + 7) / 8 * 8; }

// Backward scratch: dz, then the three GEMMs' tile counters.
static inline size_t dz_bytes(int64_t N, int64_t V) { return align_up((size_t)N * (size_t)dz_ld(V) * 2, 256); }

TT_API size_t tt_lmhead_logprob_bwd_workspace_bytes(int64_t N, int64_t V) {
  if (N < 1 || V < 1) return 0;
  return dz_bytes(N, V) + 256;
}

TT_API int tt_lmhead_logprob_bwd(const tt_bf16* hidden, const tt_bf16* w_vocab, int64_t N, int64_t V, int Hd,
                                 const int32_t* targets, const float* weights, float g, const float* lse,
                                 tt_bf16* d_hidden, float* d_w_vocab, void* ws, size_t ws_bytes, int32_t* err,
                                 tt_stream_t stream) {
  int rc = lh_check(hidden, w_vocab, N, V, Hd, targets, err);
  if (rc) return rc;
  if (!lse || !d_hidden || !d_w_vocab || !ws || !aligned16(ws) || !aligned16(d_hidden) || !aligned16(d_w_vocab))
    return TT_ERR_INVALID_ARG;
  if (ws_bytes < tt_lmhead_logprob_bwd_workspace_bytes(N, V)) return TT_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  __nv_bfloat16* dz = static_cast<__nv_bfloat16*>(ws);
  const int64_t ldz = dz_ld(V);
  int* ctr = ws_at<int>(ws, dz_bytes(N, V));  // [3]: dz, dH, dW
  if (cudaMemsetAsync(ctr, 0, 3 * sizeof(int), st) != cudaSuccess) return TT_ERR_CUDA;
  // 1. dz = g·w·(softmax(H·Wᵀ) − onehot): the forward's tiles with the dz epilogue
  CUtensorMap mh, mw;
  if (!make_tmap_bf16(&mh, hidden, (uint64_t)Hd, (uint64_t)N, kBM) ||
      !make_tmap_bf16(&mw, w_vocab, (uint64_t)Hd, (uint64_t)V, kBN))
    return TT_ERR_CUDA;
  LhArgs a = lh_args(N, V, Hd, 1, err);
  a.targets = targets; a.weights = weights; a.g = g; a.lse = lse; a.ob = dz; a.ldo = ldz; a.counter = ctr;
  rc = launch_gemm<EPI_DZ, false, false>(mh, mw, a, st);
  if (rc) return rc;
  // 2. dH = dz·W: A = dz [N][V] (K-major, K = V); B = W [V][Hd] read MN-major; token-major tiles
  CUtensorMap mdz, mw_mn;
  if (!make_tmap_bf16_ld(&mdz, dz, (uint64_t)V, (uint64_t)N, (uint64_t)ldz, kBM) ||
      !make_tmap_bf16(&mw_mn, w_vocab, (uint64_t)Hd, (uint64_t)V, 64))
    return TT_ERR_CUDA;
  LhArgs b = lh_args(N, Hd, V, 0, err);
  b.ob = reinterpret_cast<__nv_bfloat16*>(d_hidden); b.ldo = Hd; b.counter = ctr + 1;
  // 3. dW = dzᵀ·H: A = dz read MN-major ([K = tokens][M = vocabulary]), B = H [N][Hd] read MN-major
  CUtensorMap mdz_mn, mh_mn;
  if (!make_tmap_bf16_ld(&mdz_mn, dz, (uint64_t)V, (uint64_t)N, (uint64_t)ldz, 64) ||
      !make_tmap_bf16(&mh_mn, hidden, (uint64_t)Hd, (uint64_t)N, 64))
    return TT_ERR_CUDA;
  LhArgs c = lh_args(V, Hd, N, 0, err);
  c.of = d_w_vocab; c.ldo = Hd; c.counter = ctr + 2;
  // dH and dW both only read dz: dW runs on a second stream forked after dz,
  // so that its CTAs (which claim tiles as they free up) take the SMs that
  // dH's last round of tiles (792 tiles of K = V at the benchmarked shape,
  // 5.2 per SM) leaves idle; joined back before returning. Not while the
  // caller's stream is being captured into a graph (the second stream is
  // destroyed here, before such a capture would end).
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  const bool two = cudaStreamIsCapturing(st, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusNone &&
                   cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking) == cudaSuccess &&
                   cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) == cudaSuccess &&
                   cudaEventCreateWithFlags(&join, cudaEventDisableTiming) == cudaSuccess &&
                   cudaEventRecord(fork, st) == cudaSuccess && cudaStreamWaitEvent(side, fork, 0) == cudaSuccess;
  if (!two) (void)cudaGetLastError();
  rc = launch_gemm<EPI_BF16, false, true>(mdz, mw_mn, b, st);
  int rc2 = rc ? rc : launch_gemm<EPI_F32, true, true>(mdz_mn, mh_mn, c, two ? side : st);
  if (two && (cudaEventRecord(join, side) != cudaSuccess || cudaStreamWaitEvent(st, join, 0) != cudaSuccess))
    rc2 = rc2 ? rc2 : TT_ERR_CUDA;
  if (join) cudaEventDestroy(join);
  if (fork) cudaEventDestroy(fork);
  if (side) cudaStreamDestroy(side);
  return rc ? rc : rc2;
}
