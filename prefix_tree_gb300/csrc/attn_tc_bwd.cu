// Tree attention backward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// AReaL-DTA, Key Contributions 1: a shared prefix is backpropagated once with
// the gradients of all descendant leaves accumulated. With the DFS layout the
// queries that see key block b form the contiguous range [b·128, max send_b),
// so each key block's dK/dV is accumulated by one CTA over that range (and over
// the query heads of its group) with no atomics; dQ is accumulated by
// query-tile-major CTAs over the forward's key-block schedule. Both kinds of
// CTA run in ONE launch (bwd_tc_kernel: the kind with the longer CTAs first,
// each kind longest first), so each kind fills the SMs the other leaves idle. Chunk mode (query chunk at path offset s0 against a path K/V)
// uses the same kernel and accumulates fp32 path dK/dV.
//
// Inputs per query row: lse2 = LSE·log2(e) and dsum = Σ_d dO·O, written by a
// small pre-kernel into [Hq][ldp] arrays (ldp = N rounded up to 128; padding
// rows carry lse2 = +inf so their probabilities are exactly zero).
//
// dQ CTA  (one 128-row query tile x one query head, 11 warps)
//   warp 0 TMA (dO once; K and V per 128-key block, 4 and 2 stages), warp 1
//   S/dP MMAs, warp 10 dQ MMAs, warps 2..9 softmax (two per TMEM lane
//   quarter, 64 keys each; they also write Q into TMEM at the start).
//   TMEM: S [0, 128), dP [128, 256), dQ [256, 256+D), dS (bf16) [384, 448),
//   Q (bf16) [448, 448+D/2).
//   S = Q·Kᵀ (A from TMEM), dP = dO·Vᵀ (SS); P = exp2(S·c − lse2),
//   dS = P⊙(dP − dsum) as bf16 in TMEM; dQ += dS·K (A from TMEM, K as an
//   MN-major B operand).
// dK/dV CTA (one 128-key block x one KV head, warps 0..6; 7..10 idle)
//   warp 0 TMA (K, V once; Q, dO, lse2, dsum per 64-row query tile, 4 stages),
//   warp 1 Sᵀ/dPᵀ MMAs, warp 6 dV/dK MMAs, warps 2..5 one thread per key row.
//   TMEM: Sᵀ_b [64b, 64b+64) and dPᵀ_b [128+64b, ...) double buffered, Pᵀ_b
//   and dSᵀ_b (bf16) written over the first 32 columns of their buffers,
//   dV [256, 256+D), dK [384, 384+D).
//   Sᵀ = K·Qᵀ, dPᵀ = V·dOᵀ (SS); dV += Pᵀ·dO, dK += dSᵀ·Q (A from TMEM).
#include <type_traits>

#include "attn.cuh"
#include "tc_common.cuh"

namespace tt {
namespace tc {
namespace {

constexpr int kTreeM = 0, kChunkM = 1;
constexpr int kKvWarps = 6;     // dK/dV CTA: TMA, Sᵀ/dPᵀ MMA, 4 softmax (warps 0..5)
constexpr int kKvMmaWarp2 = 6;  // ... and the warp that issues the dV/dK MMAs
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kChunk = 128 * 128;  // one [128 rows][64 cols] bf16 box (bytes)

struct BwdTc {
  int64_t nq, nk, q_off, ldp;
  const float* lse2;   // [hq][ldp]
  const float* dsum;   // [hq][ldp]
  const int32_t* send;
  const int32_t* blk_min;
  const int32_t* blk_max;
  const int32_t* order_dq;  // tree: longest-first query-tile order (dQ CTAs)
  const int32_t* order_kv;  // tree: longest-first key-block order (dK/dV CTAs)
  const int64_t* hdr;
  const __nv_bfloat16* qp;  // Q rows (the dQ CTAs write them into TMEM)
  __nv_bfloat16 *dq, *dk, *dv;
  float *dk_acc, *dv_acc;
  int hq, hkv;
  float scale, scale_log2;
  int32_t* err;
};

__device__ __forceinline__ bool tree_header_ok(const BwdTc& a) {
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

// *p += (a, b, c, d) as one vector reduction in L2 (16-byte aligned p).
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}


// ---------------------------------------------------------------- dQ CTA
// Whole 128-key blocks, so that S = Q·Kᵀ and dP = dO·Vᵀ are N = 128 MMAs (an
// N = 64 MMA reads more shared memory per flop than the SM can deliver). Q
// sits in TMEM as the A operand of S (written there by the softmax threads at
// the start), which halves the shared-memory reads of S and leaves room for a
// 4-stage K ring: a K stage is freed only once dQ += dS·K of its block is
// done, and the ring keeps about three blocks of loads in flight ahead of the
// MMAs (a 32 KB tile takes over a microsecond to arrive under load). S and dP
// are single-buffered; the MMA thread issues, per block i,
//   S(i) [once S(i−1) has been read], dP(i) [once dP(i−1) has been read],
//   dQ += dS(i−1)·K(i−1) [once dS(i−1) is written],
// so the softmax warps read S(i) while dP(i) is formed and dP(i) while
// dQ(i−1) runs, and the pipe need not drain between blocks. dS (bf16, single
// buffer) is written once dQ(i−1) has read the previous one. Eight softmax
// warps: two per TMEM lane quarter, each thread one query row and 64 of the
// 128 keys. Two threads issue MMAs: one S and dP, the other dQ. A thread
// blocks in every wait and commit while the tensor pipe holds only a few of
// its MMAs, so with one issuer the pipe ran dry at each of the block's five
// waits; with two, one thread's MMAs keep the pipe busy while the other
// waits. No TMEM or shared buffer is handed between the two threads without
// a barrier of the softmax warps in between (dQ of a block is issued only
// after its dS is written, i.e. after its S and dP were read).

constexpr int kStages = 4;                                           // dK/dV query-tile stages
constexpr uint32_t kChunk64 = 64 * 128;                              // one [64 rows][64 cols] bf16 box (bytes)
constexpr int kDqWarps = 11;                                          // TMA, S/dP MMA, 8 softmax, dQ MMA
constexpr int kDqMmaWarp2 = 10;                                       // the warp that issues the dQ MMAs
constexpr int kDqKSt = 4, kDqVSt = 2;                                 // K stages, V stages
// TMEM columns: S, dP, dQ, dS (bf16 pairs), Q (bf16 pairs, A operand of S)
constexpr uint32_t kDqS = 0, kDqP = 128, kDqQ = 256, kDqDS = 384, kDqQA = 448;
// mbarrier slots. S and dP have barriers of their own, so that the softmax
// warps read S out of TMEM while dP is still being formed, and S of the next
// block can be issued as soon as S has been read (not once both are):
//   DO         dO tile loaded;
//   QA         every softmax thread has written its part of Q into TMEM;
//   KF[s]      K stage s loaded (its block index published with it);
//   KE[s]      dQ of the block in K stage s done (s = i % kDqKSt): frees the
//              K stage and the dS buffer;
//   VF[b]      V stage b loaded;
//   SFS        S of block i done;
//   SFP[b]     dP of block i done (b = i & 1); also frees V stage b;
//   SES / SEP  every softmax thread has loaded S / dP of the block (the TMEM
//              columns may be overwritten);
//   DSR        dS of the block written;
//   FINAL      both MMA threads' MMAs done (count 2).
// Each tcgen05.commit costs the MMA thread tens of cycles while the tensor
// pipe holds only a few queued MMAs, so one barrier serves every waiter of the
// same event.
constexpr int DQ_DO = 0, DQ_QA = 1, DQ_KF = 2, DQ_KE = DQ_KF + kDqKSt, DQ_VF = DQ_KE + kDqKSt,
              DQ_SFS = DQ_VF + kDqVSt, DQ_SFP = DQ_SFS + 1, DQ_SES = DQ_SFP + 2, DQ_SEP = DQ_SES + 1,
              DQ_DSR = DQ_SEP + 1, DQ_FINAL = DQ_DSR + 1, DQ_NBAR = DQ_FINAL + 1;
static_assert(kDqVSt == 2, "a V stage is released by the dP barrier of the same parity");

template <int D>
struct DqSmem {
  static constexpr uint32_t kTile = (D / 64) * kChunk;  // 128 rows
  static constexpr uint32_t dO = 0;
  static constexpr uint32_t k0 = dO + kTile;
  static constexpr uint32_t v0 = k0 + kDqKSt * kTile;
  static constexpr uint32_t kidx = v0 + kDqVSt * kTile;  // [kDqKSt] key block of each K stage (-1: end)
  static constexpr uint32_t kmin = kidx + 16;             // [kDqKSt] its minimum send (tree mode)
  static constexpr uint32_t bars = kmin + 16;
  static constexpr uint32_t misc = bars + DQ_NBAR * 8;
  static constexpr uint32_t total = misc + 16 + 1024;
};

// Chunk mode: the next 128-key block after b (b = -1 for the first) that the
// query rows [q0, q1) of the chunk see (every block up to the causal limit of
// the last row), or -1.
__device__ __forceinline__ int next_chunk_block(const BwdTc& a, int64_t q1, int b) {
  const int64_t kmax = min(a.nk, a.q_off + q1);
  return (int64_t)(b + 1) * 128 < kmax ? b + 1 : -1;
}

template <int D, int MODE>
__device__ __forceinline__ void dq_cta(const CUtensorMap& tmdO, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                       const BwdTc& a, int cta) {
  using L = DqSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::misc + 4);
  volatile int32_t* kidx = reinterpret_cast<volatile int32_t*>(sm + L::kidx);
  volatile int32_t* kmin = reinterpret_cast<volatile int32_t*>(sm + L::kmin);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (MODE == kTreeM && !tree_header_ok(a)) return;
  const int h = cta % a.hq;
  const int nT = (int)((a.nq + 127) / 128);
  const int T = MODE == kTreeM ? a.order_dq[cta / a.hq] : nT - 1 - cta / a.hq;
  const int g = h / (a.hq / a.hkv);
  const int64_t q0 = (int64_t)T * 128, q1 = min(q0 + 128, a.nq);
  // packed chunk (a.send set): several sibling subtrees after the path, key k
  // visible to path position p iff k <= p < send[k]
  const bool packed = MODE == kChunkM && a.send != nullptr;

  if (threadIdx.x == 0) {
    mbar_init(&bar[DQ_DO], 1);
    mbar_init(&bar[DQ_QA], 256);
    for (int i = 0; i < kDqKSt; ++i) {
      mbar_init(&bar[DQ_KF + i], 1);
      mbar_init(&bar[DQ_KE + i], 1);
    }
    for (int i = 0; i < kDqVSt; ++i) {
      mbar_init(&bar[DQ_VF + i], 1);
    }
    mbar_init(&bar[DQ_SFS], 1);
    mbar_init(&bar[DQ_SFP], 1);
    mbar_init(&bar[DQ_SFP + 1], 1);
    mbar_init(&bar[DQ_SES], 256);
    mbar_init(&bar[DQ_SEP], 256);
    mbar_init(&bar[DQ_DSR], 256);
    mbar_init(&bar[DQ_FINAL], 2);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    // TMA producer: the whole warp finds the next key block (32 candidates
    // per coalesced load of the per-block maxima, a ballot picks the first),
    // lane 0 waits for free stages and issues the copies. (A one-thread scan
    // walked up to a few hundred blocks between the root's and the leaf's
    // blocks with one dependent load each, and the MMAs ran dry meanwhile.)
    if (lane == 0) {
      mbar_expect_tx(&bar[DQ_DO], 128 * D * 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_2d(sm + L::dO + c * kChunk, &tmdO, &bar[DQ_DO], h * D + c * 64, (int)q0);
    }
    auto next_block = [&](int b) -> int {
      if constexpr (MODE != kTreeM) {
        if (!packed) return next_chunk_block(a, q1, b);
        // a block holding a path key, or whose maximum send exceeds the tile's
        // first query
        const int nbk = (int)((min(a.nk, a.q_off + q1) + 127) / 128);
        const int64_t qa0 = a.q_off + q0;
        for (int base = b + 1; base < nbk; base += 32) {
          const int x = base + lane;
          const int64_t kx = (int64_t)x * 128;
          const bool keep = x < nbk && (kx < a.q_off || a.blk_max[x] > qa0);
          const uint32_t m = __ballot_sync(0xffffffffu, keep);
          if (m) return base + __ffs(m) - 1;
        }
        return -1;
      } else {
        for (int base = b + 1; base <= T; base += 32) {
          const int x = base + lane;
          const uint32_t m = __ballot_sync(0xffffffffu, x <= T && a.blk_max[x] > q0);
          if (m) return base + __ffs(m) - 1;
        }
        return -1;
      }
    };
    // The block of each K stage is published with it (kidx), so the MMA and
    // softmax roles never scan the per-block maxima; after the last block a
    // stage carrying -1 (and no data) ends their loops.
    int i = 0, nk = 0, nv = 0;  // blocks started; K and V loads issued (lane 0)
    bool ok = true;
    for (int b = next_block(-1); b >= 0; b = next_block(b), ++i) {
      if (lane == 0) {
        const int ks = i % kDqKSt, vs = i % kDqVSt;
        ok = i < kDqKSt || mbar_wait(&bar[DQ_KE + ks], ((i - kDqKSt) / kDqKSt) & 1, abort_flag, 20);
        if (ok) {
          ++nk;
          kidx[ks] = b;
          if (MODE == kTreeM) kmin[ks] = a.blk_min[b];
          mbar_expect_tx(&bar[DQ_KF + ks], 128 * D * 2);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_2d(sm + L::k0 + ks * L::kTile + c * kChunk, &tmK, &bar[DQ_KF + ks], g * D + c * 64, b * 128);
          ok = i < kDqVSt || mbar_wait(&bar[DQ_SFP + vs], ((i - kDqVSt) >> 1) & 1, abort_flag, 21);
        }
        if (ok) {
          ++nv;
          mbar_expect_tx(&bar[DQ_VF + vs], 128 * D * 2);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_2d(sm + L::v0 + vs * L::kTile + c * kChunk, &tmV, &bar[DQ_VF + vs], g * D + c * 64, b * 128);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
    }
    if (lane == 0) {
      // every copy issued has landed before the CTA may leave (waited for
      // before the end marker below, which completes one more phase of a K
      // stage's barrier and would make the parity of that stage's last load
      // name the next, never completing, phase)
      mbar_drain(&bar[DQ_DO], 0, abort_flag);
      for (int j = nk - 1; j >= 0 && j >= nk - kDqKSt; --j)
        mbar_drain(&bar[DQ_KF + j % kDqKSt], (j / kDqKSt) & 1, abort_flag);
      for (int j = nv - 1; j >= 0 && j >= nv - kDqVSt; --j)
        mbar_drain(&bar[DQ_VF + j % kDqVSt], (j / kDqVSt) & 1, abort_flag);
      if (ok) {
        const int ks = i % kDqKSt;
        if (i < kDqKSt || mbar_wait(&bar[DQ_KE + ks], ((i - kDqKSt) / kDqKSt) & 1, abort_flag, 19)) {
          kidx[ks] = -1;
          mbar_arrive(&bar[DQ_KF + ks]);
        }
      }
    }
  } else if (warp == 1) {
    // S(i) and dP(i) of every block
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, 128, 0, 0);
      const uint64_t dob = smem_desc(smem_u32(sm + L::dO), 16, 1024);
      bool ok = mbar_wait(&bar[DQ_DO], 0, abort_flag, 22) && mbar_wait(&bar[DQ_QA], 0, abort_flag, 17);
      for (int i = 0; ok; ++i) {
        const int ks = i % kDqKSt, vs = i % kDqVSt;
        if (!mbar_wait(&bar[DQ_KF + ks], (i / kDqKSt) & 1, abort_flag, 24)) break;
        if (kidx[ks] < 0) break;
        // S of block i − 1 loaded by every softmax thread
        if (i >= 1 && !mbar_wait(&bar[DQ_SES], (i - 1) & 1, abort_flag, 26)) break;
        tc_fence_after();
        const uint64_t dk = smem_desc(smem_u32(sm + L::k0 + ks * L::kTile), 16, 1024);
        const uint64_t dv = smem_desc(smem_u32(sm + L::v0 + vs * L::kTile), 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kChunk + (k & 3) * 32;
          umma_ts(tbase + kDqS, tbase + kDqQA + k * 8, desc_at(dk, off), idS, k > 0);
        }
        umma_commit(&bar[DQ_SFS]);  // S ready
        if (!mbar_wait(&bar[DQ_VF + vs], (i / kDqVSt) & 1, abort_flag, 25)) break;
        // dP of block i − 1 loaded by every softmax thread
        if (i >= 1 && !mbar_wait(&bar[DQ_SEP], (i - 1) & 1, abort_flag, 18)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kChunk + (k & 3) * 32;
          umma_ss(tbase + kDqP, desc_at(dob, off), desc_at(dv, off), idS, k > 0);
        }
        umma_commit(&bar[DQ_SFP + vs]);  // dP ready, V stage vs free
      }
      umma_commit(&bar[DQ_FINAL]);  // completes once both MMA threads' MMAs are done
      mbar_drain(&bar[DQ_FINAL], 0, abort_flag);
    }
  } else if (warp == kDqMmaWarp2) {
    // dQ += dS(i)·K(i) of every block, once dS(i) is written
    if (lane == 0) {
      constexpr uint32_t idQ = idesc_bf16(128, D, 0, 1);
      for (int i = 0;; ++i) {
        const int ks = i % kDqKSt;
        if (!mbar_wait(&bar[DQ_KF + ks], (i / kDqKSt) & 1, abort_flag, 16)) break;
        if (kidx[ks] < 0) break;
        if (!mbar_wait(&bar[DQ_DSR], i & 1, abort_flag, 23)) break;
        tc_fence_after();
        const uint64_t dk = smem_desc(smem_u32(sm + L::k0 + ks * L::kTile), kChunk, 1024);
#pragma unroll
        for (int k = 0; k < 128 / 16; ++k)
          umma_ts(tbase + kDqQ, tbase + kDqDS + k * 8, desc_at(dk, k * 2048), idQ, (i > 0 || k > 0));
        umma_commit(&bar[DQ_KE + ks]);  // frees K stage ks and the dS buffer
      }
      umma_commit(&bar[DQ_FINAL]);
      mbar_drain(&bar[DQ_FINAL], 0, abort_flag);
    }
  } else {
    static_assert(kDqMmaWarp2 == 10, "softmax warps are 2..9");
    const int wq = warp & 3;
    const int half = (warp - 2) >> 2;  // keys [64·half, 64·half + 64) of each block
    const int r = wq * 32 + lane;
    const int64_t q = q0 + r;
    const uint32_t lb = (uint32_t)(wq * 32) << 16;
    // This thread's half of its Q row into TMEM (bf16 pairs, zero past the
    // last row): the A operand of S = Q·Kᵀ.
    {
      constexpr int kW = D / 4;  // 32-bit words of half a row
      uint32_t w[kW];
      if (q < a.nq) {
        const uint4* src = reinterpret_cast<const uint4*>(a.qp + (q * a.hq + h) * (int64_t)D + (D / 2) * half);
#pragma unroll
        for (int v = 0; v < kW / 4; ++v) {
          const uint4 x = src[v];
          w[4 * v] = x.x; w[4 * v + 1] = x.y; w[4 * v + 2] = x.z; w[4 * v + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int v = 0; v < kW; ++v) w[v] = 0u;
      }
      if constexpr (kW == 32) tmem_st32(tbase + lb + kDqQA + kW * half, w);
      else tmem_st16(tbase + lb + kDqQA + kW * half, w);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[DQ_QA]);
    }
    const float lse2 = a.lse2[(int64_t)h * a.ldp + q];
    const float dsum = a.dsum[(int64_t)h * a.ldp + q];
    const float2 c2 = make_float2(a.scale_log2, a.scale_log2), nl2 = make_float2(-lse2, -lse2);
    const float2 nd2 = make_float2(-dsum, -dsum);
    int i = 0;
    bool ok = true;
    for (;; ++i) {
      const int ks = i % kDqKSt;
      // the block arrives with its K
      if (!mbar_wait(&bar[DQ_KF + ks], (i / kDqKSt) & 1, abort_flag, 27)) { ok = false; break; }
      const int b = kidx[ks];
      if (b < 0) break;
      const int64_t kb = (int64_t)b * 128;
      bool full;
      if (MODE == kTreeM) {
        full = kb + 127 <= q0 && kb + 128 <= a.nk && kmin[ks] >= q1;
      } else if (packed) {
        full = kb + 128 <= a.q_off;  // path keys only
      } else {
        full = kb + 127 <= a.q_off + q0 && kb + 128 <= a.nk;
      }
      if (!mbar_wait(&bar[DQ_SFS], i & 1, abort_flag, 28)) { ok = false; break; }
      tc_fence_after();
      // Visibility of key column col (partial blocks only): tree mode and
      // packed chunks need col <= qk and qi < send (path positions; q_off = 0
      // in tree mode); chunk mode col <= cmax.
      const int qk = (int)(a.q_off + q - kb);
      int cmax = 127;
      if (MODE != kTreeM) {
        const int64_t lim = a.q_off + q - kb, lim2 = a.nk - 1 - kb;
        cmax = q < a.nq ? (int)(lim < lim2 ? lim : lim2) : -1;
      }
      const int32_t qi = (int32_t)(a.q_off + q);
      const uint32_t col0 = 64 * half;
      // P = exp2(S·c − lse2) of this thread's 64 columns, read while dP is formed
      float2 p[32];
      {
        uint32_t s0[32], s1[32];
        tmem_ld32(tbase + lb + kDqS + col0, s0);
        tmem_ld32(tbase + lb + kDqS + col0 + 32, s1);
        tmem_ld_wait();
        tmem_pin(s0);
        tmem_pin(s1);
        tc_fence_before();
        mbar_arrive(&bar[DQ_SES]);  // S may be overwritten
        // send of the block's keys (zero-padded past N), partial blocks only
        const int32_t* bsend = a.send + kb + col0;
        // Packed chunks, warp-uniform case: when this half of the block
        // precedes the warp's 32 rows and no key's send falls inside them,
        // every row of the warp sees the same keys, those whose send passes the
        // warp's last row. Lane l tests keys 2l and 2l+1 of the half; column
        // 2j+e is bit j of vb[e]. (On whole trees the test cost as much as it
        // saved.)
        bool uni = false;
        uint32_t vb0 = 0u, vb1 = 0u;
        if (MODE == kChunkM && packed && !full) {
          const int qf = (int)(a.q_off + q0) + wq * 32, ql = qf + 31;
          const int2 se = *reinterpret_cast<const int2*>(bsend + 2 * lane);
          const bool mixed = (se.x > qf && se.x <= ql) || (se.y > qf && se.y <= ql);
          vb0 = __ballot_sync(0xffffffffu, se.x > ql);
          vb1 = __ballot_sync(0xffffffffu, se.y > ql);
          uni = kb + col0 + 63 <= qf && !__any_sync(0xffffffffu, mixed);
        }
        // The mask kind is uniform over the warp: one branch per block, none per element.
        constexpr int kFullP = 0, kUniP = 1, kElemP = 2;
        auto probs = [&](auto mode_tag) {
          constexpr int kMode = decltype(mode_tag)::value;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const uint32_t x0 = j < 16 ? s0[2 * j] : s1[2 * j - 32];
            const uint32_t x1 = j < 16 ? s0[2 * j + 1] : s1[2 * j - 31];
            const float2 xx = __ffma2_rn(make_float2(__uint_as_float(x0), __uint_as_float(x1)), c2, nl2);
            float2 pv = make_float2(fast_exp2(xx.x), fast_exp2(xx.y));
            if constexpr (kMode == kUniP) {
              pv.x = (vb0 >> j) & 1u ? pv.x : 0.f;
              pv.y = (vb1 >> j) & 1u ? pv.y : 0.f;
            } else if constexpr (kMode == kElemP) {
              const int col = (int)col0 + 2 * j;
              bool v0, v1;
              if (MODE == kTreeM || packed) {
                const int2 se = *reinterpret_cast<const int2*>(bsend + 2 * j);
                v0 = col <= qk && qi < se.x;
                v1 = col + 1 <= qk && qi < se.y;
              } else {
                v0 = col <= cmax;
                v1 = col + 1 <= cmax;
              }
              pv.x = v0 ? pv.x : 0.f;
              pv.y = v1 ? pv.y : 0.f;
            }
            p[j] = pv;
          }
        };
        if (full) probs(std::integral_constant<int, kFullP>{});
        else if (MODE == kChunkM && uni) probs(std::integral_constant<int, kUniP>{});
        else probs(std::integral_constant<int, kElemP>{});
      }
      // dS = P ⊙ (dP − dsum), packed to bf16
      uint32_t pk[32];
      if (!mbar_wait(&bar[DQ_SFP + (i & 1)], (i >> 1) & 1, abort_flag, 32)) { ok = false; break; }
      tc_fence_after();
      {
        uint32_t d0[32], d1[32];
        tmem_ld32(tbase + lb + kDqP + col0, d0);
        tmem_ld32(tbase + lb + kDqP + col0 + 32, d1);
        tmem_ld_wait();
        tmem_pin(d0);
        tmem_pin(d1);
        tc_fence_before();
        mbar_arrive(&bar[DQ_SEP]);  // dP may be overwritten
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const uint32_t y0 = j < 16 ? d0[2 * j] : d1[2 * j - 32];
          const uint32_t y1 = j < 16 ? d0[2 * j + 1] : d1[2 * j - 31];
          const float2 ds = __fmul2_rn(p[j], __fadd2_rn(make_float2(__uint_as_float(y0), __uint_as_float(y1)), nd2));
          pk[j] = pack_bf16(ds.x, ds.y);
        }
      }
      // the dS buffer was last read by the dQ MMAs of block i − 1
      if (i >= 1 && !mbar_wait(&bar[DQ_KE + (i - 1) % kDqKSt], ((i - 1) / kDqKSt) & 1, abort_flag, 30)) {
        ok = false;
        break;
      }
      tmem_st32(tbase + lb + kDqDS + 32 * half, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[DQ_DSR]);
    }
    const int n = i;
    // dQ columns [64·half, 64·half + 64) of this thread's row (the loads are
    // warp-collective and run on every lane; only the stores are guarded)
    if (ok && n > 0 && mbar_wait(&bar[DQ_FINAL], 0, abort_flag, 31)) {
      tc_fence_after();
      __nv_bfloat16* row = a.dq + q * (int64_t)a.hq * D + (int64_t)h * D;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int cc = (D / 64) * half + c;  // 32-column chunk of dQ
        uint32_t o[32];
        tmem_ld32(tbase + lb + kDqQ + cc * 32, o);
        tmem_ld_wait();
        tmem_pin(o);
        if (q < a.nq) {
          uint4* dst = reinterpret_cast<uint4*>(row + cc * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * a.scale, __uint_as_float(o[8 * v + 1]) * a.scale);
            w.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * a.scale, __uint_as_float(o[8 * v + 3]) * a.scale);
            w.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * a.scale, __uint_as_float(o[8 * v + 5]) * a.scale);
            w.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * a.scale, __uint_as_float(o[8 * v + 7]) * a.scale);
            dst[v] = w;
          }
        }
      }
    } else if (n == 0 && q < a.nq) {
      uint4* dst = reinterpret_cast<uint4*>(a.dq + q * (int64_t)a.hq * D + (int64_t)h * D + (D / 2) * half);
      for (int v = 0; v < D / 16; ++v) dst[v] = make_uint4(0, 0, 0, 0);
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

// ---------------------------------------------------------------- dK/dV CTA
// Query tiles of 64 rows so that Sᵀ/dPᵀ are double buffered in TMEM next to the
// dV and dK accumulators: Sᵀ/dPᵀ of tile t+1 are formed while the softmax
// warps turn tile t into Pᵀ / dSᵀ. As in the dQ CTA, two threads issue the
// MMAs (Sᵀ/dPᵀ, and dV/dK), so that one thread's waits do not leave the
// tensor pipe idle; Sᵀ/dPᵀ of tile t + 2 wait until dV/dK of tile t (the
// other thread's MMAs) have read Pᵀ / dSᵀ from the same TMEM buffer.
// mbarrier slots: KV (K, V loaded), QF[s] / QE[s] (query-tile stage s loaded /
// free), SDS[b] / SDP[b] (Sᵀ_b / dPᵀ_b formed: separate, so that the softmax
// turns Sᵀ into P while dPᵀ is still being formed), PDS[b] (Pᵀ_b / dSᵀ_b
// written), FINAL (both MMA threads' MMAs done).
constexpr int KV_KV = 0, KV_QF = 1, KV_QE = KV_QF + kStages, KV_SDS = KV_QE + kStages, KV_SDP = KV_SDS + 2,
              KV_PDS = KV_SDP + 2, KV_FINAL = KV_PDS + 2, KV_NBAR = KV_FINAL + 1;
constexpr uint32_t kKvS = 0, kKvP = 128, kKvV = 256, kKvK = 384;  // Sᵀ_b at 64b, dPᵀ_b at 128+64b

template <int D>
struct KvSmem {
  static constexpr uint32_t kTileK = (D / 64) * kChunk;    // 128 rows
  static constexpr uint32_t kTileQ = (D / 64) * kChunk64;  // 64 rows
  static constexpr uint32_t k = 0;
  static constexpr uint32_t v = k + kTileK;
  static constexpr uint32_t q0 = v + kTileK;
  static constexpr uint32_t o0 = q0 + kStages * kTileQ;
  static constexpr uint32_t lse = o0 + kStages * kTileQ;  // [kStages][64] f32
  static constexpr uint32_t ds = lse + kStages * 64 * 4;   // [kStages][64] f32
  static constexpr uint32_t bars = ds + kStages * 64 * 4;
  static constexpr uint32_t misc = bars + KV_NBAR * 8;
  static constexpr uint32_t total = misc + 16 + 1024;
};

template <int D, int MODE>
__device__ __forceinline__ void dkdv_cta(const CUtensorMap& tmQ, const CUtensorMap& tmdO, const CUtensorMap& tmK,
                                         const CUtensorMap& tmV, const BwdTc& a, int cta) {
  using L = KvSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::misc + 4);
  const float* sL = reinterpret_cast<const float*>(sm + L::lse);
  const float* sD = reinterpret_cast<const float*>(sm + L::ds);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (MODE == kTreeM && !tree_header_ok(a)) return;
  const int g = cta % a.hkv;
  const int bi = cta / a.hkv;
  const int B = MODE == kTreeM ? a.order_kv[bi] : bi;
  const int G = a.hq / a.hkv;
  const int64_t kb0 = (int64_t)B * 128;
  // packed chunk (a.send set): key k visible to path position p iff k <= p < send[k]
  const bool packed = MODE == kChunkM && a.send != nullptr;
  // 64-row query tiles that see this key block
  int t0, t1;
  if (MODE == kTreeM) {
    t0 = 2 * B;
    t1 = (a.blk_max[B] + 63) / 64;
  } else {
    const int64_t qs = kb0 > a.q_off ? kb0 - a.q_off : 0;
    int64_t qe = a.nq;
    if (packed && kb0 >= a.q_off) {
      // chunk keys only: the block's maximum send ends the rows that see it
      const int64_t e = (int64_t)a.blk_max[B] - a.q_off;
      qe = e < qe ? (e > 0 ? e : 0) : qe;
    }
    t0 = (int)(qs / 64);
    t1 = (int)((qe + 63) / 64);
  }
  const int ntile = t1 > t0 ? t1 - t0 : 0;
  const int niter = ntile * G;

  if (threadIdx.x == 0) {
    mbar_init(&bar[KV_KV], 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar[KV_QF + i], 1);
      mbar_init(&bar[KV_QE + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[KV_SDS + i], 1);
      mbar_init(&bar[KV_SDP + i], 1);
      mbar_init(&bar[KV_PDS + i], 128);
    }
    mbar_init(&bar[KV_FINAL], 2);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    if (lane == 0 && niter > 0) {
      mbar_expect_tx(&bar[KV_KV], 2 * 128 * D * 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_2d(sm + L::k + c * kChunk, &tmK, &bar[KV_KV], g * D + c * 64, (int)kb0);
        tma_load_2d(sm + L::v + c * kChunk, &tmV, &bar[KV_KV], g * D + c * 64, (int)kb0);
      }
      int nq = 0;  // query-tile loads issued
      for (int it = 0; it < niter; ++it, ++nq) {
        const int st = it % kStages;
        if (it >= kStages && !mbar_wait(&bar[KV_QE + st], ((it - kStages) / kStages) & 1, abort_flag, 30)) break;
        const int h = g * G + it / ntile;
        const int64_t q0 = (int64_t)(t0 + it % ntile) * 64;
        mbar_expect_tx(&bar[KV_QF + st], 2 * 64 * D * 2 + 512);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_2d(sm + L::q0 + st * L::kTileQ + c * kChunk64, &tmQ, &bar[KV_QF + st], h * D + c * 64, (int)q0);
          tma_load_2d(sm + L::o0 + st * L::kTileQ + c * kChunk64, &tmdO, &bar[KV_QF + st], h * D + c * 64, (int)q0);
        }
        bulk_load(sm + L::lse + st * 256, a.lse2 + (int64_t)h * a.ldp + q0, 256, &bar[KV_QF + st]);
        bulk_load(sm + L::ds + st * 256, a.dsum + (int64_t)h * a.ldp + q0, 256, &bar[KV_QF + st]);
      }
      // every copy issued has landed before the CTA may leave
      mbar_drain(&bar[KV_KV], 0, abort_flag);
      for (int j = nq - 1; j >= 0 && j >= nq - kStages; --j) mbar_drain(&bar[KV_QF + j % kStages], (j / kStages) & 1, abort_flag);
    }
  } else if (warp == 1) {
    // Sᵀ(it) and dPᵀ(it) of every query tile
    if (lane == 0 && niter > 0) {
      constexpr uint32_t idS = idesc_bf16(128, 64, 0, 0);
      const uint64_t dks = smem_desc(smem_u32(sm + L::k), 16, 1024), dvs = smem_desc(smem_u32(sm + L::v), 16, 1024);
      bool ok = mbar_wait(&bar[KV_KV], 0, abort_flag, 32);
      for (int it = 0; ok && it < niter; ++it) {
        const int bb = it & 1, st = it % kStages;
        if (!mbar_wait(&bar[KV_QF + st], (it / kStages) & 1, abort_flag, 33)) break;
        // Sᵀ_b / dPᵀ_b hold Pᵀ / dSᵀ of tile it − 2 until its dV/dK MMAs
        // (issued by the other MMA thread) have read them
        if (it >= 2 && !mbar_wait(&bar[KV_QE + (it - 2) % kStages], ((it - 2) / kStages) & 1, abort_flag, 34)) break;
        tc_fence_after();
        const uint64_t dq = smem_desc(smem_u32(sm + L::q0 + st * L::kTileQ), 16, 1024);
        const uint64_t dob = smem_desc(smem_u32(sm + L::o0 + st * L::kTileQ), 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t offk = (k >> 2) * kChunk + (k & 3) * 32, offq = (k >> 2) * kChunk64 + (k & 3) * 32;
          umma_ss(tbase + kKvS + 64 * bb, desc_at(dks, offk), desc_at(dq, offq), idS, k > 0);
        }
        umma_commit(&bar[KV_SDS + bb]);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t offk = (k >> 2) * kChunk + (k & 3) * 32, offq = (k >> 2) * kChunk64 + (k & 3) * 32;
          umma_ss(tbase + kKvP + 64 * bb, desc_at(dvs, offk), desc_at(dob, offq), idS, k > 0);
        }
        umma_commit(&bar[KV_SDP + bb]);
      }
    }
    if (lane == 0) {
      umma_commit(&bar[KV_FINAL]);  // completes once both MMA threads' MMAs are done
      mbar_drain(&bar[KV_FINAL], 0, abort_flag);
    }
  } else if (warp == kKvMmaWarp2) {
    // dV += Pᵀ(it)·dO(it) and dK += dSᵀ(it)·Q(it) of every query tile, once
    // the softmax has written Pᵀ / dSᵀ
    if (lane == 0 && niter > 0) {
      constexpr uint32_t idG = idesc_bf16(128, D, 0, 1);
      for (int it = 0; it < niter; ++it) {
        const int bb = it & 1, st = it % kStages;
        if (!mbar_wait(&bar[KV_PDS + bb], (it >> 1) & 1, abort_flag, 31)) break;
        tc_fence_after();
        const uint64_t dqg = smem_desc(smem_u32(sm + L::q0 + st * L::kTileQ), kChunk64, 1024);
        const uint64_t dog = smem_desc(smem_u32(sm + L::o0 + st * L::kTileQ), kChunk64, 1024);
#pragma unroll
        for (int k = 0; k < 64 / 16; ++k)
          umma_ts(tbase + kKvV, tbase + kKvS + 64 * bb + k * 8, desc_at(dog, k * 2048), idG, (it > 0 || k > 0));
#pragma unroll
        for (int k = 0; k < 64 / 16; ++k)
          umma_ts(tbase + kKvK, tbase + kKvP + 64 * bb + k * 8, desc_at(dqg, k * 2048), idG, (it > 0 || k > 0));
        umma_commit(&bar[KV_QE + st]);  // frees the Q/dO stage and Sᵀ_b / dPᵀ_b
      }
    }
    if (lane == 0) {
      umma_commit(&bar[KV_FINAL]);
      mbar_drain(&bar[KV_FINAL], 0, abort_flag);
    }
  } else if (warp < kKvWarps) {
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int64_t k = kb0 + r;
    const uint32_t lb = (uint32_t)(wq * 32) << 16;
    // tree: zero-padded past N; packed: read for blocks holding a chunk key (path keys hold >= s0 + C)
    const int32_t ksend = MODE == kTreeM || (packed && kb0 + 128 > a.q_off) ? a.send[k] : INT32_MAX;
    const float2 c2 = make_float2(a.scale_log2, a.scale_log2);
    bool ok = true;
    for (int it = 0; it < niter; ++it) {
      const int bb = it & 1, st = it % kStages;
      const int64_t q0 = (int64_t)(t0 + it % ntile) * 64;
      if (!mbar_wait(&bar[KV_QF + st], (it / kStages) & 1, abort_flag, 35) ||
          !mbar_wait(&bar[KV_SDS + bb], (it >> 1) & 1, abort_flag, 36)) {
        ok = false;
        break;
      }
      tc_fence_after();
      bool full;
      if (MODE == kTreeM) full = q0 >= kb0 + 127 && q0 + 64 <= a.nq && kb0 + 128 <= a.nk && q0 + 64 <= a.blk_min[B];
      else if (packed) full = kb0 + 128 <= a.q_off && q0 + 64 <= a.nq;  // path keys only
      else full = a.q_off + q0 >= kb0 + 127 && q0 + 64 <= a.nq && kb0 + 128 <= a.nk;
      const float* cL = sL + st * 64;
      const float* cD = sD + st * 64;
      // Partial tiles: query column col is visible iff lo <= col < hi.
      int lo = 0, hi = 64;
      if (MODE == kTreeM) {
        const int64_t e = (int64_t)ksend < a.nq ? (int64_t)ksend : a.nq;  // ksend = 0 past N
        lo = (int)(k - q0 > 0 ? (k - q0 < 64 ? k - q0 : 64) : 0);
        hi = (int)(e - q0 > 0 ? (e - q0 < 64 ? e - q0 : 64) : 0);
      } else {
        int64_t e = a.nq;  // packed: rows past the key's segment do not see it
        if (packed && (int64_t)ksend - a.q_off < e) e = (int64_t)ksend - a.q_off;
        const int64_t l = k - a.q_off - q0, h2 = e - q0;
        lo = (int)(l > 0 ? (l < 64 ? l : 64) : 0);
        hi = k < a.nk ? (int)(h2 > 0 ? (h2 < 64 ? h2 : 64) : 0) : 0;
      }
      // P = exp2(Sᵀ·c − lse2) of the thread's 64 query columns, written to
      // TMEM as bf16 (over Sᵀ_b columns [0, 32), already read) and kept in
      // fp32 for dS; `full` is uniform over the CTA: one branch per tile, none
      // per element.
      float2 p[32];
      auto probs = [&](auto full_tag) {
        constexpr bool kFull = decltype(full_tag)::value;
        uint32_t s0[32], s1[32];
        tmem_ld32(tbase + lb + kKvS + 64 * bb, s0);
        tmem_ld32(tbase + lb + kKvS + 64 * bb + 32, s1);
        tmem_ld_wait();
        tmem_pin(s0);
        tmem_pin(s1);
        uint32_t pk[32];
        float4 l4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int col = 2 * j;
          // the tile's lse2 (the same for every thread: broadcast loads, 16 bytes at a time)
          if ((j & 1) == 0) l4 = *reinterpret_cast<const float4*>(cL + col);
          const float2 l2 = (j & 1) ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y);
          const uint32_t x0 = j < 16 ? s0[2 * j] : s1[2 * j - 32];
          const uint32_t x1 = j < 16 ? s0[2 * j + 1] : s1[2 * j - 31];
          const float2 xx = __ffma2_rn(make_float2(__uint_as_float(x0), __uint_as_float(x1)), c2,
                                       make_float2(-l2.x, -l2.y));
          float2 pv = make_float2(fast_exp2(xx.x), fast_exp2(xx.y));
          if constexpr (!kFull) {
            pv.x = (col >= lo && col < hi) ? pv.x : 0.f;
            pv.y = (col + 1 >= lo && col + 1 < hi) ? pv.y : 0.f;
          }
          p[j] = pv;
          pk[j] = pack_bf16(pv.x, pv.y);
        }
        tmem_st32(tbase + lb + kKvS + 64 * bb, pk);
      };
      if (full) probs(std::true_type{});
      else probs(std::false_type{});
      // dS = P ⊙ (dPᵀ − dsum), 32 columns at a time; dSᵀ (bf16) of chunk c
      // goes over dPᵀ_b columns [16c, 16c + 16), which chunk 0 has read
      if (!mbar_wait(&bar[KV_SDP + bb], (it >> 1) & 1, abort_flag, 40)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t dp[32];
        tmem_ld32(tbase + lb + kKvP + 64 * bb + c * 32, dp);
        tmem_ld_wait();
        tmem_pin(dp);
        uint32_t dk[16];
        float4 d4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int col = c * 32 + 2 * j;
          if ((j & 1) == 0) d4 = *reinterpret_cast<const float4*>(cD + col);
          const float2 d2 = (j & 1) ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y);
          const float2 ds = __fmul2_rn(
              p[c * 16 + j],
              __fadd2_rn(make_float2(__uint_as_float(dp[2 * j]), __uint_as_float(dp[2 * j + 1])),
                         make_float2(-d2.x, -d2.y)));
          dk[j] = pack_bf16(ds.x, ds.y);
        }
        tmem_st16(tbase + lb + kKvP + 64 * bb + 16 * c, dk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[KV_PDS + bb]);
    }
    const bool have = ok && niter > 0 && mbar_wait(&bar[KV_FINAL], 0, abort_flag, 38);
    if (have) tc_fence_after();
    {
      // The TMEM loads are warp-collective: every lane runs them, only the
      // stores are limited to existing key rows.
      const int64_t base = k * (int64_t)a.hkv * D + (int64_t)g * D;
      const bool row_ok = k < a.nk;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t vv[32], kk[32];
        if (have) {
          tmem_ld32(tbase + lb + kKvV + c * 32, vv);
          tmem_ld32(tbase + lb + kKvK + c * 32, kk);
          tmem_ld_wait();
          tmem_pin(vv);
          tmem_pin(kk);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) vv[j] = kk[j] = 0u;
        }
        if (MODE == kTreeM) {
          if (!row_ok) continue;
          uint4* dvp = reinterpret_cast<uint4*>(a.dv + base + c * 32);
          uint4* dkp = reinterpret_cast<uint4*>(a.dk + base + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 wv, wk;
            wv.x = pack_bf16(__uint_as_float(vv[8 * v + 0]), __uint_as_float(vv[8 * v + 1]));
            wv.y = pack_bf16(__uint_as_float(vv[8 * v + 2]), __uint_as_float(vv[8 * v + 3]));
            wv.z = pack_bf16(__uint_as_float(vv[8 * v + 4]), __uint_as_float(vv[8 * v + 5]));
            wv.w = pack_bf16(__uint_as_float(vv[8 * v + 6]), __uint_as_float(vv[8 * v + 7]));
            wk.x = pack_bf16(__uint_as_float(kk[8 * v + 0]) * a.scale, __uint_as_float(kk[8 * v + 1]) * a.scale);
            wk.y = pack_bf16(__uint_as_float(kk[8 * v + 2]) * a.scale, __uint_as_float(kk[8 * v + 3]) * a.scale);
            wk.z = pack_bf16(__uint_as_float(kk[8 * v + 4]) * a.scale, __uint_as_float(kk[8 * v + 5]) * a.scale);
            wk.w = pack_bf16(__uint_as_float(kk[8 * v + 6]) * a.scale, __uint_as_float(kk[8 * v + 7]) * a.scale);
            dvp[v] = wv;
            dkp[v] = wk;
          }
        } else if (have) {
          // fp32 path accumulators: fire-and-forget vector adds in L2 (this
          // CTA is the only writer of these rows in the launch, so the sums
          // are the same as a load-add-store, without the load latency). The
          // warp's 32 rows of this 32-column slice go through shared memory
          // (the query-tile ring, idle once every MMA is done; 16-byte chunks
          // XOR-swizzled by row, so neither side has bank conflicts), and
          // eight lanes then add one row's 128 contiguous bytes: an
          // instruction covers four whole lines instead of 32 scattered
          // 16-byte pieces. (A CTA that gave up adds nothing: its sums would
          // be zero.)
          float4* stg = reinterpret_cast<float4*>(sm + L::q0 + wq * 8192);  // [dV, dK][32 rows][8 chunks]
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            const int p = lane * 8 + (x ^ (lane & 7));
            stg[p] = make_float4(__uint_as_float(vv[4 * x + 0]), __uint_as_float(vv[4 * x + 1]),
                                 __uint_as_float(vv[4 * x + 2]), __uint_as_float(vv[4 * x + 3]));
            stg[256 + p] = make_float4(__uint_as_float(kk[4 * x + 0]) * a.scale, __uint_as_float(kk[4 * x + 1]) * a.scale,
                                       __uint_as_float(kk[4 * x + 2]) * a.scale, __uint_as_float(kk[4 * x + 3]) * a.scale);
          }
          __syncwarp();
          const int x = lane & 7;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int row = j * 4 + (lane >> 3);
            const int64_t kr = kb0 + wq * 32 + row;
            if (kr < a.nk) {
              const int p = row * 8 + (x ^ (row & 7));
              const float4 v4 = stg[p], k4 = stg[256 + p];
              const int64_t off = kr * (int64_t)a.hkv * D + (int64_t)g * D + c * 32 + x * 4;
              red_add_v4(a.dv_acc + off, v4.x, v4.y, v4.z, v4.w);
              red_add_v4(a.dk_acc + off, k4.x, k4.y, k4.z, k4.w);
            }
          }
          __syncwarp();  // the next slice overwrites the staging rows
        }
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

// One launch for both kinds of CTA, each kind in its own longest-first
// order: the kind whose longest CTA takes longer comes first (blocks
// [0, n_first)), so that the other kind's shorter CTAs fill the tail.
// Launched with kDqWarps warps and the larger of the two shared-memory layouts.
template <int D>
constexpr uint32_t bwd_smem_bytes() {
  return DqSmem<D>::total > KvSmem<D>::total ? DqSmem<D>::total : KvSmem<D>::total;
}
static_assert(bwd_smem_bytes<128>() <= 232448, "backward shared memory exceeds the per-CTA limit");
static_assert(kKvMmaWarp2 < kDqWarps && kKvWarps <= kKvMmaWarp2, "the dK/dV CTA runs on the first warps of the launch");

template <int D, int MODE>
__global__ void __launch_bounds__(kDqWarps * 32, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmQ64, const __grid_constant__ CUtensorMap tmdO64,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const BwdTc a,
                  int n_first, int dq_first) {
  const int b = (int)blockIdx.x;
  const bool first = b < n_first;
  const int idx = first ? b : b - n_first;
  if (first != (dq_first != 0)) dkdv_cta<D, MODE>(tmQ64, tmdO64, tmK, tmV, a, idx);
  else dq_cta<D, MODE>(tmdO, tmK, tmV, a, idx);
}

// lse2 = LSE·log2(e), dsum = Σ_d dO·O, both [hq][ldp]; padding rows: lse2 = +inf, dsum = 0.
// One warp per query row t: the row's hq·D values of O and of dO are
// contiguous, so lanes read them 16 bytes at a time (kPrepUnroll loads of
// each in flight per lane), and the D/8 lanes that hold one head reduce
// their partial sums with shuffles inside their group.
constexpr int kPrepUnroll = 4;
template <int D>
__global__ void prep_kernel(const __nv_bfloat16* o, const __nv_bfloat16* dO, const float* lse, int64_t lse_ld,
                            int64_t nq, int hq, int64_t ldp, float* lse2, float* dsum) {
  constexpr int kLph = D / 8;  // lanes (16-byte chunks) per head
  static_assert(32 % kLph == 0, "a head's chunks must not straddle a warp's chunk block");
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= ldp) return;
  if (t >= nq) {
    for (int h = lane; h < hq; h += 32) {
      lse2[h * ldp + t] = INFINITY;
      dsum[h * ldp + t] = 0.f;
    }
    return;
  }
  const int nchunk = hq * kLph;
  const uint4* orow = reinterpret_cast<const uint4*>(o + t * hq * D);
  const uint4* drow = reinterpret_cast<const uint4*>(dO + t * hq * D);
  for (int base = 0; base < nchunk; base += 32 * kPrepUnroll) {
    uint4 x[kPrepUnroll], y[kPrepUnroll];
#pragma unroll
    for (int u = 0; u < kPrepUnroll; ++u) {
      const int c = base + u * 32 + lane;
      x[u] = c < nchunk ? drow[c] : make_uint4(0u, 0u, 0u, 0u);
      y[u] = c < nchunk ? orow[c] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kPrepUnroll; ++u) {
      const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&x[u]);
      const __nv_bfloat162* yp = reinterpret_cast<const __nv_bfloat162*>(&y[u]);
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 xf = __bfloat1622float2(xp[e]), yf = __bfloat1622float2(yp[e]);
        acc += xf.x * yf.x + xf.y * yf.y;
      }
#pragma unroll
      for (int off = kLph / 2; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      const int c = base + u * 32 + lane;
      if (c < nchunk && lane % kLph == 0) {
        const int h = c / kLph;
        dsum[h * ldp + t] = acc;
        lse2[h * ldp + t] = lse[h * lse_ld + t] * 1.4426950408889634f;
      }
    }
  }
}

template <int D, int MODE>
int launch_bwd(BwdTc a, const void* Q, const void* K, const void* V, const void* O, const float* LSE, int64_t lse_ld,
               const void* dO, const int32_t* dq_order, const int32_t* kv_order, cudaStream_t st) {
  const unsigned pblocks = (unsigned)((a.ldp * 32 + 255) / 256);  // one warp per query row
  prep_kernel<D><<<pblocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO),
                                         LSE, lse_ld, a.nq, a.hq, a.ldp, const_cast<float*>(a.lse2),
                                         const_cast<float*>(a.dsum));
  if (cudaGetLastError() != cudaSuccess) return TT_ERR_CUDA;
  // dQ CTAs: 128-row dO, K, V boxes (Q goes to TMEM from global memory); dK/dV CTAs:
  // 128-row K/V, 64-row Q/dO boxes.
  CUtensorMap mo, mk, mv, mq64, mo64;
  const uint64_t cq = (uint64_t)a.hq * D, ck = (uint64_t)a.hkv * D;
  if (!make_tmap_bf16(&mo, dO, cq, a.nq, 128) ||
      !make_tmap_bf16(&mk, K, ck, a.nk, 128) || !make_tmap_bf16(&mv, V, ck, a.nk, 128) ||
      !make_tmap_bf16(&mq64, Q, cq, a.nq, 64) || !make_tmap_bf16(&mo64, dO, cq, a.nq, 64))
    return TT_ERR_CUDA;
  auto kern = bwd_tc_kernel<D, MODE>;
  const int smem = (int)bwd_smem_bytes<D>();
  if (!smem_attr_set<bwd_tc_kernel<D, MODE>>(smem)) return TT_ERR_CUDA;
  BwdTc b = a;
  b.order_dq = dq_order;
  b.order_kv = kv_order;
  b.qp = static_cast<const __nv_bfloat16*>(Q);
  const int n_kv = (int)((a.nk + 127) / 128) * a.hkv;
  const int n_dq = (int)((a.nq + 127) / 128) * a.hq;
  // Tree mode: the root's key blocks are seen by the whole tree, so dK/dV
  // CTAs are the longest. Chunk mode: the longest dQ CTA runs over every key
  // block of the path, the longest dK/dV CTA over G query heads × every
  // 64-row tile of the chunk (about 2100 and 1950 cycles per unit).
  int dq_first = 0;
  if (MODE == kChunkM) {
    const double dq_cost = 2100.0 * (double)((a.nk + 127) / 128);
    const double kv_cost = 1950.0 * (double)((a.nq + 63) / 64) * (double)(a.hq / a.hkv);
    dq_first = dq_cost > kv_cost;
  }
  KtScope kt(TT_KT_BWD, st);
  kern<<<(unsigned)(n_kv + n_dq), kDqWarps * 32, smem, st>>>(mo, mq64, mo64, mk, mv, b, dq_first ? n_dq : n_kv,
                                                            dq_first);
  if (cudaGetLastError() != cudaSuccess) return TT_ERR_CUDA;
  return TT_OK;
}

}  // namespace

size_t bwd_ws_bytes(int64_t nq, int hq) { return 2 * (size_t)hq * (size_t)((nq + 127) / 128 * 128) * sizeof(float); }

int bwd_tree(const void* ws, const void* Q, const void* K, const void* V, const void* O, const float* LSE,
             const void* dO, void* dQ, void* dK, void* dV, int64_t N, int Hq, int Hkv, int d, float scale,
             void* bws, int32_t* err, cudaStream_t st) {
  const TreeWs Lw = tree_ws_layout(0, N);
  BwdTc a = {};
  a.nq = N; a.nk = N; a.q_off = 0; a.ldp = (N + 127) / 128 * 128;
  a.lse2 = static_cast<const float*>(bws);
  a.dsum = static_cast<const float*>(bws) + (size_t)Hq * a.ldp;
  a.send = ws_at<int32_t>(ws, Lw.send);
  a.blk_min = ws_at<int32_t>(ws, Lw.blk_min);
  a.blk_max = ws_at<int32_t>(ws, Lw.blk_max);
  a.hdr = ws_at<int64_t>(ws, Lw.hdr);
  a.dq = static_cast<__nv_bfloat16*>(dQ); a.dk = static_cast<__nv_bfloat16*>(dK); a.dv = static_cast<__nv_bfloat16*>(dV);
  a.hq = Hq; a.hkv = Hkv; a.scale = scale; a.scale_log2 = scale * 1.4426950408889634f; a.err = err;
  const int32_t* fo = ws_at<int32_t>(ws, Lw.fwd_order);
  const int32_t* bo = ws_at<int32_t>(ws, Lw.bwd_order);
  return d == 64 ? launch_bwd<64, kTreeM>(a, Q, K, V, O, LSE, N, dO, fo, bo, st)
                 : launch_bwd<128, kTreeM>(a, Q, K, V, O, LSE, N, dO, fo, bo, st);
}

int bwd_chunk(const void* q, int64_t C, int64_t s0, const void* k, const void* v, const int32_t* send,
              const int32_t* blk_max, const void* o, const float* lse, int64_t lse_ld, const void* dO, void* dq,
              float* dk_acc, float* dv_acc, int Hq, int Hkv, int d, float scale, void* bws, int32_t* err,
              cudaStream_t st) {
  BwdTc a = {};
  a.nq = C; a.nk = s0 + C; a.q_off = s0; a.ldp = (C + 127) / 128 * 128; a.send = send; a.blk_max = blk_max;
  a.lse2 = static_cast<const float*>(bws);
  a.dsum = static_cast<const float*>(bws) + (size_t)Hq * a.ldp;
  a.dq = static_cast<__nv_bfloat16*>(dq); a.dk_acc = dk_acc; a.dv_acc = dv_acc;
  a.hq = Hq; a.hkv = Hkv; a.scale = scale; a.scale_log2 = scale * 1.4426950408889634f; a.err = err;
  return d == 64 ? launch_bwd<64, kChunkM>(a, q, k, v, o, lse, lse_ld, dO, nullptr, nullptr, st)
                 : launch_bwd<128, kChunkM>(a, q, k, v, o, lse, lse_ld, dO, nullptr, nullptr, st);
}

}  // namespace tc
}  // namespace tt

