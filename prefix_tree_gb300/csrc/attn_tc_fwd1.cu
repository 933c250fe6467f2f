// Tree attention forward on the 5th-generation tensor cores, one query tile
// per CTA: the schedule for launches too small to fill the GPU with tile
// pairs (short query chunks, small trees), where twice the CTAs beat the
// paired kernel's better per-tile overlap.
//
// "Tree Training", Abstract: every token attends only to its root-to-token
// path of the DFS-serialised tree, which reproduces independent per-branch
// attention exactly. Key k is visible to query t iff k <= t < send[k].
// AReaL-DTA, Key Contributions 1–2: the same kernel serves a query chunk at
// path offset s0 against a contiguous path K/V (query i sees keys 0..s0+i).
//
// One CTA = one 128-row query tile of one query head; 10 warps:
//   warp 0      TMA producers: lane 0 loads Q once and then K of each
//               scheduled 128-key block into a 3-stage ring; lane 1 loads V
//               (and the keys' send values) into a 2-stage ring of its own;
//   warp 1      MMA issuer (one thread): S = Q·Kᵀ into one of two TMEM S
//               buffers, then O += P·V with P read from TMEM (A operand);
//   warps 2..9  softmax / epilogue: two warps per TMEM lane quarter, each
//               thread one query row (= TMEM lane) and 64 of a block's 128
//               keys; the two halves of a row agree on the row maximum
//               through shared memory (an mbarrier per lane quarter);
//               masked online softmax with lazy rescaling (the running max
//               only moves when it grows by more than 2^8), P written back
//               to TMEM as bf16, O rescaled in TMEM when the max moves,
//               final O / l and LSE written to global memory.
// Key blocks with no ancestor pair are never loaded (per-block max of send);
// the element mask runs only on blocks that are not fully visible.
// TMEM: S0 [0,128) S1 [128,256) O [256,256+D) P0 [384,448) P1 [448,512).
//
// Key-range split (chunk mode, for launches whose tiles x heads leave SMs
// idle or spill into a short second wave): the P CTAs of a thread-block
// cluster share one tile and head, CTA p taking key blocks [p·nb/P,
// (p+1)·nb/P) of the tile's nb. Each leaves its unnormalised O, running
// maximum m_p and row sum l_p in its own shared memory (the K ring, idle by
// then); after a cluster barrier CTA p finalises rows [p·128/P, (p+1)·128/P)
// from all P partials over distributed shared memory: M = max_p m_p,
// w_p = 2^(m_p − M), L = Σ_p w_p·l_p, O = Σ_p w_p·O_p / L, LSE = (M + log2 L)·ln 2
// (the online-softmax merge of disjoint key sets).
#include "attn.cuh"
#include "tc_common.cuh"

namespace tt {
namespace tc {

namespace {

constexpr int kTreeM = 0, kChunkM = 1;
constexpr int kFwdWarps = 10;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP0 = 384, kColP1 = 448;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 2^8 between rescales
// Tree mode: the tile's key blocks (those with an ancestor pair) are listed in
// shared memory once per CTA, so that no role scans the per-block maxima in
// global memory on its critical path; tiles past kMaxList blocks scan instead.
constexpr int kMaxList = 4096;

// mbarrier slots
// FINAL completes once, after the last MMA of the CTA: the epilogue reads O
// after it and no MMA is in flight when the CTA exits.
// K and V have rings of their own (kKStages, kVStages): a K stage is free once
// S = Q·Kᵀ of its block is done, a V stage once O += P·V is done (the P_FREE
// barrier of the same parity: each tcgen05.commit costs the MMA thread tens
// of cycles, while the tensor pipe holds only a few queued MMAs), so the
// loads of later blocks do not wait for the softmax of earlier ones. The
// keys' send values travel with V (they are read by the softmax).
constexpr int kKStages = 3, kVStages = 2;
static_assert(kVStages == 2, "a V stage is released by the P-buffer barrier of the same parity");
// S_FULL[i % kKStages] completes when S of block i is done; it also frees K
// stage i % kKStages (one commit for both).
constexpr int Q_FULL = 0, K_FULL = 1, V_FULL = K_FULL + kKStages, S_FULL = V_FULL + kVStages,
              S_FREE = S_FULL + kKStages, P_READY = S_FREE + 2,
              P_FREE = P_READY + 2, FINAL = P_FREE + 2, XMAX = FINAL + 1,
              XL = XMAX + 8, STALL = XL + 4, NBAR = STALL + 1;  // XMAX: [parity][lane quarter], XL: [lane quarter]

struct FwdTc {
  int64_t nq, nk, q_off, lse_ld;
  const int32_t* send;     // tree and packed chunk: per-key subtree end, zero-padded to a multiple of 128
  const int32_t* blk_min;  // tree: per-128-key-block min / max of send (packed chunk: max only)
  const int32_t* blk_max;
  const int32_t* order;    // tree: longest-first query-tile order
  const int64_t* hdr;
  __nv_bfloat16* o;
  float* lse;
  int hq, hkv;
  int nsplit;  // chunk mode: CTAs (one cluster) per tile and head, each a key range; 1 = no split
  float scale_log2;
  int32_t* err;
  // Test hook, 0 in normal calls: the MMA thread waits stall_ns on a barrier
  // nothing arrives at before its second key block, so that the timeout path
  // (abort, drain, TT_ERR_TIMEOUT) runs in the middle of the pipeline.
  uint64_t stall_ns;
};

template <int D>
struct FwdSmem {
  static constexpr uint32_t kChunk = 128 * 128;  // one [128 rows][64 cols] bf16 box
  static constexpr uint32_t kTileB = (D / 64) * kChunk;
  static constexpr uint32_t q = 0;
  static constexpr uint32_t k0 = q + kTileB;
  static constexpr uint32_t v0 = k0 + kKStages * kTileB;
  static constexpr uint32_t send = v0 + kVStages * kTileB;
  static constexpr uint32_t xch = send + kVStages * 128 * 4;  // [2][2][128] f32 partial row maxima
  static constexpr uint32_t xl = xch + 2 * 2 * 128 * 4;       // [2][128] f32 partial row sums
  static constexpr uint32_t blist = xl + 2 * 128 * 4;         // [kMaxList] u16 key blocks of the tile
  static constexpr uint32_t bars = blist + kMaxList * 2;
  static constexpr uint32_t misc = bars + NBAR * 8;
  static constexpr uint32_t total = misc + 16 + 1024;  // + slack for 1024-byte alignment
  // key-range split: the CTA's partial O, [128][kPartLd] fp32 over the K ring
  // (row stride padded by 16 bytes: the rows written by consecutive threads
  // fall in different banks), and [2][128] fp32 (m, l) over the send slots
  static constexpr uint32_t kPartLd = D + 4;
  static_assert(128 * kPartLd * 4 <= kKStages * kTileB, "partial O exceeds the K ring");
  static_assert(2 * 128 * 4 <= kVStages * 128 * 4, "partial (m, l) exceed the send slots");
};
constexpr int kMaxSplit = 4;

// Tree mode, tiles past the listed range: the next key block after b with an ancestor pair.
__device__ __forceinline__ int next_tree_block(const FwdTc& a, int T, int64_t q0, int b) {
  for (int x = b + 1; x <= T; ++x)
    if (a.blk_max[x] > q0) return x;
  return -1;
}

// Key-range split: CTA `part` of the cluster finalises rows [part·128/P,
// (part+1)·128/P) of the tile from the P partials (threads 64..319).
template <int D>
__device__ __forceinline__ void split_combine(const FwdTc& a, uint8_t* sm, int P, int part, int64_t q0, int h) {
  using L = FwdSmem<D>;
  constexpr float kLn2c = 0.6931471805599453f;
  const int t = (int)threadIdx.x - 64;
  const int r_lo = part * 128 / P, r_hi = (part + 1) * 128 / P, nr = r_hi - r_lo;
  float* wl = reinterpret_cast<float*>(sm + L::xch);  // [128][kMaxSplit] w_p / L
  const uint32_t pml = smem_u32(sm + L::send), po = smem_u32(sm + L::k0);
  if (t < nr) {
    const int r = r_lo + t;
    float m[kMaxSplit], l[kMaxSplit], M = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxSplit; ++j) {
      m[j] = -INFINITY;
      l[j] = 0.f;
      if (j < P) {
        m[j] = dsmem_ld_f32(dsmem_addr(pml + r * 4, j));
        l[j] = dsmem_ld_f32(dsmem_addr(pml + (128 + r) * 4, j));
      }
      M = fmaxf(M, m[j]);
    }
    float w[kMaxSplit], Ls = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxSplit; ++j) {
      w[j] = m[j] == -INFINITY ? 0.f : fast_exp2(m[j] - M);
      Ls += w[j] * l[j];
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
    for (int j = 0; j < kMaxSplit; ++j) wl[r * kMaxSplit + j] = w[j] * inv;
    const int64_t q = q0 + r;
    if (q < a.nq) a.lse[(int64_t)h * a.lse_ld + q] = Ls > 0.f ? (M + __log2f(Ls)) * kLn2c : -INFINITY;
  }
  named_barrier(1, 256);
  constexpr int kC8 = D / 8;  // 8-column groups of a row (one 16-byte bf16 store)
  for (int e = t; e < nr * kC8; e += 256) {
    const int r = r_lo + e / kC8, c = (e % kC8) * 8;
    const int64_t q = q0 + r;
    if (q >= a.nq) continue;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const uint32_t off = po + (uint32_t)(r * L::kPartLd + c) * 4;
    for (int j = 0; j < P; ++j) {
      const float wj = wl[r * kMaxSplit + j];
      if (wj == 0.f) continue;  // no visible key of this row in split j (its O is not written)
      const uint32_t src = dsmem_addr(off, j);
      const float4 x = dsmem_ld_f32x4(src), y = dsmem_ld_f32x4(src + 16);
      acc[0] += wj * x.x; acc[1] += wj * x.y; acc[2] += wj * x.z; acc[3] += wj * x.w;
      acc[4] += wj * y.x; acc[5] += wj * y.y; acc[6] += wj * y.z; acc[7] += wj * y.w;
    }
    uint4 o;
    o.x = pack_bf16(acc[0], acc[1]);
    o.y = pack_bf16(acc[2], acc[3]);
    o.z = pack_bf16(acc[4], acc[5]);
    o.w = pack_bf16(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(a.o + q * (int64_t)a.hq * D + (int64_t)h * D + c) = o;
  }
}

template <int D, int MODE>
__global__ void __launch_bounds__(kFwdWarps * 32, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdTc a) {
  using L = FwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::misc + 4);
  int32_t* sSend = reinterpret_cast<int32_t*>(sm + L::send);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (MODE == kTreeM) {
    if (a.hdr[0] != kTreeMagic || a.hdr[1] != a.nq) {
      if (threadIdx.x == 0) set_err(a.err, TT_ERR_INVALID_ARG);
      return;
    }
    if (a.hdr[3] == 0) {
      if (threadIdx.x == 0) set_err(a.err, TT_ERR_INVALID_TREE);
      return;
    }
  }
  // blockIdx.x = (tile-head) · P + part; a cluster is the P CTAs of one tile-head
  const int P = MODE == kChunkM ? a.nsplit : 1;
  const int th = (int)blockIdx.x / P, part = (int)blockIdx.x % P;
  const int h = th % a.hq;
  const int nT = (int)((a.nq + 127) / 128);
  const int T = MODE == kTreeM ? a.order[th / a.hq] : nT - 1 - th / a.hq;
  const int g = h / (a.hq / a.hkv);
  const int64_t q0 = (int64_t)T * 128, q1 = min(q0 + 128, a.nq);
  // chunk mode: this CTA's key blocks [c_lo, c_hi) of the tile's nb (query i sees keys 0..s0+i); a packed
  // chunk (a.send set) lists the blocks the tile sees and splits positions [c_lo, c_hi) of that list
  const bool packed = MODE == kChunkM && a.send != nullptr;
  int c_lo = 0, c_hi = 0, nb = 0;
  if (MODE == kChunkM) {
    const int64_t kmax = min(a.nk, a.q_off + q1);
    nb = (int)((kmax + 127) / 128);
    c_lo = (int)((int64_t)part * nb / P);
    c_hi = (int)((int64_t)(part + 1) * nb / P);
  }
  const bool plist = packed && nb <= kMaxList;

  if (threadIdx.x == 0) {
    mbar_init(&bar[Q_FULL], 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bar[K_FULL + i], 1);
      mbar_init(&bar[S_FULL + i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bar[V_FULL + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[S_FREE + i], 256);
      mbar_init(&bar[P_READY + i], 256);
      mbar_init(&bar[P_FREE + i], 1);
    }
    mbar_init(&bar[FINAL], 1);
    for (int i = 0; i < 8; ++i) mbar_init(&bar[XMAX + i], 64);
    for (int i = 0; i < 4; ++i) mbar_init(&bar[XL + i], 64);
    mbar_init(&bar[STALL], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  uint16_t* blist = reinterpret_cast<uint16_t*>(sm + L::blist);
  int* nlist = reinterpret_cast<int*>(sm + L::misc + 8);
  const bool use_list = (MODE == kTreeM && T < kMaxList) || plist;
  if (warp == 0 && plist) {
    // packed chunk: a block is seen by the tile if it holds a path key or the
    // maximum send over its keys exceeds the tile's first query; bit 15: path
    // keys only
    const int64_t qa0 = a.q_off + q0;
    int cnt = 0;
    for (int base = 0; base < nb; base += 32) {
      const int x = base + lane;
      const int64_t kx = (int64_t)x * 128;
      const bool keep = x < nb && (kx < a.q_off || a.blk_max[x] > qa0);
      const uint32_t m = __ballot_sync(0xffffffffu, keep);
      if (keep) blist[cnt + __popc(m & ((1u << lane) - 1u))] = (uint16_t)(x | (kx + 128 <= a.q_off ? 0x8000 : 0));
      cnt += __popc(m);
    }
    if (lane == 0) *nlist = cnt;
  } else if (warp == 0 && use_list) {
    int cnt = 0;
    for (int base = 0; base <= T; base += 32) {
      const int x = base + lane;
      const bool keep = x <= T && a.blk_max[x] > q0;
      const uint32_t m = __ballot_sync(0xffffffffu, keep);
      // bit 15: every key of the block is visible to every query of the tile
      const bool full = keep && (int64_t)x * 128 + 127 <= q0 && (int64_t)x * 128 + 128 <= a.nk && a.blk_min[x] >= q1;
      if (keep) blist[cnt + __popc(m & ((1u << lane) - 1u))] = (uint16_t)(x | (full ? 0x8000 : 0));
      cnt += __popc(m);
    }
    if (lane == 0) *nlist = cnt;
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const int n_list = use_list ? *nlist : 0;
  if (plist) {
    c_lo = (int)((int64_t)part * n_list / P);
    c_hi = (int)((int64_t)(part + 1) * n_list / P);
  }
  // block at position idx of the schedule (prev = the block at idx - 1)
  auto nextb = [&](int idx, int prev) -> int {
    if (MODE == kChunkM) {
      if (plist) return c_lo + idx < c_hi ? (int)(blist[c_lo + idx] & 0x7fff) : -1;
      const int x = prev < 0 ? c_lo : prev + 1;
      return x < c_hi ? x : -1;
    }
    if (use_list) return idx < n_list ? (int)(blist[idx] & 0x7fff) : -1;
    return next_tree_block(a, T, q0, prev);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producers
    // lane 0: Q, then the K ring; lane 1: the V ring (with the keys' send values)
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      mbar_expect_tx(&bar[Q_FULL], 128 * D * 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_load_2d(sm + L::q + c * L::kChunk, &tmQ, &bar[Q_FULL], h * D + c * 64, (int)q0);
      int i = 0;
      for (int b = nextb(0, -1); b >= 0; b = nextb(i + 1, b), ++i) {
        const int st = i % kKStages;
        if (i >= kKStages && !mbar_wait(&bar[S_FULL + st], ((i - kKStages) / kKStages) & 1, abort_flag, 10)) break;
        mbar_expect_tx(&bar[K_FULL + st], 128 * D * 2);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sm + L::k0 + st * L::kTileB + c * L::kChunk, &tmK, &bar[K_FULL + st], g * D + c * 64, b * 128);
      }
      // every copy issued has landed before the CTA may leave
      mbar_drain(&bar[Q_FULL], 0, abort_flag);
      for (int j = i - 1; j >= 0 && j >= i - kKStages; --j) mbar_drain(&bar[K_FULL + j % kKStages], (j / kKStages) & 1, abort_flag);
    } else if (lane == 1) {
      prefetch_tmap(&tmV);
      int i = 0;
      for (int b = nextb(0, -1); b >= 0; b = nextb(i + 1, b), ++i) {
        const int st = i % kVStages;
        // V stage st = i & 1 is free once O += P·V of block i − 2 is done: the
        // same event (and phase) as P buffer st being free
        if (i >= kVStages && !mbar_wait(&bar[P_FREE + st], ((i - kVStages) >> 1) & 1, abort_flag, 9)) break;
        // send values of the block: tree mode, and packed blocks holding a chunk key
        const bool ld_send = MODE == kTreeM || (packed && (int64_t)b * 128 + 128 > a.q_off);
        mbar_expect_tx(&bar[V_FULL + st], 128 * D * 2 + (ld_send ? 512 : 0));
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sm + L::v0 + st * L::kTileB + c * L::kChunk, &tmV, &bar[V_FULL + st], g * D + c * 64, b * 128);
        if (ld_send) bulk_load(sSend + st * 128, a.send + (int64_t)b * 128, 512, &bar[V_FULL + st]);
      }
      for (int j = i - 1; j >= 0 && j >= i - kVStages; --j) mbar_drain(&bar[V_FULL + j % kVStages], (j / kVStages) & 1, abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idPV = idesc_bf16(128, D, 0, 1);
      const uint64_t dq = smem_desc(smem_u32(sm + L::q), 16, 1024);
      bool ok = mbar_wait(&bar[Q_FULL], 0, abort_flag, 11);
      auto issue_pv = [&](int ip) -> bool {
        const int bb = ip & 1, st = ip % kVStages;
        if (!mbar_wait(&bar[P_READY + bb], (ip >> 1) & 1, abort_flag, 12)) return false;
        if (!mbar_wait(&bar[V_FULL + st], (ip / kVStages) & 1, abort_flag, 8)) return false;
        tc_fence_after();
        const uint64_t dv = smem_desc(smem_u32(sm + L::v0 + st * L::kTileB), L::kChunk, 1024);
        const uint32_t pcol = tbase + (bb ? kColP1 : kColP0);
#pragma unroll
        for (int k = 0; k < 128 / 16; ++k)
          umma_ts(tbase + kColO, pcol + k * 8, desc_at(dv, k * 2048), idPV, (ip > 0 || k > 0));
        umma_commit(&bar[P_FREE + bb]);  // also frees V stage bb (kVStages == 2)
        return true;
      };
      int i = 0;
      if (ok) {
        for (int b = nextb(0, -1); b >= 0; b = nextb(i + 1, b), ++i) {
          const int bb = i & 1, st = i % kKStages;
          if (i == 1 && a.stall_ns && !mbar_wait(&bar[STALL], 0, abort_flag, 6, a.stall_ns)) { ok = false; break; }
          if (!mbar_wait(&bar[K_FULL + st], (i / kKStages) & 1, abort_flag, 13)) { ok = false; break; }
          if (i >= 2 && !mbar_wait(&bar[S_FREE + bb], ((i - 2) >> 1) & 1, abort_flag, 14)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dk = smem_desc(smem_u32(sm + L::k0 + st * L::kTileB), 16, 1024);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * L::kChunk + (k & 3) * 32;
            umma_ss(tbase + (bb ? kColS1 : kColS0), desc_at(dq, off), desc_at(dk, off), idS, k > 0);
          }
          umma_commit(&bar[S_FULL + st]);  // S ready; K stage st free
          if (i >= 1 && !issue_pv(i - 1)) { ok = false; break; }
        }
        if (ok && i >= 1) issue_pv(i - 1);
      }
      // completes after every MMA of this CTA: O is final, nothing in flight
      // (waited for even after an abort: TMEM and shared memory must outlive the MMAs)
      umma_commit(&bar[FINAL]);
      mbar_drain(&bar[FINAL], 0, abort_flag);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int wq = warp & 3;
    const int hf = (warp - 2) >> 2;  // keys [64·hf, 64·hf + 64) of each block, O columns [D/2·hf, D/2·hf + D/2)
    const int r = wq * 32 + lane;
    const int64_t q = q0 + r;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    float* xmax = reinterpret_cast<float*>(sm + L::xch);  // [parity][half][row]
    float* xl = reinterpret_cast<float*>(sm + L::xl);     // [half][row]
    float m_used = -INFINITY, l = 0.f;
    int i = 0;
    bool ok = true;
    for (int b = nextb(0, -1); b >= 0; b = nextb(i + 1, b), ++i) {
      const int bb = i & 1;
      if (!mbar_wait(&bar[S_FULL + i % kKStages], (i / kKStages) & 1, abort_flag, 15)) { ok = false; break; }
      tc_fence_after();
      uint32_t s[2][32];
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_ld32(tbase + lane_base + (bb ? kColS1 : kColS0) + 64 * hf + c * 32, s[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_pin(s[c]);
      tc_fence_before();
      mbar_arrive(&bar[S_FREE + bb]);

      const int64_t kb = (int64_t)b * 128;
      bool full;
      if (MODE == kTreeM) {
        full = use_list ? (blist[i] >> 15) != 0 : (kb + 127 <= q0 && kb + 128 <= a.nk && a.blk_min[b] >= q1);
        // the keys' send values arrive with this block's V
        if (!full && !mbar_wait(&bar[V_FULL + i % kVStages], (i / kVStages) & 1, abort_flag, 7)) { ok = false; break; }
      } else if (packed) {
        full = kb + 128 <= a.q_off;  // path keys only
        if (!full && !mbar_wait(&bar[V_FULL + i % kVStages], (i / kVStages) & 1, abort_flag, 7)) { ok = false; break; }
      } else {
        full = kb + 127 <= a.q_off + q0 && kb + 128 <= a.nk;
      }
      // Row maximum on the raw scores (scaling by a positive constant commutes
      // with max); masked scores become -inf and so contribute exp2(-inf) = 0.
      // The uniform `full` test is taken once per block (not per element) and
      // the mask is applied with selects; four independent maxima shorten the
      // dependency chain.
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (full) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int j = 0; j < 16; ++j)
            mx4[j & 3] = fmax3f(mx4[j & 3], __uint_as_float(s[c][2 * j]), __uint_as_float(s[c][2 * j + 1]));
      } else if (MODE == kTreeM || packed) {
        const int4* sv = reinterpret_cast<const int4*>(sSend + (i % kVStages) * 128 + 64 * hf);
        const int64_t qa = a.q_off + q;    // path position of the query (q_off = 0 in tree mode)
        const int64_t dq = qa - kb - 64 * hf;  // key column col of this half is visible iff col <= dq and qa < send
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const int4 se = sv[c * 8 + j4];
            const int sj[4] = {se.x, se.y, se.z, se.w};
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int col = c * 32 + j4 * 4 + e;
              const bool vis = col <= dq && qa < sj[e];
              v[e] = vis ? __uint_as_float(s[c][j4 * 4 + e]) : -INFINITY;
              s[c][j4 * 4 + e] = __float_as_uint(v[e]);
            }
            mx4[(j4 & 1) * 2] = fmax3f(mx4[(j4 & 1) * 2], v[0], v[1]);
            mx4[(j4 & 1) * 2 + 1] = fmax3f(mx4[(j4 & 1) * 2 + 1], v[2], v[3]);
          }
      } else {
        const int64_t lim = a.q_off + q - kb - 64 * hf;  // visible iff col <= lim
        const int64_t lim2 = a.nk - 1 - kb - 64 * hf;    // and col < nk - kb - 64·hf
        const int64_t cmax = lim < lim2 ? lim : lim2;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float x0 = (c * 32 + 2 * j) <= cmax ? __uint_as_float(s[c][2 * j]) : -INFINITY;
            const float x1 = (c * 32 + 2 * j + 1) <= cmax ? __uint_as_float(s[c][2 * j + 1]) : -INFINITY;
            s[c][2 * j] = __float_as_uint(x0);
            s[c][2 * j + 1] = __float_as_uint(x1);
            mx4[j & 3] = fmax3f(mx4[j & 3], x0, x1);
          }
      }
      // the row maximum from both halves (slot parity bb is reused two blocks
      // later, after both halves have passed the next block's exchange)
      {
        const float pm = fmax3f(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
        xmax[(bb * 2 + hf) * 128 + r] = pm;
        mbar_arrive(&bar[XMAX + bb * 4 + wq]);
        if (!mbar_wait(&bar[XMAX + bb * 4 + wq], (i >> 1) & 1, abort_flag, 20)) { ok = false; break; }
        mx4[0] = fmaxf(pm, xmax[(bb * 2 + (hf ^ 1)) * 128 + r]);
      }
      const float mx = mx4[0] * a.scale_log2;
      bool resc = false;
      float alpha = 1.f;
      if (mx > m_used + kRescaleThreshold) {
        alpha = fast_exp2(m_used - mx);  // 0 on the first visible block
        l *= alpha;
        resc = i > 0;
        m_used = mx;
      }
      const float mu = m_used == -INFINITY ? 0.f : m_used;
      // p = exp2(s·scale·log2e − m), two lanes per packed fp32 instruction
      const float2 c2 = make_float2(a.scale_log2, a.scale_log2), nm2 = make_float2(-mu, -mu);
      float2 rs2 = make_float2(0.f, 0.f);
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[c][2 * j]), __uint_as_float(s[c][2 * j + 1])), c2, nm2);
          const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          rs2 = __fadd2_rn(rs2, pp);
          pk[c * 16 + j] = pack_bf16(pp.x, pp.y);
        }
      }
      l += rs2.x + rs2.y;
      if (i >= 2 && !mbar_wait(&bar[P_FREE + bb], ((i - 2) >> 1) & 1, abort_flag, 16)) { ok = false; break; }
      if (__any_sync(0xffffffffu, resc)) {
        // O += P·V of block i − 1 done (P buffer (i − 1) & 1 free)
        if (!mbar_wait(&bar[P_FREE + ((i - 1) & 1)], ((i - 1) >> 1) & 1, abort_flag, 17)) { ok = false; break; }
        tc_fence_after();
        const float f = resc ? alpha : 1.f;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          const uint32_t col = kColO + (D / 2) * hf + c * 32;
          uint32_t o[32];
          tmem_ld32(tbase + lane_base + col, o);
          tmem_ld_wait();
          tmem_pin(o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
          tmem_st32(tbase + lane_base + col, o);
        }
      }
      tmem_st32(tbase + lane_base + (bb ? kColP1 : kColP0) + 32 * hf, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[P_READY + bb]);
    }
    const int n = i;
    // the row sum from both halves
    bool have = ok && n > 0;
    if (have) {
      xl[hf * 128 + r] = l;
      mbar_arrive(&bar[XL + wq]);
      have = mbar_wait(&bar[XL + wq], 0, abort_flag, 21);
      if (have) l += xl[(hf ^ 1) * 128 + r];
    }
    if (have) have = mbar_wait(&bar[FINAL], 0, abort_flag, 18);
    if (P > 1) {
      // Key-range split: publish this CTA's unnormalised O and (m, l) in its
      // own shared memory (FINAL has completed: no MMA reads the K ring any
      // more and every K copy issued has landed). A row with no visible key
      // here, or an aborted CTA, publishes m = -inf and is left out.
      float* part_o = reinterpret_cast<float*>(sm + L::k0);
      float* pml = reinterpret_cast<float*>(sm + L::send);
      if (have) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          const int cc = (D / 64) * hf + c;
          uint32_t o[32];
          tmem_ld32(tbase + lane_base + kColO + cc * 32, o);
          tmem_ld_wait();
          tmem_pin(o);
          float4* dst = reinterpret_cast<float4*>(part_o + r * L::kPartLd + cc * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]), __uint_as_float(o[4 * v + 2]),
                                 __uint_as_float(o[4 * v + 3]));
        }
      }
      if (hf == 0) {
        pml[r] = have && l > 0.f ? m_used : -INFINITY;
        pml[128 + r] = have ? l : 0.f;
      }
    } else if (have) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = a.o + q * (int64_t)a.hq * D + (int64_t)h * D;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int cc = (D / 64) * hf + c;  // 32-column chunk of O
        uint32_t o[32];
        tmem_ld32(tbase + lane_base + kColO + cc * 32, o);
        tmem_ld_wait();
        tmem_pin(o);
        if (q < a.nq) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
            dst[v] = w;
          }
        }
      }
      if (q < a.nq && hf == 0) a.lse[(int64_t)h * a.lse_ld + q] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
    }
  }
  if (MODE == kChunkM && P > 1) {
    // Every thread of every CTA of the cluster passes both barriers (no role
    // returns early in chunk mode and every wait above is bounded).
    __syncwarp();
    cluster_barrier();  // all partials published
    if (warp >= 2) split_combine<D>(a, sm, P, part, q0, h);
    __syncwarp();
    cluster_barrier();  // no CTA leaves while a peer may still read its shared memory
  }
  if (*abort_flag && threadIdx.x == 0) set_err(a.err, TT_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

template <int D, int MODE>
int launch_fwd(const FwdTc& a, const void* q, const void* k, const void* v, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!make_tmap_bf16(&mq, q, (uint64_t)a.hq * D, a.nq, 128) || !make_tmap_bf16(&mk, k, (uint64_t)a.hkv * D, a.nk, 128) ||
      !make_tmap_bf16(&mv, v, (uint64_t)a.hkv * D, a.nk, 128))
    return TT_ERR_CUDA;
  const int smem = (int)FwdSmem<D>::total;
  auto kern = fwd_tc_kernel<D, MODE>;
  if (!smem_attr_set<fwd_tc_kernel<D, MODE>>(smem)) return TT_ERR_CUDA;
  const unsigned grid = (unsigned)((a.nq + 127) / 128) * a.hq * a.nsplit;
  if (a.nsplit == 1) {
    KtScope kt(TT_KT_FWD, st);
    kern<<<grid, kFwdWarps * 32, smem, st>>>(mq, mk, mv, a);
    return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFwdWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.nsplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  KtScope kt(TT_KT_FWD, st);
  return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, a) == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

// CTAs of the chunk kernel resident at once in clusters of P (queried once
// per device, head size and P; a cluster lives on one GPC, so P > 1 can leave
// SMs of a GPC idle).
template <int D>
int split_slots(int P) {
  static std::atomic<int> cache[kMaxDevices][kMaxSplit + 1];
  const int dev = current_device();
  const int sms = sm_count();
  if (dev < 0 || sms < 1) return 0;
  if (P == 1) return sms;
  int v = cache[dev][P].load(std::memory_order_relaxed);
  if (v == 0) {
    const int smem = (int)FwdSmem<D>::total;
    int n = 0;
    if (smem_attr_set<fwd_tc_kernel<D, kChunkM>>(smem)) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(P * sms));
      cfg.blockDim = dim3(kFwdWarps * 32);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = P;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, fwd_tc_kernel<D, kChunkM>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
      }
    }
    v = n > 0 ? n * P : -1;  // -1: clusters of P unavailable
    cache[dev][P].store(v, std::memory_order_relaxed);
  }
  return v;
}

// Splits per tile for a chunk launch: each of the n = tiles x heads units
// costs about nb key blocks plus a fixed cost per CTA (launch, Q load,
// pipeline fill and drain, epilogue: kCtaOverhead block-equivalents, about
// 8.5 us against about 1 us per 128-key block on a GB300), and a split CTA
// kMergeOverhead more (publishing the partial, two cluster barriers, the
// merge); P splits cost ceil(n·P / slots_P) waves of ceil(nb / P) + those.
// The smallest estimate wins (ties: fewer splits), so splits are taken for
// launches too small to fill the GPU once, not to even out a second wave.
constexpr int kCtaOverhead = 8, kMergeOverhead = 5;
template <int D>
int choose_splits(int64_t C, int64_t s0, int hq) {
  const int64_t n = (C + 127) / 128 * hq;
  const int64_t nb = (s0 + C + 127) / 128;
  int best = 1;
  double best_cost = 0.0;
  for (int P = 1; P <= kMaxSplit && P <= nb; ++P) {
    const int slots = split_slots<D>(P);
    if (slots < 1) continue;
    const double cost = (double)((n * P + slots - 1) / slots) *
                        (double)((nb + P - 1) / P + kCtaOverhead + (P > 1 ? kMergeOverhead : 0));
    if (P == 1 || cost < best_cost) {
      best = P;
      best_cost = cost;
    }
  }
  return best;
}

}  // namespace

// One-tile entry points (attn_tc.cu chooses between these and the paired kernel).
int fwd_tree_1tile(const void* ws, const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t N, int Hq,
             int Hkv, int d, float scale, int32_t* err, cudaStream_t st, uint64_t stall_ns) {
  const TreeWs Lw = tree_ws_layout(0, N);
  FwdTc a = {};
  a.nq = N; a.nk = N; a.q_off = 0; a.lse_ld = N;
  a.send = ws_at<int32_t>(ws, Lw.send);
  a.blk_min = ws_at<int32_t>(ws, Lw.blk_min);
  a.blk_max = ws_at<int32_t>(ws, Lw.blk_max);
  a.order = ws_at<int32_t>(ws, Lw.fwd_order);
  a.hdr = ws_at<int64_t>(ws, Lw.hdr);
  a.o = static_cast<__nv_bfloat16*>(O); a.lse = LSE; a.hq = Hq; a.hkv = Hkv;
  a.scale_log2 = scale * 1.4426950408889634f; a.err = err; a.stall_ns = stall_ns; a.nsplit = 1;
  return d == 64 ? launch_fwd<64, kTreeM>(a, Q, K, V, st) : launch_fwd<128, kTreeM>(a, Q, K, V, st);
}

int fwd_chunk_1tile(const void* q, int64_t C, int64_t s0, const void* k, const void* v, const int32_t* send,
                    const int32_t* blk_max, void* o, float* lse, int64_t lse_ld, int Hq, int Hkv, int d, float scale,
                    int32_t* err, cudaStream_t st, int splits, uint64_t stall_ns) {
  if (splits < 0 || splits > kMaxSplit) return TT_ERR_INVALID_ARG;
  FwdTc a = {};
  a.nq = C; a.nk = s0 + C; a.q_off = s0; a.lse_ld = lse_ld; a.send = send; a.blk_max = blk_max;
  a.o = static_cast<__nv_bfloat16*>(o); a.lse = lse; a.hq = Hq; a.hkv = Hkv;
  a.scale_log2 = scale * 1.4426950408889634f; a.err = err; a.stall_ns = stall_ns;
  a.nsplit = splits > 0 ? splits : d == 64 ? choose_splits<64>(C, s0, Hq) : choose_splits<128>(C, s0, Hq);
  if (splits > 1 && (d == 64 ? split_slots<64>(splits) : split_slots<128>(splits)) < 1) return TT_ERR_UNSUPPORTED;
  return d == 64 ? launch_fwd<64, kChunkM>(a, q, k, v, st) : launch_fwd<128, kChunkM>(a, q, k, v, st);
}

}  // namespace tc
}  // namespace tt
