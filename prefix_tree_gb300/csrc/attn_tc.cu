// Tree attention forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// "Tree Training", Abstract: every token attends only to its root-to-token
// path of the DFS-serialised tree, which reproduces independent per-branch
// attention exactly. Key k is visible to query t iff k <= t < send[k].
// AReaL-DTA, Key Contributions 1–2: the same kernel serves a query chunk at
// path offset s0 against a contiguous path K/V (query i sees keys 0..s0+i).
//
// One CTA = two 128-row query tiles that read the same K/V blocks: two query
// heads of one KV group over the same rows; when the group size is odd, its
// last head takes two adjacent query tiles of that head instead (the CTA's
// key blocks are the union of the two tiles'; the element mask covers the
// difference). 12 warps:
//   warp 0      TMA producer: both Q tiles once, then K of each scheduled
//               128-key block into a 2-stage ring;
//   warp 2      TMA producer: V (and the keys' send values) into a 2-stage ring;
//   warp 1      MMA issuer (one thread), per block i:
//               O_0 += P_0·V(i), S_0 = Q_0·K(i+1)ᵀ, O_1 += P_1·V(i),
//               S_1 = Q_1·K(i+1)ᵀ, so the tensor pipe works on one tile
//               while the softmax of the other runs;
//   warp 3      idle (warps 0..3 form the warpgroup that hands registers
//               to the softmax warpgroups);
//   warps 4..7  softmax / epilogue of tile 0, warps 8..11 of tile 1: one
//               thread per query row (= TMEM lane), all 128 keys of a block;
//               masked online softmax with lazy rescaling (the running max
//               only moves when it grows by more than 2^8), P written back
//               to TMEM as bf16 over S, O rescaled in TMEM when the max
//               moves, final O / l and LSE written to global memory.
// Key blocks with no ancestor pair are never loaded (per-block max of send);
// the element mask runs only on blocks that are not fully visible. A masked
// block that lies wholly before a warp's 32 rows, with no key's send inside
// them, gives every row of the warp the same visible keys: four ballots make
// the warp's column pattern, fully visible 32-column chunks take the plain
// maximum and the others a one-bit select. Other masked blocks test each
// score (k <= t < send[k]).
// TMEM: S_0 [0,128) S_1 [128,256) O_0 [256,256+D) O_1 [384,384+D); P_x over
// the first 64 columns of S_x. The MMAs of one thread run in issue order, so
// S_x of the next block overwrites P_x only after O_x += P_x·V has read it.

#include "attn.cuh"
#include "tc_common.cuh"

namespace tt {
namespace tc {

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  return make_tmap_bf16_ld(map, base, cols, rows, cols, box_rows);
}

bool make_tmap_bf16_ld(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t ld,
                       uint32_t box_rows) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static Encode encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<Encode>(fn);
  }
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// kPackM: a chunk of several sibling subtrees (chunk mode with the tree mask on the chunk's keys)
constexpr int kTreeM = 0, kChunkM = 1, kPackM = 2;
constexpr int kFwdWarps = 12;
// Registers: 12 warps launch with 168 each (three warps per SM sub-partition);
// the producer / MMA warpgroup then gives registers back so that the softmax
// warpgroups, which hold a row's 128 scores, can grow:
// 128·96 + 256·200 = 63,488 <= 384·168 = 64,512 launched.
constexpr uint32_t kRegsCtl = 96, kRegsSoftmax = 200;
static_assert(128 * kRegsCtl + 256 * kRegsSoftmax <= 384 * 168, "register split exceeds the launch's registers");
constexpr uint32_t kTmemCols = 512;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 2^8 between rescales
// Tree mode: the key blocks of the CTA's query rows (those with an ancestor
// pair) are listed in shared memory once per CTA, so that no role scans the
// per-block maxima in global memory on its critical path; CTAs whose rows lie
// past kMaxList blocks scan instead.
constexpr int kMaxList = 4096;

// TMEM of tile x (0 or 1): S_x in columns [128x, 128x + 128), P_x (bf16 pairs)
// over the first 64 of them once the softmax has read S_x, O_x in columns
// [256 + 128x, 256 + 128x + D).
__device__ __forceinline__ uint32_t col_s(int x) { return 128u * (uint32_t)x; }
__device__ __forceinline__ uint32_t col_o(int x) { return 256u + 128u * (uint32_t)x; }

// mbarrier slots. The MMA thread issues, per key block i,
//   O_0 += P_0·V(i), S_0 = Q_0·K(i+1)ᵀ, O_1 += P_1·V(i), S_1 = Q_1·K(i+1)ᵀ,
// so the tensor pipe works on one tile while the softmax warps of the other
// run. (One issuer per tile is slower: the two tiles' MMAs then interleave in
// the pipe and each tile's S arrives later.) A commit tracks every earlier MMA
// of the thread, so:
//   S0        S_0 of a block is done (and with it O_0 += P_0·V of the block
//             before: the softmax may rescale O_0 after this wait);
//   KS[st]    S_1 of the block in K stage st is done: tile 1's S is ready and
//             the K stage is free;
//   VF[st]    O_1 += P_1·V of the block in V stage st is done: the V stage is free;
//   P_RDY[x]  the 128 softmax threads of tile x wrote P_x;
//   FINAL     every MMA of the CTA is done (epilogue; nothing in flight at exit).
constexpr int kKStages = 2, kVStages = 2;
constexpr int Q_FULL = 0, K_FULL = 1, V_FULL = K_FULL + kKStages, S0 = V_FULL + kVStages, KS = S0 + 1,
              VF = KS + kKStages, P_RDY = VF + kVStages, FINAL = P_RDY + 2, STALL = FINAL + 1, NBAR = STALL + 1;

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
  int n_adj;  // CTAs [0, n_adj): two adjacent query tiles of a group's last head (odd group sizes); the rest:
              // two query heads of one KV group over the same rows
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
  static constexpr uint32_t q = 0;  // [2] tiles
  static constexpr uint32_t k0 = q + 2 * kTileB;
  static constexpr uint32_t v0 = k0 + kKStages * kTileB;
  static constexpr uint32_t send = v0 + kVStages * kTileB;
  static constexpr uint32_t blist = send + kVStages * 128 * 4;  // [kMaxList] u16 key blocks of the CTA
  static constexpr uint32_t bars = blist + kMaxList * 2;
  static constexpr uint32_t misc = bars + NBAR * 8;
  static constexpr uint32_t total = misc + 16 + 1024;  // + slack for 1024-byte alignment
};
static_assert(FwdSmem<128>::total <= 232448, "forward shared memory exceeds the per-CTA limit");

// Next key block after b with an ancestor pair for query rows [q0, q1)
// (tree: blocks up to the one holding row q1 − 1; chunk: every block up to
// the causal limit of the last row).
template <int MODE>
__device__ __forceinline__ int next_block(const FwdTc& a, int64_t q0, int64_t q1, int b) {
  if (MODE == kTreeM) {
    const int last = (int)((q1 - 1) / 128);
    for (int x = b + 1; x <= last; ++x)
      if (a.blk_max[x] > q0) return x;
    return -1;
  }
  const int64_t kmax = min(a.nk, a.q_off + q1);
  const int nb = (int)((kmax + 127) / 128);
  return b + 1 < nb ? b + 1 : -1;
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
  // The CTA's two tiles: tile x is query head h0 + x·dh, rows q0 + x·dq .. + 127.
  const int nT = (int)((a.nq + 127) / 128);
  int h0, dh;
  int64_t q0, dq;
  const int G = a.hq / a.hkv;
  if ((int)blockIdx.x >= a.n_adj) {
    // head pair hp: heads 2·(hp mod G/2) and the next one of group hp / (G/2)
    const int np = a.hkv * (G / 2);
    const int b = (int)blockIdx.x - a.n_adj;
    const int hp = b % np;
    const int ti = b / np;
    const int T = MODE == kTreeM ? a.order[ti] : nT - 1 - ti;
    h0 = (hp / (G / 2)) * G + 2 * (hp % (G / 2)); dh = 1;
    q0 = (int64_t)T * 128; dq = 0;
  } else {
    // the last head of each group when G is odd: tile pair p
    const int nP = (nT + 1) / 2;
    const int pi = (int)blockIdx.x / a.hkv;
    const int p = MODE == kTreeM ? pi : nP - 1 - pi;
    h0 = ((int)blockIdx.x % a.hkv) * G + G - 1; dh = 0;
    q0 = (int64_t)p * 256; dq = 128;
  }
  const bool has1 = q0 + dq < a.nq;  // tile 1 holds rows (only the last tile pair may lack it)
  const int g = h0 / G;
  const int64_t q1 = min(q0 + (has1 ? dq : 0) + 128, a.nq);  // the CTA's query rows are [q0, q1)

  if (threadIdx.x == 0) {
    mbar_init(&bar[Q_FULL], 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bar[K_FULL + i], 1);
      mbar_init(&bar[KS + i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bar[V_FULL + i], 1);
      mbar_init(&bar[VF + i], 1);
    }
    mbar_init(&bar[S0], 1);
    for (int x = 0; x < 2; ++x) mbar_init(&bar[P_RDY + x], 128);
    mbar_init(&bar[FINAL], 1);
    mbar_init(&bar[STALL], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  uint16_t* blist = reinterpret_cast<uint16_t*>(sm + L::blist);
  int* nlist = reinterpret_cast<int*>(sm + L::misc + 8);
  const int last_blk = (int)((q1 - 1) / 128);
  // packed chunk: the blocks the CTA's rows see are listed too
  constexpr bool packed = MODE == kPackM;
  const int nbk = MODE != kTreeM ? (int)((min(a.nk, a.q_off + q1) + 127) / 128) : 0;
  const bool plist = packed && nbk <= kMaxList;
  const bool use_list = (MODE == kTreeM && last_blk < kMaxList) || plist;
  if (warp == 0 && plist) {
    // a block is seen if it holds a path key or the maximum send over its
    // keys exceeds the CTA's first query; bit 15: path keys only
    const int64_t qa0 = a.q_off + q0;
    int cnt = 0;
    for (int base = 0; base < nbk; base += 32) {
      const int x = base + lane;
      const int64_t kx = (int64_t)x * 128;
      const bool keep = x < nbk && (kx < a.q_off || a.blk_max[x] > qa0);
      const uint32_t m = __ballot_sync(0xffffffffu, keep);
      if (keep) blist[cnt + __popc(m & ((1u << lane) - 1u))] = (uint16_t)(x | (kx + 128 <= a.q_off ? 0x8000 : 0));
      cnt += __popc(m);
    }
    if (lane == 0) *nlist = cnt;
  } else if (warp == 0 && use_list) {
    int cnt = 0;
    for (int base = 0; base <= last_blk; base += 32) {
      const int x = base + lane;
      const bool keep = x <= last_blk && a.blk_max[x] > q0;
      const uint32_t m = __ballot_sync(0xffffffffu, keep);
      // bit 15: every key of the block is visible to every query row of the CTA
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
  // block at position idx of the schedule (prev = the block at idx - 1)
  auto nextb = [&](int idx, int prev) -> int {
    if (use_list) return idx < n_list ? (int)(blist[idx] & 0x7fff) : -1;
    return next_block<MODE>(a, q0, q1, prev);
  };

  if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ TMA producers
    // warp 0: both Q tiles, then the K ring; warp 2: the V ring (with the keys'
    // send values). One thread each, in warps of their own: a thread suspended
    // in an mbarrier wait holds up the other lanes of its warp.
    if (warp == 0 && lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      mbar_expect_tx(&bar[Q_FULL], (has1 ? 2 : 1) * 128 * D * 2);
      for (int x = 0; x < (has1 ? 2 : 1); ++x)
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sm + L::q + x * L::kTileB + c * L::kChunk, &tmQ, &bar[Q_FULL], (h0 + x * dh) * D + c * 64,
                      (int)(q0 + x * dq));
      int i = 0;
      for (int b = nextb(0, -1); b >= 0; b = nextb(i + 1, b), ++i) {
        const int st = i % kKStages;
        if (i >= kKStages && !mbar_wait(&bar[KS + st], ((i - kKStages) / kKStages) & 1, abort_flag, 10)) break;
        mbar_expect_tx(&bar[K_FULL + st], 128 * D * 2);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sm + L::k0 + st * L::kTileB + c * L::kChunk, &tmK, &bar[K_FULL + st], g * D + c * 64, b * 128);
      }
      // every copy issued has landed before the CTA may leave
      mbar_drain(&bar[Q_FULL], 0, abort_flag);
      for (int j = i - 1; j >= 0 && j >= i - kKStages; --j) mbar_drain(&bar[K_FULL + j % kKStages], (j / kKStages) & 1, abort_flag);
    } else if (warp == 2 && lane == 0) {
      prefetch_tmap(&tmV);
      int i = 0;
      for (int b = nextb(0, -1); b >= 0; b = nextb(i + 1, b), ++i) {
        const int st = i % kVStages;
        if (i >= kVStages && !mbar_wait(&bar[VF + st], ((i - kVStages) / kVStages) & 1, abort_flag, 9)) break;
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
      const uint64_t dq0 = smem_desc(smem_u32(sm + L::q), 16, 1024);
      const uint64_t dk0 = smem_desc(smem_u32(sm + L::k0), 16, 1024);
      const uint64_t dv0 = smem_desc(smem_u32(sm + L::v0), L::kChunk, 1024);
      // S_x = Q_x · Kᵀ of the block in K stage st
      auto issue_s = [&](int x, int st) {
        const uint64_t dq = desc_at(dq0, x * L::kTileB), dk = desc_at(dk0, st * L::kTileB);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * L::kChunk + (k & 3) * 32;
          umma_ss(tbase + col_s(x), desc_at(dq, off), desc_at(dk, off), idS, k > 0);
        }
      };
      // O_x += P_x · V of the block in V stage st (P_x read from TMEM)
      auto issue_pv = [&](int x, int st, bool acc) {
        const uint64_t dv = desc_at(dv0, st * L::kTileB);
#pragma unroll
        for (int k = 0; k < 128 / 16; ++k)
          umma_ts(tbase + col_o(x), tbase + col_s(x) + k * 8, desc_at(dv, k * 2048), idPV, acc || k > 0);
      };
      bool ok = mbar_wait(&bar[Q_FULL], 0, abort_flag, 11);
      int b = nextb(0, -1);
      if (ok && b >= 0) {
        ok = mbar_wait(&bar[K_FULL], 0, abort_flag, 13);
        if (ok) {
          tc_fence_after();
          issue_s(0, 0);
          umma_commit(&bar[S0]);
          if (has1) issue_s(1, 0);
          umma_commit(&bar[KS]);
        }
      }
      for (int i = 0; ok && b >= 0; ++i) {
        const int bn = nextb(i + 1, b);
        const int sv = i % kVStages, sk = (i + 1) % kKStages;
        if (i == 1 && a.stall_ns && !mbar_wait(&bar[STALL], 0, abort_flag, 6, a.stall_ns)) { ok = false; break; }
        ok = mbar_wait(&bar[P_RDY], i & 1, abort_flag, 12) &&
             mbar_wait(&bar[V_FULL + sv], (i / kVStages) & 1, abort_flag, 8);
        if (!ok) break;
        tc_fence_after();
        issue_pv(0, sv, i > 0);
        if (bn >= 0) {
          if (!mbar_wait(&bar[K_FULL + sk], ((i + 1) / kKStages) & 1, abort_flag, 14)) { ok = false; break; }
          tc_fence_after();
          issue_s(0, sk);
          umma_commit(&bar[S0]);  // S_0 ready (and O_0 += P_0·V of block i done)
        }
        if (has1) {
          if (!mbar_wait(&bar[P_RDY + 1], i & 1, abort_flag, 15)) { ok = false; break; }
          tc_fence_after();
          issue_pv(1, sv, i > 0);
        }
        umma_commit(&bar[VF + sv]);  // V stage sv free
        if (bn >= 0) {
          if (has1) issue_s(1, sk);
          umma_commit(&bar[KS + sk]);  // S_1 ready; K stage sk free
        }
        b = bn;
      }
      // completes after every MMA of this CTA: O is final, nothing in flight
      // (waited for even after an abort: TMEM and shared memory must outlive the MMAs)
      umma_commit(&bar[FINAL]);
      mbar_drain(&bar[FINAL], 0, abort_flag);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------ softmax + epilogue
    // warps 4..7: tile 0, warps 8..11: tile 1; warp w reads TMEM lanes 32·(w % 4) ..
    const int x = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int hx = h0 + x * dh;
    const int64_t q = q0 + x * dq + r;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t ts = tbase + lane_base + col_s(x), to = tbase + lane_base + col_o(x);
    float m_used = -INFINITY, l = 0.f;
    int i = 0;
    bool ok = x == 0 || has1;
    for (int b = ok ? nextb(0, -1) : -1; b >= 0; b = nextb(i + 1, b), ++i) {
      // S_x of block i (this also means O_x += P_x·V of block i − 1 is done)
      ok = x == 0 ? mbar_wait(&bar[S0], i & 1, abort_flag, 16)
                  : mbar_wait(&bar[KS + i % kKStages], (i / kKStages) & 1, abort_flag, 17);
      if (!ok) break;
      tc_fence_after();
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
      // The uniform `full` test is taken once per block, the mask is applied
      // with selects, and four independent maxima shorten the dependency chain.
      // S arrives in two halves: the first half's mask and maximum overlap the
      // load of the second.
      const int4* sv = reinterpret_cast<const int4*>(sSend + (i % kVStages) * 128);
      // tree and packed chunks: col visible iff col <= dqk and q32 < send (path positions; q_off = 0 in tree mode)
      const int dqk = (int)(a.q_off + q - kb), q32 = (int)(a.q_off + q);
      int64_t lim = min(a.q_off + q - kb, a.nk - 1 - kb);  // chunk: col visible iff col <= lim
      const int cmax = (int)(lim < -1 ? -1 : (lim > 127 ? 127 : lim));
      // Tree mask, warp-uniform case: when the whole block precedes the warp's
      // 32 rows and no key's send falls inside them (the rows sit in one
      // subtree), every row of the warp sees the same keys, those whose send
      // passes the warp's last row. Lane l tests keys 4l..4l+3; ballot e has
      // bit l for key 4l+e, so column 32c+4j+e of a row is bit 8c+j of vb[e].
      bool uni = false;
      uint32_t vb[4] = {0u, 0u, 0u, 0u};
      if ((MODE == kTreeM || packed) && !full) {
        const int qf = (int)(a.q_off + q0 + x * dq) + wq * 32, ql = qf + 31;
        const int4 se = sv[lane];
        const int sj[4] = {se.x, se.y, se.z, se.w};
        bool mixed = false;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          mixed |= sj[e] > qf && sj[e] <= ql;
          vb[e] = __ballot_sync(0xffffffffu, sj[e] > ql);
        }
        uni = kb + 127 <= qf && !__any_sync(0xffffffffu, mixed);
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      uint32_t s[4][32];
      tmem_ld32(ts, s[0]);
      tmem_ld32(ts + 32, s[1]);
      tmem_ld_wait();
      tmem_pin(s[0]);
      tmem_pin(s[1]);
      tmem_ld32(ts + 64, s[2]);
      tmem_ld32(ts + 96, s[3]);
      // the full case on its own, so that its four chunks are one straight run of code
      if (full) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c == 2) {
            tmem_ld_wait();
            tmem_pin(s[2]);
            tmem_pin(s[3]);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j)
            mx4[j & 3] = fmax3f(mx4[j & 3], __uint_as_float(s[c][2 * j]), __uint_as_float(s[c][2 * j + 1]));
        }
      } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (c == 2) {
          tmem_ld_wait();
          tmem_pin(s[2]);
          tmem_pin(s[3]);
        }
        if ((MODE == kTreeM || packed) && uni) {
          if (((vb[0] & vb[1] & vb[2] & vb[3]) >> (8 * c) & 0xffu) == 0xffu) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              mx4[j & 3] = fmax3f(mx4[j & 3], __uint_as_float(s[c][2 * j]), __uint_as_float(s[c][2 * j + 1]));
          } else {
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              float v[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                v[e] = (vb[e] >> (8 * c + j4)) & 1u ? __uint_as_float(s[c][j4 * 4 + e]) : -INFINITY;
                s[c][j4 * 4 + e] = __float_as_uint(v[e]);
              }
              mx4[(j4 & 1) * 2] = fmax3f(mx4[(j4 & 1) * 2], v[0], v[1]);
              mx4[(j4 & 1) * 2 + 1] = fmax3f(mx4[(j4 & 1) * 2 + 1], v[2], v[3]);
            }
          }
        } else if (MODE == kTreeM || packed) {
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const int4 se = sv[c * 8 + j4];
            const int sj[4] = {se.x, se.y, se.z, se.w};
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int col = c * 32 + j4 * 4 + e;
              const bool vis = col <= dqk && q32 < sj[e];
              v[e] = vis ? __uint_as_float(s[c][j4 * 4 + e]) : -INFINITY;
              s[c][j4 * 4 + e] = __float_as_uint(v[e]);
            }
            mx4[(j4 & 1) * 2] = fmax3f(mx4[(j4 & 1) * 2], v[0], v[1]);
            mx4[(j4 & 1) * 2 + 1] = fmax3f(mx4[(j4 & 1) * 2 + 1], v[2], v[3]);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float v0 = (c * 32 + 2 * j) <= cmax ? __uint_as_float(s[c][2 * j]) : -INFINITY;
            const float v1 = (c * 32 + 2 * j + 1) <= cmax ? __uint_as_float(s[c][2 * j + 1]) : -INFINITY;
            s[c][2 * j] = __float_as_uint(v0);
            s[c][2 * j + 1] = __float_as_uint(v1);
            mx4[j & 3] = fmax3f(mx4[j & 3], v0, v1);
          }
        }
      }
      }
      const float mx = fmax3f(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3])) * a.scale_log2;
      bool resc = false;
      float alpha = 1.f;
      if (mx > m_used + kRescaleThreshold) {
        alpha = fast_exp2(m_used - mx);  // 0 on the first visible block
        l *= alpha;
        resc = i > 0;
        m_used = mx;
      }
      if (__any_sync(0xffffffffu, resc)) {
        const float f = resc ? alpha : 1.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(to + c * 32, o);
          tmem_ld_wait();
          tmem_pin(o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
          tmem_st32(to + c * 32, o);
        }
      }
      const float mu = m_used == -INFINITY ? 0.f : m_used;
      // p = exp2(s·scale·log2e − m), two lanes per packed fp32 instruction;
      // P (bf16 pairs) overwrites the first 64 columns of S_x
      const float2 c2 = make_float2(a.scale_log2, a.scale_log2), nm2 = make_float2(-mu, -mu);
      float2 rs2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 v = __ffma2_rn(make_float2(__uint_as_float(s[c][2 * j]), __uint_as_float(s[c][2 * j + 1])), c2, nm2);
          const float2 pp = make_float2(fast_exp2(v.x), fast_exp2(v.y));
          rs2 = __fadd2_rn(rs2, pp);
          pk[j] = pack_bf16(pp.x, pp.y);
        }
        tmem_st16(ts + c * 16, pk);
      }
      l += rs2.x + rs2.y;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[P_RDY + x]);
    }
    const int n = i;
    if (ok && n > 0 && mbar_wait(&bar[FINAL], 0, abort_flag, 18)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = a.o + q * (int64_t)a.hq * D + (int64_t)hx * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(to + c * 32, o);
        tmem_ld_wait();
        tmem_pin(o);
        if (q < a.nq) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
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
      if (q < a.nq) a.lse[(int64_t)hx * a.lse_ld + q] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
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

template <int D, int MODE>
int launch_fwd(FwdTc a, const void* q, const void* k, const void* v, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!make_tmap_bf16(&mq, q, (uint64_t)a.hq * D, a.nq, 128) || !make_tmap_bf16(&mk, k, (uint64_t)a.hkv * D, a.nk, 128) ||
      !make_tmap_bf16(&mv, v, (uint64_t)a.hkv * D, a.nk, 128))
    return TT_ERR_CUDA;
  const int smem = (int)FwdSmem<D>::total;
  auto kern = fwd_tc_kernel<D, MODE>;
  if (!smem_attr_set<fwd_tc_kernel<D, MODE>>(smem)) return TT_ERR_CUDA;
  // two query heads of a KV group share every K/V block: pair them; an odd
  // group's last head pairs adjacent query tiles instead (their CTAs first,
  // so that the head pairs' longest-first order fills the tail)
  const int64_t nT = (a.nq + 127) / 128;
  const int G = a.hq / a.hkv;
  a.n_adj = G % 2 ? (int)((nT + 1) / 2 * a.hkv) : 0;
  const unsigned grid = (unsigned)(a.n_adj + nT * a.hkv * (G / 2));
  {
    KtScope kt(TT_KT_FWD, st);
    kern<<<grid, kFwdWarps * 32, smem, st>>>(mq, mk, mv, a);
  }
  return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

}  // namespace

namespace {
// Paired tiles halve the CTA count. Measured on chunk forwards (32 query
// heads against a 5,120-key path): the paired grid is about 10 % faster from
// 0.6 of a wave on (one wave of paired CTAs beats two of single tiles), except
// just past a whole wave, where its second wave holds a few long CTAs and the
// single tiles, twice as many, spread more evenly (2–3 % alone); below 0.6 of
// a wave the single tiles (split over key ranges when that pays) win. On the
// path-at-a-time pass, whose second path stack fills part of a launch's tail,
// that band is narrower: ending it at 1.2 waves was 0.2 % faster than at
// 1.35, and 2–4 % faster than at 1.5 or 1.7 (two-tile packs of 1.4–1.7 waves).
bool pairs_fill_gpu(int64_t nq, int hq, int hkv) {
  const int64_t nT = (nq + 127) / 128;
  const int G = hq / hkv;
  const int64_t ctas = nT * hkv * (G / 2) + (G % 2 ? (nT + 1) / 2 * hkv : 0);
  const int64_t nsm = sm_count();
  if (ctas * 10 < nsm * 6) return false;
  if (ctas > nsm && ctas * 100 < nsm * 120) return false;
  return true;
}
bool use_pairs(int tiles, int64_t nq, int hq, int hkv) { return tiles == 0 ? pairs_fill_gpu(nq, hq, hkv) : tiles == 2; }
}  // namespace

// Entry points used by the C ABI (attn_api.cu).
int fwd_tree(const void* ws, const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t N, int Hq,
             int Hkv, int d, float scale, int32_t* err, cudaStream_t st, int tiles, uint64_t stall_ns) {
  if (!use_pairs(tiles, N, Hq, Hkv))
    return fwd_tree_1tile(ws, Q, K, V, O, LSE, N, Hq, Hkv, d, scale, err, st, stall_ns);
  const TreeWs Lw = tree_ws_layout(0, N);
  FwdTc a = {};
  a.nq = N; a.nk = N; a.q_off = 0; a.lse_ld = N;
  a.send = ws_at<int32_t>(ws, Lw.send);
  a.blk_min = ws_at<int32_t>(ws, Lw.blk_min);
  a.blk_max = ws_at<int32_t>(ws, Lw.blk_max);
  a.order = ws_at<int32_t>(ws, Lw.fwd_order);
  a.hdr = ws_at<int64_t>(ws, Lw.hdr);
  a.o = static_cast<__nv_bfloat16*>(O); a.lse = LSE; a.hq = Hq; a.hkv = Hkv;
  a.scale_log2 = scale * 1.4426950408889634f; a.err = err; a.stall_ns = stall_ns;
  return d == 64 ? launch_fwd<64, kTreeM>(a, Q, K, V, st) : launch_fwd<128, kTreeM>(a, Q, K, V, st);
}

int fwd_chunk(const void* q, int64_t C, int64_t s0, const void* k, const void* v, const int32_t* send,
              const int32_t* blk_max, void* o, float* lse, int64_t lse_ld, int Hq, int Hkv, int d, float scale,
              int32_t* err, cudaStream_t st, int tiles, int splits, uint64_t stall_ns) {
  if (splits > 0 || !use_pairs(tiles, C, Hq, Hkv))
    return fwd_chunk_1tile(q, C, s0, k, v, send, blk_max, o, lse, lse_ld, Hq, Hkv, d, scale, err, st, splits,
                           stall_ns);
  FwdTc a = {};
  a.nq = C; a.nk = s0 + C; a.q_off = s0; a.lse_ld = lse_ld; a.send = send; a.blk_max = blk_max;
  a.o = static_cast<__nv_bfloat16*>(o); a.lse = lse; a.hq = Hq; a.hkv = Hkv;
  a.scale_log2 = scale * 1.4426950408889634f; a.err = err; a.stall_ns = stall_ns;
  if (send) return d == 64 ? launch_fwd<64, kPackM>(a, q, k, v, st) : launch_fwd<128, kPackM>(a, q, k, v, st);
  return d == 64 ? launch_fwd<64, kChunkM>(a, q, k, v, st) : launch_fwd<128, kChunkM>(a, q, k, v, st);
}

}  // namespace tc
}  // namespace tt
