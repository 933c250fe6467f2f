/*
 * tt.h — C ABI of libtt, the GB300 (sm_103a) hot path of prefix-tree training.
 *
 * The method ("Tree Training: Accelerating Agentic LLMs Training via Shared
 * Prefix Reuse", Abstract; "AREAL-DTA: Dynamic Tree Attention for Efficient
 * Reinforcement Learning of Large Language Models", Key Contributions 1–2 and
 * "Methodology in Plain English"): the rollouts of one task form a prefix tree
 * of token segments; the tree is serialised in DFS order so every token is
 * computed exactly once; attention lets each token see only its root-to-token
 * path; the branch-average loss is the per-token loss weighted by the fraction
 * of branches through the token.
 *
 * Conventions shared by every call:
 *  - Pointers named *_host are host memory; every other pointer is DEVICE
 *    memory owned by the caller. The library never allocates, frees or
 *    retains caller memory, and keeps no state between calls (except the
 *    launch-timing records, off by default; see tt_kernel_timing).
 *  - bf16 tensors are passed as tt_bf16 (raw IEEE bfloat16 bits, uint16).
 *  - Attention tensors are token-major and contiguous: Q, O, dO, dQ are
 *    [rows][Hq][d]; K, V, dK, dV are [rows][Hkv][d]; LSE is [Hq][lse_ld]
 *    (lse_ld = N for whole-tree calls). Base pointers must be 16-byte
 *    aligned. Query head h uses key/value head h / (Hq / Hkv).
 *  - Supported head_dim d: 64 and 128. Hq % Hkv must be 0.
 *  - Every call is asynchronous on `stream` (NULL = legacy default stream)
 *    and returns a tt status: TT_OK once the work is enqueued, or a negative
 *    code for errors found on the host (nothing is enqueued then).
 *  - `err` is a caller-owned device int32 that kernels set (first error
 *    wins) when they detect an error in device data: invalid tree, target
 *    out of range, interval capacity too small. Zero it before a call, read
 *    it after synchronising; tt_status_string() names the code. Kernels never
 *    trap: a failed check writes `err` and the affected outputs are left
 *    unspecified (documented per call).
 *  - Scores are scale·q·k; LSE is the natural-log log-sum-exp of the scaled
 *    scores of the token's visible keys, in fp32.
 */
#ifndef TT_H_
#define TT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
#define TT_EXTERN extern "C"
#else
#define TT_EXTERN extern
#endif
#define TT_API TT_EXTERN __attribute__((visibility("default")))

typedef uint16_t tt_bf16;
typedef struct CUstream_st* tt_stream_t; /* identical to cudaStream_t */

enum {
  TT_OK = 0,
  TT_ERR_INVALID_ARG = -1,  /* bad pointer, size, stride, alignment or target id */
  TT_ERR_INVALID_TREE = -2, /* parent/length arrays do not form a topological tree */
  TT_ERR_UNSUPPORTED = -3,  /* head_dim or head grouping outside what the kernels cover */
  TT_ERR_WORKSPACE = -4,    /* workspace or interval capacity too small */
  TT_ERR_CUDA = -5,         /* a CUDA runtime call failed */
  TT_ERR_TIMEOUT = -6       /* a bounded device wait gave up */
};

/* Outputs of tt_tree_build: caller-allocated device arrays (all int32 unless
 * stated). S = number of segments, N = number of tokens. */
typedef struct tt_tree_out {
  int32_t* seg_start;       /* [S] DFS token offset of each segment */
  int32_t* seg_subtree_end; /* [S] end of the DFS span of the segment's subtree */
  int32_t* seg_depth;       /* [S] number of strict ancestor segments (root 0) */
  int32_t* seg_pathlen;     /* [S] tokens on the root path before the segment */
  int32_t* seg_leafcnt;     /* [S] leaves (childless segments) in the subtree */
  int32_t* iv_ptr;          /* [S+1] CSR offsets into iv, in interval pairs */
  int32_t* iv;              /* [2*iv_capacity] (begin, end) half-open DFS ranges */
  int32_t* tok_seg;         /* [N] segment of each token */
  int32_t* tok_pos;         /* [N] 0-based depth along the token's path (RoPE position) */
  int32_t* tok_send;        /* [N] subtree end of the token's segment: k is an
                               ancestor of t  <=>  k <= t < tok_send[k] */
  int32_t* tok_leafcnt;     /* [N] leaves below the token's segment (n_t) */
  float* tok_weight;        /* [N] fp32(n_t) / fp32(B), correctly rounded */
  int64_t* stats;           /* [8] B, N, sum of branch lengths, ancestor pairs,
                               non-empty 128x128 tile pairs, interval pairs,
                               max segment depth, max path length */
} tt_tree_out;

/* ---------------------------------------------------------------- tree build
 * DFS serialisation of a rollout tree ("Tree Training", Abstract: DFS
 * serialization; loss weight = fraction of branches through a token).
 * Input: seg_parent[S] (−1 for segment 0, else 0 <= parent < s), seg_len[S]
 * (>= 1, summing to N); children are visited in ascending segment index.
 * Writes every field of *out (a host struct of device pointers), and the
 * tile schedules the attention calls read into `ws` (size from
 * tt_tree_workspace_bytes; keep it alive and unmodified while attention
 * calls use it). The ancestor interval list of segment s is the merged,
 * ascending list of its root-to-s segments' ranges; a token t of s uses that
 * list with the last end clipped to t+1. If the list needs more than
 * iv_capacity pairs, `err` = TT_ERR_WORKSPACE, iv is not written and
 * stats[5] holds the pairs needed. An invalid tree sets `err` =
 * TT_ERR_INVALID_TREE; the outputs are then unspecified and attention calls
 * given this `ws` set the same error and write nothing. */
TT_API size_t tt_tree_workspace_bytes(int32_t S, int64_t N);
TT_API int tt_tree_build(const int32_t* seg_parent, const int32_t* seg_len, int32_t S, int64_t N,
                         const tt_tree_out* out, int64_t iv_capacity, void* ws, size_t ws_bytes,
                         int32_t* err, tt_stream_t stream);

/* The tile schedules a tree build wrote into `ws`, copied into caller device
 * arrays for inspection (any pointer may be NULL to skip it). With nT =
 * ceil(N / 128) query tiles and key blocks of 128 rows: send[nT·128] =
 * tok_send zero-padded to whole blocks; blk_min[nT], blk_max[nT] = min / max
 * of send over each block's real keys; fwd_cnt[T] = key blocks with an
 * ancestor pair for query tile T; bwd_cnt[b] = query tiles with an ancestor
 * pair for key block b; fwd_order / bwd_order = tiles / blocks by decreasing
 * count, ties by increasing index (the order in which the attention kernels'
 * CTAs take them). N must be the N of the build. Asynchronous on `stream`. */
TT_API int tt_tree_schedules(const void* ws, int64_t N, int32_t* send, int32_t* blk_min, int32_t* blk_max,
                             int32_t* fwd_cnt, int32_t* fwd_order, int32_t* bwd_cnt, int32_t* bwd_order,
                             tt_stream_t stream);

/* ---------------------------------------------------------- tree attention
 * Forward ("Tree Training", Abstract: attention adapted so each token's
 * result equals independent per-branch causal attention):
 *   O_t = Σ_{k ∈ anc(t)} softmax_k(scale·q_t·k_k) v_k,  LSE_t in fp32,
 * with anc(t) the root-to-t path (including t). ws = the tree's workspace. */
TT_API int tt_tree_attn_fwd(const void* ws, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V,
                            tt_bf16* O, float* LSE, int64_t N, int Hq, int Hkv, int d, float scale,
                            int32_t* err, tt_stream_t stream);

/* Same as tt_tree_attn_fwd with the forward schedule fixed: tiles = 1 runs
 * one 128-row query tile per CTA, tiles = 2 two tiles per CTA (two query
 * heads of a KV group; an odd group's last head takes two adjacent query
 * tiles), tiles = 0 chooses as tt_tree_attn_fwd does (two tiles from 0.6 of
 * a wave of paired CTAs on, except between 1.0 and 1.2 waves, where the
 * single tiles' second wave is better filled). For tuning and for tests that
 * run both schedules on the same inputs; any other value returns
 * TT_ERR_INVALID_ARG. */
TT_API int tt_tree_attn_fwd_tiles(const void* ws, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V, tt_bf16* O,
                                  float* LSE, int64_t N, int Hq, int Hkv, int d, float scale, int tiles,
                                  int32_t* err, tt_stream_t stream);

/* Test of the timeout path (no counterpart on the pages): runs
 * tt_tree_attn_fwd_tiles, except that the MMA-issuing thread of every CTA
 * waits, before its second key block, on a barrier that nothing arrives at,
 * with a limit of stall_ns nanoseconds (1 .. 10^10) instead of the normal 2 s.
 * The wait expires; the CTA's other roles stop at their next wait, every TMA
 * copy and tensor-core operation already issued is waited for, tensor memory
 * is freed, and `err` receives TT_ERR_TIMEOUT. O and LSE are unspecified
 * afterwards; the context and stream stay usable. A CTA with a single key
 * block never reaches the stall and finishes normally. */
TT_API int tt_tree_attn_fwd_stall_test(const void* ws, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V,
                                       tt_bf16* O, float* LSE, int64_t N, int Hq, int Hkv, int d, float scale,
                                       int tiles, int64_t stall_ns, int32_t* err, tt_stream_t stream);

/* Backward (AReaL-DTA, Key Contributions 1: a shared prefix is
 * backpropagated once with the gradients of all descendant leaves): the VJP
 * of Σ_t <dO_t, O_t>; dK/dV of a prefix token sum over every descendant
 * query (and over the query heads of its group). Overwrites dQ, dK, dV
 * (bf16; fp32 accumulation). O and LSE are the forward's outputs.
 * bwd_ws: scratch of tt_tree_attn_bwd_workspace_bytes(N, Hq) bytes. */
TT_API size_t tt_tree_attn_bwd_workspace_bytes(int64_t N, int Hq);
TT_API int tt_tree_attn_bwd(const void* ws, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V,
                            const tt_bf16* O, const float* LSE, const tt_bf16* dO, tt_bf16* dQ,
                            tt_bf16* dK, tt_bf16* dV, int64_t N, int Hq, int Hkv, int d, float scale,
                            void* bwd_ws, size_t bwd_ws_bytes, int32_t* err, tt_stream_t stream);

/* ------------------------------------------------------ chunk-vs-path mode
 * Path-at-a-time attention (AReaL-DTA, Key Contributions 1–2): a chunk of C
 * query rows sitting at path positions s0 .. s0+C−1 attends to the first
 * s0+C rows of a contiguous path K/V (the chunk's own keys are the last C
 * rows): query i sees path keys 0 .. s0+i.
 *   q, o: [C][Hq][d];  k_path, v_path: [s0+C][Hkv][d];  lse: [Hq][lse_ld].
 * The backward writes dq (bf16) and ACCUMULATES (+=) fp32 dk_acc, dv_acc
 * [s0+C][Hkv][d], so chunks processed right to left and descendant leaves
 * sum into the shared path prefix. ws: tt_tree_attn_chunk_bwd_workspace_bytes. */
TT_API int tt_tree_attn_chunk_fwd(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                  const tt_bf16* v_path, tt_bf16* o, float* lse, int64_t lse_ld, int Hq,
                                  int Hkv, int d, float scale, int32_t* err, tt_stream_t stream);
/* tt_tree_attn_chunk_fwd with the forward schedule fixed (tiles as in
 * tt_tree_attn_fwd_tiles). */
TT_API int tt_tree_attn_chunk_fwd_tiles(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                        const tt_bf16* v_path, tt_bf16* o, float* lse, int64_t lse_ld, int Hq,
                                        int Hkv, int d, float scale, int tiles, int32_t* err, tt_stream_t stream);
/* tt_tree_attn_chunk_fwd on the one-tile schedule with each tile's key range
 * split over `splits` CTAs of a thread-block cluster (1 <= splits <= 4; 0 =
 * chosen from the launch size, as tt_tree_attn_chunk_fwd does when the
 * paired schedule would not fill the GPU). The CTAs' partial softmax results
 * are merged in distributed shared memory (max, rescaled sums); O and LSE
 * agree with the unsplit call up to fp32 rounding. Returns
 * TT_ERR_INVALID_ARG for splits outside 0..4 and TT_ERR_UNSUPPORTED if the
 * device cannot co-schedule a cluster of that size. */
TT_API int tt_tree_attn_chunk_fwd_split(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                        const tt_bf16* v_path, tt_bf16* o, float* lse, int64_t lse_ld, int Hq,
                                        int Hkv, int d, float scale, int splits, int32_t* err, tt_stream_t stream);
TT_API size_t tt_tree_attn_chunk_bwd_workspace_bytes(int64_t C, int Hq);
TT_API int tt_tree_attn_chunk_bwd(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                  const tt_bf16* v_path, const tt_bf16* o, const float* lse, int64_t lse_ld,
                                  const tt_bf16* dO, tt_bf16* dq, float* dk_acc, float* dv_acc, int Hq,
                                  int Hkv, int d, float scale, void* ws, size_t ws_bytes, int32_t* err,
                                  tt_stream_t stream);

/* Packed chunk: the C chunk rows are several sibling subtrees laid out one
 * after the other behind their shared path of s0 rows (for example a run of
 * leaves of one segment, or a tree partition of tt_tree_partition, as the
 * DFS layout stores them), and each query sees the path and its own
 * ancestors within the chunk only — the tree rule of "Tree Training",
 * Abstract (key k is visible to the query at path position p iff
 * k <= p < send[k]), over path positions.
 *   send: device int32, indexed by path position, at least
 *         roundup(s0 + C, 128) entries, 16-byte aligned. Entries from
 *         128·floor(s0/128) on are read: those below s0 (path keys) must be
 *         >= s0 + C; entry s0 + i (chunk row i) is s0 + the end (exclusive,
 *         within the chunk) of the subtree of the segment holding row i (for
 *         a leaf, the end of the leaf), which exceeds its own index; entries
 *         from s0 + C on must be 0. Entries below 128·floor(s0/128) are never
 *         read.
 *   blk_max: device int32, one entry per 128-key block b (key positions
 *         128·b .. 128·b + 127): the maximum of those send entries; entries
 *         floor(s0/128) .. ceil((s0 + C)/128) − 1 are read.
 * The caller owns both; they are not validated on the device (a wrong value
 * gives wrong results, not a fault: every read stays inside the entries
 * above, and every range derived from them is clamped to the chunk).
 * Everything else as tt_tree_attn_chunk_fwd / tt_tree_attn_chunk_bwd: the
 * same layouts, the same dk_acc / dv_acc accumulation over all s0 + C rows,
 * the same workspace. With one segment spanning the chunk the results equal
 * the unpacked calls up to fp32 rounding. send or blk_max == NULL returns
 * TT_ERR_INVALID_ARG. */
TT_API int tt_tree_attn_chunk_fwd_packed(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                         const tt_bf16* v_path, const int32_t* send, const int32_t* blk_max,
                                         tt_bf16* o, float* lse, int64_t lse_ld, int Hq, int Hkv, int d, float scale,
                                         int32_t* err, tt_stream_t stream);
TT_API int tt_tree_attn_chunk_bwd_packed(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                         const tt_bf16* v_path, const int32_t* send, const int32_t* blk_max,
                                         const tt_bf16* o, const float* lse, int64_t lse_ld, const tt_bf16* dO,
                                         tt_bf16* dq, float* dk_acc, float* dv_acc, int Hq, int Hkv, int d,
                                         float scale, void* ws, size_t ws_bytes, int32_t* err, tt_stream_t stream);

/* Chunk backward that allocates nothing. The pages have no counterpart for
 * this call: it is for callers that cannot allocate device memory when they
 * call, such as a runtime that owns every device allocation through its own
 * pool, or a latency path that cannot afford cudaMalloc's implicit device
 * synchronisation. Same arguments and results as tt_tree_attn_chunk_bwd
 * without the workspace: its scratch (2 · Hq · roundup(C, 128) floats) lives
 * in a 2 MiB static device array that every GPU loading the library holds
 * until the process exits. Limit: Hq · roundup(C, 128) <= 262144 (for example
 * C <= 4096 at Hq <= 64); larger calls return TT_ERR_WORKSPACE and enqueue
 * nothing. The first call on a device looks up the array's device address
 * (once per device, with that device current); make that first call before
 * any stream capture. The looked-up address is cached per device and not
 * refreshed after cudaDeviceReset: do not call this entry point after a
 * reset in the same process. All calls share the array and each call
 * rewrites what it reads, so it needs no clearing; calls that overlap on the
 * GPU (other streams, other host threads) race on it. */
TT_API int tt_tree_attn_chunk_bwd_noalloc(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                          const tt_bf16* v_path, const tt_bf16* o, const float* lse, int64_t lse_ld,
                                          const tt_bf16* dO, tt_bf16* dq, float* dk_acc, float* dv_acc, int Hq,
                                          int Hkv, int d, float scale, int32_t* err, tt_stream_t stream);

/* Whole-tree attention forward + backward by path-at-a-time traversal
 * (AReaL-DTA, "Methodology in Plain English"): segments are visited in DFS
 * order with their root path kept as a contiguous K/V stack; entering a
 * segment forwards its tokens in chunks of at most `chunk` queries; leaving
 * it (after all descendants) backpropagates those chunks right to left, and
 * its key/value gradients are then complete and written out. Produces the
 * same O, LSE, dQ, dK, dV as tt_tree_attn_fwd + tt_tree_attn_bwd. Children
 * are entered in the greedy order (TT_DTA_ORDER_GREEDY below).
 * Packs: each run of consecutive leaf children of a segment is cut into
 * packs of leaves that lie next to each other in the DFS layout (at most
 * `chunk` rows and 32 leaves each), and a pack of two or more leaves runs as
 * one packed chunk (tt_tree_attn_chunk_fwd_packed / _bwd_packed) behind the
 * shared path: the same attention pairs, fewer and fuller launches.
 * Slots: the packs of a run are spread over `slots` path stacks (pack i of
 * the run on slot i mod slots), and when a segment's children are balanced
 * (no child subtree or pack holds more than half of their attention work) all
 * of them are spread at once, longest first onto the least-loaded stack. Each
 * stack has its own K/V copy of the path and fp32 gradient accumulators and
 * its own stream; afterwards the stacks' sums over the shared prefix are
 * added into stack 0 in stack order, so the results do not depend on timing
 * (they differ from another slot count or chunk size only in the order of
 * fp32 sums). Scratch per slot: a stack of max(longest root-to-leaf path,
 * a parent's path + one chunk of its leaves) rows; slots = 1 is the
 * one-stack traversal. tt_dta_tree_attn and tt_dta_tree_attn_ordered use
 * TT_DTA_DEFAULT_SLOTS.
 * seg_parent_host / seg_len_host: the tree on the host (same rules as
 * tt_tree_build; an invalid tree returns TT_ERR_INVALID_TREE before any
 * work). ws: tt_dta_workspace_bytes(...) bytes of device scratch
 * (tt_dta_workspace_bytes_slots for another slot count, 1..8; 0 for an
 * invalid tree or argument). */
enum { TT_DTA_DEFAULT_SLOTS = 2 };
TT_API size_t tt_dta_workspace_bytes(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S,
                                     int64_t chunk, int Hq, int Hkv, int d);
TT_API size_t tt_dta_workspace_bytes_slots(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S,
                                           int64_t chunk, int Hq, int Hkv, int d, int slots);
TT_API int tt_dta_tree_attn(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int64_t N,
                            int64_t chunk, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V,
                            const tt_bf16* dO, tt_bf16* O, float* LSE, tt_bf16* dQ, tt_bf16* dK, tt_bf16* dV,
                            int Hq, int Hkv, int d, float scale, void* ws, size_t ws_bytes, int32_t* err,
                            tt_stream_t stream);
/* Visiting orders of the traversal (AReaL-DTA, "Key Contributions" 2 and
 * "Methodology in Plain English": visits reordered so that each leaf and the
 * next one have the longest possible common prefix). Every DFS order gives consecutive leaves
 * the same total shared prefix, so the greedy rule only settles ties: GREEDY
 * (the order of tt_dta_tree_attn) enters, at every segment, the child whose
 * subtree holds the deepest leaf (most tokens on its root path) first, ties by
 * the lower index of that leaf; INDEX enters children in ascending segment
 * index (the order of the DFS layout). Results are the same up to the order
 * of the fp32 gradient accumulations. */
enum { TT_DTA_ORDER_INDEX = 0, TT_DTA_ORDER_GREEDY = 1 };
/* tt_dta_tree_attn with the visiting order chosen (TT_DTA_ORDER_*; any other
 * value returns TT_ERR_INVALID_ARG). */
TT_API int tt_dta_tree_attn_ordered(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int64_t N,
                                    int64_t chunk, int order, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V,
                                    const tt_bf16* dO, tt_bf16* O, float* LSE, tt_bf16* dQ, tt_bf16* dK, tt_bf16* dV,
                                    int Hq, int Hkv, int d, float scale, void* ws, size_t ws_bytes, int32_t* err,
                                    tt_stream_t stream);
/* tt_dta_tree_attn with the visiting order and the slot count (1..8; other
 * values return TT_ERR_INVALID_ARG) chosen; ws of
 * tt_dta_workspace_bytes_slots(..., slots) bytes. */
TT_API int tt_dta_tree_attn_slots(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int64_t N,
                                  int64_t chunk, int order, int slots, const tt_bf16* Q, const tt_bf16* K,
                                  const tt_bf16* V, const tt_bf16* dO, tt_bf16* O, float* LSE, tt_bf16* dQ,
                                  tt_bf16* dK, tt_bf16* dV, int Hq, int Hkv, int d, float scale, void* ws,
                                  size_t ws_bytes, int32_t* err, tt_stream_t stream);
/* A plan of the path-at-a-time pass: tt_dta_tree_attn_slots's device work
 * for one tree, chunk size, order, slot count, set of buffers, scale and err
 * word, captured once into a CUDA graph (the slots' streams become parallel
 * branches). tt_dta_plan_launch enqueues the whole
 * pass on `stream` with one call (no host work per segment); results are
 * those of tt_dta_tree_attn_slots with the same arguments, bitwise. The
 * pointers are baked in: the buffers must stay allocated and keep their
 * addresses while the plan exists, and new inputs are written into them.
 * Create and launch with the device current that owns the buffers (a launch
 * with another current device returns TT_ERR_INVALID_ARG). Creation enqueues
 * nothing and runs no kernel; it returns the errors of
 * tt_dta_tree_attn_slots's host checks, or TT_ERR_CUDA if the capture or
 * the graph instantiation fails. Launches of a plan are not timed by
 * tt_kernel_timing. tt_dta_plan_destroy frees the graph (NULL is a no-op);
 * a plan must not be destroyed while a launch of it may still run. */
typedef struct tt_dta_plan_s* tt_dta_plan;
TT_API int tt_dta_plan_create(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int64_t N,
                              int64_t chunk, int order, int slots, const tt_bf16* Q, const tt_bf16* K,
                              const tt_bf16* V, const tt_bf16* dO, tt_bf16* O, float* LSE, tt_bf16* dQ, tt_bf16* dK,
                              tt_bf16* dV, int Hq, int Hkv, int d, float scale, void* ws, size_t ws_bytes,
                              int32_t* err, tt_dta_plan* plan_out);
TT_API int tt_dta_plan_launch(tt_dta_plan plan, tt_stream_t stream);
TT_API int tt_dta_plan_destroy(tt_dta_plan plan);
/* The leaves (segment ids) in the order the traversal reaches them. Host
 * memory; returns the number of leaves written, TT_ERR_INVALID_TREE,
 * TT_ERR_INVALID_ARG (unknown order) or TT_ERR_WORKSPACE (capacity too small
 * or leaves_host NULL). */
TT_API int tt_dta_leaf_order(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int order,
                             int32_t* leaves_host, int32_t capacity);
/* Redundancy-free tree partitioning ("Tree Training", Abstract: a tree too
 * large for GPU memory is split so that no attention pair is computed twice
 * and the device holds at most one root-to-leaf path; the pages give no
 * algorithm, the rule is this library's): the partitions the path-at-a-time traversal
 * processes for a token budget (its `chunk`). A subtree is packable when it
 * holds at most `budget` rows and 64 segments. If the root's subtree is
 * packable, the whole tree is one partition with an empty path. Otherwise
 * every segment that is not packable contributes its own rows in chunks of
 * at most `budget` (kind 1: chunk i of the segment attends to the segment's
 * root path and the segment's earlier rows), and the children of such a
 * segment, in `order`, are taken in runs of consecutive packable children,
 * each run cut into packs of whole sibling subtrees adjacent in the DFS
 * layout (taken in layout order), at most `budget` rows and 64 segments per
 * pack (kind 0: a packed chunk behind the parent's root path). Every row lies
 * in exactly one partition and attends only to its root path and its own
 * partition, so each ancestor pair is computed once, and a partition needs
 * its path plus at most `budget` rows on the device.
 * Partition i (in DFS layout order): rows first_host[i] .. + rows_host[i]
 * of the layout, path_host[i] rows of cached root path before them,
 * kind_host[i]. Returns the number of partitions; with capacity 0 and all
 * four arrays NULL it only counts them. TT_ERR_INVALID_TREE,
 * TT_ERR_INVALID_ARG (budget < 1, unknown order, an array NULL) or
 * TT_ERR_WORKSPACE (capacity too small). Host only. */
TT_API int tt_tree_partition(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int64_t budget,
                             int order, int64_t* first_host, int64_t* rows_host, int64_t* path_host,
                             int32_t* kind_host, int32_t capacity);

/* -------------------------------------------------- weighted log-prob loss
 * ("Tree Training", Abstract: branch-average loss == per-token weighted loss)
 *   lse_t = log Σ_v exp(z_tv);  logp_t = z_{t,y_t} − lse_t;
 *   loss  = −Σ_t w_t logp_t  (fp64, fixed-order reduction: deterministic);
 *   dlogits_tv = g·w_t·(exp(z_tv − lse_t) − [v == y_t])  (bf16).
 * logits: [N][ld] bf16 rows (ld >= V); targets int32 [N]; weights fp32 [N]
 * (NULL = all ones); logp fp32 [N]; loss: one device double; dlogits [N][ld]
 * or NULL for the forward only. A target outside [0, V) sets `err` =
 * TT_ERR_INVALID_ARG and that row's logp (hence the loss) to NaN; its
 * dlogits row then omits the one-hot term.
 * Execution: with 16-byte aligned rows (ld a multiple of 8), each row is
 * split over a thread-block cluster; when the resident clusters leave SMs
 * idle and N is at least four rows per SM, the last rows of the batch run on
 * those SMs, on a library-owned stream that the call forks from `stream` and
 * joins back before it returns (work queued on `stream` afterwards sees every
 * row). While `stream` is being captured into a graph the clusters take all
 * rows. Which rows run where depends only on N, V and the device, so repeated
 * calls give bitwise-equal results. */
TT_API int tt_weighted_logprob(const tt_bf16* logits, int64_t N, int64_t V, int64_t ld, const int32_t* targets,
                               const float* weights, float g, float* logp, double* loss, tt_bf16* dlogits,
                               int32_t* err, tt_stream_t stream);

/* ---------------------------------------------------------------- trie build (host)
 * The step before tt_tree_build: the prefix tree of a task's rollouts from
 * their token sequences ("Tree Training", Abstract: a task's tokens form a
 * tree with shared prefixes; AReaL-DTA "Main Findings": rollouts that are
 * prefixes of others are collapsed, fully-contained prefix sequences merged).
 * Host memory throughout; no GPU work. Input: R >= 1 rollouts, rollout r =
 * tokens_host[offsets_host[r] .. offsets_host[r+1]) (offsets_host[0] = 0,
 * every rollout non-empty, all sharing their first token). A node is a
 * distinct prefix; children are ordered by first appearance (rollout order,
 * then position); a segment is a maximal chain of nodes in which every node
 * but the last has one child (a rollout ending inside a chain does not split
 * it); segments are numbered in DFS preorder, so the outputs are valid
 * tt_tree_build inputs and its DFS token order equals tok_host.
 * Outputs (arrays of `capacity` entries; capacity = offsets_host[R] always
 * suffices): seg_parent_host[S], seg_len_host[S], tok_host[N] (token ids in
 * DFS order); rollout_end_host[R] = DFS index of each rollout's last token;
 * counts_host[4] = {S, N, total tokens Σ rollout lengths, leaf tokens Σ
 * lengths of the distinct rollouts that are not prefixes of others}.
 * Returns TT_OK; TT_ERR_INVALID_ARG (bad pointer or offsets[0] != 0);
 * TT_ERR_INVALID_TREE (an empty rollout, or rollouts with different first
 * tokens); TT_ERR_WORKSPACE if S or N exceeds capacity (counts_host and
 * rollout_end_host are still written). */
TT_API int tt_trie_build(const int32_t* tokens_host, const int64_t* offsets_host, int32_t R, int64_t capacity,
                         int32_t* seg_parent_host, int32_t* seg_len_host, int32_t* tok_host,
                         int64_t* rollout_end_host, int64_t* counts_host);

/* ------------------------------------ LM head fused with the weighted log-prob
 * ("Tree Training", Abstract: every token's log-probability once, weighted by
 * the share of branches through it; the LM head in front is the plain product
 * z = H·Wᵀ). The logits are formed tile by tile on the tensor cores and never
 * written to memory:
 *   z_tv = <H_t, W_v>;  lse_t = log Σ_v exp(z_tv);  logp_t = z_{t,y_t} − lse_t;
 *   loss = −Σ_t w_t logp_t  (fp64, fixed-order reduction: deterministic).
 * hidden: [N][Hd] bf16 rows; w_vocab: [V][Hd] bf16 rows (a linear layer's
 * weight layout); Hd a multiple of 64; both 16-byte aligned. targets int32
 * [N]; weights fp32 [N] (NULL = all ones); logp fp32 [N]; lse fp32 [N] or
 * NULL; loss: one device double. ws: device scratch of
 * tt_lmhead_logprob_workspace_bytes(N, V) bytes (per-row partial log-sum-exp
 * of every 256-entry vocabulary tile: 8·N·ceil(V/256) bytes + 4·N), 16-byte
 * aligned. A target outside [0, V) sets `err` = TT_ERR_INVALID_ARG and that
 * row's logp (hence the loss) to NaN. Returns TT_ERR_UNSUPPORTED when Hd is
 * not a multiple of 64. */
TT_API size_t tt_lmhead_logprob_workspace_bytes(int64_t N, int64_t V);
TT_API int tt_lmhead_logprob(const tt_bf16* hidden, const tt_bf16* w_vocab, int64_t N, int64_t V, int Hd,
                             const int32_t* targets, const float* weights, float* logp, float* lse, double* loss,
                             void* ws, size_t ws_bytes, int32_t* err, tt_stream_t stream);
/* Backward of tt_lmhead_logprob: the gradients of g·loss,
 *   dz_tv = g·w_t·(exp(z_tv − lse_t) − [v == y_t]),
 *   d_hidden = dz·W  ([N][Hd] bf16, written),  d_w_vocab = dzᵀ·H  ([V][Hd] fp32, written).
 * lse: the forward's [N] output. Three tensor-core GEMMs; dz is the one
 * intermediate kept, in ws (bf16 [N][V rounded up to 8]:
 * tt_lmhead_logprob_bwd_workspace_bytes(N, V) bytes, 16-byte aligned; 3.85 GB
 * at N = 12,669, V = 151,936). Same argument rules as the forward; a target
 * outside [0, V) sets `err` = TT_ERR_INVALID_ARG and its row's dz omits the
 * one-hot term. */
TT_API size_t tt_lmhead_logprob_bwd_workspace_bytes(int64_t N, int64_t V);
TT_API int tt_lmhead_logprob_bwd(const tt_bf16* hidden, const tt_bf16* w_vocab, int64_t N, int64_t V, int Hd,
                                 const int32_t* targets, const float* weights, float g, const float* lse,
                                 tt_bf16* d_hidden, float* d_w_vocab, void* ws, size_t ws_bytes, int32_t* err,
                                 tt_stream_t stream);

/* ---------------------------------------------------------------- launch timing
 * A measurement aid, off by default, and the one state the library keeps
 * between calls. While on, every launch of the kernels below is bracketed by
 * two CUDA events recorded on the stream it runs on, so that a caller can
 * time one kernel class inside larger calls (the path-at-a-time driver's
 * chunk launches). Classes: TT_KT_FWD (attention forward, whole-tree and
 * chunk), TT_KT_BWD (the attention backward's main kernel, whose dQ and
 * dK/dV CTAs share one launch; its small pre-kernel is not timed),
 * TT_KT_LOGPROB (the weighted log-prob kernel), TT_KT_LMHEAD (the LM-head GEMM
 * kernels, forward and backward; the forward's small combine kernel is not
 * timed).
 * tt_kernel_timing(1) clears the records and turns timing on; (0) turns it
 * off and keeps the records. tt_kernel_timing_read waits for the recorded
 * events and writes, for classes c < n, the summed event time ms_host[c]
 * (milliseconds) and launch count launches_host[c] of the records since the
 * last tt_kernel_timing(1); launches beyond 65536 records (or whose events
 * could not be recorded) are not timed and are counted in *dropped_host
 * (may be NULL). Host arrays; returns TT_OK, TT_ERR_INVALID_ARG or
 * TT_ERR_CUDA. Not meant for concurrent use from several host threads. */
enum { TT_KT_FWD = 0, TT_KT_BWD = 1, TT_KT_LOGPROB = 2, TT_KT_LMHEAD = 3, TT_KT_CLASSES = 4 };
TT_API int tt_kernel_timing(int on);
TT_API int tt_kernel_timing_read(double* ms_host, int64_t* launches_host, int n, int64_t* dropped_host);

/* Name of a status code (static string). */
TT_API const char* tt_status_string(int code);
/* ABI version of this header (major*100 + minor). */
TT_API int tt_version(void);

#endif /* TT_H_ */
