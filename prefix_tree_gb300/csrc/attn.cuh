// Internal entry points of the tensor-memory attention kernels, called by the
// C ABI (attn_api.cu), the path-at-a-time driver and the no-allocation chunk
// backward. Arguments are validated by the callers.
#pragma once

#include "common.cuh"

namespace tt {
namespace tc {

// Forward query tiles per CTA: 0 = chosen from the grid size (two tiles when
// the paired grid still gives every SM a CTA), 1 or 2 = fixed. stall_ns is a
// test hook (0 in normal calls): the MMA thread of each CTA waits that long
// on a barrier nothing arrives at before its second key block, so that a
// bounded wait expires in the middle of the pipeline.
int fwd_tree(const void* ws, const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t N, int Hq,
             int Hkv, int d, float scale, int32_t* err, cudaStream_t st, int tiles, uint64_t stall_ns = 0);
// Chunk mode: splits = key-range splits per tile on the one-tile schedule
// (0 = chosen from the launch size, 1..4 fixed). `send` (nullptr: query i of
// the chunk sees keys 0..s0+i) packs several sibling subtrees into one chunk:
// key k is visible to the query at path position p iff k <= p < send[k];
// send is indexed by path position, holds at least roundup(s0 + C, 128)
// entries, and only entries from 128·floor(s0/128) on are read (path keys
// among them hold >= s0 + C, chunk keys s0 + the end of their subtree within
// the chunk, and the padding past s0 + C holds 0); blk_max[b] is the maximum
// of send over 128-key block b (read for the blocks from floor(s0/128) on).
int fwd_chunk(const void* q, int64_t C, int64_t s0, const void* k, const void* v, const int32_t* send,
              const int32_t* blk_max, void* o, float* lse, int64_t lse_ld, int Hq, int Hkv, int d, float scale,
              int32_t* err, cudaStream_t st, int tiles, int splits = 0, uint64_t stall_ns = 0);
int fwd_tree_1tile(const void* ws, const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t N, int Hq,
                   int Hkv, int d, float scale, int32_t* err, cudaStream_t st, uint64_t stall_ns = 0);
int fwd_chunk_1tile(const void* q, int64_t C, int64_t s0, const void* k, const void* v, const int32_t* send,
                    const int32_t* blk_max, void* o, float* lse, int64_t lse_ld, int Hq, int Hkv, int d, float scale,
                    int32_t* err, cudaStream_t st, int splits = 0, uint64_t stall_ns = 0);

// Backward scratch: lse·log2 e and Σ_d dO·O per query row, [2][Hq][roundup(nq, 128)] fp32.
size_t bwd_ws_bytes(int64_t nq, int hq);
int bwd_tree(const void* ws, const void* Q, const void* K, const void* V, const void* O, const float* LSE,
             const void* dO, void* dQ, void* dK, void* dV, int64_t N, int Hq, int Hkv, int d, float scale,
             void* bws, int32_t* err, cudaStream_t st);
int bwd_chunk(const void* q, int64_t C, int64_t s0, const void* k, const void* v, const int32_t* send,
              const int32_t* blk_max, const void* o, const float* lse, int64_t lse_ld, const void* dO, void* dq,
              float* dk_acc, float* dv_acc, int Hq, int Hkv, int d, float scale, void* bws, int32_t* err,
              cudaStream_t st);

}  // namespace tc
}  // namespace tt
