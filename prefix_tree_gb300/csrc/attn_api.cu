// C ABI of the tree-attention calls: host-side argument checks, then the
// tensor-memory (tcgen05 / TMEM / TMA) kernels of attn_tc*.cu.
//
// "Tree Training", Abstract: each token attends only to its root-to-token
// path, so the DFS-serialised tree reproduces independent per-branch causal
// attention exactly; with the DFS layout key k is an ancestor of query t iff
// k <= t < send[k]. AReaL-DTA, Key Contributions 1–2: chunk mode runs a query
// chunk at path offset s0 against a contiguous path K/V (query i sees keys
// 0..s0+i) and accumulates key/value gradients into the path; a packed chunk
// holds several sibling subtrees after their shared path, each token seeing
// the path and its own ancestors within the chunk (the same rule
// k <= p < send[k] over path positions).
#include "attn.cuh"

namespace tt {
namespace {

constexpr int64_t kRowSlack = 128;  // row indices stay below INT32_MAX with a tile of slack

int check_heads(int Hq, int Hkv, int d) {
  if (Hq < 1 || Hkv < 1) return TT_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return TT_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return TT_ERR_UNSUPPORTED;
  return TT_OK;
}

int tree_fwd(const void* ws, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V, tt_bf16* O, float* LSE, int64_t N,
             int Hq, int Hkv, int d, float scale, int32_t* err, tt_stream_t stream, int tiles,
             uint64_t stall_ns = 0) {
  int rc = check_heads(Hq, Hkv, d);
  if (rc) return rc;
  if (tiles < 0 || tiles > 2) return TT_ERR_INVALID_ARG;
  if (!ws || !Q || !K || !V || !O || !LSE || !err || N < 1 || N > INT32_MAX - kRowSlack) return TT_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return TT_ERR_INVALID_ARG;
  return tc::fwd_tree(ws, Q, K, V, O, LSE, N, Hq, Hkv, d, scale, err, reinterpret_cast<cudaStream_t>(stream), tiles,
                      stall_ns);
}

int chunk_fwd(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path, const tt_bf16* v_path,
              const int32_t* send, const int32_t* blk_max, tt_bf16* o, float* lse, int64_t lse_ld, int Hq, int Hkv,
              int d, float scale, int32_t* err, tt_stream_t stream, int tiles, int splits = 0) {
  int rc = check_heads(Hq, Hkv, d);
  if (rc) return rc;
  if (tiles < 0 || tiles > 2 || splits < 0 || splits > 4) return TT_ERR_INVALID_ARG;
  if (!q || !k_path || !v_path || !o || !lse || !err || C < 1 || s0 < 0 || lse_ld < C ||
      s0 + C > (int64_t)INT32_MAX - kRowSlack)
    return TT_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_path) || !aligned16(v_path) || !aligned16(o)) return TT_ERR_INVALID_ARG;
  if (send && (!aligned16(send) || !blk_max)) return TT_ERR_INVALID_ARG;
  return tc::fwd_chunk(q, C, s0, k_path, v_path, send, blk_max, o, lse, lse_ld, Hq, Hkv, d, scale, err,
                       reinterpret_cast<cudaStream_t>(stream), tiles, splits);
}

int chunk_bwd(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path, const tt_bf16* v_path,
              const int32_t* send, const int32_t* blk_max, const tt_bf16* o, const float* lse, int64_t lse_ld,
              const tt_bf16* dO, tt_bf16* dq, float* dk_acc, float* dv_acc, int Hq, int Hkv, int d, float scale,
              void* ws, size_t ws_bytes, int32_t* err, tt_stream_t stream) {
  int rc = check_heads(Hq, Hkv, d);
  if (rc) return rc;
  if (!q || !k_path || !v_path || !o || !lse || !dO || !dq || !dk_acc || !dv_acc || !ws || !err || C < 1 || s0 < 0 ||
      lse_ld < C || s0 + C > (int64_t)INT32_MAX - kRowSlack)
    return TT_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_path) || !aligned16(v_path) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk_acc) || !aligned16(dv_acc))
    return TT_ERR_INVALID_ARG;
  if (send && (!aligned16(send) || !blk_max)) return TT_ERR_INVALID_ARG;
  if (ws_bytes < tt_tree_attn_chunk_bwd_workspace_bytes(C, Hq)) return TT_ERR_WORKSPACE;
  if (!aligned16(ws)) return TT_ERR_INVALID_ARG;
  return tc::bwd_chunk(q, C, s0, k_path, v_path, send, blk_max, o, lse, lse_ld, dO, dq, dk_acc, dv_acc, Hq, Hkv, d,
                       scale, ws, err, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace tt

using namespace tt;

TT_API int tt_tree_attn_fwd(const void* ws, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V, tt_bf16* O,
                            float* LSE, int64_t N, int Hq, int Hkv, int d, float scale, int32_t* err,
                            tt_stream_t stream) {
  return tree_fwd(ws, Q, K, V, O, LSE, N, Hq, Hkv, d, scale, err, stream, 0);
}

TT_API int tt_tree_attn_fwd_tiles(const void* ws, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V, tt_bf16* O,
                                  float* LSE, int64_t N, int Hq, int Hkv, int d, float scale, int tiles,
                                  int32_t* err, tt_stream_t stream) {
  return tree_fwd(ws, Q, K, V, O, LSE, N, Hq, Hkv, d, scale, err, stream, tiles);
}

TT_API int tt_tree_attn_fwd_stall_test(const void* ws, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V,
                                       tt_bf16* O, float* LSE, int64_t N, int Hq, int Hkv, int d, float scale,
                                       int tiles, int64_t stall_ns, int32_t* err, tt_stream_t stream) {
  if (stall_ns < 1 || stall_ns > 10000000000LL) return TT_ERR_INVALID_ARG;
  return tree_fwd(ws, Q, K, V, O, LSE, N, Hq, Hkv, d, scale, err, stream, tiles, (uint64_t)stall_ns);
}

TT_API size_t tt_tree_attn_bwd_workspace_bytes(int64_t N, int Hq) {
  if (N < 1 || Hq < 1) return 0;
  return align_up(tc::bwd_ws_bytes(N, Hq), 256);
}

TT_API int tt_tree_attn_bwd(const void* ws, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V, const tt_bf16* O,
                            const float* LSE, const tt_bf16* dO, tt_bf16* dQ, tt_bf16* dK, tt_bf16* dV, int64_t N,
                            int Hq, int Hkv, int d, float scale, void* bwd_ws, size_t bwd_ws_bytes, int32_t* err,
                            tt_stream_t stream) {
  int rc = check_heads(Hq, Hkv, d);
  if (rc) return rc;
  if (!ws || !Q || !K || !V || !O || !LSE || !dO || !dQ || !dK || !dV || !bwd_ws || !err || N < 1 ||
      N > INT32_MAX - kRowSlack)
    return TT_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(dQ) ||
      !aligned16(dK) || !aligned16(dV))
    return TT_ERR_INVALID_ARG;
  if (bwd_ws_bytes < tt_tree_attn_bwd_workspace_bytes(N, Hq)) return TT_ERR_WORKSPACE;
  if (!aligned16(bwd_ws)) return TT_ERR_INVALID_ARG;
  return tc::bwd_tree(ws, Q, K, V, O, LSE, dO, dQ, dK, dV, N, Hq, Hkv, d, scale, bwd_ws, err,
                      reinterpret_cast<cudaStream_t>(stream));
}

TT_API int tt_tree_attn_chunk_fwd(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                  const tt_bf16* v_path, tt_bf16* o, float* lse, int64_t lse_ld, int Hq, int Hkv,
                                  int d, float scale, int32_t* err, tt_stream_t stream) {
  return chunk_fwd(q, C, s0, k_path, v_path, nullptr, nullptr, o, lse, lse_ld, Hq, Hkv, d, scale, err, stream, 0);
}

TT_API int tt_tree_attn_chunk_fwd_tiles(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                        const tt_bf16* v_path, tt_bf16* o, float* lse, int64_t lse_ld, int Hq,
                                        int Hkv, int d, float scale, int tiles, int32_t* err, tt_stream_t stream) {
  return chunk_fwd(q, C, s0, k_path, v_path, nullptr, nullptr, o, lse, lse_ld, Hq, Hkv, d, scale, err, stream, tiles);
}

TT_API int tt_tree_attn_chunk_fwd_split(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                        const tt_bf16* v_path, tt_bf16* o, float* lse, int64_t lse_ld, int Hq,
                                        int Hkv, int d, float scale, int splits, int32_t* err, tt_stream_t stream) {
  if (splits < 0 || splits > 4) return TT_ERR_INVALID_ARG;
  return chunk_fwd(q, C, s0, k_path, v_path, nullptr, nullptr, o, lse, lse_ld, Hq, Hkv, d, scale, err, stream, 1,
                   splits);
}

TT_API size_t tt_tree_attn_chunk_bwd_workspace_bytes(int64_t C, int Hq) {
  if (C < 1 || Hq < 1) return 0;
  return align_up(tc::bwd_ws_bytes(C, Hq), 256);
}

TT_API int tt_tree_attn_chunk_bwd(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                  const tt_bf16* v_path, const tt_bf16* o, const float* lse, int64_t lse_ld,
                                  const tt_bf16* dO, tt_bf16* dq, float* dk_acc, float* dv_acc, int Hq, int Hkv,
                                  int d, float scale, void* ws, size_t ws_bytes, int32_t* err, tt_stream_t stream) {
  return chunk_bwd(q, C, s0, k_path, v_path, nullptr, nullptr, o, lse, lse_ld, dO, dq, dk_acc, dv_acc, Hq, Hkv, d,
                   scale, ws, ws_bytes, err, stream);
}

TT_API int tt_tree_attn_chunk_fwd_packed(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                         const tt_bf16* v_path, const int32_t* send, const int32_t* blk_max,
                                         tt_bf16* o, float* lse, int64_t lse_ld, int Hq, int Hkv, int d, float scale,
                                         int32_t* err, tt_stream_t stream) {
  if (!send || !blk_max) return TT_ERR_INVALID_ARG;
  return chunk_fwd(q, C, s0, k_path, v_path, send, blk_max, o, lse, lse_ld, Hq, Hkv, d, scale, err, stream, 0);
}

TT_API int tt_tree_attn_chunk_bwd_packed(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                         const tt_bf16* v_path, const int32_t* send, const int32_t* blk_max,
                                         const tt_bf16* o, const float* lse, int64_t lse_ld, const tt_bf16* dO,
                                         tt_bf16* dq, float* dk_acc, float* dv_acc, int Hq, int Hkv, int d,
                                         float scale, void* ws, size_t ws_bytes, int32_t* err, tt_stream_t stream) {
  if (!send || !blk_max) return TT_ERR_INVALID_ARG;
  return chunk_bwd(q, C, s0, k_path, v_path, send, blk_max, o, lse, lse_ld, dO, dq, dk_acc, dv_acc, Hq, Hkv, d,
                   scale, ws, ws_bytes, err, stream);
}
