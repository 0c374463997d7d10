// tcgen05 (5th-generation tensor core) kernels of the bf16 path: indexer scores and the gathered
// sparse attention, dispatched by the C ABI for bf16 storage with H = 64 / H_idx = 64.
#pragma once

#include <cuda.h>

#include "kernels.h"

namespace csa {

bool tc_index_available();                                    // the tcgen05 indexer is built
bool tc_attn_available();                                     // the tcgen05 attention is built
int tc_attn_split_len();                                      // candidates per attention CTA (decode)
int tc_attn_splits(int window, int top_k, int64_t n_cap, int rows);   // CTAs per query (rows = B * S)
size_t tc_workspace_bytes(int B, int S, int64_t n_cap, int top_k);
int tc_sm_count();

// 2-D bf16 tensor map over [rows][cols] with a 64-element x box_rows box and the 128-byte swizzle.
cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, int64_t rows, uint32_t cols, uint32_t box_rows);

// s_i = sum_h w_h relu(rope(q_h, t) . cidx_i) for i < visible(t), bf16 operands, fp32 accumulate.
// `close` (decode, S = 1; null otherwise): the compressor's close step for both caches (job[0] the
// 512-channel KV cache, job[1] the index cache) runs inside this kernel, before the scores that
// need it; the kernel is then the step's first and must not be a dependent launch.
cudaError_t tc_index_scores(int B, int S, const int64_t* pos, const void* q_idx, const float* w,
                            const void* cidx, int64_t n_cap, int ratio, const RopeTab& rope,
                            float* scores, void* ws, int32_t* err, cudaStream_t st, bool pdl,
                            const CompressParams* close = nullptr, int64_t entry_base = 0);

// Decode indexer and selection fused (S = 1): one cluster of C CTAs per request scores its visible
// entries and selects the top_k (ascending entry index, -1 padded) into topk [B, top_k]; scores
// [B, n_cap] is written only when non-null. `close`: as for tc_index_scores. `ckv_prefetch`
// (nullable): the compressed KV cache, whose selected rows are requested into L2 once selected.
// `test_stall`: the timeout test hook (csa.h, CSA_FLAG_TEST_STALL). `lowp`: cidx (and ckv_prefetch, and
// the entries the close step writes) are in the low-precision format of lowp.cuh.
// tc_index_select_cluster gives C for B requests of capacity n_cap, or 0 when the kernel does not apply.
int tc_index_select_cluster(int B, int64_t n_cap);
cudaError_t tc_index_select(int B, int C, const int64_t* pos, const void* q_idx, const float* w, const void* cidx,
                            int64_t n_cap, int ratio, int top_k, const RopeTab& rope, float* scores, int32_t* topk,
                            int32_t* err, cudaStream_t st, bool pdl, const CompressParams* close = nullptr,
                            const void* ckv_prefetch = nullptr, bool test_stall = false, bool lowp = false);

// Many-query attention (prefill): one CTA per query over all of its candidates (at most
// tc_attn_prefill_max_tiles() tiles of 128), final output written directly.
int tc_attn_prefill_max_tiles();
cudaError_t tc_attn_prefill(int B, const AttnParams& p, cudaStream_t st, bool pdl);

// Decode attention fused with the split merge, the sink and the inverse RoPE (S = 1, CSA top-k):
// one cluster of C CTAs per query, each with Wc window rows and Kc selection slots (R rows padded
// to 16), bf16 output written directly. tc_attn_fused_plan gives C (and the shares), or 0 when the
// kernel does not apply.
// The kernel exchanges its partials through `ws` (tc_attn_fused_workspace bytes).
int tc_attn_fused_plan(int B, int window, int top_k, int* Wc, int* Kc, int* R);
size_t tc_attn_fused_workspace(int B, int C);
// `lowp`: p.ckv is in the low-precision format of lowp.cuh (raw rows, q and out stay bf16).
cudaError_t tc_attn_fused(int B, int C, int Wc, int Kc, int R, const AttnParams& p, void* ws, cudaStream_t st,
                          bool pdl, bool lowp = false);

// Sparse attention (split partials when p.n_split > 1, else the final output).
cudaError_t tc_sparse_attn(int B, const AttnParams& p, void* ws, cudaStream_t st, bool pdl);

}  // namespace csa
