// Internal launch interface of the CSA / HCA kernels (not part of the C ABI).
#pragma once

#include "common.cuh"

namespace csa {

// ------------------------------------------------------------------ K1 compressor
struct CompressJob {
  const void* src;       // [B, N, C] raw rows
  const void* gate;      // [B, N, C] gate logits
  const float* bias;     // [2m, C]
  void* dst;             // [B, n_cap, C]
  int C;                 // 512 (kv) or 128 (index keys)
};

struct CompressParams {
  CompressJob job[2];    // job[1] used when n_jobs == 2
  int n_jobs;
  int64_t N, n_cap;
  int64_t first_entry, n_entries;   // range mode
  const int64_t* pos;    // close mode when non-null: entry pos[b]/m if (pos[b]+1) % m == 0
  int ratio;
  int epb;               // range mode: entries per CTA (set by the launcher)
  float eps;
  RopeTab rope;
  int32_t* err;
};

// Storage of the compressed caches: float32, bf16, or the low-precision format of lowp.cuh (FP4 E2M1
// latent + FP8 E4M3 tail, raw rows in bf16).
enum StoreKind { kStoreF32 = 0, kStoreBf16 = 1, kStoreLowp = 2 };

// `pdl`: launch as a programmatic dependent of the previous kernel in the stream.
cudaError_t launch_compress(int kind, int B, const CompressParams& p, cudaStream_t st, bool pdl);

// Low-precision caches -> bf16 [B, n_cap, C] copies of entries [0, n) of every request, n =
// min(n_cap, n_max), further limited to (pos[b] + 1) / ratio when pos is non-null (one position per
// request).
cudaError_t launch_dequant_cache(int B, int C, int d_rope, const void* src, int64_t n_cap, int64_t n_max,
                                 const int64_t* pos, int ratio, void* dst, cudaStream_t st, bool pdl);

// ------------------------------------------------------------------ K2 / K6 indexer scores (SIMT)
struct IndexParams {
  const void* q_idx;     // [B, S, H_idx, d_idx]
  const float* w;        // [B, S, H_idx]
  const void* cidx;      // [B, n_cap, d_idx]
  float* scores;         // [B, S, n_cap]
  const int64_t* pos;    // [B, S]; null: t = s
  int64_t n_cap;
  int64_t entry_base;    // cidx holds the entries [entry_base, entry_base + n_cap) (0: all)
  int S, H_idx, ratio;
  RopeTab rope;
};

cudaError_t launch_index_simt(bool bf16, int B, const IndexParams& p, cudaStream_t st, bool pdl);

// ------------------------------------------------------------------ K3 top-k
struct TopkParams {
  const float* scores;   // [B, S, n_cap]
  int32_t* topk;         // [B, S, k]
  const int64_t* pos;    // [B, S]; null: t = s
  int64_t n_cap;
  int64_t entry_base;    // the scores are those of entries [entry_base, entry_base + n_cap); the
                         // selected indices are local (0 .. n_cap - 1)
  int S, k, ratio;
  void* ws;              // candidate buffers of the multi-level selection (topk_workspace_bytes)
};

size_t topk_workspace_bytes(int64_t rows, int64_t n_cap, int k);
cudaError_t launch_topk(int B, const TopkParams& p, cudaStream_t st, bool pdl);

// ------------------------------------------------------------------ K4 / K5 attention (SIMT)
struct AttnParams {
  const void* q;         // [B, S, H, d]
  const void* kv;        // [B, N, d]
  const void* ckv;       // [B, n_cap, d]
  const int32_t* topk;   // [B, S, k] or null (HCA)
  const float* sink;     // [H]
  void* out;             // [B, S, H, d]
  const int64_t* pos;    // [B, S]; null: t = s
  float* part_o;         // [B, S, n_split, H, d]   (n_split > 1)
  float* part_ml;        // [B, S, n_split, H, 2]
  int64_t N, n_cap;
  int64_t entry_base;    // ckv holds the entries [entry_base, entry_base + n_cap); topk is local
  int S, H, k, ratio, window, n_split, split_len;
  int no_window;         // CUDA-core kernel: leave the raw window out of the candidates
  int partial;           // CUDA-core kernel: write the (max, sum, unnormalised o) partials even unsplit
  float scale;
  RopeTab rope;
  int32_t* err;
};

cudaError_t launch_attn_simt(bool bf16, int B, const AttnParams& p, cudaStream_t st, bool pdl);

// ------------------------------------------------------------------ exchange over entry-range shards
constexpr int kMaxShards = 8;
constexpr int kMaxMergeCandidates = 4096;    // G * k per request

struct MergeParams {
  const float* score;                        // [B, G, k] candidate scores (-inf / NaN: empty)
  const int32_t* idx;                        // [B, G, k] candidate entries, local to their shard (-1 empty)
  int64_t base[kMaxShards];                  // first entry of each shard
  int64_t n_shard[kMaxShards];               // entries of each shard
  int G, k;
  int32_t* topk;                             // [B, k] the global selection, ascending, -1 padded
  int32_t* shard_sel;                        // [B, G, k] nullable: each shard's selected entries (local)
};

size_t topk_merge_smem(int G, int k);
cudaError_t launch_pack_candidates(int B, const float* scores, int64_t n_shard, const int32_t* idx, float* cand_score,
                                   int k, cudaStream_t st, bool pdl);
cudaError_t launch_topk_merge(int B, const MergeParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_attn_merge(bool bf16, int B, const AttnParams& p, cudaStream_t st, bool pdl);

}  // namespace csa
