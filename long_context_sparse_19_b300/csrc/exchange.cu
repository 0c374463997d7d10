// The exchange step of one request whose compressed caches are split by entry range over G shards
// (G devices in a multi-device deployment; the kernels here are each device's share of the work).
//
// [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", section "少读 KV 之前，Indexer 仍要给历史打分": the
// selection is made on the combined scores. Sharded by entry range, every shard scores its own
// entries and keeps its local top k as (score, entry) candidates; the global top k under the order
// (-score, index) is the top k of the union of those candidates, since an entry outside its shard's
// local top k has k entries of its shard above it. The attention ("局部和压缩记忆，共用一次归一化")
// splits the same way: each shard reduces its selected rows (and the owner of the raw window the
// window) to per-head partials (max logit, sum of exponentials, unnormalised weighted sum), and the
// partials merge with the sink counted once, followed by the inverse RoPE.
//
// This file holds the two steps that exist only because of the split: packing a shard's candidates
// (their scores) and merging G candidate lists into the global selection (with each shard's local
// list of the selected entries it holds). Scoring a shard, its local top k, the attention partials
// and their merge use the indexer, top-k and CUDA-core attention kernels with an entry offset.
#include "kernels.h"

namespace csa {
namespace {

constexpr int kMergeThreads = 1024;

__device__ __forceinline__ uint32_t cand_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;                        // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);   // order-preserving, >= 0x007FFFFF for -inf
}

// cand_score[b, j] = scores[b, idx[b, j]] (-inf for an empty slot)
__global__ void pack_candidates_kernel(const float* scores, int64_t n_shard, const int32_t* idx, float* cand_score,
                                       int k) {
  griddep_launch();
  griddep_wait();
  const int b = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= k) return;
  const int32_t i = idx[(int64_t)b * k + j];
  cand_score[(int64_t)b * k + j] = (i >= 0 && i < n_shard) ? scores[(int64_t)b * n_shard + i] : -INFINITY;
}

// One CTA per request. Candidate c = (shard g, slot j) holds key (order key of its score, then the
// complement of its global index): distinct keys, larger = earlier under (-score, index). A valid
// candidate is selected when fewer than k keys are larger; its output slot is the number of selected
// candidates with a smaller global index (ascending output), and likewise inside its shard.
__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(const MergeParams p) {
  extern __shared__ unsigned long long mkey[];                  // [G k]
  int32_t* gidx = reinterpret_cast<int32_t*>(mkey + p.G * p.k); // [G k]
  uint8_t* sel = reinterpret_cast<uint8_t*>(gidx + p.G * p.k);  // [G k]
  __shared__ int32_t n_sel[kMaxShards + 1];
  griddep_launch();
  griddep_wait();
  const int b = blockIdx.x, tid = threadIdx.x;
  const int n = p.G * p.k;
  if (tid <= kMaxShards) n_sel[tid] = 0;
  for (int c = tid; c < n; c += kMergeThreads) {
    const int g = c / p.k;
    const int64_t at = ((int64_t)b * p.G + g) * p.k + (c % p.k);
    const int32_t li = p.idx[at];
    const float sc = p.score[at];
    const bool valid = li >= 0 && li < p.n_shard[g] && sc == sc;
    const int64_t gi = valid ? p.base[g] + li : -1;
    mkey[c] = valid ? ((unsigned long long)cand_key(sc) << 32) | (uint32_t)(0x7FFFFFFF - gi) : 0ull;
    gidx[c] = (int32_t)gi;
  }
  __syncthreads();
  for (int c = tid; c < n; c += kMergeThreads) {
    const unsigned long long kc = mkey[c];
    int above = 0;
    if (kc != 0ull)
      for (int j = 0; j < n && above < p.k; ++j) above += mkey[j] > kc;
    sel[c] = kc != 0ull && above < p.k;
  }
  __syncthreads();
  for (int c = tid; c < n; c += kMergeThreads) {
    if (!sel[c]) continue;
    const int g = c / p.k, gi = gidx[c];
    int before = 0, before_g = 0;
    for (int j = 0; j < n; ++j) {
      const bool lower = sel[j] && gidx[j] < gi;
      before += lower;
      before_g += lower && j / p.k == g;
    }
    p.topk[(int64_t)b * p.k + before] = gi;
    if (p.shard_sel) p.shard_sel[((int64_t)b * p.G + g) * p.k + before_g] = (int32_t)(gi - p.base[g]);
    atomicAdd(&n_sel[g], 1);
    atomicAdd(&n_sel[kMaxShards], 1);
  }
  __syncthreads();
  for (int j = n_sel[kMaxShards] + tid; j < p.k; j += kMergeThreads) p.topk[(int64_t)b * p.k + j] = -1;
  if (p.shard_sel)
    for (int g = 0; g < p.G; ++g)
      for (int j = n_sel[g] + tid; j < p.k; j += kMergeThreads) p.shard_sel[((int64_t)b * p.G + g) * p.k + j] = -1;
}

}  // namespace

size_t topk_merge_smem(int G, int k) { return (size_t)G * k * (8 + 4 + 1); }

cudaError_t launch_pack_candidates(int B, const float* scores, int64_t n_shard, const int32_t* idx, float* cand_score,
                                   int k, cudaStream_t st, bool pdl) {
  if (B == 0 || k == 0) return cudaSuccess;
  dim3 grid((unsigned)((k + 255) / 256), (unsigned)B);
  return launch_kernel(pdl, pack_candidates_kernel, grid, dim3(256), 0, st, scores, n_shard, idx, cand_score, k);
}

cudaError_t launch_topk_merge(int B, const MergeParams& p, cudaStream_t st, bool pdl) {
  if (B == 0) return cudaSuccess;
  const size_t smem = topk_merge_smem(p.G, p.k);
  cudaError_t e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(pdl, topk_merge_kernel, dim3((unsigned)B), dim3(kMergeThreads), smem, st, p);
}

}  // namespace csa
