// K3: top-k selection of indexer scores, one CTA per query row.
//
// [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", section "少读 KV 之前，Indexer 仍要给历史打分":
// top-k fixes how many compressed entries the main attention reads. The selection is exact: the
// k largest visible scores, ordered by (-score, index) (equal scores keep the lower index first);
// when fewer than k entries are visible every visible entry is taken and the tail holds -1.
//
// Method: float scores map to order-preserving 32-bit keys; a 4-pass MSB radix select (8-bit
// digits, shared-memory histograms) finds the k-th largest key T and how many keys equal to T are
// needed; one more pass gathers keys > T and, in index order, the first needed keys == T; a
// bitonic sort in shared memory orders the k winners.
#include "kernels.h"

namespace csa {
namespace {

constexpr int kThreads = 1024;
constexpr int kMaxK = 2048;

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;                        // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// a precedes b: larger key first, then smaller index
__device__ __forceinline__ bool before(uint32_t ka, int32_t ia, uint32_t kb, int32_t ib) {
  return ka > kb || (ka == kb && ia < ib);
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkParams p) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t sel_key[kMaxK];
  __shared__ int32_t sel_idx[kMaxK];
  __shared__ uint32_t s_prefix, s_need;
  __shared__ uint32_t s_gt;
  __shared__ uint32_t warp_cnt[32];

  const int b = blockIdx.y, s = blockIdx.x;
  const int64_t row = (int64_t)b * p.S + s;
  const int64_t t = p.pos ? p.pos[row] : s;
  const int64_t V = min(visible_entries(t, p.ratio), p.n_cap);
  const float* sc = p.scores + row * p.n_cap;
  int32_t* out = p.topk + row * p.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kk = (int)((int64_t)p.k < V ? (int64_t)p.k : V);

  if (kk == 0) {
    for (int j = tid; j < p.k; j += kThreads) out[j] = -1;
    return;
  }

  uint32_t prefix = 0, pmask = 0, need = (uint32_t)kk;
  if (kk < V) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      if (tid < 256) hist[tid] = 0;
      __syncthreads();
      for (int64_t i = tid; i < V; i += kThreads) {
        const uint32_t key = order_key(sc[i]);
        if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // bins in descending digit order; lane l owns digits 255-8l .. 248-8l
        uint32_t c[8], tot = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) { c[u] = hist[255 - 8 * lane - u]; tot += c[u]; }
        uint32_t incl = tot;                                   // inclusive scan over lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const uint32_t excl = incl - tot;
        if (excl < need && need <= incl) {                     // exactly one lane
          uint32_t run = excl;
          for (int u = 0; u < 8; ++u) {
            if (run + c[u] >= need) {
              s_prefix = prefix | ((uint32_t)(255 - 8 * lane - u) << shift);
              s_need = need - run;
              break;
            }
            run += c[u];
          }
        }
      }
      __syncthreads();
      prefix = s_prefix;
      need = s_need;
      pmask |= 255u << shift;
      __syncthreads();
    }
  } else {
    prefix = 0; need = 0;            // take everything: every key is > the (virtual) threshold
  }
  const bool take_all = (kk >= V);
  // gather: keys > T anywhere; keys == T in index order until `need` are taken
  if (tid == 0) s_gt = 0;
  __syncthreads();
  const uint32_t n_gt = (uint32_t)kk - need;
  uint32_t tie_base = 0;
  for (int64_t base = 0; base < V; base += kThreads) {
    const int64_t i = base + tid;
    uint32_t key = 0;
    bool gt = false, eq = false;
    if (i < V) {
      key = order_key(sc[i]);
      gt = take_all || key > prefix;
      eq = !take_all && key == prefix;
    }
    if (gt) {
      const uint32_t slot = atomicAdd(&s_gt, 1u);
      if (slot < (uint32_t)kMaxK) { sel_key[slot] = key; sel_idx[slot] = (int32_t)i; }
    }
    const unsigned bal = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) warp_cnt[warp] = __popc(bal);
    __syncthreads();
    uint32_t before_me = 0, total = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      const uint32_t c = warp_cnt[w];
      if (w < warp) before_me += c;
      total += c;
    }
    if (eq) {
      const uint32_t r = tie_base + before_me + __popc(bal & ((1u << lane) - 1u));
      if (r < need && n_gt + r < (uint32_t)kMaxK) { sel_key[n_gt + r] = key; sel_idx[n_gt + r] = (int32_t)i; }
    }
    tie_base += total;
    __syncthreads();
  }
  // bitonic sort of the kk winners (padded to a power of two)
  int n = 1;
  while (n < kk) n <<= 1;
  for (int j = kk + tid; j < n; j += kThreads) { sel_key[j] = 0u; sel_idx[j] = 0x7fffffff; }
  __syncthreads();
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int j = tid; j < n / 2; j += kThreads) {
        const int lo = 2 * j - (j & (stride - 1));
        const int hi = lo + stride;
        const bool up = ((lo & size) == 0);              // this run sorts in "precedes" order
        const uint32_t ka = sel_key[lo], kb = sel_key[hi];
        const int32_t ia = sel_idx[lo], ib = sel_idx[hi];
        const bool swap = up ? before(kb, ib, ka, ia) : before(ka, ia, kb, ib);
        if (swap) { sel_key[lo] = kb; sel_key[hi] = ka; sel_idx[lo] = ib; sel_idx[hi] = ia; }
      }
      __syncthreads();
    }
  }
  for (int j = tid; j < p.k; j += kThreads) out[j] = j < kk ? sel_idx[j] : -1;
}

}  // namespace

cudaError_t launch_topk(int B, const TopkParams& p, cudaStream_t st) {
  if (B == 0 || p.S == 0) return cudaSuccess;
  dim3 grid((unsigned)p.S, (unsigned)B);
  topk_kernel<<<grid, kThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace csa
