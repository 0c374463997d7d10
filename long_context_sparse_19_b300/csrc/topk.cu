// K3: top-k selection of indexer scores.
//
// [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", section "少读 KV 之前，Indexer 仍要给历史打分":
// top-k fixes how many compressed entries the main attention reads. The selection is exact: the
// k largest visible scores under the order (-score, index) (of equal scores the lower index is
// taken first); when fewer than k entries are visible every visible entry is taken. The selected
// entries are written in ascending entry index, followed by -1 in the unused slots.
//
// Method. Float scores map to order-preserving 32-bit keys. One CTA selects from at most `cap`
// items, loaded into shared memory once:
//   1. an 11-bit histogram of the keys (shared-memory atomics) locates the bin
//      that holds the k-th largest key;
//   2. the items of that bin are listed and an MSB radix select over their lower 21 bits finds
//      the exact threshold key T and how many items equal to T are taken;
//   3. one order-preserving compaction (warp ballots and scans, four items per lane) writes every
//      item above T and the first needed items equal to T, in index order.
// Rows longer than one CTA's capacity are cut into chunks; each chunk's winners (a superset of
// the row's winners inside the chunk) become (key, index) candidates, still in index order, and
// a further level selects among them until one CTA holds the whole row.
#include "kernels.h"

namespace csa {
namespace {

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;                        // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SelParams {
  const float* scores;       // level 0: [rows, n_in] scores (entry index = position in the row)
  const uint32_t* in_key;    // level > 0: [rows, n_in] candidate keys
  const int32_t* in_idx;     // level > 0: [rows, n_in] candidate entry indices (-1 = empty)
  int64_t n_in;              // items per row of the input (n_cap at level 0)
  const int64_t* pos;        // [rows] query positions (level 0 visibility); null: t = row % S
  int S, ratio, k;
  int chunk;                 // items per CTA (blockIdx.x selects the chunk), a multiple of 4
  int n_chunks;
  int32_t* topk;             // final level: [rows, k], ascending entry index, -1 padded
  uint32_t* out_key;         // otherwise: [rows, n_chunks * k] candidates (-1 padded)
  int32_t* out_idx;
};

constexpr int kBins = 2048;                 // first-level histogram: the top 11 key bits
constexpr int kShift0 = 21;

template <int kThreads>
struct SelSmem {
  static size_t bytes(int cap, bool with_idx) {
    // keys, (indices), bin list, histogram, scan scratch
    return (size_t)cap * 4 * (with_idx ? 3 : 2) + kBins * 4 + 4 * 64 * 4 + 64;
  }
};

// block-wide exclusive scan of one value per thread (kThreads <= 1024); returns the exclusive
// prefix and writes the block total to *total. `scratch` holds 32 words.
template <int kThreads>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* scratch, uint32_t* total) {
  constexpr int kWarps = kThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  uint32_t wo = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t s = scratch[w];
    wo += (w < warp) ? s : 0u;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return wo + incl - v;
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads) topk_select_kernel(const SelParams p, int cap) {
  constexpr int kWarps = kThreads / 32;
  extern __shared__ __align__(16) uint8_t sm[];
  const bool level0 = p.scores != nullptr;
  uint32_t* keys = reinterpret_cast<uint32_t*>(sm);                              // [cap]
  int32_t* idxs = reinterpret_cast<int32_t*>(keys + cap);                        // [cap] (levels > 0)
  uint32_t* list = level0 ? reinterpret_cast<uint32_t*>(idxs) : reinterpret_cast<uint32_t*>(idxs + cap);  // [cap]
  uint32_t* hist = list + cap;                                                   // [kBins]
  uint32_t* scr = hist + kBins;                                                  // [4][64]
  __shared__ uint32_t s_T, s_need, s_cls, s_nlist, s_nvalid, s_bin, s_need_bin;

  griddep_launch();
  griddep_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.y;
  const int64_t c0 = (int64_t)blockIdx.x * p.chunk;

  // ---- load the items of this CTA: level 0 = visible entries of the chunk, else the candidates
  int n;
  if (level0) {
    const int64_t t = p.pos ? p.pos[row] : (row % p.S);
    const int64_t V = t < 0 ? 0 : min(visible_entries(t, p.ratio), p.n_in);
    n = (int)max((int64_t)0, min((int64_t)p.chunk, V - c0));
  } else {
    n = (int)max((int64_t)0, min((int64_t)p.chunk, p.n_in - c0));
  }
  const int n4 = (n + 3) & ~3;
  for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
  if (tid == 0) { s_nlist = 0; s_nvalid = 0; }
  __syncthreads();
  {
    const bool vec = ((row * p.n_in + c0) & 3) == 0;      // 16-byte aligned score rows
    uint32_t nv = 0;
    for (int i = 4 * tid; i < n4; i += 4 * kThreads) {
      uint32_t kq[4];
      int32_t iq[4] = {0, 0, 0, 0};
      if (level0) {
        const float* sc = p.scores + row * p.n_in + c0 + i;
        if (vec && i + 4 <= n) {
          const float4 f = __ldg(reinterpret_cast<const float4*>(sc));
          kq[0] = order_key(f.x); kq[1] = order_key(f.y); kq[2] = order_key(f.z); kq[3] = order_key(f.w);
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u) kq[u] = (i + u < n) ? order_key(__ldg(sc + u)) : 0u;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) nv += (i + u < n);
      } else {
        const uint32_t* ik = p.in_key + row * p.n_in + c0 + i;
        const int32_t* ii = p.in_idx + row * p.n_in + c0 + i;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          iq[u] = (i + u < n) ? __ldg(ii + u) : -1;
          kq[u] = iq[u] >= 0 ? __ldg(ik + u) : 0u;
          nv += iq[u] >= 0;
        }
        *reinterpret_cast<int4*>(idxs + i) = make_int4(iq[0], iq[1], iq[2], iq[3]);
      }
      *reinterpret_cast<uint4*>(keys + i) = make_uint4(kq[0], kq[1], kq[2], kq[3]);
      // histogram of the top 11 bits (valid items have keys > 0)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (kq[u] != 0u) atomicAdd(&hist[kq[u] >> kShift0], 1u);
      }
    }
    nv = __reduce_add_sync(0xffffffffu, nv);
    if (lane == 0 && nv) atomicAdd(&s_nvalid, nv);
  }
  __syncthreads();
  const uint32_t n_valid = s_nvalid;
  const uint32_t kk = min((uint32_t)p.k, n_valid);
  const bool take_all = kk >= n_valid;

  // take keys with (key & pmask) > T, and the first need_t with (key & pmask) == T
  uint32_t T = 0, need_t = 0, pmask = ~0u;
  if (!take_all) {
    // ---- 1. the bin of the kk-th largest key: thread t scans bins in descending order
    constexpr int kPer = kBins / kThreads;      // bins per thread
    uint32_t c[kPer], tot = 0;
#pragma unroll
    for (int u = 0; u < kPer; ++u) { c[u] = hist[kBins - 1 - kPer * tid - u]; tot += c[u]; }
    uint32_t all;
    const uint32_t excl = block_excl_scan<kThreads>(tot, scr, &all);
    if (excl < kk && kk <= excl + tot) {
      uint32_t run = excl;
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        if (run < kk && kk <= run + c[u]) { s_bin = kBins - 1 - kPer * tid - u; s_need_bin = kk - run; }
        run += c[u];
      }
    }
    __syncthreads();
    const uint32_t bin = s_bin;
    uint32_t need = s_need_bin;                  // items still needed from the bin
    // ---- 2. list the bin's keys, then radix-select the need-th largest among them
    for (int i = tid; i < n; i += kThreads) {
      const unsigned am = __activemask();
      const uint32_t key = keys[i];
      const bool in = key != 0u && (key >> kShift0) == bin;
      const unsigned b = __ballot_sync(am, in);
      if (b) {
        const int leader = __ffs(b) - 1;
        uint32_t base = 0;
        if (lane == leader) base = atomicAdd(&s_nlist, (uint32_t)__popc(b));
        base = __shfl_sync(am, base, leader);
        if (in) list[base + __popc(b & ((1u << lane) - 1u))] = key;
      }
    }
    __syncthreads();
    const uint32_t nl = s_nlist;
    uint32_t prefix = bin << kShift0;
    pmask = ~0u << kShift0;
    uint32_t cls = nl;                           // items of the current class (masked key == prefix)
    // digits of 7 bits: bits 20..14, 13..7, 6..0
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = 14 - 7 * pass;
      if (cls == need) break;                    // every item of the class is taken
      for (int i = tid; i < 128; i += kThreads) hist[i] = 0;
      __syncthreads();
      for (uint32_t i = tid; i < nl; i += kThreads) {
        const uint32_t key = list[i];
        if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 127u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        uint32_t cc[4], tt = 0;                  // lane l owns digits 127-4l .. 124-4l
#pragma unroll
        for (int u = 0; u < 4; ++u) { cc[u] = hist[127 - 4 * lane - u]; tt += cc[u]; }
        uint32_t incl = tt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += x;
        }
        const uint32_t ex = incl - tt;
        if (ex < need && need <= incl) {
          uint32_t run = ex;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (run < need && need <= run + cc[u]) {
              s_T = prefix | ((uint32_t)(127 - 4 * lane - u) << shift);
              s_need = need - run;
              s_cls = cc[u];
            }
            run += cc[u];
          }
        }
      }
      __syncthreads();
      prefix = s_T;
      need = s_need;
      cls = s_cls;
      pmask |= 127u << shift;
      __syncthreads();
    }
    // Keys of the final class: (key & pmask) == prefix. If the class was fully determined
    // before the last pass (nl == need at some point), its members differ in their low bits;
    // comparing the masked key keeps them together and all of them are taken.
    T = prefix;
    need_t = need;
  }
  const uint32_t mask = pmask;

  // ---- 3. order-preserving compaction: gt = (key & mask) > T, eq = (key & mask) == T
  // warp w owns items [w*seg, (w+1)*seg), seg a multiple of 128; lane l takes 4 consecutive items
  const int seg = ((n4 + kWarps - 1) / kWarps + 127) & ~127;
  const int s0 = min(n4, warp * seg), s1 = min(n4, s0 + seg);
  auto classify = [&](int i, uint32_t (&kq)[4], uint32_t& g, uint32_t& e) {
    const uint4 v = *reinterpret_cast<const uint4*>(keys + i);
    kq[0] = v.x; kq[1] = v.y; kq[2] = v.z; kq[3] = v.w;
    g = 0; e = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool ok = kq[u] != 0u;
      const uint32_t km = kq[u] & mask;
      g |= (uint32_t)(ok && (take_all || km > T)) << u;
      e |= (uint32_t)(ok && !take_all && km == T) << u;
    }
  };
  uint32_t cg = 0, ce = 0;
  for (int b = s0; b < s1; b += 128) {
    const int i = b + 4 * lane;
    if (i < s1) {
      uint32_t kq[4], g, e;
      classify(i, kq, g, e);
      cg += __popc(g); ce += __popc(e);
    }
  }
  cg = __reduce_add_sync(0xffffffffu, cg);
  ce = __reduce_add_sync(0xffffffffu, ce);
  if (lane == 0) { scr[warp] = cg; scr[64 + warp] = ce; }
  __syncthreads();
  uint32_t og = 0, oe = 0;
  for (int w = 0; w < warp; ++w) { og += scr[w]; oe += scr[64 + w]; }
  int32_t* out_final = p.topk ? p.topk + row * p.k : nullptr;
  const int64_t cand = row * ((int64_t)p.n_chunks * p.k) + (int64_t)blockIdx.x * p.k;
  for (int b = s0; b < s1; b += 128) {
    const int i = b + 4 * lane;
    uint32_t kq[4] = {0, 0, 0, 0}, g = 0, e = 0;
    if (i < s1) classify(i, kq, g, e);
    // lane-exclusive prefix of the gt / eq counts
    const uint32_t lg = __popc(g), le = __popc(e);
    uint32_t ig = lg, ie = le;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t xg = __shfl_up_sync(0xffffffffu, ig, o);
      const uint32_t xe = __shfl_up_sync(0xffffffffu, ie, o);
      if (lane >= o) { ig += xg; ie += xe; }
    }
    uint32_t rg = og + ig - lg, re = oe + ie - le;     // ranks of this lane's first item
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool gt = (g >> u) & 1u, eq = (e >> u) & 1u;
      if (gt || (eq && re < need_t)) {
        const uint32_t slot = rg + min(re, need_t);
        const int32_t id = level0 ? (int32_t)(c0 + i + u) : idxs[i + u];
        if (out_final) out_final[slot] = id;
        else { p.out_key[cand + slot] = kq[u]; p.out_idx[cand + slot] = id; }
      }
      rg += gt;
      re += eq;
    }
    og += __shfl_sync(0xffffffffu, ig, 31);
    oe += __shfl_sync(0xffffffffu, ie, 31);
  }
  // unused slots
  for (int j = kk + tid; j < p.k; j += kThreads) {
    if (out_final) out_final[j] = -1;
    else { p.out_key[cand + j] = 0u; p.out_idx[cand + j] = -1; }
  }
}

template <int kThreads>
cudaError_t launch_select(const SelParams& p, int64_t rows, int cap, cudaStream_t st, bool pdl) {
  const bool with_idx = p.scores == nullptr;
  const size_t smem = SelSmem<kThreads>::bytes(cap, with_idx);
  cudaError_t e = cudaFuncSetAttribute(topk_select_kernel<kThreads>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.n_chunks, (unsigned)rows);
  return launch_kernel(pdl, topk_select_kernel<kThreads>, grid, dim3(kThreads), smem, st, p, cap);
}

// Items one CTA holds: the large variant (1024 threads) serves the later levels of very long rows;
// the small one (512 threads for decode rows, 256 for the many short rows of a prefill) the first
// level and every short row. Cutting decode rows into 4096-entry chunks spreads the first level
// over many SMs; its winners (k per chunk) are then few enough for one small CTA per row.
constexpr int kCapLarge = 16384;
constexpr int kCapSmall = 4096;

}  // namespace

size_t topk_workspace_bytes(int64_t rows, int64_t n_cap, int k) {
  // candidates of the intermediate levels: two ping-pong buffers of (key, index) pairs, each large
  // enough for the first level's output
  if (n_cap <= kCapSmall || k <= 0) return 0;
  const int64_t chunks = (n_cap + kCapSmall - 1) / kCapSmall;
  return 2 * (size_t)rows * chunks * k * 8;
}

cudaError_t launch_topk(int B, const TopkParams& p, cudaStream_t st, bool pdl) {
  if (B == 0 || p.S == 0) return cudaSuccess;
  const int64_t rows = (int64_t)B * p.S;
  SelParams s;
  s.scores = p.scores; s.in_key = nullptr; s.in_idx = nullptr; s.n_in = p.n_cap; s.pos = p.pos;
  s.S = p.S; s.ratio = p.ratio; s.k = p.k;
  uint8_t* ws = static_cast<uint8_t*>(p.ws);
  const size_t half = topk_workspace_bytes(rows, p.n_cap, p.k) / 2;
  int64_t n_in = p.n_cap;
  for (int level = 0;; ++level) {
    const bool first_launch = level == 0;
    const bool dep = pdl || !first_launch;
    if (n_in <= kCapSmall) {                                   // one small CTA holds the row: final level
      s.chunk = (int)((n_in + 3) & ~3ll); s.n_chunks = 1;
      s.topk = p.topk; s.out_key = nullptr; s.out_idx = nullptr;
      if (p.S > 1) return launch_select<256>(s, rows, kCapSmall, st, dep);
      return launch_select<512>(s, rows, kCapSmall, st, dep);
    }
    if (level > 0 && n_in <= kCapLarge) {                      // one large CTA holds the row: final level
      s.chunk = (int)((n_in + 3) & ~3ll); s.n_chunks = 1;
      s.topk = p.topk; s.out_key = nullptr; s.out_idx = nullptr;
      return launch_select<1024>(s, rows, kCapLarge, st, dep);
    }
    if (!ws) return cudaErrorInvalidValue;
    const int64_t cap = level == 0 ? kCapSmall : kCapLarge;
    const int64_t chunks = (n_in + cap - 1) / cap;
    const int64_t n_out = chunks * p.k;
    uint8_t* buf = ws + (level & 1) * half;
    s.chunk = (int)cap; s.n_chunks = (int)chunks;
    s.topk = nullptr;
    s.out_key = reinterpret_cast<uint32_t*>(buf);
    s.out_idx = reinterpret_cast<int32_t*>(buf + (size_t)rows * n_out * 4);
    cudaError_t e = level == 0 ? launch_select<512>(s, rows, kCapSmall, st, dep)
                               : launch_select<1024>(s, rows, kCapLarge, st, dep);
    if (e != cudaSuccess) return e;
    s.scores = nullptr; s.pos = nullptr;
    s.in_key = s.out_key; s.in_idx = s.out_idx; s.n_in = n_out;
    n_in = n_out;
  }
}

}  // namespace csa
