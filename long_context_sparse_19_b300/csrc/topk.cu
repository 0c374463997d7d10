// K3: top-k selection of indexer scores.
//
// [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", section "少读 KV 之前，Indexer 仍要给历史打分":
// top-k fixes how many compressed entries the main attention reads. The selection is exact: the
// k largest visible scores under the order (-score, index) (of equal scores the lower index is
// taken first); when fewer than k entries are visible every visible entry is taken. The selected
// entries are written in ascending entry index, followed by -1 in the unused slots.
//
// Method. Float scores map to order-preserving 32-bit keys (0 marks an empty item). One CTA holds
// up to 16 items per thread in registers, thread t owning items 16t .. 16t+15, so index order is
// thread order. An MSB radix select finds the threshold key T: digits of 11, 11 and 10 bits, each
// a shared-memory histogram over the items still matching the prefix (the first, over all items,
// in per-warp private histograms so that warps never contend), a block-wide scan of the bins, and
// an early exit once the threshold digit's bin holds exactly the items still needed. One
// order-preserving compaction (block scans of per-thread counts) then writes every item above T and
// the first needed items equal to T. Long rows are cut into chunks; each chunk's winners (a
// superset of the row's winners inside the chunk) become (key, index) candidates, still in index
// order, and a further level selects among them.
#include "kernels.h"

namespace csa {
namespace {

constexpr int kItems = 16;                  // items per thread
constexpr int kBins = 2048;                 // 11-bit digits

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
  int64_t entry_base;        // level 0: the row holds the entries [entry_base, entry_base + n_in)
  int S, ratio, k;
  int chunk;                 // items per CTA (blockIdx.x selects the chunk)
  int n_chunks;
  int32_t* topk;             // final level: [rows, k], ascending entry index, -1 padded
  uint32_t* out_key;         // otherwise: [rows, n_chunks * k] candidates (-1 padded)
  int32_t* out_idx;
};

template <int kThreads>
struct SelSmem {
  static constexpr int kWarps = kThreads / 32;
  // per-warp histograms of the first digit: two 16-bit counters per word
  static constexpr size_t kWarpHist = (size_t)kWarps * (kBins / 2) * 4;
  static constexpr size_t kBytes = kWarpHist + kBins * 4 + 4 * 32 * 4 + 64;
};

// block-wide exclusive scan of two counters per thread (kThreads <= 1024), thread order;
// scratch holds 64 words. Returns the exclusive prefixes and the totals.
template <int kThreads>
__device__ __forceinline__ void block_scan2(uint32_t a, uint32_t b, uint32_t* scratch, uint32_t& ea,
                                            uint32_t& eb, uint32_t& ta, uint32_t& tb) {
  constexpr int kWarps = kThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t xa = __shfl_up_sync(0xffffffffu, ia, o);
    const uint32_t xb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) { ia += xa; ib += xb; }
  }
  if (lane == 31) { scratch[warp] = ia; scratch[32 + warp] = ib; }
  __syncthreads();
  uint32_t wa = 0, wb = 0, sa = 0, sb = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t va = scratch[w], vb = scratch[32 + w];
    if (w < warp) { wa += va; wb += vb; }
    sa += va; sb += vb;
  }
  __syncthreads();
  ea = wa + ia - a; eb = wb + ib - b; ta = sa; tb = sb;
}

// Finds the bin holding the need-th largest item: bins are scanned from the top; thread t owns
// kBins / kThreads consecutive bins (descending). Writes the bin, the items still needed from it
// and that bin's count to out[0..2] (then visible to the whole block).
template <int kThreads>
__device__ __forceinline__ void find_bin(const uint32_t* hist, uint32_t need, uint32_t* scratch, uint32_t* out) {
  constexpr int kPer = kBins / kThreads;
  uint32_t c[kPer], tot = 0;
#pragma unroll
  for (int u = 0; u < kPer; ++u) { c[u] = hist[kBins - 1 - kPer * threadIdx.x - u]; tot += c[u]; }
  uint32_t ex, dummy, all, dummy2;
  block_scan2<kThreads>(tot, 0u, scratch, ex, dummy, all, dummy2);
  if (ex < need && need <= ex + tot) {
    uint32_t run = ex;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      if (run < need && need <= run + c[u]) {
        out[0] = kBins - 1 - kPer * threadIdx.x - u;
        out[1] = need - run;
        out[2] = c[u];
      }
      run += c[u];
    }
  }
  __syncthreads();
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads) topk_select_kernel(const SelParams p) {
  constexpr int kWarps = kThreads / 32;
  extern __shared__ __align__(16) uint8_t sm[];
  uint32_t* whist = reinterpret_cast<uint32_t*>(sm);                // [kWarps][kBins / 2]
  uint32_t* hist = whist + kWarps * (kBins / 2);                    // [kBins]
  uint32_t* scr = hist + kBins;                                     // [128]
  uint32_t* res = scr + 128;                                        // [16]

  if (threadIdx.x == 0) CSA_STAMP(54);
  if (threadIdx.x == 0) CSA_STAMP(gridDim.x > 1 ? 45 : 47);
  griddep_launch();
  griddep_wait();
  if (threadIdx.x == 0) CSA_STAMP(55);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.y;
  const int64_t c0 = (int64_t)blockIdx.x * p.chunk;
  const bool level0 = p.scores != nullptr;

  // ---- the items of this CTA: level 0 = visible entries of the chunk, else the candidates
  int n;
  if (level0) {
    const int64_t t = p.pos ? p.pos[row] : (row % p.S);
    const int64_t V = visible_local(t, p.ratio, p.entry_base, p.n_in);
    n = (int)max((int64_t)0, min((int64_t)p.chunk, V - c0));
  } else {
    n = (int)max((int64_t)0, min((int64_t)p.chunk, p.n_in - c0));
  }
  uint32_t key[kItems];
  int32_t id[kItems];
  const int i0 = tid * kItems;
  if (level0) {
    const float* sc = p.scores + row * p.n_in + c0 + i0;
    if (((row * p.n_in + c0) & 3) == 0 && i0 + kItems <= n) {       // 16-byte aligned, all in range
#pragma unroll
      for (int q = 0; q < kItems / 4; ++q) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(sc) + q);
        key[4 * q] = order_key(f.x); key[4 * q + 1] = order_key(f.y);
        key[4 * q + 2] = order_key(f.z); key[4 * q + 3] = order_key(f.w);
      }
    } else {
#pragma unroll
      for (int u = 0; u < kItems; ++u) key[u] = i0 + u < n ? order_key(__ldg(sc + u)) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kItems; ++u) id[u] = (int32_t)(c0 + i0 + u);
  } else {
    const uint32_t* ik = p.in_key + row * p.n_in + c0 + i0;
    const int32_t* ii = p.in_idx + row * p.n_in + c0 + i0;
#pragma unroll
    for (int u = 0; u < kItems; ++u) id[u] = i0 + u < n ? __ldg(ii + u) : -1;
#pragma unroll
    for (int u = 0; u < kItems; ++u) key[u] = id[u] >= 0 ? __ldg(ik + u) : 0u;
  }

  // ---- first digit (key bits 31..21): per-warp private histograms, then summed
  if (tid == 0) CSA_STAMP(56);
  {
    uint4* z = reinterpret_cast<uint4*>(whist);
    for (int i = tid; i < kWarps * (kBins / 2) / 4; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
    if (tid < 16) res[tid] = 0;
  }
  __syncthreads();
  {
    uint32_t* wh = whist + warp * (kBins / 2);
    uint32_t nv = 0;
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      if (key[u] != 0u) {
        const uint32_t b = key[u] >> 21;
        atomicAdd(&wh[b >> 1], 1u << ((b & 1u) * 16));
        ++nv;
      }
    }
    nv = __reduce_add_sync(0xffffffffu, nv);
    if (lane == 0 && nv) atomicAdd(&res[8], nv);
  }
  __syncthreads();
  if (tid == 0) CSA_STAMP(57);
  for (int b2 = tid; b2 < kBins / 2; b2 += kThreads) {
    uint32_t lo = 0, hi = 0;
#pragma unroll 4
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t v = whist[w * (kBins / 2) + b2];
      lo += v & 0xffffu;
      hi += v >> 16;
    }
    hist[2 * b2] = lo;
    hist[2 * b2 + 1] = hi;
  }
  __syncthreads();
  if (tid == 0) CSA_STAMP(58);
  const uint32_t n_valid = res[8];
  const uint32_t kk = min((uint32_t)p.k, n_valid);
  const bool take_all = kk >= n_valid;

  // ---- radix select of the threshold: taken = (key & pmask) > prefix, or == prefix for the first
  // `need` such items in index order
  uint32_t prefix = 0, pmask = 0, need = kk;
  if (!take_all) {
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const uint32_t dmask = pass < 2 ? 2047u : 1023u;
      if (pass > 0) {
        for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kItems; ++u)
          if (key[u] != 0u && (key[u] & pmask) == prefix) atomicAdd(&hist[(key[u] >> shift) & dmask], 1u);
        __syncthreads();
      }
      find_bin<kThreads>(hist, need, scr, res);
      if (tid == 0) CSA_STAMP(59 + pass);
      const uint32_t bin = res[0], cnt = res[2];
      need = res[1];
      prefix |= bin << shift;
      pmask |= dmask << shift;
      if (cnt == need) break;                                 // the whole class is taken
    }
  }

  // ---- order-preserving compaction of the winners
  uint32_t ngt = 0, neq = 0;
#pragma unroll
  for (int u = 0; u < kItems; ++u) {
    const bool valid = key[u] != 0u;
    const uint32_t m = key[u] & pmask;
    ngt += valid && (take_all || m > prefix);
    neq += valid && !take_all && m == prefix;
  }
  uint32_t rg, re, tgt, teq;
  block_scan2<kThreads>(ngt, neq, scr, rg, re, tgt, teq);
  if (tid == 0) CSA_STAMP(62);
  int32_t* out_final = p.topk ? p.topk + row * p.k : nullptr;
  const int64_t cand = row * ((int64_t)p.n_chunks * p.k) + (int64_t)blockIdx.x * p.k;
#pragma unroll
  for (int u = 0; u < kItems; ++u) {
    const bool valid = key[u] != 0u;
    const uint32_t m = key[u] & pmask;
    const bool gt = valid && (take_all || m > prefix);
    const bool eq = valid && !take_all && m == prefix;
    if (gt || (eq && re < need)) {
      const uint32_t slot = rg + min(re, need);
      if (out_final) {
        out_final[slot] = id[u];
      } else {
        p.out_key[cand + slot] = key[u];
        p.out_idx[cand + slot] = id[u];
      }
    }
    rg += gt;
    re += eq;
  }
  for (int j = (int)kk + tid; j < p.k; j += kThreads) {
    if (out_final) out_final[j] = -1;
    else { p.out_key[cand + j] = 0u; p.out_idx[cand + j] = -1; }
  }
  if (tid == 0) CSA_STAMP(63);
  if (tid == 0) CSA_STAMP(gridDim.x > 1 ? 46 : 48);
}

// ------------------------------------------------------------------ one row, one cluster
// A row of up to 8 x 2048 items is selected by one thread-block cluster in a single launch. CTA r
// of the cluster holds items 2048 r .. 2048 r + 2047 (16 per thread, in registers). The CTAs share
// what they find by writing into each other's shared memory (remote adds and stores: no round
// trips) followed by a cluster barrier. A remote request costs a few hundred nanoseconds and one
// thread's requests do not overlap, so each CTA sends as few as it can:
//   1. every CTA adds its histogram of the keys' top 11 bits into every CTA's copy of the cluster
//      histogram, and into a second array of the higher-ranked CTAs only, but only from the bin
//      of its own k-th largest key upwards (the row's k-th largest key is at least as large, so
//      lower bins cannot hold it). After the barrier each CTA finds the same threshold bin, and
//      the second array tells it how many items above the bin and in it the lower-ranked CTAs
//      hold: where its own winners go in the output;
//   2. when only part of the bin is taken, every CTA stores its in-bin keys into every CTA's list
//      at those offsets (row order); after the barrier each finds the remaining digits of the
//      threshold on its own and takes the first `need` in-bin keys in (-key, position) order;
// then every CTA writes its winners in ascending index order. A bin of more than kListCap items
// (a very flat distribution) is first refined by the next digits through further exchanges, with
// the offsets then exchanged as counts. No CTA writes to another after the last barrier it takes
// part in, so none can exit while another still writes to it. Shared memory is kept near 45 KB: a
// larger footprint delays placing the 8-CTA clusters beside the CTAs of neighbouring launches.
constexpr int kCluThreads = 128;
constexpr int kCluChunk = kCluThreads * kItems;          // 2048 items per CTA
constexpr int kCluMax = 8;                                // portable cluster size
constexpr int kListCap = 1024;                            // in-bin items split locally (cluster total)
constexpr int kListPer = kListCap / kCluThreads;          // list positions per thread in the final order
static_assert(kListCap % kCluThreads == 0, "the final order gives each thread the same number of list positions");

struct CluSmem {
  uint32_t full[3][kBins];              // cluster histogram of each digit pass (remote adds)
  uint32_t before[kBins];               // first digit, lower-ranked CTAs only (remote adds)
  uint32_t hist[kBins];                 // this CTA's histogram; later the local digit passes
  alignas(16) uint32_t list[kListCap];  // the cluster's in-bin keys in row order (remote stores)
  uint32_t src_cnt[kCluMax][2];         // per source CTA: (items above, in the class) (remote stores)
  uint32_t n_valid;                     // the row's valid items (remote adds)
  uint32_t scr[64];
  uint32_t res[4];
  uint8_t taken[kListCap];              // in-bin item (row order) is selected
};

__global__ void __launch_bounds__(kCluThreads) topk_cluster_kernel(const SelParams p) {
  extern __shared__ __align__(16) uint8_t clu_raw[];
  CluSmem& sm = *reinterpret_cast<CluSmem*>(clu_raw);
  if (threadIdx.x == 0) CSA_STAMP(47);
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t rank = cluster_rank(), C = gridDim.x;
  for (int i = tid; i < 4 * kBins; i += kCluThreads) (&sm.full[0][0])[i] = 0;   // full and before
  if (tid == 0) sm.n_valid = 0;
  cluster_arrive();                                       // the zeroed counters may be added into
  griddep_launch();
  griddep_wait();
  if (tid == 0) CSA_STAMP(54);
  const int64_t row = blockIdx.y;
  const int64_t c0 = (int64_t)rank * kCluChunk;
  const bool level0 = p.scores != nullptr;
  int n;
  if (level0) {
    const int64_t t = p.pos ? p.pos[row] : (row % p.S);
    const int64_t V = visible_local(t, p.ratio, p.entry_base, p.n_in);
    n = (int)max((int64_t)0, min((int64_t)kCluChunk, V - c0));
  } else {
    n = (int)max((int64_t)0, min((int64_t)kCluChunk, p.n_in - c0));
  }
  uint32_t key[kItems];
  int32_t id[kItems];
  const int i0 = tid * kItems;
  if (level0) {
    const float* sc = p.scores + row * p.n_in + c0 + i0;
    if (((row * p.n_in + c0) & 3) == 0 && i0 + kItems <= n) {
#pragma unroll
      for (int q = 0; q < kItems / 4; ++q) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(sc) + q);
        key[4 * q] = order_key(f.x); key[4 * q + 1] = order_key(f.y);
        key[4 * q + 2] = order_key(f.z); key[4 * q + 3] = order_key(f.w);
      }
    } else {
#pragma unroll
      for (int u = 0; u < kItems; ++u) key[u] = i0 + u < n ? order_key(__ldg(sc + u)) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kItems; ++u) id[u] = (int32_t)(c0 + i0 + u);
  } else {
    const uint32_t* ik = p.in_key + row * p.n_in + c0 + i0;
    const int32_t* ii = p.in_idx + row * p.n_in + c0 + i0;
#pragma unroll
    for (int u = 0; u < kItems; ++u) id[u] = i0 + u < n ? __ldg(ii + u) : -1;
#pragma unroll
    for (int u = 0; u < kItems; ++u) key[u] = id[u] >= 0 ? __ldg(ik + u) : 0u;
  }


  if (tid == 0) CSA_STAMP(55);
  // ---- threshold class: digits of 11, 11, 10 bits over the cluster's summed histograms
  uint32_t prefix = 0, pmask = 0, need = 0, n_valid = 0, class_cnt = 0;
  bool take_all = false;
  int pass = 0;
  for (; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dmask = pass < 2 ? 2047u : 1023u;
    for (int i = tid; i < kBins; i += kCluThreads) sm.hist[i] = 0;
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kItems; ++u)
      if (key[u] != 0u && (key[u] & pmask) == prefix) atomicAdd(&sm.hist[(key[u] >> shift) & dmask], 1u);
    __syncthreads();
    uint32_t floor_bin = 0;                               // bins below it are not sent
    if (pass == 0) {
      uint32_t nl = 0;
#pragma unroll
      for (int u = 0; u < kItems; ++u) nl += key[u] != 0u;
      uint32_t d0, d1, d2;
      block_scan2<kCluThreads>(nl, 0u, sm.scr, d0, d1, nl, d2);   // this CTA's valid items
      if (nl > (uint32_t)p.k) {
        find_bin<kCluThreads>(sm.hist, (uint32_t)p.k, sm.scr, sm.res);
        floor_bin = sm.res[0];
      }
      cluster_wait();                                     // every CTA has zeroed its counters
      if (tid < (int)C && nl != 0u) dsmem_add(dsmem_addr(&sm.n_valid, (uint32_t)tid), nl);
      if (tid == 0) CSA_STAMP(56);
    } else if (tid == 0) {
      CSA_STAMP(52);
    }
    for (int i = tid; i < kBins; i += kCluThreads) {
      const uint32_t v = sm.hist[i];
      if (v != 0u && (uint32_t)i >= floor_bin) {
        for (uint32_t r = 0; r < C; ++r) dsmem_add(dsmem_addr(&sm.full[pass][i], r), v);
        if (pass == 0)
          for (uint32_t r = rank + 1; r < C; ++r) dsmem_add(dsmem_addr(&sm.before[i], r), v);
      }
    }
    cluster_sync();                                       // every CTA's additions have landed
    if (tid == 0) CSA_STAMP(pass == 0 ? 57 : 53);
    if (pass == 0) {
      n_valid = sm.n_valid;
      need = min((uint32_t)p.k, n_valid);
      take_all = need >= n_valid;
      if (take_all) break;
    }
    find_bin<kCluThreads>(sm.full[pass], need, sm.scr, sm.res);
    prefix |= sm.res[0] << shift;
    pmask |= dmask << shift;
    need = sm.res[1];
    class_cnt = sm.res[2];
    __syncthreads();                                      // res is written again by the next search
    if (tid == 0) CSA_STAMP(58 + pass);
    if (class_cnt == need || class_cnt <= kListCap) break;   // wholly taken, or split locally
  }
  const uint32_t kk = min((uint32_t)p.k, n_valid);

  // ---- this CTA's items above the class and in it, and their offsets within the CTA
  uint32_t ngt = 0, neq = 0;
#pragma unroll
  for (int u = 0; u < kItems; ++u) {
    const bool valid = key[u] != 0u;
    const uint32_t m = key[u] & pmask;
    ngt += valid && (take_all || m > prefix);
    neq += valid && !take_all && m == prefix;
  }
  uint32_t rg, re, GT, EQ;
  block_scan2<kCluThreads>(ngt, neq, sm.scr, rg, re, GT, EQ);
  // the class is split locally when only part of it is taken and digits remain (the same in every CTA)
  const bool split = !take_all && class_cnt > need && pmask != 0xFFFFFFFFu;
  uint32_t gt_off = 0, eq_off = 0, eq_total = take_all ? 0u : class_cnt;
  if (pass == 0) {
    // resolved by the first digit: the lower-ranked CTAs' counts are in `before` (every bin above
    // the threshold bin, or every bin when all is taken, was sent by every CTA)
    const uint32_t bstar = prefix >> 21;
    uint32_t above = 0;
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const uint32_t bin = kBins - 1 - kItems * tid - u;
      if (take_all || bin > bstar) above += sm.before[bin];
    }
    uint32_t d0, d1, d2;
    block_scan2<kCluThreads>(above, 0u, sm.scr, d0, d1, gt_off, d2);
    eq_off = take_all ? 0u : sm.before[bstar];
  } else {
    // refined by further digits: exchange the counts
    if (tid < (int)C) {
      const uint32_t at = dsmem_addr(&sm.src_cnt[rank][0], (uint32_t)tid);
      dsmem_st(at, GT);
      dsmem_st(at + 4, EQ);
    }
    cluster_sync();                                       // every CTA's counts have landed
    for (uint32_t r = 0; r < rank; ++r) { gt_off += sm.src_cnt[r][0]; eq_off += sm.src_cnt[r][1]; }
  }
  if (tid == 0) CSA_STAMP(61);
  const bool all_eq_taken = take_all || eq_total <= need;
  const bool by_position = !all_eq_taken && !split;       // all 32 bits fixed: equal keys, first `need`
  if (split) {                                            // eq_total <= kListCap here
    // this CTA's in-bin keys go to their row-order positions [eq_off, eq_off + EQ) of the local
    // list first, then to every other CTA, spread evenly over the threads: 16-byte stores for the
    // aligned middle of the segment, single words at its two ends
    uint32_t e = eq_off + re;
#pragma unroll
    for (int u = 0; u < kItems; ++u)
      if (key[u] != 0u && (key[u] & pmask) == prefix) sm.list[e++] = key[u];
    __syncthreads();
    const uint32_t lo = eq_off, hi = eq_off + EQ;
    const uint32_t qlo = min((lo + 3u) & ~3u, hi), qhi = max(hi & ~3u, qlo);
    const uint32_t nq = (qhi - qlo) / 4, n_lo = qlo - lo, items = nq + n_lo + (hi - qhi);
    for (uint32_t w = tid; w < items * (C - 1); w += kCluThreads) {
      const uint32_t item = w / (C - 1), d = w % (C - 1), r = d < rank ? d : d + 1;
      if (item < nq) {
        const uint32_t at = qlo + 4 * item;
        dsmem_st4(dsmem_addr(&sm.list[at], r), *reinterpret_cast<const uint4*>(&sm.list[at]));
      } else {
        const uint32_t j = item - nq, at = j < n_lo ? lo + j : qhi + (j - n_lo);
        dsmem_st(dsmem_addr(&sm.list[at], r), sm.list[at]);
      }
    }
    cluster_sync();                                       // the list is complete: the last barrier
    if (tid == 0) CSA_STAMP(49);
    // the remaining digits of the threshold, over the class's keys only
    uint32_t lp = prefix, lm = pmask, ln = need;
    for (int dp = pass + 1; dp < 3; ++dp) {
      const int shift = dp == 1 ? 10 : 0;
      const uint32_t dmask = dp == 1 ? 2047u : 1023u;
      for (int i = tid; i < kBins; i += kCluThreads) sm.hist[i] = 0;
      __syncthreads();
      for (uint32_t gpos = tid; gpos < eq_total; gpos += kCluThreads) {
        const uint32_t kv = sm.list[gpos];
        if ((kv & lm) == lp) atomicAdd(&sm.hist[(kv >> shift) & dmask], 1u);
      }
      __syncthreads();
      find_bin<kCluThreads>(sm.hist, ln, sm.scr, sm.res);
      lp |= sm.res[0] << shift;
      lm |= dmask << shift;
      ln = sm.res[1];
      const uint32_t cls = sm.res[2];
      __syncthreads();
      if (cls == ln) break;
    }
    // taken: above the final class, or in it and among its first `ln` in row order
    const uint32_t q0 = kListPer * tid;
    uint32_t c = 0;
#pragma unroll
    for (int j = 0; j < kListPer; ++j)
      c += q0 + j < eq_total && (sm.list[q0 + j] & lm) == lp;
    uint32_t ce, d0, d1, d2;
    block_scan2<kCluThreads>(c, 0u, sm.scr, ce, d0, d1, d2);
#pragma unroll
    for (int j = 0; j < kListPer; ++j)
      if (q0 + j < eq_total) {
        const uint32_t m = sm.list[q0 + j] & lm;
        sm.taken[q0 + j] = m > lp || (m == lp && ce++ < ln);
      }
    __syncthreads();
    if (tid == 0) CSA_STAMP(62);
  }
  auto eq_taken = [&](uint32_t gpos) -> bool {
    return all_eq_taken ? true : (by_position ? gpos < need : sm.taken[gpos] != 0);
  };
  // taken in-bin items of the CTAs before this one
  uint32_t tb = 0;
  if (all_eq_taken) tb = eq_off;
  else if (by_position) tb = min(eq_off, need);
  else {
    uint32_t c = 0;
    for (uint32_t gpos = tid; gpos < eq_off; gpos += kCluThreads) c += sm.taken[gpos];
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) sm.scr[tid >> 5] = c;
    __syncthreads();
    for (int w = 0; w < kCluThreads / 32; ++w) tb += sm.scr[w];
    __syncthreads();
  }
  if (tid == 0) CSA_STAMP(63);
  // ---- write the winners in ascending index order
  uint32_t mine = ngt;
  {
    uint32_t e = eq_off + re;
#pragma unroll
    for (int u = 0; u < kItems; ++u)
      if (key[u] != 0u && !take_all && (key[u] & pmask) == prefix) mine += eq_taken(e++);
  }
  uint32_t wex, d2, wtot, d3;
  block_scan2<kCluThreads>(mine, 0u, sm.scr, wex, d2, wtot, d3);
  uint32_t slot = gt_off + tb + wex;
  uint32_t e = eq_off + re;
  int32_t* out = p.topk + row * p.k;
#pragma unroll
  for (int u = 0; u < kItems; ++u) {
    const bool valid = key[u] != 0u;
    const uint32_t m = key[u] & pmask;
    const bool gt = valid && (take_all || m > prefix);
    const bool eq = valid && !take_all && m == prefix;
    bool t_ = gt;
    if (eq) t_ = eq_taken(e++);
    if (t_) out[slot++] = id[u];
  }
  for (int j = (int)kk + (int)(rank * kCluThreads) + tid; j < p.k; j += (int)(C * kCluThreads)) out[j] = -1;
  if (tid == 0) CSA_STAMP(48);
}

cudaError_t launch_cluster_select(const SelParams& p, int64_t rows, int C, cudaStream_t st, bool pdl) {
  cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(CluSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C, (unsigned)rows);
  cfg.blockDim = dim3(kCluThreads);
  cfg.dynamicSmemBytes = sizeof(CluSmem);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  int na = 1;
  if (pdl) {
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    na = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, topk_cluster_kernel, p);
}

template <int kThreads>
cudaError_t launch_select(const SelParams& p, int64_t rows, cudaStream_t st, bool pdl) {
  const size_t smem = SelSmem<kThreads>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(topk_select_kernel<kThreads>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.n_chunks, (unsigned)rows);
  return launch_kernel(pdl, topk_select_kernel<kThreads>, grid, dim3(kThreads), smem, st, p);
}

constexpr int kCapLarge = 1024 * kItems;     // 16384 items: one CTA of 1024 threads
constexpr int kCapMid = 256 * kItems;        // 4096
constexpr int kCapSmall = 128 * kItems;      // 2048

}  // namespace

// A row longer than one small CTA is first cut into 2048-item chunks, one 128-thread CTA each: one
// SM moves only tens of GB/s, so spreading the first pass over many SMs is what makes it fast. The
// chunks' winners (k per chunk, in index order) then go through further levels (2048-item chunks for
// k <= 512, else 16384-item chunks) until one cluster (or CTA) holds a row.
static int64_t first_level_chunks(int64_t n_cap) { return (n_cap + kCapSmall - 1) / kCapSmall; }

size_t topk_workspace_bytes(int64_t rows, int64_t n_cap, int k) {
  // candidates of the intermediate levels: two ping-pong buffers of (key, index) pairs, each large
  // enough for the first level's output. Rows of up to 16384 entries are selected in one launch
  // (one CTA or one cluster) and need none.
  if (n_cap <= (int64_t)kCluMax * kCluChunk || k <= 0) return 0;
  return 2 * (size_t)rows * first_level_chunks(n_cap) * k * 8;
}

cudaError_t launch_topk(int B, const TopkParams& p, cudaStream_t st, bool pdl) {
  if (B == 0 || p.S == 0) return cudaSuccess;
  const int64_t rows = (int64_t)B * p.S;
  SelParams s;
  s.scores = p.scores; s.in_key = nullptr; s.in_idx = nullptr; s.n_in = p.n_cap; s.pos = p.pos;
  s.entry_base = p.entry_base;
  s.S = p.S; s.ratio = p.ratio; s.k = p.k;
  uint8_t* ws = static_cast<uint8_t*>(p.ws);
  const size_t half = topk_workspace_bytes(rows, p.n_cap, p.k) / 2;
  int64_t n_in = p.n_cap;
  for (int level = 0;; ++level) {
    const bool dep = pdl || level > 0;
    const bool fits = n_in <= (int64_t)kCluMax * kCluChunk || (level > 0 && n_in <= kCapLarge);
    if (fits) {                                                // one CTA holds the row: final level
      s.chunk = (int)n_in; s.n_chunks = 1;
      s.topk = p.topk; s.out_key = nullptr; s.out_idx = nullptr;
      if (n_in <= kCapSmall) return launch_select<128>(s, rows, st, dep);
      if (n_in <= (int64_t)kCluMax * kCluChunk)                // one cluster of 2048-item CTAs per row
        return launch_cluster_select(s, rows, (int)((n_in + kCluChunk - 1) / kCluChunk), st, dep);
      if (n_in <= kCapMid) return launch_select<256>(s, rows, st, dep);
      return launch_select<1024>(s, rows, st, dep);
    }
    if (!ws) return cudaErrorInvalidValue;
    // an intermediate level cuts its input into 2048-item chunks, one 128-thread CTA each, while
    // that shrinks it at least 4x (k <= 512: the 1M-token decode goes 262,144 -> 65,536 -> 16,384
    // candidates, then one cluster per row; one 1024-thread CTA per 16,384 items had left 16 CTAs
    // busy for ~39 us there); larger k takes 16,384-item chunks, which shrink it at least 8x
    const bool small = level == 0 || 4 * (int64_t)p.k <= kCapSmall;
    const int64_t cap = small ? kCapSmall : kCapLarge;
    const int64_t chunks = (n_in + cap - 1) / cap;
    const int64_t n_out = chunks * p.k;
    uint8_t* buf = ws + (level & 1) * half;
    s.chunk = (int)cap; s.n_chunks = (int)chunks;
    s.topk = nullptr;
    s.out_key = reinterpret_cast<uint32_t*>(buf);
    s.out_idx = reinterpret_cast<int32_t*>(buf + (size_t)rows * n_out * 4);
    cudaError_t e = small ? launch_select<128>(s, rows, st, dep) : launch_select<1024>(s, rows, st, dep);
    if (e != cudaSuccess) return e;
    s.scores = nullptr; s.pos = nullptr;
    s.in_key = s.out_key; s.in_idx = s.out_idx; s.n_in = n_out;
    n_in = n_out;
  }
}

}  // namespace csa
