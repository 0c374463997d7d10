// K2 + K3 fused for decode: indexer scores on the tensor cores and the exact top-k selection, in
// one launch (bf16 storage, H_idx = 64, d_idx = 128, one query per request).
//
// [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", section "少读 KV 之前，Indexer 仍要给历史打分":
//     s_i = sum_h w_h * max(0, rope(q_h, t) . cidx_i),   i < (t+1)/m,
// w signed, summed over the heads; then the top_k entries are selected (exact, under the order
// (-s_i, i)) and listed in ascending entry index, -1 padded.
//
// One request is one thread-block cluster of C CTAs (one CTA per SM). CTA r of the cluster scores
// the r-th contiguous run of the request's visible 128-entry tiles (TMA ring of cache tiles ->
// tcgen05.mma M = 128 entries x N = 128 (the rotated query as bf16 value and bf16 remainder) x
// K = 128 -> TMEM -> thread-per-entry head reduction), but keeps
// its scores (at most 4096) in shared memory. When every CTA of the cluster has scored its run, the
// cluster selects the request's winners through distributed shared memory, with no global round
// trip and no further launch. The scores become order-preserving 32-bit keys (thread t holds 16
// consecutive entries, so thread order is entry order, and CTA rank order is entry order too) and
// the k-th largest key is found by radix select over 8-bit digits, most significant first:
//   * in each pass every CTA histograms the keys of the current class (those matching the digits
//     fixed so far) into 256 bins and stores the histogram into its row of every CTA's table;
//   * after one cluster barrier every CTA holds the same C rows, finds the same threshold bin,
//     and also reads how many winners above it the lower-ranked CTAs hold;
//   * a pass ends the search when the threshold bin is taken whole; after four passes every bit
//     is fixed and the first keys equal to the threshold, in entry order, fill the remaining slots;
// then every CTA writes its winners at their ascending-index positions (its offset follows from
// the tables, so no further exchange is needed). Every CTA takes part in every cluster barrier on
// every path (the path is decided by data that is identical in all CTAs), so no barrier can wait
// for a CTA that left, and after the last barrier no CTA touches another's shared memory.
//
// The compressor's close step of a decode step runs here too ([FLASH] "压缩是逐通道的 learned
// pooling": when t completes a group, entry t / m is pooled): warps 6 and 7, idle while the cache
// streams, pool the new index entry in the CTA that scores the request's last tile (its TMA load
// waits for it) and the new KV entry in CTA 0 (the attention reads it later).
//
// With the low-precision cache (FP4 E2M1 dims 0..63 with two block scales, FP8 E4M3 dims 64..127;
// lowp.cuh) a tile is three bulk copies (4 KB + 8 KB + 256 B of the cache's planes, 98 instead of 256
// bytes per entry) into a staging ring, and each epilogue thread first expands its TMEM lane's entry
// of tile i into f16 (exact: an E2M1 code times a power of two and an E4M3 code are f16 values, and
// the hardware converts both to f16 in one instruction per pair) and stores it into TMEM, where the
// MMA takes its A operand from, before it reduces tile i-1. Shared-memory bandwidth is what an
// expanded operand in shared memory would cost (32 KB written and read again per tile on top of the
// query operand the MMA reads): TMEM keeps it off that path. The query operand is then f16 as well
// (value and remainder, both f16, of the query scaled per head by a power of two that puts its
// largest element in [256, 512); the head weight carries the inverse scale).
//
// Warps: 0 = TMA producer, 1 = TMEM owner and MMA issuer, 2..5 = query operand and score epilogue
// (TMEM lane quadrant = warp % 4; with the low-precision cache also the expansion of each tile),
// 6..7 = close step; all eight select.
#include <cudaTypedefs.h>

#include "close_entry.cuh"
#include "lowp.cuh"
#include "tc.h"
#include "tc_ptx.cuh"

namespace csa {
namespace {

using namespace tc;

constexpr int kDI = 128;
constexpr int kTileM = 128;
constexpr int kStages = 4;
constexpr uint32_t kTileBytes = kTileM * kDI * 2;           // 32 KB: two 16 KB swizzle blocks
constexpr uint32_t kBlockBytes = 16384;
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 256;                         // two accumulators of 128 columns
// M = 128 entries x N = 128: columns 0..63 the heads' products with the query's value, 64..127 with
// its remainder
constexpr uint32_t kIdesc = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescF16 = idesc_f16(128, 128, false, false);   // low-precision cache: f16 operands
constexpr int kMaxTiles = 32;                               // tiles per CTA
constexpr int kCap = kMaxTiles * kTileM;                    // 4096 entries per CTA
constexpr int kItems = kCap / kThreads;                     // 16 keys per thread
constexpr int kBins8 = 256;                                 // 8-bit digits: one bin per thread
constexpr int kCluMax = 8;
static_assert(kCap % kThreads == 0 && kBins8 == kThreads, "one bin per thread");
// low-precision cache: per tile 128 entries x (32 B of E2M1 codes + 64 B of E4M3 codes + 2 scale bytes)
constexpr uint32_t kQFp8Off = kTileM * 32;                 // 4 KB
constexpr uint32_t kQScaleOff = kQFp8Off + kTileM * 64;    // 12 KB
constexpr uint32_t kQStageBytes = kQScaleOff + kTileM * 2; // 12,544 B
// the expanded f16 tile goes to TMEM (A operand of the MMA): two slots of 64 columns after the two
// 128-column accumulators
constexpr uint32_t kQTmemCols = 512;
constexpr uint32_t kQACol = 256;
// the low-precision tiles are small (12.5 KB): more are kept in flight
constexpr int kQStages = 10;

// Selection tables: row r of a pass's table holds CTA r's histogram of that pass (remote stores).
// The first pass's table is written while this CTA may still be streaming: its own region. The
// later ones, and the local scratch, are written only after the first cluster barrier, when every
// CTA of the cluster has finished streaming: they overlay the TMA ring.
struct SelShared {
  uint32_t hall0[kCluMax * kBins8];
};
struct SelScratch {
  uint32_t hallx[3][kCluMax * kBins8];
  uint32_t hist[kBins8];
  uint32_t scr[64];
  uint32_t res[4];
};


constexpr size_t kOffRing = kTileBytes;                                  // after the query operand

// shared-memory layout of each variant: [query operand][ring][scores][selection tables][barriers ...]
template <bool kLowp>
struct Layout {
  static constexpr int kSt = kLowp ? kQStages : kStages;                 // loads in flight
  static constexpr size_t kRing = kLowp ? kQStages * kQStageBytes : kStages * kTileBytes;
  static constexpr size_t kOffScores = kOffRing + kRing;
  static constexpr size_t kOffSel = kOffScores + kCap * sizeof(float);
  static constexpr size_t kOffBars = kOffSel + sizeof(SelShared);
  static constexpr size_t kSmem = 1024 /*align*/ + kOffBars + 1536;   // barriers, weights, tables
  static_assert(kSmem <= 232448, "shared memory of one CTA");
  static_assert(kRing >= sizeof(SelScratch), "the selection scratch overlays the ring");
};

struct IndexSelParams {
  const __nv_bfloat16* q_idx;   // [B, 64, 128]
  const float* w;               // [B, 64]
  float* scores;                // [B, n_cap] or null (not stored)
  int32_t* topk;                // [B, k]
  const int64_t* pos;           // [B]
  int64_t n_cap;
  int ratio, k;
  RopeTab rope;
  int32_t* err;
  // the entry that t closes is pooled here (close.job[0].src non-null): KV entry by CTA 0, index
  // entry by the CTA that scores the last tile
  CompressParams close;
  // the compressed KV cache (bf16 [B, n_cap, 512] or the low-precision planes), or null: each winner's
  // row is requested into L2 as soon as it is known, so that the attention's gather finds it there
  const void* ckv_prefetch;
  const uint8_t* cidx_q;        // the low-precision index cache (kLowp)
  // timeout test hook: skip the first cache-tile load and wait at most wait_ns (else 1 s)
  int test_stall;
  uint64_t wait_ns;
};

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;                        // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// block-wide exclusive scan of two counters per thread, thread order; scratch holds 64 words
__device__ __forceinline__ void block_scan2(uint32_t a, uint32_t b, uint32_t* scratch, uint32_t& ea, uint32_t& eb,
                                            uint32_t& ta, uint32_t& tb) {
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

template <bool kLowp>
__global__ void __launch_bounds__(kThreads, 1)
    index_select_kernel(const __grid_constant__ CUtensorMap cmap, const IndexSelParams p) {
  using Lay = Layout<kLowp>;
  constexpr int kSt = Lay::kSt;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* qop = smem;                                      // [2 blocks][128 rows][128 B]
  uint8_t* stage_base = smem + kOffRing;                    // kSt x [2 blocks][128 rows][128 B]
  float* sc = reinterpret_cast<float*>(smem + Lay::kOffScores);  // [kCap] scores of this CTA's entries
  SelShared& sh = *reinterpret_cast<SelShared*>(smem + Lay::kOffSel);
  SelScratch& sx = *reinterpret_cast<SelScratch*>(stage_base);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBars);
  uint64_t* full = bars;                                    // [kSt]
  uint64_t* empty = bars + kSt;                         // [kSt]
  uint64_t* tfull = bars + 2 * kSt;                     // [2]
  uint64_t* tempty = bars + 2 * kSt + 2;                // [2]
  uint64_t* qready = bars + 2 * kSt + 4;
  uint64_t* closed = bars + 2 * kSt + 5;                // the index entry is in global memory
  uint64_t* opfull = bars + 2 * kSt + 6;                // [2] kLowp: TMEM operand slot written
  uint64_t* opempty = bars + 2 * kSt + 8;               // [2] kLowp: operand slot read by the MMA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kSt + 10);
  uint8_t* qstage = stage_base;                             // kLowp: kSt x kQStageBytes
  float* w_s = reinterpret_cast<float*>(tmem_slot + 4);    // [64]
  float* red = w_s + 64;                                    // [4]
  float* hsc = red + 4;                                     // [64] kLowp: inverse query scale per head
  float* q_cs = hsc + 64;                                   // [32] cos / sin of the query's RoPE angles
  float* q_sn = q_cs + 32;                                  // [32]

  if (threadIdx.x == 0) CSA_STAMP(42);
  griddep_launch();
  griddep_wait();                                           // a no-op unless launched as a dependent
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int b = blockIdx.y;
  const uint32_t rank = cluster_rank(), C = gridDim.x;
  const int64_t t = p.pos[b];
  const int64_t V = t < 0 ? 0 : min(visible_entries(t, p.ratio), p.n_cap);
  const int64_t T = (V + kTileM - 1) / kTileM;
  const int64_t tile0 = (int64_t)rank * T / C;
  const int64_t tile1 = (int64_t)(rank + 1) * T / C;
  const int ntiles = (int)(tile1 - tile0);                  // <= kMaxTiles (checked by the launcher)
  const int n_local = (int)max((int64_t)0, min(V, tile1 * kTileM) - tile0 * kTileM);
  const bool fused = p.close.job[0].src != nullptr;
  const bool group_done = fused && t >= 0 && t < p.close.N && (t + 1) % p.ratio == 0;
  if (fused && rank == 0 && threadIdx.x == 0 &&
      (t < 0 || t >= p.close.N || (group_done && t / p.ratio >= p.n_cap)))
    set_error(p.err, DEVERR_BAD_POS);
  const bool closes = group_done && t / p.ratio < p.n_cap;  // then entry e = V - 1 is the last visible
  const bool close_kv = closes && rank == 0;
  const bool close_idx = closes && tile1 == T && ntiles > 0;   // the CTA that scores entry e

  // the query loads go out first: they are the longest latency of the prologue
  const int et = tid - 64;                                  // epilogue thread 0..127 (warps 2..5)
  const int qc = et & 15, qh0 = et >> 4;                    // 8-dim chunk qc of heads qh0 + 8 i
  float xs[8][8];
  float wv = 0.f;
  if (warp >= 2 && warp < 6) {
    const __nv_bfloat16* q = p.q_idx + (int64_t)b * 64 * kDI;
#pragma unroll
    for (int i = 0; i < 8; ++i) load8(q + (qh0 + 8 * i) * kDI + qc * 8, xs[i]);
    if (et < 64) wv = p.w[(int64_t)b * 64 + et];
  }
  if (threadIdx.x == 0) {
    // kLowp: a staging slot is released by the 128 expanding threads, not by the MMA
    for (int i = 0; i < kSt; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], kLowp ? 128 : 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&tfull[i], 1); mbar_init(&tempty[i], 128); }
    for (int i = 0; i < 2; ++i) { mbar_init(&opfull[i], 128); mbar_init(&opempty[i], 1); }
    mbar_init(qready, 128);
    mbar_init(closed, 64);
    fence_mbar_init();
  }
  constexpr uint32_t kCols = kLowp ? kQTmemCols : kTmemCols;
  if (warp == 1) { tmem_alloc(tmem_slot, kCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive();                                         // this CTA runs: its tables may be written
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && ntiles > 0) {
      if (!kLowp) prefetch_tensormap(&cmap);
      const uint64_t policy = l2_evict_first_policy();      // the cache streams through once
      const LowpLayout lay = lowp_layout(kDI, p.n_cap, 64);
      const uint8_t* qb = kLowp ? p.cidx_q + (int64_t)b * lay.stride : nullptr;
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % kSt;
        if (i >= kSt && !mbar_wait(&empty[st], ((i / kSt) & 1) ^ 1, p.err, p.wait_ns)) break;
        if (close_idx && i == ntiles - 1 && !mbar_wait(closed, 0, p.err, p.wait_ns)) break;   // holds entry e
        if (p.test_stall && i == 0) continue;                // the timeout test hook
        if constexpr (kLowp) {
          // the tile's entries of each plane (never past n_cap; the scale run rounded up to 8
          // entries, which the plane's 16-byte padding holds)
          const int64_t e0 = (tile0 + i) * kTileM;
          const uint32_t ne = (uint32_t)min((int64_t)kTileM, p.n_cap - e0), ne8 = (ne + 7) & ~7u;
          uint8_t* dst = qstage + st * kQStageBytes;
          mbar_arrive_expect_tx(&full[st], ne * 32 + ne * 64 + ne8 * 2);
          bulk_load_hint(dst, qb + e0 * 32, ne * 32, &full[st], policy);
          bulk_load_hint(dst + kQFp8Off, qb + lay.fp8 + e0 * 64, ne * 64, &full[st], policy);
          bulk_load_hint(dst + kQScaleOff, qb + lay.scale + e0 * 2, ne8 * 2, &full[st], policy);
        } else {
          mbar_arrive_expect_tx(&full[st], kTileBytes);
          const int32_t y = (int32_t)(b * p.n_cap + (tile0 + i) * kTileM);
          uint8_t* dst = stage_base + st * kTileBytes;
          tma_load_2d_hint(dst, &cmap, &full[st], 0, y, policy);
          tma_load_2d_hint(dst + kBlockBytes, &cmap, &full[st], 64, y, policy);
        }
        issued = i + 1;
        if (i == 16) CSA_STAMP(55);
      }
      // no copy may still be landing in the ring when the selection reuses it (after a wait that
      // ran out, loads can be left unconsumed): wait, bounded, for the last load of every stage
      for (int i = issued > kSt ? issued - kSt : 0; i < issued; ++i)
        if (!(p.test_stall && i == 0)) mbar_wait(&full[i % kSt], (i / kSt) & 1, p.err, p.wait_ns);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && ntiles > 0 && mbar_wait(qready, 0, p.err, p.wait_ns)) {
      tc_fence_after();
      const uint32_t q_addr = smem_u32(qop);
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % kSt, acc = i & 1;
        if (kLowp ? !mbar_wait(&opfull[acc], (i >> 1) & 1, p.err, p.wait_ns)
                  : !mbar_wait(&full[st], (i / kSt) & 1, p.err, p.wait_ns))
          break;
        if (i >= 2 && !mbar_wait(&tempty[acc], ((i >> 1) & 1) ^ 1, p.err, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * 128;
        if constexpr (kLowp) {                                // A (the expanded tile) in TMEM
          const uint32_t a_tm = tmem + kQACol + acc * 64;
#pragma unroll
          for (int kk = 0; kk < kDI / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBlockBytes + (kk & 3) * 32;
            mma_f16_tmem_a(d, a_tm + kk * 8, desc_kmajor_sw128(q_addr + off), kIdescF16, kk > 0);
          }
        } else {
          const uint32_t a_addr = smem_u32(stage_base + st * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kDI / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBlockBytes + (kk & 3) * 32;
            mma_bf16(d, desc_kmajor_sw128(a_addr + off), desc_kmajor_sw128(q_addr + off), kIdesc, kk > 0);
          }
        }
        mma_commit(kLowp ? &opempty[acc] : &empty[st]);
        mma_commit(&tfull[acc]);
      }
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------------- query operand + epilogue
    // rotated query (RoPE on dims 64..127 at t), split into bf16 value (rows 0..63) and bf16
    // remainder (rows 64..127) of the N = 128 operand
    const int r0 = kDI - p.rope.d_rope;
    // each of the d_rope / 2 angles once (thread et), shared through shared memory
    if (et < p.rope.d_rope / 2) rope_cs(t, p.rope, et, q_cs[et], q_sn[et]);
    named_barrier(1, 128);
    float cs4[4], sn4[4];
    const bool rot = qc * 8 >= r0;
    if (rot) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        cs4[k] = q_cs[(qc * 8 - r0) / 2 + k];
        sn4[k] = q_sn[(qc * 8 - r0) / 2 + k];
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float* x = xs[i];
      if (rot) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float a = x[2 * k], bb = x[2 * k + 1];
          x[2 * k] = a * cs4[k] - bb * sn4[k];
          x[2 * k + 1] = a * sn4[k] + bb * cs4[k];
        }
      }
      const int h = qh0 + 8 * i, blk = qc >> 3, ch = qc & 7;
      if constexpr (kLowp) {
        // head h's 128 dims sit in the 16 lanes that share qh0: scale them by 2^sh so that the
        // largest lies in [256, 512), then split into f16 value and f16 remainder
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int ef = (int)((__float_as_uint(amax) >> 23) & 255u) - 127;
        const int sh = amax > 0.f ? max(-126, min(126, 8 - ef)) : 0;
        const float scl = __uint_as_float((uint32_t)(sh + 127) << 23);
        uint4 uh, ul;
        uint32_t* ph = &uh.x;
        uint32_t* pl = &ul.x;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float a = x[2 * k] * scl, bb = x[2 * k + 1] * scl;
          const __half2 hv = __floats2half2_rn(a, bb);
          const float2 hf = __half22float2(hv);
          const __half2 lv = __floats2half2_rn(a - hf.x, bb - hf.y);
          ph[k] = *reinterpret_cast<const uint32_t*>(&hv);
          pl[k] = *reinterpret_cast<const uint32_t*>(&lv);
        }
        *reinterpret_cast<uint4*>(qop + blk * kBlockBytes + sw128_offset(h, ch)) = uh;
        *reinterpret_cast<uint4*>(qop + blk * kBlockBytes + sw128_offset(64 + h, ch)) = ul;
        if (qc == 0) hsc[h] = __uint_as_float((uint32_t)(127 - sh) << 23);
      } else {
        float hi[8], lo[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          hi[k] = __bfloat162float(__float2bfloat16_rn(x[k]));
          lo[k] = x[k] - hi[k];
        }
        store8(reinterpret_cast<__nv_bfloat16*>(qop + blk * kBlockBytes + sw128_offset(h, ch)), hi);
        store8(reinterpret_cast<__nv_bfloat16*>(qop + blk * kBlockBytes + sw128_offset(64 + h, ch)), lo);
      }
    }
    if constexpr (kLowp) {
      named_barrier(1, 128);                                // every head's scale is in hsc
      if (et < 64) w_s[et] = wv * hsc[et];
    } else {
      if (et < 64) w_s[et] = wv;
    }
    if (et == 0) CSA_STAMP(43);
    fence_proxy_async_smem();
    mbar_arrive(qready);
    named_barrier(1, 128);                                  // w_s visible to every epilogue thread

    const uint32_t quad = warp & 3;                         // TMEM lanes 32*quad .. 32*quad+31
    const int row_in_tile = quad * 32 + lane;
    float* gout = p.scores ? p.scores + (int64_t)b * p.n_cap : nullptr;
#ifdef CSA_TRACE
    unsigned long long tw_tf = 0;
#endif
    auto epilogue = [&](int i) -> bool {
      const int acc = i & 1;
#ifdef CSA_TRACE
      const unsigned long long e0_ = global_timer_ns();
#endif
      if (!mbar_wait_warp(&tfull[acc], (i >> 1) & 1, p.err, p.wait_ns)) return false;   // uniform over the warp
#ifdef CSA_TRACE
      tw_tf += global_timer_ns() - e0_;
      if (et == 0 && i == ntiles - 1) CSA_TRACE_VAL(36, tw_tf);
#endif
      tc_fence_after();
      const uint32_t ta = tmem + ((quad * 32) << 16) + acc * 128;
      // four partial sums (heads h = k mod 4): four short dependency chains instead of one of 64.
      // The loop over the two halves stays rolled: this loop and the expansion run once per tile
      // on the same SMs as the other roles' loops, and what limits them is instruction fetch
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
      const float4* w4 = reinterpret_cast<const float4*>(w_s);
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t hv[32], lv[32];
        tmem_ld32(ta + half * 32, hv);
        tmem_ld32(ta + 64 + half * 32, lv);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 wj = w4[half * 8 + j];
          const float wv4[4] = {wj.x, wj.y, wj.z, wj.w};
#pragma unroll
          for (int k = 0; k < 4; ++k)
            s4[k] = fmaf(wv4[k], fmaxf(__uint_as_float(hv[4 * j + k]) + __uint_as_float(lv[4 * j + k]), 0.f), s4[k]);
        }
      }
      const float s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      const int li = i * kTileM + row_in_tile;
      sc[li] = s;
      if (gout && li < n_local) gout[tile0 * kTileM + li] = s;
      return true;
    };
    if constexpr (kLowp) {
      // tile i: this thread expands its TMEM lane's entry row of the staged codes (dims 0..63: E2M1 x
      // the block's scale, dims 64..127: E4M3) into f16 operand slot i % 2 in TMEM (the A operand of
      // the MMA: no shared-memory round trip), then reduces tile i-1
#ifdef CSA_TRACE
      unsigned long long tw_full = 0, tw_op = 0;
#endif
      auto expand = [&](int i) -> bool {
        const int st = i % kSt, slot = i & 1;
#ifdef CSA_TRACE
        const unsigned long long w0_ = global_timer_ns();
#endif
        if (!mbar_wait_warp(&full[st], (i / kSt) & 1, p.err, p.wait_ns)) return false;
#ifdef CSA_TRACE
        const unsigned long long w1_ = global_timer_ns();
#endif
        if (i >= 2 && !mbar_wait_warp(&opempty[slot], ((i >> 1) & 1) ^ 1, p.err, p.wait_ns)) return false;
#ifdef CSA_TRACE
        if (et == 0) {
          tw_full += w1_ - w0_;
          tw_op += global_timer_ns() - w1_;
        }
#endif
        tc_fence_after();                                   // the MMA that read this slot is done
        const uint8_t* sp = qstage + st * kQStageBytes;
        const int r = row_in_tile;                          // this thread's TMEM lane
        const uint32_t sc2 = *reinterpret_cast<const uint16_t*>(sp + kQScaleOff + r * 2);
        const uint32_t s0 = e8m0_to_h2(sc2 & 255u), s1 = e8m0_to_h2(sc2 >> 8);
        const uint32_t a_tm = tmem + ((quad * 32) << 16) + kQACol + slot * 64;
        uint32_t v[32];
        {                                                   // dims 0..63: columns 0..31 of the slot
          const uint4 c0 = *reinterpret_cast<const uint4*>(sp + r * 32);
          const uint4 c1 = *reinterpret_cast<const uint4*>(sp + r * 32 + 16);
          const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 h = expand_fp4x8_f16(cw[c], c < 4 ? s0 : s1);
            v[4 * c] = h.x; v[4 * c + 1] = h.y; v[4 * c + 2] = h.z; v[4 * c + 3] = h.w;
          }
          tmem_st32(a_tm, v);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {                       // dims 64..127: columns 32..63
          const uint4 f = *reinterpret_cast<const uint4*>(sp + kQFp8Off + r * 64 + j * 16);
          const uint4 h0 = expand_fp8x8_f16(f.x, f.y), h1 = expand_fp8x8_f16(f.z, f.w);
          v[8 * j] = h0.x; v[8 * j + 1] = h0.y; v[8 * j + 2] = h0.z; v[8 * j + 3] = h0.w;
          v[8 * j + 4] = h1.x; v[8 * j + 5] = h1.y; v[8 * j + 6] = h1.z; v[8 * j + 7] = h1.w;
        }
        tmem_st32(a_tm + 32, v);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&empty[st]);
        mbar_arrive(&opfull[slot]);
        return true;
      };
#ifdef CSA_TRACE
      unsigned long long t_exp = 0, t_epi = 0;
#endif
      for (int i = 0; i <= ntiles; ++i) {
#ifdef CSA_TRACE
        const unsigned long long ta_ = global_timer_ns();
#endif
        if (i < ntiles && !expand(i)) break;
        if (et == 0 && (i == 8 || i == 16 || i == 24)) CSA_STAMP(50 + i / 8);
#ifdef CSA_TRACE
        const unsigned long long tb_ = global_timer_ns();
#endif
        if (i >= 1 && !epilogue(i - 1)) break;
#ifdef CSA_TRACE
        t_exp += tb_ - ta_;
        t_epi += global_timer_ns() - tb_;
#endif
      }
#ifdef CSA_TRACE
      if (et == 0) {
        CSA_TRACE_VAL(32, t_exp);
        CSA_TRACE_VAL(33, t_epi);
        CSA_TRACE_VAL(34, tw_full);
        CSA_TRACE_VAL(35, tw_op);
      }
#endif
    } else {
      for (int i = 0; i < ntiles; ++i)
        if (!epilogue(i)) break;
    }
  } else {
    // ---------------------------------------------------------------- close step (warps 6, 7)
    const int ct = tid - 192;                               // 0..63
    const int64_t e = t / p.ratio;
    if (close_kv)
      close_entry_bf16<512, 64, kLowp>(p.close.job[0], p.close.N, p.n_cap, p.ratio, p.close.eps, p.close.rope, b, e,
                                       ct, red, 2);
    if (close_idx) {
      close_entry_bf16<128, 64, kLowp>(p.close.job[1], p.close.N, p.n_cap, p.ratio, p.close.eps, p.close.rope, b, e,
                                       ct, red + 2, 2);
      fence_proxy_async_global();                           // the TMA load of the last tile reads it
      mbar_arrive(closed);
    }
  }
  tc_fence_before();
  __syncthreads();                                          // every score of this CTA is in sc
  if (threadIdx.x == 0) CSA_STAMP(44);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }

  // ==================================================================== cluster selection
  // Radix select over 8-bit digits of the keys, most significant first. In each pass every CTA
  // histograms its keys of the current class (the keys that match the digits fixed so far) and
  // stores the histogram into its own row of every CTA's table; after the cluster barrier every
  // CTA holds all C histograms, so every CTA finds the same threshold bin and also knows how many
  // of the winners above it lie in lower-ranked CTAs (their entries come first in the output).
  uint32_t key[kItems];
  const int i0 = tid * kItems;
#pragma unroll
  for (int u = 0; u < kItems; ++u) key[u] = i0 + u < n_local ? order_key(sc[i0 + u]) : 0u;
  const uint32_t k = (uint32_t)p.k;
  uint32_t prefix = 0, pmask = 0, need = 0, n_valid = 0;
  uint32_t gt_lower = 0;                 // winners above the final class held by lower-ranked CTAs
  uint32_t eq_lower = 0;                 // keys of the final class held by lower-ranked CTAs
  bool take_all = false;
  const int bin = (kBins8 - 1) - tid;    // this thread's bin (threads scan the bins top down)
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    uint32_t* hall = pass == 0 ? sh.hall0 : sx.hallx[pass - 1];      // [kCluMax][kBins8]
    sx.hist[tid] = 0u;
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kItems; ++u)
      if (key[u] != 0u && (key[u] & pmask) == prefix) atomicAdd(&sx.hist[(key[u] >> shift) & 255u], 1u);
    __syncthreads();
    const uint32_t v = sx.hist[tid];
    if (pass == 0) cluster_wait();       // every CTA of the cluster is running
    for (uint32_t r = 0; r < C; ++r) dsmem_st(dsmem_addr(&hall[rank * kBins8 + tid], r), v);
    cluster_sync();                      // every CTA's histogram is in every table
    if (tid == 0) CSA_STAMP(45 + pass);
    uint32_t tot = 0, low = 0;
    for (uint32_t r = 0; r < C; ++r) {
      const uint32_t h = hall[r * kBins8 + bin];
      tot += h;
      if (r < rank) low += h;
    }
    uint32_t ex_tot, ex_low, all_tot, all_low;
    block_scan2(tot, low, sx.scr, ex_tot, ex_low, all_tot, all_low);
    if (pass == 0) {
      n_valid = all_tot;
      need = min(k, n_valid);
      if (need == n_valid) {             // every visible entry is selected (uniform over the cluster)
        take_all = true;
        gt_lower = all_low;
        break;
      }
    }
    if (ex_tot < need && need <= ex_tot + tot) {
      sx.res[0] = (uint32_t)bin;
      sx.res[1] = need - ex_tot;
      sx.res[2] = tot;
      sx.res[3] = ex_low;
    }
    __syncthreads();
    const uint32_t bstar = sx.res[0], cls = sx.res[2];
    need = sx.res[1];
    gt_lower += sx.res[3];
    prefix |= bstar << shift;
    pmask |= 255u << shift;
    eq_lower = 0;
    for (uint32_t r = 0; r < rank; ++r) eq_lower += hall[r * kBins8 + bstar];
    if (cls == need) break;              // the whole class is taken (uniform over the cluster)
    // after the last pass every bit is fixed: the class holds equal keys, the first `need` of them
    // in entry order are taken
  }
  if (tid == 0) CSA_STAMP(49);
  // ---- this CTA's winners: keys above the class, and class keys whose cluster-wide position in
  // entry order is below `need`; they go to the output in ascending entry index
  uint32_t na = 0, nc = 0;
#pragma unroll
  for (int u = 0; u < kItems; ++u) {
    const bool valid = key[u] != 0u;
    const uint32_t m = key[u] & pmask;
    na += valid && (take_all || m > prefix);
    nc += valid && !take_all && m == prefix;
  }
  uint32_t ea, ec, ta, tcl;
  block_scan2(na, nc, sx.scr, ea, ec, ta, tcl);
  uint32_t cpos = eq_lower + ec;         // cluster-wide class position of this thread's next class key
  uint32_t slot = gt_lower + min(eq_lower, need) + ea + (need > eq_lower ? min(need - eq_lower, ec) : 0u);
  int32_t* out = p.topk + (int64_t)b * p.k;
  const int64_t id0 = tile0 * kTileM + i0;                  // entry index of key[0]
#pragma unroll
  for (int u = 0; u < kItems; ++u) {
    const bool valid = key[u] != 0u;
    const uint32_t m = key[u] & pmask;
    bool win = valid && (take_all || m > prefix);
    if (valid && !take_all && m == prefix) win = cpos++ < need;
    if (win && slot < k) {
      out[slot++] = (int32_t)(id0 + u);
      if (p.ckv_prefetch) {
        const int64_t e = id0 + u;
        if constexpr (kLowp) {                 // the entry's three pieces: 224 + 64 + 16 bytes
          const LowpLayout kl = lowp_layout(512, p.n_cap, 64);
          const uint8_t* kb = static_cast<const uint8_t*>(p.ckv_prefetch) + (int64_t)b * kl.stride;
          prefetch_l2(kb + e * 224, 224);
          prefetch_l2(kb + kl.fp8 + e * 64, 64);
          prefetch_l2(kb + kl.scale + e * 16, 16);
        } else {
          prefetch_l2(static_cast<const __nv_bfloat16*>(p.ckv_prefetch) + ((int64_t)b * p.n_cap + e) * 512, 1024);
        }
      }
    }
  }
  const uint32_t kk = min(k, n_valid);
  for (int j = (int)kk + (int)(rank * kThreads) + tid; j < p.k; j += (int)(C * kThreads)) out[j] = -1;
  if (tid == 0) CSA_STAMP(63);
}

}  // namespace

// Cluster size for B requests whose visible entries are at most n_cap, or 0 when the fused kernel
// does not apply (a request needs more than kCluMax CTAs of kMaxTiles tiles, or the cluster cannot
// be placed). One CTA per SM: as many CTAs per request as keep the batch in one wave, at least
// enough for the tiles, at most kCluMax.
int tc_index_select_cluster(int B, int64_t n_cap) {
  if (B <= 0) return 0;
  const int64_t tiles = (n_cap + kTileM - 1) / kTileM;
  const int c_min = (int)((tiles + kMaxTiles - 1) / kMaxTiles);
  if (c_min > kCluMax) return 0;
  int c = tc_sm_count() / B;
  if (c > kCluMax) c = kCluMax;
  if (c < c_min) c = c_min;
  if (c < 1) c = 1;
  static int fits[kCluMax + 1] = {0};                       // 1 = placeable, -1 = not, 0 = unknown
  if (!fits[c]) {
    cudaError_t e = cudaFuncSetAttribute(index_select_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Layout<false>::kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(index_select_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)Layout<true>::kSmem);
    int n = 0;
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)c, 1);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = Layout<true>::kSmem;              // the larger of the two variants
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)c;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&n, index_select_kernel<true>, &cfg);
    }
    if (e != cudaSuccess) (void)cudaGetLastError();
    fits[c] = (e == cudaSuccess && n > 0) ? 1 : -1;
  }
  return fits[c] > 0 ? c : 0;
}

cudaError_t tc_index_select(int B, int C, const int64_t* pos, const void* q_idx, const float* w, const void* cidx,
                            int64_t n_cap, int ratio, int top_k, const RopeTab& rope, float* scores, int32_t* topk,
                            int32_t* err, cudaStream_t st, bool pdl, const CompressParams* close,
                            const void* ckv_prefetch, bool test_stall, bool lowp) {
  if (C < 1 || C > kCluMax || top_k < 1) return cudaErrorInvalidValue;
  const int64_t tiles = (n_cap + kTileM - 1) / kTileM;
  if ((tiles + C - 1) / C > kMaxTiles) return cudaErrorInvalidValue;
  if ((int64_t)B * n_cap >= (int64_t)1 << 31) return cudaErrorInvalidValue;
  const size_t smem = lowp ? Layout<true>::kSmem : Layout<false>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(lowp ? index_select_kernel<true> : index_select_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  CUtensorMap map;
  memset(&map, 0, sizeof map);                                // unused with the low-precision cache
  if (!lowp) {
    e = make_tmap_2d(&map, cidx, (int64_t)B * n_cap, kDI, kTileM);
    if (e != cudaSuccess) return e;
  }
  IndexSelParams p;
  p.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  p.w = w; p.scores = scores; p.topk = topk; p.pos = pos; p.n_cap = n_cap; p.ratio = ratio; p.k = top_k;
  p.rope = rope; p.err = err;
  p.ckv_prefetch = ckv_prefetch;
  p.cidx_q = lowp ? static_cast<const uint8_t*>(cidx) : nullptr;
  p.test_stall = test_stall ? 1 : 0;
  p.wait_ns = test_stall ? 2000000ull : kWaitTimeoutNs;
  memset(&p.close, 0, sizeof p.close);
  if (close) {
    if (close->n_jobs != 2 || close->job[0].C != 512 || close->job[1].C != kDI) return cudaErrorInvalidValue;
    p.close = *close;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C, (unsigned)B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
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
  return cudaLaunchKernelEx(&cfg, lowp ? index_select_kernel<true> : index_select_kernel<false>, map, p);
}

}  // namespace csa
