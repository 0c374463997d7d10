// K4: sparse joint attention on the 5th-generation tensor cores (bf16 storage, H = 64, d = 512).
//
// [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", section "局部和压缩记忆，共用一次归一化": the raw
// window entries and the selected compressed entries form ONE candidate set under one softmax, and
// each head's sink only enlarges the denominator (the merge kernel adds it). One shared 512-dim KV
// head serves all 64 query heads (K = V), so a tile of 128 candidates is a dense contraction:
//     S^T[c, h] = sum_d KV[c, d] Q[h, d]            (M = 128 candidates, N = 64 heads, K = 512)
//     O^T[d, h] = sum_c KV[c, d] P[h, c]            (M = 4 x 128 dims,   N = 64 heads, K = 128)
// The same shared-memory KV data is the K-major A operand of the first product and, read along
// the other axis, the MN-major A operand of the second.
//
// One CTA = one query and one or two 128-candidate tiles (window tiles first, then compressed
// tiles). Decode batches use one tile per CTA: the grid lists every query's window tile first and
// those CTAs never wait for the selection kernel, so under programmatic dependent launch they run
// while the selection is still being computed; the compressed tiles follow, and every CTA asks L2
// for all of its rows at once before its first gather. A tile streams through a 4-stage ring in
// 32 KB K-chunks (128 candidates x 128 dims); with two tiles per CTA the last tile of the S^T phase
// stays resident for the O^T phase and only the other one is gathered again (an L2 hit).
// Warps:
//   0    loads Q by TMA and issues every tcgen05.mma (one thread);
//   1..5 gather the candidate rows with 16-byte cp.async straight into the 128-byte swizzled layout
//        (random 1 KB rows: an SM sustains only tens of GB/s of such gathers, so many threads issue
//        them and several chunks stay in flight); empty slots are zero-filled. Warp 1 also owns
//        TMEM. Warps 2..5 (thread = candidate row = TMEM lane) then run the softmax on S^T read from
//        TMEM: per-head max and sum by a butterfly reduce-scatter across lanes plus a 4-warp
//        combine, P^T (bf16) into shared memory, and finally write the split partial (max, sum, O);
//   6    rotates the query at t (RoPE on dims 448..511) in shared memory. Raw window rows are
//        rotated at their own positions by the gather threads, each in the pieces it copied;
//   7..  only gather: one SM issues scattered 16-byte copies faster with more warps issuing them
//        (the CTA holds the whole SM, so the extra warps cost no occupancy).
// HCA takes every visible entry, so a compressed tile whose 128 rows are all visible is one
// contiguous run of the cache: it is loaded by TMA (two 64-column boxes per chunk, straight into the
// swizzled layout) instead of 2,048 scattered copies; a partly visible tile keeps the gather, which
// zero-fills its empty rows.
#include <cudaTypedefs.h>

#include "tc.h"
#include "tc_ptx.cuh"

namespace csa {
namespace {

using namespace tc;

constexpr int kD = 512;
constexpr int kH = 64;
constexpr int kTile = 128;
constexpr int kMaxTiles = 2;                        // tiles per CTA
constexpr int kGatherOnlyWarps = 4;                // warps 7.. : gather only
constexpr int kThreads = 224 + 32 * kGatherOnlyWarps;
constexpr int kStages = 4;                          // = chunks per tile: chunk c always uses stage c
constexpr uint32_t kBlk = kTile * 128;              // 16 KB: [128 rows][64 dims] swizzled
constexpr uint32_t kChunkBytes = 2 * kBlk;          // 32 KB: 128 rows x 128 dims
constexpr uint32_t kQBlock = kH * 128;              // 8 KB: [64 heads][64 dims]
constexpr uint32_t kQBytes = 8 * kQBlock;           // 64 KB
constexpr uint32_t kPBytes = kTile * 128;           // 16 KB per tile: P^T, one 128-byte line per candidate
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = kMaxTiles * kH;          // O^T[dc] at kColO + 64 dc
constexpr uint32_t kIdescS = idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdescO = idesc_bf16(128, 64, true, true);
constexpr int kGatherThreads = 160 + 32 * kGatherOnlyWarps;   // warps 1..5 and 7..
constexpr size_t kAuxBytes = 2048;                   // barriers, row table, RoPE table (< 1.5 KB)
constexpr size_t kSmemBytes = 1024 + kQBytes + kStages * kChunkBytes + kMaxTiles * kPBytes + kAuxBytes;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnTcParams {
  const __nv_bfloat16* kv;   // [B, N, 512] raw rows (for L2 prefetch; loads go through the tensor maps)
  const __nv_bfloat16* ckv;  // [B, n_cap, 512]
  const int32_t* topk;       // [B, S, k] or null (HCA)
  const int64_t* pos;        // [B, S] or null (t = s)
  float* part_o;             // [B, S, n_split, H, 512]
  float* part_ml;            // [B, S, n_split, H, 2]
  int64_t N, n_cap;
  int S, k, ratio, window, n_split, win_tiles, tiles_per_cta;
  float scale;
  RopeTab rope;
  int32_t* err;
};

// The loads of one CTA, in order: S^T phase i = 0 .. 4 nt - 1 (tile slot i / 4, chunk i % 4, fill
// i / 4 of stage i % 4), then, for two tiles, the re-gather of tile slot 0 (fill 2 of stages 0..3).
struct LoadSeq {
  int nt;
  __device__ int count() const { return 4 * nt + (nt > 1 ? 4 : 0); }
  __device__ void at(int i, int& j, int& c, int& fill) const {
    if (i < 4 * nt) { j = i >> 2; c = i & 3; fill = i >> 2; }
    else { j = 0; c = i - 4 * nt; fill = 2; }
  }
};

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap cmap,
                   const AttnTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* qs = smem;                                          // [8 blocks][64 heads][128 B]
  uint8_t* ring = qs + kQBytes;                                // kStages x [2 blocks][128 rows][128 B]
  uint8_t* ps = ring + kStages * kChunkBytes;                  // kMaxTiles x [128 rows][128 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ps + kMaxTiles * kPBytes);
  uint64_t* full = bars;                                       // [kStages] (kGatherThreads arrivals)
  uint64_t* empty = bars + kStages;                            // [kStages] (MMA commit)
  uint64_t* bar_q = bars + 2 * kStages;                        // Q bytes landed (tx)
  uint64_t* bar_qrot = bar_q + 1;                              // Q rotated (32 arrivals)
  uint64_t* bar_s = bar_q + 2;                                 // S^T complete
  uint64_t* bar_p = bar_q + 3;                                 // P^T written (128 arrivals)
  uint64_t* bar_o = bar_q + 4;                                 // O^T complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_q + 6);
  int32_t* rows_s = reinterpret_cast<int32_t*>(bar_q + 8);     // [kMaxTiles][128] global row (-1 = empty)
  float* th_hi = reinterpret_cast<float*>(rows_s + kMaxTiles * kTile);   // [32]
  float* th_lo = th_hi + 32;                                   // [32]
  int* tile_id = reinterpret_cast<int*>(th_lo + 32);           // [kMaxTiles] (+ [kMaxTiles] TMA flags)
  float* q_cs = reinterpret_cast<float*>(tile_id + 4);         // [32] cos / sin of the query's angles
  float* q_sn = q_cs + 32;                                     // [32]
  // softmax scratch lives in the Q buffer, which is dead once S^T is complete
  float* red = reinterpret_cast<float*>(qs);                   // [4][64]
  float* m_s = red + 4 * kH;                                   // [64]

  if (threadIdx.x == 0) CSA_STAMP(0);
  griddep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // grid (rows, splits): every query's first tile (its window) is scheduled before any second tile
  const int64_t row = blockIdx.x;
  const int b = (int)(row / p.S), s = (int)(row % p.S), cta = blockIdx.y;
  const int64_t t = p.pos ? p.pos[row] : s;
  if (t < 0 || t >= p.N) {                                     // uniform over the CTA
    if (threadIdx.x == 0) set_error(p.err, DEVERR_BAD_POS);
    return;
  }
  const int64_t V = min(visible_entries(t, p.ratio), p.n_cap);
  const int64_t lo = t - p.window + 1 > 0 ? t - p.window + 1 : 0;
  const int64_t n_win = t - lo + 1;
  const int comp_tiles = p.topk ? (p.k + kTile - 1) / kTile : (int)((p.n_cap + kTile - 1) / kTile);
  const int total_tiles = p.win_tiles + comp_tiles;
  const int first_tile = cta * p.tiles_per_cta;
  const int nt = min(p.tiles_per_cta, total_tiles - first_tile);   // >= 1 by construction of the grid
  const LoadSeq seq{nt};
  // Processing order of the S^T phase: a window tile last, so that it is the resident tile of the
  // O^T phase and is rotated only once.
  if (threadIdx.x < kMaxTiles) {
    int id = first_tile + (int)threadIdx.x;
    if (nt == 2 && first_tile < p.win_tiles) id = first_tile + 1 - (int)threadIdx.x;
    tile_id[threadIdx.x] = threadIdx.x < nt ? id : -1;
    // HCA: a compressed tile whose rows are all visible is one contiguous run, loaded by TMA
    const int64_t first = ((int64_t)id - p.win_tiles) * kTile;
    tile_id[kMaxTiles + threadIdx.x] =
        threadIdx.x < nt && !p.topk && id >= p.win_tiles && first + kTile <= V ? 1 : 0;
  }
  if (threadIdx.x < 32) { th_hi[threadIdx.x] = p.rope.th_hi[threadIdx.x]; th_lo[threadIdx.x] = p.rope.th_lo[threadIdx.x]; }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) { mbar_init(&full[i], kGatherThreads); mbar_init(&empty[i], 1); }
    mbar_init(bar_q, 1);
    mbar_init(bar_qrot, 32);
    mbar_init(bar_s, 1);
    mbar_init(bar_p, 128);
    mbar_init(bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 32) {                                     // Q is an input of the call: load it now
    prefetch_tensormap(&qmap);
    mbar_arrive_expect_tx(bar_q, kQBytes);
    for (int kb = 0; kb < 8; ++kb) tma_load_2d(qs + kb * kQBlock, &qmap, bar_q, kb * 64, (int32_t)(row * kH));
  }
  // Only compressed tiles read the selection written by the previous kernel; window tiles read
  // nothing it writes and proceed at once.
  bool any_comp = false;
  for (int j = 0; j < nt; ++j) any_comp |= tile_id[j] >= p.win_tiles;
  if (any_comp) griddep_wait();

  // ---------------------------------------------------------------- candidate rows of the tiles
  for (int i = threadIdx.x; i < kMaxTiles * kTile; i += kThreads) {
    const int j = i / kTile, r = i % kTile;
    const int tid_ = tile_id[j];
    int64_t g = -1;
    if (tid_ >= 0) {
      if (tid_ < p.win_tiles) {
        const int64_t c = (int64_t)tid_ * kTile + r;
        if (c < n_win) g = (int64_t)b * p.N + lo + c;
      } else {
        const int64_t slot = (int64_t)(tid_ - p.win_tiles) * kTile + r;
        int64_t idx = -1;
        if (p.topk) {
          if (slot < p.k) idx = p.topk[row * p.k + slot];
        } else if (slot < V) {
          idx = slot;
        }
        if (idx >= V) { set_error(p.err, DEVERR_BAD_INDEX); idx = -1; }
        if (idx >= 0) g = (int64_t)b * p.n_cap + idx;
      }
    }
    rows_s[i] = (int32_t)g;
    // the gathers below are limited by how many requests one SM keeps in flight: have L2 fetch
    // every row of the CTA at once
    if (g >= 0) prefetch_l2((tid_ < p.win_tiles ? p.kv : p.ckv) + g * kD, kD * 2);
  }
  __syncthreads();
  if (threadIdx.x == 0) CSA_STAMP(1);
  const uint32_t tmem = *tmem_slot;
  auto is_win = [&](int j) { return tile_id[j] < p.win_tiles; };
  auto is_tma = [&](int j) { return tile_id[kMaxTiles + j] != 0; };
  // ---------------------------------------------------------------- the gather (warps 1..5)
  // Load i brings chunk c (dims 128c..128c+127) of the 128 rows of tile slot j into stage c: 2048
  // pieces of 16 bytes, consecutive threads on consecutive pieces of a row. Empty slots are zeros.
  const int gt = warp >= 7 ? threadIdx.x - 64 : threadIdx.x - 32;   // gather thread: warps 1..5, then 7..
  auto gather_issue = [&](int j, int c) {
    uint8_t* stage = ring + c * kChunkBytes;
    if (is_tma(j)) {                                           // one thread, two boxes; the rest just arrive
      if (gt == 0) {
        mbar_arrive_expect_tx(&full[c], kChunkBytes);
        const int32_t y = (int32_t)((int64_t)b * p.n_cap + (int64_t)(tile_id[j] - p.win_tiles) * kTile);
        tma_load_2d(stage, &cmap, &full[c], c * 128, y);
        tma_load_2d(stage + kBlk, &cmap, &full[c], c * 128 + 64, y);
      }
      cp_async_commit();
      return;
    }
    const __nv_bfloat16* base = is_win(j) ? p.kv : p.ckv;
    for (int u = gt; u < 2048; u += kGatherThreads) {
      const int rr = u >> 4, piece = u & 15;
      uint8_t* dst = stage + (piece >> 3) * kBlk + sw128_offset(rr, piece & 7);
      const int32_t g = rows_s[j * kTile + rr];
      if (g >= 0) cp_async16(dst, base + (int64_t)g * kD + c * 128 + piece * 8);
      else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
  };
  // this thread's copies of load i landed: a raw window tile's chunk 3 holds the rotary dims
  // 448..511 (block 1), which each thread rotates in the pieces it copied itself, at the row's own
  // position; then the chunk is published to the tensor core
  auto gather_complete = [&](int i) {
    int j, c, fill;
    seq.at(i, j, c, fill);
    if (c == 3 && is_win(j)) {
      uint8_t* blk1 = ring + 3 * kChunkBytes + kBlk;
      for (int u = gt; u < 2048; u += kGatherThreads) {
        const int rr = u >> 4, piece = u & 15;
        if (piece < 8 || rows_s[j * kTile + rr] < 0) continue;
        uint4* q16 = reinterpret_cast<uint4*>(blk1 + sw128_offset(rr, piece - 8));
        uint4 v = *q16;
        uint32_t* w = reinterpret_cast<uint32_t*>(&v);
        const int64_t pos = lo + (int64_t)tile_id[j] * kTile + rr;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int pair = (piece - 8) * 4 + k;
          float cs, sn;
          rope_cs(pos, th_hi[pair], th_lo[pair], cs, sn);
          const float a = bf16lo(w[k]), bb = bf16hi(w[k]);
          w[k] = pack_bf16(a * cs - bb * sn, a * sn + bb * cs);
        }
        *q16 = v;
      }
    }
    fence_proxy_async_smem();
    if (!(is_tma(j) && gt == 0)) mbar_arrive(&full[c]);        // the TMA issuer arrived with the bytes
  };
  // loads [i0, i1) in order, up to kStages - 1 in flight per thread
  auto gather_loads = [&](int i0, int i1, bool& ok) {
    for (int i = i0; i < i1; ++i) {
      int j, c, fill;
      seq.at(i, j, c, fill);
      if (fill > 0 && ok) ok = mbar_wait(&empty[c], (fill - 1) & 1, p.err);
      if (ok) gather_issue(j, c);
      else cp_async_commit();
      if (gt == 0) CSA_STAMP(16 + i);
      if (i - i0 >= kStages - 1) {
        cp_async_wait<kStages - 1>();
        gather_complete(i - (kStages - 1));
      }
    }
    cp_async_wait<0>();
    for (int i = i1 - (kStages - 1) > i0 ? i1 - (kStages - 1) : i0; i < i1; ++i) gather_complete(i);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      bool ok = mbar_wait(bar_q, 0, p.err) && mbar_wait(bar_qrot, 0, p.err);
      CSA_STAMP(8);
      const uint32_t q_addr = smem_u32(qs), ring_addr = smem_u32(ring), p_addr = smem_u32(ps);
      auto wait_load = [&](int i) {                            // load i landed (and was rotated if needed)
        int j, c, fill;
        seq.at(i, j, c, fill);
        return mbar_wait(&full[c], fill & 1, p.err);
      };
      // S^T phase
      for (int q = 0; q < 4 * nt && ok; ++q) {
        const int j = q >> 2, c = q & 3;
        ok = wait_load(q);
        if (!ok) break;
        CSA_STAMP(32 + q);
        tc_fence_after();
        const uint32_t a0 = ring_addr + c * kChunkBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kBlk + (kk & 3) * 32;
          const uint32_t qoff = (2 * c + (kk >> 2)) * kQBlock + (kk & 3) * 32;
          mma_bf16(tmem + j * kH, desc_kmajor_sw128(a0 + off), desc_kmajor_sw128(q_addr + qoff), kIdescS,
                   (c > 0 || kk > 0) ? 1u : 0u);
        }
        if (j < nt - 1) mma_commit(&empty[c]);                 // the last tile stays resident
      }
      if (ok) mma_commit(bar_s);
      CSA_STAMP(9);
      if (ok) ok = mbar_wait(bar_p, 0, p.err);
      CSA_STAMP(10);
      // O^T phase: the resident tile (slot nt-1), then slot 0 again
      for (int jj = 0; jj < nt && ok; ++jj) {
        const int j = nt - 1 - jj;
        for (int c = 0; c < 4 && ok; ++c) {
          if (jj > 0) {
            ok = wait_load(4 * nt + c);
            if (!ok) break;
          }
          tc_fence_after();
          const uint32_t a0 = ring_addr + c * kChunkBytes;
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks) {
            mma_bf16(tmem + kColO + c * kH, desc_mnmajor_sw128(a0 + ks * 2048, kBlk),
                     desc_mnmajor_sw128(p_addr + j * kPBytes + ks * 2048, kBlk), kIdescO,
                     (jj > 0 || ks > 0) ? 1u : 0u);
          }
          if (jj == 0 && nt > 1) mma_commit(&empty[c]);        // frees the stage for the re-gather
        }
      }
      if (ok) mma_commit(bar_o);
      CSA_STAMP(11);
    }
  } else if (warp == 1 || warp >= 7) {
    // ---------------------------------------------------------------- gather (these warps only gather)
    // Drain the S^T phase before the re-gather: its loads wait for the O^T MMAs, which need the
    // softmax, which needs every S^T phase load completed by all gather threads.
    bool ok = true;
    gather_loads(0, 4 * nt, ok);
    gather_loads(4 * nt, seq.count(), ok);
  } else if (warp == 6) {
    // ---------------------------------------------------------------- RoPE of the query
    // every head is rotated at t: lane i computes pair i's cos / sin once, shared through registers
    float cs_i, sn_i;
    rope_cs(t, th_hi[lane], th_lo[lane], cs_i, sn_i);
    q_cs[lane] = cs_i;
    q_sn[lane] = sn_i;
    __syncwarp();
    bool ok = mbar_wait_warp(bar_q, 0, p.err);
    if (ok) {
      rope_line_tab(qs + 7 * kQBlock + lane * 128, lane, q_cs, q_sn);
      rope_line_tab(qs + 7 * kQBlock + (lane + 32) * 128, lane + 32, q_cs, q_sn);
    }
    fence_proxy_async_smem();
    mbar_arrive(bar_qrot);
    if (lane == 0) CSA_STAMP(2);
  } else {
    // ---------------------------------------------------------------- softmax / epilogue warps (2..5)
    const int et = threadIdx.x - 64;                           // 0..127
    const int wq = warp & 3;                                   // TMEM lane quadrant
    const int r = 32 * wq + lane;                              // candidate row = TMEM lane
    const int wi = warp - 2;
    bool gok = true;
    gather_loads(0, 4 * nt, gok);                              // the S^T phase loads
    // TMEM loads are warp-collective: every lane loads, empty rows are masked afterwards
    bool ok = mbar_wait_warp(bar_s, 0, p.err) && __all_sync(0xffffffffu, gok);
    if (et == 0) CSA_STAMP(4);
    tc_fence_after();
    const uint32_t lane_base = tmem + ((wq * 32) << 16);
    float v[64];
#pragma unroll
    for (int h = 0; h < 64; ++h) v[h] = -INFINITY;
    for (int j = 0; j < nt && ok; ++j) {
      const bool valid = rows_s[j * kTile + r] >= 0;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float sv[32];
        tmem_row32(lane_base + j * kH + half * 32, sv);
#pragma unroll
        for (int h = 0; h < 32; ++h) v[half * 32 + h] = fmaxf(v[half * 32 + h], valid ? sv[h] : -INFINITY);
      }
    }
    reduce_scatter64<true>(v, lane);
    red[wi * kH + 2 * lane] = v[0];
    red[wi * kH + 2 * lane + 1] = v[1];
    named_barrier(1, 128);
    if (et < kH) m_s[et] = fmaxf(fmaxf(red[et], red[kH + et]), fmaxf(red[2 * kH + et], red[3 * kH + et]));
    named_barrier(1, 128);
    const float c2 = p.scale * kLog2e;
#pragma unroll
    for (int h = 0; h < 64; ++h) v[h] = 0.f;
    for (int j = 0; j < nt; ++j) {
      const bool valid = ok && rows_s[j * kTile + r] >= 0;
      uint8_t* line = ps + j * kPBytes;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float sv[32];
        if (ok) tmem_row32(lane_base + j * kH + half * 32, sv);     // ok is warp-uniform
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          const float m = m_s[half * 32 + h];
          const float e = (valid && m != -INFINITY) ? fast_exp2((sv[h] - m) * c2) : 0.f;
          sv[h] = e;
          v[half * 32 + h] += e;
        }
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint4 u;
          u.x = pack_bf16(sv[8 * ch + 0], sv[8 * ch + 1]);
          u.y = pack_bf16(sv[8 * ch + 2], sv[8 * ch + 3]);
          u.z = pack_bf16(sv[8 * ch + 4], sv[8 * ch + 5]);
          u.w = pack_bf16(sv[8 * ch + 6], sv[8 * ch + 7]);
          *reinterpret_cast<uint4*>(line + sw128_offset(r, half * 4 + ch)) = u;
        }
      }
    }
    tc_fence_before();
    fence_proxy_async_smem();
    mbar_arrive(bar_p);
    if (et == 0) CSA_STAMP(5);
    gather_loads(4 * nt, seq.count(), gok);                    // two tiles: tile slot 0 again
    reduce_scatter64<false>(v, lane);
    red[wi * kH + 2 * lane] = v[0];
    red[wi * kH + 2 * lane + 1] = v[1];
    named_barrier(1, 128);
    const int64_t pi = (row * p.n_split + cta) * kH;
    if (et < kH) {
      const float l = (red[et] + red[kH + et]) + (red[2 * kH + et] + red[3 * kH + et]);
      p.part_ml[2 * (pi + et)] = m_s[et] == -INFINITY ? -INFINITY : m_s[et] * p.scale;
      p.part_ml[2 * (pi + et) + 1] = l;
    }
    // split partial O: thread = dim 128 dc + r, 64 heads
    ok = mbar_wait_warp(bar_o, 0, p.err) && ok;
    if (et == 0) CSA_STAMP(6);
    if (ok) {
      tc_fence_after();
#pragma unroll 1
      for (int dc = 0; dc < 4; ++dc) {
        float* dst = p.part_o + pi * kD + dc * 128 + r;
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          float ov[32];
          tmem_row32(lane_base + kColO + dc * kH + hh * 32, ov);
#pragma unroll
          for (int j = 0; j < 32; ++j) dst[(int64_t)(hh * 32 + j) * kD] = ov[j];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) CSA_STAMP(12);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool tc_attn_available() { return true; }
int tc_attn_split_len() { return kTile; }
size_t tc_workspace_bytes(int, int, int64_t, int) { return 0; }

// tiles of one query: window tiles + compressed tiles
static int attn_tiles(int window, int top_k, int64_t n_cap) {
  const int wt = (window + kTile - 1) / kTile;
  const int64_t ct = top_k > 0 ? (top_k + kTile - 1) / kTile : (n_cap + kTile - 1) / kTile;
  return wt + (int)ct;
}

// Tiles per CTA: one (no tile is ever gathered twice) while the batch's tiles fit in the waves the
// launch can overlap with earlier work, else two. With a selection (CSA) the window tiles, listed
// first, run during the selection kernel, so two waves of one-tile CTAs still pay off; without one
// (HCA) every tile waits for the same closing step, so the CTAs must fit one wave (one per SM).
static int attn_tiles_per_cta(int rows, int tiles, bool selection) {
  return (int64_t)rows * tiles <= (selection ? 2 : 1) * (int64_t)tc_sm_count() ? 1 : 2;
}

int tc_attn_splits(int window, int top_k, int64_t n_cap, int rows) {
  const int tiles = attn_tiles(window, top_k, n_cap);
  const int per = attn_tiles_per_cta(rows, tiles, top_k > 0);
  return (tiles + per - 1) / per;
}

cudaError_t tc_sparse_attn(int B, const AttnParams& a, void*, cudaStream_t st, bool pdl) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int rows = B * a.S;
  const int tiles = attn_tiles(a.window, a.k, a.n_cap);
  const int per = attn_tiles_per_cta(rows, tiles, a.k > 0);
  if (a.n_split != (tiles + per - 1) / per || !a.part_o) return cudaErrorInvalidValue;
  if ((int64_t)B * a.N >= (int64_t)1 << 31 || (int64_t)B * a.n_cap >= (int64_t)1 << 31) return cudaErrorInvalidValue;
  CUtensorMap qmap, cmap;
  cudaError_t e = make_tmap_2d(&qmap, a.q, (int64_t)B * a.S * kH, kD, kH);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d(&cmap, a.ckv, (int64_t)B * a.n_cap, kD, kTile);   // HCA's whole compressed tiles
  if (e != cudaSuccess) return e;
  AttnTcParams p;
  p.kv = static_cast<const __nv_bfloat16*>(a.kv);
  p.ckv = static_cast<const __nv_bfloat16*>(a.ckv);
  p.topk = a.topk; p.pos = a.pos; p.part_o = a.part_o; p.part_ml = a.part_ml; p.N = a.N; p.n_cap = a.n_cap;
  p.S = a.S; p.k = a.k; p.ratio = a.ratio; p.window = a.window; p.n_split = a.n_split;
  p.win_tiles = (a.window + kTile - 1) / kTile; p.tiles_per_cta = per;
  p.scale = a.scale; p.rope = a.rope; p.err = a.err;
  dim3 grid((unsigned)rows, (unsigned)a.n_split);
  return launch_kernel(pdl, attn_tc_kernel, grid, dim3(kThreads), kSmemBytes, st, qmap, cmap, p);
}

}  // namespace csa
