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
// One CTA = one query and up to two 128-candidate tiles (window tiles first, then compressed
// tiles), so that a decode step of 32 requests x 5 tiles fits one wave of CTAs. A tile streams
// through a 4-stage ring in 32 KB K-chunks (128 candidates x 128 dims): the last tile of the
// S^T phase stays resident for the O^T phase and only the other tile is gathered again (an L2
// hit). Rows are gathered by warps 2..5 with 16-byte cp.async straight into the 128-byte
// swizzled tensor-core layout; empty slots are zero-filled; raw window rows are rotated at their
// own positions (RoPE on dims 448..511) in shared memory. Warp 0 loads Q by TMA and issues every
// tcgen05.mma; warps 2..5 (thread = candidate row = TMEM lane) run the softmax on S^T read from
// TMEM: per-head max and sum by a butterfly reduce-scatter across lanes plus a 4-warp combine,
// P^T (bf16) into shared memory. They finally write the split partial (max, sum, O) in fp32.
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
constexpr int kThreads = 192;
constexpr int kStages = 4;
constexpr uint32_t kBlk = kTile * 128;              // 16 KB: [128 rows][64 dims] swizzled
constexpr uint32_t kChunkBytes = 2 * kBlk;          // 32 KB: 128 rows x 128 dims
constexpr uint32_t kQBlock = kH * 128;              // 8 KB: [64 heads][64 dims]
constexpr uint32_t kQBytes = 8 * kQBlock;           // 64 KB
constexpr uint32_t kPBytes = kTile * 128;           // 16 KB per tile: P^T, one 128-byte line per candidate
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = kMaxTiles * kH;          // O^T[dc] at kColO + 64 dc
constexpr uint32_t kIdescS = idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdescO = idesc_bf16(128, 64, true, true);
constexpr size_t kAuxBytes = 2048;                   // barriers, row table, RoPE table (< 1.5 KB)
constexpr size_t kSmemBytes = 1024 + kQBytes + kStages * kChunkBytes + kMaxTiles * kPBytes + kAuxBytes;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnTcParams {
  const __nv_bfloat16* kv;   // [B, N, 512] raw rows
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

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap qmap, const AttnTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qs = smem;                                          // [8 blocks][64 heads][128 B]
  uint8_t* ring = qs + kQBytes;                                // kStages x [2 blocks][128 rows][128 B]
  uint8_t* ps = ring + kStages * kChunkBytes;                  // kMaxTiles x [128 rows][128 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ps + kMaxTiles * kPBytes);
  uint64_t* full = bars;                                       // [kStages] (128 arrivals)
  uint64_t* empty = bars + kStages;                            // [kStages] (MMA commit)
  uint64_t* bar_q = bars + 2 * kStages;                        // Q bytes landed (tx)
  uint64_t* bar_qrot = bar_q + 1;                              // Q rotated (64 arrivals)
  uint64_t* bar_s = bar_q + 2;                                 // S^T complete
  uint64_t* bar_p = bar_q + 3;                                 // P^T written (128 arrivals)
  uint64_t* bar_o = bar_q + 4;                                 // O^T complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_q + 6);
  int32_t* rows_s = reinterpret_cast<int32_t*>(bar_q + 8);     // [kMaxTiles][128] global row (-1 = empty)
  float* th_hi = reinterpret_cast<float*>(rows_s + kMaxTiles * kTile);   // [32]
  float* th_lo = th_hi + 32;                                   // [32]
  int* tile_id = reinterpret_cast<int*>(th_lo + 32);           // [kMaxTiles]
  // softmax scratch lives in the Q buffer, which is dead once S^T is complete
  float* red = reinterpret_cast<float*>(qs);                   // [4][64]
  float* m_s = red + 4 * kH;                                   // [64]

  griddep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, s = blockIdx.y, cta = blockIdx.x;
  const int64_t row = (int64_t)b * p.S + s;
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
  // Processing order of the S^T phase: a window tile last, so that it is the resident tile of the
  // O^T phase and never has to be rotated twice.
  if (threadIdx.x < kMaxTiles) {
    int id = first_tile + (int)threadIdx.x;
    if (nt == 2 && first_tile < p.win_tiles) id = first_tile + 1 - (int)threadIdx.x;
    tile_id[threadIdx.x] = threadIdx.x < nt ? id : -1;
  }
  __syncthreads();

  if (threadIdx.x < 32) { th_hi[threadIdx.x] = p.rope.th_hi[threadIdx.x]; th_lo[threadIdx.x] = p.rope.th_lo[threadIdx.x]; }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) { mbar_init(&full[i], 128); mbar_init(&empty[i], 1); }
    mbar_init(bar_q, 1);
    mbar_init(bar_qrot, 64);
    mbar_init(bar_s, 1);
    mbar_init(bar_p, 128);
    mbar_init(bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {                                      // Q is an input of the call: load it now
    prefetch_tensormap(&qmap);
    mbar_arrive_expect_tx(bar_q, kQBytes);
    for (int kb = 0; kb < 8; ++kb) tma_load_2d(qs + kb * kQBlock, &qmap, bar_q, kb * 64, (int32_t)(row * kH));
  }
  griddep_wait();                                              // the selection comes from the previous kernel

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
  }
  __syncthreads();
  const uint32_t tmem = *tmem_slot;
  // loads: S^T phase = nt tiles x 4 chunks (fills 0, 1); O^T phase re-gathers tile 0 when nt == 2 (fill 2)
  const int n_loads_s = 4 * nt;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- the MMA issuer
      bool ok = mbar_wait(bar_q, 0, p.err) && mbar_wait(bar_qrot, 0, p.err);
      const uint32_t q_addr = smem_u32(qs), ring_addr = smem_u32(ring), p_addr = smem_u32(ps);
      // S^T phase
      for (int q = 0; q < n_loads_s && ok; ++q) {
        const int st = q % kStages, fill = q / kStages, j = q / 4, c = q % 4;
        ok = mbar_wait(&full[st], fill & 1, p.err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a0 = ring_addr + st * kChunkBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kBlk + (kk & 3) * 32;
          const uint32_t qoff = (2 * c + (kk >> 2)) * kQBlock + (kk & 3) * 32;
          mma_bf16(tmem + j * kH, desc_kmajor_sw128(a0 + off), desc_kmajor_sw128(q_addr + qoff), kIdescS,
                   (c > 0 || kk > 0) ? 1u : 0u);
        }
        if (j < nt - 1) mma_commit(&empty[st]);                // the last tile stays resident
      }
      if (ok) mma_commit(bar_s);
      if (ok) ok = mbar_wait(bar_p, 0, p.err);
      // O^T phase: the resident tile (tile nt-1, fill (nt-1) of stages 0..3), then tile 0 again
      for (int jj = 0; jj < nt && ok; ++jj) {
        const int j = nt - 1 - jj;
        for (int c = 0; c < 4 && ok; ++c) {
          const int st = c;
          if (jj > 0) {                                        // re-gathered chunk: fill 2
            ok = mbar_wait(&full[st], 0, p.err);
            if (!ok) break;
          }
          tc_fence_after();
          const uint32_t a0 = ring_addr + st * kChunkBytes;
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks) {
            mma_bf16(tmem + kColO + c * kH, desc_mnmajor_sw128(a0 + ks * 2048, kBlk),
                     desc_mnmajor_sw128(p_addr + j * kPBytes + ks * 2048, kBlk), kIdescO,
                     (jj > 0 || ks > 0) ? 1u : 0u);
          }
          if (jj == 0 && nt > 1) mma_commit(&empty[st]);       // frees the stage for the re-gather
        }
      }
      if (ok) mma_commit(bar_o);
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- gather / softmax / epilogue warps
    const int pt = threadIdx.x - 64;                           // 0..127
    const int wq = warp & 3;                                   // TMEM lane quadrant
    const int r = 32 * wq + lane;                              // candidate row = TMEM lane
    bool ok = true;
    // Q rotation at t: thread h < 64 rotates head h's dims 448..511 once the TMA bytes landed
    if (pt < kH) {
      ok = mbar_wait(bar_q, 0, p.err);
      if (ok) rope_line(qs + 7 * kQBlock + pt * 128, pt, t, th_hi, th_lo);
      fence_proxy_async_smem();
      mbar_arrive(bar_qrot);
    }
    // one load = 128 rows x 256 B of chunk c of tile slot j into ring stage st
    auto issue = [&](int j, int c, int st) {
      uint8_t* stage = ring + st * kChunkBytes;
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int u = pt + 128 * i;                            // (row, piece) pairs, 2 rows per warp
        const int rr = u >> 4, piece = u & 15;
        uint8_t* dst = stage + (piece >> 3) * kBlk + sw128_offset(rr, piece & 7);
        const int32_t g = rows_s[j * kTile + rr];
        const __nv_bfloat16* base = tile_id[j] < p.win_tiles ? p.kv : p.ckv;
        if (g >= 0) cp_async16(dst, base + (int64_t)g * kD + c * 128 + piece * 8);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
      cp_async_commit();
    };
    // completes load (j, c) in stage st: rotate window rows (chunk 3), publish to the async proxy
    auto finish = [&](int j, int c, int st) {
      if (c == 3 && tile_id[j] < p.win_tiles) {
        named_barrier(1, 128);                                 // every thread's copies of the chunk landed
        const int32_t g = rows_s[j * kTile + pt];
        if (g >= 0) rope_line(ring + st * kChunkBytes + kBlk + pt * 128, pt, lo + (int64_t)tile_id[j] * kTile + pt,
                              th_hi, th_lo);
      }
      fence_proxy_async_smem();
      mbar_arrive(&full[st]);
    };
    // S^T phase loads: q -> (tile q/4, chunk q%4), stage q%4, fill q/4; up to kStages - 1 loads stay
    // in flight while the oldest one is completed
    for (int q = 0; q < n_loads_s; ++q) {
      const int st = q % kStages, fill = q / kStages;
      if (fill > 0 && ok) ok = mbar_wait(&empty[st], (fill - 1) & 1, p.err);
      if (ok) issue(q / 4, q % 4, st);
      else cp_async_commit();
      if (q >= kStages - 1) {
        cp_async_wait<kStages - 1>();
        const int d = q - (kStages - 1);
        finish(d / 4, d % 4, d % kStages);
      }
    }
    cp_async_wait<0>();
    for (int d = n_loads_s - (kStages - 1) > 0 ? n_loads_s - (kStages - 1) : 0; d < n_loads_s; ++d)
      finish(d / 4, d % 4, d % kStages);

    // ---------------------------------------------------------------- softmax over the CTA's candidates
    // TMEM loads are warp-collective: every lane loads, empty rows are masked afterwards
    ok = mbar_wait_warp(bar_s, 0, p.err) && __all_sync(0xffffffffu, ok);
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
    const int wi = warp - 2;
    reduce_scatter64<true>(v, lane);
    red[wi * kH + 2 * lane] = v[0];
    red[wi * kH + 2 * lane + 1] = v[1];
    named_barrier(1, 128);
    if (pt < kH) m_s[pt] = fmaxf(fmaxf(red[pt], red[kH + pt]), fmaxf(red[2 * kH + pt], red[3 * kH + pt]));
    named_barrier(1, 128);
    const float c2 = p.scale * kLog2e;
#pragma unroll
    for (int h = 0; h < 64; ++h) v[h] = 0.f;
    for (int j = 0; j < kMaxTiles; ++j) {
      if (j >= nt) break;
      const bool valid = ok && rows_s[j * kTile + r] >= 0;
      uint8_t* line = ps + j * kPBytes;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float sv[32];
        if (ok) tmem_row32(lane_base + j * kH + half * 32, sv);     // ok is warp-uniform
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          const float m = m_s[half * 32 + h];
          const float e = (valid && m != -INFINITY) ? exp2f((sv[h] - m) * c2) : 0.f;
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
    // O^T phase: re-gather tile 0 of a two-tile CTA into stages 0..3 (fill 2)
    if (nt > 1) {
      for (int c = 0; c < 4; ++c) {
        if (ok) ok = mbar_wait(&empty[c], 1, p.err);
        if (ok) issue(0, c, c);
        else cp_async_commit();
      }
      cp_async_wait<3>(); finish(0, 0, 0);
      cp_async_wait<2>(); finish(0, 1, 1);
      cp_async_wait<1>(); finish(0, 2, 2);
      cp_async_wait<0>(); finish(0, 3, 3);
    }
    reduce_scatter64<false>(v, lane);
    red[wi * kH + 2 * lane] = v[0];
    red[wi * kH + 2 * lane + 1] = v[1];
    named_barrier(1, 128);
    const int64_t pi = (row * p.n_split + cta) * kH;
    if (pt < kH) {
      const float l = (red[pt] + red[kH + pt]) + (red[2 * kH + pt] + red[3 * kH + pt]);
      p.part_ml[2 * (pi + pt)] = m_s[pt] == -INFINITY ? -INFINITY : m_s[pt] * p.scale;
      p.part_ml[2 * (pi + pt) + 1] = l;
    }
    // split partial O: thread = dim 128 dc + r, 64 heads
    ok = mbar_wait_warp(bar_o, 0, p.err) && __all_sync(0xffffffffu, ok);
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

// Tiles per CTA: one when every tile of the batch fits one wave of CTAs, otherwise two.
static int attn_tiles_per_cta(int rows, int tiles) {
  return (int64_t)rows * tiles <= tc_sm_count() ? 1 : 2;
}

int tc_attn_splits(int window, int top_k, int64_t n_cap, int rows) {
  const int tiles = attn_tiles(window, top_k, n_cap);
  const int per = attn_tiles_per_cta(rows, tiles);
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
  const int per = attn_tiles_per_cta(rows, tiles);
  if (a.n_split != (tiles + per - 1) / per || !a.part_o) return cudaErrorInvalidValue;
  if ((int64_t)B * a.N >= (int64_t)1 << 31 || (int64_t)B * a.n_cap >= (int64_t)1 << 31) return cudaErrorInvalidValue;
  CUtensorMap qmap;
  cudaError_t e = make_tmap_2d(&qmap, a.q, (int64_t)B * a.S * kH, kD, kH);
  if (e != cudaSuccess) return e;
  AttnTcParams p;
  p.kv = static_cast<const __nv_bfloat16*>(a.kv);
  p.ckv = static_cast<const __nv_bfloat16*>(a.ckv);
  p.topk = a.topk; p.pos = a.pos; p.part_o = a.part_o; p.part_ml = a.part_ml; p.N = a.N; p.n_cap = a.n_cap;
  p.S = a.S; p.k = a.k; p.ratio = a.ratio; p.window = a.window; p.n_split = a.n_split;
  p.win_tiles = (a.window + kTile - 1) / kTile; p.tiles_per_cta = per;
  p.scale = a.scale; p.rope = a.rope; p.err = a.err;
  dim3 grid((unsigned)a.n_split, (unsigned)a.S, (unsigned)B);
  return launch_kernel(pdl, attn_tc_kernel, grid, dim3(kThreads), kSmemBytes, st, qmap, p);
}

}  // namespace csa
