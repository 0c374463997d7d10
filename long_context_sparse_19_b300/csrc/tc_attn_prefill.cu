// K7: sparse joint attention for many queries (causal prefill) on the tensor cores (bf16, H = 64,
// d = 512), one CTA per query owning its whole candidate set (at most 5 tiles of 128 candidates).
//
// [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", sections "局部和压缩记忆，共用一次归一化" (one
// softmax over the raw window and the selected compressed entries; the per-head sink enlarges the
// denominator only) and "输出投影也分组，并且降低中间维度" (o = inverse_RoPE(o)).
//
// Because the CTA sees every candidate of its query, the softmax is exact in one pass and no split
// partials exist:
//   phase S: S^T[j] = KV_j Q^T for every tile j (M = 128 candidates, N = 64 heads, K = 512), all
//            tiles kept in TMEM (5 x 64 columns);
//   softmax: per-head max over every candidate and the sink, P^T = exp(scale s - max) in bf16 (it
//            reuses the Q buffer, dead by then), per-head denominators;
//   phase O: O^T[dims] = sum_j KV_j^T P^T_j in two halves of 256 dims (2 x 64 TMEM columns each:
//            half 0 after the S^T tiles, half 1 in the S^T columns, dead once P^T is written), each
//            half normalised and written as the final output (inverse RoPE on dims 448..511).
// The KV data streams through a 4-stage ring of 32 KB K-chunks twice (phase S, then phase O; the
// second pass hits L2). The rows are gathered with 16-byte cp.async by six warps, up to three
// chunks in flight per thread: measured on this part, one SM gathers random 1 KB rows from L2 at
// about 110 GB/s this way and at under 20 GB/s with tile::gather4 TMA loads. Warps: 0 = Q TMA +
// tcgen05.mma issuer, 1 = TMEM owner + Q rotation, 2..5 = softmax / epilogue (thread = TMEM lane),
// 6..11 = gather (each thread rotates the raw window pieces it copied, at the row's own position).
#include <cudaTypedefs.h>

#include "tc.h"
#include "tc_ptx.cuh"

namespace csa {
namespace {

using namespace tc;

constexpr int kD = 512;
constexpr int kH = 64;
constexpr int kTile = 128;
constexpr int kMaxTiles = 5;
constexpr int kThreads = 384;
constexpr int kGatherThreads = 192;                 // warps 6..11
constexpr int kSThreads = 320;                      // warps 2..11 during phase S
static_assert(11 * kGatherThreads >= 2048 && kSThreads >= kGatherThreads, "a chunk in 11 rounds");
constexpr int kStages = 4;
constexpr uint32_t kBlk = kTile * 128;              // 16 KB: [128 rows][64 dims] swizzled
constexpr uint32_t kChunkBytes = 2 * kBlk;          // 32 KB: 128 rows x 128 dims
constexpr uint32_t kQBlock = kH * 128;              // 8 KB: [64 heads][64 dims]
constexpr uint32_t kQBytes = 8 * kQBlock;           // 64 KB
constexpr uint32_t kPBytes = kTile * 128;           // 16 KB per tile
constexpr uint32_t kQPBytes = kMaxTiles * kPBytes;  // 80 KB: Q (phase S), then P^T (phase O)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = kMaxTiles * kH;          // 320: O^T half, 2 x 64 columns
constexpr uint32_t kIdescS = idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdescO = idesc_bf16(128, 64, true, true);
constexpr size_t kAuxBytes = 5120;
constexpr size_t kOutStageBytes = 32 * kTile * 2;   // 8 KB: one block of 32 heads x 128 dims (bf16)
constexpr size_t kSmemBytes = 1024 + kQPBytes + kStages * kChunkBytes + kAuxBytes + kOutStageBytes;
static_assert(kSmemBytes <= 232448, "shared memory of one CTA");
constexpr float kLog2e = 1.4426950408889634f;

struct PrefillParams {
  const __nv_bfloat16* kv;   // [B, N, 512] raw rows
  const __nv_bfloat16* ckv;  // [B, n_cap, 512]
  const int32_t* topk;       // [B, S, k] or null (HCA)
  const int64_t* pos;        // [B, S] or null (t = s)
  const float* sink;         // [64]
  __nv_bfloat16* out;        // [B, S, 64, 512]
  int64_t N, n_cap;
  int S, k, ratio, window, win_tiles, n_tiles;
  float scale;
  RopeTab rope;
  int32_t* err;
};

__global__ void __launch_bounds__(kThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap qmap, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* qs = smem;                                          // Q: [8 blocks][64 heads][128 B]
  uint8_t* ps = smem;                                          // P^T: [5 tiles][128 rows][128 B] (after phase S)
  uint8_t* ring = smem + kQPBytes;                             // kStages x [2 blocks][128 rows][128 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + kStages * kChunkBytes);
  uint64_t* full = bars;                                       // [kStages] phase O (kGatherThreads arrivals)
  uint64_t* empty = bars + kStages;                            // [kStages] (MMA commit)
  uint64_t* bar_q = bars + 2 * kStages;                        // Q landed (tx)
  uint64_t* bar_qrot = bar_q + 1;                              // Q rotated (32 arrivals)
  uint64_t* bar_s = bar_q + 2;                                 // S^T complete
  uint64_t* bar_p = bar_q + 3;                                 // P^T written (128 arrivals)
  uint64_t* bar_o0 = bar_q + 4;                                // O^T half 0 complete
  uint64_t* bar_o1 = bar_q + 6;                                // O^T half 1 complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_q + 8);
  uint64_t* full_s = bar_q + 10;                               // [kStages] phase S (kSThreads arrivals)
  int32_t* rows_s = reinterpret_cast<int32_t*>(bar_q + 14);    // [5][128] global row (-1 = empty)
  float* th_hi = reinterpret_cast<float*>(rows_s + kMaxTiles * kTile);   // [32]
  float* th_lo = th_hi + 32;                                   // [32]
  float* red = th_lo + 32;                                     // [4][64]
  float* mx_s = red + 4 * kH;                                  // [64] max of scale * s and the sink
  float* il_s = mx_s + kH;                                     // [64] 1 / denominator
  float* q_cs = il_s + kH;                                     // [32] cos / sin of the query's angles
  float* q_sn = q_cs + 32;                                     // [32]
  __nv_bfloat16* ostage = reinterpret_cast<__nv_bfloat16*>(ring + kStages * kChunkBytes + kAuxBytes);  // [32][128]

  if (threadIdx.x == 0) CSA_STAMP(0);
  griddep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y, s = blockIdx.x;
  const int64_t row = (int64_t)b * p.S + s;
  const int64_t t = p.pos ? p.pos[row] : s;
  if (t < 0 || t >= p.N) {
    if (threadIdx.x == 0) set_error(p.err, DEVERR_BAD_POS);
    return;
  }
  const int64_t V = min(visible_entries(t, p.ratio), p.n_cap);
  const int64_t lo = t - p.window + 1 > 0 ? t - p.window + 1 : 0;
  const int64_t n_win = t - lo + 1;
  const int nt = p.n_tiles;

  if (threadIdx.x < 32) { th_hi[threadIdx.x] = p.rope.th_hi[threadIdx.x]; th_lo[threadIdx.x] = p.rope.th_lo[threadIdx.x]; }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], kGatherThreads);
      mbar_init(&full_s[i], kSThreads);
      mbar_init(&empty[i], 1);
    }
    mbar_init(bar_q, 1);
    mbar_init(bar_qrot, 32);
    mbar_init(bar_s, 1);
    mbar_init(bar_p, 128);
    mbar_init(bar_o0, 1);
    mbar_init(bar_o1, 1);
    fence_mbar_init();
  }
  if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    prefetch_tensormap(&qmap);
    mbar_arrive_expect_tx(bar_q, kQBytes);
    for (int kb = 0; kb < 8; ++kb) tma_load_2d(qs + kb * kQBlock, &qmap, bar_q, kb * 64, (int32_t)(row * kH));
  }
  griddep_wait();                                              // the selection comes from the previous kernel
  for (int i = threadIdx.x; i < kMaxTiles * kTile; i += kThreads) {
    const int j = i / kTile, r = i % kTile;
    int64_t g = -1;
    if (j < nt) {
      if (j < p.win_tiles) {
        const int64_t c = (int64_t)j * kTile + r;
        if (c < n_win) g = (int64_t)b * p.N + lo + c;
      } else {
        const int64_t slot = (int64_t)(j - p.win_tiles) * kTile + r;
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
  if (threadIdx.x == 0) CSA_STAMP(1);
  const uint32_t tmem = *tmem_slot;
  const int n_loads = 4 * nt;                                  // per phase
  // load q of phase S: tile q/4, chunk q%4; load q of phase O (half = q / (2 nt)): tile (q % (2 nt)) / 2,
  // chunk 2 half + q % 2
  auto load_of = [&](int q, int& j, int& c) {
    if (q < n_loads) { j = q >> 2; c = q & 3; return; }
    const int u = q - n_loads, half = u / (2 * nt), v = u % (2 * nt);
    j = v >> 1;
    c = 2 * half + (v & 1);
  };

  // ------------------------------------------------------------------ gather pipeline
  // Load q brings chunk c (dims 128c .. 128c+127) of the 128 rows of tile j into stage q % kStages:
  // 2048 pieces of 16 bytes, consecutive threads on consecutive pieces of a row; empty rows are
  // zeros. A chunk of phase S is split over the 320 threads of warps 2..11 (the softmax warps have
  // nothing else to do until S is complete), a chunk of phase O over the 192 threads of warps
  // 6..11. After a raw window tile's chunk 3 lands (block 1 = dims 448..511), each thread rotates
  // the pieces it copied at the row's own position.
  auto split_of = [&](int q, int& tid, int& nth) {
    if (q < n_loads) { tid = (int)threadIdx.x - 64; nth = kSThreads; }
    else { tid = (int)threadIdx.x - 192; nth = kGatherThreads; }
  };
  auto issue = [&](int q) {
    int j, c, tid, nth;
    load_of(q, j, c);
    split_of(q, tid, nth);
    uint8_t* stage = ring + (q % kStages) * kChunkBytes;
    const __nv_bfloat16* base = j < p.win_tiles ? p.kv : p.ckv;
    // 11 x 192 >= 2048 pieces: every row-table read is issued before the first copy (a copy's
    // memory clobber would otherwise hold each read behind the previous copy)
    int32_t g[11];
#pragma unroll
    for (int i = 0; i < 11; ++i) {
      const int u = tid + i * nth;
      g[i] = u < 2048 ? rows_s[j * kTile + (u >> 4)] : -1;
    }
#pragma unroll
    for (int i = 0; i < 11; ++i) {
      const int u = tid + i * nth;
      if (u < 2048) {
        const int rr = u >> 4, piece = u & 15;
        uint8_t* dst = stage + (piece >> 3) * kBlk + sw128_offset(rr, piece & 7);
        if (g[i] >= 0) cp_async16(dst, base + (int64_t)g[i] * kD + c * 128 + piece * 8);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_commit();
  };
  auto complete = [&](int q) {
    int j, c, tid, nth;
    load_of(q, j, c);
    split_of(q, tid, nth);
    const int st = q % kStages;
    if (c == 3 && j < p.win_tiles) {
      uint8_t* blk1 = ring + st * kChunkBytes + kBlk;
#pragma unroll 1
      for (int u = tid; u < 2048; u += nth) {
        const int rr = u >> 4, piece = u & 15;
        if (piece < 8 || rows_s[j * kTile + rr] < 0) continue;
        uint4* q16 = reinterpret_cast<uint4*>(blk1 + sw128_offset(rr, piece - 8));
        uint4 v = *q16;
        uint32_t* w = reinterpret_cast<uint32_t*>(&v);
        const int64_t pos_r = lo + (int64_t)j * kTile + rr;
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
          const int pair = (piece - 8) * 4 + k;
          const float2 cs = rope_cs_nl(pos_r, th_hi[pair], th_lo[pair]);
          const float a = bf16lo(w[k]), bb = bf16hi(w[k]);
          w[k] = pack_bf16(a * cs.x - bb * cs.y, a * cs.y + bb * cs.x);
        }
        *q16 = v;
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(q < n_loads ? &full_s[st] : &full[st]);
  };
  // Loads [0, q_end). A landed chunk is handed to the MMA before the thread waits for a free stage:
  // that wait is for the MMA of an older chunk, so the MMAs never wait on the issue of next loads.
  auto gather = [&](int q_end) {
    bool ok = true;
#pragma unroll 1
    for (int q = 0; q < q_end; ++q) {
      const int st = q % kStages, fill = q / kStages;
      if (q >= kStages - 1) {
        cp_async_wait<kStages - 2>();                          // load q - (kStages - 1) landed
        if (threadIdx.x == 192 && q >= 8 && q < 16) CSA_STAMP(10 + 3 * (q - 8));
        complete(q - (kStages - 1));
      }
      if (fill > 0 && ok) ok = mbar_wait(&empty[st], (fill - 1) & 1, p.err);
      if (threadIdx.x == 192 && q >= 8 && q < 16) CSA_STAMP(11 + 3 * (q - 8));
      if (ok) issue(q);
      else cp_async_commit();
      if (threadIdx.x == 192 && q >= 8 && q < 16) CSA_STAMP(12 + 3 * (q - 8));
    }
    cp_async_wait<0>();
#pragma unroll 1
    for (int q = q_end > kStages - 1 ? q_end - (kStages - 1) : 0; q < q_end; ++q) complete(q);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      bool ok = mbar_wait(bar_q, 0, p.err) && mbar_wait(bar_qrot, 0, p.err);
      const uint32_t q_addr = smem_u32(qs), ring_addr = smem_u32(ring), p_addr = smem_u32(ps);
      for (int q = 0; q < 2 * n_loads && ok; ++q) {
        const int st = q % kStages, fill = q / kStages;
        int j, c;
        load_of(q, j, c);
        if (q == n_loads) {                                     // phase O needs P^T
          mma_commit(bar_s);
          ok = mbar_wait(bar_p, 0, p.err);
          if (!ok) break;
        }
        if (q == n_loads + 2 * nt) mma_commit(bar_o0);          // half 1 goes to the dead S^T columns
        ok = q < n_loads ? mbar_wait(&full_s[st], fill & 1, p.err)
                         : mbar_wait(&full[st], ((q - n_loads) / kStages) & 1, p.err);
        if (!ok) break;
        if (q >= 5 && q < 13) CSA_STAMP(34 + (q - 5));
        tc_fence_after();
        const uint32_t a0 = ring_addr + st * kChunkBytes;
        if (q < n_loads) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kBlk + (kk & 3) * 32;
            const uint32_t qoff = (2 * c + (kk >> 2)) * kQBlock + (kk & 3) * 32;
            mma_bf16(tmem + j * kH, desc_kmajor_sw128(a0 + off), desc_kmajor_sw128(q_addr + qoff), kIdescS,
                     (c > 0 || kk > 0) ? 1u : 0u);
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks) {
            mma_bf16(tmem + (c < 2 ? kColO : 0u) + (c & 1) * kH, desc_mnmajor_sw128(a0 + ks * 2048, kBlk),
                     desc_mnmajor_sw128(p_addr + j * kPBytes + ks * 2048, kBlk), kIdescO,
                     (j > 0 || ks > 0) ? 1u : 0u);
          }
        }
        mma_commit(&empty[st]);
      }
      if (ok) mma_commit(bar_o1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- Q rotation at t
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
  } else if (warp >= 6) {
    gather(2 * n_loads);                                       // warps 6..11: phases S and O
  } else {
    // ---------------------------------------------------------------- softmax / epilogue (warps 2..5)
    gather(n_loads);                                           // phase S, with the gather warps
    const int et = threadIdx.x - 64;                           // 0..127
    const int wq = warp & 3;
    const int r = 32 * wq + lane;                              // TMEM lane
    const int wi = warp - 2;
    const uint32_t lane_base = tmem + ((wq * 32) << 16);
    // TMEM loads are warp-collective: every lane loads, empty rows are masked afterwards
    bool ok = mbar_wait_warp(bar_s, 0, p.err);
    if (et == 0) CSA_STAMP(2);
    tc_fence_after();
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
    if (et < kH) {
      const float m = fmaxf(fmaxf(red[et], red[kH + et]), fmaxf(red[2 * kH + et], red[3 * kH + et]));
      mx_s[et] = fmaxf(m == -INFINITY ? -INFINITY : m * p.scale, p.sink[et]);   // logit units
    }
    named_barrier(1, 128);
#pragma unroll
    for (int h = 0; h < 64; ++h) v[h] = 0.f;
    const float c2 = p.scale * kLog2e;
    for (int j = 0; j < nt; ++j) {
      const bool valid = ok && rows_s[j * kTile + r] >= 0;
      uint8_t* line = ps + j * kPBytes;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float sv[32];
        if (ok) tmem_row32(lane_base + j * kH + half * 32, sv);     // ok is warp-uniform
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          const float e = valid ? fast_exp2(fmaf(sv[h], c2, -mx_s[half * 32 + h] * kLog2e)) : 0.f;
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
    if (et == 0) CSA_STAMP(3);
    reduce_scatter64<false>(v, lane);
    red[wi * kH + 2 * lane] = v[0];
    red[wi * kH + 2 * lane + 1] = v[1];
    named_barrier(1, 128);
    if (et < kH) {
      const float l = (red[et] + red[kH + et]) + (red[2 * kH + et] + red[3 * kH + et]);
      il_s[et] = 1.f / (l + expf(p.sink[et] - mx_s[et]));
    }
    named_barrier(1, 128);
    // two halves of O^T: thread = dim 128 c + r, 64 heads; each block of 32 heads x 128 dims passes
    // through shared memory and leaves as 16-byte stores (256 contiguous bytes per head)
    __nv_bfloat16* orow = p.out + row * kH * kD;
    for (int half = 0; half < 2; ++half) {
      ok = mbar_wait_warp(half == 0 ? bar_o0 : bar_o1, 0, p.err) && ok;
      if (et == 0) CSA_STAMP(4 + half);
      tc_fence_after();
      for (int cc = 0; cc < 2; ++cc) {
        const int dim = (2 * half + cc) * 128 + r;
        const bool rot = dim >= kD - p.rope.d_rope;
        float cs = 1.f, sn = 0.f;
        if (rot) rope_cs(t, th_hi[(dim - (kD - p.rope.d_rope)) / 2], th_lo[(dim - (kD - p.rope.d_rope)) / 2], cs, sn);
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          float ov[32];
          if (ok) tmem_row32(lane_base + (half == 0 ? kColO : 0u) + cc * kH + hh * 32, ov);
          else {
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = 0.f;
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int h = hh * 32 + j;
            float x = ov[j] * il_s[h];
            if (rot) {                                         // inverse RoPE: the pair partner is lane ^ 1
              const float y = __shfl_xor_sync(0xffffffffu, x, 1);
              x = (lane & 1) ? (x * cs - y * sn) : (x * cs + y * sn);
            }
            ostage[j * kTile + r] = __float2bfloat16_rn(x);
          }
          named_barrier(1, 128);                                 // staged: [32 heads][128 dims]
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int u = et + 128 * i, h = u >> 4, piece = u & 15;
            *reinterpret_cast<uint4*>(orow + (int64_t)(hh * 32 + h) * kD + (2 * half + cc) * 128 + piece * 8) =
                *reinterpret_cast<const uint4*>(ostage + h * kTile + piece * 8);
          }
          named_barrier(1, 128);                                 // the stage is free again
          if (et == 0) CSA_STAMP(48 + 4 * half + 2 * cc + hh);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    CSA_STAMP(6);
#ifdef CSA_TRACE
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    CSA_TRACE_VAL(7, smid + 1);
#endif
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int tc_attn_prefill_max_tiles() { return kMaxTiles; }

cudaError_t tc_attn_prefill(int B, const AttnParams& a, cudaStream_t st, bool pdl) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int win_tiles = (a.window + kTile - 1) / kTile;
  const int64_t comp = a.k > 0 ? (a.k + kTile - 1) / kTile : (a.n_cap + kTile - 1) / kTile;
  if (win_tiles + comp > kMaxTiles) return cudaErrorInvalidValue;
  if ((int64_t)B * a.N >= (int64_t)1 << 31 || (int64_t)B * a.n_cap >= (int64_t)1 << 31) return cudaErrorInvalidValue;
  CUtensorMap qmap;
  cudaError_t e = make_tmap_2d(&qmap, a.q, (int64_t)B * a.S * kH, kD, kH);
  if (e != cudaSuccess) return e;
  PrefillParams p;
  p.kv = static_cast<const __nv_bfloat16*>(a.kv);
  p.ckv = static_cast<const __nv_bfloat16*>(a.ckv);
  p.topk = a.topk; p.pos = a.pos; p.sink = a.sink; p.out = static_cast<__nv_bfloat16*>(a.out);
  p.N = a.N; p.n_cap = a.n_cap; p.S = a.S; p.k = a.k; p.ratio = a.ratio; p.window = a.window;
  p.win_tiles = win_tiles; p.n_tiles = win_tiles + (int)comp; p.scale = a.scale; p.rope = a.rope; p.err = a.err;
  dim3 grid((unsigned)a.S, (unsigned)B);
  return launch_kernel(pdl, attn_prefill_kernel, grid, dim3(kThreads), kSmemBytes, st, qmap, p);
}

}  // namespace csa
