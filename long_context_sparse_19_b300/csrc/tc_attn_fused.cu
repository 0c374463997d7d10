// K4 + K5 fused for decode: sparse joint attention with the sink and the inverse RoPE, one query per
// thread-block cluster, bf16 output written directly (bf16 storage, H = 64, d = 512, CSA top-k).
//
// [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", sections "局部和压缩记忆，共用一次归一化" (the raw
// window and the selected compressed entries form ONE candidate set under one softmax; each head's
// sink logit enlarges the denominator and owns no value) and "输出投影也分组，并且降低中间维度"
// (o = inverse_RoPE(o) at t). One shared 512-dim KV head serves the 64 query heads (K = V).
//
// The candidates of the query at t are the raw window rows lo..t (lo = max(0, t-W+1)), rotated at
// their own positions, and the top_k selected compressed rows. CTA r of the query's cluster of C
// takes the r-th share of each: window rows [r Wc, (r+1) Wc) and selection slots [r Kc, (r+1) Kc),
// R <= 160 rows in all, every one resident in shared memory at once (K = V: the same tile serves
// both products):
//   S = Q KV^T     M = 64 heads, N = R rows, K = 512: 32 tcgen05.mma into TMEM (an M = 64 accumulator
//                  puts head h on TMEM lane 32 (h / 16) + h % 16, columns = rows);
//   softmax        thread = head: the max over this CTA's rows, P = exp(scale (s - max)) in bf16
//                  (K-major, the A operand of the next product) and the row sum l, each a loop over
//                  32-column TMEM loads, with no cross-thread reduction;
//   O = P KV       M = 64 heads, N = 2 x 256 dims, K = R rows, into the same TMEM columns;
//   partials       thread = head: O / l (a weighted mean of this CTA's rows, so fp16 keeps 11 bits)
//                  and (max, l) go to a global workspace, which stays in L2;
//   merge          after one cluster barrier CTA r owns the output dims [r 512/C, (r+1) 512/C): it
//                  weights the C partials with e^(max_i - M) l_i / L, where M is the overall max with
//                  the sink and L = e^(sink - M) + sum_i e^(max_i - M) l_i, applies the inverse RoPE
//                  and stores bf16.
// Measured on this part, one SM reads L2 several times faster than another CTA's shared memory,
// hence the exchange through L2. The window rows and the query do not depend on the selection:
// under programmatic dependent launch they are fetched (and rotated) before the kernel waits for
// the selection kernel. The code on this path runs once per CTA, where instruction fetch
// dominates, so it is kept to short loops.
// With the low-precision cache (FP4 E2M1 latent + FP8 E4M3 tail, lowp.cuh; 304 instead of 1024
// bytes per entry) each selected row is loaded into one thread's registers (14 E2M1 pieces of one
// 32-dim block each, the scale record, 4 E4M3 pieces) and expanded into the same bf16 tile (exact).
// Warps: 0 = Q TMA and tcgen05.mma issuer (one lane), 1..7 gather the window rows, 1 = TMEM owner
// and RoPE of the query, 2..7 gather the selected rows, 4..7 then run the softmax and the O
// epilogue (lanes 0..15: one head each, TMEM lane quadrant = warp % 4); all eight merge.
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "lowp.cuh"
#include "tc.h"
#include "tc_ptx.cuh"

namespace csa {
namespace {

using namespace tc;

constexpr int kD = 512;
constexpr int kH = 64;
constexpr int kThreads = 256;
constexpr int kMaxRows = 160;                        // candidate rows per CTA
constexpr int kCluMax = 8;
constexpr uint32_t kRowBytes = 128;                  // one 64-dim block of one row
constexpr uint32_t kBlkStride = kMaxRows * kRowBytes;   // 20 KB: [160 rows][128 B] swizzled, per 64 dims
constexpr uint32_t kKvBytes = 8 * kBlkStride;        // 160 KB
constexpr uint32_t kQBlock = kH * 128;               // 8 KB: [64 heads][64 dims]
constexpr uint32_t kQBytes = 8 * kQBlock;            // 64 KB: Q, then P
constexpr uint32_t kPBlock = kH * 128;               // 8 KB: P of 64 rows, [64 heads][64 rows] swizzled
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescO = idesc_bf16(64, 256, false, true);
constexpr size_t kAuxBytes = 1536;                   // row table, barriers, RoPE tables
constexpr size_t kSmemBytes = 1024 + kKvBytes + kQBytes + kAuxBytes;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kGather = kThreads - 64;               // warps 2..7 gather the selected rows
static_assert(kMaxRows <= 3 * 64 && 3 * kPBlock + kCluMax * kH * 4 <= kQBytes, "P and the weights fit");

struct FusedParams {
  const __nv_bfloat16* kv;   // [B, N, 512] raw rows
  const void* ckv;           // [B, n_cap, 512] bf16, or the low-precision planes (kLowp)
  const int32_t* topk;       // [B, k]
  const int64_t* pos;        // [B]
  const float* sink;         // [64]
  __nv_bfloat16* out;        // [B, 64, 512]
  __half* part;              // [B, C, 64, 512] O / l of each CTA (workspace)
  float* pstat;              // [B, C, 64, 2] (max, l) of each CTA (workspace)
  int64_t N, n_cap;
  int k, ratio, window, Wc, Kc, R;
  float scale;
  RopeTab rope;
  int32_t* err;
};

// The merge of one output slice: dims [rank 512/C, (rank+1) 512/C) of the 64 heads. Thread t takes
// the 8-dim pieces t + kThreads j (j < PER); the loads of all C partials (C PER = 16) are issued
// before any is used.
template <int PER>
__device__ __forceinline__ void merge_slice(const FusedParams& p, const float* wgt, const float* th_hi,
                                            const float* th_lo, uint32_t rank, int b, int64_t t) {
  constexpr int C = 16 / PER;
  constexpr int Dc = kD / C, q8 = Dc / 8;                      // 8-dim pieces per head row of the slice
  const int D0 = (int)rank * Dc;
  const __half* part = p.part + (int64_t)b * C * kH * kD;
  uint4 o[C * PER];
#pragma unroll
  for (int i = 0; i < C * PER; ++i) {
    const int r = i / PER, idx = threadIdx.x + kThreads * (i % PER);
    o[i] = __ldcg(reinterpret_cast<const uint4*>(part + ((int64_t)r * kH + idx / q8) * kD + D0 + 8 * (idx % q8)));
  }
  const int r0 = kD - p.rope.d_rope;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int idx = threadIdx.x + kThreads * j;
    const int hh = idx / q8, d = D0 + 8 * (idx % q8);
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = 0.f;
#pragma unroll
    for (int r = 0; r < C; ++r) {
      const float w = wgt[r * kH + hh];
      const __half2* hv = reinterpret_cast<const __half2*>(&o[r * PER + j]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(hv[e]);
        v[2 * e] = fmaf(w, f.x, v[2 * e]);
        v[2 * e + 1] = fmaf(w, f.y, v[2 * e + 1]);
      }
    }
    if (d >= r0) {                                             // inverse RoPE at t, pairs (d + 2e, d + 2e + 1)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 cs = rope_cs_nl(t, th_hi[(d - r0) / 2 + e], th_lo[(d - r0) / 2 + e]);
        const float x = v[2 * e], y = v[2 * e + 1];
        v[2 * e] = x * cs.x + y * cs.y;
        v[2 * e + 1] = -x * cs.y + y * cs.x;
      }
    }
    store8(p.out + ((int64_t)b * kH + hh) * kD + d, v);
  }
}

template <bool kLowp>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fused_kernel(const __grid_constant__ CUtensorMap qmap, const FusedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* kvs = smem;                                         // [8 blocks][160 rows][128 B]
  uint8_t* qs = smem + kKvBytes;                               // Q: [8 blocks][64 heads][128 B]
  uint8_t* ps = qs;                                            // P: [3 blocks][64 heads][128 B] (after S)
  float* wgt = reinterpret_cast<float*>(qs + 3 * kPBlock);     // [C][64] merge weights
  uint8_t* aux = qs + kQBytes;
  int32_t* rows_s = reinterpret_cast<int32_t*>(aux);           // [160] global row (-1 = empty)
  uint64_t* bars = reinterpret_cast<uint64_t*>(aux + kMaxRows * 4 + 32);
  uint64_t* bar_q = bars;                                      // Q landed (tx)
  uint64_t* bar_qrot = bars + 1;                               // Q and warp 1's window pieces rotated (32)
  uint64_t* bar_kv = bars + 2;                                 // the selected rows landed (kGather arrivals)
  uint64_t* bar_s = bars + 3;                                  // S complete
  uint64_t* bar_p = bars + 4;                                  // P written (64 arrivals)
  uint64_t* bar_o = bars + 5;                                  // O complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 6);
  float* th_hi = reinterpret_cast<float*>(bars + 8);           // [32]
  float* th_lo = th_hi + 32;                                   // [32]
  float* q_cs = th_lo + 32;                                    // [32]
  float* q_sn = q_cs + 32;                                     // [32]

  if (threadIdx.x == 0) CSA_STAMP(0);
  griddep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int b = blockIdx.y;
  const uint32_t rank = cluster_rank(), C = gridDim.x;
  const int R = p.R;
  int64_t t = p.pos[b];
  const bool bad_pos = t < 0 || t >= p.N;
  if (bad_pos) {                                               // no early exit: the cluster barrier follows
    if (tid == 0 && rank == 0) set_error(p.err, DEVERR_BAD_POS);
    t = 0;
  }
  const int64_t V = min(visible_entries(t, p.ratio), p.n_cap);
  const int64_t lo = t - p.window + 1 > 0 ? t - p.window + 1 : 0;
  const int64_t n_win = bad_pos ? 0 : t - lo + 1;

  if (tid < 32) { th_hi[tid] = p.rope.th_hi[tid]; th_lo[tid] = p.rope.th_lo[tid]; }
  if (tid == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_qrot, 32);
    mbar_init(bar_kv, kGather);
    mbar_init(bar_s, 1);
    mbar_init(bar_p, 64);
    mbar_init(bar_o, 1);
    fence_mbar_init();
  }
  // window rows of this CTA: known before the selection
  for (int i = tid; i < p.Wc; i += kThreads) {
    const int64_t w = (int64_t)rank * p.Wc + i;
    rows_s[i] = w < n_win ? (int32_t)((int64_t)b * p.N + lo + w) : -1;
  }
  for (int i = p.Wc + p.Kc + tid; i < R; i += kThreads) rows_s[i] = -1;   // K padding rows
  if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // piece u of the row range: row u / 64, 16-byte piece u % 64 (dim block (u % 64) / 8); empty rows
  // are zero-filled (the O product reads every row up to R). Eight row-table reads are issued ahead
  // of their eight copies (a copy's memory clobber would otherwise hold each read behind it).
  auto gather = [&](int r0, int r1, const __nv_bfloat16* base, int g, int ng) {
    const int u_end = r1 * 64;
#pragma unroll 1
    for (int u0 = r0 * 64 + g; u0 < u_end; u0 += 8 * ng) {
      int32_t gr[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int u = u0 + k * ng;
        gr[k] = u < u_end ? rows_s[u >> 6] : -1;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int u = u0 + k * ng;
        if (u < u_end) {
          const int rr = u >> 6, piece = u & 63;
          uint8_t* dst = kvs + (piece >> 3) * kBlkStride + sw128_offset(rr, piece & 7);
          if (gr[k] >= 0) cp_async16(dst, base + (int64_t)gr[k] * kD + piece * 8);
          else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
      }
    }
    cp_async_commit();
  };

  // kLowp: rows [r0, r1) from the low-precision cache, one row per thread: its 14 E2M1 pieces (one
  // 32-dim block each), its scale record and its 4 E4M3 pieces are all loaded before any is expanded.
  // Empty rows read as zero codes, which expand to zeros.
  auto gather_lowp = [&](int r0, int r1, int g, int ng) {
    const LowpLayout kl = lowp_layout(kD, p.n_cap, 64);
    const uint8_t* kb = static_cast<const uint8_t*>(p.ckv) + (int64_t)b * kl.stride;
#pragma unroll 1
    for (int rr = r0 + g; rr < r1; rr += ng) {
      const int32_t gr = rows_s[rr];
      uint4 v4[14], v8[4], sr = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < 14; ++j) v4[j] = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < 4; ++j) v8[j] = make_uint4(0, 0, 0, 0);
      if (gr >= 0) {
        const int64_t e = gr - (int64_t)b * p.n_cap;
        const uint4* p4 = reinterpret_cast<const uint4*>(kb + e * 224);
        const uint4* p8 = reinterpret_cast<const uint4*>(kb + kl.fp8 + e * 64);
#pragma unroll
        for (int j = 0; j < 14; ++j) v4[j] = __ldcg(p4 + j);
#pragma unroll
        for (int j = 0; j < 4; ++j) v8[j] = __ldcg(p8 + j);
        sr = __ldcg(reinterpret_cast<const uint4*>(kb + kl.scale + e * 16));
      }
      if (g == 0 && rr == r0) CSA_STAMP(8);
      const uint32_t sw[4] = {sr.x, sr.y, sr.z, sr.w};
#pragma unroll
      for (int j = 0; j < 14; ++j) {                           // dims 32 j .. 32 j + 31
        const float sc = e8m0_to_f32((sw[j >> 2] >> (8 * (j & 3))) & 255u);
        uint8_t* dst = kvs + (j >> 1) * kBlkStride;
        const int c0 = (j & 1) * 4;
        *reinterpret_cast<uint4*>(dst + sw128_offset(rr, c0 + 0)) = dequant_fp4x8(v4[j].x, sc);
        *reinterpret_cast<uint4*>(dst + sw128_offset(rr, c0 + 1)) = dequant_fp4x8(v4[j].y, sc);
        *reinterpret_cast<uint4*>(dst + sw128_offset(rr, c0 + 2)) = dequant_fp4x8(v4[j].z, sc);
        *reinterpret_cast<uint4*>(dst + sw128_offset(rr, c0 + 3)) = dequant_fp4x8(v4[j].w, sc);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {                            // dims 448 + 16 q .. + 15
        uint8_t* dst = kvs + 7 * kBlkStride;
        *reinterpret_cast<uint4*>(dst + sw128_offset(rr, 2 * q)) = dequant_fp8x8(v8[q].x, v8[q].y);
        *reinterpret_cast<uint4*>(dst + sw128_offset(rr, 2 * q + 1)) = dequant_fp8x8(v8[q].z, v8[q].w);
      }
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- Q load + MMA issuer
      prefetch_tensormap(&qmap);
      mbar_arrive_expect_tx(bar_q, kQBytes);
      for (int kb = 0; kb < 8; ++kb) tma_load_2d(qs + kb * kQBlock, &qmap, bar_q, kb * 64, b * kH);
      bool ok = mbar_wait(bar_q, 0, p.err) && mbar_wait(bar_qrot, 0, p.err) && mbar_wait(bar_kv, 0, p.err);
      CSA_STAMP(11);
      if (ok) {
        tc_fence_after();
        const uint32_t q_addr = smem_u32(qs), kv_addr = smem_u32(kvs), p_addr = smem_u32(ps);
        const uint32_t idesc_s = idesc_bf16(64, R, false, false);
#pragma unroll 1
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;
          mma_bf16(tmem, desc_kmajor_sw128(q_addr + (kk >> 2) * kQBlock + off),
                   desc_kmajor_sw128(kv_addr + (kk >> 2) * kBlkStride + off), idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_s);
        CSA_STAMP(3);
        ok = mbar_wait(bar_p, 0, p.err);                       // also: every read of S is done
        CSA_STAMP(19);
        if (ok) {
          tc_fence_after();
#pragma unroll 1
          for (int ks = 0; ks < R / 16; ++ks) {
            const uint64_t a = desc_kmajor_sw128(p_addr + (ks >> 2) * kPBlock + (ks & 3) * 32);
            mma_bf16(tmem, a, desc_mnmajor_sw128(kv_addr + ks * 2048, kBlkStride), kIdescO, ks > 0 ? 1u : 0u);
            mma_bf16(tmem + 256, a, desc_mnmajor_sw128(kv_addr + 4 * kBlkStride + ks * 2048, kBlkStride), kIdescO,
                     ks > 0 ? 1u : 0u);
          }
          CSA_STAMP(20);
          mma_commit(bar_o);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- rows (warps 1..7)
    // the window rows first (known before the selection), then, for warps 2..7 after the wait for
    // the selection kernel, the selected rows; every thread rotates the dims 448..511 pieces of
    // window rows that it copied itself, at each row's own position
    const int g = tid - 32;
    gather(0, p.Wc, p.kv, g, kThreads - 32);
    auto rotate_own_window_pieces = [&]() {
#pragma unroll 1
      for (int u = g; u < p.Wc * 64; u += kThreads - 32) {
        const int rr = u >> 6, piece = u & 63;
        if (piece < 56 || rows_s[rr] < 0) continue;
        uint4* q16 = reinterpret_cast<uint4*>(kvs + 7 * kBlkStride + sw128_offset(rr, piece - 56));
        uint4 v = *q16;
        uint32_t* w = reinterpret_cast<uint32_t*>(&v);
        const int64_t pos_r = lo + (int64_t)rank * p.Wc + rr;
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
          const int pair = (piece - 56) * 4 + k;
          const float2 cs = rope_cs_nl(pos_r, th_hi[pair], th_lo[pair]);
          const float a = bf16lo(w[k]), bb = bf16hi(w[k]);
          w[k] = pack_bf16(a * cs.x - bb * cs.y, a * cs.y + bb * cs.x);
        }
        *q16 = v;
      }
    };
    if (warp == 1) {
      // RoPE of the query at t (every head: lane i computes pair i's cos / sin once)
      const float2 cs_i = rope_cs_nl(t, th_hi[lane], th_lo[lane]);
      q_cs[lane] = cs_i.x;
      q_sn[lane] = cs_i.y;
      __syncwarp();
      if (mbar_wait_warp(bar_q, 0, p.err)) {
        rope_line_tab(qs + 7 * kQBlock + lane * 128, lane, q_cs, q_sn);
        rope_line_tab(qs + 7 * kQBlock + (lane + 32) * 128, lane + 32, q_cs, q_sn);
      }
      cp_async_wait<0>();
      rotate_own_window_pieces();
      fence_proxy_async_smem();
      mbar_arrive(bar_qrot);
      if (lane == 0) CSA_STAMP(16);
    } else {
      const int gs = tid - 64;                                 // selected rows: warps 2..7
      griddep_wait();                                          // the selection (and the closed entry) is ready
      if (gs == 0) CSA_STAMP(1);
      for (int i = gs; i < p.Kc; i += kGather) {
        const int64_t slot = (int64_t)rank * p.Kc + i;
        int64_t idx = slot < p.k ? p.topk[(int64_t)b * p.k + slot] : -1;
        if (idx >= V) { set_error(p.err, DEVERR_BAD_INDEX); idx = -1; }
        rows_s[p.Wc + i] = idx >= 0 && !bad_pos ? (int32_t)((int64_t)b * p.n_cap + idx) : -1;
      }
      named_barrier(2, kGather);                               // the row table is complete
      if constexpr (kLowp) {
        gather_lowp(p.Wc, R, gs, kGather);
        if (gs == 0) CSA_STAMP(9);
        cp_async_wait<0>();                                    // this thread's window pieces landed
        if (gs == 0) CSA_STAMP(10);
        rotate_own_window_pieces();
      } else {
        gather(p.Wc, R, static_cast<const __nv_bfloat16*>(p.ckv), gs, kGather);
        cp_async_wait<1>();                                    // this thread's window pieces landed
        rotate_own_window_pieces();
        cp_async_wait<0>();
      }
      fence_proxy_async_smem();
      mbar_arrive(bar_kv);
      if (gs == 0) CSA_STAMP(2);
    }
  }
  if (warp >= 4) {
    const int wq = warp & 3;                                   // TMEM lane quadrant
    const uint32_t lane_base = tmem + ((wq * 32) << 16);
    bool ok = mbar_wait_warp(bar_s, 0, p.err);                 // warp-uniform
    if (tid == 128) CSA_STAMP(17);
    tc_fence_after();
    // ---------------------------------------------------------------- softmax: thread = head
    // head h = 16 wq + lane sits on TMEM lane 32 wq + lane (lanes 16..31 of the warp load what the
    // M = 64 products leave unused and discard it); columns are the CTA's rows
    const int h = 16 * wq + lane;
    const bool head = lane < 16;
    const int n_ch = (R + 31) / 32;
    float m = -INFINITY;
#pragma unroll 1
    for (int ch = 0; ch < n_ch && ok; ++ch) {
      float sv[32];
      tmem_row32(lane_base + ch * 32, sv);
      const int rw = 32 * ch + lane;                           // valid rows of the chunk, one bit each
      const uint32_t vb = __ballot_sync(0xffffffffu, rw < R && rows_s[rw] >= 0);
#pragma unroll
      for (int j = 0; j < 32; ++j) m = fmaxf(m, (vb >> j) & 1u ? sv[j] : -INFINITY);
    }
    if (tid == 128) CSA_STAMP(18);
    const float c2 = p.scale * kLog2e;
    float l = 0.f;
#pragma unroll 1
    for (int ch = 0; ch < n_ch; ++ch) {
      float sv[32];
      if (ok) tmem_row32(lane_base + ch * 32, sv);             // ok is warp-uniform
      const int rw = 32 * ch + lane;
      const uint32_t vb = ok ? __ballot_sync(0xffffffffu, rw < R && rows_s[rw] >= 0) : 0u;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float e = (vb >> j) & 1u ? fast_exp2((sv[j] - m) * c2) : 0.f;
        sv[j] = e;
        l += e;
      }
      if (head) {                                              // rows 32 ch .. 32 ch + 31 of P (K-major)
        uint8_t* blk = ps + (ch >> 1) * kPBlock;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 u;
          u.x = pack_bf16(sv[8 * q + 0], sv[8 * q + 1]);
          u.y = pack_bf16(sv[8 * q + 2], sv[8 * q + 3]);
          u.z = pack_bf16(sv[8 * q + 4], sv[8 * q + 5]);
          u.w = pack_bf16(sv[8 * q + 6], sv[8 * q + 7]);
          *reinterpret_cast<uint4*>(blk + sw128_offset(h, (ch & 1) * 4 + q)) = u;
        }
      }
    }
    tc_fence_before();
    if (head) {
      fence_proxy_async_smem();
      mbar_arrive(bar_p);
    }
    if (tid == 128) CSA_STAMP(4);
    // ---------------------------------------------------------------- partials (thread = head)
    if (head) {
      float* st = p.pstat + (((int64_t)b * C + rank) * kH + h) * 2;
      st[0] = m == -INFINITY ? -INFINITY : m * p.scale;        // max in logit units
      st[1] = l;
    }
    const float il = l > 0.f ? 1.f / l : 0.f;
    __half* prow = p.part + (((int64_t)b * C + rank) * kH + (head ? h : 0)) * kD;
    ok = mbar_wait_warp(bar_o, 0, p.err) && ok;
    if (tid == 128) CSA_STAMP(5);
    tc_fence_after();
#pragma unroll 1
    for (int ch = 0; ch < kD / 32; ++ch) {                     // dims 32 ch .. 32 ch + 31
      float ov[32];
      if (ok) tmem_row32(lane_base + ch * 32, ov);
      else {
#pragma unroll
        for (int j = 0; j < 32; ++j) ov[j] = 0.f;
      }
      if (head) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 u;
          __half2* hv = reinterpret_cast<__half2*>(&u);
#pragma unroll
          for (int e = 0; e < 4; ++e) hv[e] = __floats2half2_rn(ov[8 * q + 2 * e] * il, ov[8 * q + 2 * e + 1] * il);
          *reinterpret_cast<uint4*>(prow + ch * 32 + 8 * q) = u;
        }
      }
    }
    if (tid == 128) CSA_STAMP(21);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();                                              // every CTA's partials are in memory
  if (tid == 0) CSA_STAMP(6);

  // ---------------------------------------------------------------- merge (all threads)
  //   w_i = e^(max_i - M) l_i / (e^(sink - M) + sum_j e^(max_j - M) l_j),  M = max(sink, max_j)
  if (tid < kH) {
    const int h = tid;
    const float sk = p.sink[h];
    const float* st = p.pstat + ((int64_t)b * C * kH + h) * 2;
    float2 ml[kCluMax];
#pragma unroll
    for (int r = 0; r < kCluMax; ++r)
      if (r < (int)C) ml[r] = __ldcg(reinterpret_cast<const float2*>(st + (int64_t)r * kH * 2));
    float M = sk;
#pragma unroll
    for (int r = 0; r < kCluMax; ++r)
      if (r < (int)C) M = fmaxf(M, ml[r].x);
    float L = expf(sk - M);
#pragma unroll
    for (int r = 0; r < kCluMax; ++r) {
      if (r < (int)C) {
        const float e = ml[r].x == -INFINITY ? 0.f : expf(ml[r].x - M) * ml[r].y;
        wgt[r * kH + h] = e;
        L += e;
      }
    }
    const float inv = 1.f / L;
#pragma unroll
    for (int r = 0; r < kCluMax; ++r)
      if (r < (int)C) wgt[r * kH + h] *= inv;
  }
  __syncthreads();
  if (tid == 0) CSA_STAMP(22);
  if (C == 2) merge_slice<8>(p, wgt, th_hi, th_lo, rank, b, t);
  else if (C == 4) merge_slice<4>(p, wgt, th_hi, th_lo, rank, b, t);
  else merge_slice<2>(p, wgt, th_hi, th_lo, rank, b, t);
  if (tid == 0) CSA_STAMP(7);
}

}  // namespace

// Shares of one query's candidates over a cluster of C CTAs: window rows Wc, selection slots Kc,
// rows R (padded to 16). Returns C (2, 4 or 8), or 0 when the fused kernel does not apply.
int tc_attn_fused_plan(int B, int window, int top_k, int* Wc, int* Kc, int* R) {
  if (top_k <= 0 || B <= 0) return 0;
  int c = 0;
  for (int cc = 2; cc <= kCluMax; cc *= 2) {
    const int wc = (window + cc - 1) / cc, kc = (top_k + cc - 1) / cc;
    if (((wc + kc + 15) / 16) * 16 <= kMaxRows) { c = cc; break; }
  }
  if (!c) return 0;
  // spread a small batch over more SMs
  while (c < kCluMax && (int64_t)B * (c * 2) <= tc_sm_count()) c *= 2;
  *Wc = (window + c - 1) / c;
  *Kc = (top_k + c - 1) / c;
  *R = ((*Wc + *Kc + 15) / 16) * 16;
  static int fits[kCluMax + 1] = {0};                          // 1 = placeable, -1 = not
  if (!fits[c]) {
    cudaError_t e = cudaFuncSetAttribute(attn_fused_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_fused_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    int n = 0;
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)c, 1);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = kSmemBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)c;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&n, attn_fused_kernel<false>, &cfg);
    }
    if (e != cudaSuccess) (void)cudaGetLastError();
    fits[c] = (e == cudaSuccess && n > 0) ? 1 : -1;
  }
  return fits[c] > 0 ? c : 0;
}

size_t tc_attn_fused_workspace(int B, int C) {
  return (size_t)B * C * kH * (kD * sizeof(__half) + 2 * sizeof(float));
}

cudaError_t tc_attn_fused(int B, int C, int Wc, int Kc, int R, const AttnParams& a, void* ws, cudaStream_t st,
                          bool pdl, bool lowp) {
  if ((C != 2 && C != 4 && C != 8) || R > kMaxRows || R % 16 != 0 || Wc + Kc > R || a.S != 1 || !a.topk ||
      a.H != kH || !ws)
    return cudaErrorInvalidValue;
  if ((int64_t)B * a.N >= (int64_t)1 << 31 || (int64_t)B * a.n_cap >= (int64_t)1 << 31) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(lowp ? attn_fused_kernel<true> : attn_fused_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  CUtensorMap qmap;
  e = make_tmap_2d(&qmap, a.q, (int64_t)B * kH, kD, kH);
  if (e != cudaSuccess) return e;
  FusedParams p;
  p.kv = static_cast<const __nv_bfloat16*>(a.kv);
  p.ckv = a.ckv;
  p.topk = a.topk; p.pos = a.pos; p.sink = a.sink; p.out = static_cast<__nv_bfloat16*>(a.out);
  p.part = static_cast<__half*>(ws);
  p.pstat = reinterpret_cast<float*>(static_cast<char*>(ws) + (size_t)B * C * kH * kD * sizeof(__half));
  p.N = a.N; p.n_cap = a.n_cap; p.k = a.k; p.ratio = a.ratio; p.window = a.window;
  p.Wc = Wc; p.Kc = Kc; p.R = R; p.scale = a.scale; p.rope = a.rope; p.err = a.err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C, (unsigned)B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
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
  return cudaLaunchKernelEx(&cfg, lowp ? attn_fused_kernel<true> : attn_fused_kernel<false>, qmap, p);
}

}  // namespace csa
