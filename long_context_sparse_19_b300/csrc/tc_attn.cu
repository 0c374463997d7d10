// K4: sparse joint attention on the 5th-generation tensor cores (bf16 storage, H = 64, d = 512).
//
// [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", section "局部和压缩记忆，共用一次归一化": the raw
// window entries and the selected compressed entries form ONE candidate set under one softmax, and
// each head's sink only enlarges the denominator (it is added by the merge kernel). One shared
// 512-dim KV head serves all 64 query heads (K = V), so a tile of candidates is a dense contraction:
//     S^T[c, h] = sum_d KV[c, d] Q[h, d]            (M = 128 candidates, N = 64 heads, K = 512)
//     O^T[d, h] = sum_c KV[c, d] P[h, c]            (M = 4 x 128 dims,   N = 64 heads, K = 128)
// The same shared-memory KV tile is the K-major A operand of the first product and, read along
// the other axis, the MN-major A operand of the second.
//
// One CTA = one query and one 128-candidate tile (window tiles first, then compressed tiles):
//   * warp 0 issues TMA: Q (8 tiled 64 x 64 boxes) and, when the tile is 128 consecutive valid rows
//     (a full window tile, an HCA tile), the rows as 8 tiled 64 x 128 boxes; gathered tiles (top-k
//     selections, partial tiles) are copied by warps 2..5 with 16-byte cp.async, one row per warp
//     instruction pair (fully coalesced), straight into the swizzled tensor-core layout;
//   * warps 2..5 (thread = candidate row = TMEM lane) rotate the raw window rows at their own
//     positions and the query at t (RoPE on dims 448..511, in shared memory), zero rows that are
//     not candidates, then run the softmax on S^T from TMEM: per-head max and sum over the 128
//     candidates by a butterfly reduce-scatter across lanes plus a 4-warp combine, P^T (bf16) into
//     shared memory;
//   * warp 1 issues the two tcgen05.mma chains;
//   * warps 2..5 finally read O^T from TMEM and write the split partial (o, max, sum) in fp32.
#include <cudaTypedefs.h>

#include "tc.h"
#include "tc_ptx.cuh"

namespace csa {
namespace {

using namespace tc;

constexpr int kD = 512;
constexpr int kH = 64;
constexpr int kTile = 128;
constexpr int kThreads = 192;
constexpr uint32_t kKvBlock = kTile * 128;          // 16 KB: one 64-dim column block of the tile
constexpr uint32_t kKvBytes = 8 * kKvBlock;         // 128 KB
constexpr uint32_t kQBlock = kH * 128;              // 8 KB
constexpr uint32_t kQBytes = 8 * kQBlock;           // 64 KB
constexpr uint32_t kPBytes = kTile * 128;           // 16 KB: P^T, one 128-byte line per candidate
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescS = idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdescO = idesc_bf16(128, 64, true, true);
constexpr size_t kSmemBytes = 1024 + kKvBytes + kQBytes + kPBytes + 4096;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnTcParams {
  const __nv_bfloat16* kv;   // [B, N, 512] raw rows
  const __nv_bfloat16* ckv;  // [B, n_cap, 512]
  const int32_t* topk;       // [B, S, k] or null (HCA)
  const int64_t* pos;        // [B, S] or null (t = s)
  float* part_o;             // [B, S, n_split, H, 512]
  float* part_ml;            // [B, S, n_split, H, 2]
  int64_t N, n_cap;
  int S, k, ratio, window, n_split, win_tiles;
  float scale;
  RopeTab rope;
  int32_t* err;
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// rotate the 32 interleaved pairs of one 128-byte swizzled line (dims 448..511) by angle pos*theta_i
__device__ __forceinline__ void rope_line(uint8_t* line_base, uint32_t row, int64_t pos, const float* th_hi,
                                          const float* th_lo) {
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    uint4* p = reinterpret_cast<uint4*>(line_base + ((ch ^ (row & 7u)) << 4));
    uint4 u = *p;
    uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float c, s;
      rope_cs(pos, th_hi[ch * 4 + k], th_lo[ch * 4 + k], c, s);
      const float a = bf16lo(w[k]), b = bf16hi(w[k]);
      w[k] = pack_bf16(a * c - b * s, a * s + b * c);
    }
    *p = u;
  }
}

// butterfly reduce-scatter of 64 per-lane values over the 32 lanes: afterwards lane l holds the
// reduction of heads 2l and 2l+1 in v[0], v[1].
template <bool kMax>
__device__ __forceinline__ void reduce_scatter64(float (&v)[64], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int half = 32 >> step;            // values still held: 2*half -> half
    const int bit = 16 >> step;
    const bool upper = (lane & bit) != 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < half) {
        const float keep = upper ? v[j + half] : v[j];
        const float send = upper ? v[j] : v[j + half];
        const float got = __shfl_xor_sync(0xffffffffu, send, bit);
        v[j] = kMax ? fmaxf(keep, got) : keep + got;
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kvmap,
                   const __grid_constant__ CUtensorMap ckvmap, const AttnTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int n_valid_s;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kvs = smem;                                   // [8 blocks][128 rows][128 B]
  uint8_t* qs = smem + kKvBytes;                         // [8 blocks][64 rows][128 B]
  uint8_t* ps = qs + kQBytes;                            // [128 rows][128 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ps + kPBytes);
  uint64_t* bar_load = bars + 0;      // Q (+ KV when tiled) bytes landed
  uint64_t* bar_ready = bars + 1;     // rope / zeroing done (128 arrivals)
  uint64_t* bar_s = bars + 2;         // S^T in TMEM
  uint64_t* bar_p = bars + 3;         // P^T in smem (128 arrivals)
  uint64_t* bar_o = bars + 4;         // O^T in TMEM
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 6);
  int32_t* rows_s = reinterpret_cast<int32_t*>(bars + 8);           // [128] global row per candidate
  int32_t* valid_s = rows_s + kTile;                                 // [128]
  float* red = reinterpret_cast<float*>(valid_s + kTile);            // [4][64]
  float* m_s = red + 4 * kH;                                         // [64]
  float* l_s = m_s + kH;                                             // [64]
  float* th_hi = l_s + kH;                                           // [32]
  float* th_lo = th_hi + 32;                                         // [32]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, s = blockIdx.y, split = blockIdx.x;
  const int64_t row = (int64_t)b * p.S + s;
  const int64_t t = p.pos ? p.pos[row] : s;
  if (t < 0 || t >= p.N) {                                // uniform over the CTA
    if (threadIdx.x == 0) set_error(p.err, DEVERR_BAD_POS);
    return;
  }
  const int64_t V = min(visible_entries(t, p.ratio), p.n_cap);
  const int64_t lo = t - p.window + 1 > 0 ? t - p.window + 1 : 0;
  const int64_t n_win = t - lo + 1;
  const bool is_win = split < p.win_tiles;

  // ---------------------------------------------------------------- candidate rows of this tile
  if (threadIdx.x == 0) n_valid_s = 0;
  __syncthreads();
  if (threadIdx.x >= 64) {
    const int r = threadIdx.x - 64;
    int64_t g = -1;
    if (is_win) {
      const int64_t c = (int64_t)split * kTile + r;
      if (c < n_win) g = (int64_t)b * p.N + lo + c;
    } else {
      const int64_t slot = (int64_t)(split - p.win_tiles) * kTile + r;
      int64_t idx = -1;
      if (p.topk) {
        if (slot < p.k) idx = p.topk[row * p.k + slot];
      } else if (slot < V) {
        idx = slot;
      }
      if (idx >= V) { set_error(p.err, DEVERR_BAD_INDEX); idx = -1; }
      if (idx >= 0) g = (int64_t)b * p.n_cap + idx;
    }
    valid_s[r] = g >= 0;
    rows_s[r] = (int32_t)g;
    if (g >= 0) atomicAdd(&n_valid_s, 1);
  }
  if (threadIdx.x < 32) { th_hi[threadIdx.x] = p.rope.th_hi[threadIdx.x]; th_lo[threadIdx.x] = p.rope.th_lo[threadIdx.x]; }
  if (threadIdx.x == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_ready, 128);
    mbar_init(bar_s, 1);
    mbar_init(bar_p, 128);
    mbar_init(bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // 128 valid rows that are consecutive in global memory (full window and HCA tiles): tiled TMA
  const bool tiled = n_valid_s == kTile && (is_win || !p.topk);

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tensormap(&qmap);
      mbar_arrive_expect_tx(bar_load, kQBytes + (tiled ? kKvBytes : 0u));
      for (int kb = 0; kb < 8; ++kb) tma_load_2d(qs + kb * kQBlock, &qmap, bar_load, kb * 64, (int32_t)(row * kH));
      if (tiled) {
        const CUtensorMap* map = is_win ? &kvmap : &ckvmap;
        for (int kb = 0; kb < 8; ++kb) tma_load_2d(kvs + kb * kKvBlock, map, bar_load, kb * 64, rows_s[0]);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(bar_ready, 0, p.err);
      if (ok) {
        tc_fence_after();
        const uint32_t kv_addr = smem_u32(kvs), q_addr = smem_u32(qs);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t kb = kk >> 2, in = (kk & 3) * 32;
          mma_bf16(tmem, desc_kmajor_sw128(kv_addr + kb * kKvBlock + in),
                   desc_kmajor_sw128(q_addr + kb * kQBlock + in), kIdescS, kk > 0);
        }
        mma_commit(bar_s);
        ok = mbar_wait(bar_p, 0, p.err);
      }
      if (ok) {
        tc_fence_after();
        const uint32_t kv_addr = smem_u32(kvs), p_addr = smem_u32(ps);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks) {
            mma_bf16(tmem + 64 + mt * 64, desc_mnmajor_sw128(kv_addr + 2 * mt * kKvBlock + ks * 2048, kKvBlock),
                     desc_mnmajor_sw128(p_addr + ks * 2048, kKvBlock), kIdescO, ks > 0);
          }
        }
        mma_commit(bar_o);
      }
    }
  } else {
    // ---------------------------------------------------------------- softmax / epilogue warps
    const int wq = warp & 3;                             // TMEM lane quadrant of this warp
    const int r = 32 * wq + lane;                        // candidate row = TMEM lane of this thread
    const int wi = warp - 2;                             // 0..3
    if (!tiled) {
      // warp wi copies rows wi, wi+4, ...: lane l moves 16-byte chunks l and l+32 of the 1 KB row
      const __nv_bfloat16* base = is_win ? p.kv : p.ckv;
      for (int c = wi; c < kTile; c += 4) {
        if (!valid_s[c]) continue;                       // zeroed below by its owner thread
        const uint8_t* src = reinterpret_cast<const uint8_t*>(base + (int64_t)rows_s[c] * kD);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int gc = lane + 32 * i;                  // 16-byte chunk of the row: dims 8gc..8gc+7
          cp_async16(kvs + (gc >> 3) * kKvBlock + sw128_offset(c, gc & 7), src + gc * 16);
        }
      }
      cp_async_wait_all();
      named_barrier(1, 128);
    }
    bool ok = mbar_wait(bar_load, 0, p.err);
    const bool valid = valid_s[r] != 0;
    if (ok) {
      if (!valid) {                                      // not a candidate: zero its row
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          uint4* line = reinterpret_cast<uint4*>(kvs + kb * kKvBlock + r * 128);
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) line[ch] = make_uint4(0, 0, 0, 0);
        }
      } else if (is_win) {                               // raw row: RoPE at its own position
        rope_line(kvs + 7 * kKvBlock + r * 128, r, lo + (int64_t)split * kTile + r, th_hi, th_lo);
      }
      if (r < kH) rope_line(qs + 7 * kQBlock + r * 128, r, t, th_hi, th_lo);
      fence_proxy_async_smem();
    }
    mbar_arrive(bar_ready);
    if (ok) ok = mbar_wait(bar_s, 0, p.err);
    float sv[64];
    if (ok) {
      tc_fence_after();
      const uint32_t ta = tmem + ((wq * 32) << 16);
      uint32_t u[32];
      tmem_ld32(ta, u);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) sv[j] = valid ? __uint_as_float(u[j]) : -INFINITY;
      tmem_ld32(ta + 32, u);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) sv[32 + j] = valid ? __uint_as_float(u[j]) : -INFINITY;
    } else {
#pragma unroll
      for (int j = 0; j < 64; ++j) sv[j] = -INFINITY;
    }
    // per-head max over the 128 candidates
    float v[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) v[j] = sv[j];
    reduce_scatter64<true>(v, lane);
    red[wi * kH + 2 * lane] = v[0];
    red[wi * kH + 2 * lane + 1] = v[1];
    named_barrier(1, 128);
    if (r < kH) m_s[r] = fmaxf(fmaxf(red[r], red[kH + r]), fmaxf(red[2 * kH + r], red[3 * kH + r]));
    named_barrier(1, 128);
    // probabilities exp(scale * (s - m)), the P^T line of this candidate, per-head sums
    const float c2 = p.scale * kLog2e;
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      const float m = m_s[j];
      v[j] = (m == -INFINITY) ? 0.f : exp2f((sv[j] - m) * c2);
    }
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      uint4 u;
      u.x = pack_bf16(v[8 * ch + 0], v[8 * ch + 1]);
      u.y = pack_bf16(v[8 * ch + 2], v[8 * ch + 3]);
      u.z = pack_bf16(v[8 * ch + 4], v[8 * ch + 5]);
      u.w = pack_bf16(v[8 * ch + 6], v[8 * ch + 7]);
      *reinterpret_cast<uint4*>(ps + sw128_offset(r, ch)) = u;
    }
    fence_proxy_async_smem();
    mbar_arrive(bar_p);
    reduce_scatter64<false>(v, lane);
    red[wi * kH + 2 * lane] = v[0];
    red[wi * kH + 2 * lane + 1] = v[1];
    named_barrier(1, 128);
    if (r < kH) l_s[r] = (red[r] + red[kH + r]) + (red[2 * kH + r] + red[3 * kH + r]);
    named_barrier(1, 128);
    // split partial: max in natural-log units, sum, and the unnormalised o
    const int64_t pi = (row * p.n_split + split) * kH;
    if (r < kH) {
      p.part_ml[2 * (pi + r)] = m_s[r] == -INFINITY ? -INFINITY : m_s[r] * p.scale;
      p.part_ml[2 * (pi + r) + 1] = l_s[r];
    }
    if (ok) ok = mbar_wait(bar_o, 0, p.err);
    if (ok) {
      tc_fence_after();
#pragma unroll 1
      for (int mt = 0; mt < 4; ++mt) {
        const uint32_t ta = tmem + ((wq * 32) << 16) + 64 + mt * 64;
        float* dst = p.part_o + pi * kD + mt * 128 + wq * 32 + lane;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t u[32];
          tmem_ld32(ta + hh * 32, u);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) dst[(int64_t)(hh * 32 + j) * kD] = __uint_as_float(u[j]);
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

int tc_attn_splits(int window, int top_k, int64_t n_cap) {
  const int wt = (window + kTile - 1) / kTile;
  const int64_t ct = top_k > 0 ? (top_k + kTile - 1) / kTile : (n_cap + kTile - 1) / kTile;
  return wt + (int)ct;
}

cudaError_t tc_sparse_attn(int B, const AttnParams& a, void*, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  if (a.n_split != tc_attn_splits(a.window, a.k, a.n_cap) || !a.part_o) return cudaErrorInvalidValue;
  CUtensorMap qmap, kvmap, ckvmap;
  cudaError_t e = make_tmap_2d(&qmap, a.q, (int64_t)B * a.S * kH, kD, kH);
  if (e == cudaSuccess) e = make_tmap_2d(&kvmap, a.kv, (int64_t)B * a.N, kD, kTile);
  if (e == cudaSuccess) e = make_tmap_2d(&ckvmap, a.ckv, (int64_t)B * a.n_cap, kD, kTile);
  if (e != cudaSuccess) return e;
  AttnTcParams p;
  p.kv = static_cast<const __nv_bfloat16*>(a.kv);
  p.ckv = static_cast<const __nv_bfloat16*>(a.ckv);
  p.topk = a.topk; p.pos = a.pos; p.part_o = a.part_o; p.part_ml = a.part_ml; p.N = a.N; p.n_cap = a.n_cap;
  p.S = a.S; p.k = a.k; p.ratio = a.ratio; p.window = a.window; p.n_split = a.n_split;
  p.win_tiles = (a.window + kTile - 1) / kTile; p.scale = a.scale; p.rope = a.rope; p.err = a.err;
  dim3 grid((unsigned)a.n_split, (unsigned)a.S, (unsigned)B);
  attn_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(qmap, kvmap, ckvmap, p);
  return cudaGetLastError();
}

}  // namespace csa
