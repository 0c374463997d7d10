// K2 / K6: indexer scores on the 5th-generation tensor cores (bf16 storage, H_idx = 64, d_idx = 128).
//
// [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", section "少读 KV 之前，Indexer 仍要给历史打分":
//     s_i = sum_h w_h * max(0, rope(q_h, t) . cidx_i),   i < (t+1)/m,
// w signed (not a softmax), summed over the 64 heads before selection.
//
// One CTA scores a contiguous run of 128-entry tiles of one query's visible index cache:
//   * warp 0 (one lane) streams the cache tiles with TMA (two 64-dim boxes per tile, 128-byte
//     swizzle) through a 2-stage shared-memory ring;
//   * warp 1 (one lane) issues tcgen05.mma M=128 (entries) x N=128 x K=128 into a double-buffered
//     TMEM accumulator. The N dimension holds the rotated query twice: rows 0..63 its bf16 value
//     per head (hi) and rows 64..127 the bf16 rounding remainder (lo), so hi + lo carries the
//     rotated fp32 query to ~16 bits and the scores keep fp32-level accuracy (over the unrotated
//     dims the remainder is zero, and those K-slices run with N=64);
//   * warps 2..5 first build that query operand in shared memory (RoPE at t, hi/lo split,
//     swizzled K-major layout), then run the epilogue: thread = entry, 2 x 64 TMEM columns ->
//     sum_h w_h * relu(hi_h + lo_h) -> one coalesced fp32 score store.
// The cache stream is the only large traffic (256 B per visible entry), so the kernel is bound by
// HBM bandwidth; two CTAs share an SM (about 98 KB shared memory and 256 TMEM columns each).
//
// In a decode step this kernel is the first launch and also runs the compressor's close step
// ([FLASH] "压缩是逐通道的 learned pooling": when t completes a group, entry t / m is pooled):
// right after building the query, the epilogue threads of the CTA that scores the request's last
// tile pool the new index entry, store it, order the store before the async proxy and release an
// mbarrier that gates the TMA load of that tile; the CTA that owns tile 0 pools the new KV entry
// (the attention reads it later) and takes one tile fewer to make up for it. A separate close
// kernel would hold 64 SMs' registers while this kernel's CTAs wait to start.
#include <cudaTypedefs.h>

#include <mutex>

#include "close_entry.cuh"
#include "tc.h"
#include "tc_ptx.cuh"

namespace csa {
namespace {

using namespace tc;

constexpr int kDI = 128;
constexpr int kTileM = 128;
constexpr int kStages = 2;
constexpr uint32_t kTileBytes = kTileM * kDI * 2;           // 32 KB: two 16 KB swizzle blocks
constexpr uint32_t kBlockBytes = 16384;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kIdesc = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescHi = idesc_bf16(128, 64, false, false);   // the value rows only
constexpr size_t kSmemBytes = 1024 /*align*/ + kTileBytes /*query operand*/ + kStages * kTileBytes + 512;

struct IndexTcParams {
  const __nv_bfloat16* q_idx;   // [B, S, 64, 128]
  const float* w;               // [B, S, 64]
  float* scores;                // [B, S, n_cap]
  const int64_t* pos;           // [B, S] or null (t = s)
  int64_t n_cap;
  int64_t entry_base;           // cidx holds the entries [entry_base, entry_base + n_cap)
  int S, ratio, chunks;
  RopeTab rope;
  int32_t* err;
  // decode only (close.job[0].src non-null): the entry that t closes is pooled here first, the
  // index entry by the CTA that scores it and the KV entry by the CTA that owns tile 0
  CompressParams close;
};

__global__ void __launch_bounds__(kThreads, 2)
    index_tc_kernel(const __grid_constant__ CUtensorMap cmap, const IndexTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* qop = smem;                                      // [2 blocks][128 rows][128 B]
  uint8_t* stage_base = smem + kTileBytes;                  // kStages x [2 blocks][128 rows][128 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage_base + kStages * kTileBytes);
  uint64_t* full = bars;                                    // [kStages]
  uint64_t* empty = bars + kStages;                         // [kStages]
  uint64_t* tfull = bars + 2 * kStages;                     // [2]
  uint64_t* tempty = bars + 2 * kStages + 2;                // [2]
  uint64_t* qready = bars + 2 * kStages + 4;
  uint64_t* closed = bars + 2 * kStages + 5;                // the index entry is in global memory
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 6);
  float* w_s = reinterpret_cast<float*>(tmem_slot + 4);    // [64]
  float* red = w_s + 64;                                    // [2][4]

  if (threadIdx.x == 0) CSA_STAMP(42);
  griddep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, s = blockIdx.y;
  const int64_t row = (int64_t)b * p.S + s;
  const int64_t t = p.pos ? p.pos[row] : s;
  const int64_t V = visible_local(t, p.ratio, p.entry_base, p.n_cap);
  const int64_t T = (V + kTileM - 1) / kTileM;
  // decode close: t completes group e = t / m, which makes entry e = V - 1 visible (uniform per CTA)
  const bool fused = p.close.job[0].src != nullptr;
  const bool group_done = fused && t >= 0 && t < p.close.N && (t + 1) % p.ratio == 0;
  if (fused && blockIdx.x == 0 && threadIdx.x == 0 && (t < 0 || t >= p.close.N || (group_done && t / p.ratio >= p.n_cap)))
    set_error(p.err, DEVERR_BAD_POS);
  const bool closes = group_done && t / p.ratio < p.n_cap;  // then V = e + 1: entry e is the last visible
  // pooling the KV entry costs the tile-0 CTA about one tile: with a close, that CTA gets one
  // tile fewer (the split runs over T + 1 tiles, the first of them virtual)
  const int64_t Tv = closes && p.chunks > 1 ? T + 1 : T;
  const int64_t sh = Tv - T;
  const int64_t tile0 = max((int64_t)blockIdx.x * Tv / p.chunks - sh, (int64_t)0);
  const int64_t tile1 = max((int64_t)(blockIdx.x + 1) * Tv / p.chunks - sh, (int64_t)0);
  const int ntiles = (int)(tile1 - tile0);
  if (ntiles <= 0) return;                                  // uniform over the CTA
  const bool close_kv = closes && tile0 == 0;               // pools ckv entry e
  const bool close_idx = closes && tile1 == T;              // pools cidx entry e, scored in its last tile

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&tfull[i], 1); mbar_init(&tempty[i], 128); }
    mbar_init(qready, 128);
    mbar_init(closed, 128);
    fence_mbar_init();
  }
  if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tensormap(&cmap);
      griddep_wait();                                       // the cache may come from the previous kernel
      // the cache streams through once: keep it from evicting the scores the selection reads next
      const uint64_t policy = l2_evict_first_policy();
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % kStages;
        if (i >= kStages && !mbar_wait(&empty[st], ((i / kStages) & 1) ^ 1, p.err)) break;
        if (close_idx && i == ntiles - 1 && !mbar_wait(closed, 0, p.err)) break;   // holds entry e
        mbar_arrive_expect_tx(&full[st], kTileBytes);
        const int32_t y = (int32_t)(b * p.n_cap + (tile0 + i) * kTileM);
        uint8_t* dst = stage_base + st * kTileBytes;
        tma_load_2d_hint(dst, &cmap, &full[st], 0, y, policy);
        tma_load_2d_hint(dst + kBlockBytes, &cmap, &full[st], 64, y, policy);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && mbar_wait(qready, 0, p.err)) {
      tc_fence_after();
      const uint32_t q_addr = smem_u32(qop);
      const bool hi_only0 = p.rope.d_rope <= kDI / 2;
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % kStages, acc = i & 1;
        if (!mbar_wait(&full[st], (i / kStages) & 1, p.err)) break;
        if (i >= 2 && !mbar_wait(&tempty[acc], ((i >> 1) & 1) ^ 1, p.err)) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(stage_base + st * kTileBytes);
        const uint32_t d = tmem + acc * 128;
        // Dims 0..63 are not rotated when d_rope <= 64: the query there is its bf16 input, so its
        // remainder rows are zero and those four K-slices take the value rows only (N = 64). The
        // rotated block goes first, so that its first product initialises all 128 columns.
#pragma unroll
        for (int u = 0; u < kDI / 16; ++u) {
          const int kk = (u + 4) % (kDI / 16);
          const uint32_t off = (kk >> 2) * kBlockBytes + (kk & 3) * 32;
          mma_bf16(d, desc_kmajor_sw128(a_addr + off), desc_kmajor_sw128(q_addr + off),
                   (kk < 4 && hi_only0) ? kIdescHi : kIdesc, u > 0);
        }
        mma_commit(&empty[st]);
        mma_commit(&tfull[acc]);
      }
    }
  } else {
    // ---------------------------------------------------------------- query operand + epilogue
    const int et = threadIdx.x - 64;                        // 0..127
    const __nv_bfloat16* q = p.q_idx + row * 64 * kDI;
    const int r0 = kDI - p.rope.d_rope;
    // thread et owns the 8-dim chunk c = et % 16 of heads et/16 + 8 i, i < 8: all loads first
    const int c = et % (kDI / 8), h0 = et / (kDI / 8);
    float xs[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) load8(q + (h0 + 8 * i) * kDI + c * 8, xs[i]);
    const float wv = et < 64 ? p.w[row * 64 + et] : 0.f;
    float cs4[4], sn4[4];
    const bool rot = c * 8 >= r0;
    if (rot) {
#pragma unroll
      for (int k = 0; k < 4; ++k) rope_cs(t, p.rope, (c * 8 - r0) / 2 + k, cs4[k], sn4[k]);
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
      float hi[8], lo[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        hi[k] = __bfloat162float(__float2bfloat16_rn(x[k]));
        lo[k] = x[k] - hi[k];
      }
      const int h = h0 + 8 * i, blk = c >> 3, ch = c & 7;
      store8(reinterpret_cast<__nv_bfloat16*>(qop + blk * kBlockBytes + sw128_offset(h, ch)), hi);
      store8(reinterpret_cast<__nv_bfloat16*>(qop + blk * kBlockBytes + sw128_offset(64 + h, ch)), lo);
    }
    if (et < 64) w_s[et] = wv;
    if (et == 0) CSA_STAMP(43);
    fence_proxy_async_smem();
    mbar_arrive(qready);
    named_barrier(1, 128);                                  // w_s visible to every epilogue thread
    const int64_t e = t / p.ratio;
    if (close_kv)
      close_entry_bf16<512>(p.close.job[0], p.close.N, p.n_cap, p.ratio, p.close.eps, p.close.rope, b, e, et,
                            red, 2);
    if (close_idx) {
      close_entry_bf16<128>(p.close.job[1], p.close.N, p.n_cap, p.ratio, p.close.eps, p.close.rope, b, e, et,
                            red + 4, 2);
      fence_proxy_async_global();                           // the TMA load of the last tile reads it
      mbar_arrive(closed);
    }

    const uint32_t quad = warp & 3;                         // TMEM lanes 32*quad .. 32*quad+31
    float* out = p.scores + row * p.n_cap;
    griddep_wait();
    for (int i = 0; i < ntiles; ++i) {
      const int acc = i & 1;
      if (!mbar_wait_warp(&tfull[acc], (i >> 1) & 1, p.err)) break;    // uniform over the warp
      tc_fence_after();
      const uint32_t ta = tmem + ((quad * 32) << 16) + acc * 128;
      // four partial sums (heads h = j mod 4): four short dependency chains instead of one of 64
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t hv[32], lv[32];
        tmem_ld32(ta + half * 32, hv);
        tmem_ld32(ta + 64 + half * 32, lv);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          s4[j & 3] = fmaf(w_s[half * 32 + j], fmaxf(__uint_as_float(hv[j]) + __uint_as_float(lv[j]), 0.f), s4[j & 3]);
      }
      const float sc = (s4[0] + s4[1]) + (s4[2] + s4[3]);
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      const int64_t e = (tile0 + i) * kTileM + quad * 32 + lane;
      if (e < V) out[e] = sc;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) CSA_STAMP(44);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace

// 2-D bf16 tensor map [rows][cols] with a 64 x box_rows box and the 128-byte swizzle.
cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, int64_t rows, uint32_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool tc_index_available() { return true; }

int tc_sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

cudaError_t tc_index_scores(int B, int S, const int64_t* pos, const void* q_idx, const float* w, const void* cidx,
                            int64_t n_cap, int ratio, const RopeTab& rope, float* scores, void*, int32_t* err,
                            cudaStream_t st, bool pdl, const CompressParams* close, int64_t entry_base) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(index_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  CUtensorMap map;
  cudaError_t e = make_tmap_2d(&map, cidx, (int64_t)B * n_cap, kDI, kTileM);
  if (e != cudaSuccess) return e;
  IndexTcParams p;
  p.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  p.w = w; p.scores = scores; p.pos = pos; p.n_cap = n_cap; p.S = S; p.ratio = ratio; p.rope = rope; p.err = err;
  p.entry_base = entry_base;
  memset(&p.close, 0, sizeof p.close);
  if (close && entry_base != 0) return cudaErrorInvalidValue;
  if (close) {
    if (S != 1 || close->n_jobs != 2 || close->job[0].C != 512 || close->job[1].C != kDI) return cudaErrorInvalidValue;
    p.close = *close;
  }
  const int64_t tiles = (n_cap + kTileM - 1) / kTileM;
  const int64_t rows = (int64_t)B * S;
  int64_t chunks = (2 * (int64_t)tc_sm_count()) / (rows > 0 ? rows : 1);   // two CTAs per SM, one wave
  if (chunks < 1) chunks = 1;
  if (chunks > tiles) chunks = tiles;
  p.chunks = (int)chunks;
  dim3 grid((unsigned)chunks, (unsigned)S, (unsigned)B);
  return launch_kernel(pdl, index_tc_kernel, grid, dim3(kThreads), kSmemBytes, st, map, p);
}

}  // namespace csa
