// Sparse joint attention with sink on CUDA cores (the float32-storage path, and any shape without a
// tcgen05 kernel), plus the split merge with sink and inverse RoPE (K5).
//
// [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", section "局部和压缩记忆，共用一次归一化": the local
// raw entries and the selected compressed entries form ONE candidate set under one softmax; each
// head also has a learned sink that enlarges the denominator and owns no value output. Section
// "输出投影也分组，并且降低中间维度": o = inverse_RoPE(o). HCA ([ATLAS] "LLM Atlas — DeepSeek", section
// 19) keeps every visible compressed entry instead of a top-k subset.
//
// Candidates of the query at t, in order: raw tokens lo..t (lo = max(0, t-W+1)), each raw row
// rotated at its own position; then compressed slots (CSA: topk slots, -1 = empty; HCA: entries
// 0..visible-1). K = V = the candidate row. A CTA handles one query, one split of candidates and
// a group of 16 heads: warp w owns head 16g + w, a lane owns dims lane + 32u, and each warp keeps
// an online softmax. One split writes the final output; several splits write partial
// (max, sum, o) that the merge kernel combines with the sink.
#include "kernels.h"

namespace csa {
namespace {

constexpr int kD = 512;
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 16;           // candidates staged in shared memory at a time
constexpr int kHG = kWarps;          // heads per CTA (one per warp)
constexpr int kDPL = kD / 32;        // dims per lane

struct Cand {
  const void* rowp;   // null = empty slot
  int64_t rope_pos;   // raw rows: rotate at this position; -1: already rotated
};

template <typename T>
__device__ __forceinline__ Cand candidate(const AttnParams& p, int b, int64_t row, int64_t t,
                                          int64_t V, int64_t lo, int64_t n_win, int64_t c) {
  Cand r{nullptr, -1};
  if (c < n_win) {
    const int64_t j = lo + c;
    r.rowp = reinterpret_cast<const T*>(p.kv) + ((int64_t)b * p.N + j) * kD;
    r.rope_pos = j;
  } else {
    const int64_t slot = c - n_win;
    int64_t idx = p.topk ? (int64_t)p.topk[row * p.k + slot] : slot;
    if (idx >= 0) {
      if (idx >= V) { set_error(p.err, DEVERR_BAD_INDEX); return r; }
      r.rowp = reinterpret_cast<const T*>(p.ckv) + ((int64_t)b * p.n_cap + idx) * kD;
    }
  }
  return r;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) attn_simt_kernel(const AttnParams p) {
  __shared__ __align__(16) float qs[kHG * kD];        // rotated query of this head group
  __shared__ __align__(16) float rows[kChunk * kD];   // staged candidate rows
  __shared__ int valid[kChunk];
  __shared__ float th_hi[32], th_lo[32];
  griddep_launch();
  griddep_wait();
  if (threadIdx.x < 32) { th_hi[threadIdx.x] = p.rope.th_hi[threadIdx.x]; th_lo[threadIdx.x] = p.rope.th_lo[threadIdx.x]; }
  __syncthreads();

  const int b = blockIdx.z, s = blockIdx.y;
  const int n_hg = (p.H + kHG - 1) / kHG;
  const int split = blockIdx.x / n_hg, hg = blockIdx.x % n_hg;
  const int h0 = hg * kHG;
  const int64_t row = (int64_t)b * p.S + s;
  const int64_t t = p.pos ? p.pos[row] : s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (t < 0 || t >= p.N) {                   // the raw window would leave the cache
    if (tid == 0) set_error(p.err, DEVERR_BAD_POS);
    return;
  }
  const int64_t V = visible_local(t, p.ratio, p.entry_base, p.n_cap);
  const int64_t lo = t - p.window + 1 > 0 ? t - p.window + 1 : 0;
  const int64_t n_win = p.no_window ? 0 : t - lo + 1;
  const int64_t n_comp = p.topk ? p.k : V;
  const int64_t C = n_win + n_comp;
  const int64_t c_begin = (int64_t)split * p.split_len;
  const int64_t c_end = min(C, c_begin + p.split_len);
  const int r0 = kD - p.rope.d_rope;

  // rotated query of heads h0 .. h0 + 15 (missing heads are zero)
  const T* q = reinterpret_cast<const T*>(p.q) + row * p.H * kD;
  for (int e = tid; e < kHG * kD / 2; e += kThreads) {
    const int h = e / (kD / 2), pr = e % (kD / 2);
    float a = 0.f, c2 = 0.f;
    if (h0 + h < p.H) { a = to_f32(q[(h0 + h) * kD + 2 * pr]); c2 = to_f32(q[(h0 + h) * kD + 2 * pr + 1]); }
    if (2 * pr >= r0) {
      float c, sn;
      rope_cs(t, th_hi[(2 * pr - r0) / 2], th_lo[(2 * pr - r0) / 2], c, sn);
      const float x = a * c - c2 * sn, y = a * sn + c2 * c;
      a = x; c2 = y;
    }
    qs[h * kD + 2 * pr] = a;
    qs[h * kD + 2 * pr + 1] = c2;
  }

  const int h = h0 + warp;                 // this warp's head (h >= H: idle warp)
  float m_ = -INFINITY, l_ = 0.f, o_[kDPL], qv[kDPL];
#pragma unroll
  for (int u = 0; u < kDPL; ++u) o_[u] = 0.f;

  for (int64_t cb = c_begin; cb < c_end; cb += kChunk) {
    __syncthreads();                          // previous chunk fully consumed (and qs written)
    {
      const int cc = tid / 32;                // 16 candidates x 32 lanes x 16 dims
      const int d0 = (tid % 32) * 16;
      const int64_t c = cb + cc;
      Cand cd{nullptr, -1};
      if (c < c_end) cd = candidate<T>(p, b, row, t, V, lo, n_win, c);
      float v[16];
      if (cd.rowp) {
        float a8[8], b8[8];
        load8(reinterpret_cast<const T*>(cd.rowp) + d0, a8);
        load8(reinterpret_cast<const T*>(cd.rowp) + d0 + 8, b8);
#pragma unroll
        for (int k = 0; k < 8; ++k) { v[k] = a8[k]; v[8 + k] = b8[k]; }
        if (cd.rope_pos >= 0 && d0 >= r0) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float c, sn;
            rope_cs(cd.rope_pos, th_hi[(d0 - r0) / 2 + k], th_lo[(d0 - r0) / 2 + k], c, sn);
            const float x = v[2 * k], y = v[2 * k + 1];
            v[2 * k] = x * c - y * sn;
            v[2 * k + 1] = x * sn + y * c;
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = 0.f;
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) rows[cc * kD + d0 + k] = v[k];
      if ((tid % 32) == 0) valid[cc] = cd.rowp != nullptr;
    }
    __syncthreads();
    if (h < p.H) {
      if (cb == c_begin) {                    // the rotated query row stays in registers
#pragma unroll
        for (int u = 0; u < kDPL; ++u) qv[u] = qs[warp * kD + lane + 32 * u];
      }
      float my_lg = -INFINITY, cm = -INFINITY;     // lane c < 16 keeps candidate c's logit
#pragma unroll 2
      for (int cc = 0; cc < kChunk; ++cc) {
        float part = 0.f;
#pragma unroll
        for (int u = 0; u < kDPL; ++u) part = fmaf(qv[u], rows[cc * kD + lane + 32 * u], part);
        part = warp_sum(part) * p.scale;
        const float lgv = valid[cc] ? part : -INFINITY;
        if (lane == cc) my_lg = lgv;
        cm = fmaxf(cm, lgv);
      }
      if (cm != -INFINITY) {
        const float nm = fmaxf(m_, cm);
        const float so = (m_ == -INFINITY) ? 0.f : expf(m_ - nm);
        const float pl = expf(my_lg - nm);           // exp(-inf) = 0 for empty slots / lanes >= 16
        l_ = l_ * so + warp_sum(pl);
#pragma unroll
        for (int u = 0; u < kDPL; ++u) o_[u] *= so;
#pragma unroll 4
        for (int cc = 0; cc < kChunk; ++cc) {
          const float pw = __shfl_sync(0xffffffffu, pl, cc);
#pragma unroll
          for (int u = 0; u < kDPL; ++u) o_[u] = fmaf(pw, rows[cc * kD + lane + 32 * u], o_[u]);
        }
        m_ = nm;
      }
    }
  }

  if (h < p.H) {
    if (p.n_split > 1 || p.partial) {
      const int64_t pi = (row * p.n_split + split) * p.H + h;
#pragma unroll
      for (int u = 0; u < kDPL; ++u) p.part_o[pi * kD + lane + 32 * u] = o_[u];
      if (lane == 0) { p.part_ml[2 * pi] = m_; p.part_ml[2 * pi + 1] = l_; }
      return;
    }
    const float sk = p.sink[h];
    const float M = fmaxf(m_, sk);
    const float a = (m_ == -INFINITY) ? 0.f : expf(m_ - M);
    const float L = l_ * a + expf(sk - M);
    const float f = a / L;
    T* op = reinterpret_cast<T*>(p.out) + (row * p.H + h) * kD;
#pragma unroll
    for (int u = 0; u < kDPL; ++u) {
      const int dim = lane + 32 * u;
      float x = o_[u] * f;
      if (dim >= r0) {                        // inverse RoPE: pair partner is the neighbouring lane
        const float y = __shfl_xor_sync(0xffffffffu, x, 1);
        float c, sn;
        rope_cs(t, th_hi[(dim - r0) / 2], th_lo[(dim - r0) / 2], c, sn);
        x = (lane & 1) ? (y * -sn + x * c) : (x * c + y * sn);
      }
      from_f32(op[dim], x);
    }
  }
}

// Merge of split partials: M = max(m_i, sink), L = sum_i l_i e^(m_i - M) + e^(sink - M),
// o = sum_i e^(m_i - M) o_i / L, then the inverse RoPE at t. One CTA per (query, 8 heads): warp w
// owns head 8 blockIdx.x + w, lane l owns dims 16 l .. 16 l + 15. The split statistics (lane i
// holds split i) and the partial outputs of up to kMergeBatch splits are loaded in one round, so
// the kernel pays the L2 latency once per batch instead of once per dependent step.
constexpr int kMergeHeads = 8;
constexpr int kMergeBatch = 4;

template <typename T>
__global__ void __launch_bounds__(32 * kMergeHeads) attn_merge_kernel(const AttnParams p) {
  if (threadIdx.x == 0) CSA_STAMP(50);
  griddep_launch();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * kMergeHeads + warp;
  const int s = blockIdx.y, b = blockIdx.z;
  if (h >= p.H) return;
  const int64_t row = (int64_t)b * p.S + s;
  const int64_t t = p.pos ? p.pos[row] : s;
  const float sk = p.sink[h];
  const float* ml = p.part_ml + (row * p.n_split * p.H + h) * 2;     // split i at ml[2 * i * H]
  const int64_t mstride = 2 * (int64_t)p.H;
  const int d0 = lane * 16;
  const float* po = p.part_o + (row * p.n_split * p.H + h) * kD + d0;
  const int64_t ostride = (int64_t)p.H * kD;
  // the first batch of partial outputs is requested together with the split statistics
  float4 v[kMergeBatch][4];
  auto load_batch = [&](int first) {
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      if (first + u < p.n_split) {
        const float4* src = reinterpret_cast<const float4*>(po + (int64_t)(first + u) * ostride);
#pragma unroll
        for (int q = 0; q < 4; ++q) v[u][q] = src[q];
      }
    }
  };
  load_batch(0);
  float M = sk;
  for (int i = lane; i < p.n_split; i += 32) M = fmaxf(M, ml[i * mstride]);
  M = warp_max(M);
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float L = 0.f;
  for (int i0 = 0; i0 < p.n_split; i0 += 32) {
    const int i = i0 + lane;
    float mi = -INFINITY, li = 0.f;
    if (i < p.n_split) { mi = ml[i * mstride]; li = ml[i * mstride + 1]; }
    const float wgt = mi == -INFINITY ? 0.f : expf(mi - M);
    L = fmaf(li, wgt, L);
    const int cnt = min(32, p.n_split - i0);
    for (int u0 = 0; u0 < cnt; u0 += kMergeBatch) {
      if (i0 + u0 > 0) load_batch(i0 + u0);
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const float a = __shfl_sync(0xffffffffu, wgt, (u0 + u) & 31);
        if (u0 + u < cnt && a != 0.f) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc[4 * q + 0] = fmaf(a, v[u][q].x, acc[4 * q + 0]);
            acc[4 * q + 1] = fmaf(a, v[u][q].y, acc[4 * q + 1]);
            acc[4 * q + 2] = fmaf(a, v[u][q].z, acc[4 * q + 2]);
            acc[4 * q + 3] = fmaf(a, v[u][q].w, acc[4 * q + 3]);
          }
        }
      }
    }
  }
  L = warp_sum(L) + expf(sk - M);
  const float inv = 1.f / L;
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] *= inv;
  const int r0 = kD - p.rope.d_rope;
  if (d0 >= r0) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float c, sn;
      rope_cs(t, p.rope, (d0 - r0) / 2 + q, c, sn);
      const float x = acc[2 * q], y = acc[2 * q + 1];
      acc[2 * q] = x * c + y * sn;
      acc[2 * q + 1] = -x * sn + y * c;
    }
  }
  T* op = reinterpret_cast<T*>(p.out) + (row * p.H + h) * kD + d0;
  float a8[8], b8[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) { a8[k] = acc[k]; b8[k] = acc[8 + k]; }
  store8(op, a8);
  store8(op + 8, b8);
  if (threadIdx.x == 0) CSA_STAMP(51);
}

}  // namespace

cudaError_t launch_attn_simt(bool bf16, int B, const AttnParams& p, cudaStream_t st, bool pdl) {
  if (B == 0 || p.S == 0) return cudaSuccess;
  const int n_hg = (p.H + kHG - 1) / kHG;
  dim3 grid((unsigned)(p.n_split * n_hg), (unsigned)p.S, (unsigned)B);
  if (bf16) return launch_kernel(pdl, attn_simt_kernel<__nv_bfloat16>, grid, dim3(kThreads), 0, st, p);
  return launch_kernel(pdl, attn_simt_kernel<float>, grid, dim3(kThreads), 0, st, p);
}

cudaError_t launch_attn_merge(bool bf16, int B, const AttnParams& p, cudaStream_t st, bool pdl) {
  if (B == 0 || p.S == 0 || p.n_split <= 1) return cudaSuccess;
  dim3 grid((unsigned)((p.H + kMergeHeads - 1) / kMergeHeads), (unsigned)p.S, (unsigned)B);
  if (bf16) return launch_kernel(pdl, attn_merge_kernel<__nv_bfloat16>, grid, dim3(32 * kMergeHeads), 0, st, p);
  return launch_kernel(pdl, attn_merge_kernel<float>, grid, dim3(32 * kMergeHeads), 0, st, p);
}

}  // namespace csa
