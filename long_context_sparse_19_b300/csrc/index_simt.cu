// Indexer scores on CUDA cores (the float32-storage path, and any shape without a tcgen05 kernel).
//
// [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", section "少读 KV 之前，Indexer 仍要给历史打分":
// H_idx heads of 128 dims score the one shared compressed index cache; the head weights are signed
// and are not a softmax; the heads are summed before selection:
//     s_i = sum_h w_h * max(0, rope(q_h, t) . cidx_i),   i < (t+1)/m.
// One CTA scores 128 entries for one query; one thread per entry keeps all head dot products in
// registers while it streams its cache row in 32-dim slices; the rotated query sits in shared memory.
#include "kernels.h"

namespace csa {
namespace {

constexpr int kDI = 128;
constexpr int kMaxHI = 64;
constexpr int kTile = 128;

template <typename T>
__global__ void __launch_bounds__(kTile) index_simt_kernel(const IndexParams p) {
  __shared__ float qs[kMaxHI][kDI];
  __shared__ float ws[kMaxHI];
  griddep_launch();
  griddep_wait();
  const int b = blockIdx.z, s = blockIdx.y;
  const int64_t t = p.pos ? p.pos[(int64_t)b * p.S + s] : s;
  const int64_t V = visible_local(t, p.ratio, p.entry_base, p.n_cap);
  const int64_t i0 = (int64_t)blockIdx.x * kTile;
  if (i0 >= V) return;

  // rotated query (float32) and weights; heads >= H_idx are zero
  const T* q = reinterpret_cast<const T*>(p.q_idx) + ((int64_t)b * p.S + s) * p.H_idx * kDI;
  for (int e = threadIdx.x; e < kMaxHI * kDI / 2; e += kTile) {
    const int h = e / (kDI / 2), pr = e % (kDI / 2);
    float a = 0.f, c2 = 0.f;
    if (h < p.H_idx) {
      a = to_f32(q[h * kDI + 2 * pr]);
      c2 = to_f32(q[h * kDI + 2 * pr + 1]);
      const int r0 = kDI - p.rope.d_rope;
      if (2 * pr >= r0) {
        float c, sn;
        rope_cs(t, p.rope, (2 * pr - r0) / 2, c, sn);
        const float x = a * c - c2 * sn, y = a * sn + c2 * c;
        a = x; c2 = y;
      }
    }
    qs[h][2 * pr] = a;
    qs[h][2 * pr + 1] = c2;
  }
  if (threadIdx.x < kMaxHI)
    ws[threadIdx.x] = threadIdx.x < p.H_idx ? p.w[((int64_t)b * p.S + s) * p.H_idx + threadIdx.x] : 0.f;
  __syncthreads();

  const int64_t i = i0 + threadIdx.x;
  if (i >= V) return;
  const T* row = reinterpret_cast<const T*>(p.cidx) + ((int64_t)b * p.n_cap + i) * kDI;
  float acc[kMaxHI];
#pragma unroll
  for (int h = 0; h < kMaxHI; ++h) acc[h] = 0.f;
  for (int dc = 0; dc < kDI; dc += 32) {
    float r[32];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float v[8];
      load8(row + dc + 8 * u, v);
#pragma unroll
      for (int k = 0; k < 8; ++k) r[8 * u + k] = v[k];
    }
#pragma unroll
    for (int h = 0; h < kMaxHI; ++h) {
      float a = acc[h];
#pragma unroll
      for (int j = 0; j < 32; ++j) a = fmaf(qs[h][dc + j], r[j], a);
      acc[h] = a;
    }
  }
  float sc = 0.f;
#pragma unroll
  for (int h = 0; h < kMaxHI; ++h) sc = fmaf(ws[h], fmaxf(acc[h], 0.f), sc);
  p.scores[((int64_t)b * p.S + s) * p.n_cap + i] = sc;
}

}  // namespace

cudaError_t launch_index_simt(bool bf16, int B, const IndexParams& p, cudaStream_t st, bool pdl) {
  const int64_t nx = (p.n_cap + kTile - 1) / kTile;
  if (nx == 0 || B == 0 || p.S == 0) return cudaSuccess;
  dim3 grid((unsigned)nx, (unsigned)p.S, (unsigned)B);
  if (bf16) return launch_kernel(pdl, index_simt_kernel<__nv_bfloat16>, grid, dim3(kTile), 0, st, p);
  return launch_kernel(pdl, index_simt_kernel<float>, grid, dim3(kTile), 0, st, p);
}

}  // namespace csa
