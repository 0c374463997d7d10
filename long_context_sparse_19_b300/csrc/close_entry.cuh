// The decode compressor's closing entry, computed by one group of threads of a CTA that has other work.
//
// [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", sections "压缩是逐通道的 learned pooling" and
// "一个通道，逐项算出压缩结果": when position t closes a group (t + 1 divisible by m), entry
// e = t / m pools the raw tokens [(e-1)m, (e+1)m) of every channel with its own softmax over
// gate + bias row (a token before position 0 takes weight 0), then RMSNorm over the C channels,
// then RoPE of the last d_rope channels at position e*m. Same arithmetic as the compressor's
// close kernel (one online-softmax state per channel, tokens in order), with the 2m tokens'
// loads issued before any is used. bf16 raw rows; the entry is stored as bf16 or, with kLowp, in the
// low-precision cache format of lowp.cuh.
#pragma once

#include "kernels.h"
#include "lowp.cuh"

namespace csa {

template <int P>
__device__ __forceinline__ void load_row_part(const __nv_bfloat16* p, float (&v)[P]) {
  static_assert(P == 1 || P == 2 || P == 4 || P == 8, "1, 2, 4 or 8 channels per thread");
  if constexpr (P == 1) {
    v[0] = __bfloat162float(p[0]);
  } else if constexpr (P == 2) {
    const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(p));
    v[0] = bf16lo(u); v[1] = bf16hi(u);
  } else if constexpr (P == 4) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
  } else {
    load8(p, v);
  }
}

template <int P>
__device__ __forceinline__ void load_row_part(const float* p, float (&v)[P]) {
  if constexpr (P == 1) {
    v[0] = __ldg(p);
  } else if constexpr (P == 2) {
    const float2 f = __ldg(reinterpret_cast<const float2*>(p));
    v[0] = f.x; v[1] = f.y;
  } else if constexpr (P == 4) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  } else {
    load8(p, v);
  }
}

// Pools entry e of request b of `job` (C channels, bf16 rows) and stores it. Called by all kT
// threads `tid` = 0..kT-1 of one group (whole warps), which synchronise on named barrier `bar_id`;
// `red` is kT / 32 floats of shared memory. Returns after this thread's part of the entry is stored.
template <int C, int kT = 128, bool kLowp = false>
__device__ __forceinline__ void close_entry_bf16(const CompressJob& job, int64_t N, int64_t n_cap, int m,
                                                 float eps, const RopeTab& rope, int64_t b, int64_t e, int tid,
                                                 float* red, int bar_id) {
  constexpr int P = C / kT;                      // channels per thread
  static_assert(C % kT == 0 && (P == 1 || P == 2 || P == 4 || P == 8) && kT % 32 == 0, "channels per thread");
  constexpr int kU = P >= 8 ? 4 : 8;             // tokens whose loads are in flight together
  const int c0 = tid * P;
  const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(job.src) + b * N * C + c0;
  const __nv_bfloat16* gate = static_cast<const __nv_bfloat16*>(job.gate) + b * N * C + c0;
  const float* bias = job.bias + c0;
  float mx[P], sum[P], acc[P];
#pragma unroll
  for (int k = 0; k < P; ++k) { mx[k] = -INFINITY; sum[k] = 0.f; acc[k] = 0.f; }
  const int64_t j0 = (e - 1) * m;                // window position q holds token j0 + q
  for (int q0 = 0; q0 < 2 * m; q0 += kU) {
    float v[kU][P], g[kU][P], bq[kU][P];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int q = q0 + u;
      if (q < 2 * m && j0 + q >= 0) {
        load_row_part<P>(src + (j0 + q) * C, v[u]);
        load_row_part<P>(gate + (j0 + q) * C, g[u]);
        load_row_part<P>(bias + (int64_t)q * C, bq[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int q = q0 + u;
      if (q < 2 * m && j0 + q >= 0) {
#pragma unroll
        for (int k = 0; k < P; ++k) {
          const float l = g[u][k] + bq[u][k];
          if (l > mx[k]) {
            const float sc = expf(mx[k] - l);    // exp(-inf) = 0 on the first token
            sum[k] = sum[k] * sc + 1.f;
            acc[k] = acc[k] * sc + v[u][k];
            mx[k] = l;
          } else {
            const float w = expf(l - mx[k]);
            sum[k] += w;
            acc[k] = fmaf(w, v[u][k], acc[k]);
          }
        }
      }
    }
  }
  float x[P], ss = 0.f;
#pragma unroll
  for (int k = 0; k < P; ++k) { x[k] = acc[k] / sum[k]; ss = fmaf(x[k], x[k], ss); }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  named_barrier(bar_id, kT);
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kT / 32; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)C + eps);
#pragma unroll
  for (int k = 0; k < P; ++k) x[k] *= inv;
  const int r0 = C - rope.d_rope;
  if constexpr (P == 1) {
    const float xp = __shfl_xor_sync(0xffffffffu, x[0], 1);     // the other channel of the pair
    if (c0 >= r0) {
      float cs, sn;
      rope_cs(e * m, rope, (c0 - r0) / 2, cs, sn);
      x[0] = (c0 & 1) ? fmaf(xp, sn, x[0] * cs) : fmaf(-xp, sn, x[0] * cs);
    }
    if constexpr (kLowp) {
      const LowpLayout lay = lowp_layout(C, n_cap, rope.d_rope);
      store_entry_lowp<1>(static_cast<uint8_t*>(job.dst) + b * lay.stride, lay, e, c0, x);
    } else {
      static_cast<__nv_bfloat16*>(job.dst)[(b * n_cap + e) * C + c0] = __float2bfloat16_rn(x[0]);
    }
  } else {
    if (c0 >= r0) {
#pragma unroll
      for (int q = 0; q < P / 2; ++q) {
        float cs, sn;
        rope_cs(e * m, rope, (c0 - r0) / 2 + q, cs, sn);
        const float a = x[2 * q], bb = x[2 * q + 1];
        x[2 * q] = a * cs - bb * sn;
        x[2 * q + 1] = a * sn + bb * cs;
      }
    }
    if constexpr (kLowp) {
      const LowpLayout lay = lowp_layout(C, n_cap, rope.d_rope);
      store_entry_lowp<P>(static_cast<uint8_t*>(job.dst) + b * lay.stride, lay, e, c0, x);
      return;
    }
    __nv_bfloat16* d = static_cast<__nv_bfloat16*>(job.dst) + (b * n_cap + e) * C + c0;
    if constexpr (P == 2) {
      *reinterpret_cast<uint32_t*>(d) = pack_bf16(x[0], x[1]);
    } else if constexpr (P == 4) {
      uint2 u;
      u.x = pack_bf16(x[0], x[1]);
      u.y = pack_bf16(x[2], x[3]);
      *reinterpret_cast<uint2*>(d) = u;
    } else {
      store8(d, x);
    }
  }
}

}  // namespace csa
