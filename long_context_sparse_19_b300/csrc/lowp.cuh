// The low-precision compressed cache: FP4 E2M1 latent with one power-of-two scale per 32 dims, and
// an FP8 E4M3 RoPE tail.
//
// [LAB41] "Lab tổng hợp DeepSeek-V4.1-Flash — chạy toàn trình 1A → 6B bằng NumPy", section
// "3 Giải pháp": the KV budget per token is priced with FP4 E2M1 for the latent part of a cache entry
// and FP8 E4M3 for its RoPE tail. E2M1 is applied as its published definition applies it (OCP
// Microscaling, MXFP4): blocks of 32 latent dims share the scale 2^E, stored as the E8M0 byte E + 127,
// with E = floor(log2 max|x|) - 2 clamped to [-127, 127] (-127 for an all-zero block); an element is
// x / 2^E rounded to nearest even and saturated to +-6. The tail is E4M3 (bias 7, largest finite 448),
// rounded to nearest even and saturated, with no scale. Both conversions are the hardware's
// cvt.rn.satfinite instructions on the fp32 value.
//
// Layout of one request's cache of n_cap entries of C dims (L = C - d_rope latent dims), three planes,
// entry-major inside each:
//   plane 0 at 0:                  n_cap x L/2 bytes; byte j of an entry = dims 2j (low nibble), 2j+1
//   plane 1 at n_cap L/2:          n_cap x d_rope bytes, E4M3 codes of the tail dims
//   plane 2 at n_cap (L/2+d_rope): n_cap x sb bytes, byte k < L/32 = E8M0 scale of dims 32k..32k+31
// with sb the next power of two >= L/32 (16 for C = 512, 2 for C = 128); requests follow one another
// at a stride of n_cap (L/2 + d_rope) + round_up(n_cap sb, 16) bytes (304 and 98 bytes per entry).
// Every plane offset is a multiple of 16, so a run of consecutive entries of one plane is one bulk
// copy, and a KV entry's pieces (224, 64 and 16 bytes) are whole 16-byte units.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace csa {

struct LowpLayout {
  int64_t fp8;       // byte offset of plane 1 inside a request
  int64_t scale;     // byte offset of plane 2
  int64_t stride;    // bytes per request
  int L, R, nb, sb;  // latent dims, tail dims, scale blocks, scale bytes per entry
};

__host__ __device__ inline LowpLayout lowp_layout(int C, int64_t n_cap, int d_rope) {
  LowpLayout l;
  l.L = C - d_rope;
  l.R = d_rope;
  l.nb = l.L / 32;
  int sb = 1;
  while (sb < l.nb) sb <<= 1;
  l.sb = sb;
  l.fp8 = n_cap * (l.L / 2);
  l.scale = l.fp8 + n_cap * d_rope;
  l.stride = l.scale + (n_cap * sb + 15) / 16 * 16;
  return l;
}

// E of a block whose max |x| is amax (fp32): the exponent field gives floor(log2 amax) for a normal
// amax; a subnormal or zero amax lands on the clamp.
__device__ __forceinline__ int mx_exponent(float amax) {
  if (!(amax > 0.f)) return -127;
  const int ef = (int)((__float_as_uint(amax) >> 23) & 255u) - 127;
  return max(-127, min(127, ef - 2));
}

// 2^s for s in [-126, 127], built from the exponent field.
__device__ __forceinline__ float exp2_int(int s) { return __uint_as_float((uint32_t)(s + 127) << 23); }

// 2^(byte - 127) of an E8M0 scale byte (byte 0 is the subnormal 2^-127; 255, never written, is NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t byte) {
  return byte == 0 ? __uint_as_float(0x00400000u) : byte == 255 ? __uint_as_float(0x7fc00000u)
                                                                : __uint_as_float(byte << 23);
}

// One byte: E2M1 codes of lo (bits 0..3) and hi (bits 4..7).
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two bytes: E4M3 codes of lo (bits 0..7) and hi (bits 8..15).
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// The two E2M1 codes of byte `b` (low nibble first) as fp32.
__device__ __forceinline__ float2 e2m1x2_to_f2(uint32_t b) {
  uint32_t h;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h) : "r"(b));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// The two E4M3 codes of the 16-bit `v` (low byte first) as fp32.
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t v) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)v));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// 8 latent dims: 4 bytes of E2M1 codes times 2^E -> 8 bf16 (exact).
__device__ __forceinline__ uint4 dequant_fp4x8(uint32_t codes, float scale) {
  uint4 o;
  uint32_t* w = &o.x;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 f = e2m1x2_to_f2(codes >> (8 * j));
    w[j] = pack_bf16(f.x * scale, f.y * scale);
  }
  return o;
}

// 8 tail dims: 8 bytes of E4M3 codes -> 8 bf16 (exact).
__device__ __forceinline__ uint4 dequant_fp8x8(uint32_t c0, uint32_t c1) {
  uint4 o;
  float2 f = e4m3x2_to_f2(c0);
  o.x = pack_bf16(f.x, f.y);
  f = e4m3x2_to_f2(c0 >> 16);
  o.y = pack_bf16(f.x, f.y);
  f = e4m3x2_to_f2(c1);
  o.z = pack_bf16(f.x, f.y);
  f = e4m3x2_to_f2(c1 >> 16);
  o.w = pack_bf16(f.x, f.y);
  return o;
}

// f16x2 (both halves) of 2^(byte - 127): exact for E in [-24, 15] (a subnormal below 2^-14); 0 below,
// which the codes of a block with E < -24 (values under 2^-21) then expand to.
__device__ __forceinline__ uint32_t e8m0_to_h2(uint32_t byte) {
  const int E = (int)byte - 127;
  const uint32_t h = E >= -14 ? (uint32_t)(E + 15) << 10 : E >= -24 ? 1u << (E + 24) : 0u;
  return h | (h << 16);
}

// 8 latent dims: 4 bytes of E2M1 codes times 2^E -> 8 f16 (exact for E in [-23, 13]; the expanded
// products are exact in f16, subnormals included).
__device__ __forceinline__ uint4 expand_fp4x8_f16(uint32_t codes, uint32_t scale2) {
  uint4 o;
  uint32_t* w = &o.x;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t h;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h) : "r"(codes >> (8 * j)));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(w[j]) : "r"(h), "r"(scale2));
  }
  return o;
}

// 8 tail dims: 8 bytes of E4M3 codes -> 8 f16 (exact: every E4M3 value is an f16 value).
__device__ __forceinline__ uint4 expand_fp8x8_f16(uint32_t c0, uint32_t c1) {
  uint4 o;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o.x) : "h"((uint16_t)c0));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o.y) : "h"((uint16_t)(c0 >> 16)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o.z) : "h"((uint16_t)c1));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o.w) : "h"((uint16_t)(c1 >> 16)));
  return o;
}

// Stores this thread's P consecutive dims c0 .. c0+P-1 (P in {1, 2, 4, 8}) of entry e into the
// request's low-precision cache at `base`. The lanes in `mask` call it together; they hold whole
// 32-dim blocks, in lane order (lane i of an aligned group of 32 / P lanes holds dims P i .. P i + P - 1
// of one block).
template <int P>
__device__ __forceinline__ void store_entry_lowp(uint8_t* base, const LowpLayout& lay, int64_t e, int c0,
                                                 const float (&x)[P], unsigned mask = 0xffffffffu) {
  static_assert(P == 1 || P == 2 || P == 4 || P == 8, "1, 2, 4 or 8 dims per thread");
  constexpr int kLanes = 32 / P;                         // lanes of one 32-dim block
  const bool latent = c0 < lay.L;                        // uniform over a block's lanes
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < P; ++k) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
  for (int o = 1; o < kLanes; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(mask, amax, o));
  // the neighbour's value for the pairs that straddle two lanes (P == 1)
  const float xn = __shfl_xor_sync(mask, x[0], 1);
  if (latent) {
    const int E = mx_exponent(amax);
    const float inv = exp2_int(-E);
    uint8_t* d = base + e * (lay.L / 2) + c0 / 2;
    if constexpr (P == 1) {
      if ((c0 & 1) == 0) *d = (uint8_t)cvt_e2m1x2(x[0] * inv, xn * inv);
    } else {
      uint32_t v = 0;
#pragma unroll
      for (int k = 0; k < P / 2; ++k) v |= cvt_e2m1x2(x[2 * k] * inv, x[2 * k + 1] * inv) << (8 * k);
      if constexpr (P == 2) *d = (uint8_t)v;
      else if constexpr (P == 4) *reinterpret_cast<uint16_t*>(d) = (uint16_t)v;
      else *reinterpret_cast<uint32_t*>(d) = v;
    }
    if ((c0 & 31) == 0) {                                // the block's first lane writes the scale
      uint8_t* s = base + lay.scale + e * lay.sb;
      s[c0 / 32] = (uint8_t)(E + 127);
      if (c0 / 32 == lay.nb - 1)
        for (int k = lay.nb; k < lay.sb; ++k) s[k] = 0;  // padding of the scale record
    }
  } else {
    uint8_t* d = base + lay.fp8 + e * (int64_t)lay.R + (c0 - lay.L);
    if constexpr (P == 1) {
      if ((c0 & 1) == 0) *reinterpret_cast<uint16_t*>(d) = (uint16_t)cvt_e4m3x2(x[0], xn);
    } else if constexpr (P == 2) {
      *reinterpret_cast<uint16_t*>(d) = (uint16_t)cvt_e4m3x2(x[0], x[1]);
    } else if constexpr (P == 4) {
      *reinterpret_cast<uint32_t*>(d) = cvt_e4m3x2(x[0], x[1]) | (cvt_e4m3x2(x[2], x[3]) << 16);
    } else {
      uint2 v;
      v.x = cvt_e4m3x2(x[0], x[1]) | (cvt_e4m3x2(x[2], x[3]) << 16);
      v.y = cvt_e4m3x2(x[4], x[5]) | (cvt_e4m3x2(x[6], x[7]) << 16);
      *reinterpret_cast<uint2*>(d) = v;
    }
  }
}

}  // namespace csa
