// K1: the compressor — overlapped per-channel softmax pooling, RMSNorm, partial RoPE.
//
// [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", sections "压缩是逐通道的 learned pooling"
// (every channel runs its own softmax along the token axis; RMSNorm after pooling; RoPE on the last
// 64 dims) and "一个通道，逐项算出压缩结果" (the first group has no previous group: its rows take
// gate -inf, weight 0). Entry i pools tokens [(i-1)m, (i+1)m) with gate bias row p = j - (i-1)m.
//
// Design: a team of C/8 threads owns one request's run of consecutive entries; each thread owns
// 8 adjacent channels and loads 16-byte vectors, so a team reads each raw row fully coalesced.
// Each raw group g is read ONCE: its tokens update two online-softmax states at the same time,
// one with the second-half bias rows (for entry g) and one with the first-half bias rows (for
// entry g+1). An entry is the merge of the two states, which are exact softmax partials.
// With the low-precision cache (kLowp) the raw rows are bf16 and each finished entry is stored as
// FP4 E2M1 latent blocks + an FP8 E4M3 tail (lowp.cuh).
#include "kernels.h"
#include "lowp.cuh"

namespace csa {
namespace {

constexpr int kThreads = 256;
constexpr int kEntriesPerBlock = 64;   // large builds; small ones use 16 so that the grid fills the GPU

struct Stat8 {
  float mx[8], sum[8], acc[8];
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int k = 0; k < 8; ++k) { mx[k] = -INFINITY; sum[k] = 0.f; acc[k] = 0.f; }
  }
  __device__ __forceinline__ void add(int k, float l, float v) {
    if (l > mx[k]) {
      const float sc = expf(mx[k] - l);       // exp(-inf) = 0 on the first token
      sum[k] = sum[k] * sc + 1.f;
      acc[k] = acc[k] * sc + v;
      mx[k] = l;
    } else {
      const float e = expf(l - mx[k]);
      sum[k] += e;
      acc[k] = fmaf(e, v, acc[k]);
    }
  }
};

// Reads group g (tokens g*m .. g*m+m-1) once; updates `lo` with bias rows [0, m) and, when
// `want_hi`, `hi` with bias rows [m, 2m).
template <typename T, int C>
__device__ __forceinline__ void scan_group(const T* src, const T* gate, const float* bias, int64_t g,
                                           int m, int c0, Stat8& lo, Stat8& hi, bool want_hi) {
  for (int r = 0; r < m; ++r) {
    const int64_t j = g * m + r;
    float v[8], gt[8], bl[8], bh[8];
    load8(src + j * C + c0, v);
    load8(gate + j * C + c0, gt);
    load8(bias + (int64_t)r * C + c0, bl);
    if (want_hi) load8(bias + (int64_t)(m + r) * C + c0, bh);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      lo.add(k, gt[k] + bl[k], v[k]);
      if (want_hi) hi.add(k, gt[k] + bh[k], v[k]);
    }
  }
}

template <typename T, int C, bool kLowp>
__device__ void compress_run(const CompressParams& p, const CompressJob& job, int b, int64_t e_begin,
                             int64_t e_end, int team, int tt, float* red) {
  constexpr int TPE = C / 8;               // threads per entry team
  const int m = p.ratio;
  const int c0 = tt * 8;
  const T* src = reinterpret_cast<const T*>(job.src) + (int64_t)b * p.N * C;
  const T* gate = reinterpret_cast<const T*>(job.gate) + (int64_t)b * p.N * C;
  T* dst = reinterpret_cast<T*>(job.dst) + (int64_t)b * p.n_cap * C;
  const int lane = threadIdx.x & 31;
  const LowpLayout lay = lowp_layout(C, p.n_cap, p.rope.d_rope);
  uint8_t* lbase = static_cast<uint8_t*>(job.dst) + (int64_t)b * lay.stride;
  // lanes of this team inside the warp (teams narrower than a warp share it)
  const unsigned tmask = TPE >= 32 ? 0xffffffffu : ((1u << (TPE & 31)) - 1u) << (lane & ~(TPE - 1));

  Stat8 prev, lo, hi;
  prev.clear();
  if (e_begin >= 1) scan_group<T, C>(src, gate, job.bias, e_begin - 1, m, c0, prev, hi, false);

  for (int64_t e = e_begin; e < e_end; ++e) {
    lo.clear();
    hi.clear();
    scan_group<T, C>(src, gate, job.bias, e, m, c0, lo, hi, true);
    float x[8];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float M = fmaxf(prev.mx[k], hi.mx[k]);
      const float a = (prev.mx[k] == -INFINITY) ? 0.f : expf(prev.mx[k] - M);
      const float bb = expf(hi.mx[k] - M);
      x[k] = (prev.acc[k] * a + hi.acc[k] * bb) / (prev.sum[k] * a + hi.sum[k] * bb);
      ss = fmaf(x[k], x[k], ss);
      prev.mx[k] = lo.mx[k]; prev.sum[k] = lo.sum[k]; prev.acc[k] = lo.acc[k];
    }
    // RMSNorm over the C channels of the entry: reduce within the team.
    if constexpr (TPE >= 32) {
      ss = warp_sum(ss);
      if constexpr (TPE > 32) {
        constexpr int W = TPE / 32;
        const int wit = tt >> 5;
        if (lane == 0) red[team * W + wit] = ss;
        named_barrier(1 + team, TPE);
        ss = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) ss += red[team * W + w];
        named_barrier(1 + team, TPE);
      }
    } else {
      const unsigned mask = ((1u << (TPE & 31)) - 1u) << (lane & ~(TPE - 1));
#pragma unroll
      for (int o = TPE / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(mask, ss, o);
    }
    const float inv = 1.0f / sqrtf(ss / (float)C + p.eps);
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] *= inv;
    // RoPE of the last d_rope channels at position e*m (interleaved pairs).
    const int r0 = C - p.rope.d_rope;
    if (c0 >= r0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float c, s;
        rope_cs(e * m, p.rope, (c0 - r0) / 2 + q, c, s);
        const float a = x[2 * q], bq = x[2 * q + 1];
        x[2 * q] = a * c - bq * s;
        x[2 * q + 1] = a * s + bq * c;
      }
    }
    if constexpr (kLowp) store_entry_lowp<8>(lbase, lay, e, c0, x, tmask);
    else store8(dst + e * C + c0, x);
  }
}

template <typename T, int C, bool kLowp>
__device__ void compress_block(const CompressParams& p, const CompressJob& job, float* red) {
  constexpr int TPE = C / 8;
  constexpr int TEAMS = kThreads / TPE;
  const int team = threadIdx.x / TPE;
  const int tt = threadIdx.x % TPE;
  const int b = blockIdx.y;
  const int EPT = p.epb / TEAMS;                  // entries per team (epb is a multiple of 16)
  const int64_t e_begin = p.first_entry + (int64_t)blockIdx.x * p.epb + (int64_t)team * EPT;
  const int64_t e_end = min(e_begin + EPT, p.first_entry + p.n_entries);
  if (e_begin >= e_end) return;
  compress_run<T, C, kLowp>(p, job, b, e_begin, e_end, team, tt, red);
}

template <typename T, bool kLowp>
__global__ void __launch_bounds__(kThreads) compress_kernel(const CompressParams p) {
  __shared__ float red[16];
  griddep_launch();
  griddep_wait();
  const CompressJob& job = p.job[blockIdx.z];
  if (job.C == 512) compress_block<T, 512, kLowp>(p, job, red);
  else compress_block<T, 128, kLowp>(p, job, red);
}

// ------------------------------------------------------------------ decode: the closing entry only
// One CTA per (request, cache): when t closes a group, entry e = t/m is pooled from its 2m tokens.
// The tokens are spread over G groups of threads (each thread: 8 channels of every G-th token,
// one online-softmax state), so the loads of all tokens are in flight at once; the G partial
// states per channel are then merged in shared memory, one thread per channel.
constexpr int kCloseThreads = 512;

template <typename T, int C, bool kLowp>
__device__ void compress_close(const CompressParams& p, const CompressJob& job, float* sm) {
  constexpr int CH = C / 8;                  // channel chunks
  constexpr int G = kCloseThreads / CH;      // token groups
  const int b = blockIdx.x;
  const int64_t t = p.pos[b];
  if (t < 0 || t >= p.N) { if (threadIdx.x == 0) set_error(p.err, DEVERR_BAD_POS); return; }
  if ((t + 1) % p.ratio != 0) return;
  const int64_t e = t / p.ratio;
  if (e >= p.n_cap) { if (threadIdx.x == 0) set_error(p.err, DEVERR_BAD_POS); return; }
  const int m = p.ratio;
  const int chunk = threadIdx.x % CH, g = threadIdx.x / CH;
  const int c0 = chunk * 8;
  const T* src = reinterpret_cast<const T*>(job.src) + (int64_t)b * p.N * C;
  const T* gate = reinterpret_cast<const T*>(job.gate) + (int64_t)b * p.N * C;
  Stat8 st;
  st.clear();
  const int64_t j0 = (e - 1) * m;                  // window position q holds token j0 + q
  for (int pp = g; pp < 2 * m; pp += 4 * G) {
    float v[4][8], gt[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {                  // issue up to four tokens' loads first
      const int q = pp + u * G;
      if (q < 2 * m && j0 + q >= 0) {
        load8(src + (j0 + q) * C + c0, v[u]);
        load8(gate + (j0 + q) * C + c0, gt[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = pp + u * G;
      if (q < 2 * m && j0 + q >= 0) {
        float bq[8];
        load8(job.bias + (int64_t)q * C + c0, bq);
#pragma unroll
        for (int k = 0; k < 8; ++k) st.add(k, gt[u][k] + bq[k], v[u][k]);
      }
    }
  }
  // partial states -> shared memory [3][G][C]
  float* smx = sm;
  float* ssum = sm + G * C;
  float* sacc = sm + 2 * G * C;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    smx[g * C + c0 + k] = st.mx[k];
    ssum[g * C + c0 + k] = st.sum[k];
    sacc[g * C + c0 + k] = st.acc[k];
  }
  __syncthreads();
  float* xs = sm + 3 * G * C;                      // [C] pooled values
  float* red = xs + C;                             // [32]
  float ss = 0.f;
  if (threadIdx.x < C) {
    const int c = threadIdx.x;
    float M = -INFINITY;
    for (int q = 0; q < G; ++q) M = fmaxf(M, smx[q * C + c]);
    float num = 0.f, den = 0.f;
    for (int q = 0; q < G; ++q) {
      const float mq = smx[q * C + c];
      if (mq == -INFINITY) continue;
      const float a = expf(mq - M);
      num = fmaf(sacc[q * C + c], a, num);
      den = fmaf(ssum[q * C + c], a, den);
    }
    const float x = num / den;
    xs[c] = x;
    ss = x * x;
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < CH) {
    float tot = 0.f;
    for (int w = 0; w < kCloseThreads / 32; ++w) tot += red[w];
    const float inv = 1.0f / sqrtf(tot / (float)C + p.eps);
    float x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = xs[c0 + k] * inv;
    const int r0 = C - p.rope.d_rope;
    if (c0 >= r0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float cs, sn;
        rope_cs(e * m, p.rope, (c0 - r0) / 2 + q, cs, sn);
        const float a = x[2 * q], bq = x[2 * q + 1];
        x[2 * q] = a * cs - bq * sn;
        x[2 * q + 1] = a * sn + bq * cs;
      }
    }
    if constexpr (kLowp) {
      const LowpLayout lay = lowp_layout(C, p.n_cap, p.rope.d_rope);
      store_entry_lowp<8>(static_cast<uint8_t*>(job.dst) + (int64_t)b * lay.stride, lay, e, c0, x,
                          CH >= 32 ? 0xffffffffu : (1u << CH) - 1u);
    } else {
      T* dst = reinterpret_cast<T*>(job.dst) + ((int64_t)b * p.n_cap + e) * C;
      store8(dst + c0, x);
    }
  }
}

// A long window (2m >= 128 tokens, HCA's m = 128: 256 tokens x 1 KB of kv and of gate per request)
// is split over a cluster of P CTAs: CTA r folds the tokens [r 2m/P, (r+1) 2m/P) into per-channel
// online-softmax states, CTA 0 merges the P states through distributed shared memory and stores the
// entry. (One CTA per request left the step waiting ~37 us for 16 CTAs' 512 KB each.)
constexpr int kCloseClusterMax = 8;

template <typename T, int C, bool kLowp>
__device__ void compress_close_split(const CompressParams& p, const CompressJob& job, float* sm) {
  constexpr int CH = C / 8;                  // channel chunks
  constexpr int G = kCloseThreads / CH;      // token groups
  const int b = blockIdx.y;
  const uint32_t rank = cluster_rank(), P = gridDim.x;
  const int64_t t = p.pos[b];
  // the early exits are uniform over the cluster (every CTA reads the same t): no CTA waits at a
  // cluster barrier for one that left
  if (t < 0 || t >= p.N) { if (threadIdx.x == 0 && rank == 0) set_error(p.err, DEVERR_BAD_POS); return; }
  if ((t + 1) % p.ratio != 0) return;
  const int64_t e = t / p.ratio;
  if (e >= p.n_cap) { if (threadIdx.x == 0 && rank == 0) set_error(p.err, DEVERR_BAD_POS); return; }
  const int m = p.ratio;
  const int chunk = threadIdx.x % CH, g = threadIdx.x / CH;
  const int c0 = chunk * 8;
  const T* src = reinterpret_cast<const T*>(job.src) + (int64_t)b * p.N * C;
  const T* gate = reinterpret_cast<const T*>(job.gate) + (int64_t)b * p.N * C;
  const int q_lo = (int)(rank * 2 * m / P), q_hi = (int)((rank + 1) * 2 * m / P);
  Stat8 st;
  st.clear();
  const int64_t j0 = (e - 1) * m;                  // window position q holds token j0 + q
  for (int pp = q_lo + g; pp < q_hi; pp += 4 * G) {
    float v[4][8], gt[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {                  // issue up to four tokens' loads first
      const int q = pp + u * G;
      if (q < q_hi && j0 + q >= 0) {
        load8(src + (j0 + q) * C + c0, v[u]);
        load8(gate + (j0 + q) * C + c0, gt[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = pp + u * G;
      if (q < q_hi && j0 + q >= 0) {
        float bq[8];
        load8(job.bias + (int64_t)q * C + c0, bq);
#pragma unroll
        for (int k = 0; k < 8; ++k) st.add(k, gt[u][k] + bq[k], v[u][k]);
      }
    }
  }
  float* smx = sm;
  float* ssum = sm + G * C;
  float* sacc = sm + 2 * G * C;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    smx[g * C + c0 + k] = st.mx[k];
    ssum[g * C + c0 + k] = st.sum[k];
    sacc[g * C + c0 + k] = st.acc[k];
  }
  __syncthreads();
  float* part = sm + 3 * G * C;                    // [3][C] this CTA's merged state (read remotely)
  if (threadIdx.x < C) {
    const int c = threadIdx.x;
    float M = -INFINITY;
    for (int q = 0; q < G; ++q) M = fmaxf(M, smx[q * C + c]);
    float num = 0.f, den = 0.f;
    for (int q = 0; q < G; ++q) {
      const float mq = smx[q * C + c];
      if (mq == -INFINITY) continue;
      const float a = expf(mq - M);
      num = fmaf(sacc[q * C + c], a, num);
      den = fmaf(ssum[q * C + c], a, den);
    }
    part[c] = M;
    part[C + c] = den;
    part[2 * C + c] = num;
  }
  cluster_sync();                                  // every CTA's state is in its shared memory
  if (rank == 0) {
    float* xs = part + 3 * C;                      // [C] pooled values
    float* red = xs + C;                           // [32]
    float ss = 0.f;
    if (threadIdx.x < C) {
      const int c = threadIdx.x;
      float mr[kCloseClusterMax], dr[kCloseClusterMax], nr[kCloseClusterMax];
#pragma unroll
      for (int r = 0; r < kCloseClusterMax; ++r) {
        if (r < (int)P) {
          mr[r] = dsmem_ldf(dsmem_addr(&part[c], r));
          dr[r] = dsmem_ldf(dsmem_addr(&part[C + c], r));
          nr[r] = dsmem_ldf(dsmem_addr(&part[2 * C + c], r));
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < kCloseClusterMax; ++r)
        if (r < (int)P) M = fmaxf(M, mr[r]);
      float num = 0.f, den = 0.f;
#pragma unroll
      for (int r = 0; r < kCloseClusterMax; ++r) {
        if (r < (int)P && mr[r] != -INFINITY) {
          const float a = expf(mr[r] - M);
          num = fmaf(nr[r], a, num);
          den = fmaf(dr[r], a, den);
        }
      }
      const float x = num / den;
      xs[c] = x;
      ss = x * x;
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < CH) {
      float tot = 0.f;
      for (int w = 0; w < kCloseThreads / 32; ++w) tot += red[w];
      const float inv = 1.0f / sqrtf(tot / (float)C + p.eps);
      float x[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = xs[c0 + k] * inv;
      const int r0 = C - p.rope.d_rope;
      if (c0 >= r0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float cs, sn;
          rope_cs(e * m, p.rope, (c0 - r0) / 2 + q, cs, sn);
          const float a = x[2 * q], bq = x[2 * q + 1];
          x[2 * q] = a * cs - bq * sn;
          x[2 * q + 1] = a * sn + bq * cs;
        }
      }
      if constexpr (kLowp) {
        const LowpLayout lay = lowp_layout(C, p.n_cap, p.rope.d_rope);
        store_entry_lowp<8>(static_cast<uint8_t*>(job.dst) + (int64_t)b * lay.stride, lay, e, c0, x,
                            CH >= 32 ? 0xffffffffu : (1u << CH) - 1u);
      } else {
        T* dst = reinterpret_cast<T*>(job.dst) + ((int64_t)b * p.n_cap + e) * C;
        store8(dst + c0, x);
      }
    }
  }
  cluster_sync();                                  // CTA 0 has read every CTA's state
}

template <typename T, bool kLowp>
__global__ void __launch_bounds__(kCloseThreads) compress_close_split_kernel(const CompressParams p) {
  extern __shared__ float sm[];
  if (threadIdx.x == 0) CSA_STAMP(40);
  griddep_launch();
  griddep_wait();
  const CompressJob& job = p.job[blockIdx.z];
  if (job.C == 512) compress_close_split<T, 512, kLowp>(p, job, sm);
  else compress_close_split<T, 128, kLowp>(p, job, sm);
  if (threadIdx.x == 0) CSA_STAMP(41);
}

template <typename T, bool kLowp>
__global__ void __launch_bounds__(kCloseThreads) compress_close_kernel(const CompressParams p) {
  extern __shared__ float sm[];
  if (threadIdx.x == 0) CSA_STAMP(40);
  griddep_launch();
  griddep_wait();
  const CompressJob& job = p.job[blockIdx.y];
  if (job.C == 512) compress_close<T, 512, kLowp>(p, job, sm);
  else compress_close<T, 128, kLowp>(p, job, sm);
  if (threadIdx.x == 0) CSA_STAMP(41);
}

template <typename T, bool kLowp>
cudaError_t launch_compress_t(int B, const CompressParams& p, cudaStream_t st, bool pdl) {
  if (p.pos && 2 * p.ratio >= 128) {
    // long windows: a cluster of P CTAs per (request, cache), 64 tokens or more each; shared memory:
    // the partial states, this CTA's merged state [3][512], the pooled row and reduction scratch
    // P = 4 for m = 128: the clusters of one step fit on the GPU at once (with P = 8, of 16
    // clusters of 8 full-SM CTAs a part waited for a second wave)
    int P = 2 * p.ratio / 64;
    if (P > kCloseClusterMax / 2) P = kCloseClusterMax / 2;
    const size_t smem = (size_t)(3 * kCloseThreads * 8 + 3 * 512 + 512 + 32) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(compress_close_split_kernel<T, kLowp>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P, (unsigned)B, (unsigned)p.n_jobs);
    cfg.blockDim = dim3(kCloseThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)P;
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
    return cudaLaunchKernelEx(&cfg, compress_close_split_kernel<T, kLowp>, p);
  }
  if (p.pos) {
    // shared memory: 3 partial states x (token groups x channels), which is kCloseThreads * 8 for
    // both caches, plus the pooled row and reduction scratch
    const size_t smem = (size_t)(3 * kCloseThreads * 8 + 512 + 32) * sizeof(float);
    dim3 grid((unsigned)B, (unsigned)p.n_jobs);
    cudaError_t e = cudaFuncSetAttribute(compress_close_kernel<T, kLowp>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(pdl, compress_close_kernel<T, kLowp>, grid, dim3(kCloseThreads), smem, st, p);
  }
  CompressParams q = p;
  q.epb = kEntriesPerBlock;
  if ((p.n_entries + kEntriesPerBlock - 1) / kEntriesPerBlock * B * p.n_jobs < 4 * 148) q.epb = 16;
  const int64_t nb = (p.n_entries + q.epb - 1) / q.epb;
  if (nb == 0) return cudaSuccess;
  dim3 grid((unsigned)nb, (unsigned)B, (unsigned)p.n_jobs);
  return launch_kernel(pdl, compress_kernel<T, kLowp>, grid, dim3(kThreads), 0, st, q);
}

// ------------------------------------------------------------------ low-precision cache -> bf16
// One thread per (entry, 8 dims): 4 bytes of E2M1 codes and their block's scale byte, or 8 bytes of
// E4M3 codes, become one 16-byte bf16 store (exact: every E2M1 value times a power of two and every
// E4M3 value is a bf16 value).
__global__ void __launch_bounds__(256) dequant_cache_kernel(const uint8_t* src, int C, int d_rope, int64_t n_cap,
                                                            int64_t n_max, const int64_t* pos, int ratio,
                                                            __nv_bfloat16* dst) {
  griddep_launch();
  griddep_wait();
  const int b = blockIdx.y;
  const LowpLayout lay = lowp_layout(C, n_cap, d_rope);
  int64_t n = min(n_cap, n_max);
  if (pos) {
    const int64_t t = pos[b];
    n = t < 0 ? 0 : min(n, (t + 1) / ratio);
  }
  const int cpe = C / 8;
  const int64_t total = n * cpe;
  const uint8_t* base = src + (int64_t)b * lay.stride;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = u / cpe;
    const int c0 = (int)(u % cpe) * 8;
    uint4 o;
    if (c0 < lay.L) {
      const uint32_t codes = __ldg(reinterpret_cast<const uint32_t*>(base + e * (lay.L / 2) + c0 / 2));
      o = dequant_fp4x8(codes, e8m0_to_f32(__ldg(base + lay.scale + e * lay.sb + c0 / 32)));
    } else {
      const uint2 c = __ldg(reinterpret_cast<const uint2*>(base + lay.fp8 + e * lay.R + (c0 - lay.L)));
      o = dequant_fp8x8(c.x, c.y);
    }
    *reinterpret_cast<uint4*>(dst + ((int64_t)b * n_cap + e) * C + c0) = o;
  }
}

}  // namespace

cudaError_t launch_dequant_cache(int B, int C, int d_rope, const void* src, int64_t n_cap, int64_t n_max,
                                 const int64_t* pos, int ratio, void* dst, cudaStream_t st, bool pdl) {
  if (n_max > n_cap) n_max = n_cap;
  if (B == 0 || n_max <= 0) return cudaSuccess;
  const int64_t units = n_max * (C / 8);
  int64_t blocks = (units + 255) / 256;
  if (blocks > 148 * 8) blocks = 148 * 8;
  dim3 grid((unsigned)blocks, (unsigned)B);
  return launch_kernel(pdl, dequant_cache_kernel, grid, dim3(256), 0, st, static_cast<const uint8_t*>(src), C,
                       d_rope, n_cap, n_max, pos, ratio, static_cast<__nv_bfloat16*>(dst));
}

cudaError_t launch_compress(int kind, int B, const CompressParams& p, cudaStream_t st, bool pdl) {
  if (B == 0) return cudaSuccess;
  if (kind == kStoreLowp) return launch_compress_t<__nv_bfloat16, true>(B, p, st, pdl);
  if (kind == kStoreBf16) return launch_compress_t<__nv_bfloat16, false>(B, p, st, pdl);
  return launch_compress_t<float, false>(B, p, st, pdl);
}

}  // namespace csa
