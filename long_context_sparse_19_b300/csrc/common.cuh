// Device helpers shared by the kernels of the CSA / HCA path (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <math.h>

namespace csa {

// Device error word values (written with atomicCAS so the first error wins).
enum DevErr : int32_t {
  DEVERR_NONE = 0,
  DEVERR_BAD_INDEX = 1,      // a selected entry index outside [0, visible)
  DEVERR_TIMEOUT = 2,        // a bounded mbarrier wait ran out
  DEVERR_BAD_POS = 3,        // a position outside the raw capacity
};

__device__ __forceinline__ void set_error(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

// ------------------------------------------------------------------ 8-element vector load / store
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
  v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
}

__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);   // .x = a (low half), .y = b
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 u;
  u.x = pack_bf16(v[0], v[1]); u.y = pack_bf16(v[2], v[3]);
  u.z = pack_bf16(v[4], v[5]); u.w = pack_bf16(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = u;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f32(float& d, float x) { d = x; }
__device__ __forceinline__ void from_f32(__nv_bfloat16& d, float x) { d = __float2bfloat16_rn(x); }

// ------------------------------------------------------------------ RoPE
// Rotary table. theta_i = base^(-2i/d_rope); the kernels use theta_i / pi split into two floats
// (hi + lo, about 48 significant bits), computed in double on the host.
struct RopeTab {
  float th_hi[32];
  float th_lo[32];
  int d_rope;      // <= 64
};

// cos / sin of pos * theta_i without double arithmetic. u = pos * theta_i / pi is formed as an
// unevaluated float sum: TwoProduct with FMA (Ogita, Rump and Oishi, "Accurate sum and dot
// product", 2005) gives pos * th_hi exactly as p + e, and pos * th_lo is added to the error term.
// Subtracting the even integer nearest to p is exact, which reduces u to [-1, 1] half-turns
// (Cody and Waite style reduction with an exactly representable period); sincospif then needs no
// argument reduction of its own. Positions must be < 2^24 (exact in float).
__device__ __forceinline__ void rope_cs(int64_t pos, float th_hi, float th_lo, float& c, float& s) {
  const float x = (float)pos;
  const float p = x * th_hi;
  const float e = fmaf(x, th_hi, -p);
  const float lo = fmaf(x, th_lo, e);
  const float r = (p - 2.0f * rintf(0.5f * p)) + lo;
  sincospif(r, &s, &c);
}

__device__ __forceinline__ void rope_cs(int64_t pos, const RopeTab& tab, int i, float& c, float& s) {
  rope_cs(pos, tab.th_hi[i], tab.th_lo[i], c, s);
}

// rope_cs out of line, (cos, sin) returned in registers: for code that runs once per CTA, where every
// inlined copy of the sine / cosine evaluation is fetched from memory again
static __device__ __noinline__ float2 rope_cs_nl(int64_t pos, float th_hi, float th_lo) {
  float c, s;
  rope_cs(pos, th_hi, th_lo, c, s);
  return make_float2(c, s);
}

// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32: relative error about 2^-22, 2^-inf = 0,
// subnormal results flushed to zero). For softmax weights that are rounded to bf16 / fp16 next; the
// library's exp2f also handles subnormal inputs and costs several times more per element.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ programmatic dependent launch
// A kernel launched with programmatic stream serialization may start while the previous kernel of
// the stream is still running; griddep_wait() blocks until that kernel has completed and its
// memory is visible (a no-op for a normal launch). griddep_launch() lets the next kernel start.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Asks L2 to fetch `bytes` (a multiple of 16, 16-byte aligned) starting at p; nothing waits for it.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ thread-block clusters
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Cluster barrier in two halves, so that independent work can run between them. The arrive
// releases this thread's earlier shared-memory writes (local and remote) at cluster scope; the
// wait acquires every other thread's. All threads of every CTA of the cluster take part.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() { cluster_arrive(); cluster_wait(); }

// shared::cluster address of the variable at local shared address `p` in CTA `rank`
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t remote;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}
// fire-and-forget writes into another CTA's shared memory (visible there after a cluster barrier)
__device__ __forceinline__ void dsmem_add(uint32_t addr, uint32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void dsmem_st(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void dsmem_st4(uint32_t addr, uint4 v) {   // addr 16-byte aligned
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w) : "memory");
}

// loads from another CTA's shared memory (a shared::cluster address from dsmem_addr)
__device__ __forceinline__ float dsmem_ldf(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 dsmem_ld4f(uint32_t addr) {   // addr 16-byte aligned
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr) : "memory");
  return v;
}

// ------------------------------------------------------------------ phase stamps
// CSA_STAMP(slot) records %globaltimer for (CTA, slot) in a device table when the library is
// compiled with -DCSA_TRACE (a timing build that also defines g_trace); otherwise it is nothing.
#ifdef CSA_TRACE
extern __device__ unsigned long long g_trace[8192][64];
#define CSA_STAMP(slot)                                                                            \
  do {                                                                                             \
    unsigned long long t_;                                                                         \
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                                         \
    const int c_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);                 \
    if (c_ < 8192 && (slot) < 64) ::csa::g_trace[c_][(slot)] = t_;                                 \
  } while (0)
// CSA_TRACE_VAL(slot, v): the value v itself in the same table (timing build only).
#define CSA_TRACE_VAL(slot, v)                                                                     \
  do {                                                                                             \
    const int c_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);                 \
    if (c_ < 8192 && (slot) < 64) ::csa::g_trace[c_][(slot)] = (unsigned long long)(v);            \
  } while (0)
#else
#define CSA_STAMP(slot) ((void)0)
#define CSA_TRACE_VAL(slot, v) ((void)0)
#endif

// visible compressed entries of a query at t
__device__ __forceinline__ int64_t visible_entries(int64_t t, int ratio) { return (t + 1) / ratio; }

// visible entries of a cache that holds the entry run [base, base + n) of a request at rows 0 .. n-1
// (a shard of the entry range; base = 0 for a whole cache)
__device__ __forceinline__ int64_t visible_local(int64_t t, int ratio, int64_t base, int64_t n) {
  if (t < 0) return 0;
  const int64_t v = visible_entries(t, ratio) - base;
  return v < 0 ? 0 : (v < n ? v : n);
}

}  // namespace csa
