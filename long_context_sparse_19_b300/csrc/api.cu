// C ABI of the CSA / HCA path: argument checks, workspace carving, kernel dispatch.
// Every entry point only enqueues kernels on the caller's stream; nothing here allocates.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/csa.h"
#include "kernels.h"
#include "lowp.cuh"
#include "tc.h"

namespace {

using namespace csa;

thread_local std::string g_last_error;

__device__ int32_t g_device_error;      // per-device error word (first error wins)

int32_t* device_error_word() {
  static std::mutex mu;
  static int32_t* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int32_t*>(p);
  }
  return addr[dev];
}

// Scratch of csa_index_topk_static: one fixed device array (every device that loads the library
// holds it until the process exits); no call ever allocates it or frees it.
__device__ __align__(256) uint8_t g_static_scratch[CSA_STATIC_SCRATCH_BYTES];

// Device address of g_static_scratch on the current device, looked up once per device with that
// device current (host code must not pass the symbol itself to a kernel).
uint8_t* static_scratch(cudaError_t* err) {
  static std::mutex mu;
  static uint8_t* addr[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess && (dev < 0 || dev >= 64)) e = cudaErrorInvalidDevice;
  if (e != cudaSuccess) { *err = e; return nullptr; }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) { *err = e; return nullptr; }
    addr[dev] = static_cast<uint8_t*>(ptr);
  }
  return addr[dev];
}

csa_status fail(csa_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
csa_status fail(csa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

csa_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return CSA_OK;
  return fail(CSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define CHECK_PTR(p)                                                                       \
  do {                                                                                     \
    if (!(p)) return fail(CSA_ERR_INVALID_ARG, "%s is NULL", #p);                          \
    if (!aligned16(p)) return fail(CSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p);  \
  } while (0)

#define CHECK_OPT_PTR(p)                                                                   \
  do {                                                                                     \
    if ((p) && !aligned16(p)) return fail(CSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p); \
  } while (0)

csa_status check_config(const csa_config* c) {
  if (!c) return fail(CSA_ERR_INVALID_ARG, "cfg is NULL");
  if (c->storage != CSA_F32 && c->storage != CSA_BF16 && c->storage != CSA_FP4)
    return fail(CSA_ERR_DTYPE, "storage dtype %d", (int)c->storage);
  if (c->d != 512) return fail(CSA_ERR_SHAPE, "d = %d (supported: 512)", c->d);
  if (c->d_rope != 64) return fail(CSA_ERR_SHAPE, "d_rope = %d (supported: 64)", c->d_rope);
  if (c->H < 1 || c->H > 64) return fail(CSA_ERR_SHAPE, "H = %d (supported: 1..64)", c->H);
  if (c->ratio < 1 || c->ratio > 256) return fail(CSA_ERR_SHAPE, "ratio = %d (supported: 1..256)", c->ratio);
  if (c->top_k < 0 || c->top_k > 2048) return fail(CSA_ERR_SHAPE, "top_k = %d (supported: 0..2048)", c->top_k);
  if (c->window < 1 || c->window > 1024) return fail(CSA_ERR_SHAPE, "window = %d (supported: 1..1024)", c->window);
  if (c->top_k > 0) {
    if (c->d_idx != 128) return fail(CSA_ERR_SHAPE, "d_idx = %d (supported: 128)", c->d_idx);
    if (c->H_idx < 1 || c->H_idx > 64) return fail(CSA_ERR_SHAPE, "H_idx = %d (supported: 1..64)", c->H_idx);
  }
  if (!(c->rope_base > 0.f)) return fail(CSA_ERR_INVALID_ARG, "rope_base must be > 0");
  if (!(c->rms_eps >= 0.f)) return fail(CSA_ERR_INVALID_ARG, "rms_eps must be >= 0");
  return CSA_OK;
}

RopeTab make_rope(const csa_config* c) {
  RopeTab r;
  memset(&r, 0, sizeof r);
  r.d_rope = c->d_rope;
  const double inv_pi = 0.31830988618379067153776752674503;
  for (int i = 0; i < c->d_rope / 2; ++i) {
    const double tp = pow((double)c->rope_base, -2.0 * i / c->d_rope) * inv_pi;
    r.th_hi[i] = (float)tp;
    r.th_lo[i] = (float)(tp - (double)r.th_hi[i]);
  }
  return r;
}

float softmax_scale(const csa_config* c) {
  return c->softmax_scale > 0.f ? c->softmax_scale : (float)(1.0 / sqrt((double)c->d));
}

// Low-precision caches (raw rows, queries and outputs in bf16).
bool lowp(const csa_config* c) { return c->storage == CSA_FP4; }
// Raw rows, queries and outputs in bf16 (every storage but float32).
bool bf16_io(const csa_config* c) { return c->storage != CSA_F32; }
int store_kind(const csa_config* c) {
  return c->storage == CSA_FP4 ? kStoreLowp : c->storage == CSA_BF16 ? kStoreBf16 : kStoreF32;
}

bool use_tc_index(const csa_config* c) {
  return tc_index_available() && bf16_io(c) && !(c->flags & CSA_FLAG_SIMT) && c->top_k > 0 && c->H_idx == 64 &&
         c->d_idx == 128;
}

bool use_tc_attn(const csa_config* c) {
  return tc_attn_available() && bf16_io(c) && !(c->flags & CSA_FLAG_SIMT) && c->H == 64 && c->d == 512;
}

// Cluster size of the fused decode indexer + selection for this call, or 0 when it does not apply.
int fused_select_cluster(const csa_config* c, int B, int S, int64_t n_cap) {
  if (S != 1 || !use_tc_index(c)) return 0;
  return tc_index_select_cluster(B, n_cap);
}

// ------------------------------------------------------------------ launch counting / stage profiling
enum Stage { ST_COMPRESS = 0, ST_INDEX = 1, ST_TOPK = 2, ST_ATTN = 3, ST_MERGE = 4, ST_COUNT = 5 };

std::atomic<int64_t> g_launches{0};

struct ProfRec {
  int stage;
  cudaEvent_t a, b;
};

struct Profiler {
  std::mutex mu;
  bool on = false;
  int cap = 0;
  std::vector<ProfRec> recs;
  std::vector<cudaEvent_t> pool;
  int extra[ST_COUNT] = {0};     // launches counted beyond the recording cap
} g_prof;

// Wraps one kernel launch: counts it and, while profiling, brackets it with an event pair.
template <typename F>
cudaError_t launch_stage(int stage, cudaStream_t st, F&& f) {
  ProfRec rec{stage, nullptr, nullptr};
  bool recorded = false;
  {
    std::lock_guard<std::mutex> lock(g_prof.mu);
    if (g_prof.on) {
      if ((int)g_prof.recs.size() < g_prof.cap && g_prof.pool.size() >= 2) {
        rec.a = g_prof.pool.back(); g_prof.pool.pop_back();
        rec.b = g_prof.pool.back(); g_prof.pool.pop_back();
        recorded = true;
      } else {
        g_prof.extra[stage]++;
      }
    }
  }
  if (recorded) cudaEventRecord(rec.a, st);
  const cudaError_t e = f();
  if (recorded) {
    cudaEventRecord(rec.b, st);
    std::lock_guard<std::mutex> lock(g_prof.mu);
    g_prof.recs.push_back(rec);
  }
  if (e == cudaSuccess) g_launches.fetch_add(1);
  return e;
}

// ------------------------------------------------------------------ workspace plan
constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Plan {
  bool tc_attn = false;
  bool tc_prefill = false;           // one CTA per query over all candidates, no partials
  int fused = 0;                     // decode: cluster size of the fused attention + merge (0: split path)
  int f_wc = 0, f_kc = 0, f_rows = 0;
  int n_split = 1, split_len = 0;
  // low-precision caches: the one-launch indexer reads cidx directly (idx_direct); otherwise the
  // entries a call reads are first expanded into bf16 copies in the workspace (dq_idx, dq_kv)
  bool idx_direct = false, dq_idx = false, dq_kv = false;
  size_t off_scores = 0, off_topk = 0, off_tksel = 0, off_po = 0, off_pml = 0, off_tc = 0, total = 0;
  size_t off_dq_idx = 0, off_dq_kv = 0;
};

Plan make_plan(const csa_config* c, int B, int S, int64_t n_cap) {
  Plan p;
  const bool hca = c->top_k == 0;
  const int64_t c_max = (int64_t)c->window + (hca ? n_cap : c->top_k);
  if (S == 1) {                               // decode: split the candidates across CTAs
    p.tc_attn = use_tc_attn(c);
    if (p.tc_attn && !hca) p.fused = tc_attn_fused_plan(B, c->window, c->top_k, &p.f_wc, &p.f_kc, &p.f_rows);
    if (p.fused) {
      p.tc_attn = false;                      // one cluster per query merges on chip: no partials
      p.n_split = 1;
      p.split_len = (int)c_max;
    } else if (p.tc_attn) {
      p.split_len = tc_attn_split_len();
      p.n_split = tc_attn_splits(c->window, c->top_k, n_cap, B * S);
    } else {
      p.split_len = 64;
      p.n_split = (int)((c_max + p.split_len - 1) / p.split_len);
    }
    if (p.n_split < 1) p.n_split = 1;
  } else {
    p.split_len = (int)c_max;
    p.n_split = 1;
    const int64_t tiles = (c->window + 127) / 128 + (hca ? (n_cap + 127) / 128 : (c->top_k + 127) / 128);
    p.tc_prefill = use_tc_attn(c) && tiles <= tc_attn_prefill_max_tiles();
  }
  size_t o = 0;
  const size_t rows = (size_t)B * (size_t)S;
  if (!hca) {
    p.off_scores = o; o = up(o + rows * (size_t)n_cap * sizeof(float));
    p.off_topk = o;   o = up(o + rows * (size_t)c->top_k * sizeof(int32_t));
    p.off_tksel = o;  o = up(o + topk_workspace_bytes((int64_t)rows, n_cap, c->top_k));
  }
  if (p.fused) {                              // fp16 partials of each CTA of a query's cluster
    p.off_po = o;  o = up(o + tc_attn_fused_workspace(B, p.fused));
  } else if (p.n_split > 1 || p.tc_attn) {
    p.off_po = o;  o = up(o + rows * p.n_split * (size_t)c->H * c->d * sizeof(float));
    p.off_pml = o; o = up(o + rows * p.n_split * (size_t)c->H * 2 * sizeof(float));
  }
  p.off_tc = o;
  o = up(o + tc_workspace_bytes(B, S, n_cap, c->top_k));
  if (lowp(c)) {
    if (S == 1 && !hca) {
      p.idx_direct = fused_select_cluster(c, B, S, n_cap) > 0;
      p.dq_idx = !p.idx_direct;
      p.dq_kv = !p.fused;
    } else {
      p.dq_idx = !hca;
      p.dq_kv = true;
    }
    if (p.dq_idx) { p.off_dq_idx = o; o = up(o + (size_t)B * (size_t)n_cap * c->d_idx * 2); }
    if (p.dq_kv) { p.off_dq_kv = o; o = up(o + (size_t)B * (size_t)n_cap * c->d * 2); }
  }
  p.total = o;
  return p;
}

template <typename T>
T* carve(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

csa_status check_ws(const Plan& pl, void* ws, size_t ws_bytes) {
  if (ws_bytes < pl.total) return fail(CSA_ERR_WORKSPACE, "workspace %zu bytes < required %zu", ws_bytes, pl.total);
  if (pl.total && !ws) return fail(CSA_ERR_INVALID_ARG, "ws is NULL");
  if (ws && !aligned16(ws)) return fail(CSA_ERR_INVALID_ARG, "ws is not 16-byte aligned");
  return CSA_OK;
}

// ------------------------------------------------------------------ stage launchers
CompressParams compress_params(const csa_config* c, const csa_cache* k, int64_t first, int64_t n,
                               const int64_t* pos) {
  CompressParams p;
  memset(&p, 0, sizeof p);
  p.job[0] = CompressJob{k->kv, k->gate, k->gate_bias, k->ckv, c->d};
  p.n_jobs = 1;
  if (c->top_k > 0 && k->idx_k) {
    p.job[1] = CompressJob{k->idx_k, k->idx_gate, k->idx_bias, k->cidx, c->d_idx};
    p.n_jobs = 2;
  }
  p.N = k->N; p.n_cap = k->n_cap; p.first_entry = first; p.n_entries = n; p.pos = pos;
  p.ratio = c->ratio; p.eps = c->rms_eps; p.rope = make_rope(c); p.err = device_error_word();
  return p;
}

csa_status run_compress(const csa_config* c, int B, const csa_cache* k, int64_t first, int64_t n,
                        const int64_t* pos, cudaStream_t st) {
  const CompressParams p = compress_params(c, k, first, n, pos);
  // the compressor is the first kernel of every call that runs it: a normal (fully ordered) launch
  return cuda_status(
      launch_stage(ST_COMPRESS, st, [&] { return launch_compress(store_kind(c), B, p, st, false); }),
      "compress launch");
}

// `scores`: where the scores go; `scores_out`: the caller's score output (nullable), the only
// scores the fused decode kernel writes (it keeps its own in shared memory).
csa_status run_index_topk(const csa_config* c, int B, int S, const int64_t* pos, const void* q_idx,
                          const float* w, const void* cidx, int64_t n_cap, int32_t* topk,
                          float* scores, float* scores_out, void* tk_ws, void* tc_ws, cudaStream_t st,
                          bool pdl, const CompressParams* close = nullptr, const void* ckv_prefetch = nullptr,
                          int64_t entry_base = 0) {
  const bool bf16 = bf16_io(c);
  // with lowp(c): cidx is the low-precision cache; a shard of the entry range takes the general path
  const int clu = entry_base == 0 ? fused_select_cluster(c, B, S, n_cap) : 0;
  if (clu > 0) {
    const RopeTab rope = make_rope(c);
    int32_t* err = device_error_word();
    return cuda_status(launch_stage(ST_INDEX, st, [&] {
                         return tc_index_select(B, clu, pos, q_idx, w, cidx, n_cap, c->ratio, c->top_k, rope,
                                                scores_out, topk, err, st, pdl, close, ckv_prefetch,
                                                (c->flags & CSA_FLAG_TEST_STALL) != 0, lowp(c));
                       }),
                       "fused indexer + selection launch");
  }
  if (use_tc_index(c)) {
    const RopeTab rope = make_rope(c);
    int32_t* err = device_error_word();
    cudaError_t e = launch_stage(ST_INDEX, st, [&] {
      return tc_index_scores(B, S, pos, q_idx, w, cidx, n_cap, c->ratio, rope, scores, tc_ws, err, st, pdl, close,
                             entry_base);
    });
    if (e != cudaSuccess) return cuda_status(e, "tcgen05 indexer launch");
  } else {
    IndexParams ip;
    memset(&ip, 0, sizeof ip);
    ip.q_idx = q_idx; ip.w = w; ip.cidx = cidx; ip.scores = scores; ip.pos = pos; ip.n_cap = n_cap;
    ip.S = S; ip.H_idx = c->H_idx; ip.ratio = c->ratio; ip.rope = make_rope(c); ip.entry_base = entry_base;
    csa_status s = cuda_status(launch_stage(ST_INDEX, st, [&] { return launch_index_simt(bf16, B, ip, st, pdl); }),
                               "indexer launch");
    if (s != CSA_OK) return s;
  }
  TopkParams tp;
  memset(&tp, 0, sizeof tp);
  tp.scores = scores; tp.topk = topk; tp.pos = pos; tp.n_cap = n_cap; tp.S = S; tp.k = c->top_k;
  tp.ratio = c->ratio; tp.ws = tk_ws; tp.entry_base = entry_base;
  return cuda_status(launch_stage(ST_TOPK, st, [&] { return launch_topk(B, tp, st, true); }), "top-k launch");
}

csa_status run_attn(const csa_config* c, const Plan& pl, int B, int S, const int64_t* pos,
                    const void* q, const void* kv, int64_t N, const void* ckv, int64_t n_cap,
                    const int32_t* topk, const float* sink, void* out, void* ws, cudaStream_t st, bool pdl) {
  AttnParams ap;
  memset(&ap, 0, sizeof ap);
  ap.q = q; ap.kv = kv; ap.ckv = ckv; ap.topk = c->top_k > 0 ? topk : nullptr; ap.sink = sink;
  ap.out = out; ap.pos = pos; ap.N = N; ap.n_cap = n_cap; ap.S = S; ap.H = c->H; ap.k = c->top_k;
  ap.ratio = c->ratio; ap.window = c->window; ap.n_split = pl.n_split; ap.split_len = pl.split_len;
  ap.scale = softmax_scale(c); ap.rope = make_rope(c); ap.err = device_error_word();
  if (pl.n_split > 1 || pl.tc_attn) { ap.part_o = carve<float>(ws, pl.off_po); ap.part_ml = carve<float>(ws, pl.off_pml); }
  const bool bf16 = bf16_io(c);
  cudaError_t e;
  if (pl.fused) {                             // with lowp(c): ckv is the low-precision cache
    e = launch_stage(ST_ATTN, st, [&] {
      return tc_attn_fused(B, pl.fused, pl.f_wc, pl.f_kc, pl.f_rows, ap, carve<char>(ws, pl.off_po), st, pdl,
                           lowp(c));
    });
    return cuda_status(e, "fused decode attention launch");
  }
  if (pl.tc_prefill) {
    e = launch_stage(ST_ATTN, st, [&] { return tc_attn_prefill(B, ap, st, pdl); });
    return cuda_status(e, "prefill attention launch");
  }
  if (pl.tc_attn) e = launch_stage(ST_ATTN, st, [&] { return tc_sparse_attn(B, ap, carve<char>(ws, pl.off_tc), st, pdl); });
  else e = launch_stage(ST_ATTN, st, [&] { return launch_attn_simt(bf16, B, ap, st, pdl); });
  if (e != cudaSuccess) return cuda_status(e, "attention launch");
  if (pl.n_split <= 1 && !pl.tc_attn) return CSA_OK;
  return cuda_status(launch_stage(ST_MERGE, st, [&] { return launch_attn_merge(bf16, B, ap, st, true); }),
                     "merge launch");
}

csa_status check_cache_ptrs(const csa_config* c, const csa_cache* k, bool need_idx) {
  if (!k) return fail(CSA_ERR_INVALID_ARG, "cache is NULL");
  CHECK_PTR(k->kv); CHECK_PTR(k->gate); CHECK_PTR(k->gate_bias); CHECK_PTR(k->ckv);
  if (need_idx) { CHECK_PTR(k->idx_k); CHECK_PTR(k->idx_gate); CHECK_PTR(k->idx_bias); CHECK_PTR(k->cidx); }
  if (k->N < 1 || k->n_cap < 1) return fail(CSA_ERR_SHAPE, "cache N = %lld, n_cap = %lld", (long long)k->N, (long long)k->n_cap);
  (void)c;
  return CSA_OK;
}

// Low-precision cache -> its bf16 copy in the workspace (entries < n_max, limited to the visible ones
// of pos[b] when pos is non-null).
csa_status run_dequant(const csa_config* c, int B, int which, const void* src, int64_t n_cap, int64_t n_max,
                       const int64_t* pos, void* dst, cudaStream_t st, bool pdl) {
  const int C = which ? c->d_idx : c->d;
  return cuda_status(launch_stage(ST_COMPRESS, st, [&] {
                       return launch_dequant_cache(B, C, c->d_rope, src, n_cap, n_max, pos, c->ratio, dst, st, pdl);
                     }),
                     "cache expansion launch");
}

}  // namespace

// ================================================================== C ABI
extern "C" {

const char* csa_status_string(csa_status s) {
  switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARG: return "invalid argument";
    case CSA_ERR_SHAPE: return "unsupported or inconsistent shape";
    case CSA_ERR_DTYPE: return "unsupported dtype";
    case CSA_ERR_WORKSPACE: return "workspace too small";
    case CSA_ERR_CUDA: return "CUDA error";
    case CSA_ERR_DEVICE: return "device-side error";
    case CSA_ERR_NOT_IMPLEMENTED: return "not implemented";
    case CSA_ERR_DEVICE_TIMEOUT: return "a device-side wait ran out";
  }
  return "unknown status";
}

const char* csa_last_error(void) { return g_last_error.c_str(); }

csa_status csa_get_device_status(cudaStream_t stream, int reset, int32_t* code) {
  int32_t* w = device_error_word();
  if (!w) return fail(CSA_ERR_CUDA, "device error word unavailable");
  csa_status s = cuda_status(cudaStreamSynchronize(stream), "stream synchronize");
  if (s != CSA_OK) return s;
  int32_t v = 0;
  s = cuda_status(cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost), "read error word");
  if (s != CSA_OK) return s;
  if (reset) {
    s = cuda_status(cudaMemset(w, 0, sizeof v), "clear error word");
    if (s != CSA_OK) return s;
    s = cuda_status(cudaDeviceSynchronize(), "clear error word");
    if (s != CSA_OK) return s;
  }
  if (code) *code = v;
  if (!v) return CSA_OK;
  return v == DEVERR_TIMEOUT ? CSA_ERR_DEVICE_TIMEOUT : CSA_ERR_DEVICE;
}

csa_status csa_sync_status(cudaStream_t stream) { return csa_get_device_status(stream, 0, nullptr); }

size_t csa_cache_bytes(const csa_config* cfg, int32_t which, int64_t n_cap) {
  if (check_config(cfg) != CSA_OK || n_cap < 0 || (which != 0 && which != 1)) return 0;
  const int C = which ? cfg->d_idx : cfg->d;
  if (cfg->storage == CSA_FP4) return (size_t)lowp_layout(C, n_cap, cfg->d_rope).stride;
  return (size_t)n_cap * C * (cfg->storage == CSA_F32 ? 4 : 2);
}

size_t csa_workspace_bytes(const csa_config* cfg, int32_t B, int32_t S, int64_t n_cap) {
  if (check_config(cfg) != CSA_OK || B < 0 || S < 0 || n_cap < 0) return 0;
  return make_plan(cfg, B, S, n_cap).total;
}

csa_status csa_compress(const csa_config* cfg, int32_t B, const csa_cache* cache, int64_t first_entry,
                        int64_t n_entries, cudaStream_t stream) {
  csa_status s = check_config(cfg);
  if (s != CSA_OK) return s;
  if (B < 0 || B > 65535) return fail(CSA_ERR_SHAPE, "B = %d", B);
  s = check_cache_ptrs(cfg, cache, cfg->top_k > 0 && cache && cache->idx_k);
  if (s != CSA_OK) return s;
  if (first_entry < 0 || n_entries < 0) return fail(CSA_ERR_INVALID_ARG, "negative entry range");
  if ((first_entry + n_entries) * cfg->ratio > cache->N)
    return fail(CSA_ERR_SHAPE, "entries up to %lld need %lld raw tokens > N = %lld",
                (long long)(first_entry + n_entries), (long long)((first_entry + n_entries) * cfg->ratio),
                (long long)cache->N);
  if (first_entry + n_entries > cache->n_cap) return fail(CSA_ERR_SHAPE, "entry range exceeds n_cap");
  if (B == 0 || n_entries == 0) return CSA_OK;
  return run_compress(cfg, B, cache, first_entry, n_entries, nullptr, stream);
}

csa_status csa_index_topk(const csa_config* cfg, int32_t B, int32_t S, const int64_t* pos,
                          const void* q_idx, const float* w, const void* cidx, int64_t n_cap,
                          int32_t* topk, float* scores, void* ws, size_t ws_bytes, cudaStream_t stream) {
  csa_status s = check_config(cfg);
  if (s != CSA_OK) return s;
  if (cfg->top_k == 0) return fail(CSA_ERR_INVALID_ARG, "top_k == 0 (HCA) has no indexer");
  if (B < 0 || B > 65535 || S < 0 || S > 65535) return fail(CSA_ERR_SHAPE, "B = %d, S = %d", B, S);
  if (n_cap < 1) return fail(CSA_ERR_SHAPE, "n_cap = %lld", (long long)n_cap);
  CHECK_PTR(pos); CHECK_PTR(q_idx); CHECK_PTR(w); CHECK_PTR(cidx); CHECK_PTR(topk); CHECK_OPT_PTR(scores);
  const Plan pl = make_plan(cfg, B, S, n_cap);
  s = check_ws(pl, ws, ws_bytes);
  if (s != CSA_OK) return s;
  if (B == 0 || S == 0) return CSA_OK;
  float* sc = scores ? scores : carve<float>(ws, pl.off_scores);
  const void* ci = cidx;
  bool pdl = false;
  if (pl.dq_idx) {
    s = run_dequant(cfg, B, 1, cidx, n_cap, n_cap, S == 1 ? pos : nullptr, carve<char>(ws, pl.off_dq_idx), stream,
                    false);
    if (s != CSA_OK) return s;
    ci = carve<char>(ws, pl.off_dq_idx);
    pdl = true;
  }
  return run_index_topk(cfg, B, S, pos, q_idx, w, ci, n_cap, topk, sc, scores, carve<char>(ws, pl.off_tksel),
                        carve<char>(ws, pl.off_tc), stream, pdl);
}

csa_status csa_index_topk_static(const csa_config* cfg, int32_t B, int32_t S, const int64_t* pos,
                                 const void* q_idx, const float* w, const void* cidx, int64_t n_cap,
                                 int32_t* topk, float* scores, cudaStream_t stream) {
  csa_status s = check_config(cfg);
  if (s != CSA_OK) return s;
  if (cfg->top_k == 0) return fail(CSA_ERR_INVALID_ARG, "top_k == 0 (HCA) has no indexer");
  if (B < 0 || B > 65535 || S < 0 || S > 65535) return fail(CSA_ERR_SHAPE, "B = %d, S = %d", B, S);
  if (n_cap < 1) return fail(CSA_ERR_SHAPE, "n_cap = %lld", (long long)n_cap);
  CHECK_PTR(pos); CHECK_PTR(q_idx); CHECK_PTR(w); CHECK_PTR(cidx); CHECK_PTR(topk); CHECK_OPT_PTR(scores);
  // Scratch actually used: nothing on the fused decode path (scores stay on chip); otherwise the
  // float32 scores when the caller passes none, then the candidate lists of long rows.
  const bool fused = fused_select_cluster(cfg, B, S, n_cap) > 0;
  if (lowp(cfg) && !fused)
    return fail(CSA_ERR_WORKSPACE,
                "csa_index_topk_static: a low-precision index cache outside the one-launch decode indexer needs "
                "a bf16 copy in a workspace; call csa_index_topk with a workspace instead");
  const size_t rows = (size_t)B * (size_t)S;
  const size_t sc_bytes = (fused || scores) ? 0 : up(rows * (size_t)n_cap * sizeof(float));
  const size_t tk_bytes = fused ? 0 : topk_workspace_bytes((int64_t)rows, n_cap, cfg->top_k);
  const size_t need = sc_bytes + tk_bytes;
  if (need > (size_t)CSA_STATIC_SCRATCH_BYTES)
    return fail(CSA_ERR_WORKSPACE,
                "csa_index_topk_static: B = %d, S = %d, n_cap = %lld need %zu bytes of scratch, more than the "
                "static %u-byte array; call csa_index_topk with a workspace instead",
                B, S, (long long)n_cap, need, (unsigned)CSA_STATIC_SCRATCH_BYTES);
  cudaError_t e = cudaSuccess;
  uint8_t* ws = static_scratch(&e);
  if (!ws) return cuda_status(e, "csa_index_topk_static: device address of the static scratch");
  if (B == 0 || S == 0) return CSA_OK;
  float* sc = scores ? scores : reinterpret_cast<float*>(ws);
  return run_index_topk(cfg, B, S, pos, q_idx, w, cidx, n_cap, topk, sc, scores, ws + sc_bytes, nullptr, stream,
                        false);
}

csa_status csa_sparse_attn(const csa_config* cfg, int32_t B, int32_t S, const int64_t* pos, const void* q,
                           const void* kv, int64_t N, const void* ckv, int64_t n_cap, const int32_t* topk,
                           const float* sink, void* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  csa_status s = check_config(cfg);
  if (s != CSA_OK) return s;
  if (B < 0 || B > 65535 || S < 0 || S > 65535) return fail(CSA_ERR_SHAPE, "B = %d, S = %d", B, S);
  if (N < 1 || n_cap < 1) return fail(CSA_ERR_SHAPE, "N = %lld, n_cap = %lld", (long long)N, (long long)n_cap);
  CHECK_PTR(pos); CHECK_PTR(q); CHECK_PTR(kv); CHECK_PTR(ckv); CHECK_PTR(sink); CHECK_PTR(out);
  if (cfg->top_k > 0) CHECK_PTR(topk);
  const Plan pl = make_plan(cfg, B, S, n_cap);
  s = check_ws(pl, ws, ws_bytes);
  if (s != CSA_OK) return s;
  if (B == 0 || S == 0) return CSA_OK;
  const void* ck = ckv;
  bool pdl = false;
  if (pl.dq_kv) {
    s = run_dequant(cfg, B, 0, ckv, n_cap, n_cap, S == 1 ? pos : nullptr, carve<char>(ws, pl.off_dq_kv), stream,
                    false);
    if (s != CSA_OK) return s;
    ck = carve<char>(ws, pl.off_dq_kv);
    pdl = true;
  }
  return run_attn(cfg, pl, B, S, pos, q, kv, N, ck, n_cap, topk, sink, out, ws, stream, pdl);
}

csa_status csa_decode(const csa_config* cfg, int32_t B, const int64_t* pos, const csa_cache* cache,
                      const void* q, const void* q_idx, const float* w, const float* sink, void* out,
                      int32_t* topk_out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  csa_status s = check_config(cfg);
  if (s != CSA_OK) return s;
  const bool hca = cfg->top_k == 0;
  if (B < 0 || B > 65535) return fail(CSA_ERR_SHAPE, "B = %d", B);
  s = check_cache_ptrs(cfg, cache, !hca);
  if (s != CSA_OK) return s;
  CHECK_PTR(pos); CHECK_PTR(q); CHECK_PTR(sink); CHECK_PTR(out); CHECK_OPT_PTR(topk_out);
  if (!hca) { CHECK_PTR(q_idx); CHECK_PTR(w); }
  const Plan pl = make_plan(cfg, B, 1, cache->n_cap);
  s = check_ws(pl, ws, ws_bytes);
  if (s != CSA_OK) return s;
  if (B == 0) return CSA_OK;
  // CSA with the tensor-core indexer: the step's first kernel is the indexer, which also pools the
  // entries that t closes (both caches) before the scores need them. Otherwise the compressor's
  // close kernel runs first. With low-precision caches the indexer pools them only when it is the
  // one-launch kernel that reads the low-precision index cache itself; every cache that a later
  // kernel cannot read directly is then expanded into its bf16 copy (the visible entries only).
  const bool fused_close = !hca && use_tc_index(cfg) && (!lowp(cfg) || pl.idx_direct);
  const CompressParams close = compress_params(cfg, cache, 0, 0, pos);
  bool after_first = false;
  if (!fused_close) {
    s = run_compress(cfg, B, cache, 0, 0, pos, stream);
    if (s != CSA_OK) return s;
    after_first = true;
  }
  const void* ci = cache->cidx;
  const void* ck = cache->ckv;
  if (pl.dq_idx) {
    s = run_dequant(cfg, B, 1, cache->cidx, cache->n_cap, cache->n_cap, pos, carve<char>(ws, pl.off_dq_idx), stream,
                    after_first);
    if (s != CSA_OK) return s;
    ci = carve<char>(ws, pl.off_dq_idx);
    after_first = true;
  }
  if (pl.dq_kv && hca) {                      // with CSA the KV copy waits for the indexer's close
    s = run_dequant(cfg, B, 0, cache->ckv, cache->n_cap, cache->n_cap, pos, carve<char>(ws, pl.off_dq_kv), stream,
                    after_first);
    if (s != CSA_OK) return s;
    ck = carve<char>(ws, pl.off_dq_kv);
    after_first = true;
  }
  int32_t* tk = nullptr;
  if (!hca) {
    tk = topk_out ? topk_out : carve<int32_t>(ws, pl.off_topk);
    s = run_index_topk(cfg, B, 1, pos, q_idx, w, ci, cache->n_cap, tk,
                       carve<float>(ws, pl.off_scores), nullptr, carve<char>(ws, pl.off_tksel),
                       carve<char>(ws, pl.off_tc), stream, after_first, fused_close ? &close : nullptr,
                       pl.fused ? cache->ckv : nullptr);
    if (s != CSA_OK) return s;
    if (pl.dq_kv) {
      s = run_dequant(cfg, B, 0, cache->ckv, cache->n_cap, cache->n_cap, pos, carve<char>(ws, pl.off_dq_kv), stream,
                      true);
      if (s != CSA_OK) return s;
      ck = carve<char>(ws, pl.off_dq_kv);
    }
  }
  return run_attn(cfg, pl, B, 1, pos, q, cache->kv, cache->N, ck, cache->n_cap, tk, sink, out, ws, stream, true);
}

csa_status csa_prefill(const csa_config* cfg, int32_t B, int32_t S, const csa_cache* cache, const void* q,
                       const void* q_idx, const float* w, const float* sink, void* out, int32_t* topk_out,
                       void* ws, size_t ws_bytes, cudaStream_t stream) {
  csa_status s = check_config(cfg);
  if (s != CSA_OK) return s;
  const bool hca = cfg->top_k == 0;
  if (B < 0 || B > 65535 || S < 0 || S > 65535) return fail(CSA_ERR_SHAPE, "B = %d, S = %d", B, S);
  s = check_cache_ptrs(cfg, cache, !hca);
  if (s != CSA_OK) return s;
  if (S > cache->N) return fail(CSA_ERR_SHAPE, "S = %d > N = %lld", S, (long long)cache->N);
  if (S / cfg->ratio > cache->n_cap) return fail(CSA_ERR_SHAPE, "S / ratio entries exceed n_cap");
  CHECK_PTR(q); CHECK_PTR(sink); CHECK_PTR(out); CHECK_OPT_PTR(topk_out);
  if (!hca) { CHECK_PTR(q_idx); CHECK_PTR(w); }
  const Plan pl = make_plan(cfg, B, S, cache->n_cap);
  s = check_ws(pl, ws, ws_bytes);
  if (s != CSA_OK) return s;
  if (B == 0 || S == 0) return CSA_OK;
  s = run_compress(cfg, B, cache, 0, S / cfg->ratio, nullptr, stream);
  if (s != CSA_OK) return s;
  const void* ci = cache->cidx;
  const void* ck = cache->ckv;
  if (pl.dq_idx) {                            // low-precision caches: bf16 copies of the S / ratio entries
    s = run_dequant(cfg, B, 1, cache->cidx, cache->n_cap, S / cfg->ratio, nullptr, carve<char>(ws, pl.off_dq_idx),
                    stream, true);
    if (s != CSA_OK) return s;
    ci = carve<char>(ws, pl.off_dq_idx);
  }
  if (pl.dq_kv) {
    s = run_dequant(cfg, B, 0, cache->ckv, cache->n_cap, S / cfg->ratio, nullptr, carve<char>(ws, pl.off_dq_kv),
                    stream, true);
    if (s != CSA_OK) return s;
    ck = carve<char>(ws, pl.off_dq_kv);
  }
  int32_t* tk = nullptr;
  if (!hca) {
    tk = topk_out ? topk_out : carve<int32_t>(ws, pl.off_topk);
    s = run_index_topk(cfg, B, S, nullptr, q_idx, w, ci, cache->n_cap, tk,
                       carve<float>(ws, pl.off_scores), nullptr, carve<char>(ws, pl.off_tksel),
                       carve<char>(ws, pl.off_tc), stream, true);
    if (s != CSA_OK) return s;
  }
  return run_attn(cfg, pl, B, S, nullptr, q, cache->kv, cache->N, ck, cache->n_cap, tk, sink, out,
                  ws, stream, true);
}

// ---- the exchange over entry-range shards
csa_status csa_index_topk_shard(const csa_config* cfg, int32_t B, const int64_t* pos, const void* q_idx, const float* w,
                                const void* cidx_shard, int64_t n_shard, int64_t entry_base, int32_t* cand_idx,
                                float* cand_score, void* ws, size_t ws_bytes, cudaStream_t stream) {
  csa_status s = check_config(cfg);
  if (s != CSA_OK) return s;
  if (cfg->top_k == 0) return fail(CSA_ERR_INVALID_ARG, "top_k == 0 (HCA) has no indexer");
  if (lowp(cfg)) return fail(CSA_ERR_NOT_IMPLEMENTED, "shard calls read bf16 or float32 caches");
  if (B < 0 || B > 65535 || n_shard < 1 || entry_base < 0)
    return fail(CSA_ERR_SHAPE, "B = %d, n_shard = %lld, entry_base = %lld", B, (long long)n_shard, (long long)entry_base);
  CHECK_PTR(pos); CHECK_PTR(q_idx); CHECK_PTR(w); CHECK_PTR(cidx_shard); CHECK_PTR(cand_idx); CHECK_PTR(cand_score);
  const Plan pl = make_plan(cfg, B, 1, n_shard);
  s = check_ws(pl, ws, ws_bytes);
  if (s != CSA_OK) return s;
  if (B == 0) return CSA_OK;
  float* sc = carve<float>(ws, pl.off_scores);
  s = run_index_topk(cfg, B, 1, pos, q_idx, w, cidx_shard, n_shard, cand_idx, sc, sc, carve<char>(ws, pl.off_tksel),
                     carve<char>(ws, pl.off_tc), stream, false, nullptr, nullptr, entry_base);
  if (s != CSA_OK) return s;
  return cuda_status(launch_stage(ST_TOPK, stream, [&] {
                       return launch_pack_candidates(B, sc, n_shard, cand_idx, cand_score, cfg->top_k, stream, true);
                     }),
                     "candidate pack launch");
}

csa_status csa_topk_merge(const csa_config* cfg, int32_t B, int32_t G, const float* cand_score, const int32_t* cand_idx,
                          const int64_t* entry_base, const int64_t* n_shard, int32_t* topk, int32_t* shard_sel,
                          cudaStream_t stream) {
  csa_status s = check_config(cfg);
  if (s != CSA_OK) return s;
  if (cfg->top_k == 0) return fail(CSA_ERR_INVALID_ARG, "top_k == 0 (HCA) has no selection");
  if (B < 0 || B > 65535 || G < 1 || G > kMaxShards) return fail(CSA_ERR_SHAPE, "B = %d, G = %d (1..%d)", B, G, kMaxShards);
  if ((int64_t)G * cfg->top_k > kMaxMergeCandidates)
    return fail(CSA_ERR_SHAPE, "G * top_k = %d exceeds %d candidates", G * cfg->top_k, kMaxMergeCandidates);
  if (!entry_base || !n_shard) return fail(CSA_ERR_INVALID_ARG, "entry_base / n_shard is NULL");
  CHECK_PTR(cand_score); CHECK_PTR(cand_idx); CHECK_PTR(topk); CHECK_OPT_PTR(shard_sel);
  MergeParams mp;
  memset(&mp, 0, sizeof mp);
  for (int g = 0; g < G; ++g) {
    if (entry_base[g] < 0 || n_shard[g] < 0 || entry_base[g] + n_shard[g] > INT32_MAX)
      return fail(CSA_ERR_SHAPE, "shard %d: entries [%lld, %lld)", g, (long long)entry_base[g],
                  (long long)(entry_base[g] + n_shard[g]));
    for (int h = 0; h < g; ++h)
      if (entry_base[g] < entry_base[h] + n_shard[h] && entry_base[h] < entry_base[g] + n_shard[g])
        return fail(CSA_ERR_SHAPE, "shards %d and %d overlap", h, g);
    mp.base[g] = entry_base[g];
    mp.n_shard[g] = n_shard[g];
  }
  if (B == 0) return CSA_OK;
  mp.score = cand_score; mp.idx = cand_idx; mp.G = G; mp.k = cfg->top_k; mp.topk = topk; mp.shard_sel = shard_sel;
  return cuda_status(launch_stage(ST_TOPK, stream, [&] { return launch_topk_merge(B, mp, stream, false); }),
                     "candidate merge launch");
}

csa_status csa_sparse_attn_shard(const csa_config* cfg, int32_t B, const int64_t* pos, const void* q, const void* kv,
                                 int64_t N, const void* ckv_shard, int64_t n_shard, int64_t entry_base,
                                 const int32_t* sel, int32_t with_window, float* part_o, float* part_ml,
                                 cudaStream_t stream) {
  csa_status s = check_config(cfg);
  if (s != CSA_OK) return s;
  if (lowp(cfg)) return fail(CSA_ERR_NOT_IMPLEMENTED, "shard calls read bf16 or float32 caches");
  if (B < 0 || B > 65535 || N < 1 || n_shard < 1 || entry_base < 0)
    return fail(CSA_ERR_SHAPE, "B = %d, N = %lld, n_shard = %lld", B, (long long)N, (long long)n_shard);
  CHECK_PTR(pos); CHECK_PTR(q); CHECK_PTR(kv); CHECK_PTR(ckv_shard); CHECK_PTR(part_o); CHECK_PTR(part_ml);
  if (cfg->top_k > 0) CHECK_PTR(sel);
  if (B == 0) return CSA_OK;
  AttnParams ap;
  memset(&ap, 0, sizeof ap);
  ap.q = q; ap.kv = kv; ap.ckv = ckv_shard; ap.topk = cfg->top_k > 0 ? sel : nullptr; ap.pos = pos;
  ap.part_o = part_o; ap.part_ml = part_ml; ap.N = N; ap.n_cap = n_shard; ap.entry_base = entry_base; ap.S = 1;
  ap.H = cfg->H; ap.k = cfg->top_k; ap.ratio = cfg->ratio; ap.window = cfg->window; ap.n_split = 1;
  ap.split_len = cfg->window + (cfg->top_k > 0 ? cfg->top_k : (int)n_shard);
  ap.no_window = with_window ? 0 : 1; ap.partial = 1;
  ap.scale = softmax_scale(cfg); ap.rope = make_rope(cfg); ap.err = device_error_word();
  return cuda_status(
      launch_stage(ST_ATTN, stream, [&] { return launch_attn_simt(bf16_io(cfg), B, ap, stream, false); }),
      "shard attention launch");
}

csa_status csa_attn_merge(const csa_config* cfg, int32_t B, int32_t G, const int64_t* pos, const float* part_o,
                          const float* part_ml, const float* sink, void* out, cudaStream_t stream) {
  csa_status s = check_config(cfg);
  if (s != CSA_OK) return s;
  if (B < 0 || B > 65535 || G < 1 || G > 65535) return fail(CSA_ERR_SHAPE, "B = %d, G = %d", B, G);
  CHECK_PTR(pos); CHECK_PTR(part_o); CHECK_PTR(part_ml); CHECK_PTR(sink); CHECK_PTR(out);
  if (B == 0) return CSA_OK;
  AttnParams ap;
  memset(&ap, 0, sizeof ap);
  ap.part_o = const_cast<float*>(part_o); ap.part_ml = const_cast<float*>(part_ml); ap.pos = pos; ap.sink = sink;
  ap.out = out; ap.S = 1; ap.H = cfg->H; ap.n_split = G; ap.rope = make_rope(cfg); ap.err = device_error_word();
  return cuda_status(
      launch_stage(ST_MERGE, stream, [&] { return launch_attn_merge(bf16_io(cfg), B, ap, stream, false); }),
      "partial merge launch");
}

int64_t csa_launch_count(void) { return g_launches.load(); }

csa_status csa_profile_begin(int32_t max_launches) {
  if (max_launches < 0) return fail(CSA_ERR_INVALID_ARG, "max_launches < 0");
  std::lock_guard<std::mutex> lock(g_prof.mu);
  for (auto& r : g_prof.recs) { g_prof.pool.push_back(r.a); g_prof.pool.push_back(r.b); }
  g_prof.recs.clear();
  for (int s = 0; s < ST_COUNT; ++s) g_prof.extra[s] = 0;
  while ((int)g_prof.pool.size() < 2 * max_launches) {
    cudaEvent_t ev;
    if (cudaEventCreate(&ev) != cudaSuccess) return fail(CSA_ERR_CUDA, "cudaEventCreate failed");
    g_prof.pool.push_back(ev);
  }
  g_prof.cap = max_launches;
  g_prof.recs.reserve(max_launches);
  g_prof.on = true;
  return CSA_OK;
}

csa_status csa_profile_end(float* ms, int32_t* launches, int32_t n_stages) {
  std::lock_guard<std::mutex> lock(g_prof.mu);
  g_prof.on = false;
  for (int s = 0; s < n_stages; ++s) {
    if (ms) ms[s] = 0.f;
    if (launches) launches[s] = s < ST_COUNT ? g_prof.extra[s] : 0;
  }
  csa_status st = CSA_OK;
  for (auto& r : g_prof.recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) { st = fail(CSA_ERR_CUDA, "event synchronize failed"); continue; }
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) { st = fail(CSA_ERR_CUDA, "event elapsed failed"); continue; }
    if (r.stage < n_stages) {
      if (ms) ms[r.stage] += t;
      if (launches) launches[r.stage] += 1;
    }
  }
  return st;
}

}  // extern "C"
