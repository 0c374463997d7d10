/*
 * csa.h — C ABI of the compressed-sparse-attention (CSA / HCA) hot path.
 *
 * The operations follow the DeepSeek-V4-Flash attention as described in
 *   [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程" (hs-black.github.io/posts/deepseek-v4-flash)
 *   [LAB41] "Lab tổng hợp DeepSeek-V4.1-Flash — chạy toàn trình 1A → 6B bằng NumPy" (openarchlab.com)
 *   [ATLAS] "LLM Atlas — DeepSeek" (llm-atlas.k1412.top/deepseek), section 19
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every tensor pointer is caller-owned DEVICE memory, dense row-major (last index fastest),
 *    at least 16-byte aligned. Storage tensors (raw kv / gates / keys, caches, q, out) have the
 *    dtype csa_config.storage (float32 or bfloat16); gate biases, indexer weights, sinks and
 *    scores are float32; positions are int64; selected indices are int32.
 *  - No call allocates device memory. Temporary buffers live in the caller's workspace
 *    (ws, ws_bytes), sized by csa_workspace_bytes(); the workspace must not be shared by calls
 *    that may run concurrently.
 *  - Every call only enqueues work on `stream` and returns without synchronising. Arguments are
 *    checked before anything is launched; on an argument error nothing is written and the
 *    status says why (csa_last_error() gives a one-line message for the calling thread).
 *  - A device-side problem detected by a kernel (an index outside the cache, a bounded wait that
 *    ran out) sets a per-device error word instead of trapping; csa_get_device_status() reads it.
 *  - Positions are absolute token indices t. A query at t may read compressed entries
 *    i < (t + 1) / ratio ([FLASH] "压缩条目必须等整组完成后才可见") and raw tokens
 *    max(0, t - window + 1) .. t.
 *  - q and q_idx are passed before RoPE; the library rotates them at t.
 *  - The library looks up the device addresses of its own device variables (the error word, the
 *    scratch of csa_index_topk_static) once per device and keeps them: resetting a device
 *    (cudaDeviceReset) while the library is loaded is not supported.
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = 1,     /* null pointer, negative size, misaligned pointer          */
  CSA_ERR_SHAPE = 2,           /* unsupported or inconsistent shape                         */
  CSA_ERR_DTYPE = 3,           /* unsupported storage dtype                                 */
  CSA_ERR_WORKSPACE = 4,       /* ws_bytes smaller than csa_workspace_bytes()               */
  CSA_ERR_CUDA = 5,            /* a CUDA runtime call or launch failed                      */
  CSA_ERR_DEVICE = 6,          /* a kernel reported a device-side error (see error word)    */
  CSA_ERR_NOT_IMPLEMENTED = 7, /* valid request that this build does not support            */
  CSA_ERR_DEVICE_TIMEOUT = 8   /* a kernel's bounded wait ran out (error word DEVERR 2)     */
} csa_status;

/* Storage of the compressed caches. CSA_FP4 (the low-precision cache of [LAB41] "Lab tổng hợp
 * DeepSeek-V4.1-Flash", section "3 Giải pháp": FP4 E2M1 for the latent, FP8 E4M3 for the RoPE tail):
 * raw rows, q, q_idx and out are bfloat16; ckv and cidx are byte buffers of csa_cache_bytes() bytes
 * per request laid out as below. Of a compressed entry of C dims (C = d or d_idx), the first
 * L = C - d_rope dims are E2M1 codes in blocks of 32 dims that share the scale 2^E (E8M0 byte E + 127,
 * E = floor(log2 max|x|) - 2 clamped to [-127, 127], -127 for an all-zero block; x / 2^E rounded to
 * nearest even, saturated to +-6: the OCP MXFP4 rule), the last d_rope dims are E4M3 codes (rounded
 * to nearest even, saturated to +-448). One request's cache of n_cap entries is three planes:
 *   plane 0, offset 0:                    n_cap x L/2 bytes; byte j of an entry = dims 2j (low
 *                                          nibble) and 2j+1 (high nibble)
 *   plane 1, offset n_cap L/2:            n_cap x d_rope bytes of E4M3 codes
 *   plane 2, offset n_cap (L/2 + d_rope): n_cap x sb bytes, byte k < L/32 = the scale byte of dims
 *                                          32k .. 32k+31, the rest 0; sb = 16 for C = 512, 2 for C = 128
 * and requests follow one another at the stride csa_cache_bytes() (304 bytes per KV entry, 98 per
 * index entry, plus the padding of plane 2 to 16 bytes). The decode calls (S = 1, CSA) read this
 * format inside their kernels when the one-launch indexer and the fused attention apply (see
 * csa_decode); every other call that reads a low-precision cache first expands the entries it
 * reads into bf16 copies in the workspace (csa_workspace_bytes counts them). */
typedef enum { CSA_F32 = 0, CSA_BF16 = 1, CSA_FP4 = 2 } csa_dtype;

/* csa_config.flags */
#define CSA_FLAG_SIMT 1u       /* use the CUDA-core kernels even where a tcgen05 kernel exists */
/* Test hook for the timeout path, never set in production: the one-launch decode indexer (bf16,
 * one query per request) skips its first cache-tile load and gives each of its waits 2 ms instead
 * of 1 s, so the waits run out, the kernel records the timeout in the device error word and
 * returns; the call's selection is then meaningless and csa_sync_status reports
 * CSA_ERR_DEVICE_TIMEOUT. */
#define CSA_FLAG_TEST_STALL (1u << 30)

/* Shape and hyper-parameters of one layer (tensor contract of [FLASH] "每个算子先对齐四个维度").
 * Supported: d = 512, d_rope = 64, d_idx = 128, 1 <= H <= 64, 1 <= H_idx <= 64,
 * 1 <= ratio <= 256, 0 <= top_k <= 2048 (0 = HCA, every visible entry), 1 <= window <= 1024. */
typedef struct {
  int32_t H;             /* query heads                                                  */
  int32_t d;             /* width of the single shared KV head (K = V), 512               */
  int32_t d_rope;        /* rotary tail width, 64 (the last d_rope dims are rotated)       */
  int32_t H_idx;         /* indexer heads                                                */
  int32_t d_idx;         /* indexer width, 128                                            */
  int32_t ratio;         /* compression ratio m (CSA 4, HCA 128)                          */
  int32_t top_k;         /* selected compressed entries per query; 0 = HCA                */
  int32_t window;        /* raw sliding-window length W                                   */
  float rope_base;       /* RoPE base, 10000                                              */
  float softmax_scale;   /* attention logit scale; <= 0 selects 1/sqrt(d)                 */
  float rms_eps;         /* RMSNorm epsilon after pooling, 1e-6                           */
  csa_dtype storage;     /* storage dtype of kv, gates, keys, caches, q, q_idx, out       */
  uint32_t flags;        /* CSA_FLAG_*                                                    */
} csa_config;

/* Raw per-token inputs and compressed caches of B requests.
 *   kv, gate        [B, N, d]        storage   raw shared KV head rows and compressor gate logits
 *   gate_bias       [2*ratio, d]     float32   positional gate bias, index p = j - (i-1)*ratio
 *   idx_k, idx_gate [B, N, d_idx]    storage   raw index keys and their gate logits (NULL for HCA)
 *   idx_bias        [2*ratio, d_idx] float32   (NULL for HCA)
 *   ckv             [B, n_cap, d]    storage   compressed KV cache (entry i rotated at i*ratio)
 *   cidx            [B, n_cap, d_idx] storage  compressed index cache (NULL for HCA)
 * (with CSA_FP4 storage the raw rows are bfloat16 and ckv / cidx are the byte layout of csa_dtype) */
typedef struct {
  const void* kv;
  const void* gate;
  const float* gate_bias;
  const void* idx_k;
  const void* idx_gate;
  const float* idx_bias;
  int64_t N;             /* raw tokens held per request (row stride of kv / gate / idx_*)   */
  void* ckv;
  void* cidx;
  int64_t n_cap;         /* compressed entries held per request (row stride of ckv / cidx) */
} csa_cache;

/* One-line description of a status code (static storage). */
const char* csa_status_string(csa_status s);

/* Message of the last argument error raised in the calling thread ("" if none). */
const char* csa_last_error(void);

/* Reads (and with reset != 0 clears) the device error word of the current device after
 * synchronising `stream`. Returns CSA_OK, CSA_ERR_DEVICE_TIMEOUT (a bounded wait ran out) or
 * CSA_ERR_DEVICE (another device-side error); *code (nullable) receives the raw word (0 = no
 * error, 1 = a selected index outside the visible entries, 2 = a wait ran out, 3 = a position
 * outside the raw capacity). The first error since the last reset is the one kept. */
csa_status csa_get_device_status(cudaStream_t stream, int reset, int32_t* code);

/* Synchronises `stream` and returns the device status as csa_get_device_status(stream, 0, NULL)
 * does, leaving the error word as it is. */
csa_status csa_sync_status(cudaStream_t stream);

/* Bytes of one request's compressed cache of n_cap entries: which = 0 for ckv (d dims), 1 for cidx
 * (d_idx dims). n_cap * C * 4 for float32, * 2 for bf16, the plane layout of csa_dtype for CSA_FP4.
 * Returns 0 for an invalid configuration. */
size_t csa_cache_bytes(const csa_config* cfg, int32_t which, int64_t n_cap);

/* Workspace bytes needed by csa_index_topk / csa_sparse_attn / csa_decode / csa_prefill for
 * B requests, S queries per request and a compressed capacity of n_cap entries. Returns 0 for
 * an invalid configuration. */
size_t csa_workspace_bytes(const csa_config* cfg, int32_t B, int32_t S, int64_t n_cap);

/* Compressor ([FLASH] "压缩是逐通道的 learned pooling", "一个通道，逐项算出压缩结果").
 * Writes entries i in [first_entry, first_entry + n_entries) of every request:
 *   for each channel c, softmax over p in [0, 2m) of gate[j, c] + gate_bias[p, c] with
 *   j = (i-1)m + p (rows j < 0 take weight 0), pooled kv[j, c]; then RMSNorm over the channels
 *   (unit weight, eps = rms_eps); then RoPE of the last d_rope dims at position i*m.
 * The same rule builds cidx from idx_k / idx_gate / idx_bias when those are non-NULL.
 * Requires (first_entry + n_entries) * ratio <= cache->N and first_entry + n_entries <= n_cap. */
csa_status csa_compress(const csa_config* cfg, int32_t B, const csa_cache* cache,
                        int64_t first_entry, int64_t n_entries, cudaStream_t stream);

/* Indexer and selection ([FLASH] "少读 KV 之前，Indexer 仍要给历史打分").
 *   pos     [B, S] int64     query positions t
 *   q_idx   [B, S, H_idx, d_idx] storage (before RoPE; rotated at t inside)
 *   w       [B, S, H_idx] float32 signed head weights
 *   cidx    [B, n_cap, d_idx] storage
 *   topk    [B, S, top_k] int32 out: the top_k visible entries under the order (-s_i, i) with
 *           s_i = sum_h w_h * max(0, rope(q_h, t) . cidx_i) (of equal scores the lower index wins),
 *           written in ascending entry index; when fewer than top_k entries are visible, every
 *           visible entry is taken and the tail holds -1.
 *   scores  [B, S, n_cap] float32 out, nullable: s_i for i < visible(t); other entries untouched.
 * Requires top_k > 0. */
csa_status csa_index_topk(const csa_config* cfg, int32_t B, int32_t S, const int64_t* pos,
                          const void* q_idx, const float* w, const void* cidx, int64_t n_cap,
                          int32_t* topk, float* scores, void* ws, size_t ws_bytes,
                          cudaStream_t stream);

/* Sparse joint attention with sink and inverse RoPE ([FLASH] "局部和压缩记忆，共用一次归一化",
 * "输出投影也分组，并且降低中间维度"; [LAB41] "attn_sink"; HCA: [ATLAS] section 19).
 *   pos   [B, S] int64; q [B, S, H, d] storage (before RoPE)
 *   kv    [B, N, d] raw rows; candidate raw token j is kv[j] rotated at j
 *   ckv   [B, n_cap, d]; topk [B, S, top_k] int32 (-1 = empty slot), or NULL when top_k == 0 (HCA:
 *         every visible entry is a candidate)
 *   sink  [H] float32 per-head sink logit (adds exp(sink_h) to the denominator, owns no value)
 *   out   [B, S, H, d] storage: o_h = sum_c exp(l_hc) e_c / (exp(sink_h) + sum_c exp(l_hc)) with
 *         l_hc = softmax_scale * rope(q_h, t) . e_c, then rotated back by -t.
 * A selected index outside [0, visible(t)) is skipped and flagged in the device error word. */
csa_status csa_sparse_attn(const csa_config* cfg, int32_t B, int32_t S, const int64_t* pos,
                           const void* q, const void* kv, int64_t N, const void* ckv, int64_t n_cap,
                           const int32_t* topk, const float* sink, void* out, void* ws,
                           size_t ws_bytes, cudaStream_t stream);

/* One decode step of B requests, one query each at pos[b] ([FLASH] "压缩条目必须等整组完成后才可见"):
 * the caller has already written token t = pos[b] into the raw rows of `cache`. If t closes a
 * group ((t + 1) % ratio == 0) entry t / ratio of ckv (and cidx) is written before anything reads
 * it (with bf16 storage and top_k > 0 the indexer kernel pools both entries itself, the index
 * entry ahead of the tile that scores it); the indexer, top-k (skipped for HCA) and the sparse
 * attention run for the query at t. Stream order holds as for any call: the first kernel starts
 * after the caller's earlier work on `stream`.
 *   pos   [B] int64 (device); q [B, H, d]; q_idx [B, H_idx, d_idx]; w [B, H_idx] (NULL for HCA)
 *   out   [B, H, d] storage; topk_out [B, top_k] int32, nullable (the selection used). */
csa_status csa_decode(const csa_config* cfg, int32_t B, const int64_t* pos, const csa_cache* cache,
                      const void* q, const void* q_idx, const float* w, const float* sink,
                      void* out, int32_t* topk_out, void* ws, size_t ws_bytes,
                      cudaStream_t stream);

/* Causal prefill of S = cache->N tokens at positions 0 .. S-1 of B requests: every compressed
 * entry 0 .. S/ratio - 1 is built at once, then each query t keeps its own visibility mask
 * ([FLASH] "压缩条目必须等整组完成后才可见": prefill computes all entries in parallel, and each
 * query still applies its causal mask).
 *   q [B, S, H, d]; q_idx [B, S, H_idx, d_idx]; w [B, S, H_idx]; out [B, S, H, d];
 *   topk_out [B, S, top_k] int32, nullable. */
csa_status csa_prefill(const csa_config* cfg, int32_t B, int32_t S, const csa_cache* cache,
                       const void* q, const void* q_idx, const float* w, const float* sink,
                       void* out, int32_t* topk_out, void* ws, size_t ws_bytes,
                       cudaStream_t stream);

/* ---- The exchange over entry-range shards ------------------------------------------------------
 * One long request's compressed caches split by entry range over G shards (in a multi-device
 * deployment, one per device; [FLASH] "少读 KV 之前，Indexer 仍要给历史打分": the selection is made on
 * the combined scores). Shard g holds the entries [entry_base_g, entry_base_g + n_shard_g) of every
 * request at rows 0 .. n_shard_g - 1 of its own caches. The exact global top k is the top k of the
 * union of the shards' local top k (an entry outside its shard's local top k has k entries of its
 * own shard above it), and the attention ("局部和压缩记忆，共用一次归一化") splits into per-shard partials
 * merged with the sink counted once. Between the calls below, a multi-device caller all-gathers the
 * candidates ([B, k] scores and indices per shard) and the partials ([B, H, d] and [B, H, 2] per
 * shard); on one device the shards' outputs are simply laid out side by side. Storage bf16 or
 * float32; one query per request. Every call is asynchronous like the others.
 *
 * csa_index_topk_shard: a shard's candidates: the top_k of its visible entries (visibility of the
 *   query at pos[b], counted in global entries) under (-s, i), as local indices in ascending order
 *   (-1 padded) in cand_idx [B, top_k] int32, and their scores in cand_score [B, top_k] float32 (-inf
 *   for padding). Arguments otherwise as csa_index_topk with S = 1 (q_idx [B, H_idx, d_idx], w
 *   [B, H_idx]); ws of csa_workspace_bytes(cfg, B, 1, n_shard) bytes. */
csa_status csa_index_topk_shard(const csa_config* cfg, int32_t B, const int64_t* pos, const void* q_idx,
                                const float* w, const void* cidx_shard, int64_t n_shard, int64_t entry_base,
                                int32_t* cand_idx, float* cand_score, void* ws, size_t ws_bytes,
                                cudaStream_t stream);

/* csa_topk_merge: the global selection from G shards' candidates (cand_score, cand_idx: [B, G, top_k]
 * device, as csa_index_topk_shard writes them; entry_base, n_shard: [G] HOST arrays of disjoint
 * ranges; 1 <= G <= 8, G * top_k <= 4096): topk [B, top_k] = the top_k of all candidates under
 * (-s, global index), global indices in ascending order, -1 padded (exactly what csa_index_topk
 * selects on the unsharded cache with the same scores); shard_sel [B, G, top_k] (nullable) = each
 * shard's selected entries as its local indices, ascending, -1 padded. */
csa_status csa_topk_merge(const csa_config* cfg, int32_t B, int32_t G, const float* cand_score,
                          const int32_t* cand_idx, const int64_t* entry_base, const int64_t* n_shard,
                          int32_t* topk, int32_t* shard_sel, cudaStream_t stream);

/* csa_sparse_attn_shard: a shard's attention partials for the query at pos[b] over its selected rows
 * sel [B, top_k] (local indices, -1 = empty; ignored for HCA, which takes every visible entry of the
 * shard) and, when with_window != 0, the raw window rows of kv (one shard owns the window):
 *   part_ml [B, H, 2] float32 = (m_h, l_h): m_h the largest logit softmax_scale * rope(q_h, t) . e_c
 *   (-inf when the shard contributes nothing), l_h = sum_c exp(l_hc - m_h);
 *   part_o  [B, H, d] float32 = sum_c exp(l_hc - m_h) e_c (unnormalised, in the rotated frame). */
csa_status csa_sparse_attn_shard(const csa_config* cfg, int32_t B, const int64_t* pos, const void* q,
                                 const void* kv, int64_t N, const void* ckv_shard, int64_t n_shard,
                                 int64_t entry_base, const int32_t* sel, int32_t with_window, float* part_o,
                                 float* part_ml, cudaStream_t stream);

/* csa_attn_merge: out [B, H, d] (storage dtype) from G shards' partials (part_o [B, G, H, d],
 * part_ml [B, G, H, 2], as csa_sparse_attn_shard writes them): with M = max(sink_h, m_g),
 * o = sum_g e^(m_g - M) part_o_g / (e^(sink_h - M) + sum_g e^(m_g - M) l_g), rotated back by -t. */
csa_status csa_attn_merge(const csa_config* cfg, int32_t B, int32_t G, const int64_t* pos, const float* part_o,
                          const float* part_ml, const float* sink, void* out, cudaStream_t stream);

/* ---- For callers that cannot allocate device memory ------------------------------------------
 * The source pages have no counterpart of this call: it is a deployment convenience of the
 * library, computing exactly what csa_index_topk computes.
 *
 * csa_index_topk needs a caller workspace. Some callers have no way to provide one: an engine
 * whose device memory was reserved up front by another allocator has none left to hand out, a
 * latency-critical serving loop must not call cudaMalloc / cudaFree (they can synchronise the
 * device and take unbounded time), and some plugin hosts do not let a library allocate at all.
 * csa_index_topk_static takes the arguments of csa_index_topk minus (ws, ws_bytes) and allocates
 * nothing: its temporary buffers (the float32 scores when `scores` is NULL, the selection, and the
 * candidate lists of rows longer than 16,384 entries) live in one fixed device array of
 * CSA_STATIC_SCRATCH_BYTES inside this library. Every device that loads the library holds that
 * array until the process exits.
 *  - Limit: a request whose temporary buffers exceed CSA_STATIC_SCRATCH_BYTES (about
 *    4 * B * S * n_cap bytes of scores plus the selections) is rejected with CSA_ERR_WORKSPACE
 *    before anything is launched; use csa_index_topk with a workspace for it.
 *  - Set-up: the first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current. Make that first call before any stream
 *    capture begins.
 *  - Sharing: every call uses the same array and leaves its contents there; nothing in it has to
 *    start at zero (a call writes every byte it later reads). Calls that can overlap on the GPU
 *    (other streams, other host threads) race on the array: the caller must serialise them.
 * Arguments, results and other errors are those of csa_index_topk. */
#define CSA_STATIC_SCRATCH_BYTES (8u << 20)
csa_status csa_index_topk_static(const csa_config* cfg, int32_t B, int32_t S, const int64_t* pos,
                                 const void* q_idx, const float* w, const void* cidx, int64_t n_cap,
                                 int32_t* topk, float* scores, cudaStream_t stream);

/* ---- Instrumentation (host side; never changes results) -------------------------------------
 * Stage ids used below: 0 compressor, 1 indexer scores, 2 top-k, 3 sparse attention, 4 split merge. */

/* Number of kernel launches this library has issued in the process so far. */
int64_t csa_launch_count(void);

/* Starts recording a CUDA event pair on the launching stream around each kernel launch of every
 * following call (at most max_launches launches are recorded; later ones are counted only).
 * Not for use while a stream is being captured into a CUDA graph. */
csa_status csa_profile_begin(int32_t max_launches);

/* Stops recording, waits for the recorded events, and writes for each stage s < n_stages the total
 * device milliseconds ms[s] and the launch count launches[s] (either pointer may be NULL). */
csa_status csa_profile_end(float* ms, int32_t* launches, int32_t n_stages);

#ifdef __cplusplus
}
#endif

#endif /* CSA_H_ */
