/*
 * pa.h - paged GQA decode / speculative-verify attention for one GB300 GPU.
 *
 * C ABI of libpa.  Every entry point takes plain pointers and sizes; no C++ or
 * PyTorch type crosses this boundary.  Unless a comment says "host", a pointer
 * is a DEVICE pointer on the current CUDA device.  The caller owns every
 * buffer; the library allocates no device memory, keeps no per-call state
 * (it caches only the SM count of each device it has launched on), never
 * synchronises inside a decode call, and may be called from several host
 * threads at once.  The decode calls are stream-ordered and can be captured
 * in a CUDA graph: every launch parameter is passed by value, so a graph never
 * refers to host memory that a later call could overwrite ("SM70 attention and
 * quantized projection coverage across TP sizes", section "Graph replay and
 * long-prefill follow-up": symbol values as kernel arguments, no captured
 * host stack addresses).
 *
 * Operation (every variant).  For request b < batch, verify query
 * qi < q_len and query head h < num_q_heads, with G = num_q_heads /
 * num_kv_heads, KV head g = h / G and L = ctx_lens[b]:
 *
 *     key j (0 <= j <= L - q_len + qi) lives in page block_table[b][j / page_size],
 *     slot j % page_size;  s_j = (q . k_j) / sqrt(head_dim);
 *     out[b][qi][h] = sum_j softmax(s)_j v_j.
 *
 * The q_len verify queries are the last q_len tokens of the context, so query
 * qi sees one more key than query qi - 1 (causal speculative verify:
 * "DFlash2 concurrent long-context attention", sections "Why the
 * single-request optimization was missing from concurrent decode" and
 * "Matched endpoint gate": q7/q8 verify steps over a paged E4M3 cache).  A row
 * that sees no key (L = 0, a padded slot, or L < q_len - qi) is written as
 * +0.0 in every element and Q for it is never read; a request with L = 0 never
 * reads its block-table row ("padded requests and zero-length rows remain
 * safe", same section).
 *
 * The G query heads x q_len queries that share one KV head are computed as one
 * packed tile, so every KV byte is read once per KV head rather than once per
 * query head ("perf(fa2): port decode GQA group-swap into d128 varlen
 * launcher", vllm.cpp pull request #48, description: KV is read once per
 * group).  Long contexts are cut into splits whose count depends only on that
 * request's length; each split writes FP32 (m, l, O) partials into the
 * request-major workspace and a log-sum-exp merge (the last phase of the same
 * kernel, once every split of the request has arrived) combines them in ascending
 * split order ("DFlash2 concurrent long-context attention", same section:
 * independent request-major workspace panels).  Results therefore do not
 * depend on batch composition: a batched call writes, bit for bit, what one
 * call per request writes ("Operator validation": batched results equal
 * independent single-request execution bitwise).
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_ABI_VERSION 2

/* Return codes.  Every host-detectable problem is reported before any launch;
 * nothing is written to out, lse or workspace in that case. */
typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_NULL = -1,        /* a required pointer (or params/caps struct) is NULL */
  PA_ERR_SHAPE = -2,       /* batch, heads, q_len, page size, pool, lengths or strides out of range */
  PA_ERR_UNSUPPORTED = -3, /* head_dim or GQA geometry this library does not implement */
  PA_ERR_ALIGN = -4,       /* a pointer or stride is not a multiple of 8 bytes (16 for q/out/lse) */
  PA_ERR_WORKSPACE = -5,   /* workspace NULL, not 256-byte aligned, or smaller than *_workspace_bytes() */
  PA_ERR_CUDA = -6         /* a CUDA runtime call or a kernel launch failed */
} pa_status;

/* Bits of the 32-bit status word at the start of the workspace.  Kernels OR
 * them in when a data-dependent check fails; the affected request's rows are
 * then written as zeros instead of reading out of range.  The word is sticky:
 * it keeps its bits across calls until pa_clear_status(). */
#define PA_FLAG_BAD_PAGE 0x1u   /* a block-table entry for a visible key is outside [0, num_pages) */
#define PA_FLAG_BAD_LENGTH 0x2u /* ctx_lens[b] < 0 or ctx_lens[b] > max_ctx_len */
#define PA_FLAG_TIMEOUT 0x4u    /* an internal pipeline wait exceeded its bound; output of that call is invalid */

/* Capabilities of the loaded library (host struct).  A caller compares these
 * with what it is about to pass, so a stale binary is never handed shapes it
 * cannot serve ("DFlash2 concurrent long-context attention", section "Why the
 * single-request optimization was missing from concurrent decode": the loaded
 * extension reports its batch capacity; "SM70 attention and quantized
 * projection coverage across TP sizes", section "Compiled-library precision
 * admission": the library reports its QK/PV accumulation bits, and section
 * "Additional findings": positive 16-aligned page sizes are admitted and
 * advertised by a capability query). */
typedef struct pa_caps {
  int32_t abi_version;   /* PA_ABI_VERSION */
  int32_t max_batch;     /* largest batch (request slots) per call */
  int32_t max_q_len;     /* largest verify window q_len */
  int32_t max_group;     /* largest num_q_heads / num_kv_heads */
  int32_t page_multiple; /* page_size must be a positive multiple of this */
  int32_t max_ctx;       /* largest max_ctx_len */
  int32_t accum_bits;    /* width of the QK and PV accumulators: 32 */
  int32_t fp8_head_dim;  /* head_dim of pa_decode_fp8, pa_decode_e5m2, pa_decode_f16, pa_decode_bf16_d256: 256 */
  int32_t bf16_head_dim; /* head_dim of pa_decode_bf16_d128: 128 */
  int32_t max_splits;    /* most splits one request is cut into (pa_split_plan's *num_splits) */
  int32_t reserved[6];
} pa_caps;

/* Geometry of one call (host struct, read during the call only). */
typedef struct pa_params {
  int32_t batch;             /* request slots B, 1 .. max_batch (padded slots have ctx_lens 0) */
  int32_t num_kv_heads;      /* Hkv >= 1 */
  int32_t num_q_heads;       /* Hq = G * Hkv, 1 <= G <= max_group */
  int32_t head_dim;          /* D: 128 for pa_decode_bf16_d128, 256 for every other decode call */
  int32_t q_len;             /* verify queries per request, 1 .. max_q_len (bf16: 1 .. max_q_len too) */
  int32_t page_size;         /* tokens per page, a positive multiple of page_multiple */
  int32_t max_pages_per_req; /* block_table row length; >= ceil(max_ctx_len / page_size) */
  int32_t num_pages;         /* pages in the pool; valid page ids are 0 .. num_pages-1 */
  int32_t max_ctx_len;       /* host upper bound of every ctx_lens[b]; sizes grid and workspace */
  int32_t reserved0;
  /* byte strides of K and V: element (page p, slot t, kv head g, d) of K is at
   * k_pages + p*k_page_stride + t*k_token_stride + g*k_head_stride + d*elem_bytes,
   * V likewise.  Any layout is accepted (separate K/V tensors [pages, page_size,
   * Hkv, D], or K and V interleaved per token and head) as long as every stride
   * and both base pointers are multiples of 8 bytes; 16-byte multiples select
   * 16-byte vector loads ("DFlash2 concurrent long-context attention",
   * section "Operator validation": interleaved and eight-byte-only aligned KV
   * strides). */
  int64_t k_page_stride, k_token_stride, k_head_stride;
  int64_t v_page_stride, v_token_stride, v_head_stride;
} pa_params;

/* Fills *out (host).  Returns PA_OK or PA_ERR_NULL. */
int pa_get_capabilities(pa_caps* out);

/* Static description of a status code (host string, never NULL). */
const char* pa_status_string(int status);

/* Host copy of the split planner the kernels run on the device: a request of
 * ctx_len keys, read for each of num_kv_heads KV heads, is cut into
 * *num_splits consecutive splits of *chunk keys (the last one shorter).
 * Depends on ctx_len and num_kv_heads (the packed geometry, "perf(fa2): port
 * decode GQA group-swap into d128 varlen launcher", vllm.cpp pull request
 * #48: the split count is chosen on the packed geometry), never on the batch:
 * about 512 * min(num_kv_heads, 4) keys per split, at most max_splits splits,
 * whole 128-key tiles.  ctx_len 0 gives 0 splits.  Returns PA_ERR_NULL or
 * PA_ERR_SHAPE (ctx_len < 0 or num_kv_heads < 1). */
int pa_split_plan(int32_t ctx_len, int32_t num_kv_heads, int32_t* num_splits, int32_t* chunk);

/* ---- FP16 Q x E4M3 K/V, head_dim 256 ---------------------------------------
 *
 * Workspace bytes a pa_decode_fp8 call with this geometry needs (0 when the
 * geometry is invalid).  The workspace holds the status word, per-call
 * counters and flags, and the request-major FP32 split partials.  It must
 * be zero-filled before its first use (for example one cudaMemset after
 * allocation); every call leaves the counters and flags at zero again, so
 * between calls only the status word carries information. */
size_t pa_decode_fp8_workspace_bytes(const pa_params* p);

/* q           FP16 [batch][q_len][num_q_heads][256], contiguous, 16-byte aligned.
 * k_pages     E4M3 bytes, addressed through the strides in *p (8-byte aligned).
 * v_pages     E4M3 bytes, same.
 * block_table int32 [batch][max_pages_per_req]; entries past ceil(L/page_size) are never read.
 * ctx_lens    int32 [batch]; 0 marks an empty or padded slot.
 * k_scale     one FP32 in device memory: a K element is E4M3(byte) * *k_scale.
 * v_scale     one FP32 in device memory: a V element is E4M3(byte) * *v_scale.
 *             (Device pointers, so a captured graph can be replayed with new scales.)
 * out         FP16 [batch][q_len][num_q_heads][256], contiguous, 16-byte aligned; fully written.
 * workspace   device buffer of at least pa_decode_fp8_workspace_bytes(p) bytes, 256-byte aligned,
 *             zero-filled before its first use; two calls in flight at the same time must use
 *             different workspaces.
 * stream      cudaStream_t (NULL = legacy default stream).
 * QK^T and PV run on the tensor cores with FP16 inputs and FP32 accumulation
 * ("SM70 attention and quantized projection coverage across TP sizes", section
 * "Scope": FP16 inputs with FP32 accumulation for both QK and PV).
 * Returns PA_OK after enqueueing the kernels, or a negative pa_status. */
int pa_decode_fp8(const pa_params* p, const void* q, const void* k_pages, const void* v_pages,
                  const int32_t* block_table, const int32_t* ctx_lens, const float* k_scale,
                  const float* v_scale, void* out, void* workspace, size_t workspace_bytes, void* stream);

/* ---- FP16 Q x E4M3 K/V without a caller workspace ---------------------------
 * Same operation, arguments and results as pa_decode_fp8, for callers that
 * cannot allocate device memory: code running under another framework's
 * memory manager, which gives a library no allocator of its own and would
 * see a raw cudaMalloc bypass its pool (and cudaMalloc/cudaFree may
 * synchronise the whole device), or a latency-critical host thread that must
 * not block in the allocator.  The pages describe no such entry point; it is
 * an addition of this library.
 *
 * Scratch memory: a PA_NOALLOC_SCRATCH_BYTES (16 MiB) array in device global
 * memory, declared in the library, which every GPU that loads the library
 * holds until the process exits.  The call allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine).  Geometries whose workspace
 * (pa_decode_fp8_workspace_bytes) exceeds the array are rejected with
 * PA_ERR_WORKSPACE before anything is enqueued (B8 x 131072 keys, GQA 6,
 * q_len 8 needs 12.7 MB and fits).  Every call looks up the array's device
 * address (cudaGetSymbolAddress) in the current context.  The first call on a
 * device is special: under CUDA's lazy module loading it is the lookup that
 * loads the array's module, and the driver commits the 16 MiB at that moment,
 * so that first call can block like an allocation.  Make one warm-up call per
 * device at set-up, before any stream capture and before the latency-critical
 * phase; from the second call on nothing is allocated or loaded.  Every call
 * on a device shares the one array, which keeps the last call's contents;
 * each call clears the status word first, and its kernel returns the
 * per-request flags and counters to zero as it finishes (the array starts at
 * zero), so a bad input flagged by one call does not carry into the next.
 * Calls that overlap on the GPU (different streams, or several host threads)
 * race on the array and give undefined results: serialise them.  The status
 * word is cleared at the start of every call and cannot be read back.
 * Returns PA_OK after enqueueing, or a negative pa_status. */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)
int pa_decode_fp8_noalloc(const pa_params* p, const void* q, const void* k_pages, const void* v_pages,
                          const int32_t* block_table, const int32_t* ctx_lens, const float* k_scale,
                          const float* v_scale, void* out, void* stream);

/* ---- FP16 Q x E5M2 K/V, head_dim 256 ---------------------------------------
 *
 * The same decode for a cache stored as E5M2 (1 sign bit, 5 exponent bits
 * with bias 15, 2 mantissa bits; the OCP 8-bit floating point E5M2 format).
 * E5M2 KV is one of the cache types that keeps its own graph set beside the
 * E4M3 one ("DFlash2 concurrent long-context attention", section "Why the
 * single-request optimization was missing from concurrent decode"), and the
 * E5M2 graphs are checked against an FP64 reference as well ("SM70 attention
 * and quantized projection coverage across TP sizes", section "Additional
 * findings").  Arguments, layouts, alignment, workspace
 * (pa_decode_fp8_workspace_bytes), errors and results are those of
 * pa_decode_fp8, with one difference: a K element is E5M2(byte) * *k_scale
 * and a V element E5M2(byte) * *v_scale.  Codes with an all-ones exponent
 * (infinities and NaNs) are outside the contract: they propagate through the
 * arithmetic and the affected rows are undefined. */
int pa_decode_e5m2(const pa_params* p, const void* q, const void* k_pages, const void* v_pages,
                   const int32_t* block_table, const int32_t* ctx_lens, const float* k_scale,
                   const float* v_scale, void* out, void* workspace, size_t workspace_bytes, void* stream);

/* ---- 16-bit K/V, head_dim 256 ----------------------------------------------
 *
 * The same decode over caches that keep K and V in 16 bits: FP16 Q/K/V
 * (pa_decode_f16; FP16 KV is one of the cache types that keeps its own graph
 * set, "DFlash2 concurrent long-context attention", section "Why the
 * single-request optimization was missing from concurrent decode", and whose
 * graphs "SM70 attention and quantized projection coverage across TP sizes",
 * section "Additional findings", checks against FP64) and BF16 Q/K/V
 * (pa_decode_bf16_d256, the head-dim-256 counterpart of pa_decode_bf16_d128,
 * "perf(fa2): port decode GQA group-swap into d128 varlen launcher", vllm.cpp
 * pull request #48).  Arguments, layouts, alignment, workspace
 * (pa_decode_fp8_workspace_bytes: the workspace depends on head_dim, not on
 * the element type), errors and results are those of pa_decode_fp8 with
 * these differences: K and V elements are 2 bytes (512 bytes per key row),
 * there are no scales, the softmax scale is 1/16, and out is FP16
 * (pa_decode_f16) or BF16 (pa_decode_bf16_d256).  For BF16 the V values are
 * rounded to FP16 for the PV product, as in pa_decode_bf16_d128.
 * lse         (pa_decode_bf16_d256) optional, as in pa_decode_bf16_d128. */
int pa_decode_f16(const pa_params* p, const void* q, const void* k_pages, const void* v_pages,
                  const int32_t* block_table, const int32_t* ctx_lens, void* out, void* workspace,
                  size_t workspace_bytes, void* stream);

int pa_decode_bf16_d256(const pa_params* p, const void* q, const void* k_pages, const void* v_pages,
                        const int32_t* block_table, const int32_t* ctx_lens, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream);

/* ---- BF16 Q/K/V, head_dim 128 ----------------------------------------------
 *
 * The head-dim-128 BF16 decode with group packing ("perf(fa2): port decode GQA
 * group-swap into d128 varlen launcher", vllm.cpp pull request #48,
 * description: the query heads of one KV group are packed together, the grid
 * runs over (batch, kv_heads), and the split count is chosen on the packed
 * geometry).  Same conventions as pa_decode_fp8 with BF16 elements (2 bytes),
 * no scales, and softmax scale 1/sqrt(128).
 * lse         optional (NULL to skip) FP32 [batch][q_len][num_q_heads], 16-byte aligned:
 *             natural-log log-sum-exp of the row's scores, -inf for a row with no key. */
size_t pa_decode_bf16_d128_workspace_bytes(const pa_params* p);

int pa_decode_bf16_d128(const pa_params* p, const void* q, const void* k_pages, const void* v_pages,
                        const int32_t* block_table, const int32_t* ctx_lens, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream);

/* ---- causal prefill, FP16 Q/K/V, head_dim 256 ---------------------------------
 *
 * The long-prefill phase of the same attention ("SM70 attention and quantized
 * projection coverage across TP sizes", sections "Scope" and "Accumulation
 * audit and rejected tuning": Q8192 x KV262144 causal prefill for GQA-6,
 * head_dim 256, FP16 inputs and intermediates, FP32 accumulation of both QK
 * and PV).  For request b, query i < q_len and query head h (KV head
 * h / (num_q_heads / num_kv_heads)), the q_len queries are the last q_len
 * positions of a context of kv_len keys, so query i sees keys
 * 0 .. kv_len - q_len + i:
 *   out[b][i][h] = sum_j exp(s_j - max s) v_j / sum_j exp(s_j - max s),
 *   s_j = q . k_j / 16,  lse[b][i][h] = max s + log(sum_j exp(s_j - max s)).
 * A query that sees no key (kv_len < q_len, i < q_len - kv_len) gets zeros
 * and lse = -inf.  The keys are cut into splits whose length depends on
 * kv_len alone (pa_prefill_plan); each (128-query tile, split) is computed
 * with P = exp(s - m) rounded to FP16 before the PV product, and the splits
 * are merged in ascending order, so every output row's bits are independent
 * of batch and of num_q_heads / num_kv_heads. */
typedef struct pa_prefill_params {
  int32_t batch;        /* requests, 1 .. 64 */
  int32_t q_len;        /* queries per request, 1 .. 65536 */
  int32_t kv_len;       /* keys per request, 1 .. 4194304 */
  int32_t num_q_heads;  /* Hq, a multiple of num_kv_heads, at most 256 */
  int32_t num_kv_heads; /* Hkv >= 1 */
  int32_t head_dim;     /* 256 */
  /* element strides of K and V: element (b, key t, kv head g, d) of K is at
   * k + b*k_batch_stride + t*k_token_stride + g*k_head_stride + d (FP16
   * elements); V likewise.  Every stride a positive multiple of 8 elements
   * (16 bytes) or, for an extent of 1 (batch 1, one KV head), any value. */
  int64_t k_batch_stride, k_token_stride, k_head_stride;
  int64_t v_batch_stride, v_token_stride, v_head_stride;
} pa_prefill_params;

/* Key split of the prefill for kv_len keys: *num_splits splits of *split_len
 * keys (the last one shorter): split_len = 32768 above 32768 keys, else
 * kv_len / 8 rounded up to a multiple of 128 and at least 1024.  Returns
 * PA_ERR_NULL or PA_ERR_SHAPE (kv_len < 1). */
int pa_prefill_plan(int32_t kv_len, int32_t* num_splits, int32_t* split_len);

/* Workspace bytes a pa_prefill_f16 call with this geometry needs (0 when the
 * geometry is invalid): the status word and the FP32 split partials. */
size_t pa_prefill_f16_workspace_bytes(const pa_prefill_params* p);

/* q         FP16 [batch][q_len][num_q_heads][256], contiguous, 16-byte aligned.
 * k, v      FP16, addressed through the strides in *p, 16-byte aligned.
 * out       FP16 [batch][q_len][num_q_heads][256], contiguous, 16-byte aligned; fully written.
 * lse       nullable FP32 [batch][q_len][num_q_heads] (natural log).
 * workspace device buffer of at least pa_prefill_f16_workspace_bytes(p) bytes,
 *           256-byte aligned, status word zero; two calls in flight at the
 *           same time must use different workspaces.
 * stream    cudaStream_t (NULL = legacy default stream).
 * Two kernels run on the stream: the tcgen05 attention kernel over (tile,
 * split) work items, then the merge of the split partials.  A pipeline wait
 * that exceeds its bound sets PA_FLAG_TIMEOUT in the workspace's status word
 * (pa_read_status).  Returns PA_OK after enqueueing, or a negative pa_status
 * (PA_ERR_UNSUPPORTED for head_dim != 256). */
int pa_prefill_f16(const pa_prefill_params* p, const void* q, const void* k, const void* v, void* out, float* lse,
                   void* workspace, size_t workspace_bytes, void* stream);

/* ---- workspace bank ---------------------------------------------------------
 *
 * A host object that hands out decode workspaces ("panels") so that CUDA
 * graphs can be captured for several batch sizes without one workspace per
 * graph ("DFlash2 concurrent long-context attention", section "Why the
 * single-request optimization was missing from concurrent decode":
 * workspaces are shared across compatible batch sizes on the same device,
 * stream and context contract; descending capture allocates the largest
 * panel once; when a call grows the bank, older panels stay alive because
 * earlier graphs can still reference them; different streams never share a
 * panel; section "Operator validation": growing the bank preserves every
 * pointer handed out before).
 *
 * Key of a panel: (device, stream, head_dim, num_kv_heads, num_q_heads,
 * q_len, max_ctx_len).  pa_bank_workspace returns the key's current panel
 * when it is large enough for *p (any batch up to the one it was made for),
 * otherwise it obtains a panel of exactly the needed size from the caller's
 * allocator, makes it the key's current panel and keeps the older ones.  No
 * panel is released before pa_bank_destroy.  The bank itself allocates no
 * device memory, makes no CUDA call and is safe to use from several host
 * threads; `device` and `stream` are only compared, never used.
 *
 * pa_bank_alloc_fn  returns `bytes` bytes of ZERO-FILLED device memory on
 *                   `device`, 256-byte aligned (a decode workspace must be
 *                   zero before its first use), or NULL.  Called with the bank's
 *                   lock held: it must not call back into the bank.
 * pa_bank_free_fn   returns a panel to the caller (NULL: the caller keeps
 *                   ownership of every panel). */
typedef struct pa_bank pa_bank;
typedef void* (*pa_bank_alloc_fn)(size_t bytes, int32_t device, void* user);
typedef void (*pa_bank_free_fn)(void* ptr, size_t bytes, int32_t device, void* user);

/* New empty bank (host), or NULL when alloc is NULL or host memory runs out. */
pa_bank* pa_bank_create(pa_bank_alloc_fn alloc, pa_bank_free_fn release, void* user);

/* Workspace for a decode call with geometry *p (head_dim 256: pa_decode_fp8 /
 * pa_decode_e5m2; 128: pa_decode_bf16_d128) on `device` and `stream`:
 * *workspace and *workspace_bytes (host outputs) are the panel to pass to the
 * decode call.  Returns PA_OK; PA_ERR_NULL; PA_ERR_SHAPE (device < 0 or a
 * geometry the decode calls reject); PA_ERR_UNSUPPORTED (head_dim);
 * PA_ERR_WORKSPACE (the allocator returned NULL); PA_ERR_ALIGN (the allocator
 * returned memory that is not 256-byte aligned; it is handed back through
 * pa_bank_free_fn). */
int pa_bank_workspace(pa_bank* bank, const pa_params* p, int32_t device, void* stream, void** workspace,
                      size_t* workspace_bytes);

/* Number of panels the bank holds and their total bytes (host outputs). */
int pa_bank_stats(pa_bank* bank, int64_t* panels, int64_t* bytes);

/* Releases every panel through pa_bank_free_fn and frees the bank.  No decode
 * call or graph that uses one of its panels may run afterwards. */
int pa_bank_destroy(pa_bank* bank);

/* ---- status word ------------------------------------------------------------
 * pa_read_status synchronises `stream`, then copies the status word of
 * `workspace` to *flags (host).  pa_clear_status enqueues a reset of it. */
int pa_read_status(const void* workspace, uint32_t* flags, void* stream);
int pa_clear_status(void* workspace, void* stream);

/* ---- bookkeeping checks -------------------------------------------------------
 * pa_debug_worklist runs the kernels' own device-side split planner over
 * ctx_lens and writes, for every work item the split kernel would execute,
 * one int4 {request, kv_head, key_begin, key_end} into items (device,
 * capacity max_items) in the order the persistent CTAs take them, and the
 * item count into *count (device int32).  Returns PA_ERR_SHAPE if max_items
 * is too small for max_ctx_len.
 *
 * pa_debug_gather_fp8 reads, through the kernels' own block-table addressing,
 * the K (which = 0) or V (which = 1) bytes of every visible key of request b
 * and KV head g, and writes them densely as dst[b][g][j][256] (device,
 * [batch][num_kv_heads][max_ctx_len][256] bytes); slots past ctx_lens[b] are
 * left untouched. */
int pa_debug_worklist(const pa_params* p, const int32_t* ctx_lens, int32_t* items, int32_t max_items,
                      int32_t* count, void* stream);
int pa_debug_gather_fp8(const pa_params* p, const void* k_pages, const void* v_pages,
                        const int32_t* block_table, const int32_t* ctx_lens, int32_t which, void* dst,
                        void* stream);

/* pa_debug_kv_load_path writes to *path how a decode call with this geometry
 * and these K/V base pointers moves K and V rows into shared memory:
 *   1  TMA boxes: both bases and every stride 16-byte aligned;
 *   2  TMA windows: both bases 8 bytes past a 16-byte boundary and every
 *      stride a multiple of 16 (each key's 256 row bytes of a fill arrive in a
 *      272-byte window that starts 8 bytes before them);
 *   0  8-byte cp.async copies: any other 8-byte aligned layout, or a layout
 *      whose tensor maps the CUDA driver refused to encode.
 * head_dim is 128 or 256, elem_bytes the K/V element size (1 for E4M3/E5M2,
 * 2 for FP16/BF16).  Nothing is launched; the pointers are not dereferenced.
 * Returns PA_ERR_NULL, PA_ERR_SHAPE, PA_ERR_UNSUPPORTED (head_dim or
 * elem_bytes) or PA_ERR_ALIGN (a base or stride not a multiple of 8). */
int pa_debug_kv_load_path(const pa_params* p, int32_t head_dim, int32_t elem_bytes, const void* k_pages,
                          const void* v_pages, int32_t* path);

/* ---- wait-bound check --------------------------------------------------------
 * Test hook for the kernels' bounded waits.  The next pa_decode_* call made in
 * this process (by any thread) runs its split kernel with every pipeline wait
 * bounded by wait_limit_cycles SM cycles and never signals that its Q tile is
 * ready, so the tensor-core issuer's wait runs out: every CTA abandons its
 * work, frees its tensor memory, sets PA_FLAG_TIMEOUT in the status word and
 * exits; the output of that call is invalid and the CUDA context stays usable.
 * Returns PA_ERR_SHAPE if wait_limit_cycles <= 0. */
int pa_debug_stall_next(int64_t wait_limit_cycles);

/* ---- kernel timing ------------------------------------------------------------
 * pa_timing_enable(1) makes every later decode or prefill call record CUDA
 * events around its attention kernel (on the call's stream; a decode call is
 * one kernel: split-KV attention followed by the log-sum-exp merge of the
 * split partials).
 * pa_timing_collect synchronises those events and returns, for kernel 0 (the
 * decode kernel) or kernel 1 (the attention kernel of pa_prefill_f16, without
 * its merge), the summed device time in milliseconds and the number of
 * launches timed since the previous collect, then resets them.  Recording
 * stops while disabled.  At most 4096 launches per kernel are kept. */
int pa_timing_enable(int on);
int pa_timing_collect(int kernel, double* total_ms, int64_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
