/*
 * bia.h - batch-invariant paged-KV grouped-query attention for one GB300
 * (sm_103a).  C ABI of libbia.so.
 *
 * The operation is the paged-KV prefill / decode attention that the pages
 * describe as FlashInfer's BatchPrefillWithPagedKVCacheWrapper and decode
 * wrapper run with a fixed split-KV tile ("sglang PR #43612", Summary;
 * "sglang PR #10417 [POC] Support deterministic inference", Modifications:
 * paged prefill for every prefill, split-KV fixed to 2048 for decode and
 * 4096 for prefill).  A request's output bits depend only on its own
 * q/k/v values and lengths, head_dim, the GQA group size and the split size:
 * never on the batch it is in, the order of that batch, the physical pages
 * it occupies, the number of SMs or the launch grid, or where a chunk
 * boundary falls ("sglang PR #43612", Summary: chunked prefill must
 * reproduce the unchunked one when chunks start on the 128-row q-tile grid,
 * 128 / gqa_group tokens; this library also reproduces it off that grid
 * unless an off-grid chunk leaves a q tile holding a single token, which is
 * computed by the streaming path; callers may only rely on the grid).
 *
 * Layouts (all row-major, all device pointers unless named *_host):
 *   q        [total_q, num_qo_heads, head_dim] bf16 (decode: [batch, ...])
 *   k_cache  [num_pages, page_size, num_kv_heads, head_dim] bf16
 *   v_cache  same as k_cache
 *   out      [total_q, num_qo_heads, head_dim] bf16
 *   lse      [total_q, num_qo_heads] fp32, natural log; may be NULL
 *   qo_indptr [batch+1] int32: request b owns q tokens
 *            qo_indptr[b] .. qo_indptr[b+1]-1 (qo_indptr[0] == 0)
 *   kv_indptr [batch+1] int32: request b owns pages
 *            kv_indices[kv_indptr[b] .. kv_indptr[b+1]-1], in key order
 *   kv_last_page_len [batch] int32 in 1..page_size (ignored for a request
 *            that owns no page)
 * Request b has kv_len = (n_pages-1)*page_size + kv_last_page_len[b] keys;
 * key j sits at page kv_indices[kv_indptr[b] + j/page_size], slot
 * j % page_size.  Its q tokens are the LAST q_len positions of the sequence:
 * in-call token t is at absolute position kv_len - q_len + t, and a causal
 * row sees keys 0..that position.  q head h reads kv head
 * h / (num_qo_heads / num_kv_heads).  sm_scale <= 0 selects 1/sqrt(head_dim).
 *
 * Ownership: the caller owns every buffer and the stream; the library never
 * allocates device memory and never synchronises the stream.  Every device
 * pointer must be device memory (cudaMalloc or a pool carved from it) of the
 * current device: the prefill kernels multicast each gathered K/V row into
 * the CTAs of a thread-block cluster, which this library does for this GPU's
 * own memory only, so a host, managed or peer-mapped pointer is refused with
 * BIA_ERR_INVALID_ARG (bia_last_error names it) before anything is enqueued.
 * The *_host
 * arrays are read synchronously during the call (to validate and to size the
 * launch) and must equal their device copies.  All work is enqueued on
 * `stream` (a cudaStream_t; NULL = legacy default stream) on the current
 * device, with one exception that keeps the same ordering: a prefill call
 * with both tensor-core q tiles and streamed single-token tiles runs the
 * streamed tiles on a library-owned stream (one per host thread and device,
 * created on first use and never destroyed) that waits for the call's plan
 * on `stream`, and `stream` waits for it before the merge, so everything the
 * call does comes after the work already on `stream` and before the work
 * enqueued there next.  During a graph capture of `stream` the fork is
 * captured with the call (if that thread's side stream does not exist yet,
 * the call stays on `stream`).  A process drives one GPU: each kernel's shared-memory limit is
 * raised on its first launch, for the device current then, and a later
 * launch on another device fails with BIA_ERR_CUDA (one process per GPU is
 * the intended deployment).
 *
 * Errors: every entry point returns BIA_OK or a negative bia_status and never
 * aborts.  Host-side checks run before anything is enqueued.  A page index
 * outside [0, num_pages) is caught on the device: the row is read as zeros and
 * bit 0 of the workspace status word is set (bia_read_status).  The device
 * planner also checks the device index arrays (lengths, page counts, and the
 * bounds of a bounded call); when a check fails it computes nothing, fills
 * out and lse with NaN (so the failure shows in the data, also under graph
 * replay) and sets bit 1 of the status word.
 *
 * Alignment: q, out, the caches and every bf16 row buffer start on a 16-byte
 * boundary; int32 and fp32 arrays on 4 bytes, int64 arrays on 8; a call
 * given a pointer off its boundary returns BIA_ERR_INVALID_ARG.
 *
 * Supported: head_dim 64, 96, 128 or 256 (96 runs zero-padded on the 128
 * kernels);
 * num_qo_heads / num_kv_heads in {1,2,4,8};
 * page_size a power of two in 1..256; split sizes positive multiples of 128.
 */
#ifndef BIA_H
#define BIA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define BIA_API __attribute__((visibility("default")))
#else
#define BIA_API
#endif

/* Rows of one prefill q tile: (token, q head of the group) pairs, GQA-packed
 * ("sglang PR #43612", Summary: the 128-row q-tile grid). */
#define BIA_Q_TILE_ROWS 128
/* Default fixed split-KV sizes ("sglang PR #10417", Modifications). */
#define BIA_PREFILL_SPLIT 4096
#define BIA_DECODE_SPLIT 2048

typedef enum bia_status {
    BIA_OK = 0,
    BIA_ERR_INVALID_ARG = -1,         /* null pointer, bad indptr, q_len > kv_len (causal) ... */
    BIA_ERR_UNSUPPORTED = -2,         /* head_dim, GQA group, page size or split not supported */
    BIA_ERR_WORKSPACE_TOO_SMALL = -3, /* workspace_bytes below the *_workspace_size answer */
    BIA_ERR_CUDA = -4                 /* a CUDA call or launch failed */
} bia_status;

typedef struct bia_attn_desc {
    int32_t num_qo_heads;
    int32_t num_kv_heads;
    int32_t head_dim;  /* 64, 96 or 128 */
    int32_t page_size; /* power of two, 1..256 */
    float sm_scale;    /* <= 0: 1/sqrt(head_dim) */
} bia_attn_desc;

/*
 * Causal (or full) prefill / chunked-prefill extend of a batch of requests
 * against the paged KV cache.  Rows are processed in 128-row q tiles
 * (128/G tokens x G heads of one kv head), keys in 128-key blocks anchored at
 * absolute key 0, and each row's keys in fixed split-KV tiles of split_size
 * keys (also anchored at key 0); a row's split partials are merged in
 * ascending split order by log-sum-exp ("sglang PR #10417", Modifications;
 * "sglang PR #43612", Summary).
 *   causal:     1 = causal extend, 0 = every row sees all kv_len keys
 *   split_size: keys per split-KV tile, multiple of 128; 0 = BIA_PREFILL_SPLIT
 *   workspace:  >= bia_prefill_workspace_size(...) bytes, 256-byte aligned;
 *               its contents on entry do not matter
 *   out / lse:  written for every q row (lse may be NULL)
 */
BIA_API int bia_prefill_paged(const bia_attn_desc *desc, const void *q, const void *k_cache,
                      const void *v_cache, int64_t num_pages, const int32_t *qo_indptr,
                      const int32_t *kv_indptr, const int32_t *kv_indices,
                      const int32_t *kv_last_page_len, const int32_t *qo_indptr_host,
                      const int32_t *kv_indptr_host, const int32_t *kv_last_page_len_host,
                      int32_t batch, int32_t causal, int32_t split_size, void *workspace,
                      size_t workspace_bytes, void *out, float *lse, void *stream);

/*
 * bia_prefill_paged with a custom attention mask: key j is visible to in-call
 * token t of request b only if bit mask_indptr[b] + t*kv_len(b) + j of the
 * mask is 1 (and, when causal, also j <= the token's position).  The mask is a
 * little-endian bit string (bit k = (byte k/8 >> k%8) & 1), like the packed
 * per-request [q_len, kv_len] masks of paged prefill wrappers; the pages name
 * no custom mask, so this is the next-row extension of the same extend path
 * ("sglang PR #43612", Summary: BatchPrefillWithPagedKVCacheWrapper).
 *   mask:        device, 4-byte aligned, mask_bytes long; every request's
 *                q_len*kv_len bits must lie in its first mask_bytes/4 words
 *   mask_indptr: device int64 [batch+1] bit offsets (mask_indptr_host: the
 *                host mirror, validated)
 * A row that the mask leaves without keys gets out 0 and lse -inf.  The
 * workspace is bia_prefill_workspace_size's.  Results for a request depend on
 * its own mask bits, never on the batch.
 */
BIA_API int bia_prefill_paged_mask(const bia_attn_desc *desc, const void *q, const void *k_cache,
                           const void *v_cache, int64_t num_pages, const int32_t *qo_indptr,
                           const int32_t *kv_indptr, const int32_t *kv_indices,
                           const int32_t *kv_last_page_len, const int32_t *qo_indptr_host,
                           const int32_t *kv_indptr_host, const int32_t *kv_last_page_len_host,
                           int32_t batch, int32_t causal, int32_t split_size,
                           const void *mask, size_t mask_bytes, const int64_t *mask_indptr,
                           const int64_t *mask_indptr_host, void *workspace,
                           size_t workspace_bytes, void *out, float *lse, void *stream);

/* Workspace bytes bia_prefill_paged needs for this call (0 on invalid input). */
BIA_API size_t bia_prefill_workspace_size(const bia_attn_desc *desc, const int32_t *qo_indptr_host,
                                  const int32_t *kv_indptr_host,
                                  const int32_t *kv_last_page_len_host, int32_t batch,
                                  int32_t causal, int32_t split_size);

/*
 * Decode: one query token per request (q [batch, Hq, D]) against its whole
 * paged context, in fixed split-KV tiles of split_size keys (0 =
 * BIA_DECODE_SPLIT) whose partials are merged in ascending order
 * ("sglang PR #10417", Modifications: split-KV fixed to 2048 for decode).
 * Every request must own at least one key.
 */
BIA_API int bia_decode_paged(const bia_attn_desc *desc, const void *q, const void *k_cache,
                     const void *v_cache, int64_t num_pages, const int32_t *kv_indptr,
                     const int32_t *kv_indices, const int32_t *kv_last_page_len,
                     const int32_t *kv_indptr_host, const int32_t *kv_last_page_len_host,
                     int32_t batch, int32_t split_size, void *workspace, size_t workspace_bytes,
                     void *out, float *lse, void *stream);

/* Workspace bytes bia_decode_paged needs for this call (0 on invalid input). */
BIA_API size_t bia_decode_workspace_size(const bia_attn_desc *desc, const int32_t *kv_indptr_host,
                                 const int32_t *kv_last_page_len_host, int32_t batch,
                                 int32_t split_size);

/*
 * Bounded calls: a prefill or decode whose launch is sized from upper bounds
 * instead of the host mirrors, so that one captured CUDA graph replays across
 * serving steps while the lengths and page tables in the device arrays change
 * (each decode step adds a key; each chunk of a chunked prefill adds its
 * tokens).  The pages keep split-KV under CUDA graphs only by turning it off
 * during capture and replay ("sglang PR #10417 [POC] Support deterministic
 * inference", Modifications); here the fixed split tiles stay: the device
 * planner lays out the units the actual lengths need in the same order as the
 * exact call and retires the rest, so a bounded call's out and lse bits equal
 * those of bia_prefill_paged / bia_decode_paged on the same inputs.  Nothing
 * is read from the host: the index arrays are read only on the device, and a
 * request beyond the bounds (or malformed arrays) sets status bit 1 and
 * computes nothing.  The price is a launch sized for the bounds (retired
 * units exit at once) and a workspace sized for them.
 */
typedef struct bia_bounds {
    int32_t max_q_len;   /* q tokens of any one request (prefill; decode ignores it) */
    int32_t max_kv_len;  /* keys of any one request, >= 1 for decode */
    int64_t max_total_q; /* q tokens of the whole call (prefill; decode ignores it):
                            q, out and lse must hold this many token rows */
} bia_bounds;

/*
 * bia_prefill_paged sized from `bounds` (see above): request b's lengths come
 * from qo_indptr / kv_indptr / kv_last_page_len on the device only, within
 * max_q_len, max_kv_len and qo_indptr[batch] <= max_total_q; kv_indices must
 * hold kv_indptr[batch] entries.  The workspace is
 * bia_prefill_bounded_workspace_size's; everything else as for
 * bia_prefill_paged.
 */
BIA_API int bia_prefill_paged_bounded(const bia_attn_desc *desc, const bia_bounds *bounds,
                                      const void *q, const void *k_cache, const void *v_cache,
                                      int64_t num_pages, const int32_t *qo_indptr,
                                      const int32_t *kv_indptr, const int32_t *kv_indices,
                                      const int32_t *kv_last_page_len, int32_t batch,
                                      int32_t causal, int32_t split_size, void *workspace,
                                      size_t workspace_bytes, void *out, float *lse,
                                      void *stream);

/* Workspace bytes of every bounded prefill of `batch` requests within
 * `bounds` (0 on invalid input). */
BIA_API size_t bia_prefill_bounded_workspace_size(const bia_attn_desc *desc,
                                                  const bia_bounds *bounds, int32_t batch,
                                                  int32_t causal, int32_t split_size);

/*
 * bia_decode_paged sized from `bounds` (max_kv_len; see above): every request
 * owns 1 .. max_kv_len keys, read from the device arrays only.  The workspace
 * is bia_decode_bounded_workspace_size's.
 */
BIA_API int bia_decode_paged_bounded(const bia_attn_desc *desc, const bia_bounds *bounds,
                                     const void *q, const void *k_cache, const void *v_cache,
                                     int64_t num_pages, const int32_t *kv_indptr,
                                     const int32_t *kv_indices, const int32_t *kv_last_page_len,
                                     int32_t batch, int32_t split_size, void *workspace,
                                     size_t workspace_bytes, void *out, float *lse,
                                     void *stream);

/* Workspace bytes of every bounded decode of `batch` requests within
 * `bounds` (0 on invalid input). */
BIA_API size_t bia_decode_bounded_workspace_size(const bia_attn_desc *desc,
                                                 const bia_bounds *bounds, int32_t batch,
                                                 int32_t split_size);

/* Size of the library-owned scratch array behind bia_decode_paged_noalloc. */
#define BIA_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * bia_decode_paged without a workspace argument, for callers that cannot
 * allocate device memory: plugin / extension hooks of inference engines whose
 * enqueue step may not call cudaMalloc (it can synchronise the device, break
 * a CUDA-graph capture in progress or exceed a memory budget fixed up front),
 * and hosts that account for all device memory before serving.  There is no
 * counterpart on the pages; it is a packaging of the same decode path.
 *
 * Arguments, layouts and results are those of bia_decode_paged.  The scratch
 * space lives in a statically sized __device__ array of
 * BIA_DECODE_NOALLOC_SCRATCH_BYTES that every GPU loading this library holds
 * until the process exits; a call whose bia_decode_workspace_size exceeds it
 * returns BIA_ERR_WORKSPACE_TOO_SMALL without enqueuing anything.  Nothing is
 * allocated (no cudaMalloc / cudaFree).  The first call on each device looks
 * up the array's device address with that device current and keeps it for
 * the life of the process; make that first call before any stream capture,
 * and do not call this entry point after a cudaDeviceReset (the kept address
 * would be stale).  All calls share the one array, which keeps the previous
 * call's contents (every call rewrites what it reads), so calls whose work
 * overlaps on the GPU - different streams, or different host threads - race
 * and must be serialised by the caller.  The device status word (bad page
 * indices, a failed device plan) lives in that array, whose address the
 * caller never sees, so it cannot be read with bia_read_status: a caller that
 * needs those checks uses bia_decode_paged.
 */
BIA_API int bia_decode_paged_noalloc(const bia_attn_desc *desc, const void *q, const void *k_cache,
                             const void *v_cache, int64_t num_pages, const int32_t *kv_indptr,
                             const int32_t *kv_indices, const int32_t *kv_last_page_len,
                             const int32_t *kv_indptr_host, const int32_t *kv_last_page_len_host,
                             int32_t batch, int32_t split_size, void *out, float *lse,
                             void *stream);

/* Multi-head latent attention: the latent (value) width and its rope width. */
#define BIA_MLA_CKV_DIM 512
#define BIA_MLA_KPE_DIM 64

typedef struct bia_mla_desc {
    int32_t num_heads; /* q heads; a multiple of 8 */
    int32_t page_size; /* power of two, 1..256 */
    float sm_scale;    /* <= 0: 1/sqrt(512 + 64) */
} bia_mla_desc;

/*
 * Batch-invariant multi-head latent attention (MLA) decode over a paged latent
 * cache: the paged MLA wrapper the pages name, which has no deterministic mode
 * there ("sglang PR #43612", Summary), with the decode path's fixed split-KV
 * tiles and ascending merge ("sglang PR #10417", Modifications).  Every q head
 * attends to the one shared latent cache:
 *   s_j = sm_scale * (<q_nope, ckv_j> + <q_pe, kpe_j>),
 *   out = sum_j softmax(s)_j * ckv_j,  lse = natural-log LSE of s.
 *   q_nope    [batch, num_heads, 512] bf16, q_pe [batch, num_heads, 64] bf16
 *   ckv_cache [num_pages, page_size, 512] bf16, kpe_cache [num_pages, page_size, 64]
 *   out       [batch, num_heads, 512] bf16, lse [batch, num_heads] fp32 or NULL
 * The page table, split_size (0 = BIA_DECODE_SPLIT), workspace, ownership and
 * error rules are those of bia_decode_paged; every request owns at least one
 * key.  batch * num_heads and num_pages * page_size must stay below 2^31
 * (else BIA_ERR_UNSUPPORTED).  Outputs of a request never depend on the batch.
 */
BIA_API int bia_mla_decode_paged(const bia_mla_desc *desc, const void *q_nope, const void *q_pe,
                         const void *ckv_cache, const void *kpe_cache, int64_t num_pages,
                         const int32_t *kv_indptr, const int32_t *kv_indices,
                         const int32_t *kv_last_page_len, const int32_t *kv_indptr_host,
                         const int32_t *kv_last_page_len_host, int32_t batch, int32_t split_size,
                         void *workspace, size_t workspace_bytes, void *out, float *lse,
                         void *stream);

/* Workspace bytes bia_mla_decode_paged needs for this call (0 on invalid input). */
BIA_API size_t bia_mla_decode_workspace_size(const bia_mla_desc *desc,
                                     const int32_t *kv_indptr_host,
                                     const int32_t *kv_last_page_len_host, int32_t batch,
                                     int32_t split_size);

/*
 * Causal MLA extend (chunked prefill) over the same paged latent cache: the
 * MLA counterpart of bia_prefill_paged, which the pages leave open ("sglang
 * PR #43612", Summary: the flashinfer MLA path has no deterministic mode).
 * Request b's q tokens are the last q_len = qo_indptr[b+1] - qo_indptr[b]
 * positions of its kv_len keys (the rule of bia_prefill_paged); in-call token
 * t sees keys 0 .. kv_len - q_len + t.
 *   q_nope [total_q, num_heads, 512] bf16, q_pe [total_q, num_heads, 64] bf16
 *   out    [total_q, num_heads, 512] bf16, lse [total_q, num_heads] fp32 or NULL
 *   split_size: keys per split-KV tile, a multiple of 128; 0 = BIA_PREFILL_SPLIT
 * Each q token is computed as its own query against its own keys (the decode
 * kernel's fixed split tiles and ascending merge; with 8 or 16 heads, 32 /
 * num_heads consecutive tokens share a CTA and each key block it reads, every
 * token in its own MMA columns), so its bits depend only on
 * its request's keys up to its position and on split_size: the same in any
 * batch and under any chunking of the extend, on the q-tile grid or off it;
 * with equal split_size a token's bits equal those of bia_mla_decode_paged
 * for that position.  A request may have q_len = 0.  total_q * num_heads and
 * num_pages * page_size must stay below 2^31 (else BIA_ERR_UNSUPPORTED).
 * Arguments, ownership and errors otherwise as for bia_prefill_paged
 * (causal only).  The keys are read once per q token (once per group of
 * 32 / num_heads tokens with 8 or 16 heads): this path suits short extends
 * (speculative tokens, small chunks), not long prompts.
 */
BIA_API int bia_mla_prefill_paged(const bia_mla_desc *desc, const void *q_nope, const void *q_pe,
                          const void *ckv_cache, const void *kpe_cache, int64_t num_pages,
                          const int32_t *qo_indptr, const int32_t *kv_indptr,
                          const int32_t *kv_indices, const int32_t *kv_last_page_len,
                          const int32_t *qo_indptr_host, const int32_t *kv_indptr_host,
                          const int32_t *kv_last_page_len_host, int32_t batch, int32_t split_size,
                          void *workspace, size_t workspace_bytes, void *out, float *lse,
                          void *stream);

/* Workspace bytes bia_mla_prefill_paged needs for this call (0 on invalid input). */
BIA_API size_t bia_mla_prefill_workspace_size(const bia_mla_desc *desc,
                                      const int32_t *qo_indptr_host,
                                      const int32_t *kv_indptr_host,
                                      const int32_t *kv_last_page_len_host, int32_t batch,
                                      int32_t split_size);

/*
 * Fixed-order log-sum-exp merge of attention states (the merge the split-KV
 * partials of "sglang PR #10417", Modifications, need; the pages fix only
 * that its order is fixed).  For row (i, h) the states s = 0..count-1 are
 * folded left to right:
 *   M = max(L, lse_s); a = e^{L-M}; b = e^{lse_s-M};
 *   o = (a*o + b*v_s) / (a+b); L = M + ln(a+b)
 * starting from the first state; a state with lse = -inf is skipped, and a
 * row with no finite state yields out 0 and lse -inf.
 *   v:          [n, num_states_max, num_heads, head_dim] fp32
 *   s:          [n, num_states_max, num_heads] fp32, natural-log LSE
 *   num_states: [n] int32 device array of counts <= num_states_max, or NULL
 *   out:        [n, num_heads, head_dim] bf16 (round to nearest even)
 *   out_lse:    [n, num_heads] fp32 or NULL
 * head_dim: a multiple of 4 up to 512.
 */
BIA_API int bia_merge_states(const float *v, const float *s, const int32_t *num_states, int64_t n,
                     int32_t num_states_max, int32_t num_heads, int32_t head_dim, void *out,
                     float *out_lse, void *stream);

/*
 * Paged-KV append: writes the key and value rows of a call's new tokens into
 * their pages, the step that precedes an extend over the same page tables
 * (the pages' chunked prefill attends each chunk against a cache that already
 * holds that chunk: "sglang PR #43612", Summary; they never spell the write
 * out, so it is defined here).  Request b's page table already covers its
 * n_new(b) = append_indptr[b+1] - append_indptr[b] new tokens as the LAST
 * n_new(b) of its kv_len keys (the convention bia_prefill_paged uses for q):
 * new token t of request b is written to position
 *   kv_len(b) - n_new(b) + (t - append_indptr[b]),
 * i.e. page kv_indices[kv_indptr[b] + pos / page_size], slot pos % page_size,
 * all num_kv_heads heads.  Nothing else in the caches is touched.
 *   k_new, v_new:  [total_new, num_kv_heads, head_dim] bf16, total_new =
 *                  append_indptr[batch]; 16-byte aligned (as are the caches)
 *   append_indptr: [batch+1] int32, append_indptr[0] == 0, n_new(b) <= kv_len(b)
 *   kv_*:          the page table of bia_prefill_paged (num_qo_heads and
 *                  sm_scale of desc are not used)
 *   status:        NULL, or a device int32 the call zeroes and then sets bit 0
 *                  of when a page index is outside [0, num_pages) (that token
 *                  is skipped); readable with bia_read_status(status, ...)
 * Two positions that map to the same page slot are the caller's error (which
 * write lands is then unspecified).
 */
BIA_API int bia_append_paged_kv(const bia_attn_desc *desc, const void *k_new, const void *v_new,
                        void *k_cache, void *v_cache, int64_t num_pages,
                        const int32_t *append_indptr, const int32_t *kv_indptr,
                        const int32_t *kv_indices, const int32_t *kv_last_page_len,
                        const int32_t *append_indptr_host, const int32_t *kv_indptr_host,
                        const int32_t *kv_last_page_len_host, int32_t batch, int32_t *status,
                        void *stream);

/* Tokens per q tile for GQA group size G = num_qo_heads / num_kv_heads:
 * 128 / G, the chunk grid on which chunked prefill is guaranteed to be
 * bit-identical ("sglang PR #43612", Summary).  0 if G does not divide 128. */
BIA_API int32_t bia_q_tile_tokens(int32_t gqa_group);

/* Static text for a bia_status value. */
BIA_API const char *bia_status_string(int status);

/* Detail of the last failure in the calling thread: the CUDA or driver call
 * behind a BIA_ERR_CUDA and its error, or the pointer a residency check
 * refused; empty if none. */
BIA_API const char *bia_last_error(void);

/*
 * Copies the device status word of the last call that used `workspace`
 * (bit 0: a page index was out of range; bit 1: the device index arrays
 * disagreed with the host-sized launch, broke a rule of the call or exceeded
 * the bounds of a bounded call, and nothing was computed; bit 2: a device wait
 * timed out) into *status_out.  Synchronises `stream`.
 */
BIA_API int bia_read_status(const void *workspace, int32_t *status_out, void *stream);

/*
 * Measurement hooks (not part of the computation).
 * bia_set_profile_events: when both are non-NULL, every later prefill /
 * decode call records `attn_begin` just before and `attn_end` just after its
 * attention kernel on the call's stream (cudaEvent_t handles owned by the
 * caller), so the kernel alone can be timed; NULL, NULL turns this off.
 * Process-wide, not thread-safe.
 * bia_launch_count: kernels this library has launched since it was loaded.
 */
BIA_API void bia_set_profile_events(void *attn_begin, void *attn_end);
BIA_API uint64_t bia_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* BIA_H */
