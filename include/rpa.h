/*
 * rpa.h -- C ABI of the GB300 (sm_103a) ragged paged attention library.
 *
 * Four operations, each one asynchronous call on a caller-supplied CUDA stream:
 *
 *   rpa_forward          ragged paged attention over a packed prefill+decode batch
 *                        (tpu-inference "ragged_paged_attention/v2/kernel.py",
 *                        ref_ragged_paged_attention and ragged_paged_attention).
 *   rpa_update_kv_cache  scatter of the batch's new K/V tokens into their pages
 *                        (no counterpart on the pages beyond the v2 wrapper's TODO for a
 *                        cache-write kernel; defined like the MLA update_kv_cache).
 *                        rpa_forward_update does both in one call.
 *   mla_rpa_forward      MLA latent attention with its cache update
 *                        (tpu-inference "mla/v1/kernel.py", update_kv_cache and
 *                        mla_ragged_paged_attention / ref_mla_ragged_paged_attention).
 *   sparse_mla_forward   DSA sparse MLA over selected units of a paged latent cache
 *                        (sglang-jax "dsa/sparse_mla_prefill.py", sparse_mla_attention and
 *                        _sparse_mla_kernel_chunked_hminor).
 *
 * Conventions shared by every entry point
 *   - Every tensor argument is a DEVICE pointer owned by the caller; the library
 *     never frees or retains it.  Row-major, densely packed, 16-byte aligned.
 *   - The library allocates no memory.  Scratch (work lists, split-KV partials,
 *     the device error word) lives in a caller-provided workspace whose size the
 *     matching *_workspace_size() call returns; the workspace must be 256-byte
 *     aligned, must be zero-filled once after it is allocated (the library keeps it
 *     consistent from then on), and must not be shared by two calls in flight at once.
 *   - Calls are asynchronous on `stream` and never synchronise with the host, so
 *     they can be captured in a CUDA graph.  Sizes read from device memory
 *     (num_seqs, cu_q_lens, kv_lens, page tables, indices) are validated on the
 *     device: a bad value sets a bit in the workspace's error word, the offending
 *     sequence/query is skipped (its output rows are left untouched), and no
 *     out-of-range address is ever formed.  rpa_check_device_status() reads the word.
 *   - Host-side arguments (shapes, dtypes, options) are validated before any launch;
 *     a bad one returns a negative status and launches nothing.
 *   - Optional values use a "none" encoding: sliding_window = 0, soft_cap = 0,
 *     k_scale = v_scale = 0, mask_value = NaN (meaning -0.7 * FLT_MAX, the pages'
 *     DEFAULT_MASK_VALUE).
 *   - Masking follows the pages: RPA adds mask_value to a masked logit, MLA
 *     substitutes it.  With a mask value at or below -1e30 a masked key's weight
 *     underflows to exactly zero in float32 (the key at the query's own position is
 *     always visible), so the kernels skip masked keys outright.  Any larger finite
 *     mask_value leaves masked keys real weight: then every key below kv_len takes
 *     part (future keys of a prefill chunk and keys outside the window alike) with
 *     mask_value added or substituted.  +inf is rejected with RPA_ERR_VALUE.
 */
#ifndef RPA_GB300_RPA_H_
#define RPA_GB300_RPA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RPA_ABI_VERSION 1

/* Every entry point below is exported from the shared library. */
#if defined(__GNUC__)
#define RPA_API __attribute__((visibility("default")))
#else
#define RPA_API
#endif

/* Status codes returned by every call. */
typedef enum {
    RPA_OK = 0,
    RPA_ERR_NULL = -1,          /* a required pointer is NULL */
    RPA_ERR_SHAPE = -2,         /* inconsistent sizes (Hq % Hkv, odd combined heads, ...) */
    RPA_ERR_DTYPE = -3,         /* unsupported dtype combination */
    RPA_ERR_VALUE = -4,         /* bad option value (sliding_window < 0, soft_cap < 0, ...) */
    RPA_ERR_UNSUPPORTED = -5,   /* valid on the pages but not implemented here */
    RPA_ERR_CUDA = -6,          /* a CUDA runtime call failed (see rpa_last_error) */
    RPA_ERR_DEVICE_CHECK = -7,  /* rpa_check_device_status found a device-side error */
    RPA_ERR_WORKSPACE = -8      /* workspace NULL, misaligned or too small */
} rpa_status;

/* Element types. */
typedef enum {
    RPA_DTYPE_BF16 = 1,
    RPA_DTYPE_FP8_E4M3 = 2,
    RPA_DTYPE_F32 = 3,
    RPA_DTYPE_INT8 = 4,          /* two's-complement bytes (RPA K/V only) */
    RPA_DTYPE_INT4 = 5           /* two's-complement 4-bit values, two to a byte along the head
                                  * dimension: element 2i of a row in the low nibble (bits 0-3) of
                                  * the row's byte i, element 2i+1 in the high nibble (RPA K/V only;
                                  * a head row is head_dim / 2 bytes) */
} rpa_dtype;

/* Bits of the device error word (OR-ed together). */
#define RPA_DEV_ERR_NUM_SEQS   0x01u  /* num_seqs / distribution outside [0, max_num_seqs] */
#define RPA_DEV_ERR_Q_LEN      0x02u  /* q_len < 0 or q_len > kv_len for some sequence */
#define RPA_DEV_ERR_KV_LEN     0x04u  /* cdiv(kv_len, page_size) > pages_per_seq */
#define RPA_DEV_ERR_PAGE       0x08u  /* a used page index outside [0, total_num_pages) */
#define RPA_DEV_ERR_TOKENS     0x10u  /* cu_q_lens[num_seqs] > max_num_tokens or not monotone */
#define RPA_DEV_ERR_POSITION   0x20u  /* sparse: query position outside [0, seq_len) */
#define RPA_DEV_ERR_TIMEOUT    0x40u  /* a pipeline wait gave up after its time limit (2 s) */
#define RPA_DEV_ERR_BATCH_KIND 0x80u  /* a sequence of the class rpa_params.batch_kind excludes */

/* rpa_params.batch_kind: what the caller knows of the batch's mix (the MLA v1 page keys its
 * decode-only, prefill-only and mixed kernels on its `distribution`).  A sequence is decode-class
 * when q_len * (num_q_heads / num_kv_heads) <= 16, prefill-class otherwise. */
#define RPA_BATCH_MIXED        0      /* unknown or mixed: every kernel is launched */
#define RPA_BATCH_DECODE_ONLY  1      /* no prefill-class sequence: the prefill launches are skipped */
#define RPA_BATCH_PREFILL_ONLY 2      /* no decode-class sequence: the decode launch is skipped */

/* CUDA stream handle (ABI-compatible with cudaStream_t). */
typedef struct CUstream_st* rpa_stream_t;

/* ---------------------------------------------------------------------- */
/* Standard ragged paged attention                                         */
/* ---------------------------------------------------------------------- */

/* Problem description shared by rpa_forward / rpa_update_kv_cache.
 * Layouts (tpu-inference RPA v2, ref_ragged_paged_attention):
 *   q          [max_num_tokens, num_q_heads, head_dim]               q_dtype (bf16)
 *   kv_pages   [total_num_pages, page_size, num_combined_kv_heads, head_dim]  kv_dtype;
 *              combined head 2j holds K and 2j+1 holds V of KV head j
 *   kv_lens    int32 [max_num_seqs]   keys of each sequence, including its new tokens
 *   page_indices int32 [max_num_seqs, pages_per_seq]   logical -> physical page
 *   cu_q_lens  int32 [max_num_seqs + 1]   sequence i owns tokens [cu_q_lens[i], cu_q_lens[i+1])
 *   num_seqs   int32 [1] (device)   only the first num_seqs sequences are processed
 *   out        [max_num_tokens, num_q_heads, head_dim]   q_dtype; rows of tokens
 *              >= cu_q_lens[num_seqs] are not written
 * Query j of sequence i sits at position kv_len - q_len + j; key k is visible when
 * k <= q_pos and (sliding_window == 0 or k > q_pos - sliding_window).  Q head h reads
 * KV head h / (num_q_heads / num_kv_heads).  Logits: sm_scale * q.k, then
 * soft_cap * tanh(x / soft_cap) when soft_cap != 0.  When k_scale (v_scale) != 0 the
 * keys (values) are dequantised as bf16(float(k) * k_scale) before the dot products.
 * kv_dtype int8 and int4 (the v2 kernel's packed integer KV): two's-complement integers, read
 * as their exact value without a scale and dequantised like any other dtype with one; int4
 * packs two values a byte (RPA_DTYPE_INT4), so kv_pages (and new_k / new_v) rows are
 * head_dim / 2 bytes. */
typedef struct {
    uint32_t struct_size;        /* sizeof(rpa_params) */
    uint32_t version;            /* RPA_ABI_VERSION */
    int32_t max_num_tokens;
    int32_t num_q_heads;
    int32_t num_combined_kv_heads;
    int32_t head_dim;            /* 64, 128 or 256; 96 or 192 for attention over a bf16 cache without
                                    scales, with a power-of-two page_size >= 8 and a mask_value at or
                                    below -1e30 (the cache write takes any of the five) */
    int32_t total_num_pages;
    int32_t page_size;
    int32_t max_num_seqs;
    int32_t pages_per_seq;
    int32_t q_dtype;             /* RPA_DTYPE_BF16 */
    int32_t kv_dtype;            /* RPA_DTYPE_BF16, RPA_DTYPE_FP8_E4M3, RPA_DTYPE_INT8 or RPA_DTYPE_INT4 */
    float sm_scale;
    int32_t sliding_window;      /* 0 = none */
    float soft_cap;              /* 0 = none */
    float mask_value;            /* NaN = default */
    float k_scale;               /* 0 = none */
    float v_scale;               /* 0 = none */
    /* RPA_BATCH_*; a sequence the hint excludes is skipped (its rows are not written) and sets
     * RPA_DEV_ERR_BATCH_KIND.  Optional: a struct_size that ends before this field means
     * RPA_BATCH_MIXED. */
    int32_t batch_kind;
} rpa_params;

/* Bytes of workspace rpa_forward needs for these maxima. */
RPA_API int rpa_workspace_size(const rpa_params* p, size_t* bytes);

/* Ragged paged attention over the whole batch (every sequence, prefill and decode,
 * in one call).  `out` must not alias `q` or `kv_pages`. */
RPA_API int rpa_forward(const rpa_params* p, const void* q, const void* kv_pages, const int32_t* kv_lens,
                const int32_t* page_indices, const int32_t* cu_q_lens, const int32_t* num_seqs,
                void* out, void* workspace, size_t workspace_bytes, rpa_stream_t stream);

/* rpa_forward without a workspace argument, for callers that cannot allocate device
 * memory (for example a plugin inside an application whose memory manager owns the
 * whole GPU, or a serving loop that must not call cudaMalloc, which can synchronise
 * the device, once it is running).  The pages have no counterpart: it is a packaging
 * of rpa_forward, with the same arguments minus the workspace and the same results.
 *   - Scratch is a fixed array of RPA_NOALLOC_SCRATCH_BYTES inside the library; every
 *     GPU that loads the library holds it until the process exits.  Problems whose
 *     rpa_workspace_size() exceeds it are rejected with RPA_ERR_WORKSPACE before any
 *     launch.  The call allocates nothing itself.
 *   - Every call looks up the array's device address in the context current on the
 *     calling thread, so a host application's own (non-primary) context and a device
 *     reset between calls are both handled.  The first call in a context also loads
 *     the library's device code there; make that first call before any stream capture.
 *   - All calls share the one array and it keeps the previous call's contents; the
 *     kernels reset what they need.  Calls that overlap on the GPU (two streams, or
 *     two threads) race on it: serialise them.
 *   - Device-side metadata errors skip the offending sequence as in rpa_forward, but
 *     the error word is not reported (there is no workspace to pass to
 *     rpa_check_device_status). */
#define RPA_NOALLOC_SCRATCH_BYTES (64u << 20)
RPA_API int rpa_forward_noalloc(const rpa_params* p, const void* q, const void* kv_pages, const int32_t* kv_lens,
                                const int32_t* page_indices, const int32_t* cu_q_lens, const int32_t* num_seqs,
                                void* out, rpa_stream_t stream);

/* Write token j of sequence i (position kv_len - q_len + j) into slot
 * page_indices[i, pos / page_size], pos % page_size of kv_pages, in place:
 * new_k[t, g, :] to combined head 2g and new_v[t, g, :] to 2g+1.
 *   new_k, new_v  [max_num_tokens, num_combined_kv_heads / 2, head_dim]  kv_dtype
 * Bytes are copied unchanged; every other byte of kv_pages is left as it was.
 * `workspace` is optional (may be NULL): when given, device-side metadata errors are
 * recorded in its error word (it needs at least 256 bytes). */
RPA_API int rpa_update_kv_cache(const rpa_params* p, const void* new_k, const void* new_v, void* kv_pages,
                        const int32_t* kv_lens, const int32_t* page_indices, const int32_t* cu_q_lens,
                        const int32_t* num_seqs, void* workspace, size_t workspace_bytes,
                        rpa_stream_t stream);

/* rpa_update_kv_cache followed by rpa_forward, in one call with one launch fewer: the cache
 * write of the batch's new K/V rows (exactly as rpa_update_kv_cache: bit-exact, in place)
 * runs in the same launch as the work-list plan, and the attention launches read the cache
 * only after both have ended, so the new tokens attend to themselves. The tpu-inference RPA
 * v2 wrapper leaves this write inside the attention call as a TODO; this is that fused form.
 * Arguments as in the two calls; `workspace` is rpa_forward's (its error word also records the
 * cache write's metadata errors). `out` must not alias q, kv_pages, new_k or new_v. */
RPA_API int rpa_forward_update(const rpa_params* p, const void* q, const void* new_k, const void* new_v,
                               void* kv_pages, const int32_t* kv_lens, const int32_t* page_indices,
                               const int32_t* cu_q_lens, const int32_t* num_seqs, void* out, void* workspace,
                               size_t workspace_bytes, rpa_stream_t stream);

/* ---------------------------------------------------------------------- */
/* MLA latent ragged paged attention                                       */
/* ---------------------------------------------------------------------- */

/* Layouts (tpu-inference MLA v1, mla_ragged_paged_attention):
 *   ql_nope    [max_num_tokens, num_q_heads, lkv_dim]        bf16, or fp8 e4m3 (q_dtype)
 *   q_pe       [max_num_tokens, num_q_heads, r_dim]          same dtype as ql_nope
 *   new_kv_c   [max_num_tokens, lkv_dim]                     bf16
 *   new_k_pe   [max_num_tokens, r_dim]                       bf16
 *   cache_kv_c [total_num_pages, page_size / kv_packing, kv_packing, lkv_dim_pad] bf16
 *   cache_k_pe [total_num_pages, page_size / kv_packing, kv_packing, r_dim_pad]   bf16
 *              (token t of a page is row t of the page: same bytes as [P, page_size, D])
 *   kv_lens    int32 [max_num_seqs]; page_indices int32 [max_num_seqs * pages_per_seq]
 *   cu_q_lens  int32 [max_num_seqs + 1]; distribution int32 [3] (device):
 *              (decode_end, prefill_end, num_seqs); only distribution[2] bounds the work
 *   out        [max_num_tokens, num_q_heads, lkv_dim]        bf16
 * Key = [kv_c | k_pe], value = kv_c, one latent head shared by all q heads; masked
 * logits are replaced by mask_value (see the header note on masking).  fp8 queries are
 * widened exactly to bf16 before the products; the output stays bf16 (the MLA v1 page
 * writes it in the query dtype, which for fp8 would throw away most of its precision). */
typedef struct {
    uint32_t struct_size;        /* sizeof(mla_params) */
    uint32_t version;            /* RPA_ABI_VERSION */
    int32_t max_num_tokens;
    int32_t num_q_heads;         /* multiple of 128 (one two-CTA tile) */
    int32_t lkv_dim;             /* 512 */
    int32_t r_dim;               /* 64 */
    int32_t lkv_dim_pad;         /* align(lkv_dim, 128) */
    int32_t r_dim_pad;           /* align(r_dim, 128) */
    int32_t total_num_pages;
    int32_t page_size;
    int32_t kv_packing;          /* 2 for bf16 */
    int32_t max_num_seqs;
    int32_t pages_per_seq;
    float sm_scale;
    int32_t sliding_window;      /* 0 = none */
    float soft_cap;              /* 0 = none */
    float mask_value;            /* NaN = default */
    /* Optional (read only when struct_size covers them, else bf16 queries): */
    int32_t q_dtype;             /* RPA_DTYPE_BF16 (0 is taken as bf16) or RPA_DTYPE_FP8_E4M3 for
                                    ql_nope and q_pe */
    float q_scale;               /* fp8 queries: every score is multiplied by it after sm_scale
                                    (0 = 1); must be 0 for bf16 queries */
} mla_params;

RPA_API int mla_workspace_size(const mla_params* p, size_t* bytes);

/* Scatter the batch's new latent rows into the caches, in place (update_kv_cache):
 * token j of sequence i < distribution[2] goes to position kv_len - q_len + j; its
 * kv_c row is copied to cache_kv_c and its k_pe row to cache_k_pe with columns
 * [r_dim, r_dim_pad) written as zero.  `workspace` is optional, as for
 * rpa_update_kv_cache. */
RPA_API int mla_update_kv_cache(const mla_params* p, const void* new_kv_c, const void* new_k_pe, void* cache_kv_c,
                        void* cache_k_pe, const int32_t* kv_lens, const int32_t* page_indices,
                        const int32_t* cu_q_lens, const int32_t* distribution, void* workspace,
                        size_t workspace_bytes, rpa_stream_t stream);

/* mla_update_kv_cache followed by attention of every query token over the updated
 * caches (the caches are modified in place).  The cache write runs in the same launch as
 * the work-list plan (the MLA v1 page leaves fusing it as a TODO); attention starts once
 * both have ended. */
RPA_API int mla_rpa_forward(const mla_params* p, const void* ql_nope, const void* q_pe, const void* new_kv_c,
                    const void* new_k_pe, void* cache_kv_c, void* cache_k_pe, const int32_t* kv_lens,
                    const int32_t* page_indices, const int32_t* cu_q_lens, const int32_t* distribution,
                    void* out, void* workspace, size_t workspace_bytes, rpa_stream_t stream);

/* ---------------------------------------------------------------------- */
/* DSA sparse MLA                                                           */
/* ---------------------------------------------------------------------- */

/* Layouts (sglang-jax sparse_mla_attention, paged per-request mode):
 *   q          [batch, num_queries, num_heads, dk]    bf16 (dk = 576 = 512 + 64)
 *   cache      [total_num_pages * page_size, row_stride]  bf16 (row_stride >= dk; the
 *              [P, page_size / packing, packing, row_stride] cache has these bytes)
 *   indices    int32 [batch, num_queries, topk]   unit ids, -1 = empty slot
 *   positions  int32 [batch, num_queries]         query positions (causal bound)
 *   page_table int32 [batch, max_pages]           logical -> physical page
 *   out        [batch, num_queries, num_heads, dv]  float32 (dv = 512)
 * A unit u covers tokens [u * read_block, (u + 1) * read_block).  Token kp of slot i
 * is a key when u >= 0, kp <= position and kp < seq_len; it is read from row
 * page_table[b, kp / page_size] * page_size + kp % page_size.  Keys form a multiset
 * (a unit named twice counts twice); a query with no key outputs zeros.
 * read_block must divide page_size. */
typedef struct {
    uint32_t struct_size;        /* sizeof(sparse_params) */
    uint32_t version;            /* RPA_ABI_VERSION */
    int32_t batch;
    int32_t num_queries;
    int32_t num_heads;           /* multiple of 128 (one two-CTA tile) */
    int32_t dk;                  /* 576 */
    int32_t dv;                  /* 512 */
    int32_t row_stride;          /* elements per cache row (640) */
    int32_t topk;
    int32_t read_block;
    int32_t page_size;
    int32_t max_pages;
    int32_t total_num_pages;
    int32_t seq_len;
    float sm_scale;              /* required, > 0 */
} sparse_params;

RPA_API int sparse_mla_workspace_size(const sparse_params* p, size_t* bytes);

RPA_API int sparse_mla_forward(const sparse_params* p, const void* q, const void* cache, const int32_t* indices,
                       const int32_t* positions, const int32_t* page_table, float* out, void* workspace,
                       size_t workspace_bytes, rpa_stream_t stream);

/* Packed-ragged mode with the self-write (sglang-jax "dsa/sparse_mla_prefill.py",
 * prefill_write_and_attend_ragged and the ragged branch of sparse_mla_attention): several
 * requests' tokens packed along one axis.
 *   ql         [num_tokens, num_heads, dv]      bf16 absorbed latent query (dv = 512)
 *   qpe        [num_tokens, num_heads, rope]    bf16 rope query (rope = 64); the query is
 *              their concatenation (dk = dv + rope = 576)
 *   kvc, kpe   [num_tokens, dv], [num_tokens, rope]  bf16 new latent rows (both NULL: no write)
 *   cache      [total_num_pages * page_size, row_stride]  bf16, written in place
 *   topk       int32 [num_tokens, topk]   request-local unit ids, -1 = empty slot
 *   positions  int32 [num_tokens]         absolute query positions
 *   loc        int32 [num_tokens]         flat cache row of each token's new row (-1 = none;
 *              NULL with kvc/kpe NULL)
 *   seq_lens   int32 [num_seqs]           each request's key length (causal bound)
 *   cu_q_lens  int32 [num_seqs + 1]       request r owns tokens [cu_q_lens[r], cu_q_lens[r+1])
 *   cu_kv_lens int32 [num_seqs + 1]       page-aligned key offsets into page_indices' runs
 *   page_indices int32 [num_page_ids]     packed physical page ids
 *   out        [num_tokens, num_heads, dv]  float32
 * First every token's row [kvc | kpe | zeros] is written to cache row loc[t] (rows outside
 * the cache are dropped; two tokens naming one row leave either's). Then token t attends as
 * in sparse_mla_forward, where its request r is the number of cu_q_lens[1..num_seqs]
 * entries <= t (clipped to num_seqs - 1), the causal bound is seq_lens[r], and key kp sits
 * in page page_indices[min(cu_kv_lens[r] / page_size + kp / page_size, num_page_ids - 1)].
 * read_block must divide page_size. */
typedef struct {
    uint32_t struct_size;        /* sizeof(sparse_ragged_params) */
    uint32_t version;            /* RPA_ABI_VERSION */
    int32_t num_tokens;
    int32_t num_seqs;
    int32_t num_heads;           /* multiple of 128 */
    int32_t dv;                  /* 512 */
    int32_t rope;                /* 64 */
    int32_t row_stride;          /* elements per cache row (>= dv + rope, multiple of 8) */
    int32_t topk;
    int32_t read_block;
    int32_t page_size;
    int32_t num_page_ids;
    int32_t total_num_pages;
    float sm_scale;              /* required, > 0 */
} sparse_ragged_params;

RPA_API int sparse_mla_ragged_workspace_size(const sparse_ragged_params* p, size_t* bytes);

RPA_API int sparse_mla_write_and_attend_ragged(const sparse_ragged_params* p, const void* ql, const void* qpe,
                                               const void* kvc, const void* kpe, void* cache, const int32_t* topk,
                                               const int32_t* positions, const int32_t* loc,
                                               const int32_t* seq_lens, const int32_t* cu_q_lens,
                                               const int32_t* cu_kv_lens, const int32_t* page_indices, float* out,
                                               void* workspace, size_t workspace_bytes, rpa_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Status and diagnostics                                                   */
/* ---------------------------------------------------------------------- */

/* Synchronises `stream`, reads the workspace's device error word into *bits (may be
 * NULL) and clears it.  Returns RPA_ERR_DEVICE_CHECK when any bit was set. */
RPA_API int rpa_check_device_status(void* workspace, uint32_t* bits, rpa_stream_t stream);

/* Failure-path check (diagnostics): launches one thread that waits, through the same bounded
 * wait every pipeline of the library uses, on a barrier nothing arrives on.  The wait gives up
 * after its limit (2 s), sets RPA_DEV_ERR_TIMEOUT in the workspace's error word and the kernel
 * returns: rpa_check_device_status then reports it, and the context stays usable.
 * `workspace` needs at least 256 bytes. */
RPA_API int rpa_selftest_bounded_wait(void* workspace, size_t workspace_bytes, rpa_stream_t stream);

/* Per-kernel timing (diagnostics).  While enabled, every kernel the library launches
 * is bracketed by two CUDA events on its launch stream (a GPU-side timestamp pair; no
 * host synchronisation).  rpa_profile_read synchronises on the recorded events and
 * reports, per kernel name, the number of launches and their summed duration since
 * the last rpa_profile_reset.  Entries are written to out[0 .. max_entries) in name
 * order; *n_entries receives the total number of kernel names. */
typedef struct {
    char name[48];
    int64_t launches;
    double total_ms;
} rpa_kernel_time;

RPA_API int rpa_profile_enable(int on);
RPA_API int rpa_profile_reset(void);
RPA_API int rpa_profile_read(rpa_kernel_time* out, int max_entries, int* n_entries);

/* Number of kernels the library has launched since it was loaded, counted whether or not
 * timing is enabled (a host-side counter; no synchronisation). */
RPA_API int64_t rpa_launch_count(void);

/* Thread-local description of the last failed call ("" if none). */
RPA_API const char* rpa_last_error(void);

/* RPA_ABI_VERSION of the loaded library. */
RPA_API int rpa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RPA_GB300_RPA_H_ */
