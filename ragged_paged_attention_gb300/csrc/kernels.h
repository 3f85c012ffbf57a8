// Kernel argument blocks and launch entry points shared by the C ABI (api.cu)
// and the kernel translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <utility>

namespace rpa {

struct WsHeader;

// Tiling constants of the RPA kernels.
constexpr int kMaxDecodeHeads = 4;      // most KV heads a decode CTA covers (one warp each)
constexpr int kDecodeBK = 16;           // keys per decode pipeline stage
constexpr int kDecodeRows = 8;          // query rows (q_len x G) per decode item (mma N)
constexpr int kCuCache = 4096;          // metadata ints the cache-write kernels stage in shared memory
// Shared-memory ints the RPA cache write stages (cu_q_lens and kv_lens of every sequence slot),
// or 0 when they do not fit and it reads them from global memory.
__host__ __device__ inline int update_cache_ints(int max_num_seqs) {
    return 2 * max_num_seqs + 1 <= kCuCache ? 2 * max_num_seqs + 1 : 0;
}
constexpr int kPrefillRows = 128;       // (token, q-head) rows per prefill item (one TMEM tile)
constexpr int kMinChunk = 256;          // smallest split-KV chunk (keys)
constexpr int kMaxDecodeCtas = 2048;    // most decode shares (static, one per CTA, and pooled)
// Pool: the part of the line left after the static shares (here only their rounding
// remainder: measured on the Llama-3 and Gemma-2 batches, pooled shares of 64-256 keys cost
// more in per-item start-up than they recover in balance)
constexpr int kPoolPercent = 0;         // share of the decode work left to the pool
constexpr int kMinPoolChunk = 64;       // smallest pooled decode share (keys)
constexpr int kPoolPerCta = 3;          // pooled shares per decode CTA (about)
// Each decode group also costs its items a fixed start (descriptor, metadata, Q and the first
// stage's latency) and, when split, a fence, ticket and merge. Counted in keys, that cost is laid
// on the line ahead of the group's keys, so shares that cross more groups get fewer keys and all
// shares still end together. Measured on GB300: 128 keys takes the Llama-3 bf16 decode kernel from
// 190.7 to 182.3 us; the converting (fp8 or scaled) kernel, slower per key, ends best at 0
// (Gemma-2 fp8: 204 us, 210 us at 128).
inline int rpa_item_cost_keys(bool converting) { return converting ? 0 : 128; }

// Prefill beside decode: the prefill items are tensor-core bound and the decode items HBM
// bound, so the plan kernel gives prefill the share of the SMs that makes both lists end
// together, from the batch's prefill FLOPs and decode bytes and these measured rates
// (a mis-estimate costs a short tail: prefill left over when decode ends runs on every SM).
constexpr float kDecHbmBytesPerNs = 5800.f;   // decode kernel with HBM saturated
// the prefill grid beside decode takes no new item once this share of the decode CTAs with a
// share are out of work (equal shares end within a few percent of one another)
constexpr int kPrefillStopPercent = 90;

// Per-SM rates of the two kernels by head size and cache type: prefill FLOPs per ns per SM,
// decode bytes per ns per SM while the SMs (not HBM) limit it. Measured on GB300 for head_dim
// 128 bf16 (Llama-3 batch) and 256 fp8 (Gemma-2 batch); the other entries are scaled from
// those. Only the SM split depends on them, never a result.
inline void rpa_rates(int head_dim, bool fp8, bool scale, bool pow2, float* pre, float* dec) {
    const bool conv = fp8 || scale;
    *pre = conv ? (head_dim >= 256 ? 1800.f : 2200.f) : (head_dim >= 256 ? 3000.f : head_dim >= 128 ? 3800.f : 2400.f);
    // (one-byte caches with power-of-two scales decode through the f16 fragment path)
    *dec = conv ? (fp8 && pow2 ? 38.f : 26.f) : 60.f;
}

// A scale the f16 paths may take: a power of two with e4m3 * scale inside bf16's normal range
// (bf16(float(x) * scale) is then exactly x * scale, so the scale can move onto S and O).
inline bool rpa_pow2_scale(float s) {
    int e = 0;
    const float m = frexpf(s, &e);
    return s > 0.f && m == 0.5f && e >= -40 && e <= 40;
}

// One unit of work for a persistent attention CTA (32 bytes).
struct __align__(16) WorkItem {
    int seq;         // sequence (RPA/MLA) or flat query b*S+s (sparse)
    int head;        // first KV head (RPA) or first q head (latent) of the tile
    int row_begin;   // first row of the tile (RPA prefill) / token in sequence (MLA)
    int key_begin;   // key range [key_begin, key_end)
    int key_end;
    int first_item;  // item index of split 0 of this group (ticket / partial base)
    int num_splits;
    int split;
};

struct RpaArgs {
    const __nv_bfloat16* q;
    const void* kv_pages;
    const int32_t* kv_lens;
    const int32_t* page_indices;
    const int32_t* cu_q_lens;
    const int32_t* num_seqs;
    __nv_bfloat16* out;
    int max_num_tokens, num_q_heads, num_kv_heads, head_dim;
    int total_num_pages, page_size, max_num_seqs, pages_per_seq;
    int kv_byte;                // narrow K/V elements: e4m3, int8 (kv_int8) or int4 (kv_int4)
    int kv_int8;
    int kv_int4;                // two 4-bit values a byte, element 2i in the low nibble of byte i
    float sm_scale, soft_cap;
    int sliding_window;
    // a mask_value that leaves masked keys real weight (above -1e30): every key of a sequence
    // takes part, a masked one with mask_value added to its logit (the RPA reference's form);
    // otherwise masked keys are skipped (their weight is exactly zero either way)
    int mask_mild;
    float mask_value;
    int batch_kind;             // RPA_BATCH_*: a decode-only or prefill-only batch skips the other launches
    int has_scale;              // k_scale or v_scale given
    float k_scale_or_one, v_scale_or_one;
    int decode_per_sm;          // decode CTAs resident per SM (occupancy of the chosen kernel)
    int decode_heads;           // KV heads per decode item (decode_heads_for)
    int num_sms;
    int overlap;                // run prefill beside decode (off while kernels are timed one by one)
    float pre_flops_per_ns_sm;  // prefill kernel rate per SM (this head size and cache type)
    float dec_bytes_per_ns_sm;  // decode kernel rate per SM while SMs, not HBM, limit it
    int item_cost_keys;         // per-group cost on the decode line (a multiple of 16 keys)
    // workspace
    WsHeader* hdr;
    WorkItem* dec_items;
    WorkItem* pre_items;
    int* tickets;
    int* cta_first;             // [kMaxDecodeCtas + 1] first decode item of each decode share
    float* partial_ml;
    float* partial_o;
    int max_dec_items, max_pre_items;
};

struct RpaUpdateArgs {
    const void* new_k;
    const void* new_v;
    void* kv_pages;
    const int32_t* kv_lens;
    const int32_t* page_indices;
    const int32_t* cu_q_lens;
    const int32_t* num_seqs;
    uint32_t* err;  // may be null
    int max_num_tokens, num_kv_heads, head_dim, row_bytes;  // row_bytes: one head row of K or V
    int total_num_pages, page_size, max_num_seqs, pages_per_seq;
};

// Latent (MLA and sparse MLA) attention.
constexpr int kLatRows = 128;     // q heads per (two-CTA) tile
constexpr int kLatBK = 64;        // keys per block
constexpr int kLatDk = 576;       // 512 latent + 64 rope
constexpr int kLatDv = 512;
constexpr int kLatMinChunk = 512;
// most items the MLA plan aims for (the workspace bound); it aims for two per SM (one per CTA of
// each two-CTA cluster, twice over): a split costs its partial O and a merge, and a decode batch
// split finer spends more on those than it gains in balance (64 decode queries: 1104 us at up to
// 512 items, measured)
constexpr int kLatTargetCtas = 512;
// sparse MLA splits a query's selected keys only down to about this many items in all (half
// the two-CTA clusters): its per-item cost (Q slice, pipeline fill, fp32 partial and merge)
// outweighs the extra parallelism on decode-sized batches (64 single-query sequences: 127 us
// unsplit, 197 us in two splits, 361 us in four; measured)
constexpr int kSparseTargetCtas = 38;

struct LatentArgs {
    int sparse;                     // 0 = MLA (paged, causal), 1 = DSA sparse
    int num_heads;
    float sm_scale, soft_cap;
    int sliding_window;
    // mask_value above -1e30: every key of a sequence takes part and a masked logit is replaced
    // by mask_value (the MLA reference's form); otherwise masked keys are skipped
    int mask_mild;
    float mask_value;
    // MLA
    const __nv_bfloat16* ql_nope;   // [T, H, 512]
    const __nv_bfloat16* q_pe;      // [T, H, 64]
    int q_fp8;                      // ql_nope and q_pe hold fp8 e4m3 bytes (same shapes)
    const __nv_bfloat16* cache_kv_c;  // rows of lkv_pad
    const __nv_bfloat16* cache_k_pe;  // rows of r_pad
    const int32_t* kv_lens;
    const int32_t* page_indices;
    const int32_t* cu_q_lens;
    const int32_t* distribution;
    int max_num_tokens, max_num_seqs, pages_per_seq, lkv_pad, r_pad;
    int target_items;               // MLA plan: about this many items in all (<= kLatTargetCtas)
    __nv_bfloat16* out_bf16;        // [T, H, 512]
    // sparse
    const __nv_bfloat16* q;         // [B, S, H, 576]
    const __nv_bfloat16* cache;     // rows of row_stride
    const int32_t* indices;         // [B, S, K]
    const int32_t* positions;       // [B, S]
    const int32_t* page_table;      // [B, max_pages]
    int batch, num_queries, topk, read_block, max_pages, seq_len, row_stride, sparse_splits;
    // sparse, packed-ragged mode (q_base != nullptr): B = 1, S = tokens; query s's causal bound
    // and its base in the packed page list (page_table, max_pages entries) come from these
    // (written by the prep kernel); Q comes from ql_nope and q_pe when q is null
    const int32_t* q_bound;
    const int32_t* q_base;
    float* out_f32;                 // [B, S, H, 512]
    // common
    int total_num_pages, page_size;
    // workspace
    WsHeader* hdr;
    WorkItem* items;
    int* tickets;
    float* partial_ml;
    float* partial_o;
    int max_items;
};

// Packed-ragged sparse MLA: each token's request, causal bound and page base, and the
// self-write of its latent row.
struct SparseRaggedPrepArgs {
    const __nv_bfloat16* kvc;       // [T, dv] (null: no self-write)
    const __nv_bfloat16* kpe;       // [T, rope]
    __nv_bfloat16* cache;           // rows of row_stride
    const int32_t* loc;             // [T] flat slot per token (-1: none)
    const int32_t* seq_lens;        // [S]
    const int32_t* cu_q_lens;       // [S + 1]
    const int32_t* cu_kv_lens;      // [S + 1]
    int32_t* q_bound;               // [T] out
    int32_t* q_base;                // [T] out
    int num_tokens, num_seqs, dv, rope, row_stride, page_size, total_num_pages;
};

struct MlaUpdateArgs {
    const __nv_bfloat16* new_kv_c;
    const __nv_bfloat16* new_k_pe;
    __nv_bfloat16* cache_kv_c;
    __nv_bfloat16* cache_k_pe;
    const int32_t* kv_lens;
    const int32_t* page_indices;
    const int32_t* cu_q_lens;
    const int32_t* distribution;
    uint32_t* err;
    int max_num_tokens, lkv_dim, r_dim, lkv_pad, r_pad;
    int total_num_pages, page_size, max_num_seqs, pages_per_seq;
};

cudaError_t launch_rpa_forward(const RpaArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_wait_selftest(uint32_t* err, cudaStream_t stream);
cudaError_t launch_rpa_forward_update(const RpaArgs& a, const RpaUpdateArgs& u, int num_sms, cudaStream_t stream);
cudaError_t launch_mla_forward_update(const LatentArgs& a, const MlaUpdateArgs& u, int num_sms, cudaStream_t stream);
// Launch with programmatic stream serialization when pdl (the kernel may start before the
// previous launch of the stream ends; it orders itself with griddepcontrol), else plainly.
template <typename... P, typename... A>
cudaError_t launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                       A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}

cudaError_t launch_rpa_decode(const RpaArgs& a, int num_sms, cudaStream_t stream);
int rpa_decode_ctas_per_sm(const RpaArgs& a);  // resident CTAs per SM of the kernel launch_rpa_decode picks
cudaError_t launch_rpa_prefill(const RpaArgs& a, int num_sms, cudaStream_t stream, int tail);
int decode_heads_for(int head_dim, bool fp8);
cudaError_t launch_rpa_update(const RpaUpdateArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_mla_update(const MlaUpdateArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_sparse_forward(const LatentArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_sparse_ragged(const SparseRaggedPrepArgs& pa, const LatentArgs& a, int num_sms,
                                 cudaStream_t stream);
cudaError_t launch_mla_attention(const LatentArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_sparse_attention(const LatentArgs& a, int num_sms, cudaStream_t stream);

// Sparse split count the host chooses from static sizes (no device metadata needed).
inline int sparse_num_splits(int batch, int num_queries, int heads, int slots) {
    long long tiles = (long long)batch * num_queries * (heads / kLatRows);
    long long total = tiles * slots;
    long long chunk = (total + kSparseTargetCtas - 1) / kSparseTargetCtas;
    if (chunk < kLatMinChunk) chunk = kLatMinChunk;
    chunk = (chunk + kLatBK - 1) / kLatBK * kLatBK;
    long long n = (slots + chunk - 1) / chunk;
    return n < 1 ? 1 : (int)n;
}

}  // namespace rpa

#ifdef __CUDACC__
#include "common.cuh"
namespace rpa {
// Validates one sequence's metadata (the reference's dynamic checks); on failure
// records the error bit and returns false so the sequence is skipped.
__device__ __forceinline__ bool seq_shape(const RpaArgs& a, int s, int& ql, int& kl) {
    const int c0 = a.cu_q_lens[s], c1 = a.cu_q_lens[s + 1];
    ql = c1 - c0;
    kl = a.kv_lens[s];
    uint32_t bad = 0;
    if (c0 < 0 || c1 < c0 || c1 > a.max_num_tokens)
        bad = RPA_DEV_ERR_TOKENS;
    else if (ql > kl)
        bad = RPA_DEV_ERR_Q_LEN;
    else if (cdiv(kl, a.page_size) > a.pages_per_seq)
        bad = RPA_DEV_ERR_KV_LEN;
    if (bad) {
        set_error(&a.hdr->error_bits, bad);
        return false;
    }
    return true;
}

// Sequence of token t: the last s in [0, num) with cu[s] <= t (cu = cu_q_lens, in global or
// shared memory; callers check that t really lies in [cu[s], cu[s+1])).
__device__ __forceinline__ int seq_of_token(const int32_t* cu, int num, int t) {
    int lo = 0, hi = num - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Whether the caller's batch_kind admits a sequence of this class (decode: q_len * G <= 16).
__device__ __forceinline__ bool kind_allows(const RpaArgs& a, bool decode_class) {
    return !(a.batch_kind == RPA_BATCH_DECODE_ONLY && !decode_class) &&
           !(a.batch_kind == RPA_BATCH_PREFILL_ONLY && decode_class);
}

// First key any query of a decode-class sequence can see (aligned down to a stage).
__device__ __forceinline__ int decode_key_begin(const RpaArgs& a, int ql, int kl) {
    if (a.sliding_window <= 0 || a.mask_mild) return 0;
    const int lo = kl - ql - a.sliding_window + 1;
    return lo <= 0 ? 0 : lo / kDecodeBK * kDecodeBK;
}
}  // namespace rpa
#endif
