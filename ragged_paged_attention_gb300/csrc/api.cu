// C ABI of the library (declared in include/rpa.h): host-side validation, workspace
// layout and kernel launches.  Nothing here touches tensor data on the host.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "profile.h"

using namespace rpa;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* where) {
    return fail(RPA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

int num_sms_current() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

float resolve_mask(float m) { return isnan(m) ? -0.7f * 3.402823466e38f : m; }
// A mask value above -1e30 leaves masked keys real weight (exp(s + mask - m) does not underflow
// for the logits attention sees), so the kernels then take every key and apply it literally.
bool mild_mask(float m) { return resolve_mask(m) > -1e30f; }

// ---------------------------- RPA ----------------------------------------
// batch_kind, or RPA_BATCH_MIXED when the caller's struct ends before it
int rpa_batch_kind(const rpa_params* p) {
    return p->struct_size >= offsetof(rpa_params, batch_kind) + sizeof(int32_t) ? p->batch_kind : RPA_BATCH_MIXED;
}

struct RpaLayout {
    size_t items_dec, items_pre, tickets, cta_first, pml, po, total;
    int max_dec, max_pre;
};

int check_rpa_params(const rpa_params* p) {
    if (!p) return fail(RPA_ERR_NULL, "params is NULL");
    if (p->struct_size < offsetof(rpa_params, batch_kind)) return fail(RPA_ERR_VALUE, "rpa_params.struct_size too small");
    if (rpa_batch_kind(p) < RPA_BATCH_MIXED || rpa_batch_kind(p) > RPA_BATCH_PREFILL_ONLY)
        return fail(RPA_ERR_VALUE, "batch_kind %d is not an RPA_BATCH_* value", rpa_batch_kind(p));
    if (p->version != RPA_ABI_VERSION) return fail(RPA_ERR_VALUE, "rpa_params.version %u != %d", p->version, RPA_ABI_VERSION);
    if (p->max_num_tokens <= 0 || p->num_q_heads <= 0 || p->num_combined_kv_heads <= 0 || p->total_num_pages <= 0 ||
        p->page_size <= 0 || p->max_num_seqs <= 0 || p->pages_per_seq <= 0)
        return fail(RPA_ERR_SHAPE, "all sizes must be positive");
    if (p->num_combined_kv_heads % 2) return fail(RPA_ERR_SHAPE, "num_combined_kv_heads must be even (K and V interleaved)");
    const int hkv = p->num_combined_kv_heads / 2;
    if (p->num_q_heads % hkv) return fail(RPA_ERR_SHAPE, "num_q_heads %d not divisible by num_kv_heads %d", p->num_q_heads, hkv);
    if (p->head_dim != 64 && p->head_dim != 96 && p->head_dim != 128 && p->head_dim != 192 && p->head_dim != 256)
        return fail(RPA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 96, 128, 192, 256)", p->head_dim);
    if (p->q_dtype != RPA_DTYPE_BF16) return fail(RPA_ERR_DTYPE, "q_dtype must be bf16");
    if (p->kv_dtype != RPA_DTYPE_BF16 && p->kv_dtype != RPA_DTYPE_FP8_E4M3 && p->kv_dtype != RPA_DTYPE_INT8 &&
        p->kv_dtype != RPA_DTYPE_INT4)
        return fail(RPA_ERR_DTYPE, "kv_dtype must be bf16, fp8 e4m3, int8 or int4");
    if (!isfinite(p->sm_scale)) return fail(RPA_ERR_VALUE, "sm_scale must be finite");
    if (p->sliding_window < 0) return fail(RPA_ERR_VALUE, "sliding_window must be positive (0 = none)");
    if (!isfinite(p->soft_cap)) return fail(RPA_ERR_VALUE, "soft_cap must be finite (0 = none)");
    if (!isfinite(p->k_scale) || !isfinite(p->v_scale)) return fail(RPA_ERR_VALUE, "k_scale/v_scale must be finite");
    if (isinf(p->mask_value) && p->mask_value > 0.f) return fail(RPA_ERR_VALUE, "mask_value must not be +inf");
    if ((long long)p->max_num_seqs * p->pages_per_seq > INT32_MAX) return fail(RPA_ERR_SHAPE, "page table too large");
    return RPA_OK;
}

RpaLayout rpa_layout(const rpa_params* p) {
    RpaLayout L;
    const int hkv = p->num_combined_kv_heads / 2;
    const int G = p->num_q_heads / hkv;
    const int dh = decode_heads_for(p->head_dim, p->kv_dtype != RPA_DTYPE_BF16);
    const int groups = cdiv(hkv, dh);
    // pieces: one per CTA share plus one more per group a share boundary cuts (groups: up to two
    // 8-row halves per sequence and KV-head group)
    L.max_dec = kMaxDecodeCtas + 2 * groups * p->max_num_seqs;
    L.max_pre = hkv * (int)((long long)p->max_num_tokens * G / kPrefillRows + p->max_num_seqs + 1);
    size_t off = kWsHeaderBytes;
    L.items_dec = off;
    off = align_up(off + sizeof(WorkItem) * (size_t)L.max_dec);
    L.items_pre = off;
    off = align_up(off + sizeof(WorkItem) * (size_t)L.max_pre);
    L.tickets = off;
    off = align_up(off + sizeof(int) * (size_t)L.max_dec);
    L.cta_first = off;
    off = align_up(off + sizeof(int) * (size_t)(kMaxDecodeCtas + 1));
    L.pml = off;
    off = align_up(off + sizeof(float) * 2 * dh * kDecodeRows * (size_t)L.max_dec);
    L.po = off;
    off = align_up(off + sizeof(float) * (size_t)p->head_dim * dh * kDecodeRows * (size_t)L.max_dec);
    L.total = off;
    return L;
}

int check_workspace(const void* ws, size_t have, size_t need) {
    if (!ws) return fail(RPA_ERR_WORKSPACE, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(ws) % kAlign) return fail(RPA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (have < need) return fail(RPA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", have, need);
    return RPA_OK;
}

// ---------------------------- MLA ----------------------------------------
struct LatLayout {
    size_t items, tickets, pml, po, total;
    int max_items;
};

// q_dtype and q_scale sit at the end of mla_params; a caller built against the struct
// without them passes a struct_size that ends before them and gets bf16 queries
int mla_q_dtype(const mla_params* p) {
    if (p->struct_size < offsetof(mla_params, q_dtype) + sizeof(int32_t) || p->q_dtype == 0) return RPA_DTYPE_BF16;
    return p->q_dtype;
}

float mla_q_scale(const mla_params* p) {
    return p->struct_size >= offsetof(mla_params, q_scale) + sizeof(float) ? p->q_scale : 0.f;
}

int check_mla_params(const mla_params* p) {
    if (!p) return fail(RPA_ERR_NULL, "params is NULL");
    if (p->struct_size < offsetof(mla_params, q_dtype)) return fail(RPA_ERR_VALUE, "mla_params.struct_size too small");
    if (p->version != RPA_ABI_VERSION) return fail(RPA_ERR_VALUE, "mla_params.version %u != %d", p->version, RPA_ABI_VERSION);
    if (p->max_num_tokens <= 0 || p->num_q_heads <= 0 || p->total_num_pages <= 0 || p->page_size <= 0 ||
        p->max_num_seqs <= 0 || p->pages_per_seq <= 0 || p->kv_packing <= 0)
        return fail(RPA_ERR_SHAPE, "all sizes must be positive");
    if (p->page_size % p->kv_packing) return fail(RPA_ERR_SHAPE, "page_size must be divisible by kv_packing");
    if (p->kv_packing != 2) return fail(RPA_ERR_DTYPE, "kv_packing %d does not match bf16 (2)", p->kv_packing);
    if (p->lkv_dim_pad != (p->lkv_dim + 127) / 128 * 128 || p->r_dim_pad != (p->r_dim + 127) / 128 * 128)
        return fail(RPA_ERR_SHAPE, "cache widths must be align(dim, 128)");
    if (p->lkv_dim % 8 || p->r_dim % 8) return fail(RPA_ERR_SHAPE, "lkv_dim and r_dim must be multiples of 8");
    if (!isfinite(p->sm_scale)) return fail(RPA_ERR_VALUE, "sm_scale must be finite");
    if (p->sliding_window < 0) return fail(RPA_ERR_VALUE, "sliding_window must be positive (0 = none)");
    if (!isfinite(p->soft_cap)) return fail(RPA_ERR_VALUE, "soft_cap must be finite (0 = none)");
    if (isinf(p->mask_value) && p->mask_value > 0.f) return fail(RPA_ERR_VALUE, "mask_value must not be +inf");
    if ((long long)p->max_num_seqs * p->pages_per_seq > INT32_MAX) return fail(RPA_ERR_SHAPE, "page table too large");
    const int qd = mla_q_dtype(p);
    if (qd != RPA_DTYPE_BF16 && qd != RPA_DTYPE_FP8_E4M3)
        return fail(RPA_ERR_DTYPE, "mla q_dtype %d: queries are bf16 or fp8 e4m3", qd);
    const float qs = mla_q_scale(p);
    if (!isfinite(qs) || qs < 0.f) return fail(RPA_ERR_VALUE, "q_scale must be finite and >= 0 (0 = 1)");
    if (qd == RPA_DTYPE_BF16 && qs != 0.f) return fail(RPA_ERR_VALUE, "q_scale applies to fp8 queries only");
    return RPA_OK;
}

int check_mla_attn_shape(const mla_params* p) {
    if (p->lkv_dim != 512 || p->r_dim != 64)
        return fail(RPA_ERR_UNSUPPORTED, "MLA attention supports lkv_dim 512 and r_dim 64 (got %d, %d)", p->lkv_dim, p->r_dim);
    if (p->num_q_heads % kLatRows) return fail(RPA_ERR_UNSUPPORTED, "num_q_heads must be a multiple of %d", kLatRows);
    return RPA_OK;
}

LatLayout lat_layout(long long max_items) {
    LatLayout L;
    L.max_items = (int)max_items;
    size_t off = kWsHeaderBytes;
    L.items = off;
    off = align_up(off + sizeof(WorkItem) * (size_t)max_items);
    L.tickets = off;
    off = align_up(off + sizeof(int) * 2 * (size_t)max_items);  // one ticket per CTA of a pair
    L.pml = off;
    off = align_up(off + sizeof(float) * 2 * kLatRows * (size_t)max_items);
    L.po = off;
    off = align_up(off + sizeof(float) * (size_t)kLatRows * kLatDv * (size_t)max_items);
    L.total = off;
    return L;
}

LatLayout mla_layout(const mla_params* p) {
    const long long tiles = p->num_q_heads / kLatRows;
    return lat_layout(kLatTargetCtas + tiles * (long long)p->max_num_tokens + tiles);
}

// ---------------------------- sparse --------------------------------------
int check_sparse_params(const sparse_params* p) {
    if (!p) return fail(RPA_ERR_NULL, "params is NULL");
    if (p->struct_size < sizeof(sparse_params)) return fail(RPA_ERR_VALUE, "sparse_params.struct_size too small");
    if (p->version != RPA_ABI_VERSION) return fail(RPA_ERR_VALUE, "sparse_params.version %u != %d", p->version, RPA_ABI_VERSION);
    if (p->batch <= 0 || p->num_queries <= 0 || p->num_heads <= 0 || p->topk <= 0 || p->read_block <= 0 ||
        p->page_size <= 0 || p->max_pages <= 0 || p->total_num_pages <= 0 || p->seq_len < 0)
        return fail(RPA_ERR_SHAPE, "all sizes must be positive");
    if (p->dk != kLatDk || p->dv != kLatDv)
        return fail(RPA_ERR_UNSUPPORTED, "sparse MLA supports dk 576 and dv 512 (got %d, %d)", p->dk, p->dv);
    if (p->row_stride < p->dk || p->row_stride % 8) return fail(RPA_ERR_SHAPE, "row_stride must be >= dk and a multiple of 8");
    if (p->num_heads % kLatRows) return fail(RPA_ERR_UNSUPPORTED, "num_heads must be a multiple of %d", kLatRows);
    if (p->page_size % p->read_block) return fail(RPA_ERR_SHAPE, "read_block must divide page_size");
    if (!(p->sm_scale > 0.f) || !isfinite(p->sm_scale)) return fail(RPA_ERR_VALUE, "sm_scale is required (> 0)");
    if ((long long)p->topk * p->read_block > INT32_MAX / 2) return fail(RPA_ERR_SHAPE, "topk * read_block too large");
    if ((long long)p->max_pages * p->page_size < p->seq_len) return fail(RPA_ERR_SHAPE, "max_pages * page_size < seq_len");
    return RPA_OK;
}

LatLayout sparse_layout(const sparse_params* p, int* splits) {
    const int sp = sparse_num_splits(p->batch, p->num_queries, p->num_heads, p->topk * p->read_block);
    if (splits) *splits = sp;
    const long long items = (long long)p->batch * p->num_queries * (p->num_heads / kLatRows) * sp;
    return lat_layout(sp > 1 ? items : 0);
}

// The packed-ragged mode as a sparse problem of one batch entry and num_tokens queries
// (checked by check_sparse_params), plus its own checks.
int ragged_as_sparse(const sparse_ragged_params* p, sparse_params& sp) {
    if (!p) return fail(RPA_ERR_NULL, "params is NULL");
    if (p->struct_size < sizeof(sparse_ragged_params)) return fail(RPA_ERR_VALUE, "sparse_ragged_params.struct_size too small");
    if (p->version != RPA_ABI_VERSION) return fail(RPA_ERR_VALUE, "sparse_ragged_params.version %u != %d", p->version, RPA_ABI_VERSION);
    if (p->num_seqs <= 0 || p->num_page_ids <= 0) return fail(RPA_ERR_SHAPE, "all sizes must be positive");
    if (p->dv % 8 || p->rope % 8) return fail(RPA_ERR_SHAPE, "dv and rope must be multiples of 8");
    memset(&sp, 0, sizeof sp);
    sp.struct_size = sizeof(sparse_params);
    sp.version = RPA_ABI_VERSION;
    sp.batch = 1;
    sp.num_queries = p->num_tokens;
    sp.num_heads = p->num_heads;
    sp.dk = p->dv + p->rope;
    sp.dv = p->dv;
    sp.row_stride = p->row_stride;
    sp.topk = p->topk;
    sp.read_block = p->read_block;
    sp.page_size = p->page_size;
    sp.max_pages = p->num_page_ids;
    sp.total_num_pages = p->total_num_pages;
    sp.seq_len = 0;
    sp.sm_scale = p->sm_scale;
    return check_sparse_params(&sp);
}

struct RaggedLayout {
    LatLayout lat;
    size_t q_bound, q_base, total;
};

RaggedLayout ragged_layout(const sparse_params& sp, int* splits) {
    RaggedLayout L;
    L.lat = sparse_layout(&sp, splits);
    size_t off = align_up(L.lat.total);
    L.q_bound = off;
    off = align_up(off + sizeof(int32_t) * (size_t)sp.num_queries);
    L.q_base = off;
    off = align_up(off + sizeof(int32_t) * (size_t)sp.num_queries);
    L.total = off;
    return L;
}

}  // namespace

extern "C" {

int rpa_version(void) { return RPA_ABI_VERSION; }

const char* rpa_last_error(void) { return g_err; }

int rpa_workspace_size(const rpa_params* p, size_t* bytes) {
    int rc = check_rpa_params(p);
    if (rc) return rc;
    if (!bytes) return fail(RPA_ERR_NULL, "bytes is NULL");
    *bytes = rpa_layout(p).total;
    return RPA_OK;
}

// Validates an rpa_forward call and fills the kernels' argument block.
static int rpa_prepare(const rpa_params* p, const void* q, const void* kv_pages, const int32_t* kv_lens,
                       const int32_t* page_indices, const int32_t* cu_q_lens, const int32_t* num_seqs, void* out,
                       void* workspace, size_t workspace_bytes, RpaArgs& a, int& sms) {
    int rc = check_rpa_params(p);
    if (rc) return rc;
    if (!q || !kv_pages || !kv_lens || !page_indices || !cu_q_lens || !num_seqs || !out)
        return fail(RPA_ERR_NULL, "a tensor pointer is NULL");
    if (!aligned16(q) || !aligned16(kv_pages) || !aligned16(out)) return fail(RPA_ERR_VALUE, "q, kv_pages and out must be 16-byte aligned");
    if (out == q || out == kv_pages) return fail(RPA_ERR_VALUE, "out must not alias q or kv_pages");
    if (p->head_dim == 96 || p->head_dim == 192) {
        // the prefill kernel runs these at the next multiple of 128 with the tensor maps'
        // zero fill for the missing dims, which needs its TMA path
        const int ps = p->page_size;
        if (p->kv_dtype != RPA_DTYPE_BF16 || p->k_scale != 0.f || p->v_scale != 0.f || mild_mask(p->mask_value) ||
            (ps & (ps - 1)) != 0 || ps < 8)
            return fail(RPA_ERR_UNSUPPORTED,
                        "head_dim %d attention needs a bf16 cache without scales, a power-of-two page_size >= 8 "
                        "and a mask_value at or below -1e30", p->head_dim);
    }
    const RpaLayout L = rpa_layout(p);
    rc = check_workspace(workspace, workspace_bytes, L.total);
    if (rc) return rc;
    sms = num_sms_current();
    if (!sms) return fail(RPA_ERR_CUDA, "no CUDA device");
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    memset(&a, 0, sizeof a);
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.kv_pages = kv_pages;
    a.kv_lens = kv_lens;
    a.page_indices = page_indices;
    a.cu_q_lens = cu_q_lens;
    a.num_seqs = num_seqs;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.max_num_tokens = p->max_num_tokens;
    a.num_q_heads = p->num_q_heads;
    a.num_kv_heads = p->num_combined_kv_heads / 2;
    a.head_dim = p->head_dim;
    a.total_num_pages = p->total_num_pages;
    a.page_size = p->page_size;
    a.max_num_seqs = p->max_num_seqs;
    a.pages_per_seq = p->pages_per_seq;
    a.kv_byte = p->kv_dtype != RPA_DTYPE_BF16;
    a.kv_int8 = p->kv_dtype == RPA_DTYPE_INT8;
    a.kv_int4 = p->kv_dtype == RPA_DTYPE_INT4;
    a.sm_scale = p->sm_scale;
    a.soft_cap = p->soft_cap;
    a.sliding_window = p->sliding_window;
    a.mask_mild = mild_mask(p->mask_value) ? 1 : 0;
    a.mask_value = resolve_mask(p->mask_value);
    a.batch_kind = rpa_batch_kind(p);
    a.has_scale = p->k_scale != 0.f || p->v_scale != 0.f;
    a.k_scale_or_one = p->k_scale != 0.f ? p->k_scale : 1.f;
    a.v_scale_or_one = p->v_scale != 0.f ? p->v_scale : 1.f;
    a.decode_heads = decode_heads_for(p->head_dim, p->kv_dtype != RPA_DTYPE_BF16);
    a.num_sms = sms;
    a.overlap = prof_enabled() ? 0 : 1;
    rpa_rates(p->head_dim, a.kv_byte != 0, a.has_scale != 0,
              rpa_pow2_scale(a.k_scale_or_one) && rpa_pow2_scale(a.v_scale_or_one), &a.pre_flops_per_ns_sm,
              &a.dec_bytes_per_ns_sm);
    a.item_cost_keys = rpa_item_cost_keys(a.kv_byte || a.has_scale);
    a.decode_per_sm = rpa_decode_ctas_per_sm(a);
    if (a.decode_per_sm <= 0) return fail(RPA_ERR_CUDA, "decode kernel occupancy query failed");
    a.hdr = reinterpret_cast<WsHeader*>(ws);
    a.dec_items = reinterpret_cast<WorkItem*>(ws + L.items_dec);
    a.pre_items = reinterpret_cast<WorkItem*>(ws + L.items_pre);
    a.tickets = reinterpret_cast<int*>(ws + L.tickets);
    a.cta_first = reinterpret_cast<int*>(ws + L.cta_first);
    a.partial_ml = reinterpret_cast<float*>(ws + L.pml);
    a.partial_o = reinterpret_cast<float*>(ws + L.po);
    a.max_dec_items = L.max_dec;
    a.max_pre_items = L.max_pre;
    return RPA_OK;
}

// Validates an rpa_update_kv_cache call (the workspace is checked by the caller) and fills the
// cache-write kernel's argument block.
static int rpa_update_prepare(const rpa_params* p, const void* new_k, const void* new_v, void* kv_pages,
                              const int32_t* kv_lens, const int32_t* page_indices, const int32_t* cu_q_lens,
                              const int32_t* num_seqs, uint32_t* err, RpaUpdateArgs& a) {
    int rc = check_rpa_params(p);
    if (rc) return rc;
    if (!new_k || !new_v || !kv_pages || !kv_lens || !page_indices || !cu_q_lens || !num_seqs)
        return fail(RPA_ERR_NULL, "a tensor pointer is NULL");
    if (!aligned16(new_k) || !aligned16(new_v) || !aligned16(kv_pages))
        return fail(RPA_ERR_VALUE, "new_k, new_v and kv_pages must be 16-byte aligned");
    a.new_k = new_k;
    a.new_v = new_v;
    a.kv_pages = kv_pages;
    a.kv_lens = kv_lens;
    a.page_indices = page_indices;
    a.cu_q_lens = cu_q_lens;
    a.num_seqs = num_seqs;
    a.err = err;
    a.max_num_tokens = p->max_num_tokens;
    a.num_kv_heads = p->num_combined_kv_heads / 2;
    a.head_dim = p->head_dim;
    a.row_bytes = p->kv_dtype == RPA_DTYPE_BF16 ? p->head_dim * 2 : p->kv_dtype == RPA_DTYPE_INT4 ? p->head_dim / 2 : p->head_dim;
    a.total_num_pages = p->total_num_pages;
    a.page_size = p->page_size;
    a.max_num_seqs = p->max_num_seqs;
    a.pages_per_seq = p->pages_per_seq;
    return RPA_OK;
}

int rpa_forward(const rpa_params* p, const void* q, const void* kv_pages, const int32_t* kv_lens,
                const int32_t* page_indices, const int32_t* cu_q_lens, const int32_t* num_seqs, void* out,
                void* workspace, size_t workspace_bytes, rpa_stream_t stream) {
    RpaArgs a;
    int sms = 0;
    const int rc = rpa_prepare(p, q, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs, out, workspace,
                               workspace_bytes, a, sms);
    if (rc) return rc;
    cudaError_t e = launch_rpa_forward(a, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "rpa_forward launch");
    return RPA_OK;
}

int rpa_update_kv_cache(const rpa_params* p, const void* new_k, const void* new_v, void* kv_pages,
                        const int32_t* kv_lens, const int32_t* page_indices, const int32_t* cu_q_lens,
                        const int32_t* num_seqs, void* workspace, size_t workspace_bytes, rpa_stream_t stream) {
    if (workspace && workspace_bytes < (size_t)kWsHeaderBytes) return fail(RPA_ERR_WORKSPACE, "workspace smaller than 256 bytes");
    RpaUpdateArgs a;
    const int rc = rpa_update_prepare(p, new_k, new_v, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs,
                                      workspace ? &reinterpret_cast<WsHeader*>(workspace)->error_bits : nullptr, a);
    if (rc) return rc;
    const int sms = num_sms_current();
    if (!sms) return fail(RPA_ERR_CUDA, "no CUDA device");
    cudaError_t e = launch_rpa_update(a, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "rpa_update_kv_cache launch");
    return RPA_OK;
}

int rpa_forward_update(const rpa_params* p, const void* q, const void* new_k, const void* new_v, void* kv_pages,
                       const int32_t* kv_lens, const int32_t* page_indices, const int32_t* cu_q_lens,
                       const int32_t* num_seqs, void* out, void* workspace, size_t workspace_bytes,
                       rpa_stream_t stream) {
    RpaArgs a;
    int sms = 0;
    int rc = rpa_prepare(p, q, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs, out, workspace, workspace_bytes,
                         a, sms);
    if (rc) return rc;
    if (out == new_k || out == new_v) return fail(RPA_ERR_VALUE, "out must not alias new_k or new_v");
    RpaUpdateArgs u;
    rc = rpa_update_prepare(p, new_k, new_v, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs,
                            &a.hdr->error_bits, u);
    if (rc) return rc;
    cudaError_t e = launch_rpa_forward_update(a, u, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "rpa_forward_update launch");
    return RPA_OK;
}

int mla_workspace_size(const mla_params* p, size_t* bytes) {
    int rc = check_mla_params(p);
    if (rc) return rc;
    if (!bytes) return fail(RPA_ERR_NULL, "bytes is NULL");
    *bytes = mla_layout(p).total;
    return RPA_OK;
}

static void mla_update_args(const mla_params* p, const void* new_kv_c, const void* new_k_pe, void* cache_kv_c,
                            void* cache_k_pe, const int32_t* kv_lens, const int32_t* page_indices,
                            const int32_t* cu_q_lens, const int32_t* distribution, uint32_t* err, MlaUpdateArgs& a) {
    a.new_kv_c = static_cast<const __nv_bfloat16*>(new_kv_c);
    a.new_k_pe = static_cast<const __nv_bfloat16*>(new_k_pe);
    a.cache_kv_c = static_cast<__nv_bfloat16*>(cache_kv_c);
    a.cache_k_pe = static_cast<__nv_bfloat16*>(cache_k_pe);
    a.kv_lens = kv_lens;
    a.page_indices = page_indices;
    a.cu_q_lens = cu_q_lens;
    a.distribution = distribution;
    a.err = err;
    a.max_num_tokens = p->max_num_tokens;
    a.lkv_dim = p->lkv_dim;
    a.r_dim = p->r_dim;
    a.lkv_pad = p->lkv_dim_pad;
    a.r_pad = p->r_dim_pad;
    a.total_num_pages = p->total_num_pages;
    a.page_size = p->page_size;
    a.max_num_seqs = p->max_num_seqs;
    a.pages_per_seq = p->pages_per_seq;
}

int mla_update_kv_cache(const mla_params* p, const void* new_kv_c, const void* new_k_pe, void* cache_kv_c,
                        void* cache_k_pe, const int32_t* kv_lens, const int32_t* page_indices,
                        const int32_t* cu_q_lens, const int32_t* distribution, void* workspace,
                        size_t workspace_bytes, rpa_stream_t stream) {
    int rc = check_mla_params(p);
    if (rc) return rc;
    if (!new_kv_c || !new_k_pe || !cache_kv_c || !cache_k_pe || !kv_lens || !page_indices || !cu_q_lens ||
        !distribution)
        return fail(RPA_ERR_NULL, "a tensor pointer is NULL");
    if (!aligned16(new_kv_c) || !aligned16(new_k_pe) || !aligned16(cache_kv_c) || !aligned16(cache_k_pe))
        return fail(RPA_ERR_VALUE, "tensors must be 16-byte aligned");
    if (workspace && workspace_bytes < (size_t)kWsHeaderBytes) return fail(RPA_ERR_WORKSPACE, "workspace smaller than 256 bytes");
    const int sms = num_sms_current();
    if (!sms) return fail(RPA_ERR_CUDA, "no CUDA device");
    MlaUpdateArgs a;
    mla_update_args(p, new_kv_c, new_k_pe, cache_kv_c, cache_k_pe, kv_lens, page_indices, cu_q_lens, distribution,
                    workspace ? &reinterpret_cast<WsHeader*>(workspace)->error_bits : nullptr, a);
    cudaError_t e = launch_mla_update(a, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "mla_update_kv_cache launch");
    return RPA_OK;
}

int mla_rpa_forward(const mla_params* p, const void* ql_nope, const void* q_pe, const void* new_kv_c,
                    const void* new_k_pe, void* cache_kv_c, void* cache_k_pe, const int32_t* kv_lens,
                    const int32_t* page_indices, const int32_t* cu_q_lens, const int32_t* distribution, void* out,
                    void* workspace, size_t workspace_bytes, rpa_stream_t stream) {
    int rc = check_mla_params(p);
    if (rc) return rc;
    rc = check_mla_attn_shape(p);
    if (rc) return rc;
    if (!ql_nope || !q_pe || !new_kv_c || !new_k_pe || !cache_kv_c || !cache_k_pe || !kv_lens || !page_indices ||
        !cu_q_lens || !distribution || !out)
        return fail(RPA_ERR_NULL, "a tensor pointer is NULL");
    if (!aligned16(ql_nope) || !aligned16(q_pe) || !aligned16(new_kv_c) || !aligned16(new_k_pe) ||
        !aligned16(cache_kv_c) || !aligned16(cache_k_pe) || !aligned16(out))
        return fail(RPA_ERR_VALUE, "tensors must be 16-byte aligned");
    if (out == ql_nope || out == cache_kv_c) return fail(RPA_ERR_VALUE, "out must not alias an input");
    const LatLayout L = mla_layout(p);
    rc = check_workspace(workspace, workspace_bytes, L.total);
    if (rc) return rc;
    const int sms = num_sms_current();
    if (!sms) return fail(RPA_ERR_CUDA, "no CUDA device");
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    MlaUpdateArgs u;
    mla_update_args(p, new_kv_c, new_k_pe, cache_kv_c, cache_k_pe, kv_lens, page_indices, cu_q_lens, distribution,
                    &reinterpret_cast<WsHeader*>(ws)->error_bits, u);
    LatentArgs a;
    memset(&a, 0, sizeof a);
    a.sparse = 0;
    a.num_heads = p->num_q_heads;
    // fp8 queries: the scores carry q_scale on top of sm_scale (one product, as a float)
    a.q_fp8 = mla_q_dtype(p) == RPA_DTYPE_FP8_E4M3 ? 1 : 0;
    a.sm_scale = mla_q_scale(p) != 0.f ? p->sm_scale * mla_q_scale(p) : p->sm_scale;
    a.soft_cap = p->soft_cap;
    a.sliding_window = p->sliding_window;
    a.mask_mild = mild_mask(p->mask_value) ? 1 : 0;
    a.mask_value = resolve_mask(p->mask_value);
    a.ql_nope = static_cast<const __nv_bfloat16*>(ql_nope);
    a.q_pe = static_cast<const __nv_bfloat16*>(q_pe);
    a.cache_kv_c = static_cast<const __nv_bfloat16*>(cache_kv_c);
    a.cache_k_pe = static_cast<const __nv_bfloat16*>(cache_k_pe);
    a.kv_lens = kv_lens;
    a.page_indices = page_indices;
    a.cu_q_lens = cu_q_lens;
    a.distribution = distribution;
    a.max_num_tokens = p->max_num_tokens;
    a.max_num_seqs = p->max_num_seqs;
    a.pages_per_seq = p->pages_per_seq;
    a.lkv_pad = p->lkv_dim_pad;
    a.r_pad = p->r_dim_pad;
    a.out_bf16 = static_cast<__nv_bfloat16*>(out);
    a.target_items = sms;
    a.total_num_pages = p->total_num_pages;
    a.page_size = p->page_size;
    a.hdr = reinterpret_cast<WsHeader*>(ws);
    a.items = reinterpret_cast<WorkItem*>(ws + L.items);
    a.tickets = reinterpret_cast<int*>(ws + L.tickets);
    a.partial_ml = reinterpret_cast<float*>(ws + L.pml);
    a.partial_o = reinterpret_cast<float*>(ws + L.po);
    a.max_items = L.max_items;
    // the cache write shares the plan's launch; attention starts once both have ended
    cudaError_t e = launch_mla_forward_update(a, u, sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "mla_rpa_forward launch");
    return RPA_OK;
}

int sparse_mla_workspace_size(const sparse_params* p, size_t* bytes) {
    int rc = check_sparse_params(p);
    if (rc) return rc;
    if (!bytes) return fail(RPA_ERR_NULL, "bytes is NULL");
    *bytes = sparse_layout(p, nullptr).total;
    return RPA_OK;
}

int sparse_mla_forward(const sparse_params* p, const void* q, const void* cache, const int32_t* indices,
                       const int32_t* positions, const int32_t* page_table, float* out, void* workspace,
                       size_t workspace_bytes, rpa_stream_t stream) {
    int rc = check_sparse_params(p);
    if (rc) return rc;
    if (!q || !cache || !indices || !positions || !page_table || !out) return fail(RPA_ERR_NULL, "a tensor pointer is NULL");
    if (!aligned16(q) || !aligned16(cache) || !aligned16(out)) return fail(RPA_ERR_VALUE, "q, cache and out must be 16-byte aligned");
    int splits = 1;
    const LatLayout L = sparse_layout(p, &splits);
    rc = check_workspace(workspace, workspace_bytes, L.total);
    if (rc) return rc;
    const int sms = num_sms_current();
    if (!sms) return fail(RPA_ERR_CUDA, "no CUDA device");
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    LatentArgs a;
    memset(&a, 0, sizeof a);
    a.sparse = 1;
    a.num_heads = p->num_heads;
    a.sm_scale = p->sm_scale;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.cache = static_cast<const __nv_bfloat16*>(cache);
    a.indices = indices;
    a.positions = positions;
    a.page_table = page_table;
    a.batch = p->batch;
    a.num_queries = p->num_queries;
    a.topk = p->topk;
    a.read_block = p->read_block;
    a.max_pages = p->max_pages;
    a.seq_len = p->seq_len;
    a.row_stride = p->row_stride;
    a.sparse_splits = splits;
    a.out_f32 = out;
    a.total_num_pages = p->total_num_pages;
    a.page_size = p->page_size;
    a.hdr = reinterpret_cast<WsHeader*>(ws);
    a.items = nullptr;
    a.tickets = reinterpret_cast<int*>(ws + L.tickets);
    a.partial_ml = reinterpret_cast<float*>(ws + L.pml);
    a.partial_o = reinterpret_cast<float*>(ws + L.po);
    a.max_items = L.max_items;
    cudaError_t e = launch_sparse_forward(a, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_forward launch");
    return RPA_OK;
}

int sparse_mla_ragged_workspace_size(const sparse_ragged_params* p, size_t* bytes) {
    sparse_params sp;
    int rc = ragged_as_sparse(p, sp);
    if (rc) return rc;
    if (!bytes) return fail(RPA_ERR_NULL, "bytes is NULL");
    *bytes = ragged_layout(sp, nullptr).total;
    return RPA_OK;
}

int sparse_mla_write_and_attend_ragged(const sparse_ragged_params* p, const void* ql, const void* qpe,
                                       const void* kvc, const void* kpe, void* cache, const int32_t* topk,
                                       const int32_t* positions, const int32_t* loc, const int32_t* seq_lens,
                                       const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                                       const int32_t* page_indices, float* out, void* workspace,
                                       size_t workspace_bytes, rpa_stream_t stream) {
    sparse_params sp;
    int rc = ragged_as_sparse(p, sp);
    if (rc) return rc;
    if (!ql || !qpe || !cache || !topk || !positions || !seq_lens || !cu_q_lens || !cu_kv_lens || !page_indices ||
        !out)
        return fail(RPA_ERR_NULL, "a tensor pointer is NULL");
    const bool write = kvc || kpe;
    if (write && (!kvc || !kpe || !loc)) return fail(RPA_ERR_NULL, "kvc, kpe and loc go together");
    if (!aligned16(ql) || !aligned16(qpe) || !aligned16(cache) || !aligned16(out) ||
        (write && (!aligned16(kvc) || !aligned16(kpe))))
        return fail(RPA_ERR_VALUE, "ql, qpe, kvc, kpe, cache and out must be 16-byte aligned");
    int splits = 1;
    const RaggedLayout L = ragged_layout(sp, &splits);
    rc = check_workspace(workspace, workspace_bytes, L.total);
    if (rc) return rc;
    const int sms = num_sms_current();
    if (!sms) return fail(RPA_ERR_CUDA, "no CUDA device");
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    SparseRaggedPrepArgs pa;
    pa.kvc = write ? static_cast<const __nv_bfloat16*>(kvc) : nullptr;
    pa.kpe = static_cast<const __nv_bfloat16*>(kpe);
    pa.cache = static_cast<__nv_bfloat16*>(cache);
    pa.loc = loc;
    pa.seq_lens = seq_lens;
    pa.cu_q_lens = cu_q_lens;
    pa.cu_kv_lens = cu_kv_lens;
    pa.q_bound = reinterpret_cast<int32_t*>(ws + L.q_bound);
    pa.q_base = reinterpret_cast<int32_t*>(ws + L.q_base);
    pa.num_tokens = p->num_tokens;
    pa.num_seqs = p->num_seqs;
    pa.dv = p->dv;
    pa.rope = p->rope;
    pa.row_stride = p->row_stride;
    pa.page_size = p->page_size;
    pa.total_num_pages = p->total_num_pages;
    LatentArgs a;
    memset(&a, 0, sizeof a);
    a.sparse = 1;
    a.num_heads = p->num_heads;
    a.sm_scale = p->sm_scale;
    a.q = nullptr;  // split query: ql_nope and q_pe
    a.ql_nope = static_cast<const __nv_bfloat16*>(ql);
    a.q_pe = static_cast<const __nv_bfloat16*>(qpe);
    a.cache = static_cast<const __nv_bfloat16*>(cache);
    a.indices = topk;
    a.positions = positions;
    a.page_table = page_indices;
    a.q_bound = pa.q_bound;
    a.q_base = pa.q_base;
    a.batch = 1;
    a.num_queries = p->num_tokens;
    a.topk = p->topk;
    a.read_block = p->read_block;
    a.max_pages = p->num_page_ids;
    a.seq_len = 0;
    a.row_stride = p->row_stride;
    a.sparse_splits = splits;
    a.out_f32 = out;
    a.total_num_pages = p->total_num_pages;
    a.page_size = p->page_size;
    a.hdr = reinterpret_cast<WsHeader*>(ws);
    a.items = nullptr;
    a.tickets = reinterpret_cast<int*>(ws + L.lat.tickets);
    a.partial_ml = reinterpret_cast<float*>(ws + L.lat.pml);
    a.partial_o = reinterpret_cast<float*>(ws + L.lat.po);
    a.max_items = L.lat.max_items;
    cudaError_t e = launch_sparse_ragged(pa, a, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_write_and_attend_ragged launch");
    return RPA_OK;
}

int rpa_selftest_bounded_wait(void* workspace, size_t workspace_bytes, rpa_stream_t stream) {
    if (!workspace) return fail(RPA_ERR_NULL, "workspace is NULL");
    if (workspace_bytes < (size_t)kWsHeaderBytes) return fail(RPA_ERR_WORKSPACE, "workspace smaller than 256 bytes");
    cudaError_t e = launch_wait_selftest(&reinterpret_cast<WsHeader*>(workspace)->error_bits,
                                         reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "rpa_selftest_bounded_wait launch");
    return RPA_OK;
}

int rpa_check_device_status(void* workspace, uint32_t* bits, rpa_stream_t stream) {
    if (!workspace) return fail(RPA_ERR_NULL, "workspace is NULL");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "rpa_check_device_status sync");
    e = cudaMemcpy(&v, &reinterpret_cast<WsHeader*>(workspace)->error_bits, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "rpa_check_device_status read");
    if (v) {
        e = cudaMemset(&reinterpret_cast<WsHeader*>(workspace)->error_bits, 0, sizeof v);
        if (e != cudaSuccess) return cuda_fail(e, "rpa_check_device_status clear");
    }
    if (bits) *bits = v;
    if (v) return fail(RPA_ERR_DEVICE_CHECK, "device-side check failed: bits 0x%x", v);
    return RPA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// rpa_forward_noalloc: rpa_forward for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a plugin running inside a host application
// whose memory manager owns all of the device memory, or a serving loop that must not
// allocate after start-up because cudaMalloc can synchronise the device.  This entry
// point gives them rpa_forward without a workspace argument: its scratch (work lists,
// split-KV partials, counters) is the fixed file-scope array below, which every GPU
// that loads this library holds until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = RPA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch in the context current on this thread (the host-side
// name of the array is only a stand-in, never a device address). It is looked up on every
// call rather than cached: a host application may make its own (non-primary) context
// current, or reset the device between calls, and either gives the array another address.
// The lookup is a host-side table read once the library's device code is loaded in that
// context (the first call there loads it).
void* noalloc_scratch_ptr(int* rc) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
        *rc = cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol, "rpa_forward_noalloc: cudaGetSymbolAddress");
        return nullptr;
    }
    return p;
}

}  // namespace

extern "C" int rpa_forward_noalloc(const rpa_params* p, const void* q, const void* kv_pages, const int32_t* kv_lens,
                                   const int32_t* page_indices, const int32_t* cu_q_lens, const int32_t* num_seqs,
                                   void* out, rpa_stream_t stream) {
    int rc = check_rpa_params(p);
    if (rc) return rc;
    const size_t need = rpa_layout(p).total;
    if (need > kNoAllocScratchBytes)
        return fail(RPA_ERR_WORKSPACE,
                    "rpa_forward_noalloc: these maxima need %zu bytes of scratch but the library's static scratch "
                    "holds %zu; use rpa_forward with a caller-allocated workspace",
                    need, kNoAllocScratchBytes);
    rc = RPA_OK;
    void* scratch = noalloc_scratch_ptr(&rc);
    if (!scratch) return rc;
    return rpa_forward(p, q, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs, out, scratch, kNoAllocScratchBytes,
                       stream);
}
