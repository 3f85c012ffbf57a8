/*
 * Float64 CPU oracle for ragged paged attention and its two variants.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * statement of what the GPU library computes.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the product
 * path never links, imports or calls it, and it shares no code, header or
 * constant table with the CUDA sources.
 *
 * Every function follows one passage of the source pages:
 *   - oracle_rpa                  : tpu-inference "ragged_paged_attention/v2/kernel.py",
 *                                   function ref_ragged_paged_attention (the
 *                                   reference semantics of the RPA v2 kernel).
 *   - oracle_rpa_update_kv_cache  : no passage on the pages (the v2 wrapper only
 *                                   carries a TODO for a cache-write kernel); defined
 *                                   by analogy with the MLA update_kv_cache below.
 *   - oracle_mla_update_kv_cache  : tpu-inference "mla/v1/kernel.py", update_kv_cache.
 *   - oracle_mla                  : tpu-inference "mla/v1/kernel.py",
 *                                   ref_mla_ragged_paged_attention.
 *   - oracle_sparse_mla           : sglang-jax "dsa/sparse_mla_prefill.py",
 *                                   _sparse_mla_kernel_chunked_hminor (validity rule,
 *                                   -inf-safe softmax) and units_to_token_ids.
 *   - oracle_sparse_ragged_write,   same page, prefill_write_and_attend_ragged (the
 *     oracle_sparse_mla_ragged      self-write, the request of each token, its causal
 *                                   bound and page base) and the ragged branch of
 *                                   sparse_mla_attention.
 *
 * Arithmetic is IEEE binary64 except where the pages fix a precision: the RPA
 * reference dequantises K and V as float32(k) * k_scale rounded to the query
 * dtype (bfloat16) before the dot products, and this file does exactly that.
 * Scores are exact-order float64 sums; no blocking, no online softmax.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_PAGE (-2)
#define ORACLE_ERR_LEN (-3)

/* dtype codes understood by the oracle */
#define ORACLE_BF16 1
#define ORACLE_E4M3 2
#define ORACLE_INT8 3
#define ORACLE_INT4 4

/* ------------------------------------------------------------------ */
/* Number formats, decoded from their definitions.                     */
/* ------------------------------------------------------------------ */

/* bfloat16 is the upper 16 bits of an IEEE binary32 value. */
static float bf16_bits_to_f32(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* float8 e4m3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities, S.1111.111 is NaN, exponent 0 is
 * subnormal with scale 2^-6. */
static float e4m3_bits_to_f32(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9); /* (m/8) * 2^(1-7) */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return (float)(sign ? -v : v); /* exact: at most 4 significant bits */
}

/* Round a binary32 value to the nearest bfloat16, ties to even. */
static float f32_round_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) return f; /* NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    u &= 0xFFFF0000u;
    float r;
    memcpy(&r, &u, sizeof r);
    return r;
}

/* int8: a two's-complement byte; the RPA reference promotes it exactly (it is a bfloat16
 * value) or, with a scale, multiplies float32(x) by it like any other KV dtype. */
static float int8_to_f32(uint8_t b) { return (float)(b < 128 ? (int)b : (int)b - 256); }

/* int4: a two's-complement nibble (values -8 .. 7), two to a byte along the head dimension:
 * element 2i of a row is the low nibble of the row's byte i, element 2i+1 the high nibble (the
 * v2 kernel's packed integer loads unpack several values from one word the same way, lowest
 * bits first).  Like int8 it is promoted exactly, or scaled in float32. */
static float int4_to_f32(uint8_t nib) { return (float)(nib < 8 ? (int)nib : (int)nib - 16); }

static float load_elem(const void* base, size_t idx, int dtype) {
    if (dtype == ORACLE_E4M3) return e4m3_bits_to_f32(((const uint8_t*)base)[idx]);
    if (dtype == ORACLE_INT8) return int8_to_f32(((const uint8_t*)base)[idx]);
    if (dtype == ORACLE_INT4) {
        const uint8_t b = ((const uint8_t*)base)[idx >> 1];
        return int4_to_f32((idx & 1) ? (uint8_t)(b >> 4) : (uint8_t)(b & 15));
    }
    return bf16_bits_to_f32(((const uint16_t*)base)[idx]);
}

/* K or V element as the RPA reference sees it: optionally scaled in float32
 * and rounded back to the query dtype (bfloat16). */
static double rpa_kv_value(const void* base, size_t idx, int dtype, float scale) {
    float x = load_elem(base, idx, dtype);
    if (scale != 0.0f) {
        volatile float prod = x * scale; /* one binary32 multiply */
        x = f32_round_to_bf16(prod);
    }
    return (double)x;
}

/* Exported for the pin tests: decode / round a single value. */
double oracle_decode_bf16(uint16_t bits) { return (double)bf16_bits_to_f32(bits); }
double oracle_decode_e4m3(uint8_t bits) { return (double)e4m3_bits_to_f32(bits); }
double oracle_decode_int8(uint8_t bits) { return (double)int8_to_f32(bits); }
double oracle_decode_int4(uint8_t nibble) { return (double)int4_to_f32((uint8_t)(nibble & 15)); }
double oracle_round_f32_to_bf16(float f) { return (double)f32_round_to_bf16(f); }

/* ------------------------------------------------------------------ */
/* Softmax of one score row followed by the weighted sum of value rows. */
/* ------------------------------------------------------------------ */

/* p_k = exp(x_k - max x); out = sum_k p_k v_k / sum_k p_k.
 * A row whose scores are all -inf (nothing selected) returns zeros, the
 * convention the sparse kernel states with its (l == 0 ? 1 : l) divide. */
static void softmax_weights(double* x, int n, double* l_out) {
    double m = -INFINITY;
    for (int k = 0; k < n; ++k)
        if (x[k] > m) m = x[k];
    double l = 0.0;
    if (m == -INFINITY) {
        for (int k = 0; k < n; ++k) x[k] = 0.0;
    } else {
        for (int k = 0; k < n; ++k) {
            x[k] = exp(x[k] - m);
            l += x[k];
        }
    }
    *l_out = l;
}

static int find_seq(const int32_t* cu_q_lens, int num_seqs, int t) {
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) { /* last s with cu_q_lens[s] <= t */
        int mid = (lo + hi + 1) / 2;
        if (cu_q_lens[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

static int default_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
    nthreads = 1;
#endif
    return nthreads;
}

/* ------------------------------------------------------------------ */
/* Standard ragged paged attention (RPA v2 reference semantics).       */
/* ------------------------------------------------------------------ */

typedef struct {
    int32_t num_q_heads;
    int32_t num_combined_kv_heads; /* K at even, V at odd combined heads */
    int32_t head_dim;
    int32_t total_num_pages;
    int32_t page_size;
    int32_t max_num_seqs;
    int32_t pages_per_seq;
    int32_t kv_dtype;       /* ORACLE_BF16, ORACLE_E4M3 or ORACLE_INT8 */
    double sm_scale;
    int32_t sliding_window; /* 0 = none */
    double soft_cap;        /* 0 = none */
    double mask_value;      /* added to masked logits */
    float k_scale;          /* 0 = none */
    float v_scale;          /* 0 = none */
} oracle_rpa_params;

/* q: bf16 [*, Hq, D]; kv_pages: [P, ps, 2*Hkv, D]; page_indices [max_num_seqs, pps];
 * out: float64 [*, Hq, D], written only for the listed tokens (all tokens
 * < cu_q_lens[num_seqs] when tokens == NULL). */
int oracle_rpa(const oracle_rpa_params* p, const uint16_t* q, const void* kv_pages,
               const int32_t* kv_lens, const int32_t* page_indices, const int32_t* cu_q_lens,
               int32_t num_seqs, const int32_t* tokens, int32_t n_tokens, double* out,
               int nthreads) {
    if (!p || !q || !kv_pages || !kv_lens || !page_indices || !cu_q_lens || !out) return ORACLE_ERR_ARG;
    const int Hq = p->num_q_heads, C = p->num_combined_kv_heads, D = p->head_dim;
    const int ps = p->page_size, pps = p->pages_per_seq;
    if (C % 2 || Hq % (C / 2) || num_seqs < 0 || num_seqs > p->max_num_seqs) return ORACLE_ERR_ARG;
    const int group = Hq / (C / 2);
    for (int s = 0; s < num_seqs; ++s) { /* the reference's dynamic validation */
        int q_len = cu_q_lens[s + 1] - cu_q_lens[s], kv_len = kv_lens[s];
        if (q_len < 0 || q_len > kv_len) return ORACLE_ERR_LEN;
        int np = (kv_len + ps - 1) / ps;
        if (np > pps) return ORACLE_ERR_LEN;
        for (int pg = 0; pg < np; ++pg) {
            int32_t idx = page_indices[(size_t)s * pps + pg];
            if (idx < 0 || idx >= p->total_num_pages) return ORACLE_ERR_PAGE;
        }
    }
    const int total = num_seqs > 0 ? cu_q_lens[num_seqs] : 0;
    const int n = tokens ? n_tokens : total;
    int err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1) num_threads(default_threads(nthreads))
    for (int it = 0; it < n * Hq; ++it) {
        const int t = tokens ? tokens[it / Hq] : it / Hq;
        const int h = it % Hq;
        if (t < 0 || t >= total) {
#pragma omp atomic write
            err = ORACLE_ERR_ARG;
            continue;
        }
        const int s = find_seq(cu_q_lens, num_seqs, t);
        const int q_len = cu_q_lens[s + 1] - cu_q_lens[s];
        const int kv_len = kv_lens[s];
        const int q_pos = kv_len - q_len + (t - cu_q_lens[s]);
        const int kvh = h / group;
        double* x = (double*)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
        const uint16_t* qrow = q + ((size_t)t * Hq + h) * D;
        for (int k = 0; k < kv_len; ++k) {
            const size_t page = (size_t)page_indices[(size_t)s * pps + k / ps];
            const size_t krow = ((page * ps + k % ps) * C + 2 * kvh) * (size_t)D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += (double)bf16_bits_to_f32(qrow[d]) *
                       rpa_kv_value(kv_pages, krow + d, p->kv_dtype, p->k_scale);
            double v = p->sm_scale * dot;
            if (p->soft_cap != 0.0) v = p->soft_cap * tanh(v / p->soft_cap);
            int masked = q_pos < k;
            if (p->sliding_window > 0 && q_pos - p->sliding_window >= k) masked = 1;
            if (masked) v += p->mask_value;
            x[k] = v;
        }
        double l;
        softmax_weights(x, kv_len, &l);
        double* o = out + ((size_t)t * Hq + h) * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int k = 0; k < kv_len; ++k) {
            if (x[k] == 0.0) continue;
            const size_t page = (size_t)page_indices[(size_t)s * pps + k / ps];
            const size_t vrow = ((page * ps + k % ps) * C + 2 * kvh + 1) * (size_t)D;
            for (int d = 0; d < D; ++d)
                o[d] += x[k] * rpa_kv_value(kv_pages, vrow + d, p->kv_dtype, p->v_scale);
        }
        const double inv = l > 0.0 ? 1.0 / l : 0.0;
        for (int d = 0; d < D; ++d) o[d] *= inv;
        free(x);
    }
    return err;
}

/* Write token j of sequence i (absolute position kv_len - q_len + j) into its
 * page slot: K of KV head g to combined head 2g, V to 2g+1.  Element bytes are
 * copied unchanged.  new_k / new_v: [*, Hkv, D] in the cache dtype. */
int oracle_rpa_update_kv_cache(const oracle_rpa_params* p, const void* new_k, const void* new_v,
                               void* kv_pages, const int32_t* kv_lens, const int32_t* page_indices,
                               const int32_t* cu_q_lens, int32_t num_seqs) {
    if (!p || !new_k || !new_v || !kv_pages) return ORACLE_ERR_ARG;
    const int C = p->num_combined_kv_heads, Hkv = C / 2, D = p->head_dim, ps = p->page_size;
    /* bytes of one head row: D elements of 2, 1 or (int4) 1/2 byte */
    const size_t rowb = p->kv_dtype == ORACLE_BF16 ? (size_t)D * 2 : p->kv_dtype == ORACLE_INT4 ? (size_t)D / 2 : (size_t)D;
    for (int i = 0; i < num_seqs; ++i) {
        const int q_start = cu_q_lens[i], q_len = cu_q_lens[i + 1] - cu_q_lens[i];
        const int kv_len = kv_lens[i];
        if (q_len < 0 || q_len > kv_len) return ORACLE_ERR_LEN;
        for (int j = 0; j < q_len; ++j) {
            const int pos = kv_len - q_len + j;
            if (pos / ps >= p->pages_per_seq) return ORACLE_ERR_LEN;
            const int32_t page = page_indices[(size_t)i * p->pages_per_seq + pos / ps];
            if (page < 0 || page >= p->total_num_pages) return ORACLE_ERR_PAGE;
            for (int g = 0; g < Hkv; ++g) {
                const size_t src = ((size_t)(q_start + j) * Hkv + g) * rowb;
                const size_t dk = (((size_t)page * ps + pos % ps) * C + 2 * g) * rowb;
                memcpy((char*)kv_pages + dk, (const char*)new_k + src, rowb);
                memcpy((char*)kv_pages + dk + rowb, (const char*)new_v + src, rowb);
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* MLA latent attention (MLA v1 reference semantics).                  */
/* ------------------------------------------------------------------ */

typedef struct {
    int32_t num_q_heads;
    int32_t lkv_dim;      /* actual latent width (512); cache row is lkv_dim_pad */
    int32_t lkv_dim_pad;  /* align(lkv_dim, 128) */
    int32_t r_dim;        /* actual rope width (64) */
    int32_t r_dim_pad;    /* align(r_dim, 128) */
    int32_t total_num_pages;
    int32_t page_size;
    int32_t max_num_seqs;
    int32_t pages_per_seq;
    double sm_scale;
    int32_t sliding_window; /* 0 = none */
    double soft_cap;        /* 0 = none */
    double mask_value;      /* replaces masked logits */
    int32_t q_dtype;        /* ORACLE_BF16, or ORACLE_E4M3 for fp8 queries (ql_nope, q_pe) */
    double q_scale;         /* 0 = none; else the scores are multiplied by it (after sm_scale) */
} oracle_mla_params;

/* Query element: bfloat16, or an fp8 e4m3 byte decoded exactly. */
static double mla_q_elem(const void* base, size_t idx, int dtype) {
    if (dtype == ORACLE_E4M3) return (double)e4m3_bits_to_f32(((const uint8_t*)base)[idx]);
    return (double)bf16_bits_to_f32(((const uint16_t*)base)[idx]);
}

/* new_kv_c: bf16 [*, lkv]; new_k_pe: bf16 [*, r]; caches viewed as
 * [P, ps, lkv_pad] and [P, ps, r_pad] (the [P, ps/pk, pk, D] layout has the
 * same row-major bytes).  Columns past the actual widths are written as 0. */
int oracle_mla_update_kv_cache(const oracle_mla_params* p, const uint16_t* new_kv_c,
                               const uint16_t* new_k_pe, uint16_t* cache_kv_c, uint16_t* cache_k_pe,
                               const int32_t* kv_lens, const int32_t* page_indices,
                               const int32_t* cu_q_lens, int32_t num_seqs) {
    if (!p || !new_kv_c || !new_k_pe || !cache_kv_c || !cache_k_pe) return ORACLE_ERR_ARG;
    const int ps = p->page_size;
    for (int i = 0; i < num_seqs; ++i) {
        const int q_start = cu_q_lens[i], q_len = cu_q_lens[i + 1] - cu_q_lens[i];
        const int kv_len = kv_lens[i];
        if (q_len < 0 || q_len > kv_len) return ORACLE_ERR_LEN;
        for (int j = 0; j < q_len; ++j) {
            const int pos = kv_len - q_len + j;
            if (pos / ps >= p->pages_per_seq) return ORACLE_ERR_LEN;
            const int32_t page = page_indices[(size_t)i * p->pages_per_seq + pos / ps];
            if (page < 0 || page >= p->total_num_pages) return ORACLE_ERR_PAGE;
            const size_t slot = (size_t)page * ps + pos % ps;
            uint16_t* c = cache_kv_c + slot * p->lkv_dim_pad;
            uint16_t* r = cache_k_pe + slot * p->r_dim_pad;
            for (int d = 0; d < p->lkv_dim_pad; ++d)
                c[d] = d < p->lkv_dim ? new_kv_c[(size_t)(q_start + j) * p->lkv_dim + d] : 0;
            for (int d = 0; d < p->r_dim_pad; ++d)
                r[d] = d < p->r_dim ? new_k_pe[(size_t)(q_start + j) * p->r_dim + d] : 0;
        }
    }
    return ORACLE_OK;
}

/* ql_nope: bf16 [*, H, lkv]; q_pe: bf16 [*, H, r]; caches as above (already
 * updated).  Key = [kv_c | k_pe], value = kv_c, one latent head for all q
 * heads.  Masked logits are replaced by mask_value.  out: float64 [*, H, lkv]. */
int oracle_mla(const oracle_mla_params* p, const void* ql_nope, const void* q_pe,
               const uint16_t* cache_kv_c, const uint16_t* cache_k_pe, const int32_t* kv_lens,
               const int32_t* page_indices, const int32_t* cu_q_lens, int32_t num_seqs,
               const int32_t* tokens, int32_t n_tokens, double* out, int nthreads) {
    if (!p || !ql_nope || !q_pe || !cache_kv_c || !cache_k_pe || !out) return ORACLE_ERR_ARG;
    const int H = p->num_q_heads, L = p->lkv_dim, R = p->r_dim, ps = p->page_size;
    const int pps = p->pages_per_seq;
    if (num_seqs < 0 || num_seqs > p->max_num_seqs) return ORACLE_ERR_ARG;
    for (int s = 0; s < num_seqs; ++s) {
        int q_len = cu_q_lens[s + 1] - cu_q_lens[s], kv_len = kv_lens[s];
        if (q_len < 0 || q_len > kv_len) return ORACLE_ERR_LEN;
        int np = (kv_len + ps - 1) / ps;
        if (np > pps) return ORACLE_ERR_LEN;
        for (int pg = 0; pg < np; ++pg) {
            int32_t idx = page_indices[(size_t)s * pps + pg];
            if (idx < 0 || idx >= p->total_num_pages) return ORACLE_ERR_PAGE;
        }
    }
    const int total = num_seqs > 0 ? cu_q_lens[num_seqs] : 0;
    const int n = tokens ? n_tokens : total;
    int err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1) num_threads(default_threads(nthreads))
    for (int it = 0; it < n * H; ++it) {
        const int t = tokens ? tokens[it / H] : it / H;
        const int h = it % H;
        if (t < 0 || t >= total) {
#pragma omp atomic write
            err = ORACLE_ERR_ARG;
            continue;
        }
        const int s = find_seq(cu_q_lens, num_seqs, t);
        const int q_len = cu_q_lens[s + 1] - cu_q_lens[s];
        const int kv_len = kv_lens[s];
        const int q_pos = kv_len - q_len + (t - cu_q_lens[s]);
        const size_t qn = ((size_t)t * H + h) * L, qr = ((size_t)t * H + h) * R;  /* element offsets */
        double* x = (double*)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
        for (int k = 0; k < kv_len; ++k) {
            const size_t slot = (size_t)page_indices[(size_t)s * pps + k / ps] * ps + k % ps;
            const uint16_t* c = cache_kv_c + slot * p->lkv_dim_pad;
            const uint16_t* r = cache_k_pe + slot * p->r_dim_pad;
            double dot = 0.0;
            for (int d = 0; d < L; ++d) dot += mla_q_elem(ql_nope, qn + d, p->q_dtype) * bf16_bits_to_f32(c[d]);
            for (int d = 0; d < R; ++d) dot += mla_q_elem(q_pe, qr + d, p->q_dtype) * bf16_bits_to_f32(r[d]);
            /* the MLA kernel's order: sm_scale, then (fp8 queries) q_scale */
            double v = p->sm_scale * dot;
            if (p->q_scale != 0.0) v *= p->q_scale;
            if (p->soft_cap != 0.0) v = p->soft_cap * tanh(v / p->soft_cap);
            int masked = q_pos < k;
            if (p->sliding_window > 0 && q_pos - p->sliding_window >= k) masked = 1;
            x[k] = masked ? p->mask_value : v;
        }
        double l;
        softmax_weights(x, kv_len, &l);
        double* o = out + ((size_t)t * H + h) * L;
        for (int d = 0; d < L; ++d) o[d] = 0.0;
        for (int k = 0; k < kv_len; ++k) {
            if (x[k] == 0.0) continue;
            const size_t slot = (size_t)page_indices[(size_t)s * pps + k / ps] * ps + k % ps;
            const uint16_t* c = cache_kv_c + slot * p->lkv_dim_pad;
            for (int d = 0; d < L; ++d) o[d] += x[k] * bf16_bits_to_f32(c[d]);
        }
        const double inv = l > 0.0 ? 1.0 / l : 0.0;
        for (int d = 0; d < L; ++d) o[d] *= inv;
        free(x);
    }
    return err;
}

/* ------------------------------------------------------------------ */
/* DSA sparse MLA over a paged latent cache (per-batch page table).    */
/* ------------------------------------------------------------------ */

typedef struct {
    int32_t batch;        /* B */
    int32_t num_queries;  /* S per batch entry */
    int32_t num_heads;    /* H */
    int32_t dk;           /* 576 = 512 + 64 */
    int32_t dv;           /* 512: value = first dv latent columns */
    int32_t row_stride;   /* stored row width of the cache (640) */
    int32_t topk;         /* K unit slots per query */
    int32_t read_block;   /* RB tokens per unit */
    int32_t page_size;
    int32_t max_pages;    /* page_table row width */
    int32_t total_num_pages;
    int32_t seq_len;      /* causal bound T */
    double sm_scale;
} oracle_sparse_params;

/* q: bf16 [B, S, H, dk]; cache: bf16 [P*ps, row_stride]; indices [B, S, K]
 * unit ids (-1 = none); positions [B, S]; page_table [B, max_pages].
 * out: float64 [B, S, H, dv], written for the listed (b*S+s) queries (all
 * when queries == NULL).  Keys form a multiset: a unit named twice counts
 * twice.  A query with no valid key outputs zeros. */
int oracle_sparse_mla(const oracle_sparse_params* p, const uint16_t* q, const uint16_t* cache,
                      const int32_t* indices, const int32_t* positions, const int32_t* page_table,
                      const int32_t* queries, int32_t n_queries, double* out, int nthreads) {
    if (!p || !q || !cache || !indices || !positions || !page_table || !out) return ORACLE_ERR_ARG;
    const int B = p->batch, S = p->num_queries, H = p->num_heads, K = p->topk, RB = p->read_block;
    const int ps = p->page_size;
    const int n = queries ? n_queries : B * S;
    int err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1) num_threads(default_threads(nthreads))
    for (int it = 0; it < n; ++it) {
        const int bs = queries ? queries[it] : it;
        if (bs < 0 || bs >= B * S) {
#pragma omp atomic write
            err = ORACLE_ERR_ARG;
            continue;
        }
        const int b = bs / S;
        const int qpos = positions[bs];
        /* units -> token ids, kept when causal and inside the sequence */
        int32_t* keys = (int32_t*)malloc(sizeof(int32_t) * (size_t)K * RB + 4);
        int nk = 0;
        for (int i = 0; i < K; ++i) {
            const int u = indices[(size_t)bs * K + i];
            if (u < 0) continue;
            for (int r = 0; r < RB; ++r) {
                const long kp = (long)u * RB + r;
                if (kp <= qpos && kp < p->seq_len) keys[nk++] = (int32_t)kp;
            }
        }
        size_t* rows = (size_t*)malloc(sizeof(size_t) * (size_t)(nk > 0 ? nk : 1));
        int bad = 0;
        for (int i = 0; i < nk; ++i) {
            const int lp = keys[i] / ps;
            const int32_t page = lp < p->max_pages ? page_table[(size_t)b * p->max_pages + lp] : -1;
            if (page < 0 || page >= p->total_num_pages) bad = 1;
            rows[i] = (size_t)(page < 0 ? 0 : page) * ps + keys[i] % ps;
        }
        if (bad) {
#pragma omp atomic write
            err = ORACLE_ERR_PAGE;
            free(keys);
            free(rows);
            continue;
        }
        double* x = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
        for (int h = 0; h < H; ++h) {
            const uint16_t* qh = q + ((size_t)bs * H + h) * p->dk;
            for (int i = 0; i < nk; ++i) {
                const uint16_t* row = cache + rows[i] * p->row_stride;
                double dot = 0.0;
                for (int d = 0; d < p->dk; ++d)
                    dot += (double)bf16_bits_to_f32(qh[d]) * bf16_bits_to_f32(row[d]);
                x[i] = p->sm_scale * dot;
            }
            double l;
            softmax_weights(x, nk, &l);
            double* o = out + ((size_t)bs * H + h) * p->dv;
            for (int d = 0; d < p->dv; ++d) o[d] = 0.0;
            for (int i = 0; i < nk; ++i) {
                const uint16_t* row = cache + rows[i] * p->row_stride;
                for (int d = 0; d < p->dv; ++d) o[d] += x[i] * bf16_bits_to_f32(row[d]);
            }
            const double inv = l > 0.0 ? 1.0 / l : 0.0;
            for (int d = 0; d < p->dv; ++d) o[d] *= inv;
        }
        free(x);
        free(keys);
        free(rows);
    }
    return err;
}

/* ------------------------------------------------------------------ */
/* DSA sparse MLA, packed-ragged mode with the self-write              */
/* (sglang-jax "dsa/sparse_mla_prefill.py", prefill_write_and_attend_  */
/* ragged and the ragged branch of sparse_mla_attention).              */
/* ------------------------------------------------------------------ */

typedef struct {
    int32_t num_tokens;   /* T: queries packed along one axis */
    int32_t num_seqs;     /* S: requests (length of seq_lens) */
    int32_t num_heads;    /* H */
    int32_t dv;           /* 512: kv_lora_rank, the value width */
    int32_t rope;         /* 64: k_rope width; dk = dv + rope */
    int32_t row_stride;   /* stored row width of the cache (>= dv + rope) */
    int32_t topk;         /* K unit slots per query */
    int32_t read_block;   /* RB tokens per unit */
    int32_t page_size;
    int32_t num_page_ids; /* PTW: length of the packed page_indices list */
    int32_t total_num_pages;
    double sm_scale;
} oracle_ragged_params;

/* Self-write: token t's row [kvc[t] (dv) | kpe[t] (rope) | zeros] goes to flat cache row
 * loc[t]; a slot outside [0, P * page_size) (the -1 padding included) is dropped and the
 * cache is left as it was there. */
int oracle_sparse_ragged_write(const oracle_ragged_params* p, const uint16_t* kvc, const uint16_t* kpe,
                               uint16_t* cache, const int32_t* loc) {
    if (!p || !kvc || !kpe || !cache || !loc) return ORACLE_ERR_ARG;
    const long slots = (long)p->total_num_pages * p->page_size;
    for (int t = 0; t < p->num_tokens; ++t) {
        const long slot = loc[t];
        if (slot < 0 || slot >= slots) continue;
        uint16_t* row = cache + (size_t)slot * p->row_stride;
        for (int d = 0; d < p->row_stride; ++d) row[d] = 0;
        for (int d = 0; d < p->dv; ++d) row[d] = kvc[(size_t)t * p->dv + d];
        for (int d = 0; d < p->rope; ++d) row[p->dv + d] = kpe[(size_t)t * p->rope + d];
    }
    return ORACLE_OK;
}

/* Request of token t: the number of cu_q_lens[1..S] entries <= t (searchsorted, right
 * side, over cu_q_lens[1:]), clipped to [0, S - 1]. */
static int ragged_request(const int32_t* cu_q_lens, int S, int t) {
    int n = 0;
    for (int i = 1; i <= S; ++i)
        if (cu_q_lens[i] <= t) ++n;
    return n < 0 ? 0 : (n > S - 1 ? S - 1 : n);
}

/* ql bf16 [T, H, dv], qpe bf16 [T, H, rope] (the query is their concatenation); cache bf16
 * [P * page_size, row_stride] (already written); topk [T, K] request-local unit ids (-1 =
 * none); positions [T]; seq_lens [S]; cu_q_lens [S + 1]; cu_kv_lens [S + 1] (page-aligned
 * key offsets); page_indices [PTW].  Token t of request r = request(t) attends to key kp =
 * u * RB + j of each selected unit u when kp <= positions[t] and kp < seq_lens[r]; the key's
 * page is page_indices[min(cu_kv_lens[r] / page_size + kp / page_size, PTW - 1)].
 * out float64 [T, H, dv] for the listed tokens (all when queries == NULL). */
int oracle_sparse_mla_ragged(const oracle_ragged_params* p, const uint16_t* ql, const uint16_t* qpe,
                             const uint16_t* cache, const int32_t* topk, const int32_t* positions,
                             const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                             const int32_t* page_indices, const int32_t* queries, int32_t n_queries, double* out,
                             int nthreads) {
    if (!p || !ql || !qpe || !cache || !topk || !positions || !seq_lens || !cu_q_lens || !cu_kv_lens ||
        !page_indices || !out || p->num_seqs < 1 || p->num_page_ids < 1)
        return ORACLE_ERR_ARG;
    const int T = p->num_tokens, H = p->num_heads, K = p->topk, RB = p->read_block, ps = p->page_size;
    const int dk = p->dv + p->rope;
    const int n = queries ? n_queries : T;
    int err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1) num_threads(default_threads(nthreads))
    for (int it = 0; it < n; ++it) {
        const int t = queries ? queries[it] : it;
        if (t < 0 || t >= T) {
#pragma omp atomic write
            err = ORACLE_ERR_ARG;
            continue;
        }
        const int r = ragged_request(cu_q_lens, p->num_seqs, t);
        const long bound = seq_lens[r];
        const long base = cu_kv_lens[r] / ps;
        const int qpos = positions[t];
        size_t* rows = (size_t*)malloc(sizeof(size_t) * (size_t)K * RB + 8);
        int nk = 0, bad = 0;
        for (int i = 0; i < K; ++i) {
            const int u = topk[(size_t)t * K + i];
            if (u < 0) continue;
            for (int j = 0; j < RB; ++j) {
                const long kp = (long)u * RB + j;
                if (!(kp <= qpos && kp < bound)) continue;
                long pidx = base + kp / ps;
                if (pidx > p->num_page_ids - 1) pidx = p->num_page_ids - 1;
                if (pidx < 0) {
                    bad = 1;
                    continue;
                }
                const int32_t page = page_indices[pidx];
                if (page < 0 || page >= p->total_num_pages) {
                    bad = 1;
                    continue;
                }
                rows[nk++] = (size_t)page * ps + (size_t)(kp % ps);
            }
        }
        if (bad) {
#pragma omp atomic write
            err = ORACLE_ERR_PAGE;
            free(rows);
            continue;
        }
        double* x = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
        for (int h = 0; h < H; ++h) {
            const uint16_t* qn = ql + ((size_t)t * H + h) * p->dv;
            const uint16_t* qr = qpe + ((size_t)t * H + h) * p->rope;
            for (int i = 0; i < nk; ++i) {
                const uint16_t* row = cache + rows[i] * p->row_stride;
                double dot = 0.0;
                for (int d = 0; d < dk; ++d)
                    dot += (double)bf16_bits_to_f32(d < p->dv ? qn[d] : qr[d - p->dv]) * bf16_bits_to_f32(row[d]);
                x[i] = p->sm_scale * dot;
            }
            double l;
            softmax_weights(x, nk, &l);
            double* o = out + ((size_t)t * H + h) * p->dv;
            for (int d = 0; d < p->dv; ++d) o[d] = 0.0;
            for (int i = 0; i < nk; ++i) {
                const uint16_t* row = cache + rows[i] * p->row_stride;
                for (int d = 0; d < p->dv; ++d) o[d] += x[i] * bf16_bits_to_f32(row[d]);
            }
            const double inv = l > 0.0 ? 1.0 / l : 0.0;
            for (int d = 0; d < p->dv; ++d) o[d] *= inv;
        }
        free(x);
        free(rows);
    }
    return err;
}
