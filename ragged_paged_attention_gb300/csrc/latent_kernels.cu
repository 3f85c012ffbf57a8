// MLA latent ragged paged attention (tpu-inference "mla/v1/kernel.py") and DSA sparse
// MLA (sglang-jax "dsa/sparse_mla_prefill.py") for sm_103a.
//
// Both are MQA over one latent head: every q head of a token reads the same 576-wide
// key rows ([kv_c | k_pe]) and the value is the first 512 columns of the same row.  A
// CTA owns 64 q heads of one query, so each gathered key row feeds a 64 x 576 x 32
// score tile and a 64 x 32 x 512 value tile: the key stream is shared by all rows and
// the whole mask is per key (one query position per tile).
//   * MLA: keys are the causal (and windowed) prefix of the sequence, gathered page by
//     page; a plan kernel turns cu_q_lens/kv_lens into per-token work items and splits
//     long key ranges.
//   * Sparse: keys are the selected units (read_block tokens each) of indices[b, s, :];
//     slot i is token indices[i / RB] * RB + i % RB, valid when the unit id is >= 0 and
//     the token is causal and inside seq_len; items are arithmetic (no plan kernel).
// The attention itself runs on tcgen05 in latent_tc.cu; this file holds the MLA cache
// update and the plan kernel that turns the ragged metadata into per-token work items.
#include "common.cuh"
#include "kernels.h"
#include "profile.h"

namespace rpa {

// ---------------------------------------------------------------------------
// MLA cache update: one warp per token, 16-byte copies, rope pad written as zeros
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mla_update_body(const MlaUpdateArgs& a, int block, int nblocks) {
    extern __shared__ int s_cu[];  // cu_q_lens[0..num] when it fits (kCuCache entries)
    __shared__ int s_num;
    if (threadIdx.x == 0) {
        int n = a.distribution[2];
        const int i = a.distribution[0], j = a.distribution[1];
        if (!(0 <= i && i <= j && j <= n && n <= a.max_num_seqs)) {
            set_error(a.err, RPA_DEV_ERR_NUM_SEQS);
            n = 0;
        }
        s_num = n;
    }
    __syncthreads();
    const int num = s_num;
    if (num == 0) return;
    // one global round trip for the metadata the per-token search reads
    const bool cached = num + 1 <= kCuCache;
    if (cached)
        for (int i = threadIdx.x; i <= num; i += blockDim.x) s_cu[i] = a.cu_q_lens[i];
    __syncthreads();
    const int32_t* cu = cached ? s_cu : a.cu_q_lens;
    const int total = cu[num];
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    const int kv_chunks = a.lkv_pad / 8, pe_chunks = a.r_pad / 8;
    for (int t = block * warps + (threadIdx.x >> 5); t < min(total, a.max_num_tokens); t += nblocks * warps) {
        const int s = seq_of_token(cu, num, t);
        const int q_start = cu[s], q_len = cu[s + 1] - q_start, kv_len = a.kv_lens[s];
        if (t < q_start || t >= q_start + q_len) continue;
        if (q_len > kv_len) {
            if (lane == 0) set_error(a.err, RPA_DEV_ERR_Q_LEN);
            continue;
        }
        const int pos = kv_len - q_len + (t - q_start);
        if (pos / a.page_size >= a.pages_per_seq) {
            if (lane == 0) set_error(a.err, RPA_DEV_ERR_KV_LEN);
            continue;
        }
        const int page = a.page_indices[(size_t)s * a.pages_per_seq + pos / a.page_size];
        if ((unsigned)page >= (unsigned)a.total_num_pages) {
            if (lane == 0) set_error(a.err, RPA_DEV_ERR_PAGE);
            continue;
        }
        const size_t slot = (size_t)page * a.page_size + pos % a.page_size;
        // up to 4 chunks per lane in flight: all loads of a batch before its stores
        for (int c0 = lane; c0 < kv_chunks + pe_chunks; c0 += 32 * 4) {
            uint4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = c0 + 32 * j;
                v[j] = make_uint4(0, 0, 0, 0);
                if (c < kv_chunks) {
                    if (c * 8 < a.lkv_dim) v[j] = __ldg(reinterpret_cast<const uint4*>(a.new_kv_c + (size_t)t * a.lkv_dim + c * 8));
                } else if (c < kv_chunks + pe_chunks) {
                    const int cc = c - kv_chunks;
                    if (cc * 8 < a.r_dim) v[j] = __ldg(reinterpret_cast<const uint4*>(a.new_k_pe + (size_t)t * a.r_dim + cc * 8));
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = c0 + 32 * j;
                if (c < kv_chunks)
                    *reinterpret_cast<uint4*>(a.cache_kv_c + slot * a.lkv_pad + c * 8) = v[j];
                else if (c < kv_chunks + pe_chunks)
                    *reinterpret_cast<uint4*>(a.cache_k_pe + slot * a.r_pad + (c - kv_chunks) * 8) = v[j];
            }
        }
    }
}

__global__ void __launch_bounds__(256) mla_update_kernel(MlaUpdateArgs a) { mla_update_body(a, blockIdx.x, gridDim.x); }

// ---------------------------------------------------------------------------
// MLA plan: one item per (token, 64-head tile, key chunk)
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool mla_token(const LatentArgs& a, int num, int t, int& s, int& klo, int& khi) {
    int lo = 0, hi = num - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.cu_q_lens[mid] <= t) lo = mid; else hi = mid - 1;
    }
    s = lo;
    const int q_start = a.cu_q_lens[s], q_len = a.cu_q_lens[s + 1] - q_start, kv_len = a.kv_lens[s];
    if (t < q_start || t >= q_start + q_len) return false;
    if (q_len > kv_len) {
        set_error(&a.hdr->error_bits, RPA_DEV_ERR_Q_LEN);
        return false;
    }
    if (cdiv(kv_len, a.page_size) > a.pages_per_seq) {
        set_error(&a.hdr->error_bits, RPA_DEV_ERR_KV_LEN);
        return false;
    }
    const int qpos = kv_len - q_len + (t - q_start);
    // the causal (windowed) range, or every key of the sequence with a mild mask
    khi = a.mask_mild ? kv_len : qpos + 1;
    klo = a.sliding_window > 0 && !a.mask_mild ? max(0, qpos - a.sliding_window + 1) : 0;
    klo = klo / kLatBK * kLatBK;
    return true;
}

__device__ __forceinline__ void mla_plan_body(const LatentArgs& a) {
    __shared__ int scan_scratch[40];
    __shared__ long long red[32];
    __shared__ int s_num, s_total, s_chunk, s_bad;
    constexpr int kLenBuckets = 1024;  // item lengths in 64-key blocks (longer ones share the last)
    __shared__ int hist[kLenBuckets];
    WsHeader* hdr = a.hdr;
    const int tid = threadIdx.x;
    if (tid == 0) {
        int n = a.distribution[2];
        const int i = a.distribution[0], j = a.distribution[1];
        if (!(0 <= i && i <= j && j <= n && n <= a.max_num_seqs)) {
            set_error(&hdr->error_bits, RPA_DEV_ERR_NUM_SEQS);
            n = 0;
        }
        s_num = n;
        s_bad = 0;
    }
    __syncthreads();
    // cu_q_lens must be non-decreasing from a non-negative start and end within max_num_tokens
    for (int s = tid; s < s_num; s += blockDim.x) {
        const int c0 = a.cu_q_lens[s], c1 = a.cu_q_lens[s + 1];
        if (c0 < 0 || c1 < c0 || c1 > a.max_num_tokens) s_bad = 1;
    }
    __syncthreads();
    if (tid == 0) {
        if (s_bad) {
            set_error(&hdr->error_bits, RPA_DEV_ERR_TOKENS);
            s_num = 0;
        }
        s_total = s_num > 0 ? a.cu_q_lens[s_num] : 0;
    }
    __syncthreads();
    const int num = s_num, total = s_total;
    const int tiles = a.num_heads / kLatRows;
    long long work = 0;
    for (int t = tid; t < total; t += blockDim.x) {
        int s, klo, khi;
        if (mla_token(a, num, t, s, klo, khi)) work += (long long)(khi - klo) * tiles;
    }
    for (int o = 16; o > 0; o >>= 1) work += __shfl_xor_sync(0xffffffffu, work, o);
    if ((tid & 31) == 0) red[tid >> 5] = work;
    __syncthreads();
    if (tid == 0) {
        long long w = 0;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) w += red[i];
        const int tgt = max(1, min(kLatTargetCtas, a.target_items));
        long long c = (w + tgt - 1) / tgt;
        if (c < kLatMinChunk) c = kLatMinChunk;
        c = (c + kLatBK - 1) / kLatBK * kLatBK;
        s_chunk = (int)c;
        hdr->chunk_keys = (int)c;
    }
    __syncthreads();
    const int chunk = s_chunk;
    // Items are listed longest first (a counting sort on their 64-key blocks, kLenBuckets
    // buckets): the attention kernel takes them from a queue in list order, so the short ones
    // fill in at the end. A split group keeps its partials at its group slots (split 0's
    // running index in token order plus the split), whatever the items' places in the list.
    auto bucket = [&](int len) { return kLenBuckets - 1 - min(kLenBuckets - 1, (len + kLatBK - 1) / kLatBK); };
    for (int i = tid; i < kLenBuckets; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int t0 = 0; t0 < total; t0 += blockDim.x) {
        const int t = t0 + tid;
        int s = 0, klo = 0, khi = 0;
        if (t < total && mla_token(a, num, t, s, klo, khi)) {
            const int nsplit = cdiv(khi - klo, chunk);
            for (int i = 0; i < nsplit; ++i)
                atomicAdd(&hist[bucket(min(khi, klo + (i + 1) * chunk) - (klo + i * chunk))], tiles);
        }
    }
    __syncthreads();
    {
        // exclusive offsets of the buckets (one thread per bucket: the plan runs 1024 threads)
        int tot;
        const int v = tid < kLenBuckets ? hist[tid] : 0;
        const int o = block_exclusive_scan(v, scan_scratch, &tot);
        if (tid < kLenBuckets) hist[tid] = o;
        __syncthreads();
    }
    int base = 0;
    for (int t0 = 0; t0 < total; t0 += blockDim.x) {
        const int t = t0 + tid;
        int s = 0, klo = 0, khi = 0, nsplit = 0;
        if (t < total && mla_token(a, num, t, s, klo, khi)) nsplit = cdiv(khi - klo, chunk);
        int tot;
        const int off = block_exclusive_scan(nsplit * tiles, scan_scratch, &tot) + base;
        for (int h = 0; h < tiles && nsplit; ++h) {
            for (int i = 0; i < nsplit; ++i) {
                const int g = off + h * nsplit + i;  // group slot of this split
                if (g >= a.max_items) break;
                WorkItem w;
                w.seq = s;
                w.head = h * kLatRows;
                w.row_begin = t;
                w.key_begin = klo + i * chunk;
                w.key_end = min(khi, klo + (i + 1) * chunk);
                w.first_item = off + h * nsplit;
                w.num_splits = nsplit;
                w.split = i;
                const int it = atomicAdd(&hist[bucket(w.key_end - w.key_begin)], 1);  // place in the list
                if (it < a.max_items) a.items[it] = w;
                a.tickets[2 * g] = 0;  // one ticket per CTA rank of the cluster pair
                a.tickets[2 * g + 1] = 0;
            }
        }
        base += tot;
    }
    if (tid == 0) {
        hdr->num_items[2] = min(base, a.max_items);
        hdr->next_item[2] = 0;
    }
}

// The cache write and the plan in one launch (mla_rpa_forward): block 0 plans, the others write
// the batch's new latent rows; the attention launch behind starts once this whole grid has ended.
__global__ void __launch_bounds__(1024) mla_plan_update_kernel(LatentArgs a, MlaUpdateArgs u) {
    if (blockIdx.x == 0)
        mla_plan_body(a);
    else
        mla_update_body(u, blockIdx.x - 1, gridDim.x - 1);
}

cudaError_t launch_mla_update(const MlaUpdateArgs& a, int num_sms, cudaStream_t stream) {
    const int grid = min(cdiv(a.max_num_tokens, 8), num_sms * 8);
    if (grid <= 0) return cudaSuccess;
    const int smem = min(a.max_num_seqs + 1, kCuCache) * (int)sizeof(int);
    ProfScope ps("mla_update", stream);
    mla_update_kernel<<<grid, 256, smem, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_mla_forward_update(const LatentArgs& a, const MlaUpdateArgs& u, int num_sms, cudaStream_t stream) {
    // one warp per new token in 1024-thread blocks, behind the plan's block
    const int ublocks = max(1, min(cdiv(u.max_num_tokens, 32), num_sms * 2));
    const int smem = min(u.max_num_seqs + 1, kCuCache) * (int)sizeof(int);
    {
        ProfScope ps("mla_plan_update", stream);
        mla_plan_update_kernel<<<1 + ublocks, 1024, smem, stream>>>(a, u);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return launch_mla_attention(a, num_sms, stream);
}

// ---------------------------------------------------------------------------
// Packed-ragged sparse MLA (sglang-jax "dsa/sparse_mla_prefill.py",
// prefill_write_and_attend_ragged): one warp per token finds its request (the number of
// cu_q_lens[1..S] entries <= t, as searchsorted, clipped to the last request), records that
// request's causal bound (seq_lens) and page base (cu_kv_lens / page_size), and writes the
// token's latent row [c_kv | k_rope | zeros] into cache slot loc[t] (a slot outside the cache,
// the -1 padding included, is dropped).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) sparse_ragged_prep_kernel(SparseRaggedPrepArgs a) {
    const int lane = threadIdx.x & 31, warps = blockDim.x >> 5;
    const long long slots = (long long)a.total_num_pages * a.page_size;
    const int chunks = a.row_stride / 8;  // 16-byte chunks of a row
    for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < a.num_tokens; t += gridDim.x * warps) {
        if (lane == 0) {
            int lo = 1, hi = a.num_seqs + 1;  // first i in [1, S] with cu_q_lens[i] > t (S + 1: none)
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (a.cu_q_lens[mid] > t) hi = mid; else lo = mid + 1;
            }
            const int r = min(lo - 1, a.num_seqs - 1);
            a.q_bound[t] = a.seq_lens[r];
            const int kvo = a.cu_kv_lens[r];
            a.q_base[t] = kvo >= 0 ? kvo / a.page_size : -1;
        }
        if (!a.kvc) continue;
        const long long slot = a.loc[t];
        if (slot < 0 || slot >= slots) continue;
        uint4* row = reinterpret_cast<uint4*>(a.cache + slot * a.row_stride);
        for (int c = lane; c < chunks; c += 32) {
            const int e = c * 8;  // dv and rope are multiples of 8: no chunk straddles two parts
            uint4 v = make_uint4(0, 0, 0, 0);
            if (e < a.dv)
                v = __ldg(reinterpret_cast<const uint4*>(a.kvc + (size_t)t * a.dv + e));
            else if (e < a.dv + a.rope)
                v = __ldg(reinterpret_cast<const uint4*>(a.kpe + (size_t)t * a.rope + (e - a.dv)));
            row[c] = v;
        }
    }
}

cudaError_t launch_sparse_ragged(const SparseRaggedPrepArgs& pa, const LatentArgs& a, int num_sms,
                                 cudaStream_t stream) {
    {
        ProfScope ps("sparse_ragged_prep", stream);
        const int grid = max(1, min(cdiv(pa.num_tokens, 8), num_sms * 8));
        sparse_ragged_prep_kernel<<<grid, 256, 0, stream>>>(pa);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return launch_sparse_attention(a, num_sms, stream);
}

cudaError_t launch_sparse_forward(const LatentArgs& a, int num_sms, cudaStream_t stream) {
    return launch_sparse_attention(a, num_sms, stream);
}

}  // namespace rpa
