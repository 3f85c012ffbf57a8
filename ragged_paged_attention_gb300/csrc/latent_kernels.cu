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
// Eight warps split the work: QK^T as 4 x 4 m16n8 tiles over the 36 k-steps, the score
// tile goes through shared memory for the softmax, and each warp accumulates a 64 x 64
// slice of O in registers.  Split items merge through the log-sum-exp rule.
#include "common.cuh"
#include "kernels.h"
#include "profile.h"

namespace rpa {

// ---------------------------------------------------------------------------
// MLA cache update: one warp per token, 16-byte copies, rope pad written as zeros
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) mla_update_kernel(MlaUpdateArgs a) {
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
    const int total = a.cu_q_lens[num];
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    const int kv_chunks = a.lkv_pad / 8, pe_chunks = a.r_pad / 8;
    for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < min(total, a.max_num_tokens); t += gridDim.x * warps) {
        int lo = 0, hi = num - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.cu_q_lens[mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int s = lo;
        const int q_start = a.cu_q_lens[s], q_len = a.cu_q_lens[s + 1] - q_start, kv_len = a.kv_lens[s];
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
        for (int c = lane; c < kv_chunks + pe_chunks; c += 32) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (c < kv_chunks) {
                if (c * 8 < a.lkv_dim)
                    v = __ldg(reinterpret_cast<const uint4*>(a.new_kv_c + (size_t)t * a.lkv_dim + c * 8));
                *reinterpret_cast<uint4*>(a.cache_kv_c + slot * a.lkv_pad + c * 8) = v;
            } else {
                const int cc = c - kv_chunks;
                if (cc * 8 < a.r_dim)
                    v = __ldg(reinterpret_cast<const uint4*>(a.new_k_pe + (size_t)t * a.r_dim + cc * 8));
                *reinterpret_cast<uint4*>(a.cache_k_pe + slot * a.r_pad + cc * 8) = v;
            }
        }
    }
}

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
    khi = qpos + 1;
    klo = a.sliding_window > 0 ? max(0, qpos - a.sliding_window + 1) : 0;
    klo = klo / kLatBK * kLatBK;
    return true;
}

__global__ void __launch_bounds__(1024) mla_plan_kernel(LatentArgs a) {
    __shared__ int scan_scratch[40];
    __shared__ long long red[32];
    __shared__ int s_num, s_total, s_chunk, s_bad;
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
        long long c = (w + kLatTargetCtas - 1) / kLatTargetCtas;
        if (c < kLatMinChunk) c = kLatMinChunk;
        c = (c + kLatBK - 1) / kLatBK * kLatBK;
        s_chunk = (int)c;
        hdr->chunk_keys = (int)c;
    }
    __syncthreads();
    const int chunk = s_chunk;
    int base = 0;
    for (int t0 = 0; t0 < total; t0 += blockDim.x) {
        const int t = t0 + tid;
        int s = 0, klo = 0, khi = 0, nsplit = 0;
        if (t < total && mla_token(a, num, t, s, klo, khi)) nsplit = cdiv(khi - klo, chunk);
        int tot;
        const int off = block_exclusive_scan(nsplit * tiles, scan_scratch, &tot) + base;
        for (int h = 0; h < tiles && nsplit; ++h) {
            for (int i = 0; i < nsplit; ++i) {
                const int it = off + h * nsplit + i;
                if (it >= a.max_items) break;
                WorkItem w;
                w.seq = s;
                w.head = h * kLatRows;
                w.row_begin = t;
                w.key_begin = klo + i * chunk;
                w.key_end = min(khi, klo + (i + 1) * chunk);
                w.first_item = off + h * nsplit;
                w.num_splits = nsplit;
                w.split = i;
                a.items[it] = w;
                a.tickets[it] = 0;
            }
        }
        base += tot;
    }
    if (tid == 0) {
        hdr->num_items[2] = min(base, a.max_items);
        hdr->next_item[2] = 0;
    }
}

// ---------------------------------------------------------------------------
// Latent attention
// ---------------------------------------------------------------------------
constexpr int kLatRowBytes = kLatDk * 2;          // 1152: one Q or key row in shared memory
constexpr int kLatChunks = kLatDk / 8;            // 72 16-byte chunks per row
constexpr int kLatSStride = kLatBK + 4;           // fp32 score row stride (floats)
constexpr int kLatPStride = (kLatBK + 8) * 2;     // bf16 probability row stride (bytes): 80
constexpr int kLatQBytes = kLatRows * kLatRowBytes;
constexpr int kLatStageBytes = kLatBK * kLatRowBytes;
constexpr int kLatSmem = kLatQBytes + 2 * kLatStageBytes + kLatRows * kLatSStride * 4 + kLatRows * kLatPStride +
                         3 * kLatRows * 4 + 2 * kLatBK * 4;

template <bool SPARSE>
__global__ void __launch_bounds__(256, 1) latent_attn_kernel(LatentArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* qs = smem;
    uint8_t* kvs = qs + kLatQBytes;
    float* S = reinterpret_cast<float*>(kvs + 2 * kLatStageBytes);
    uint8_t* Ps = reinterpret_cast<uint8_t*>(S + kLatRows * kLatSStride);
    float* m_run = reinterpret_cast<float*>(Ps + kLatRows * kLatPStride);
    float* l_run = m_run + kLatRows;
    float* alpha_s = l_run + kLatRows;
    int* key_ok = reinterpret_cast<int*>(alpha_s + kLatRows);  // [2][kLatBK]
    __shared__ WorkItem s_item;
    __shared__ int s_item_idx, s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    WsHeader* hdr = a.hdr;
    const int H = a.num_heads;
    const int tiles = H / kLatRows;
    int sparse_items = 0, slots = 0, sparse_chunk = 0;
    if (SPARSE) {
        slots = a.topk * a.read_block;
        sparse_items = a.batch * a.num_queries * tiles * a.sparse_splits;
        sparse_chunk = cdiv(cdiv(slots, a.sparse_splits), kLatBK) * kLatBK;
    }

    while (true) {
        __syncthreads();
        if (tid == 0) {
            const int it = atomicAdd(&hdr->next_item[SPARSE ? 3 : 2], 1);
            s_item.seq = -1;
            s_item_idx = it;
            if (SPARSE) {
                if (it < sparse_items) {
                    const int per_q = tiles * a.sparse_splits;
                    const int bs = it / per_q, rem = it % per_q;
                    const int tile = rem / a.sparse_splits, sp = rem % a.sparse_splits;
                    WorkItem w;
                    w.seq = bs;
                    w.head = tile * kLatRows;
                    w.row_begin = 0;
                    w.key_begin = sp * sparse_chunk;
                    w.key_end = min(slots, (sp + 1) * sparse_chunk);
                    w.first_item = it - sp;
                    w.num_splits = a.sparse_splits;
                    w.split = sp;
                    s_item = w;
                }
            } else if (it < hdr->num_items[2]) {
                s_item = a.items[it];
            }
        }
        __syncthreads();
        const WorkItem w = s_item;
        if (w.seq < 0) break;
        const int self = s_item_idx;
        const int h0 = w.head;

        // per-item query context
        int qpos = 0, b = 0, seq = 0, t = 0, wlo = 0;
        if (SPARSE) {
            b = w.seq / a.num_queries;
            qpos = a.positions[w.seq];
        } else {
            seq = w.seq;
            t = w.row_begin;
            const int q_start = a.cu_q_lens[seq];
            qpos = a.kv_lens[seq] - (a.cu_q_lens[seq + 1] - q_start) + (t - q_start);
            wlo = a.sliding_window > 0 ? qpos - a.sliding_window + 1 : 0;
        }
        const int kb = w.key_begin, ke = w.key_end;
        const int n_blocks = ke > kb ? cdiv(ke - kb, kLatBK) : 0;

        // ---- Q tile ----
        for (int i = tid; i < kLatRows * kLatChunks; i += 256) {
            const int r = i / kLatChunks, c = i % kLatChunks;
            const __nv_bfloat16* src;
            if (SPARSE) {
                src = a.q + ((size_t)w.seq * H + h0 + r) * kLatDk + c * 8;
            } else {
                src = c < 64 ? a.ql_nope + ((size_t)t * H + h0 + r) * 512 + c * 8
                             : a.q_pe + ((size_t)t * H + h0 + r) * 64 + (c - 64) * 8;
            }
            cp_async16(smem_u32(qs + swz(r, c, kLatRowBytes)), src, true);
        }
        if (tid < kLatRows) {
            m_run[tid] = -INFINITY;
            l_run[tid] = 0.f;
        }

        auto load_block = [&](int blk, int stage) {
            uint8_t* dst = kvs + stage * kLatStageBytes;
            const int key0 = kb + blk * kLatBK;
            for (int i = tid; i < kLatBK * kLatChunks; i += 256) {
                const int kk = i / kLatChunks, c = i % kLatChunks;
                const int key = key0 + kk;
                bool v = key < ke;
                const __nv_bfloat16* src = SPARSE ? a.cache : a.cache_kv_c;
                if (v) {
                    if (SPARSE) {
                        const int u = a.indices[(size_t)w.seq * a.topk + key / a.read_block];
                        const long long kp = (long long)u * a.read_block + key % a.read_block;
                        v = u >= 0 && kp <= qpos && kp < a.seq_len;
                        if (v) {
                            const int lp = (int)(kp / a.page_size);
                            const int page = lp < a.max_pages ? a.page_table[(size_t)b * a.max_pages + lp] : -1;
                            if ((unsigned)page >= (unsigned)a.total_num_pages) {
                                set_error(&hdr->error_bits, RPA_DEV_ERR_PAGE);
                                v = false;
                            } else {
                                src = a.cache + ((size_t)page * a.page_size + kp % a.page_size) * a.row_stride + c * 8;
                            }
                        }
                    } else if (key < wlo) {
                        v = false;  // outside the sliding window (the causal bound is ke)
                    } else {
                        const int page = a.page_indices[(size_t)seq * a.pages_per_seq + key / a.page_size];
                        if ((unsigned)page >= (unsigned)a.total_num_pages) {
                            set_error(&hdr->error_bits, RPA_DEV_ERR_PAGE);
                            v = false;
                        } else {
                            const size_t slot = (size_t)page * a.page_size + key % a.page_size;
                            src = c < 64 ? a.cache_kv_c + slot * a.lkv_pad + c * 8
                                         : a.cache_k_pe + slot * a.r_pad + (c - 64) * 8;
                        }
                    }
                }
                if (c == 0) key_ok[stage * kLatBK + kk] = v;
                cp_async16(smem_u32(dst + swz(kk, c, kLatRowBytes)), src, v);
            }
        };

        if (n_blocks > 0) load_block(0, 0);
        cp_async_commit();

        // this warp's slice of O: 4 m-tiles x 8 n-tiles (columns 64*warp .. +64)
        float o[4][8][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) o[i][j][0] = o[i][j][1] = o[i][j][2] = o[i][j][3] = 0.f;

        const int mt_s = warp >> 1, nt_s = (warp & 1) * 2;  // score tile of this warp
        const uint32_t q_base = smem_u32(qs);
        const uint32_t p_base = smem_u32(Ps);
        const float scale = a.sm_scale, cap = a.soft_cap;

        for (int blk = 0; blk < n_blocks; ++blk) {
            if (blk + 1 < n_blocks) load_block(blk + 1, (blk + 1) & 1);
            cp_async_commit();
            cp_async_wait<1>();
            __syncthreads();
            const int stage = blk & 1;
            const uint32_t kv_base = smem_u32(kvs + stage * kLatStageBytes);

            // ---- S = Q K^T (64 x 32) ----
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 4
            for (int ks = 0; ks < kLatDk / 16; ++ks) {
                uint32_t af[4], b0, b1, b2, b3;
                ldsm_x4(q_base + swz(mt_s * 16 + (lane & 15), ks * 2 + (lane >> 4), kLatRowBytes), af[0], af[1], af[2],
                        af[3]);
                const int key = nt_s * 8 + ((lane >> 4) << 3) + (lane & 7);
                ldsm_x4(kv_base + swz(key, ks * 2 + ((lane >> 3) & 1), kLatRowBytes), b0, b1, b2, b3);
                mma_bf16(acc[0], af, b0, b1);
                mma_bf16(acc[1], af, b2, b3);
            }
            {
                const int r0 = mt_s * 16 + (lane >> 2);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int col = (nt_s + j) * 8 + 2 * (lane & 3);
                    *reinterpret_cast<float2*>(S + r0 * kLatSStride + col) = make_float2(acc[j][0], acc[j][1]);
                    *reinterpret_cast<float2*>(S + (r0 + 8) * kLatSStride + col) = make_float2(acc[j][2], acc[j][3]);
                }
            }
            __syncthreads();
            // ---- online softmax: 4 threads per row, 8 keys each ----
            {
                const int row = tid >> 2, qd = tid & 3;
                const float m_old = m_run[row];
                float x[8];
                float mx = -INFINITY;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int k = qd * 8 + e;
                    float v = S[row * kLatSStride + k] * scale;
                    if (cap != 0.f) v = cap * tanhf(v / cap);
                    v *= kLog2e;
                    v = key_ok[stage * kLatBK + k] ? v : -INFINITY;
                    x[e] = v;
                    mx = fmaxf(mx, v);
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_old, mx);
                const float mu = m_new == -INFINITY ? 0.f : m_new;
                float sum = 0.f;
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float p0 = fast_exp2(x[e] - mu), p1 = fast_exp2(x[e + 1] - mu);
                    sum += p0 + p1;
                    pk[e / 2] = pack_bf16(p0, p1);
                }
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                *reinterpret_cast<uint4*>(Ps + row * kLatPStride + qd * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                if (qd == 0) {
                    const float al = fast_exp2(m_old - mu);
                    alpha_s[row] = al;
                    m_run[row] = m_new;
                    l_run[row] = l_run[row] * al + sum;
                }
            }
            __syncthreads();
            // ---- O = alpha * O + P V ----
            {
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    const float a0 = alpha_s[mt * 16 + (lane >> 2)], a1 = alpha_s[mt * 16 + (lane >> 2) + 8];
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt) {
                        o[mt][nt][0] *= a0;
                        o[mt][nt][1] *= a0;
                        o[mt][nt][2] *= a1;
                        o[mt][nt][3] *= a1;
                    }
                }
#pragma unroll
                for (int kk = 0; kk < kLatBK / 16; ++kk) {
                    uint32_t bf[8][2];
#pragma unroll
                    for (int np = 0; np < 4; ++np) {
                        const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                        const int chunk = warp * 8 + np * 2 + (lane >> 4);
                        ldsm_x4_t(kv_base + swz(key, chunk, kLatRowBytes), bf[2 * np][0], bf[2 * np][1],
                                  bf[2 * np + 1][0], bf[2 * np + 1][1]);
                    }
#pragma unroll
                    for (int mt = 0; mt < 4; ++mt) {
                        uint32_t af[4];
                        ldsm_x4(p_base + (mt * 16 + (lane & 15)) * kLatPStride + (kk * 2 + (lane >> 4)) * 16, af[0],
                                af[1], af[2], af[3]);
#pragma unroll
                        for (int nt = 0; nt < 8; ++nt) mma_bf16(o[mt][nt], af, bf[nt][0], bf[nt][1]);
                    }
                }
            }
            __syncthreads();
        }
        cp_async_wait<0>();
        __syncthreads();

        // ---- finalise ----
        const int g8 = lane >> 2, q4 = lane & 3;
        if (w.num_splits == 1) {
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int row = mt * 16 + g8 + e * 8;
                    const float l = l_run[row];
                    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt) {
                        const int col = warp * 64 + nt * 8 + 2 * q4;
                        const float v0 = o[mt][nt][2 * e] * inv, v1 = o[mt][nt][2 * e + 1] * inv;
                        if (SPARSE) {
                            *reinterpret_cast<float2*>(a.out_f32 + ((size_t)w.seq * H + h0 + row) * kLatDv + col) =
                                make_float2(v0, v1);
                        } else {
                            *reinterpret_cast<uint32_t*>(a.out_bf16 + ((size_t)t * H + h0 + row) * kLatDv + col) =
                                pack_bf16(v0, v1);
                        }
                    }
                }
            }
            continue;
        }
        // split: partial (m, l, unnormalised O), then the last CTA of the group merges
        float* po = a.partial_o + (size_t)self * kLatRows * kLatDv;
        float* pml = a.partial_ml + (size_t)self * kLatRows * 2;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int row = mt * 16 + g8 + e * 8;
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
                    *reinterpret_cast<float2*>(po + (size_t)row * kLatDv + warp * 64 + nt * 8 + 2 * q4) =
                        make_float2(o[mt][nt][2 * e], o[mt][nt][2 * e + 1]);
            }
        if (tid < kLatRows) {
            pml[tid * 2] = m_run[tid];
            pml[tid * 2 + 1] = l_run[tid];
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last = atomicAdd(&a.tickets[w.first_item], 1) == w.num_splits - 1;
        __syncthreads();
        if (!s_last) continue;
        __threadfence();
        for (int i = tid; i < kLatRows * (kLatDv / 4); i += 256) {
            const int row = i / (kLatDv / 4), c4 = (i % (kLatDv / 4)) * 4;
            float M = -INFINITY;
            for (int sp = 0; sp < w.num_splits; ++sp)
                M = fmaxf(M, __ldcg(a.partial_ml + (size_t)(w.first_item + sp) * kLatRows * 2 + row * 2));
            const float Mu = M == -INFINITY ? 0.f : M;
            float L = 0.f;
            float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int sp = 0; sp < w.num_splits; ++sp) {
                const size_t it = (size_t)(w.first_item + sp);
                const float m = __ldcg(a.partial_ml + it * kLatRows * 2 + row * 2);
                const float l = __ldcg(a.partial_ml + it * kLatRows * 2 + row * 2 + 1);
                const float f = fast_exp2(m - Mu);
                L += f * l;
                const float4 v = __ldcg(reinterpret_cast<const float4*>(a.partial_o + it * kLatRows * kLatDv +
                                                                        (size_t)row * kLatDv + c4));
                acc4.x += f * v.x;
                acc4.y += f * v.y;
                acc4.z += f * v.z;
                acc4.w += f * v.w;
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            if (SPARSE) {
                *reinterpret_cast<float4*>(a.out_f32 + ((size_t)w.seq * H + h0 + row) * kLatDv + c4) =
                    make_float4(acc4.x * inv, acc4.y * inv, acc4.z * inv, acc4.w * inv);
            } else {
                __nv_bfloat16* dst = a.out_bf16 + ((size_t)t * H + h0 + row) * kLatDv + c4;
                *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16(acc4.x * inv, acc4.y * inv),
                                                            pack_bf16(acc4.z * inv, acc4.w * inv));
            }
        }
        if (tid == 0) a.tickets[w.first_item] = 0;
    }
}

// sets the sparse work counter (no plan kernel on that path)
__global__ void sparse_reset_kernel(WsHeader* hdr) {
    hdr->next_item[3] = 0;
}

template <bool SPARSE>
static cudaError_t launch_latent(const LatentArgs& a, int grid, cudaStream_t stream) {
    auto kern = latent_attn_kernel<SPARSE>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kLatSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    ProfScope ps(SPARSE ? "sparse_attn" : "mla_attn", stream);
    kern<<<grid, 256, kLatSmem, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_mla_update(const MlaUpdateArgs& a, int num_sms, cudaStream_t stream) {
    const int grid = min(cdiv(a.max_num_tokens, 8), num_sms * 8);
    if (grid <= 0) return cudaSuccess;
    ProfScope ps("mla_update", stream);
    mla_update_kernel<<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_mla_forward(const LatentArgs& a, int num_sms, cudaStream_t stream) {
    cudaError_t e;
    {
        ProfScope ps("mla_plan", stream);
        mla_plan_kernel<<<1, 1024, 0, stream>>>(a);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    return launch_latent<false>(a, num_sms, stream);
}

cudaError_t launch_sparse_forward(const LatentArgs& a, int num_sms, cudaStream_t stream) {
    cudaError_t e;
    {
        ProfScope ps("sparse_reset", stream);
        sparse_reset_kernel<<<1, 1, 0, stream>>>(a.hdr);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    return launch_latent<true>(a, num_sms, stream);
}

}  // namespace rpa
