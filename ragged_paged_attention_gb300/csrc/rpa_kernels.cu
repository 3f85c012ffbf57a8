// Standard ragged paged attention (tpu-inference "ragged_paged_attention/v2/kernel.py")
// and its cache write, for sm_103a.
//
// One rpa_forward call = plan kernel + attention kernel(s), all on the caller's stream:
//   * rpa_plan_kernel reads the device metadata (num_seqs, cu_q_lens, kv_lens),
//     validates it, and writes two work lists into the workspace: "decode" items
//     (sequences whose q_len * G rows fit one 16-row tile, split along the keys and, past
//     8 rows, into two 8-row halves) and
//     "prefill" items (128-row tiles of one KV head over the whole causal key range)
//     (prefill items are 128 rows of one KV head: kPrefillRows).
//   * the prefill items run on tcgen05/TMEM (rpa_prefill_tc.cu), the decode items on
//     the streaming split-KV kernel (rpa_decode.cu); both are persistent CTAs that
//     steal items from their list.
#include "common.cuh"
#include "kernels.h"
#include "profile.h"

namespace rpa {

// ---------------------------------------------------------------------------
// Plan
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) rpa_plan_kernel(RpaArgs a) {
    __shared__ int scan_scratch[40];
    __shared__ long long red[32];
    __shared__ int s_num;
    __shared__ int s_chunk;
    // per sequence of the current group of blockDim.x: item end offsets and decode shape
    __shared__ int e_dend[1024], e_pend[1024], e_klo[1024], e_kl[1024], e_ns[1024], e_nrh[1024];
    WsHeader* hdr = a.hdr;
    const int tid = threadIdx.x;
    if (tid == 0) {
        int n = a.num_seqs[0];
        if (n < 0 || n > a.max_num_seqs) {
            set_error(&hdr->error_bits, RPA_DEV_ERR_NUM_SEQS);
            n = 0;
        }
        s_num = n;
    }
    __syncthreads();
    const int num = s_num;
    const int G = a.num_q_heads / a.num_kv_heads;
    const int n_groups = cdiv(a.num_kv_heads, a.decode_heads);

    // pass 1: total decode work (keys x head groups)
    long long dec_keys = 0;
    for (int s = tid; s < num; s += blockDim.x) {
        int ql, kl, klo;
        if (seq_shape(a, s, ql, kl) && ql >= 1 && ql * G <= 16) {
            klo = decode_key_begin(a, ql, kl);
            dec_keys += (long long)(kl - klo) * n_groups * cdiv(ql * G, kDecodeRows);
        }
    }
    for (int o = 16; o > 0; o >>= 1) dec_keys += __shfl_xor_sync(0xffffffffu, dec_keys, o);
    if ((tid & 31) == 0) red[tid >> 5] = dec_keys;
    __syncthreads();
    if (tid == 0) {
        long long t = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
        long long c = (t + a.decode_target_ctas - 1) / a.decode_target_ctas;
        if (c < kMinChunk) c = kMinChunk;
        c = (c + kDecodeBK - 1) / kDecodeBK * kDecodeBK;
        s_chunk = (int)c;
        hdr->chunk_keys = (int)c;
    }
    __syncthreads();
    const int chunk = s_chunk;

    // pass 2: item counts, scan, emit
    int dec_base = 0, pre_base = 0;
    for (int s0 = 0; s0 < num; s0 += blockDim.x) {
        const int s = s0 + tid;
        int ql = 0, kl = 0, nd = 0, np = 0, klo = 0, nsplit = 0, nrh = 0;
        bool ok = s < num && seq_shape(a, s, ql, kl);
        if (ok && ql >= 1) {
            if (ql * G <= 16) {
                klo = decode_key_begin(a, ql, kl);
                nsplit = cdiv(kl - klo, chunk);
                nrh = cdiv(ql * G, kDecodeRows);
                nd = nsplit * n_groups * nrh;
            } else {
                np = cdiv(ql * G, kPrefillRows) * a.num_kv_heads;
            }
        }
        int tot_d, tot_p;
        const int od = block_exclusive_scan(nd, scan_scratch, &tot_d);
        const int op = block_exclusive_scan(np, scan_scratch, &tot_p);
        // every thread then emits items: a thread per item, not per sequence (a long prefill
        // sequence has hundreds); item idx belongs to the first sequence whose end offset
        // (exclusive prefix + count) exceeds it
        e_dend[tid] = od + nd;
        e_pend[tid] = op + np;
        e_klo[tid] = klo;
        e_kl[tid] = kl;
        e_ns[tid] = nsplit;
        e_nrh[tid] = nrh;
        __syncthreads();
        const int nseq = min((int)blockDim.x, num - s0);
        auto owner = [&](const int* ends, int idx) {
            int lo = 0, hi = nseq - 1;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (ends[mid] > idx) hi = mid; else lo = mid + 1;
            }
            return lo;
        };
        for (int idx = tid; idx < tot_d; idx += blockDim.x) {
            const int it = dec_base + idx;
            if (it >= a.max_dec_items) break;  // cannot happen: the host bound covers it
            const int k = owner(e_dend, idx);
            const int ns = e_ns[k], nh = e_nrh[k];
            const int beg = e_dend[k] - ns * n_groups * nh;
            const int rel = idx - beg, gh = rel / ns, i = rel - gh * ns;
            const int g = gh / nh, rh = gh - g * nh;
            WorkItem w;
            w.seq = s0 + k;
            w.head = g * a.decode_heads;
            w.key_begin = e_klo[k] + i * chunk;
            w.key_end = min(e_kl[k], e_klo[k] + (i + 1) * chunk);
            w.first_item = dec_base + beg + gh * ns;
            w.num_splits = ns;
            w.split = i;
            w.row_begin = rh * kDecodeRows;
            a.dec_items[it] = w;
            a.tickets[it] = 0;
        }
        for (int idx = tid; idx < tot_p; idx += blockDim.x) {
            const int it = pre_base + idx;
            if (it >= a.max_pre_items) break;
            const int k = owner(e_pend, idx);
            const int kprev = k > 0 ? e_pend[k - 1] : 0;  // this sequence's items start here
            const int tiles = (e_pend[k] - kprev) / a.num_kv_heads;
            const int rel = idx - kprev, h = rel / tiles, r = rel - h * tiles;
            WorkItem w;
            w.seq = s0 + k;
            w.head = h;
            w.row_begin = r * kPrefillRows;
            w.key_begin = 0;
            w.key_end = e_kl[k];
            w.first_item = it;
            w.num_splits = 1;
            w.split = 0;
            a.pre_items[it] = w;
        }
        __syncthreads();  // the next group of sequences reuses the e_* arrays
        dec_base += tot_d;
        pre_base += tot_p;
    }
    if (tid == 0) {
        hdr->num_items[0] = min(dec_base, a.max_dec_items);
        hdr->num_items[1] = min(pre_base, a.max_pre_items);
        hdr->next_item[0] = 0;
        hdr->next_item[1] = 0;
    }
}

// ---------------------------------------------------------------------------
// Cache write: new K/V rows -> their page slots (16-byte copies, bit exact)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) rpa_update_kernel(RpaUpdateArgs a) {
    extern __shared__ int s_cu[];  // cu_q_lens[0..num] when it fits (kCuCache entries)
    __shared__ int s_num;
    if (threadIdx.x == 0) {
        int n = a.num_seqs[0];
        if (n < 0 || n > a.max_num_seqs) {
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
    const int lane = threadIdx.x & 31, warps = blockDim.x >> 5;
    const int Hkv = a.num_kv_heads, C = 2 * Hkv;
    const int row_chunks = a.head_dim * a.esz / 16;  // 16-byte chunks per head row
    const int chunks = Hkv * 2 * row_chunks;
    // one warp per token
    for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < min(total, a.max_num_tokens); t += gridDim.x * warps) {
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
        uint8_t* slot = static_cast<uint8_t*>(a.kv_pages) +
                        ((size_t)page * a.page_size + pos % a.page_size) * C * a.head_dim * a.esz;
        // up to 8 chunks per lane in flight: all loads of a batch before its stores
        for (int i0 = lane; i0 < chunks; i0 += 32 * 8) {
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = i0 + 32 * j;
                if (i < chunks) {
                    const int head = i / (2 * row_chunks), part = (i / row_chunks) & 1, c = i % row_chunks;
                    v[j] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(part ? a.new_v : a.new_k) +
                                                                 (((size_t)t * Hkv + head) * a.head_dim * a.esz) + c * 16));
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = i0 + 32 * j;
                if (i < chunks) {
                    const int head = i / (2 * row_chunks), part = (i / row_chunks) & 1, c = i % row_chunks;
                    *reinterpret_cast<uint4*>(slot + ((size_t)(2 * head + part) * a.head_dim * a.esz) + c * 16) = v[j];
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Launch helpers
// ---------------------------------------------------------------------------
cudaError_t launch_rpa_forward(const RpaArgs& a, int num_sms, cudaStream_t stream) {
    cudaError_t e;
    {
        ProfScope ps("rpa_plan", stream);
        rpa_plan_kernel<<<1, 1024, 0, stream>>>(a);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    e = launch_rpa_prefill(a, num_sms, stream);
    if (e != cudaSuccess) return e;
    return launch_rpa_decode(a, num_sms, stream);
}

cudaError_t launch_rpa_update(const RpaUpdateArgs& a, int num_sms, cudaStream_t stream) {
    const int grid = min(cdiv(a.max_num_tokens, 8), num_sms * 8);
    if (grid <= 0) return cudaSuccess;
    const int smem = min(a.max_num_seqs + 1, kCuCache) * (int)sizeof(int);
    ProfScope ps("rpa_update", stream);
    rpa_update_kernel<<<grid, 256, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace rpa
