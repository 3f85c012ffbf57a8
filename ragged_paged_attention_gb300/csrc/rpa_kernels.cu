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
        const int od = block_exclusive_scan(nd, scan_scratch, &tot_d) + dec_base;
        const int op = block_exclusive_scan(np, scan_scratch, &tot_p) + pre_base;
        for (int gh = 0; gh < n_groups * nrh && nd; ++gh) {
            const int g = gh / nrh, rh = gh % nrh;
            for (int i = 0; i < nsplit; ++i) {
                const int it = od + gh * nsplit + i;
                if (it >= a.max_dec_items) break;  // cannot happen: the host bound covers it
                WorkItem w;
                w.seq = s;
                w.head = g * a.decode_heads;
                w.key_begin = klo + i * chunk;
                w.key_end = min(kl, klo + (i + 1) * chunk);
                w.first_item = od + gh * nsplit;
                w.num_splits = nsplit;
                w.split = i;
                w.row_begin = rh * kDecodeRows;
                a.dec_items[it] = w;
                a.tickets[it] = 0;
            }
        }
        const int tiles = np ? np / a.num_kv_heads : 0;
        for (int h = 0; h < a.num_kv_heads && np; ++h) {
            for (int r = 0; r < tiles; ++r) {
                const int it = op + h * tiles + r;
                if (it >= a.max_pre_items) break;
                WorkItem w;
                w.seq = s;
                w.head = h;
                w.row_begin = r * kPrefillRows;
                w.key_begin = 0;
                w.key_end = kl;
                w.first_item = it;
                w.num_splits = 1;
                w.split = 0;
                a.pre_items[it] = w;
            }
        }
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
    const int total = a.cu_q_lens[num];
    const int Hkv = a.num_kv_heads, C = 2 * Hkv;
    const int row_chunks = a.head_dim * a.esz / 16;  // 16-byte chunks per head row
    const int chunks = Hkv * 2 * row_chunks;
    for (int t = blockIdx.x; t < min(total, a.max_num_tokens); t += gridDim.x) {
        // sequence of token t: last s with cu_q_lens[s] <= t
        int lo = 0, hi = num - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.cu_q_lens[mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int s = lo;
        const int q_start = a.cu_q_lens[s], q_len = a.cu_q_lens[s + 1] - q_start, kv_len = a.kv_lens[s];
        if (t < q_start || t >= q_start + q_len) continue;
        if (q_len > kv_len) {
            if (threadIdx.x == 0) set_error(a.err, RPA_DEV_ERR_Q_LEN);
            continue;
        }
        const int pos = kv_len - q_len + (t - q_start);
        if (pos / a.page_size >= a.pages_per_seq) {
            if (threadIdx.x == 0) set_error(a.err, RPA_DEV_ERR_KV_LEN);
            continue;
        }
        const int page = a.page_indices[(size_t)s * a.pages_per_seq + pos / a.page_size];
        if ((unsigned)page >= (unsigned)a.total_num_pages) {
            if (threadIdx.x == 0) set_error(a.err, RPA_DEV_ERR_PAGE);
            continue;
        }
        uint8_t* slot = static_cast<uint8_t*>(a.kv_pages) +
                        ((size_t)page * a.page_size + pos % a.page_size) * C * a.head_dim * a.esz;
        for (int i = threadIdx.x; i < chunks; i += blockDim.x) {
            const int head = i / (2 * row_chunks);
            const int part = (i / row_chunks) & 1;
            const int c = i % row_chunks;
            const uint8_t* src = static_cast<const uint8_t*>(part ? a.new_v : a.new_k) +
                                 (((size_t)t * Hkv + head) * a.head_dim * a.esz) + c * 16;
            *reinterpret_cast<uint4*>(slot + ((size_t)(2 * head + part) * a.head_dim * a.esz) + c * 16) =
                __ldg(reinterpret_cast<const uint4*>(src));
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
    const int grid = min(a.max_num_tokens, num_sms * 8);
    if (grid <= 0) return cudaSuccess;
    ProfScope ps("rpa_update", stream);
    rpa_update_kernel<<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace rpa
