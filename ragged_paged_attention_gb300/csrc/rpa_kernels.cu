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
// Decode work is cut into shares of one line: every decode group (sequence x KV-head group x
// 8-row half) is a stream of its keys rounded up to 16, and the streams lie end to end. The
// first three quarters of the line are R equal shares, one per decode CTA resident at once;
// the rest is cut into small shares that CTAs take from a pool once their own is done. The
// pieces of a group that fall to different shares are its splits (merged by whichever
// finishes last). Equal shares remove the tail a queue of long items leaves (a few CTAs
// finishing while the rest of the GPU idles); the pool evens out CTAs that stream faster
// than others.
__device__ __forceinline__ void plan_body(const RpaArgs& a) {
    __shared__ long long scan_ll[40];
    __shared__ long long red[32], red_g[32];
    __shared__ float red_f[32];
    __shared__ int s_num;
    __shared__ long long s_q1, s_q2, s_ls;  // static share size, pooled share size, static part
    __shared__ int s_r;                     // static shares
    __shared__ float s_pf, s_db, best_t[32];
    __shared__ int best_n[32];
    // per sequence of the current group of blockDim.x: item end offsets, decode shape and the
    // line position of its first decode group
    __shared__ int e_dend[1024], e_pend[1024], e_klo[1024], e_kl[1024], e_nrh[1024];
    __shared__ long long e_pos[1024];
    WsHeader* hdr = a.hdr;
    const int tid = threadIdx.x;
    // the prefill grid behind may become resident now; it waits for this grid's end
    pdl_launch_dependents();
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
    auto round_bk = [](int keys) { return (long long)cdiv(keys, kDecodeBK) * kDecodeBK; };

    // pass 1: decode work (line length: keys and per-group cost), decode groups and the prefill
    // (query, key) pairs
    long long work = 0, ngrp = 0;
    float pre_pairs = 0.f;
    // this thread's first sequence's shape, kept for pass 2 (its first group of sequences)
    bool c_ok = false;
    int c_ql = 0, c_kl = 0;
    for (int s = tid; s < num; s += blockDim.x) {
        int ql, kl;
        const bool sok = seq_shape(a, s, ql, kl);
        if (s == tid) {
            c_ok = sok;
            c_ql = ql;
            c_kl = kl;
        }
        if (sok && ql >= 1 && !kind_allows(a, ql * G <= 16)) {
            set_error(&a.hdr->error_bits, RPA_DEV_ERR_BATCH_KIND);  // skipped: its launch is not made
        } else if (sok && ql >= 1) {
            if (ql * G <= 16) {
                const int klo = decode_key_begin(a, ql, kl);
                const long long g = (long long)n_groups * cdiv(ql * G, kDecodeRows);
                work += (round_bk(kl - klo) + a.item_cost_keys) * g;
                ngrp += g;
            } else {
                // causal: query i of the chunk sees kl - ql + i + 1 keys (at most the window)
                float seen = (float)kl - 0.5f * (float)(ql - 1);
                if (a.sliding_window > 0) seen = fminf(seen, (float)a.sliding_window);
                pre_pairs += (float)ql * seen;
            }
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        work += __shfl_xor_sync(0xffffffffu, work, o);
        ngrp += __shfl_xor_sync(0xffffffffu, ngrp, o);
        pre_pairs += __shfl_xor_sync(0xffffffffu, pre_pairs, o);
    }
    if ((tid & 31) == 0) {
        red[tid >> 5] = work;
        red_g[tid >> 5] = ngrp;
        red_f[tid >> 5] = pre_pairs;
    }
    __syncthreads();
    // the per-warp partials summed by warp 0 with shuffles (a serial loop over them is a
    // chain of dependent shared-memory loads)
    if (tid < 32) {
        const int nw = (int)(blockDim.x >> 5);
        long long W = tid < nw ? red[tid] : 0, NG = tid < nw ? red_g[tid] : 0;
        float pp = tid < nw ? red_f[tid] : 0.f;
        for (int o = 16; o > 0; o >>= 1) {
            W += __shfl_xor_sync(0xffffffffu, W, o);
            NG += __shfl_xor_sync(0xffffffffu, NG, o);
            pp += __shfl_xor_sync(0xffffffffu, pp, o);
        }
        __syncwarp();
        if (tid == 0) red[0] = W;
        if (tid == 0) {
            s_pf = pp * 4.f * (float)a.num_q_heads * (float)a.head_dim;
            s_db = (float)(W - NG * a.item_cost_keys) * (float)a.decode_heads * 2.f * (float)a.head_dim *
                   (a.kv_byte ? 1.f : 2.f);
        }
    }
    __syncthreads();
    // SMs for the prefill kernel beside decode: the n minimising max(prefill time on n SMs,
    // decode time on the rest), one candidate n = tid + 1 per thread
    const int S = a.num_sms;
    {
        const float pre_flops = s_pf, dec_bytes = s_db;
        float tt = INFINITY;
        int nn = S;
        if (a.overlap && pre_flops > 0.f && dec_bytes > 0.f && tid + 1 < S) {
            nn = tid + 1;
            const float tp = pre_flops / (a.pre_flops_per_ns_sm * (float)nn);
            const float td = dec_bytes / fminf(kDecHbmBytesPerNs, a.dec_bytes_per_ns_sm * (float)(S - nn));
            tt = fmaxf(tp, td);
        }
        for (int o = 16; o > 0; o >>= 1) {
            const float t2 = __shfl_xor_sync(0xffffffffu, tt, o);
            const int n2 = __shfl_xor_sync(0xffffffffu, nn, o);
            if (t2 < tt || (t2 == tt && n2 < nn)) {
                tt = t2;
                nn = n2;
            }
        }
        if ((tid & 31) == 0) {
            best_t[tid >> 5] = tt;
            best_n[tid >> 5] = nn;
        }
    }
    __syncthreads();
    float bt = INFINITY;
    int bn = S;
    if (tid < 32) {  // the best of the warps' candidates, by warp 0
        if (tid < (int)(blockDim.x >> 5)) {
            bt = best_t[tid];
            bn = best_n[tid];
        }
        for (int o = 16; o > 0; o >>= 1) {
            const float t2 = __shfl_xor_sync(0xffffffffu, bt, o);
            const int n2 = __shfl_xor_sync(0xffffffffu, bn, o);
            if (t2 < bt || (t2 == bt && n2 < bn)) {
                bt = t2;
                bn = n2;
            }
        }
    }
    if (tid == 0) {
        const long long W = red[0];
        const float pre_flops = s_pf, dec_bytes = s_db;
        // all SMs to prefill first unless the split beats the serial order by 10%
        int n_pre = S;
        if (pre_flops <= 0.f) {
            n_pre = 0;
        } else if (a.overlap && dec_bytes > 0.f && S > 1) {
            const float serial = pre_flops / (a.pre_flops_per_ns_sm * (float)S) +
                                 dec_bytes / fminf(kDecHbmBytesPerNs, a.dec_bytes_per_ns_sm * (float)S);
            if (bt < 0.9f * serial) n_pre = bn;
        }
        hdr->prefill_ctas = n_pre;
        // decode CTAs resident at once: beside the prefill share, or every slot
        int ctas = (n_pre > 0 && n_pre < S ? S - n_pre : S) * a.decode_per_sm;
        ctas = max(1, min(ctas, kMaxDecodeCtas / 2));
        // static shares: all but the pool's part of the line, none under kMinChunk keys
        const long long w_static = W * (100 - kPoolPercent) / 100;
        long long q1 = div_nn(w_static, ctas) / kDecodeBK * kDecodeBK;
        int r = ctas;
        if (q1 < kMinChunk) {
            q1 = kMinChunk;
            r = (int)min((long long)ctas, div_nn(w_static, kMinChunk));
        }
        const long long ls = (long long)r * q1;
        // pooled shares: about kPoolPerCta per CTA, at least kMinPoolChunk keys, within the bound
        const long long rest = W - ls;
        long long q2 = div_nn(rest, (long long)kPoolPerCta * ctas);
        q2 = max(q2, div_nn(rest + (kMaxDecodeCtas - r) - 1, kMaxDecodeCtas - r));
        q2 = max((long long)kMinPoolChunk, (q2 + kDecodeBK - 1) / kDecodeBK * kDecodeBK);
        // (every share longer than a group's cost holds at least one key)
        q2 = max(q2, (long long)(a.item_cost_keys + kDecodeBK));
        s_q1 = q1;
        s_q2 = q2;
        s_ls = ls;
        s_r = r;
        hdr->chunk_keys = (int)min(q1, (long long)0x7fffffff);
        hdr->dec_ctas = r;
        hdr->dec_shares = r + (int)div_nn(rest + q2 - 1, q2);
    }
    __syncthreads();
    const long long q1 = s_q1, q2 = s_q2, ls = s_ls;
    const int n_static = s_r;
    // share holding line position p, and where share c starts
    auto share_of = [&](long long p) { return p < ls ? div_nn(p, q1) : n_static + div_nn(p - ls, q2); };
    auto share_start = [&](long long c) { return c < n_static ? c * q1 : ls + (c - n_static) * q2; };
    // pass 2: item counts, scan, emit
    int dec_base = 0, pre_base = 0;
    long long pos_base = 0;  // line position of the current group of sequences
    for (int s0 = 0; s0 < num; s0 += blockDim.x) {
        const int s = s0 + tid;
        int ql = 0, kl = 0, nd = 0, np = 0, klo = 0, nrh = 0;
        long long wk = 0;  // this sequence's decode work (all its groups)
        bool ok = false;
        if (s0 == 0) {
            ok = s < num && c_ok;
            ql = c_ql;
            kl = c_kl;
        } else {
            ok = s < num && seq_shape(a, s, ql, kl);
        }
        if (ok && ql >= 1 && kind_allows(a, ql * G <= 16)) {
            if (ql * G <= 16) {
                klo = decode_key_begin(a, ql, kl);
                nrh = cdiv(ql * G, kDecodeRows);
                wk = (round_bk(kl - klo) + a.item_cost_keys) * n_groups * nrh;
            } else {
                np = cdiv(ql * G, kPrefillRows) * a.num_kv_heads;
            }
        }
        long long tot_w;
        const long long pos = pos_base + block_exclusive_scan(wk, scan_ll, &tot_w);
        // splits of each group: the number of shares its keys' stretch of the line meets (a group
        // spans its cost, then its keys)
        if (wk > 0) {
            const long long len = round_bk(kl - klo);
            for (int j = 0; j < n_groups * nrh; ++j) {
                const long long kr0 = pos + j * (len + a.item_cost_keys) + a.item_cost_keys;
                nd += (int)(share_of(kr0 + len - 1) - share_of(kr0) + 1);
            }
        }
        // both item counts in one scan: decode in the high word, prefill in the low (each total
        // is far below 2^31, so the low word never carries)
        long long tot_dp;
        const long long odp = block_exclusive_scan(((long long)nd << 32) | (long long)np, scan_ll, &tot_dp);
        const int od = (int)(odp >> 32), op = (int)(odp & 0xffffffffll);
        const int tot_d = (int)(tot_dp >> 32), tot_p = (int)(tot_dp & 0xffffffffll);
        // every thread then emits items: a thread per item, not per sequence (a long prefill
        // sequence has hundreds); item idx belongs to the first sequence whose end offset
        // (exclusive prefix + count) exceeds it
        e_dend[tid] = od + nd;
        e_pend[tid] = op + np;
        e_klo[tid] = klo;
        e_kl[tid] = kl;
        e_nrh[tid] = nrh;
        e_pos[tid] = pos;
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
            const int nh = e_nrh[k], kl_k = e_kl[k], klo_k = e_klo[k];
            const long long len = round_bk(kl_k - klo_k);
            const int seq_first = k > 0 ? e_dend[k - 1] : 0;
            // the group j of this sequence holding the item, and the item's split in it
            int rel = idx - seq_first, first = dec_base + seq_first, j = 0;
            long long p0 = e_pos[k], kr0 = p0 + a.item_cost_keys;  // group start, its keys' start
            int ns = (int)(share_of(kr0 + len - 1) - share_of(kr0) + 1);
            while (rel >= ns) {
                rel -= ns;
                first += ns;
                ++j;
                p0 += len + a.item_cost_keys;
                kr0 = p0 + a.item_cost_keys;
                ns = (int)(share_of(kr0 + len - 1) - share_of(kr0) + 1);
            }
            const long long c = share_of(kr0) + rel;  // the share holding this piece
            const long long c_lo = share_start(c);
            const long long b0 = max(kr0, c_lo) - kr0, b1 = min(kr0 + len, share_start(c + 1)) - kr0;
            WorkItem w;
            w.seq = s0 + k;
            w.head = (j / nh) * a.decode_heads;
            w.row_begin = (j % nh) * kDecodeRows;
            w.key_begin = klo_k + (int)b0;
            w.key_end = min(kl_k, klo_k + (int)b1);
            w.first_item = first;
            w.num_splits = ns;
            w.split = rel;
            a.dec_items[it] = w;
            a.tickets[it] = 0;
            // the piece that opens share c: a later piece of a group, or its first when the share
            // began within this group's stretch
            if (rel > 0 || c_lo >= p0) a.cta_first[c] = it;
        }
        for (int idx = tid; idx < tot_p; idx += blockDim.x) {
            const int it = pre_base + idx;
            if (it >= a.max_pre_items) break;
            const int k = owner(e_pend, idx);
            const int kprev = k > 0 ? e_pend[k - 1] : 0;  // this sequence's items start here
            const int tiles = (e_pend[k] - kprev) / a.num_kv_heads;
            // a sequence's tiles longest first (a later tile sees more keys), the KV heads of one
            // tile together: persistent CTAs take the long items first and the short ones fill
            // in at the end
            const int rel = idx - kprev, h = rel % a.num_kv_heads, r = tiles - 1 - rel / a.num_kv_heads;
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
        pos_base += tot_w;
    }
    if (tid == 0) {
        hdr->num_items[0] = min(dec_base, a.max_dec_items);
        hdr->num_items[1] = min(pre_base, a.max_pre_items);
        a.cta_first[hdr->dec_shares] = hdr->num_items[0];
        hdr->next_item[0] = 0;
        hdr->next_item[1] = 0;  // prefill queue
        hdr->next_item[2] = 0;  // pooled decode shares taken
        // started beside the cache write (programmatic launch): end after it, so that the
        // attention grids behind see the new rows (no-op on an ordinary launch)
        pdl_wait();
    }
}

__global__ void __launch_bounds__(1024) rpa_plan_kernel(RpaArgs a) { plan_body(a); }

// ---------------------------------------------------------------------------
// Cache write: new K/V rows -> their page slots (16-byte copies, bit exact)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void update_body(const RpaUpdateArgs& a, int block, int nblocks) {
    // cu_q_lens[0..max_num_seqs] then kv_lens[0..max_num_seqs), when they fit (update_cache_ints)
    extern __shared__ int s_cu[];
    __shared__ int s_num;
    // an rpa_forward plan kernel behind may start now: it reads only metadata this kernel does
    // not write, and it ends after this grid has
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, warps = blockDim.x >> 5;
    const int Hkv = a.num_kv_heads, C = 2 * Hkv;
    const int row_chunks = a.row_bytes / 16;  // 16-byte chunks per head row
    const int chunks = Hkv * 2 * row_chunks;
    // one warp per token; each lane moves up to kBatch 16-byte chunks of the token's rows at a
    // time, loaded before the sequence and page lookups (they depend on the token index only)
    constexpr int kBatch = 8;
    auto load_batch = [&](int t, int i0, uint4 (&v)[kBatch]) {
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int i = i0 + 32 * j;
            if (i < chunks) {
                const int head = i / (2 * row_chunks), part = (i / row_chunks) & 1, c = i % row_chunks;
                v[j] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(part ? a.new_v : a.new_k) +
                                                             (((size_t)t * Hkv + head) * a.row_bytes) + c * 16));
            }
        }
    };
    // the metadata in one round trip, issued first: the sequence count and, for every sequence
    // slot the arrays have (cu_q_lens holds max_num_seqs + 1 entries, kv_lens max_num_seqs),
    // the query offsets and KV lengths, read before the count is known
    const bool cached = update_cache_ints(a.max_num_seqs) > 0;
    const int ms = a.max_num_seqs;
    if (threadIdx.x == 0) {
        int n = a.num_seqs[0];
        if (n < 0 || n > ms) {
            set_error(a.err, RPA_DEV_ERR_NUM_SEQS);
            n = 0;
        }
        s_num = n;
    }
    if (cached) {
        for (int i = threadIdx.x; i <= ms; i += blockDim.x) s_cu[i] = a.cu_q_lens[i];
        for (int i = threadIdx.x; i < ms; i += blockDim.x) s_cu[ms + 1 + i] = a.kv_lens[i];
    }
    // tokens interleaved over the blocks (warp w of block b starts at token w * nblocks + b),
    // so a small batch still spreads over every block; the first token's rows are in flight
    // while the metadata arrives
    const int t_first = (threadIdx.x >> 5) * nblocks + block;
    uint4 v[kBatch];
    if (t_first < a.max_num_tokens) load_batch(t_first, lane, v);
    __syncthreads();
    const int num = s_num;
    if (num == 0) return;
    const int32_t* cu = cached ? s_cu : a.cu_q_lens;
    const int32_t* kvl = cached ? s_cu + ms + 1 : a.kv_lens;
    const int total = cu[num];
    for (int t = t_first; t < min(total, a.max_num_tokens); t += nblocks * warps) {
        if (t != t_first) load_batch(t, lane, v);
        const int s = seq_of_token(cu, num, t);
        const int q_start = cu[s], q_len = cu[s + 1] - q_start, kv_len = kvl[s];
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
                        ((size_t)page * a.page_size + pos % a.page_size) * C * a.row_bytes;
        for (int i0 = lane; i0 < chunks; i0 += 32 * kBatch) {
            if (i0 != lane) load_batch(t, i0, v);
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int i = i0 + 32 * j;
                if (i < chunks) {
                    const int head = i / (2 * row_chunks), part = (i / row_chunks) & 1, c = i % row_chunks;
                    *reinterpret_cast<uint4*>(slot + ((size_t)(2 * head + part) * a.row_bytes) + c * 16) = v[j];
                }
            }
        }
    }
}

__global__ void __launch_bounds__(256) rpa_update_kernel(RpaUpdateArgs a) { update_body(a, blockIdx.x, gridDim.x); }

// The cache write and the plan in one launch (rpa_forward_update): block 0 plans, the others
// write the batch's new K/V rows. The attention grids behind start reading only once this whole
// grid has ended, so they see the new rows.
__global__ void __launch_bounds__(1024) rpa_plan_update_kernel(RpaArgs a, RpaUpdateArgs u) {
    if (blockIdx.x == 0)
        plan_body(a);
    else
        update_body(u, blockIdx.x - 1, gridDim.x - 1);
}

// ---------------------------------------------------------------------------
// Failure path check: one thread waits, through the bounded wait every pipeline uses, on an
// mbarrier nothing ever arrives on; the wait gives up after its limit, records
// RPA_DEV_ERR_TIMEOUT and the kernel returns (no fault, the context stays usable).
// ---------------------------------------------------------------------------
__global__ void rpa_wait_selftest_kernel(uint32_t* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, err);
}

cudaError_t launch_wait_selftest(uint32_t* err, cudaStream_t stream) {
    rpa_wait_selftest_kernel<<<1, 32, 0, stream>>>(err);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Launch helpers
// ---------------------------------------------------------------------------
// the attention launches behind the plan: with overlap, prefill on the plan's share of the SMs,
// decode started early (programmatic launch) on the rest and finishing after that prefill grid,
// then the prefill items still queued when decode ran dry, on every SM; otherwise prefill then
// decode
// A batch_kind hint drops the launches of the class it excludes: a decode-only batch launches
// decode alone, a prefill-only batch one prefill grid on every SM, each an ordinary launch behind
// the plan (it reads the plan's lists at its start, and later work on the stream starts only
// once it has ended).
static cudaError_t launch_attention(const RpaArgs& a, int num_sms, cudaStream_t stream) {
    if (a.batch_kind == RPA_BATCH_DECODE_ONLY) {
        RpaArgs d = a;
        d.overlap = 0;
        return launch_rpa_decode(d, num_sms, stream);
    }
    if (a.batch_kind == RPA_BATCH_PREFILL_ONLY) return launch_rpa_prefill(a, num_sms, stream, 2);
    cudaError_t e = launch_rpa_prefill(a, num_sms, stream, 0);
    if (e != cudaSuccess) return e;
    e = launch_rpa_decode(a, num_sms, stream);
    if (e != cudaSuccess || !a.overlap) return e;
    return launch_rpa_prefill(a, num_sms, stream, 1);
}

cudaError_t launch_rpa_forward(const RpaArgs& a, int num_sms, cudaStream_t stream) {
    cudaError_t e;
    {
        ProfScope ps("rpa_plan", stream);
        e = launch_pdl(rpa_plan_kernel, dim3(1), dim3(1024), 0, stream, a.overlap != 0, a);
    }
    if (e != cudaSuccess) return e;
    return launch_attention(a, num_sms, stream);
}

cudaError_t launch_rpa_forward_update(const RpaArgs& a, const RpaUpdateArgs& u, int num_sms, cudaStream_t stream) {
    // one warp per new token in 1024-thread blocks beside the plan's block, over as many SMs as
    // the batch fills (the tokens are interleaved over the blocks)
    const int ublocks = max(1, min(u.max_num_tokens, max(num_sms - 1, min(cdiv(u.max_num_tokens, 32), num_sms * 2))));
    const int smem = update_cache_ints(u.max_num_seqs) * (int)sizeof(int);
    {
        ProfScope ps("rpa_plan_update", stream);
        rpa_plan_update_kernel<<<1 + ublocks, 1024, smem, stream>>>(a, u);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return launch_attention(a, num_sms, stream);
}

cudaError_t launch_rpa_update(const RpaUpdateArgs& a, int num_sms, cudaStream_t stream) {
    const int grid = min(cdiv(a.max_num_tokens, 8), num_sms * 8);
    if (grid <= 0) return cudaSuccess;
    const int smem = update_cache_ints(a.max_num_seqs) * (int)sizeof(int);
    ProfScope ps("rpa_update", stream);
    rpa_update_kernel<<<grid, 256, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace rpa
