// Standard ragged paged attention (tpu-inference "ragged_paged_attention/v2/kernel.py")
// and its cache write, for sm_103a.
//
// One rpa_forward call = plan kernel + attention kernel(s), all on the caller's stream:
//   * rpa_plan_kernel reads the device metadata (num_seqs, cu_q_lens, kv_lens),
//     validates it, and writes two work lists into the workspace: "decode" items
//     (sequences whose q_len * G rows fit one 16-row tile, split along the keys) and
//     "prefill" items (64-row tiles of one KV head over the whole causal key range).
//   * rpa_attn_kernel<DECODE=true/false> are persistent CTAs that steal items from
//     their list.  K/V rows are gathered page by page with cp.async into swizzled
//     shared-memory stages; QK^T and PV run on bf16 tensor-core tiles with fp32
//     accumulation and an online softmax in the log2 domain.
//   * Split decode items store (m, l, unnormalised O) partials; the last CTA of a
//     group (atomic ticket) merges them with the log-sum-exp rule.
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
            dec_keys += (long long)(kl - klo) * n_groups;
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
        int ql = 0, kl = 0, nd = 0, np = 0, klo = 0, nsplit = 0;
        bool ok = s < num && seq_shape(a, s, ql, kl);
        if (ok && ql >= 1) {
            if (ql * G <= 16) {
                klo = decode_key_begin(a, ql, kl);
                nsplit = cdiv(kl - klo, chunk);
                nd = nsplit * n_groups;
            } else {
                np = cdiv(ql * G, kPrefillRows) * a.num_kv_heads;
            }
        }
        int tot_d, tot_p;
        const int od = block_exclusive_scan(nd, scan_scratch, &tot_d) + dec_base;
        const int op = block_exclusive_scan(np, scan_scratch, &tot_p) + pre_base;
        for (int g = 0; g < n_groups && nd; ++g) {
            for (int i = 0; i < nsplit; ++i) {
                const int it = od + g * nsplit + i;
                if (it >= a.max_dec_items) break;  // cannot happen: the host bound covers it
                WorkItem w;
                w.seq = s;
                w.head = g * a.decode_heads;
                w.key_begin = klo + i * chunk;
                w.key_end = min(kl, klo + (i + 1) * chunk);
                w.first_item = od + g * nsplit;
                w.num_splits = nsplit;
                w.split = i;
                w.row_begin = 0;
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
// Attention
// ---------------------------------------------------------------------------
template <int D, int NH, int BK, int STAGES, bool FP8>
struct RpaTile {
    static constexpr int kEsz = FP8 ? 1 : 2;
    static constexpr int kRowBytes = NH * 2 * D * kEsz;          // one key, NH heads, K and V
    static constexpr int kRowBytesBf16 = NH * 2 * D * 2;
    static constexpr int kChunksPerPart = D * kEsz / 16;         // 16-byte chunks in one K (or V) row
    static constexpr int kStageBytes = BK * kRowBytes;
    static constexpr int kConvBytes = FP8 ? BK * kRowBytesBf16 : 0;
    static constexpr int kQBytes = 64 * D * 2;
    static constexpr int kSmem = STAGES * kStageBytes + kConvBytes + kQBytes;
    static_assert(kRowBytes % 128 == 0, "swizzle needs 128-byte rows");
};

template <int D, int NH, int BK, int STAGES, bool FP8, bool DECODE>
__global__ void __launch_bounds__(128) rpa_attn_kernel(RpaArgs a) {
    using T = RpaTile<D, NH, BK, STAGES, FP8>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* stages = smem;
    uint8_t* conv = smem + STAGES * T::kStageBytes;
    uint8_t* qs = conv + T::kConvBytes;
    __shared__ WorkItem s_item;
    __shared__ int s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.num_q_heads / a.num_kv_heads;
    const int C = 2 * a.num_kv_heads;
    const int list = DECODE ? 0 : 1;
    const WorkItem* items = DECODE ? a.dec_items : a.pre_items;
    WsHeader* hdr = a.hdr;
    const uint8_t* kv = static_cast<const uint8_t*>(a.kv_pages);
    // the bf16 operand tile the MMAs read: the conversion buffer for fp8, the stage otherwise
    constexpr int kOpRowBytes = T::kRowBytesBf16;

    while (true) {
        __syncthreads();
        if (tid == 0) {
            const int it = atomicAdd(&hdr->next_item[list], 1);
            s_item.seq = -1;
            if (it < hdr->num_items[list]) {
                s_item = items[it];
                s_item.first_item = DECODE ? s_item.first_item : it;
                s_item.row_begin = DECODE ? it : s_item.row_begin;  // decode: remember own index
            }
        }
        __syncthreads();
        const WorkItem w = s_item;
        if (w.seq < 0) break;
        const int s = w.seq;
        const int q_start = a.cu_q_lens[s];
        const int q_len = a.cu_q_lens[s + 1] - q_start;
        const int kv_len = a.kv_lens[s];
        const int n_rows = q_len * G;  // rows of one KV head in this sequence

        // rows owned by this warp: 16 rows of one KV head
        const int my_head = DECODE ? w.head + warp : w.head;
        const int row0 = DECODE ? 0 : w.row_begin + warp * 16;
        const bool head_ok = my_head < a.num_kv_heads;
        // per-thread rows (g, g + 8) -> query position and window start
        int qpos[2], wlo[2];
        bool rv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int R = row0 + (lane >> 2) + e * 8;
            rv[e] = head_ok && R < n_rows;
            const int j = rv[e] ? R / G : 0;
            qpos[e] = kv_len - q_len + j;
            wlo[e] = a.sliding_window > 0 ? qpos[e] - a.sliding_window + 1 : 0;
            if (!rv[e]) qpos[e] = -1;
        }
        // key range of the whole CTA
        int kb, ke;
        if (DECODE) {
            kb = w.key_begin;
            ke = w.key_end;
        } else {
            const int R0 = w.row_begin;
            const int R1 = min(n_rows, w.row_begin + 64) - 1;
            const int qmin = kv_len - q_len + R0 / G;
            const int qmax = kv_len - q_len + R1 / G;
            kb = a.sliding_window > 0 ? max(0, qmin - a.sliding_window + 1) : 0;
            kb = kb / BK * BK;
            ke = qmax + 1;
        }
        const int n_blocks = ke > kb ? cdiv(ke - kb, BK) : 0;

        // ---- Q tile -> shared (rows of invalid tokens/heads are zero) ----
        {
            constexpr int kQChunks = D * 2 / 16;
            for (int i = tid; i < 64 * kQChunks; i += 128) {
                const int r = i / kQChunks, c = i % kQChunks;
                const int wr = r / 16;  // warp that owns the row
                const int head = DECODE ? w.head + wr : w.head;
                const int R = (DECODE ? 0 : w.row_begin + wr * 16) + (r % 16);
                const bool v = head < a.num_kv_heads && R < n_rows;
                const int j = v ? R / G : 0, g = v ? R % G : 0;
                const __nv_bfloat16* src = a.q + ((size_t)(q_start + j) * a.num_q_heads + head * G + g) * D + c * 8;
                cp_async16(smem_u32(qs + swz(r, c, D * 2)), v ? (const void*)src : (const void*)a.q, v);
            }
        }

        auto load_block = [&](int blk, int stage) {
            uint8_t* dst = stages + stage * T::kStageBytes;
            const int key0 = kb + blk * BK;
            constexpr int kChunksPerKey = NH * 2 * T::kChunksPerPart;
            for (int i = tid; i < BK * kChunksPerKey; i += 128) {
                const int kk = i / kChunksPerKey, c = i % kChunksPerKey;
                const int hh = c / (2 * T::kChunksPerPart);
                const int part = (c / T::kChunksPerPart) & 1;
                const int cc = c % T::kChunksPerPart;
                const int key = key0 + kk;
                const int head = (DECODE ? w.head : w.head) + hh;
                bool v = key < ke && key < kv_len && head < a.num_kv_heads;
                const uint8_t* src = kv;
                if (v) {
                    const int page = a.page_indices[(size_t)s * a.pages_per_seq + key / a.page_size];
                    if ((unsigned)page >= (unsigned)a.total_num_pages) {
                        set_error(&hdr->error_bits, RPA_DEV_ERR_PAGE);
                        v = false;
                    } else {
                        src = kv + ((((size_t)page * a.page_size + key % a.page_size) * C + 2 * head + part) * D) *
                                       T::kEsz +
                              cc * 16;
                    }
                }
                cp_async16(smem_u32(dst + swz(kk, c, T::kRowBytes)), src, v);
            }
        };

        // ---- prologue ----
#pragma unroll
        for (int st = 0; st < STAGES - 1; ++st) {
            if (st < n_blocks) load_block(st, st);
            cp_async_commit();
        }

        float o[D / 8][4];
#pragma unroll
        for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
        const float scale = a.sm_scale;
        const float cap = a.soft_cap;
        const uint32_t q_base = smem_u32(qs) ;
        const int kv_head_chunk = DECODE ? warp * 2 * (D * 2 / 16) : 0;  // chunk offset of this warp's K in a bf16 row

        for (int blk = 0; blk < n_blocks; ++blk) {
            {
                const int nb = blk + STAGES - 1;
                if (nb < n_blocks) load_block(nb, nb % STAGES);
                cp_async_commit();
            }
            cp_async_wait<STAGES - 1>();
            __syncthreads();
            const uint8_t* stage = stages + (blk % STAGES) * T::kStageBytes;
            const uint8_t* op = stage;
            if (FP8 || a.has_scale) {
                // dequantise: bf16(float(x) * scale), the reference's K/V conversion
                constexpr int kIn = T::kRowBytes / 16;  // 16-byte chunks per key row (input)
                uint8_t* dst = FP8 ? conv : const_cast<uint8_t*>(stage);
                for (int i = tid; i < BK * kIn; i += 128) {
                    const int kk = i / kIn, c = i % kIn;
                    const int part = (c / T::kChunksPerPart) & 1;
                    const float sc = part ? a.v_scale_or_one : a.k_scale_or_one;
                    const uint4 raw = *reinterpret_cast<const uint4*>(stage + swz(kk, c, T::kRowBytes));
                    if (FP8) {
                        const uint16_t* h = reinterpret_cast<const uint16_t*>(&raw);
                        uint32_t outw[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            float2 f = e4m3x2_to_float2(h[e]);
                            outw[e] = pack_bf16(f.x * sc, f.y * sc);
                        }
                        // input chunk c (16 fp8) -> output chunks 2c, 2c+1 (8 bf16 each)
                        *reinterpret_cast<uint4*>(dst + swz(kk, 2 * c, kOpRowBytes)) =
                            make_uint4(outw[0], outw[1], outw[2], outw[3]);
                        *reinterpret_cast<uint4*>(dst + swz(kk, 2 * c + 1, kOpRowBytes)) =
                            make_uint4(outw[4], outw[5], outw[6], outw[7]);
                    } else {
                        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
                        uint32_t outw[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float2 f = __bfloat1622float2(h[e]);
                            outw[e] = pack_bf16(f.x * sc, f.y * sc);
                        }
                        *reinterpret_cast<uint4*>(dst + swz(kk, c, T::kRowBytes)) =
                            make_uint4(outw[0], outw[1], outw[2], outw[3]);
                    }
                }
                __syncthreads();
                op = FP8 ? conv : stage;
            }
            const uint32_t op_base = smem_u32(op);
            const int key0 = kb + blk * BK;

            // ---- S = Q K^T ----
            float sc[BK / 8][4];
#pragma unroll
            for (int i = 0; i < BK / 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t af[4];
                ldsm_x4(q_base + swz(warp * 16 + (lane & 15), ks * 2 + (lane >> 4), D * 2), af[0], af[1], af[2], af[3]);
#pragma unroll
                for (int np = 0; np < BK / 16; ++np) {
                    uint32_t b0, b1, b2, b3;
                    const int key = np * 16 + ((lane >> 4) << 3) + (lane & 7);
                    ldsm_x4(op_base + swz(key, kv_head_chunk + ks * 2 + ((lane >> 3) & 1), kOpRowBytes), b0, b1, b2, b3);
                    mma_bf16(sc[2 * np], af, b0, b1);
                    mma_bf16(sc[2 * np + 1], af, b2, b3);
                }
            }
            // ---- scale, soft cap, mask ----
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nt = 0; nt < BK / 8; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = e >> 1;
                    const int key = key0 + nt * 8 + 2 * (lane & 3) + (e & 1);
                    float x = sc[nt][e] * scale;
                    if (cap != 0.f) x = cap * tanhf(x / cap);
                    x *= kLog2e;
                    const bool ok = key <= qpos[r] && key >= wlo[r] && key < kv_len;
                    x = ok ? x : -INFINITY;
                    sc[nt][e] = x;
                    mx[r] = fmaxf(mx[r], x);
                }
            }
            float alpha[2], muse[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                const float mn = fmaxf(m_run[r], mx[r]);
                muse[r] = mn == -INFINITY ? 0.f : mn;
                alpha[r] = fast_exp2(m_run[r] - muse[r]);
                m_run[r] = mn;
                l_run[r] *= alpha[r];
            }
#pragma unroll
            for (int nt = 0; nt < BK / 8; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p = fast_exp2(sc[nt][e] - muse[e >> 1]);
                    sc[nt][e] = p;
                    l_run[e >> 1] += p;
                }
            }
#pragma unroll
            for (int dt = 0; dt < D / 8; ++dt) {
                o[dt][0] *= alpha[0];
                o[dt][1] *= alpha[0];
                o[dt][2] *= alpha[1];
                o[dt][3] *= alpha[1];
            }
            // ---- O += P V ----
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                uint32_t pf[4];
                pf[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
                pf[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
                pf[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
                pf[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp) {
                    uint32_t b0, b1, b2, b3;
                    const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                    const int chunk = kv_head_chunk + (D * 2 / 16) + dp * 2 + (lane >> 4);
                    ldsm_x4_t(op_base + swz(key, chunk, kOpRowBytes), b0, b1, b2, b3);
                    mma_bf16(o[2 * dp], pf, b0, b1);
                    mma_bf16(o[2 * dp + 1], pf, b2, b3);
                }
            }
            __syncthreads();  // the stage (and conversion buffer) may be refilled now
        }
        cp_async_wait<0>();

        // ---- finalise ----
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
            l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
        }
        const int g8 = lane >> 2, q4 = lane & 3;
        if (!DECODE || w.num_splits == 1) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                if (!rv[e]) continue;
                const int R = row0 + g8 + e * 8;
                const int j = R / G, qh = my_head * G + R % G;
                const float inv = l_run[e] > 0.f ? 1.f / l_run[e] : 0.f;
                __nv_bfloat16* dst = a.out + ((size_t)(q_start + j) * a.num_q_heads + qh) * D;
#pragma unroll
                for (int dt = 0; dt < D / 8; ++dt)
                    *reinterpret_cast<uint32_t*>(dst + dt * 8 + 2 * q4) =
                        pack_bf16(o[dt][2 * e] * inv, o[dt][2 * e + 1] * inv);
            }
            continue;
        }
        // split decode: store the partial, then the last CTA of the group merges
        const int self = w.row_begin;  // own item index (set above)
        float* po = a.partial_o + (size_t)self * (NH * 16 * D);
        float* pml = a.partial_ml + (size_t)self * (NH * 16 * 2);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = warp * 16 + g8 + e * 8;
#pragma unroll
            for (int dt = 0; dt < D / 8; ++dt)
                *reinterpret_cast<float2*>(po + (size_t)r * D + dt * 8 + 2 * q4) = make_float2(o[dt][2 * e], o[dt][2 * e + 1]);
            if (q4 == 0) {
                pml[r * 2 + 0] = m_run[e];
                pml[r * 2 + 1] = l_run[e];
            }
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const int old = atomicAdd(&a.tickets[w.first_item], 1);
            s_last = old == w.num_splits - 1;
        }
        __syncthreads();
        if (!s_last) continue;
        __threadfence();
        // merge: warp `warp` handles head slot `warp`, rows 0..15 of it
        if (head_ok) {
            for (int r = 0; r < 16; ++r) {
                const int R = r;
                if (R >= n_rows) break;
                const int row = warp * 16 + r;
                float M = -INFINITY;
                for (int sp = 0; sp < w.num_splits; ++sp)
                    M = fmaxf(M, __ldcg(a.partial_ml + (size_t)(w.first_item + sp) * (NH * 16 * 2) + row * 2));
                const float Mu = M == -INFINITY ? 0.f : M;
                float L = 0.f;
                float acc[D / 32];
#pragma unroll
                for (int i = 0; i < D / 32; ++i) acc[i] = 0.f;
                for (int sp = 0; sp < w.num_splits; ++sp) {
                    const size_t it = (size_t)(w.first_item + sp);
                    const float m = __ldcg(a.partial_ml + it * (NH * 16 * 2) + row * 2);
                    const float l = __ldcg(a.partial_ml + it * (NH * 16 * 2) + row * 2 + 1);
                    const float f = fast_exp2(m - Mu);
                    L += f * l;
                    const float* src = a.partial_o + it * (NH * 16 * D) + (size_t)row * D;
#pragma unroll
                    for (int i = 0; i < D / 32; ++i) acc[i] += f * __ldcg(src + i * 32 + lane);
                }
                const float inv = L > 0.f ? 1.f / L : 0.f;
                const int j = R / G, qh = my_head * G + R % G;
                __nv_bfloat16* dst = a.out + ((size_t)(q_start + j) * a.num_q_heads + qh) * D;
#pragma unroll
                for (int i = 0; i < D / 32; ++i) dst[i * 32 + lane] = __float2bfloat16_rn(acc[i] * inv);
            }
        }
        if (tid == 0) a.tickets[w.first_item] = 0;
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
template <int D, int NH, int BK, int STAGES, bool FP8, bool DECODE>
static cudaError_t launch_attn(const RpaArgs& a, int grid, cudaStream_t stream) {
    using T = RpaTile<D, NH, BK, STAGES, FP8>;
    auto kern = rpa_attn_kernel<D, NH, BK, STAGES, FP8, DECODE>;
    static int per_sm = 0;  // resident CTAs per SM, computed once per process
    if (per_sm == 0) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmem);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 128, T::kSmem);
        if (e != cudaSuccess) return e;
        per_sm = n > 0 ? n : 1;
    }
    ProfScope ps(DECODE ? "rpa_decode_attn" : "rpa_prefill_attn", stream);
    kern<<<grid * (per_sm > 0 ? per_sm : 1), 128, T::kSmem, stream>>>(a);
    return cudaGetLastError();
}

template <int D, bool FP8>
static cudaError_t launch_rpa_d(const RpaArgs& a, int num_sms, cudaStream_t stream) {
    constexpr int kPreBK = D >= 256 ? 32 : 64;
    cudaError_t e = launch_attn<D, 1, kPreBK, 3, FP8, false>(a, num_sms, stream);
    if (e != cudaSuccess) return e;
    return launch_rpa_decode(a, num_sms, stream);
}

cudaError_t launch_rpa_forward(const RpaArgs& a, int num_sms, cudaStream_t stream) {
    cudaError_t e;
    {
        ProfScope ps("rpa_plan", stream);
        rpa_plan_kernel<<<1, 1024, 0, stream>>>(a);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    const bool fp8 = a.kv_fp8 != 0;
    switch (a.head_dim) {
        case 64: return fp8 ? launch_rpa_d<64, true>(a, num_sms, stream) : launch_rpa_d<64, false>(a, num_sms, stream);
        case 128: return fp8 ? launch_rpa_d<128, true>(a, num_sms, stream) : launch_rpa_d<128, false>(a, num_sms, stream);
        case 256: return fp8 ? launch_rpa_d<256, true>(a, num_sms, stream) : launch_rpa_d<256, false>(a, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_rpa_update(const RpaUpdateArgs& a, int num_sms, cudaStream_t stream) {
    const int grid = min(a.max_num_tokens, num_sms * 8);
    if (grid <= 0) return cudaSuccess;
    ProfScope ps("rpa_update", stream);
    rpa_update_kernel<<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace rpa
