// Decode-class work of ragged paged attention (tpu-inference "ragged_paged_attention/v2/
// kernel.py": sequences whose q_len * G query rows fit one 16-row tile), for sm_103a.
//
// Decode attention reads every visible key once and does ~2 flops per byte, so it is
// bound by HBM.  The kernel is a warp-specialised streaming pipeline:
//   * a producer warp walks the page table (lane t resolves token t of a 16-key stage,
//     one stage ahead) and issues one bulk (TMA 1-D) copy per token: the contiguous K/V
//     segment of HG KV heads of that token (HG * 2 * D elements) lands in a padded
//     shared-memory row (padding keeps ldmatrix conflict free); a full/empty mbarrier
//     pair per stage orders producer and consumers;
//   * HG consumer warps, one per KV head, run the contractions transposed so that the
//     16 keys of a stage fill the M side of the m16n8k16 tile and the item's <= 8 query
//     rows (G heads x q_len tokens) its N side: S^T = K Q^T with Q^T held as B fragments
//     in registers, then O^T += V^T P^T with V^T loaded by a transposing ldmatrix and
//     P^T moved into B-fragment layout by movmatrix; the online softmax runs per column
//     (a query row) across the 8 lanes that share it.  Half the tensor-core work and
//     half the accumulator registers of rows-on-M tiles, whose 16 rows would be mostly
//     padding; fp8 or int8 (or scaled bf16) K/V are dequantised by the warp into its own
//     bf16 rows as bf16(float(x) * scale): K first, then (after QK) V into the same rows;
//   * slots past kv_len are never copied: the stage memory is zeroed once at start, so
//     a skipped row holds finite data whose probability is exactly zero.
// Items split the keys of a sequence (flash-decoding); split partials (m, l, O) are
// merged by the last CTA of the group (atomic ticket), as in rpa_kernels.cu.
#include "common.cuh"
#include "kernels.h"
#include "profile.h"

namespace rpa {

template <int D, int HG, int ESZ, bool CONV, bool F16 = false, bool I4 = false>
struct DecTile {
    static constexpr int BK = kDecodeBK;                 // keys per stage
    // bytes of one token's segment (I4: half a byte an element)
    static constexpr int kSeg = I4 ? HG * D : HG * 2 * D * ESZ;
    static constexpr int kRow = kSeg + 16;               // padded shared-memory row
    static constexpr int kStage = BK * kRow;
    static constexpr int kConvRow = D * 2 + 16;          // one head's K (then V) in bf16, padded
    // (the f16 path converts straight into MMA fragments: no conversion rows)
    static constexpr int kConv = CONV && !F16 ? HG * BK * kConvRow : 0;
    // shared memory per CTA: two stages and (fp8) the conversion rows fit four fp8 or three
    // bf16 CTAs on an SM (with ~150 / ~95 registers a thread); measured on the Gemma-2 and
    // Llama decode batches, occupancy beats deeper rings here
    static constexpr int kBudget = CONV ? 56 * 1024 : 72 * 1024;
    static constexpr int kFit = (kBudget - kConv) / kStage;
    static constexpr int STAGES = kFit < 2 ? 2 : (kFit > 4 ? 4 : kFit);
    static constexpr int kBarOff = STAGES * kStage + kConv;
    static constexpr int kSmem = kBarOff + 2 * STAGES * 8;
    static constexpr int kThreads = (HG + 1) * 32;
    static_assert(kSeg % 16 == 0, "bulk copies move 16-byte multiples");
};

// 8 elements (K or V of one head) -> 8 bf16 of bf16(float(x) * scale), packed in a uint4
// (one-byte elements: e4m3, or int8 when I8).
template <int ESZ, bool I8 = false>
__device__ __forceinline__ uint4 dequant8(const uint8_t* src, float sc) {
    uint32_t w[4];
    if (ESZ == 1 && I8) {
        const uint2 raw = *reinterpret_cast<const uint2*>(src);
        const int8_t* b = reinterpret_cast<const int8_t*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = pack_bf16((float)b[2 * e] * sc, (float)b[2 * e + 1] * sc);
    } else if (ESZ == 1) {
        const uint2 raw = *reinterpret_cast<const uint2*>(src);
        const uint16_t* h = reinterpret_cast<const uint16_t*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = e4m3x2_to_float2(h[e]);
            w[e] = pack_bf16(f.x * sc, f.y * sc);
        }
    } else {
        const uint4 raw = *reinterpret_cast<const uint4*>(src);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            w[e] = pack_bf16(f.x * sc, f.y * sc);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// 8 int4 elements (4 bytes; element 2i in the low nibble of byte i) -> 8 bf16 of
// bf16(float(x) * scale), packed in a uint4.
__device__ __forceinline__ uint4 dequant_i4x8(const uint8_t* src, float sc) {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(src);
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int lo = (int)(v << (28 - 8 * e)) >> 28;  // nibble 2e, sign-extended
        const int hi = (int)(v << (24 - 8 * e)) >> 28;  // nibble 2e + 1
        w[e] = pack_bf16((float)lo * sc, (float)hi * sc);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// 8 one-byte elements (e4m3, or int8 when I8) -> 8 f16 (exact, unscaled), packed in a uint4.
template <bool I8>
__device__ __forceinline__ uint4 byte8_to_f16(const uint8_t* src) {
    const uint2 raw = *reinterpret_cast<const uint2*>(src);
    const uint16_t* h = reinterpret_cast<const uint16_t*>(&raw);
    if (I8) return make_uint4(s8x2_to_f16x2(h[0]), s8x2_to_f16x2(h[1]), s8x2_to_f16x2(h[2]), s8x2_to_f16x2(h[3]));
    return make_uint4(e4m3x2_to_f16x2(h[0]), e4m3x2_to_f16x2(h[1]), e4m3x2_to_f16x2(h[2]), e4m3x2_to_f16x2(h[3]));
}

// Two one-byte elements (the low 16 bits of v) -> an f16 pair, exactly.
template <bool I8>
__device__ __forceinline__ uint32_t byte2_to_f16x2(uint32_t v) {
    return I8 ? s8x2_to_f16x2((uint16_t)(v & 0xFFFFu)) : e4m3x2_to_f16x2((uint16_t)(v & 0xFFFFu));
}

// f16 path, fragment layouts.  A dot product is the same under any order of its terms, so K and
// Q use one permutation of the head dims chosen for the loads: lane (g8, q4) of the S^T = K Q^T
// MMA reads, per K row, the 16-byte chunks kchunk(q4, i) (spread so a quarter-warp hits eight
// distinct bank groups), and k-step ks takes bytes 4 (ks & 3).. of chunk kchunk(q4, ks >> 2).
template <int D>
__device__ __forceinline__ int kchunk(int q4, int i) {
    if constexpr (D >= 256)
        return 2 * q4 + 8 * (i & 1) + (i >> 1);
    else if constexpr (D == 128)
        return 2 * q4 + i;
    else
        return q4;
}
// O^T = V^T P^T permutes the output dims instead (undone by the stores): lane g8 of tile t holds
// dims vdim(g8, 2t) and vdim(g8, 2t + 1), the bytes 2t, 2t + 1 of its D/8 bytes of each V row
// (16-byte chunks g8 + 8i, or 8 bytes at 8 g8 when D = 64).
template <int D>
__device__ __forceinline__ int vdim(int g8, int j) {
    if constexpr (D >= 128)
        return 16 * (g8 + 8 * (j >> 4)) + (j & 15);
    else
        return 8 * g8 + j;
}

// F16 (fp8 or int8 caches whose k_scale and v_scale are powers of two): bf16(float(x) * scale)
// is then exactly x * scale, so K and V go to the tensor cores as exact f16 values and the
// scales are applied to S and O instead; each query row is brought into f16 range by a power
// of two (undone on its scores), which keeps its bf16 values exact.  The one-byte K and V rows
// are converted straight into MMA fragments (permuted head dims, see kchunk / vdim): no
// conversion rows in shared memory, no ldmatrix.  I8: the one-byte elements are int8.
// I4: int4 caches (two elements a byte), dequantised into the bf16 conversion rows.
template <int D, int HG, int ESZ, bool CONV, bool F16 = false, bool I8 = false, bool I4 = false>
__global__ void __launch_bounds__(DecTile<D, HG, ESZ, CONV, F16, I4>::kThreads) rpa_decode_kernel(RpaArgs a) {
    using T = DecTile<D, HG, ESZ, CONV, F16, I4>;
    static_assert(!F16 || (CONV && ESZ == 1 && !I4), "the f16 path takes one-byte caches");
    static_assert(!I8 || (CONV && ESZ == 1), "int8 caches take the converting path");
    static_assert(!I4 || (CONV && !F16 && !I8), "int4 caches take the bf16 converting path");
    constexpr int kRowB = I4 ? D / 2 : D * ESZ;  // bytes of one head row of K or V
    constexpr int BK = T::BK, STAGES = T::STAGES;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem;
    uint8_t* conv = smem + STAGES * T::kStage;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::kBarOff);
    uint64_t* empty = full + STAGES;
    __shared__ WorkItem s_item;
    __shared__ int s_item_idx, s_last;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool producer = warp == HG;
    WsHeader* hdr = a.hdr;
    uint32_t* err = &hdr->error_bits;
    const int Hkv = a.num_kv_heads, G = a.num_q_heads / Hkv, C = 2 * Hkv;
    const uint8_t* kv = static_cast<const uint8_t*>(a.kv_pages);

    // zero the stages once: rows that are never copied (slots past kv_len) stay finite
    for (int i = tid * 16; i < STAGES * T::kStage; i += blockDim.x * 16)
        *reinterpret_cast<uint4*>(stages + i) = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int st = 0; st < STAGES; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], HG);
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    fence_proxy_async_smem();
    __syncthreads();

    uint32_t pipe = 0;            // blocks this CTA has pushed through the ring so far
    uint32_t issued_phase[4] = {0, 0, 0, 0};  // producer: last phase issued per stage (+1)

    // prefill first (the plan gave it every SM): start once it has ended, so that the CTAs
    // begin their equal shares together (no-op on an ordinary launch)
    if (hdr->prefill_ctas >= a.num_sms && hdr->num_items[1] > 0) pdl_wait();
    // shares are runs of consecutive items laid out by the plan kernel: this CTA's own (the
    // first dec_ctas CTAs have one), then shares taken from the pool (thread 0 keeps the run)
    const int n_items = hdr->num_items[0], n_static = hdr->dec_ctas, n_shares = hdr->dec_shares;
    int my_it = 0, my_end = 0;
    bool pool_left = true;
    if (tid == 0 && (int)blockIdx.x < n_static) {
        my_it = min(max(a.cta_first[blockIdx.x], 0), n_items);
        my_end = min(max(a.cta_first[blockIdx.x + 1], my_it), n_items);
    }
    while (true) {
        if (tid == 0) {
            while (my_it >= my_end && pool_left) {
                const int c = n_static + atomicAdd(&hdr->next_item[2], 1);
                if (c >= n_shares) {
                    pool_left = false;
                } else {
                    my_it = min(max(a.cta_first[c], 0), n_items);
                    my_end = min(max(a.cta_first[c + 1], my_it), n_items);
                }
            }
            const int it = my_it < my_end ? my_it++ : -1;
            s_item.seq = -1;
            s_item_idx = it;
            if (it >= 0) s_item = a.dec_items[it];
        }
        __syncthreads();
        const WorkItem w = s_item;
        const int self = s_item_idx;
        if (w.seq < 0 || s_abort) break;
        const int s = w.seq;
        const int q_start = a.cu_q_lens[s];
        const int q_len = a.cu_q_lens[s + 1] - q_start;
        const int kv_len = a.kv_lens[s];
        const int n_rows = q_len * G;
        const int kb = w.key_begin, ke = w.key_end;
        const int n_blocks = ke > kb ? cdiv(ke - kb, BK) : 0;
        const int h0 = w.head;
        const int seg_heads = min(HG, Hkv - h0);
        const uint32_t seg_bytes = seg_heads * 2 * kRowB;

        if (producer) {
            // lane t < BK owns token t of every stage: it resolves that token's page (the
            // next stage's entry is fetched while this stage's slot is still busy) and
            // issues the token's bulk copy, so the 16 copies of a stage go out together.
            const size_t tbl = (size_t)s * a.pages_per_seq;
            auto page_of = [&](int blk) -> int {
                const int key = kb + blk * BK + lane;
                return (lane < BK && blk < n_blocks && key < ke) ? __ldg(a.page_indices + tbl + key / a.page_size)
                                                                 : -1;
            };
            int page_next = page_of(0);
            for (int blk = 0; blk < n_blocks; ++blk) {
                const uint32_t q = pipe + blk, st = q % STAGES, ph = (q / STAGES) & 1;
                const int page = page_next;
                page_next = page_of(blk + 1);
                const int key = kb + blk * BK + lane;
                const bool want = lane < BK && key < ke;
                const bool ok = want && (unsigned)page < (unsigned)a.total_num_pages;
                if (want && !ok) set_error(err, RPA_DEV_ERR_PAGE);
                const uint32_t mask = __ballot_sync(0xffffffffu, ok);
                int go = 1;
                if (lane == 0) {
                    go = mbar_wait(&empty[st], ph ^ 1, err);
                    if (go) {
                        mbar_arrive_expect_tx(&full[st], __popc(mask) * seg_bytes);
                        issued_phase[st] = ph + 1;
                    } else {
                        s_abort = 1;
                    }
                }
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) break;
                if (ok) {
                    const uint8_t* src =
                        kv + (((size_t)page * a.page_size + key % a.page_size) * C + 2 * h0) * (size_t)kRowB;
                    bulk_g2s(smem_u32(stages + st * T::kStage + lane * T::kRow), src, seg_bytes, &full[st]);
                }
            }
        } else {
            // ---------------- consumer warp: KV head h0 + warp ----------------
            // C-fragment columns of this thread: rows rb + 2*q4 + {0,1}; B-fragment column: row rb + g8
            const bool head_ok = warp < seg_heads;
            const int head = h0 + warp;
            const int g8 = lane >> 2, q4 = lane & 3;
            const int rb = w.row_begin;
            int qpos[2], wlo[2];
            bool rv[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int R = rb + 2 * q4 + j;
                rv[j] = head_ok && R < n_rows;
                qpos[j] = rv[j] ? kv_len - q_len + R / G : -1;
                wlo[j] = a.sliding_window > 0 ? qpos[j] - a.sliding_window + 1 : 0;
            }
            const int Rb = rb + g8;
            const bool rvb = head_ok && Rb < n_rows;
            // Q^T as B fragments: column g8, k = dims 2*q4.. and 2*q4+8.. of each 16-wide step
            uint32_t qb[D / 16][2];
            {
                const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                    a.q + ((size_t)(q_start + (rvb ? Rb / G : 0)) * a.num_q_heads + head * G + (rvb ? Rb % G : 0)) * D);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    // (f16 path: the dims of K's permuted A fragments, kchunk)
                    const int w0 = F16 ? 8 * kchunk<D>(q4, ks >> 2) + 2 * (ks & 3) : ks * 8 + q4;
                    const int w1 = F16 ? w0 + 1 : ks * 8 + 4 + q4;
                    qb[ks][0] = rvb ? __ldg(qrow + w0) : 0u;
                    qb[ks][1] = rvb ? __ldg(qrow + w1) : 0u;
                }
            }
            // F16: the row's power-of-two range factor (its 4 lanes hold its D values), the
            // fragments re-packed as f16, and each C column's factor back on its scores
            float colmul[2] = {1.f, 1.f};
            if (F16) {
                float mabs = 0.f;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qb[ks][h]));
                        mabs = fmaxf(mabs, fmaxf(fabsf(f.x), fabsf(f.y)));
                    }
                mabs = fmaxf(mabs, __shfl_xor_sync(0xffffffffu, mabs, 1));
                mabs = fmaxf(mabs, __shfl_xor_sync(0xffffffffu, mabs, 2));
                int ex = 0;
                frexpf(mabs, &ex);                               // mabs < 2^ex
                const int k = max(-30, min(100, ex - 15));       // mabs * 2^-k in [2^14, 2^15)
                const float qs = ldexpf(1.f, -k);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qb[ks][h]));
                        qb[ks][h] = pack_f16(f.x * qs, f.y * qs);
                    }
                const float rowmul = ldexpf(1.f, k);
#pragma unroll
                for (int j = 0; j < 2; ++j) colmul[j] = __shfl_sync(0xffffffffu, rowmul, (2 * q4 + j) * 4) * a.k_scale_or_one;
            }
            // O^T tiles: rows (dims) 16*dm + g8 and +8, columns (query rows) 2*q4, 2*q4+1
            float o[D / 16][4];
#pragma unroll
            for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
            float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
            const float scale = a.sm_scale, cap = a.soft_cap;
            const float cap_k2 = cap != 0.f ? 2.f * kLog2e / cap : 0.f;

            for (int blk = 0; blk < n_blocks; ++blk) {
                const uint32_t qn = pipe + blk, st = qn % STAGES, ph = (qn / STAGES) & 1;
                if (!mbar_wait(&full[st], ph, err)) {
                    s_abort = 1;
                    break;
                }
                const uint8_t* stg = stages + st * T::kStage;
                uint32_t kbase, vbase;
                int rowb;
                uint8_t* cb = conv + warp * BK * T::kConvRow;
                // CONV: dequantise 16 rows of K (part 0) or V (part 1) of this warp's head into cb
                auto convert = [&](int part) {
                    constexpr int kChunks = D / 8;  // 8-element chunks of K or V per key
                    const float sc = part == 0 ? a.k_scale_or_one : a.v_scale_or_one;
#pragma unroll 4
                    for (int i = lane; i < BK * kChunks; i += 32) {
                        const int kk = i / kChunks, c = i % kChunks;
                        const uint8_t* src = stg + kk * T::kRow + (warp * 2 + part) * kRowB + c * 8 * kRowB / D;
                        *reinterpret_cast<uint4*>(cb + kk * T::kConvRow + c * 16) =
                            I4 ? dequant_i4x8(src, sc) : F16 ? byte8_to_f16<I8>(src) : dequant8<ESZ, I8>(src, sc);
                    }
                    __syncwarp();
                };
                if (CONV && !F16) {
                    if (head_ok) convert(0);
                    kbase = vbase = smem_u32(cb);
                    rowb = T::kConvRow;
                } else if (F16) {
                    kbase = vbase = 0u;  // (fragments come straight from the stage rows)
                    rowb = T::kRow;
                } else {
                    kbase = smem_u32(stg) + warp * 2 * D * 2;
                    vbase = kbase + D * 2;
                    rowb = T::kRow;
                }
                if (head_ok) {
                    const int key0 = kb + blk * BK;
                    // S^T [16 keys x 8 rows] = K Q^T; A = K rows (ldmatrix: keys 0-7 / 8-15, dims 0-7 / 8-15)
                    float sc[4] = {0.f, 0.f, 0.f, 0.f};
                    if constexpr (F16) {
                        // K rows g8 and g8 + 8 of this warp's head, converted into A fragments
                        const uint8_t* kr0 = stg + g8 * T::kRow + warp * 2 * D;
                        const uint8_t* kr1 = kr0 + 8 * T::kRow;
#pragma unroll
                        for (int i = 0; i < D / 64; ++i) {
                            const int c = kchunk<D>(q4, i);
                            const uint4 u0 = *reinterpret_cast<const uint4*>(kr0 + c * 16);
                            const uint4 u1 = *reinterpret_cast<const uint4*>(kr1 + c * 16);
                            const uint32_t x0[4] = {u0.x, u0.y, u0.z, u0.w}, x1[4] = {u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                uint32_t ka4[4];
                                ka4[0] = byte2_to_f16x2<I8>(x0[e]);        // key g8, dims d, d + 1
                                ka4[1] = byte2_to_f16x2<I8>(x1[e]);        // key g8 + 8
                                ka4[2] = byte2_to_f16x2<I8>(x0[e] >> 16);  // key g8, dims d + 2, d + 3
                                ka4[3] = byte2_to_f16x2<I8>(x1[e] >> 16);
                                mma_f16(sc, ka4, qb[4 * i + e][0], qb[4 * i + e][1]);
                            }
                        }
                    } else {
                        const uint32_t ka = kbase + ((lane & 7) + ((lane >> 3) & 1) * 8) * rowb + (lane >> 4) * 16;
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            uint32_t ka4[4];
                            ldsm_x4(ka + ks * 32, ka4[0], ka4[1], ka4[2], ka4[3]);
                            mma_bf16(sc, ka4, qb[ks][0], qb[ks][1]);
                        }
                    }
                    if (CONV && !F16) {
                        __syncwarp();  // every lane is done reading K out of cb
                        convert(1);
                    }
                    // sc[e]: key g8 + 8*(e>>1), row 2*q4 + (e&1)
                    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = e & 1;
                        const int key = key0 + g8 + (e >> 1) * 8;
                        float x = sc[e] * (F16 ? scale * colmul[j] : scale);
                        if (cap != 0.f) x = soft_cap(x, cap, cap_k2);
                        x *= kLog2e;
                        const bool ok = key <= qpos[j] && key >= wlo[j] && key < ke;
                        // a mild mask adds mask_value to a masked logit of a key in the range
                        x = ok ? x : (a.mask_mild && key < ke) ? x + a.mask_value * kLog2e : -INFINITY;
                        sc[e] = x;
                        mx[j] = fmaxf(mx[j], x);
                    }
                    float alpha[2], muse[2];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 4));
                        mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 8));
                        mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 16));
                        const float mn = fmaxf(m_run[j], mx[j]);
                        muse[j] = mn == -INFINITY ? 0.f : mn;
                        alpha[j] = fast_exp2(m_run[j] - muse[j]);
                        m_run[j] = mn;
                        l_run[j] *= alpha[j];
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float p = fast_exp2(sc[e] - muse[e & 1]);
                        sc[e] = p;
                        l_run[e & 1] += p;
                    }
                    // P^T as B fragments (k = keys 2*q4.., n = row g8): transpose the 8x8 blocks
                    const uint32_t pb0 = movmatrix_t(F16 ? pack_f16(sc[0], sc[1]) : pack_bf16(sc[0], sc[1]));
                    const uint32_t pb1 = movmatrix_t(F16 ? pack_f16(sc[2], sc[3]) : pack_bf16(sc[2], sc[3]));
                    // O^T [16 dims x 8 rows] += V^T P^T
                    if constexpr (F16) {
                        // A = V^T from keys 2 q4, 2 q4 + 1, 2 q4 + 8, 2 q4 + 9: a byte permute pairs
                        // two keys' elements of one dim, one convert makes the f16 pair
                        const uint8_t* vr = stg + warp * 2 * D + D;
                        const uint8_t* v0 = vr + (2 * q4) * T::kRow;
                        const uint8_t* v1 = v0 + T::kRow;
                        const uint8_t* v2 = v0 + 8 * T::kRow;
                        const uint8_t* v3 = v2 + T::kRow;
                        constexpr int kVW = D / 32;  // 32-bit words of this lane's D/8 bytes per row
                        uint32_t w0[kVW], w1[kVW], w2[kVW], w3[kVW];
                        if constexpr (D >= 128) {
#pragma unroll
                            for (int i = 0; i < D / 128; ++i) {
                                const int off = 16 * (g8 + 8 * i);
                                const uint4 r0 = *reinterpret_cast<const uint4*>(v0 + off);
                                const uint4 r1 = *reinterpret_cast<const uint4*>(v1 + off);
                                const uint4 r2 = *reinterpret_cast<const uint4*>(v2 + off);
                                const uint4 r3 = *reinterpret_cast<const uint4*>(v3 + off);
                                w0[4 * i] = r0.x; w0[4 * i + 1] = r0.y; w0[4 * i + 2] = r0.z; w0[4 * i + 3] = r0.w;
                                w1[4 * i] = r1.x; w1[4 * i + 1] = r1.y; w1[4 * i + 2] = r1.z; w1[4 * i + 3] = r1.w;
                                w2[4 * i] = r2.x; w2[4 * i + 1] = r2.y; w2[4 * i + 2] = r2.z; w2[4 * i + 3] = r2.w;
                                w3[4 * i] = r3.x; w3[4 * i + 1] = r3.y; w3[4 * i + 2] = r3.z; w3[4 * i + 3] = r3.w;
                            }
                        } else {
                            const int off = 8 * g8;
                            const uint2 r0 = *reinterpret_cast<const uint2*>(v0 + off);
                            const uint2 r1 = *reinterpret_cast<const uint2*>(v1 + off);
                            const uint2 r2 = *reinterpret_cast<const uint2*>(v2 + off);
                            const uint2 r3 = *reinterpret_cast<const uint2*>(v3 + off);
                            w0[0] = r0.x; w0[1] = r0.y; w1[0] = r1.x; w1[1] = r1.y;
                            w2[0] = r2.x; w2[1] = r2.y; w3[0] = r3.x; w3[1] = r3.y;
                        }
#pragma unroll
                        for (int wd = 0; wd < kVW; ++wd) {
                            // bytes 4 wd .. 4 wd + 3: tiles 2 wd (bytes 0, 1) and 2 wd + 1 (bytes 2, 3)
                            const uint32_t lo01 = __byte_perm(w0[wd], w1[wd], 0x5140), hi01 = __byte_perm(w0[wd], w1[wd], 0x7362);
                            const uint32_t lo23 = __byte_perm(w2[wd], w3[wd], 0x5140), hi23 = __byte_perm(w2[wd], w3[wd], 0x7362);
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int dm = 2 * wd + h;
                                const uint32_t p01 = h ? hi01 : lo01, p23 = h ? hi23 : lo23;
                                o[dm][0] *= alpha[0];
                                o[dm][1] *= alpha[1];
                                o[dm][2] *= alpha[0];
                                o[dm][3] *= alpha[1];
                                uint32_t va4[4];
                                va4[0] = byte2_to_f16x2<I8>(p01);        // dim vdim(g8, 2 dm), keys 2 q4, 2 q4 + 1
                                va4[1] = byte2_to_f16x2<I8>(p01 >> 16);  // dim vdim(g8, 2 dm + 1)
                                va4[2] = byte2_to_f16x2<I8>(p23);        // keys 2 q4 + 8, 2 q4 + 9
                                va4[3] = byte2_to_f16x2<I8>(p23 >> 16);
                                mma_f16(o[dm], va4, pb0, pb1);
                            }
                        }
                    } else {
                        // A = V^T by a transposing ldmatrix of V rows
                        const uint32_t va = vbase + ((lane & 7) + ((lane >> 4) << 3)) * rowb + ((lane >> 3) & 1) * 16;
#pragma unroll
                        for (int dm = 0; dm < D / 16; ++dm) {
                            o[dm][0] *= alpha[0];
                            o[dm][1] *= alpha[1];
                            o[dm][2] *= alpha[0];
                            o[dm][3] *= alpha[1];
                            uint32_t va4[4];
                            ldsm_x4_t(va + dm * 32, va4[0], va4[1], va4[2], va4[3]);
                            mma_bf16(o[dm], va4, pb0, pb1);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);  // (CONV: free once V was converted)
            }
            // ---- results of this warp's rows ----
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 4);
                l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 8);
                l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 16);
            }
            // (warp-uniform: the movmatrix below is warp-collective)
            if (!__any_sync(0xffffffffu, s_abort != 0) && head_ok) {
                if (F16 && w.num_splits == 1) {
                    // the thread's two columns are query rows 2 q4 + j; each tile's pair of C rows
                    // is two adjacent head dims (vdim): one 32-bit store per row and tile
                    const float vs = a.v_scale_or_one;  // (V went in unscaled)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        if (!rv[j]) continue;
                        const int R = rb + 2 * q4 + j;
                        const float inv = l_run[j] > 0.f ? vs / l_run[j] : 0.f;
                        __nv_bfloat16* dst = a.out + ((size_t)(q_start + R / G) * a.num_q_heads + head * G + R % G) * D;
#pragma unroll
                        for (int dm = 0; dm < D / 16; ++dm)
                            *reinterpret_cast<uint32_t*>(dst + vdim<D>(g8, 2 * dm)) =
                                pack_bf16(o[dm][j] * inv, o[dm][2 + j] * inv);
                    }
                } else if (w.num_splits == 1) {
                    // normalise per column, transpose each 8x8 block back to rows: thread then
                    // holds row rb + g8, dims 2*q4, 2*q4+1 of the block (32-bit stores)
                    const float vs = F16 ? a.v_scale_or_one : 1.f;  // (F16: V went in unscaled)
                    const float inv0 = l_run[0] > 0.f ? vs / l_run[0] : 0.f;
                    const float inv1 = l_run[1] > 0.f ? vs / l_run[1] : 0.f;
                    __nv_bfloat16* dst = a.out + ((size_t)(q_start + (rvb ? Rb / G : 0)) * a.num_q_heads + head * G +
                                                  (rvb ? Rb % G : 0)) * D;
#pragma unroll
                    for (int dm = 0; dm < D / 16; ++dm) {
                        const uint32_t t0 = movmatrix_t(pack_bf16(o[dm][0] * inv0, o[dm][1] * inv1));
                        const uint32_t t1 = movmatrix_t(pack_bf16(o[dm][2] * inv0, o[dm][3] * inv1));
                        if (rvb) {
                            *reinterpret_cast<uint32_t*>(dst + dm * 16 + 2 * q4) = t0;
                            *reinterpret_cast<uint32_t*>(dst + dm * 16 + 8 + 2 * q4) = t1;
                        }
                    }
                } else {
                    // partials: kDecodeRows rows per KV head, numbered from the item's first row
                    float* po = a.partial_o + (size_t)self * (a.decode_heads * kDecodeRows * D);
                    float* pml = a.partial_ml + (size_t)self * (a.decode_heads * kDecodeRows * 2);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        if (!rv[j]) continue;
                        const int r = warp * kDecodeRows + 2 * q4 + j;
                        const float vs = F16 ? a.v_scale_or_one : 1.f;
#pragma unroll
                        for (int dm = 0; dm < D / 16; ++dm) {
                            const int d0 = F16 ? vdim<D>(g8, 2 * dm) : dm * 16 + g8;
                            const int d1 = F16 ? d0 + 1 : dm * 16 + 8 + g8;
                            po[(size_t)r * D + d0] = o[dm][j] * vs;
                            po[(size_t)r * D + d1] = o[dm][2 + j] * vs;
                        }
                        if (g8 == 0) {
                            pml[r * 2] = m_run[j];
                            pml[r * 2 + 1] = l_run[j];
                        }
                    }
                }
            }
        }
        pipe += n_blocks;
        __syncthreads();
        if (s_abort) break;
        if (w.num_splits == 1) continue;
        // ---- split merge: the last CTA of the group combines every split ----
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last = atomicAdd(&a.tickets[w.first_item], 1) == w.num_splits - 1;
        __syncthreads();
        if (!s_last) continue;
        __threadfence();
        if (!producer && warp < seg_heads) {
            const int head = h0 + warp;
            for (int R = w.row_begin; R < min(n_rows, w.row_begin + kDecodeRows); ++R) {
                const int row = warp * kDecodeRows + (R - w.row_begin);
                float M = -INFINITY;
                for (int sp = 0; sp < w.num_splits; ++sp)
                    M = fmaxf(M, __ldcg(a.partial_ml + (size_t)(w.first_item + sp) * (a.decode_heads * kDecodeRows * 2) + row * 2));
                const float Mu = M == -INFINITY ? 0.f : M;
                float L = 0.f;
                float acc[D / 32];
#pragma unroll
                for (int i = 0; i < D / 32; ++i) acc[i] = 0.f;
                for (int sp = 0; sp < w.num_splits; ++sp) {
                    const size_t it = (size_t)(w.first_item + sp);
                    const float m = __ldcg(a.partial_ml + it * (a.decode_heads * kDecodeRows * 2) + row * 2);
                    const float l = __ldcg(a.partial_ml + it * (a.decode_heads * kDecodeRows * 2) + row * 2 + 1);
                    const float f = fast_exp2(m - Mu);
                    L += f * l;
                    const float* src = a.partial_o + it * (a.decode_heads * kDecodeRows * D) + (size_t)row * D;
#pragma unroll
                    for (int i = 0; i < D / 32; ++i) acc[i] += f * __ldcg(src + i * 32 + lane);
                }
                const float inv = L > 0.f ? 1.f / L : 0.f;
                __nv_bfloat16* dst = a.out + ((size_t)(q_start + R / G) * a.num_q_heads + head * G + R % G) * D;
#pragma unroll
                for (int i = 0; i < D / 32; ++i) dst[i * 32 + lane] = __float2bfloat16_rn(acc[i] * inv);
            }
        }
        if (tid == 0) a.tickets[w.first_item] = 0;
    }
    // after an abort, wait (bounded) until no bulk copy can still land in this CTA's memory
    if (producer && lane == 0 && s_abort) {
        for (int st = 0; st < STAGES; ++st)
            if (issued_phase[st]) mbar_wait(&full[st], issued_phase[st] - 1, err);
    }
    // a CTA with a share is out of decode work (the prefill grid's signal when there is no pool)
    if (tid == 0 && (int)blockIdx.x < n_static) atomicAdd(&hdr->next_item[0], 1);
    // started early beside the prefill grid: end after it, so that the stream order seen by
    // later launches is the plain one (no-op on an ordinary launch)
    if (tid == 0) pdl_wait();
}

// per_sm_out != nullptr: only report the kernel's resident CTAs per SM (no launch)
template <int D, int HG, int ESZ, bool CONV, bool F16 = false, bool I8 = false, bool I4 = false>
static cudaError_t launch_decode(const RpaArgs& a, int num_sms, cudaStream_t stream, int* per_sm_out) {
    using T = DecTile<D, HG, ESZ, CONV, F16, I4>;
    auto kern = rpa_decode_kernel<D, HG, ESZ, CONV, F16, I8, I4>;
    static int per_sm = 0;
    if (per_sm == 0) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmem);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, T::kThreads, T::kSmem);
        if (e != cudaSuccess) return e;
        per_sm = n > 0 ? n : 1;
    }
    if (per_sm_out) {
        *per_sm_out = per_sm;
        return cudaSuccess;
    }
    ProfScope ps("rpa_decode_attn", stream);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms * per_sm);
    cfg.blockDim = dim3(T::kThreads);
    cfg.dynamicSmemBytes = T::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

int decode_heads_for(int head_dim, bool fp8) {
    (void)fp8;
    return head_dim >= 256 ? 2 : 4;
}

template <int D>
static cudaError_t launch_decode_d(const RpaArgs& a, int num_sms, cudaStream_t stream, int* per_sm_out) {
    constexpr int HG = D >= 256 ? 2 : 4;
    const bool pow2 = rpa_pow2_scale(a.k_scale_or_one) && rpa_pow2_scale(a.v_scale_or_one);
    if (a.kv_int4) return launch_decode<D, HG, 1, true, false, false, true>(a, num_sms, stream, per_sm_out);
    if (a.kv_int8 && pow2) return launch_decode<D, HG, 1, true, true, true>(a, num_sms, stream, per_sm_out);
    if (a.kv_int8) return launch_decode<D, HG, 1, true, false, true>(a, num_sms, stream, per_sm_out);
    if (a.kv_byte && pow2) return launch_decode<D, HG, 1, true, true>(a, num_sms, stream, per_sm_out);
    if (a.kv_byte) return launch_decode<D, HG, 1, true>(a, num_sms, stream, per_sm_out);
    if (a.has_scale) return launch_decode<D, HG, 2, true>(a, num_sms, stream, per_sm_out);
    return launch_decode<D, HG, 2, false>(a, num_sms, stream, per_sm_out);
}

static cudaError_t decode_dispatch(const RpaArgs& a, int num_sms, cudaStream_t stream, int* per_sm_out) {
    switch (a.head_dim) {
        case 64: return launch_decode_d<64>(a, num_sms, stream, per_sm_out);
        // head_dim 96 and 192: bf16 caches without scales (the host admits nothing else)
        case 96: return launch_decode<96, 4, 2, false>(a, num_sms, stream, per_sm_out);
        case 128: return launch_decode_d<128>(a, num_sms, stream, per_sm_out);
        case 192: return launch_decode<192, 4, 2, false>(a, num_sms, stream, per_sm_out);
        case 256: return launch_decode_d<256>(a, num_sms, stream, per_sm_out);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_rpa_decode(const RpaArgs& a, int num_sms, cudaStream_t stream) {
    return decode_dispatch(a, num_sms, stream, nullptr);
}

int rpa_decode_ctas_per_sm(const RpaArgs& a) {
    int n = 0;
    return decode_dispatch(a, 0, nullptr, &n) == cudaSuccess ? n : 0;
}

}  // namespace rpa
