// Prefill-class work of ragged paged attention (tpu-inference "ragged_paged_attention/v2/
// kernel.py": sequences whose q_len * G query rows exceed one 16-row tile) on the
// 5th-generation tensor cores of sm_103a.
//
// A work item is 128 query rows of one KV head (rows are (token, q head of the GQA
// group), token-major) against its causal / windowed key range.  Per CTA:
//   * producers gather the item's Q rows and, per key block, the K
//     and V rows of that KV head page by page into 128-byte-swizzled K-major panels.
//     bf16 caches go by TMA (one 3-D tensor copy per page-sized box and 64-wide panel,
//     issued by the lanes of two warps per operand, pages looked up one block ahead; the
//     partial last page is copied by those warps through registers); one-byte and scaled
//     caches go through registers in the same warps 8-11 and are converted there
//     (bf16(float(x) * scale), or exact f16 with power-of-two scales).  Rows past the key range are never copied: the stage
//     memory is zeroed at start, so such rows hold finite data with zero probability;
//   * warp 12 issues tcgen05.mma S = Q K^T into one of two TMEM score buffers, warp 13
//     O += P V into the TMEM output accumulator (V read MN-major from the same panels, P
//     the A operand from one of two TMEM P buffers);
//   * warps 0-7 turn S into P, two warps per TMEM lane quarter (one thread per row, each
//     warp of the pair half of the row's columns; the row max is exchanged through
//     shared memory): scale (folded into the exponent's FFMA when there is no soft cap),
//     soft cap, mask (only on blocks that cross a row's causal or window limit), online
//     softmax in the log2 domain with lazy rescaling (the running max only moves when it
//     grows by more than 2^8, and then O is rescaled in TMEM), P written as bf16 pairs into
//     the block's P buffer (shared memory holds only Q and the K/V rings); at the end they
//     read O, divide by l, store bf16 rows.
// Barriers: k_full/k_empty and v_full/v_empty (producers <-> MMA; separate K and V rings
// of NSK / NSV stages, so a K slot frees as soon as its QK is done); per score buffer s_full
// (QK -> softmax) and s_free (the softmax has loaded the scores: the next QK into that buffer
// may start while the softmax is still computing); per P buffer p_full (softmax -> PV) and
// p_empty (PV has read P); q_full, o_full; q_empty (the item's QKs are done and its softmax
// warps have started it: Q may be refilled) and o_empty (the epilogue has read O: the next
// item's first PV may overwrite it); item_full/item_empty, a two-slot ring through which the
// first producer thread hands items to every warp, so each role runs its own item loop and
// the producers and QK issuer start item n+1 during item n's epilogue.  Blocks are 128 keys
// (64 for D = 256).
// Every wait is bounded (common.cuh); on a timeout the CTA records an error and stops.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "profile.h"

namespace rpa {

template <int D, bool RAW = false>
struct PreTc {
    static constexpr int BK = D >= 256 ? 64 : 128;       // keys per block
    static constexpr int DP = D / 64;                    // 64-wide panels of the head dim
    // Q tile: DP panels of [128 rows x 128 B] in shared memory, or (RAW) in TMEM
    static constexpr int kQ = RAW ? 0 : DP * 128 * 128;
    static constexpr int kPanel = BK * 128;              // one K or V panel: [BK rows x 128 B]
    static constexpr int kStage = DP * kPanel;           // K (or V) of one block
    // RAW (one-byte caches staged by TMA): a block's raw K (or V) rows as D / 128 halves of
    // [BK rows x 128 B], 128-byte swizzled like the panels
    static constexpr int NH = D / 128;
    static constexpr int kRawHalf = BK * 128;
    static constexpr int kRaw = RAW ? NH * kRawHalf : 0;
    static constexpr int kReserve = 3072;                // barriers, scratch, row factors, item ring
    // stages of the K ring and of the V ring: as many as fit (P lives in TMEM), V's ring the
    // deeper one when the count is odd (a V slot is held from its load until PV, K's only until
    // QK); RAW: two f16 stages each and the raw rings (three stages each) in the rest
    static constexpr int kFitS = RAW ? 4 : (232448 - kQ - kReserve) / kStage;
    static constexpr int kTotS = kFitS > 8 ? 8 : kFitS;
    static constexpr int NSK = kTotS / 2;
    static constexpr int NSV = kTotS - NSK;
    static constexpr int NR = RAW ? (232448 - kReserve - kTotS * kStage) / (2 * (kRaw > 0 ? kRaw : 1)) : 0;
    static constexpr int kOffK = kQ;
    static constexpr int kOffV = kOffK + NSK * kStage;
    static constexpr int kOffRawK = kOffV + NSV * kStage;
    static constexpr int kOffRawV = kOffRawK + NR * kRaw;
    static constexpr int kOffBar = kOffRawV + NR * kRaw;
    // rings (+ raw rings), S/P barriers, q_full, o_full, fin, q_empty, o_empty, item ring full/empty [2] each
    static constexpr int kNumBars = 2 * (NSK + NSV) + 4 * NR + 4 * 2 + 3 + 2 + 4 + (RAW ? 1 : 0);
    // RAW: the item's Q tile (DP panels of [128 rows x 128 B]) is staged by TMA in the free K
    // slot (kQinK panels) and V slot (the rest) of the item's first block
    static constexpr int kQinK = kStage / 16384;
    static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr int kOffRed = (kOffTmemSlot + 16 + 127) / 128 * 128;  // [2 parities][2 halves][128 rows] float
    static constexpr int kOffQmul = kOffRed + 2 * 2 * 128 * 4;           // [128] float: Q row factors (f16 path)
    static constexpr int kOffItem = kOffQmul + 128 * 4;                  // [2] WorkItem ring (16-byte aligned) + abort flag
    static constexpr int kSmem = kOffItem + 2 * 32 + 16 + 32;  // + each softmax warp's kv_len
    static_assert(kOffBar % 8 == 0 && kOffRed % 16 == 0 && kOffItem % 16 == 0, "shared-memory alignment");
    static_assert(NSK >= 2 && NSV >= 2 && kOffK % 1024 == 0 && kOffV % 1024 == 0, "stages / swizzle-atom alignment");
    static_assert(!RAW || (NR >= 2 && kOffRawK % 1024 == 0 && kOffRawV % 1024 == 0 && (D == 128 || D == 256)),
                  "raw rings");
    // TMEM: kSB score buffers of BK columns, two P buffers of BK/2 columns (bf16 pairs), O and
    // (RAW) Q (D/2 columns of element pairs).  S and P live apart, so QK of block j+kSB may
    // overwrite S as soon as the softmax has loaded block j's scores, while PV of block j still
    // reads P(j) from its own buffer.  RAW keeps one score buffer (the softmax loads a block's
    // scores at once, so the next QK waits only for that) to make room for Q.
    static constexpr int kSB = RAW ? 1 : 2;
    static constexpr int kPB = 2;
    static constexpr int kColP = kSB * BK;
    static constexpr int kColO = kColP + kPB * (BK / 2);
    static constexpr int kColQ = kColO + D;
    static constexpr int kTmemCols = (RAW ? kColQ + D / 2 : kColO + D) <= 256 ? 256 : 512;
    static constexpr int kSoftWarps = 8;                 // two per TMEM lane quarter (column halves)
    static constexpr int kHalf = BK / 2;                 // score columns per softmax warp
    static_assert((RAW ? kColQ + D / 2 : kColO + D) <= kTmemCols, "TMEM budget");
    static_assert(kSmem <= 232448, "shared memory budget");
};

// Raw 8-element chunk of a K/V row: 8 bytes of e4m3 or 16 bytes of bf16.
template <bool FP8>
struct KvRaw {
    using type = uint4;
    __device__ static uint4 zero() { return make_uint4(0, 0, 0, 0); }
};
template <>
struct KvRaw<true> {
    using type = uint2;
    __device__ static uint2 zero() { return make_uint2(0, 0); }
};
template <bool FP8>
__device__ __forceinline__ typename KvRaw<FP8>::type kv_load_raw(const uint8_t* row, int c) {
    if constexpr (FP8)
        return __ldg(reinterpret_cast<const uint2*>(row + c * 8));
    else
        return __ldg(reinterpret_cast<const uint4*>(row + c * 16));
}
// Raw chunk -> 16 bytes of bf16: e4m3 or int8 (I8) (or scaled bf16) values become
// bf16(float(x) * scale).
template <bool FP8, bool SCALE, bool I8 = false>
__device__ __forceinline__ uint4 kv_convert(typename KvRaw<FP8>::type raw, float sc) {
    uint32_t w[4];
    if constexpr (FP8 && I8) {
        const int8_t* b = reinterpret_cast<const int8_t*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = pack_bf16((float)b[2 * e] * sc, (float)b[2 * e + 1] * sc);
        return make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (FP8) {
        const uint16_t* h = reinterpret_cast<const uint16_t*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = e4m3x2_to_float2(h[e]);
            w[e] = pack_bf16(f.x * sc, f.y * sc);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        if (!SCALE) return raw;
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            w[e] = pack_bf16(f.x * sc, f.y * sc);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// 8 int4 elements (4 bytes; element 2i in the low nibble of byte i) -> 16 bytes of bf16 of
// bf16(float(x) * scale).
__device__ __forceinline__ uint4 kv_convert_i4(uint32_t v, float sc) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int lo = (int)(v << (28 - 8 * e)) >> 28;  // nibble 2e, sign-extended
        const int hi = (int)(v << (24 - 8 * e)) >> 28;  // nibble 2e + 1
        w[e] = pack_bf16((float)lo * sc, (float)hi * sc);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Raw chunk of 8 one-byte elements -> 8 f16, exact and unscaled (the f16 path).
template <bool I8>
__device__ __forceinline__ uint4 kv_convert_f16(uint2 raw) {
    const uint16_t* h = reinterpret_cast<const uint16_t*>(&raw);
    if constexpr (I8)
        return make_uint4(s8x2_to_f16x2(h[0]), s8x2_to_f16x2(h[1]), s8x2_to_f16x2(h[2]), s8x2_to_f16x2(h[3]));
    else
        return make_uint4(e4m3x2_to_f16x2(h[0]), e4m3x2_to_f16x2(h[1]), e4m3x2_to_f16x2(h[2]), e4m3x2_to_f16x2(h[3]));
}

// softmax, producers (2 for K, 2 for V), QK and PV issuers, and (RAW) the raw-row TMA warp
template <bool RAW>
constexpr int prefill_warps() { return 8 + 4 + 2 + (RAW ? 1 : 0); }

// 16 raw one-byte values (dims 16c .. 16c+15 of a row) -> two 16-byte chunks of f16 (exact,
// unscaled: the f16 path) or bf16(float(x) * scale) values.
template <bool F16, bool I8>
__device__ __forceinline__ void raw16_convert(uint4 r, float sc, uint4& lo, uint4& hi) {
    const uint2 a = make_uint2(r.x, r.y), b = make_uint2(r.z, r.w);
    if constexpr (F16) {
        lo = kv_convert_f16<I8>(a);
        hi = kv_convert_f16<I8>(b);
    } else {
        lo = kv_convert<true, false, I8>(a, sc);
        hi = kv_convert<true, false, I8>(b, sc);
    }
}

// F16 (one-byte caches whose k_scale and v_scale are powers of two): K and V go to the tensor
// cores as exact f16 values (one convert per pair), each Q row is brought into f16 range by a
// power of two found from its largest element (its bf16 values stay exact), P is f16, and the
// row factor with k_scale goes onto the scores, v_scale onto O.
// RAW (one-byte caches, page boxes of >= 8 rows): warp 14 lands each block's raw K and V rows
// by TMA (128-byte swizzled halves of [BK x 128 B]) in rings of NR stages, warps 8-11 convert
// them shared memory to shared memory into the f16/bf16 panels and put Q into TMEM (the QK
// MMAs read A from there), and S has one TMEM buffer.
// I4 (int4 caches, two elements a byte): the register path, each 8-element chunk 4 bytes.
// MILD: a mask value that leaves masked keys weight (rare: its own, register-path instantiations,
// so that the common ones carry none of its code)
template <int D, bool FP8, bool SCALE, bool TMA, bool I8 = false, bool F16 = false, bool RAW = false, bool I4 = false,
          bool MILD = false>
__global__ void __launch_bounds__(prefill_warps<RAW>() * 32, 1)
    rpa_prefill_tc_kernel(RpaArgs a, const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_q,
                          int box_rows, int q_tma, int tail) {
    using T = PreTc<D, RAW>;
    constexpr int BK = T::BK;
    // first launch (tail == 0): started early behind the plan kernel, it waits for it, then lets
    // the decode grid behind start; only the plan's share of its CTAs works. Either launch
    // leaves at once when the list is empty.
    if (!tail) {
        pdl_wait();
        pdl_launch_dependents();
    }
    extern __shared__ __align__(1024) uint8_t smem[];
    {
        // one decision for the whole CTA: the queue counter moves while other CTAs take items,
        // so threads reading it on their own could disagree, and a CTA whose item-fetching
        // thread left would leave its other warps waiting for an item
        volatile int& s_exit = *reinterpret_cast<volatile int*>(smem + T::kOffItem + 68);
        if (threadIdx.x == 0) {
            const WsHeader* h = a.hdr;
            s_exit = (!tail && (int)blockIdx.x >= h->prefill_ctas) ||
                     *(volatile const int*)&h->next_item[1] >= h->num_items[1];
        }
        __syncthreads();
        if (s_exit) return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::kOffBar);
    constexpr int NSK = T::NSK, NSV = T::NSV;
    uint64_t* k_full = bars;                       // [NSK] K block landed
    uint64_t* k_empty = bars + NSK;                // [NSK] QK of that block done
    uint64_t* v_full = bars + 2 * NSK;             // [NSV] V block landed
    uint64_t* v_empty = bars + 2 * NSK + NSV;      // [NSV] PV of that block done
    uint64_t* const bars_s = bars + 2 * (NSK + NSV);
    constexpr int SB = T::kSB, PB = T::kPB, NR = T::NR;
    constexpr uint32_t NRd = NR > 0 ? NR : 1;  // ring divisor (the raw rings exist only with RAW)
    static_assert(T::kPB == 2 && T::kSB <= 2, "barrier layout");
    uint64_t* s_full = bars_s;            // [SB] S buffer written by QK
    uint64_t* s_free = bars_s + 2;        // [SB] the softmax has loaded that buffer's scores
    uint64_t* p_full = bars_s + 4;        // [PB] P buffer written (and O rescaled)
    uint64_t* p_empty = bars_s + 6;       // [PB] PV of that buffer's P done (buffer free again)
    uint64_t* q_full = bars_s + 8;
    uint64_t* o_full = q_full + 1;
    uint64_t* fin = q_full + 2;
    uint64_t* q_empty = q_full + 3;     // the item's QKs are done and the softmax warps have started it
    uint64_t* o_empty = q_full + 4;     // the epilogue has read O out of TMEM
    uint64_t* item_full = q_full + 5;   // [2] ring slot written
    uint64_t* item_empty = q_full + 7;  // [2] ring slot read by every warp
    uint64_t* rawk_full = q_full + 9;             // [NR] (RAW) a block's raw K rows landed
    uint64_t* rawk_empty = rawk_full + NR;        // [NR] converted (slot free)
    uint64_t* rawv_full = rawk_full + 2 * NR;     // [NR] raw V rows landed
    uint64_t* rawv_empty = rawk_full + 3 * NR;    // [NR] converted
    uint64_t* q_stage = rawk_full + 4 * NR;       // (RAW) the item's Q tile landed in its staging slots
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + T::kOffTmemSlot);
    float* red = reinterpret_cast<float*>(smem + T::kOffRed);
    // producer warps [8, 12): warps 8-9 stream K, 10-11 V; then the MMA warp
    // warp 12 issues the QK MMAs (and owns the TMEM allocation), warp 13 the PV MMAs: two issuing
    // threads, so neither stream waits behind the other's inputs (an MMA issue blocks while the
    // tensor pipe's short queue is full)
    constexpr int kProdW0 = 8, kProdW1 = 12, kMmaW = kProdW1, kPvW = kProdW1 + 1, kRawW = kProdW1 + 2;
    // (no static shared variables: with the 1024-byte aligned dynamic block they would
    // round up to 1 KB and push the kernel past the 227 KB limit)
    static_assert(!F16 || (FP8 && !TMA), "the f16 path takes one-byte caches through registers");
    static_assert(!RAW || (FP8 && !TMA && !SCALE && !I4), "the raw-staging path is for one-byte caches");
    static_assert(!I4 || (FP8 && !TMA && !RAW && !F16 && !I8), "int4 caches take the bf16 register path");
    float* qmul = reinterpret_cast<float*>(smem + T::kOffQmul);
    WorkItem* s_items = reinterpret_cast<WorkItem*>(smem + T::kOffItem);
    volatile int& s_abort = *reinterpret_cast<volatile int*>(smem + T::kOffItem + 64);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    WsHeader* hdr = a.hdr;
    uint32_t* err = &hdr->error_bits;
    const int Hkv = a.num_kv_heads, G = a.num_q_heads / Hkv, C = 2 * Hkv;
    constexpr int kEsz = FP8 ? 1 : 2;
    const uint8_t* kvp = static_cast<const uint8_t*>(a.kv_pages);

    // zero Q and the K/V stages once: rows no copy ever writes stay finite
    for (int i = tid * 16; i < T::kOffBar; i += blockDim.x * 16) *reinterpret_cast<uint4*>(smem + i) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid == 0) {
        for (int i = 0; i < NSK; ++i) {
            mbar_init(&k_full[i], 64);  // the two warps streaming K
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < NSV; ++i) {
            mbar_init(&v_full[i], 64);  // the two warps streaming V
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < SB; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], T::kSoftWarps * 32);
        }
        for (int i = 0; i < PB; ++i) {
            mbar_init(&p_full[i], T::kSoftWarps * 32);
            mbar_init(&p_empty[i], 1);
        }
        for (int i = 0; i < NR; ++i) {
            mbar_init(&rawk_full[i], 1);   // the TMA warp's arrive + the copies' bytes
            mbar_init(&rawk_empty[i], 2);  // one arrival per converting warp
            mbar_init(&rawv_full[i], 1);
            mbar_init(&rawv_empty[i], 2);
        }
        if (RAW) mbar_init(q_stage, 1);
        // Q by TMA: the issuing thread alone; through registers: every producer thread
        mbar_init(q_full, (TMA && q_tma) ? 1 : (kProdW1 - kProdW0) * 32);
        mbar_init(o_full, 1);
        mbar_init(fin, 2);                         // both issuing threads
        mbar_init(q_empty, 1 + T::kSoftWarps);     // QK issuer's commit + each softmax warp
        mbar_init(o_empty, T::kSoftWarps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&item_full[i], 1);
            mbar_init(&item_empty[i], prefill_warps<RAW>());
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaW) tmem_alloc(tmem_slot, T::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Items reach the warps through a two-slot ring. The first producer thread (its role runs
    // furthest ahead) takes item n when it gets to it; every warp reads the slot and frees it.
    // Each role then runs its own item loop: the producers and the QK issuer start item n + 1
    // while the softmax warps finish item n (its last blocks and its epilogue). The Q buffer
    // is refilled once item n's QKs are done and the softmax warps have started it (q_empty),
    // and PV overwrites O once the epilogue has read it (o_empty); the K/V, S and P rings are
    // indexed by the CTA's running block count and need nothing at item boundaries.
    uint32_t jb = 0;     // key blocks this CTA has processed (ring positions)
    uint32_t items = 0;  // items this CTA has processed (ring slots, q / o phases)
    while (true) {
        const uint32_t islot = items & 1, iring = (items >> 1) & 1;
        // the fetching thread: the first producer thread, or (RAW) the raw-row TMA warp's
        if (tid == (RAW ? kRawW : kProdW0) * 32) {
            WorkItem nw;
            nw.seq = -1;
            if (!mbar_wait(&item_empty[islot], iring ^ 1, err)) s_abort = 1;
            // beside decode, take no new item once most decode CTAs with a share are out of
            // work (decode is ending): what is left goes to the launch after decode, on every SM
            const bool stop = s_abort || (!tail && a.overlap && hdr->dec_ctas > 0 &&
                                          *(volatile const int*)&hdr->next_item[0] >=
                                              max(1, hdr->dec_ctas * kPrefillStopPercent / 100));
            if (!stop) {
                const int it = atomicAdd(&hdr->next_item[1], 1);
                if (it < hdr->num_items[1]) nw = a.pre_items[it];
            }
            s_items[islot] = nw;
            mbar_arrive(&item_full[islot]);
        }
        WorkItem w;
        w.seq = -1;
        if (mbar_wait(&item_full[islot], iring, err)) w = s_items[islot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_empty[islot]);
        if (w.seq < 0 || s_abort) break;
        const int s = w.seq;
        const int q_start = a.cu_q_lens[s];
        const int q_len = a.cu_q_lens[s + 1] - q_start;
        const int kv_len = a.kv_lens[s];
        const int n_rows = q_len * G;
        const int kvh = w.head;
        const int R0 = w.row_begin;
        const int R1 = min(n_rows, R0 + 128) - 1;
        const int qmin = kv_len - q_len + R0 / G, qmax = kv_len - q_len + R1 / G;
        // keys the tile's rows see: the causal (windowed) range, or every key with a mild mask
        int kb = a.sliding_window > 0 && !MILD ? max(0, qmin - a.sliding_window + 1) : 0;
        kb = kb / BK * BK;
        const int ke = MILD ? kv_len : qmax + 1;
        const int nb = cdiv(ke - kb, BK);
        const uint32_t iph = items & 1;

        if (RAW && warp >= kProdW0 && warp < kProdW1) {
            // ---------------- converters (RAW) ----------------
            // Q: this warp's 32 rows (its TMEM lane quarter), once the previous item's QKs have
            // read Q and its softmax warps have started it (q_empty). With q_tma the tile has been
            // staged by TMA in the item's first K and V slots (128-byte swizzled panels) and is
            // read from there; otherwise each thread loads its row from global memory.
            {
                const int r = (warp - kProdW0) * 32 + lane;
                const uint32_t lane_off = (uint32_t)((warp - kProdW0) * 32) << 16;
                if (!mbar_wait(q_empty, iph ^ 1, err)) s_abort = 1;
                if (q_tma && !mbar_wait(q_stage, iph, err)) s_abort = 1;
                tc_fence_after();
                const int R = R0 + r;
                const bool rv = R < n_rows;
                const uint8_t* src = reinterpret_cast<const uint8_t*>(
                    a.q + ((size_t)(q_start + (rv ? R / G : 0)) * a.num_q_heads + kvh * G + (rv ? R % G : 0)) * D);
                // this row in the staged tile: panel p at base(p) + r * 128, 16-byte chunk cc of it
                // at position cc ^ (r % 8)
                const uint32_t kst = smem_u32(smem + T::kOffK + (jb % NSK) * T::kStage) + r * 128;
                const uint32_t vst = smem_u32(smem + T::kOffV + (jb % NSV) * T::kStage) + r * 128;
                // 16-byte chunk c (elements 8c .. 8c+7) of this row; rows past the item are zeros
                auto qchunk = [&](int c) -> uint4 {
                    if (!rv) return make_uint4(0, 0, 0, 0);
                    if (!q_tma) return __ldg(reinterpret_cast<const uint4*>(src + c * 16));
                    const int p = c >> 3;
                    return lds128((p < T::kQinK ? kst + p * 16384 : vst + (p - T::kQinK) * 16384) +
                                  (((c & 7) ^ (r & 7)) << 4));
                };
                float qs = 1.f;
                if (F16) {
                    // the row's largest |q| < 2^ex; 2^-k brings it into [2^14, 2^15) (f16 range);
                    // eight chunks in flight, four independent maxima
                    float m4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
                    for (int c0 = 0; c0 < D / 8; c0 += 8) {
                        uint4 v8[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) v8[u] = qchunk(c0 + u);
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v8[u]);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = __bfloat1622float2(h2[e]);
                                m4[e] = fmax3(m4[e], fabsf(f.x), fabsf(f.y));
                            }
                        }
                    }
                    const float mabs = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                    int ex = 0;
                    frexpf(mabs, &ex);
                    const int k = max(-30, min(100, ex - 15));
                    qs = ldexpf(1.f, -k);
                    qmul[r] = ldexpf(1.f, k);
                }
                // 32 elements (16 TMEM columns of element pairs) per store, two stores per batch
#pragma unroll 1
                for (int g = 0; g < D / 32; g += 2) {
                    uint4 v8[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) v8[u] = qchunk(g * 4 + u);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t v[16];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint4 u = v8[h * 4 + c];
                            if (F16) {
                                const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
                                uint32_t w4[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float2 f = __bfloat1622float2(h2[e]);
                                    w4[e] = pack_f16(f.x * qs, f.y * qs);
                                }
                                u = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                            }
                            v[4 * c] = u.x;
                            v[4 * c + 1] = u.y;
                            v[4 * c + 2] = u.z;
                            v[4 * c + 3] = u.w;
                        }
                        tmem_st16_nowait(tmem + lane_off + T::kColQ + (g + h) * 16, v);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                // every converter thread has read the staged tile before block jb's K and V are
                // converted into the same slots
                if (q_tma) asm volatile("bar.sync 5, 128;" ::: "memory");
                mbar_arrive(q_full);
            }
            // K (warps 8-9) or V (warps 10-11) of every block: raw rows -> panels. The part's 64
            // threads work in phases of 8 lanes, each phase one 16-byte raw chunk of 8 consecutive
            // rows (distinct swizzled positions for the raw reads and the panel writes alike).
            const int part = (warp - kProdW0) >> 1;
            const int ph = (((warp - kProdW0) & 1) << 2) | (lane >> 3), l8 = lane & 7;
            uint64_t* fbar = part ? v_full : k_full;
            uint64_t* ebar = part ? v_empty : k_empty;
            uint64_t* rfull = part ? rawv_full : rawk_full;
            uint64_t* rempty = part ? rawv_empty : rawk_empty;
            const float sc = part ? a.v_scale_or_one : a.k_scale_or_one;
            constexpr int kChunks = D / 16;                    // 16-byte raw chunks per row
            constexpr int kIters = (BK / 8) * kChunks / 8;     // (row group, chunk) pairs per phase
            constexpr int kCB = kChunks / 8 > 0 ? kChunks / 8 : 1;  // raw halves (8-chunk groups) per row
            // iteration `it` of a phase covers chunk c = (it % kCB) * 8 + ph of rows
            // (it / kCB) * 8 + l8: its raw half is it % kCB, its panels (it % kCB) * 2 + ph / 4,
            // so every address is a per-thread base plus a compile-time offset
            const uint32_t raw_base = l8 * 128 + ((ph ^ l8) << 4);
            const uint32_t dst_base = (ph >> 2) * T::kPanel + l8 * 128;
            const uint32_t pos0 = ((2 * (ph & 3)) ^ l8) << 4, pos1 = ((2 * (ph & 3) + 1) ^ l8) << 4;
            for (int j = 0; j < nb; ++j) {
                const uint32_t q = jb + j, slot = part ? q % NSV : q % NSK, par = (part ? q / NSV : q / NSK) & 1;
                const uint32_t rs = q % NRd, rp = (q / NRd) & 1;
                if (!mbar_wait(&rfull[rs], rp, err) || !mbar_wait(&ebar[slot], par ^ 1, err)) {
                    s_abort = 1;
                    break;
                }
                const uint8_t* raw = smem + (part ? T::kOffRawV : T::kOffRawK) + rs * T::kRaw + raw_base;
                uint8_t* stage = smem + (part ? T::kOffV : T::kOffK) + slot * T::kStage + dst_base;
                const int nvalid = ke - (kb + j * BK);  // rows of this block inside the key range (>= 1)
                const bool full = nvalid >= BK;
                // a batch's raw chunks are all loaded before any is converted and stored (the
                // compiler cannot tell the raw ring from the panels, so it would otherwise keep
                // every load behind the previous store)
                constexpr int kBatch = 8;
                static_assert(kIters % kBatch == 0, "converter batches");
#pragma unroll
                for (int it0 = 0; it0 < kIters; it0 += kBatch) {
                    uint4 r16[kBatch];
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) {
                        const int it = it0 + u;
                        const int row = (it / kCB) * 8 + l8;
                        r16[u] = (full || row < nvalid)
                                     ? *reinterpret_cast<const uint4*>(raw + (it % kCB) * T::kRawHalf + (it / kCB) * 1024)
                                     : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) {
                        const int it = it0 + u;
                        uint4 lo, hi;
                        raw16_convert<F16, I8>(r16[u], sc, lo, hi);  // zero bytes convert to zeros
                        uint8_t* drow = stage + (it % kCB) * 2 * T::kPanel + (it / kCB) * 1024;
                        *reinterpret_cast<uint4*>(drow + pos0) = lo;
                        *reinterpret_cast<uint4*>(drow + pos1) = hi;
                    }
                }
                fence_proxy_async_smem();  // panels written by threads, read by the tensor core
                mbar_arrive(&fbar[slot]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&rempty[rs]);
            }
        } else if (RAW && warp == kRawW) {
            // ---------------- raw-row TMA (RAW) ----------------
            // lane l owns box l (box_rows keys of one page) of every block, looked up one block
            // ahead; a box with any row inside the key range is copied whole (its rows past the
            // range are slots of the same page, converted to zeros), K then V of each block
            const int nbox = BK / box_rows;
            const int lbr = __ffs(box_rows) - 1, lps = __ffs(a.page_size) - 1, pmask_ps = a.page_size - 1;
            const uint32_t box_bytes = (uint32_t)box_rows * 128 * T::NH;
            const int* tbl = a.page_indices + (size_t)s * a.pages_per_seq;
            auto page_of = [&](int j) -> int {
                const int key = kb + j * BK + lane * box_rows;
                return (lane < nbox && j < nb && key < ke) ? __ldg(tbl + (key >> lps)) : 0;
            };
            int page_next = page_of(0);
            bool go = true;
            for (int j = 0; go && j < nb; ++j) {
                const uint32_t q = jb + j, rs = q % NRd, rp = (q / NRd) & 1;
                int page = page_next;
                page_next = page_of(j + 1);
                const int kbj = kb + j * BK;
                const int nvb = min(nbox, (ke - kbj + box_rows - 1) >> lbr);  // boxes with a row in range
                if (lane < nvb && (unsigned)page >= (unsigned)a.total_num_pages) {
                    set_error(err, RPA_DEV_ERR_PAGE);
                    page = 0;  // an in-bounds page keeps the barrier's byte count; the error is recorded
                }
                const int z0 = (page << lps) + ((kbj + lane * box_rows) & pmask_ps);
#pragma unroll 1
                for (int part = 0; part < 2; ++part) {
                    uint64_t* rfull = part ? rawv_full : rawk_full;
                    uint64_t* rempty = part ? rawv_empty : rawk_empty;
                    int g = 1;
                    if (lane == 0) {
                        g = mbar_wait(&rempty[rs], rp ^ 1, err);
                        if (g)
                            mbar_arrive_expect_tx(&rfull[rs], (uint32_t)nvb * box_bytes);
                        else
                            s_abort = 1;
                    }
                    if (!__shfl_sync(0xffffffffu, g, 0)) {
                        go = false;
                        break;
                    }
                    uint8_t* dst = smem + (part ? T::kOffRawV : T::kOffRawK) + rs * T::kRaw + lane * box_rows * 128;
                    if (lane < nvb) {
#pragma unroll
                        for (int h = 0; h < T::NH; ++h)
                            tma_load_3d(smem_u32(dst + h * T::kRawHalf), &tm_kv, 128 * h, 2 * kvh + part, z0, &rfull[rs]);
                    }
                }
                if (go && j == 0 && q_tma) {
                    // the item's Q tile into the K and V slots of its first block once those are
                    // free (QK and PV of block jb - 2 done); the converters read it from there
                    int g = 1;
                    if (lane == 0) {
                        const uint32_t ks = jb % NSK, kp = (jb / NSK) & 1, vs = jb % NSV, vp = (jb / NSV) & 1;
                        g = mbar_wait(&k_empty[ks], kp ^ 1, err) &&
                            (T::DP <= T::kQinK || mbar_wait(&v_empty[vs], vp ^ 1, err));
                        if (g) {
                            mbar_arrive_expect_tx(q_stage, (uint32_t)D * 256);
#pragma unroll
                            for (int p = 0; p < T::DP; ++p) {
                                uint8_t* qd = p < T::kQinK ? smem + T::kOffK + ks * T::kStage + p * 16384
                                                           : smem + T::kOffV + vs * T::kStage + (p - T::kQinK) * 16384;
                                tma_load_3d(smem_u32(qd), &tm_q, 64 * p, kvh * G, q_start + R0 / G, q_stage);
                            }
                        } else {
                            s_abort = 1;
                        }
                    }
                    if (!__shfl_sync(0xffffffffu, g, 0)) go = false;
                }
            }
        } else if (warp >= kProdW0 && warp < kProdW1) {
            // ---------------- producers ----------------
            const int pt = tid - kProdW0 * 32;
            if (TMA && q_tma) {
                // the 128 rows are 128/G consecutive tokens x the G heads of this KV head
                // issued from a V-streaming thread: its loads have the most slack, while the K
                // streamers (and the item fetch) run on into this item ahead of its Q
                if (pt == 64) {
                    if (mbar_wait(q_empty, iph ^ 1, err)) {  // the previous item's QKs read Q
                        mbar_arrive_expect_tx(q_full, D * 256);
#pragma unroll
                        for (int p = 0; p < T::DP; ++p)
                            tma_load_3d(smem_u32(smem + p * 16384), &tm_q, 64 * p, kvh * G, q_start + R0 / G, q_full);
                    } else {
                        s_abort = 1;
                    }
                }
            } else {
                // the previous item's QKs have read Q and its softmax warps its row factors
                if (!mbar_wait(q_empty, iph ^ 1, err)) s_abort = 1;
                const int nprod = (kProdW1 - kProdW0) * 32;
                for (int r = pt; r < 128; r += nprod) {
                    const int R = R0 + r;
                    const bool rv = R < n_rows;
                    // rows are a.head_dim wide (below D when the kernel runs at the next multiple
                    // of 128: the dims past it are zeros)
                    const int dq8 = a.head_dim / 8;
                    const uint8_t* src = reinterpret_cast<const uint8_t*>(
                        a.q + ((size_t)(q_start + (rv ? R / G : 0)) * a.num_q_heads + kvh * G + (rv ? R % G : 0)) * a.head_dim);
                    float qs = 1.f;
                    if (F16) {
                        // the row's largest |q| < 2^ex; 2^-k brings it into [2^14, 2^15) (f16 range)
                        float mabs = 0.f;
#pragma unroll 8
                        for (int c = 0; c < D / 8; ++c) {
                            const uint4 v = rv ? __ldg(reinterpret_cast<const uint4*>(src + c * 16)) : make_uint4(0, 0, 0, 0);
                            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = __bfloat1622float2(h2[e]);
                                mabs = fmax3(mabs, fabsf(f.x), fabsf(f.y));
                            }
                        }
                        int ex = 0;
                        frexpf(mabs, &ex);
                        const int k = max(-30, min(100, ex - 15));
                        qs = ldexpf(1.f, -k);
                        qmul[r] = ldexpf(1.f, k);
                    }
#pragma unroll 8
                    for (int c = 0; c < D / 8; ++c) {
                        uint4 v = rv && c < dq8 ? __ldg(reinterpret_cast<const uint4*>(src + c * 16)) : make_uint4(0, 0, 0, 0);
                        if (F16) {
                            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v);
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = __bfloat1622float2(h2[e]);
                                w[e] = pack_f16(f.x * qs, f.y * qs);
                            }
                            v = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                        *reinterpret_cast<uint4*>(smem + (c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(q_full);
            }
            if (TMA) {
                // warps 8-9 stream K, 10-11 V, each warp half of the 64-wide panels (a TMA
                // issue costs ~65 cycles and is serial within a warp, so small page boxes need
                // several issuing warps).  Lane l owns box l (box_rows keys of one page,
                // box_rows >= 8) of every block; its page is looked up one block ahead.  Full
                // boxes are one TMA per panel; the rows of a partial last box are copied by the
                // warp through registers.  Each full barrier takes TMA bytes + 64 arrivals.
                const int part = (warp - kProdW0) >> 1, pw = (warp - kProdW0) & 1;
                constexpr int kPW = (T::DP + 1) / 2;  // panels per warp
                const int p0 = pw * kPW, p1 = min(T::DP, p0 + kPW);
                uint64_t* fbar = part ? v_full : k_full;
                uint64_t* ebar = part ? v_empty : k_empty;
                // box_rows and page_size are powers of two (the host's condition for this path) and
                // a box never crosses a page, so the per-block bookkeeping is shifts and one compare
                // per lane: the number of full boxes is the same on every lane (no shuffles)
                const int nbox = BK / box_rows;
                const int lbr = __ffs(box_rows) - 1, lps = __ffs(a.page_size) - 1, pmask_ps = a.page_size - 1;
                const uint32_t box_bytes = (uint32_t)box_rows * (p1 - p0) * 128;
                const int* tbl = a.page_indices + (size_t)s * a.pages_per_seq;
                auto page_of = [&](int j) -> int {
                    const int key = kb + j * BK + lane * box_rows;
                    return (lane < nbox && j < nb && key < ke) ? __ldg(tbl + (key >> lps)) : 0;
                };
                int page_next = page_of(0);
                for (int j = 0; j < nb; ++j) {
                    const uint32_t q = jb + j, slot = part ? q % NSV : q % NSK, par = (part ? q / NSV : q / NSK) & 1;
                    int page = page_next;
                    page_next = page_of(j + 1);
                    const int kbj = kb + j * BK, avail = ke - kbj;  // avail >= 1
                    const int nfull = min(nbox, avail >> lbr);
                    const int prow = nfull < nbox ? avail - (nfull << lbr) : 0;  // rows of a partial box
                    if (lane <= nfull && lane < nbox && (unsigned)page >= (unsigned)a.total_num_pages) {
                        if (part == 0) set_error(err, RPA_DEV_ERR_PAGE);
                        page = 0;  // an in-bounds page keeps the barrier's byte count; the error is recorded
                    }
                    const int kbx = kbj + lane * box_rows;
                    const int z0 = (page << lps) + (kbx & pmask_ps);
                    int g = 1;
                    if (lane == 0) {
                        g = mbar_wait(&ebar[slot], par ^ 1, err);
                        if (g)
                            mbar_expect_tx(&fbar[slot], (uint32_t)nfull * box_bytes);
                        else
                            s_abort = 1;
                    }
                    if (!__shfl_sync(0xffffffffu, g, 0)) break;
                    uint8_t* stage = smem + (part ? T::kOffV : T::kOffK) + slot * T::kStage;
                    if (lane < nfull) {
                        for (int p = p0; p < p1; ++p)
                            tma_load_3d(smem_u32(stage + p * T::kPanel + lane * box_rows * 128), &tm_kv, 64 * p,
                                        2 * kvh + part, z0, &fbar[slot]);
                    }
                    const bool wrote = prow > 0 && p1 > p0;
                    if (wrote) {
                        // the partial last box: its rows by cp.async, all in flight at once (the
                        // whole warp; dims past a.head_dim, when the kernel runs at the next
                        // multiple of 128, are filled with zeros)
                        const int pz0 = __shfl_sync(0xffffffffu, z0, nfull);
                        constexpr int kCh = kPW * 8;  // this warp's 16-byte chunks of a row
                        for (int i = lane; i < prow * kCh; i += 32) {
                            const int tr = i / kCh, c = p0 * 8 + i % kCh;
                            if (c >= D / 8) continue;
                            const int kk = nfull * box_rows + tr;
                            const bool in = c * 8 < a.head_dim;
                            const uint8_t* src = kvp + ((size_t)(pz0 + tr) * C + 2 * kvh + part) * (size_t)(a.head_dim * 2) +
                                                 (in ? c * 16 : 0);
                            cp_async16(smem_u32(stage + (c >> 3) * T::kPanel + kk * 128 + (((c & 7) ^ (kk & 7)) << 4)), src, in);
                        }
                        cp_async_commit();
                        cp_async_wait<0>();
                        fence_proxy_async_smem();  // thread-copied rows, read by the tensor core
                    }
                    mbar_arrive(&fbar[slot]);
                }
            } else {
                // register path (fp8 / scaled caches): warps 8-9 stream K, warps 10-11 V.  A thread
                // owns BK / 64 key rows of every block; the next block's pages are looked up
                // ahead, and all of a row's loads are issued before it is converted and stored.
                constexpr int kRowChunks = D / 8;  // 8-element chunks per K (or V) row
                constexpr int kRpt = BK / 64;      // rows per thread
                const int part = (warp - kProdW0) >> 1;
                const int gt = pt & 63;
                uint64_t* fbar = part ? v_full : k_full;
                uint64_t* ebar = part ? v_empty : k_empty;
                const float sc = part ? a.v_scale_or_one : a.k_scale_or_one;
                auto page_of = [&](int j, int i) -> int {
                    const int key = kb + j * BK + gt + 64 * i;
                    return (j < nb && key < ke) ? __ldg(a.page_indices + (size_t)s * a.pages_per_seq + key / a.page_size)
                                                : -1;
                };
                int page_next[kRpt];
#pragma unroll
                for (int i = 0; i < kRpt; ++i) page_next[i] = page_of(0, i);
                for (int j = 0; j < nb; ++j) {
                    const uint32_t q = jb + j, slot = part ? q % NSV : q % NSK, par = (part ? q / NSV : q / NSK) & 1;
                    int page[kRpt];
#pragma unroll
                    for (int i = 0; i < kRpt; ++i) {
                        page[i] = page_next[i];
                        page_next[i] = page_of(j + 1, i);
                    }
                    if (!mbar_wait(&ebar[slot], par ^ 1, err)) {
                        s_abort = 1;
                        break;
                    }
                    uint8_t* stage = smem + (part ? T::kOffV : T::kOffK) + slot * T::kStage;
#pragma unroll 1
                    for (int i = 0; i < kRpt; ++i) {
                        const int kk = gt + 64 * i;
                        const int key = kb + j * BK + kk;
                        bool v = key < ke;
                        if (v && (unsigned)page[i] >= (unsigned)a.total_num_pages) {
                            if (part == 0) set_error(err, RPA_DEV_ERR_PAGE);
                            v = false;
                        }
                        const uint8_t* row =
                            v ? kvp + (((size_t)page[i] * a.page_size + key % a.page_size) * C + 2 * kvh + part) *
                                          (size_t)(I4 ? D / 2 : D * kEsz)
                              : nullptr;
                        if constexpr (I4) {
                            // 8 int4 elements (4 bytes) a chunk: a whole row's loads in flight
                            uint32_t raw4[kRowChunks];
#pragma unroll
                            for (int c = 0; c < kRowChunks; ++c) raw4[c] = v ? __ldg(reinterpret_cast<const uint32_t*>(row + c * 4)) : 0u;
#pragma unroll
                            for (int c = 0; c < kRowChunks; ++c)
                                *reinterpret_cast<uint4*>(stage + (c >> 3) * T::kPanel + kk * 128 + (((c & 7) ^ (kk & 7)) << 4)) =
                                    kv_convert_i4(raw4[c], sc);
                            continue;
                        }
                        // loads in flight per pass: a whole row for fp8 (8-byte chunks), 16 chunks for bf16
                        constexpr int kGroup = FP8 ? kRowChunks : (kRowChunks < 16 ? kRowChunks : 16);
#pragma unroll 1
                        for (int c0 = 0; c0 < kRowChunks; c0 += kGroup) {
                            // raw loads first (all in flight), then dequantise and store
                            typename KvRaw<FP8>::type raw[kGroup];
#pragma unroll
                            for (int c = 0; c < kGroup; ++c) raw[c] = v ? kv_load_raw<FP8>(row, c0 + c) : KvRaw<FP8>::zero();
#pragma unroll
                            for (int c = 0; c < kGroup; ++c) {
                                const int cc = c0 + c;
                                uint4 cv;
                                if constexpr (F16)
                                    cv = kv_convert_f16<I8>(raw[c]);
                                else
                                    cv = kv_convert<FP8, SCALE, I8>(raw[c], sc);
                                *reinterpret_cast<uint4*>(stage + (cc >> 3) * T::kPanel + kk * 128 + (((cc & 7) ^ (kk & 7)) << 4)) = cv;
                            }
                        }
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(&fbar[slot]);
                }
            }
        } else if (warp == kMmaW) {
            // ---------------- QK issuer ----------------
            if (lane == 0) {
                constexpr uint32_t idesc_qk = umma_idesc_16(128, BK, false, false, F16);
                // descriptors of the operand bases; a byte offset d within shared memory adds
                // d >> 4 to the start-address field (no carry: every address is below 256 KB)
                const uint64_t qdesc = umma_desc_sw128(smem_u32(smem), 16, 1024);
                const uint64_t kdesc = umma_desc_sw128(smem_u32(smem + T::kOffK), 16, 1024);
                bool ok = mbar_wait(q_full, iph, err);
                for (int j = 0; ok && j < nb; ++j) {
                    const uint32_t q = jb + j, sb = q % SB, sp = (q / SB) & 1, slot = q % NSK, par = (q / NSK) & 1;
                    // K landed, and the score buffer's previous scores (block q - SB) loaded by the softmax
                    ok = mbar_wait(&k_full[slot], par, err) && mbar_wait(&s_free[sb], sp ^ 1, err);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t kb0 = kdesc + (uint64_t)((slot * T::kStage) >> 4);
                    if constexpr (RAW) {
                        // Q from TMEM: one K=16 step spans 8 columns of element pairs
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks)
                            umma_bf16_ta(tmem + sb * BK, tmem + T::kColQ + ks * 8,
                                         kb0 + (((ks >> 2) * T::kPanel + (ks & 3) * 32) >> 4), idesc_qk, ks > 0 ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks)
                            umma_bf16(tmem + sb * BK, qdesc + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4),
                                      kb0 + (((ks >> 2) * T::kPanel + (ks & 3) * 32) >> 4), idesc_qk, ks > 0 ? 1u : 0u);
                    }
                    umma_commit(&s_full[sb]);
                    umma_commit(&k_empty[slot]);
                }
                umma_commit(q_empty);  // Q may be refilled once these QKs have completed
                if (!ok) s_abort = 1;
            }
        } else if (warp == kPvW) {
            // ---------------- PV issuer ----------------
            if (lane == 0) {
                constexpr uint32_t idesc_pv = umma_idesc_16(128, D, false, true, F16);
                const uint64_t vdesc = umma_desc_sw128(smem_u32(smem + T::kOffV), T::kPanel, 1024);
                // the first PV overwrites O: the previous item's epilogue has read it
                bool ok = mbar_wait(o_empty, iph ^ 1, err);
                for (int j = 0; ok && j < nb; ++j) {
                    const uint32_t q = jb + j, pb = q % PB, pp = (q / PB) & 1, slot = q % NSV, par = (q / NSV) & 1;
                    ok = mbar_wait(&p_full[pb], pp, err) && mbar_wait(&v_full[slot], par, err);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t vb0 = vdesc + (uint64_t)((slot * T::kStage) >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16_ta(tmem + T::kColO, tmem + T::kColP + pb * (BK / 2) + kk * 8, vb0 + ((kk * 16 * 128) >> 4),
                                     idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(&p_empty[pb]);
                    umma_commit(&v_empty[slot]);
                }
                umma_commit(o_full);
                if (!ok) s_abort = 1;
            }
        } else if (warp < T::kSoftWarps) {
            // ------- softmax / epilogue: row = TMEM lane, warps w and w+4 split its columns -------
            const int quarter = warp & 3, half = warp >> 2;
            const int r = quarter * 32 + lane;
            const int R = R0 + r;
            const bool rv = R < n_rows;
            const int qpos = rv ? kv_len - q_len + R / G : -1;
            const int wlo = a.sliding_window > 0 ? qpos - a.sliding_window + 1 : INT_MIN;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            // kv_len is needed again only by a mild mask: this warp's copy waits in shared memory
            // instead of a register held through the block loop
            volatile int* s_kvl = reinterpret_cast<volatile int*>(smem + T::kOffItem + 80) + warp;
            if constexpr (MILD) {
                if (lane == 0) *s_kvl = kv_len;
                __syncwarp();
            }
            // F16: the row's power of two (set by the producers with Q) and k_scale go onto its scores
            float srow = 1.f;
            bool q_ok = true;
            if (F16) {
                q_ok = mbar_wait(q_full, iph, err);
                srow = a.k_scale_or_one * qmul[r];
            }
            // this warp has started the item (and read its row factor): the producers may
            // refill Q for the next one once the QKs are done too
            __syncwarp();
            if (lane == 0) mbar_arrive(q_empty);
            const float scale = a.sm_scale * srow, cap = a.soft_cap, c_log2 = a.sm_scale * srow * kLog2e;
            const float cap_k2 = cap != 0.f ? 2.f * kLog2e / cap : 0.f;
            // without a soft cap (and with a positive scale) the row max is taken on the raw
            // scores and the scale goes into the exponent's one FFMA: 2^(s * c - m)
            const bool fold = cap == 0.f && c_log2 > 0.f;
            const float cs = fold ? c_log2 : 1.f;
            constexpr int HB = T::kHalf;
            float m_use = -INFINITY, l_half = 0.f;
            bool ok = q_ok;
            for (int j = 0; ok && j < nb; ++j) {
                const uint32_t q = jb + j, sslot = q % SB, spar = (q / SB) & 1;  // S buffer
                const uint32_t slot = q % PB, par = (q / PB) & 1;                 // P buffer
                if (!mbar_wait(&s_full[sslot], spar, err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float x[HB];
#pragma unroll
                for (int c = 0; c < HB / 32; ++c) {
                    float t32[32];
                    tmem_ld32(tmem + lane_off + sslot * BK + half * HB + c * 32, t32);
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[c * 32 + i] = t32[i];
                }
                tc_fence_before();
                mbar_arrive(&s_free[sslot]);  // QK of block q + SB may overwrite these scores
                const int key0 = kb + j * BK + half * HB;
                if (cap != 0.f) {
                    // small logits (the warp's every |x * scale| <= |cap| / 4): the series form,
                    // on the FMA pipe; otherwise the exponential identity
                    float am = 0.f;
#pragma unroll
                    for (int i = 0; i < HB; i += 2) am = fmax3(am, fabsf(x[i]), fabsf(x[i + 1]));
                    if (__all_sync(0xffffffffu, am * fabsf(scale) <= 0.25f * fabsf(cap))) {
                        const float sl2 = scale * kLog2e, ic = 1.f / (cap * kLog2e);
#pragma unroll
                        for (int i = 0; i < HB; i += 2) {
                            const float2 y = soft_cap_small2(fmul2(make_float2(x[i], x[i + 1]), make_float2(sl2, sl2)), ic);
                            x[i] = y.x;
                            x[i + 1] = y.y;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < HB; ++i) x[i] = soft_cap(x[i] * scale, cap, cap_k2) * kLog2e;
                    }
                } else if (!fold) {
#pragma unroll
                    for (int i = 0; i < HB; ++i) x[i] *= c_log2;
                }
                // the causal / window mask only matters on blocks crossing a row's limits; a mild
                // mask adds mask_value to a masked logit (in x's units: raw scores when the scale
                // is folded into the exponent, log2 units otherwise) and only keys past the
                // sequence are dropped
                const bool inside = key0 >= wlo && key0 + HB - 1 <= qpos;
                if (__any_sync(0xffffffffu, !inside)) {
                    if constexpr (!MILD) {
#pragma unroll
                        for (int i = 0; i < HB; ++i) {
                            const int key = key0 + i;
                            x[i] = (key <= qpos && key >= wlo) ? x[i] : -INFINITY;
                        }
                    } else {
                        const float madd = fold ? a.mask_value / scale : a.mask_value * kLog2e;
                        const int kvl = *s_kvl;
#pragma unroll
                        for (int i = 0; i < HB; ++i) {
                            const int key = key0 + i;
                            const bool vis = key <= qpos && key >= wlo;
                            x[i] = vis ? x[i] : key < kvl ? x[i] + madd : -INFINITY;
                        }
                    }
                }
                float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int i = 0; i < HB; i += 2) mx4[(i >> 1) & 3] = fmax3(mx4[(i >> 1) & 3], x[i], x[i + 1]);
                float* red_j = red + (q & 1) * 256;
                red_j[half * 128 + r] = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
                asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
                tc_fence_after();
                const float mx = fmaxf(red_j[r], red_j[128 + r]) * cs;  // log2 units
                float alpha = 1.f;
                const bool had = m_use > -INFINITY;  // O already holds earlier blocks of this row
                const bool rescale = mx > m_use + 8.f;
                if (rescale) {
                    alpha = fast_exp2(m_use - mx);
                    m_use = mx;
                }
                const float nmu = m_use == -INFINITY ? 0.f : -m_use;
                // P (bf16 pairs) into this block's P buffer once PV of block q - SB has read it:
                // this warp's HB keys are its columns half * HB / 2 ..
                if (!mbar_wait(&p_empty[slot], par ^ 1, err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                const float2 cs2 = make_float2(cs, cs), nmu2 = make_float2(nmu, nmu);
#pragma unroll
                for (int c16 = 0; c16 < HB / 32; ++c16) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float2 a2 = ffma2(make_float2(x[c16 * 32 + 2 * e], x[c16 * 32 + 2 * e + 1]), cs2, nmu2);
                        a2.x = fast_exp2(a2.x);
                        a2.y = fast_exp2(a2.y);
                        sum2[e & 1] = fadd2(sum2[e & 1], a2);
                        pk[e] = F16 ? pack_f16(a2.x, a2.y) : pack_bf16(a2.x, a2.y);
                    }
                    tmem_st16_nowait(tmem + lane_off + T::kColP + slot * (BK / 2) + half * (HB / 2) + c16 * 16, pk);
                }
                // O already holds this row's earlier blocks when l was positive before
                const bool row_rescale = rescale && had;
                l_half = l_half * alpha + ((sum2[0].x + sum2[1].x) + (sum2[0].y + sum2[1].y));
                // tcgen05.ld/st are warp-collective: the warp rescales together when any of its
                // rows needs it (the others multiply by 1); each warp of the pair owns D/2 columns
                if (__any_sync(0xffffffffu, row_rescale)) {
                    const float f = row_rescale ? alpha : 1.f;
                    const uint32_t qp = q - 1, sp = qp % PB, pp = (qp / PB) & 1;
                    if (!mbar_wait(&p_empty[sp], pp, err)) {  // PV(j-1) has finished writing O
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < D / 64; ++c) {
                        float o32[32];
                        const uint32_t col = T::kColO + half * (D / 2) + c * 32;
                        tmem_ld32(tmem + lane_off + col, o32);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o32[i] *= f;
                        tmem_st32(tmem + lane_off + col, o32);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&p_full[slot]);
            }
            // epilogue: l = both halves; each warp of the pair writes D/2 output columns
            float l_run = 0.f;
            if (ok) {
                // the other parity's exchange buffer: both warps are past its last use
                float* red_l = red + ((jb + nb) & 1) * 256;
                red_l[half * 128 + r] = l_half;
                asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
                l_run = red_l[r] + red_l[128 + r];
                asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
            }
            if (ok && mbar_wait(o_full, iph, err)) {
                tc_fence_after();
                const float inv = l_run > 0.f ? (F16 ? a.v_scale_or_one : 1.f) / l_run : 0.f;
                __nv_bfloat16* dst = a.out +
                                     ((size_t)(q_start + (rv ? R / G : 0)) * a.num_q_heads + kvh * G + (rv ? R % G : 0)) *
                                         a.head_dim +
                                     half * (D / 2);
                // every lane runs the (warp-collective) TMEM loads; only real rows store
#pragma unroll 1
                for (int c = 0; c < D / 64; ++c) {
                    float o32[32];
                    tmem_ld32(tmem + lane_off + T::kColO + half * (D / 2) + c * 32, o32);
                    if (rv && half * (D / 2) + c * 32 < a.head_dim) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(o32[2 * i] * inv, o32[2 * i + 1] * inv);
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
                // O has been read: the next item's first PV may overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_empty);
            } else {
                s_abort = 1;
            }
            tc_fence_before();
        }
        __syncwarp();  // the issuer warps' idle lanes wait here for lane 0, not at the next slot
        jb += nb;
        ++items;
    }
    // every role has left its loop (the softmax warps' last TMEM reads included)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // drain: every MMA this CTA issued has completed before TMEM is released
    if (warp == kPvW && lane == 0) umma_commit(fin);
    if (warp == kMmaW) {
        if (lane == 0) {
            umma_commit(fin);
            mbar_wait(fin, 0, err);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, T::kTmemCols);
    }
}

// Tensor maps (built on the host per call: they embed the caller's pointers).
static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 3-D bf16 tensor [d2][d1][d0] (d0 contiguous) with a box of {64, b1, b2}, 128-byte swizzle.
static bool make_tmap_bf16(CUtensorMap* tm, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b1,
                           uint32_t b2) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    const cuuint32_t box[3] = {64, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D one-byte tensor [d2][d1][d0] (d0 contiguous) with a box of {128, 1, b2}, 128-byte swizzle:
// half of a raw K or V row per copy (the raw-staging path).
static bool make_tmap_u8(CUtensorMap* tm, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b2) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0, d0 * d1};
    const cuuint32_t box[3] = {128, 1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool FP8, bool SCALE, bool TMA, bool I8 = false, bool F16 = false, bool RAW = false, bool I4 = false,
          bool MILD = false>
static cudaError_t launch_pre(const RpaArgs& a, int num_sms, cudaStream_t stream, const CUtensorMap& tkv,
                              const CUtensorMap& tq, int box_rows, int q_tma, int tail) {
    using T = PreTc<D, RAW>;
    auto kern = rpa_prefill_tc_kernel<D, FP8, SCALE, TMA, I8, F16, RAW, I4, MILD>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    // tail 1: the launch after decode; 2: the only attention launch of a prefill-only batch
    ProfScope ps(tail == 1 ? "rpa_prefill_tail" : "rpa_prefill_attn", stream);
    return launch_pdl(kern, dim3(num_sms), dim3(prefill_warps<RAW>() * 32), T::kSmem, stream, a.overlap && !tail, a,
                      tkv, tq, box_rows, q_tma, tail);
}

template <int D>
static cudaError_t launch_pre_d(const RpaArgs& a, int num_sms, cudaStream_t stream, int tail) {
    constexpr int BK = PreTc<D>::BK;
    CUtensorMap tkv, tq;
    memset(&tkv, 0, sizeof tkv);
    memset(&tq, 0, sizeof tq);
    const int ps = a.page_size, G = a.num_q_heads / a.num_kv_heads, C = 2 * a.num_kv_heads;
    // box of one page (or of one block when pages are longer); page sizes that do not tile
    // the block, or boxes too small for one lane each, take the register path
    const int box_rows = ps < BK ? ps : BK;
    // (boxes of >= 8 rows keep every TMA destination on a 1024-byte swizzle-atom boundary)
    if (a.head_dim != D && (a.mask_mild || a.kv_byte || a.has_scale)) return cudaErrorInvalidValue;
    if (a.mask_mild) {
        // mild masks: the register path for every cache type (one-byte caches dequantised to bf16)
        if (a.kv_int4) return launch_pre<D, true, false, false, false, false, false, true, true>(a, num_sms, stream, tkv, tq, 0, 0, tail);
        if (a.kv_int8) return launch_pre<D, true, false, false, true, false, false, false, true>(a, num_sms, stream, tkv, tq, 0, 0, tail);
        if (a.kv_byte) return launch_pre<D, true, false, false, false, false, false, false, true>(a, num_sms, stream, tkv, tq, 0, 0, tail);
        if (a.has_scale) return launch_pre<D, false, true, false, false, false, false, false, true>(a, num_sms, stream, tkv, tq, 0, 0, tail);
        return launch_pre<D, false, false, false, false, false, false, false, true>(a, num_sms, stream, tkv, tq, 0, 0, tail);
    }
    bool tma = !a.kv_byte && !a.has_scale && (ps & (ps - 1)) == 0 && box_rows >= 8 && BK / box_rows <= 32;
    const uint64_t tokens = (uint64_t)a.total_num_pages * ps;
    // (the maps are a.head_dim wide: at head_dim 96 or 192 the boxes' columns past it read
    // the fill value, zero, so the kernel runs at D = the next multiple of 128 unchanged)
    if (tma) tma = make_tmap_bf16(&tkv, a.kv_pages, a.head_dim, C, tokens, 1, box_rows);
    int q_tma = 0;
    if (tma && 128 % G == 0)
        q_tma = make_tmap_bf16(&tq, a.q, a.head_dim, a.num_q_heads, a.max_num_tokens, G, 128 / G) ? 1 : 0;
    if (tma) return launch_pre<D, false, false, true>(a, num_sms, stream, tkv, tq, box_rows, q_tma, tail);
    if (a.head_dim != D) return cudaErrorInvalidValue;  // (the host admits such shapes only where TMA runs)
    // int4 caches: dequantised to bf16 through registers
    if (a.kv_int4) return launch_pre<D, true, false, false, false, false, false, true>(a, num_sms, stream, tkv, tq, box_rows, 0, tail);
    // one-byte caches with power-of-two scales: exact f16 operands, scales on S and O
    const bool pow2 = rpa_pow2_scale(a.k_scale_or_one) && rpa_pow2_scale(a.v_scale_or_one);
    if constexpr (D == 128 || D == 256) {
        // one-byte caches whose pages tile the block in boxes of >= 8 rows: raw rows by TMA,
        // converted in shared memory, Q in TMEM
        bool raw = a.kv_byte && (ps & (ps - 1)) == 0 && box_rows >= 8 && BK / box_rows <= 32;
        if (raw) raw = make_tmap_u8(&tkv, a.kv_pages, D, C, tokens, box_rows);
        if (raw) {
            // Q staged by TMA (boxes of G heads x 128 / G tokens) when G divides the tile
            const int qt = (128 % G == 0 && make_tmap_bf16(&tq, a.q, D, a.num_q_heads, a.max_num_tokens, G, 128 / G)) ? 1 : 0;
            if (a.kv_int8 && pow2)
                return launch_pre<D, true, false, false, true, true, true>(a, num_sms, stream, tkv, tq, box_rows, qt, tail);
            if (a.kv_int8) return launch_pre<D, true, false, false, true, false, true>(a, num_sms, stream, tkv, tq, box_rows, qt, tail);
            if (pow2) return launch_pre<D, true, false, false, false, true, true>(a, num_sms, stream, tkv, tq, box_rows, qt, tail);
            return launch_pre<D, true, false, false, false, false, true>(a, num_sms, stream, tkv, tq, box_rows, qt, tail);
        }
    }
    if (a.kv_int8 && pow2) return launch_pre<D, true, false, false, true, true>(a, num_sms, stream, tkv, tq, box_rows, 0, tail);
    if (a.kv_int8) return launch_pre<D, true, false, false, true>(a, num_sms, stream, tkv, tq, box_rows, 0, tail);
    if (a.kv_byte && pow2) return launch_pre<D, true, false, false, false, true>(a, num_sms, stream, tkv, tq, box_rows, 0, tail);
    if (a.kv_byte) return launch_pre<D, true, false, false>(a, num_sms, stream, tkv, tq, box_rows, 0, tail);
    if (a.has_scale) return launch_pre<D, false, true, false>(a, num_sms, stream, tkv, tq, box_rows, 0, tail);
    return launch_pre<D, false, false, false>(a, num_sms, stream, tkv, tq, box_rows, 0, tail);
}

cudaError_t launch_rpa_prefill(const RpaArgs& a, int num_sms, cudaStream_t stream, int tail) {
    switch (a.head_dim) {
        case 64: return launch_pre_d<64>(a, num_sms, stream, tail);
        case 96:
        case 128: return launch_pre_d<128>(a, num_sms, stream, tail);
        case 192:
        case 256: return launch_pre_d<256>(a, num_sms, stream, tail);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rpa
