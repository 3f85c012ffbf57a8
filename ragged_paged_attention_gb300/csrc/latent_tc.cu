// MLA latent attention (tpu-inference "mla/v1/kernel.py") and DSA sparse MLA (sglang-jax
// "dsa/sparse_mla_prefill.py") on the 5th-generation tensor cores of sm_103a.
//
// Both are MQA over one latent head: the 128 q heads of a query read the same key rows
// [kv_c (512) | k_pe (64)] and the value is kv_c.  A 128-head Q slice of 576 bf16 is 144 KB
// and the fp32 output [128 x 512] fills all of TMEM, so one query is worked by a cluster
// of two CTAs that split the latent dimensions:
//   rank 0: score dims 0-255 and the 64 rope dims, output dims 0-255;
//   rank 1: score dims 256-511,                    output dims 256-511.
// Each CTA keeps its Q slice in tensor memory (the MMA's A operand), gathers only its dims
// of each key row into a 4-deep shared-memory ring and computes a partial score tile
// S_r = Q_r K_r^T (tcgen05, 128 x 64 per block).  The softmax of the 128 rows is split
// between the two CTAs: rank r owns rows 64r..64r+63.  For the peer's rows, a CTA only
// sends its partial scores (fp32, through distributed shared memory: st.async into a
// double-buffered receive area, completing on the receiver's mbarrier) and later receives
// those rows' P (bf16) and rescale factor; for its own rows it adds the peer's partial,
// runs the online softmax, keeps P and sends it to the peer.  Both CTAs then accumulate
// O_r += P V_r into their own 256 TMEM columns (P is the A operand, in TMEM).  This moves
// 24 KB per block each way instead of 32 (the SM-to-SM link, not the tensor core, bounds
// a block) and halves the exponentials per CTA.  Receive buffers are reused two blocks
// later: readers arrive on a local barrier and a signalling warp (with no remote stores of
// its own in flight) passes that on to the peer with one cluster-scope release arrive.
// Row statistics (m, l) of the owned rows go to the peer once per item.
// Warps per CTA: 0-7 softmax (two per TMEM lane quarter, 32 of the 64 columns each; a
// quarter's warps are owners or helpers), 8-11 producers, 12 MMA issuer, 13 signalling.
// MLA keys are the causal (windowed) prefix, brought page by page with TMA boxes (the
// partial last page through registers); sparse keys are the selected units' rows, four at a
// time by TMA tile::gather4 copies, with their validity recorded for the softmax.  Items
// split long key ranges; partials merge by the log-sum-exp rule.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "profile.h"

namespace rpa {

namespace lat {
constexpr int BK = 64;                        // keys per block
constexpr int NQP_MAX = 5;                    // score panels of rank 0 (4 latent + 1 rope)
constexpr int kPanel = BK * 128;              // one key panel: [64 rows x 64 dims]
constexpr int kStage = NQP_MAX * kPanel;
constexpr int NS = 4;                         // key stages
// receive buffers (in the receiving CTA), a warp's 32 rows of one 16-byte chunk contiguous:
constexpr int kSRecv = 2 * 8 * 64 * 16;       // peer's partial S of my 64 rows: [half][8 chunks][row]
constexpr int kPRecv = 2 * 4 * 64 * 16 + 64 * 4;  // P of the peer's 64 rows [half][4 chunks][row] + alpha[row]
constexpr int kOffKV = 0;
constexpr int kOffSRecv = kOffKV + NS * kStage;    // [2]
constexpr int kOffPRecv = kOffSRecv + 2 * kSRecv;  // [2]
constexpr int kOffStat = kOffPRecv + 2 * kPRecv;   // (m, l) of the peer's rows
constexpr int kOffBar = kOffStat + 64 * 8;
constexpr int kNumBars = 3 * NS + 26;
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffRed = (kOffTmemSlot + 16 + 127) / 128 * 128;
constexpr int kOffVld = kOffRed + 2 * 2 * 128 * 4;
constexpr int kOffItem = kOffVld + NS * BK;
constexpr int kSmem = kOffItem + 64;  // item, abort flag, item index, index ring [2], merge flag
// TMEM columns: S [128 x 64] fp32 at 0, the Q slice (bf16 pairs, 160 or 128 columns) at 64,
// P [128 x 64] bf16 pairs at 224, the O half [128 x 256] fp32 at 256.
constexpr int kColS = 0, kColQ = BK, kColP = 224, kColO = 256;
constexpr int kTmemCols = 512;
// split merges keep their weights [split][128 rows] in the idle key ring (up to this many splits)
constexpr int kMergeSplits = NS * kStage / (128 * 4);
constexpr int kWarps = 14;
constexpr int kProdW0 = 8, kMmaW = 12, kSigW = 13;
static_assert(kSmem <= 232448, "shared memory budget");
static_assert(kOffKV % 1024 == 0 && kOffSRecv % 16 == 0 && kOffPRecv % 16 == 0 && kPRecv % 16 == 0 &&
                  kOffBar % 8 == 0 && kOffItem % 16 == 0, "alignment");
static_assert(kColQ + NQP_MAX * 32 <= kColP && kColP + BK / 2 <= kColO, "TMEM columns");
}  // namespace lat

// Column (in elements) of latent row data that panel p of CTA `rank` holds.
__device__ __forceinline__ int lat_panel_col(int rank, int p) { return rank == 0 ? (p < 4 ? 64 * p : 512) : 256 + 64 * p; }

template <bool SPARSE>
__global__ void __launch_bounds__(lat::kWarps * 32, 1)
    latent_tc_kernel(LatentArgs a, const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_kr,
                     const __grid_constant__ CUtensorMap tm_kc3, const __grid_constant__ CUtensorMap tm_qa,
                     const __grid_constant__ CUtensorMap tm_qb, int kv_tma, int box_rows, int q_tma) {
    using namespace lat;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* kv_full = bars + 0;           // [NS] this CTA's key panels landed
    uint64_t* kv_empty = bars + NS;         // [NS] PV of that block done
    uint64_t* vld_full = bars + 2 * NS;     // [NS] (sparse) key validity written
    uint64_t* s_full = bars + 3 * NS;       // partial S written by QK
    uint64_t* s_empty = bars + 3 * NS + 1;  // partial S read by the softmax
    uint64_t* p_full = bars + 3 * NS + 2;     // P written to TMEM (and O rescaled)
    uint64_t* p_empty = bars + 3 * NS + 3;    // PV done with P
    uint64_t* q_full = bars + 3 * NS + 4;     // the Q slice is in TMEM
    uint64_t* o_full = bars + 3 * NS + 5;
    uint64_t* fin = bars + 3 * NS + 6;
    uint64_t* srecv_full = bars + 3 * NS + 7;   // [2] the peer's partial S of my rows landed (bytes)
    uint64_t* srecv_used = bars + 3 * NS + 9;   // [2] my owner threads have read it
    uint64_t* s_free = bars + 3 * NS + 11;      // [2] the peer has read the S buffer I write next
    uint64_t* precv_full = bars + 3 * NS + 13;  // [2] P + alpha of the peer's rows landed (bytes)
    uint64_t* precv_used = bars + 3 * NS + 15;  // [2] my helper threads have read it
    uint64_t* p_free = bars + 3 * NS + 17;      // [2] the peer has read the P buffer I write next
    uint64_t* stat_full = bars + 3 * NS + 19;   // (m, l) of the peer's rows landed (bytes)
    uint64_t* itm_full = bars + 3 * NS + 20;    // [2] (MLA, rank 1) the item index from rank 0 landed
    uint64_t* itm_free = bars + 3 * NS + 22;    // [2] (MLA, rank 0) rank 1 has read that slot's index
    uint64_t* q_land = bars + 3 * NS + 24;      // (Q by TMA) the Q slice's boxes landed in the ring
    uint64_t* q_free = bars + 3 * NS + 25;      // (Q by TMA) the softmax threads have read them
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
    float* red = reinterpret_cast<float*>(smem + kOffRed);
    uint8_t* vld = smem + kOffVld;
    WorkItem& s_item = *reinterpret_cast<WorkItem*>(smem + kOffItem);
    volatile int& s_abort = *reinterpret_cast<volatile int*>(smem + kOffItem + 32);
    volatile int* s_itm = reinterpret_cast<volatile int*>(smem + kOffItem + 40);  // [2] item index slots

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
    const int nqp = rank == 0 ? 5 : 4;
    WsHeader* hdr = a.hdr;
    uint32_t* err = &hdr->error_bits;
    const int H = a.num_heads;
    const int tiles = H / 128;

    for (int i = tid * 16; i < kOffSRecv; i += blockDim.x * 16) *reinterpret_cast<uint4*>(smem + i) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&kv_full[i], (kv_tma == 1 || kv_tma == 2) ? 32 : 128);  // MLA TMA: warp 8; gathers: all producers
            mbar_init(&kv_empty[i], 1);
            mbar_init(&vld_full[i], 128);
        }
        mbar_init(p_full, 256);
        mbar_init(p_empty, 1);
        mbar_init(s_full, 1);
        mbar_init(s_empty, 256);
        mbar_init(q_full, 256);
        mbar_init(o_full, 1);
        mbar_init(fin, 1);
        for (int i = 0; i < 2; ++i) {
            // *_full: one local thread arms the bytes, the peer's st.async complete them;
            // *_free: the peer's signalling thread arrives
            mbar_init(&srecv_full[i], 1);
            mbar_init(&srecv_used[i], 128);
            mbar_init(&s_free[i], 1);
            mbar_init(&precv_full[i], 1);
            mbar_init(&precv_used[i], 128);
            mbar_init(&p_free[i], 1);
        }
        mbar_init(stat_full, 1);
        mbar_init(q_land, 1);
        mbar_init(q_free, 256);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&itm_full[i], 1);  // rank 1 arms the 4 bytes rank 0's st.async delivers
            mbar_init(&itm_free[i], 1);  // rank 1's release arrive
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaW) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // items are dealt round-robin to clusters: both CTAs of a cluster see the same sequence
    int sparse_items = 0, slots = 0, sparse_chunk = 0;
    if (SPARSE) {
        slots = a.topk * a.read_block;
        sparse_items = a.batch * a.num_queries * tiles * a.sparse_splits;
        sparse_chunk = cdiv(cdiv(slots, a.sparse_splits), BK) * BK;
    }
    const int n_items = SPARSE ? sparse_items : hdr->num_items[2];
    uint32_t jb = 0, items = 0, nstat = 0;
    // Sparse items are dealt round-robin to the clusters (every query selects the same number of
    // units). MLA items differ in length, so they are taken from a queue that the plan sorted
    // longest first: rank 0 of a cluster takes the next index and hands it to rank 1 through that
    // CTA's shared memory (st.async on a two-slot ring, bounded waits on both sides), so both
    // CTAs work the same item.
    const uint32_t itm_slot_peer = mapa_shared(smem_u32((const void*)s_itm), peer);
    const uint32_t itm_full_peer = mapa_shared(smem_u32(itm_full), peer);
    const uint32_t itm_free_peer = mapa_shared(smem_u32(itm_free), peer);
    for (uint32_t k = 0;; ++k) {
        volatile int& s_it = *reinterpret_cast<volatile int*>(smem + kOffItem + 36);
        if (tid == 0) {
            int it;
            if (SPARSE) {
                it = (int)cluster_id_x() + (int)k * (int)cluster_count_x();
            } else {
                const uint32_t sl = k & 1, ph = (k >> 1) & 1;
                if (rank == 0) {
                    it = n_items;
                    if (mbar_wait_cluster(&itm_free[sl], ph ^ 1, err)) {  // rank 1 has read index k - 2
                        const int q = atomicAdd(&hdr->next_item[2], 1);
                        it = q < n_items ? q : n_items;
                    } else {
                        s_abort = 1;
                    }
                    st_async_f32(itm_slot_peer + sl * 4, __int_as_float(it), itm_full_peer + sl * 8);
                } else {
                    mbar_arrive_expect_tx(&itm_full[sl], 4);
                    if (mbar_wait_cluster(&itm_full[sl], ph, err)) {
                        it = s_itm[sl];
                        mbar_arrive_cluster(itm_free_peer + sl * 8);
                    } else {
                        it = n_items;
                        s_abort = 1;
                    }
                }
            }
            s_it = it;
            if (it < n_items) {
                WorkItem w;
                if (SPARSE) {
                    const int per_q = tiles * a.sparse_splits;
                    const int bs = it / per_q, rem = it % per_q;
                    const int tile = rem / a.sparse_splits, sp = rem % a.sparse_splits;
                    w.seq = bs;
                    w.head = tile * 128;
                    w.row_begin = 0;
                    w.key_begin = sp * sparse_chunk;
                    w.key_end = min(slots, (sp + 1) * sparse_chunk);
                    w.first_item = it - sp;
                    w.num_splits = a.sparse_splits;
                    w.split = sp;
                } else {
                    w = a.items[it];
                }
                s_item = w;
            }
        }
        __syncthreads();
        const int it = s_it;
        if (it >= n_items) break;
        const WorkItem w = s_item;
        if (s_abort) break;
        const int h0 = w.head;
        int qpos, b = 0, seq = 0, t = 0, wlo = INT_MIN, q_start = 0;
        int kbound = 0, kbase = 0;  // sparse: the query's causal bound and packed page base
        if (SPARSE) {
            b = w.seq / a.num_queries;
            qpos = a.positions[w.seq];
            kbound = a.q_bound ? a.q_bound[w.seq] : a.seq_len;
            kbase = a.q_base ? a.q_base[w.seq] : 0;
        } else {
            seq = w.seq;
            t = w.row_begin;
            q_start = a.cu_q_lens[seq];
            qpos = a.kv_lens[seq] - (a.cu_q_lens[seq + 1] - q_start) + (t - q_start);
            if (a.sliding_window > 0) wlo = qpos - a.sliding_window + 1;
        }
        const int kb = w.key_begin, ke = w.key_end;
        const int nb = ke > kb ? cdiv(ke - kb, BK) : 0;
        const uint32_t iph = items & 1;
        const int qrow0 = (SPARSE ? w.seq : t) * H + h0;  // first Q row of the tile

        if (warp >= kProdW0 && warp < kMmaW) {
            // ---------------- producers ----------------
            const int pt = tid - kProdW0 * 32;
            if (SPARSE && kv_tma == 3) {
                // selected rows by TMA gathers: warp w of the four resolves keys 16w .. 16w+15 of
                // each block (one per lane, one block ahead) and its lanes 0-3 each gather one group
                // of four rows, one 4-row copy per 64-column panel, straight into the swizzled
                // panels; a key that is not valid gathers a row past the cache (zeros). Every
                // block's copies go out as soon as its slot is free, so up to NS blocks are in flight.
                const int wsub = warp - kProdW0, kk = wsub * 16 + (lane & 15);
                const bool rb_p2 = (a.read_block & (a.read_block - 1)) == 0, ps_p2 = (a.page_size & (a.page_size - 1)) == 0;
                const int rb_sh = __ffs(a.read_block) - 1, ps_sh = __ffs(a.page_size) - 1;
                const int oob_row = a.total_num_pages * a.page_size;  // gathers zeros
                // A key is resolved in three steps an iteration apart, so that no step waits on
                // the load of the one before: its unit (index load), then its token, validity and
                // page-table entry (page load), then its row.
                auto idx_load = [&](int j, int& u, int& key) {
                    key = kb + j * BK + kk;
                    const bool in = lane < 16 && j < nb && key < ke;
                    const int kc = in ? key : kb;  // a slot of this query: kb < ke when nb > 0
                    if (!in) key = -1;
                    u = __ldg(a.indices + (size_t)w.seq * a.topk + (rb_p2 ? kc >> rb_sh : kc / a.read_block));
                };
                auto page_load = [&](int u, int key, int& page, int& po, int& st) {
                    // st: 0 no key, 1 key with a page-table entry (page loaded), 2 key past the table
                    const int kc = key >= 0 ? key : 0;
                    const int ur = rb_p2 ? kc & (a.read_block - 1) : kc % a.read_block;
                    const long long kp = (long long)u * a.read_block + ur;
                    const bool v = key >= 0 && u >= 0 && kp <= qpos && kp < kbound;
                    const long long kpc = v ? kp : 0;
                    const int lp = ps_p2 ? (int)(kpc >> ps_sh) : (int)(kpc / a.page_size);
                    po = ps_p2 ? (int)(kpc & (a.page_size - 1)) : (int)(kpc % a.page_size);
                    long long pidx;
                    bool pin;
                    if (a.q_base) {  // packed list: the request's run, clamped to the list's end
                        pidx = min((long long)kbase + lp, (long long)a.max_pages - 1);
                        pin = pidx >= 0;
                    } else {
                        pin = lp < a.max_pages;
                        pidx = (long long)b * a.max_pages + lp;
                    }
                    st = !v ? 0 : pin ? 1 : 2;
                    page = __ldg(a.page_table + (st == 1 ? pidx : 0));
                };
                auto row_of = [&](int page, int po, int st) -> int {
                    if (st == 0) return oob_row;
                    const int pg = st == 1 ? page : -1;
                    if ((unsigned)pg >= (unsigned)a.total_num_pages) {
                        set_error(err, RPA_DEV_ERR_PAGE);
                        return oob_row;
                    }
                    return pg * a.page_size + po;
                };
                int gu, gkey, gpage, gpo, gst;
                idx_load(0, gu, gkey);
                page_load(gu, gkey, gpage, gpo, gst);
                idx_load(1, gu, gkey);
                const uint32_t grp_bytes = 4u * nqp * 128;  // one group's four rows, every panel
                for (int j = 0; j < nb; ++j) {
                    const uint32_t q = jb + j, st = q % NS, par = (q / NS) & 1;
                    const int row = row_of(gpage, gpo, gst);
                    const bool v = row != oob_row;
                    page_load(gu, gkey, gpage, gpo, gst);  // block j + 1
                    idx_load(j + 2, gu, gkey);
                    int g = 1;
                    if (lane == 0) {
                        g = mbar_wait(&kv_empty[st], par ^ 1, err) && (j != NS - 2 || !q_tma || mbar_wait(q_free, iph, err));
                        if (g)
                            mbar_expect_tx(&kv_full[st], 4 * grp_bytes);
                        else
                            s_abort = 1;
                    }
                    if (!__shfl_sync(0xffffffffu, g, 0)) break;
                    if (lane < 16) vld[st * BK + kk] = v ? 1 : 0;
                    mbar_arrive(&vld_full[st]);  // (read by the softmax through plain loads)
                    // group gi = lane & 3: the rows of lanes 4gi .. 4gi+3
                    const int gi = lane & 3;
                    const int r0 = __shfl_sync(0xffffffffu, row, 4 * gi), r1 = __shfl_sync(0xffffffffu, row, 4 * gi + 1);
                    const int r2 = __shfl_sync(0xffffffffu, row, 4 * gi + 2), r3 = __shfl_sync(0xffffffffu, row, 4 * gi + 3);
                    if (lane < 4) {
                        uint8_t* dst = smem + kOffKV + st * kStage + (wsub * 16 + gi * 4) * 128;
#pragma unroll
                        for (int p = 0; p < NQP_MAX; ++p)
                            if (p < nqp)
                                tma_gather4(smem_u32(dst + p * kPanel), &tm_kc, lat_panel_col(rank, p), r0, r1, r2, r3,
                                            &kv_full[st]);
                    }
                    mbar_arrive(&kv_full[st]);
                }
            } else if (!SPARSE && kv_tma) {
                if (warp == kProdW0) {
                    const int nbox = BK / box_rows;
                    const size_t tbl = (size_t)seq * a.pages_per_seq;
                    auto page_of = [&](int j) -> int {
                        const int key = kb + j * BK + lane * box_rows;
                        return (lane < nbox && j < nb && key < ke) ? __ldg(a.page_indices + tbl + key / a.page_size) : -1;
                    };
                    int page_next = page_of(0);
                    for (int j = 0; j < nb; ++j) {
                        const uint32_t q = jb + j, st = q % NS, par = (q / NS) & 1;
                        const int page = page_next;
                        page_next = page_of(j + 1);
                        const int kbx = kb + j * BK + lane * box_rows;
                        int rows = lane < nbox ? min(box_rows, ke - kbx) : 0;
                        if (rows < 0) rows = 0;
                        if (rows > 0 && (unsigned)page >= (unsigned)a.total_num_pages) {
                            set_error(err, RPA_DEV_ERR_PAGE);
                            rows = 0;
                        }
                        const bool full = rows == box_rows;
                        uint32_t bytes = full ? (uint32_t)box_rows * nqp * 128 : 0u;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
                        int g = 1;
                        if (lane == 0) {
                            g = mbar_wait(&kv_empty[st], par ^ 1, err) && (j != NS - 2 || !q_tma || mbar_wait(q_free, iph, err));
                            if (g)
                                mbar_expect_tx(&kv_full[st], bytes);
                            else
                                s_abort = 1;
                        }
                        if (!__shfl_sync(0xffffffffu, g, 0)) break;
                        uint8_t* stage = smem + kOffKV + st * kStage;
                        const int row0 = page * a.page_size + kbx % a.page_size;
                        if (full && kv_tma == 2) {
                            // whole block in one box: the four latent panels of this rank in one
                            // 3-D copy ([panel][row][64] lands as the stage layout), rope apart
                            tma_load_3d(smem_u32(stage), &tm_kc3, 0, row0, rank == 0 ? 0 : 4, &kv_full[st]);
                            if (rank == 0) tma_load_2d(smem_u32(stage + 4 * kPanel), &tm_kr, 0, row0, &kv_full[st]);
                        } else if (full) {
                            for (int p = 0; p < nqp; ++p) {
                                const uint32_t dst = smem_u32(stage + p * kPanel + lane * box_rows * 128);
                                if (rank == 0 && p == 4)
                                    tma_load_2d(dst, &tm_kr, 0, row0, &kv_full[st]);
                                else
                                    tma_load_2d(dst, &tm_kc, lat_panel_col(rank, p), row0, &kv_full[st]);
                            }
                        }
                        // a box that is not full (the sequence's last keys): its rows by cp.async,
                        // all of them in flight at once.  Past the range the mask drops the scores
                        // (a select, whatever the bytes), but P = 0 multiplies the value rows, and
                        // 0 * v is 0 only for finite v: those rows' value panels get zeros (the
                        // ring's stale bytes may be fp32 words of an output tile or merge weights)
                        uint32_t pm = __ballot_sync(0xffffffffu, rows > 0 && !full);
                        uint32_t pz = __ballot_sync(0xffffffffu, lane < nbox && !full);
                        const bool wrote = pz != 0;
                        while (pm) {
                            const int src = __ffs(pm) - 1;
                            pm &= pm - 1;
                            const int prow = __shfl_sync(0xffffffffu, rows, src);
                            const int pr0 = __shfl_sync(0xffffffffu, row0, src);
                            for (int i = lane; i < prow * nqp * 8; i += 32) {
                                const int r = i / (nqp * 8), rem = i % (nqp * 8), p = rem / 8, c = rem % 8;
                                const int kk = src * box_rows + r;
                                const __nv_bfloat16* s_row = (rank == 0 && p == 4)
                                                                  ? a.cache_k_pe + (size_t)(pr0 + r) * a.r_pad
                                                                  : a.cache_kv_c + (size_t)(pr0 + r) * a.lkv_pad + lat_panel_col(rank, p);
                                cp_async16(smem_u32(stage + p * kPanel + kk * 128 + ((c ^ (kk & 7)) << 4)), s_row + c * 8, true);
                            }
                        }
                        while (pz) {
                            const int src = __ffs(pz) - 1;
                            pz &= pz - 1;
                            const int prow = __shfl_sync(0xffffffffu, rows, src);
                            for (int i = lane; i < (box_rows - prow) * 32; i += 32) {
                                const int kk = src * box_rows + prow + (i >> 5), p = (i >> 3) & 3, c = i & 7;
                                *reinterpret_cast<uint4*>(stage + p * kPanel + kk * 128 + ((c ^ (kk & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                            }
                        }
                        if (wrote) {
                            cp_async_commit();
                            cp_async_wait<0>();
                            fence_proxy_async_smem();  // thread-copied rows, read by the tensor core
                        }
                        mbar_arrive(&kv_full[st]);
                    }
                }
            } else {
                // row gather: two threads per key row, each half of the row's panels.  The row
                // of the next block is resolved (index -> token -> page) while this block's slot
                // is still busy.
                const int kk = pt >> 1, hh = pt & 1;
                const int nch = nqp * 4;  // chunks of this thread (20 or 16)
                // read_block and page_size are powers of two in practice: shifts and masks then
                // replace the divisions (two of them 64-bit) this thread runs for every block
                const bool rb_p2 = (a.read_block & (a.read_block - 1)) == 0, ps_p2 = (a.page_size & (a.page_size - 1)) == 0;
                const int rb_sh = __ffs(a.read_block) - 1, ps_sh = __ffs(a.page_size) - 1;
                auto resolve = [&](int j, bool& v) -> const __nv_bfloat16* {
                    const int key = kb + j * BK + kk;
                    v = j < nb && key < ke;
                    if (!v) return nullptr;
                    if (SPARSE) {
                        const int ui = rb_p2 ? key >> rb_sh : key / a.read_block;
                        const int ur = rb_p2 ? key & (a.read_block - 1) : key % a.read_block;
                        const int u = __ldg(a.indices + (size_t)w.seq * a.topk + ui);
                        const long long kp = (long long)u * a.read_block + ur;
                        v = u >= 0 && kp <= qpos && kp < kbound;
                        if (!v) return nullptr;
                        // kp >= 0 here (u >= 0)
                        const int lp = ps_p2 ? (int)(kp >> ps_sh) : (int)(kp / a.page_size);
                        const int po = ps_p2 ? (int)(kp & (a.page_size - 1)) : (int)(kp % a.page_size);
                        int page;
                        if (a.q_base) {  // packed list: the request's run, clamped to the list's end
                            const long long pidx = min((long long)kbase + lp, (long long)a.max_pages - 1);
                            page = pidx >= 0 ? __ldg(a.page_table + pidx) : -1;
                        } else {
                            page = lp < a.max_pages ? __ldg(a.page_table + (size_t)b * a.max_pages + lp) : -1;
                        }
                        if ((unsigned)page >= (unsigned)a.total_num_pages) {
                            set_error(err, RPA_DEV_ERR_PAGE);
                            v = false;
                            return nullptr;
                        }
                        return a.cache + ((size_t)page * a.page_size + po) * a.row_stride;
                    }
                    const int page = __ldg(a.page_indices + (size_t)seq * a.pages_per_seq + key / a.page_size);
                    if ((unsigned)page >= (unsigned)a.total_num_pages) {
                        set_error(err, RPA_DEV_ERR_PAGE);
                        v = false;
                        return nullptr;
                    }
                    return a.cache_kv_c + ((size_t)page * a.page_size + key % a.page_size) * a.lkv_pad;
                };
                bool v_next;
                const __nv_bfloat16* row_next = resolve(0, v_next);
                // copies go by cp.async (no register staging): a thread keeps one block's copies
                // in flight while it issues the next, and publishes a block (proxy fence, arrive)
                // once that block's copies have landed
                int prev_st = -1;
                for (int j = 0; j < nb; ++j) {
                    const uint32_t q = jb + j, st = q % NS, par = (q / NS) & 1;
                    const bool v = v_next;
                    const __nv_bfloat16* row = row_next;
                    row_next = resolve(j + 1, v_next);
                    if (!mbar_wait(&kv_empty[st], par ^ 1, err) || (j == NS - 2 && q_tma && !mbar_wait(q_free, iph, err))) {
                        s_abort = 1;
                        break;
                    }
                    uint8_t* stage = smem + kOffKV + st * kStage;
                    if (v) {
                        // MLA rope panel (rank 0, panel 4) comes from the k_pe cache row
                        const __nv_bfloat16* pe_row =
                            SPARSE ? nullptr : a.cache_k_pe + (size_t)((row - a.cache_kv_c) / a.lkv_pad) * a.r_pad;
#pragma unroll
                        for (int i = 0; i < 20; ++i) {
                            if (i < nch) {
                                const int c = hh * nch + i, p = c >> 3, cc = c & 7;
                                const __nv_bfloat16* src = (!SPARSE && rank == 0 && p == 4) ? pe_row + cc * 8
                                                                                           : row + lat_panel_col(rank, p) + cc * 8;
                                cp_async16(smem_u32(stage + p * kPanel + kk * 128 + ((cc ^ (kk & 7)) << 4)), src, true);
                            }
                        }
                    } else {
                        // a key that is not valid: zeros in its value panels (its P is 0, and
                        // 0 * v is 0 only for finite v)
                        for (int c = hh * 16; c < hh * 16 + 16; ++c)
                            *reinterpret_cast<uint4*>(stage + (c >> 3) * kPanel + kk * 128 + (((c & 7) ^ (kk & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                    }
                    cp_async_commit();
                    if (SPARSE) {
                        if (hh == 0) vld[st * BK + kk] = v ? 1 : 0;
                        mbar_arrive(&vld_full[st]);  // (read by the softmax through plain loads)
                    }
                    if (prev_st >= 0) {
                        cp_async_wait<1>();  // the previous block's copies have landed
                        fence_proxy_async_smem();
                        mbar_arrive(&kv_full[prev_st]);
                    }
                    prev_st = (int)st;
                }
                cp_async_wait<0>();
                if (prev_st >= 0 && !s_abort) {
                    fence_proxy_async_smem();
                    mbar_arrive(&kv_full[prev_st]);
                }
            }
        } else if (warp == kMmaW) {
            // ---------------- MMA issuer ----------------
            if (lane == 0) {
                constexpr uint32_t idesc_qk = umma_idesc_bf16(128, BK, false, false);
                constexpr uint32_t idesc_pv = umma_idesc_bf16(128, 256, false, true);
                // descriptors of stage 0; a byte offset d within shared memory adds d >> 4 to
                // the start-address field (no carry: every address is below 256 KB)
                const uint64_t kdesc0 = umma_desc_sw128(smem_u32(smem + kOffKV), 16, 1024);
                const uint64_t vdesc0 = umma_desc_sw128(smem_u32(smem + kOffKV), kPanel, 1024);
                bool ok = mbar_wait(q_full, iph, err);
                tc_fence_after();
                // issue QK(next) and PV(next) in whichever order their inputs become ready
                int nq = 0, np = 0;
                unsigned long long t0 = 0;
                uint32_t idle = 0;
                while (ok && np < nb) {
                    bool moved = false;
                    if (nq < nb) {
                        // S is single-buffered: QK(q) needs the softmax to have read S(q-1)
                        const uint32_t q = jb + nq, st = q % NS, par = (q / NS) & 1;
                        if (mbar_test(&kv_full[st], par) && mbar_test(s_empty, (q & 1) ^ 1)) {
                            tc_fence_after();
                            const uint64_t bd = kdesc0 + (uint64_t)((st * kStage) >> 4);
                            const uint32_t sa = tmem + kColS, qa = tmem + kColQ;
#pragma unroll
                            for (int p = 0; p < NQP_MAX; ++p) {
                                if (p < nqp) {
#pragma unroll
                                    for (int ks = 0; ks < 4; ++ks)
                                        umma_bf16_ta(sa, qa + p * 32 + ks * 8, bd + ((p * kPanel + ks * 32) >> 4), idesc_qk,
                                                     (p > 0 || ks > 0) ? 1u : 0u);
                                }
                            }
                            umma_commit(s_full);
                            ++nq;
                            moved = true;
                        }
                    }
                    if (np < nq) {
                        const uint32_t q = jb + np, st = q % NS;
                        if (mbar_test(p_full, q & 1)) {
                            tc_fence_after();
                            const uint64_t bd = vdesc0 + (uint64_t)((st * kStage) >> 4);
#pragma unroll
                            for (int kk = 0; kk < BK / 16; ++kk)
                                umma_bf16_ta(tmem + kColO, tmem + kColP + kk * 8, bd + ((kk * 16 * 128) >> 4), idesc_pv,
                                             (np > 0 || kk > 0) ? 1u : 0u);
                            umma_commit(p_empty);
                            umma_commit(&kv_empty[st]);
                            ++np;
                            moved = true;
                        }
                    }
                    // the wait limit is checked every 256 idle polls (the clock read is not free)
                    if (moved) {
                        t0 = 0;
                        idle = 0;
                    } else if (++idle == 256) {
                        idle = 0;
                        if (t0 == 0) {
                            t0 = global_ns();
                        } else if (global_ns() - t0 > kWaitLimitNs) {
                            set_error(err, RPA_DEV_ERR_TIMEOUT);
                            ok = false;
                        }
                    }
                }
                umma_commit(o_full);
                if (!ok) s_abort = 1;
            }
        } else if (warp == kSigW) {
            // ---------------- exchange signalling ----------------
            // once this CTA has read receive buffer rb of block q, tell the peer it may write
            // it again (block q+2); the release carries the readers' loads (cumulativity)
            if (lane == 0) {
                const uint32_t sfree_peer = mapa_shared(smem_u32(s_free), peer);
                const uint32_t pfree_peer = mapa_shared(smem_u32(p_free), peer);
                for (int j = 0; j < nb; ++j) {
                    const uint32_t q = jb + j, rb = q & 1, rp = (q >> 1) & 1;
                    if (!mbar_wait(&srecv_used[rb], rp, err)) {
                        s_abort = 1;
                        break;
                    }
                    mbar_arrive_cluster(sfree_peer + rb * 8);
                    if (!mbar_wait(&precv_used[rb], rp, err)) {
                        s_abort = 1;
                        break;
                    }
                    mbar_arrive_cluster(pfree_peer + rb * 8);
                }
            }
        } else {
            // ------- softmax: row = TMEM lane, warps w and w+4 take 32 of the 64 columns each -------
            const int quarter = warp & 3, half = warp >> 2;
            const int r = quarter * 32 + lane;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            const float scale = a.sm_scale, cap = a.soft_cap, c_log2 = a.sm_scale * kLog2e;
            const float cap_k2 = cap != 0.f ? 2.f * kLog2e / cap : 0.f;
            // rows 64*rank.. are owned here; `orow` is the row within the owned (or peer-owned) 64
            const bool owner = (quarter >> 1) == (int)rank;
            const int orow = (quarter & 1) * 32 + lane;
            const bool lead = (quarter & 1) == 0 && half == 0 && lane == 0;  // arms this role's receive barriers
            const uint32_t srecv_peer = mapa_shared(smem_u32(smem + kOffSRecv), peer);
            const uint32_t precv_peer = mapa_shared(smem_u32(smem + kOffPRecv), peer);
            const uint32_t srecv_full_peer = mapa_shared(smem_u32(srecv_full), peer);
            const uint32_t precv_full_peer = mapa_shared(smem_u32(precv_full), peer);
            bool ok = true;
            if (q_tma) {
                // Q slice by TMA, 64-row boxes of one 64-dim panel each, into the ring stages of
                // blocks jb+NS-2 and jb+NS-1 (five boxes a stage): the producers hold back from
                // those two stages until this CTA's softmax threads have moved the slice on.
                const uint32_t stA = (jb + NS - 2) % NS, stB = (jb + NS - 1) % NS;
                auto box_at = [&](int bi) -> uint8_t* {
                    return smem + kOffKV + (bi < 5 ? stA : stB) * kStage + (bi < 5 ? bi : bi - 5) * kPanel;
                };
                if (tid == 0) {
                    mbar_arrive_expect_tx(q_land, (uint32_t)nqp * 2 * kPanel);
                    for (int bi = 0; bi < 2 * nqp; ++bi) {
                        const int p = bi >> 1, y = qrow0 + (bi & 1) * 64;
                        if (rank == 0 && p == 4 && !(SPARSE && a.q))
                            tma_load_2d(smem_u32(box_at(bi)), &tm_qb, 0, y, q_land);
                        else
                            tma_load_2d(smem_u32(box_at(bi)), &tm_qa, lat_panel_col(rank, p), y, q_land);
                    }
                }
                if (!mbar_wait(q_land, iph, err)) {
                    s_abort = 1;
                    ok = false;
                }
                // this thread's row, half of its 16-byte chunks, four chunks (16 columns) a store;
                // 128-byte swizzle: chunk c of box row rr sits at slot c ^ (rr & 7)
                const int nch = nqp * 4, c0 = half * nch, rr = r & 63;
#pragma unroll
                for (int i = 0; i < 20; i += 4) {
                    if (i < nch) {
                        uint32_t v[16];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int c = c0 + i + u, p = c >> 3, cc = c & 7;
                            const int bi = 2 * p + (r >> 6);
                            const uint8_t* src = box_at(bi) + rr * 128 + ((cc ^ (rr & 7)) << 4);
                            const uint4 x = *reinterpret_cast<const uint4*>(src);
                            v[4 * u] = x.x;
                            v[4 * u + 1] = x.y;
                            v[4 * u + 2] = x.z;
                            v[4 * u + 3] = x.w;
                        }
                        tmem_st16_nowait(tmem + lane_off + kColQ + (c0 + i) * 4, v);
                    }
                }
                fence_proxy_async_smem();  // these reads before the producers' copies into the stages
                mbar_arrive(q_free);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(q_full);
            } else {
                // Q slice -> TMEM: this thread's row, half of its 16-byte chunks (8 dims = 4
                // columns each).  The previous item's MMAs have all completed (o_full).
                const int nch = nqp * 4, c0 = half * nch;
                const size_t qrow = (size_t)qrow0 + r;
                uint4 buf[20];
#pragma unroll
                for (int i = 0; i < 20; ++i) {
                    if (i < nch && !SPARSE && a.q_fp8) {  // fp8 queries: 8 bytes per chunk, widened
                        const int c = c0 + i, p = c >> 3, cc = c & 7;
                        const uint8_t* src = (rank == 0 && p == 4)
                                                 ? reinterpret_cast<const uint8_t*>(a.q_pe) + qrow * 64 + cc * 8
                                                 : reinterpret_cast<const uint8_t*>(a.ql_nope) + qrow * kLatDv +
                                                       lat_panel_col(rank, p) + cc * 8;
                        buf[i] = e4m3x8_to_bf16x8(__ldg(reinterpret_cast<const uint2*>(src)));
                    } else if (i < nch) {
                        const int c = c0 + i, p = c >> 3, cc = c & 7;
                        const __nv_bfloat16* src = (SPARSE && a.q) ? a.q + qrow * kLatDk + lat_panel_col(rank, p) + cc * 8
                                                   : (rank == 0 && p == 4) ? a.q_pe + qrow * 64 + cc * 8
                                                                           : a.ql_nope + qrow * kLatDv + lat_panel_col(rank, p) + cc * 8;
                        buf[i] = __ldg(reinterpret_cast<const uint4*>(src));
                    }
                }
#pragma unroll
                for (int i = 0; i < 20; i += 4) {
                    if (i < nch) {
                        const uint32_t v[16] = {buf[i].x,     buf[i].y,     buf[i].z,     buf[i].w,
                                                buf[i + 1].x, buf[i + 1].y, buf[i + 1].z, buf[i + 1].w,
                                                buf[i + 2].x, buf[i + 2].y, buf[i + 2].z, buf[i + 2].w,
                                                buf[i + 3].x, buf[i + 3].y, buf[i + 3].z, buf[i + 3].w};
                        tmem_st16_nowait(tmem + lane_off + kColQ + (c0 + i) * 4, v);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(q_full);
            }
            float m_use = -INFINITY, l_half = 0.f;
            // common tail of a block: once PV of the previous block is done with P and has
            // written O, rescale this row of O by f and store this row's P
            auto finish = [&](uint32_t q, const uint32_t (&pk)[16], float f) -> bool {
                if (!mbar_wait(p_empty, (q & 1) ^ 1, err)) return false;
                tc_fence_after();
                if (__any_sync(0xffffffffu, f != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        float o32[32];
                        const uint32_t col = kColO + half * 128 + c * 32;
                        tmem_ld32(tmem + lane_off + col, o32);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o32[i] *= f;
                        tmem_st32(tmem + lane_off + col, o32);
                    }
                }
                tmem_st16_nowait(tmem + lane_off + kColP + half * 16, pk);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(p_full);
                return true;
            };
            if (!owner) {
                // ---- helper rows (owned by the peer): send my partial S as soon as it exists,
                // then take the row's P and rescale factor back; block q+1's partial goes out
                // before block q's P is awaited, so neither CTA waits on a round trip ----
                auto send_s = [&](uint32_t q) -> bool {
                    const uint32_t rb = q & 1, rp = (q >> 1) & 1;
                    if (!mbar_wait(s_full, q & 1, err)) return false;
                    tc_fence_after();
                    float x[32];
                    tmem_ld32(tmem + lane_off + kColS + half * 32, x);
                    tc_fence_before();
                    mbar_arrive(s_empty);
                    if (!mbar_wait_cluster(&s_free[rb], rp ^ 1, err)) return false;  // the peer has read block q-2
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        st_async_v4(srecv_peer + rb * kSRecv + ((half * 8 + i) * 64 + orow) * 16, x[4 * i], x[4 * i + 1],
                                    x[4 * i + 2], x[4 * i + 3], srecv_full_peer + rb * 8);
                    return true;
                };
                if (nb > 0 && !send_s(jb)) ok = false;
                for (int j = 0; j < nb && ok; ++j) {
                    const uint32_t q = jb + j, rb = q & 1, rp = (q >> 1) & 1;
                    if (j + 1 < nb && !send_s(q + 1)) {
                        ok = false;
                        break;
                    }
                    if (lead) mbar_arrive_expect_tx(&precv_full[rb], kPRecv);  // phase of block q-2 consumed here
                    if (!mbar_wait_cluster(&precv_full[rb], rp, err)) {
                        ok = false;
                        break;
                    }
                    const uint8_t* pr = smem + kOffPRecv + rb * kPRecv;
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 v = *reinterpret_cast<const uint4*>(pr + ((half * 4 + i) * 64 + orow) * 16);
                        pk[4 * i] = v.x;
                        pk[4 * i + 1] = v.y;
                        pk[4 * i + 2] = v.z;
                        pk[4 * i + 3] = v.w;
                    }
                    const float f = reinterpret_cast<const float*>(pr + 2 * 4 * 64 * 16)[orow];
                    mbar_arrive(&precv_used[rb]);
                    if (!finish(q, pk, f)) {
                        ok = false;
                        break;
                    }
                }
            } else {
                // ---- owned rows: add the peer's partial, online softmax, P to the peer ----
                for (int j = 0; j < nb; ++j) {
                    const uint32_t q = jb + j, st = q % NS, par = (q / NS) & 1, rb = q & 1, rp = (q >> 1) & 1;
                    if (!mbar_wait(s_full, q & 1, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    float x[32];
                    tmem_ld32(tmem + lane_off + kColS + half * 32, x);
                    tc_fence_before();
                    mbar_arrive(s_empty);
                    if (lead) mbar_arrive_expect_tx(&srecv_full[rb], kSRecv);  // phase of block q-2 consumed here
                    if (!mbar_wait_cluster(&srecv_full[rb], rp, err)) {
                        ok = false;
                        break;
                    }
                    {
                        const uint8_t* sr = smem + kOffSRecv + rb * kSRecv;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float4 v = *reinterpret_cast<const float4*>(sr + ((half * 8 + i) * 64 + orow) * 16);
                            x[4 * i] += v.x;
                            x[4 * i + 1] += v.y;
                            x[4 * i + 2] += v.z;
                            x[4 * i + 3] += v.w;
                        }
                    }
                    mbar_arrive(&srecv_used[rb]);
                    // scale, soft cap, key validity
                    if (cap != 0.f) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) x[i] = soft_cap(x[i] * scale, cap, cap_k2) * kLog2e;
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) x[i] *= c_log2;
                    }
                    const int key0 = kb + j * BK + half * 32;
                    if (SPARSE) {
                        if (!mbar_wait(&vld_full[st], par, err)) {
                            ok = false;
                            break;
                        }
                        const uint8_t* vb = vld + st * BK + half * 32;
#pragma unroll
                        for (int i = 0; i < 32; ++i) x[i] = vb[i] ? x[i] : -INFINITY;
                    } else if (!(key0 >= wlo && key0 + 31 <= qpos && key0 + 31 < ke)) {
                        // a mild mask replaces a masked logit of a key in the range by mask_value
                        const float mrep = a.mask_value * kLog2e;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int key = key0 + i;
                            const bool vis = key <= qpos && key >= wlo;
                            x[i] = key < ke ? (vis ? x[i] : a.mask_mild ? mrep : -INFINITY) : -INFINITY;
                        }
                    }
                    float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int i = 0; i < 32; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], x[i]);
                    float* red_j = red + (q & 1) * 256;
                    red_j[half * 128 + r] = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
                    asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
                    const float mx = fmaxf(red_j[r], red_j[128 + r]);
                    float alpha = 1.f;
                    const bool had = m_use > -INFINITY;
                    const bool rescale = mx > m_use + 8.f;
                    if (rescale) {
                        alpha = fast_exp2(m_use - mx);
                        m_use = mx;
                    }
                    const float mu = m_use == -INFINITY ? 0.f : m_use;
                    float sum4[4] = {0.f, 0.f, 0.f, 0.f};
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float p0 = fast_exp2(x[2 * e] - mu), p1 = fast_exp2(x[2 * e + 1] - mu);
                        sum4[e & 3] += p0 + p1;
                        pk[e] = pack_bf16(p0, p1);
                    }
                    const float f = (rescale && had) ? alpha : 1.f;
                    l_half = l_half * alpha + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
                    if (!mbar_wait_cluster(&p_free[rb], rp ^ 1, err)) {  // the peer has read block q-2 out of it
                        ok = false;
                        break;
                    }
                    const uint32_t pdst = precv_peer + rb * kPRecv;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        st_async_u4(pdst + ((half * 4 + i) * 64 + orow) * 16,
                                    make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]),
                                    precv_full_peer + rb * 8);
                    if (half == 0) st_async_f32(pdst + 2 * 4 * 64 * 16 + orow * 4, f, precv_full_peer + rb * 8);
                    if (!finish(q, pk, f)) {
                        ok = false;
                        break;
                    }
                }
            }
            // ---- row statistics: owners reduce l over the pair and send (m, l) to the peer ----
            float l_run = 0.f;
            if (ok && nb > 0) {
                const uint32_t sph = nstat & 1;
                if (owner) {
                    float* red_l = red + ((jb + nb) & 1) * 256;
                    red_l[half * 128 + r] = l_half;
                    asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
                    l_run = red_l[r] + red_l[128 + r];
                    asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
                    if (half == 0)
                        st_async_v2(mapa_shared(smem_u32(smem + kOffStat + orow * 8), peer), m_use, l_run,
                                    mapa_shared(smem_u32(stat_full), peer));
                } else {
                    if (lead) mbar_arrive_expect_tx(stat_full, 64 * 8);
                    if (mbar_wait_cluster(stat_full, sph, err)) {
                        const float2 ml = *reinterpret_cast<const float2*>(smem + kOffStat + orow * 8);
                        m_use = ml.x;
                        l_run = ml.y;
                    } else {
                        ok = false;
                    }
                }
            }
            // ---- epilogue: this CTA's O half goes row-major through the idle key ring (16-byte
            // chunks XOR-swizzled by the row, so neither side conflicts), then out a row at a time,
            // 512 contiguous bytes a warp store.  Every softmax thread reaches the barrier.
            const bool eok = ok && mbar_wait(o_full, iph, err);
            if (!eok) s_abort = 1;
            const bool split = w.num_splits > 1;
            const bool f32 = SPARSE || split;  // fp32 rows (1 KB), else bf16 rows (512 bytes)
            const size_t pslot = (size_t)w.first_item + w.split;  // split: the group's slot plus the split
            uint8_t* tile = smem + kOffKV;
            if (eok) {
                tc_fence_after();
                const float inv = split ? 1.f : (l_run > 0.f ? 1.f / l_run : 0.f);
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    float o32[32];
                    tmem_ld32(tmem + lane_off + kColO + half * 128 + c * 32, o32);
                    if (f32) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int k = half * 32 + c * 8 + i;
                            *reinterpret_cast<float4*>(tile + r * 1024 + ((k ^ (r & 7)) << 4)) =
                                make_float4(o32[4 * i] * inv, o32[4 * i + 1] * inv, o32[4 * i + 2] * inv, o32[4 * i + 3] * inv);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int k = half * 16 + c * 4 + i;
                            *reinterpret_cast<uint4*>(tile + r * 512 + ((k ^ (r & 7)) << 4)) =
                                make_uint4(pack_bf16(o32[8 * i] * inv, o32[8 * i + 1] * inv), pack_bf16(o32[8 * i + 2] * inv, o32[8 * i + 3] * inv),
                                           pack_bf16(o32[8 * i + 4] * inv, o32[8 * i + 5] * inv), pack_bf16(o32[8 * i + 6] * inv, o32[8 * i + 7] * inv));
                        }
                    }
                }
                if (split && half == 0) {
                    a.partial_ml[(pslot * 128 + r) * 2] = m_use;
                    a.partial_ml[(pslot * 128 + r) * 2 + 1] = l_run;
                }
            }
            tc_fence_before();
            asm volatile("bar.sync 5, 256;" ::: "memory");
            // rows warp, warp + 8, ...: the lanes take consecutive chunks of a row
#pragma unroll 1
            for (int rr = warp; rr < 128; rr += 8) {
                if (h0 + rr >= H) continue;
                if (f32) {
                    float* dst = split ? a.partial_o + (pslot * 128 + rr) * kLatDv + rank * 256
                                       : a.out_f32 + ((size_t)w.seq * H + h0 + rr) * kLatDv + rank * 256;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int k = hh * 32 + lane;
                        reinterpret_cast<uint4*>(dst)[k] = *reinterpret_cast<const uint4*>(tile + rr * 1024 + ((k ^ (rr & 7)) << 4));
                    }
                } else {
                    __nv_bfloat16* dst = a.out_bf16 + ((size_t)t * H + h0 + rr) * kLatDv + rank * 256;
                    reinterpret_cast<uint4*>(dst)[lane] = *reinterpret_cast<const uint4*>(tile + rr * 512 + ((lane ^ (rr & 7)) << 4));
                }
            }
            fence_proxy_async_smem();  // the ring is refilled by TMA for the next item
        }
        jb += nb;
        ++items;
        if (nb > 0) ++nstat;
        __syncthreads();
        tc_fence_after();
        if (w.num_splits > 1 && !s_abort) {
            // the last CTA of this rank to finish a split group merges the group's halves
            volatile int& s_last = *reinterpret_cast<volatile int*>(smem + kOffItem + 48);
            __threadfence();
            __syncthreads();
            if (tid == 0) s_last = atomicAdd(&a.tickets[w.first_item * 2 + rank], 1) == w.num_splits - 1;
            __syncthreads();
            if (s_last) {
                __threadfence();
                const int ns = w.num_splits;
                const size_t ib = (size_t)w.first_item * 128;
                if (ns <= kMergeSplits) {
                    // merge, row-parallel: the key ring is idle between items and holds the
                    // weights [split][row]. Thread r < 128 owns row r: its splits' (m, l) loads in
                    // flight together, then the row's max, sum and each split's weight
                    float* wgt = reinterpret_cast<float*>(smem + kOffKV);
                    if (tid < 128) {
                        float M = -INFINITY;
#pragma unroll 4
                        for (int s0 = 0; s0 < ns; ++s0) M = fmaxf(M, __ldcg(a.partial_ml + (ib + (size_t)s0 * 128 + tid) * 2));
                        const float Mu = M == -INFINITY ? 0.f : M;
                        float L = 0.f;
#pragma unroll 4
                        for (int s0 = 0; s0 < ns; ++s0) {
                            const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.partial_ml + (ib + (size_t)s0 * 128 + tid) * 2));
                            const float e = fast_exp2(ml.x - Mu);
                            wgt[s0 * 128 + tid] = e;
                            L += e * ml.y;
                        }
                        const float inv = L > 0.f ? 1.f / L : 0.f;
                        for (int s0 = 0; s0 < ns; ++s0) wgt[s0 * 128 + tid] *= inv;
                    }
                    __syncthreads();
                    // O: this rank's [128 x 256] as 8192 float4 chunks (row c / 64, columns
                    // 4 (c % 64) of this rank's half); a thread takes eight chunks at a time, their
                    // eight loads of one split in flight together
                    constexpr int kPer = 8;
                    const int nthr = (int)blockDim.x;
                    for (int c0 = tid; c0 < 128 * 64; c0 += nthr * kPer) {
                        float4 acc[kPer];
#pragma unroll
                        for (int j = 0; j < kPer; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
                        for (int s0 = 0; s0 < ns; ++s0) {
                            float4 v[kPer];
#pragma unroll
                            for (int j = 0; j < kPer; ++j) {
                                const int c = c0 + j * nthr;
                                const bool in = c < 128 * 64;
                                const int rr = in ? c >> 6 : 0;
                                v[j] = in ? __ldcg(reinterpret_cast<const float4*>(a.partial_o + (ib + (size_t)s0 * 128 + rr) * kLatDv +
                                                                                   rank * 256 + (c & 63) * 4))
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
#pragma unroll
                            for (int j = 0; j < kPer; ++j) {
                                const int c = c0 + j * nthr;
                                const float f = wgt[s0 * 128 + (c < 128 * 64 ? c >> 6 : 0)];
                                acc[j].x += f * v[j].x;
                                acc[j].y += f * v[j].y;
                                acc[j].z += f * v[j].z;
                                acc[j].w += f * v[j].w;
                            }
                        }
#pragma unroll
                        for (int j = 0; j < kPer; ++j) {
                            const int c = c0 + j * nthr;
                            if (c >= 128 * 64) continue;
                            const int rr = c >> 6, col = (int)rank * 256 + (c & 63) * 4;
                            if (h0 + rr >= H) continue;
                            if (SPARSE) {
                                *reinterpret_cast<float4*>(a.out_f32 + ((size_t)w.seq * H + h0 + rr) * kLatDv + col) = acc[j];
                            } else {
                                *reinterpret_cast<uint2*>(a.out_bf16 + ((size_t)t * H + h0 + rr) * kLatDv + col) =
                                    make_uint2(pack_bf16(acc[j].x, acc[j].y), pack_bf16(acc[j].z, acc[j].w));
                            }
                        }
                    }
                    fence_proxy_async_smem();  // the ring is refilled by TMA for the next item
                } else {
                    // (more splits than the ring holds weights for) a warp per row at a time; each
                    // lane holds one split's (m, l) and two float4 of this rank's 256 output columns,
                    // four splits' loads in flight at once
                    const int cbase = (int)rank * 256 + lane * 4;
                    for (int rr = warp; rr < 128; rr += lat::kWarps) {
                        if (h0 + rr >= H) continue;
                        float M = -INFINITY;
                        for (int s0 = lane; s0 < ns; s0 += 32) M = fmaxf(M, __ldcg(a.partial_ml + ((ib + (size_t)s0 * 128 + rr) * 2)));
                        M = warp_max(M);
                        const float Mu = M == -INFINITY ? 0.f : M;
                        float L = 0.f;
                        for (int s0 = lane; s0 < ns; s0 += 32) {
                            const size_t base = (ib + (size_t)s0 * 128 + rr) * 2;
                            L += fast_exp2(__ldcg(a.partial_ml + base) - Mu) * __ldcg(a.partial_ml + base + 1);
                        }
                        L = warp_sum(L);
                        const float inv = L > 0.f ? 1.f / L : 0.f;
                        float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
                        for (int s0 = 0; s0 < ns; s0 += 32) {
                            // lane l: the factor of split s0 + l
                            const int sl = s0 + lane;
                            const float fl = sl < ns ? fast_exp2(__ldcg(a.partial_ml + (ib + (size_t)sl * 128 + rr) * 2) - Mu) * inv : 0.f;
                            const int cnt = min(32, ns - s0);
                            for (int j = 0; j < cnt; j += 4) {
                                float4 v[8];
                                float f[4];
    #pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    f[u] = __shfl_sync(0xffffffffu, fl, (j + u) & 31);
                                    const bool in = j + u < cnt;
                                    const float* po = a.partial_o + (ib + (size_t)(s0 + j + u) * 128 + rr) * kLatDv + cbase;
                                    v[2 * u] = in ? __ldcg(reinterpret_cast<const float4*>(po)) : make_float4(0.f, 0.f, 0.f, 0.f);
                                    v[2 * u + 1] = in ? __ldcg(reinterpret_cast<const float4*>(po + 128)) : make_float4(0.f, 0.f, 0.f, 0.f);
                                    if (!in) f[u] = 0.f;
                                }
    #pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    acc0.x += f[u] * v[2 * u].x;
                                    acc0.y += f[u] * v[2 * u].y;
                                    acc0.z += f[u] * v[2 * u].z;
                                    acc0.w += f[u] * v[2 * u].w;
                                    acc1.x += f[u] * v[2 * u + 1].x;
                                    acc1.y += f[u] * v[2 * u + 1].y;
                                    acc1.z += f[u] * v[2 * u + 1].z;
                                    acc1.w += f[u] * v[2 * u + 1].w;
                                }
                            }
                        }
                        if (SPARSE) {
                            float* o = a.out_f32 + ((size_t)w.seq * H + h0 + rr) * kLatDv + cbase;
                            *reinterpret_cast<float4*>(o) = acc0;
                            *reinterpret_cast<float4*>(o + 128) = acc1;
                        } else {
                            __nv_bfloat16* o = a.out_bf16 + ((size_t)t * H + h0 + rr) * kLatDv + cbase;
                            *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16(acc0.x, acc0.y), pack_bf16(acc0.z, acc0.w));
                            *reinterpret_cast<uint2*>(o + 128) = make_uint2(pack_bf16(acc1.x, acc1.y), pack_bf16(acc1.z, acc1.w));
                        }
                    }
                }
                if (tid == 0) a.tickets[w.first_item * 2 + rank] = 0;
            }
            __syncthreads();
        }
    }
    // drain the tensor core, then make sure the peer no longer touches this CTA's memory
    if (warp == kMmaW) {
        if (lane == 0) {
            umma_commit(fin);
            mbar_wait(fin, 0, err);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    __syncthreads();
    cluster_sync_all();
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 lat_tmap_encoder() {
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

// 2-D bf16 [rows][cols] with a row stride of `stride` elements; box {64, box_rows}, 128-byte swizzle.
static bool make_tmap_2d(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint64_t stride,
                         uint32_t box_rows) {
    auto enc = lat_tmap_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {stride * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The latent row [rows][lkv_pad] bf16 viewed as [panel (8)][rows][64]: dims {64, rows, 8},
// strides {row, 128 bytes}; box {64, 64 rows, 4 panels} lands as four [64 x 64] panels.
static bool make_tmap_panels(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t stride) {
    auto enc = lat_tmap_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {64, rows, kLatDv / 64};
    const cuuint64_t strides[2] = {stride * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)lat::BK, 4};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool SPARSE>
static cudaError_t launch_latent_tc(const LatentArgs& a, int num_sms, cudaStream_t stream) {
    using namespace lat;
    CUtensorMap kc, kr, kc3;
    memset(&kc, 0, sizeof kc);
    memset(&kr, 0, sizeof kr);
    memset(&kc3, 0, sizeof kc3);
    int kv_tma = 0, box_rows = 0;  // without usable key maps the register gather runs
    if (SPARSE) {
        // kv_tma 3: the fused latent rows [rows][row_stride] by 4-row TMA gathers of 64 columns
        const uint64_t rows = (uint64_t)a.total_num_pages * a.page_size;
        if (rows < 0x7fffffffull && make_tmap_2d(&kc, a.cache, a.row_stride, rows, a.row_stride, 1)) kv_tma = 3;
    } else {
        const int ps = a.page_size;
        box_rows = ps < BK ? ps : BK;
        if ((ps & (ps - 1)) == 0 && box_rows >= 8) {
            const uint64_t rows = (uint64_t)a.total_num_pages * ps;
            kv_tma = make_tmap_2d(&kc, a.cache_kv_c, a.lkv_pad, rows, a.lkv_pad, box_rows) &&
                     make_tmap_2d(&kr, a.cache_k_pe, a.r_pad, rows, a.r_pad, box_rows);
            // kv_tma 2: a block is one box per panel group (pages of at least a block)
            if (kv_tma && box_rows == BK && make_tmap_panels(&kc3, a.cache_kv_c, rows, a.lkv_pad)) kv_tma = 2;
        }
    }
    // Q slices by TMA (bf16 queries): [rows][512 or 576] and the rope part [rows][64], 64-row boxes
    CUtensorMap qa, qb;
    memset(&qa, 0, sizeof qa);
    memset(&qb, 0, sizeof qb);
    int q_tma = 0;
    {
        const uint64_t qrows = SPARSE ? (uint64_t)a.batch * a.num_queries * a.num_heads : (uint64_t)a.max_num_tokens * a.num_heads;
        if (qrows < 0x7fffffffull) {
            if (SPARSE && a.q)
                q_tma = make_tmap_2d(&qa, a.q, kLatDk, qrows, kLatDk, 64);
            else if (!a.q_fp8)
                q_tma = make_tmap_2d(&qa, a.ql_nope, kLatDv, qrows, kLatDv, 64) && make_tmap_2d(&qb, a.q_pe, 64, qrows, 64, 64);
        }
    }
    auto kern = latent_tc_kernel<SPARSE>;
    static int max_clusters = 0;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (max_clusters == 0) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(2 * (num_sms / 2));
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
        max_clusters = n > 0 ? n : 1;
    }
    cfg.gridDim = dim3(2 * max_clusters);
    ProfScope ps(SPARSE ? "sparse_attn" : "mla_attn", stream);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, kc, kr, kc3, qa, qb, kv_tma, box_rows, q_tma);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_mla_attention(const LatentArgs& a, int num_sms, cudaStream_t stream) {
    return launch_latent_tc<false>(a, num_sms, stream);
}
cudaError_t launch_sparse_attention(const LatentArgs& a, int num_sms, cudaStream_t stream) {
    return launch_latent_tc<true>(a, num_sms, stream);
}

}  // namespace rpa
