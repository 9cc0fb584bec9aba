// Persistent latent-space decode attention for CTA pairs (d_c > 256, bf16
// cache): the balanced plan.
//
// The arithmetic per tile is that of attn_tc.cu (same pair split of the score
// contraction and of O by latent channel, same fp16 partial-score exchange,
// online softmax in log2 units, P . V into tensor memory; "Why MLA and MTP
// Fight Each Other", section 4: each cache byte read once and used by both
// contractions).  What differs is the work: the grid is persist_groups x
// (128-row blocks) pairs, and each group takes an equal contiguous range of the
// batch's sequence tiles (sequences in batch order), so that every pair slot of
// the GPU streams the same number of tiles whatever the lengths.  A pair walks
// the sequences its range touches (work items), and its tiles run through the
// operand ring, the score exchange and the barrier phases without a break at
// item boundaries.
//
// Four epilogue warps (12-15, one per TMEM lane quadrant) take the item
// boundaries off the softmax warps: once an item's last score chain has run
// they load the next item's queries into tensor memory; once its last P . V
// has landed they drain O (normalised by the (m, l) the softmax warps leave in
// global scratch) and free O for the next item's first P . V.  A sequence that
// one range holds whole is written out directly.  The pieces of a sequence
// split between ranges (only a range's first and last items can be) are written
// normalised (bf16) with their (m, l), kept in L2 by an evict_last policy while
// the streamed cache goes in evict_first; the CTA that writes a sequence's last
// piece (per-sequence counters) owes its merge, which all 16 warps do once
// every item of the CTA is done, the pieces' rows staged in the idle operand
// ring by bulk copies:
//   M = max_s m_s,  w_s = l_s e^(m_s - M),  o = sum_s w_s o_s / sum_s w_s,
//   lse = M + ln sum_s w_s
// (each CTA of a pair merges its own half of the columns, relative to its own
// (m, l); the first CTA also writes lse).
#include <cuda_fp16.h>

#include "attn_common.cuh"
#include "attn_tc.cuh"
#include "common.cuh"
#include "launch.h"
#include "sm100.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace sm100;
using namespace attn;

constexpr int kPThreads = 512;  // softmax 0-7, producer 8, score MMAs 9, exchange 10, sums 11, epilogue 12-15
constexpr int kEpiWarp0 = 12;
constexpr uint32_t kBarEpi = 6;    // named barrier of the epilogue warps (128 threads)
constexpr uint32_t kBarMerge = 7;  // named barrier of the whole block, for the merges at the end
constexpr int kMergeBatch = 8;       // pieces whose (m, l) one thread loads at once
constexpr int kMergeRowsStep = 64;   // rows of a merge block (one piece's half of the 128)
constexpr uint64_t kMergeWaitNs = 1000000000ull;  // bound of a merge wave's wait for its copies
static_assert(kPThreads / 32 * 4 == kMergeRowsStep, "a merge step gives each warp 4 rows");
// Register split of the 512-thread launch (128 a thread): the softmax warpgroups
// take 152, the role and epilogue warpgroups 104 (2 x 128 x 152 + 2 x 128 x 104 =
// 65536, the launch's total).
constexpr int kPRegSoftmax = 152, kPRegOther = 104;
static_assert(2 * 128 * kPRegSoftmax + 2 * 128 * kPRegOther == 65536, "register split must equal the launch's total");

// A work item: tokens [t0, t1) of sequence b for this pair's row block, in
// ntiles 64-token tiles; S its first tile in the batch's tile order; out -1 when
// the item covers its sequence whole, else the pair's partial slot (0 / 1).
struct PItem {
    int b, L, t0, t1, ntiles, out;
    long long S, E;  // the sequence's tiles [S, E) in the batch's tile order
};
struct PWalk {
    int b;        // next sequence to look at
    long long S;  // its first tile
};

// The pieces' rows in the workspace: for each (pair, slot) 128 rows of d_c
// columns, stored as the first CTA's 128 x 256 block (its columns [0, 256)) and
// then the second CTA's 128 x (d_c - 256), so that a CTA's rows of a piece are
// contiguous (a merge fetches 64 of them with one bulk copy).  row0: the piece's
// first row ((pair * 2 + slot) * 128); row r of the CTA's block at + r * g.vn.
template <class T>
__device__ __forceinline__ T *piece_rows(T *part16, long long row0, int d_c, uint32_t rank) {
    return part16 + row0 * d_c + (long long)rank * kRows * 256;
}

// Bounded wait for a merge wave's copies (global to this CTA's shared memory,
// so they end by themselves; the bound does not give up on an abort, as no copy
// may still be landing when the CTA exits).
__device__ __forceinline__ void merge_wait(Smem &sm, const AttnParams &p, uint32_t parity) {
    if (mbar_try_wait(&sm.merge_full, parity)) return;
    const uint64_t t0 = globaltimer_ns();
    const long long c0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(&sm.merge_full, parity)) return;
        if ((it & 63u) == 0 && (globaltimer_ns() - t0 > kMergeWaitNs || clock64() - c0 > 2 * (long long)kMergeWaitNs)) {
            set_status(p.status, MLA_ERR_TIMEOUT);
            return;
        }
    }
}

// The merges this CTA owes, once every warp has left its role (all 512 threads
// call this).  A merge works in blocks of 64 rows of one piece (half h of the
// 128 rows, piece j; h-major): each block's rows (this CTA's latent columns) and
// its rows' (m, l) come into the idle operand ring by bulk copies, as many
// blocks at once as the ring holds (one barrier phase a wave).  While the first
// wave lands, one thread a row finds M = max_s m_s and 1 / sum_s l_s e^(m_s - M)
// over the pieces (the first CTA also writes lse).  Warp w then adds rows
// 4w..4w+3 of each block, weighted by l_s e^(m_s - M) / sum, with its lanes along
// the latent columns, and writes a half's rows once its last piece is in.
__device__ __forceinline__ void merge_pending(Smem &sm, const AttnParams &p, const Geo &g, uint32_t rank, int rb,
                                              int n_rb, int G, long long T, int rows_total) {
    named_bar(kBarMerge, kPThreads);  // every item of every warp done: the list is complete, the ring idle
    const int npend = sm.n_pending;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const __nv_bfloat16 *part16 = reinterpret_cast<const __nv_bfloat16 *>(p.part_acc);
    float2 *row_ms = reinterpret_cast<float2 *>(sm.rx[0]);  // [row]: M, 1 / sum
    float4 *blk_ml = reinterpret_cast<float4 *>(sm.rx[1]);  // [block of the wave][row]: (m, l) of both CTAs
    const uint32_t row_bytes = (uint32_t)g.vn * 2;
    const int wave = min((int)(sizeof(sm.kv) / (kMergeRowsStep * row_bytes)),
                         (int)(sizeof(sm.rx[1]) / (kMergeRowsStep * sizeof(float4))));
    uint8_t *stage = &sm.kv[0][0];
    uint32_t phase = 0;
    for (int q = 0; q < npend; ++q) {
        const int b = sm.pend_b[q];
        const long long S = sm.pend_S[q];
        const int L = __ldg(p.seq_lens + b);
        const long long E = S + (seq_len_ok(p, L) ? (L + kTile - 1) / kTile : 0);
        const int g0r = group_of_tile(S, G, T);
        const int np = group_of_tile(E - 1, G, T) - g0r + 1;
        // first row (over the pieces' [pair][slot][row] layout) of piece j
        auto piece_row = [&](int j) -> long long {
            const int gg = g0r + j;
            return ((long long)(gg * n_rb + rb) * 2 + persist_slot(S, gg, G, T)) * kRows;
        };
        const int nblocks = 2 * np;
        float acc[4][8];
        for (int w0 = 0; w0 < nblocks; w0 += wave) {
            const int nb = min(wave, nblocks - w0);
            if (threadIdx.x == 0) {
                uint32_t bytes = 0;
                for (int bi = w0; bi < w0 + nb; ++bi) {
                    const int rows_here = max(0, min(kMergeRowsStep, rows_total - (rb * kRows + (bi / np) * kMergeRowsStep)));
                    bytes += (uint32_t)rows_here * (row_bytes + (uint32_t)sizeof(float4));
                }
                mbar_arrive_expect_tx(&sm.merge_full, bytes);
            }
            named_bar(kBarMerge, kPThreads);  // the ring and the (m, l) buffer are free again
            if (threadIdx.x < nb) {  // one thread a block: its rows are contiguous, one copy each
                const int slot = threadIdx.x;
                const int bi = w0 + slot, h = (bi / np) * kMergeRowsStep, j = bi % np;
                const int rows_here = max(0, min(kMergeRowsStep, rows_total - (rb * kRows + h)));
                const long long pr0 = piece_row(j);
                if (rows_here > 0) {
                    bulk_load(stage + (size_t)slot * kMergeRowsStep * row_bytes, piece_rows(part16, pr0, p.d_c, rank) + (long long)h * g.vn,
                              (uint32_t)rows_here * row_bytes, &sm.merge_full);
                    bulk_load(blk_ml + slot * kMergeRowsStep, p.part_ml + (pr0 + h) * 4, (uint32_t)rows_here * sizeof(float4),
                              &sm.merge_full);
                }
            }
            if (w0 == 0 && threadIdx.x < kRows) {  // under the first wave's copies
                const int r = threadIdx.x;
                float M = -INFINITY, Ls = 0.f;
                for (int j0 = 0; j0 < np; j0 += kMergeBatch) {
                    float mv[kMergeBatch], lv[kMergeBatch];
#pragma unroll
                    for (int j = 0; j < kMergeBatch; ++j) {
                        mv[j] = -INFINITY;
                        lv[j] = 0.f;
                        if (j0 + j < np) {
                            const long long pr = piece_row(j0 + j) + r;
                            mv[j] = __ldcg(p.part_ml + (pr * 2 + rank) * 2);
                            lv[j] = __ldcg(p.part_ml + (pr * 2 + rank) * 2 + 1);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < kMergeBatch; ++j) {
                        if (mv[j] == -INFINITY) continue;
                        const float Mn = fmaxf(M, mv[j]);
                        Ls = Ls * __expf(M - Mn) + lv[j] * __expf(mv[j] - Mn);
                        M = Mn;
                    }
                }
                row_ms[r] = make_float2(M, Ls > 0.f ? 1.f / Ls : 0.f);
                const int gr = rb * kRows + r;
                if (rank == 0 && gr < rows_total)
                    p.lse[(long long)b * rows_total + gr] = Ls > 0.f ? M + __logf(Ls) : -INFINITY;
            }
            named_bar(kBarMerge, kPThreads);  // the rows' (M, 1 / sum) are in
            merge_wait(sm, p, phase & 1);
            ++phase;
            for (int slot = 0; slot < nb; ++slot) {
                const int bi = w0 + slot, h = (bi / np) * kMergeRowsStep, j = bi % np;
                const int rows_here = max(0, min(kMergeRowsStep, rows_total - (rb * kRows + h)));
                if (j == 0) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
                }
                if (lane * 8 < g.vn) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int rr = warp * 4 + i;
                        if (rr >= rows_here) continue;
                        const float4 ml = blk_ml[slot * kMergeRowsStep + rr];
                        const float m = rank == 0 ? ml.x : ml.z, l = rank == 0 ? ml.y : ml.w;
                        // a piece with no visible token never wrote its rows: weight 0, rows unread
                        if (m == -INFINITY) continue;
                        const float2 ms = row_ms[h + rr];
                        const float w = l * __expf(m - ms.x) * ms.y;
                        const uint4 v =
                            *reinterpret_cast<const uint4 *>(stage + (size_t)(slot * kMergeRowsStep + rr) * row_bytes + lane * 16);
                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[e]));
                            acc[i][2 * e] += w * f.x;
                            acc[i][2 * e + 1] += w * f.y;
                        }
                    }
                }
                if (j == np - 1 && lane * 8 < g.vn) {  // the half's last piece: its rows are done
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int rr = warp * 4 + i;
                        if (rr >= rows_here) continue;
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) pk[e] = pack_bf16x2(acc[i][2 * e], acc[i][2 * e + 1]);
                        const long long gr = rb * kRows + h + rr;
                        *reinterpret_cast<uint4 *>(p.o_lat + ((long long)b * rows_total + gr) * p.d_c + g.k0 + lane * 8) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
            }
        }
    }
    named_bar(kBarMerge, kPThreads);  // the last wave's reads of the ring and of the (m, l) are done
}

template <bool kPaged>
__global__ void __launch_bounds__(kPThreads, 1)
    attn_persist(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1, const AttnParams p,
                 const Geo g0, const Geo g1) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // the swizzled operand tiles need a 1 KB boundary
        if (threadIdx.x == 0) set_status(p.status, MLA_ERR_UNSUPPORTED);
        return;
    }
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (p.pdl) pdl_launch_dependents();
    const uint32_t rank = cluster_rank();
    const uint32_t peer = rank ^ 1u;
    const Geo g = rank == 0 ? g0 : g1;
    const CUtensorMap *tm = rank == 0 ? &tm0 : &tm1;
    const int rows_total = p.s_q * p.H;
    const int n_rb = (rows_total + kRows - 1) / kRows;
    const int pair = blockIdx.x / 2;
    const int rb = pair % n_rb, grp = pair / n_rb;
    const int q_last_rb = min(p.s_q - 1, ((rb + 1) * kRows - 1) / p.H);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.q_ready, kSoftmaxThreads);
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_free, kSoftmaxThreads);
        mbar_init(&sm.p_ready, kSoftmaxThreads);
        mbar_init(&sm.o_done, 1);
        mbar_init(&sm.drain, 2);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.staged[i], kSoftmaxThreads);
            mbar_init(&sm.rx_full[i], 1);
            mbar_init(&sm.ml_ready[i], kSoftmaxThreads);
        }
        mbar_init(&sm.q_next, 128);
        mbar_init(&sm.s_last, 1);
        mbar_init(&sm.o_last, 1);
        mbar_init(&sm.o_free, 128);
        mbar_init(&sm.merge_full, 1);
        for (int q = 0; q < 4; ++q) sm.pair_stop[q][0] = sm.pair_stop[q][1] = 0;
        sm.abort = 0;
        sm.wait_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
        sm.armed = sm.received = -1;
        sm.n_pending = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm0);
        tma_prefetch_desc(&tm1);
    }
    if (warp == kMmaWarp) tmem_alloc<512>(&sm.tmem_base);
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    // Every CTA computes the batch's tile prefix (sequence b has ceil(L_b / 64)
    // tiles, none if its length lies outside [s_q, capacity]) in the staging
    // buffer, idle until the first tile: a run of sequences per thread, the runs'
    // totals scanned by warp shuffles and then over the warps.
    {
        int *pre = reinterpret_cast<int *>(sm.tx[0]);   // B + 1 entries (the host keeps B below 4096)
        int *wsum = reinterpret_cast<int *>(sm.tx[1]);  // one total per warp
        const int nt = blockDim.x;
        const int per = (p.B + nt - 1) / nt;
        const int lo = min(p.B, (int)threadIdx.x * per), hi = min(p.B, lo + per);
        int mine = 0;
        for (int c = lo; c < hi; ++c) {
            const int Lc = __ldg(p.seq_lens + c);
            const int tc = seq_len_ok(p, Lc) ? (Lc + kTile - 1) / kTile : 0;
            if (tc == 0 && pair == 0 && rank == 0) set_status(p.status, MLA_ERR_SEQLEN);
            pre[c] = tc;
            mine += tc;
        }
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        int before = 0;
        for (int k = 0; k < warp; ++k) before += wsum[k];
        if (threadIdx.x == nt - 1) pre[p.B] = before + incl;
        int run = before + incl - mine;
        for (int c = lo; c < hi; ++c) {
            const int v = pre[c];
            pre[c] = run;
            run += v;
        }
        __syncthreads();
    }
    const int *pre = reinterpret_cast<const int *>(sm.tx[0]);
    const long long T = pre[p.B];
    const int G = persist_groups(p.persist_groups, T);
    long long R0 = 0, R1 = 0;  // this group's range of tiles
    if (grp < G && T > 0) {
        R0 = group_first_tile(grp, G, T);
        R1 = group_first_tile(grp + 1, G, T);
    }
    if (threadIdx.x == 0) {
        // the last sequence starting at or before R0 holds it (sequences without
        // tiles start where the next one does and are passed over by the walk)
        int lo_b = 0, hi_b = p.B - 1;
        while (lo_b < hi_b) {
            const int mid = (lo_b + hi_b + 1) / 2;
            if (pre[mid] <= R0) lo_b = mid;
            else hi_b = mid - 1;
        }
        sm.walk_b = lo_b;
        sm.walk_S = pre[lo_b];
    }
    if (pair == 0 && rank == 0)  // the merges and the host read the prefix from the workspace
        for (int c = threadIdx.x; c <= p.B; c += blockDim.x) p.prefix[c] = pre[c];
    __syncthreads();
    const PWalk walk0 = {sm.walk_b, sm.walk_S};
    auto next_item = [&](PWalk &w, PItem &it) -> bool {
        while (w.b < p.B && w.S < R1) {
            const int bb = w.b;
            const int L = __ldg(p.seq_lens + bb);
            const int tiles = seq_len_ok(p, L) ? (L + kTile - 1) / kTile : 0;
            const long long S = w.S;
            w.S += tiles;
            ++w.b;
            const long long a = max(R0, S), e = min(R1, S + tiles);
            if (e <= a) continue;
            it.b = bb;
            it.L = L;
            it.S = S;
            it.E = S + tiles;
            it.t0 = (int)(a - S) * kTile;
            const int t1 = min(L, (int)(e - S) * kTile);
            it.t1 = max(it.t0, min(t1, L - p.s_q + q_last_rb + 1));  // no row of the block sees past this
            it.ntiles = (it.t1 - it.t0 + kTile - 1) / kTile;
            it.out = (a == S && e == S + tiles) ? -1 : persist_slot(S, grp, G, T);
            return true;
        }
        return false;
    };
    int total_tiles = 0;
    {
        PWalk w = walk0;
        PItem it;
        while (next_item(w, it)) total_tiles += it.ntiles;
    }
    auto row_index = [&](int bb, int gr) -> long long { return (long long)bb * rows_total + gr; };

    if (warp >= kSoftmaxWarps) {
    regs_dec<kPRegOther>();
    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        // The tiles of all items stream through the ring without a break (n: the
        // tile's position over all of them, which fixes its stage and phase).
        if (lane == 0) {
            const uint64_t pol_stream = l2_evict_first();
            int issued = 0;
            bool go = true;
            PWalk w = walk0;
            PItem it;
            int n = 0;
            int next_page = 0;  // paged: the block-table entry of the item's next tile
            while (go && next_item(w, it)) {
                for (int i = 0; i < it.ntiles; ++i, ++n) {
                    const int s = n % kRing;
                    // The first tile goes out at once, the rest of the ring only after the
                    // first item's queries are in (without a preceding grid, every CTA
                    // starts at once and its whole ring would queue in HBM ahead of them).
                    if (n == 1 && i == 1 && !p.pdl && !wait_bar(sm, &sm.q_ready, 0)) {
                        raise_abort<true>(sm, p, peer);
                        go = false;
                        break;
                    }
                    if (n >= kRing && !wait_bar(sm, &sm.empty[s], ((n / kRing) - 1) & 1)) {
                        raise_abort<true>(sm, p, peer);
                        go = false;
                        break;
                    }
                    // this tile's page id was looked up while the loop waited for its stage
                    int y, z;
                    bool page_ok = true;
                    if (kPaged) {
                        const int tok = it.t0 + i * kTile;
                        const int page = i == 0 ? __ldg(p.block_table + (long long)it.b * p.max_pages + tok / p.page_size)
                                                : next_page;
                        page_ok = page >= 0 && page < p.num_pages;
                        y = page * p.page_size + tok % p.page_size;
                        z = 0;
                    } else {
                        y = it.t0 + i * kTile;
                        z = it.b;
                    }
                    if (!page_ok) {
                        set_status(p.status, MLA_ERR_PAGE);
                        y = p.num_pages * p.page_size;  // wholly out of range: the box reads as zeros
                    }
                    mbar_arrive_expect_tx(&sm.full[s], g.nbox * kBoxBytes);
                    for (int bx = 0; bx < g.nbox; ++bx) {  // each cache line is read once: first out of L2
                        if (kPaged) tma_load_2d_hint(sm.kv[s] + bx * kBoxBytes, tm, &sm.full[s], g.k0 + 64 * bx, y, pol_stream);
                        else tma_load_3d_hint(sm.kv[s] + bx * kBoxBytes, tm, &sm.full[s], g.k0 + 64 * bx, y, z, pol_stream);
                    }
                    issued = n + 1;
                    if (kPaged && i + 1 < it.ntiles)
                        next_page = __ldg(p.block_table + (long long)it.b * p.max_pages + (it.t0 + (i + 1) * kTile) / p.page_size);
                    // eight tiles before an item ends, the next item's queries go to L2 for
                    // the epilogue warps that load them at the hand-over
                    if (i == max(0, it.ntiles - 8)) {
                        PWalk w2 = w;
                        PItem nx;
                        while (next_item(w2, nx)) {
                            if (nx.ntiles == 0) continue;
                            const int QW = p.d_c + p.d_rope;
                            const int nrows = min(kRows, rows_total - rb * kRows);
                            const uint8_t *q0 = reinterpret_cast<const uint8_t *>(p.q_cat + row_index(nx.b, rb * kRows) * QW);
                            const uint32_t bytes = (uint32_t)nrows * QW * 2;
                            for (uint32_t o = 0; o < bytes; o += 16384) prefetch_l2_bulk(q0 + o, min(16384u, bytes - o));
                            break;
                        }
                    }
                }
            }
            const int first = issued > kRing ? issued - kRing : 0;
            for (int m = first; m < issued; ++m) mbar_wait(&sm.full[m % kRing], (m / kRing) & 1);
        }
    } else if (warp == kMmaWarp || warp == kSumWarp) {
        // ------------------------------------------------------------ MMA issuers
        // Scores (warp 9): each item's chains wait for its queries (the first
        // item's from the softmax warps, q_ready; later ones from the epilogue
        // warps, one q_next phase per item); the item's last chain also completes
        // s_last.  Sums (warp 11): an item's first P . V starts O afresh, once the
        // epilogue warps have drained the previous item's (o_free); its last also
        // completes o_last.
        const bool scores = warp == kMmaWarp;
        const uint32_t idesc_qk = idesc_of<false>(kRows, kTile, false, false);
        const uint32_t idesc_pv = idesc_of<false>(kRows, g.vn, false, true);
        const uint64_t qk_desc0 = smem_desc_sw128(smem_u32(sm.kv[0]), 16, 1024);
        const uint64_t pv_desc0 = smem_desc_sw128(smem_u32(sm.kv[0]), kBoxBytes, 1024);
        const int nks = g.sw / 16;
        bool ok = true;
        PWalk w = walk0;
        PItem it;
        int n = 0, k = 0;
        while (ok && next_item(w, it)) {
            if (it.ntiles == 0) continue;
            if (scores && !(k == 0 ? warp_wait(sm, &sm.q_ready, 0) : warp_wait(sm, &sm.q_next, (k - 1) & 1))) {
                ok = false;
                break;
            }
            for (int i = 0; i < it.ntiles; ++i, ++n) {
                const int s = n % kRing;
                const bool last = i + 1 == it.ntiles;
                if (scores) {
                    if (!warp_wait(sm, &sm.full[s], (n / kRing) & 1) || (n > 0 && !warp_wait(sm, &sm.s_free, (n - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    // tokens at or past the sequence end may hold anything (even NaN): zero
                    // them so that 0-weight products stay 0
                    const int valid = min(kTile, it.L - (it.t0 + i * kTile));
                    if (valid < kTile) {
                        for (int e = lane; e < (kTile - valid) * 8 * g.nbox; e += 32) {
                            const int bx = e / ((kTile - valid) * 8);
                            const int rr = valid + (e / 8) % (kTile - valid);
                            reinterpret_cast<uint4 *>(sm.kv[s] + bx * kBoxBytes + rr * 128)[e % 8] = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint64_t db = qk_desc0 + (uint64_t)((s * kStageBytes) >> 4);
                        const uint32_t d_s = tmem + kColS, a_q = tmem + kColQ;
#pragma unroll
                        for (int ks = 0; ks < kMaxBoxes * 4; ++ks)
                            if (ks < nks)
                                mma_ts(d_s, a_q + ks * 8, db + (uint64_t)(((ks >> 2) * kBoxBytes + (ks & 3) * 32) >> 4),
                                       idesc_qk, ks > 0);
                        mma_commit(&sm.s_full);
                        if (last) mma_commit(&sm.s_last);
                    }
                } else {
                    if (!warp_wait(sm, &sm.p_ready, n & 1) || (i == 0 && k > 0 && !warp_wait(sm, &sm.o_free, (k - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint64_t db = pv_desc0 + (uint64_t)((s * kStageBytes) >> 4);
#pragma unroll
                        for (int kt = 0; kt < kTile / 16; ++kt)
                            mma_ts(tmem + kColO, tmem + kColP + kt * 8, db + (uint64_t)(kt * (16 * 128 / 16)), idesc_pv,
                                   (i > 0) || kt > 0);
                        mma_commit(&sm.o_done);
                        mma_commit(&sm.empty[s]);
                        if (last) mma_commit(&sm.o_last);
                    }
                }
                __syncwarp();
            }
            ++k;
        }
        if (!ok) raise_abort<true>(sm, p, peer);
        if (lane == 0) mma_commit(&sm.drain);
        __syncwarp();
        mbar_wait(&sm.drain, 0);
        __syncwarp();
    } else if (warp == kExchangeWarp) {
        // ------------------------------------------------------------ score exchange
        // As in attn_tc.cu, over the tiles of all items: ship each staged tile of
        // partial scores to the peer with one bulk copy, arming this CTA's own
        // receive of the tile first.
        if (lane == 0) {
            const uint32_t rx_peer0 = map_to_rank(smem_u32(sm.rx[0]), peer);
            const uint32_t rxfull_peer0 = map_to_rank(smem_u32(&sm.rx_full[0]), peer);
            for (int u = 0; u < total_tiles; ++u) {
                const int pb = u & 1;
                if (!wait_bar(sm, &sm.staged[pb], (u >> 1) & 1)) {
                    raise_abort<true>(sm, p, peer);
                    break;
                }
                mbar_arrive_expect_tx(&sm.rx_full[pb], kXBytes);
                *(volatile int *)&sm.armed = u;
                bulk_copy_to_peer(rx_peer0 + pb * (uint32_t)sizeof(sm.rx[0]), sm.tx[pb], kXBytes,
                                  rxfull_peer0 + pb * (uint32_t)sizeof(uint64_t));
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue warps (12-15)
        // Warp 12 + q owns TMEM lane quadrant q: row r = 32 q + lane, all of this
        // CTA's latent columns.
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const int gr = rb * kRows + r;
        const bool in_rows = gr < rows_total;
        const uint32_t lane_base = tmem_lane_base(quad);
        const float scale_log2 = p.scale * 1.4426950408889634f;
        const int W = p.d_c + p.d_rope;
        const float ln2 = 0.6931471805599453f;
        __nv_bfloat16 *const part16 = reinterpret_cast<__nv_bfloat16 *>(p.part_acc);
        const int et = threadIdx.x - kEpiWarp0 * 32;  // 0..127
        if (p.pdl) pdl_wait();

        // sequences without tiles (length out of range) get zero rows and lse -inf,
        // written by the pairs of group 0, each its row block and half
        if (grp == 0) {
            for (int bb = 0; bb < p.B; ++bb) {
                const int Lb = __ldg(p.seq_lens + bb);
                if (seq_len_ok(p, Lb) || !in_rows) continue;
                uint4 *dst = reinterpret_cast<uint4 *>(p.o_lat + row_index(bb, gr) * p.d_c + g.k0);
                for (int v = 0; v < g.vn / 8; ++v) dst[v] = make_uint4(0, 0, 0, 0);
                if (rank == 0) p.lse[row_index(bb, gr)] = -INFINITY;
            }
        }

        // this thread's query row of item bq -> TMEM (pre-scaled), 96 channels a round
        // (12 loads in flight): the first round's loads go out before the wait for
        // the item's last score chain, as they do not touch TMEM
        constexpr int kQRound = 96;
        uint4 qin[kQRound / 8];
        auto q_fetch = [&](int bq, int c0) {
            const __nv_bfloat16 *src = p.q_cat + row_index(bq, in_rows ? gr : 0) * W + g.qk0;
#pragma unroll
            for (int j = 0; j < kQRound / 8; ++j) {
                const int c = c0 + 8 * j;
                qin[j] = (in_rows && c < g.sw && g.qk0 + c < W) ? *reinterpret_cast<const uint4 *>(src + c)
                                                                : make_uint4(0, 0, 0, 0);
            }
        };
        auto q_put = [&](int c0) {
#pragma unroll
            for (int s4 = 0; s4 < kQRound / 32; ++s4) {
                if (c0 + 32 * s4 >= g.sw) break;
                uint32_t v[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 u = qin[4 * s4 + j];
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[e]));
                        v[4 * j + e] = pack_bf16x2(f.x * scale_log2, f.y * scale_log2);
                    }
                }
                tmem_st16(tmem + lane_base + kColQ + (c0 + 32 * s4) / 2, v);
            }
        };

        bool ok = true;
        int k = 0;  // items with tiles so far
        PWalk w = walk0;
        PItem it;
        while (ok && next_item(w, it)) {
            const long long prow = ((long long)pair * 2 + (it.out < 0 ? 0 : it.out)) * kRows + r;
            if (it.ntiles > 0) {
                PWalk w2 = w;
                PItem nx;
                bool has_nx = false;
                while (next_item(w2, nx))
                    if (nx.ntiles > 0) {
                        has_nx = true;
                        break;
                    }
                // A wait that runs out fails this warp's item (nothing more of it is
                // done); the four warps agree below and leave together, so that none is
                // left at a barrier the others have passed.
                bool fail = false;
                if (has_nx) {  // the next item's queries, once this item's last score chain has run
                    q_fetch(nx.b, 0);
                    fail = !warp_wait(sm, &sm.s_last, k & 1);
                    if (!fail) {
                        tc_fence_after();
                        q_put(0);
                        for (int c0 = kQRound; c0 < g.sw; c0 += kQRound) {
                            q_fetch(nx.b, c0);
                            q_put(c0);
                        }
                        tmem_st_wait();
                        tc_fence_before();
                        mbar_arrive(&sm.q_next);
                    }
                }
                fail = fail || !warp_wait(sm, &sm.o_last, k & 1) || !warp_wait(sm, &sm.ml_ready[k & 1], (k >> 1) & 1);
                if (named_bar_or(kBarEpi, 128, fail)) {
                    raise_abort<true>(sm, p, peer);
                    ok = false;
                    break;
                }
                tc_fence_after();
                // written by this CTA's softmax warps in this launch: plain (not read-only) loads
                const volatile float *ml = p.ml + ((((long long)pair * 2 + rank) * 2 + (k & 1)) * kRows + r) * 3;
                const float m2 = ml[0], l_row = ml[1] + ml[2];
                const bool any = l_row > 0.f;
                const float inv = any ? 1.f / l_row : 0.f;
                __nv_bfloat16 *dst = it.out < 0 ? p.o_lat + row_index(it.b, gr) * p.d_c + g.k0
                                                : piece_rows(part16, prow - r, p.d_c, rank) + (long long)r * g.vn;
                for (int c = 0; c < g.vn; c += 32) {
                    uint32_t u[2][16];
#pragma unroll
                    for (int j = 0; j < 2; ++j) tmem_ld16(tmem + lane_base + kColO + c + 16 * j, u[j]);
                    tmem_ld_wait();
                    if (in_rows) {
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            uint32_t o8[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                o8[e] = pack_bf16x2(__uint_as_float(u[j][2 * e]) * inv, __uint_as_float(u[j][2 * e + 1]) * inv);
                            // pieces stay in L2 for the merge (evict_last); sequences held whole leave as usual
                            const uint64_t pol = it.out < 0 ? l2_evict_normal() : l2_evict_last();
                            uint4 *d4 = reinterpret_cast<uint4 *>(dst + c + 16 * j);
                            st_global_hint(d4, make_uint4(o8[0], o8[1], o8[2], o8[3]), pol);
                            st_global_hint(d4 + 1, make_uint4(o8[4], o8[5], o8[6], o8[7]), pol);
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&sm.o_free);  // the next item's first P . V may overwrite O
                if (in_rows) {
                    if (it.out < 0) {
                        if (rank == 0) p.lse[row_index(it.b, gr)] = any ? (m2 + __log2f(l_row)) * ln2 : -INFINITY;
                    } else {
                        st_global_hint(p.part_ml + (prow * 2 + rank) * 2 + 0, any ? m2 * ln2 : -INFINITY, l2_evict_last());
                        st_global_hint(p.part_ml + (prow * 2 + rank) * 2 + 1, any ? l_row : 0.f, l2_evict_last());
                    }
                }
                ++k;
            } else if (in_rows) {  // an empty piece (the causal limit cut its tiles): all in its (m, l)
                st_global_hint(p.part_ml + (prow * 2 + rank) * 2 + 0, -INFINITY, l2_evict_last());
                st_global_hint(p.part_ml + (prow * 2 + rank) * 2 + 1, 0.f, l2_evict_last());
            }
            if (it.out < 0) continue;
            // A piece of a sequence split between ranges: count it; the CTA that writes
            // the last one (for its half of the columns) owes the merge, done once all
            // of its items are (merge_pending).
            const int g0r = group_of_tile(it.S, G, T), g1r = group_of_tile(it.E - 1, G, T);
            __threadfence();
            named_bar(kBarEpi, 128);
            if (et == 0) {
                const int old = atomicAdd(p.counters + ((long long)it.b * n_rb + rb) * 2 + rank, 1);
                if (old == g1r - g0r && sm.n_pending < 2) {
                    sm.pend_b[sm.n_pending] = it.b;
                    sm.pend_S[sm.n_pending] = it.S;
                    ++sm.n_pending;
                }
            }
        }
        if (!ok) raise_abort<true>(sm, p, peer);
        tc_fence_before();
    }
    merge_pending(sm, p, g, rank, rb, n_rb, G, T, rows_total);

    } else {
        regs_inc<kPRegSoftmax>();
        // ------------------------------------------------------------ softmax
        const int quad = warp & 3, hf = warp >> 2;
        const int r = quad * 32 + lane;  // this thread's row == TMEM lane
        const int gr = rb * kRows + r;
        const bool in_rows = gr < rows_total;
        const int qi = in_rows ? gr / p.H : 0;
        const int q_first = (rb * kRows) / p.H;  // the block's earliest query
        const uint32_t lane_base = tmem_lane_base(quad);
        const float scale_log2 = p.scale * 1.4426950408889634f;
        const int W = p.d_c + p.d_rope;
        const uint32_t pair_bar = kBarPairBase + quad;
        const int sw = r & 7;  // chunk swizzle of this row in tx / rx
        const uint32_t s_addr = tmem + lane_base + kColS + kHalf * hf;
        if (p.pdl) pdl_wait();  // q_cat comes from the grid this one overlaps

        // The first item's queries -> TMEM, pre-multiplied by scale * log2(e), as in
        // attn_tc.cu: each warp reads 8 rows x 64 contiguous bytes per instruction
        // and turns them row-per-lane through its 2 KB of the idle staging buffer.
        auto load_q = [&](int bq) {
            const int lr = lane >> 2, lj = lane & 3;
            const __nv_bfloat16 *src[4];
            bool src_ok[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int gq = rb * kRows + quad * 32 + 8 * k + lr;
                src_ok[k] = gq < rows_total;
                src[k] = p.q_cat + (src_ok[k] ? row_index(bq, gq) * W : 0);
            }
            uint4 qv[kMaxBoxes][4];
#pragma unroll
            for (int i = 0; i < kMaxBoxes; ++i) {
                const int c = 32 * hf + 64 * i + lj * 8;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    qv[i][k] = make_uint4(0, 0, 0, 0);
                    if (src_ok[k] && c < g.sw && g.qk0 + c < W) qv[i][k] = *reinterpret_cast<const uint4 *>(src[k] + g.qk0 + c);
                }
            }
            uint8_t *slot = reinterpret_cast<uint8_t *>(sm.tx[0]) + warp * 2048;
#pragma unroll
            for (int i = 0; i < kMaxBoxes; ++i) {
                const int c0 = 32 * hf + 64 * i;
                if (c0 >= g.sw) break;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int R = 8 * k + lr;
                    *reinterpret_cast<uint4 *>(slot + R * 64 + ((lj ^ ((R >> 1) & 3)) << 4)) = qv[i][k];
                }
                __syncwarp();
                uint32_t v[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(slot + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4));
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[e]));
                        v[j * 4 + e] = pack_bf16x2(f.x * scale_log2, f.y * scale_log2);
                    }
                }
                __syncwarp();
                tmem_st16(tmem + lane_base + kColQ + c0 / 2, v);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.q_ready);
        };
        auto stage = [&](int u, const float (&sp)[kHalf]) {
            uint32_t h16[kHalf / 2];
#pragma unroll
            for (int j = 0; j < kHalf / 2; ++j) h16[j] = pack_f16x2(sp[2 * j], sp[2 * j + 1]);
            uint4 *txrow = reinterpret_cast<uint4 *>(sm.tx[u & 1] + r * kTile);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                txrow[(4 * hf + c) ^ sw] = make_uint4(h16[4 * c], h16[4 * c + 1], h16[4 * c + 2], h16[4 * c + 3]);
            fence_proxy_async_smem();
            mbar_arrive(&sm.staged[u & 1]);
        };

        {  // the first item with tiles: its queries, before the loop over items
            PWalk w1 = walk0;
            PItem f;
            while (next_item(w1, f))
                if (f.ntiles > 0) {
                    load_q(f.b);
                    break;
                }
        }
        bool ok = true;
        int n = 0, k = 0;  // tiles and items with tiles so far
        PWalk w = walk0;
        PItem it;
        while (ok && next_item(w, it)) {
            if (it.ntiles == 0) continue;
            const int L = it.L;
            const int lim = L - p.s_q + qi;  // last visible token of this row
            float m2 = -INFINITY, l = 0.f;
            float sc[kHalf];
            {
                float s0[kHalf];
                if (!warp_wait(sm, &sm.s_full, n & 1)) raise_abort<true>(sm, p, peer);
                tc_fence_after();
                load_scores(s_addr, s0);
                tc_fence_before();
                mbar_arrive(&sm.s_free);
                stage(n, s0);
#pragma unroll
                for (int j = 0; j < kHalf; ++j) sc[j] = s0[j];
            }
            // paged: the block-table entry of the current tile, loaded one tile ahead
            int page_cur = kPaged ? __ldg(p.block_table + (long long)it.b * p.max_pages + it.t0 / p.page_size) : 0;
            for (int i = 0; i < it.ntiles; ++i, ++n) {
                float sn[kHalf];
                const bool more = i + 1 < it.ntiles;
                const int page_n = page_cur;
                if (kPaged && more)
                    page_cur = __ldg(p.block_table + (long long)it.b * p.max_pages + (it.t0 + (i + 1) * kTile) / p.page_size);
                if (more) {
                    if (!warp_wait(sm, &sm.s_full, (n + 1) & 1)) raise_abort<true>(sm, p, peer);
                    tc_fence_after();
                    load_scores(s_addr, sn);
                    tc_fence_before();
                    mbar_arrive(&sm.s_free);
                }
                float x[kHalf];
                if (warp_wait<true>(sm, &sm.rx_full[n & 1], (n >> 1) & 1)) {
                    if (threadIdx.x == 0) *(volatile int *)&sm.received = n;
                } else {
                    raise_abort<true>(sm, p, peer);
                }
                const uint4 *rxrow = reinterpret_cast<const uint4 *>(sm.rx[n & 1] + r * kTile);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 v = rxrow[(4 * hf + c) ^ sw];
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        x[8 * c + 2 * e] = sc[8 * c + 2 * e];
                        x[8 * c + 2 * e + 1] = sc[8 * c + 2 * e + 1];
                        add_f16x2_to(w4[e], x[8 * c + 2 * e], x[8 * c + 2 * e + 1]);
                    }
                }
                if (more) stage(n + 1, sn);
#pragma unroll
                for (int j = 0; j < kHalf; ++j) sc[j] = sn[j];
                // mask (only tiles that reach past a limit) and half-row maximum
                const int tok0 = it.t0 + i * kTile;
                bool tile_ok = true;
                if (kPaged) tile_ok = page_n >= 0 && page_n < p.num_pages;
                const bool whole = tile_ok && tok0 + kTile <= it.t1 && tok0 + kTile - 1 <= L - p.s_q + q_first;
                float mx0 = -INFINITY, mx1 = -INFINITY;
                if (whole) {
#pragma unroll
                    for (int j = 0; j < kHalf; j += 2) {
                        mx0 = fmaxf(mx0, x[j]);
                        mx1 = fmaxf(mx1, x[j + 1]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < kHalf; ++j) {
                        const int tok = tok0 + kHalf * hf + j;
                        const bool vis = tile_ok && in_rows && tok < it.t1 && tok <= lim;
                        x[j] = vis ? x[j] : -INFINITY;
                        mx0 = fmaxf(mx0, x[j]);
                    }
                }
                sm.pair[n & 1][hf][r] = fmaxf(mx0, mx1);
                if (hf == 0 && lane == 0) sm.pair_stop[quad][n & 1] = *(volatile int *)&sm.abort;
                named_bar(pair_bar, 64);
                if (*(volatile int *)&sm.pair_stop[quad][n & 1]) {
                    ok = false;
                    break;
                }
                const float tmax = fmaxf(sm.pair[n & 1][0][r], sm.pair[n & 1][1][r]);
                float m_use = m2, alpha = 1.f;
                bool rescale = false;
                if (tmax > m2 + kRescaleLog2 || (m2 == -INFINITY && tmax > -INFINITY)) {
                    m_use = tmax;
                    if (m2 != -INFINITY) {
                        alpha = ex2(m2 - m_use);
                        rescale = true;
                    }
                }
                float sum0 = 0.f, sum1 = 0.f;
                uint32_t pk[16];
                if (m_use == -INFINITY) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) pk[j] = 0u;
                } else {
#pragma unroll
                    for (int j = 0; j < kHalf; j += 2) {
                        const float a = ex2(x[j] - m_use);
                        const float c = ex2(x[j + 1] - m_use);
                        sum0 += a;
                        sum1 += c;
                        pk[j / 2] = pack_bf16x2(a, c);
                    }
                }
                l = l * alpha + (sum0 + sum1);
                m2 = m_use;
                // the previous P . V (of this item, or the last of the previous one) must
                // be done before O is rescaled or P overwritten
                if (n >= 1) {
                    if (!warp_wait(sm, &sm.o_done, (n - 1) & 1)) raise_abort<true>(sm, p, peer);
                    tc_fence_after();
                }
                if (i >= 1 && __any_sync(0xffffffffu, rescale)) {
                    if (!rescale) alpha = 1.f;
                    const int half_cols = g.vn / 2;
                    for (int c = half_cols * hf; c < half_cols * (hf + 1); c += 16) {
                        uint32_t u[16];
                        tmem_ld16(tmem + lane_base + kColO + c, u);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
                        tmem_st16(tmem + lane_base + kColO + c, u);
                    }
                }
                tmem_st16(tmem + lane_base + kColP + 16 * hf, pk);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&sm.p_ready);
            }
            // this row half's (m, l) for the epilogue warps (m2 is the same in both halves)
            float *ml = p.ml + ((((long long)pair * 2 + rank) * 2 + (k & 1)) * kRows + r) * 3;
            if (hf == 0) ml[0] = m2;
            ml[1 + hf] = l;
            mbar_arrive(&sm.ml_ready[k & 1]);
            ++k;
        }
        tc_fence_before();
        merge_pending(sm, p, g, rank, rb, n_rb, G, T, rows_total);
    }

    __syncthreads();
    // no incoming copy may land in this CTA's shared memory after it exits
    if (threadIdx.x == 0) {
        for (int u = *(volatile int *)&sm.received + 1; u <= *(volatile int *)&sm.armed; ++u)
            mbar_wait(&sm.rx_full[u & 1], (u >> 1) & 1);
    }
    cluster_sync();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_free<512>(tmem);
    }
}

}  // namespace

// The balanced plan's launch: persist_groups x (128-row blocks) CTA pairs (see
// the file comment), dense bf16 caches at d_c > 256, B below 4096.
cudaError_t launch_attn_persist(const AttnParams &p, cudaStream_t st) {
    const int W = p.d_c + p.d_rope;
    if (p.d_c <= 256 || p.kv_fp8 || p.indices != nullptr || p.B >= 4096 || p.persist_groups < 1)
        return cudaErrorNotSupported;
    const Geo g0 = make_geo(p, 0, true), g1 = make_geo(p, 1, true);
    if (g0.nbox > kMaxBoxes || g1.nbox > kMaxBoxes || g0.kw % 16 || g1.kw % 16) return cudaErrorNotSupported;
    CUtensorMap tm;
    if (p.block_table) {
        uint64_t dims[2] = {(uint64_t)W, (uint64_t)p.num_pages * p.page_size};
        uint64_t strides[1] = {(uint64_t)W * 2};
        uint32_t box[2] = {64, kTile};
        if (!encode_bf16_sw128(&tm, p.kv, 2, dims, strides, box)) return cudaErrorInvalidValue;
    } else {
        uint64_t dims[3] = {(uint64_t)W, (uint64_t)p.capacity, (uint64_t)p.B};
        uint64_t strides[2] = {(uint64_t)W * 2, (uint64_t)p.seq_stride * 2};
        uint32_t box[3] = {64, kTile, 1};
        if (!encode_bf16_sw128(&tm, p.kv, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    const int smem = (int)sizeof(Smem);
    auto kern = p.block_table ? attn_persist<true> : attn_persist<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // the register split hands out exactly the registers of a 128-per-thread launch
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || fa.numRegs != 128) return cudaErrorNotSupported;
    const int n_rb = (p.s_q * p.H + kRows - 1) / kRows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * n_rb * p.persist_groups, 1, 1);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, tm, tm, p, g0, g1);
}

}  // namespace mla
