// Latent-space decode attention on the tcgen05 tensor cores.
//
// One work item = (sequence b, history split, block of 128 query rows), where
// rows r = i*H + h run over the s_q new tokens and the H heads.  The latent
// cache is streamed in 64-token tiles [c_kv | k_rope] by TMA, each byte read
// from HBM once and used by both contractions ("Why MLA and MTP Fight Each
// Other", section 4: the fused, streaming condition; "MLA, dim by dim", "MLA
// Decode": stream the cache blocks, online softmax, accumulate p.C):
//   S   = q_cat . tile^T             (M=128 rows, N=64 tokens, K = d_c + d_rope)
//   P   = exp(scale*S - m)           online softmax, causal among the s_q queries
//   O  += P . tile[:, 0:d_c]         (M=128, N = d_c slice, K = 64 tokens)
//
// The fp32 accumulator of 128 rows x 512 latent columns would fill all of an
// SM's tensor memory, so when d_c > 256 a cluster of two CTAs shares the work
// item: CTA 0 owns latent columns [0, 256), CTA 1 owns [256, d_c) plus the RoPE
// key.  Each CTA loads only its own channel slice of every tile and computes
// the partial score over that slice; the pair swaps partial scores (sent as
// fp16) with one bulk shared-memory copy per tile and direction, and each CTA
// adds the peer's to its own fp32 partial.  Each CTA then runs the softmax of
// all rows and accumulates its half of O; its running (m, l) describe that half
// (the two CTAs' scores differ only by the fp16 rounding of the other CTA's
// partial, so split partials carry one (m, l) per CTA).  The swap of tile n+1
// is in flight while tile n's softmax runs.  Send and receive buffers are
// double (by tile parity), and a CTA stages tile n+1 only after it has
// received and consumed the peer's tile n.  That order frees both buffers
// without a signal across the cluster: the peer shipped its tile n only after
// consuming this CTA's tile n-1, whose copy had therefore finished reading the
// staging buffer that tile n+1 now takes (a copy into the peer completes on
// the peer's barrier alone), and the peer ships tile n+2 into a receive buffer
// only after receiving tile n+1, which this CTA stages after consuming tile n.
// (Staging tile n+1 before waiting for the peer's tile n, with a "consumed"
// signal across the cluster, measured slower: the softmax of tile n, on which
// the operand ring waits, then starts later.)
//
// Three ways of feeding the tensor cores.
//  - Dense bf16 cache: the producer's TMA tile loads write the 128-byte-swizzled
//    operand tiles straight into a 4-stage ring.
//  - Sparse lists over a bf16 cache: the listed rows are gathered straight into
//    the same 4-stage ring by two engines at once -- the producer's
//    tile::gather4 copies (four rows of one 128-byte box per copy) take the
//    leading boxes of a row, and four loader warps the last two with 16-byte
//    cp.async copies, on both CTAs of a pair (the one with the RoPE key's fifth
//    box gathers three) (the tensor-memory-access unit alone moves one 4-row box in
//    about 70 cycles, too slow for 80 boxes a tile).  Entries that take no part
//    are gathered from row -1, which the copy engine fills with zeros.
//  - FP8 caches: the producer copies each tile's row-major E4M3 codes into the
//    top of the operand stage the tile will occupy -- one TMA copy per tile
//    (dense), or one tile::gather4 copy per 4 listed rows (sparse), each moving
//    this CTA's whole channel slice of a row as 32-bit elements -- and four
//    converter warps rewrite the stage in place as swizzled fp16 tiles (the
//    codes are exact in fp16), zeroing the rows that take no part.  The warps
//    first load all their codes into registers and wait until every converter
//    has, then store, so no code is overwritten before it is read; the 4-stage
//    ring and the shared-memory footprint stay those of the bf16 kernel.  The
//    MMAs run in fp16 (Q, P and the tile) and the cache's scale is folded into
//    Q's pre-scale and into the final normalisation.
//
// Tensor memory (512 columns): O [0, 256), S [256, 320), P (16-bit) [320, 352),
// Q slice (16-bit, the A operand of the score MMA) [352, 512).
// Warps 0-7: softmax and epilogue, two warps per TMEM lane quadrant (warp w
// owns rows 32*(w%4) .. +31 and token columns 32*(w/4) .. +31 of each tile);
// warp 8: TMA producer; warp 9: TMEM owner, issues the score MMAs; warp 10:
// ships the staged partial scores to the peer; warp 11: issues the sum MMAs;
// warps 12-15: converters (FP8) or loaders (bf16 sparse).
// Every wait is bounded; a lost wait records MLA_ERR_TIMEOUT, drains what is in
// flight, and the CTA returns.
//
// Work order (grid z): item z is sequence z, piece blockIdx.y of num_splits; with
// a tail (tail_splits > 1) items past tail_b0 are the pieces of the last
// sequences, so that they fill the last wave; with the longest-first order (dense
// bf16) item positions map to sequences by rank of length, every CTA ranking
// the lengths itself.  Around the tile loop: the producer holds the ring after
// the first tile until the queries are in (no preceding grid), the queries load
// coalesced and turn row-per-lane through shared memory, and O leaves through a
// shared-memory copy as whole-row stores.
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory"); }

// Four E4M3 codes (the bytes of u, lowest first) as four fp16 values (two
// f16x2 words); every E4M3 value is an fp16 number, so this is exact.
__device__ __forceinline__ uint2 e4m3x4_to_f16x4(uint32_t u) {
    uint2 r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(r.x), "=r"(r.y)
        : "r"(u));
    return r;
}

// Converter warp cw (of kNConv) turns its share of a raw FP8 tile (64 rows of
// `pitch` bytes) into the fp16 operand stage.  Input chunk f of the tile (16
// codes: row f / ncin, codes 16 (f % ncin) ..) becomes output chunks 2 (f % ncin)
// and 2 (f % ncin) + 1 of that row (8 fp16 each); output chunk c of row r lands
// at chunk (c % 8) ^ (r % 8) of row r of box c / 8.  The warp's input chunks are
// all loaded first, so the loads overlap; `all_read()` then waits until every
// converter holds its codes (the raw tile lies inside the stage being written)
// and, if it returns false, nothing is stored.  Rows whose bit in vmask is
// clear are written as zeros.
template <int kNConv, class AllRead>
__device__ __forceinline__ void convert_fp8_tile(uint8_t *dst, const uint8_t *src, int pitch, int ncin,
                                                 unsigned long long vmask, int cw, int lane, AllRead &&all_read) {
    constexpr int kMax = kTile * 20 / (32 * kNConv);  // input chunks per lane at 320 codes a row
    const int per = kTile * ncin / kNConv;             // input chunks of this warp
    // f / ncin through a float reciprocal: (f + 0.5) / ncin is at least 0.5 / 20
    // away from an integer and the product errs by less than 1280 * 2^-23, so the
    // truncation is the exact quotient (a division would cost a loop per chunk)
    const float inv = 1.0f / (float)ncin;
    auto row_of = [&](int i) { return (int)(((float)(cw * per + lane + 32 * i) + 0.5f) * inv); };
    uint4 in[kMax];
#pragma unroll
    for (int i = 0; i < kMax; ++i) {
        const int r = row_of(i), c = cw * per + lane + 32 * i - r * ncin;
        in[i] = make_uint4(0, 0, 0, 0);
        if (lane + 32 * i < per && ((vmask >> r) & 1ull)) in[i] = *reinterpret_cast<const uint4 *>(src + r * pitch + c * 16);
    }
    if (!all_read()) return;
#pragma unroll
    for (int i = 0; i < kMax; ++i) {
        if (lane + 32 * i < per) {
            const int r = row_of(i), c = cw * per + lane + 32 * i - r * ncin;
            const uint2 a = e4m3x4_to_f16x4(in[i].x), b = e4m3x4_to_f16x4(in[i].y);
            const uint2 d = e4m3x4_to_f16x4(in[i].z), e = e4m3x4_to_f16x4(in[i].w);
            const int o0 = 2 * c, sw = r & 7;
            uint8_t *row = dst + (o0 >> 3) * kBoxBytes + r * 128;
            *reinterpret_cast<uint4 *>(row + (((o0 & 7) ^ sw) << 4)) = make_uint4(a.x, a.y, b.x, b.y);
            *reinterpret_cast<uint4 *>(row + ((((o0 & 7) + 1) ^ sw) << 4)) = make_uint4(d.x, d.y, e.x, e.y);
        }
    }
}

// Dense FP8 tiles arrive box by box: the 64 codes of each row of box b (64
// channels) land, 64 rows x 64 B, in the upper half of the box's own 8 KB output
// region.  convert_fp8_rows turns rows [r0, r0 + 16 * kRowGroups) of such a raw
// box into the swizzled fp16 box: raw chunk c (16 codes) of row r becomes output
// chunks 2c and 2c + 1 of row r, at chunks (2c) ^ (r % 8) and (2c + 1) ^ (r % 8).
// Lane l takes raw chunk l % 4 of row r0 + l / 4 (+ 8 per step): two
// neighbouring rows land in disjoint bank groups, so the stores do not conflict.
// All loads come first; `all_read()` then returns whether to store (the raw box
// lies inside the output box).  Rows whose bit in vmask is clear become zeros.
template <int kRowGroups, class AllRead>
__device__ __forceinline__ void convert_fp8_rows(uint8_t *box, int r0, unsigned long long vmask, int lane,
                                                 AllRead &&all_read) {
    constexpr int kSteps = kRowGroups * 2;  // 8 rows per step
    const uint8_t *raw = box + 4096;
    uint4 in[kSteps];
#pragma unroll
    for (int i = 0; i < kSteps; ++i) {
        const int r = r0 + 8 * i + (lane >> 2), c = lane & 3;
        in[i] = ((vmask >> r) & 1ull) ? *reinterpret_cast<const uint4 *>(raw + r * 64 + c * 16) : make_uint4(0, 0, 0, 0);
    }
    if (!all_read()) return;
#pragma unroll
    for (int i = 0; i < kSteps; ++i) {
        const int r = r0 + 8 * i + (lane >> 2), c = lane & 3, sw = r & 7;
        const uint2 a = e4m3x4_to_f16x4(in[i].x), b = e4m3x4_to_f16x4(in[i].y);
        const uint2 d = e4m3x4_to_f16x4(in[i].z), e = e4m3x4_to_f16x4(in[i].w);
        uint8_t *row = box + r * 128;
        *reinterpret_cast<uint4 *>(row + (((2 * c) ^ sw) << 4)) = make_uint4(a.x, a.y, b.x, b.y);
        *reinterpret_cast<uint4 *>(row + (((2 * c + 1) ^ sw) << 4)) = make_uint4(d.x, d.y, e.x, e.y);
    }
}

// bf16 sparse: 128-byte boxes of a row the producer gathers (tile::gather4);
// the loader warps copy the last two, so both CTAs of a pair load the same.
__device__ __forceinline__ int tma_boxes_of(const Geo &g) { return min(g.nbox, max(kTmaBoxes, g.nbox - 2)); }

template <bool kSplit, bool kPaged, bool kSparse, bool kFp8>
__global__ void __launch_bounds__(threads_of(kSparse, kFp8), 1)
    attn_tc(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1, const AttnParams p,
            const Geo g0, const Geo g1) {
    constexpr bool kStaged = kFp8;                // converter warps
    constexpr bool kLoaders = kSparse && !kFp8;   // loader warps share the gather
    constexpr int kMma = kMmaWarp;
    constexpr int kExch = kExchangeWarp;
    constexpr int kNConv = kStaged ? kFp8ConvWarps : kConvWarps;
    constexpr bool kRegSplit = threads_of(kSparse, kFp8) == 512;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the launch reserves no slack for realignment (the block is within a few
    // hundred bytes of the limit): a window that does not start on a 1 KB
    // boundary (the swizzled operand tiles need one) is reported, not used;
    // both CTAs of a pair see the same offset, so both leave here
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) set_status(p.status, MLA_ERR_UNSUPPORTED);
        return;
    }
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (p.pdl) pdl_launch_dependents();
    const uint32_t rank = kSplit ? cluster_rank() : 0;
    const uint32_t peer = rank ^ 1u;
    const Geo g = rank == 0 ? g0 : g1;
    const CUtensorMap *tm = rank == 0 ? &tm0 : &tm1;
    const int rb = kSplit ? blockIdx.x / 2 : blockIdx.x;
    // work item -> sequence, piece of it and the sequence's piece count; part_seq
    // indexes the sequence's partials
    int split = blockIdx.y, b = blockIdx.z, nsplit = p.num_splits, part_seq = blockIdx.z;
    if (p.tail_splits > 1 && b >= p.tail_b0) {
        const int i = b - p.tail_b0;
        nsplit = p.tail_splits;
        split = i % nsplit;
        part_seq = i / nsplit;
        b = p.tail_b0 + part_seq;
    }
    // longest-first order (dense bf16 variants only: compiled into the 512-thread
    // FP8 kernel it cost 3 %): every length is requested now and used after the
    // setup below, which hides the load
    constexpr bool kOrdered = !kFp8 && !kSparse;
    const bool lpt = kOrdered && p.lpt;
    constexpr int kLensPerThread = 3;  // 3 x 384 threads >= 1024 sequences
    int lens_reg[kLensPerThread];
#pragma unroll
    for (int k = 0; k < kLensPerThread; ++k) {
        const int c = threadIdx.x + k * blockDim.x;
        lens_reg[k] = lpt && c < p.B ? __ldg(p.seq_lens + c) : 0;
    }
    // expanded attention: work-item sequence b is head hsub of sequence bseq
    const int hps = p.heads_per_seq > 1 ? p.heads_per_seq : 1;
    const int L_pre = lpt ? 0 : __ldg(p.seq_lens + b / hps);  // the sequence's length, likewise early

    if (threadIdx.x == 0) {
        // the loaders of a CTA whose slice has no box past the gathered ones stay idle
        const bool loading = kLoaders && g.nbox > tma_boxes_of(g);
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&sm.full[s], kStaged ? kNConv : (loading ? 1 + kConvWarps : 1));
            mbar_init(&sm.empty[s], 1);
        }
        if constexpr (kStaged) {
            for (int s = 0; s < kRing; ++s) {
                mbar_init(&sm.landed[s], 1);
                mbar_init(&sm.read[s], kNConv);
            }
        }
        mbar_init(&sm.q_ready, kSoftmaxThreads);
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_free, kSoftmaxThreads);
        mbar_init(&sm.p_ready, kSoftmaxThreads);
        mbar_init(&sm.o_done, 1);
        mbar_init(&sm.drain, 2);  // one commit from each MMA issuer
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.staged[i], kSoftmaxThreads);
            mbar_init(&sm.rx_full[i], 1);
        }
        for (int q = 0; q < 4; ++q) sm.pair_stop[q][0] = sm.pair_stop[q][1] = 0;
        sm.abort = 0;
        sm.wait_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
        sm.armed = sm.received = -1;
        fence_mbar_init();
        tma_prefetch_desc(&tm0);
        if (kSplit) tma_prefetch_desc(&tm1);
    }
    if (warp == kMma) tmem_alloc<512>(&sm.tmem_base);
    tc_fence_before();
    if (kSplit) cluster_sync();
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    if (lpt) {
        // longest first: position b of the work order is the sequence of rank b by
        // (length descending, index ascending), so that over several waves the long
        // sequences start first and the short ones fill in behind them; every CTA
        // ranks the lengths itself (B is small: the host enables this up to 1024)
        int *lens = reinterpret_cast<int *>(sm.tx[0]);
#pragma unroll
        for (int k = 0; k < kLensPerThread; ++k) {
            const int c = threadIdx.x + k * blockDim.x;
            if (c < p.B) lens[c] = lens_reg[k];
        }
        __syncthreads();
        for (int c = threadIdx.x; c < p.B; c += blockDim.x) {
            const int lc = lens[c];
            int r = 0;
            for (int d = 0; d < p.B; ++d) r += (lens[d] > lc) || (lens[d] == lc && d < c);
            if (r == b) {
                sm.lpt_b = c;
                sm.lpt_L = lc;
            }
        }
        __syncthreads();
        // the merge of split pieces finds a position's sequence here
        if (p.order != nullptr && threadIdx.x == 0 && rb == 0 && split == 0 && rank == 0) p.order[b] = sm.lpt_b;
        b = sm.lpt_b;
    }
    const int rows_total = p.s_q * p.H;
    const int bseq = b / hps, hsub = b % hps;
    auto row_index = [&](int gr) -> long long { return ((long long)bseq * rows_total + gr) * hps + hsub; };

    const int L = lpt ? sm.lpt_L : L_pre;
    const bool seq_ok = seq_len_ok(p, L);
    // [t0, t1): token positions (dense) or positions in the sparse list
    int t0 = 0, t1 = 0;
    if (seq_ok) split_range(kSparse ? p.topk : L, nsplit, split, t0, t1);
    if (!kSparse && seq_ok) {
        // no row of this block sees a token past its last query's causal limit:
        // those tiles are not streamed at all (with many new tokens -- a prefill --
        // this halves the work)
        const int q_last = min(p.s_q - 1, ((rb + 1) * kRows - 1) / p.H);
        t1 = max(t0, min(t1, L - p.s_q + q_last + 1));
    }
    const int ntiles = (t1 - t0 + kTile - 1) / kTile;
    if (!seq_ok && split == 0 && rb == 0 && rank == 0 && threadIdx.x == 0) set_status(p.status, MLA_ERR_SEQLEN);

    if (warp >= kSoftmaxWarps) {
        if constexpr (kRegSplit) regs_dec<kRegOther>();
        if (warp == kProducerWarp && kSparse) {
            // ------------------------------------------------------------ producer, sparse
            // Tile n = listed entries e = t0 + 64 n + r.  The whole warp resolves them
            // (lanes r and r + 32): an entry takes part if it names a token this row
            // block's query may see, 0 <= j <= L - s_q + i (all rows of a block share
            // i), on a page inside the pool.  Lanes 0-15 then gather rows 4q .. 4q+3
            // with tile::gather4: FP8, the whole slice of each row into the raw ring;
            // bf16, the first tma_boxes_of(g) 128-byte boxes of each row into the operand
            // stage (the loader warps copy the rest).  Entries that take no part are
            // gathered from row -1, which reads as zeros.  The next tile's entries are
            // loaded one tile ahead, so their latency hides behind the wait for a
            // free stage.
            const int W = p.d_c + p.d_rope;
            const int iq = (rb * kRows) / p.H;
            const int lim = L - p.s_q + iq;
            const int *list = p.indices + ((long long)b * p.s_q + iq) * p.topk;
            const long long seq_rows = p.seq_stride / W;  // contiguous: rows between sequences
            const int nbt = kLoaders ? tma_boxes_of(g) : min(g.nbox, kTmaBoxes);
            auto fetch = [&](int n, int (&j)[2]) {
    #pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int e = t0 + n * kTile + lane + 32 * h2;
                    j[h2] = (n < ntiles && e < t1) ? __ldg(list + e) : -1;
                }
            };
            int nxt[2];
            fetch(0, nxt);
            int issued = 0;
            for (int n = 0; n < ntiles; ++n) {
                const int s = n % kRing;
                const int cur[2] = {nxt[0], nxt[1]};
                fetch(n + 1, nxt);
                if (n >= kRing && !warp_wait(sm, &sm.empty[s], ((n / kRing) - 1) & 1)) {
                    if (lane == 0) raise_abort<kSplit>(sm, p, peer);
                    break;
                }
                int rows[2];
                bool vis[2];
    #pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int j = cur[h2];
                    vis[h2] = j >= 0 && j <= lim;
                    long long row = -1;
                    if (vis[h2]) {
                        if (kPaged) {
                            const int page = __ldg(p.block_table + (long long)b * p.max_pages + j / p.page_size);
                            if (page >= 0 && page < p.num_pages) {
                                row = (long long)page * p.page_size + j % p.page_size;
                            } else {
                                set_status(p.status, MLA_ERR_PAGE);
                                vis[h2] = false;
                            }
                        } else {
                            row = b * seq_rows + j;
                        }
                    }
                    rows[h2] = vis[h2] ? (int)row : -1;
                }
                const unsigned lo = __ballot_sync(0xffffffffu, vis[0]), hi = __ballot_sync(0xffffffffu, vis[1]);
                const unsigned long long vmask = (unsigned long long)hi << 32 | lo;
                if (lane == 0) {
                    sm.valid[s] = vmask;
                    if (kStaged) mbar_arrive_expect_tx(&sm.landed[s], kTile * g.pitch);
                    else mbar_arrive_expect_tx(&sm.full[s], nbt * kBoxBytes);
                }
                __syncwarp();
                // lane q (< 16) gathers rows 4q .. 4q + 3
                int r4[4];
    #pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = 4 * (lane & 15) + k;
                    const int a0 = __shfl_sync(0xffffffffu, rows[0], r & 31);
                    const int a1 = __shfl_sync(0xffffffffu, rows[1], r & 31);
                    r4[k] = r < 32 ? a0 : a1;
                }
                if (lane < 16) {
                    if (kStaged) {
                        tma_gather4(sm.kv[s] + kStageBytes - kTile * g.pitch + lane * 4 * g.pitch, tm, &sm.landed[s], g.x_u32, r4[0],
                                    r4[1], r4[2], r4[3]);
                    } else {
                        for (int bx = 0; bx < nbt; ++bx)
                            tma_gather4(sm.kv[s] + bx * kBoxBytes + lane * 4 * 128, tm, &sm.full[s], g.k0 + 64 * bx, r4[0],
                                        r4[1], r4[2], r4[3]);
                    }
                }
                issued = n + 1;
            }
            // every issued copy must land before this CTA may exit
            const int first = issued > kRing ? issued - kRing : 0;
            for (int n = first; n < issued; ++n)
                mbar_wait(kStaged ? &sm.landed[n % kRing] : &sm.full[n % kRing], (n / kRing) & 1);
        } else if (warp == kProducerWarp) {
            // ------------------------------------------------------------ TMA producer, dense
            if (lane == 0) {
                // every cache line is read once: it leaves L2 first, ahead of the
                // queries and outputs the projections around this kernel reuse
                const uint64_t pol = l2_evict_first();
                // y / z coordinates of tile n's box, or false if its page is outside the pool
                auto coords = [&](int n, int &y, int &z) -> bool {
                    const int tok = t0 + n * kTile;
                    if (kPaged) {
                        const int page = __ldg(p.block_table + (long long)b * p.max_pages + tok / p.page_size);
                        y = page * p.page_size + tok % p.page_size;
                        z = 0;
                        return page >= 0 && page < p.num_pages;
                    }
                    y = tok;
                    z = b;
                    return true;
                };
                int issued = 0;
                // tile n's coordinates are looked up while the loop waits for its stage
                // (a paged cache's block-table entry is a load of its own)
                int y = 0, z = 0;
                bool page_ok = ntiles > 0 && coords(0, y, z);
                for (int n = 0; n < ntiles; ++n) {
                    const int s = n % kRing;
                    // Without a preceding grid, every CTA starts at once: the first tile
                    // goes out, the rest of the ring waits until the queries are in,
                    // which otherwise queue in HBM behind every CTA's whole ring.
                    if (n == 1 && !p.pdl && !wait_bar(sm, &sm.q_ready, 0)) {
                        raise_abort<kSplit>(sm, p, peer);
                        break;
                    }
                    if (n >= kRing && !wait_bar(sm, &sm.empty[s], ((n / kRing) - 1) & 1)) {
                        raise_abort<kSplit>(sm, p, peer);
                        break;
                    }
                    if (!page_ok) {
                        set_status(p.status, MLA_ERR_PAGE);
                        y = p.num_pages * p.page_size;  // wholly out of range: the box reads as zeros
                    }
                    if constexpr (kStaged) {
                        // one box of 64 rows of this CTA's slice; rows past the sequence end
                        // (which may hold anything) and a bad page's rows are zeroed by the converters
                        const int cnt = page_ok ? min(kTile, L - (t0 + n * kTile)) : 0;
                        sm.valid[s] = cnt >= kTile ? ~0ull : ((1ull << cnt) - 1ull);
                        // box by box: 64 rows x 64 codes into the upper half of each output box
                        mbar_arrive_expect_tx(&sm.landed[s], g.nbox * 4096);
                        for (int bx = 0; bx < g.nbox; ++bx) {
                            uint8_t *raw = sm.kv[s] + bx * kBoxBytes + 4096;
                            // (no L2 policy here: evict_first measured 1 % slower on the FP8 codes)
                            if (kPaged) tma_load_2d(raw, tm, &sm.landed[s], g.x_u32 + 16 * bx, y);
                            else tma_load_3d(raw, tm, &sm.landed[s], g.x_u32 + 16 * bx, y, z);
                        }
                    } else {
                        mbar_arrive_expect_tx(&sm.full[s], g.nbox * kBoxBytes);
                        for (int bx = 0; bx < g.nbox; ++bx) {
                            if (kPaged) tma_load_2d_hint(sm.kv[s] + bx * kBoxBytes, tm, &sm.full[s], g.k0 + 64 * bx, y, pol);
                            else tma_load_3d_hint(sm.kv[s] + bx * kBoxBytes, tm, &sm.full[s], g.k0 + 64 * bx, y, z, pol);
                        }
                    }
                    issued = n + 1;
                    if (n + 1 < ntiles) page_ok = coords(n + 1, y, z);
                }
                // every issued copy must land before this CTA may exit
                const int first = issued > kRing ? issued - kRing : 0;
                for (int n = first; n < issued; ++n)
                    mbar_wait(kStaged ? &sm.landed[n % kRing] : &sm.full[n % kRing], (n / kRing) & 1);
            }
        } else if (warp == kMma || warp == kSumWarp) {
            // ------------------------------------------------------------ MMA issuers
            // Two independent streams share the tensor pipe: the scores (warp 9: tile
            // k needs tile k loaded and S(k-1) read by the softmax) and the sums (warp
            // 11: tile k needs P(k)).  Each score MMA accumulates into the previous
            // one's result and waits out its latency; with the sums issued from a
            // warp of their own they run in those gaps instead of queueing behind the
            // whole chain (an issuing thread's next shared-memory operation waits for
            // its queued MMAs, so one thread cannot keep both streams in flight).
            const bool scores = warp == kMma;
            const uint32_t idesc_qk = idesc_of<kFp8>(kRows, kTile, false, false);
            const uint32_t idesc_pv = idesc_of<kFp8>(kRows, g.vn, false, true);
            // descriptors of stage 0; a stage's are 16-byte-unit offsets of these
            const uint64_t qk_desc0 = smem_desc_sw128(smem_u32(sm.kv[0]), 16, 1024);
            const uint64_t pv_desc0 = smem_desc_sw128(smem_u32(sm.kv[0]), kBoxBytes, 1024);
            const int nks = g.sw / 16;
            bool ok = ntiles == 0 || warp_wait(sm, &sm.q_ready, 0);
            for (int n = 0; ok && n < ntiles; ++n) {
                const int s = n % kRing;
                if (scores) {
                    if (!warp_wait(sm, &sm.full[s], (n / kRing) & 1) || (n > 0 && !warp_wait(sm, &sm.s_free, (n - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    // tokens at or past the sequence end may hold anything (even NaN):
                    // zero them so that 0-weight products stay 0 (the converters, and
                    // the sparse gathers, already wrote zeros there)
                    const int tok = t0 + n * kTile;
                    const int valid = min(kTile, L - tok);
                    if (!kStaged && !kSparse && valid < kTile) {
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
                        // fully unrolled: each MMA is an immediate add to the descriptor and
                        // the A address
                        const uint64_t db = qk_desc0 + (uint64_t)((s * kStageBytes + (g.sk0 >> 6) * kBoxBytes) >> 4);
                        const uint32_t d_s = tmem + kColS, a_q = tmem + kColQ;
    #pragma unroll
                        for (int ks = 0; ks < kMaxBoxes * 4; ++ks)
                            if (ks < nks)
                                mma_ts(d_s, a_q + ks * 8, db + (uint64_t)(((ks >> 2) * kBoxBytes + (ks & 3) * 32) >> 4),
                                       idesc_qk, ks > 0);
                        mma_commit(&sm.s_full);
                    }
                } else {
                    if (!warp_wait(sm, &sm.p_ready, n & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {  // O += P(n) . V(n), then release the tile's stage
                        const uint64_t db = pv_desc0 + (uint64_t)((s * kStageBytes) >> 4);
    #pragma unroll
                        for (int kt = 0; kt < kTile / 16; ++kt)
                            mma_ts(tmem + kColO, tmem + kColP + kt * 8, db + (uint64_t)(kt * (16 * 128 / 16)), idesc_pv,
                                   (n > 0) || kt > 0);
                        mma_commit(&sm.o_done);
                        mma_commit(&sm.empty[s]);
                    }
                }
                __syncwarp();
            }
            if (!ok) raise_abort<kSplit>(sm, p, peer);
            // every MMA issued above must finish before tensor memory is released
            if (lane == 0) mma_commit(&sm.drain);
            __syncwarp();
            mbar_wait(&sm.drain, 0);  // time-bounded only: in-flight MMAs must land
            __syncwarp();
        } else if (warp == kExch) {
            // ------------------------------------------------------------ score exchange (split mode)
            // Ships each staged tile of partial scores to the peer with one bulk copy
            // that completes on the peer's receive barrier of the tile's parity.  This
            // CTA's own receive of tile u is armed first: the receive of tile u - 2
            // has completed by then (the softmax warps consume it before they stage
            // tile u), and bytes of tile u that land before the arm only take the
            // barrier's transaction count below zero for a while.
            if (kSplit && lane == 0) {
                const uint32_t rx_peer0 = map_to_rank(smem_u32(sm.rx[0]), peer);
                const uint32_t rxfull_peer0 = map_to_rank(smem_u32(&sm.rx_full[0]), peer);
                for (int u = 0; u < ntiles; ++u) {
                    const int pb = u & 1;
                    if (!wait_bar(sm, &sm.staged[pb], (u >> 1) & 1)) {
                        raise_abort<kSplit>(sm, p, peer);
                        break;
                    }
                    mbar_arrive_expect_tx(&sm.rx_full[pb], kXBytes);
                    *(volatile int *)&sm.armed = u;
                    bulk_copy_to_peer(rx_peer0 + pb * (uint32_t)sizeof(sm.rx[0]), sm.tx[pb], kXBytes,
                                      rxfull_peer0 + pb * (uint32_t)sizeof(uint64_t));
                }
            }
        } else if (warp >= kConvWarp0 && kLoaders) {
            // ------------------------------------------------------------ loaders (bf16 sparse)
            // Boxes tma_boxes_of(g) .. nbox-1 of every listed row, copied 16 bytes at a time
            // with cp.async straight into the swizzled stage (chunk c of row r goes to
            // chunk (c % 8) ^ (r % 8) of row r of box c / 8).  Loader warp lw owns rows
            // 16 lw .. 16 lw + 15 and resolves their entries itself (lanes 0-15, one
            // tile ahead), the lanes running along a row's chunks; rows of entries that
            // take no part are written as zeros.  Each iteration first announces tile
            // n - 2, once its copies have landed (wait_group 1) and a proxy fence has
            // made them visible to the tensor cores, and only then waits for a free
            // stage, so two tiles of copies stay in flight.
            const int lw = warp - kConvWarp0;
            const int W = p.d_c + p.d_rope;
            const int iq = (rb * kRows) / p.H;
            const int lim = L - p.s_q + iq;
            const int *list = p.indices + ((long long)b * p.s_q + iq) * p.topk;
            const long long seq_rows = p.seq_stride / W;
            const int c0 = 8 * tma_boxes_of(g);  // first chunk of a row the loaders copy
            const int nl = g.kw / 8 - c0;  // chunks per row they copy (even)
            const __nv_bfloat16 *kvb = static_cast<const __nv_bfloat16 *>(p.kv);
            auto entry = [&](int n) -> int {  // lanes 0-15: list entry of row 16 lw + lane of tile n
                const int e = t0 + n * kTile + 16 * lw + (lane & 15);
                return (n < ntiles && e < t1) ? __ldg(list + e) : -1;
            };
            if (nl > 0) {
                int nxt = entry(0);
                for (int n = 0; n < ntiles + 2; ++n) {
                    if (n >= 2) {  // announce tile n - 2 (n groups committed so far)
                        cp_async_wait<1>();
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sm.full[(n - 2) % kRing]);
                    }
                    bool stop = false;
                    if (n < ntiles) {
                        const int j = nxt;
                        nxt = entry(n + 1);
                        long long myrow = -1;  // row of this lane's entry, -1: takes no part
                        if (j >= 0 && j <= lim) {
                            if (kPaged) {
                                const int page = __ldg(p.block_table + (long long)b * p.max_pages + j / p.page_size);
                                if (page >= 0 && page < p.num_pages) myrow = (long long)page * p.page_size + j % p.page_size;
                            } else {
                                myrow = b * seq_rows + j;
                            }
                        }
                        const int s = n % kRing;
                        if (n >= kRing && !warp_wait(sm, &sm.empty[s], ((n / kRing) - 1) & 1)) {
                            if (lane == 0) raise_abort<kSplit>(sm, p, peer);
                            stop = true;
                        } else {
                            const uint32_t stage = smem_u32(sm.kv[s]);
                            int r = lane / nl, c = lane % nl;  // element lane of 16 rows x nl chunks
                            for (int it = 0; it < 16 * nl / 32; ++it) {
                                const long long grow = __shfl_sync(0xffffffffu, myrow, r);
                                const int rr = 16 * lw + r, cc = c0 + c;
                                const uint32_t dst = stage + (cc >> 3) * kBoxBytes + rr * 128 + (((cc & 7) ^ (rr & 7)) << 4);
                                if (grow >= 0) {
                                    cp_async16(dst, kvb + grow * W + g.k0 + cc * 8);
                                } else {
                                    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0) : "memory");
                                }
                                c += 32;
                                while (c >= nl) {
                                    c -= nl;
                                    ++r;
                                }
                            }
                        }
                    }
                    cp_async_commit();
                    if (__any_sync(0xffffffffu, stop)) break;
                }
                cp_async_wait<0>();  // no copy may land after this CTA exits
            }
        } else if (warp >= kConvWarp0 && kStaged) {
            // ------------------------------------------------------------ converters (FP8)
            // Tile n's codes land at the top of stage n % 4 (the producer copied them
            // there once the stage was free); the converters load them, agree that
            // all have (mbarrier read[s]), rewrite the stage as fp16 operand tiles
            // and announce it.
            const int cw = warp - kConvWarp0;
            const int ncin = g.kw / 16;  // 16-byte input chunks (16 codes) of a row
            for (int n = 0; n < ntiles; ++n) {
                const int s = n % kRing;
                const uint32_t par = (n / kRing) & 1;
                if (!warp_wait(sm, &sm.landed[s], par)) {
                    if (lane == 0) raise_abort<kSplit>(sm, p, peer);
                    break;
                }
                bool ok = true;
                auto all_read = [&]() {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.read[s]);  // release: the loads are done
                    ok = warp_wait(sm, &sm.read[s], par);
                    return ok;
                };
                if constexpr (kSparse) {
                    // whole row slices: every converter's codes may lie under any output
                    convert_fp8_tile<kNConv>(sm.kv[s], sm.kv[s] + kStageBytes - kTile * g.pitch, g.pitch, ncin,
                                             sm.valid[s], cw, lane, all_read);
                } else {
                    // box cw (if any) alone, in place; a fifth box (the RoPE key's) shared by all
                    // four, 16 rows each, behind the read barrier
                    const unsigned long long vm = sm.valid[s];
                    if (cw < g.nbox && cw < 4)  // the warp's own loads precede its stores
                        convert_fp8_rows<4>(sm.kv[s] + cw * kBoxBytes, 0, vm, lane, [] {
                            __syncwarp();
                            return true;
                        });
                    if (g.nbox > 4) convert_fp8_rows<1>(sm.kv[s] + 4 * kBoxBytes, 16 * cw, vm, lane, all_read);
                }
                if (!ok) {
                    if (lane == 0) raise_abort<kSplit>(sm, p, peer);
                    break;
                }
                fence_proxy_async_smem();  // the MMAs read the stage through the async proxy
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.full[s]);
            }
        }
    } else {
        if constexpr (kRegSplit) regs_inc<kRegSoftmax>();
        // ------------------------------------------------------------ softmax + epilogue
        const int quad = warp & 3, hf = warp >> 2;
        const int r = quad * 32 + lane;  // this thread's row == TMEM lane
        const int gr = rb * kRows + r;
        const bool row_ok = seq_ok && gr < rows_total;
        const int qi = row_ok ? gr / p.H : 0;
        // the block's earliest query: a tile it sees whole, every row of the block sees whole
        const int q_first = (rb * kRows) / p.H;
        const int lim = L - p.s_q + qi;  // last visible token of this row
        const uint32_t lane_base = tmem_lane_base(quad);
        // an FP8 cache's scale multiplies every key element: fold it into Q
        const float scale_log2 = p.scale * 1.4426950408889634f * (kFp8 ? p.kv_scale : 1.f);
        const int W = p.d_c + p.d_rope;
        const uint32_t pair_bar = kBarPairBase + quad;

        // Q slice -> TMEM (bf16 pairs, fp16 with an FP8 cache), pre-multiplied by
        // scale * log2(e) (* kv_scale) so that the score MMAs produce exponents in
        // log2 units directly; the two warps of a quadrant take alternate
        // 32-channel chunks; padding rows and channels are zero.  A warp reads a
        // chunk of its 32 rows as 8 rows x 64 contiguous bytes per instruction (one
        // row per lane would touch 32 lines per instruction), every chunk's loads in
        // flight at once, and turns it into one row per lane through its own 2 KB
        // of the score staging buffer (idle until the first tile's scores),
        // 16-byte pieces XOR-swizzled by row so both passes are conflict-free.
        {
            if (p.pdl) pdl_wait();  // q_cat comes from the grid this one overlaps
            const int QW = p.q_w > 0 ? p.q_w : W;
            const int lr = lane >> 2, lj = lane & 3;  // load pass: row (of 8) and 16-byte piece
            const __nv_bfloat16 *src[4];
            bool src_ok[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int gq = rb * kRows + quad * 32 + 8 * k + lr;
                src_ok[k] = seq_ok && gq < rows_total;
                src[k] = p.q_cat + (src_ok[k] ? row_index(gq) * QW : 0);
            }
            uint4 qv[kMaxBoxes][4];
#pragma unroll
            for (int i = 0; i < kMaxBoxes; ++i) {
                const int c = 32 * hf + 64 * i + lj * 8;  // first channel of this lane's piece
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    qv[i][k] = make_uint4(0, 0, 0, 0);
                    if (src_ok[k] && c < g.sw && g.qk0 + c < QW)
                        qv[i][k] = *reinterpret_cast<const uint4 *>(src[k] + g.qk0 + c);
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
                        const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&w4[e]);
                        const float2 f = __bfloat1622float2(h);
                        v[j * 4 + e] = kFp8 ? pack_f16x2(f.x * scale_log2, f.y * scale_log2)
                                            : pack_bf16x2(f.x * scale_log2, f.y * scale_log2);
                    }
                }
                __syncwarp();
                tmem_st16(tmem + lane_base + kColQ + c0 / 2, v);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.q_ready);
        }

        const int sw = r & 7;  // chunk swizzle of this row in tx / rx
        const uint32_t s_addr = tmem + lane_base + kColS + kHalf * hf;

        // Split mode: round this thread's partial scores to fp16, stage them for the
        // exchange warp and move on.
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

        float m2 = -INFINITY;  // running (possibly stale) row maximum, log2 units (same in both halves)
        float l = 0.f;         // this half-row's sum of weights
        bool ok = true;
        int last_bar = -1;       // last tile whose pair barrier this thread passed
        float sc[kHalf];  // this CTA's (split: partial) scores of the current tile
        // paged: the block-table entry of the current tile, loaded one tile ahead
        int page_cur = (kPaged && !kSparse && ntiles > 0) ? __ldg(p.block_table + (long long)b * p.max_pages + t0 / p.page_size) : 0;
        if (ntiles > 0) {
            float s0[kHalf];
            if (!warp_wait(sm, &sm.s_full, 0)) raise_abort<kSplit>(sm, p, peer);
            tc_fence_after();
            load_scores(s_addr, s0);
            tc_fence_before();
            mbar_arrive(&sm.s_free);
            if (kSplit) stage(0, s0);
#pragma unroll
            for (int j = 0; j < kHalf; ++j) sc[j] = s0[j];
        }
        for (int n = 0; n < ntiles; ++n) {
            const int page_n = page_cur;
            if (kPaged && !kSparse && n + 1 < ntiles)
                page_cur = __ldg(p.block_table + (long long)b * p.max_pages + (t0 + (n + 1) * kTile) / p.page_size);
            // next tile's scores (the MMA computes S(n+1) as soon as S(n) was read)
            float sn[kHalf];
            const bool more = n + 1 < ntiles;
            if (more) {
                if (!warp_wait(sm, &sm.s_full, (n + 1) & 1)) raise_abort<kSplit>(sm, p, peer);
                tc_fence_after();
                load_scores(s_addr, sn);
                tc_fence_before();
                mbar_arrive(&sm.s_free);
            }
            float x[kHalf];  // scaled scores of tile n
            if (kSplit) {
                // the peer's partial of tile n
                if (warp_wait<true>(sm, &sm.rx_full[n & 1], (n >> 1) & 1)) {
                    if (threadIdx.x == 0) *(volatile int *)&sm.received = n;
                } else {
                    raise_abort<kSplit>(sm, p, peer);
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
            } else {
#pragma unroll
                for (int j = 0; j < kHalf; ++j) x[j] = sc[j];
            }
#pragma unroll
            for (int j = 0; j < kHalf; ++j) sc[j] = sn[j];
            // mask (only tiles that reach past a limit) and half-row maximum
            const int tok0 = t0 + n * kTile;
            bool tile_ok = true;
            if (kPaged && !kSparse) tile_ok = page_n >= 0 && page_n < p.num_pages;  // tokens of a bad page are skipped
            // sparse: the producer's per-row flags (listed, visible to this block's query, good page)
            const unsigned long long vmask = kSparse ? sm.valid[n % kRing] : 0ull;
            const bool whole = kSparse ? vmask == ~0ull
                                       : tile_ok && tok0 + kTile <= t1 && tok0 + kTile - 1 <= L - p.s_q + q_first;
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
                    const bool vis = kSparse ? ((vmask >> (kHalf * hf + j)) & 1ull) != 0
                                             : tile_ok && row_ok && tok < t1 && tok <= lim;
                    x[j] = vis ? x[j] : -INFINITY;
                    mx0 = fmaxf(mx0, x[j]);
                }
            }
            // the two halves of the row agree on the maximum, and on whether to go on
            sm.pair[n & 1][hf][r] = fmaxf(mx0, mx1);
            if (hf == 0 && lane == 0) sm.pair_stop[quad][n & 1] = *(volatile int *)&sm.abort;
            named_bar(pair_bar, 64);
            last_bar = n;
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
                    pk[j / 2] = kFp8 ? pack_f16x2(a, c) : pack_bf16x2(a, c);
                }
            }
            l = l * alpha + (sum0 + sum1);
            m2 = m_use;
            // the previous P . V must be done before O is rescaled or P overwritten
            if (n >= 1) {
                if (!warp_wait(sm, &sm.o_done, (n - 1) & 1)) raise_abort<kSplit>(sm, p, peer);
                tc_fence_after();
            }
            // tcgen05.ld/st are warp-collective: the whole warp takes the rescale
            // path if any of its rows needs it (alpha = 1 for the others); each warp
            // of the quadrant rescales its half of O's columns
            if (n >= 1 && __any_sync(0xffffffffu, rescale)) {
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
        ok = __shfl_sync(0xffffffffu, ok, 0);

        // ------------------------------------------------------------ epilogue
        bool have_o = ok && ntiles > 0;
        if (have_o) {
            if (!warp_wait(sm, &sm.o_done, (ntiles - 1) & 1)) {
                have_o = false;
                raise_abort<kSplit>(sm, p, peer);
            }
            tc_fence_after();
        }
        // the slot of the parity after the last pair barrier is free for the sums
        const int ls = (last_bar + 1) & 1;
        sm.pair[ls][hf][r] = l;
        named_bar(pair_bar, 64);
        const float l_row = sm.pair[ls][0][r] + sm.pair[ls][1][r];
        // TMEM reads below are warp-collective, so every lane runs them; only the
        // stores are guarded by the row bound
        const bool store = gr < rows_total;
        const float ln2 = 0.6931471805599453f;
        const int half_cols = g.vn / 2;
        const bool any = have_o && l_row > 0.f;
        // an FP8 cache's scale multiplies every value element
        const float vscale = kFp8 ? p.kv_scale : 1.f;
        // O leaves through shared memory: each thread writes its row's columns into a
        // staging copy (the operand ring is idle once the last sum has landed), then
        // the softmax warps store whole rows, consecutive lanes on consecutive 16-byte
        // chunks, instead of one 16-byte piece of 32 different rows per instruction.
        uint8_t *stg = &sm.kv[0][0];
        const int eb = nsplit == 1 ? 2 : 4;  // bf16 output or fp32 partial
        const int row_bytes = g.vn * eb, pitch = row_bytes + 16;
        if (nsplit == 1) {
            const float inv = any ? vscale / l_row : 0.f;
            for (int c = half_cols * hf; c < half_cols * (hf + 1); c += 16) {
                uint32_t u[16];
                tmem_ld16(tmem + lane_base + kColO + c, u);
                tmem_ld_wait();
                uint32_t o8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    o8[e] = pack_bf16x2(any ? __uint_as_float(u[2 * e]) * inv : 0.f,
                                        any ? __uint_as_float(u[2 * e + 1]) * inv : 0.f);
                uint4 *d4 = reinterpret_cast<uint4 *>(stg + r * pitch + c * 2);
                d4[0] = make_uint4(o8[0], o8[1], o8[2], o8[3]);
                d4[1] = make_uint4(o8[4], o8[5], o8[6], o8[7]);
            }
            if (store && rank == 0 && hf == 0)
                p.lse[row_index(gr)] = any ? (m2 + __log2f(l_row)) * ln2 : -INFINITY;
        } else {
            const long long prow = ((long long)part_seq * nsplit + split) * rows_total + gr;
            for (int c = half_cols * hf; c < half_cols * (hf + 1); c += 16) {
                uint32_t u[16];
                tmem_ld16(tmem + lane_base + kColO + c, u);
                tmem_ld_wait();
                float4 *d4 = reinterpret_cast<float4 *>(stg + r * pitch + c * 4);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    d4[e] = any ? make_float4(__uint_as_float(u[4 * e]) * vscale, __uint_as_float(u[4 * e + 1]) * vscale,
                                              __uint_as_float(u[4 * e + 2]) * vscale,
                                              __uint_as_float(u[4 * e + 3]) * vscale)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (store && hf == 0) {  // this CTA's (m, l): its half of the columns is relative to them
                p.part_ml[(prow * 2 + rank) * 2 + 0] = any ? m2 * ln2 : -INFINITY;
                p.part_ml[(prow * 2 + rank) * 2 + 1] = any ? l_row : 0.f;
            }
        }
        named_bar(kBarEpilogue, kSoftmaxThreads);
        {
            const int cpr = row_bytes / 16;  // 16-byte chunks of a row
            for (int idx = threadIdx.x; idx < kRows * cpr; idx += kSoftmaxThreads) {
                const int rr = idx / cpr, ch = idx - rr * cpr;
                const int grr = rb * kRows + rr;
                if (grr >= rows_total) continue;
                const uint4 v = *reinterpret_cast<const uint4 *>(stg + rr * pitch + ch * 16);
                uint8_t *dst = nsplit == 1
                    ? reinterpret_cast<uint8_t *>(p.o_lat + row_index(grr) * p.d_c + g.k0)
                    : reinterpret_cast<uint8_t *>(p.part_acc + (((long long)part_seq * nsplit + split) * rows_total + grr) * p.d_c + g.k0);
                *reinterpret_cast<uint4 *>(dst + ch * 16) = v;
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    // no incoming copy may land in this CTA's shared memory after it exits
    if (kSplit && threadIdx.x == 0) {
        for (int u = *(volatile int *)&sm.received + 1; u <= *(volatile int *)&sm.armed; ++u)
            mbar_wait(&sm.rx_full[u & 1], (u >> 1) & 1);
    }
    if (kSplit) cluster_sync();  // the peer may still touch this CTA's shared memory until here
    if (warp == kMma) {
        tc_fence_after();
        tmem_free<512>(tmem);
    }
}

template <bool kSplit, bool kPaged, bool kSparse, bool kFp8>
cudaError_t launch_variant(const CUtensorMap &tm0, const CUtensorMap &tm1, const AttnParams &p, const Geo &g0,
                           const Geo &g1, cudaStream_t st) {
    constexpr bool kStaged = kFp8;
    const int smem = (int)sizeof(Smem);
    auto kern = attn_tc<kSplit, kPaged, kSparse, kFp8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (threads_of(kSparse, kFp8) == 512) {
        // the register split hands out exactly the registers of a 128-per-thread
        // launch; with any other allocation the kernel is not run
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || fa.numRegs != 128) return cudaErrorNotSupported;
    }
    const int row_blocks = (p.s_q * p.H + kRows - 1) / kRows;
    cudaLaunchConfig_t cfg = {};
    const int items = p.tail_splits > 1 ? p.tail_b0 + (p.B - p.tail_b0) * p.tail_splits : p.B;
    cfg.gridDim = dim3(row_blocks * (kSplit ? 2 : 1), p.tail_splits > 1 ? 1 : p.num_splits, items);
    cfg.blockDim = dim3(threads_of(kSparse, kFp8));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSplit ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, tm0, tm1, p, g0, g1);
}

template <bool kSplit, bool kSparse, bool kFp8>
cudaError_t launch_paged(const CUtensorMap &tm0, const CUtensorMap &tm1, const AttnParams &p, const Geo &g0,
                         const Geo &g1, cudaStream_t st) {
    return p.block_table ? launch_variant<kSplit, true, kSparse, kFp8>(tm0, tm1, p, g0, g1, st)
                         : launch_variant<kSplit, false, kSparse, kFp8>(tm0, tm1, p, g0, g1, st);
}

template <bool kSplit>
cudaError_t launch_split(const CUtensorMap &tm0, const CUtensorMap &tm1, const AttnParams &p, const Geo &g0,
                         const Geo &g1, cudaStream_t st) {
    const bool sparse = p.indices != nullptr;
    if (p.kv_fp8)
        return sparse ? launch_paged<kSplit, true, true>(tm0, tm1, p, g0, g1, st)
                      : launch_paged<kSplit, false, true>(tm0, tm1, p, g0, g1, st);
    return sparse ? launch_paged<kSplit, true, false>(tm0, tm1, p, g0, g1, st)
                  : launch_paged<kSplit, false, false>(tm0, tm1, p, g0, g1, st);
}

// Tensor map of the FP8 variants for one CTA's slice: rows of 32-bit
// elements, a box of one row (sparse gathers) or of one 64-token tile.
bool encode_slice_map(CUtensorMap *tm, const AttnParams &p, const Geo &g, bool sparse) {
    const int W = p.d_c + p.d_rope;
    const uint64_t eb = p.kv_fp8 ? 1 : 2;
    const uint64_t row_u32 = (uint64_t)W * eb / 4;
    const uint32_t box_x = (uint32_t)(g.pitch / 4);
    if (sparse) {
        const uint64_t rows = p.block_table ? (uint64_t)p.num_pages * p.page_size
                                            : (uint64_t)p.B * (uint64_t)(p.seq_stride / W);
        uint64_t dims[2] = {row_u32, rows};
        uint64_t strides[1] = {(uint64_t)W * eb};
        uint32_t box[2] = {box_x, 1};
        return encode_u32_plain(tm, p.kv, 2, dims, strides, box);
    }
    // dense: one 64-channel box (64 codes = 16 words) of 64 rows per copy
    if (p.block_table) {
        uint64_t dims[2] = {row_u32, (uint64_t)p.num_pages * p.page_size};
        uint64_t strides[1] = {(uint64_t)W * eb};
        uint32_t box[2] = {16, kTile};
        return encode_u32_plain(tm, p.kv, 2, dims, strides, box);
    }
    uint64_t dims[3] = {row_u32, (uint64_t)p.capacity, (uint64_t)p.B};
    uint64_t strides[2] = {(uint64_t)W * eb, (uint64_t)p.seq_stride * eb};
    uint32_t box[3] = {16, kTile, 1};
    return encode_u32_plain(tm, p.kv, 3, dims, strides, box);
}

}  // namespace

// Per-head attention over an expanded buffer (the prefill "expand" form): p.kv
// holds, for each (sequence, head) pair b' = b * heads_per_seq + h, capacity rows
// [V_h (d_c = d_v) | K_h (d_nope) | k_rope (d_rope_cache)] of W = p.d_c + p.d_rope
// elements; the score contracts q row [q_nope | q_rope] (p.q_w = d_nope + d_rope
// elements) with the row's channels [d_v, W), the sum runs over [0, d_v).  One
// CTA per (128 query tokens, head, sequence), no history split.
cudaError_t launch_attn_expand(const AttnParams &p, cudaStream_t st) {
    const int W = p.d_c + p.d_rope;
    if (p.num_splits != 1 || p.block_table != nullptr || p.indices != nullptr || p.kv_fp8) return cudaErrorNotSupported;
    if (p.d_c % 64 || p.d_c > 256 || W > kMaxBoxes * 64 || p.q_w != W - p.d_c || p.q_w % 16) return cudaErrorNotSupported;
    Geo g;
    g.k0 = 0;
    g.kw = W;
    g.vn = p.d_c;
    g.nbox = (W + 63) / 64;
    g.pitch = 0;
    g.x_u32 = 0;
    g.sk0 = p.d_c;
    g.sw = p.q_w;
    g.qk0 = 0;
    CUtensorMap tm;
    uint64_t dims[3] = {(uint64_t)W, (uint64_t)p.capacity, (uint64_t)p.B};
    uint64_t strides[2] = {(uint64_t)W * 2, (uint64_t)p.seq_stride * 2};
    uint32_t box[3] = {64, kTile, 1};
    if (!encode_bf16_sw128(&tm, p.kv, 3, dims, strides, box)) return cudaErrorInvalidValue;
    return launch_variant<false, false, false, false>(tm, tm, p, g, g, st);
}

cudaError_t launch_attn_tc(const AttnParams &p, cudaStream_t st) {
    const int W = p.d_c + p.d_rope;
    const bool split = p.d_c > 256;
    const bool sparse = p.indices != nullptr;
    const Geo g0 = make_geo(p, 0, split), g1 = make_geo(p, 1, split);
    if (g0.nbox > kMaxBoxes || g1.nbox > kMaxBoxes || g0.kw % 16 || g1.kw % 16) return cudaErrorNotSupported;
    CUtensorMap tm0, tm1;
    if (p.kv_fp8) {
        // the raw codes sit at the top of a stage: 64 rows of at most half a stage
        if (kTile * g0.pitch > kStageBytes / 2 || kTile * g1.pitch > kStageBytes / 2) return cudaErrorNotSupported;
        if (!encode_slice_map(&tm0, p, g0, sparse)) return cudaErrorInvalidValue;
        if (split && !encode_slice_map(&tm1, p, g1, sparse)) return cudaErrorInvalidValue;
        if (!split) tm1 = tm0;
    } else if (sparse) {
        // every cache row of the contiguous cache or the pool, gathered one row per entry
        const uint64_t rows = p.block_table ? (uint64_t)p.num_pages * p.page_size
                                            : (uint64_t)p.B * (uint64_t)(p.seq_stride / W);
        uint64_t dims[2] = {(uint64_t)W, rows};
        uint64_t strides[1] = {(uint64_t)W * 2};
        uint32_t box[2] = {64, 1};
        if (!encode_bf16_sw128(&tm0, p.kv, 2, dims, strides, box)) return cudaErrorInvalidValue;
        tm1 = tm0;
    } else if (p.block_table) {
        uint64_t dims[2] = {(uint64_t)W, (uint64_t)p.num_pages * p.page_size};
        uint64_t strides[1] = {(uint64_t)W * 2};
        uint32_t box[2] = {64, kTile};
        if (!encode_bf16_sw128(&tm0, p.kv, 2, dims, strides, box)) return cudaErrorInvalidValue;
        tm1 = tm0;
    } else {
        uint64_t dims[3] = {(uint64_t)W, (uint64_t)p.capacity, (uint64_t)p.B};
        uint64_t strides[2] = {(uint64_t)W * 2, (uint64_t)p.seq_stride * 2};
        uint32_t box[3] = {64, kTile, 1};
        if (!encode_bf16_sw128(&tm0, p.kv, 3, dims, strides, box)) return cudaErrorInvalidValue;
        tm1 = tm0;
    }
    cudaError_t e = split ? launch_split<true>(tm0, tm1, p, g0, g1, st) : launch_split<false>(tm0, tm1, p, g0, g1, st);
    if (e != cudaSuccess) return e;
    if (p.tail_splits > 1) {
        // merge the tail's pieces: work-order positions tail_b0.. (their sequences
        // through p.order when the order is longest first)
        AttnParams t = p;
        t.B = p.B - p.tail_b0;
        t.num_splits = p.tail_splits;
        t.combine_b0 = p.tail_b0;
        return launch_attn_combine(t, st);
    }
    if (p.num_splits == 1) return e;
    return launch_attn_combine(p, st);
}

}  // namespace mla
