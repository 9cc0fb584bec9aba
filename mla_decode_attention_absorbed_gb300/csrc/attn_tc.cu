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
// key.  Each CTA loads only its own channel slice of every tile, computes the
// partial score over that slice, and the pair swaps partial scores through
// distributed shared memory; both then run the identical softmax (same sums in
// the same order, so the same P) and each accumulates its half of O.
//
// Tensor memory (512 columns): O [0, 256), S [256, 320), P (bf16) [320, 352),
// Q slice (bf16, MMA A operand) [352, 512).
// Warps: 0-3 softmax / epilogue (thread = row = TMEM lane), 4 TMA producer,
// 5 TMEM owner + MMA issuer.  Every wait is bounded; a lost wait records
// MLA_ERR_TIMEOUT, drains what is in flight, and the CTA returns.
#include "common.cuh"
#include "launch.h"
#include "sm100.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace sm100;

constexpr int kRows = 128;        // query rows per work item (MMA M)
constexpr int kTile = 64;         // tokens per tile (MMA N of the score, K of the sum)
constexpr int kStages = 4;        // tiles in flight
constexpr int kMaxBoxes = 5;      // 64-channel boxes per tile and CTA (320 channels)
constexpr int kBoxBytes = kTile * 128;
constexpr int kStageBytes = kMaxBoxes * kBoxBytes;  // 40 KB
constexpr int kXBytes = kRows * kTile * 4;  // one partial-score tile, fp32 (32 KB)
constexpr int kThreads = 192;
constexpr uint32_t kColO = 0, kColS = 256, kColP = 320, kColQ = 352;
constexpr float kRescaleLog2 = 8.0f;  // keep a stale maximum until scores exceed it by 2^8

struct Geo {
    int k0;      // first channel of this CTA's contraction slice (= first latent column of its O slice)
    int kw;      // contraction width (multiple of 16)
    int nbox;    // 64-channel boxes loaded per tile
    int vn;      // latent columns this CTA accumulates (multiple of 64, <= 256)
};

struct Smem {
    uint8_t kv[kStages][kStageBytes];
    // split mode: this CTA's partial scores staged for the bulk copy to the peer,
    // and the peer's partial scores received.  Row r's 16-byte chunk c sits at
    // chunk c ^ (r % 16), so that a warp's row-per-thread accesses do not collide.
    float tx[kRows * kTile];
    float rx[kRows * kTile];
    uint64_t full[kStages], empty[kStages];
    uint64_t q_ready, s_full, s_free, p_ready, o_done, rx_full, peer_rx_free, drain;
    uint32_t tmem_base;
    int abort;  // set by this CTA or, remotely, by the peer
    int stop;   // the softmax warps' common decision to leave the tile loop
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bounded wait that also gives up once the CTA is aborting.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(Smem &sm, uint64_t *bar, uint32_t parity) {
    if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const long long c0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*(volatile int *)&sm.abort) return false;
            if (wait_expired(t0, c0)) return false;
        }
    }
}

// Every lane waits; the warp proceeds only if all lanes saw the phase complete,
// so warp-collective tcgen05 instructions that follow stay converged.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(Smem &sm, uint64_t *bar, uint32_t parity) {
    const bool ok = wait_bar<kCluster>(sm, bar, parity);
    return __all_sync(0xffffffffu, ok);
}

template <bool kSplit>
__device__ __forceinline__ void raise_abort(Smem &sm, const AttnParams &p, uint32_t peer) {
    *(volatile int *)&sm.abort = 1;
    set_status(p.status, MLA_ERR_TIMEOUT);
    if (kSplit) {
        uint32_t remote = map_to_rank(smem_u32(&sm.abort), peer);
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(1) : "memory");
    }
}

template <bool kSplit, bool kPaged>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc(const __grid_constant__ CUtensorMap tm_kv, const AttnParams p, const Geo g0, const Geo g1) {
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = kSplit ? cluster_rank() : 0;
    const uint32_t peer = rank ^ 1u;
    const Geo g = rank == 0 ? g0 : g1;
    const int rb = kSplit ? blockIdx.x / 2 : blockIdx.x;
    const int split = blockIdx.y, b = blockIdx.z;
    const int rows_total = p.s_q * p.H;

    const int L = __ldg(p.seq_lens + b);
    const bool seq_ok = seq_len_ok(p, L);
    int t0 = 0, t1 = 0;
    if (seq_ok) split_range(L, p.num_splits, split, t0, t1);
    const int ntiles = (t1 - t0 + kTile - 1) / kTile;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.q_ready, 128);
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_free, 128);
        mbar_init(&sm.p_ready, 128);
        mbar_init(&sm.o_done, 1);
        mbar_init(&sm.rx_full, 1);
        mbar_init(&sm.peer_rx_free, 1);
        mbar_init(&sm.drain, 1);
        sm.abort = 0;
        sm.stop = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_kv);
    }
    if (!seq_ok && split == 0 && rb == 0 && rank == 0 && threadIdx.x == 0) set_status(p.status, MLA_ERR_SEQLEN);
    if (warp == 5) tmem_alloc<512>(&sm.tmem_base);
    tc_fence_before();
    if (kSplit) cluster_sync();
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 4) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int n = 0; n < ntiles; ++n) {
                const int s = n % kStages;
                if (n >= kStages && !wait_bar(sm, &sm.empty[s], ((n / kStages) - 1) & 1)) {
                    raise_abort<kSplit>(sm, p, peer);
                    break;
                }
                const int tok = t0 + n * kTile;
                int x0 = g.k0, y = 0, z = 0;
                if (kPaged) {
                    int page = __ldg(p.block_table + (long long)b * p.max_pages + tok / p.page_size);
                    if (page < 0 || page >= p.num_pages) {
                        set_status(p.status, MLA_ERR_PAGE);
                        page = p.num_pages;  // wholly out of range: the box reads as zeros
                    }
                    y = page * p.page_size + tok % p.page_size;
                } else {
                    y = tok;
                    z = b;
                }
                mbar_arrive_expect_tx(&sm.full[s], g.nbox * kBoxBytes);
                for (int bx = 0; bx < g.nbox; ++bx) {
                    if (kPaged) tma_load_2d(sm.kv[s] + bx * kBoxBytes, &tm_kv, &sm.full[s], x0 + 64 * bx, y);
                    else tma_load_3d(sm.kv[s] + bx * kBoxBytes, &tm_kv, &sm.full[s], x0 + 64 * bx, y, z);
                }
                issued = n + 1;
            }
            // drain: every issued copy must land before this CTA may exit
            const int first = issued > kStages ? issued - kStages : 0;
            for (int n = first; n < issued; ++n) mbar_wait(&sm.full[n % kStages], (n / kStages) & 1);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t idesc_qk = idesc_bf16(kRows, kTile, false, false);
        const uint32_t idesc_pv = idesc_bf16(kRows, g.vn, false, true);
        bool ok = ntiles == 0 || warp_wait(sm, &sm.q_ready, 0);
        for (int n = 0; n < ntiles && ok; ++n) {
            const int s = n % kStages;
            if (!warp_wait(sm, &sm.full[s], (n / kStages) & 1)) { ok = false; break; }
            // tokens at or past the sequence end may hold anything (even NaN): zero
            // them so that 0-weight products stay 0
            const int tok = t0 + n * kTile;
            const int valid = min(kTile, L - tok);
            if (valid < kTile) {
                for (int e = lane; e < (kTile - valid) * 8 * g.nbox; e += 32) {
                    const int bx = e / ((kTile - valid) * 8);
                    const int rr = valid + (e / 8) % (kTile - valid);
                    reinterpret_cast<uint4 *>(sm.kv[s] + bx * kBoxBytes + rr * 128)[e % 8] = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (n >= 1 && !warp_wait(sm, &sm.s_free, (n - 1) & 1)) { ok = false; break; }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t kvs = smem_u32(sm.kv[s]);
                for (int ks = 0; ks < g.kw / 16; ++ks) {
                    const uint64_t db = smem_desc_sw128(kvs + (ks / 4) * kBoxBytes + (ks % 4) * 32, 16, 1024);
                    mma_ts(tmem + kColS, tmem + kColQ + ks * 8, db, idesc_qk, ks > 0);
                }
                mma_commit(&sm.s_full);
            }
            __syncwarp();
            if (n >= 1) {
                if (!warp_wait(sm, &sm.p_ready, (n - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    const int sp = (n - 1) % kStages;
                    const uint32_t kvs = smem_u32(sm.kv[sp]);
                    for (int kt = 0; kt < kTile / 16; ++kt) {
                        const uint64_t db = smem_desc_sw128(kvs + kt * 16 * 128, kBoxBytes, 1024);
                        mma_ts(tmem + kColO, tmem + kColP + kt * 8, db, idesc_pv, (n - 1 > 0) || kt > 0);
                    }
                    mma_commit(&sm.o_done);
                    mma_commit(&sm.empty[sp]);
                }
                __syncwarp();
            }
        }
        if (ok && ntiles > 0) {
            if (!warp_wait(sm, &sm.p_ready, (ntiles - 1) & 1)) {
                ok = false;
            } else {
                tc_fence_after();
                if (lane == 0) {
                    const int sp = (ntiles - 1) % kStages;
                    const uint32_t kvs = smem_u32(sm.kv[sp]);
                    for (int kt = 0; kt < kTile / 16; ++kt) {
                        const uint64_t db = smem_desc_sw128(kvs + kt * 16 * 128, kBoxBytes, 1024);
                        mma_ts(tmem + kColO, tmem + kColP + kt * 8, db, idesc_pv, (ntiles - 1 > 0) || kt > 0);
                    }
                    mma_commit(&sm.o_done);
                    mma_commit(&sm.empty[sp]);
                }
                __syncwarp();
            }
        }
        if (!ok) raise_abort<kSplit>(sm, p, peer);
        // every MMA issued above must finish before tensor memory is released
        if (lane == 0) mma_commit(&sm.drain);
        __syncwarp();
        mbar_wait(&sm.drain, 0);  // time-bounded only: in-flight MMAs must land
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue (rows)
        const int r = threadIdx.x;  // 0..127 == TMEM lane
        const int gr = rb * kRows + r;
        const bool row_ok = seq_ok && gr < rows_total;
        const int qi = row_ok ? gr / p.H : 0;
        const int lim = L - p.s_q + qi;  // last visible token of this row
        const uint32_t lane_base = tmem_lane_base(warp);
        const float scale_log2 = p.scale * 1.4426950408889634f;
        const int W = p.d_c + p.d_rope;

        // Q slice -> TMEM (bf16 pairs), zero for padding rows / channels
        {
            const __nv_bfloat16 *qrow = p.q_cat + ((long long)b * rows_total + gr) * W;
            for (int c0 = 0; c0 < g.kw; c0 += 32) {
                uint32_t v[16];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint4 u = make_uint4(0, 0, 0, 0);
                    const int ch = g.k0 + c0 + e * 8;
                    if (row_ok && ch < W && c0 + e * 8 < g.kw) u = *reinterpret_cast<const uint4 *>(qrow + ch);
                    v[e * 4 + 0] = u.x; v[e * 4 + 1] = u.y; v[e * 4 + 2] = u.z; v[e * 4 + 3] = u.w;
                }
                tmem_st16(tmem + lane_base + kColQ + c0 / 2, v);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.q_ready);
        }

        uint32_t rx_peer = 0, rxfull_peer = 0, rxfree_peer = 0;
        if (kSplit) {
            rx_peer = map_to_rank(smem_u32(sm.rx), peer);
            rxfull_peer = map_to_rank(smem_u32(&sm.rx_full), peer);
            rxfree_peer = map_to_rank(smem_u32(&sm.peer_rx_free), peer);
        }
        const int sw = r & 15;  // chunk swizzle of this row in tx / rx

        float m2 = -INFINITY;  // running (possibly stale) maximum, log2 units
        float l = 0.f;
        bool ok = true;
        int armed = -1, received = -1;  // last receive this CTA armed / completed (split mode)
        for (int n = 0; n < ntiles; ++n) {
            bool good = warp_wait(sm, &sm.s_full, n & 1);
            tc_fence_after();
            float s[kTile];
            {
                uint32_t u0[16], u1[16], u2[16], u3[16];
                tmem_ld16(tmem + lane_base + kColS + 0, u0);
                tmem_ld16(tmem + lane_base + kColS + 16, u1);
                tmem_ld16(tmem + lane_base + kColS + 32, u2);
                tmem_ld16(tmem + lane_base + kColS + 48, u3);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    s[e] = __uint_as_float(u0[e]);
                    s[16 + e] = __uint_as_float(u1[e]);
                    s[32 + e] = __uint_as_float(u2[e]);
                    s[48 + e] = __uint_as_float(u3[e]);
                }
            }
            tc_fence_before();
            mbar_arrive(&sm.s_free);
            if (kSplit) {
                // Swap partial scores with the peer: stage locally, one bulk copy
                // each way (completing bytes on the receiver's barrier), sum.
                // Named barriers keep the 128 threads in step; nobody leaves the loop
                // between them, and the decision to stop is taken jointly.
                float4 *txrow = reinterpret_cast<float4 *>(sm.tx + r * kTile);
#pragma unroll
                for (int c = 0; c < kTile / 4; ++c)
                    txrow[c ^ sw] = make_float4(s[4 * c], s[4 * c + 1], s[4 * c + 2], s[4 * c + 3]);
                fence_proxy_async_smem();
                named_bar(1, 128);
                if (threadIdx.x == 0) {
                    bool go = !*(volatile int *)&sm.abort;
                    if (go && n >= 1 && !wait_bar<true>(sm, &sm.peer_rx_free, (n - 1) & 1)) {
                        raise_abort<kSplit>(sm, p, peer);
                        go = false;
                    }
                    mbar_arrive_expect_tx(&sm.rx_full, kXBytes);  // arm this CTA's receive of tile n
                    armed = n;
                    if (go) {
                        bulk_copy_to_peer(rx_peer, sm.tx, kXBytes, rxfull_peer);
                        bulk_commit();
                    }
                }
                if (warp_wait<true>(sm, &sm.rx_full, n & 1)) {
                    if (threadIdx.x == 0) received = n;
                } else {
                    good = false;
                }
                const float4 *rxrow = reinterpret_cast<const float4 *>(sm.rx + r * kTile);
#pragma unroll
                for (int c = 0; c < kTile / 4; ++c) {
                    const float4 v = rxrow[c ^ sw];
                    s[4 * c] += v.x; s[4 * c + 1] += v.y; s[4 * c + 2] += v.z; s[4 * c + 3] += v.w;
                }
                if (!good) raise_abort<kSplit>(sm, p, peer);
                if (threadIdx.x == 0) {
                    bulk_wait_read_all();  // tx may be rewritten next tile
                    sm.stop = *(volatile int *)&sm.abort;
                }
                named_bar(1, 128);
                const bool stop = *(volatile int *)&sm.stop;
                if (threadIdx.x == 0 && !stop) mbar_arrive_remote(rxfree_peer);  // the peer may refill rx
                if (stop) {
                    ok = false;
                    break;
                }
            } else if (!good) {
                ok = false;
                break;
            }
            // scale, mask (only tiles that reach past a limit), tile maximum
            const int tok0 = t0 + n * kTile;
            bool tile_ok = true;
            if (kPaged) {
                const int page = __ldg(p.block_table + (long long)b * p.max_pages + tok0 / p.page_size);
                tile_ok = page >= 0 && page < p.num_pages;  // tokens of a bad page are skipped
            }
            const bool whole = tile_ok && tok0 + kTile <= t1 && tok0 + kTile - 1 <= L - p.s_q;
            float tmax = -INFINITY;
            if (whole) {
#pragma unroll
                for (int j = 0; j < kTile; ++j) {
                    s[j] *= scale_log2;
                    tmax = fmaxf(tmax, s[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < kTile; ++j) {
                    const int tok = tok0 + j;
                    const bool vis = tile_ok && row_ok && tok < t1 && tok <= lim;
                    s[j] = vis ? s[j] * scale_log2 : -INFINITY;
                    tmax = fmaxf(tmax, s[j]);
                }
            }
            float m_use = m2, alpha = 1.f;
            bool rescale = false;
            if (tmax > m2 + kRescaleLog2 || (m2 == -INFINITY && tmax > -INFINITY)) {
                m_use = tmax;
                if (m2 != -INFINITY) {
                    alpha = ex2(m2 - m_use);
                    rescale = true;
                }
            }
            float sum = 0.f;
            uint32_t pk[kTile / 2];
            if (m_use == -INFINITY) {
#pragma unroll
                for (int j = 0; j < kTile / 2; ++j) pk[j] = 0u;
            } else {
#pragma unroll
                for (int j = 0; j < kTile; j += 2) {
                    const float a = ex2(s[j] - m_use);
                    const float c = ex2(s[j + 1] - m_use);
                    sum += a + c;
                    pk[j / 2] = pack_bf16x2(a, c);
                }
            }
            l = l * alpha + sum;
            m2 = m_use;
            // the previous P . V must be done before O is rescaled or P overwritten
            if (n >= 1) {
                if (!warp_wait(sm, &sm.o_done, (n - 1) & 1)) {
                    if (!kSplit) {
                        ok = false;
                        break;
                    }
                    raise_abort<kSplit>(sm, p, peer);  // the loop stops at the next joint decision
                }
                tc_fence_after();
            }
            // tcgen05.ld/st are warp-collective: the whole warp takes the rescale
            // path if any of its rows needs it (alpha = 1 for the others)
            if (n >= 1 && __any_sync(0xffffffffu, rescale)) {
                if (!rescale) alpha = 1.f;
                for (int c = 0; c < g.vn; c += 16) {
                    uint32_t u[16];
                    tmem_ld16(tmem + lane_base + kColO + c, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
                    tmem_st16(tmem + lane_base + kColO + c, u);
                }
            }
            {
                uint32_t h0[16], h1[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) { h0[e] = pk[e]; h1[e] = pk[16 + e]; }
                tmem_st16(tmem + lane_base + kColP, h0);
                tmem_st16(tmem + lane_base + kColP + 16, h1);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.p_ready);
        }
        if (kSplit) {
            if (threadIdx.x == 0 && armed > received) mbar_wait(&sm.rx_full, armed & 1);  // no copy may land after exit
            ok = ok && !*(volatile int *)&sm.abort;
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        if (!ok) raise_abort<kSplit>(sm, p, peer);

        // ------------------------------------------------------------ epilogue
        bool have_o = ok && ntiles > 0;
        if (have_o) {
            if (!warp_wait(sm, &sm.o_done, (ntiles - 1) & 1)) {
                have_o = false;
                raise_abort<kSplit>(sm, p, peer);
            }
            tc_fence_after();
        }
        // TMEM reads below are warp-collective, so every lane runs them; only the
        // stores are guarded by the row bound
        const bool store = gr < rows_total;
        const float ln2 = 0.6931471805599453f;
        if (p.num_splits == 1) {
            const float inv = (have_o && l > 0.f) ? 1.f / l : 0.f;
            __nv_bfloat16 *dst = p.o_lat + ((long long)b * rows_total + gr) * p.d_c + g.k0;
            for (int c = 0; c < g.vn; c += 16) {
                uint32_t u[16];
                tmem_ld16(tmem + lane_base + kColO + c, u);
                tmem_ld_wait();
                uint32_t o8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    o8[e] = pack_bf16x2(inv == 0.f ? 0.f : __uint_as_float(u[2 * e]) * inv,
                                        inv == 0.f ? 0.f : __uint_as_float(u[2 * e + 1]) * inv);
                if (store) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
                    d4[0] = make_uint4(o8[0], o8[1], o8[2], o8[3]);
                    d4[1] = make_uint4(o8[4], o8[5], o8[6], o8[7]);
                }
            }
            if (store && rank == 0)
                p.lse[(long long)b * rows_total + gr] = (have_o && l > 0.f) ? (m2 + __log2f(l)) * ln2 : -INFINITY;
        } else {
            const long long prow = ((long long)b * p.num_splits + split) * rows_total + gr;
            float *dst = p.part_acc + prow * p.d_c + g.k0;
            for (int c = 0; c < g.vn; c += 16) {
                uint32_t u[16];
                tmem_ld16(tmem + lane_base + kColO + c, u);
                tmem_ld_wait();
                if (store) {
                    float4 *d4 = reinterpret_cast<float4 *>(dst + c);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        d4[e] = have_o ? make_float4(__uint_as_float(u[4 * e]), __uint_as_float(u[4 * e + 1]),
                                                     __uint_as_float(u[4 * e + 2]), __uint_as_float(u[4 * e + 3]))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            if (store && rank == 0) {
                const bool any = have_o && l > 0.f;
                p.part_ml[prow * 2 + 0] = any ? m2 * ln2 : -INFINITY;
                p.part_ml[prow * 2 + 1] = any ? l : 0.f;
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    if (kSplit) cluster_sync();  // the peer may still touch this CTA's shared memory until here
    if (warp == 5) {
        tc_fence_after();
        tmem_free<512>(tmem);
    }
}

Geo make_geo(const AttnParams &p, int rank, bool split) {
    const int W = p.d_c + p.d_rope;
    Geo g;
    if (!split) {
        g.k0 = 0;
        g.kw = W;
        g.vn = p.d_c;
    } else if (rank == 0) {
        g.k0 = 0;
        g.kw = 256;
        g.vn = 256;
    } else {
        g.k0 = 256;
        g.kw = W - 256;
        g.vn = p.d_c - 256;
    }
    g.nbox = (g.kw + 63) / 64;
    return g;
}

template <bool kSplit, bool kPaged>
cudaError_t launch_variant(const CUtensorMap &tm, const AttnParams &p, const Geo &g0, const Geo &g1, cudaStream_t st) {
    const int smem = (int)sizeof(Smem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(attn_tc<kSplit, kPaged>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int row_blocks = (p.s_q * p.H + kRows - 1) / kRows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(row_blocks * (kSplit ? 2 : 1), p.num_splits, p.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSplit ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_tc<kSplit, kPaged>, tm, p, g0, g1);
}

}  // namespace

cudaError_t launch_attn_tc(const AttnParams &p, cudaStream_t st) {
    const int W = p.d_c + p.d_rope;
    const bool split = p.d_c > 256;
    const Geo g0 = make_geo(p, 0, split), g1 = make_geo(p, 1, split);
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
    cudaError_t e;
    if (split) e = p.block_table ? launch_variant<true, true>(tm, p, g0, g1, st) : launch_variant<true, false>(tm, p, g0, g1, st);
    else e = p.block_table ? launch_variant<false, true>(tm, p, g0, g1, st) : launch_variant<false, false>(tm, p, g0, g1, st);
    if (e != cudaSuccess || p.num_splits == 1) return e;
    return launch_attn_combine(p, st);
}

}  // namespace mla
