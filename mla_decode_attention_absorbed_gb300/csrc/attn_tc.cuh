// Layout shared by the attention kernels (attn_tc.cu, attn_persist.cu): tile
// and work-item sizes, warp roles, tensor-memory columns, the shared-memory
// block, each CTA's channel slice of a pair, and two small device helpers.
#pragma once

#include <cuda_fp16.h>

#include "attn_common.cuh"
#include "common.cuh"
#include "sm100.cuh"

namespace mla {
namespace attn {

using namespace sm100;

constexpr int kRows = 128;        // query rows per work item (MMA M)
constexpr int kTile = 64;         // tokens per tile (MMA N of the score, K of the sum)
constexpr int kHalf = kTile / 2;  // tokens per softmax thread
constexpr int kMaxBoxes = 5;      // 64-channel boxes per tile and CTA (320 channels)
constexpr int kBoxBytes = kTile * 128;
constexpr int kStageBytes = kMaxBoxes * kBoxBytes;  // 40 KB
constexpr int kXBytes = kRows * kTile * 2;          // one partial-score tile in fp16 (16 KB)
constexpr int kSoftmaxThreads = 256;
constexpr int kSoftmaxWarps = kSoftmaxThreads / 32;
constexpr int kProducerWarp = 8, kMmaWarp = 9, kExchangeWarp = 10, kSumWarp = 11, kConvWarp0 = 12;
constexpr int kConvWarps = 4;     // loader warps (bf16 sparse)
constexpr int kFp8ConvWarps = 4;  // converter warps (FP8)
constexpr int kTmaBoxes = 2;      // bf16 sparse: boxes of a row gathered by tile::gather4, at least

constexpr int kRing = 4;          // operand-ring stages (tiles in flight into the MMAs)

// threads of a variant
__host__ __device__ constexpr int extra_warps(bool sparse, bool fp8) { return fp8 ? kFp8ConvWarps : (sparse ? kConvWarps : 0); }
__host__ __device__ constexpr int threads_of(bool sparse, bool fp8) {
    return kSoftmaxThreads + 128 + 32 * extra_warps(sparse, fp8);
}


// Register split of the 512-thread variants: the launch gives every thread
// 65536 / 512 = 128 registers; the two softmax warpgroups raise theirs to 136
// and the other two lower theirs to 120 (2 x 128 x 136 + 2 x 128 x 120 = 65536,
// exactly the launch's total, so the raise never waits on registers nobody
// gives up).  Each warpgroup runs its instruction once, on entering its roles.
constexpr int kRegSoftmax = 136, kRegOther = 120;
static_assert(2 * 128 * kRegSoftmax + 2 * 128 * kRegOther == 65536, "register split must equal the launch's total");

constexpr uint32_t kColO = 0, kColS = 256, kColP = 320, kColQ = 352;
constexpr float kRescaleLog2 = 8.0f;  // keep a stale maximum until scores exceed it by 2^8
constexpr uint32_t kBarPairBase = 1;  // named barrier 1 + quadrant: the two warps of a quadrant (64 threads)
constexpr uint32_t kBarEpilogue = 5;  // all softmax warps: O rows staged in shared memory

struct Geo {
    int k0;      // first channel of this CTA's contraction slice (= first latent column of its O slice)
    int kw;      // contraction width (multiple of 16)
    int nbox;    // 64-channel boxes loaded per tile
    int vn;      // latent columns this CTA accumulates (multiple of 64, <= 256)
    int pitch;   // FP8: bytes of one raw row (the slice, rounded up to 32 B)
    int x_u32;   // FP8: first 32-bit element of the slice within a cache row
    int sk0;     // first channel of the score contraction, counted from k0 (a multiple of 64)
    int sw;      // score contraction width (multiple of 16; = kw unless the row carries values apart)
    int qk0;     // first channel of this CTA's query slice within a q_cat row
};

struct Smem {
    uint8_t kv[kRing][kStageBytes];  // swizzled operand tiles (FP8: raw codes first land at the top)
    // split mode: this CTA's scaled partial scores (fp16) staged for the bulk copy
    // to the peer, and the peer's received, both by tile parity.  Row r is 128 B
    // (64 fp16); its 16-byte chunk c sits at chunk c ^ (r % 8).
    alignas(128) __half tx[2][kRows * kTile];
    __half rx[2][kRows * kTile];
    // per half-row values the two warps of a quadrant exchange, by tile parity:
    // tile maxima in the loop, softmax sums in the epilogue
    float pair[2][2][kRows];
    int pair_stop[4][2];  // each quadrant's joint decision to leave the tile loop, by tile parity
    // sparse and FP8: per stage, bit r set when row r of the tile takes part
    unsigned long long valid[kRing];
    uint64_t full[kRing], empty[kRing];
    uint64_t landed[kRing], read[kRing];  // FP8: raw codes landed; every converter holds its codes
    uint64_t q_ready, s_full, s_free, p_ready, o_done, drain;
    // staged[i]: the softmax warps staged the tile of parity i; rx_full[i]: the
    // peer's tile of parity i landed
    uint64_t staged[2], rx_full[2];
    uint32_t tmem_base;
    int abort;    // set by this CTA or, remotely, by the peer
    uint64_t wait_ns;  // bound of the waits for work (the launch's, else the default)
    int lpt_b, lpt_L;  // longest-first order: the sequence of this CTA's work item, its length
    int armed;    // last tile whose receive the exchange warp armed
    int received; // last tile the softmax warps received
    // persistent kernel only (attn_persist.cu): one phase per work item with tiles
    uint64_t q_next;       // the epilogue warps loaded the next item's queries
    uint64_t s_last;       // the item's last score chain completed
    uint64_t o_last;       // the item's last P . V completed
    uint64_t o_free;       // the epilogue warps drained the item's O
    uint64_t ml_ready[2];  // by item parity: the softmax warps left the item's (m, l)
    uint64_t merge_full;   // a merge wave's rows and (m, l) landed in the ring
    int walk_b;            // the sequence holding the first tile of this pair's range
    int n_pending;         // merges this CTA owes (it wrote the sequence's last piece): at most 2
    int pend_b[2];         // their sequences
    long long walk_S;      // walk_b's first tile in the batch's tile order
    long long pend_S[2];   // the pending sequences' first tiles
};

// the whole block, with no realignment slack, within the 227 KB a CTA may use
static_assert(sizeof(Smem) <= 232448, "shared memory block over the per-CTA limit");

// This thread's 32 scores of the tile in S (tensor memory).
__device__ __forceinline__ void load_scores(uint32_t taddr, float (&s)[kHalf]) {
    uint32_t u0[16], u1[16];
    tmem_ld16(taddr, u0);
    tmem_ld16(taddr + 16, u1);
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        s[e] = __uint_as_float(u0[e]);
        s[16 + e] = __uint_as_float(u1[e]);
    }
}

// Instruction descriptor of the kernel's MMAs: bf16 operands, or fp16 for an FP8 cache.
template <bool kFp8>
__device__ __forceinline__ uint32_t idesc_of(int M, int N, bool a_mn, bool b_mn) {
    const uint32_t d = idesc_bf16(M, N, a_mn, b_mn);
    return kFp8 ? (d & ~((7u << 7) | (7u << 10))) : d;  // A / B format 0 = f16
}

inline Geo make_geo(const AttnParams &p, int rank, bool split) {
    const int W = p.d_c + p.d_rope;
    const int eb = p.kv_fp8 ? 1 : 2;  // bytes per cache element
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
    g.pitch = (g.kw * eb + 31) / 32 * 32;
    g.x_u32 = g.k0 * eb / 4;
    g.sk0 = 0;
    g.sw = g.kw;
    g.qk0 = g.k0;
    return g;
}

}  // namespace attn
}  // namespace mla
