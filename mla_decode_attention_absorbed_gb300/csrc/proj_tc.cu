// Per-head projection GEMMs on the 5th-generation tensor cores (tcgen05):
//   absorb:  q_cat[m,h,0:d_c] = q_nope[m,h,:] . W_UK[h]^T          (B operand K-major)
//   out:     out[m,h,:]       = o_lat[m,h,:]  . W_UV[h]            (B operand MN-major)
//   append:  c[m,:]           = x[m,:] . W_DKV                     (B operand MN-major, split K)
// ("MLA, dim by dim", "MLA Decode": absorb W_UK^T into the current query, apply
// W_UV once to the latent-space output, and compress the new token's hidden
// state into its latent, which is appended to the cache.)  m = b*s_q + i runs
// over the batch's query tokens; one CTA computes a 128-row x BN-column tile of
// one head, over all of K or, split K, over a run of K chunks whose fp32 tile
// it stores as that split's partial.
//
// Warp roles (320 threads): warp 0 issues TMA loads, warp 1 owns tensor memory
// and issues the MMAs, warps 2-9 drain the fp32 accumulator from TMEM (two warps
// per lane quadrant, one half of the columns each), round to bf16 and stage the
// rows in the idle operand ring, then store them as whole rows (consecutive
// lanes on consecutive 16-byte chunks).  K is streamed in 64-wide chunks through
// a 4-stage ring.
#include "common.cuh"
#include "launch.h"
#include "sm100.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace sm100;

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 320;
constexpr int kEpiThreads = kThreads - 64;  // warps 2-9
constexpr uint32_t kBarEpi = 1;             // named barrier of the epilogue warps

struct ProjArgs {
    int M;                 // query tokens (B * s_q)
    int H;                 // heads = batch of the GEMM
    int N;                 // output width per head
    int K;                 // contraction width
    __nv_bfloat16 *out;    // row m, head h, column n at out + (m*H + h)*out_row + n
    int out_row;           // elements per (m, h) output row
    const __nv_bfloat16 *rope_src;  // absorb only: q_rope [M][H][d_rope], copied after column d_c
    int d_rope;
    float *acc;            // split K: fp32 partials [splits][M][N] instead of `out`
    int kc_per_cta;        // split K: 64-wide K chunks per CTA
    int splits;            // split K: CTAs along K (grid z)
    // programmatic dependent launch inside a fused decode step: this grid may start
    // while the previous one runs and reads A (its output) only after it completed;
    // and / or lets the next grid start its CTAs right away
    bool wait_a;
    bool trigger;
};

// BN = 512 (a whole d_c = 512 head per CTA) would run two N = 256 MMAs per K step
// into the two halves of tensor memory.  The absorb GEMM (K-major B, K = d_nope:
// two chunks) at BN = 256 takes a 2-stage ring, so that two CTAs fit an SM: its
// 2 x H CTAs at d_c = 512 run in one wave (measured against one CTA a head: the
// dsv3 step 116.4 -> 114.6 us).
template <int BN, bool kBMN>
struct ProjSmem {
    static constexpr uint32_t kTmemCols = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : BN <= 256 ? 256 : 512;
    static constexpr int kStagesN = (BN > 256 || (!kBMN && BN == 256)) ? 2 : kStages;
    static constexpr int kHalves = BN > 256 ? 2 : 1;   // MMAs of N = BN / kHalves per K step
    static constexpr int kABytes = kBM * kBK * 2;  // 16 KB
    static constexpr int kBBytes = BN * kBK * 2;   // 32 KB at BN = 256
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kBytes = kStagesN * kStageBytes + 1024 /* barriers */ + 1024 /* alignment */;
    static_assert(kBM * (BN * 2 + 16) <= kStagesN * kStageBytes, "the bf16 rows are staged in the operand ring");
};

template <int BN, bool kBMN>
__global__ void __launch_bounds__(kThreads, 1)
    proj_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, ProjArgs g) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment: the 128-byte swizzle pattern repeats every 8 rows of 128 B
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using L = ProjSmem<BN, kBMN>;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kStagesN * L::kStageBytes);
    uint64_t *empty = full + L::kStagesN;
    uint64_t *acc_full = empty + L::kStagesN;
    uint32_t *tmem_base_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_base_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * kBM;
    const int nk_all = (g.K + kBK - 1) / kBK;  // the last chunk's columns past K read as zero
    const int h = g.acc ? 0 : blockIdx.z;
    const int kc0 = g.acc ? blockIdx.z * g.kc_per_cta : 0;
    const int nk = g.acc ? min(g.kc_per_cta, nk_all - kc0) : nk_all;
    if (g.trigger) pdl_launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::kStagesN; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) tmem_alloc<L::kTmemCols>(tmem_base_slot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_slot;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        // After a programmatic launch the weight chunks of the first stages are
        // fetched while the previous grid still runs; A, its output, only once it
        // has completed.
        const int early = g.wait_a ? min(nk, L::kStagesN) : 0;
        auto load_b = [&](int kc) {
            const int s = kc % L::kStagesN;
            uint8_t *sb = smem + s * L::kStageBytes + L::kABytes;
            const int kx = (kc0 + kc) * kBK;
            if (kBMN) {
                for (int j = 0; j < BN / 64; ++j) tma_load_3d(sb + j * 64 * 128, &tmB, &full[s], n0 + 64 * j, kx, h);
            } else {
                for (int j = 0; j < L::kHalves; ++j)
                    tma_load_3d(sb + j * (BN / L::kHalves) * 128, &tmB, &full[s], kx, n0 + j * (BN / L::kHalves), h);
            }
        };
        for (int kc = 0; kc < early; ++kc) {
            mbar_arrive_expect_tx(&full[kc], L::kStageBytes);
            load_b(kc);
        }
        if (g.wait_a) pdl_wait();
        for (int kc = 0; kc < nk; ++kc) {
            const int s = kc % L::kStagesN;
            if (kc >= L::kStagesN && !mbar_wait(&empty[s], ((kc / L::kStagesN) - 1) & 1)) {
                *abort_flag = 1;
                break;
            }
            if (*abort_flag) break;
            uint8_t *sa = smem + s * L::kStageBytes;
            const int kx = (kc0 + kc) * kBK;
            if (kc >= early) mbar_arrive_expect_tx(&full[s], L::kStageBytes);
            tma_load_3d(sa, &tmA, &full[s], kx, h, m0);
            if (kc >= early) load_b(kc);
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        constexpr uint32_t idesc = idesc_bf16(kBM, BN / L::kHalves, false, kBMN);
        bool ok = true;
        for (int kc = 0; kc < nk && ok; ++kc) {
            const int s = kc % L::kStagesN;
            if (!mbar_wait(&full[s], (kc / L::kStagesN) & 1)) {
                *abort_flag = 1;
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + s * L::kStageBytes);
            const uint32_t sb = sa + L::kABytes;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
                const uint64_t da = smem_desc_sw128(sa + kk * 32, 16, 1024);
#pragma unroll
                for (int j = 0; j < L::kHalves; ++j) {
                    const uint64_t db = kBMN ? smem_desc_sw128(sb + kk * 16 * 128, 64 * 128, 1024)
                                             : smem_desc_sw128(sb + j * (BN / L::kHalves) * 128 + kk * 32, 16, 1024);
                    mma_ss(tmem + j * (BN / L::kHalves), da, db, idesc, (kc | kk) != 0);
                }
            }
            mma_commit(&empty[s]);  // the stage is free once these MMAs have read it
        }
        mma_commit(acc_full);
    } else if (warp >= 2) {
        // ---------------- epilogue: TMEM -> bf16 -> shared staging -> global
        const int q = warp & 3;             // TMEM lane quadrant this warp may access
        const int c_lo = ((warp - 2) >> 2) * (BN / 2), c_hi = c_lo + BN / 2;  // its columns
        const int row = q * 32 + lane;
        const int m = m0 + row;
        // a quadrant without a valid row (fewer than 128 tokens) has nothing to drain
        const bool live = m0 + q * 32 < g.M;
        const int t = threadIdx.x - 64;
        // absorb: the q_rope chunks this thread copies are read while the MMAs run
        constexpr int kRopeMax = 4;  // 16-byte chunks per thread: 128 rows x d_rope <= 128
        uint4 rope[kRopeMax];
        const bool copy_rope = !g.acc && g.rope_src != nullptr && blockIdx.x == 0 && g.d_rope > 0;
        const int rpr = copy_rope ? g.d_rope / 8 : 1;  // 16-byte chunks of a q_rope row
        if (copy_rope) {
#pragma unroll
            for (int i = 0; i < kRopeMax; ++i) {
                const int idx = t + i * kEpiThreads, rr = idx / rpr, ch = idx - rr * rpr;
                rope[i] = make_uint4(0, 0, 0, 0);
                if (rr < kBM && m0 + rr < g.M)
                    rope[i] = __ldg(reinterpret_cast<const uint4 *>(g.rope_src + ((long long)(m0 + rr) * g.H + h) * g.d_rope) + ch);
            }
        }
        const bool ok = live && (nk <= 0 || mbar_wait(acc_full, 0)) && !*abort_flag;
        tc_fence_after();
        const int n_valid = g.N - n0;  // a multiple of 16
        if (g.acc && live) {
            // split K: this CTA's fp32 tile is split blockIdx.z's partial (zeros if it has no K)
            float *prow = g.acc + ((long long)blockIdx.z * g.M + m) * g.N + n0;
            for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(tmem + tmem_lane_base(q) + c0, r);
                tmem_ld_wait();
                if (m < g.M && c0 < n_valid) {
                    float4 *a4 = reinterpret_cast<float4 *>(prow + c0);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        a4[e] = nk <= 0 ? make_float4(0.f, 0.f, 0.f, 0.f)
                                        : make_float4(ok ? __uint_as_float(r[4 * e]) : __int_as_float(0x7fc00000),
                                                      __uint_as_float(r[4 * e + 1]), __uint_as_float(r[4 * e + 2]),
                                                      __uint_as_float(r[4 * e + 3]));
                }
            }
        }
        if (!g.acc) {
            // every MMA has read the ring (acc_full), so it holds the bf16 rows now;
            // the pitch's extra 16 bytes keep the row-per-lane writes conflict-free
            constexpr int kPitch = BN * 2 + 16;
            // two 16-column loads in flight per wait where the half is a multiple of 32
            constexpr int kStep = (BN / 2) % 32 == 0 ? 32 : 16;
            for (int c0 = c_lo; live && c0 < c_hi; c0 += kStep) {
                uint32_t r[kStep];
                tmem_ld16(tmem + tmem_lane_base(q) + c0, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
                if (kStep == 32) tmem_ld16(tmem + tmem_lane_base(q) + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&r[kStep - 16]));
                tmem_ld_wait();
#pragma unroll
                for (int hb = 0; hb < kStep / 16; ++hb) {
                    uint32_t pk[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float lo = ok ? __uint_as_float(r[16 * hb + 2 * e]) : __int_as_float(0x7fc00000);
                        float hi = ok ? __uint_as_float(r[16 * hb + 2 * e + 1]) : __int_as_float(0x7fc00000);
                        pk[e] = pack_bf16x2(lo, hi);
                    }
                    uint4 *d4 = reinterpret_cast<uint4 *>(smem + row * kPitch + (c0 + 16 * hb) * 2);
                    d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
            }
            named_bar(kBarEpi, kEpiThreads);
            const int cpr = min(BN, n_valid) / 8;  // 16-byte chunks of a row
            for (int idx = t; idx < kBM * cpr; idx += kEpiThreads) {
                const int rr = idx / cpr, ch = idx - rr * cpr;
                if (m0 + rr >= g.M) break;  // rows only grow with idx
                *reinterpret_cast<uint4 *>(g.out + ((long long)(m0 + rr) * g.H + h) * g.out_row + n0 + ch * 8) =
                    *reinterpret_cast<const uint4 *>(smem + rr * kPitch + ch * 16);
            }
            if (copy_rope) {
#pragma unroll
                for (int i = 0; i < kRopeMax; ++i) {
                    const int idx = t + i * kEpiThreads, rr = idx / rpr, ch = idx - rr * rpr;
                    if (rr < kBM && m0 + rr < g.M)
                        reinterpret_cast<uint4 *>(g.out + ((long long)(m0 + rr) * g.H + h) * g.out_row + g.N)[ch] = rope[i];
                }
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_free<L::kTmemCols>(tmem);
    }
}

template <int BN, bool kBMN>
cudaError_t launch_proj(const CUtensorMap &tA, const CUtensorMap &tB, const ProjArgs &g, cudaStream_t st) {
    const int smem = ProjSmem<BN, kBMN>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(proj_gemm_tc<BN, kBMN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((g.N + BN - 1) / BN, (g.M + kBM - 1) / kBM, g.acc ? g.splits : g.H);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g.wait_a ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, proj_gemm_tc<BN, kBMN>, tA, tB, g);
}

// A operand [M][H][K] bf16 (K contiguous), box 64 x 1 x 128.
bool map_rows(CUtensorMap *m, const void *base, int M, int H, int K) {
    uint64_t dims[3] = {(uint64_t)K, (uint64_t)H, (uint64_t)M};
    uint64_t strides[2] = {(uint64_t)K * 2, (uint64_t)H * K * 2};
    uint32_t box[3] = {64, 1, kBM};
    return encode_bf16_sw128(m, base, 3, dims, strides, box);
}

}  // namespace

// q_cat = [q_nope . W_UK^T | q_rope]
cudaError_t launch_absorb_q_tc(const mla_dims &d, const void *q_nope, const void *q_rope, const void *w_uk,
                               void *q_cat, cudaStream_t st, bool trigger) {
    const int M = d.B * d.s_q;
    CUtensorMap tA, tB;
    if (!map_rows(&tA, q_nope, M, d.H, d.d_nope)) return cudaErrorInvalidValue;
    // W_UK [H][d_c][d_nope]: K-major B, box 64 (k) x BN (n) x 1
    const int BN = d.d_c >= 256 ? 256 : d.d_c;  // d_c is a multiple of 64: N tiles of 256 (two CTAs an SM)
    uint64_t dims[3] = {(uint64_t)d.d_nope, (uint64_t)d.d_c, (uint64_t)d.H};
    uint64_t strides[2] = {(uint64_t)d.d_nope * 2, (uint64_t)d.d_c * d.d_nope * 2};
    uint32_t box[3] = {64, (uint32_t)(BN > 256 ? 256 : BN), 1};
    if (!encode_bf16_sw128(&tB, w_uk, 3, dims, strides, box)) return cudaErrorInvalidValue;
    ProjArgs g{M, d.H, d.d_c, d.d_nope, (__nv_bfloat16 *)q_cat, d.d_c + d.d_rope,
               d.d_rope ? (const __nv_bfloat16 *)q_rope : nullptr, d.d_rope, nullptr, 0, 1, false, trigger};
    switch (BN) {
        case 256: return launch_proj<256, false>(tA, tB, g, st);
        case 192: return launch_proj<192, false>(tA, tB, g, st);
        case 128: return launch_proj<128, false>(tA, tB, g, st);
        case 64: return launch_proj<64, false>(tA, tB, g, st);
        default: return cudaErrorInvalidValue;
    }
}

// out = o_lat . W_UV
cudaError_t launch_out_proj_tc(const mla_dims &d, const void *o_lat, const void *w_uv, void *out, cudaStream_t st,
                               bool wait_prev) {
    const int M = d.B * d.s_q;
    CUtensorMap tA, tB;
    if (!map_rows(&tA, o_lat, M, d.H, d.d_c)) return cudaErrorInvalidValue;
    // W_UV [H][d_c][d_v]: MN-major B, box 64 (n) x 64 (k) x 1
    uint64_t dims[3] = {(uint64_t)d.d_v, (uint64_t)d.d_c, (uint64_t)d.H};
    uint64_t strides[2] = {(uint64_t)d.d_v * 2, (uint64_t)d.d_c * d.d_v * 2};
    uint32_t box[3] = {64, 64, 1};
    if (!encode_bf16_sw128(&tB, w_uv, 3, dims, strides, box)) return cudaErrorInvalidValue;
    ProjArgs g{M, d.H, d.d_v, d.d_c, (__nv_bfloat16 *)out, d.d_v, nullptr, 0, nullptr, 0, 1, wait_prev, false};
    switch ((d.d_v + 63) / 64 * 64) {  // MMA width: d_v rounded up to whole 64-column boxes
        case 256: return launch_proj<256, true>(tA, tB, g, st);
        case 192: return launch_proj<192, true>(tA, tB, g, st);
        case 128: return launch_proj<128, true>(tA, tB, g, st);
        case 64: return launch_proj<64, true>(tA, tB, g, st);
        default: return cudaErrorNotSupported;
    }
}

// Writes row m = b*s_q + i of the new latents (the sum of the splits' fp32
// partials, rounded to bf16) and its RoPE key into the cache at position
// L_b - s_q + i, contiguous or paged.  One CTA per row: 64 threads per group of
// 8-column chunks, four groups each summing every fourth split, summed through
// shared memory (the partials' loads are independent, not one chain).
constexpr int kScatterThreads = 256;
// Four values as E4M3 codes (value 0 in the low byte): round to nearest even,
// saturating at +-448.
__device__ __forceinline__ uint32_t pack_e4m3x4(float v0, float v1, float v2, float v3) {
    unsigned short lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(v1), "f"(v0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(v3), "f"(v2));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

__global__ void __launch_bounds__(kScatterThreads) append_scatter(AttnParams p, const float *part, int splits,
                                                                  const __nv_bfloat16 *k_rope) {
    __shared__ float red[3][512];
    const int m = blockIdx.x;
    const int M = p.B * p.s_q;
    const int b = m / p.s_q, i = m % p.s_q;
    const int L = __ldg(p.seq_lens + b);
    if (!seq_len_ok(p, L)) {
        if (threadIdx.x == 0) set_status(p.status, MLA_ERR_SEQLEN);
        return;
    }
    // the row's element offset in the cache (bf16 values or E4M3 codes)
    const int pos = L - p.s_q + i;
    const long long W = p.d_c + p.d_rope;
    long long at;
    if (p.block_table == nullptr) {
        at = (long long)b * p.seq_stride + (long long)pos * W;
    } else {
        const int page = __ldg(p.block_table + (long long)b * p.max_pages + pos / p.page_size);
        if (page < 0 || page >= p.num_pages) {
            if (threadIdx.x == 0) set_status(p.status, MLA_ERR_PAGE);
            return;
        }
        at = ((long long)page * p.page_size + pos % p.page_size) * W;
    }
    const int grp = threadIdx.x / 64, c = 8 * (threadIdx.x % 64);  // d_c <= 512: one chunk per thread
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (c < p.d_c) {
        for (int s = grp; s < splits; s += 4) {
            const float *src = part + ((long long)s * M + m) * p.d_c + c;
            const float4 u = *reinterpret_cast<const float4 *>(src);
            const float4 w = *reinterpret_cast<const float4 *>(src + 4);
            a[0] += u.x; a[1] += u.y; a[2] += u.z; a[3] += u.w;
            a[4] += w.x; a[5] += w.y; a[6] += w.z; a[7] += w.w;
        }
        if (grp > 0)
            for (int e = 0; e < 8; ++e) red[grp - 1][c + e] = a[e];
    }
    __syncthreads();
    if (p.kv_fp8) {
        // FP8 cache: the code of value / kv_scale for every element, RoPE key included
        uint8_t *dst = const_cast<uint8_t *>(static_cast<const uint8_t *>(p.kv)) + at;
        const float s = p.kv_scale;
        if (grp == 0 && c < p.d_c) {
            for (int e = 0; e < 8; ++e) a[e] += red[0][c + e] + red[1][c + e] + red[2][c + e];
            *reinterpret_cast<uint2 *>(dst + c) = make_uint2(pack_e4m3x4(a[0] / s, a[1] / s, a[2] / s, a[3] / s),
                                                             pack_e4m3x4(a[4] / s, a[5] / s, a[6] / s, a[7] / s));
        }
        if (grp == 1 && c < p.d_rope) {
            const uint4 u = *reinterpret_cast<const uint4 *>(k_rope + (long long)m * p.d_rope + c);
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
            float f[8];
            for (int e = 0; e < 4; ++e) {
                const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[e]));
                f[2 * e] = v.x / s;
                f[2 * e + 1] = v.y / s;
            }
            *reinterpret_cast<uint2 *>(dst + p.d_c + c) =
                make_uint2(pack_e4m3x4(f[0], f[1], f[2], f[3]), pack_e4m3x4(f[4], f[5], f[6], f[7]));
        }
        return;
    }
    __nv_bfloat16 *dst = const_cast<__nv_bfloat16 *>(static_cast<const __nv_bfloat16 *>(p.kv)) + at;
    if (grp == 0 && c < p.d_c) {
        for (int e = 0; e < 8; ++e) a[e] += red[0][c + e] + red[1][c + e] + red[2][c + e];
        *reinterpret_cast<uint4 *>(dst + c) = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                                                          pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
    }
    if (grp == 1 && c < p.d_rope)
        *reinterpret_cast<uint4 *>(dst + p.d_c + c) =
            *reinterpret_cast<const uint4 *>(k_rope + (long long)m * p.d_rope + c);
}

// c = x . W_DKV for the batch's new tokens, appended with their RoPE keys.  The
// GEMM is weight-bound (every W_DKV byte read once), so K is split over enough
// CTAs to stream the weight at full bandwidth (append_splits); each split stores
// its fp32 partial tile in `part`, and the scatter sums them into the cache rows.
cudaError_t launch_cache_append_tc(const AttnParams &p, int d_model, const void *x, const void *w_dkv,
                                   const void *k_rope, float *part, cudaStream_t st) {
    const int M = p.B * p.s_q;
    if (M == 0) return cudaSuccess;
    CUtensorMap tA, tB;
    if (!map_rows(&tA, x, M, 1, d_model)) return cudaErrorInvalidValue;
    // W_DKV [d_model][d_c]: MN-major B, box 64 (n) x 64 (k) x 1
    uint64_t dims[3] = {(uint64_t)p.d_c, (uint64_t)d_model, 1};
    uint64_t strides[2] = {(uint64_t)p.d_c * 2, (uint64_t)d_model * p.d_c * 2};
    uint32_t box[3] = {64, 64, 1};
    if (!encode_bf16_sw128(&tB, w_dkv, 3, dims, strides, box)) return cudaErrorInvalidValue;
    const AppendPlan plan = append_plan(M, p.d_c, d_model);
    ProjArgs g{M, 1, p.d_c, d_model, nullptr, 0, nullptr, 0, part, plan.kc_per_cta, plan.splits, false, false};
    cudaError_t e = launch_proj<64, true>(tA, tB, g, st);
    if (e != cudaSuccess) return e;
    append_scatter<<<M, kScatterThreads, 0, st>>>(p, part, plan.splits, (const __nv_bfloat16 *)k_rope);
    return cudaGetLastError();
}

}  // namespace mla
