// The prefill "expand" form's projections ("Why MLA and MTP Fight Each Other",
// sections 5.3 and 5.5; "MLA, dim by dim", MLA prefill: materialise K, V from
// the latent, then run standard attention).  For every cached token j < L_b of
// every sequence b and every head h:
//   K_h[j] = c_kv[j] . W_UK[h]   (d_nope)     V_h[j] = c_kv[j] . W_UV[h]   (d_v)
// written as one expanded row [V_h | K_h | k_rope_j] of W_e = d_v + d_nope + d_rope
// elements at exp[b][h][j]; the per-head attention (launch_attn_expand) then
// contracts [q_nope | q_rope] with the row's channels [d_v, W_e) and sums P over
// its first d_v channels.
//
// One CTA per (128 tokens, head, sequence): D[128 x (d_v + d_nope)] =
// C[128 x d_c] . [W_UV[h] | W_UK[h]] on the tcgen05 tensor cores, the fp32
// accumulator in tensor memory, a 4-stage TMA ring of 64-wide K slices (A: two
// 64-row boxes of cache rows, through the block table when paged; B: 64-column
// boxes of the two weights, MN-major).  Warp 0 loads, warp 1 owns tensor memory
// and issues the MMAs, warps 2-5 write the rows.
#include "common.cuh"
#include "launch.h"
#include "sm100.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace sm100;

constexpr int kBM = 128, kBK = 64, kStages = 4, kThreads = 192;
constexpr int kBN = 256;  // d_v + d_nope at most
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kBN * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 1024;

struct ExpandArgs {
    AttnParams p;
    int d_nope, d_v, W, We;     // cache row width W = d_c + d_rope, expanded row width We
    __nv_bfloat16 *exp;         // [B][H][capacity][We]
};

__global__ void __launch_bounds__(kThreads, 1)
    expand_kv_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmK, const ExpandArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint64_t *empty = full + kStages;
    uint64_t *acc_full = empty + kStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const AttnParams &p = a.p;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t0 = blockIdx.x * kBM, h = blockIdx.y, b = blockIdx.z;
    const int L = __ldg(p.seq_lens + b);
    if (!seq_len_ok(p, L)) {
        if (threadIdx.x == 0 && t0 == 0 && h == 0) set_status(p.status, MLA_ERR_SEQLEN);
        return;
    }
    if (t0 >= L) return;  // no token of this tile is cached yet
    const int N = a.d_v + a.d_nope;
    const int nk = (p.d_c + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmK);
    }
    if (warp == 1) tmem_alloc<256>(tmem_slot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        // row coordinate of the 64 tokens from t: the contiguous cache (y = t, z = b)
        // or the pool row of its page (pages hold whole 64-token tiles); rows past
        // the table or on a page outside the pool read as zeros
        int y[2];
        for (int hb = 0; hb < 2; ++hb) {
            const int t = t0 + 64 * hb;
            if (p.block_table == nullptr) {
                y[hb] = t;
            } else {
                const int pi = t / p.page_size;
                const int page = pi < p.max_pages ? __ldg(p.block_table + (long long)b * p.max_pages + pi) : -1;
                if (page >= 0 && page < p.num_pages) {
                    y[hb] = page * p.page_size + t % p.page_size;
                } else {
                    if (t < L) set_status(p.status, MLA_ERR_PAGE);
                    y[hb] = p.num_pages * p.page_size;
                }
            }
        }
        for (int kc = 0; kc < nk; ++kc) {
            const int s = kc % kStages;
            if (kc >= kStages && !mbar_wait(&empty[s], ((kc / kStages) - 1) & 1)) {
                *abort_flag = 1;
                break;
            }
            uint8_t *sa = smem + s * kStageBytes;
            uint8_t *sb = sa + kABytes;
            const int kx = kc * kBK;
            mbar_arrive_expect_tx(&full[s], kABytes + N * kBK * 2);
            for (int hb = 0; hb < 2; ++hb) {
                if (p.block_table == nullptr) tma_load_3d(sa + hb * 64 * 128, &tmA, &full[s], kx, y[hb], b);
                else tma_load_2d(sa + hb * 64 * 128, &tmA, &full[s], kx, y[hb]);
            }
            for (int j = 0; j < a.d_v / 64; ++j) tma_load_3d(sb + j * 64 * 128, &tmV, &full[s], 64 * j, kx, h);
            for (int j = 0; j < a.d_nope / 64; ++j)
                tma_load_3d(sb + (a.d_v / 64 + j) * 64 * 128, &tmK, &full[s], 64 * j, kx, h);
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        const uint32_t idesc = idesc_bf16(kBM, N, false, true);
        bool ok = true;
        for (int kc = 0; kc < nk && ok; ++kc) {
            const int s = kc % kStages;
            if (!mbar_wait(&full[s], (kc / kStages) & 1)) {
                *abort_flag = 1;
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + s * kStageBytes);
            const uint32_t sb = sa + kABytes;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
                mma_ss(tmem, smem_desc_sw128(sa + kk * 32, 16, 1024), smem_desc_sw128(sb + kk * 16 * 128, 64 * 128, 1024),
                       idesc, (kc | kk) != 0);
            mma_commit(&empty[s]);
        }
        mma_commit(acc_full);
    } else if (warp >= 2) {
        // ---------------- epilogue: TMEM -> bf16 expanded rows
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const int row = q * 32 + lane;
        const int t = t0 + row;
        const bool ok = mbar_wait(acc_full, 0) && !*abort_flag;
        tc_fence_after();
        const bool store = ok && t < L;
        __nv_bfloat16 *dst = a.exp + (((long long)b * p.H + h) * p.capacity + t) * a.We;
        for (int c0 = 0; c0 < N; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(tmem + tmem_lane_base(q) + c0, r);
            tmem_ld_wait();
            if (store) {
                uint32_t pk[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + c0);  // V_h then K_h: TMEM columns = row channels
                d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
        }
        if (store && p.d_rope > 0) {  // the token's RoPE key, shared by every head
            const __nv_bfloat16 *src = kv_row(p, b, t);
            if (src != nullptr) {
                const uint4 *s4 = reinterpret_cast<const uint4 *>(src + p.d_c);
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + N);
                for (int e = 0; e < p.d_rope / 8; ++e) d4[e] = s4[e];
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_free<256>(tmem);
    }
}

__global__ void concat_q(const __nv_bfloat16 *q_nope, const __nv_bfloat16 *q_rope, __nv_bfloat16 *q_exp,
                         long long rows, int d_nope, int d_rope) {
    const int w = d_nope + d_rope;
    const long long total = rows * (w / 8);
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
        const long long r = i / (w / 8);
        const int c = (int)(i % (w / 8)) * 8;
        const uint4 v = c < d_nope ? *reinterpret_cast<const uint4 *>(q_nope + r * d_nope + c)
                                   : *reinterpret_cast<const uint4 *>(q_rope + r * d_rope + (c - d_nope));
        *reinterpret_cast<uint4 *>(q_exp + r * w + c) = v;
    }
}

}  // namespace

cudaError_t launch_expand_kv(const AttnParams &p, int d_nope, int d_v, const void *w_uk, const void *w_uv, void *exp,
                             cudaStream_t st) {
    const int W = p.d_c + p.d_rope;
    if (d_v % 64 || d_nope % 64 || d_v + d_nope > kBN || p.kv_fp8) return cudaErrorNotSupported;
    ExpandArgs a{p, d_nope, d_v, W, d_v + d_nope + p.d_rope, static_cast<__nv_bfloat16 *>(exp)};
    CUtensorMap tA, tV, tK;
    if (p.block_table == nullptr) {
        uint64_t dims[3] = {(uint64_t)W, (uint64_t)p.capacity, (uint64_t)p.B};
        uint64_t strides[2] = {(uint64_t)W * 2, (uint64_t)p.seq_stride * 2};
        uint32_t box[3] = {64, 64, 1};
        if (!encode_bf16_sw128(&tA, p.kv, 3, dims, strides, box)) return cudaErrorInvalidValue;
    } else {
        uint64_t dims[2] = {(uint64_t)W, (uint64_t)p.num_pages * p.page_size};
        uint64_t strides[1] = {(uint64_t)W * 2};
        uint32_t box[2] = {64, 64};
        if (!encode_bf16_sw128(&tA, p.kv, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    // W_UV [H][d_c][d_v] and W_UK [H][d_c][d_nope]: MN-major B, boxes of 64 (n) x 64 (k) x 1
    {
        uint64_t dims[3] = {(uint64_t)d_v, (uint64_t)p.d_c, (uint64_t)p.H};
        uint64_t strides[2] = {(uint64_t)d_v * 2, (uint64_t)p.d_c * d_v * 2};
        uint32_t box[3] = {64, 64, 1};
        if (!encode_bf16_sw128(&tV, w_uv, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        uint64_t dims[3] = {(uint64_t)d_nope, (uint64_t)p.d_c, (uint64_t)p.H};
        uint64_t strides[2] = {(uint64_t)d_nope * 2, (uint64_t)p.d_c * d_nope * 2};
        uint32_t box[3] = {64, 64, 1};
        if (!encode_bf16_sw128(&tK, w_uk, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(expand_kv_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid((p.capacity + kBM - 1) / kBM, p.H, p.B);
    expand_kv_tc<<<grid, kThreads, kSmemBytes, st>>>(tA, tV, tK, a);
    return cudaGetLastError();
}

cudaError_t launch_concat_q(const mla_dims &d, const void *q_nope, const void *q_rope, void *q_exp, cudaStream_t st) {
    const long long rows = (long long)d.B * d.s_q * d.H;
    if (rows == 0) return cudaSuccess;
    const long long units = rows * ((d.d_nope + d.d_rope) / 8);
    const int blocks = (int)((units + 255) / 256 < 4096 ? (units + 255) / 256 : 4096);
    concat_q<<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(q_nope),
                                     static_cast<const __nv_bfloat16 *>(q_rope), static_cast<__nv_bfloat16 *>(q_exp),
                                     rows, d.d_nope, d.d_rope);
    return cudaGetLastError();
}

}  // namespace mla
