// CUDA-core split attention (the first, correctness-first version) and the
// cross-split log-sum-exp combine.
#include "common.cuh"
#include "launch.h"

namespace mla {

// ----------------------------------------------------------------------------
// Split attention, one CTA per (row block of 16 query rows, split, sequence).
// Rows r = i*H + h of sequence b.  Online softmax over 32-token tiles; masked
// and out-of-range tokens are never multiplied (their cache rows may hold NaN).
// ----------------------------------------------------------------------------
constexpr int kSR = 16;   // query rows per CTA
constexpr int kST = 32;   // tokens per tile

__global__ void __launch_bounds__(256) attn_split_simple(AttnParams p) {
    extern __shared__ float dyn[];
    const int W = p.d_c + p.d_rope;
    const int KS = W + 2;  // padded row stride of the token tile (conflict-free column reads)
    float (*ps)[kST] = reinterpret_cast<float (*)[kST]>(dyn);          // [kSR][kST]
    float *alpha_s = dyn + kSR * kST;                                   // [kSR]
    float *m_s = alpha_s + kSR, *l_s = m_s + kSR;                       // [kSR] each
    int *tok_ok = reinterpret_cast<int *>(l_s + kSR);                   // [kST]
    float *qs_flat = reinterpret_cast<float *>(tok_ok + kST);           // [kSR][W]
    __nv_bfloat16 *ks_flat = reinterpret_cast<__nv_bfloat16 *>(qs_flat + kSR * W);  // [kST][KS]
#define qs(r, k) qs_flat[(r) * W + (k)]
#define ks(j, k) ks_flat[(j) * KS + (k)]

    const int b = blockIdx.z, split = blockIdx.y, r0 = blockIdx.x * kSR;
    const int rows = p.s_q * p.H;
    const int tid = threadIdx.x;
    const int L = __ldg(p.seq_lens + b);
    const bool valid = seq_len_ok(p, L);
    if (!valid && split == 0 && r0 == 0 && tid == 0) set_status(p.status, MLA_ERR_SEQLEN);

    int t0 = 0, t1 = 0;
    if (valid) split_range(L, p.num_splits, split, t0, t1);

    for (int e = tid; e < kSR * W; e += blockDim.x) {
        int r = e / W, k = e % W;
        int rr = r0 + r;
        qs(r, k) = rr < rows ? __bfloat162float(p.q_cat[((long long)b * rows + rr) * W + k]) : 0.f;
    }
    if (tid < kSR) { m_s[tid] = -INFINITY; l_s[tid] = 0.f; }

    // accumulators: thread owns columns c = tid + 256*u (u < 2) for all kSR rows
    float acc[kSR][2];
#pragma unroll
    for (int r = 0; r < kSR; ++r) { acc[r][0] = 0.f; acc[r][1] = 0.f; }
    __syncthreads();

    for (int j0 = t0; j0 < t1; j0 += kST) {
        // load the tile; tokens outside [t0, t1) or on a bad page are flagged off
        if (tid < kST) {
            int j = j0 + tid;
            int ok = 0;
            if (j < t1) {
                const __nv_bfloat16 *row = kv_row(p, b, j);
                if (row) ok = 1;
                else set_status(p.status, MLA_ERR_PAGE);
            }
            tok_ok[tid] = ok;
        }
        __syncthreads();
        for (int e = tid; e < kST * W; e += blockDim.x) {
            int jj = e / W, k = e % W;
            __nv_bfloat16 v = __float2bfloat16_rn(0.f);
            if (tok_ok[jj]) v = kv_row(p, b, j0 + jj)[k];
            ks(jj, k) = v;
        }
        __syncthreads();
        // scores
        for (int e = tid; e < kSR * kST; e += blockDim.x) {
            int r = e / kST, jj = e % kST;
            int rr = r0 + r;
            int i = rr / p.H;
            int j = j0 + jj;
            float s = -INFINITY;
            if (rr < rows && tok_ok[jj] && j <= L - p.s_q + i) {
                float d = 0.f;
                for (int k = 0; k < W; ++k) d += qs(r, k) * __bfloat162float(ks(jj, k));
                s = d * p.scale;
            }
            ps[r][jj] = s;
        }
        __syncthreads();
        // online softmax: warp w handles rows 2w, 2w+1; lane = token
        {
            int warp = tid / 32, lane = tid % 32;
            for (int r = warp * 2; r < warp * 2 + 2; ++r) {
                float s = ps[r][lane];
                float mx = s;
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                float m_old = m_s[r];
                float m_new = fmaxf(m_old, mx);
                float pj = (s == -INFINITY) ? 0.f : __expf(s - m_new);
                float sum = pj;
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                float a = (m_old == -INFINITY) ? 0.f : __expf(m_old - m_new);
                __syncwarp();
                ps[r][lane] = pj;
                if (lane == 0) {
                    alpha_s[r] = a;
                    m_s[r] = m_new;
                    l_s[r] = l_s[r] * a + sum;
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            int c = tid + 256 * u;
            if (c < p.d_c) {
#pragma unroll
                for (int r = 0; r < kSR; ++r) {
                    float a = acc[r][u] * alpha_s[r];
                    for (int jj = 0; jj < kST; ++jj) {
                        float pj = ps[r][jj];
                        if (pj != 0.f) a += pj * __bfloat162float(ks(jj, c));
                    }
                    acc[r][u] = a;
                }
            }
        }
        __syncthreads();
    }

    // epilogue
    for (int r = 0; r < kSR; ++r) {
        int rr = r0 + r;
        if (rr >= rows) break;
        float m = m_s[r], l = l_s[r];
        long long grow = (long long)b * rows + rr;
        if (p.num_splits == 1) {
            float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                int c = tid + 256 * u;
                if (c < p.d_c) p.o_lat[grow * p.d_c + c] = __float2bfloat16_rn(acc[r][u] * inv);
            }
            if (tid == 0) p.lse[grow] = l > 0.f ? m + __logf(l) : -INFINITY;
        } else {
            long long prow = ((long long)b * p.num_splits + split) * rows + rr;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                int c = tid + 256 * u;
                if (c < p.d_c) p.part_acc[prow * p.d_c + c] = acc[r][u];
            }
            if (tid == 0) {
                p.part_ml[prow * 2 + 0] = m;
                p.part_ml[prow * 2 + 1] = l;
            }
        }
    }
#undef qs
#undef ks
}

// Cross-split merge, one CTA (128 threads) per (b, row):
//   M = max m_s,  L = sum l_s e^{m_s - M},  o = sum acc_s e^{m_s - M} / L,  lse = M + ln L.
__global__ void attn_combine(AttnParams p) {
    const int rows = p.s_q * p.H;
    const long long grow = blockIdx.x;
    const int b = (int)(grow / rows), rr = (int)(grow % rows);
    const int S = p.num_splits;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) {
        long long prow = ((long long)b * S + s) * rows + rr;
        M = fmaxf(M, p.part_ml[prow * 2]);
    }
    float Lsum = 0.f;
    for (int s = 0; s < S; ++s) {
        long long prow = ((long long)b * S + s) * rows + rr;
        float m = p.part_ml[prow * 2];
        if (m != -INFINITY) Lsum += p.part_ml[prow * 2 + 1] * __expf(m - M);
    }
    float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    for (int c = threadIdx.x; c < p.d_c; c += blockDim.x) {
        float o = 0.f;
        for (int s = 0; s < S; ++s) {
            long long prow = ((long long)b * S + s) * rows + rr;
            float m = p.part_ml[prow * 2];
            if (m != -INFINITY) o += p.part_acc[prow * p.d_c + c] * __expf(m - M);
        }
        p.o_lat[grow * p.d_c + c] = __float2bfloat16_rn(o * inv);
    }
    if (threadIdx.x == 0) p.lse[grow] = Lsum > 0.f ? M + __logf(Lsum) : -INFINITY;
}

// ----------------------------------------------------------------------------
cudaError_t launch_attn_simple(const AttnParams &p, cudaStream_t st) {
    int rows = p.s_q * p.H;
    dim3 grid((rows + kSR - 1) / kSR, p.num_splits, p.B);
    const int W = p.d_c + p.d_rope;
    size_t smem = sizeof(float) * (kSR * kST + 3 * kSR) + sizeof(int) * kST + sizeof(float) * kSR * W +
                  sizeof(__nv_bfloat16) * kST * (W + 2);
    cudaError_t e0 = cudaFuncSetAttribute(attn_split_simple, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e0 != cudaSuccess) return e0;
    attn_split_simple<<<grid, 256, smem, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.num_splits == 1) return e;
    return launch_attn_combine(p, st);
}

cudaError_t launch_attn_combine(const AttnParams &p, cudaStream_t st) {
    const long long rows = (long long)p.B * p.s_q * p.H;
    attn_combine<<<(unsigned)rows, 128, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace mla
