// Naive decompress-then-attend decode: the comparison path.
// ("The MLA decode speedup hiding in your model card", "The naive form, written
// out": up-project every cached latent to per-head K and V, then attend.)
#include "common.cuh"
#include "launch.h"

namespace mla {

// K[b,h,j,:] = c_kv[b,j,:] . W_UK[h]  and  V[b,h,j,:] = c_kv[b,j,:] . W_UV[h]
// for j < seq_lens[b]; a 64x64 output tile per CTA, 256 threads, 4x4 per thread.
// grid (ceil(capacity/64), ceil(max(d_nope, d_v)/64) * 2, B*H); y picks K or V.
__global__ void __launch_bounds__(256) naive_decompress(AttnParams p, int d_nope, int d_v,
                                                        const __nv_bfloat16 *__restrict__ w_uk,
                                                        const __nv_bfloat16 *__restrict__ w_uv,
                                                        __nv_bfloat16 *__restrict__ Kbuf,
                                                        __nv_bfloat16 *__restrict__ Vbuf) {
    __shared__ float As[16][64 + 1];
    __shared__ float Bs[16][64 + 1];
    const int bh = blockIdx.z, b = bh / p.H, h = bh % p.H;
    const int L = __ldg(p.seq_lens + b);
    if (!seq_len_ok(p, L)) return;
    const int j0 = blockIdx.x * 64;
    if (j0 >= L) return;
    const int nblk = (max(d_nope, d_v) + 63) / 64;
    const bool isV = blockIdx.y >= nblk;
    const int n0 = (blockIdx.y % nblk) * 64;
    const int N = isV ? d_v : d_nope;
    if (n0 >= N) return;
    const __nv_bfloat16 *Wm = (isV ? w_uv : w_uk) + (long long)h * p.d_c * N;
    __nv_bfloat16 *out = (isV ? Vbuf : Kbuf) + (long long)bh * p.capacity * N;

    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < p.d_c; k0 += 16) {
        for (int e = threadIdx.x; e < 64 * 16; e += 256) {
            int jj = e / 16, kk = e % 16;
            int j = j0 + jj;
            float v = 0.f;
            if (j < L) {
                const __nv_bfloat16 *row = kv_row(p, b, j);
                if (row) v = __bfloat162float(row[k0 + kk]);
            }
            As[kk][jj] = v;
            int kk2 = e / 64, nn = e % 64;
            Bs[kk2][nn] = (n0 + nn < N) ? __bfloat162float(Wm[(long long)(k0 + kk2) * N + n0 + nn]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], bb[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) { a[u] = As[kk][ty * 4 + u]; bb[u] = Bs[kk][tx * 4 + u]; }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] += a[u] * bb[v];
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        int j = j0 + ty * 4 + u;
        if (j >= L) continue;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            int n = n0 + tx * 4 + v;
            if (n < N) out[(long long)j * N + n] = __float2bfloat16_rn(acc[u][v]);
        }
    }
}

// Standard attention over the materialised K, V with the shared RoPE key appended:
//   s_j = scale (q_nope . K_j + q_rope . k_rope_j),  out = sum_j softmax(s)_j V_j.
// One CTA (128 threads) per (b, i, h); 128-token chunks with an online softmax.
__global__ void __launch_bounds__(128) naive_attend(AttnParams p, int d_nope, int d_v,
                                                    const __nv_bfloat16 *__restrict__ q_nope,
                                                    const __nv_bfloat16 *__restrict__ q_rope,
                                                    const __nv_bfloat16 *__restrict__ Kbuf,
                                                    const __nv_bfloat16 *__restrict__ Vbuf,
                                                    __nv_bfloat16 *__restrict__ out, float *__restrict__ lse) {
    __shared__ float qn[256], qr[64];
    __shared__ float pj[128];
    __shared__ float red[4];
    const long long grow = blockIdx.x;  // (b*s_q + i)*H + h
    const int h = (int)(grow % p.H);
    const long long bi = grow / p.H;
    const int i = (int)(bi % p.s_q), b = (int)(bi / p.s_q);
    const int L = __ldg(p.seq_lens + b);
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    if (!seq_len_ok(p, L)) {
        if (tid == 0) set_status(p.status, MLA_ERR_SEQLEN);
        for (int v = tid; v < d_v; v += 128) out[grow * d_v + v] = __float2bfloat16_rn(0.f);
        if (tid == 0) lse[grow] = -INFINITY;
        return;
    }
    for (int n = tid; n < d_nope; n += 128) qn[n] = __bfloat162float(q_nope[grow * d_nope + n]);
    for (int k = tid; k < p.d_rope; k += 128) qr[k] = __bfloat162float(q_rope[grow * p.d_rope + k]);
    __syncthreads();
    const long long bh = (long long)b * p.H + h;
    const __nv_bfloat16 *K = Kbuf + bh * p.capacity * d_nope;
    const __nv_bfloat16 *V = Vbuf + bh * p.capacity * d_v;
    const int n_vis = L - p.s_q + i + 1;
    float m = -INFINITY, l = 0.f;
    float acc[2] = {0.f, 0.f};  // columns v = tid, tid + 128
    for (int j0 = 0; j0 < n_vis; j0 += 128) {
        int j = j0 + tid;
        float s = -INFINITY;
        if (j < n_vis) {
            float d = 0.f;
            for (int n = 0; n < d_nope; ++n) d += qn[n] * __bfloat162float(K[(long long)j * d_nope + n]);
            const __nv_bfloat16 *row = kv_row(p, b, j);
            if (row) {
                for (int k = 0; k < p.d_rope; ++k) d += qr[k] * __bfloat162float(row[p.d_c + k]);
            } else {
                set_status(p.status, MLA_ERR_PAGE);
            }
            s = d * p.scale;
        }
        float mx = s;
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) red[warp] = mx;
        __syncthreads();
        mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
        __syncthreads();
        float m_new = fmaxf(m, mx);
        float e = (s == -INFINITY) ? 0.f : __expf(s - m_new);
        pj[tid] = e;
        float sum = e;
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) red[warp] = sum;
        __syncthreads();
        sum = red[0] + red[1] + red[2] + red[3];
        float a = (m == -INFINITY) ? 0.f : __expf(m - m_new);
        l = l * a + sum;
        m = m_new;
        int jn = min(128, n_vis - j0);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            int v = tid + 128 * u;
            if (v < d_v) {
                float x = acc[u] * a;
                for (int jj = 0; jj < jn; ++jj) {
                    float w = pj[jj];
                    if (w != 0.f) x += w * __bfloat162float(V[(long long)(j0 + jj) * d_v + v]);
                }
                acc[u] = x;
            }
        }
        __syncthreads();
    }
    float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        int v = tid + 128 * u;
        if (v < d_v) out[grow * d_v + v] = __float2bfloat16_rn(acc[u] * inv);
    }
    if (tid == 0) lse[grow] = l > 0.f ? m + __logf(l) : -INFINITY;
}

cudaError_t launch_naive(const AttnParams &p, int d_nope, int d_v, const void *q_nope, const void *q_rope,
                         const void *w_uk, const void *w_uv, void *out, float *lse, void *kv_scratch,
                         cudaStream_t st) {
    __nv_bfloat16 *Kbuf = (__nv_bfloat16 *)kv_scratch;
    __nv_bfloat16 *Vbuf = Kbuf + (long long)p.B * p.H * p.capacity * d_nope;
    int nblk = (max(d_nope, d_v) + 63) / 64;
    dim3 g1((p.capacity + 63) / 64, 2 * nblk, p.B * p.H);
    naive_decompress<<<g1, 256, 0, st>>>(p, d_nope, d_v, (const __nv_bfloat16 *)w_uk,
                                         (const __nv_bfloat16 *)w_uv, Kbuf, Vbuf);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    naive_attend<<<(unsigned)((long long)p.B * p.s_q * p.H), 128, 0, st>>>(
        p, d_nope, d_v, (const __nv_bfloat16 *)q_nope, (const __nv_bfloat16 *)q_rope, Kbuf, Vbuf,
        (__nv_bfloat16 *)out, lse);
    return cudaGetLastError();
}

}  // namespace mla
