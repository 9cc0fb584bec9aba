// Cross-split log-sum-exp combine of the attention partials ("Why MLA and MTP
// Fight Each Other", section 4: flash decoding splits the history and merges
// the partial softmax states).  For every row, the splits' (acc, m, l) merge as
//   M = max_s m_s,  L = sum_s l_s e^(m_s - M),  o = sum_s acc_s e^(m_s - M) / L,
//   lse = M + ln L.
// Rows of a pair-split attention carry one (m, l) per CTA: columns [0, 256) use
// the first, the rest the second.
#include "common.cuh"
#include "launch.h"

namespace mla {

__global__ void attn_combine(AttnParams p) {
    const int rows = p.s_q * p.H;
    // partial sequence b (its pieces' rows) and the sequence bo it belongs to
    const int b = (int)(blockIdx.x / rows), rr = (int)(blockIdx.x % rows);
    const int pos = p.combine_b0 + b;
    const int bo = p.order != nullptr ? p.order[pos] : pos;
    if (bo < 0 || bo >= p.combine_b0 + p.B) return;  // positions and sequences are both 0 .. B-1
    const long long grow = (long long)bo * rows + rr;
    const int S = p.num_splits;
    // columns [0, 256) are relative to the (m, l) of half 0, the rest to half 1
    const int halves = p.d_c > 256 ? 2 : 1;
    float M[2] = {-INFINITY, -INFINITY}, Lsum[2] = {0.f, 0.f};
    for (int h = 0; h < halves; ++h) {
        for (int s = 0; s < S; ++s) {
            const long long prow = ((long long)b * S + s) * rows + rr;
            M[h] = fmaxf(M[h], p.part_ml[(prow * 2 + h) * 2]);
        }
        for (int s = 0; s < S; ++s) {
            const long long prow = ((long long)b * S + s) * rows + rr;
            const float m = p.part_ml[(prow * 2 + h) * 2];
            if (m != -INFINITY) Lsum[h] += p.part_ml[(prow * 2 + h) * 2 + 1] * __expf(m - M[h]);
        }
    }
    for (int c = threadIdx.x; c < p.d_c; c += blockDim.x) {
        const int h = c < 256 ? 0 : 1;
        float o = 0.f;
        for (int s = 0; s < S; ++s) {
            const long long prow = ((long long)b * S + s) * rows + rr;
            const float m = p.part_ml[(prow * 2 + h) * 2];
            if (m != -INFINITY) o += p.part_acc[prow * p.d_c + c] * __expf(m - M[h]);
        }
        p.o_lat[grow * p.d_c + c] = __float2bfloat16_rn(Lsum[h] > 0.f ? o / Lsum[h] : 0.f);
    }
    if (threadIdx.x == 0) p.lse[grow] = Lsum[0] > 0.f ? M[0] + __logf(Lsum[0]) : -INFINITY;
}

cudaError_t launch_attn_combine(const AttnParams &p, cudaStream_t st) {
    const long long rows = (long long)p.B * p.s_q * p.H;
    attn_combine<<<(unsigned)rows, 128, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace mla
