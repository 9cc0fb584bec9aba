// Kernel launchers shared between translation units of the MLA library.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {

// trigger: let the next grid (launched programmatically) start its CTAs at once;
// wait_prev: this grid is launched programmatically after the attention and
// reads o_lat only once that grid has completed.
cudaError_t launch_absorb_q_tc(const mla_dims &d, const void *q_nope, const void *q_rope, const void *w_uk,
                               void *q_cat, cudaStream_t st, bool trigger = false);
cudaError_t launch_out_proj_tc(const mla_dims &d, const void *o_lat, const void *w_uv, void *out, cudaStream_t st,
                               bool wait_prev = false);
// Split-K plan of the cache append's down-projection: 64-column N tiles, and
// K (d_model, in 64-wide chunks) cut so that all tiles together make about one
// CTA per SM.  Partials: splits * M * d_c fp32.
struct AppendPlan {
    int kc_per_cta, splits;
};
inline AppendPlan append_plan(int M, int d_c, int d_model) {
    const int nk = (d_model + 63) / 64;
    const int tiles = ((d_c + 63) / 64) * ((M + 127) / 128);
    int per = (nk * tiles + 147) / 148;
    if (per < 1) per = 1;
    return AppendPlan{per, (nk + per - 1) / per};
}
cudaError_t launch_cache_append_tc(const AttnParams &p, int d_model, const void *x, const void *w_dkv,
                                   const void *k_rope, float *part, cudaStream_t st);
cudaError_t launch_attn_tc(const AttnParams &p, cudaStream_t st);
cudaError_t launch_attn_persist(const AttnParams &p, cudaStream_t st);
cudaError_t launch_attn_expand(const AttnParams &p, cudaStream_t st);
// Expanded rows [V_h | K_h | k_rope] of every cached token < seq_lens[b] of every
// sequence and head (the prefill "expand" form), into exp [B][H][capacity][W_e].
cudaError_t launch_expand_kv(const AttnParams &p, int d_nope, int d_v, const void *w_uk, const void *w_uv, void *exp,
                             cudaStream_t st);
// q_exp [B][s_q][H][d_nope + d_rope] = [q_nope | q_rope]
cudaError_t launch_concat_q(const mla_dims &d, const void *q_nope, const void *q_rope, void *q_exp, cudaStream_t st);

cudaError_t launch_attn_combine(const AttnParams &p, cudaStream_t st);
cudaError_t launch_naive(const AttnParams &p, int d_nope, int d_v, const void *q_nope, const void *q_rope,
                         const void *w_uk, const void *w_uv, void *out, float *lse, void *kv_scratch,
                         cudaStream_t st);

}  // namespace mla
