// Kernel launchers shared between translation units of the MLA library.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {

cudaError_t launch_absorb_q_tc(const mla_dims &d, const void *q_nope, const void *q_rope, const void *w_uk,
                               void *q_cat, cudaStream_t st);
cudaError_t launch_out_proj_tc(const mla_dims &d, const void *o_lat, const void *w_uv, void *out, cudaStream_t st);
cudaError_t launch_attn_tc(const AttnParams &p, cudaStream_t st);
cudaError_t launch_attn_combine(const AttnParams &p, cudaStream_t st);
cudaError_t launch_naive(const AttnParams &p, int d_nope, int d_v, const void *q_nope, const void *q_rope,
                         const void *w_uk, const void *w_uv, void *out, float *lse, void *kv_scratch,
                         cudaStream_t st);

}  // namespace mla
