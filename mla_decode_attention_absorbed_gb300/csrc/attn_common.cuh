// Device helpers of the attention kernels (attn_tc.cu):
// bounded waits that also give up once the CTA aborts, the abort broadcast to
// the peer CTA of a pair, fp16 packing of partial scores, register hand-over
// between warpgroups.  No method arithmetic here.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"
#include "sm100.cuh"

namespace mla {
namespace attn {

using namespace sm100;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bounded wait that also gives up once the CTA is aborting (S: the kernel's
// shared-memory block, with an `abort` flag and the launch's wait bound
// `wait_ns`; the cycle bound is twice it, about the SM clock in GHz, so the
// bound holds even if one of the two clocks does not advance).
template <bool kCluster = false, class S>
__device__ __forceinline__ bool wait_bar(S &sm, uint64_t *bar, uint32_t parity) {
    if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const long long c0 = clock64();
    const uint64_t lim_ns = sm.wait_ns;
    const long long lim_cyc = (long long)(lim_ns > (1ull << 61) ? (1ull << 62) : 2 * lim_ns);
    for (uint32_t it = 1;; ++it) {
        if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
        // the clocks are read after the first retry (a try_wait suspends in hardware,
        // so a short bound is seen at once) and then every 64
        if (it == 1 || (it & 63u) == 0) {
            if (*(volatile int *)&sm.abort) return false;
            if (globaltimer_ns() - t0 > lim_ns || clock64() - c0 > lim_cyc) return false;
        }
    }
}

// Every lane waits; the warp proceeds only if all lanes saw the phase complete,
// so warp-collective tcgen05 instructions that follow stay converged.
template <bool kCluster = false, class S>
__device__ __forceinline__ bool warp_wait(S &sm, uint64_t *bar, uint32_t parity) {
    const bool ok = wait_bar<kCluster>(sm, bar, parity);
    return __all_sync(0xffffffffu, ok);
}

// Marks this CTA (and, in a pair, the peer) as aborting and records the timeout.
template <bool kSplit, class S>
__device__ __forceinline__ void raise_abort(S &sm, const AttnParams &p, uint32_t peer) {
    *(volatile int *)&sm.abort = 1;
    set_status(p.status, MLA_ERR_TIMEOUT);
    if (kSplit) {
        uint32_t remote = map_to_rank(smem_u32(&sm.abort), peer);
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(1) : "memory");
    }
}

// Two scores to fp16 (lo in the low half), saturating at +-65504 instead of
// overflowing to infinity.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t u) {
    __half2 h = *reinterpret_cast<__half2 *>(&u);
    return __half22float2(h);
}

// lo += the low fp16 half of h, hi += the high half, each in one fp32 add (the
// fp16 value widens exactly).
__device__ __forceinline__ void add_f16x2_to(uint32_t h, float &lo, float &hi) {
    asm("{\n\t.reg .b16 l16, h16;\n\tmov.b32 {l16, h16}, %2;\n\t"
        "add.rn.f32.f16 %0, l16, %0;\n\tadd.rn.f32.f16 %1, h16, %1;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "r"(h));
}

// Register hand-over between warpgroups (all four warps of a warpgroup run it).
template <int kRegs>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs)); }
template <int kRegs>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs)); }

}  // namespace attn
}  // namespace mla
