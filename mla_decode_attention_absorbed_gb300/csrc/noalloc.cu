// mla_decode_attn_noalloc: the latent-space decode attention for callers that
// cannot hand the library any scratch memory.
//
// Some callers hold only their input and output buffers: a plain C or FFI
// host with no device allocator of its own, or a serving loop whose device
// memory is owned by a framework pool, where calling cudaMalloc (which can
// synchronise the whole device) is not allowed while decoding.  For them the
// split partials and the status word live in one fixed array compiled into
// this library instead of a caller-provided workspace.
#include "common.cuh"

namespace {

// Scratch of the no-allocation entry point.  Every GPU on which this library's
// kernels are loaded holds these bytes until the process exits.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB

}  // namespace

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

namespace {

// Device address of g_decode_scratch on the current device.  In host code the
// symbol's name only stands for it; the address comes from cudaGetSymbolAddress
// with the device current.  It is looked up on every call (cheap once the
// library's module is loaded on the device), so a reset device or a recreated
// context, where the module and its array are loaded anew, gets the new address.
int static_scratch(void **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    *out = p;
    return MLA_OK;
}

}  // namespace

extern "C" {

MLA_API int mla_decode_attn_noalloc(const mla_dims *dims, const void *q_cat, const mla_cache *cache, void *o_lat,
                                    float *lse, int num_splits, int *device_status, void *stream) {
    if (!dims || !cache) return MLA_ERR_NULL;
    if (num_splits < MLA_SPLITS_BALANCED) return MLA_ERR_SHAPE;
    if (device_status && ((uintptr_t)device_status & 3u)) return MLA_ERR_ALIGN;
    // The library's plan keeps its split partials to about one wave of work items
    // (about 20 MB at most), so it fits the array; a plan or an explicit split
    // count that does not is refused.
    const size_t need = mla_decode_workspace_size(dims, cache, num_splits);
    if (need > kStaticScratchBytes) return MLA_ERR_WORKSPACE;
    void *scratch = nullptr;
    int s = static_scratch(&scratch);
    if (s != MLA_OK) return s;
    s = mla_decode_attn(dims, q_cat, cache, o_lat, lse, scratch, kStaticScratchBytes, num_splits, stream);
    if (s != MLA_OK) return s;
    if (device_status &&
        cudaMemcpyAsync(device_status, scratch, sizeof(int), cudaMemcpyDeviceToDevice,
                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MLA_ERR_CUDA;
    return MLA_OK;
}

}  // extern "C"
