// no_alloc.cu -- fdpp_decode_attn_noalloc: the decode step without a caller-supplied workspace.
//
// Some callers cannot allocate device memory at all: a plugin living inside a host runtime or
// inference engine that owns every device allocation and hands its plugins no allocator, or a
// serving loop whose memory budget is fixed at start-up so that nothing may call cudaMalloc (or
// any allocating library, torch included) afterwards. This entry point serves them: its scratch
// (split partials, plan, flags, fallback list) lives in one file-scope device array that every
// GPU loading this library holds until the process exits.
//
// The array is shared by every call on a device, and keeps the last call's contents. Each call
// clears the part that must start at zero (header counters and the fallback list) on the
// caller's stream, so calls issued on one stream follow one another safely; calls that overlap
// on the GPU (different streams, or other threads, without ordering between them) race on the
// array and give wrong results.
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "fdpp.h"
#include "fdpp_internal.h"

namespace {

// The library-owned scratch. In host code this name is only a host-side stand-in: its device
// address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FDPP_NOALLOC_WORKSPACE_BYTES];

std::mutex g_mutex;
void* g_scratch_ptr[64];

fdpp_status setup_failed(fdpp_status s, const char* what)
{
    fdpp::set_last_error(what);
    return s;
}

}  // namespace

extern "C" fdpp_status fdpp_decode_attn_noalloc(const void* q, const void* k_cache,
                                                const void* v_cache, const int32_t* block_table,
                                                const int32_t* seq_lens, const fdpp_params* p,
                                                void* out, fdpp_stream stream)
{
    size_t need = 0;
    fdpp_status st = fdpp_workspace_size(p, &need);
    if (st != FDPP_OK) return st;
    if (need > (size_t)FDPP_NOALLOC_WORKSPACE_BYTES) {
        char msg[256];
        std::snprintf(msg, sizeof msg,
                      "fdpp_decode_attn_noalloc: this problem needs %zu bytes of scratch, the "
                      "static workspace holds %zu; use fdpp_decode_attn with a workspace",
                      need, (size_t)FDPP_NOALLOC_WORKSPACE_BYTES);
        return setup_failed(FDPP_ERR_WORKSPACE, msg);
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return setup_failed(FDPP_ERR_CUDA, "fdpp_decode_attn_noalloc: cudaGetDevice failed");
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mutex);
        if (!g_scratch_ptr[dev]) {
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
                return setup_failed(FDPP_ERR_CUDA,
                                    "fdpp_decode_attn_noalloc: cudaGetSymbolAddress failed");
            g_scratch_ptr[dev] = ptr;
        }
        scratch = g_scratch_ptr[dev];
    }
    const size_t zero = fdpp::workspace_zero_prefix(*p);
    if (cudaMemsetAsync(scratch, 0, zero, (cudaStream_t)stream) != cudaSuccess)
        return setup_failed(FDPP_ERR_CUDA, "fdpp_decode_attn_noalloc: cudaMemsetAsync failed");
    return fdpp_decode_attn(q, k_cache, v_cache, block_table, seq_lens, p, scratch,
                            (size_t)FDPP_NOALLOC_WORKSPACE_BYTES, out, stream);
}
