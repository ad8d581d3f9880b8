// no_alloc.cu -- fdpp_decode_attn_noalloc: the decode step without a caller-supplied workspace,
// and fdpp_read_diag_noalloc, which reads what such a call left behind.
//
// Some callers cannot allocate device memory at all: a plugin living inside a host runtime or
// inference engine that owns every device allocation and hands its plugins no allocator, or a
// serving loop whose memory budget is fixed at start-up so that nothing may call cudaMalloc (or
// any allocating library, torch included) afterwards. This entry point serves them: its scratch
// (split partials, plan, flags, fallback lists) lives in one file-scope device array that every
// GPU loading this library holds until the process exits.
//
// The array is shared by every call on a device, and keeps the last call's contents. Each call
// clears, on the caller's stream, the header, the plan and the fallback lists (the state that
// must start at zero, whatever shape the previous call had); the start-up hint of the tensor
// kernel behind them is kept, since a stale hint only costs a useless L2 prefetch. Calls issued
// on one stream follow one another safely; calls that overlap on the GPU (different streams, or
// other threads, without ordering between them) race on the array and give wrong results.
#include <cstdio>

#include <cuda_runtime.h>

#include "fdpp.h"
#include "fdpp_internal.h"

namespace {

// The library-owned scratch. In host code this name is only a host-side stand-in: its device
// address comes from cudaGetSymbolAddress, looked up on every call for the current device (a
// cached address would go stale if the caller reset the device's primary context).
static __device__ __align__(256) unsigned char g_noalloc_scratch[FDPP_NOALLOC_WORKSPACE_BYTES];

fdpp_status setup_failed(fdpp_status s, const char* what)
{
    fdpp::set_last_error(what);
    return s;
}

// The scratch's device address on the current device, after checking that a problem of `p`
// fits in it.
fdpp_status scratch_for(const fdpp_params* p, const char* who, void** scratch)
{
    size_t need = 0;
    fdpp_status st = fdpp_workspace_size(p, &need);
    if (st != FDPP_OK) return st;
    if (need > (size_t)FDPP_NOALLOC_WORKSPACE_BYTES) {
        char msg[256];
        std::snprintf(msg, sizeof msg,
                      "%s: this problem needs %zu bytes of scratch, the static workspace holds "
                      "%zu; use fdpp_decode_attn with a workspace",
                      who, need, (size_t)FDPP_NOALLOC_WORKSPACE_BYTES);
        return setup_failed(FDPP_ERR_WORKSPACE, msg);
    }
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
        char msg[256];
        std::snprintf(msg, sizeof msg, "%s: cudaGetSymbolAddress: %s", who, cudaGetErrorString(e));
        return setup_failed(FDPP_ERR_CUDA, msg);
    }
    *scratch = ptr;
    return FDPP_OK;
}

}  // namespace

extern "C" fdpp_status fdpp_decode_attn_noalloc(const void* q, const void* k_cache,
                                                const void* v_cache, const int32_t* block_table,
                                                const int32_t* seq_lens, const fdpp_params* p,
                                                void* out, fdpp_stream stream)
{
    void* scratch = nullptr;
    const fdpp_status st = scratch_for(p, "fdpp_decode_attn_noalloc", &scratch);
    if (st != FDPP_OK) return st;
    // header (error bits of this call only), plan and fallback lists; not the start-up hint
    const size_t zero = fdpp::workspace_hint_offset(*p);
    if (cudaMemsetAsync(scratch, 0, zero, (cudaStream_t)stream) != cudaSuccess)
        return setup_failed(FDPP_ERR_CUDA, "fdpp_decode_attn_noalloc: cudaMemsetAsync failed");
    return fdpp_decode_attn(q, k_cache, v_cache, block_table, seq_lens, p, scratch,
                            (size_t)FDPP_NOALLOC_WORKSPACE_BYTES, out, stream);
}

extern "C" fdpp_status fdpp_read_diag_noalloc(const fdpp_params* p, fdpp_diag* diag,
                                              uint8_t* flags_host, int32_t* nsplit_host)
{
    void* scratch = nullptr;
    const fdpp_status st = scratch_for(p, "fdpp_read_diag_noalloc", &scratch);
    if (st != FDPP_OK) return st;
    return fdpp_read_diag(scratch, (size_t)FDPP_NOALLOC_WORKSPACE_BYTES, p, diag, flags_host,
                          nsplit_host);
}
