// kda_noalloc.cu -- kda_prefill_noalloc: the prefill for callers that cannot
// allocate device memory.
//
// kda_prefill needs a caller-provided device workspace.  Some callers cannot
// call cudaMalloc at the point where they run the prefill: code inside a
// framework that owns every allocation through its own pool, plugins handed
// only input and output buffers, or code running where an allocation would
// synchronise the device.  For them this entry point uses a fixed scratch area
// that lives in the library itself: a file-scope __device__ array of
// KDA_PREFILL_NOALLOC_SCRATCH_BYTES.  It allocates nothing and frees nothing;
// the CUDA runtime reserves the array on a device when this module is first
// used there and keeps it until the process exits.
//
// Host code cannot use the array's name as a device address (on the host it
// only names a stand-in object), so every call asks the runtime for the
// array's device address with cudaGetSymbolAddress, with the caller's device
// current, and passes that address to the kernels.  The lookup is host-side
// work with no stream operation; nothing is cached, so a context that was
// destroyed and re-created (cudaDeviceReset) or a different context on the
// same device gets its own address.  The first call in a context may make the
// runtime load the library's kernels there, so make it before any stream
// capture.
//
// Every call on a device shares the one array.  The prefill writes every byte
// of scratch it later reads (status word, sequence table, per-chunk records),
// so nothing has to start at zero and the previous call's leftovers are
// harmless; but calls whose GPU work overlaps (different streams, or
// different host threads, without ordering between them) race on the array.
#include "kda_common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_kda_noalloc_scratch[KDA_PREFILL_NOALLOC_SCRATCH_BYTES];

}  // namespace

extern "C" int kda_prefill_noalloc(const kda_desc* desc, const void* q, const void* k, const void* v,
                                   const void* log_alpha, const void* beta, const int32_t* cu_seqlens,
                                   const float* initial_state, void* out, float* final_state,
                                   kda_stream_t stream) {
    if (!desc) return KDA_ERR_INVALID_ARGUMENT;
    kda_desc d = *desc;
    d.workspace = nullptr;
    d.workspace_bytes = 0;
    const size_t need = kda_prefill_workspace_bytes(&d);
    if (need == 0)                                   // invalid or unsupported description:
        return kda_prefill(&d, q, k, v, log_alpha, beta, cu_seqlens, initial_state, out, final_state,
                           stream);                  // let the regular checks name the problem
    if (need > (size_t)KDA_PREFILL_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;

    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_kda_noalloc_scratch) != cudaSuccess || ptr == nullptr) return KDA_ERR_CUDA;
    d.workspace = ptr;
    d.workspace_bytes = (size_t)KDA_PREFILL_NOALLOC_SCRATCH_BYTES;
    return kda_prefill(&d, q, k, v, log_alpha, beta, cu_seqlens, initial_state, out, final_state, stream);
}
