// Verify step for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run the verify step: inference engines that plan every device byte up
// front and treat a later allocation as a failure, plugins hosted inside a
// framework that owns the allocator, or decode loops that must not take the
// device-wide synchronization an allocation can cause.  For them this file
// keeps the step's scratch (split partials and chunk classes) in a fixed,
// file-scope device array instead of a caller-provided tmp buffer.
//
// The array is 16 MiB and is held on every GPU that loads the library until
// the process exits.  Its device address belongs to the CUDA context, not to
// the device number (a cudaDeviceReset, or another context made current on the
// same device, reloads the module at a new address), so every call asks the
// runtime for it (cudaGetSymbolAddress allocates nothing).  The first call in
// a context also loads the module there; make that first call before any
// stream capture.  Every call shares the one array and leaves the last call's
// contents in it: nothing in it needs to start at zero (each call writes every
// partial and class it later reads), but calls whose work overlaps on the GPU
// (other streams, or graphs replayed concurrently) race on it.
#include "ta_internal.cuh"
#include "tree_attn.h"

#define TA_EXPORT extern "C" __attribute__((visibility("default")))

namespace ta {
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch in the current context.  Host code may
// not use the symbol itself: its host-side name is a stand-in, not a device
// address.
cudaError_t static_scratch_address(void **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

}  // namespace
}  // namespace ta

using namespace ta;

TA_EXPORT ta_status tree_attn_fwd_noalloc(const ta_tree_params *p, const ta_buf *q, const ta_buf *k,
                                          const ta_buf *v, const ta_buf *mask, const ta_buf *out,
                                          void *stream) {
    const size_t need = tree_attn_workspace_bytes(p);
    if (need == SIZE_MAX) {
        // report the parameter problem the regular entry point would report
        ta_buf none = {nullptr, 0, TA_F32, 0};
        ta_status st = tree_attn_fwd(p, q, k, v, mask, &none, out, stream);
        return st != TA_OK ? st : TA_ERR_INVALID_ARGUMENT;
    }
    if (need > kStaticScratchBytes) {
        set_last_error("tree_attn_fwd_noalloc: these parameters need %zu bytes of scratch but the "
                       "static scratch holds %zu; lower nwg or use tree_attn_fwd with a tmp buffer",
                       need, kStaticScratchBytes);
        return TA_ERR_UNSUPPORTED;
    }
    void *base = nullptr;
    cudaError_t e = static_scratch_address(&base);
    if (e != cudaSuccess) {
        set_last_error("tree_attn_fwd_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
        return TA_ERR_CUDA;
    }
    const ta_buf tmp = {base, kStaticScratchBytes, TA_F32, 0};
    ta_status st = tree_attn_fwd(p, q, k, v, mask, &tmp, out, stream);
    if (st != TA_OK) return st;
    return tree_attn_reduce(p, &tmp, out, stream);
}
