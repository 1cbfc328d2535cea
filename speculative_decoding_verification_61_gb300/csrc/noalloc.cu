// noalloc.cu -- the allocation-free verify entry point, spec_verify_noalloc
// (include/spec_verify.h).  The web pages have no counterpart: this is a
// deployment convenience of the library.
//
// Some callers cannot allocate device memory at the moment they verify: a
// serving loop that forbids allocation on its hot path so that latency stays
// predictable, or a runtime whose own memory pool owns all device memory and
// gives out nothing else.  spec_verify_noalloc runs the kernels of
// spec_verify, but its scratch memory is a fixed array compiled into this
// library, so the call allocates nothing.
//
// The array is a file-scope device variable in a translation unit of its
// own, so it lives in a module of its own: with the CUDA runtime's lazy
// module loading (the default) a device holds it only once a process has
// called this entry point there, and then until the process exits; with
// eager loading every device that loads the library holds it.  In host code
// its name only stands in for the device object: the host looks its device
// address up with cudaGetSymbolAddress, once per device, with that device
// current, and passes that address to the kernels.

#include <cstdio>
#include <mutex>

#include "host_common.h"

namespace specv {

constexpr size_t kNoAllocScratchBytes = SPEC_NOALLOC_SCRATCH_BYTES;  // 48 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
void *g_noalloc_addr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

}  // namespace specv

using namespace specv;

extern "C" {

size_t spec_noalloc_bytes(int B, int V, int dtype) { return spec_workspace_bytes(B, V, dtype); }

int spec_verify_noalloc(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                        const float *u_accept, const float *u_resample, const float *temperature, int B,
                        const int32_t *k_offsets, int V, int dtype, int32_t *out_tokens,
                        int32_t *out_num_accepted, void *stream) {
    int rc = check_common(B, V, dtype);
    if (rc != SPEC_OK) return rc;
    if (B == 0) return SPEC_OK;
    if (!target_logits || !draft_logits || !draft_tokens || !u_accept || !u_resample || !temperature ||
        !k_offsets || !out_tokens || !out_num_accepted)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || !aligned16(draft_logits)) return SPEC_ERR_ALIGNMENT;
    const size_t need = spec_workspace_bytes(B, V, dtype);
    if (need > kNoAllocScratchBytes) {
        snprintf(g_last_error, sizeof g_last_error,
                 "spec_verify_noalloc: B=%d, V=%d needs %zu bytes of scratch, the fixed array holds %zu", B, V,
                 need, kNoAllocScratchBytes);
        return SPEC_ERR_WORKSPACE;
    }
    int dev = 0;
    if (!cuda_ok(cudaGetDevice(&dev), "cudaGetDevice") || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
    void *ws;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_addr[dev]) {
            // first call on this device (current): resolve the array's device address
            void *p = nullptr;
            if (!cuda_ok(cudaGetSymbolAddress(&p, g_noalloc_scratch), "cudaGetSymbolAddress(g_noalloc_scratch)"))
                return SPEC_ERR_CUDA;
            g_noalloc_addr[dev] = p;
        }
        ws = g_noalloc_addr[dev];
    }
    // the array keeps the previous call's contents: the status word and the
    // unit-ticket words that follow it must start at zero (one memset, no
    // allocation); the kernels zero the rest of what they count with
    if (!cuda_ok(cudaMemsetAsync(static_cast<unsigned char *>(ws) + kStatusOffset, 0,
                                 (kCounterWords - kStatus) * sizeof(int), static_cast<cudaStream_t>(stream)),
                 "cudaMemsetAsync(noalloc status and tickets)"))
        return SPEC_ERR_CUDA;
    return verify_call(target_logits, draft_logits, nullptr, draft_tokens, u_accept, u_resample, temperature, B,
                       k_offsets, V, dtype, out_tokens, out_num_accepted, nullptr, ws, kNoAllocScratchBytes, stream,
                       false);
}

}  // extern "C"
