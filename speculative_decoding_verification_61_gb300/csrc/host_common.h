// host_common.h -- host-side helpers shared by the verify translation units:
// per-device state, the workspace counter block, launches with programmatic
// dependent launch, and the helpers defined in spec_verify.cu.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

#include "verify_common.cuh"

namespace specv {

struct DeviceState {
    bool init = false;
    int sms = 0;
    int smem_per_sm = 0;
    int smem_optin = 0;
    int fuse_per_sm[2] = {0, 0};  // resident decide_stream_kernel CTAs per SM, by dtype
    void *ws = nullptr;
    size_t ws_bytes = 0;
    void *stage = nullptr;
    size_t stage_bytes = 0;
    cudaStream_t host_stream = nullptr;       // spec_round_host's second copy stream
    cudaEvent_t host_ev[2] = {nullptr, nullptr};
};

constexpr int kMaxDevices = 64;
extern DeviceState g_dev[kMaxDevices];

// The counters block opens every workspace, so that the status word has a
// fixed offset (kStatusOffset) whatever B and V are.
constexpr size_t kStatusOffset = sizeof(int) * kStatus;
constexpr size_t kTicketOffset = sizeof(int) * kTicket;  // the ticket words up to kCounterWords
constexpr size_t kCountersBytes = 256;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Last CUDA failure seen by the calling thread (call site + CUDA error name).
constexpr int kLastErrorBytes = 256;
extern thread_local char g_last_error[kLastErrorBytes];
bool cuda_ok(cudaError_t e, const char *what);

bool make_geometry(int V, int dtype, Geometry *g);
// Per-device state of the chain kernels (attributes set once per device).
DeviceState *device_state(int *dev_out);

// The streaming kernel copies its rows evict-first in L2 (chain and tree
// passes; the vocab-sharded pass measured no better with it).
#ifndef SPEC_STREAM_EVICT_FIRST
#define SPEC_STREAM_EVICT_FIRST 1
#endif
// Ring depth, dynamic shared memory and CTAs per SM of stats_kernel for a
// call with B sequences (ns = 0 if nothing fits).
void pick_ring(const DeviceState &st, int B, int *ns, size_t *smem, int *ctas_per_sm);
// The library-owned workspace of a device, grown to at least `need` bytes
// (zero-filled when allocated).  Calls that share it must be ordered on one
// stream.
void *get_internal_ws(DeviceState &st, size_t need);
// Zero the unit-ticket words of a caller workspace on the stream.
bool reset_tickets(void *ws, cudaStream_t stream);
bool aligned16(const void *p);
int check_common(int B, int V, int dtype);
// One verify call (spec_verify, spec_verify_ex, spec_verify_lse): the
// caller's workspace if given (checked; its ticket words zeroed on the
// stream unless reset_counters is false, when the caller has cleared them),
// else the library-owned one.
int verify_call(const void *target_logits, const void *draft_logits, const double *draft_lse2,
                const int32_t *draft_tokens, const float *u_accept, const float *u_resample, const float *temperature,
                int B, const int32_t *k_offsets, int V, int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
                const spec_verify_aux_t *aux, void *workspace, size_t workspace_bytes, void *stream,
                bool reset_counters);

// Launch with programmatic stream serialization: the kernel may begin
// while its predecessor on the stream drains; it orders itself with
// grid_dependency_wait() before touching the predecessor's outputs.
// The first kernel of a call reads the caller's inputs before it waits, so
// it is launched without the attribute (plain stream order): only kernels
// whose predecessor is one of ours start early.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace specv
