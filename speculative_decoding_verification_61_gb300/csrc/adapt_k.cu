// adapt_k.cu -- device-side adaptive draft length (the next round's k per
// sequence from this round's accept counts), behind the C ABI of
// include/spec_verify.h.
//
// The rule follows sxl-space.tk "【大模型】- 推测解码", 自适应推测解码
// (AdaptiveSpeculativeDecoder.adapt_k), applied to every sequence of the
// batch on its own:
//   * a round's acceptance rate is n / k, the accepted drafted tokens over
//     the round's draft length;
//   * the rate joins the sequence's history (its last 100 rates; only the
//     last 10 are ever read);
//   * once the history holds 10 rates, their mean decides: above 0.8 the
//     length grows by one (up to max_k), below 0.5 it shrinks by one (down to
//     min_k), else it stays;
//   * the first length is (min_k + max_k) / 2, rounded down.
// The mean is compared exactly: every rate is a multiple of 1 / L with
// L = lcm(1..32), so sums of ten rates are integers (of L-ths) and the
// thresholds become integer comparisons; ties at exactly 0.8 or 0.5 change
// nothing.  A round that carries no rate (a data error, n < 0, or a
// sequence drafted with k = 0, or n > k) leaves that sequence's state as it
// was.
//
// The whole update is one small kernel (one block) that also writes the
// next round's k_offsets, so a serving loop never copies counts to the host.

#include <cstdint>

#include <cuda_runtime.h>

#include "spec_verify.h"

namespace specadapt {

constexpr int kWindow = 10;     // rates the decision reads
constexpr int kHistory = 100;   // rates the history keeps (caps the count)
constexpr int kThreads = 1024;  // one block: B <= SPEC_MAX_B = 4096
constexpr long long kL = 144403552893600LL;  // lcm(1, ..., 32)

// L / k for k = 0..32 (entry 0 unused): the rate n / k is n * (L / k) L-ths.
__constant__ long long kLOver[SPEC_MAX_K + 1] = {
    0,           kL / 1,  kL / 2,  kL / 3,  kL / 4,  kL / 5,  kL / 6,  kL / 7,  kL / 8,  kL / 9,  kL / 10,
    kL / 11,     kL / 12, kL / 13, kL / 14, kL / 15, kL / 16, kL / 17, kL / 18, kL / 19, kL / 20, kL / 21,
    kL / 22,     kL / 23, kL / 24, kL / 25, kL / 26, kL / 27, kL / 28, kL / 29, kL / 30, kL / 31, kL / 32};

// Per-sequence state, structure of arrays in the caller's device buffer.
struct State {
    int32_t *k;      // [B] the length of the next round
    int32_t *count;  // [B] rates in the history (<= kHistory)
    int32_t *head;   // [B] slot of the next rate in the window ring
    int32_t *hn;     // [B * kWindow] accepted counts of the last rates
    int32_t *hk;     // [B * kWindow] their draft lengths
};

__host__ __device__ inline State state_at(void *base, int B) {
    int32_t *p = static_cast<int32_t *>(base);
    State s;
    s.k = p;
    s.count = p + B;
    s.head = p + 2 * B;
    s.hn = p + 3 * B;
    s.hk = p + 3 * B + static_cast<size_t>(kWindow) * B;
    return s;
}

inline size_t state_bytes(int B) { return static_cast<size_t>(3 + 2 * kWindow) * B * sizeof(int32_t); }

// Exclusive prefix sum of k over the block, written as k_offsets[0..B].
__device__ void write_offsets(const int32_t *k, int B, int32_t *k_offsets) {
    __shared__ int s_warp[kThreads / 32 + 1];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int seg = (B + kThreads - 1) / kThreads;
    const int b0 = min(B, tid * seg), b1 = min(B, b0 + seg);
    int sum = 0;
    for (int b = b0; b < b1; ++b) sum += k[b];
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += n;
    }
    if (lane == 31) s_warp[w] = incl;
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int i = 0; i < kThreads / 32; ++i) {
            const int t = s_warp[i];
            s_warp[i] = acc;
            acc += t;
        }
        s_warp[kThreads / 32] = acc;
    }
    __syncthreads();
    int base = incl - sum + s_warp[w];
    for (int b = b0; b < b1; ++b) {
        k_offsets[b] = base;
        base += k[b];
    }
    if (tid == 0) k_offsets[B] = s_warp[kThreads / 32];
}

__global__ void __launch_bounds__(kThreads) init_kernel(State s, int B, int k0, int32_t *k_offsets) {
    for (int b = threadIdx.x; b < B; b += kThreads) {
        s.k[b] = k0;
        s.count[b] = 0;
        s.head[b] = 0;
        for (int j = 0; j < kWindow; ++j) {
            s.hn[static_cast<size_t>(j) * B + b] = 0;
            s.hk[static_cast<size_t>(j) * B + b] = 1;
        }
    }
    __syncthreads();
    write_offsets(s.k, B, k_offsets);
}

__global__ void __launch_bounds__(kThreads) update_kernel(State s, const int32_t *__restrict__ num_accepted, int B,
                                                          int min_k, int max_k, int32_t *k_offsets) {
    int32_t *__restrict__ sk = s.k;
    int32_t *__restrict__ scount = s.count;
    int32_t *__restrict__ shead = s.head;
    int32_t *__restrict__ hn = s.hn;
    int32_t *__restrict__ hk = s.hk;
    for (int b = threadIdx.x; b < B; b += kThreads) {
        const int k = sk[b];
        const int n = num_accepted[b];
        if (n < 0 || k <= 0 || n > k) continue;  // no rate this round
        const int head = shead[b];
        const int count = min(scount[b] + 1, kHistory);
        // the window after appending n / k at `head`: its sum in L-ths
        long long sum = static_cast<long long>(n) * kLOver[k];
#pragma unroll
        for (int j = 0; j < kWindow; ++j) {
            if (j == head) continue;
            sum += static_cast<long long>(hn[static_cast<size_t>(j) * B + b]) * kLOver[hk[static_cast<size_t>(j) * B + b]];
        }
        hn[static_cast<size_t>(head) * B + b] = n;
        hk[static_cast<size_t>(head) * B + b] = k;
        shead[b] = head + 1 == kWindow ? 0 : head + 1;
        scount[b] = count;
        if (count < kWindow) continue;
        // mean > 4/5  <=>  sum > 8 L;  mean < 1/2  <=>  sum < 5 L
        int knew = k;
        if (sum > 8 * kL) knew = min(k + 1, max_k);
        else if (sum < 5 * kL) knew = max(k - 1, min_k);
        sk[b] = knew;
    }
    __syncthreads();
    write_offsets(sk, B, k_offsets);
}

}  // namespace specadapt

using namespace specadapt;

namespace specv {
// spec_verify.cu: records a CUDA failure for spec_last_error()
bool cuda_ok(cudaError_t e, const char *what);
}  // namespace specv

namespace {
bool adapt_args_ok(const void *state, int B, int min_k, int max_k, const int32_t *k_offsets_out) {
    return state && k_offsets_out && B > 0 && B <= SPEC_MAX_B && min_k >= 1 && min_k <= max_k &&
           max_k <= SPEC_MAX_K;
}

int launch_status(cudaError_t e, const char *what) { return specv::cuda_ok(e, what) ? SPEC_OK : SPEC_ERR_CUDA; }
}  // namespace

extern "C" {

size_t spec_adapt_state_bytes(int B) {
    if (B <= 0 || B > SPEC_MAX_B) return 0;
    return state_bytes(B);
}

int spec_adapt_init(void *state, int B, int min_k, int max_k, int32_t *k_offsets_out, void *stream) {
    if (!adapt_args_ok(state, B, min_k, max_k, k_offsets_out)) return SPEC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(state) & 7u) != 0) return SPEC_ERR_ALIGNMENT;
    init_kernel<<<1, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(state_at(state, B), B, (min_k + max_k) / 2,
                                                                       k_offsets_out);
    return launch_status(cudaGetLastError(), "launch init_kernel");
}

int spec_adapt_update(void *state, const int32_t *num_accepted, int B, int min_k, int max_k,
                      int32_t *k_offsets_out, void *stream) {
    if (!adapt_args_ok(state, B, min_k, max_k, k_offsets_out) || !num_accepted) return SPEC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(state) & 7u) != 0) return SPEC_ERR_ALIGNMENT;
    update_kernel<<<1, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(state_at(state, B), num_accepted, B, min_k,
                                                                         max_k, k_offsets_out);
    return launch_status(cudaGetLastError(), "launch update_kernel");
}

}  // extern "C"
