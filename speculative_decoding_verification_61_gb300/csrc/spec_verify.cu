// spec_verify.cu -- GB300 (sm_103a) verify-and-resample step of speculative
// decoding, behind the C ABI of include/spec_verify.h.
//
// The method (web pages, cited by title and section):
//   docs.ifdog.com "投机解码": 投机解码的三步流程 step 3 (accept with
//     min(1, p/q), resample from norm(max(0, p - q)), bonus after k
//     acceptances); 动手实践 (temperature-scaled softmax, greedy branch);
//   bbs.huaweicloud.com "大模型推理无损加速:投机采样...": 二.1 (alpha), 二.2
//     (residual distribution), 三 (speculative_sampling_step);
//   sxl-space.tk "【大模型】- 推测解码": 批量推测解码 (one verify per sequence
//     of a batch, different accepted lengths).
//
// Pipeline of one spec_verify call (all on the caller's stream, no host sync):
//   1. stats_kernel    persistent; streams every needed logit row through a
//                      shared-memory ring filled by 1-D bulk copies (TMA
//                      engine) and reduces each 2 KB sub-chunk to an online
//                      softmax partial (max m, sum 2^(x c - m)) or, for
//                      greedy rows, an arg-max partial.  Each row is read
//                      from HBM once.
//   2. resolve_kernel  kSub blocks per sequence: each combines the partials
//                      of the sequence's rows, forms alpha_i and finds the
//                      first rejection with a warp ballot; on a rejection the
//                      blocks share the residual mass max(0, p - q) of the two
//                      rows at that position, and the last warp to finish
//                      locates the sub-chunk where the cumulative mass crosses
//                      u * Z, re-reads only that piece and finds the token
//                      with a warp scan.  The bonus draw uses the partials of
//                      row k the same way.
// spec_draft_sample runs stats_kernel over the draft rows, then
// draft_select_kernel (arg-max, or the same locate + scan per row).

#include <algorithm>
#include <climits>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <utility>

#include "device_utils.cuh"

namespace specv {

constexpr int kSlotBytes = 16384;        // one chunk of one row per ring slot
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxSlots = 6;
constexpr int kSub = kConsumerWarps;                // sub-chunks per chunk (one per consumer warp)
constexpr int kSubVecs = kSlotBytes / 16 / kSub;    // 16-byte vectors per sub-chunk (2 KB)

enum UnitKind : int { kEnd = 0, kSoft = 1, kArg = 2 };
enum DrawKind : int { kJobNone = 0, kJobResid = 1, kJobBonus = 2 };

struct Geometry {
    int V;
    int chunk_elems;  // elements per chunk (a multiple of the 16-byte vector)
    int n_chunks;     // chunks per row
    int sub_elems;    // elements per sub-chunk (2 KB)
    int n_sub;        // sub-chunk slots per row (n_chunks * kSub; trailing ones may be empty)
};

struct UnitDesc {
    uint32_t nbytes;
    int kind;
    float c;
    int elem0;
    int64_t out_idx;
};

// Words of the workspace's counter block.
// Status word, then stats_kernel's unit tickets and count of CTAs done.
enum CounterWord : int { kStatus = 1, kTicket = 2, kDone = 3, kCounterWords = 4 };

struct WsPtrs {
    float2 *part;        // [rows_cap * n_sub] sub-chunk partials
    int *counters;       // CounterWord: status, unit tickets and CTAs done
    int *seqcnt;         // [B] resolve_kernel arrivals per sequence
    float *resid_part;   // [B * n_sub] residual mass per sub-chunk
};

// ------------------------------------------------------------------ helpers
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before its predecessor on the stream has
// finished; grid_dependency_wait() blocks until that predecessor has
// completed and its memory is visible.  grid_launch_dependents() lets the
// next kernel on the stream begin launching.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }
__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

// Exclusive block scan of one int per thread (any multiple of 32 threads).
__device__ int block_excl_scan(int v, int *s_warp, int *total) {
    const int lane = lane_id(), w = warp_id(), nw = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += n;
    }
    if (lane == 31) s_warp[w] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int i = 0; i < nw; ++i) {
            int t = s_warp[i];
            s_warp[i] = acc;
            acc += t;
        }
        s_warp[nw] = acc;
    }
    __syncthreads();
    const int r = incl - v + s_warp[w];
    *total = s_warp[nw];
    __syncthreads();
    return r;
}

// ------------------------------------------------------------ unit tickets
// stats_kernel hands out its units dynamically: an SM that streams faster
// takes more of them, so all CTAs finish together.  Ticket t (one atomic
// add on a counter) is a batch of kStatsBatch consecutive units while at
// least kStatsTailPerCta units per CTA remain after it, then a batch of
// kStatsTailBatch, which keeps the finishing times within a fraction of a
// microsecond without an atomic per unit.
#ifndef SPEC_STATS_BATCH
#define SPEC_STATS_BATCH 4
#endif
#ifndef SPEC_STATS_TAIL_BATCH
#define SPEC_STATS_TAIL_BATCH 1
#endif
#ifndef SPEC_STATS_TAIL_PER_CTA
#define SPEC_STATS_TAIL_PER_CTA 8
#endif
constexpr int kStatsBatch = SPEC_STATS_BATCH;
constexpr int kStatsTailBatch = SPEC_STATS_TAIL_BATCH;
constexpr int kStatsTailPerCta = SPEC_STATS_TAIL_PER_CTA;

__device__ __forceinline__ int64_t big_batches(int64_t total_units, int grid) {
    return max(static_cast<int64_t>(0), (total_units - static_cast<int64_t>(grid) * kStatsTailPerCta) / kStatsBatch);
}

__device__ __forceinline__ void unit_batch(int t, int64_t n_big, int64_t *u0, int *cnt) {
    if (t < n_big) {
        *u0 = static_cast<int64_t>(t) * kStatsBatch;
        *cnt = kStatsBatch;
    } else {
        *u0 = n_big * kStatsBatch + (t - n_big) * static_cast<int64_t>(kStatsTailBatch);
        *cnt = kStatsTailBatch;
    }
}

// ================================================================== kernel 1
// Streaming modes of stats_kernel (which rows it reads).
enum StatsMode : int {
    kModeVerify = 0,  // target rows, plus the draft rows of sampled sequences
    kModeDraft = 1,   // draft rows only (spec_draft_sample)
    kModeTarget = 2   // target rows only (verify with the draft rows' lse given)
};

// Persistent streaming kernel.  Unit u = (row r of the virtual row list,
// chunk ch).  Virtual row list, by sequence b in order:
//   verify mode: target rows of b (k_b + 1), then draft rows of b (k_b) if
//                b is sampled; nothing for a bad temperature;
//   draft mode:  draft rows of b (k_b); nothing for a bad temperature;
//   target mode: target rows of b (k_b + 1); nothing for a bad temperature.
// Units are taken by tickets (unit_batch).  One lane of warp 8 is the
// producer: it waits for a free ring slot and issues the bulk copy of the
// next unit into it.  Warps 0..7 consume: warp w owns the w-th 2 KB
// sub-chunk of the slot (128 16-byte vectors, lane l reading vectors
// l + 32 j), reduces it to a partial (online softmax or arg-max) and writes
// that partial straight to global memory.
// (the bound caps registers at 40, which leaves room on an SM with four
// of these CTAs for one resolve_kernel block of the other stream)
template <int DT, int MODE>
__global__ void __launch_bounds__(kThreads, 5) stats_kernel(
    const void *__restrict__ target, const void *__restrict__ draft,
    const float *__restrict__ temperature, const int *__restrict__ k_offsets, int B, Geometry g, int ns,
    float2 *__restrict__ part, int *__restrict__ counters, int *__restrict__ seqcnt) {
    using E = Elem<DT>;
    constexpr bool DRAFT = MODE == kModeDraft;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)ns * kSlotBytes);
    uint64_t *empty = full + ns;
    UnitDesc *desc = reinterpret_cast<UnitDesc *>(empty + ns);
    int *s_kofs = reinterpret_cast<int *>(desc + ns);
    int *s_rowpre = s_kofs + (B + 1);
    float *s_c = reinterpret_cast<float *>(s_rowpre + (B + 1));
    int *s_tmp = reinterpret_cast<int *>(s_c + B);  // [kThreads/32 + 1]

    const int tid = threadIdx.x;
    for (int i = tid; i <= B; i += kThreads) {
        s_kofs[i] = k_offsets[i];
        if (i < B) s_c[i] = temp_scale(temperature[i]);
    }
    __syncthreads();

    // k_offsets validation and row counts (contiguous segment per thread)
    const int seg = (B + kThreads - 1) / kThreads;
    const int b0 = min(B, tid * seg), b1 = min(B, b0 + seg);
    int bad = (tid == 0 && s_kofs[0] != 0) ? 1 : 0;
    int rows = 0;
    // rows of sequence b: none for a bad temperature
    auto seq_rows = [&](int b) -> int {
        const int k = s_kofs[b + 1] - s_kofs[b];
        const float c = s_c[b];
        if (c != c) return 0;
        if (MODE == kModeDraft) return k;
        if (MODE == kModeTarget) return k + 1;
        return c == 0.0f ? k + 1 : 2 * k + 1;
    };
    for (int b = b0; b < b1; ++b) {
        const int k = s_kofs[b + 1] - s_kofs[b];
        if (k < 0 || k > kMaxK) bad = 1;
        rows += seq_rows(b);
    }
    int total_rows;
    int base = block_excl_scan(rows, s_tmp, &total_rows);
    for (int b = b0; b < b1; ++b) {
        s_rowpre[b] = base;
        base += seq_rows(b);
    }
    if (tid == 0) s_rowpre[B] = total_rows;
    // everything above only read the inputs; from here on the workspace is
    // written, so the previous kernel on the stream must have finished
    grid_dependency_wait();
    const bool any_bad = __syncthreads_or(bad);
    if (!DRAFT)
        for (int i = blockIdx.x * kThreads + tid; i < B; i += gridDim.x * kThreads) seqcnt[i] = 0;
    // the next kernel may be scheduled as soon as SMs free up; it waits for
    // this grid's completion before it reads anything written here
    grid_launch_dependents();
    if (any_bad) return;

    if (tid == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    const int64_t R_t = static_cast<int64_t>(s_kofs[B]) + B;
    const int lane = lane_id();

    if (warp_id() == kConsumerWarps) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            // units u = r * n_chunks + ch are handed out by tickets (see
            // unit_batch); each CTA's units increase, so b only moves forward
            const int64_t total_units = static_cast<int64_t>(total_rows) * g.n_chunks;
            const int64_t n_big = big_batches(total_units, gridDim.x);
            int b = 0;
            int islot = 0;
            uint32_t iphase = 0;  // slot and use parity of the next issue
            int t = atomicAdd(counters + kTicket, 1);
            while (ok) {
                int64_t u0;
                int cnt;
                unit_batch(t, n_big, &u0, &cnt);
                if (u0 >= total_units) break;
                const int tn = atomicAdd(counters + kTicket, 1);  // next batch, in flight meanwhile
                cnt = static_cast<int>(min(static_cast<int64_t>(cnt), total_units - u0));
                int r = static_cast<int>(u0 / g.n_chunks);
                int ch = static_cast<int>(u0 - static_cast<int64_t>(r) * g.n_chunks);
                for (int q = 0; q < cnt; ++q) {
                    if (issued >= ns && !mbar_wait_bounded(&empty[islot], iphase ^ 1u)) {
                        ok = false;
                        break;
                    }
                    while (s_rowpre[b + 1] <= r) ++b;
                    const int l = r - s_rowpre[b];
                    const int k = s_kofs[b + 1] - s_kofs[b];
                    const float c = s_c[b];
                    const void *base_ptr;
                    int64_t row, slot_row;
                    if (DRAFT) {
                        row = s_kofs[b] + l;
                        base_ptr = draft;
                        slot_row = row;
                    } else if (l <= k) {
                        row = static_cast<int64_t>(s_kofs[b]) + b + l;
                        base_ptr = target;
                        slot_row = row;
                    } else {
                        row = static_cast<int64_t>(s_kofs[b]) + (l - k - 1);
                        base_ptr = draft;
                        slot_row = R_t + row;
                    }
                    const int e0 = ch * g.chunk_elems;
                    const int e1 = min(g.V, e0 + g.chunk_elems);
                    UnitDesc d;
                    d.nbytes = static_cast<uint32_t>(e1 - e0) * E::kBytes;
                    d.kind = (c == 0.0f) ? kArg : kSoft;
                    d.c = c;
                    d.elem0 = e0;
                    d.out_idx = (slot_row * g.n_chunks + ch) * kSub;
                    desc[islot] = d;
                    const unsigned char *src = static_cast<const unsigned char *>(base_ptr) +
                                               (row * g.V + e0) * static_cast<int64_t>(E::kBytes);
                    mbar_arrive_expect_tx(&full[islot], d.nbytes);
                    bulk_g2s(ring + static_cast<size_t>(islot) * kSlotBytes, src, d.nbytes, &full[islot]);
                    ++issued;
                    if (++islot == ns) {
                        islot = 0;
                        iphase ^= 1u;
                    }
                    if (++ch == g.n_chunks) {
                        ch = 0;
                        ++r;
                    }
                }
                t = tn;
            }
            if (ok && issued >= ns) ok = mbar_wait_bounded(&empty[islot], iphase ^ 1u);
            {
                // end marker (also on time-out, so that consumers leave)
                desc[islot].kind = kEnd;
                mbar_arrive(&full[islot]);
            }
            if (!ok) {
                set_status(counters + kStatus, SPEC_ERR_TIMEOUT);
                // let issued copies land before the CTA exits (bounded)
                for (int i = max(0, issued - ns); i < issued; ++i) mbar_wait_bounded(&full[i % ns], (i / ns) & 1);
            }
        }
        __syncwarp();
    } else {
    // ---------------------------------------------------------- consumers
    const int w = warp_id();
    int slot = 0;
    uint32_t phase = 0;
    for (;;) {
        if (!mbar_wait_bounded(&full[slot], phase)) {
            set_status(counters + kStatus, SPEC_ERR_TIMEOUT);
            break;
        }
        const UnitDesc d = desc[slot];
        if (d.kind == kEnd) break;
        const uint4 *v4 =
            reinterpret_cast<const uint4 *>(ring + static_cast<size_t>(slot) * kSlotBytes) + w * kSubVecs;
        const int nvec = min(kSubVecs, static_cast<int>(d.nbytes >> 4) - w * kSubVecs);  // may be <= 0
        uint4 v[4];
        bool okv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int idx = lane + 32 * j;
            okv[j] = idx < nvec;
            // vectors past the end read as -inf: no mass, never the max
            v[j] = okv[j] ? v4[idx] : make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);  // the slot's data is in registers
        if (++slot == ns) {
            slot = 0;
            phase ^= 1u;
        }
        float2 res;
        if (d.kind == kSoft) {
            // warp-wide max first (NaN-propagating), then one pass of
            // 2^(x c - m_w) against it in packed fp32 pairs
            float vmax = E::vmax4_nan(v);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) vmax = fmax_nan(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
            float m, sum;
            if (vmax != vmax) {
                m = -INFINITY;
                sum = __int_as_float(0x7fc00000);
            } else if (vmax == -INFINITY) {
                m = -INFINITY;
                sum = 0.0f;
            } else {
                m = vmax * d.c;
                const float2 cc = make_float2(d.c, d.c), mm = make_float2(-m, -m);
                float2 acc0 = make_float2(0.0f, 0.0f), acc1 = acc0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
#pragma unroll
                    for (int p = 0; p < E::kPairs; ++p) {
                        const float2 t = ffma2(E::pair(v[j], p), cc, mm);
                        const float2 e = make_float2(ex2(t.x), ex2(t.y));
                        if (p & 1) acc1 = fadd2(acc1, e); else acc0 = fadd2(acc0, e);
                    }
                }
                sum = (acc0.x + acc0.y) + (acc1.x + acc1.y);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            }
            res = make_float2(m, sum);
        } else {
            ArgPart a{-INFINITY, INT_MAX};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (!okv[j]) continue;
                const float vm = E::vmax_nan(v[j]);
                if (vm != vm) {
                    a.i = -1;
                } else if (a.i != -1 && (vm > a.v || a.i == INT_MAX)) {
                    float x[E::kPerVec];
                    E::unpack(v[j], x);
                    int e = 0;
#pragma unroll
                    for (int q = E::kPerVec - 1; q >= 0; --q)
                        if (x[q] == vm) e = q;
                    a = ArgPart{vm, d.elem0 + (w * kSubVecs + lane + 32 * j) * E::kPerVec + e};
                }
            }
            a = warp_arg(a);
            res = make_float2(a.v, __int_as_float(a.i));
        }
        if (lane == 0) part[d.out_idx + w] = res;
    }
    }
    // the last CTA out resets the ticket counters for the next launch on the
    // stream (the library zeroes them once when it allocates a workspace)
    __syncthreads();
    if (tid == 0 && atomic_add_acq_rel_gpu(counters + kDone, 1) == static_cast<int>(gridDim.x) - 1) {
        counters[kTicket] = 0;
        counters[kDone] = 0;
    }
}

// ================================================================== warp tools
// GB300's fp64 pipe is a small fraction of its fp32 rate, so every loop
// below (over partials, weights or elements) runs in fp32; fp64 appears only
// in a few per-call scalars (cumulative masses, thresholds, log-sum-exps).

// Two-sum accumulation: (hi, lo) carries the rounding error of each add.
struct Acc2 {
    float hi = 0.0f, lo = 0.0f;
    __device__ __forceinline__ void add(float b) {
        const float s = hi + b;
        const float bb = s - hi;
        lo += (hi - (s - bb)) + (b - bb);
        hi = s;
    }
    __device__ __forceinline__ float value() const { return hi + lo; }
};

// Unevaluated sum hi + lo of two fp32 values, |lo| <= ulp(hi) / 2 once
// normalised: about 44 bits of precision from fp32 operations.  The running
// masses of the inverse CDF use it instead of fp64, whose pipe is a small
// fraction of GB300's fp32 rate.  (Error-free sums after Knuth and Dekker.)
struct F2 {
    float hi, lo;
};

__device__ __forceinline__ F2 f2_two_sum(float a, float b) {  // a + b = hi + lo exactly
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    return F2{s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}

__device__ __forceinline__ F2 f2_norm(float s, float e) {  // |s| >= |e| (or s == 0)
    const float t = __fadd_rn(s, e);
    return F2{t, __fsub_rn(e, __fsub_rn(t, s))};
}

__device__ __forceinline__ F2 f2_add(F2 a, float b) {
    const F2 t = f2_two_sum(a.hi, b);
    return f2_norm(t.hi, __fadd_rn(t.lo, a.lo));
}

__device__ __forceinline__ F2 f2_sub(F2 a, F2 b) {
    const F2 t = f2_two_sum(a.hi, -b.hi);
    return f2_norm(t.hi, __fadd_rn(t.lo, __fsub_rn(a.lo, b.lo)));
}

__device__ __forceinline__ F2 f2_scale(float u, F2 a) {  // u * (hi + lo)
    const float p = __fmul_rn(u, a.hi);
    return f2_norm(p, __fmaf_rn(u, a.lo, __fmaf_rn(u, a.hi, -p)));
}

__device__ __forceinline__ bool f2_gt(F2 a, F2 b) {
    const F2 d = f2_sub(a, b);
    return d.hi > 0.0f || (d.hi == 0.0f && d.lo > 0.0f);
}

__device__ __forceinline__ F2 shfl_f2(F2 v, int src) {
    return F2{__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}

// Largest fp32 value <= hi + lo (normalised pair).
__device__ __forceinline__ float f2_round_down(F2 x) {
    return x.lo < 0.0f ? nextafterf(x.hi, -INFINITY) : x.hi;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ float warp_incl_scan_f(float v) {
    const int lane = lane_id();
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += n;
    }
    return v;
}

// log2-domain log-sum-exp M + log2(S) for S >= 1: the exponent of S is
// split off so that log2f works on the mantissa (absolute error ~1e-7).
__device__ __forceinline__ double lse2(float M, float S) {
    int e;
    const float m = frexpf(S, &e);
    return static_cast<double>(M) + static_cast<double>(e) + static_cast<double>(log2f(m));
}

// Sub-chunk partials a lane holds in registers: p[lane + 32 j], j < 8, so
// rows of up to 256 sub-chunks take one memory round trip; the rest of a
// longer row is read again where needed.
constexpr int kPartCache = 8;

__device__ __forceinline__ void load_parts(const float2 *p, int n, float2 (&c)[kPartCache]) {
    const int lane = lane_id();
#pragma unroll
    for (int j = 0; j < kPartCache; ++j) {
        const int i = lane + 32 * j;
        c[j] = (i < n) ? __ldcg(p + i) : make_float2(-INFINITY, 0.0f);
    }
}

// Row combine of the n sub-chunk partials of one row by a whole warp:
// M = max of the partial maxima, S = sum s_i 2^(m_i - M) (>= 1); lane l
// adds its partials in index order whether cached or not.
__device__ bool combine_soft(const float2 (&cache)[kPartCache], const float2 *p, int n, float *M_out,
                             float *S_out) {
    const int lane = lane_id();
    float M = -INFINITY;
    bool nan = false;
#pragma unroll
    for (int j = 0; j < kPartCache; ++j) {
        nan |= (cache[j].y != cache[j].y);
        M = fmaxf(M, cache[j].x);
    }
    for (int i = lane + 32 * kPartCache; i < n; i += 32) {
        const float2 v = __ldcg(p + i);
        nan |= (v.y != v.y);
        M = fmaxf(M, v.x);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    nan = __any_sync(0xffffffffu, nan);
    if (nan || !(M > -INFINITY) || !(M < INFINITY)) return false;
    Acc2 acc;
#pragma unroll
    for (int j = 0; j < kPartCache; ++j)
        if (cache[j].x > -INFINITY) acc.add(cache[j].y * ex2(cache[j].x - M));
    for (int i = lane + 32 * kPartCache; i < n; i += 32) {
        const float2 v = __ldcg(p + i);
        if (v.x > -INFINITY) acc.add(v.y * ex2(v.x - M));
    }
    const float S = warp_sum_f(acc.value());
    if (!(S > 0.0f) || !(S < INFINITY)) return false;
    *M_out = M;
    *S_out = S;
    return true;
}

__device__ bool warp_combine_soft(const float2 *p, int n, float *M_out, float *S_out) {
    float2 cache[kPartCache];
    load_parts(p, n, cache);
    return combine_soft(cache, p, n, M_out, S_out);
}

// Arg-max over the n sub-chunk partials of one row; -1 if a NaN was seen.
__device__ int warp_combine_arg(const float2 *p, int n) {
    ArgPart a{-INFINITY, INT_MAX};
    for (int i = lane_id(); i < n; i += 32) {
        const float2 v = __ldcg(p + i);
        a = arg_merge(a, ArgPart{v.x, __float_as_int(v.y)});
    }
    a = warp_arg(a);
    return a.i == INT_MAX ? -1 : a.i;
}

// Warp-level locate over n non-negative weights (sub-chunk masses): total
// Z, target = u * Z, and the first i whose cumulative mass exceeds the
// target, with the mass before it.  If rounding leaves no such i, the last
// i with positive weight.  Returns -1 if every weight is 0.  Weight i is
// cache[j] of lane i % 32 for i = lane + 32 j < 32 * kPartCache, wfar(i)
// beyond.
template <class WF>
__device__ int warp_locate(int n, const float (&cache)[kPartCache], WF wfar, float u, F2 *before, F2 *total,
                           F2 *target_out) {
    const int lane = lane_id();
    constexpr int kCache = kPartCache;
    Acc2 acc;
#pragma unroll
    for (int j = 0; j < kCache; ++j) acc.add(cache[j]);
    for (int j = kCache; 32 * j < n; ++j) acc.add((lane + 32 * j < n) ? wfar(lane + 32 * j) : 0.0f);
    const F2 tot = f2_two_sum(warp_sum_f(acc.hi), warp_sum_f(acc.lo));
    const F2 target = f2_scale(u, tot);
    *total = tot;
    *target_out = target;
    F2 carry{0.0f, 0.0f}, last_before{0.0f, 0.0f};
    int last = -1;
    for (int j = 0; 32 * j < n; ++j) {
        float w = 0.0f;
#pragma unroll
        for (int q = 0; q < kCache; ++q)
            if (q == j) w = cache[q];
        if (j >= kCache) w = (lane + 32 * j < n) ? wfar(lane + 32 * j) : 0.0f;
        const float incl = warp_incl_scan_f(w);
        const F2 cum = f2_add(carry, incl);
        const unsigned hit = __ballot_sync(0xffffffffu, w > 0.0f && f2_gt(cum, target));
        if (hit) {
            const int src = __ffs(hit) - 1;
            *before = shfl_f2(f2_add(carry, incl - w), src);
            return 32 * j + src;
        }
        const unsigned pos = __ballot_sync(0xffffffffu, w > 0.0f);
        if (pos) {
            const int src = 31 - __clz(pos);
            last = 32 * j + src;
            last_before = shfl_f2(f2_add(carry, incl - w), src);
        }
        carry = shfl_f2(cum, 31);
    }
    *before = last_before;
    return last;
}

#ifndef SPEC_RESID_PREFETCH
#define SPEC_RESID_PREFETCH 1
#endif
#ifndef SPEC_RESID_L2HINT
#define SPEC_RESID_L2HINT 0
#endif
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
#if SPEC_RESID_L2HINT
    uint4 v;
    asm volatile("ld.global.nc.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
#else
    return __ldg(p);
#endif
}

// Element range of sub-chunk sc of a row.
__device__ __forceinline__ void sub_range(const Geometry &g, int sc, int *a, int *b) {
    const int ch = sc / kSub, w = sc - ch * kSub;
    const int c0 = ch * g.chunk_elems;
    const int c1 = min(g.V, c0 + g.chunk_elems);
    *a = min(c1, c0 + w * g.sub_elems);
    *b = min(c1, *a + g.sub_elems);
}

// Vector j (0..3, not a compile-time constant) of four held in registers:
// a chain of selects, so that the loops over j below stay rolled.
__device__ __forceinline__ uint4 pick4(const uint4 (&r)[4], int j) {
    uint4 v = r[3];
    v = (j == 2) ? r[2] : v;
    v = (j == 1) ? r[1] : v;
    return (j == 0) ? r[0] : v;
}

// Warp-level inverse CDF inside elements [a, b) (at most one sub-chunk) of
// one or two rows: lane l owns vectors 4l .. 4l+3 (contiguous), weights are
// W(x_row1, x_row2).  Returns the first element whose cumulative mass,
// starting at `before`, exceeds `target`; else the last element with
// positive weight (rounding fallback); else -1.
// This runs once per draw, at the end of a kernel, so its code is kept
// small: the loops over a lane's four vectors are rolled (fully unrolled,
// the first pass of a draw stalled for several microseconds on
// instruction fetches).
template <int DT, class WF>
__device__ int warp_scan_elems(const void *row1, const void *row2, int a, int b, WF W, F2 before, F2 target) {
    using E = Elem<DT>;
    constexpr int PV = E::kPerVec;
    const int lane = lane_id();
    const int nvec = (b - a) / PV;  // <= 128
    const uint4 *p1 = reinterpret_cast<const uint4 *>(static_cast<const unsigned char *>(row1) +
                                                      static_cast<int64_t>(a) * E::kBytes);
    const uint4 *p2 = reinterpret_cast<const uint4 *>(static_cast<const unsigned char *>(row2) +
                                                      static_cast<int64_t>(a) * E::kBytes);
    uint4 r1[4], r2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int vi = 4 * lane + j;
        r1[j] = make_uint4(0u, 0u, 0u, 0u);
        r2[j] = r1[j];
        if (vi < nvec) {
            r1[j] = __ldg(p1 + vi);
            r2[j] = (row2 != row1) ? __ldg(p2 + vi) : r1[j];
        }
    }
    // this lane's vectors are 4 * lane .. 4 * lane + nv - 1
    const int nv = max(0, min(4, nvec - 4 * lane));
    // weights are recomputed in the second pass (same fp32 operations, same
    // order) instead of being kept live
    float lsum = 0.0f;
#pragma unroll 1
    for (int j = 0; j < nv; ++j) {
        float x1[PV], x2[PV];
        E::unpack(pick4(r1, j), x1);
        E::unpack(pick4(r2, j), x2);
#pragma unroll
        for (int q = 0; q < PV; ++q) lsum += W(x1[q], x2[q]);
    }
    const float incl = warp_incl_scan_f(lsum);
    const F2 start = f2_add(before, incl - lsum);
    const float rem = f2_round_down(f2_sub(target, start));  // acc > rem  <=>  start + acc > target
    float acc = 0.0f;
    int found = -1, lastpos = -1;
#pragma unroll 1
    for (int j = 0; j < nv; ++j) {
        float x1[PV], x2[PV];
        E::unpack(pick4(r1, j), x1);
        E::unpack(pick4(r2, j), x2);
#pragma unroll
        for (int q = 0; q < PV; ++q) {
            const float wv = W(x1[q], x2[q]);
            acc += wv;
            if (wv > 0.0f) lastpos = j * PV + q;
            if (found < 0 && wv > 0.0f && acc > rem) found = j * PV + q;
        }
    }
    const unsigned hit = __ballot_sync(0xffffffffu, found >= 0);
    if (hit) {
        const int src = __ffs(hit) - 1;
        return a + 4 * PV * src + __shfl_sync(0xffffffffu, found, src);
    }
    const unsigned pos = __ballot_sync(0xffffffffu, lastpos >= 0);
    if (!pos) return -1;
    const int src = 31 - __clz(pos);
    return a + 4 * PV * src + __shfl_sync(0xffffffffu, lastpos, src);
}

// One draw from a soft row (bonus token or draft token) by one warp:
// locate the sub-chunk from the row's partials (pc: this lane's cached ones,
// from load_parts), then scan its elements.
template <int DT>
__device__ int warp_draw_row(const void *logits, int64_t row, const float2 *part, const float2 (&pc)[kPartCache],
                             const Geometry &g, float c, float M, float u) {
    float w[kPartCache];
#pragma unroll
    for (int j = 0; j < kPartCache; ++j) w[j] = pc[j].x > -INFINITY ? pc[j].y * ex2(pc[j].x - M) : 0.0f;
    auto wfar = [&](int i) -> float {
        const float2 v = __ldcg(part + i);
        return v.x > -INFINITY ? v.y * ex2(v.x - M) : 0.0f;
    };
    F2 before, total, target;
    const int sc = warp_locate(g.n_sub, w, wfar, u, &before, &total, &target);
    if (sc < 0) return -1;
    int a, b;
    sub_range(g, sc, &a, &b);
    const void *rp = static_cast<const unsigned char *>(logits) + row * g.V * static_cast<int64_t>(Elem<DT>::kBytes);
    auto W = [&](float x, float) -> float { return prob_weight(x, c, M); };
    return warp_scan_elems<DT>(rp, rp, a, b, W, before, target);
}

// ================================================================== kernel 2
// The epilogue of spec_verify in one launch of B * nsplit blocks; block
// (b, s) serves sequence b and the s-th of nsplit slices of a row's
// sub-chunks (nsplit is sized so that the grid has a few blocks per SM).
//  1. Every block of b combines the sub-chunk partials of b's rows, forms
//     alpha_i and finds the first rejection n with a warp ballot.  All
//     blocks of b run the same arithmetic on the same data, so they reach
//     the same decision.
//  2. If a drafted token of a sampled sequence was rejected, block s sums
//     max(0, p - q) over its slice of the two rows at position n.
//  3. The warp of b that finishes step 2 last (per-sequence arrival
//     counter, zeroed by stats_kernel) draws the residual token: it locates
//     the sub-chunk where the cumulative mass crosses u * Z and scans its
//     elements.  Block s == 0 writes the accepted prefix, the count and the
//     aux outputs, and draws the bonus (all k accepted) or greedy token.
// The call's inputs (the k_offsets check, drafted tokens and their logits)
// are read before the wait on stats_kernel, which hides that latency behind
// the streaming pass's tail.
// With draft_lse2 given (the draft rows' log2-domain log-sum-exp, written by
// the draft-sampling pass from the same partials this kernel would combine),
// the draft rows were not streamed: their Ld comes from that array, bit for
// bit what the combine below would give.
struct ResolveSmem {
    float M[kMaxK + 1];       // target rows: max of z*c
    float S[kMaxK + 1];       // target rows: sum 2^(z*c - M)
    double Ld[kMaxK];         // draft rows: log2-domain log-sum-exp
    int arg[kMaxK + 1];       // greedy target rows: arg-max
    int ok[2 * kMaxK + 1];
    int n;     // accepted count, -1 on a data error
    int kind;  // kJobNone, kJobResid or kJobBonus
    float lth, ltl, ldh, ldl, u;
};

#ifndef SPEC_RESOLVE_MIN_BLOCKS
#define SPEC_RESOLVE_MIN_BLOCKS 4
#endif
template <int DT>
__global__ void __launch_bounds__(256, SPEC_RESOLVE_MIN_BLOCKS) resolve_kernel(
    const void *__restrict__ target, const void *__restrict__ draft,
    const int32_t *__restrict__ tokens, const float *__restrict__ u_accept,
    const float *__restrict__ u_resample, const float *__restrict__ temperature,
    const int *__restrict__ k_offsets, const double *__restrict__ draft_lse2, int B, Geometry g, int nsplit,
    WsPtrs ws, int32_t *__restrict__ out_tokens, int32_t *__restrict__ out_num, spec_verify_aux_t aux) {
    using E = Elem<DT>;
    __shared__ ResolveSmem sm;
    const int b = blockIdx.x / nsplit;
    const int s = blockIdx.x - b * nsplit;
    const int lane = lane_id(), warp = warp_id();

    // --- inputs only (written before this call) --------------------------
    // the same k_offsets check as stats_kernel: only with it do the row
    // indices below stay inside the caller's buffers
    int bad = 0;
    for (int i = threadIdx.x; i <= B; i += blockDim.x) {
        const int v = k_offsets[i];
        if (i == 0) {
            bad |= v != 0;
        } else {
            const int kk = v - k_offsets[i - 1];
            bad |= (kk < 0 || kk > kMaxK);
        }
    }
    bad = __syncthreads_or(bad);
    if (bad) {
        // the whole call fails; outputs of unknown size stay untouched
        grid_dependency_wait();
        if (s == 0 && threadIdx.x == 0) {
            out_num[b] = -1;
            if (aux.residual_mass) aux.residual_mass[b] = NAN;
            if (b == 0) set_status(ws.counters + kStatus, SPEC_ERR_INVALID_ARG);
        }
        return;
    }
    const int k0 = k_offsets[b];
    const int k = k_offsets[b + 1] - k0;
    const int64_t ot = static_cast<int64_t>(k0) + b;  // first target row / output slot
    const int64_t od = k0;                            // first draft row
    const int64_t R_t = static_cast<int64_t>(k_offsets[B]) + B;
    const float c = temp_scale(temperature[b]);
    const int V = g.V;
    const bool greedy = (c == 0.0f);
    const bool given = draft_lse2 != nullptr;
    int x = 0;
    bool xbad = false;
    float zt = 0.0f, zd = 0.0f, ua = 0.0f, ur = 0.0f;
    if (warp == 0 && lane <= k) {
        ur = u_resample[ot + lane];  // lane <= k <= 32 is at most lane 31 here
        if (lane < k) {
            x = tokens[od + lane];
            ua = u_accept[od + lane];
            xbad = (x < 0 || x >= V);
            if (!xbad && !greedy && c == c) {
                zt = E::load1(target, (ot + lane) * V + x);
                zd = E::load1(draft, (od + lane) * V + x);
                if (given) sm.Ld[lane] = draft_lse2[od + lane];  // read by warp 0 only
            }
        }
    }

    // --- 1. row statistics and the decision -------------------------------
    grid_dependency_wait();
    if (c == c) {
        const int nrows = (greedy || given) ? k + 1 : 2 * k + 1;
        for (int rr = warp; rr < nrows; rr += blockDim.x >> 5) {
            const bool is_t = rr <= k;
            const int i = is_t ? rr : rr - k - 1;
            const int si = is_t ? i : kMaxK + 1 + i;
            const int64_t slot_row = is_t ? ot + i : R_t + od + i;
            const float2 *p = ws.part + slot_row * g.n_sub;
            if (greedy) {
                const int am = warp_combine_arg(p, g.n_sub);
                if (lane == 0) {
                    sm.arg[si] = am;
                    sm.ok[si] = am >= 0;
                }
            } else {
                float M, S;
                const bool ok = warp_combine_soft(p, g.n_sub, &M, &S);
                if (lane == 0) {
                    if (is_t) {
                        sm.M[i] = M;
                        sm.S[i] = S;
                    } else {
                        sm.Ld[i] = ok ? lse2(M, S) : NAN;
                    }
                    sm.ok[si] = ok;
                }
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        bool err = (c != c) || __any_sync(0xffffffffu, xbad);
        int n = -1, tok = -1, kind = kJobNone;
        float alpha_out = NAN;
        double Lt = NAN, Ld = NAN;
        if (!err) {
            bool rows_ok = true;
            for (int i = lane; i <= k; i += 32) rows_ok &= sm.ok[i] != 0;
            if (!greedy) {
                if (given)
                    rows_ok &= lane >= k || isfinite(sm.Ld[lane]);
                else
                    for (int i = lane; i < k; i += 32) rows_ok &= sm.ok[kMaxK + 1 + i] != 0;
            }
            err = !__all_sync(0xffffffffu, rows_ok);
        }
        if (!err && greedy) {
            // greedy: accept while x_i == argmax p_i
            const int a = (lane <= k) ? sm.arg[lane] : 0;
            const unsigned mism = __ballot_sync(0xffffffffu, lane < k && x != a);
            n = mism ? (__ffs(mism) - 1) : k;
            tok = sm.arg[n];
        } else if (!err) {
            // alpha_i = min(1, p_i(x_i) / q_i(x_i)) in the log domain: log-ratio
            // in fp64 scalars, the exponential in fp32 (alpha abs. error ~1e-7)
            bool acc = false;
            if (lane < k) {
                Lt = lse2(sm.M[lane], sm.S[lane]);
                Ld = sm.Ld[lane];
                float alpha;
                if (zt == -INFINITY) {
                    alpha = 0.0f;
                } else if (zd == -INFINITY) {
                    alpha = 1.0f;
                } else {
                    const double cd = static_cast<double>(c);
                    const double lr = (static_cast<double>(zt) * cd - Lt) - (static_cast<double>(zd) * cd - Ld);
                    alpha = lr >= 0.0 ? 1.0f : exp2f(static_cast<float>(lr));
                }
                alpha_out = alpha;
                acc = ua < alpha;
            } else if (lane == k) {
                Lt = lse2(sm.M[k], sm.S[k]);
            }
            const unsigned rej = __ballot_sync(0xffffffffu, lane < k && !acc);
            n = rej ? (__ffs(rej) - 1) : k;
            kind = n < k ? kJobResid : kJobBonus;
            // u at position n; position 32 (k = 32, all accepted) has no lane
            float u_n = __shfl_sync(0xffffffffu, ur, n & 31);
            if (n == 32) u_n = u_resample[ot + 32];
            const double Ldn = __shfl_sync(0xffffffffu, Ld, n & 31);  // used only if n < k
            if (lane == 0) {
                if (n < k) {
                    const double Ltn = lse2(sm.M[n], sm.S[n]);
                    sm.lth = static_cast<float>(Ltn);
                    sm.ltl = static_cast<float>(Ltn - static_cast<double>(sm.lth));
                    sm.ldh = static_cast<float>(Ldn);
                    sm.ldl = static_cast<float>(Ldn - static_cast<double>(sm.ldh));
                }
                sm.u = u_n;
            }
        }
        if (lane == 0) {
            sm.n = n;
            sm.kind = kind;
        }
        if (s == 0) {
            // outputs: prefix, the greedy token at n (sampled draws are
            // written by the drawing block), -1 after; everything -1 on a
            // data error
            for (int i = lane; i <= k; i += 32) {
                if (i == n && kind != kJobNone) continue;
                int32_t o = -1;
                if (n >= 0) {
                    if (i < n) o = x;  // i < n <= 32, so i == lane: this lane's own token
                    else if (i == n && greedy) o = tok;
                }
                out_tokens[ot + i] = o;
            }
            if (lane == 0) {
                out_num[b] = n;
                if (aux.residual_mass && kind != kJobResid) aux.residual_mass[b] = NAN;
            }
            if (aux.accept_prob && lane < k) aux.accept_prob[od + lane] = (n >= 0 && !greedy) ? alpha_out : NAN;
            if (aux.lse_target)
                for (int i = lane; i <= k; i += 32) {
                    float v = NAN;
                    if (n >= 0 && !greedy) v = static_cast<float>(lse2(sm.M[i], sm.S[i]) * kLn2D);
                    aux.lse_target[ot + i] = v;
                }
            if (aux.lse_draft && lane < k)
                aux.lse_draft[od + lane] = (n >= 0 && !greedy) ? static_cast<float>(Ld * kLn2D) : NAN;
        }
    }
    __syncthreads();
    const int kind = sm.kind;
    if (kind == kJobNone) return;
    const int n = sm.n;
    const int64_t trow = ot + n;

    if (kind == kJobBonus) {
        // --- bonus draw from p at position k, by block 0 of b --------------
        if (s != 0 || warp != 0) return;
        const float2 *pr = ws.part + trow * g.n_sub;
        float2 pc[kPartCache];
        load_parts(pr, g.n_sub, pc);
        const int token = warp_draw_row<DT>(target, trow, pr, pc, g, c, sm.M[k], sm.u);
        if (lane == 0) out_tokens[trow] = token;
        return;
    }

    // --- 2. residual mass of this block's slice of sub-chunks -------------
    const int64_t drow = od + n;
    const float lth = sm.lth, ltl = sm.ltl, ldh = sm.ldh, ldl = sm.ldl;
    const float2 c2 = make_float2(c, c), nlth2 = make_float2(-lth, -lth), nltl2 = make_float2(-ltl, -ltl);
    const float2 nldh2 = make_float2(-ldh, -ldh), nldl2 = make_float2(-ldl, -ldl);
    float *rp = ws.resid_part + static_cast<int64_t>(b) * g.n_sub;
    const int per = (g.n_sub + nsplit - 1) / nsplit;
    const int sc_begin = s * per;
    const int sc_end = min(g.n_sub, (s + 1) * per);
    if (SPEC_RESID_PREFETCH && warp == 0 && sc_begin < sc_end) {
        // the slice of both rows goes to L2 in bulk (up to 32 KB per lane),
        // so the warps' loads below wait on L2, not on DRAM round trips
        int a0, a1, e0, e1;
        sub_range(g, sc_begin, &a0, &e0);
        sub_range(g, sc_end - 1, &a1, &e1);
        const int64_t nbytes = static_cast<int64_t>(e1 - a0) * E::kBytes;
        const unsigned char *t0 = static_cast<const unsigned char *>(target) + (trow * V + a0) * static_cast<int64_t>(E::kBytes);
        const unsigned char *d0 = static_cast<const unsigned char *>(draft) + (drow * V + a0) * static_cast<int64_t>(E::kBytes);
        constexpr int64_t kPiece = 32768;
        for (int64_t off = static_cast<int64_t>(lane >> 1) * kPiece; off < nbytes; off += 16 * kPiece) {
            const uint32_t len = static_cast<uint32_t>(min(kPiece, nbytes - off));
            bulk_prefetch_l2(((lane & 1) ? d0 : t0) + off, len);
        }
    }
    for (int sc = sc_begin + warp; sc < sc_end; sc += blockDim.x >> 5) {
        int a, e1;
        sub_range(g, sc, &a, &e1);
        const int nvec = (e1 - a) / E::kPerVec;  // <= 128
        const uint4 *pt = reinterpret_cast<const uint4 *>(static_cast<const unsigned char *>(target) +
                                                          (trow * V + a) * static_cast<int64_t>(E::kBytes));
        const uint4 *pd = reinterpret_cast<const uint4 *>(static_cast<const unsigned char *>(draft) +
                                                          (drow * V + a) * static_cast<int64_t>(E::kBytes));
        uint4 xt4[4], xd4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = lane + 32 * j;
            if (i < nvec) {
                xt4[j] = ld_stream(pt + i);
                xd4[j] = ld_stream(pd + i);
            }
        }
        float2 acc0 = make_float2(0.0f, 0.0f), acc1 = acc0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (lane + 32 * j >= nvec) continue;
#pragma unroll
            for (int p = 0; p < E::kPairs; ++p) {
                const float2 w2 = resid_weight2(E::pair(xt4[j], p), E::pair(xd4[j], p), c2, nlth2, nltl2, nldh2, nldl2);
                if (p & 1) acc1 = fadd2(acc1, w2); else acc0 = fadd2(acc0, w2);
            }
        }
        const float sum = warp_sum_f((acc0.x + acc0.y) + (acc1.x + acc1.y));
        if (lane == 0) rp[sc] = sum;
    }
    // arrival, one per warp (no block barrier): the warp that arrives last,
    // of all nsplit * 8 warps of b, draws
    // (acquire-release add: this warp's masses are released with it, and
    // the last warp acquires everyone's)
    bool last = false;
    if (lane == 0)
        last = atomic_add_acq_rel_gpu(ws.seqcnt + b, 1) == nsplit * static_cast<int>(blockDim.x >> 5) - 1;
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __syncwarp();  // lane 0's acquire, before the other lanes' reads

    // --- 3. the residual draw, by the last warp of b -----------------------
    float w[kPartCache];
#pragma unroll
    for (int j = 0; j < kPartCache; ++j) w[j] = (lane + 32 * j < g.n_sub) ? __ldcg(rp + lane + 32 * j) : 0.0f;
    auto wfar = [&](int i) -> float { return __ldcg(rp + i); };
    F2 before, Z, tgt;
    const int sc = warp_locate(g.n_sub, w, wfar, sm.u, &before, &Z, &tgt);
    int token = -1;
    if (sc >= 0) {
        int a, e1;
        sub_range(g, sc, &a, &e1);
        const void *rt = static_cast<const unsigned char *>(target) + trow * V * static_cast<int64_t>(E::kBytes);
        const void *rd = static_cast<const unsigned char *>(draft) + drow * V * static_cast<int64_t>(E::kBytes);
        auto W = [&](float a1, float a2) -> float { return resid_weight(a1, a2, c, lth, ltl, ldh, ldl); };
        token = warp_scan_elems<DT>(rt, rd, a, e1, W, before, tgt);
    }
    if (lane == 0) {
        out_tokens[trow] = token;
        if (aux.residual_mass) aux.residual_mass[b] = __fadd_rn(Z.hi, Z.lo);
    }
}

// Draft-side draw: one warp per draft row (grid-stride over rows).  With
// out_lse2 given, each row's log2-domain log-sum-exp (the value
// resolve_kernel would combine from the same partials) is written too: NaN
// for greedy and invalid rows.
template <int DT>
__global__ void __launch_bounds__(256) draft_select_kernel(
    const void *__restrict__ draft, const float *__restrict__ temperature, const float *__restrict__ u_draft,
    const int *__restrict__ k_offsets, int B, Geometry g, const float2 *__restrict__ part,
    int32_t *__restrict__ out, double *__restrict__ out_lse2, int *__restrict__ counters) {
    extern __shared__ int s_kofs[];  // [B+1]
    __shared__ int s_bad;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int i = threadIdx.x; i <= B; i += blockDim.x) {
        const int v = k_offsets[i];
        s_kofs[i] = v;
        if (i == 0 && v != 0) s_bad = 1;
        if (i > 0) {
            const int k = v - k_offsets[i - 1];
            if (k < 0 || k > kMaxK) s_bad = 1;
        }
    }
    __syncthreads();
    grid_dependency_wait();
    grid_launch_dependents();
    if (s_bad) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(counters + kStatus, SPEC_ERR_INVALID_ARG);
        return;
    }
    const int R = s_kofs[B];
    const int lane = lane_id();
    const int nw = (gridDim.x * blockDim.x) >> 5;
    for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < R; r += nw) {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_kofs[mid] <= r) lo = mid; else hi = mid - 1;
        }
        const float c = temp_scale(temperature[lo]);
        const float2 *pr = part + static_cast<int64_t>(r) * g.n_sub;
        int token = -1;
        double L = NAN;
        if (c == 0.0f) {
            token = warp_combine_arg(pr, g.n_sub);
        } else if (c == c) {
            float M, S;
            float2 pc[kPartCache];
            load_parts(pr, g.n_sub, pc);  // one round trip serves the combine and the draw
            if (combine_soft(pc, pr, g.n_sub, &M, &S)) {
                L = lse2(M, S);
                token = warp_draw_row<DT>(draft, r, pr, pc, g, c, M, u_draft[r]);
            }
        }
        if (lane == 0) {
            out[r] = token;
            if (out_lse2) out_lse2[r] = L;
        }
    }
}

// ================================================================== host side
struct DeviceState {
    bool init = false;
    int sms = 0;
    int smem_per_sm = 0;
    int smem_optin = 0;
    void *ws = nullptr;
    size_t ws_bytes = 0;
    void *stage = nullptr;
    size_t stage_bytes = 0;
};

constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool make_geometry(int V, int dtype, Geometry *g) {
    const int s = dtype == SPEC_F32 ? 4 : 2;
    const int pv = 16 / s;
    const int64_t vb = static_cast<int64_t>(V) * s;
    const int n0 = static_cast<int>((vb + kSlotBytes - 1) / kSlotBytes);
    int ce = (V + n0 - 1) / n0;
    ce = (ce + 2 * pv - 1) / (2 * pv) * (2 * pv);
    g->V = V;
    g->chunk_elems = ce;
    g->n_chunks = (V + ce - 1) / ce;
    g->sub_elems = kSubVecs * pv;
    g->n_sub = g->n_chunks * kSub;
    return true;
}

struct WsLayout {
    size_t part, counters, seqcnt, resid, lse2, total;
};

// Workspace layout.  The counters block comes first so that the status word
// has a fixed offset (kStatusOffset) whatever B and V are.
constexpr size_t kStatusOffset = sizeof(int) * kStatus;
constexpr size_t kTicketOffset = sizeof(int) * kTicket;  // the ticket words up to kCounterWords
constexpr size_t kCountersBytes = 256;

WsLayout ws_layout(int B, const Geometry &g) {
    WsLayout l;
    size_t off = 0;
    const size_t rows_cap = static_cast<size_t>(2 * kMaxK + 1) * B;
    l.counters = off;
    off = align_up(off + kCountersBytes, 256);
    l.part = off;
    off = align_up(off + rows_cap * g.n_sub * sizeof(float2), 256);
    l.seqcnt = off;
    off = align_up(off + B * sizeof(int), 256);
    l.resid = off;
    off = align_up(off + static_cast<size_t>(B) * g.n_sub * sizeof(float), 256);
    l.lse2 = off;  // spec_round: the draft rows' lse2 between its two passes
    off = align_up(off + static_cast<size_t>(B) * kMaxK * sizeof(double), 256);
    l.total = off;
    return l;
}

WsPtrs ws_ptrs(void *base, const WsLayout &l) {
    unsigned char *p = static_cast<unsigned char *>(base);
    WsPtrs w;
    w.part = reinterpret_cast<float2 *>(p + l.part);
    w.counters = reinterpret_cast<int *>(p + l.counters);
    w.seqcnt = reinterpret_cast<int *>(p + l.seqcnt);
    w.resid_part = reinterpret_cast<float *>(p + l.resid);
    return w;
}

// Last CUDA failure seen by this thread (call site + CUDA error name).
thread_local char g_last_error[256] = "";

bool cuda_ok(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return true;
    snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", what, cudaGetErrorName(e),
             cudaGetErrorString(e));
    return false;
}

// Allow the kernel the opt-in dynamic shared memory minus its static part.
template <int DT, int MODE>
bool set_stats_attrs(int smem_optin) {
    cudaFuncAttributes fa{};
    if (!cuda_ok(cudaFuncGetAttributes(&fa, stats_kernel<DT, MODE>), "cudaFuncGetAttributes")) return false;
    const int dyn = smem_optin - static_cast<int>(fa.sharedSizeBytes);
    return cuda_ok(cudaFuncSetAttribute(stats_kernel<DT, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn),
                   "cudaFuncSetAttribute(stats_kernel)");
}

template <int DT>
bool set_stats_attrs_all(int smem_optin) {
    return set_stats_attrs<DT, kModeVerify>(smem_optin) && set_stats_attrs<DT, kModeDraft>(smem_optin) &&
           set_stats_attrs<DT, kModeTarget>(smem_optin);
}

DeviceState *device_state(int *dev_out) {
    int dev = 0;
    if (!cuda_ok(cudaGetDevice(&dev), "cudaGetDevice") || dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceState &st = g_dev[dev];
    std::lock_guard<std::mutex> lock(g_mu);
    if (!st.init) {
        if (!cuda_ok(cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute") ||
            !cuda_ok(cudaDeviceGetAttribute(&st.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev),
                     "cudaDeviceGetAttribute") ||
            !cuda_ok(cudaDeviceGetAttribute(&st.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev),
                     "cudaDeviceGetAttribute"))
            return nullptr;
        if (!set_stats_attrs_all<SPEC_F32>(st.smem_optin) || !set_stats_attrs_all<SPEC_BF16>(st.smem_optin))
            return nullptr;
        st.smem_optin -= 1024;  // headroom for the kernels' static shared memory
        st.init = true;
    }
    *dev_out = dev;
    return &st;
}

// Dynamic shared memory of stats_kernel with ns ring slots.
size_t stats_smem(int ns, int B) {
    size_t s = static_cast<size_t>(ns) * kSlotBytes;
    s += 2 * ns * sizeof(uint64_t);
    s += ns * sizeof(UnitDesc);
    s += static_cast<size_t>(B + 1) * 2 * sizeof(int) + B * sizeof(float);
    s += (kThreads / 32 + 2) * sizeof(int);
    return align_up(s, 128);
}

// Ring depth and CTAs per SM of stats_kernel: the preferred shape
// (SPEC_STATS_CTAS_PER_SM CTAs with SPEC_STATS_SLOTS slots each; four CTAs
// of three 16 KB slots give 32 consumer warps and 192 KB in flight per SM,
// measured a little faster than three CTAs of four slots) if the tables fit
// beside it, else two CTAs with up to kMaxSlots, else one.
#ifndef SPEC_STATS_CTAS_PER_SM
#define SPEC_STATS_CTAS_PER_SM 4
#endif
#ifndef SPEC_STATS_SLOTS
#define SPEC_STATS_SLOTS 3
#endif
void pick_ring(const DeviceState &st, int B, int *ns, size_t *smem, int *ctas_per_sm) {
    struct Opt {
        int per_sm, min_ns, max_ns;
    };
    const Opt opts[] = {{SPEC_STATS_CTAS_PER_SM, SPEC_STATS_SLOTS, SPEC_STATS_SLOTS}, {2, 3, kMaxSlots}, {1, 2, kMaxSlots}};
    for (const Opt &o : opts) {
        const size_t budget = static_cast<size_t>(st.smem_per_sm) / o.per_sm - 1024;
        for (int n = o.max_ns; n >= o.min_ns; --n) {
            const size_t s = stats_smem(n, B);
            if (s <= budget && s <= static_cast<size_t>(st.smem_optin)) {
                *ns = n;
                *smem = s;
                *ctas_per_sm = o.per_sm;
                return;
            }
        }
    }
    *ns = 0;
}

void *get_internal_ws(DeviceState &st, size_t need) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (st.ws_bytes >= need) return st.ws;
    if (st.ws) {
        cudaDeviceSynchronize();
        cudaFree(st.ws);
        st.ws = nullptr;
        st.ws_bytes = 0;
    }
    void *p = nullptr;
    if (!cuda_ok(cudaMalloc(&p, need), "cudaMalloc(workspace)")) return nullptr;
    if (!cuda_ok(cudaMemset(p, 0, need), "cudaMemset(workspace)")) {
        cudaFree(p);
        return nullptr;
    }
    st.ws = p;
    st.ws_bytes = need;
    return p;
}

// A caller-owned workspace may hold anything: zero its unit-ticket words on
// the stream before the call's first kernel.  (The library-owned workspaces
// are zeroed when allocated; stats_kernel leaves the words at zero.)
bool reset_tickets(void *ws, cudaStream_t stream) {
    return cuda_ok(cudaMemsetAsync(static_cast<unsigned char *>(ws) + kTicketOffset, 0,
                                   (kCounterWords - kTicket) * sizeof(int), stream),
                   "cudaMemsetAsync(workspace tickets)");
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(int B, int V, int dtype) {
    if (B < 0 || B > SPEC_MAX_B || V <= 0 || V > SPEC_MAX_V) return SPEC_ERR_INVALID_ARG;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
    const int s = dtype == SPEC_F32 ? 4 : 2;
    if ((static_cast<int64_t>(V) * s) % 16 != 0) return SPEC_ERR_ALIGNMENT;
    return SPEC_OK;
}

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

#ifndef SPEC_RESOLVE_BLOCKS_PER_SM
#define SPEC_RESOLVE_BLOCKS_PER_SM 8
#endif
// resolve_kernel blocks per sequence for n sequences on an idle GPU:
// 1..kSub, as many as fit one wave of SPEC_RESOLVE_BLOCKS_PER_SM per SM.
int resolve_split(const DeviceState &st, const Geometry &g, int n) {
    return std::max(1, std::min({kSub, g.n_sub, (SPEC_RESOLVE_BLOCKS_PER_SM * st.sms) / std::max(n, 1)}));
}

// The verify pass: stats_kernel streams the target rows (and, without
// draft_lse2, the draft rows of sampled sequences), then resolve_kernel.
// pdl_first: the call's first kernel may start early, which is safe only
// when an earlier kernel of the same call precedes it on the stream.
template <int DT>
int launch_verify(const void *target, const void *draft, const double *draft_lse2, const int32_t *tokens,
                  const float *u_accept, const float *u_resample, const float *temperature, int B,
                  const int32_t *k_offsets, const Geometry &g, int32_t *out_tokens, int32_t *out_num,
                  const spec_verify_aux_t &aux, void *ws_base, const WsLayout &l, const DeviceState &st,
                  cudaStream_t stream, bool pdl_first = false) {
    int ns, per_sm;
    size_t smem;
    pick_ring(st, B, &ns, &smem, &per_sm);
    if (ns == 0) return SPEC_ERR_INVALID_ARG;
    const WsPtrs w = ws_ptrs(ws_base, l);
    const int grid = st.sms * per_sm;
    const int nsplit = resolve_split(st, g, B);
    const cudaError_t e1 =
        draft_lse2 ? launch_k(pdl_first, stats_kernel<DT, kModeTarget>, dim3(grid), dim3(kThreads), smem, stream,
                              target, draft, temperature, k_offsets, B, g, ns, w.part, w.counters, w.seqcnt)
                   : launch_k(pdl_first, stats_kernel<DT, kModeVerify>, dim3(grid), dim3(kThreads), smem, stream,
                              target, draft, temperature, k_offsets, B, g, ns, w.part, w.counters, w.seqcnt);
    if (!cuda_ok(e1, "launch stats_kernel") ||
        !cuda_ok(launch_k(true, resolve_kernel<DT>, dim3(B * nsplit), dim3(256), 0, stream, target, draft, tokens,
                          u_accept, u_resample, temperature, k_offsets, draft_lse2, B, g, nsplit, w, out_tokens,
                          out_num, aux),
                 "launch resolve_kernel"))
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

#ifndef SPEC_SELECT_BLOCKS_PER_SM
#define SPEC_SELECT_BLOCKS_PER_SM 8
#endif
template <int DT>
int launch_draft(const void *draft, const float *temperature, const float *u_draft, int B,
                 const int32_t *k_offsets, const Geometry &g, int32_t *out, double *out_lse2, void *ws_base,
                 const WsLayout &l, const DeviceState &st, cudaStream_t stream) {
    int ns, per_sm;
    size_t smem;
    pick_ring(st, B, &ns, &smem, &per_sm);
    if (ns == 0) return SPEC_ERR_INVALID_ARG;
    const WsPtrs w = ws_ptrs(ws_base, l);
    // one warp per draft row (grid-stride): at most B * kMaxK rows, 8 warps per block
    const int grid = static_cast<int>(
        std::min(static_cast<int64_t>(st.sms) * SPEC_SELECT_BLOCKS_PER_SM, (static_cast<int64_t>(B) * kMaxK + 7) / 8));
    if (!cuda_ok(launch_k(false, stats_kernel<DT, kModeDraft>, dim3(st.sms * per_sm), dim3(kThreads), smem, stream,
                          draft, draft, temperature, k_offsets, B, g, ns, w.part, w.counters, nullptr),
                 "launch stats_kernel") ||
        !cuda_ok(launch_k(true, draft_select_kernel<DT>, dim3(std::max(grid, 1)), dim3(256),
                          (B + 1) * sizeof(int), stream, draft, temperature, u_draft, k_offsets, B, g,
                          static_cast<const float2 *>(w.part), out, out_lse2, w.counters),
                 "launch draft_select_kernel"))
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

}  // namespace specv

using namespace specv;

extern "C" {

size_t spec_workspace_bytes(int B, int V, int dtype) {
    if (check_common(B, V, dtype) != SPEC_OK) return 0;
    Geometry g;
    make_geometry(V, dtype, &g);
    return ws_layout(std::max(B, 1), g).total;
}

size_t spec_noalloc_bytes(int B, int V, int dtype) { return spec_workspace_bytes(B, V, dtype); }

}  // extern "C"

namespace specv {

// The workspace of one call: the caller's (checked, its ticket words
// zeroed on the stream) or the library-owned one.  nullptr with *rc set on
// failure.
void *call_workspace(void *workspace, size_t workspace_bytes, const WsLayout &l, DeviceState &st,
                     cudaStream_t stream, int *rc) {
    *rc = SPEC_OK;
    if (workspace) {
        if (workspace_bytes < l.total) *rc = SPEC_ERR_WORKSPACE;
        else if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) *rc = SPEC_ERR_ALIGNMENT;
        else if (!reset_tickets(workspace, stream)) *rc = SPEC_ERR_CUDA;
        return *rc == SPEC_OK ? workspace : nullptr;
    }
    void *ws = get_internal_ws(st, l.total);
    if (!ws) *rc = SPEC_ERR_CUDA;
    return ws;
}

int verify_call(const void *target_logits, const void *draft_logits, const double *draft_lse2,
                const int32_t *draft_tokens, const float *u_accept, const float *u_resample, const float *temperature,
                int B, const int32_t *k_offsets, int V, int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
                const spec_verify_aux_t *aux, void *workspace, size_t workspace_bytes, void *stream) {
    int rc = check_common(B, V, dtype);
    if (rc != SPEC_OK) return rc;
    if (B == 0) return SPEC_OK;
    if (!target_logits || !draft_logits || !draft_tokens || !u_accept || !u_resample || !temperature ||
        !k_offsets || !out_tokens || !out_num_accepted)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || !aligned16(draft_logits)) return SPEC_ERR_ALIGNMENT;
    Geometry g;
    make_geometry(V, dtype, &g);
    const WsLayout l = ws_layout(B, g);
    int dev;
    DeviceState *st = device_state(&dev);
    if (!st) return SPEC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *ws = call_workspace(workspace, workspace_bytes, l, *st, s, &rc);
    if (!ws) return rc;
    spec_verify_aux_t a{};
    if (aux) a = *aux;
    if (dtype == SPEC_F32)
        return launch_verify<SPEC_F32>(target_logits, draft_logits, draft_lse2, draft_tokens, u_accept, u_resample,
                                       temperature, B, k_offsets, g, out_tokens, out_num_accepted, a, ws, l, *st, s);
    return launch_verify<SPEC_BF16>(target_logits, draft_logits, draft_lse2, draft_tokens, u_accept, u_resample,
                                    temperature, B, k_offsets, g, out_tokens, out_num_accepted, a, ws, l, *st, s);
}

int draft_call(const void *draft_logits, const float *temperature, const float *u_draft, int B,
               const int32_t *k_offsets, int V, int dtype, int32_t *out_draft_tokens, double *out_draft_lse2,
               void *workspace, size_t workspace_bytes, void *stream) {
    int rc = check_common(B, V, dtype);
    if (rc != SPEC_OK) return rc;
    if (B == 0) return SPEC_OK;
    if (!draft_logits || !temperature || !u_draft || !k_offsets || !out_draft_tokens) return SPEC_ERR_INVALID_ARG;
    if (!aligned16(draft_logits)) return SPEC_ERR_ALIGNMENT;
    Geometry g;
    make_geometry(V, dtype, &g);
    const WsLayout l = ws_layout(B, g);
    int dev;
    DeviceState *st = device_state(&dev);
    if (!st) return SPEC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *ws = call_workspace(workspace, workspace_bytes, l, *st, s, &rc);
    if (!ws) return rc;
    if (dtype == SPEC_F32)
        return launch_draft<SPEC_F32>(draft_logits, temperature, u_draft, B, k_offsets, g, out_draft_tokens,
                                      out_draft_lse2, ws, l, *st, s);
    return launch_draft<SPEC_BF16>(draft_logits, temperature, u_draft, B, k_offsets, g, out_draft_tokens,
                                   out_draft_lse2, ws, l, *st, s);
}

// One round on device buffers: the draft pass (tokens and the draft rows'
// lse2, kept in the workspace), then the verify pass over the target rows.
int round_call(const void *target_logits, const void *draft_logits, const float *u_draft, const float *u_accept,
               const float *u_resample, const float *temperature, int B, const int32_t *k_offsets, int V, int dtype,
               int32_t *out_draft_tokens, int32_t *out_tokens, int32_t *out_num_accepted, void *stream) {
    int rc = check_common(B, V, dtype);
    if (rc != SPEC_OK) return rc;
    if (B == 0) return SPEC_OK;
    if (!target_logits || !draft_logits || !u_draft || !u_accept || !u_resample || !temperature || !k_offsets ||
        !out_draft_tokens || !out_tokens || !out_num_accepted)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || !aligned16(draft_logits)) return SPEC_ERR_ALIGNMENT;
    Geometry g;
    make_geometry(V, dtype, &g);
    const WsLayout l = ws_layout(B, g);
    int dev;
    DeviceState *st = device_state(&dev);
    if (!st) return SPEC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *ws = call_workspace(nullptr, 0, l, *st, s, &rc);
    if (!ws) return rc;
    double *lse2 = reinterpret_cast<double *>(static_cast<unsigned char *>(ws) + l.lse2);
    const spec_verify_aux_t a{};
    if (dtype == SPEC_F32) {
        rc = launch_draft<SPEC_F32>(draft_logits, temperature, u_draft, B, k_offsets, g, out_draft_tokens, lse2, ws,
                                    l, *st, s);
        if (rc != SPEC_OK) return rc;
        return launch_verify<SPEC_F32>(target_logits, draft_logits, lse2, out_draft_tokens, u_accept, u_resample,
                                       temperature, B, k_offsets, g, out_tokens, out_num_accepted, a, ws, l, *st, s,
                                       true);
    }
    rc = launch_draft<SPEC_BF16>(draft_logits, temperature, u_draft, B, k_offsets, g, out_draft_tokens, lse2, ws, l,
                                 *st, s);
    if (rc != SPEC_OK) return rc;
    return launch_verify<SPEC_BF16>(target_logits, draft_logits, lse2, out_draft_tokens, u_accept, u_resample,
                                    temperature, B, k_offsets, g, out_tokens, out_num_accepted, a, ws, l, *st, s,
                                    true);
}

}  // namespace specv

extern "C" {

int spec_verify_ex(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                   const float *u_accept, const float *u_resample, const float *temperature, int B,
                   const int32_t *k_offsets, int V, int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
                   const spec_verify_aux_t *aux, void *workspace, size_t workspace_bytes, void *stream) {
    return verify_call(target_logits, draft_logits, nullptr, draft_tokens, u_accept, u_resample, temperature, B,
                       k_offsets, V, dtype, out_tokens, out_num_accepted, aux, workspace, workspace_bytes, stream);
}

int spec_verify(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                const float *u_accept, const float *u_resample, const float *temperature, int B,
                const int32_t *k_offsets, int V, int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
                void *stream) {
    return verify_call(target_logits, draft_logits, nullptr, draft_tokens, u_accept, u_resample, temperature, B,
                       k_offsets, V, dtype, out_tokens, out_num_accepted, nullptr, nullptr, 0, stream);
}

int spec_verify_lse(const void *target_logits, const void *draft_logits, const double *draft_lse2,
                    const int32_t *draft_tokens, const float *u_accept, const float *u_resample,
                    const float *temperature, int B, const int32_t *k_offsets, int V, int dtype,
                    int32_t *out_tokens, int32_t *out_num_accepted, const spec_verify_aux_t *aux, void *workspace,
                    size_t workspace_bytes, void *stream) {
    if (B > 0 && !draft_lse2) return SPEC_ERR_INVALID_ARG;
    return verify_call(target_logits, draft_logits, draft_lse2, draft_tokens, u_accept, u_resample, temperature, B,
                       k_offsets, V, dtype, out_tokens, out_num_accepted, aux, workspace, workspace_bytes, stream);
}

int spec_draft_sample_ex(const void *draft_logits, const float *temperature, const float *u_draft, int B,
                         const int32_t *k_offsets, int V, int dtype, int32_t *out_draft_tokens, void *workspace,
                         size_t workspace_bytes, void *stream) {
    return draft_call(draft_logits, temperature, u_draft, B, k_offsets, V, dtype, out_draft_tokens, nullptr,
                      workspace, workspace_bytes, stream);
}

int spec_draft_sample(const void *draft_logits, const float *temperature, const float *u_draft, int B,
                      const int32_t *k_offsets, int V, int dtype, int32_t *out_draft_tokens, void *stream) {
    return draft_call(draft_logits, temperature, u_draft, B, k_offsets, V, dtype, out_draft_tokens, nullptr,
                      nullptr, 0, stream);
}

int spec_draft_sample_lse(const void *draft_logits, const float *temperature, const float *u_draft, int B,
                          const int32_t *k_offsets, int V, int dtype, int32_t *out_draft_tokens,
                          double *out_draft_lse2, void *workspace, size_t workspace_bytes, void *stream) {
    if (B > 0 && !out_draft_lse2) return SPEC_ERR_INVALID_ARG;
    return draft_call(draft_logits, temperature, u_draft, B, k_offsets, V, dtype, out_draft_tokens, out_draft_lse2,
                      workspace, workspace_bytes, stream);
}

int spec_round(const void *target_logits, const void *draft_logits, const float *u_draft, const float *u_accept,
               const float *u_resample, const float *temperature, int B, const int32_t *k_offsets, int V, int dtype,
               int32_t *out_draft_tokens, int32_t *out_tokens, int32_t *out_num_accepted, void *stream) {
    return round_call(target_logits, draft_logits, u_draft, u_accept, u_resample, temperature, B, k_offsets, V,
                      dtype, out_draft_tokens, out_tokens, out_num_accepted, stream);
}

int spec_round_host(const void *target_logits_host, const void *draft_logits_host, const float *u_draft_host,
                    const float *u_accept_host, const float *u_resample_host, const float *temperature_host, int B,
                    const int32_t *k_offsets_host, int V, int dtype, int32_t *out_draft_tokens_host,
                    int32_t *out_tokens_host, int32_t *out_num_accepted_host, void *stream) {
    int rc = check_common(B, V, dtype);
    if (rc != SPEC_OK) return rc;
    if (B == 0) return SPEC_OK;
    if (!target_logits_host || !draft_logits_host || !u_draft_host || !u_accept_host || !u_resample_host ||
        !temperature_host || !k_offsets_host || !out_draft_tokens_host || !out_tokens_host ||
        !out_num_accepted_host)
        return SPEC_ERR_INVALID_ARG;
    if (k_offsets_host[0] != 0) return SPEC_ERR_INVALID_ARG;
    for (int b = 0; b < B; ++b) {
        const int k = k_offsets_host[b + 1] - k_offsets_host[b];
        if (k < 0 || k > SPEC_MAX_K) return SPEC_ERR_INVALID_ARG;
    }
    const size_t es = dtype == SPEC_F32 ? 4 : 2;
    const size_t R_d = static_cast<size_t>(k_offsets_host[B]);
    const size_t R_t = R_d + B;
    // staging layout
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    const size_t o_t = take(R_t * V * es), o_d = take(std::max<size_t>(R_d, 1) * V * es);
    const size_t o_ud = take(R_d * 4 + 4), o_ua = take(R_d * 4 + 4), o_ur = take(R_t * 4);
    const size_t o_T = take(B * 4), o_k = take((B + 1) * 4), o_xd = take(R_d * 4 + 4);
    const size_t o_ot = take(R_t * 4), o_on = take(B * 4);
    int dev;
    DeviceState *st = device_state(&dev);
    if (!st) return SPEC_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (st->stage_bytes < off) {
            if (st->stage) {
                cudaDeviceSynchronize();
                cudaFree(st->stage);
            }
            st->stage = nullptr;
            st->stage_bytes = 0;
            if (!cuda_ok(cudaMalloc(&st->stage, off), "cudaMalloc(staging)")) return SPEC_ERR_CUDA;
            st->stage_bytes = off;
        }
    }
    unsigned char *d = static_cast<unsigned char *>(st->stage);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaMemcpyAsync(d + o_t, target_logits_host, R_t * V * es, cudaMemcpyHostToDevice, s);
    if (R_d) cudaMemcpyAsync(d + o_d, draft_logits_host, R_d * V * es, cudaMemcpyHostToDevice, s);
    if (R_d) cudaMemcpyAsync(d + o_ud, u_draft_host, R_d * 4, cudaMemcpyHostToDevice, s);
    if (R_d) cudaMemcpyAsync(d + o_ua, u_accept_host, R_d * 4, cudaMemcpyHostToDevice, s);
    cudaMemcpyAsync(d + o_ur, u_resample_host, R_t * 4, cudaMemcpyHostToDevice, s);
    cudaMemcpyAsync(d + o_T, temperature_host, B * 4, cudaMemcpyHostToDevice, s);
    cudaMemcpyAsync(d + o_k, k_offsets_host, (B + 1) * 4, cudaMemcpyHostToDevice, s);
    rc = round_call(d + o_t, d + o_d, reinterpret_cast<const float *>(d + o_ud),
                    reinterpret_cast<const float *>(d + o_ua), reinterpret_cast<const float *>(d + o_ur),
                    reinterpret_cast<const float *>(d + o_T), B, reinterpret_cast<const int32_t *>(d + o_k), V, dtype,
                    reinterpret_cast<int32_t *>(d + o_xd), reinterpret_cast<int32_t *>(d + o_ot),
                    reinterpret_cast<int32_t *>(d + o_on), stream);
    if (rc != SPEC_OK) return rc;
    if (R_d) cudaMemcpyAsync(out_draft_tokens_host, d + o_xd, R_d * 4, cudaMemcpyDeviceToHost, s);
    cudaMemcpyAsync(out_tokens_host, d + o_ot, R_t * 4, cudaMemcpyDeviceToHost, s);
    cudaMemcpyAsync(out_num_accepted_host, d + o_on, B * 4, cudaMemcpyDeviceToHost, s);
    if (!cuda_ok(cudaStreamSynchronize(s), "cudaStreamSynchronize")) return SPEC_ERR_CUDA;
    return cuda_ok(cudaGetLastError(), "spec_round_host copies") ? SPEC_OK : SPEC_ERR_CUDA;
}

int spec_workspace_status(const void *workspace, int *status_out, int clear) {
    if (!status_out) return SPEC_ERR_INVALID_ARG;
    const unsigned char *base = static_cast<const unsigned char *>(workspace);
    int dev;
    DeviceState *st = device_state(&dev);
    if (!st) return SPEC_ERR_CUDA;
    if (!base) {
        if (!st->ws) {
            *status_out = SPEC_OK;
            return SPEC_OK;
        }
        base = static_cast<const unsigned char *>(st->ws);
    }
    int v = 0;
    if (!cuda_ok(cudaMemcpy(&v, base + kStatusOffset, sizeof v, cudaMemcpyDeviceToHost), "cudaMemcpy(status)"))
        return SPEC_ERR_CUDA;
    *status_out = v;
    if (clear && !cuda_ok(cudaMemset(const_cast<unsigned char *>(base) + kStatusOffset, 0, sizeof v),
                          "cudaMemset(status)"))
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

const char *spec_status_string(int status) {
    switch (status) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG";
    case SPEC_ERR_ALIGNMENT: return "SPEC_ERR_ALIGNMENT";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
    case SPEC_ERR_TIMEOUT: return "SPEC_ERR_TIMEOUT";
    case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE";
    default: return "SPEC_ERR_UNKNOWN";
    }
}

int spec_abi_version(void) { return SPEC_VERIFY_ABI_VERSION; }

const char *spec_last_error(void) { return g_last_error; }

}  // extern "C"

// ------------------------------------------------------------------
// Allocation-free verify.
//
// Some callers cannot allocate device memory at the moment they need a
// verify step: code running inside a CUDA stream capture (a cudaMalloc
// there breaks the capture), serving loops that forbid allocation on the
// hot path so that latency stays predictable, and memory pools or embedded
// runtimes that own all device memory themselves.  spec_verify_noalloc
// serves them: it runs the same kernels as spec_verify, but its scratch
// memory is a fixed array compiled into this library, so the call itself
// never allocates.
//
// The array below is a file-scope device variable.  Every GPU on which the
// library is loaded holds kNoAllocScratchBytes of it until the process
// exits.  Its name in host code only stands in for the device object, so
// the host looks its device address up with cudaGetSymbolAddress, once per
// device, with that device current.
constexpr size_t kNoAllocScratchBytes = SPEC_NOALLOC_SCRATCH_BYTES;  // 48 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
void *g_noalloc_addr[kMaxDevices] = {};

extern "C" {

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
    Geometry g;
    make_geometry(V, dtype, &g);
    const WsLayout l = ws_layout(B, g);
    if (l.total > kNoAllocScratchBytes) {
        snprintf(g_last_error, sizeof g_last_error,
                 "spec_verify_noalloc: B=%d, V=%d needs %zu bytes of scratch, the fixed array holds %zu", B, V,
                 l.total, kNoAllocScratchBytes);
        return SPEC_ERR_WORKSPACE;
    }
    int dev;
    DeviceState *st = device_state(&dev);
    if (!st) return SPEC_ERR_CUDA;
    void *ws;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_noalloc_addr[dev]) {
            // first call on this device: resolve the array's device address
            void *p = nullptr;
            if (!cuda_ok(cudaGetSymbolAddress(&p, g_noalloc_scratch), "cudaGetSymbolAddress(g_noalloc_scratch)"))
                return SPEC_ERR_CUDA;
            g_noalloc_addr[dev] = p;
        }
        ws = g_noalloc_addr[dev];
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents: the status word must
    // start at zero; the unit-ticket words, which stats_kernel leaves at
    // zero, are cleared by the same memset at no extra cost; the
    // per-sequence counters are reset by stats_kernel
    if (!cuda_ok(cudaMemsetAsync(static_cast<unsigned char *>(ws) + kStatusOffset, 0,
                                 (kCounterWords - kStatus) * sizeof(int), s),
                 "cudaMemsetAsync(noalloc status and tickets)"))
        return SPEC_ERR_CUDA;
    const spec_verify_aux_t a{};
    if (dtype == SPEC_F32)
        return launch_verify<SPEC_F32>(target_logits, draft_logits, nullptr, draft_tokens, u_accept, u_resample,
                                       temperature, B, k_offsets, g, out_tokens, out_num_accepted, a, ws, l, *st, s);
    return launch_verify<SPEC_BF16>(target_logits, draft_logits, nullptr, draft_tokens, u_accept, u_resample,
                                    temperature, B, k_offsets, g, out_tokens, out_num_accepted, a, ws, l, *st, s);
}

}  // extern "C"
