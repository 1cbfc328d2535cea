// verify_common.cuh -- device code shared by the verify translation units
// (spec_verify.cu: chain verify and draft sampling; tree_verify.cu: tree
// verify and tree drafting): the geometry of a logit row, the streaming
// statistics kernel (stats_kernel, every mode), and the warp-level tools of
// the epilogues (row combine, inverse-CDF locate and scan, one draw).
#pragma once

#include <climits>

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
// Status word, then the streaming kernels' unit tickets and count of CTAs
// done, the number of listed residual pairs (see PairRec), a second ticket
// pair for the target pass of spec_round, which streams while the draft
// pass's kernels may still hold the first, and the number of sequences the
// deferred epilogue has decided.
enum CounterWord : int {
    kStatus = 1, kTicket = 2, kDone = 3, kPairs = 4, kTicketB = 5, kDoneB = 6, kDecided = 7, kCounterWords = 8
};

// A rejected position whose residual is streamed by resid_stream_kernel:
// written by the deferred epilogue's decisions, one per rejected sequence,
// in the order the decisions land; `ready` is stored last (release), and
// stats_kernel zeroes it for the next call.
struct __align__(16) PairRec {
    int b;           // sequence
    int trow, drow;  // target and draft row at the rejected position
    float c;         // temperature scale log2(e) / T_b
    float lth, ltl;  // the target row's log2-sum-exp, fp32 hi + lo
    float ldh, ldl;  // the draft row's
    float u;         // u_resample at the rejected position
    int ready;       // 1 once the fields above are written
    int t0, k;       // the sequence's first target row and its draft length
};

// Wait (bounded, 2 s) for entry p of the deferred epilogue's pair list:
// 1 once it is listed and its ready flag is set (acquire: its fields are
// then visible), 0 once every one of the B sequences is decided and p lies
// past the list (every listing precedes its sequence's count), -1 on a
// time-out (the caller records it).
__device__ __forceinline__ int wait_pair(const int *counters, const PairRec *pairs, int p, int B) {
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        int np = ld_acquire_gpu(counters + kPairs);
        if (p < np && ld_acquire_gpu(&pairs[p].ready)) return 1;
        if (p >= np && ld_acquire_gpu(counters + kDecided) >= B) {
            np = ld_acquire_gpu(counters + kPairs);
            if (p >= np) return 0;
            continue;
        }
        if (global_timer_ns() - t0 > kWaitLimitNs) return -1;
        __nanosleep(64);
    }
}

struct WsPtrs {
    float2 *part;        // [rows_cap * n_sub] sub-chunk partials
    int *counters;       // CounterWord: status, unit tickets and CTAs done, pairs
    int *seqcnt;         // [B] resolve_kernel arrivals per sequence
    float *resid_part;   // [B * n_sub] residual mass per sub-chunk
    PairRec *pairs;      // [B] listed residual pairs (deferred mode)
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
static __device__ int block_excl_scan(int v, int *s_warp, int *total) {
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
#define SPEC_STATS_BATCH 2
#endif
#ifndef SPEC_STATS_TAIL_BATCH
#define SPEC_STATS_TAIL_BATCH 1
#endif
#ifndef SPEC_STATS_TAIL_PER_CTA
#define SPEC_STATS_TAIL_PER_CTA 1
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
    kModeVerify = 0,     // target rows, plus the draft rows of sampled sequences
    kModeDraft = 1,      // draft rows only (spec_draft_sample)
    kModeTarget = 2,     // target rows only (verify with the draft rows' lse given)
    kModeTree = 3,       // tree verify: every node's target row, plus the draft rows of
                         // the internal nodes of sampled sequences
    kModeTreeDraft = 4,  // tree drafting: the draft rows of internal nodes
    kModeShard = 5       // vocab-sharded verify: as kModeVerify, over one shard's columns
};

// Nodes per sequence of a tree call, and the per-sequence tables the tree
// setup kernel writes for stats_kernel: tree_nint[b] = internal nodes of b
// (-1: invalid parent array), tree_int[b * kMaxTreeNodes + j] = the j-th
// internal node of b (global index, ascending).
constexpr int kMaxTreeNodes = SPEC_MAX_TREE_NODES;

// Persistent streaming kernel.  Unit u = (row r of the virtual row list,
// chunk ch).  Virtual row list, by sequence b in order:
//   verify mode: target rows of b (k_b + 1), then draft rows of b (k_b) if
//                b is sampled; nothing for a bad temperature;
//   draft mode:  draft rows of b (k_b); nothing for a bad temperature;
//   target mode: target rows of b (k_b + 1); nothing for a bad temperature;
//   tree mode:   (k_offsets holds node_offsets) the n_b target rows of b's
//                nodes, then the draft rows of its internal nodes if b is
//                sampled; nothing for a bad temperature or parent array;
//   tree-draft:  the draft rows of b's internal nodes.
// Partials go to slot row r for target row r and R + r for draft row r, with
// R = R_t in the chain modes (draft rows included, so that a target pass may
// stream while the draft pass's epilogue still reads its partials) and the
// node count N in tree mode; tree-draft mode uses slot r for draft row r.
// wait_first: 1 = the kernel opens its call and waits for the stream's
// previous kernel before it reads anything; 0 = it reads the call's inputs,
// then waits before it writes the workspace; 2 = it does not wait until its
// end (its predecessor in the same call writes nothing it reads or writes,
// and its completion still implies the predecessor's).
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
    float2 *__restrict__ part, int *__restrict__ counters, int *__restrict__ seqcnt,
    const int *__restrict__ tree_nint, const int *__restrict__ tree_int, int tree_nodes, int wait_first,
    PairRec *__restrict__ pairs, int evict_first_rows) {
    using E = Elem<DT>;
    constexpr bool DRAFT = MODE == kModeDraft;
    constexpr bool TREE = MODE == kModeTree || MODE == kModeTreeDraft;
    // unit tickets and CTAs done (the target pass has its own pair)
    int *tickets = counters + (MODE == kModeTarget ? kTicketB : kTicket);
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
    // wait_first: the kernel opens its call and was launched early behind
    // whatever kernel precedes it on the stream, which may still be writing
    // the inputs: wait for it before reading them
    if (wait_first == 1) grid_dependency_wait();
    for (int i = tid; i <= B; i += kThreads) {
        s_kofs[i] = k_offsets[i];
        if (i < B) s_c[i] = temp_scale(temperature[i]);
    }
    __syncthreads();

    // k_offsets validation and row counts (contiguous segment per thread)
    const int seg = (B + kThreads - 1) / kThreads;
    const int b0 = min(B, tid * seg), b1 = min(B, b0 + seg);
    // (tree modes: the node count must be the one the workspace was sized for)
    int bad = (tid == 0 && (s_kofs[0] != 0 || (TREE && s_kofs[B] != tree_nodes))) ? 1 : 0;
    int rows = 0;
    // rows of sequence b: none for a bad temperature
    auto seq_rows = [&](int b) -> int {
        const int k = s_kofs[b + 1] - s_kofs[b];
        const float c = s_c[b];
        if (c != c) return 0;
        if (MODE == kModeDraft) return k;
        if (MODE == kModeTarget) return k + 1;
        if (TREE) {
            const int nint = tree_nint[b];
            if (nint < 0) return 0;
            if (MODE == kModeTreeDraft) return nint;
            return c == 0.0f ? k : k + nint;
        }
        return c == 0.0f ? k + 1 : 2 * k + 1;
    };
    for (int b = b0; b < b1; ++b) {
        const int k = s_kofs[b + 1] - s_kofs[b];
        if (TREE ? (k < 1 || k > kMaxTreeNodes) : (k < 0 || k > kMaxK)) bad = 1;
        if (!bad) rows += seq_rows(b);
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
    if (wait_first != 2) grid_dependency_wait();
    const bool any_bad = __syncthreads_or(bad);
    if (MODE == kModeVerify || MODE == kModeTarget) {
        for (int i = blockIdx.x * kThreads + tid; i < B; i += gridDim.x * kThreads) {
            seqcnt[i] = 0;
            if (pairs) pairs[i].ready = 0;
        }
        // the epilogue of this call lists and decides its sequences from zero
        if (blockIdx.x == 0 && tid == 0) {
            counters[kPairs] = 0;
            counters[kDecided] = 0;
        }
    }
    // the next kernel may be scheduled as soon as SMs free up; it waits for
    // this grid's completion before it reads anything written here
    grid_launch_dependents();
    if (any_bad) {
        if (wait_first == 2) grid_dependency_wait();
        return;
    }

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
            // evict_first_rows: the rows pass through L2 as its first
            // victims, so that the stream does not push out what the
            // epilogue reads back from L2 (the partials of every row, the
            // pair list, the offsets)
            const bool hints = evict_first_rows != 0;
            const uint64_t evict_first = hints ? l2_policy_evict_first() : 0ull;
            int t = atomicAdd(tickets, 1);
            while (ok) {
                int64_t u0;
                int cnt;
                unit_batch(t, n_big, &u0, &cnt);
                if (u0 >= total_units) break;
                const int tn = atomicAdd(tickets, 1);  // next batch, in flight meanwhile
                cnt = static_cast<int>(min(static_cast<int64_t>(cnt), total_units - u0));
                int r = static_cast<int>(u0 / g.n_chunks);
                int ch = static_cast<int>(u0 - static_cast<int64_t>(r) * g.n_chunks);
                if (s_rowpre[b + 1] <= r) {
                    // a new batch can lie many sequences ahead (short rows):
                    // the last b with s_rowpre[b] <= r (s_rowpre is
                    // non-decreasing and s_rowpre[b] <= r already), by
                    // binary lifting; within the batch b moves on one
                    // sequence at a time
                    for (int step = 1 << (31 - __clz(B)); step > 0; step >>= 1)
                        if (b + step < B && s_rowpre[b + step] <= r) b += step;
                }
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
                    if (MODE == kModeTreeDraft) {
                        row = tree_int[b * kMaxTreeNodes + l];
                        base_ptr = draft;
                        slot_row = row;
                    } else if (MODE == kModeTree) {
                        if (l < k) {
                            row = s_kofs[b] + l;
                            base_ptr = target;
                            slot_row = row;
                        } else {
                            row = tree_int[b * kMaxTreeNodes + (l - k)];
                            base_ptr = draft;
                            slot_row = s_kofs[B] + row;
                        }
                    } else if (DRAFT) {
                        row = s_kofs[b] + l;
                        base_ptr = draft;
                        slot_row = R_t + row;
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
                    if (hints)
                        bulk_g2s_hint(ring + static_cast<size_t>(islot) * kSlotBytes, src, d.nbytes, &full[islot],
                                      evict_first);
                    else
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
    if (wait_first == 2) grid_dependency_wait();
    __syncthreads();
    if (tid == 0 && atomic_add_acq_rel_gpu(tickets + 1, 1) == static_cast<int>(gridDim.x) - 1) {
        tickets[0] = 0;
        tickets[1] = 0;
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

#ifndef SPEC_ARG_BATCH
#define SPEC_ARG_BATCH 1
#endif

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
static __device__ bool combine_soft(const float2 (&cache)[kPartCache], const float2 *p, int n, float *M_out,
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

static __device__ bool warp_combine_soft(const float2 *p, int n, float *M_out, float *S_out) {
    float2 cache[kPartCache];
    load_parts(p, n, cache);
    return combine_soft(cache, p, n, M_out, S_out);
}

// Arg-max over the n sub-chunk partials of one row; -1 if a NaN was seen.
// The first 32 * kPartCache partials arrive in one round trip (load_parts);
// the merge is order-free (largest value, lowest index, NaN wins).
// The same from the row's first 32 * kPartCache partials already loaded
// (load_parts), the rest read here.
static __device__ int warp_combine_arg_cached(const float2 (&c)[kPartCache], const float2 *p, int n) {
    const int lane = lane_id();
    ArgPart a{-INFINITY, INT_MAX};
#pragma unroll
    for (int j = 0; j < kPartCache; ++j)
        if (lane + 32 * j < n) a = arg_merge(a, ArgPart{c[j].x, __float_as_int(c[j].y)});
    for (int i = lane + 32 * kPartCache; i < n; i += 32) {
        const float2 v = __ldcg(p + i);
        a = arg_merge(a, ArgPart{v.x, __float_as_int(v.y)});
    }
    a = warp_arg(a);
    return a.i == INT_MAX ? -1 : a.i;
}

static __device__ int warp_combine_arg(const float2 *p, int n) {
#if SPEC_ARG_BATCH
    float2 c[kPartCache];
    load_parts(p, n, c);
    return warp_combine_arg_cached(c, p, n);
#else
    const int lane = lane_id();
    ArgPart a{-INFINITY, INT_MAX};
    for (int i = lane; i < n; i += 32) {
        const float2 v = __ldcg(p + i);
        a = arg_merge(a, ArgPart{v.x, __float_as_int(v.y)});
    }
    a = warp_arg(a);
    return a.i == INT_MAX ? -1 : a.i;
#endif
}

// warp_locate: warp-level locate over n non-negative weights (sub-chunk
// masses): total Z, target = u * Z, and the first i whose cumulative mass
// exceeds the target, with the mass before it.  If rounding leaves no such
// i, the last i with positive weight.  Returns -1 if every weight is 0.
// Weight i is cache[j] of lane i % 32 for i = lane + 32 j < 32 * kPartCache,
// wfar(i) beyond.  It is warp_total (Z as an unevaluated pair, the same bits
// on every call with the same weights) followed by warp_locate_at (the scan
// against a given target).
template <class WF>
__device__ F2 warp_total(int n, const float (&cache)[kPartCache], WF wfar) {
    const int lane = lane_id();
    Acc2 acc;
#pragma unroll
    for (int j = 0; j < kPartCache; ++j) acc.add(cache[j]);
    for (int j = kPartCache; 32 * j < n; ++j) acc.add((lane + 32 * j < n) ? wfar(lane + 32 * j) : 0.0f);
    return f2_two_sum(warp_sum_f(acc.hi), warp_sum_f(acc.lo));
}

template <class WF>
__device__ int warp_locate_at(int n, const float (&cache)[kPartCache], WF wfar, F2 target, F2 *before) {
    const int lane = lane_id();
    constexpr int kCache = kPartCache;
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

template <class WF>
__device__ int warp_locate(int n, const float (&cache)[kPartCache], WF wfar, float u, F2 *before, F2 *total,
                           F2 *target_out) {
    const F2 tot = warp_total(n, cache, wfar);
    const F2 target = f2_scale(u, tot);
    *total = tot;
    *target_out = target;
    return warp_locate_at(n, cache, wfar, target, before);
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

// Block-level inverse CDF inside elements [a, b) (at most one 2 KB
// sub-chunk) of one or two rows, by a block of kDrawThreads or more threads
// (up to 1024): thread t owns the 8 bytes at element a + t * PE (4 bf16 or
// 2 fp32 elements; a sub-chunk is 1024 bf16 or 512 fp32 elements, so one
// group for each of the first 256 threads), so each thread holds a
// contiguous run and the cumulative mass is one block scan.  Weights are W(x_row1, x_row2).  Every thread returns the first
// element whose cumulative mass, starting at `before`, exceeds `target`;
// else the last element with positive weight (rounding fallback); else -1.
// The same rule as warp_scan_elems, with the work spread over 8 warps so
// that the draw is a few dependent steps long instead of 64.
constexpr int kDrawThreads = 256;
struct DrawSmem {
    float wsum[32];  // per-warp sums of the block scan
    int found, lastpos;
    int sc;             // located sub-chunk (block_draw_row)
    F2 before, target;  // its cumulative mass before it, and u * Z
};

template <int DT, class WF>
__device__ int block_scan_elems(const void *row1, const void *row2, int a, int b, WF W, F2 before, F2 target,
                                DrawSmem &ds) {
    using E = Elem<DT>;
    constexpr int PE = 8 / E::kBytes;
    const int t = threadIdx.x, lane = lane_id(), warp = warp_id();
    const int e0 = a + t * PE;
    float wv[PE];
    float tsum = 0.0f;
    if (t == 0) {
        ds.found = INT_MAX;
        ds.lastpos = -1;
    }
    if (e0 < b) {
        const uint2 v1 = __ldg(reinterpret_cast<const uint2 *>(static_cast<const unsigned char *>(row1) +
                                                             static_cast<int64_t>(e0) * E::kBytes));
        const uint2 v2 = (row2 != row1) ? __ldg(reinterpret_cast<const uint2 *>(static_cast<const unsigned char *>(row2) +
                                                                               static_cast<int64_t>(e0) * E::kBytes))
                                        : v1;
        float x1[PE], x2[PE];
        if constexpr (E::kBytes == 2) {
            x1[0] = __uint_as_float(v1.x << 16);
            x1[1] = __uint_as_float(v1.x & 0xffff0000u);
            x1[PE - 2] = __uint_as_float(v1.y << 16);
            x1[PE - 1] = __uint_as_float(v1.y & 0xffff0000u);
            x2[0] = __uint_as_float(v2.x << 16);
            x2[1] = __uint_as_float(v2.x & 0xffff0000u);
            x2[PE - 2] = __uint_as_float(v2.y << 16);
            x2[PE - 1] = __uint_as_float(v2.y & 0xffff0000u);
        } else {
            x1[0] = __uint_as_float(v1.x);
            x1[PE - 1] = __uint_as_float(v1.y);
            x2[0] = __uint_as_float(v2.x);
            x2[PE - 1] = __uint_as_float(v2.y);
        }
#pragma unroll
        for (int q = 0; q < PE; ++q) {
            wv[q] = W(x1[q], x2[q]);
            tsum += wv[q];
        }
    } else {
#pragma unroll
        for (int q = 0; q < PE; ++q) wv[q] = 0.0f;
    }
    // block exclusive scan of the per-thread sums
    const float incl = warp_incl_scan_f(tsum);
    if (lane == 31) ds.wsum[warp] = incl;
    __syncthreads();
    float wpre = 0.0f;
    for (int i = 0; i < warp; ++i) wpre += ds.wsum[i];
    const F2 start = f2_add(before, wpre + (incl - tsum));
    const float rem = f2_round_down(f2_sub(target, start));  // acc > rem  <=>  start + acc > target
    float acc = 0.0f;
    int found = -1, lastpos = -1;
#pragma unroll
    for (int q = 0; q < PE; ++q) {
        acc += wv[q];
        if (wv[q] > 0.0f) lastpos = q;
        if (found < 0 && wv[q] > 0.0f && acc > rem) found = q;
    }
    // the cumulative mass only grows, so the earliest crossing is the answer
    if (found >= 0) atomicMin(&ds.found, e0 + found);
    if (lastpos >= 0) atomicMax(&ds.lastpos, e0 + lastpos);
    __syncthreads();
    const int r = ds.found != INT_MAX ? ds.found : ds.lastpos;
    __syncthreads();  // ds may be reused right after
    return r;
}

// One draw from a soft row by a whole block: warp 0 locates the sub-chunk
// from the row's partials (as warp_draw_row), then the block scans it.
// Every thread returns the token.
template <int DT>
__device__ int block_draw_row(const void *logits, int64_t row, const float2 *part, const Geometry &g, float c,
                              float M, float u, DrawSmem &ds) {
    if (warp_id() == 0) {
        float2 pc[kPartCache];
        load_parts(part, g.n_sub, pc);
        float w[kPartCache];
#pragma unroll
        for (int j = 0; j < kPartCache; ++j) w[j] = pc[j].x > -INFINITY ? pc[j].y * ex2(pc[j].x - M) : 0.0f;
        auto wfar = [&](int i) -> float {
            const float2 v = __ldcg(part + i);
            return v.x > -INFINITY ? v.y * ex2(v.x - M) : 0.0f;
        };
        F2 before, total, target;
        const int sc = warp_locate(g.n_sub, w, wfar, u, &before, &total, &target);
        if (lane_id() == 0) {
            ds.sc = sc;
            ds.before = before;
            ds.target = target;
        }
    }
    __syncthreads();
    const int sc = ds.sc;
    if (sc < 0) return -1;
    int a, b;
    sub_range(g, sc, &a, &b);
    const void *rp = static_cast<const unsigned char *>(logits) + row * g.V * static_cast<int64_t>(Elem<DT>::kBytes);
    auto W = [&](float x, float) -> float { return prob_weight(x, c, M); };
    return block_scan_elems<DT>(rp, rp, a, b, W, ds.before, ds.target, ds);
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

}  // namespace specv
