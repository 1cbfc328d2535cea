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
//   1. stats_kernel   persistent; streams every needed logit row through a
//                     shared-memory ring filled by 1-D bulk copies (TMA
//                     engine) and reduces each 16 KB chunk to an online
//                     softmax partial (max m, sum 2^(x c - m)) or, for greedy
//                     rows, an arg-max partial.  Each row is read from HBM
//                     once.
//   2. decide_kernel  one warp per sequence: combines the chunk partials of
//                     its rows in fp64, forms alpha_i, finds the first
//                     rejection with a warp ballot, writes the accepted
//                     prefix, and queues the residual or bonus draw.
//   3. resid_kernel   for every rejected sequence, sum of max(0, p - q) over
//                     each half-chunk of the two rows at the rejected position.
//   4. select_kernel  one block per sequence: locates the half-chunk (residual)
//                     or chunk (bonus) where the cumulative mass crosses u * Z,
//                     re-reads only that piece and finds the token with a
//                     block-wide prefix scan.
// spec_draft_sample runs stats_kernel over the draft rows, then
// draft_select_kernel (arg-max, or the same locate + scan per row).

#include <algorithm>
#include <climits>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "device_utils.cuh"

namespace specv {

constexpr int kSlotBytes = 16384;        // one chunk of one row per ring slot
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxSlots = 6;
constexpr int kSelThreads = 256;

enum UnitKind : int { kEnd = 0, kSoft = 1, kArg = 2 };
enum JobKind : int { kJobNone = 0, kJobResid = 1, kJobBonus = 2 };

struct Geometry {
    int V;
    int chunk_elems;  // elements per chunk (multiple of 2 vectors)
    int n_chunks;     // chunks per row
    int half_elems;   // chunk_elems / 2
    int n_half;       // half-chunks per row
};

struct UnitDesc {
    uint32_t nbytes;
    int kind;
    float c;
    int elem0;
    int64_t out_idx;
};

// Decision left for the select kernel, one per sequence.
struct SeqJob {
    int kind;
    int list_idx;  // residual list position
    int64_t trow;  // target row = output slot of the drawn token
    float c, M, u, pad;
};

// Residual job, one per rejected sequence (list order).
struct RJob {
    int64_t trow, drow;
    float c, lth, ltl, ldh, ldl, pad;
};

struct WsPtrs {
    float2 *part;        // [rows_cap * n_chunks] chunk partials
    SeqJob *jobs;        // [B]
    RJob *rjobs;         // [B]
    int *counters;       // [0] residual count, [1] status, [2] bad k_offsets
    float *resid_part;   // [B * n_half]
};

// ------------------------------------------------------------------ helpers
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

__device__ double block_excl_scan_d(double v, double *s_warp, double *total) {
    const int lane = lane_id(), w = warp_id(), nw = blockDim.x >> 5;
    double incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        double n = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += n;
    }
    if (lane == 31) s_warp[w] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        double acc = 0.0;
        for (int i = 0; i < nw; ++i) {
            double t = s_warp[i];
            s_warp[i] = acc;
            acc += t;
        }
        s_warp[nw] = acc;
    }
    __syncthreads();
    const double r = incl - v + s_warp[w];
    *total = s_warp[nw];
    __syncthreads();
    return r;
}

__device__ int block_min_int(int v, int *s_warp) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, off));
    if (lane_id() == 0) s_warp[warp_id()] = v;
    __syncthreads();
    int r = s_warp[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) r = min(r, s_warp[i]);
    __syncthreads();
    return r;
}

__device__ int block_max_int(int v, int *s_warp) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
    if (lane_id() == 0) s_warp[warp_id()] = v;
    __syncthreads();
    int r = s_warp[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) r = max(r, s_warp[i]);
    __syncthreads();
    return r;
}

__device__ double block_sum_d(double v, double *s_warp) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane_id() == 0) s_warp[warp_id()] = v;
    __syncthreads();
    double r = 0.0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r += s_warp[i];
    __syncthreads();
    return r;
}

// Row combine of the chunk partials (fp64).  Returns false if the row has
// no valid distribution (NaN / +inf present, or entirely -inf).
struct RowSoft {
    float M;   // max of the chunk maxima (log2-scaled units, exact fp32)
    double S;  // sum 2^(x c - M)
};

__device__ bool combine_soft(const float2 *p, int n, RowSoft *out) {
    float M = -INFINITY;
    bool nan = false;
    for (int i = 0; i < n; ++i) {
        const float2 v = __ldcg(p + i);
        nan |= (v.y != v.y);
        M = fmaxf(M, v.x);
    }
    if (nan || !(M > -INFINITY) || !(M < INFINITY)) return false;
    double S = 0.0;
    for (int i = 0; i < n; ++i) {
        const float2 v = __ldcg(p + i);
        if (v.x > -INFINITY) S += static_cast<double>(v.y) * exp2(static_cast<double>(v.x) - M);
    }
    if (!(S > 0.0) || !(S < INFINITY)) return false;
    out->M = M;
    out->S = S;
    return true;
}

// Arg-max over the chunk partials; -1 if a NaN was seen.
__device__ int combine_arg(const float2 *p, int n) {
    ArgPart a{-INFINITY, INT_MAX};
    for (int i = 0; i < n; ++i) {
        const float2 v = __ldcg(p + i);
        a = arg_merge(a, ArgPart{v.x, __float_as_int(v.y)});
    }
    return a.i == INT_MAX ? -1 : a.i;
}

// ================================================================== kernel 1
// Persistent streaming kernel.  Unit u = (row r of the virtual row list,
// chunk ch).  Virtual row list, by sequence b in order:
//   verify mode: target rows of b (k_b + 1), then draft rows of b (k_b) if
//                b is sampled; nothing for a bad temperature;
//   draft mode:  draft rows of b (k_b); nothing for a bad temperature.
// CTA g takes units g, g + G, g + 2G, ...  Warp 8 (one lane) is the
// producer: it issues the bulk copy of each unit into a ring slot and, when
// the slot comes back, folds the 8 consumer-warp partials into the chunk
// partial in global memory.  Warps 0..7 consume: 16-byte vector reads from
// shared memory, NaN-propagating max, then sum of 2^(x c - m).
template <int DT, bool DRAFT>
__global__ void __launch_bounds__(kThreads) stats_kernel(
    const void *__restrict__ target, const void *__restrict__ draft,
    const float *__restrict__ temperature, const int *__restrict__ k_offsets, int B, Geometry g,
    int ns, float2 *__restrict__ part, int *__restrict__ counters) {
    using E = Elem<DT>;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)ns * kSlotBytes);
    uint64_t *empty = full + ns;
    UnitDesc *desc = reinterpret_cast<UnitDesc *>(empty + ns);
    float2 *red = reinterpret_cast<float2 *>(desc + ns);
    int *s_kofs = reinterpret_cast<int *>(red + ns * kConsumerWarps);
    int *s_rowpre = s_kofs + (B + 1);
    float *s_c = reinterpret_cast<float *>(s_rowpre + (B + 1));
    int *s_tmp = reinterpret_cast<int *>(s_c + B);  // [kThreads/32 + 1]
    __shared__ int s_abort;

    const int tid = threadIdx.x;
    for (int i = tid; i <= B; i += kThreads) {
        s_kofs[i] = k_offsets[i];
        if (i < B) s_c[i] = temp_scale(temperature[i]);
    }
    if (tid == 0) s_abort = 0;
    if (!DRAFT && blockIdx.x == 0 && tid == 0) counters[0] = 0;  // residual list
    __syncthreads();

    // k_offsets validation and row counts (contiguous segment per thread)
    const int seg = (B + kThreads - 1) / kThreads;
    const int b0 = min(B, tid * seg), b1 = min(B, b0 + seg);
    int bad = (tid == 0 && s_kofs[0] != 0) ? 1 : 0;
    int rows = 0;
    for (int b = b0; b < b1; ++b) {
        const int k = s_kofs[b + 1] - s_kofs[b];
        if (k < 0 || k > kMaxK) bad = 1;
        const float c = s_c[b];
        if (c != c) continue;
        rows += DRAFT ? k : (c == 0.0f ? k + 1 : 2 * k + 1);
    }
    int total_rows;
    int base = block_excl_scan(rows, s_tmp, &total_rows);
    for (int b = b0; b < b1; ++b) {
        s_rowpre[b] = base;
        const int k = s_kofs[b + 1] - s_kofs[b];
        const float c = s_c[b];
        if (c == c) base += DRAFT ? k : (c == 0.0f ? k + 1 : 2 * k + 1);
    }
    if (tid == 0) s_rowpre[B] = total_rows;
    if (__syncthreads_or(bad)) {
        if (!DRAFT && blockIdx.x == 0 && tid == 0) counters[2] = 1;
        return;
    }
    if (!DRAFT && blockIdx.x == 0 && tid == 0) counters[2] = 0;

    if (tid == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    const int64_t total_units = static_cast<int64_t>(total_rows) * g.n_chunks;
    const int64_t R_t = static_cast<int64_t>(s_kofs[B]) + B;
    const int lane = lane_id();

    if (warp_id() == kConsumerWarps) {
        // ------------------------------------------------------ producer
        if (lane != 0) return;
        int issued = 0;
        bool ok = true;
        auto retire = [&](int i) {
            const int slot = i % ns;
            if (!mbar_wait_bounded(&empty[slot], (i / ns) & 1)) {
                ok = false;
                return;
            }
            const UnitDesc &d = desc[slot];
            const float2 *r = red + slot * kConsumerWarps;
            float2 out;
            if (d.kind == kSoft) {
                SoftPart a{r[0].x, r[0].y};
#pragma unroll
                for (int w = 1; w < kConsumerWarps; ++w) a = soft_merge(a, SoftPart{r[w].x, r[w].y});
                out = make_float2(a.m, a.s);
            } else {
                ArgPart a{r[0].x, __float_as_int(r[0].y)};
#pragma unroll
                for (int w = 1; w < kConsumerWarps; ++w)
                    a = arg_merge(a, ArgPart{r[w].x, __float_as_int(r[w].y)});
                out = make_float2(a.v, __int_as_float(a.i));
            }
            part[d.out_idx] = out;
        };
        int b = 0;
        for (int64_t u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
            if (issued >= ns) retire(issued - ns);
            if (!ok || s_abort) break;
            const int64_t r = u / g.n_chunks;
            const int ch = static_cast<int>(u - r * g.n_chunks);
            while (s_rowpre[b + 1] <= r) ++b;
            const int l = static_cast<int>(r - s_rowpre[b]);
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
            d.out_idx = slot_row * g.n_chunks + ch;
            const int slot = issued % ns;
            desc[slot] = d;
            const unsigned char *src = static_cast<const unsigned char *>(base_ptr) +
                                       (row * g.V + e0) * static_cast<int64_t>(E::kBytes);
            mbar_arrive_expect_tx(&full[slot], d.nbytes);
            bulk_g2s(ring + static_cast<size_t>(slot) * kSlotBytes, src, d.nbytes, &full[slot]);
            ++issued;
        }
        if (ok && issued >= ns) retire(issued - ns);
        {
            // end marker (also on abort, so that consumers leave)
            const int slot = issued % ns;
            desc[slot].kind = kEnd;
            mbar_arrive(&full[slot]);
        }
        if (ok)
            for (int i = max(0, issued - ns + 1); i < issued && ok; ++i) retire(i);
        if (!ok) {
            set_status(counters + 1, SPEC_ERR_TIMEOUT);
            s_abort = 1;
            // let issued copies land before the CTA exits (bounded)
            for (int i = max(0, issued - ns); i < issued; ++i)
                mbar_wait_bounded(&full[i % ns], (i / ns) & 1);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int t = tid;  // 0..255
    const int w = warp_id();
    for (int i = 0;; ++i) {
        const int slot = i % ns;
        if (!mbar_wait_bounded(&full[slot], (i / ns) & 1)) {
            set_status(counters + 1, SPEC_ERR_TIMEOUT);
            s_abort = 1;
            break;
        }
        const UnitDesc d = desc[slot];
        if (d.kind == kEnd) break;
        const uint4 *v4 = reinterpret_cast<const uint4 *>(ring + static_cast<size_t>(slot) * kSlotBytes);
        const int nvec = static_cast<int>(d.nbytes >> 4);
        uint4 v[4];
        bool okv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int idx = t + j * kConsumers;
            okv[j] = idx < nvec;
            if (okv[j]) v[j] = v4[idx];
        }
        float2 res;
        if (d.kind == kSoft) {
            float vmax = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (okv[j]) vmax = fmax_nan(vmax, E::vmax_nan(v[j]));
            SoftPart p;
            if (vmax != vmax) {
                p = SoftPart{-INFINITY, __int_as_float(0x7fc00000)};
            } else if (vmax == -INFINITY) {
                p = SoftPart{-INFINITY, 0.0f};
            } else {
                const float c = d.c;
                const float m = vmax * c;
                float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (!okv[j]) continue;
                    float x[E::kPerVec];
                    E::unpack(v[j], x);
#pragma unroll
                    for (int e = 0; e < E::kPerVec; e += 2) {
                        s0 += ex2(__fmaf_rn(x[e], c, -m));
                        s1 += ex2(__fmaf_rn(x[e + 1], c, -m));
                    }
                }
                p = SoftPart{m, s0 + s1};
            }
            p = warp_soft(p);
            res = make_float2(p.m, p.s);
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
                    a = ArgPart{vm, d.elem0 + (t + j * kConsumers) * E::kPerVec + e};
                }
            }
            a = warp_arg(a);
            res = make_float2(a.v, __int_as_float(a.i));
        }
        if (lane == 0) red[slot * kConsumerWarps + w] = res;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
}

// ================================================================== kernel 2
// One warp per sequence.  Lane i owns drafted position i (and lane k_b the
// bonus row when k_b < 32).
template <int DT>
__global__ void __launch_bounds__(256) decide_kernel(
    const void *__restrict__ target, const void *__restrict__ draft,
    const int32_t *__restrict__ tokens, const float *__restrict__ u_accept,
    const float *__restrict__ u_resample, const float *__restrict__ temperature,
    const int *__restrict__ k_offsets, int B, Geometry g, WsPtrs ws, int32_t *__restrict__ out_tokens,
    int32_t *__restrict__ out_num, spec_verify_aux_t aux) {
    using E = Elem<DT>;
    const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = lane_id();
    if (b >= B) return;
    SeqJob job{kJobNone, -1, 0, 0.f, 0.f, 0.f, 0.f};
    if (__ldcg(ws.counters + 2) != 0) {
        // invalid k_offsets: the whole call fails, outputs of unknown size untouched
        if (lane == 0) {
            out_num[b] = -1;
            ws.jobs[b] = job;
            if (aux.residual_mass) aux.residual_mass[b] = NAN;
            if (b == 0) set_status(ws.counters + 1, SPEC_ERR_INVALID_ARG);
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

    int x = 0;
    bool err = (c != c);
    if (lane < k) {
        x = tokens[od + lane];
        err |= (x < 0 || x >= V);
    }
    err = __any_sync(0xffffffffu, err);
    int n = -1;  // accepted count; -1 = data error
    int tok = -1;
    float alpha_out = NAN;
    double Lt = 0.0, Ld = 0.0;
    bool have_t = false, have_d = false;

    if (!err && c == 0.0f) {
        // greedy: accept while x_i == argmax p_i
        int a = 0;
        if (lane <= k) a = combine_arg(ws.part + (ot + lane) * g.n_chunks, g.n_chunks);
        int a_bonus = __shfl_sync(0xffffffffu, a, k & 31);
        if (k == kMaxK) a_bonus = combine_arg(ws.part + (ot + k) * g.n_chunks, g.n_chunks);
        const bool bad_row = (lane <= k && a < 0) || a_bonus < 0;
        if (!__any_sync(0xffffffffu, bad_row)) {
            const unsigned mism = __ballot_sync(0xffffffffu, lane < k && x != a);
            n = mism ? (__ffs(mism) - 1) : k;
            tok = (n < k) ? __shfl_sync(0xffffffffu, a, n & 31) : a_bonus;
        }
    } else if (!err) {
        // sampled: alpha_i = min(1, p_i(x_i) / q_i(x_i)) in the log domain
        bool ok = true, acc = false;
        RowSoft rt{}, rd{}, rk{};
        if (lane < k) {
            ok = combine_soft(ws.part + (ot + lane) * g.n_chunks, g.n_chunks, &rt) &&
                 combine_soft(ws.part + (R_t + od + lane) * g.n_chunks, g.n_chunks, &rd);
            if (ok) {
                have_t = have_d = true;
                Lt = static_cast<double>(rt.M) + log2(rt.S);
                Ld = static_cast<double>(rd.M) + log2(rd.S);
                const float zt = E::load1(target, (ot + lane) * V + x);
                const float zd = E::load1(draft, (od + lane) * V + x);
                double alpha;
                if (zt == -INFINITY) {
                    alpha = 0.0;
                } else if (zd == -INFINITY) {
                    alpha = 1.0;
                } else {
                    const double cd = static_cast<double>(c);
                    const double lr = (static_cast<double>(zt) * cd - Lt) - (static_cast<double>(zd) * cd - Ld);
                    alpha = lr >= 0.0 ? 1.0 : exp2(lr);
                }
                alpha_out = static_cast<float>(alpha);
                acc = static_cast<double>(u_accept[od + lane]) < alpha;
            }
        }
        bool okk = true;
        if (lane == (k & 31)) {
            okk = combine_soft(ws.part + (ot + k) * g.n_chunks, g.n_chunks, &rk);
            if (okk && k < kMaxK) {
                have_t = true;
                Lt = static_cast<double>(rk.M) + log2(rk.S);
            }
        }
        if (!__any_sync(0xffffffffu, !ok || !okk)) {
            const unsigned rej = __ballot_sync(0xffffffffu, lane < k && !acc);
            n = rej ? (__ffs(rej) - 1) : k;
            const int src = n & 31;
            // the lane holding row n of the target (bonus: lane k, or lane 0 for k = 32)
            const float Mk = __shfl_sync(0xffffffffu, rk.M, k & 31);
            const double Ltn = __shfl_sync(0xffffffffu, Lt, src);
            const double Ldn = __shfl_sync(0xffffffffu, Ld, src);
            if (lane == 0) {
                if (n < k) {
                    const int e = atomicAdd(ws.counters + 0, 1);
                    RJob r;
                    r.trow = ot + n;
                    r.drow = od + n;
                    r.c = c;
                    r.lth = static_cast<float>(Ltn);
                    r.ltl = static_cast<float>(Ltn - static_cast<double>(r.lth));
                    r.ldh = static_cast<float>(Ldn);
                    r.ldl = static_cast<float>(Ldn - static_cast<double>(r.ldh));
                    r.pad = 0.f;
                    ws.rjobs[e] = r;
                    job.kind = kJobResid;
                    job.list_idx = e;
                } else {
                    job.kind = kJobBonus;
                    job.M = Mk;
                }
                job.trow = ot + n;
                job.c = c;
                job.u = u_resample[ot + n];
            }
        }
    }

    // outputs: prefix, placeholder at n (written by select_kernel for sampled
    // draws), -1 after; everything -1 on a data error
    for (int i = lane; i <= k; i += 32) {
        int32_t o = -1;
        if (n >= 0) {
            if (i < n) o = x;  // i < n <= 32, so i == lane: this lane's own token
            else if (i == n && c == 0.0f) o = tok;
        }
        out_tokens[ot + i] = o;
    }
    if (lane == 0) {
        out_num[b] = n;
        ws.jobs[b] = job;
        if (aux.residual_mass) aux.residual_mass[b] = NAN;
    }
    if (aux.accept_prob && lane < k) aux.accept_prob[od + lane] = (n >= 0) ? alpha_out : NAN;
    if (aux.lse_target && lane <= k && lane < 32)
        aux.lse_target[ot + lane] = (n >= 0 && have_t) ? static_cast<float>(Lt * kLn2D) : NAN;
    if (aux.lse_target && k == kMaxK && lane == 0) {
        RowSoft r32;
        const bool ok32 = n >= 0 && c > 0.0f &&
                          combine_soft(ws.part + (ot + k) * g.n_chunks, g.n_chunks, &r32);
        aux.lse_target[ot + k] =
            ok32 ? static_cast<float>((static_cast<double>(r32.M) + log2(r32.S)) * kLn2D) : NAN;
    }
    if (aux.lse_draft && lane < k)
        aux.lse_draft[od + lane] = (n >= 0 && have_d) ? static_cast<float>(Ld * kLn2D) : NAN;
}

// ================================================================== kernel 3
// Residual mass per half-chunk of the two rows at the rejected position.
// grid = (n_half, B); block (h, e) handles residual list entry e.
template <int DT>
__global__ void __launch_bounds__(256) resid_kernel(const void *__restrict__ target,
                                                    const void *__restrict__ draft, Geometry g,
                                                    WsPtrs ws) {
    using E = Elem<DT>;
    __shared__ double s_red[32];
    const int e = blockIdx.y;
    if (e >= __ldcg(ws.counters + 0)) return;
    const int h = blockIdx.x;
    const RJob r = ws.rjobs[e];
    const int e0 = h * g.half_elems;
    const int e1 = min(g.V, e0 + g.half_elems);
    const int nvec = (e1 - e0) / E::kPerVec;
    const uint4 *pt = reinterpret_cast<const uint4 *>(static_cast<const unsigned char *>(target) +
                                                      (r.trow * g.V + e0) * static_cast<int64_t>(E::kBytes));
    const uint4 *pd = reinterpret_cast<const uint4 *>(static_cast<const unsigned char *>(draft) +
                                                      (r.drow * g.V + e0) * static_cast<int64_t>(E::kBytes));
    float s = 0.0f;
    for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
        const uint4 a = __ldg(pt + i), bq = __ldg(pd + i);
        float xt[E::kPerVec], xd[E::kPerVec];
        E::unpack(a, xt);
        E::unpack(bq, xd);
#pragma unroll
        for (int q = 0; q < E::kPerVec; ++q) s += resid_weight(xt[q], xd[q], r.c, r.lth, r.ltl, r.ldh, r.ldl);
    }
    const double tot = block_sum_d(static_cast<double>(s), s_red);
    if (threadIdx.x == 0) ws.resid_part[static_cast<int64_t>(e) * g.n_half + h] = static_cast<float>(tot);
}

// ================================================================== select
// Block-wide inverse CDF over n weights w(i) (fp32 >= 0) that start at
// cumulative mass `base`: the first i with base + sum_{i' <= i} w > target,
// else the last i with w > 0 (else -1).  Each thread owns a contiguous run
// of indices; the per-thread sums are prefix-scanned across the block in
// fp64, and the owning thread re-walks its run in the same order.
template <class WF>
__device__ int block_select(int n, WF wfn, double base, double target, double *s_d, int *s_i) {
    const int t = threadIdx.x;
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int i0 = min(n, t * per), i1 = min(n, i0 + per);
    double sum = 0.0;
    for (int i = i0; i < i1; ++i) sum += static_cast<double>(wfn(i));
    double tot;
    double run = base + block_excl_scan_d(sum, s_d, &tot);
    int found = INT_MAX, last = -1;
    for (int i = i0; i < i1; ++i) {
        const float wv = wfn(i);
        if (wv > 0.0f) last = i;
        run += static_cast<double>(wv);
        if (found == INT_MAX && run > target) found = i;
    }
    found = block_min_int(found, s_i);
    last = block_max_int(last, s_i);
    return found != INT_MAX ? found : last;
}

// Locate + scan for one soft row (bonus or draft draw): chunk weights
// s_c * 2^(m_c - M) give the chunk where the cumulative mass crosses u * S;
// that chunk is re-read and scanned element by element.
template <int DT>
__device__ int draw_from_row(const void *logits, int64_t row, const float2 *part, Geometry g, float c,
                             float M, float u, double *s_d, int *s_i) {
    using E = Elem<DT>;
    auto wchunk = [&](int i) -> float {
        const float2 v = __ldcg(part + i);
        return v.x > -INFINITY ? static_cast<float>(static_cast<double>(v.y) * exp2(static_cast<double>(v.x) - M))
                               : 0.0f;
    };
    double S = 0.0;
    for (int i = threadIdx.x; i < g.n_chunks; i += blockDim.x) S += static_cast<double>(wchunk(i));
    S = block_sum_d(S, s_d);
    const double target = static_cast<double>(u) * S;
    const int ch = block_select(g.n_chunks, wchunk, 0.0, target, s_d, s_i);
    if (ch < 0) return -1;
    double before = 0.0;
    for (int i = threadIdx.x; i < ch; i += blockDim.x) before += static_cast<double>(wchunk(i));
    before = block_sum_d(before, s_d);
    const int e0 = ch * g.chunk_elems;
    const int e1 = min(g.V, e0 + g.chunk_elems);
    const int64_t rb = row * g.V;
    auto welem = [&](int i) -> float { return prob_weight(E::load1(logits, rb + e0 + i), c, M); };
    const int v = block_select(e1 - e0, welem, before, target, s_d, s_i);
    return v < 0 ? -1 : e0 + v;
}

template <int DT>
__global__ void __launch_bounds__(kSelThreads) select_kernel(const void *__restrict__ target,
                                                             const void *__restrict__ draft, Geometry g,
                                                             WsPtrs ws, int32_t *__restrict__ out_tokens,
                                                             spec_verify_aux_t aux) {
    using E = Elem<DT>;
    __shared__ double s_d[40];
    __shared__ int s_i[40];
    const int b = blockIdx.x;
    const SeqJob job = ws.jobs[b];
    if (job.kind == kJobNone) return;
    int token;
    if (job.kind == kJobBonus) {
        token = draw_from_row<DT>(target, job.trow, ws.part + job.trow * g.n_chunks, g, job.c, job.M, job.u,
                                  s_d, s_i);
    } else {
        const RJob r = ws.rjobs[job.list_idx];
        const float *pr = ws.resid_part + static_cast<int64_t>(job.list_idx) * g.n_half;
        auto whalf = [&](int i) -> float { return __ldcg(pr + i); };
        double Z = 0.0;
        for (int i = threadIdx.x; i < g.n_half; i += blockDim.x) Z += static_cast<double>(whalf(i));
        Z = block_sum_d(Z, s_d);
        const double tgt = static_cast<double>(job.u) * Z;
        const int h = block_select(g.n_half, whalf, 0.0, tgt, s_d, s_i);
        token = -1;
        if (h >= 0) {
            double before = 0.0;
            for (int i = threadIdx.x; i < h; i += blockDim.x) before += static_cast<double>(whalf(i));
            before = block_sum_d(before, s_d);
            const int e0 = h * g.half_elems;
            const int e1 = min(g.V, e0 + g.half_elems);
            const int64_t rt = r.trow * g.V + e0, rd = r.drow * g.V + e0;
            auto welem = [&](int i) -> float {
                return resid_weight(E::load1(target, rt + i), E::load1(draft, rd + i), r.c, r.lth, r.ltl, r.ldh,
                                    r.ldl);
            };
            const int v = block_select(e1 - e0, welem, before, tgt, s_d, s_i);
            token = v < 0 ? -1 : e0 + v;
        }
        if (threadIdx.x == 0 && aux.residual_mass) aux.residual_mass[b] = static_cast<float>(Z);
    }
    if (threadIdx.x == 0) out_tokens[job.trow] = token;
}

// Draft-side draw: one block per draft row (grid-stride over rows).
template <int DT>
__global__ void __launch_bounds__(kSelThreads) draft_select_kernel(
    const void *__restrict__ draft, const float *__restrict__ temperature, const float *__restrict__ u_draft,
    const int *__restrict__ k_offsets, int B, Geometry g, const float2 *__restrict__ part,
    int32_t *__restrict__ out, int *__restrict__ counters) {
    extern __shared__ int s_kofs[];  // [B+1]
    __shared__ double s_d[40];
    __shared__ int s_i[40];
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
    if (s_bad) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(counters + 1, SPEC_ERR_INVALID_ARG);
        return;
    }
    const int R = s_kofs[B];
    for (int r = blockIdx.x; r < R; r += gridDim.x) {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_kofs[mid] <= r) lo = mid; else hi = mid - 1;
        }
        const float c = temp_scale(temperature[lo]);
        const float2 *pr = part + static_cast<int64_t>(r) * g.n_chunks;
        int token = -1;
        if (c == 0.0f) {
            token = combine_arg(pr, g.n_chunks);
        } else if (c == c) {
            RowSoft rs;
            if (combine_soft(pr, g.n_chunks, &rs))
                token = draw_from_row<DT>(draft, r, pr, g, c, rs.M, u_draft[r], s_d, s_i);
        }
        if (threadIdx.x == 0) out[r] = token;
        __syncthreads();
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
    g->half_elems = ce / 2;
    g->n_half = (V + g->half_elems - 1) / g->half_elems;
    return true;
}

struct WsLayout {
    size_t part, jobs, rjobs, counters, resid, total;
};

// Workspace layout.  The counters block comes first so that the status word
// has a fixed offset (kStatusOffset) whatever B and V are.
constexpr size_t kStatusOffset = sizeof(int);  // counters[1]

WsLayout ws_layout(int B, const Geometry &g) {
    WsLayout l;
    size_t off = 0;
    const size_t rows_cap = static_cast<size_t>(2 * kMaxK + 1) * B;
    l.counters = off;
    off = align_up(off + 64, 256);
    l.part = off;
    off = align_up(off + rows_cap * g.n_chunks * sizeof(float2), 256);
    l.jobs = off;
    off = align_up(off + B * sizeof(SeqJob), 256);
    l.rjobs = off;
    off = align_up(off + B * sizeof(RJob), 256);
    l.resid = off;
    off = align_up(off + static_cast<size_t>(B) * g.n_half * sizeof(float), 256);
    l.total = off;
    return l;
}

WsPtrs ws_ptrs(void *base, const WsLayout &l) {
    unsigned char *p = static_cast<unsigned char *>(base);
    WsPtrs w;
    w.part = reinterpret_cast<float2 *>(p + l.part);
    w.jobs = reinterpret_cast<SeqJob *>(p + l.jobs);
    w.rjobs = reinterpret_cast<RJob *>(p + l.rjobs);
    w.counters = reinterpret_cast<int *>(p + l.counters);
    w.resid_part = reinterpret_cast<float *>(p + l.resid);
    return w;
}

template <int DT, bool DRAFT>
void set_stats_attrs(int smem_optin) {
    cudaFuncSetAttribute(stats_kernel<DT, DRAFT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
}

DeviceState *device_state(int *dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceState &st = g_dev[dev];
    std::lock_guard<std::mutex> lock(g_mu);
    if (!st.init) {
        cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&st.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        cudaDeviceGetAttribute(&st.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        set_stats_attrs<SPEC_F32, false>(st.smem_optin);
        set_stats_attrs<SPEC_F32, true>(st.smem_optin);
        set_stats_attrs<SPEC_BF16, false>(st.smem_optin);
        set_stats_attrs<SPEC_BF16, true>(st.smem_optin);
        if (cudaGetLastError() != cudaSuccess) return nullptr;
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
    s += ns * kConsumerWarps * sizeof(float2);
    s += static_cast<size_t>(B + 1) * 2 * sizeof(int) + B * sizeof(float);
    s += (kThreads / 32 + 2) * sizeof(int);
    return align_up(s, 128);
}

// Ring depth and CTAs per SM: as many slots as fit two CTAs per SM (up to
// kMaxSlots), else one CTA per SM.
void pick_ring(const DeviceState &st, int B, int *ns, size_t *smem, int *ctas_per_sm) {
    for (int per_sm = 2; per_sm >= 1; --per_sm) {
        const size_t budget = static_cast<size_t>(st.smem_per_sm) / per_sm - 1024;
        for (int n = kMaxSlots; n >= 2; --n) {
            const size_t s = stats_smem(n, B);
            if (s <= budget && s <= static_cast<size_t>(st.smem_optin)) {
                *ns = n;
                *smem = s;
                *ctas_per_sm = per_sm;
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
    if (cudaMalloc(&p, need) != cudaSuccess) return nullptr;
    if (cudaMemset(p, 0, need) != cudaSuccess) {
        cudaFree(p);
        return nullptr;
    }
    st.ws = p;
    st.ws_bytes = need;
    return p;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(int B, int V, int dtype) {
    if (B < 0 || B > SPEC_MAX_B || V <= 0 || V > SPEC_MAX_V) return SPEC_ERR_INVALID_ARG;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
    const int s = dtype == SPEC_F32 ? 4 : 2;
    if ((static_cast<int64_t>(V) * s) % 16 != 0) return SPEC_ERR_ALIGNMENT;
    return SPEC_OK;
}

template <int DT>
int launch_verify(const void *target, const void *draft, const int32_t *tokens, const float *u_accept,
                  const float *u_resample, const float *temperature, int B, const int32_t *k_offsets,
                  const Geometry &g, int32_t *out_tokens, int32_t *out_num, const spec_verify_aux_t &aux,
                  void *ws_base, const WsLayout &l, const DeviceState &st, cudaStream_t stream) {
    int ns, per_sm;
    size_t smem;
    pick_ring(st, B, &ns, &smem, &per_sm);
    if (ns == 0) return SPEC_ERR_INVALID_ARG;
    const WsPtrs w = ws_ptrs(ws_base, l);
    const int grid = st.sms * per_sm;
    stats_kernel<DT, false><<<grid, kThreads, smem, stream>>>(target, draft, temperature, k_offsets, B, g, ns,
                                                              w.part, w.counters);
    decide_kernel<DT><<<(B + 7) / 8, 256, 0, stream>>>(target, draft, tokens, u_accept, u_resample, temperature,
                                                       k_offsets, B, g, w, out_tokens, out_num, aux);
    resid_kernel<DT><<<dim3(g.n_half, B), 256, 0, stream>>>(target, draft, g, w);
    select_kernel<DT><<<B, kSelThreads, 0, stream>>>(target, draft, g, w, out_tokens, aux);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

template <int DT>
int launch_draft(const void *draft, const float *temperature, const float *u_draft, int B,
                 const int32_t *k_offsets, const Geometry &g, int32_t *out, void *ws_base, const WsLayout &l,
                 const DeviceState &st, cudaStream_t stream) {
    int ns, per_sm;
    size_t smem;
    pick_ring(st, B, &ns, &smem, &per_sm);
    if (ns == 0) return SPEC_ERR_INVALID_ARG;
    const WsPtrs w = ws_ptrs(ws_base, l);
    stats_kernel<DT, true><<<st.sms * per_sm, kThreads, smem, stream>>>(draft, draft, temperature, k_offsets, B,
                                                                         g, ns, w.part, w.counters);
    const int grid = std::min(static_cast<int64_t>(st.sms) * 8, static_cast<int64_t>(B) * kMaxK);
    draft_select_kernel<DT><<<std::max(grid, 1), kSelThreads, (B + 1) * sizeof(int), stream>>>(
        draft, temperature, u_draft, k_offsets, B, g, w.part, out, w.counters);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
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

int spec_verify_ex(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                   const float *u_accept, const float *u_resample, const float *temperature, int B,
                   const int32_t *k_offsets, int V, int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
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
    void *ws = workspace;
    if (ws) {
        if (workspace_bytes < l.total) return SPEC_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SPEC_ERR_ALIGNMENT;
    } else {
        ws = get_internal_ws(*st, l.total);
        if (!ws) return SPEC_ERR_CUDA;
    }
    spec_verify_aux_t a{};
    if (aux) a = *aux;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == SPEC_F32)
        return launch_verify<SPEC_F32>(target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                                       temperature, B, k_offsets, g, out_tokens, out_num_accepted, a, ws, l, *st,
                                       s);
    return launch_verify<SPEC_BF16>(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature,
                                    B, k_offsets, g, out_tokens, out_num_accepted, a, ws, l, *st, s);
}

int spec_verify(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                const float *u_accept, const float *u_resample, const float *temperature, int B,
                const int32_t *k_offsets, int V, int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
                void *stream) {
    return spec_verify_ex(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature, B,
                          k_offsets, V, dtype, out_tokens, out_num_accepted, nullptr, nullptr, 0, stream);
}

int spec_draft_sample_ex(const void *draft_logits, const float *temperature, const float *u_draft, int B,
                         const int32_t *k_offsets, int V, int dtype, int32_t *out_draft_tokens, void *workspace,
                         size_t workspace_bytes, void *stream) {
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
    void *ws = workspace;
    if (ws) {
        if (workspace_bytes < l.total) return SPEC_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SPEC_ERR_ALIGNMENT;
    } else {
        ws = get_internal_ws(*st, l.total);
        if (!ws) return SPEC_ERR_CUDA;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == SPEC_F32)
        return launch_draft<SPEC_F32>(draft_logits, temperature, u_draft, B, k_offsets, g, out_draft_tokens, ws, l,
                                      *st, s);
    return launch_draft<SPEC_BF16>(draft_logits, temperature, u_draft, B, k_offsets, g, out_draft_tokens, ws, l,
                                   *st, s);
}

int spec_draft_sample(const void *draft_logits, const float *temperature, const float *u_draft, int B,
                      const int32_t *k_offsets, int V, int dtype, int32_t *out_draft_tokens, void *stream) {
    return spec_draft_sample_ex(draft_logits, temperature, u_draft, B, k_offsets, V, dtype, out_draft_tokens,
                                nullptr, 0, stream);
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
            if (cudaMalloc(&st->stage, off) != cudaSuccess) return SPEC_ERR_CUDA;
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
    rc = spec_draft_sample(d + o_d, reinterpret_cast<const float *>(d + o_T), reinterpret_cast<const float *>(d + o_ud),
                           B, reinterpret_cast<const int32_t *>(d + o_k), V, dtype,
                           reinterpret_cast<int32_t *>(d + o_xd), stream);
    if (rc != SPEC_OK) return rc;
    rc = spec_verify(d + o_t, d + o_d, reinterpret_cast<const int32_t *>(d + o_xd),
                     reinterpret_cast<const float *>(d + o_ua), reinterpret_cast<const float *>(d + o_ur),
                     reinterpret_cast<const float *>(d + o_T), B, reinterpret_cast<const int32_t *>(d + o_k), V,
                     dtype, reinterpret_cast<int32_t *>(d + o_ot), reinterpret_cast<int32_t *>(d + o_on), stream);
    if (rc != SPEC_OK) return rc;
    if (R_d) cudaMemcpyAsync(out_draft_tokens_host, d + o_xd, R_d * 4, cudaMemcpyDeviceToHost, s);
    cudaMemcpyAsync(out_tokens_host, d + o_ot, R_t * 4, cudaMemcpyDeviceToHost, s);
    cudaMemcpyAsync(out_num_accepted_host, d + o_on, B * 4, cudaMemcpyDeviceToHost, s);
    if (cudaStreamSynchronize(s) != cudaSuccess) return SPEC_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
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
    if (cudaMemcpy(&v, base + kStatusOffset, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return SPEC_ERR_CUDA;
    *status_out = v;
    if (clear && cudaMemset(const_cast<unsigned char *>(base) + kStatusOffset, 0, sizeof v) != cudaSuccess)
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

}  // extern "C"
