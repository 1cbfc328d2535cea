// shard_verify.cu -- the verify step over a vocabulary split across ranks.
//
// Each rank holds a contiguous range of columns [V_r, V_{r+1}) of every
// target and draft logit row.  One verify is three calls per rank:
//   spec_shard_stats  stats_kernel over the rank's columns (the chain
//                     verify's streaming pass, unchanged), then
//                     shard_row_kernel: one 16-byte record per row
//                     (max, sum of 2^(z c - max), the drafted token's logit
//                     if the rank holds it, or the greedy arg-max);
//   spec_shard_decide shard_decide_kernel, one block per sequence: every
//                     rank combines the gathered records of a row in rank
//                     order, so that all ranks take the same accept
//                     decisions; then the rank's share of the mass to draw
//                     from (a residual pass over its columns, or the bonus
//                     row's mass from its partials);
//   spec_shard_draw   shard_draw_kernel, one block per sequence: the
//                     gathered masses locate the rank holding the crossing
//                     of the cumulative mass, and that rank alone draws
//                     inside its columns (its warp 0 locates the sub-chunk,
//                     the block scans it).
// The accept rule, residual and bonus are those of the chain verify
// (docs.ifdog.com "投机解码", 投机解码的三步流程 step 3; bbs.huaweicloud.com
// "大模型推理无损加速:投机采样(Speculative Decoding)数学原理与工业级落地实践",
// 二.1, 二.2): only where each sum is taken differs.
#include <algorithm>
#include <climits>
#include <cstdio>
#include <mutex>

#include "host_common.h"

namespace specv {

constexpr int kMaxShards = SPEC_MAX_SHARDS;

// Column bounds of the G shards, passed by value to every kernel.
struct ShardSpec {
    int G;
    int rank;
    int v0;  // this rank's first column
    int bound[kMaxShards + 1];
};

// The decision of one sequence, written by shard_decide_kernel into the
// workspace for shard_draw_kernel.
struct ShardSeq {
    int kind;   // kJobNone, kJobResid or kJobBonus
    int n;      // accepted count
    int ot;     // first target row (and output slot)
    int od;     // first draft row
    float c;    // temperature scale log2(e) / T
    float M;    // global max of z c over target row ot + n (the p weights' reference)
    float lth, ltl, ldh, ldl;  // log2-domain lse of target / draft row n, as fp32 hi + lo
};

__device__ __forceinline__ int shard_of(const int *bound, int G, int x) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (bound[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// k_offsets check shared by the shard kernels (any block size): k_offsets[0]
// must be 0 and every k_b within [0, kMaxK].
__device__ __forceinline__ bool block_bad_offsets(const int *__restrict__ k_offsets, int B) {
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
    return __syncthreads_or(bad) != 0;
}

// A row's combine over this shard's sub-chunk partials: M = the largest
// partial maximum (-inf when no column is finite), S = sum s_i 2^(m_i - M)
// (0 then).  False when a partial carries NaN (a NaN or +inf column).
// cache: the row's first 32 * kPartCache partials (load_parts).
static __device__ __forceinline__ bool shard_combine_soft(const float2 (&cache)[kPartCache], const float2 *p, int n,
                                                          float *M_out, float *S_out) {
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
    if (__any_sync(0xffffffffu, nan)) return false;
    float S = 0.0f;
    if (M > -INFINITY) {
        Acc2 acc;
#pragma unroll
        for (int j = 0; j < kPartCache; ++j)
            if (cache[j].x > -INFINITY) acc.add(cache[j].y * ex2(cache[j].x - M));
        for (int i = lane + 32 * kPartCache; i < n; i += 32) {
            const float2 v = __ldcg(p + i);
            if (v.x > -INFINITY) acc.add(v.y * ex2(v.x - M));
        }
        S = warp_sum_f(acc.value());
    }
    *M_out = M;
    *S_out = S;
    return true;
}

// ============================================================ row records
// One block per sequence; warp w takes rows w, w + 8, ... of the sequence
// (its k + 1 target rows, then its k draft rows), so that every record of
// the call is written.  The k_offsets check, the drafted tokens and their
// logits in this rank's columns (the call's inputs, complete once
// stats_kernel has passed its own wait) are read before the wait on
// stats_kernel; after it, only each row's partials.  Partials are at slot r for
// target row r and R_t + d for draft row d (the record index), as
// stats_kernel writes them in verify mode.
// (four blocks per SM: a 512-sequence batch is resident at once)
template <int DT>
__global__ void __launch_bounds__(256, 4) shard_row_kernel(
    const void *__restrict__ target, const void *__restrict__ draft, const int32_t *__restrict__ tokens,
    const float *__restrict__ temperature, const int *__restrict__ k_offsets, int B, Geometry g, int v0,
    const float2 *__restrict__ part, spec_shard_stat_t *__restrict__ out, int *__restrict__ counters) {
    using E = Elem<DT>;
    __shared__ int s_x[kMaxK];
    __shared__ float s_zx[2 * kMaxK];  // the drafted token's logit in row rr (rr < k: target, else draft)
    const int b = blockIdx.x;
    const bool bad = block_bad_offsets(k_offsets, B);
    int k0 = 0, k = 0, R_t = 0;
    float c = 0.0f;
    if (!bad) {
        k0 = k_offsets[b];
        k = k_offsets[b + 1] - k0;
        R_t = k_offsets[B] + B;
        c = temp_scale(temperature[b]);
        if (static_cast<int>(threadIdx.x) < k) s_x[threadIdx.x] = tokens[k0 + threadIdx.x];
    }
    __syncthreads();
    if (!bad && c == c && c != 0.0f) {
        // thread j < 2k: the token's logit in target row j (j < k) or draft
        // row j - k, if this rank holds its column
        const int j = threadIdx.x;
        if (j < 2 * k) {
            const bool is_t = j < k;
            const int i = is_t ? j : j - k;
            const int x = s_x[i];
            const int64_t row = is_t ? static_cast<int64_t>(k0) + b + i : static_cast<int64_t>(k0) + i;
            float zx = 0.0f;
            if (x >= v0 && x - v0 < g.V) zx = E::load1(is_t ? target : draft, row * g.V + (x - v0));
            s_zx[j] = zx;
        }
    }
    __syncthreads();
    grid_dependency_wait();
    grid_launch_dependents();
    if (bad) {
        if (b == 0 && threadIdx.x == 0) set_status(counters + kStatus, SPEC_ERR_INVALID_ARG);
        return;
    }
    const int lane = lane_id();
    const int ot = k0 + b;
    const bool greedy = c == 0.0f, valid = c == c;
    const int nrows = 2 * k + 1, nw = blockDim.x >> 5;
    // record index of row rr (target rows first) and whether it is combined
    auto rec_of = [&](int rr) -> int64_t {
        return rr <= k ? static_cast<int64_t>(ot) + rr : static_cast<int64_t>(R_t) + k0 + (rr - k - 1);
    };
    auto combined = [&](int rr) -> bool { return valid && (!greedy || rr <= k); };
    // the first 32 partials of a warp's next kAhead rows are requested
    // together (whole rows when a shard has at most 32 sub-chunks), so that
    // its rows wait on L2 once rather than one after another
    constexpr int kAhead = 3;
    auto first_part = [&](int rr) -> float2 {
        return (rr < nrows && combined(rr) && lane < g.n_sub) ? __ldcg(part + rec_of(rr) * g.n_sub + lane)
                                                               : make_float2(-INFINITY, 0.0f);
    };
    float2 ahead[kAhead];
#pragma unroll
    for (int q = 0; q < kAhead; ++q) ahead[q] = first_part(warp_id() + q * nw);
    for (int rr = warp_id(); rr < nrows; rr += nw) {
        const bool is_t = rr <= k;
        const int i = is_t ? rr : rr - k - 1;
        const int64_t r = rec_of(rr);
        const float2 *p = part + r * g.n_sub;
        // the row's cache as load_parts fills it, its first entry requested earlier
        float2 cur[kPartCache];
        cur[0] = ahead[0];
#pragma unroll
        for (int q = 0; q + 1 < kAhead; ++q) ahead[q] = ahead[q + 1];
        ahead[kAhead - 1] = first_part(rr + kAhead * nw);
#pragma unroll
        for (int j = 1; j < kPartCache; ++j) {
            const int e = lane + 32 * j;
            cur[j] = (combined(rr) && e < g.n_sub) ? __ldcg(p + e) : make_float2(-INFINITY, 0.0f);
        }
        spec_shard_stat_t rec{-INFINITY, __int_as_float(0x7fc00000), 0.0f, -1};
        if (valid && greedy && is_t) {
            ArgPart a{-INFINITY, INT_MAX};
#pragma unroll
            for (int j = 0; j < kPartCache; ++j)
                if (lane + 32 * j < g.n_sub) a = arg_merge(a, ArgPart{cur[j].x, __float_as_int(cur[j].y)});
            for (int j = lane + 32 * kPartCache; j < g.n_sub; j += 32) {
                const float2 v = __ldcg(p + j);
                a = arg_merge(a, ArgPart{v.x, __float_as_int(v.y)});
            }
            a = warp_arg(a);
            rec = spec_shard_stat_t{a.v, 0.0f, 0.0f, (a.i == -1 || a.i == INT_MAX) ? -1 : a.i + v0};
        } else if (valid && !greedy) {
            const float zx = i < k ? s_zx[is_t ? i : k + i] : 0.0f;
            float M, S;
            if (shard_combine_soft(cur, p, g.n_sub, &M, &S)) {
                rec = spec_shard_stat_t{M, S, zx, 0};
            } else {
                rec = spec_shard_stat_t{-INFINITY, __int_as_float(0x7fc00000), zx, 0};
            }
        }
        if (lane == 0) out[r] = rec;
    }
}

// ================================================================ decide
// This rank's residual masses max(0, p - q) of one (target, draft) row pair,
// per sub-chunk of its columns, by all warps of the block; warp 0 first
// moves both rows to L2 in bulk so that the loads wait on L2.  The masses
// go to rp, and the first 32 * kPartCache also to rp_s (shared memory) for
// the block's own total.
template <int DT>
__device__ void shard_resid_pass(const void *target, const void *draft, int64_t trow, int64_t drow,
                                 const Geometry &g, float c, float lth, float ltl, float ldh, float ldl, float *rp,
                                 float *rp_s) {
    using E = Elem<DT>;
    const int lane = lane_id(), warp = warp_id(), nwarps = blockDim.x >> 5;
    const unsigned char *t0 = static_cast<const unsigned char *>(target) + trow * g.V * static_cast<int64_t>(E::kBytes);
    const unsigned char *d0 = static_cast<const unsigned char *>(draft) + drow * g.V * static_cast<int64_t>(E::kBytes);
    if (warp == 0) {
        // row bytes are a multiple of 16 and rows start 16-byte aligned
        const int64_t nbytes = static_cast<int64_t>(g.V) * E::kBytes;
        constexpr int64_t kPiece = 32768;
        for (int64_t off = static_cast<int64_t>(lane >> 1) * kPiece; off < nbytes; off += 16 * kPiece)
            bulk_prefetch_l2(((lane & 1) ? d0 : t0) + off, static_cast<uint32_t>(min(kPiece, nbytes - off)));
    }
    const float2 c2 = make_float2(c, c), nlth2 = make_float2(-lth, -lth), nltl2 = make_float2(-ltl, -ltl);
    const float2 nldh2 = make_float2(-ldh, -ldh), nldl2 = make_float2(-ldl, -ldl);
    for (int sc = warp; sc < g.n_sub; sc += nwarps) {
        int a, e1;
        sub_range(g, sc, &a, &e1);
        const int nvec = (e1 - a) / E::kPerVec;  // <= 128; 0 for a trailing empty sub-chunk
        const uint4 *pt = reinterpret_cast<const uint4 *>(t0 + static_cast<int64_t>(a) * E::kBytes);
        const uint4 *pd = reinterpret_cast<const uint4 *>(d0 + static_cast<int64_t>(a) * E::kBytes);
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
                const float2 w2 =
                    resid_weight2(E::pair(xt4[j], p), E::pair(xd4[j], p), c2, nlth2, nltl2, nldh2, nldl2);
                if (p & 1) acc1 = fadd2(acc1, w2); else acc0 = fadd2(acc0, w2);
            }
        }
        const float sum = warp_sum_f((acc0.x + acc0.y) + (acc1.x + acc1.y));
        if (lane == 0) {
            rp[sc] = sum;
            if (sc < 32 * kPartCache) rp_s[sc] = sum;
        }
    }
}

// p weights of one target row's sub-chunks relative to the row's global max
// M: s_i 2^(m_i - M) (the cached first 32 * kPartCache, the rest on demand).
struct PWeights {
    const float2 *p;
    float M;
    __device__ float operator()(int i) const {
        const float2 v = __ldcg(p + i);
        return v.x > -INFINITY ? v.y * ex2(v.x - M) : 0.0f;
    }
};

__device__ __forceinline__ void p_weights_cached(const PWeights &pw, int n, float (&w)[kPartCache]) {
    float2 pc[kPartCache];
    load_parts(pw.p, n, pc);
#pragma unroll
    for (int j = 0; j < kPartCache; ++j) w[j] = pc[j].x > -INFINITY ? pc[j].y * ex2(pc[j].x - pw.M) : 0.0f;
}

struct RWeights {
    const float *r;
    __device__ float operator()(int i) const { return __ldcg(r + i); }
};

__device__ __forceinline__ void r_weights_cached(const float *r, int n, float (&w)[kPartCache]) {
    const int lane = lane_id();
#pragma unroll
    for (int j = 0; j < kPartCache; ++j) w[j] = (lane + 32 * j < n) ? __ldcg(r + lane + 32 * j) : 0.0f;
}

// the same from the block's shared copy of its first masses
__device__ __forceinline__ void r_weights_shared(const float *r_s, int n, float (&w)[kPartCache]) {
    const int lane = lane_id();
#pragma unroll
    for (int j = 0; j < kPartCache; ++j) w[j] = (lane + 32 * j < n) ? r_s[lane + 32 * j] : 0.0f;
}

struct DecideSmem {
    float M[kMaxK + 1];        // target rows: global max of z c
    float S[kMaxK + 1];        // target rows: sum of 2^(z c - M) over all ranks
    double Ld[kMaxK];          // draft rows: log2-domain log-sum-exp
    int arg[kMaxK + 1];        // greedy target rows: global arg-max
    int ok[2 * kMaxK + 1];
    float zt[kMaxK], zd[kMaxK];  // the drafted tokens' logits, from the rank holding each
    int x[kMaxK];
    int xr[kMaxK];             // the rank holding x_i
    float ua[kMaxK];
    int bound[kMaxShards + 1];
    int n, kind;
    float lth, ltl, ldh, ldl, Mn;
    float rp[32 * kPartCache];  // this rank's first residual masses (shard_resid_pass)
};

// One block per sequence.  Phase 1: the gathered records of each needed row
// are combined in rank order (one lane per rank), then warp 0 takes the
// chain verify's decision.  Phase 2 (sampled sequences): this rank's masses
// of the distribution to draw from and of p at position n.  Launched with
// programmatic dependent launch: it waits for the stream's previous kernel
// (the exchange of the records) before it reads anything, and lets the draw
// kernel be scheduled right after that wait.
template <int DT>
__global__ void __launch_bounds__(256) shard_decide_kernel(
    const void *__restrict__ target, const void *__restrict__ draft, const spec_shard_stat_t *__restrict__ all_stats,
    const int32_t *__restrict__ tokens, const float *__restrict__ u_accept, const float *__restrict__ temperature,
    const int *__restrict__ k_offsets, int B, Geometry g, ShardSpec sp, const float2 *__restrict__ part,
    float *__restrict__ resid, ShardSeq *__restrict__ seq, int32_t *__restrict__ out_tokens,
    int32_t *__restrict__ out_num, double *__restrict__ out_mass, int *__restrict__ counters) {
    __shared__ DecideSmem sm;
    const int b = blockIdx.x;
    const int lane = lane_id(), warp = warp_id();
    grid_dependency_wait();
    grid_launch_dependents();
    // the sequence's own offsets and temperature (in bounds whatever the
    // offsets hold) are requested with the check's loads
    const int kb0 = k_offsets[b], kb1 = k_offsets[b + 1], kbB = k_offsets[B];
    const float temp_b = temperature[b];
    if (block_bad_offsets(k_offsets, B)) {
        // the whole call fails; outputs of unknown size stay untouched
        if (threadIdx.x == 0) {
            out_num[b] = -1;
            seq[b].kind = kJobNone;
            out_mass[2 * b] = 0.0;
            out_mass[2 * b + 1] = 0.0;
            if (b == 0) set_status(counters + kStatus, SPEC_ERR_INVALID_ARG);
        }
        return;
    }
    const int k0 = kb0;
    const int k = kb1 - k0;
    const int ot = k0 + b, od = k0;
    const int R_t = kbB + B;
    const int64_t per_rank = static_cast<int64_t>(R_t) + kbB;  // records per rank
    const float c = temp_scale(temp_b);
    const bool greedy = c == 0.0f;
    const int G = sp.G;
    for (int i = threadIdx.x; i <= G; i += blockDim.x) sm.bound[i] = sp.bound[i];
    const int V = sp.bound[G];

    // A row's G records are combined by a group of gs lanes (the power of
    // two at or above G, one lane per rank), so that a warp takes 32 / gs
    // rows at once; with more than 32 ranks, lane l holds ranks l and l + 32.
    const int nrows = greedy ? k + 1 : 2 * k + 1;
    const int nw = blockDim.x >> 5;
    const int gs = G <= 32 ? (G <= 1 ? 1 : 1 << (32 - __clz(G - 1))) : 32;
    const int rpw = 32 / gs;  // rows per warp and round
    const int grp = lane / gs, gl = lane - grp * gs;
    // each lane's records (m, s, zx, arg) of row r0 + grp: rank gl (and gl + 32);
    // a greedy sequence's draft records are loaded too, unused (so that the
    // loads need k_offsets alone, not the temperature)
    auto load_recs = [&](int r0, int4 (&st)[2]) {
        const int rr = r0 + grp;
        const bool active = rr < 2 * k + 1;
        const bool is_t = rr <= k;
        const int i = is_t ? rr : rr - k - 1;
        const int64_t rec = is_t ? static_cast<int64_t>(ot) + i : static_cast<int64_t>(R_t) + od + i;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int h = gl + 32 * j;
            st[j] = (active && h < G) ? __ldg(reinterpret_cast<const int4 *>(all_stats + h * per_rank + rec))
                                      : make_int4(__float_as_int(-INFINITY), 0, 0, INT_MAX);
        }
    };
    // the first round's records are requested before the drafted tokens, so
    // that both wait on memory together
    int4 st0[2];
    load_recs(warp * rpw, st0);
    int xbad = 0;
    if (static_cast<int>(threadIdx.x) < k) {
        const int x = tokens[od + threadIdx.x];
        sm.x[threadIdx.x] = x;
        sm.ua[threadIdx.x] = u_accept[od + threadIdx.x];
        xbad = (x < 0 || x >= V);
    }
    const bool err0 = __syncthreads_or(xbad) || (c != c);
    if (!err0 && static_cast<int>(threadIdx.x) < k) sm.xr[threadIdx.x] = shard_of(sm.bound, G, sm.x[threadIdx.x]);
    __syncthreads();

    // --- 1. rows over all ranks -------------------------------------------
    // The group's reductions are the whole warp's with the other groups'
    // steps left out, which only ever added zeros: the same bits.
    if (!err0) {
        for (int r0 = warp * rpw; r0 < nrows; r0 += nw * rpw) {
            const int rr = r0 + grp;
            const bool active = rr < nrows;
            const bool is_t = rr <= k;
            const int i = is_t ? rr : rr - k - 1;
            const int si = is_t ? i : kMaxK + 1 + i;
            int4 st[2];
            if (r0 == warp * rpw) {
                st[0] = st0[0];
                st[1] = st0[1];
            } else {
                load_recs(r0, st);
            }
            if (greedy) {
                ArgPart a{-INFINITY, INT_MAX};
#pragma unroll
                for (int j = 0; j < 2; ++j) a = arg_merge(a, ArgPart{__int_as_float(st[j].x), st[j].w});
                for (int off = gs >> 1; off > 0; off >>= 1) a = arg_merge(a, shfl_arg(a, off));
                if (active && gl == 0) {
                    sm.arg[si] = a.i;
                    sm.ok[si] = a.i >= 0 && a.i != INT_MAX;
                }
            } else {
                float mh[2], sh[2];
                float M = -INFINITY;
                bool nan = false;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    mh[j] = __int_as_float(st[j].x);
                    sh[j] = __int_as_float(st[j].y);
                    nan |= (sh[j] != sh[j]);
                    M = fmaxf(M, mh[j]);
                }
                for (int off = gs >> 1; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
                const unsigned gmask = (gs == 32 ? 0xffffffffu : ((1u << gs) - 1u)) << (grp * gs);
                nan = (__ballot_sync(0xffffffffu, nan) & gmask) != 0u;
                Acc2 acc;
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    if (mh[j] > -INFINITY) acc.add(sh[j] * ex2(mh[j] - M));
                float S = acc.value();
                for (int off = gs >> 1; off > 0; off >>= 1) S += __shfl_xor_sync(0xffffffffu, S, off);
                const bool ok = !nan && M > -INFINITY && M < INFINITY && S > 0.0f && S < INFINITY;
                // the drafted token's logit, from the group's lane holding its rank
                const int h = (active && i < k) ? sm.xr[i] : 0;
                const float z = __shfl_sync(0xffffffffu, __int_as_float(h < 32 ? st[0].z : st[1].z),
                                            grp * gs + (h & 31) % gs);
                if (active && gl == 0) {
                    if (is_t) {
                        sm.M[i] = M;
                        sm.S[i] = S;
                    } else {
                        sm.Ld[i] = ok ? lse2(M, S) : NAN;
                    }
                    sm.ok[si] = ok;
                    if (i < k) {
                        if (is_t) sm.zt[i] = z; else sm.zd[i] = z;
                    }
                }
            }
        }
    }
    __syncthreads();

    // --- the decision (warp 0), as in the chain verify ---------------------
    if (warp == 0) {
        bool err = err0;
        int n = -1, tok = -1, kind = kJobNone;
        if (!err) {
            bool rows_ok = true;
            for (int i = lane; i <= k; i += 32) rows_ok &= sm.ok[i] != 0;
            if (!greedy)
                for (int i = lane; i < k; i += 32) rows_ok &= sm.ok[kMaxK + 1 + i] != 0;
            err = !__all_sync(0xffffffffu, rows_ok);
        }
        if (!err && greedy) {
            // accept while x_i == argmax p_i
            const int a = (lane <= k) ? sm.arg[lane] : 0;
            const int x = (lane < k) ? sm.x[lane] : 0;
            const unsigned mism = __ballot_sync(0xffffffffu, lane < k && x != a);
            n = mism ? (__ffs(mism) - 1) : k;
            tok = sm.arg[n];
        } else if (!err) {
            // alpha_i = min(1, p_i(x_i) / q_i(x_i)): log-ratio in fp64, the
            // exponential in fp32
            bool acc = false;
            double Ld = NAN;
            if (lane < k) {
                const double Lt = lse2(sm.M[lane], sm.S[lane]);
                Ld = sm.Ld[lane];
                const float zt = sm.zt[lane], zd = sm.zd[lane];
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
                acc = sm.ua[lane] < alpha;
            }
            const unsigned rej = __ballot_sync(0xffffffffu, lane < k && !acc);
            n = rej ? (__ffs(rej) - 1) : k;
            kind = n < k ? kJobResid : kJobBonus;
            const double Ldn = __shfl_sync(0xffffffffu, Ld, n & 31);  // used only if n < k
            if (lane == 0) {
                sm.Mn = sm.M[n];
                if (n < k) {
                    const double Ltn = lse2(sm.M[n], sm.S[n]);
                    sm.lth = static_cast<float>(Ltn);
                    sm.ltl = static_cast<float>(Ltn - static_cast<double>(sm.lth));
                    sm.ldh = static_cast<float>(Ldn);
                    sm.ldl = static_cast<float>(Ldn - static_cast<double>(sm.ldh));
                }
            }
        }
        // outputs: the accepted prefix, the greedy token at n, -1 after (a
        // sampled token at n is written by the drawing rank); all -1 on a
        // data error
        for (int i = lane; i <= k; i += 32) {
            int32_t o = -1;
            if (n >= 0) {
                if (i < n) o = sm.x[i];
                else if (i == n && greedy) o = tok;
            }
            out_tokens[ot + i] = o;
        }
        __syncwarp();
        if (lane == 0) {
            out_num[b] = n;
            sm.n = n;
            sm.kind = kind;
            ShardSeq q;
            q.kind = kind;
            q.n = n;
            q.ot = ot;
            q.od = od;
            q.c = c;
            q.M = kind != kJobNone ? sm.Mn : 0.0f;
            q.lth = kind == kJobResid ? sm.lth : 0.0f;
            q.ltl = kind == kJobResid ? sm.ltl : 0.0f;
            q.ldh = kind == kJobResid ? sm.ldh : 0.0f;
            q.ldl = kind == kJobResid ? sm.ldl : 0.0f;
            seq[b] = q;
        }
    }
    __syncthreads();
    const int kind = sm.kind;
    if (kind == kJobNone) {
        if (threadIdx.x == 0) {
            out_mass[2 * b] = 0.0;
            out_mass[2 * b + 1] = 0.0;
        }
        return;
    }

    // --- 2. this rank's masses ---------------------------------------------
    const int n = sm.n;
    const int64_t trow = static_cast<int64_t>(ot) + n;
    float *rp = resid + static_cast<int64_t>(b) * g.n_sub;
    const PWeights pw{part + trow * g.n_sub, sm.Mn};
    float w[kPartCache];
    if (warp == 0) p_weights_cached(pw, g.n_sub, w);  // p of row n: the bonus, or a zero residual's fallback
    if (kind == kJobResid) {
        shard_resid_pass<DT>(target, draft, trow, static_cast<int64_t>(od) + n, g, c, sm.lth, sm.ltl, sm.ldh, sm.ldl,
                             rp, sm.rp);
        __syncthreads();  // every warp's masses, before warp 0 sums them
    }
    if (warp != 0) return;
    const F2 Zp = warp_total(g.n_sub, w, pw);
    F2 Z = Zp;
    if (kind == kJobResid) {
        r_weights_shared(sm.rp, g.n_sub, w);
        Z = warp_total(g.n_sub, w, RWeights{rp});
    }
    if (lane == 0) {
        out_mass[2 * b] = static_cast<double>(Z.hi) + static_cast<double>(Z.lo);
        out_mass[2 * b + 1] = static_cast<double>(Zp.hi) + static_cast<double>(Zp.lo);
    }
}

// ================================================================ draw
// One block per sequence.  Warp 0 sums the gathered masses in rank order (the
// same operations on every rank) and finds the rank whose cumulative mass
// first exceeds u * Z; that rank alone draws, inside its columns, at the
// remaining target: warp 0 locates the sub-chunk, the block scans its
// elements (block_scan_elems).  A residual mass of 0 on every rank falls
// back to p.  Launched with programmatic dependent launch: it waits for the
// stream's previous kernel (the exchange of the masses) before it reads
// anything.
struct ShardDrawSmem {
    DrawSmem ds;
    int draw;   // this rank draws: 1 from the residual, 2 from p
    int64_t trow;
};

template <int DT>
__global__ void __launch_bounds__(kDrawThreads) shard_draw_kernel(
    const void *__restrict__ target, const void *__restrict__ draft, const double *__restrict__ all_mass,
    const float *__restrict__ u_resample, const int *__restrict__ k_offsets, int B, Geometry g, ShardSpec sp,
    const float2 *__restrict__ part, const float *__restrict__ resid, const ShardSeq *__restrict__ seq,
    int32_t *__restrict__ out_tokens) {
    using E = Elem<DT>;
    __shared__ ShardDrawSmem sm;
    const int lane = lane_id();
    const int b = blockIdx.x;
    grid_dependency_wait();
    const ShardSeq q = seq[b];
    if (warp_id() == 0) {
        if (lane == 0) sm.draw = 0;
        // everything that depends on b alone is loaded at once: the decision,
        // the sequence's offsets, its masses on every rank (lane l: ranks l
        // and l + 32, G <= 64) and its residual masses on this rank
        const int k0 = k_offsets[b], k1 = k_offsets[b + 1];
        double mr[2] = {0.0, 0.0}, mp[2] = {0.0, 0.0};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int h = lane + 32 * j;
            if (h < sp.G) {
                const double2 m2 =
                    __ldg(reinterpret_cast<const double2 *>(all_mass + (static_cast<int64_t>(h) * B + b) * 2));
                mr[j] = m2.x;
                mp[j] = m2.y;
            }
        }
        const float *rp = resid + static_cast<int64_t>(b) * g.n_sub;
        float w[kPartCache];
        r_weights_cached(rp, g.n_sub, w);
        // the decision must be the one spec_shard_decide wrote for this
        // call's k_offsets (it wrote kJobNone everywhere for an invalid array)
        const int k = k1 - k0;
        const bool valid = (q.kind == kJobResid || q.kind == kJobBonus) && k >= 0 && k <= kMaxK &&
                           q.ot == k0 + b && q.od == k0 && q.n >= 0 && q.n <= k && (q.kind == kJobResid) == (q.n < k);
        if (valid) {
            const int64_t trow = static_cast<int64_t>(q.ot) + q.n;
            const float u = u_resample[trow];
            float2 pc[kPartCache];  // p partials of row n, in case p is drawn from
            load_parts(part + trow * g.n_sub, g.n_sub, pc);
            // every lane adds the ranks' masses in rank order, so the sums
            // are the same on every lane and every rank
            auto mass_of = [&](int h, bool p) -> double {
                const double a = __shfl_sync(0xffffffffu, p ? mp[0] : mr[0], h & 31);
                const double c = __shfl_sync(0xffffffffu, p ? mp[1] : mr[1], h & 31);
                return h < 32 ? a : c;
            };
            double Z = 0.0;
            for (int h = 0; h < sp.G; ++h) Z += mass_of(h, false);
            const bool use_p = !(Z > 0.0);
            if (use_p) {
                Z = 0.0;
                for (int h = 0; h < sp.G; ++h) Z += mass_of(h, true);
            }
            // u < 1, so t < Z: the running sum, which repeats Z's additions,
            // exceeds t at the latest at the last rank with positive mass
            const double t = static_cast<double>(u) * Z;
            double C = 0.0, before = 0.0;
            int owner = -1;
            if (Z > 0.0) {
                for (int h = 0; h < sp.G; ++h) {
                    const double m = mass_of(h, use_p);
                    if (m > 0.0 && C + m > t) {
                        owner = h;
                        before = C;
                        break;
                    }
                    C += m;
                }
            }
            if (owner == sp.rank) {
                const double tl = t - before;
                F2 tgt;
                tgt.hi = static_cast<float>(tl);
                tgt.lo = static_cast<float>(tl - static_cast<double>(tgt.hi));
                F2 bef;
                int sc;
                const bool from_resid = q.kind == kJobResid && !use_p;
                if (from_resid) {
                    sc = warp_locate_at(g.n_sub, w, RWeights{rp}, tgt, &bef);
                } else {
                    const PWeights pw{part + trow * g.n_sub, q.M};
#pragma unroll
                    for (int j = 0; j < kPartCache; ++j)
                        w[j] = pc[j].x > -INFINITY ? pc[j].y * ex2(pc[j].x - pw.M) : 0.0f;
                    sc = warp_locate_at(g.n_sub, w, pw, tgt, &bef);
                }
                if (lane == 0) {
                    sm.draw = sc < 0 ? 3 : (from_resid ? 1 : 2);
                    sm.trow = trow;
                    sm.ds.sc = sc;
                    sm.ds.before = bef;
                    sm.ds.target = tgt;
                }
            }
        }
    }
    __syncthreads();
    const int draw = sm.draw;
    if (draw == 0) return;  // not this rank's draw (or nothing to draw)
    const int64_t trow = sm.trow;
    int token = -1;
    if (draw != 3) {
        int a, e1;
        sub_range(g, sm.ds.sc, &a, &e1);
        const unsigned char *rt = static_cast<const unsigned char *>(target) + trow * g.V * static_cast<int64_t>(E::kBytes);
        const float c = q.c;
        if (draw == 1) {
            const unsigned char *rd = static_cast<const unsigned char *>(draft) +
                                      (static_cast<int64_t>(q.od) + q.n) * g.V * static_cast<int64_t>(E::kBytes);
            const float lth = q.lth, ltl = q.ltl, ldh = q.ldh, ldl = q.ldl;
            auto W = [&](float a1, float a2) -> float { return resid_weight(a1, a2, c, lth, ltl, ldh, ldl); };
            token = block_scan_elems<DT>(rt, rd, a, e1, W, sm.ds.before, sm.ds.target, sm.ds);
        } else {
            const float M = q.M;
            auto W = [&](float x, float) -> float { return prob_weight(x, c, M); };
            token = block_scan_elems<DT>(rt, rt, a, e1, W, sm.ds.before, sm.ds.target, sm.ds);
        }
    }
    if (threadIdx.x == 0) out_tokens[trow] = token >= 0 ? token + sp.v0 : -1;
}

}  // namespace specv

// ================================================================== host side
namespace specv {

struct ShardWsLayout {
    size_t part, resid, seq, total;
};

// Counters (the common 256-byte block) | partials of up to (2 kMaxK + 1) B
// rows of this rank's columns | residual masses [B * n_sub] | decisions [B].
ShardWsLayout shard_ws_layout(int B, const Geometry &g) {
    ShardWsLayout l;
    size_t off = kCountersBytes;
    l.part = off;
    off = align_up(off + static_cast<size_t>(2 * kMaxK + 1) * B * g.n_sub * sizeof(float2), 256);
    l.resid = off;
    off = align_up(off + static_cast<size_t>(B) * g.n_sub * sizeof(float), 256);
    l.seq = off;
    off = align_up(off + static_cast<size_t>(B) * sizeof(ShardSeq), 256);
    l.total = off;
    return l;
}

bool g_shard_init[kMaxDevices] = {};
std::mutex g_shard_mu;

template <int DT>
bool shard_stats_attr(int smem_optin_raw) {
    cudaFuncAttributes fa{};
    if (!cuda_ok(cudaFuncGetAttributes(&fa, stats_kernel<DT, kModeShard>), "cudaFuncGetAttributes")) return false;
    return cuda_ok(cudaFuncSetAttribute(stats_kernel<DT, kModeShard>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        smem_optin_raw - static_cast<int>(fa.sharedSizeBytes)),
                   "cudaFuncSetAttribute(stats_kernel shard)");
}

DeviceState *shard_device_state(int *dev_out) {
    DeviceState *st = device_state(dev_out);
    if (!st) return nullptr;
    std::lock_guard<std::mutex> lock(g_shard_mu);
    if (!g_shard_init[*dev_out]) {
        int optin = 0;
        if (!cuda_ok(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, *dev_out),
                     "cudaDeviceGetAttribute"))
            return nullptr;
        if (!shard_stats_attr<SPEC_F32>(optin) || !shard_stats_attr<SPEC_BF16>(optin)) return nullptr;
        g_shard_init[*dev_out] = true;
    }
    return st;
}

// Host checks shared by the three calls: the shard bounds, G, rank, B and
// dtype; fills the kernels' shard spec and the geometry of this rank's
// columns.
int shard_setup(int B, const int32_t *bounds, int G, int rank, int dtype, ShardSpec *sp, Geometry *g) {
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
    if (!bounds || G < 1 || G > kMaxShards || rank < 0 || rank >= G || bounds[0] != 0) return SPEC_ERR_INVALID_ARG;
    const int per_vec = dtype == SPEC_F32 ? 4 : 8;
    for (int h = 0; h < G; ++h) {
        if (bounds[h + 1] <= bounds[h]) return SPEC_ERR_INVALID_ARG;
        if ((bounds[h + 1] - bounds[h]) % per_vec != 0) return SPEC_ERR_ALIGNMENT;
    }
    const int rc = check_common(B, bounds[G], dtype);
    if (rc != SPEC_OK) return rc;
    *sp = ShardSpec{};
    sp->G = G;
    sp->rank = rank;
    sp->v0 = bounds[rank];
    for (int h = 0; h <= G; ++h) sp->bound[h] = bounds[h];
    make_geometry(bounds[rank + 1] - bounds[rank], dtype, g);
    return SPEC_OK;
}

int shard_workspace(const void *ws, size_t bytes, const ShardWsLayout &l) {
    if (!ws) return SPEC_ERR_INVALID_ARG;
    if (bytes < l.total) return SPEC_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SPEC_ERR_ALIGNMENT;
    return SPEC_OK;
}

struct ShardWs {
    int *counters;
    float2 *part;
    float *resid;
    ShardSeq *seq;
};

ShardWs shard_ws_ptrs(void *ws, const ShardWsLayout &l) {
    unsigned char *p = static_cast<unsigned char *>(ws);
    return ShardWs{reinterpret_cast<int *>(p), reinterpret_cast<float2 *>(p + l.part),
                   reinterpret_cast<float *>(p + l.resid), reinterpret_cast<ShardSeq *>(p + l.seq)};
}

template <int DT>
int launch_shard_stats(const void *target, const void *draft, const int32_t *tokens, const float *temperature, int B,
                       const int32_t *k_offsets, const ShardSpec &sp, const Geometry &g, spec_shard_stat_t *out,
                       const ShardWs &w, const DeviceState &st, cudaStream_t stream) {
    int ns, per_sm;
    size_t smem;
    pick_ring(st, B, &ns, &smem, &per_sm);
    if (ns == 0) return SPEC_ERR_INVALID_ARG;
    // the call's first kernel: launched early behind the stream's previous
    // kernel, it waits for it before reading the inputs (wait_first)
    if (!cuda_ok(launch_k(true, stats_kernel<DT, kModeShard>, dim3(st.sms * per_sm), dim3(kThreads), smem, stream,
                          target, draft, temperature, k_offsets, B, g, ns, w.part, w.counters,
                          static_cast<int *>(nullptr), static_cast<const int *>(nullptr),
                          static_cast<const int *>(nullptr), 0, 1, static_cast<PairRec *>(nullptr), 0),
                 "launch stats_kernel (shard)") ||
        !cuda_ok(launch_k(true, shard_row_kernel<DT>, dim3(B), dim3(256), 0, stream, target,
                          draft, tokens, temperature, k_offsets, B, g, sp.v0, static_cast<const float2 *>(w.part),
                          out, w.counters),
                 "launch shard_row_kernel"))
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

}  // namespace specv

using namespace specv;

extern "C" {

size_t spec_shard_workspace_bytes(int B, int Vs, int dtype) {
    if (check_common(B, Vs, dtype) != SPEC_OK) return 0;
    Geometry g;
    make_geometry(Vs, dtype, &g);
    return shard_ws_layout(std::max(B, 1), g).total;
}

int spec_shard_stats(const void *target_shard, const void *draft_shard, const int32_t *draft_tokens,
                     const float *temperature, int B, const int32_t *k_offsets, const int32_t *shard_bounds, int G,
                     int rank, int dtype, spec_shard_stat_t *out_stats, void *workspace, size_t workspace_bytes,
                     void *stream) {
    ShardSpec sp;
    Geometry g;
    int rc = shard_setup(B, shard_bounds, G, rank, dtype, &sp, &g);
    if (rc != SPEC_OK) return rc;
    if (B == 0) return SPEC_OK;
    if (!target_shard || !draft_shard || !draft_tokens || !temperature || !k_offsets || !out_stats)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned16(target_shard) || !aligned16(draft_shard)) return SPEC_ERR_ALIGNMENT;
    const ShardWsLayout l = shard_ws_layout(B, g);
    rc = shard_workspace(workspace, workspace_bytes, l);
    if (rc != SPEC_OK) return rc;
    int dev;
    DeviceState *st = shard_device_state(&dev);
    if (!st) return SPEC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // (the ticket words: zero in a zero-filled workspace, and every
    // stats_kernel launch leaves them at zero)
    const ShardWs w = shard_ws_ptrs(workspace, l);
    if (dtype == SPEC_F32)
        return launch_shard_stats<SPEC_F32>(target_shard, draft_shard, draft_tokens, temperature, B, k_offsets, sp, g,
                                            out_stats, w, *st, s);
    return launch_shard_stats<SPEC_BF16>(target_shard, draft_shard, draft_tokens, temperature, B, k_offsets, sp, g,
                                         out_stats, w, *st, s);
}

int spec_shard_decide(const void *target_shard, const void *draft_shard, const spec_shard_stat_t *all_stats,
                      const int32_t *draft_tokens, const float *u_accept, const float *temperature, int B,
                      const int32_t *k_offsets, const int32_t *shard_bounds, int G, int rank, int dtype,
                      int32_t *out_tokens, int32_t *out_num_accepted, double *out_mass, void *workspace,
                      size_t workspace_bytes, void *stream) {
    ShardSpec sp;
    Geometry g;
    int rc = shard_setup(B, shard_bounds, G, rank, dtype, &sp, &g);
    if (rc != SPEC_OK) return rc;
    if (B == 0) return SPEC_OK;
    if (!target_shard || !draft_shard || !all_stats || !draft_tokens || !u_accept || !temperature || !k_offsets ||
        !out_tokens || !out_num_accepted || !out_mass)
        return SPEC_ERR_INVALID_ARG;
    // records are read as one 16-byte vector each
    if (!aligned16(target_shard) || !aligned16(draft_shard) || !aligned16(all_stats)) return SPEC_ERR_ALIGNMENT;
    const ShardWsLayout l = shard_ws_layout(B, g);
    rc = shard_workspace(workspace, workspace_bytes, l);
    if (rc != SPEC_OK) return rc;
    int dev;
    if (!shard_device_state(&dev)) return SPEC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const ShardWs w = shard_ws_ptrs(workspace, l);
    const cudaError_t e =
        dtype == SPEC_F32
            ? launch_k(true, shard_decide_kernel<SPEC_F32>, dim3(B), dim3(256), 0, s, target_shard, draft_shard,
                       all_stats, draft_tokens, u_accept, temperature, k_offsets, B, g, sp,
                       static_cast<const float2 *>(w.part), w.resid, w.seq, out_tokens, out_num_accepted, out_mass,
                       w.counters)
            : launch_k(true, shard_decide_kernel<SPEC_BF16>, dim3(B), dim3(256), 0, s, target_shard, draft_shard,
                       all_stats, draft_tokens, u_accept, temperature, k_offsets, B, g, sp,
                       static_cast<const float2 *>(w.part), w.resid, w.seq, out_tokens, out_num_accepted, out_mass,
                       w.counters);
    return cuda_ok(e, "launch shard_decide_kernel") ? SPEC_OK : SPEC_ERR_CUDA;
}

int spec_shard_draw(const void *target_shard, const void *draft_shard, const double *all_mass,
                    const float *u_resample, int B, const int32_t *k_offsets, const int32_t *shard_bounds, int G,
                    int rank, int dtype, int32_t *out_tokens, void *workspace, size_t workspace_bytes,
                    void *stream) {
    ShardSpec sp;
    Geometry g;
    int rc = shard_setup(B, shard_bounds, G, rank, dtype, &sp, &g);
    if (rc != SPEC_OK) return rc;
    if (B == 0) return SPEC_OK;
    if (!target_shard || !draft_shard || !all_mass || !u_resample || !k_offsets || !out_tokens)
        return SPEC_ERR_INVALID_ARG;
    // all_mass is read as 16-byte pairs
    if (!aligned16(target_shard) || !aligned16(draft_shard) || !aligned16(all_mass)) return SPEC_ERR_ALIGNMENT;
    const ShardWsLayout l = shard_ws_layout(B, g);
    rc = shard_workspace(workspace, workspace_bytes, l);
    if (rc != SPEC_OK) return rc;
    int dev;
    if (!shard_device_state(&dev)) return SPEC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const ShardWs w = shard_ws_ptrs(workspace, l);
    const cudaError_t e =
        dtype == SPEC_F32
            ? launch_k(true, shard_draw_kernel<SPEC_F32>, dim3(B), dim3(kDrawThreads), 0, s, target_shard, draft_shard,
                       all_mass, u_resample, k_offsets, B, g, sp, static_cast<const float2 *>(w.part),
                       static_cast<const float *>(w.resid), static_cast<const ShardSeq *>(w.seq), out_tokens)
            : launch_k(true, shard_draw_kernel<SPEC_BF16>, dim3(B), dim3(kDrawThreads), 0, s, target_shard, draft_shard,
                       all_mass, u_resample, k_offsets, B, g, sp, static_cast<const float2 *>(w.part),
                       static_cast<const float *>(w.resid), static_cast<const ShardSeq *>(w.seq), out_tokens);
    return cuda_ok(e, "launch shard_draw_kernel") ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"
