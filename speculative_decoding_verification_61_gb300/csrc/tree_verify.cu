// tree_verify.cu -- GB300 (sm_103a) tree (multi-candidate) verify and tree
// drafting, behind the C ABI of include/spec_verify.h.
//
// The pages draw candidate trees (docs.ifdog.com "投机解码", 进阶方案:
// Medusa and EAGLE verify a tree of drafted candidates in one target
// forward) but give no acceptance rule for them.  The rule implemented is
// the plainest lossless extension of the single-candidate test of
// 投机解码的三步流程 step 3 (bbs.huaweicloud.com 二.1-二.2) to several
// candidates drawn i.i.d. from one draft distribution: at node u (target
// distribution p, draft distribution q, from u's rows), u's children are
// tried in ascending node order; child j is accepted iff
// u_accept[child] < min(1, p^(j-1)(x)/q(x)), p^(0) = p, and each rejection
// replaces p by norm(max(0, p - q)).  An accepted child becomes u.  When
// every child is rejected, one token is drawn from the last residual at
// u_resample[u] by inverse CDF; a leaf draws the bonus token from its p.
// Greedy (T = 0): the first child whose token is argmax p is accepted, else
// argmax p is emitted.
//
// Pipeline of one spec_tree_verify call (all on the caller's stream):
//   1. tree_setup_kernel  warp per sequence: checks the parent array and
//                         lists the internal nodes (the draft rows needed);
//   2. stats_kernel       (tree mode) streams every node's target row and
//                         the internal nodes' draft rows once, to sub-chunk
//                         partials, as in the chain verify;
//   3. tree_walk_kernel   a cluster of two CTAs per sequence: a prologue
//                         (the parent array checked and the internal nodes
//                         listed again in the walk itself) combines every
//                         node's partials and loads each child's logits;
//                         the walk from the root then tests a node's
//                         children in order and, after each rejection,
//                         makes one pass over the node's two rows for the
//                         residual mass, each CTA over half the sub-chunks
//                         (the rows are prefetched into L2 at the first
//                         rejection, so later passes hit L2), the halves'
//                         sums meeting through a counter; the last draw
//                         locates the sub-chunk from the pass's
//                         per-sub-chunk masses and scans it.
// spec_tree_draft_sample runs the setup, stats_kernel over the internal
// nodes' draft rows, and tree_draft_select_kernel (warp per node: its token
// from its parent's draft row).

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "host_common.h"
#include "verify_common.cuh"

namespace specv {

// ================================================================== setup
// Warp per sequence (<= kMaxTreeNodes nodes, two per lane): a sequence
// whose parent array is not a tree in topological order (root first with
// parent -1, every other node's parent an earlier node of the sequence)
// gets nint = -1; otherwise nint = its internal nodes (nodes with a child)
// and tint[b * kMaxTreeNodes + j] = the j-th of them (global index,
// ascending).  Sequences whose node count is out of range are left to the
// whole-call check of the other kernels.  pair[b] (if given) is zeroed for
// the walk.
__global__ void __launch_bounds__(256) tree_setup_kernel(const int *__restrict__ node_offsets,
                                                         const int *__restrict__ parent, int B, int N,
                                                         int *__restrict__ nint, int *__restrict__ tint,
                                                         int *__restrict__ pair) {
    // the call's first kernel, launched early behind the stream's previous
    // kernel: wait for it before reading the inputs or writing the workspace
    grid_dependency_wait();
    const int b = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = lane_id();
    if (b >= B) return;
    if (lane == 0 && pair) pair[b] = 0;  // the walk's meeting counter of this tree
    const int g0 = node_offsets[b];
    const int n = node_offsets[b + 1] - g0;
    if (n < 1 || n > kMaxTreeNodes || g0 < 0 || g0 + n > N) {
        if (lane == 0) nint[b] = -1;
        return;
    }
    const int i0 = lane, i1 = lane + 32;
    auto local_parent = [&](int i) -> int {
        if (i >= n) return -2;
        const int pa = parent[g0 + i];
        return pa < 0 ? -1 : pa - g0;
    };
    const int p0 = local_parent(i0), p1 = local_parent(i1);
    auto valid = [&](int i, int p) { return i >= n || (i == 0 ? p == -1 : (p >= 0 && p < i)); };
    if (!__all_sync(0xffffffffu, valid(i0, p0) && valid(i1, p1))) {
        if (lane == 0) nint[b] = -1;
        return;
    }
    // internal nodes: those that are some node's parent
    bool int0 = false, int1 = false;
    for (int t = 0; t < n; ++t) {
        const unsigned m0 = __ballot_sync(0xffffffffu, p0 == t);
        const unsigned m1 = __ballot_sync(0xffffffffu, p1 == t);
        if (m0 | m1) {
            int0 |= (t == i0);
            int1 |= (t == i1);
        }
    }
    const unsigned long long m = (static_cast<unsigned long long>(__ballot_sync(0xffffffffu, int1)) << 32) |
                                 __ballot_sync(0xffffffffu, int0);
    if (int0) tint[b * kMaxTreeNodes + __popcll(m & ((1ull << i0) - 1ull))] = g0 + i0;
    if (int1) tint[b * kMaxTreeNodes + __popcll(m & ((1ull << i1) - 1ull))] = g0 + i1;
    if (lane == 0) nint[b] = __popcll(m);
}

// ================================================================== walk
#ifndef SPEC_TREE_PACKED
#define SPEC_TREE_PACKED 1
#endif
// CTAs per tree: with 2, a tree is walked by a cluster of two CTAs on two
// SMs; both take every decision (from the same data, so the same one) and
// each makes half of every pass over the node's rows.
#ifndef SPEC_TREE_CTAS
#define SPEC_TREE_CTAS 2
#endif
constexpr int kTreeCtas = SPEC_TREE_CTAS;
static_assert(kTreeCtas == 1 || kTreeCtas == 2 || kTreeCtas == 4, "one, two or four CTAs per tree");
// four CTAs per tree: 256 threads each, two per SM (a tree's quarter-pass
// shares its SM with another tree's CTA, and has it to itself while that
// tree tests, draws or has finished)
constexpr int kWalkThreads = kTreeCtas == 4 ? 256 : 512;
constexpr int kWalkMinBlocks = kTreeCtas == 4 ? 2 : 1;
constexpr int kWalkWarps = kWalkThreads / 32;

struct TreeWalkSmem {
    int par[kMaxTreeNodes];     // local parent of each node (-1: root)
    int tok[kMaxTreeNodes];     // drafted token of each node
    // per node i, from the prologue (read only when the walk visits i)
    float zt[kMaxTreeNodes];    // i's token's logit in its parent's target row
    float zd[kMaxTreeNodes];    // and in its parent's draft row
    float ua[kMaxTreeNodes];    // u_accept of i
    double Lt[kMaxTreeNodes];   // log2-domain log-sum-exp of i's target row
    double Ld[kMaxTreeNodes];   // and of its draft row (internal nodes)
    float M[kMaxTreeNodes];     // max of i's target row (z * c)
    float lth[kMaxTreeNodes], ltl[kMaxTreeNodes];  // Lt as an fp32 hi/lo pair
    float ldh[kMaxTreeNodes], ldl[kMaxTreeNodes];  // Ld likewise
    int am[kMaxTreeNodes];      // greedy: arg-max of i's target row
    int ok[kMaxTreeNodes];      // i's target row is valid
    int okd[kMaxTreeNodes];     // i's draft row is valid (or not needed)
    int path[kMaxTreeNodes];    // accepted tokens
    int isint[kMaxTreeNodes];   // i has a child (an internal node)
    int ilist[kMaxTreeNodes];   // the internal nodes in ascending order
    int nil;                    // their count
    double t;                   // residual level of the current p at the node (0: p itself)
    float S;                    // its mass S(t)
    int next;                   // accepted child (local index) or -1
    int zpos;                   // the last residual mass was > 0
    int token;                  // the drawn token
    DrawSmem ds;                // block-level draws (CTA 0)
};

// The residual chain in closed form.  With a = p and b = q of the node,
// t_0 = 0 and S(t) = sum_v max(0, a_v - t b_v), the distribution after k
// rejections is p_k = max(0, a - t_k b) / S(t_k), t_(k+1) = t_k + S(t_k)
// (induction on norm(max(0, p_(k-1) - q)); p_0 = a, S(0) = 1, t_1 = 1).
// One element's a and b at the node; operations pinned, so that a
// candidate's test, the passes and the final scan compute identical bits.
__device__ __forceinline__ void tree_pq(float zt, float zd, float c, float lth, float ltl, float ldh, float ldl,
                                        float *a, float *bq) {
    *a = ex2(__fsub_rn(__fmaf_rn(zt, c, -lth), ltl));
    *bq = ex2(__fsub_rn(__fmaf_rn(zd, c, -ldh), ldl));
}

// Weight of one element at level t: max(0, a - t b) (t = 0: a itself).
struct TreeWeight {
    float c, lth, ltl, ldh, ldl, t;
    __device__ __forceinline__ float operator()(float zt, float zd) const {
        float pa, pb;
        tree_pq(zt, zd, c, lth, ltl, ldh, ldl, &pa, &pb);
        return fmaxf(__fmaf_rn(-t, pb, pa), 0.0f);
    }
};

// TreeWeight on two elements at once in packed fp32: lane for lane the same
// operations (x - y is rounded exactly as x + (-y)), so the same bits.
struct TreeWeight2 {
    float2 c2, nlth2, nltl2, nldh2, nldl2, nt2;
    __device__ __forceinline__ explicit TreeWeight2(const TreeWeight &w)
        : c2(make_float2(w.c, w.c)), nlth2(make_float2(-w.lth, -w.lth)), nltl2(make_float2(-w.ltl, -w.ltl)),
          nldh2(make_float2(-w.ldh, -w.ldh)), nldl2(make_float2(-w.ldl, -w.ldl)), nt2(make_float2(-w.t, -w.t)) {}
    __device__ __forceinline__ float2 operator()(float2 zt, float2 zd) const {
        const float2 at = fadd2(ffma2(zt, c2, nlth2), nltl2);
        const float2 ad = fadd2(ffma2(zd, c2, nldh2), nldl2);
        const float2 w = ffma2(nt2, make_float2(ex2(ad.x), ex2(ad.y)), make_float2(ex2(at.x), ex2(at.y)));
        return make_float2(fmaxf(w.x, 0.0f), fmaxf(w.y, 0.0f));
    }
};

// One pass of the whole block over the current node's two rows: the mass of
// W over every sub-chunk, to rm[sc].  Warp w takes sub-chunks w, w + 16,
// ...; the loads of its next sub-chunk are issued before the current one is
// reduced, so that they overlap.  (Not inlined: the walk's state would
// otherwise share its registers.)
template <int DT>
__device__ __noinline__ void tree_pass(const unsigned char *rt, const unsigned char *rd, const Geometry &g, const TreeWeight &W,
                          float *rm, int sc_begin, int sc_end, float2 *wpart) {
    using E = Elem<DT>;
    const int lane = lane_id();
    auto load = [&](int sc, uint4 (&xt)[4], uint4 (&xd)[4]) -> int {
        int a, e1;
        sub_range(g, sc, &a, &e1);
        const int nvec = (e1 - a) / E::kPerVec;  // <= 128
        const uint4 *pt = reinterpret_cast<const uint4 *>(rt + static_cast<int64_t>(a) * E::kBytes);
        const uint4 *pd = reinterpret_cast<const uint4 *>(rd + static_cast<int64_t>(a) * E::kBytes);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = lane + 32 * j;
            if (i < nvec) {
                xt[j] = ld_stream(pt + i);
                xd[j] = ld_stream(pd + i);
            }
        }
        return nvec;
    };
#if SPEC_TREE_PACKED
    const TreeWeight2 W2(W);
    auto mass = [&](const uint4 (&xt)[4], const uint4 (&xd)[4], int nvec) -> float {
        float2 acc0 = make_float2(0.0f, 0.0f), acc1 = acc0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (lane + 32 * j >= nvec) continue;
#pragma unroll
            for (int p = 0; p < E::kPairs; ++p) {
                const float2 w2 = W2(E::pair(xt[j], p), E::pair(xd[j], p));
                if (p & 1) acc1 = fadd2(acc1, w2); else acc0 = fadd2(acc0, w2);
            }
        }
        return warp_sum_f((acc0.x + acc0.y) + (acc1.x + acc1.y));
    };
#else
    auto mass = [&](const uint4 (&xt)[4], const uint4 (&xd)[4], int nvec) -> float {
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (lane + 32 * j >= nvec) continue;
            float x1[E::kPerVec], x2[E::kPerVec];
            E::unpack(xt[j], x1);
            E::unpack(xd[j], x2);
#pragma unroll
            for (int q = 0; q < E::kPerVec; ++q) acc += W(x1[q], x2[q]);
        }
        return warp_sum_f(acc);
    };
#endif
    int sc = sc_begin + warp_id();
    if (sc >= sc_end) {
        if (lane == 0) wpart[warp_id()] = make_float2(0.0f, 0.0f);
        return;
    }
    Acc2 wacc;  // this warp's masses in sub-chunk order (lane 0)
    uint4 ct[4], cd[4];
    int nc = load(sc, ct, cd);
    for (;;) {
        const int sn = sc + kWalkWarps;
        uint4 nt[4], nd[4];
        int nn = 0;
        if (sn < sc_end) nn = load(sn, nt, nd);
        const float sum = mass(ct, cd, nc);
        if (lane == 0) {
            rm[sc] = sum;
            wacc.add(sum);
        }
        if (sn >= sc_end) break;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            ct[j] = nt[j];
            cd[j] = nd[j];
        }
        nc = nn;
        sc = sn;
    }
    // (the masses reach the other CTAs of the tree through the meeting's
    // release: the CTA barrier before it, then thread 0's release-add)
    if (lane == 0) wpart[warp_id()] = make_float2(wacc.hi, wacc.lo);
}

__device__ __forceinline__ unsigned cluster_ctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Meeting point of a tree's CTAs after a pass, run by thread 0 of each CTA
// once the CTA's masses and warp partials are written: the CTA's partial
// T_cr = its warps' partials added in order; with two CTAs it publishes T_cr
// (ptot: this pass's two slots), adds one to the tree's counter and waits
// (bounded) until the counter reaches `target`, then S = T_0 + T_1 added
// in rank order, so both CTAs get the same bits.  On a time-out the status
// word gets SPEC_ERR_TIMEOUT and false is returned.  Counter and partials
// are in global memory: no CTA touches the other's shared memory.
__device__ bool tree_meet_sum(int *cnt, int target, float2 *ptot, int cr, const float2 *wpart, int *status,
                              float *S_out) {
    Acc2 part;
    for (int w = 0; w < kWalkWarps; ++w) {
        part.add(wpart[w].x);
        part.add(wpart[w].y);
    }
    if (kTreeCtas == 1) {
        *S_out = part.value();
        return true;
    }
    const float2 mine = make_float2(part.hi, part.lo);
    ptot[cr] = mine;
    // release: this CTA's masses (written before the caller's barrier) and
    // its partial, to whoever acquires the count
    red_add_release_gpu(cnt, 1);
    const uint64_t t0 = global_timer_ns();
    while (ld_acquire_gpu(cnt) < target) {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            set_status(status, SPEC_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(64);
    }
    Acc2 tot;
    for (int r = 0; r < kTreeCtas; ++r) {
        const float2 v = r == cr ? mine : __ldcg(ptot + r);
        tot.add(v.x);
        tot.add(v.y);
    }
    *S_out = tot.value();
    return true;
}

// Block per sequence.  Partials: target row g at slot g, draft row g at
// slot N + g (stats_kernel tree mode); rm: this sequence's n_sub residual
// masses (scratch).  Data errors (a bad temperature, token or parent array,
// or an invalid needed row) make the whole sequence -1, as in the chain
// verify; an invalid node_offsets array fails the whole call.
template <int DT>
__global__ void __launch_bounds__(kWalkThreads, kWalkMinBlocks) tree_walk_kernel(
    const void *__restrict__ target, const void *__restrict__ draft, const int *__restrict__ node_offsets,
    const int *__restrict__ parent, const int32_t *__restrict__ tokens, const float *__restrict__ u_accept,
    const float *__restrict__ u_resample, const float *__restrict__ temperature, int B, int N, Geometry g,
    const float2 *__restrict__ part, const int *__restrict__ nint, const int *__restrict__ tint,
    float *__restrict__ resid, int *__restrict__ pair, float2 *__restrict__ ptot, int *__restrict__ counters,
    int32_t *__restrict__ out_tokens,
    int32_t *__restrict__ out_num, int32_t *__restrict__ out_last) {
    using E = Elem<DT>;
    __shared__ TreeWalkSmem sm;
    __shared__ int s_meet;                   // the last meeting succeeded (thread 0 writes)
    __shared__ float2 s_wpart[kWalkWarps];   // the last pass's warp partials
    // CTA cr of the tree's cluster (0 with one CTA per tree); CTA 0 draws
    // and writes the outputs
    const int cr = kTreeCtas > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int b = blockIdx.x / kTreeCtas;
    const int lane = lane_id(), warp = warp_id(), tid = threadIdx.x;

    // --- inputs only (written before this call) --------------------------
    // the same node_offsets check as stats_kernel: only with it do the row
    // indices below stay inside the caller's buffers
    int bad = 0;
    for (int i = tid; i <= B; i += blockDim.x) {
        const int v = node_offsets[i];
        if (i == 0) {
            bad |= v != 0;
        } else {
            const int nn = v - node_offsets[i - 1];
            bad |= (nn < 1 || nn > kMaxTreeNodes);
        }
        if (i == B) bad |= v != N;
    }
    bad = __syncthreads_or(bad);
    if (bad) {
        grid_dependency_wait();
        if (tid == 0 && cr == 0) {
            out_num[b] = -1;
            if (out_last) out_last[b] = -1;
            if (b == 0) set_status(counters + kStatus, SPEC_ERR_INVALID_ARG);
        }
        return;
    }
    const int g0 = node_offsets[b], n = node_offsets[b + 1] - g0;
    const float c = temp_scale(temperature[b]);
    const bool greedy = c == 0.0f;
    // a greedy walk makes no pass: CTA 0 does it alone
    if (greedy && cr != 0) return;
    const int V = g.V;
    bool tokbad = false, parbad = false;
    if (tid < kMaxTreeNodes) sm.isint[tid] = 0;
    if (tid < n) {
        const int pa = parent[g0 + tid];
        const int lp = pa < 0 ? -1 : pa - g0;
        sm.par[tid] = lp;
        // the setup kernel's rule: the root first (parent -1), every other
        // node's parent an earlier node of the tree
        parbad = tid == 0 ? lp != -1 : (lp < 0 || lp >= tid);
        const int x = tokens[g0 + tid];
        sm.tok[tid] = x;
        tokbad = tid > 0 && (x < 0 || x >= V);
    }
    tokbad = __syncthreads_or(tokbad);
    // the internal nodes (those with a child) in ascending order, as the
    // setup kernel lists them for the streaming pass, found here from the
    // parents so that the prologue's loads wait on nothing the setup kernel
    // wrote (its count, read below, still marks a tree it found invalid)
    if (tid > 0 && tid < n && !parbad) sm.isint[sm.par[tid]] = 1;
    parbad = __syncthreads_or(parbad);
    if (warp == 0) {
        const bool f0 = lane < n && sm.isint[lane] != 0, f1 = lane + 32 < n && sm.isint[lane + 32] != 0;
        const unsigned m0 = __ballot_sync(0xffffffffu, f0), m1 = __ballot_sync(0xffffffffu, f1);
        const unsigned below = (1u << lane) - 1u;
        if (f0) sm.ilist[__popc(m0 & below)] = lane;
        if (f1) sm.ilist[__popc(m0) + __popc(m1 & below)] = lane + 32;
        if (lane == 0) sm.nil = __popc(m0) + __popc(m1);
    }
    __syncthreads();
    grid_dependency_wait();
    const int nint_b = nint[b];  // -1: the setup kernel found the tree invalid

    bool err = (c != c) || tokbad || parbad;
    int u = 0, nacc = 0, final_token = -1;
    // per-sub-chunk masses, two buffers used in turn by successive passes
    // (a CTA may start the next pass while the other still reads the last)
    float *const rm_base = resid + static_cast<int64_t>(b) * 2 * g.n_sub;
    int passes = 0;
    float *rm = rm_base;
    // this CTA's share of every pass: a contiguous half of the sub-chunks
    const int half = (g.n_sub + kTreeCtas - 1) / kTreeCtas;
    const int sc0 = min(g.n_sub, cr * half), sc1 = min(g.n_sub, sc0 + half);
    int *const meet_cnt = pair + b;
    float2 *const ptot_b = ptot + static_cast<int64_t>(b) * 2 * kTreeCtas;
    // One pass over the node's rows at level W.t; afterwards thread 0 holds
    // the pass's whole mass in *S0 and s_meet says whether the meeting of
    // the tree's CTAs succeeded (published by the caller's next barrier).
    auto pass = [&](const unsigned char *prt, const unsigned char *prd, const TreeWeight &W, float *S0) {
        rm = rm_base + (passes & 1) * g.n_sub;
        tree_pass<DT>(prt, prd, g, W, rm, sc0, sc1, s_wpart);
        ++passes;
        __syncthreads();  // this CTA's masses and warp partials are written
        if (tid == 0)
            s_meet = tree_meet_sum(meet_cnt, kTreeCtas * passes, ptot_b + (passes & 1) * kTreeCtas, cr, s_wpart,
                                   counters + kStatus, S0);
    };
    const int64_t rb = static_cast<int64_t>(V) * E::kBytes;
    // this CTA's share of a node's two rows to L2 in 32 KB bulk prefetches
    // (one warp; sub-chunk bounds are 16-byte aligned), so that the passes
    // over them wait on L2, not on DRAM
    auto prefetch_rows = [&](const unsigned char *prt, const unsigned char *prd) {
        if (!SPEC_RESID_PREFETCH || sc0 >= sc1) return;
        int e_lo, e_hi, unused;
        sub_range(g, sc0, &e_lo, &unused);
        sub_range(g, sc1 - 1, &unused, &e_hi);
        const int64_t lo = static_cast<int64_t>(e_lo) * E::kBytes, hi = static_cast<int64_t>(e_hi) * E::kBytes;
        constexpr int64_t kPiece = 32768;
        const unsigned char *r0 = (lane & 1) ? prd : prt;
        for (int64_t off = lo + static_cast<int64_t>(lane >> 1) * kPiece; off < hi; off += 16 * kPiece)
            bulk_prefetch_l2(r0 + off, static_cast<uint32_t>(min(kPiece, hi - off)));
    };

    // --- prologue: the statistics of every node's rows (the n target rows,
    // then the internal nodes' draft rows; each warp takes two rows at a
    // time, both rows' partials loaded before either is combined) and every
    // child's logits at its token, so that the walk itself only tests
    if (!err) {
        if (tid < n) {
            sm.ua[tid] = u_accept[g0 + tid];
            // a leaf's draft row is not needed; an internal node's okd is
            // written by its row's combine below (no other write, no race)
            if (!sm.isint[tid]) sm.okd[tid] = 1;
        }
        // every child's logits at its token (two loads from HBM each): issued
        // now, stored to shared memory after the rows' combine below
        float zt_own = 0.0f, zd_own = 0.0f;
        if (tid < n && tid > 0 && !greedy) {
            const int64_t prow = g0 + sm.par[tid];
            zt_own = E::load1(target, prow * V + sm.tok[tid]);
            zd_own = E::load1(draft, prow * V + sm.tok[tid]);
        }
        const int items = n + (greedy ? 0 : sm.nil);
        // partials of item k: target row of node k, or the draft row of the
        // (k - n)-th internal node
        auto item_part = [&](int k) -> const float2 * {
            const int64_t slot = k < n ? static_cast<int64_t>(g0) + k
                                       : static_cast<int64_t>(N) + g0 + sm.ilist[k - n];
            return part + slot * g.n_sub;
        };
        auto store_soft = [&](int k, bool ok, float M, float S) {
            if (lane != 0) return;
            if (k < n) {
                sm.ok[k] = ok;
                if (ok) {
                    const double Lt = lse2(M, S);
                    sm.M[k] = M;
                    sm.Lt[k] = Lt;
                    sm.lth[k] = static_cast<float>(Lt);
                    sm.ltl[k] = static_cast<float>(Lt - static_cast<double>(sm.lth[k]));
                }
            } else {
                const int i = sm.ilist[k - n];
                sm.okd[i] = ok;
                if (ok) {
                    const double Ld = lse2(M, S);
                    sm.Ld[i] = Ld;
                    sm.ldh[i] = static_cast<float>(Ld);
                    sm.ldl[i] = static_cast<float>(Ld - static_cast<double>(sm.ldh[i]));
                }
            }
        };
        if (greedy) {
            for (int k = warp; k < n; k += kWalkWarps) {
                const int am = warp_combine_arg(item_part(k), g.n_sub);
                if (lane == 0) {
                    sm.am[k] = am;
                    sm.ok[k] = am >= 0;
                }
            }
        } else {
            for (int k0 = warp; k0 < items; k0 += 2 * kWalkWarps) {
                const int k1 = k0 + kWalkWarps;
                float2 ca[kPartCache], cb[kPartCache];
                const float2 *pa = item_part(k0);
                const float2 *pb = k1 < items ? item_part(k1) : pa;
                load_parts(pa, g.n_sub, ca);
                if (k1 < items) load_parts(pb, g.n_sub, cb);
                float M, S;
                bool ok = combine_soft(ca, pa, g.n_sub, &M, &S);
                store_soft(k0, ok, M, S);
                if (k1 < items) {
                    ok = combine_soft(cb, pb, g.n_sub, &M, &S);
                    store_soft(k1, ok, M, S);
                }
            }
        }
        if (tid < n && tid > 0 && !greedy) {
            sm.zt[tid] = zt_own;
            sm.zd[tid] = zd_own;
        }
        __syncthreads();
    }
    // the setup kernel's verdict on the parent array (the rule of parbad)
    err = err || nint_b < 0;

    for (int step = 0; !err && step < n; ++step) {
        const int64_t urow = g0 + u;
        // children of u, in ascending node order (the same mask in every warp)
        const int pa0 = lane < n ? sm.par[lane] : -2, pa1 = lane + 32 < n ? sm.par[lane + 32] : -2;
        const unsigned long long kids = (static_cast<unsigned long long>(__ballot_sync(0xffffffffu, pa1 == u)) << 32) |
                                        __ballot_sync(0xffffffffu, pa0 == u);
        const bool leaf = kids == 0ull;
        if (!sm.ok[u] || (!greedy && !leaf && !sm.okd[u])) {
            err = true;
            break;
        }
        if (greedy) {
            // the first child whose token is argmax p
            const int am = sm.am[u];
            const int t0 = lane < n ? sm.tok[lane] : -1, t1 = lane + 32 < n ? sm.tok[lane + 32] : -1;
            const unsigned long long match =
                kids & ((static_cast<unsigned long long>(__ballot_sync(0xffffffffu, t1 == am)) << 32) |
                        __ballot_sync(0xffffffffu, t0 == am));
            if (!match) {
                final_token = am;
                break;
            }
            const int ch = __ffsll(static_cast<long long>(match)) - 1;
            if (tid == 0) sm.path[nacc] = sm.tok[ch];
            ++nacc;
            u = ch;
            __syncthreads();  // sm is rewritten for the next node
            continue;
        }
        if (leaf) {
            // bonus token from p_u, as the chain's bonus draw (the whole of CTA 0)
            if (cr == 0) {
                const int tk = block_draw_row<DT>(target, urow, part + urow * g.n_sub, g, c, sm.M[u],
                                                  u_resample[urow], sm.ds);
                if (tid == 0) sm.token = tk;
            }
            __syncthreads();
            final_token = sm.token;
            break;
        }
        // the children in order
        const unsigned char *rt = static_cast<const unsigned char *>(target) + urow * rb;
        const unsigned char *rd = static_cast<const unsigned char *>(draft) + urow * rb;
        const TreeWeight base{c, sm.lth[u], sm.ltl[u], sm.ldh[u], sm.ldl[u], 0.0f};
        // the accept test of child ch, the jj-th tried (thread 0): its index
        // if accepted, else -1
        auto test = [&](int ch, int jj) -> int {
            const float zt = sm.zt[ch], zd = sm.zd[ch];
            float alpha;
            if (jj == 0) {
                // the first candidate: the log-domain ratio of the chain verify
                if (zt == -INFINITY) {
                    alpha = 0.0f;
                } else if (zd == -INFINITY) {
                    alpha = 1.0f;
                } else {
                    const double cd = static_cast<double>(c);
                    const double lr =
                        (static_cast<double>(zt) * cd - sm.Lt[u]) - (static_cast<double>(zd) * cd - sm.Ld[u]);
                    alpha = lr >= 0.0 ? 1.0f : exp2f(static_cast<float>(lr));
                }
            } else {
                // p_k(x) / q(x) = max(0, a - t b) / (S b) at the current level
                float pa, pb;
                tree_pq(zt, zd, c, sm.lth[u], sm.ltl[u], sm.ldh[u], sm.ldl[u], &pa, &pb);
                const float num = fmaxf(__fmaf_rn(-static_cast<float>(sm.t), pb, pa), 0.0f);
                alpha = (zd == -INFINITY || pb == 0.0f) ? (num > 0.0f ? 1.0f : 0.0f)
                                                        : fminf(1.0f, num / (sm.S * pb));
            }
            return sm.ua[ch] < alpha ? ch : -1;
        };
        unsigned long long rest = kids;  // the children not yet tried, lowest first
        if (tid == 0) {
            sm.t = 0.0;  // p itself
            sm.S = 1.0f;
            sm.next = test(__ffsll(static_cast<long long>(rest)) - 1, 0);
        }
        __syncthreads();
        int j = 0, next = -1;
        bool zero_last = false;
        for (;;) {
            if (sm.next >= 0) {
                next = sm.next;
                break;
            }
            // rejected: the next level t' = t + S(t), and one pass over u's
            // rows for S(t') and its per-sub-chunk masses
            if (j == 0 && warp == 0) prefetch_rows(rt, rd);  // at a node's first pass: the later ones hit L2
            const double tn = sm.t + static_cast<double>(sm.S);
            TreeWeight W = base;
            W.t = static_cast<float>(tn);
            float Sn = 0.0f;
            pass(rt, rd, W, &Sn);
            rest &= rest - 1ull;
            ++j;
            if (tid == 0 && s_meet) {
                // the new level (a mass that rounded to 0 leaves p as it was),
                // then the next child's test at it
                sm.zpos = Sn > 0.0f;
                if (Sn > 0.0f) {
                    sm.t = tn;
                    sm.S = Sn;
                }
                sm.next = rest ? test(__ffsll(static_cast<long long>(rest)) - 1, j) : -1;
            }
            __syncthreads();
            if (!s_meet) {
                err = true;
                break;
            }
            zero_last = !sm.zpos;
            if (!rest) break;
        }
        if (err) break;
        if (next >= 0) {
            if (tid == 0) sm.path[nacc] = sm.tok[next];
            ++nacc;
            u = next;
            __syncthreads();
            continue;
        }
        // every child rejected: draw from p_k = max(0, a - t b) / S at the
        // current level, whose masses the last pass left in rm (after a
        // mass that rounded to 0, they are computed again; at t = 0 the
        // draw is the bonus draw from the row's partials)
        TreeWeight W = base;
        W.t = static_cast<float>(sm.t);
        const bool from_partials = zero_last && sm.t == 0.0;
        if (zero_last && !from_partials) {
            float unused;
            pass(rt, rd, W, &unused);
            __syncthreads();
            if (!s_meet) {
                err = true;
                break;
            }
        }
        // the draw, by the whole of CTA 0: warp 0 locates the sub-chunk, the
        // block scans its elements
        if (cr == 0) {
            int tk = -1;
            if (from_partials) {
                tk = block_draw_row<DT>(target, urow, part + urow * g.n_sub, g, c, sm.M[u], u_resample[urow], sm.ds);
            } else {
                if (warp == 0) {
                    float w[kPartCache];
#pragma unroll
                    for (int q = 0; q < kPartCache; ++q)
                        w[q] = (lane + 32 * q < g.n_sub) ? __ldcg(rm + lane + 32 * q) : 0.0f;
                    auto wfar = [&](int i) -> float { return __ldcg(rm + i); };
                    F2 before, Z, tgt;
                    const int sc = warp_locate(g.n_sub, w, wfar, u_resample[urow], &before, &Z, &tgt);
                    if (lane == 0) {
                        sm.ds.sc = sc;
                        sm.ds.before = before;
                        sm.ds.target = tgt;
                    }
                }
                __syncthreads();
                const int sc = sm.ds.sc;
                if (sc >= 0) {
                    int a, e1;
                    sub_range(g, sc, &a, &e1);
                    tk = block_scan_elems<DT>(rt, rd, a, e1, W, sm.ds.before, sm.ds.target, sm.ds);
                }
            }
            if (tid == 0) sm.token = tk;
        }
        __syncthreads();
        final_token = sm.token;
        break;
    }
    // outputs (CTA 0): the accepted path, the drawn token, then -1
    if (cr != 0) return;
    for (int i = tid; i < n; i += blockDim.x) {
        int32_t o = -1;
        if (!err) o = i < nacc ? sm.path[i] : (i == nacc ? final_token : -1);
        out_tokens[g0 + i] = o;
    }
    if (tid == 0) {
        out_num[b] = err ? -1 : nacc;
        if (out_last) out_last[b] = err ? -1 : g0 + u;
    }
}

// ================================================================== self-check
// The bounded device-side waits, made to run out on purpose: one thread
// waits on an mbarrier that nothing arrives at (as a ring slot whose copy
// never lands), then meets on a counter that no other CTA completes (as a
// tree whose other CTA never arrives), then waits for an entry of the
// deferred epilogue's pair list that nobody lists while the decided count
// stays short (as a residual stream whose deciding CTA never runs).  Each
// wait gives up after its limit and the status word gets SPEC_ERR_TIMEOUT;
// the kernel then returns.
__global__ void selfcheck_wait_kernel(int *counters, int *never) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_barrier_init();
    const bool mbar_ok = mbar_wait_bounded(&bar, 0);
    if (!mbar_ok) set_status(counters + kStatus, SPEC_ERR_TIMEOUT);
    float2 wpart[kWalkWarps] = {};
    // the partials' slots are global memory, as in the walk: words 16..19
    float2 *ptot = reinterpret_cast<float2 *>(counters + 16);
    float S;
    // a count the single arrival of this CTA never reaches
    const bool meet_ok = tree_meet_sum(never, 2 * kTreeCtas, ptot, 0, wpart, counters + kStatus, &S);
    // the list and the decided count of a zero-filled block stay at 0; one
    // sequence is owed (the list's entries are never read)
    const bool pair_ok = wait_pair(counters, nullptr, 0, 1) >= 0;
    if (!pair_ok) set_status(counters + kStatus, SPEC_ERR_TIMEOUT);
    counters[8] = (mbar_ok ? 0 : 1) | (meet_ok ? 0 : 2) | (pair_ok ? 0 : 4);  // which waits gave up
    *never = 0;
}

// ================================================================== drafting
// A node's sequence (by bisection of the node offsets in shared memory),
// parent, temperature scale and drafting uniform.
struct TreeNodeIn {
    int lo, pa;
    float c, ud;
};

__device__ __forceinline__ TreeNodeIn tree_node_inputs(const int *s_no, int B, const int *__restrict__ parent,
                                                       const float *__restrict__ temperature,
                                                       const float *__restrict__ u_draft, int node) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_no[mid] <= node) lo = mid; else hi = mid - 1;
    }
    return TreeNodeIn{lo, parent[node], temp_scale(temperature[lo]), u_draft[node]};
}

// Warp per node (grid-stride): a non-root node's token from its parent's
// draft row (partials at slot parent, stats_kernel tree-draft mode):
// arg-max at T = 0, else the inverse-CDF draw at u_draft[node].  Roots,
// invalid sequences and invalid rows give -1.
template <int DT>
__global__ void __launch_bounds__(256) tree_draft_select_kernel(
    const void *__restrict__ draft, const int *__restrict__ node_offsets, const int *__restrict__ parent,
    const float *__restrict__ temperature, const float *__restrict__ u_draft, int B, int N, Geometry g,
    const float2 *__restrict__ part, const int *__restrict__ nint, int32_t *__restrict__ out,
    int *__restrict__ counters) {
    extern __shared__ int s_no[];  // [B + 1]
    __shared__ int s_bad;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int i = threadIdx.x; i <= B; i += blockDim.x) {
        const int v = node_offsets[i];
        s_no[i] = v;
        if (i == 0 && v != 0) s_bad = 1;
        if (i > 0) {
            const int nn = v - node_offsets[i - 1];
            if (nn < 1 || nn > kMaxTreeNodes) s_bad = 1;
        }
        if (i == B && v != N) s_bad = 1;
    }
    __syncthreads();
    const int lane = lane_id();
    const int nw = (gridDim.x * blockDim.x) >> 5;
    const int node0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    // a node's sequence, parent, temperature and uniform: the caller's
    // inputs, complete once the call's first kernel passed its wait, so the
    // first node's are read before this kernel's wait
    TreeNodeIn in{0, -1, 0.0f, 0.0f};
    if (!s_bad && node0 < N) in = tree_node_inputs(s_no, B, parent, temperature, u_draft, node0);
    grid_dependency_wait();
    grid_launch_dependents();
    if (s_bad) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(counters + kStatus, SPEC_ERR_INVALID_ARG);
        return;
    }
    for (int node = node0; node < N; node += nw) {
        if (node != node0) in = tree_node_inputs(s_no, B, parent, temperature, u_draft, node);
        const int lo = in.lo, pa = in.pa;
        const float c = in.c;
        int token = -1;
        // the partials of the parent's draft row (in the tree's range) are
        // requested with the setup kernel's verdict on the tree, not after it
        if (pa >= s_no[lo] && pa < node && c == c) {
            const int ni = nint[lo];
            const float2 *pr = part + static_cast<int64_t>(pa) * g.n_sub;
            if (c == 0.0f) {
                const int am = warp_combine_arg(pr, g.n_sub);
                if (ni >= 0) token = am;
            } else {
                float M, S;
                float2 pc[kPartCache];
                load_parts(pr, g.n_sub, pc);
                if (ni >= 0 && combine_soft(pc, pr, g.n_sub, &M, &S))
                    token = warp_draw_row<DT>(draft, pa, pr, pc, g, c, M, in.ud);
            }
        }
        if (lane == 0) out[node] = token;
    }
}

// ================================================================== host side
struct TreeWsLayout {
    size_t part, nint, tint, resid, pair, ptot, total;
};

// Counters (the common 256-byte block) | partials of N target and N draft
// rows | nint [B] | tint [B * kMaxTreeNodes] | residual masses, two buffers
// [B * 2 * n_sub] | the walk's meeting counters [B] | the CTAs' partial masses
// of a pass [B * 2 * kTreeCtas] (fp32 hi/lo pairs).
TreeWsLayout tree_ws_layout(int B, int N, const Geometry &g) {
    TreeWsLayout l;
    size_t off = kCountersBytes;
    l.part = off;
    off = align_up(off + static_cast<size_t>(2) * N * g.n_sub * sizeof(float2), 256);
    l.nint = off;
    off = align_up(off + static_cast<size_t>(B) * sizeof(int), 256);
    l.tint = off;
    off = align_up(off + static_cast<size_t>(B) * kMaxTreeNodes * sizeof(int), 256);
    l.resid = off;
    off = align_up(off + static_cast<size_t>(B) * 2 * g.n_sub * sizeof(float), 256);
    l.pair = off;
    off = align_up(off + static_cast<size_t>(B) * sizeof(int), 256);
    l.ptot = off;
    off = align_up(off + static_cast<size_t>(B) * 2 * kTreeCtas * sizeof(float2), 256);
    l.total = off;
    return l;
}

bool g_tree_init[kMaxDevices] = {};
std::mutex g_tree_mu;

// stats_kernel's tree modes in this translation unit: the opt-in dynamic
// shared memory, once per device.
template <int DT, int MODE>
bool tree_stats_attr(int smem_optin_raw) {
    cudaFuncAttributes fa{};
    if (!cuda_ok(cudaFuncGetAttributes(&fa, stats_kernel<DT, MODE>), "cudaFuncGetAttributes")) return false;
    return cuda_ok(cudaFuncSetAttribute(stats_kernel<DT, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        smem_optin_raw - static_cast<int>(fa.sharedSizeBytes)),
                   "cudaFuncSetAttribute(stats_kernel tree)");
}

DeviceState *tree_device_state(int *dev_out) {
    DeviceState *st = device_state(dev_out);
    if (!st) return nullptr;
    std::lock_guard<std::mutex> lock(g_tree_mu);
    if (!g_tree_init[*dev_out]) {
        int optin = 0;
        if (!cuda_ok(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, *dev_out),
                     "cudaDeviceGetAttribute"))
            return nullptr;
        if (!tree_stats_attr<SPEC_F32, kModeTree>(optin) || !tree_stats_attr<SPEC_F32, kModeTreeDraft>(optin) ||
            !tree_stats_attr<SPEC_BF16, kModeTree>(optin) || !tree_stats_attr<SPEC_BF16, kModeTreeDraft>(optin))
            return nullptr;
        g_tree_init[*dev_out] = true;
    }
    return st;
}

int check_tree_args(int B, int N, int V, int dtype) {
    const int rc = check_common(B, V, dtype);
    if (rc != SPEC_OK) return rc;
    if (N < B || static_cast<int64_t>(N) > static_cast<int64_t>(B) * kMaxTreeNodes) return SPEC_ERR_INVALID_ARG;
    return SPEC_OK;
}

template <int DT, bool VERIFY>
int launch_tree(const void *target, const void *draft, const int32_t *node_offsets, const int32_t *parent,
                const int32_t *tokens, const float *u_accept, const float *u_resample, const float *u_draft,
                const float *temperature, int B, int N, const Geometry &g, int32_t *out_tokens, int32_t *out_num,
                int32_t *out_last, DeviceState &st, cudaStream_t stream) {
    const TreeWsLayout l = tree_ws_layout(B, N, g);
    void *ws = get_internal_ws(st, l.total);
    if (!ws) return SPEC_ERR_CUDA;
    unsigned char *w = static_cast<unsigned char *>(ws);
    int *counters = reinterpret_cast<int *>(w);
    float2 *part = reinterpret_cast<float2 *>(w + l.part);
    int *nint = reinterpret_cast<int *>(w + l.nint);
    int *tint = reinterpret_cast<int *>(w + l.tint);
    float *resid = reinterpret_cast<float *>(w + l.resid);
    int *pair = reinterpret_cast<int *>(w + l.pair);
    float2 *ptot = reinterpret_cast<float2 *>(w + l.ptot);
    int ns, per_sm;
    size_t smem;
    pick_ring(st, B, &ns, &smem, &per_sm);
    if (ns == 0) return SPEC_ERR_INVALID_ARG;
    // setup (launched early; it waits first), then stats_kernel launched
    // plainly: its prologue reads the setup's tables before waiting on anything
    if (!cuda_ok(launch_k(true, tree_setup_kernel, dim3((B * 32 + 255) / 256), dim3(256), 0, stream, node_offsets,
                          parent, B, N, nint, tint, VERIFY ? pair : static_cast<int *>(nullptr)),
                 "launch tree_setup_kernel"))
        return SPEC_ERR_CUDA;
    const cudaError_t e =
        VERIFY ? launch_k(false, stats_kernel<DT, kModeTree>, dim3(st.sms * per_sm), dim3(kThreads), smem, stream,
                          target, draft, temperature, node_offsets, B, g, ns, part, counters,
                          static_cast<int *>(nullptr), static_cast<const int *>(nint), static_cast<const int *>(tint), N, 0,
                          static_cast<PairRec *>(nullptr), SPEC_STREAM_EVICT_FIRST)
               : launch_k(false, stats_kernel<DT, kModeTreeDraft>, dim3(st.sms * per_sm), dim3(kThreads), smem,
                          stream, draft, draft, temperature, node_offsets, B, g, ns, part, counters,
                          static_cast<int *>(nullptr), static_cast<const int *>(nint), static_cast<const int *>(tint), N, 0,
                          static_cast<PairRec *>(nullptr), SPEC_STREAM_EVICT_FIRST);
    if (!cuda_ok(e, "launch stats_kernel (tree)")) return SPEC_ERR_CUDA;
    if (VERIFY) {
        // kTreeCtas CTAs per tree as one cluster (co-scheduled), launched
        // with programmatic dependent launch after stats_kernel
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(B * kTreeCtas);
        cfg.blockDim = dim3(kWalkThreads);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = kTreeCtas;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = kTreeCtas > 1 ? 2 : 1;
        if (!cuda_ok(cudaLaunchKernelEx(&cfg, tree_walk_kernel<DT>, target, draft, node_offsets, parent, tokens,
                                        u_accept, u_resample, temperature, B, N, g, static_cast<const float2 *>(part),
                                        static_cast<const int *>(nint), static_cast<const int *>(tint), resid, pair,
                                        ptot, counters, out_tokens, out_num, out_last),
                     "launch tree_walk_kernel"))
            return SPEC_ERR_CUDA;
    } else {
        const int grid = std::max(1, std::min(st.sms * 8, (N + 7) / 8));
        if (!cuda_ok(launch_k(true, tree_draft_select_kernel<DT>, dim3(grid), dim3(256), (B + 1) * sizeof(int),
                              stream, draft, node_offsets, parent, temperature, u_draft, B, N, g,
                              static_cast<const float2 *>(part), static_cast<const int *>(nint), out_tokens,
                              counters),
                     "launch tree_draft_select_kernel"))
            return SPEC_ERR_CUDA;
    }
    return SPEC_OK;
}

}  // namespace specv

using namespace specv;

extern "C" {

int spec_tree_verify(const void *target_logits, const void *draft_logits, const int32_t *node_offsets,
                     const int32_t *parent, const int32_t *tokens, const float *u_accept, const float *u_resample,
                     const float *temperature, int B, int N, int V, int dtype, int32_t *out_tokens,
                     int32_t *out_num_accepted, int32_t *out_last_node, void *stream) {
    int rc = check_tree_args(B, N, V, dtype);
    if (rc != SPEC_OK) return rc;
    if (B == 0) return SPEC_OK;
    if (!target_logits || !draft_logits || !node_offsets || !parent || !tokens || !u_accept || !u_resample ||
        !temperature || !out_tokens || !out_num_accepted)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || !aligned16(draft_logits)) return SPEC_ERR_ALIGNMENT;
    Geometry g;
    make_geometry(V, dtype, &g);
    int dev;
    DeviceState *st = tree_device_state(&dev);
    if (!st) return SPEC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == SPEC_F32)
        return launch_tree<SPEC_F32, true>(target_logits, draft_logits, node_offsets, parent, tokens, u_accept,
                                           u_resample, nullptr, temperature, B, N, g, out_tokens, out_num_accepted,
                                           out_last_node, *st, s);
    return launch_tree<SPEC_BF16, true>(target_logits, draft_logits, node_offsets, parent, tokens, u_accept,
                                        u_resample, nullptr, temperature, B, N, g, out_tokens, out_num_accepted,
                                        out_last_node, *st, s);
}

int spec_selfcheck_wait_timeout(void *workspace, size_t workspace_bytes, void *stream) {
    if (!workspace) return SPEC_ERR_INVALID_ARG;
    if (workspace_bytes < kCountersBytes) return SPEC_ERR_WORKSPACE;
    if (!aligned16(workspace)) return SPEC_ERR_ALIGNMENT;
    int *counters = static_cast<int *>(workspace);
    // words 8 (result), 9 (the counter nothing completes) and 16..19 (the
    // meeting's partial slots) of the counters block
    selfcheck_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(counters, counters + 9);
    return cuda_ok(cudaGetLastError(), "launch selfcheck_wait_kernel") ? SPEC_OK : SPEC_ERR_CUDA;
}

int spec_tree_draft_sample(const void *draft_logits, const int32_t *node_offsets, const int32_t *parent,
                           const float *temperature, const float *u_draft, int B, int N, int V, int dtype,
                           int32_t *out_tokens, void *stream) {
    int rc = check_tree_args(B, N, V, dtype);
    if (rc != SPEC_OK) return rc;
    if (B == 0) return SPEC_OK;
    if (!draft_logits || !node_offsets || !parent || !temperature || !u_draft || !out_tokens)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned16(draft_logits)) return SPEC_ERR_ALIGNMENT;
    Geometry g;
    make_geometry(V, dtype, &g);
    int dev;
    DeviceState *st = tree_device_state(&dev);
    if (!st) return SPEC_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == SPEC_F32)
        return launch_tree<SPEC_F32, false>(nullptr, draft_logits, node_offsets, parent, nullptr, nullptr, nullptr,
                                            u_draft, temperature, B, N, g, out_tokens, nullptr, nullptr, *st, s);
    return launch_tree<SPEC_BF16, false>(nullptr, draft_logits, node_offsets, parent, nullptr, nullptr, nullptr,
                                         u_draft, temperature, B, N, g, out_tokens, nullptr, nullptr, *st, s);
}

}  // extern "C"
