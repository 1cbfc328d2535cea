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
//   2. the epilogue, by batch size:
//      B < 128         resolve_kernel, up to kSub blocks per sequence: each
//                      combines the partials of the sequence's rows, forms
//                      alpha_i and finds the first rejection with a warp
//                      ballot; on a rejection the blocks share the residual
//                      mass max(0, p - q) of the two rows at that position,
//                      and the last block to finish locates the sub-chunk
//                      where the cumulative mass crosses u * Z, re-reads only
//                      that piece and finds the token with a block scan.
//                      The bonus draw uses the partials of row k the same way.
//      B >= 128        decide_stream_kernel (up to two sequences per
//                      resident CTA) decides every sequence and streams the
//                      rejected positions' row pairs into residual masses in
//                      one launch; beyond that, resolve_kernel decides and
//                      resid_stream_kernel streams.  resid_draw_kernel then
//                      draws each residual token (block per pair).
// spec_draft_sample runs stats_kernel over the draft rows, then
// draft_select_kernel (arg-max, or the same locate + scan per row).
// spec_round chains both passes in one call: the target pass streams while
// the draft tokens are still being drawn.

#include <algorithm>
#include <climits>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <utility>

#include "host_common.h"
#include "verify_common.cuh"

namespace specv {

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
    int last;  // this block finished the sequence's residual slices last
    F2 Z;      // residual mass (the drawing block)
    DrawSmem ds;
};

#ifndef SPEC_RESOLVE_THREADS
#define SPEC_RESOLVE_THREADS 256
#endif
#ifndef SPEC_RESOLVE_MIN_BLOCKS
#define SPEC_RESOLVE_MIN_BLOCKS 4
#endif
// One block's part of the epilogue for sequence b (slice s of nsplit); the
// body of resolve_kernel, and the decision phase of decide_stream_kernel.
template <int DT>
__device__ __forceinline__ void resolve_block(
    const void *__restrict__ target, const void *__restrict__ draft,
    const int32_t *__restrict__ tokens, const float *__restrict__ u_accept,
    const float *__restrict__ u_resample, const float *__restrict__ temperature,
    const int *__restrict__ k_offsets, const double *__restrict__ draft_lse2, int B, const Geometry &g, int nsplit,
    const WsPtrs &ws, int32_t *__restrict__ out_tokens, int32_t *__restrict__ out_num,
    const spec_verify_aux_t &aux, int defer, int inputs_early, int b, int s, ResolveSmem &sm) {
    using E = Elem<DT>;
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
    // the drafted tokens, their logits, the uniforms and the given draft
    // normalisers: before the wait when the caller passed them
    // (inputs_early), after it when the draft pass of the same call wrote them
    auto load_inputs = [&]() {
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
    };
    if (inputs_early) load_inputs();

    // --- 1. row statistics and the decision -------------------------------
    grid_dependency_wait();
    if (!inputs_early) load_inputs();
    // (deferred mode: resid_stream_kernel may be scheduled; it waits for this
    // grid before it reads the pair list)
    grid_launch_dependents();
    // a streaming CTA that timed out leaves partials of unknown age behind:
    // every sequence then reports a data error rather than outputs that
    // look valid (the status word is read here, used in the decision)
    const int status = (warp == 0) ? __ldcg(ws.counters + kStatus) : 0;
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
        bool err = (c != c) || status == SPEC_ERR_TIMEOUT || __any_sync(0xffffffffu, xbad);
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
        if (s != 0) return;
        const int token = block_draw_row<DT>(target, trow, ws.part + trow * g.n_sub, g, c, sm.M[k], sm.u, sm.ds);
        if (threadIdx.x == 0) out_tokens[trow] = token;
        return;
    }

    const int64_t drow = od + n;
    if (defer) {
        // deferred: list the pair; resid_stream_kernel (or the stream phase
        // of decide_stream_kernel) streams its two rows and resid_draw_kernel
        // draws (nsplit is 1 in this mode)
        if (threadIdx.x == 0) {
            PairRec r{};
            r.b = b;
            r.trow = static_cast<int>(trow);
            r.drow = static_cast<int>(drow);
            r.c = c;
            r.lth = sm.lth;
            r.ltl = sm.ltl;
            r.ldh = sm.ldh;
            r.ldl = sm.ldl;
            r.u = sm.u;
            r.ready = 0;
            r.t0 = static_cast<int>(ot);
            r.k = k;
            PairRec *dst = ws.pairs + atomicAdd(ws.counters + kPairs, 1);
            *dst = r;
            st_release_gpu(&dst->ready, 1);  // the residual stream may take it now
        }
        return;
    }

    // --- 2. residual mass of this block's slice of sub-chunks -------------
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
    // arrival, one per block once all its warps are done: the block that
    // arrives last, of the nsplit blocks of b, draws (acquire-release add:
    // this block's masses are released with it, and the last block
    // acquires everyone's; the barrier after it extends that to its warps)
    __syncthreads();
    if (threadIdx.x == 0) sm.last = atomic_add_acq_rel_gpu(ws.seqcnt + b, 1) == nsplit - 1;
    __syncthreads();
    if (!sm.last) return;

    // --- 3. the residual draw, by the last block of b ----------------------
    if (warp == 0) {
        float w[kPartCache];
#pragma unroll
        for (int j = 0; j < kPartCache; ++j) w[j] = (lane + 32 * j < g.n_sub) ? __ldcg(rp + lane + 32 * j) : 0.0f;
        auto wfar = [&](int i) -> float { return __ldcg(rp + i); };
        F2 before, Z, tgt;
        const int sc = warp_locate(g.n_sub, w, wfar, sm.u, &before, &Z, &tgt);
        if (lane == 0) {
            sm.ds.sc = sc;
            sm.ds.before = before;
            sm.ds.target = tgt;
            sm.Z = Z;
        }
    }
    __syncthreads();
    int token = -1;
    const int sc = sm.ds.sc;
    if (sc >= 0) {
        int a, e1;
        sub_range(g, sc, &a, &e1);
        const void *rt = static_cast<const unsigned char *>(target) + trow * V * static_cast<int64_t>(E::kBytes);
        const void *rd = static_cast<const unsigned char *>(draft) + drow * V * static_cast<int64_t>(E::kBytes);
        auto W = [&](float a1, float a2) -> float { return resid_weight(a1, a2, c, lth, ltl, ldh, ldl); };
        token = block_scan_elems<DT>(rt, rd, a, e1, W, sm.ds.before, sm.ds.target, sm.ds);
    } else {
        // every residual weight rounded to 0: p at position n is drawn with
        // the same uniform instead
        token = block_draw_row<DT>(target, trow, ws.part + trow * g.n_sub, g, c, sm.M[n], sm.u, sm.ds);
    }
    if (threadIdx.x == 0) {
        out_tokens[trow] = token;
        if (aux.residual_mass) aux.residual_mass[b] = __fadd_rn(sm.Z.hi, sm.Z.lo);
    }
}

template <int DT>
__global__ void __launch_bounds__(SPEC_RESOLVE_THREADS, SPEC_RESOLVE_MIN_BLOCKS) resolve_kernel(
    const void *__restrict__ target, const void *__restrict__ draft,
    const int32_t *__restrict__ tokens, const float *__restrict__ u_accept,
    const float *__restrict__ u_resample, const float *__restrict__ temperature,
    const int *__restrict__ k_offsets, const double *__restrict__ draft_lse2, int B, Geometry g, int nsplit,
    WsPtrs ws, int32_t *__restrict__ out_tokens, int32_t *__restrict__ out_num, spec_verify_aux_t aux,
    int defer, int inputs_early) {
    __shared__ ResolveSmem sm;
    const int b = blockIdx.x / nsplit;
    resolve_block<DT>(target, draft, tokens, u_accept, u_resample, temperature, k_offsets, draft_lse2, B, g, nsplit,
                      ws, out_tokens, out_num, aux, defer, inputs_early, b, blockIdx.x - b * nsplit, sm);
}

// ================================================================== kernel 3
// The residual pass of the deferred epilogue, as a stream: every listed pair
// (the target and the draft row at a rejected position) is cut into units
// of one chunk of each row; lane 0 of warp 8 copies a unit's two chunks
// into a 32 KB ring slot (two 1-D bulk copies on one mbarrier), and the
// eight consumer warps each sum max(0, p - q) over their 2 KB sub-chunk of
// the pair and store that mass.  Units are taken by tickets (unit_batch),
// so every SM keeps its slots full until the last pair; the bytes read are
// the pairs' rows, at the rate of the main pass instead of the rate of
// per-block loads that wait on their decisions.
constexpr int kRSlotBytes = 2 * kSlotBytes;  // a target chunk, then the draft chunk

struct RUnit {
    uint32_t nbytes;  // bytes of each row's chunk (0: end marker)
    float c, lth, ltl, ldh, ldl;
    int64_t out;      // index of the unit's first sub-chunk mass in resid_part
};

// A streaming CTA's residual ring: ns slots of a target chunk and the
// draft chunk at the same place, their full/empty barriers and descriptors.
struct RRing {
    unsigned char *ring;
    uint64_t *full, *empty;
    RUnit *desc;
    int ns;
};
__device__ __forceinline__ RRing rring_carve(unsigned char *smem, int ns) {
    RRing q;
    q.ring = smem;
    q.full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(ns) * kRSlotBytes);
    q.empty = q.full + ns;
    q.desc = reinterpret_cast<RUnit *>(q.empty + ns);
    q.ns = ns;
    return q;
}
// (thread 0; a barrier must follow before other threads use the ring)
__device__ __forceinline__ void rring_init(const RRing &q) {
    for (int i = 0; i < q.ns; ++i) {
        mbar_init(&q.full[i], 1);
        mbar_init(&q.empty[i], kConsumerWarps);
    }
    fence_barrier_init();
}

// Producer state of a ring (lane 0 of the producer warp).
struct RProd {
    int slot = 0, issued = 0;
    uint32_t phase = 0;
};

// Issue unit (pair r, chunk ch): wait for a free slot, write its
// descriptor, copy the two chunks.  False when the wait for a slot timed out.
template <int DT>
__device__ __forceinline__ bool rring_push(const RRing &q, RProd &st, const PairRec &r, int ch, const void *target,
                                           const void *draft, const Geometry &g) {
    using E = Elem<DT>;
    if (st.issued >= q.ns && !mbar_wait_bounded(&q.empty[st.slot], st.phase ^ 1u)) return false;
    const int e0 = ch * g.chunk_elems;
    const int e1 = min(g.V, e0 + g.chunk_elems);
    RUnit d;
    d.nbytes = static_cast<uint32_t>(e1 - e0) * E::kBytes;
    d.c = r.c;
    d.lth = r.lth;
    d.ltl = r.ltl;
    d.ldh = r.ldh;
    d.ldl = r.ldl;
    d.out = static_cast<int64_t>(r.b) * g.n_sub + static_cast<int64_t>(ch) * kSub;
    q.desc[st.slot] = d;
    const int64_t off = static_cast<int64_t>(e0) * E::kBytes;
    const unsigned char *ts =
        static_cast<const unsigned char *>(target) + static_cast<int64_t>(r.trow) * g.V * E::kBytes + off;
    const unsigned char *dsrc =
        static_cast<const unsigned char *>(draft) + static_cast<int64_t>(r.drow) * g.V * E::kBytes + off;
    unsigned char *slot = q.ring + static_cast<size_t>(st.slot) * kRSlotBytes;
    mbar_arrive_expect_tx(&q.full[st.slot], 2 * d.nbytes);
    bulk_g2s(slot, ts, d.nbytes, &q.full[st.slot]);
    bulk_g2s(slot + kSlotBytes, dsrc, d.nbytes, &q.full[st.slot]);
    ++st.issued;
    if (++st.slot == q.ns) {
        st.slot = 0;
        st.phase ^= 1u;
    }
    return true;
}

// Close the ring: the end marker (also after a time-out, so that the
// consumers leave), and on a time-out the status word, after the copies in
// flight have landed.
__device__ __forceinline__ void rring_close(const RRing &q, const RProd &st, bool ok, int *counters) {
    if (ok && st.issued >= q.ns) ok = mbar_wait_bounded(&q.empty[st.slot], st.phase ^ 1u);
    q.desc[st.slot].nbytes = 0;
    mbar_arrive(&q.full[st.slot]);
    if (!ok) {
        set_status(counters + kStatus, SPEC_ERR_TIMEOUT);
        for (int i = max(0, st.issued - q.ns); i < st.issued; ++i) mbar_wait_bounded(&q.full[i % q.ns], (i / q.ns) & 1);
    }
}

// Consumer warps: each sums max(0, p - q) over its 2 KB sub-chunk of every
// unit until the end marker, and stores that mass.
template <int DT>
__device__ __forceinline__ void rring_consume(const RRing &q, float *__restrict__ resid_part, int *counters) {
    using E = Elem<DT>;
    const int w = warp_id(), lane = lane_id();
    int slot = 0;
    uint32_t phase = 0;
    for (;;) {
        if (!mbar_wait_bounded(&q.full[slot], phase)) {
            set_status(counters + kStatus, SPEC_ERR_TIMEOUT);
            break;
        }
        const RUnit d = q.desc[slot];
        if (d.nbytes == 0) break;
        const unsigned char *sl = q.ring + static_cast<size_t>(slot) * kRSlotBytes;
        const uint4 *pt = reinterpret_cast<const uint4 *>(sl) + w * kSubVecs;
        const uint4 *pd = reinterpret_cast<const uint4 *>(sl + kSlotBytes) + w * kSubVecs;
        const int nvec = min(kSubVecs, static_cast<int>(d.nbytes >> 4) - w * kSubVecs);  // may be <= 0
        uint4 xt4[4], xd4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = lane + 32 * j;
            if (i < nvec) {
                xt4[j] = pt[i];
                xd4[j] = pd[i];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&q.empty[slot]);  // the slot's data is in registers
        if (++slot == q.ns) {
            slot = 0;
            phase ^= 1u;
        }
        // (a sub-chunk past the row's end has no elements and gets mass 0)
        // the same operations, in the same order, as the residual pass of
        // resolve_kernel, so both epilogues give the same masses
        const float2 c2 = make_float2(d.c, d.c), nlth2 = make_float2(-d.lth, -d.lth);
        const float2 nltl2 = make_float2(-d.ltl, -d.ltl);
        const float2 nldh2 = make_float2(-d.ldh, -d.ldh), nldl2 = make_float2(-d.ldl, -d.ldl);
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
        if (lane == 0) resid_part[d.out + w] = sum;
    }
}

// The last CTA out resets the ticket counters for the next launch.
__device__ __forceinline__ void rring_retire(int *counters) {
    __syncthreads();
    if (threadIdx.x == 0 && atomic_add_acq_rel_gpu(counters + kDone, 1) == static_cast<int>(gridDim.x) - 1) {
        counters[kTicket] = 0;
        counters[kDone] = 0;
    }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 2) resid_stream_kernel(
    const void *__restrict__ target, const void *__restrict__ draft, Geometry g, int ns,
    const PairRec *__restrict__ pairs, float *__restrict__ resid_part, int *__restrict__ counters) {
    extern __shared__ __align__(128) unsigned char smem[];
    const RRing q = rring_carve(smem, ns);
    // the pair list is complete once resolve_kernel has finished
    grid_dependency_wait();
    grid_launch_dependents();
    const int npairs = __ldcg(counters + kPairs);
    if (threadIdx.x == 0) rring_init(q);
    __syncthreads();
    if (warp_id() == kConsumerWarps) {
        // ------------------------------------------------------ producer
        if (lane_id() == 0) {
            const int64_t total_units = static_cast<int64_t>(npairs) * g.n_chunks;
            const int64_t n_big = big_batches(total_units, gridDim.x);
            RProd st;
            bool ok = true;
            int cur = -1;
            PairRec r{};
            int t = atomicAdd(counters + kTicket, 1);
            while (ok) {
                int64_t u0;
                int cnt;
                unit_batch(t, n_big, &u0, &cnt);
                if (u0 >= total_units) break;
                const int tn = atomicAdd(counters + kTicket, 1);  // next batch, in flight meanwhile
                cnt = static_cast<int>(min(static_cast<int64_t>(cnt), total_units - u0));
                for (int qi = 0; qi < cnt && ok; ++qi) {
                    const int64_t u = u0 + qi;
                    const int p = static_cast<int>(u / g.n_chunks);
                    if (p != cur) {
                        r = pairs[p];
                        cur = p;
                    }
                    ok = rring_push<DT>(q, st, r, static_cast<int>(u - static_cast<int64_t>(p) * g.n_chunks), target,
                                        draft, g);
                }
                t = tn;
            }
            rring_close(q, st, ok, counters);
        }
        __syncwarp();
    } else {
        rring_consume<DT>(q, resid_part, counters);
    }
    rring_retire(counters);
}

// Units (consecutive chunks of one pair) per ticket of decide_stream_kernel:
// one ticket, and one check of the pair's flag, per SPEC_FUSE_UNITS copies.
// Measured (three CTAs per SM, two slots): 1 unit per ticket 4-8 µs slower
// per B=512 verify or round than 2 units; 4 units 1-2 µs slower on B=256.
#ifndef SPEC_FUSE_UNITS
#define SPEC_FUSE_UNITS 2
#endif
// The deferred epilogue's decisions and residual stream in one launch (for
// B at most twice the grid).  Each CTA first decides its sequences
// (b = blockIdx.x, blockIdx.x + gridDim.x, ...) as resolve_kernel does in
// deferred mode: a rejected position's pair is listed with a ready flag
// (release), and every decided sequence is counted (release, after its
// pair).  Then the CTA streams units of listed pairs, SPEC_FUSE_UNITS
// chunks of one pair per ticket, in the order of the list: the producer
// waits (acquire) until the ticket's pair is ready, and leaves once every
// sequence is decided and the ticket lies past the list.  The first pairs
// stream while later ones are still being decided, and no launch boundary
// lies between decision and stream.  A CTA may wait on pairs that another
// lists, so the grid never exceeds the CTAs that are resident at once (the
// occupancy the host queries); should another kernel hold SMs for longer
// than the bounded wait (2 s), the call reports a time-out, not a hang.
template <int DT>
// Resident decide_stream_kernel CTAs per SM and 32 KB ring slots per CTA:
// three CTAs of two slots decide more sequences at once than two of three
// (B=512: 1.1 sequences per CTA instead of 1.7) with the same bytes in flight
// per SM; measured 3-4 µs faster per B=512 verify, the same on B=256.
#ifndef SPEC_FUSE_CTAS_PER_SM
#define SPEC_FUSE_CTAS_PER_SM 3
#endif
#ifndef SPEC_FUSE_SLOTS
#define SPEC_FUSE_SLOTS 2
#endif
__global__ void __launch_bounds__(kThreads, SPEC_FUSE_CTAS_PER_SM) decide_stream_kernel(
    const void *__restrict__ target, const void *__restrict__ draft,
    const int32_t *__restrict__ tokens, const float *__restrict__ u_accept,
    const float *__restrict__ u_resample, const float *__restrict__ temperature,
    const int *__restrict__ k_offsets, const double *__restrict__ draft_lse2, int B, Geometry g, WsPtrs ws,
    int32_t *__restrict__ out_tokens, int32_t *__restrict__ out_num, spec_verify_aux_t aux, int inputs_early,
    int ns) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ ResolveSmem sm;
    const RRing q = rring_carve(smem, ns);
    int *counters = ws.counters;
    if (threadIdx.x == 0) rring_init(q);
    // ------------------------------------------------------------ decisions
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        resolve_block<DT>(target, draft, tokens, u_accept, u_resample, temperature, k_offsets, draft_lse2, B, g, 1, ws,
                          out_tokens, out_num, aux, 1, inputs_early && b == static_cast<int>(blockIdx.x), b, 0, sm);
        __syncthreads();  // (thread 0 listed the pair, if any, before this)
        if (threadIdx.x == 0) red_add_release_gpu(counters + kDecided, 1);
    }
    grid_dependency_wait();  // (a CTA without a sequence)
    grid_launch_dependents();
    __syncthreads();
    // ------------------------------------------------------------ residual stream
    if (warp_id() == kConsumerWarps) {
        if (lane_id() == 0) {
            RProd st;
            bool ok = true;
            int cur = -1;
            PairRec r{};
            const int per = (g.n_chunks + SPEC_FUSE_UNITS - 1) / SPEC_FUSE_UNITS;  // tickets per pair
            int t = atomicAdd(counters + kTicket, 1);
            while (ok) {
                const int p = t / per;
                const int tn = atomicAdd(counters + kTicket, 1);  // the next ticket, in flight meanwhile
                if (p != cur) {
                    // wait for pair p: listed and ready, or never listed
                    const int listed = wait_pair(counters, ws.pairs, p, B);
                    if (listed < 0) ok = false;
                    if (listed <= 0) break;
                    r = ws.pairs[p];
                    cur = p;
                }
                const int c0 = (t - p * per) * SPEC_FUSE_UNITS;
                const int c1 = min(g.n_chunks, c0 + SPEC_FUSE_UNITS);
                for (int ch = c0; ch < c1 && ok; ++ch) ok = rring_push<DT>(q, st, r, ch, target, draft, g);
                t = tn;
            }
            rring_close(q, st, ok, counters);
        }
        __syncwarp();
    } else {
        rring_consume<DT>(q, ws.resid_part, counters);
    }
    rring_retire(counters);
}

// The residual draw of the deferred epilogue: one block per listed pair.
// Warp 0 locates the sub-chunk where the cumulative residual mass crosses
// u * Z; the block scans its elements (the draw of resolve_kernel's step 3).
template <int DT>
__global__ void __launch_bounds__(kDrawThreads) resid_draw_kernel(
    const void *__restrict__ target, const void *__restrict__ draft, Geometry g,
    const PairRec *__restrict__ pairs, const float *__restrict__ resid_part, const float2 *__restrict__ part,
    const int *__restrict__ counters, int32_t *__restrict__ out_tokens, int32_t *__restrict__ out_num,
    float *__restrict__ aux_resid) {
    using E = Elem<DT>;
    __shared__ DrawSmem ds;
    __shared__ F2 sZ;
    __shared__ float sM;
    __shared__ int sok;
    grid_dependency_wait();
    const int npairs = __ldcg(counters + kPairs);
    const int p = blockIdx.x;
    if (p >= npairs) return;
    const int lane = lane_id();
    const PairRec r = pairs[p];
    if (__ldcg(counters + kStatus) == SPEC_ERR_TIMEOUT) {
        // the residual stream gave up: masses of unknown age, so the
        // sequence is a data error, not a draw that looks valid
        for (int i = threadIdx.x; i <= r.k; i += blockDim.x) out_tokens[r.t0 + i] = -1;
        if (threadIdx.x == 0) {
            out_num[r.b] = -1;
            if (aux_resid) aux_resid[r.b] = NAN;
        }
        return;
    }
    if (warp_id() == 0) {
        const float *rp = resid_part + static_cast<int64_t>(r.b) * g.n_sub;
        float w[kPartCache];
#pragma unroll
        for (int j = 0; j < kPartCache; ++j) w[j] = (lane + 32 * j < g.n_sub) ? __ldcg(rp + lane + 32 * j) : 0.0f;
        auto wfar = [&](int i) -> float { return __ldcg(rp + i); };
        F2 before, Z, tgt;
        const int sc = warp_locate(g.n_sub, w, wfar, r.u, &before, &Z, &tgt);
        float M = 0.0f, S = 0.0f;
        bool ok = true;
        if (sc < 0) ok = warp_combine_soft(part + static_cast<int64_t>(r.trow) * g.n_sub, g.n_sub, &M, &S);
        if (lane == 0) {
            ds.sc = sc;
            ds.before = before;
            ds.target = tgt;
            sZ = Z;
            sM = M;
            sok = ok;
        }
    }
    __syncthreads();
    int token = -1;
    if (ds.sc >= 0) {
        int a, e1;
        sub_range(g, ds.sc, &a, &e1);
        const void *rt = static_cast<const unsigned char *>(target) + static_cast<int64_t>(r.trow) * g.V * E::kBytes;
        const void *rd = static_cast<const unsigned char *>(draft) + static_cast<int64_t>(r.drow) * g.V * E::kBytes;
        auto W = [&](float a1, float a2) -> float { return resid_weight(a1, a2, r.c, r.lth, r.ltl, r.ldh, r.ldl); };
        token = block_scan_elems<DT>(rt, rd, a, e1, W, ds.before, ds.target, ds);
    } else if (sok) {
        // every residual weight rounded to 0: p at the position is drawn with
        // the same uniform instead
        token = block_draw_row<DT>(target, r.trow, part + static_cast<int64_t>(r.trow) * g.n_sub, g, r.c, sM, r.u, ds);
    }
    if (threadIdx.x == 0) {
        out_tokens[r.trow] = token;
        if (aux_resid) aux_resid[r.b] = __fadd_rn(sZ.hi, sZ.lo);
    }
}

// A draft row's temperature scale (its sequence by bisection of the
// offsets in shared memory) and drafting uniform.
struct DraftRowIn {
    float c, ud;
};

__device__ __forceinline__ DraftRowIn draft_row_inputs(const int *s_kofs, int B, const float *__restrict__ temperature,
                                                       const float *__restrict__ u_draft, int r) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_kofs[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return DraftRowIn{temp_scale(temperature[lo]), u_draft[r]};
}

// Draft-side draw: one warp per draft row (grid-stride over rows).  With
// out_lse2 given, each row's log2-domain log-sum-exp (the value
// resolve_kernel would combine from the same partials) is written too: NaN
// for greedy and invalid rows.
template <int DT>
__global__ void __launch_bounds__(256) draft_select_kernel(
    const void *__restrict__ draft, const float *__restrict__ temperature, const float *__restrict__ u_draft,
    const int *__restrict__ k_offsets, int B, Geometry g, const float2 *__restrict__ part,
    int32_t *__restrict__ out, double *__restrict__ out_lse2, int *__restrict__ counters, int early_trigger) {
    extern __shared__ int s_kofs[];  // [B+1]
    // spec_round: the target pass may launch at once (it streams rows of its
    // own while these draws wait for the draft pass, and waits for this grid
    // before it exits)
    if (early_trigger) grid_launch_dependents();
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
    const int R = s_kofs[B];
    const int lane = lane_id();
    const int nw = (gridDim.x * blockDim.x) >> 5;
    const int r0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    // a row's temperature scale and uniform: the caller's inputs, complete
    // once the call's first kernel passed its wait, so the first row's are
    // read before this kernel's wait (with valid offsets only: then r < R
    // stays inside the caller's arrays)
    DraftRowIn in{0.0f, 0.0f};
    if (!s_bad && r0 < R) in = draft_row_inputs(s_kofs, B, temperature, u_draft, r0);
    grid_dependency_wait();
    grid_launch_dependents();
    if (s_bad) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(counters + kStatus, SPEC_ERR_INVALID_ARG);
        return;
    }
    // the streaming pass timed out: its partials are of unknown age, so every
    // row gets -1 (and no normaliser) instead of a token that looks valid
    const bool timed_out = __ldcg(counters + kStatus) == SPEC_ERR_TIMEOUT;
    for (int r = r0; r < R; r += nw) {
        if (r != r0) in = draft_row_inputs(s_kofs, B, temperature, u_draft, r);
        const float c = timed_out ? __int_as_float(0x7fc00000) : in.c;
        // (draft row r's partials are at slot R_t + r, R_t = R + B); they are
        // requested with the status word, whatever the row's temperature (a
        // row of a bad temperature has a slot too, its contents unused)
        const float2 *pr = part + (static_cast<int64_t>(R) + B + r) * g.n_sub;
        float2 pc[kPartCache];
        load_parts(pr, g.n_sub, pc);  // one round trip serves the combine and the draw
        int token = -1;
        double L = NAN;
        if (c == 0.0f) {
            token = warp_combine_arg_cached(pc, pr, g.n_sub);
        } else if (c == c) {
            float M, S;
            if (combine_soft(pc, pr, g.n_sub, &M, &S)) {
                L = lse2(M, S);
                token = warp_draw_row<DT>(draft, r, pr, pc, g, c, M, in.ud);
            }
        }
        if (lane == 0) {
            out[r] = token;
            if (out_lse2) out_lse2[r] = L;
        }
    }
}

// ================================================================== host side
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;


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
    size_t part, counters, seqcnt, resid, lse2, pairs, total;
};

// Workspace layout.  The counters block comes first (kStatusOffset).

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
    l.pairs = off;  // the deferred epilogue's residual pairs
    off = align_up(off + static_cast<size_t>(B) * sizeof(PairRec), 256);
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
    w.pairs = reinterpret_cast<PairRec *>(p + l.pairs);
    return w;
}

// Last CUDA failure seen by this thread (call site + CUDA error name).
thread_local char g_last_error[kLastErrorBytes] = "";

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

// resid_stream_kernel: up to kResidSlots 32 KB slots.
constexpr int kResidSlots = 3;
size_t resid_smem(int ns) { return align_up(ns * (kRSlotBytes + 2 * sizeof(uint64_t) + sizeof(RUnit)), 128); }

template <int DT>
bool set_stats_attrs_all(DeviceState &st) {
    const int rs = static_cast<int>(resid_smem(kResidSlots));
    return set_stats_attrs<DT, kModeVerify>(st.smem_optin) && set_stats_attrs<DT, kModeDraft>(st.smem_optin) &&
           set_stats_attrs<DT, kModeTarget>(st.smem_optin) &&
           cuda_ok(cudaFuncSetAttribute(resid_stream_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, rs),
                   "cudaFuncSetAttribute(resid_stream_kernel)") &&
           cuda_ok(cudaFuncSetAttribute(decide_stream_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(resid_smem(SPEC_FUSE_SLOTS))),
                   "cudaFuncSetAttribute(decide_stream_kernel)") &&
           cuda_ok(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&st.fuse_per_sm[DT == SPEC_F32 ? 0 : 1],
                                                                 decide_stream_kernel<DT>, kThreads,
                                                                 resid_smem(SPEC_FUSE_SLOTS)),
                   "cudaOccupancyMaxActiveBlocksPerMultiprocessor(decide_stream_kernel)");
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
        if (!set_stats_attrs_all<SPEC_F32>(st) || !set_stats_attrs_all<SPEC_BF16>(st))
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


#ifndef SPEC_RESOLVE_BLOCKS_PER_SM
#define SPEC_RESOLVE_BLOCKS_PER_SM 8
#endif
// The epilogue's residual pass: inside resolve_kernel (blocks per sequence
// stream their slices of the two rows, then the last warp draws), or, for
// batches of at least SPEC_DEFER_MIN_B sequences, deferred: resolve_kernel
// only decides and lists the rejected positions, resid_stream_kernel streams
// their rows, resid_draw_kernel draws.
#ifndef SPEC_DEFER_MIN_B
#define SPEC_DEFER_MIN_B 128
#endif
bool defer_residual(const DeviceState &, int B) { return B >= SPEC_DEFER_MIN_B; }

// Deferred epilogues of at most SPEC_FUSE_PER_CTA sequences per resident
// CTA take decide_stream_kernel (decisions and residual stream in one
// launch); larger ones resolve_kernel, then resid_stream_kernel.
#ifndef SPEC_FUSE_PER_CTA
#define SPEC_FUSE_PER_CTA 2
#endif
template <int DT>
int fuse_grid(const DeviceState &st, int B) {
    const int g = st.sms * std::min(SPEC_FUSE_CTAS_PER_SM, st.fuse_per_sm[DT == SPEC_F32 ? 0 : 1]);
    return (g > 0 && B <= SPEC_FUSE_PER_CTA * g) ? g : 0;
}

// resolve_kernel blocks per sequence for n sequences on an idle GPU:
// 1..kSub, as many as fit one wave of SPEC_RESOLVE_BLOCKS_PER_SM per SM.
int resolve_split(const DeviceState &st, const Geometry &g, int n) {
    return std::max(1, std::min({kSub, g.n_sub, (SPEC_RESOLVE_BLOCKS_PER_SM * st.sms) / std::max(n, 1)}));
}

// The verify pass: stats_kernel streams the target rows (and, without
// draft_lse2, the draft rows of sampled sequences), then resolve_kernel.
// The streaming kernel is launched early behind the stream's previous
// kernel (programmatic dependent launch).  pdl_first: the draft pass of the
// same call precedes it (spec_round): the target rows stream at once, while
// draft_select_kernel still draws (the two use disjoint partial slots), the
// streaming kernel waits for it only before it exits, and resolve_kernel
// reads the drafted tokens and normalisers only after its own wait.
// Otherwise it opens the call and waits first (the previous kernel may be
// writing the inputs).  after_event: the stream waits on an event just
// before (another stream's copy), and the kernel is launched plainly.
template <int DT>
int launch_verify(const void *target, const void *draft, const double *draft_lse2, const int32_t *tokens,
                  const float *u_accept, const float *u_resample, const float *temperature, int B,
                  const int32_t *k_offsets, const Geometry &g, int32_t *out_tokens, int32_t *out_num,
                  const spec_verify_aux_t &aux, void *ws_base, const WsLayout &l, const DeviceState &st,
                  cudaStream_t stream, bool pdl_first = false, bool after_event = false) {
    int ns, per_sm;
    size_t smem;
    pick_ring(st, B, &ns, &smem, &per_sm);
    if (ns == 0) return SPEC_ERR_INVALID_ARG;
    const WsPtrs w = ws_ptrs(ws_base, l);
    const int grid = st.sms * per_sm;
    const bool defer = defer_residual(st, B);
    const int nsplit = defer ? 1 : resolve_split(st, g, B);
    const cudaError_t e1 =
        draft_lse2 ? launch_k(!after_event, stats_kernel<DT, kModeTarget>, dim3(grid), dim3(kThreads), smem, stream,
                              target, draft, temperature, k_offsets, B, g, ns, w.part, w.counters, w.seqcnt,
                              nullptr, nullptr, 0, pdl_first ? 2 : 1, w.pairs, SPEC_STREAM_EVICT_FIRST)
                   : launch_k(!after_event, stats_kernel<DT, kModeVerify>, dim3(grid), dim3(kThreads), smem, stream,
                              target, draft, temperature, k_offsets, B, g, ns, w.part, w.counters, w.seqcnt,
                              nullptr, nullptr, 0, pdl_first ? 2 : 1, w.pairs, SPEC_STREAM_EVICT_FIRST);
    if (!cuda_ok(e1, "launch stats_kernel")) return SPEC_ERR_CUDA;
    const int fgrid = defer ? fuse_grid<DT>(st, B) : 0;
    if (fgrid > 0) {
        if (!cuda_ok(launch_k(true, decide_stream_kernel<DT>, dim3(fgrid), dim3(kThreads), resid_smem(SPEC_FUSE_SLOTS), stream,
                              target, draft, tokens, u_accept, u_resample, temperature, k_offsets, draft_lse2, B, g, w,
                              out_tokens, out_num, aux, pdl_first ? 0 : 1, SPEC_FUSE_SLOTS),
                     "launch decide_stream_kernel"))
            return SPEC_ERR_CUDA;
    } else if (!cuda_ok(launch_k(true, resolve_kernel<DT>, dim3(B * nsplit), dim3(SPEC_RESOLVE_THREADS), 0, stream, target, draft, tokens,
                          u_accept, u_resample, temperature, k_offsets, draft_lse2, B, g, nsplit, w, out_tokens,
                          out_num, aux, defer ? 1 : 0, pdl_first ? 0 : 1),
                 "launch resolve_kernel"))
        return SPEC_ERR_CUDA;
    if (!defer) return SPEC_OK;
    // deferred epilogue: the listed pairs' rows streamed, then the draws
    const int rgrid = st.sms * std::max(1, std::min(2, st.smem_per_sm / static_cast<int>(resid_smem(kResidSlots) + 1024)));
    if ((fgrid == 0 && !cuda_ok(launch_k(true, resid_stream_kernel<DT>, dim3(rgrid), dim3(kThreads), resid_smem(kResidSlots), stream,
                          target, draft, g, kResidSlots, static_cast<const PairRec *>(w.pairs), w.resid_part,
                          w.counters),
                 "launch resid_stream_kernel")) ||
        !cuda_ok(launch_k(true, resid_draw_kernel<DT>, dim3(B), dim3(kDrawThreads), 0, stream, target, draft, g,
                          static_cast<const PairRec *>(w.pairs), static_cast<const float *>(w.resid_part),
                          static_cast<const float2 *>(w.part), static_cast<const int *>(w.counters), out_tokens,
                          out_num, aux.residual_mass),
                 "launch resid_draw_kernel"))
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

#ifndef SPEC_SELECT_BESIDE_THREADS
#define SPEC_SELECT_BESIDE_THREADS 128
#endif
#ifndef SPEC_SELECT_BESIDE_BLOCKS
#define SPEC_SELECT_BESIDE_BLOCKS 1
#endif
#ifndef SPEC_SELECT_BLOCKS_PER_SM
#define SPEC_SELECT_BLOCKS_PER_SM 8
#endif
template <int DT>
int launch_draft(const void *draft, const float *temperature, const float *u_draft, int B,
                 const int32_t *k_offsets, const Geometry &g, int32_t *out, double *out_lse2, void *ws_base,
                 const WsLayout &l, const DeviceState &st, cudaStream_t stream, bool beside_stream = false) {
    int ns, per_sm;
    size_t smem;
    pick_ring(st, B, &ns, &smem, &per_sm);
    if (ns == 0) return SPEC_ERR_INVALID_ARG;
    const WsPtrs w = ws_ptrs(ws_base, l);
    // one warp per draft row (grid-stride): at most B * kMaxK rows, 8 warps
    // per block.  beside_stream (spec_round): the target pass streams while
    // the draws run and needs them only at its end, so the draws take one
    // 4-warp block per SM and leave each SM room for four streaming CTAs
    const int threads = beside_stream ? SPEC_SELECT_BESIDE_THREADS : 256;
    const int grid = beside_stream ? st.sms * SPEC_SELECT_BESIDE_BLOCKS
                                   : static_cast<int>(std::min(static_cast<int64_t>(st.sms) * SPEC_SELECT_BLOCKS_PER_SM,
                                                               (static_cast<int64_t>(B) * kMaxK + 7) / 8));
    // the call's first kernel: launched early behind the stream's previous
    // kernel, it waits for it before reading the inputs (wait_first)
    if (!cuda_ok(launch_k(true, stats_kernel<DT, kModeDraft>, dim3(st.sms * per_sm), dim3(kThreads), smem, stream,
                          draft, draft, temperature, k_offsets, B, g, ns, w.part, w.counters, nullptr, nullptr,
                          nullptr, 0, 1, static_cast<PairRec *>(nullptr), SPEC_STREAM_EVICT_FIRST),
                 "launch stats_kernel") ||
        !cuda_ok(launch_k(true, draft_select_kernel<DT>, dim3(std::max(grid, 1)), dim3(threads),
                          (B + 1) * sizeof(int), stream, draft, temperature, u_draft, k_offsets, B, g,
                          static_cast<const float2 *>(w.part), out, out_lse2, w.counters, beside_stream ? 1 : 0),
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
                const spec_verify_aux_t *aux, void *workspace, size_t workspace_bytes, void *stream,
                bool reset_counters) {
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
    void *ws = reset_counters ? call_workspace(workspace, workspace_bytes, l, *st, s, &rc) : workspace;
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
// before_verify (optional): an event the verify pass waits for (the host
// entry's copy of the target logits); the draft pass does not wait for it.
int round_call(const void *target_logits, const void *draft_logits, const float *u_draft, const float *u_accept,
               const float *u_resample, const float *temperature, int B, const int32_t *k_offsets, int V, int dtype,
               int32_t *out_draft_tokens, int32_t *out_tokens, int32_t *out_num_accepted, void *stream,
               cudaEvent_t before_verify = nullptr) {
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
    // the verify pass chains to the draft pass by programmatic dependent
    // launch, unless it has to wait for an event first
    const bool chained = before_verify == nullptr;
    if (dtype == SPEC_F32) {
        rc = launch_draft<SPEC_F32>(draft_logits, temperature, u_draft, B, k_offsets, g, out_draft_tokens, lse2, ws,
                                    l, *st, s, chained);
        if (rc != SPEC_OK) return rc;
        if (!chained && !cuda_ok(cudaStreamWaitEvent(s, before_verify, 0), "cudaStreamWaitEvent")) return SPEC_ERR_CUDA;
        return launch_verify<SPEC_F32>(target_logits, draft_logits, lse2, out_draft_tokens, u_accept, u_resample,
                                       temperature, B, k_offsets, g, out_tokens, out_num_accepted, a, ws, l, *st, s,
                                       chained, !chained);
    }
    rc = launch_draft<SPEC_BF16>(draft_logits, temperature, u_draft, B, k_offsets, g, out_draft_tokens, lse2, ws, l,
                                 *st, s, chained);
    if (rc != SPEC_OK) return rc;
    if (!chained && !cuda_ok(cudaStreamWaitEvent(s, before_verify, 0), "cudaStreamWaitEvent")) return SPEC_ERR_CUDA;
    return launch_verify<SPEC_BF16>(target_logits, draft_logits, lse2, out_draft_tokens, u_accept, u_resample,
                                    temperature, B, k_offsets, g, out_tokens, out_num_accepted, a, ws, l, *st, s,
                                    chained, !chained);
}

}  // namespace specv

extern "C" {

int spec_verify_ex(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                   const float *u_accept, const float *u_resample, const float *temperature, int B,
                   const int32_t *k_offsets, int V, int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
                   const spec_verify_aux_t *aux, void *workspace, size_t workspace_bytes, void *stream) {
    return verify_call(target_logits, draft_logits, nullptr, draft_tokens, u_accept, u_resample, temperature, B,
                       k_offsets, V, dtype, out_tokens, out_num_accepted, aux, workspace, workspace_bytes, stream,
                       true);
}

int spec_verify(const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,
                const float *u_accept, const float *u_resample, const float *temperature, int B,
                const int32_t *k_offsets, int V, int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
                void *stream) {
    return verify_call(target_logits, draft_logits, nullptr, draft_tokens, u_accept, u_resample, temperature, B,
                       k_offsets, V, dtype, out_tokens, out_num_accepted, nullptr, nullptr, 0, stream, true);
}

int spec_verify_lse(const void *target_logits, const void *draft_logits, const double *draft_lse2,
                    const int32_t *draft_tokens, const float *u_accept, const float *u_resample,
                    const float *temperature, int B, const int32_t *k_offsets, int V, int dtype,
                    int32_t *out_tokens, int32_t *out_num_accepted, const spec_verify_aux_t *aux, void *workspace,
                    size_t workspace_bytes, void *stream) {
    if (B > 0 && !draft_lse2) return SPEC_ERR_INVALID_ARG;
    return verify_call(target_logits, draft_logits, draft_lse2, draft_tokens, u_accept, u_resample, temperature, B,
                       k_offsets, V, dtype, out_tokens, out_num_accepted, aux, workspace, workspace_bytes, stream,
                       true);
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
    // The draft pass needs only the draft logits: they go first, and the
    // draft pass runs while the target logits cross the host link on a
    // second stream (started after the draft copy, so that the two copies
    // do not share the link); the verify pass waits for that copy.
    cudaStream_t s2;
    cudaEvent_t ev_draft, ev_target;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        // created on first use; each handle on its own, so that one that
        // failed is tried again by the next call
        if (!st->host_stream &&
            !cuda_ok(cudaStreamCreateWithFlags(&st->host_stream, cudaStreamNonBlocking), "cudaStreamCreate")) {
            st->host_stream = nullptr;
            return SPEC_ERR_CUDA;
        }
        for (cudaEvent_t &e : st->host_ev)
            if (!e && !cuda_ok(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "cudaEventCreate")) {
                e = nullptr;
                return SPEC_ERR_CUDA;
            }
        s2 = st->host_stream;
        ev_draft = st->host_ev[0];
        ev_target = st->host_ev[1];
    }
    cudaMemcpyAsync(d + o_k, k_offsets_host, (B + 1) * 4, cudaMemcpyHostToDevice, s);
    cudaMemcpyAsync(d + o_T, temperature_host, B * 4, cudaMemcpyHostToDevice, s);
    if (R_d) cudaMemcpyAsync(d + o_ud, u_draft_host, R_d * 4, cudaMemcpyHostToDevice, s);
    if (R_d) cudaMemcpyAsync(d + o_d, draft_logits_host, R_d * V * es, cudaMemcpyHostToDevice, s);
    if (R_d) cudaMemcpyAsync(d + o_ua, u_accept_host, R_d * 4, cudaMemcpyHostToDevice, s);
    cudaMemcpyAsync(d + o_ur, u_resample_host, R_t * 4, cudaMemcpyHostToDevice, s);
    if (!cuda_ok(cudaEventRecord(ev_draft, s), "cudaEventRecord") ||
        !cuda_ok(cudaStreamWaitEvent(s2, ev_draft, 0), "cudaStreamWaitEvent"))
        return SPEC_ERR_CUDA;
    cudaMemcpyAsync(d + o_t, target_logits_host, R_t * V * es, cudaMemcpyHostToDevice, s2);
    if (!cuda_ok(cudaEventRecord(ev_target, s2), "cudaEventRecord")) return SPEC_ERR_CUDA;
    rc = round_call(d + o_t, d + o_d, reinterpret_cast<const float *>(d + o_ud),
                    reinterpret_cast<const float *>(d + o_ua), reinterpret_cast<const float *>(d + o_ur),
                    reinterpret_cast<const float *>(d + o_T), B, reinterpret_cast<const int32_t *>(d + o_k), V, dtype,
                    reinterpret_cast<int32_t *>(d + o_xd), reinterpret_cast<int32_t *>(d + o_ot),
                    reinterpret_cast<int32_t *>(d + o_on), stream, ev_target);
    if (rc != SPEC_OK) {
        cudaStreamWaitEvent(s, ev_target, 0);  // the staging buffer stays in use until the copy lands
        cudaStreamSynchronize(s);
        return rc;
    }
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

int spec_shutdown(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    int rc = SPEC_OK;
    for (int d = 0; d < kMaxDevices; ++d) {
        DeviceState &st = g_dev[d];
        if (!st.ws && !st.stage && !st.host_stream) continue;
        if (!cuda_ok(cudaSetDevice(d), "cudaSetDevice") || !cuda_ok(cudaDeviceSynchronize(), "cudaDeviceSynchronize")) {
            rc = SPEC_ERR_CUDA;
            continue;
        }
        if (st.ws) cudaFree(st.ws);
        if (st.stage) cudaFree(st.stage);
        st.ws = nullptr;
        st.ws_bytes = 0;
        st.stage = nullptr;
        st.stage_bytes = 0;
        for (cudaEvent_t &e : st.host_ev) {
            if (e) cudaEventDestroy(e);
            e = nullptr;
        }
        if (st.host_stream) cudaStreamDestroy(st.host_stream);
        st.host_stream = nullptr;
    }
    if (prev >= 0) cudaSetDevice(prev);
    return rc;
}

const char *spec_last_error(void) { return g_last_error; }

}  // extern "C"
