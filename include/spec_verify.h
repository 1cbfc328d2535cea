/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-decoding
 * verify-and-resample library.
 *
 * The operation (three web pages on the method, cited by title and section):
 *   docs.ifdog.com "投机解码", section 投机解码的三步流程 (three-step procedure)
 *     step 3, and section 动手实践 (speculative_decode: sampling and greedy
 *     branches);
 *   bbs.huaweicloud.com "大模型推理无损加速:投机采样(Speculative Decoding)数学原理与
 *     工业级落地实践", section 二.1 (acceptance probability
 *     alpha = min(1, p/q)), section 二.2 (residual distribution
 *     norm(max(0, p - q))), section 三 (speculative_sampling_step);
 *   sxl-space.tk "【大模型】- 推测解码", section 批量推测解码
 *     (BatchSpeculativeDecoder: one verify per sequence of a batch).
 *
 * For each of B sequences with k_b drafted tokens x_0..x_{k_b-1}:
 *   (a) temperature-scaled softmax of every target row (k_b + 1 of them) and
 *       every draft row (k_b), p_i = softmax(z_t,i / T_b), q_i = softmax(z_d,i / T_b);
 *   (b) alpha_i = min(1, p_i(x_i) / q_i(x_i)); x_i is accepted iff
 *       u_accept_i < alpha_i; n_b = index of the first rejection (k_b if none);
 *   (c) if n_b < k_b: one token drawn from norm(max(0, p_j - q_j)) at j = n_b
 *       by inverse CDF (smallest v with C_v > u * Z, ascending vocabulary
 *       order, u = u_resample at position j); else the bonus token drawn from
 *       p_{k_b} the same way;
 *   (d) T_b = 0 (greedy): accept while x_i == argmax p_i (lowest index on
 *       ties); the first mismatch emits argmax p_i, full acceptance emits
 *       argmax p_{k_b}.
 *
 * Common conventions for every entry point below
 *   - Pointers are DEVICE pointers unless the name ends in _host.  The
 *     caller owns every buffer; the library keeps no pointer after a call.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  The return value reports only what the host can
 *     check: argument errors and launch failures.
 *   - Layout, with R_d = k_offsets[B] and R_t = R_d + B (k_offsets is read
 *     on the device, so the host never needs R_d):
 *       k_offsets     int32 [B+1]   k_offsets[0] = 0, 0 <= k_b <= SPEC_MAX_K
 *       target_logits [R_t, V]      row-major; sequence b owns rows
 *                                   o_b .. o_b + k_b with o_b = k_offsets[b] + b
 *                                   (row o_b + i predicts draft position i,
 *                                   row o_b + k_b is the bonus position)
 *       draft_logits  [R_d, V]      sequence b owns rows k_offsets[b] .. +k_b-1
 *       draft_tokens  int32 [R_d]
 *       u_accept      float [R_d]   in [0,1); position i of b uses u_accept[k_offsets[b]+i]
 *       u_resample    float [R_t]   in [0,1); the resample/bonus at position j
 *                                   uses u_resample[o_b + j]; unused ones are ignored
 *       temperature   float [B]     0 = greedy, > 0 sampled
 *       out_tokens    int32 [R_t]   slots o_b .. o_b + k_b: the n_b accepted
 *                                   tokens, the resampled/bonus token, then -1
 *       out_num_accepted int32 [B]  n_b, or -1 for a data error in sequence b
 *   - dtype: SPEC_F32 or SPEC_BF16, for both logit tensors.  Both logit
 *     pointers must be 16-byte aligned and V * sizeof(element) a multiple of
 *     16 (V % 4 == 0 for fp32, V % 8 == 0 for bf16); otherwise
 *     SPEC_ERR_ALIGNMENT.
 *   - Data errors found on the device mark only their sequence
 *     (out_num_accepted[b] = -1, its token slots -1): a draft token outside
 *     [0, V), a temperature < 0 / NaN / inf, a needed logit row holding NaN
 *     or +inf or entirely -inf (a greedy row: holding NaN).  An invalid
 *     k_offsets array (k_offsets[0] != 0, or some k_b outside
 *     [0, SPEC_MAX_K]) fails the whole call on the device: every
 *     out_num_accepted = -1, out_tokens untouched, and the workspace status
 *     word set to SPEC_ERR_INVALID_ARG.
 *   - Time-outs: every device-side wait is bounded (2 s).  A wait that runs
 *     out records SPEC_ERR_TIMEOUT in the workspace status word, and while
 *     that word holds it every verify or draft-sampling call on the
 *     workspace reports all its sequences (rows) as data errors (-1) rather
 *     than outputs that look valid; clear it with spec_workspace_status.
 *     Some kernels' CTAs wait on one another (they are launched no wider
 *     than the GPU holds at once); another workload that keeps SMs busy for
 *     longer than the limit can therefore make a call time out.
 *   - Temperature: every row of sequence b, target and draft, is divided by
 *     T_b before the softmax.
 *   - Randomness is never drawn inside the library: all uniforms are inputs,
 *     so results are reproducible bit for bit.
 *   - Workspace: the entry points without a workspace argument use one
 *     library-owned device workspace per GPU, allocated (cudaMalloc,
 *     synchronous) on the first call that needs a larger one; that first
 *     call therefore must not happen during stream capture.  Concurrent
 *     calls that share a workspace (the library-owned one included) must be
 *     ordered on one stream; calls on independent streams need their own
 *     workspace through the *_ex entry points.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_VERIFY_ABI_VERSION 1
#define SPEC_MAX_K 32        /* drafted positions per sequence */
#define SPEC_MAX_B 4096      /* sequences per call */
#define SPEC_MAX_V (1 << 24) /* vocabulary size */
#define SPEC_MAX_TREE_NODES 64 /* nodes per sequence of a tree verify (root included) */

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype_t;

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = -1,  /* null pointer, B/V/dtype out of range, bad k_offsets (device) */
    SPEC_ERR_ALIGNMENT = -2,    /* logit pointer or row stride not 16-byte aligned */
    SPEC_ERR_CUDA = -3,         /* a CUDA call failed (launch, allocation, copy) */
    SPEC_ERR_TIMEOUT = -4,      /* a bounded device-side wait gave up (device status only) */
    SPEC_ERR_WORKSPACE = -5     /* caller workspace smaller than spec_workspace_bytes() */
} spec_status_t;

/* Optional parity/diagnostic outputs of spec_verify_ex; any field may be NULL.
 * Values are undefined (NaN) where the quantity does not exist. */
typedef struct {
    float *accept_prob;   /* [R_d] alpha_i of every drafted position of a sampled sequence */
    float *residual_mass; /* [B]  Z = sum max(0, p_j - q_j) at the resampled position */
    float *lse_target;    /* [R_t] log-sum-exp of z/T (natural log) per target row */
    float *lse_draft;     /* [R_d] log-sum-exp of z/T per draft row */
} spec_verify_aux_t;

/*
 * Verify-and-resample for B sequences (operations (a)-(d) above).
 * Returns SPEC_OK, or an error code for host-detectable argument errors
 * (nothing is launched then).  B = 0 is a valid no-op.
 */
int spec_verify(const void *target_logits, const void *draft_logits,
                const int32_t *draft_tokens, const float *u_accept,
                const float *u_resample, const float *temperature, int B,
                const int32_t *k_offsets, int V, int dtype, int32_t *out_tokens,
                int32_t *out_num_accepted, void *stream);

/*
 * spec_verify with optional aux outputs and a caller-owned device workspace
 * of at least spec_workspace_bytes(B, V, dtype) bytes (256-byte aligned).
 * workspace == NULL selects the library-owned one.  The workspace needs no
 * initialisation beyond being zero-filled once before its first use.
 */
int spec_verify_ex(const void *target_logits, const void *draft_logits,
                   const int32_t *draft_tokens, const float *u_accept,
                   const float *u_resample, const float *temperature, int B,
                   const int32_t *k_offsets, int V, int dtype, int32_t *out_tokens,
                   int32_t *out_num_accepted, const spec_verify_aux_t *aux,
                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * Draft-side softmax + multinomial (docs.ifdog.com "投机解码", section 动手实践,
 * drafting loop; sxl-space.tk "【大模型】- 推测解码", draft_generate): for every
 * draft row r of sequence b, out_draft_tokens[r] = argmax z (lowest index)
 * if T_b = 0, else the inverse-CDF draw from softmax(z / T_b) at u_draft[r].
 * A row with NaN (or, when sampled, +inf / entirely -inf) or a bad T_b
 * gives -1.  draft_logits [R_d, V], u_draft float [R_d], out int32 [R_d].
 */
int spec_draft_sample(const void *draft_logits, const float *temperature,
                      const float *u_draft, int B, const int32_t *k_offsets, int V,
                      int dtype, int32_t *out_draft_tokens, void *stream);

int spec_draft_sample_ex(const void *draft_logits, const float *temperature,
                         const float *u_draft, int B, const int32_t *k_offsets, int V,
                         int dtype, int32_t *out_draft_tokens, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * Draft sampling that also keeps each draft row's normaliser for the verify
 * step.  docs.ifdog.com "投机解码", section 动手实践: the drafting loop keeps
 * the draft distribution q of every position and step 3 reuses it instead
 * of recomputing it; here only q's normaliser is kept (8 bytes per row),
 * since q(v) = exp(z_v / T_b) / 2^L follows from it and the draft logits.
 *
 * Same arguments and outputs as spec_draft_sample_ex, plus
 *   out_draft_lse2  double [R_d], device: for every sampled row r of
 *                   sequence b, L_r = log2(sum_v exp(z_r,v / T_b)) (the
 *                   natural log-sum-exp divided by ln 2); NaN for greedy
 *                   rows (T_b = 0) and for rows that give token -1.
 * Pass out_draft_lse2 to spec_verify_lse with the same logits, temperature
 * and k_offsets.  SPEC_ERR_INVALID_ARG if out_draft_lse2 is NULL (B > 0).
 */
int spec_draft_sample_lse(const void *draft_logits, const float *temperature,
                          const float *u_draft, int B, const int32_t *k_offsets, int V,
                          int dtype, int32_t *out_draft_tokens, double *out_draft_lse2,
                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_verify_ex with the draft rows' normalisers given (draft_lse2, from
 * spec_draft_sample_lse on the same draft logits, temperature and
 * k_offsets): only the target rows are streamed; of the draft logits it
 * reads the drafted token's logit at each position and the one draft row
 * at a rejected position (the residual max(0, p - q) needs the whole q row
 * there).  With the same inputs its outputs equal spec_verify's bit for
 * bit (both derive L from the same partial sums).  A draft_lse2 entry that
 * is NaN or infinite, for a position of a sampled sequence, is a data error
 * of that sequence.  aux, workspace: as in spec_verify_ex (aux->lse_draft
 * echoes draft_lse2 * ln 2).  SPEC_ERR_INVALID_ARG if draft_lse2 is NULL
 * (B > 0).
 */
int spec_verify_lse(const void *target_logits, const void *draft_logits,
                    const double *draft_lse2, const int32_t *draft_tokens,
                    const float *u_accept, const float *u_resample,
                    const float *temperature, int B, const int32_t *k_offsets, int V,
                    int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
                    const spec_verify_aux_t *aux, void *workspace,
                    size_t workspace_bytes, void *stream);

/*
 * One sampling round on DEVICE buffers: spec_draft_sample_lse (filling
 * out_draft_tokens [R_d]) and then spec_verify_lse on those tokens, with the
 * draft rows' normalisers kept in the library-owned workspace between the
 * two passes, so every logit row is read once (plus the two rows at a
 * rejected position).  Arguments as in spec_draft_sample and spec_verify;
 * outputs equal those of spec_draft_sample followed by spec_verify.
 */
int spec_round(const void *target_logits, const void *draft_logits, const float *u_draft,
               const float *u_accept, const float *u_resample, const float *temperature,
               int B, const int32_t *k_offsets, int V, int dtype,
               int32_t *out_draft_tokens, int32_t *out_tokens,
               int32_t *out_num_accepted, void *stream);

/*
 * One sampling round from HOST memory: copies the inputs to the device,
 * runs spec_round (draft sampling, which fills the draft tokens, then
 * verify), copies the draft tokens and the verify outputs back, and
 * returns after the stream has finished.  All pointers are host pointers
 * (pinned memory gives full copy bandwidth); k_offsets [B+1] is read on the
 * host to size the copies.  Uses a library-owned device staging area that
 * grows on demand (synchronous cudaMalloc).  The draft-side inputs are
 * copied first on `stream`; the target logits follow on a library-owned
 * second stream of the device (ordered after everything enqueued on
 * `stream` before the call), so the draft pass runs while they are still
 * crossing the host link.  The staging area and that stream are shared by
 * all callers on a device: calls must not overlap (one host thread at a
 * time per device).
 */
int spec_round_host(const void *target_logits_host, const void *draft_logits_host,
                    const float *u_draft_host, const float *u_accept_host,
                    const float *u_resample_host, const float *temperature_host, int B,
                    const int32_t *k_offsets_host, int V, int dtype,
                    int32_t *out_draft_tokens_host, int32_t *out_tokens_host,
                    int32_t *out_num_accepted_host, void *stream);

/*
 * Allocation-free spec_verify.  The pages have no counterpart: it is a
 * deployment convenience of this library.
 *
 * For callers that cannot allocate device memory at the moment they
 * verify: a serving loop that keeps cudaMalloc off its hot path so that
 * latency stays predictable, or a runtime whose own memory pool owns all
 * device memory and hands out none.  Arguments, layout, outputs and
 * data-error behaviour are those of spec_verify; the caller still provides
 * every input and output buffer.  The scratch memory the kernels need is a
 * fixed array compiled into the library (SPEC_NOALLOC_SCRATCH_BYTES = 48
 * MiB), so the call performs no cudaMalloc, cudaFree or other allocation.
 *   - The array is held on a device from this entry point's first call
 *     there until the process exits (with the CUDA runtime's default lazy
 *     module loading; with CUDA_MODULE_LOADING=EAGER every device that
 *     loads the library holds it).
 *   - A call whose scratch need, spec_noalloc_bytes(B, V, dtype), exceeds
 *     SPEC_NOALLOC_SCRATCH_BYTES is rejected with SPEC_ERR_WORKSPACE before
 *     anything is launched (spec_last_error() names the sizes).  The limit
 *     covers, e.g., B = 512 at V = 152064 in bf16.
 *   - The first call on each device does a one-time set-up: it looks up the
 *     array's device address (with that device current).  Make that first
 *     call before any stream capture.
 *   - All calls share the one array: calls that may overlap on the GPU (on
 *     different streams without ordering) race and give wrong results.
 *     Order them on one stream.
 *   - The array keeps the previous call's contents; each call first clears
 *     (cudaMemsetAsync) the words that must start at zero, the status word
 *     among them, so a time-out shows in that call's outputs only (every
 *     sequence -1; see Time-outs above).
 */
#define SPEC_NOALLOC_SCRATCH_BYTES ((size_t)48 << 20)
int spec_verify_noalloc(const void *target_logits, const void *draft_logits,
                        const int32_t *draft_tokens, const float *u_accept,
                        const float *u_resample, const float *temperature, int B,
                        const int32_t *k_offsets, int V, int dtype, int32_t *out_tokens,
                        int32_t *out_num_accepted, void *stream);

/*
 * Tree (multi-candidate) verify.  docs.ifdog.com "投机解码", 进阶方案: Medusa
 * and EAGLE verify a tree of drafted candidates in one target forward; the
 * pages give no acceptance rule for it.  The rule implemented is the
 * single-candidate test of 投机解码的三步流程 step 3 (bbs.huaweicloud.com
 * 二.1-二.2) applied to several candidates in turn: at node u, with
 * p = softmax(target row u / T_b) and q = softmax(draft row u / T_b), u's
 * children c_1 < c_2 < ... (ascending node index; their tokens must be
 * independent draws from q, e.g. from spec_tree_draft_sample) are tested in
 * order: c_j is accepted iff u_accept[c_j] < min(1, p_j-1(x)/q(x)), with
 * p_0 = p and p_j = norm(max(0, p_j-1 - q)) after each rejection.  An
 * accepted child becomes u.  When every child of u is rejected, one token
 * is drawn from the last residual at u_resample[u] (inverse CDF, ascending
 * vocabulary); at a leaf the bonus token is drawn from p.  T_b = 0: the
 * first child whose token is argmax p (lowest index on ties) is accepted,
 * else argmax p is emitted.  Each emitted token follows the target
 * distribution of its node.
 *
 * Layout (N = node_offsets[B] nodes; every pointer a device pointer):
 *   node_offsets  int32 [B+1]  node_offsets[0] = 0; sequence b owns nodes
 *                              node_offsets[b] .. node_offsets[b+1]-1, 1 to
 *                              SPEC_MAX_TREE_NODES of them, the first is
 *                              its root
 *   parent        int32 [N]    -1 for a root; otherwise an earlier node of
 *                              the same sequence
 *   tokens        int32 [N]    each non-root node's drafted token (a
 *                              root's is ignored)
 *   target_logits [N, V]       row g: the target logits after the path to
 *                              node g (the distribution of g's children)
 *   draft_logits  [N, V]       row g: the draft logits after the path to g
 *                              (rows of leaves are not read)
 *   u_accept      float [N]    the test of node g; u_resample float [N]: a
 *                              draw at node g
 *   out_tokens    int32 [N]    from slot node_offsets[b]: the accepted path's
 *                              tokens, the drawn token, then -1
 *   out_num_accepted int32 [B] accepted tokens, -1 for a data error
 *   out_last_node int32 [B]    the node where the walk ended (NULL: skip)
 * N is passed by the host as well (it sizes the library workspace) and must
 * equal node_offsets[B].  A data error (bad temperature, token or parent
 * array, or a needed row with NaN / +inf / all -inf) marks only its
 * sequence; an invalid node_offsets array (or node_offsets[B] != N) fails
 * the whole call on the device (every out_num_accepted = -1, status
 * SPEC_ERR_INVALID_ARG).  Host errors: SPEC_ERR_INVALID_ARG for null
 * pointers or N outside [B, B * SPEC_MAX_TREE_NODES], plus the errors of
 * spec_verify.  Uses the library-owned workspace (calls ordered on one
 * stream, as for spec_verify).  Each tree is walked by a cluster of two
 * CTAs (thread-block clusters); a device-side wait between them that runs
 * out (2 s) marks the tree -1 and sets SPEC_ERR_TIMEOUT in the status word.
 */
int spec_tree_verify(const void *target_logits, const void *draft_logits,
                     const int32_t *node_offsets, const int32_t *parent,
                     const int32_t *tokens, const float *u_accept,
                     const float *u_resample, const float *temperature, int B, int N,
                     int V, int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
                     int32_t *out_last_node, void *stream);

/*
 * Tree drafting: each non-root node g takes its token from the draft row of
 * its parent (softmax(z / T_b)): the inverse-CDF draw at u_draft[g], or
 * argmax z when T_b = 0, so that siblings are independent draws from one
 * distribution, as spec_tree_verify requires.  Roots and invalid rows give
 * -1.  Layout and errors as for spec_tree_verify; u_draft float [N].
 */
int spec_tree_draft_sample(const void *draft_logits, const int32_t *node_offsets,
                           const int32_t *parent, const float *temperature,
                           const float *u_draft, int B, int N, int V, int dtype,
                           int32_t *out_tokens, void *stream);

/*
 * Vocab-sharded verify.  The vocabulary is split over G ranks (as when a
 * tensor-parallel LM head leaves each GPU the logits of its own columns):
 * rank r holds columns [V_r, V_{r+1}) of every target and draft row, with
 * shard_bounds = {V_0 = 0 < V_1 < ... < V_G = V}.  The result is that of
 * spec_verify on the whole rows (operations (a)-(d) at the top of this
 * file); only the floating-point order of the sums differs.  One verify is
 * three calls per rank with two exchanges between them, which the caller
 * makes (an all-gather each, e.g. NCCL).  (docs.ifdog.com "投机解码",
 * 实践要点, names the extra synchronisation of multi-GPU tensor parallelism
 * as a cost; the split below is this library's design, not the pages'.)
 *
 *   1. spec_shard_stats  -> out_stats, one record per row of this shard;
 *      all-gather: all_stats = the G ranks' out_stats, rank-major.
 *   2. spec_shard_decide -> every rank combines the G records of each row
 *      in rank order (so all ranks take the same decisions): accept test,
 *      n_b, the accepted prefix, the greedy token; for a draw, this rank's
 *      share of its mass: out_mass [B][2] = { mass of the distribution to
 *      draw from (the residual max(0, p_j - q_j) at j = n_b, or p_{k_b}),
 *      mass of p at position n_b } over this rank's columns;
 *      all-gather: all_mass = the G ranks' out_mass, rank-major.
 *   3. spec_shard_draw   -> Z = sum of the G masses (in rank order), target
 *      u * Z; the rank whose columns hold the crossing of the cumulative
 *      mass draws inside its columns and writes the token; the others leave
 *      -1 in that slot.  If Z is 0 the draw uses the second mass, i.e. p
 *      (as spec_verify does).
 *   The caller then combines out_tokens over ranks with an element-wise
 *   maximum (all-reduce MAX): accepted tokens and greedy tokens are equal
 *   on every rank, and the drawn token is -1 everywhere but on its owner.
 *   out_num_accepted is equal on every rank after step 2.
 *
 * The three calls of one verify must use the same workspace (device,
 * 256-byte aligned, spec_shard_workspace_bytes(B, V_{r+1} - V_r, dtype)
 * bytes, owned by the caller, zero-filled before its first use so that its
 * status word reads SPEC_OK), unmodified in between, and the same B,
 * k_offsets, temperature, shard_bounds and rank.
 *
 *   target_shard  [R_t, Vs]   rank r's columns of the target rows, row-major
 *                             (Vs = V_{r+1} - V_r); draft_shard [R_d, Vs]
 *   draft_tokens, u_accept, u_resample, temperature, k_offsets: as for
 *                             spec_verify (global token ids), the same on
 *                             every rank
 *   shard_bounds  HOST int32 [G+1], 1 <= G <= SPEC_MAX_SHARDS, 0 <= rank < G;
 *                             every shard width (V_{r+1} - V_r) a multiple
 *                             of 4 (fp32) or 8 (bf16)
 *   out_stats     spec_shard_stat_t [R_t + R_d]: target row t at index t,
 *                             draft row d at index R_t + d
 *   all_stats     spec_shard_stat_t [G][R_t + R_d], 16-byte aligned
 *   out_mass      double [B][2];  all_mass double [G][B][2], 16-byte aligned
 *   out_tokens, out_num_accepted: as for spec_verify
 * Errors: as for spec_verify (data errors mark their sequence on every
 * rank; an invalid k_offsets array fails the call on the device), plus
 * SPEC_ERR_INVALID_ARG for bad shard_bounds / G / rank or a NULL
 * workspace, SPEC_ERR_WORKSPACE for a small one.
 */
#define SPEC_MAX_SHARDS 64

/* One row's statistics over one shard's columns (16 bytes).
 *   sampled row: m = max over the columns of z * log2(e) / T (-inf when
 *     every column is -inf), s = sum of 2^(z * log2(e) / T - m) (0 then;
 *     NaN when a column holds NaN or +inf), zx = the logit of the row's
 *     drafted token if this shard holds that column (else 0), arg = 0;
 *   greedy row: m = the largest logit, arg = global column of its first
 *     occurrence (-1 when a column holds NaN), s = zx = 0;
 *   a row the verify does not need: m = -inf, s = NaN, zx = 0, arg = -1. */
typedef struct {
    float m;
    float s;
    float zx;
    int32_t arg;
} spec_shard_stat_t;

size_t spec_shard_workspace_bytes(int B, int Vs, int dtype);

int spec_shard_stats(const void *target_shard, const void *draft_shard,
                     const int32_t *draft_tokens, const float *temperature, int B,
                     const int32_t *k_offsets, const int32_t *shard_bounds, int G, int rank,
                     int dtype, spec_shard_stat_t *out_stats, void *workspace,
                     size_t workspace_bytes, void *stream);

int spec_shard_decide(const void *target_shard, const void *draft_shard,
                      const spec_shard_stat_t *all_stats, const int32_t *draft_tokens,
                      const float *u_accept, const float *temperature, int B,
                      const int32_t *k_offsets, const int32_t *shard_bounds, int G, int rank,
                      int dtype, int32_t *out_tokens, int32_t *out_num_accepted,
                      double *out_mass, void *workspace, size_t workspace_bytes, void *stream);

int spec_shard_draw(const void *target_shard, const void *draft_shard, const double *all_mass,
                    const float *u_resample, int B, const int32_t *k_offsets,
                    const int32_t *shard_bounds, int G, int rank, int dtype,
                    int32_t *out_tokens, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Adaptive draft length (sxl-space.tk "【大模型】- 推测解码", 自适应推测解码:
 * AdaptiveSpeculativeDecoder.adapt_k), per sequence and on the device.
 *
 * After each round the sequence's acceptance rate n_b / k_b (accepted drafted
 * tokens over the round's draft length) joins its history; once the history
 * holds 10 rates, a mean of the last 10 above 0.8 lengthens the next round's
 * draft by one (at most max_k), below 0.5 shortens it by one (at least
 * min_k).  The first length is (min_k + max_k) / 2, rounded down.  The mean
 * is compared exactly (rates are rationals with denominators <= 32), so a
 * mean of exactly 0.8 or 0.5 changes nothing.  A sequence whose round
 * carries no rate (num_accepted < 0, a draft length of 0, or num_accepted
 * greater than its length) keeps its state.
 *
 *   state          device buffer of spec_adapt_state_bytes(B) bytes, 8-byte
 *                  aligned, owned by the caller; spec_adapt_init fills it.
 *   num_accepted   [B] int32, device: out_num_accepted of the round just
 *                  verified, which must have used the lengths of the last
 *                  k_offsets_out this state produced.
 *   k_offsets_out  [B+1] int32, device: the next round's k_offsets.
 *   min_k, max_k   1 <= min_k <= max_k <= SPEC_MAX_K (the pages use 1, 10).
 * Both calls are asynchronous on `stream` (one single-block kernel each) and
 * return only host-checkable errors: SPEC_ERR_INVALID_ARG (null pointers,
 * B outside 1..SPEC_MAX_B, bad bounds), SPEC_ERR_ALIGNMENT, SPEC_ERR_CUDA.
 */
size_t spec_adapt_state_bytes(int B);
int spec_adapt_init(void *state, int B, int min_k, int max_k, int32_t *k_offsets_out, void *stream);
int spec_adapt_update(void *state, const int32_t *num_accepted, int B, int min_k, int max_k,
                      int32_t *k_offsets_out, void *stream);

/* Bytes of device workspace needed by spec_verify_ex / spec_draft_sample_ex
 * for a call with B sequences over vocabulary V (0 for invalid arguments). */
size_t spec_workspace_bytes(int B, int V, int dtype);

/* Bytes of the fixed scratch array a spec_verify_noalloc call with B
 * sequences over vocabulary V uses (0 for invalid arguments; the same as
 * spec_workspace_bytes, as both run the same kernels); the call is refused
 * when this exceeds SPEC_NOALLOC_SCRATCH_BYTES.  Host only. */
size_t spec_noalloc_bytes(int B, int V, int dtype);

/*
 * Device status word of a workspace (NULL: the library-owned one of the
 * current device): SPEC_OK or the first device-side error (SPEC_ERR_TIMEOUT,
 * SPEC_ERR_INVALID_ARG) since it was last cleared.  Synchronous (it waits
 * for the device).  clear != 0 resets it to SPEC_OK (needed after a
 * time-out: until then, calls on the workspace report every sequence -1).
 */
int spec_workspace_status(const void *workspace, int *status_out, int clear);

/*
 * Self-check of the device-side bounded waits (for tests): one kernel waits
 * on an mbarrier that nothing arrives at, then on a meeting counter that
 * nothing completes, then for a residual pair that is never listed, as the
 * streaming kernels, the tree walk and the deferred epilogue would when a
 * copy, a peer CTA or a deciding CTA never comes.  Each wait gives up after
 * its limit (2 s each) and SPEC_ERR_TIMEOUT is recorded in the status word
 * of `workspace` (device, >= 256 bytes, 16-byte aligned, zero-filled; word 8
 * gets 7 when all three waits gave up).  Nothing traps or faults; the
 * context stays usable.  Asynchronous on `stream`; takes about 6 s on the
 * device.
 */
int spec_selfcheck_wait_timeout(void *workspace, size_t workspace_bytes, void *stream);

/* Human-readable name of a status code (static string). */
const char *spec_status_string(int status);

/* SPEC_VERIFY_ABI_VERSION of the loaded library. */
int spec_abi_version(void);

/* Frees the library-owned device buffers of every device (the workspaces of
 * the entry points without a workspace argument, and the staging buffer of
 * spec_round_host) and spec_round_host's copy stream and events, after
 * waiting for each such device.  Later calls create them again.  Must not run while another thread calls the
 * library or during stream capture.  Returns SPEC_OK, or SPEC_ERR_CUDA if a
 * device could not be synchronised (its buffers are then kept). */
int spec_shutdown(void);

/* Description of the last CUDA failure (the call and the CUDA error name)
 * seen by the calling thread, or "" if none.  Static per-thread storage. */
const char *spec_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
