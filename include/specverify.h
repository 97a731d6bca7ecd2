/*
 * specverify.h - C ABI of libspecverify.so: target-model verification attention
 * for long-context speculative decoding, on one GB300 (sm_103a).
 *
 * The operations (source pages, by title and section):
 *   - "Riepilogo Tecnico: Dustin", Metodologia section 1 (Aggregazione Ibrida
 *     dell'Attenzione): the verification set I_verify of fixed size = an
 *     attention-sink prefix + a window of recent tokens + the top-m tokens by
 *     the draft-lookahead score + a fill by the target-historical score.
 *   - Dustin, Metodologia section 3 (Workflow di Verifica), steps 3-4: the
 *     target verifies the draft tokens against the cache restricted to the
 *     selected tokens; the full cache stays in memory (nothing is evicted).
 *   - "LongSpec", section 2.C (Hybrid Tree Attention): attention is split into
 *     the cache part (no mask) and the speculative part (tree mask), and the
 *     two are combined exactly with the log-sum-exp trick.
 *   Around that path, the steps before and after it:
 *   - Dustin, Metodologia sections 1-2: the target-historical importance of
 *     each cache token on a few semantic retrieval heads (spec_importance_scores).
 *   - Dustin, Workflow di Verifica step 5, under greedy decoding (BASTION,
 *     Risultati Sperimentali): the accepted draft tokens join the cache
 *     (spec_accept_commit).
 *   - "BASTION", Metodologia sections 1-3: the hardware-aware choice of the
 *     next tree's size (spec_budget_plan, on the host).
 *
 * Conventions shared by every entry point:
 *   - bf16 tensors are passed as `const uint16_t*` holding bf16 bit patterns.
 *   - Every tensor pointer is a DEVICE pointer on the calling thread's current
 *     CUDA device, except where a comment says "host".
 *   - Ownership: the caller owns every buffer; the library allocates nothing
 *     and keeps no state between calls, apart from the two measurement aids at
 *     the end of this file (per calling thread).
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous. Results are valid once the stream reaches
 *     the point after the call.
 *   - Host-side checks return synchronously, before anything is enqueued:
 *     SPEC_ERR_INVALID_ARG for null/misaligned pointers or impossible sizes,
 *     SPEC_ERR_UNSUPPORTED for head_dim != 128 or a device that is not
 *     compute capability 10.3, SPEC_ERR_WORKSPACE for a workspace that is
 *     too small. A failed launch returns SPEC_ERR_CUDA.
 *   - Data-dependent errors found on the device (a parent outside [-1, i), an
 *     index that is out of range or not strictly ascending, a context length
 *     outside [0, L]) never trap: the offending entry is treated as masked,
 *     the rest of the result is computed, and SPEC_ERR_BAD_INPUT is recorded
 *     in the workspace's status word. Read it with spec_read_device_status().
 *     Each call clears the status word of its workspace first. The calls
 *     without a workspace (spec_accept_commit, spec_importance_scores, the
 *     no-alloc entry point) record it in a caller-given device word instead.
 *   - Layouts (row-major, innermost last):
 *       q        [B, N, Hq, d]           bf16   (query of draft node i, head h)
 *       k_cache, v_cache [B, Hkv, L, d]  bf16   element (b,h,t,c) at
 *                b*kv_stride_b + h*kv_stride_h + t*kv_stride_t + c
 *                (strides in elements, multiples of 8; d contiguous)
 *       k_draft, v_draft [B, N, Hkv, d]  bf16   (this step's draft tokens)
 *       parent   [B, N] int32: parent[b,i] in [-1, i); -1 = child of the last
 *                cache token. Node i sees draft node j iff j == i or j is an
 *                ancestor of i.
 *       out      [B, N, Hq, d] fp32, lse [B, N, Hq] fp32 (natural log of the
 *                sum of exp(scale * q.k) over every key the row sees).
 *     Query head h reads KV head h / (Hq / Hkv) (grouped-query attention).
 *   - A row that sees no key at all gets out = 0 and lse = -inf.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1,
    SPEC_ERR_UNSUPPORTED = 2,
    SPEC_ERR_CUDA = 3,
    SPEC_ERR_WORKSPACE = 4,
    SPEC_ERR_BAD_INPUT = 5,
    SPEC_ERR_TIMEOUT = 6
} spec_status_t;

/* Human-readable name of a status code (static string, never NULL). */
const char *spec_status_string(int status);

/* ------------------------------------------------------------------------ */
/* Hybrid top-k selection of I_verify (Dustin, Metodologia section 1).
 *
 * For each sequence b with n = ctx_lens[b] (or L when ctx_lens is NULL):
 *   if budget >= n: idx[b] = 0, 1, ..., n-1, then -1 padding (full context);
 *   else, with S' = min(sink, n), W' = min(window, n - S'):
 *     C = [0, S') u [n - W', n)                   (sink and local window)
 *     R = the other tokens
 *     D = the min(top_m, budget - |C|, |R|) best of R by draft_score
 *     F = the budget - |C| - |D| best of R \ D by target_score
 *     idx[b] = C u D u F in ascending order (exactly `budget` entries).
 *   "Best" = larger score; -0 == +0; NaN ranks below every number; ties go
 *   to the lower index. The result is therefore unique (bit-exact).
 *
 * draft_score, target_score: fp32 [B, ld] device, row b at b*ld, L <= ld.
 * ctx_lens: int32 [B] device, or NULL.
 * idx: int32 [B, budget] device (output). count: int32 [B] device (output:
 *   number of valid entries, min(budget, n)) or NULL.
 * Requires 1 <= budget, 0 <= sink, window, top_m, sink + window <= budget,
 * 1 <= L <= 1572864.
 * workspace: device, >= spec_select_workspace_size() bytes, 256-byte aligned.
 * The selection kernel allows a grid launched behind it with programmatic stream
 * serialisation to start at once; such a grid must wait for it (griddepcontrol.wait)
 * before reading idx or count. The verify calls do: their first kernel waits, and so
 * their set-up runs on the SMs the selection leaves free.
 */
size_t spec_select_workspace_size(int B, int L, int budget);
spec_status_t spec_select_topk(const float *draft_score, const float *target_score, int64_t ld,
                               int B, int L, const int32_t *ctx_lens, int sink, int window,
                               int top_m, int budget, int32_t *idx, int32_t *count,
                               void *workspace, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------ */
/* Dense verification attention (full cache + tree-masked draft block).
 *
 * out[b,i,h] = softmax over { cache tokens 0..n-1 } u { draft nodes visible
 * to i } of scale * q.k, applied to the matching V rows, where
 * n = ctx_lens[b] (or L). The cache part is a split-KV pass over the whole
 * GPU; the partial results and the tree part are merged by log-sum-exp
 * (LongSpec section 2.C).
 *
 * If k_draft == NULL (then v_draft and parent must be NULL too), the tree part
 * is skipped: the result is the cache-only part, ready to be combined with
 * another part through spec_lse_merge.
 * Requires d == 128, Hq % Hkv == 0, 1 <= N <= 4096, B >= 1, L >= 0,
 * 16-byte aligned tensors; out/lse must not overlap the inputs.
 * workspace: device, >= spec_verify_workspace_size(B, N, Hq, Hkv, d, L)
 * bytes, 256-byte aligned; holds the split partials and the status word.
 */
size_t spec_verify_workspace_size(int B, int N, int Hq, int Hkv, int d, int L_or_budget);

/* The split plan the tensor-core cache kernel follows for a verify call of this shape (a
 * read-only view of host logic: it launches nothing, needs no GPU and allocates nothing). The
 * cache part of a call is cut into units (b, h_kv, group of BM query rows; row group first:
 * u = rg * B * Hkv + b * Hkv + h_kv) of tiles_per_unit 128-token tiles, numbered unit by unit;
 * CTA c covers tiles [starts[c], starts[c + 1]).
 *
 * L_or_budget: L for spec_verify_attn, budget for spec_verify_attn_sparse. sms: the
 * multiprocessor count to plan for (one CTA per SM at most). sparse: nonzero for a sparse call.
 * starts: int32 host array of max_starts entries; receives starts[0..ctas], starts[ctas] = the
 * tile total. info: int32 host array of 8: units, tiles_per_unit, row_groups, BM (query rows per
 * unit), split_tiles (1: the two pipes take alternate tiles of <= 128 rows), pipes (partial
 * slots per CTA and unit), slots (partial slots of the workspace), uniform (1: an even cut).
 * Returns the CTA count (>= 1), or -SPEC_ERR_INVALID_ARG (bad shape, NULL arrays, max_starts
 * below ctas + 1) or -SPEC_ERR_UNSUPPORTED (a shape the verify calls refuse as too large).
 */
int spec_split_plan(int B, int N, int Hq, int Hkv, int L_or_budget, int sms, int sparse, int32_t *starts,
                    int max_starts, int32_t *info);
spec_status_t spec_verify_attn(const uint16_t *q, const uint16_t *k_cache,
                               const uint16_t *v_cache, int64_t kv_stride_b,
                               int64_t kv_stride_h, int64_t kv_stride_t,
                               const uint16_t *k_draft, const uint16_t *v_draft,
                               const int32_t *parent, int B, int N, int Hq, int Hkv, int d, int L,
                               const int32_t *ctx_lens, float scale, float *out, float *lse,
                               void *workspace, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------ */
/* Sparse verification attention (Dustin, Workflow di Verifica steps 3-4).
 *
 * Same as spec_verify_attn, but the cache part only reads the rows
 * idx[b, 0..budget) (shared by all heads of sequence b). Entry j is used iff
 * 0 <= idx[b,j] < n and (j == 0 or idx[b,j] > idx[b,j-1]); -1 entries are
 * padding and are skipped silently; any other unused entry also records
 * SPEC_ERR_BAD_INPUT. The workspace size is
 * spec_verify_workspace_size(B, N, Hq, Hkv, d, budget). The cache strides
 * follow the rule of spec_verify_attn (multiples of 8 elements): every
 * gathered row starts on a 16-byte boundary.
 */
spec_status_t spec_verify_attn_sparse(const uint16_t *q, const uint16_t *k_cache,
                                      const uint16_t *v_cache, int64_t kv_stride_b,
                                      int64_t kv_stride_h, int64_t kv_stride_t,
                                      const uint16_t *k_draft, const uint16_t *v_draft,
                                      const int32_t *parent, int B, int N, int Hq, int Hkv, int d,
                                      int L, const int32_t *ctx_lens, float scale,
                                      const int32_t *idx, int budget, float *out, float *lse,
                                      void *workspace, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------ */
/* Verification attention with extensions: a paged KV cache, an fp8 KV cache and a
 * bf16 output.
 *
 * The source pages use neither; they are layouts of serving engines. With
 * idx == NULL this is spec_verify_attn, with idx != NULL (`budget` entries
 * per sequence) spec_verify_attn_sparse, and ext == NULL changes nothing.
 *
 * ext->block_table != NULL: the cache is paged. The cache of sequence b is
 * stored in fixed-size blocks of a pool: token t is row t % block_size of
 * pool block block_table[b * table_ld + t / block_size], and the three
 * strides describe the pools: element (blk, h, o, c) at blk * kv_stride_b +
 * h * kv_stride_h + o * kv_stride_t + c (elements, multiples of 8; d
 * contiguous), 0 <= blk < num_blocks. Only the blocks that hold tokens below
 * n = ctx_lens[b] are read; a block entry outside [0, num_blocks) hides its
 * tokens and sets SPEC_ERR_BAD_INPUT in the status word. block_table: int32
 * [B, table_ld] device, table_ld >= ceil(L / block_size). Requires
 * kv_stride_t >= 1 and, with idx, kv_stride_b a multiple of kv_stride_t and
 * num_blocks * (kv_stride_b / kv_stride_t) below 2^31 (else
 * SPEC_ERR_UNSUPPORTED). The dense tensor-core path takes block sizes that
 * are multiples of 128 (others run on the warp-level kernel).
 * ext->out_dtype == SPEC_OUT_BF16: out is bf16 [B, N, Hq, d] (the fp32 result
 * rounded to nearest even); lse stays fp32.
 * ext->kv_dtype == SPEC_KV_E4M3: k_cache and v_cache (contiguous or paged)
 * hold E4M3 codes of the OCP 8-bit floating-point formats, one byte an
 * element (pass the byte arrays through the uint16_t pointers; the strides
 * count bytes and must be multiples of 16). The value of element (b, h, t, c)
 * is the code's number times k_scale[b * Hkv + h] (v_scale for V): fp32
 * device arrays [B * Hkv], 4-byte aligned. Queries and the draft block stay
 * bf16. The codes are converted to bf16 in shared memory (exact: every E4M3
 * number is a bf16 number; a NaN code gives NaN) and the scales fold into the
 * softmax scale and the partial's normalisation; dense contiguous caches with
 * G a divisor of 128 run on the tcgen05 kernel, the other forms on the
 * warp-level tensor-core kernel.
 * workspace: >= spec_verify_workspace_size(B, N, Hq, Hkv, d, idx ? budget : L).
 */
typedef enum { SPEC_OUT_F32 = 0, SPEC_OUT_BF16 = 1 } spec_out_dtype_t;
typedef enum { SPEC_KV_BF16 = 0, SPEC_KV_E4M3 = 1 } spec_kv_dtype_t;
typedef struct {
    const int32_t *block_table; /* NULL: the contiguous cache of spec_verify_attn */
    int64_t table_ld;
    int block_size;
    int64_t num_blocks;
    int out_dtype;        /* spec_out_dtype_t */
    int kv_dtype;         /* spec_kv_dtype_t */
    const float *k_scale; /* E4M3 only: [B * Hkv] */
    const float *v_scale;
} spec_verify_ext;
spec_status_t spec_verify_attn_ex(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                  int64_t kv_stride_b, int64_t kv_stride_h, int64_t kv_stride_t,
                                  const uint16_t *k_draft, const uint16_t *v_draft,
                                  const int32_t *parent, int B, int N, int Hq, int Hkv, int d, int L,
                                  const int32_t *ctx_lens, float scale, const int32_t *idx,
                                  int budget, const spec_verify_ext *ext, void *out, float *lse,
                                  void *workspace, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------ */
/* Log-sum-exp merge of two normalised attention parts (LongSpec section 2.C):
 *   lse = log(exp(lse_a) + exp(lse_b)),
 *   out = exp(lse_a - lse) * o_a + exp(lse_b - lse) * o_b,
 * per row; two parts that both have lse = -inf give out = 0, lse = -inf.
 * o_a, o_b, out: fp32 [rows, d]; lse_a, lse_b, lse_out: fp32 [rows]; device.
 * out may alias o_a or o_b, lse_out may alias lse_a or lse_b (in place).
 * rows <= 8 * (2^31 - 1) (one warp per row); d >= 1; pointers 4-byte aligned.
 * SPEC_ERR_INVALID_ARG for null or misaligned pointers, rows or d out of range.
 */
spec_status_t spec_lse_merge(const float *o_a, const float *lse_a, const float *o_b,
                             const float *lse_b, float *out, float *lse_out, int64_t rows, int d,
                             void *stream);

/* ------------------------------------------------------------------------ */
/* Target-historical importance of every cache token (Dustin "Metodologia",
 * sections 1-2: the target's attention scores, estimated on a few semantic
 * retrieval heads), the target score the next step's spec_select_topk reads.
 *
 * score[b * ld + t] = sum over the nh query heads heads[0..nh) (device int32;
 * a head listed twice counts twice) and the N draft queries i of
 * exp(scale q[b,i,h] . k[b, h / G, t] - lse[b,i,h]) for t < ctx_lens[b] (all L
 * when ctx_lens is NULL), and 0 for ctx_lens[b] <= t < L. q and the cache as
 * for spec_verify_attn; lse [B, N, Hq] fp32 as spec_verify_attn returns it
 * (rows with lse = -inf add nothing). score: fp32 device, ld >= L. A head
 * index outside [0, Hq) adds nothing and sets SPEC_ERR_BAD_INPUT in *status
 * (device int32, written whole by the call: SPEC_OK, or SPEC_ERR_BAD_INPUT for a
 * listed head outside [0, Hq), or SPEC_ERR_TIMEOUT; may be NULL).
 * Requires d == 128 and N <= 512 (else SPEC_ERR_UNSUPPORTED), 1 <= B <= 65535,
 * Hq % Hkv == 0, 16-byte aligned q and cache.
 */
spec_status_t spec_importance_scores(const uint16_t *q, const uint16_t *k_cache,
                                     int64_t kv_stride_b, int64_t kv_stride_h,
                                     int64_t kv_stride_t, const float *lse, const int32_t *heads,
                                     int nh, int B, int N, int Hq, int Hkv, int d, int L,
                                     const int32_t *ctx_lens, float scale, float *score, int64_t ld,
                                     int32_t *status, void *stream);

/* ------------------------------------------------------------------------ */
/* Tree size for the next step from BASTION's hardware-aware budget controller
 * ("Metodologia", sections 1-3). Runs on the host: every pointer is a host
 * pointer and the call is synchronous.
 *
 * marginals [K, C] (row-major, values in [0, 1]): the drafter's probability of
 * candidate c at tree depth k + 1. A node at depth d reached through
 * candidates c_1..c_d scores rho = prod_k marginals[k - 1][c_k]; the tree grows
 * best-first (largest rho next, ties to the candidate that entered the
 * frontier first; a node's children enter in candidate order) up to n_max
 * nodes. T_verify(N) = a T_roof(N) + c with T_roof(N) = max((bytes0 +
 * bytes_per_node N) / bw, flops_per_node N / peak) (seconds, or any unit used
 * throughout) and (a, c) the least-squares fit of cal_t on T_roof(cal_n) over
 * the n_cal >= 1 measured samples (ratio of the means, c = 0, when the samples
 * give fewer than two distinct T_roof). S(N) = (sum of the first N rho) l_ar /
 * (t_draft + T_verify(N)); the tree grows one node at a time and *n_chosen is
 * the last N before S first decreases (or the last N grown).
 * Outputs (caller-owned host arrays of n_max entries): parents (-1 = root),
 * depth (1-based), cand, rho of the *n_eval nodes grown; speedup[N - 1] =
 * S(N) for N <= *n_eval; calib[0] = a, calib[1] = c.
 * SPEC_ERR_INVALID_ARG for null pointers, K, C, n_max or n_cal below 1,
 * non-finite inputs, bw or peak <= 0, marginals outside [0, 1], or a step
 * cost t_draft + T_verify(N) <= 0.
 */
spec_status_t spec_budget_plan(const double *marginals, int K, int C, int n_max, double t_draft,
                               double l_ar, double bytes0, double bytes_per_node,
                               double flops_per_node, double bw, double peak, const double *cal_n,
                               const double *cal_t, int n_cal, int32_t *parents, int32_t *depth,
                               int32_t *cand, double *rho, double *speedup, double *calib,
                               int32_t *n_chosen, int32_t *n_eval);

/* ------------------------------------------------------------------------ */
/* Greedy acceptance of the draft tree and commit of the accepted draft K/V
 * rows into the cache (Dustin "Workflow di Verifica", steps 4-5: accepted
 * tokens join the cache, rejected ones are dropped; greedy decoding as in
 * BASTION "Risultati Sperimentali").
 *
 * draft_token [B, N], parent [B, N] (as for spec_verify_attn) and target_next
 * [B, N + 1]: int32, device. target_next[b, 0] is the target's greedy token
 * after the last committed token, target_next[b, 1 + i] its greedy token after
 * draft node i. From the root, the next accepted node is the lowest-index
 * child c of the current node (parent[c] == current, c > current) whose
 * draft_token equals target_next[b, current + 1]; the walk stops when none
 * does.
 * Outputs (device, int32): accept_path [B, N] = the accepted nodes in order,
 * then -1; accept_len [B]; bonus_token [B] = target_next[b, last + 1].
 * Commit (optional: pass k_cache, v_cache, k_draft, v_draft and ctx_lens all
 * non-NULL, or all NULL): the caches [B, Hkv, L, d] bf16 (element strides as
 * for spec_verify_attn, multiples of 8) receive, at positions ctx_lens[b],
 * ctx_lens[b] + 1, ..., the rows k_draft/v_draft [B, N, Hkv, d] of the
 * accepted nodes, and ctx_lens[b] (device, in/out) grows by the rows copied.
 * Rows past L are not copied and a ctx_lens[b] outside [0, L] commits
 * nothing; both, and a parent outside [-1, i), set SPEC_ERR_BAD_INPUT in
 * *status (device int32, zeroed by the call first; may be NULL).
 * Requires 1 <= N <= 4096, B >= 1, d == 128 (else SPEC_ERR_UNSUPPORTED) and
 * 16-byte aligned caches and drafts. The caller owns every buffer; the call
 * is asynchronous on `stream`.
 */
spec_status_t spec_accept_commit(const int32_t *draft_token, const int32_t *parent,
                                 const int32_t *target_next, int B, int N, int32_t *accept_path,
                                 int32_t *accept_len, int32_t *bonus_token, uint16_t *k_cache,
                                 uint16_t *v_cache, int64_t kv_stride_b, int64_t kv_stride_h,
                                 int64_t kv_stride_t, const uint16_t *k_draft,
                                 const uint16_t *v_draft, int Hkv, int d, int L, int32_t *ctx_lens,
                                 int32_t *status, void *stream);

/* ------------------------------------------------------------------------ */
/* Dense verification attention without a workspace (allocates nothing).
 *
 * The source pages have no counterpart to this entry point: it is a
 * deployment convenience. Some callers cannot allocate device memory at call
 * time - serving engines that reserve almost all of HBM for the KV cache at
 * start-up and allow no later allocation, or hosts that reach this library
 * from a plain C callback with no allocator - so they cannot pass the
 * workspace spec_verify_attn needs. This variant computes the same result,
 * within the parity tolerances (not bit for bit), through the warp-level
 * tensor-core cache kernel (mma.sync) and the same merge kernel, rather than
 * the tcgen05 cache kernel spec_verify_attn uses where the shape allows; its
 * speed differs accordingly. It keeps its scratch (split partials and status
 * word) in a fixed 16 MiB array inside the library, held by every GPU that has
 * loaded the library's device code until the process exits. It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments are those of spec_verify_attn without the workspace, plus
 * status_out: int32 device pointer that receives SPEC_OK or
 * SPEC_ERR_BAD_INPUT for this call's data, or NULL.
 * Limits: the problem's split partials must fit the built-in scratch; larger
 * problems return SPEC_ERR_WORKSPACE (use spec_verify_attn). For example
 * B=4, L=32768, Hq=32, Hkv=8, N=64 fits on a 152-SM GB300; B=8, Hq=64,
 * Hkv=8, N=32 does not.
 * The first call on each device looks up the array's device address (once,
 * with that device current). With lazy module loading (the CUDA default),
 * that lookup is also when the 16 MiB array is placed in device memory, so
 * make the first call on each device before reserving HBM for anything else,
 * and before any stream capture. A failed lookup is remembered: later calls on
 * that device return SPEC_ERR_CUDA.
 * Problems whose split plan would number 2^31 tiles or more return
 * SPEC_ERR_UNSUPPORTED, as spec_verify_attn does.
 * Every call on a device shares the one array: calls that overlap on the GPU
 * (different streams or threads, not ordered by the caller) race with each
 * other and must not be issued.
 */
spec_status_t spec_verify_attn_noalloc(const uint16_t *q, const uint16_t *k_cache,
                                       const uint16_t *v_cache, int64_t kv_stride_b,
                                       int64_t kv_stride_h, int64_t kv_stride_t,
                                       const uint16_t *k_draft, const uint16_t *v_draft,
                                       const int32_t *parent, int B, int N, int Hq, int Hkv,
                                       int d, int L, const int32_t *ctx_lens, float scale,
                                       float *out, float *lse, int32_t *status_out,
                                       void *stream);

/* ------------------------------------------------------------------------ */
/* Synchronises `stream`, then returns the status word that the last call
 * using `workspace` left there: SPEC_OK or SPEC_ERR_BAD_INPUT (or
 * SPEC_ERR_TIMEOUT from a bounded wait that gave up). */
spec_status_t spec_read_device_status(const void *workspace, void *stream);

/* Text of the CUDA error behind the last SPEC_ERR_CUDA this host thread got
 * from the library ("no error" if none). The string is static; do not free. */
const char *spec_last_cuda_error(void);

/* ------------------------------------------------------------------------ */
/* Measurement aids (per calling thread; not needed for normal use).
 *
 * spec_profile_events(start, stop): when both are non-NULL cudaEvent_t
 * handles, each following spec_verify_attn / spec_verify_attn_sparse call
 * records `start` on its stream right before its cache-attention kernel and
 * `stop` right after it, so that the caller can time that kernel alone with
 * cudaEventElapsedTime. Pass NULL, NULL to stop.
 *
 * spec_kernel_launches(): number of CUDA kernels this thread has launched
 * through the library so far (memsets are not counted). */
void spec_profile_events(void *start_event, void *stop_event);
uint64_t spec_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
