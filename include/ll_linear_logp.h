/*
 * ll_linear_logp.h -- C ABI of the GB300-native fused linear log-probability.
 *
 * The operation (RL-Kernel issue #261, "Current production path" and
 * "Current accumulation"; RL-Kernel PR #495, "Summary" and "Behavior changes";
 * Liger-Kernel PR #1324, "Details"):
 *
 *   forward   z = h . W^T (+ b)                              [N, V], never stored
 *             lse[n]  = log sum_v exp z[n, v]
 *             logp[n] = z[n, y_n] - lse[n]   if 0 <= y_n < V, else 0
 *   backward  g = grad_logp[n] * (onehot(y_n) - softmax(z[n, :]))   (never stored)
 *             grad_hidden = g . W          [N, D]
 *             grad_weight = g^T . h        [V, D]  (FP32 by default)
 *             grad_bias   = sum_n g[n, :]  [V]
 *   logits-input variant: the same with the logits [N, V] given.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named as device pointers must be CUDA device (or managed)
 *   memory on one device; the call switches to that device for its duration
 *   and restores the caller's current device before returning.
 * - Every call is asynchronous on `stream` (a cudaStream_t; NULL means the
 *   legacy default stream).  Outputs are valid once the stream reaches the
 *   call.  Arguments are validated on the host before anything is launched;
 *   on an error nothing is launched and no output is touched.  Calls may be
 *   in flight on several streams at once and may be recorded by CUDA stream
 *   capture: work that overlaps a GEMM runs on a library side stream that is
 *   forked from and joined back to `stream` by events.  The first call for a
 *   given dtype and path sets kernel attributes and is best made outside a
 *   capture.
 * - The library never allocates device memory.  The caller owns every buffer,
 *   including the scratch `workspace`, whose size ll_workspace_size() gives.
 *   A workspace must not be shared by calls that may overlap on the GPU.
 * - Row-major, contiguous layouts.  Element types are given by ll_dtype:
 *   hidden, weight and bias share one dtype.  logp, lse and grad_logp are
 *   FP32.  targets are int64.
 * - Targets outside [0, V) (for instance the ignore index -100) give logp = 0
 *   and an exactly +0 gradient row (PR #495, "Behavior changes").
 * - Gradient entries that receive no non-zero contribution are +0, as with a
 *   +0-initialised gradient table (issue #261, "Correctness boundary"); a
 *   row whose grad_logp is +-0 is exactly +0.
 * - Results are deterministic: the same inputs give the same bits.  logp,
 *   lse, grad_hidden and grad_logits of a row do not depend on the other rows
 *   of the batch, on the batch size or on the row's position (batch
 *   invariance, PR #495, "Prior art & reuse decision").
 * - Indexing is 64-bit; N * V and V * D may exceed 2^31.  V must be below
 *   2^31 - 256.
 * - Device-side waits are bounded.  A wait that runs out records
 *   LL_ERR_DEVICE_TIMEOUT in a per-device status word that ll_check_status()
 *   returns; the kernel then returns without hanging the device.
 * - The library keeps per-device state for the life of the process (device
 *   properties, the device address of its status word, kernel attributes).
 *   Do not use it on a device after cudaDeviceReset of that device.
 */
#ifndef LL_LINEAR_LOGP_H
#define LL_LINEAR_LOGP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LL_OK = 0,
    LL_ERR_INVALID_ARG = 1,     /* null pointer where one is required, bad flag  */
    LL_ERR_DTYPE = 2,           /* unsupported dtype or dtype combination        */
    LL_ERR_SHAPE = 3,           /* negative or too large N, D, V, ld             */
    LL_ERR_ALIGN = 4,           /* pointer or row stride not 16-byte aligned     */
    LL_ERR_WORKSPACE = 5,       /* workspace missing, too small or misaligned    */
    LL_ERR_CUDA = 6,            /* a CUDA runtime/driver call failed             */
    LL_ERR_DEVICE_TIMEOUT = 7,  /* a bounded device-side wait ran out            */
    LL_ERR_UNSUPPORTED = 8      /* device is not sm_103 / feature not built      */
} ll_status;

typedef enum { LL_F32 = 0, LL_F16 = 1, LL_BF16 = 2 } ll_dtype;

/*
 * Per-call options of the *_ex entry points (and of the vocab-shard calls).
 * A NULL pointer means every default.  An entry point without _ex is its
 * _ex form with NULL.
 *   temperature  > 0 and finite; default 1.  The distribution is
 *                softmax(z / T): logp = z[y] / T - logsumexp(z / T), lse is
 *                that of z / T, and every gradient carries the 1 / T factor
 *                of d(z / T)/dz (the sampling temperature of RL rollouts;
 *                RL-Kernel PR #495, the vLLM provider evidence at
 *                temperatures 1.0 and 0.7).  T = 1 gives bitwise the
 *                results of the calls without options.
 *   split_s      backward with 16-bit operands: how the off-target part
 *                S = -grad_logp * p / T of g is stored before the
 *                grad_hidden / grad_weight contractions, whose operands are
 *                16-bit.  One 16-bit part loses up to 2^-9 of an entry, which
 *                matters where off-target probabilities are large (peaked
 *                rows, small vocabularies).
 *                0 (default) automatic: S_hi = S rounded, and the rounding
 *                  rest S_lo = S - S_hi (rounded) is kept for the entries
 *                  with p >= 2^-8 only, in pieces of 32 rows x 64 columns;
 *                  the contractions run a second pass over the pieces that
 *                  hold such an entry.  A row's results depend on that row
 *                  alone (batch invariance holds).  Flat distributions,
 *                  such as a freshly initialised head, write few or no
 *                  pieces (none at all where every p < 2^-8) and cost
 *                  little more than mode 2.
 *                1 every entry keeps its rest; the contractions run over S_hi
 *                  and S_lo, twice their work: S carried to ~2^-17 relative.
 *                2 never: S in one 16-bit part (no S_lo buffer needed).
 *                Modes 0 and 1 take one more S-sized buffer in the workspace
 *                (bits 1-2 of ll_workspace_size's flags give the mode).
 *                Ignored for FP32 operands (S is FP32).
 *   reserved     must be 0.
 * A bad temperature, split_s not 0 / 1 / 2 or a non-zero reserved field is
 * LL_ERR_INVALID_ARG.
 */
typedef struct {
    float temperature;
    int split_s;
    int reserved[6];
} ll_options;

/* Human-readable name of a status code (static storage). */
const char* ll_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int ll_version(void);

/*
 * Workspace bytes needed by ll_forward (is_backward = 0), ll_backward
 * (is_backward = 1) or ll_forward_backward (is_backward = 2) for these
 * sizes; `flags` bit 0 is the need_db flag of the backward (bias gradient
 * partials), bits 1-2 the split_s option of ll_options (0 = automatic, the
 * default, 1 = always, 2 = never); both are ignored for the forward.
 * Returns 0 for a split_s field above 2.
 * token_chunks: number of token chunks the backward splits N into (0 =
 * automatic, see ll_backward).  Returns 0 only for N == 0 in the forward.
 * The workspace pointer must be 256-byte aligned.
 */
size_t ll_workspace_size(int64_t N, int64_t D, int64_t V, int dtype,
                         int token_chunks, int is_backward, int flags);

/*
 * Forward.  Issue #261 "Current production path" (the linear_logp op) and
 * PR #495 "Summary" (logp of the selected token; lse is saved for backward).
 *   hidden  [N, D] dtype, device, 16-byte aligned; D a multiple of 8 (else LL_ERR_ALIGN)
 *   weight  [V, D] dtype, device, 16-byte aligned
 *   bias    [V]    dtype, device, or NULL
 *   targets [N]    int64, device
 *   logp    [N]    float, device (written)
 *   lse     [N]    float, device (written; pass it to ll_backward)
 * N == 0 launches nothing.  D >= 1, V >= 1.
 * A small problem (fewer than 128 blocks of 128 rows x 1024 vocab columns,
 * N * round_up(V, 8) FP32 logits within 4 MiB) keeps its logits in the
 * workspace and forms the per-segment partials in a second kernel with the
 * same arithmetic: the same bits as the one-kernel path of larger problems,
 * with 4x as many SMs busy.
 */
int ll_forward(const void* hidden, const void* weight, const void* bias,
               const int64_t* targets, int64_t N, int64_t D, int64_t V, int dtype,
               float* logp, float* lse, void* workspace, size_t ws_bytes,
               void* stream);

/*
 * Backward.  Issue #261 "Current accumulation" (FP32 grad_w table, per-chunk
 * accumulation; its "Static traffic model" prices the chunking); Liger-Kernel
 * PR #1324 "Details" (accumulate each chunk's contribution into grad_weight
 * with no [V, D] temporary).  The automatic chunk size is not #261's rule of
 * C = floor(2^24 / V) rows: it is a 2 GiB budget on the chunk's softmax part
 * (below).
 *   grad_logp [N] float, device.  hidden/weight/bias/targets as in ll_forward.
 *   lse       [N] float, device: the forward's lse for the same inputs.
 *   need_dh / need_dw / need_db: which gradients to produce (0 or 1).
 *   grad_hidden [N, D] of dh_dtype (written when need_dh).
 *   grad_weight [V, D] of dw_dtype (written, i.e. overwritten, when need_dw).
 *     LL_F32 accumulates and stores FP32.  A 16-bit dw_dtype equal to dtype
 *     accumulates each token chunk in FP32 and rounds the running table once
 *     per chunk (once in total when token_chunks == 1).
 *   grad_bias [V] of dw_dtype (written when need_db; requires a bias).
 *   token_chunks: 0 = automatic (one chunk when its softmax part S,
 *     [rows, round_up(V, 8)] in the operand dtype, is at most 2 GiB, otherwise
 *     the fewest chunks of a multiple of 128 rows whose S fits), else the
 *     number of chunks N is split into, in order.  logp-independent outputs (dh) are
 *     bitwise independent of token_chunks; dW/db differ by FP32 rounding.
 * N == 0: grad_weight / grad_bias (if requested) are filled with +0.
 */
int ll_backward(const float* grad_logp, const void* hidden, const void* weight,
                const void* bias, const int64_t* targets, const float* lse,
                int64_t N, int64_t D, int64_t V, int dtype,
                int need_dh, int need_dw, int need_db,
                void* grad_hidden, int dh_dtype,
                void* grad_weight, int dw_dtype,
                void* grad_bias, int token_chunks,
                void* workspace, size_t ws_bytes, void* stream);

/*
 * Forward and backward in one call, for when grad_logp is known before the
 * forward (a fixed loss weighting such as a mean cross entropy, as in the
 * fused linear cross entropy of Liger-Kernel PR #1324, "Summary").  Same
 * arguments and results as ll_forward followed by ll_backward (logp and lse
 * are written as the forward's outputs), bitwise, for the same token_chunks
 * (token_chunks = 0 chooses the same chunks as ll_backward): each token
 * chunk's forward GEMM keeps its FP32 logits in the workspace (one chunk's
 * worth, never the whole [N, V] beyond it), and the softmax part is formed
 * from them instead of recomputing the logits.
 * Workspace: ll_workspace_size(..., is_backward = 2, need_db).
 */
int ll_forward_backward(const float* grad_logp, const void* hidden, const void* weight,
                        const void* bias, const int64_t* targets, int64_t N, int64_t D,
                        int64_t V, int dtype, float* logp, float* lse, int need_dh,
                        int need_dw, int need_db, void* grad_hidden, int dh_dtype,
                        void* grad_weight, int dw_dtype, void* grad_bias, int token_chunks,
                        void* workspace, size_t ws_bytes, void* stream);

/* ll_forward, ll_backward and ll_forward_backward with options (see
 * ll_options); same workspaces. */
int ll_forward_ex(const void* hidden, const void* weight, const void* bias,
                  const int64_t* targets, int64_t N, int64_t D, int64_t V, int dtype,
                  float* logp, float* lse, void* workspace, size_t ws_bytes,
                  const ll_options* opt, void* stream);
int ll_backward_ex(const float* grad_logp, const void* hidden, const void* weight,
                   const void* bias, const int64_t* targets, const float* lse,
                   int64_t N, int64_t D, int64_t V, int dtype,
                   int need_dh, int need_dw, int need_db,
                   void* grad_hidden, int dh_dtype,
                   void* grad_weight, int dw_dtype,
                   void* grad_bias, int token_chunks,
                   void* workspace, size_t ws_bytes, const ll_options* opt, void* stream);
int ll_forward_backward_ex(const float* grad_logp, const void* hidden, const void* weight,
                           const void* bias, const int64_t* targets, int64_t N, int64_t D,
                           int64_t V, int dtype, float* logp, float* lse, int need_dh,
                           int need_dw, int need_db, void* grad_hidden, int dh_dtype,
                           void* grad_weight, int dw_dtype, void* grad_bias,
                           int token_chunks, void* workspace, size_t ws_bytes,
                           const ll_options* opt, void* stream);

/*
 * Vocab-parallel (tensor-parallel) pieces: the vocab split over ranks into
 * contiguous shards [v0, v0 + Vs) (RL-Kernel PR #495, the coordinated
 * cross entropy experiment and its follow-up commit: each tensor-parallel
 * shard must start and end on a fixed vocab tile boundary, and training
 * and rollout scoring must agree bitwise across tensor-parallel layouts,
 * which a shard-local merge broke for 282 of 1200 rows).
 *   v0 must be a multiple of LL_SEGMENT_COLS; Vs too, except for the last
 *   shard (v0 + Vs == V).  Anything else is LL_ERR_SHAPE.
 * The forward's lse is an ascending-order merge of per-segment (max,
 * sum-exp) partials, segments of LL_SEGMENT_COLS vocab entries.  A shard's
 * partials are exactly the whole-vocab run's partials of its segments, so
 * the shards' partials stacked in shard order, merged by ll_lse_merge, give
 * the logp and lse of ll_forward bitwise, for any number of shards.
 * Targets are global vocab ids throughout.
 */
#define LL_SEGMENT_COLS 1024

/* Segments of a shard of Vs vocab entries: ceil(Vs / LL_SEGMENT_COLS). */
int64_t ll_shard_segments(int64_t Vs);

/* Workspace bytes of ll_forward_shard (is_backward = 0) or
 * ll_backward_shard (is_backward = 1; flags as for ll_workspace_size),
 * 256-byte aligned. */
size_t ll_workspace_size_shard(int64_t N, int64_t D, int64_t Vs, int dtype, int token_chunks,
                               int is_backward, int flags);

/*
 * Forward of one vocab shard: the shard's segment partials, no lse.
 *   weight [Vs, D], bias [Vs] or NULL: the shard's rows of W and b.
 *   targets [N] int64, global ids.
 *   part_m, part_s [ll_shard_segments(Vs), N] float, device (written): for
 *     the shard's segment j and row n, m = max over the segment of
 *     z * log2(e) and s = sum over the segment of 2^(z * log2(e) - m).
 *   zy [N] float, device (written): z[n, y_n] where y_n lies in the shard,
 *     -inf elsewhere; the elementwise max over the shards is z[n, y_n].
 */
int ll_forward_shard(const void* hidden, const void* weight, const void* bias,
                     const int64_t* targets, int64_t N, int64_t D, int64_t Vs, int64_t v0,
                     int64_t V, int dtype, float* part_m, float* part_s, float* zy,
                     void* workspace, size_t ws_bytes, const ll_options* opt,
                     void* stream);

/*
 * Ordered merge of whole-vocab segment partials: lse[n] = M + log sum_j
 * s[j, n] 2^(m[j, n] - M) (M = max_j m[j, n], j ascending; in natural units),
 * logp[n] = zy[n] - lse[n] if 0 <= targets[n] < V, else 0.
 *   part_m, part_s [n_segs, part_ld] float, device, part_ld >= N; rows with
 *     m = -inf, s = 0 (padding between shards) change nothing, bitwise.
 *   zy [N] float: z[n, y_n] (for instance the max over the shards' zy).
 *   logp, lse [N] float, device (written).  No workspace.
 */
int ll_lse_merge(const float* part_m, const float* part_s, int64_t n_segs, int64_t part_ld,
                 const float* zy, const int64_t* targets, int64_t N, int64_t V, float* logp,
                 float* lse, void* stream);

/*
 * Backward of one vocab shard, given the merged lse.  Arguments as in
 * ll_backward with weight/bias/grad_weight/grad_bias being the shard's rows
 * ([Vs, D], [Vs]) and targets global ids.
 *   grad_hidden [N, D] (written): this shard's part, sum over v in the shard
 *     of g[n, v] W[v, :]; grad_hidden is the sum of the shards' parts (add
 *     them in a fixed order; LL_F32 keeps that sum accurate).
 *   grad_weight / grad_bias: the shard's rows of the whole gradients,
 *     bitwise those of ll_backward for the same token_chunks.
 * A row whose target lies in another shard has no one-hot entry here and
 * keeps its softmax part; invalid targets or grad_logp = 0 give +0 rows.
 */
int ll_backward_shard(const float* grad_logp, const void* hidden, const void* weight,
                      const void* bias, const int64_t* targets, const float* lse, int64_t N,
                      int64_t D, int64_t Vs, int64_t v0, int64_t V, int dtype, int need_dh,
                      int need_dw, int need_db, void* grad_hidden, int dh_dtype,
                      void* grad_weight, int dw_dtype, void* grad_bias, int token_chunks,
                      void* workspace, size_t ws_bytes, const ll_options* opt,
                      void* stream);

/*
 * Forward without a caller workspace.  No counterpart on the source pages:
 * it exists for callers that cannot allocate device memory (a framework
 * that forbids allocation during a step, plugin code without access to the
 * application's allocator).  Same arguments, results and errors as
 * ll_forward, minus the workspace (argument errors and N == 0 are answered
 * exactly as ll_forward answers them): the scratch lives in a static 8 MiB
 * (8388608-byte) device array of the library, held on every GPU that loads
 * the library until the process exits.  A problem whose forward workspace,
 * ll_workspace_size(N, D, V, dtype, 0, 0) (three regions of
 * ceil(V / 1024) * N, ceil(V / 1024) * N and N floats, each padded to 256
 * bytes, plus at most 4 MiB of logits for a small problem, see ll_forward),
 * exceeds that is rejected with LL_ERR_WORKSPACE before anything
 * runs: N <= 32262 fits at V = 32768, N <= 7013 at V = 151936.  The first
 * call on a device looks up the array's device address (cudaGetSymbolAddress
 * with the device of `hidden` current) and keeps it for the process; make
 * that first call before any stream capture, and do not call it on a device
 * after cudaDeviceReset of that device.  It allocates nothing.  All calls on
 * a device share the one array, which keeps the last call's contents: calls
 * that may overlap on the GPU (other streams, other host threads) race.
 */
int ll_forward_noalloc(const void* hidden, const void* weight, const void* bias,
                       const int64_t* targets, int64_t N, int64_t D, int64_t V, int dtype,
                       float* logp, float* lse, void* stream);

/*
 * Logits-input forward.  PR #495 "Summary" (fused logp forward: one row per
 * block, logp of the target, constant 0 for targets outside [0, V)).
 *   logits [N, ld] dtype, device; row n starts at logits + n * ld; columns
 *          [V, ld) are ignored.  ld >= V.
 *   logp, lse [N] float, device (written).
 * N == 0 launches nothing.  No workspace.
 */
int logits_logp_fwd(const void* logits, int64_t ld, int dtype, const int64_t* targets,
                    int64_t N, int64_t V, float* logp, float* lse, void* stream);

/*
 * Logits-input backward.  PR #495 "Summary" (dlogits = grad * (one_hot -
 * softmax) written in the logits dtype, no workspace) using the saved lse:
 * one read and one write of the logits.
 *   grad_logits [N, ld] dtype, device (columns [0, V) written; [V, ld)
 *               untouched).  It may not overlap logits.
 * N == 0 launches nothing.
 */
int logits_logp_bwd(const float* grad_logp, const void* logits, int64_t ld, int dtype,
                    const int64_t* targets, const float* lse, int64_t N, int64_t V,
                    void* grad_logits, void* stream);

/*
 * Logits-input forward and backward in one pass, for a grad_logp known
 * before the forward.  Same arguments as logits_logp_fwd plus
 * logits_logp_bwd together; logp, lse and grad_logits are written, bitwise
 * the results of the two calls.  Each row's gradient is computed right after
 * its lse, so the row's second read is served (mostly) by L2: HBM sees about
 * 4 V bytes per row instead of 6 V.  grad_logits may be the logits buffer
 * itself (in place); a partial overlap is LL_ERR_INVALID_ARG.
 */
int logits_logp_fwd_bwd(const float* grad_logp, const void* logits, int64_t ld, int dtype,
                        const int64_t* targets, int64_t N, int64_t V, float* logp, float* lse,
                        void* grad_logits, void* stream);

/* The logits-input calls with options (see ll_options). */
int logits_logp_fwd_ex(const void* logits, int64_t ld, int dtype, const int64_t* targets,
                       int64_t N, int64_t V, float* logp, float* lse, const ll_options* opt,
                       void* stream);
int logits_logp_bwd_ex(const float* grad_logp, const void* logits, int64_t ld, int dtype,
                       const int64_t* targets, const float* lse, int64_t N, int64_t V,
                       void* grad_logits, const ll_options* opt, void* stream);
int logits_logp_fwd_bwd_ex(const float* grad_logp, const void* logits, int64_t ld, int dtype,
                           const int64_t* targets, int64_t N, int64_t V, float* logp,
                           float* lse, void* grad_logits, const ll_options* opt,
                           void* stream);

/*
 * Device status word of the current device: synchronises `stream`, returns
 * LL_OK or the first device-side error recorded since the last call
 * (LL_ERR_DEVICE_TIMEOUT), and clears it.
 */
int ll_check_status(void* stream);

/*
 * Fixed-order sum of partial tables, the data-parallel exchange of
 * grad_weight / grad_bias.  Each rank computes its token shard's tables and
 * they must be added (issue #261, "Current accumulation": the FP32 gradient
 * table is a sum over tokens); adding them in ascending rank order on one
 * rank, for each slice of the table it owns, gives the same bits whatever
 * the transport and on every rank that receives the result.
 *   parts [nparts, ld] of dtype, device: part k at parts + k * ld elements.
 *   out   [n] of dtype, device (written): out[i] = parts[0][i] + parts[1][i]
 *         + ... + parts[nparts - 1][i], in that order, accumulated in FP32
 *         and rounded once to dtype.  n <= ld.  out may not overlap parts.
 * n == 0 launches nothing.  Asynchronous on `stream`.
 */
int ll_sum_ordered(const void* parts, int64_t nparts, int64_t n, int64_t ld, int dtype,
                   void* out, void* stream);

/*
 * Tracing.  ll_launch_count(): number of kernels this library has launched
 * in the process.  ll_profile_enable(1) clears earlier records and brackets
 * every phase of later calls (fwd_gemm, lse_merge, token_sort,
 * recompute_gemm, softmax_part, lo_plan, transpose_h, grad_gemm
 * (grad_hidden and grad_weight tiles), db_sums, logits_fwd, logits_bwd,
 * logits_fused, sum_ordered; an _f32 suffix
 * marks the GEMMs of FP32 operands, 3 x TF32 on the tensor cores) with CUDA
 * events on the call's
 * stream; ll_profile_enable(0) stops recording.  ll_profile_summary()
 * synchronises on the recorded events and writes one line per phase,
 * "label count total_ms", into buf (NUL-terminated, truncated to len);
 * it returns the number of phases, or -LL_ERR_CUDA.
 */
long long ll_launch_count(void);
void ll_profile_enable(int on);
int ll_profile_summary(char* buf, size_t len);

/*
 * Test hook for the bounded waits: when `ns` > 0 every device-side wait of
 * later launches gives up after `ns` nanoseconds (default 2e9).  Used by the
 * tests to show that a wait that can never complete returns an error status
 * instead of hanging.  Host-side setting, not thread-safe.
 */
void ll_set_wait_limit_ns(int64_t ns);

/*
 * Test hook: a kernel that waits on a device barrier nothing will ever
 * complete, bounded by the wait limit.  It must end with
 * LL_ERR_DEVICE_TIMEOUT in the status word.  `device_flag` is one int of
 * device memory the kernel writes its exit path into (1 = timed out).
 */
int ll_debug_unsatisfied_wait(int* device_flag, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LL_LINEAR_LOGP_H */
