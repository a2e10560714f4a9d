// Internal host-side interface between the C ABI (capi.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ll_linear_logp.h"

namespace ll {

// Tile shape of the tensor-core GEMMs (M rows x N columns per output tile,
// K elements per pipeline stage for 16-bit operands).
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kVocabTilesPerSeg = 4;  // vocab tiles per LSE segment (1024 vocab)

// Maximum vocab size: inner indices within a row stay below 2^31.
constexpr int64_t kMaxV = (int64_t(1) << 31) - 1 - 256;

// Vocab-parallel shards: a shard covers vocab [v0, v0 + Vs) with v0 and (but
// for the last shard) Vs multiples of one LSE segment, so its segment
// partials are those of the whole-vocab run.  Inside a shard's launches a
// target is the local index y - v0, or kTargetInOtherShard for a valid
// target of another shard: the row keeps its softmax part, it has no
// one-hot entry here (EpiArgs::shard set).  Invalid targets become -1.
constexpr int64_t kSegCols = int64_t(kBN) * kVocabTilesPerSeg;
constexpr int64_t kTargetInOtherShard = -(int64_t(1) << 62);

struct DevInfo {
    int device;
    int num_sms;
    int* status;         // device status word (static device storage)
    cudaStream_t side;   // library side stream of the device (may be null)
};

// Wait limit for bounded device-side waits, nanoseconds.
uint64_t wait_limit_ns();

// Count of kernels this library has launched (for launch accounting).
void note_launches(int n);

// --- logits-input kernels (logits_kernels.cu) --------------------------------
// inv_temp: the logits are scaled by 1 / temperature (1 = none).
cudaError_t launch_logits_fwd(const void* logits, int64_t ld, int dtype, const int64_t* targets,
                              int64_t N, int64_t V, float* logp, float* lse, float inv_temp,
                              cudaStream_t s);
cudaError_t launch_logits_bwd(const float* grad, const void* logits, int64_t ld, int dtype,
                              const int64_t* targets, const float* lse, int64_t N, int64_t V,
                              void* grad_logits, float inv_temp, cudaStream_t s);

// Logits forward + backward in one pass for a known upstream gradient
// (logits_kernels.cu): per row the forward then the backward, bitwise the
// results of the two kernels; grad_logits may be the logits buffer.
cudaError_t launch_logits_fused(const float* grad, const void* logits, int64_t ld, int dtype,
                                const int64_t* targets, int64_t N, int64_t V, float* logp,
                                float* lse, void* grad_logits, float inv_temp,
                                const DevInfo& dev, cudaStream_t s);

// --- GEMM-based linear path -------------------------------------------------
enum class EpiKind : int { Fwd = 0, Recomp = 1, Dh = 2, Dw = 3 };

// Everything an epilogue may need; unused fields are ignored by a given kind.
struct EpiArgs {
    int64_t M;            // valid rows of the output tile grid (M dimension)
    int64_t Ncols;        // valid columns (N dimension)
    int64_t V;            // vocab size
    // forward / recompute (M = tokens of the launch, N = vocab)
    const int64_t* targets;  // [M]
    const void* bias;        // [V] or nullptr
    float* part_m;           // [n_segs, part_ld] running max (log2 units)
    float* part_s;           // [n_segs, part_ld] running sum
    float* zy;               // [M] target logit
    int64_t part_ld;
    float* Z;                // forward of the single fwd+bwd call: FP32 logits [M, ldZ]
    int64_t ldZ;
    const float* lse;        // [M]
    const float* grad;       // [M] grad_logp
    void* S;                 // [M, ldS] off-target part of g (0 at the target)
    int64_t ldS;
    float* tc;               // [M] target entry of g: grad * (1 - p[y]) (Recomp writes,
                             //     Dh reads; offset to the launch's rows)
    float* db_part;          // Recomp: [ceil(M / 32), V] grad_bias partials, or nullptr
    // dh (M = tokens, N = D): adds gl * W[y] and stores
    const void* W;
    int64_t ldW;
    void* out;               // dh [M, ld_out] or dW [V, ld_out]
    int64_t ld_out;
    int out_dtype;
    // dW (M = vocab, N = D)
    int first_chunk, last_chunk;
    int dw_add_prev;         // epilogue adds the stored grad_weight (else the store reduces)
    const int* offs;         // [V + 1] token list offsets per vocab row
    const int64_t* keys;     // sorted (target << 32 | token)
    const float* tc_all;     // [N] target entry of g of every token
    const void* h_all;       // [N, D] hidden of every token
    int64_t ld_h;
    int* status;
    uint64_t wait_ns;
    int shard;               // targets may be kTargetInOtherShard (vocab shard)
    float inv_temp;          // Fwd / Recomp: logits scaled by 1 / temperature (1 = none)
    void* S_lo;              // Recomp, 16-bit: S - S_hi (the rounding rest of S) [M, ldS],
                             //   or nullptr (no hi / lo split)
    uint8_t* lo_flags;       // Recomp, automatic split: [ceil(M / 32), lo_flags_ld] bytes, one
                             //   per piece of 32 rows x 64 columns: 1 if its S_lo was
                             //   written, else 0 (every piece in the chunk gets one);
                             //   nullptr = S_lo written in full (split of every entry)
    int64_t lo_flags_ld;     // row pitch of the flags: lo_flags_cols rounded up to 16
    int64_t lo_flags_cols;   // pieces per row group: ceil(V / 64)
    int dh_part;             // Dh, K split: store the raw partial sum (no target column,
                             //   no zero rules); dh_finish_kernel completes the rows
    int z_only;              // Fwd: store the logits (bias, temperature applied) and
                             //   nothing else; fwd_fold_kernel forms the partials
};

// Row pitch of the automatic split's piece flags: ceil(V / 64) rounded up to
// 16 bytes, so that the plan reads them 16 at a time.
__host__ __device__ inline int64_t lo_flags_pitch(int64_t V) { return ((V + 63) / 64 + 15) / 16 * 16; }

// Automatic hi / lo split of S: an off-target entry keeps its rounding rest
// S - S_hi when its probability p = S / (-grad / T) is at least this.
// Smaller ones store S_hi alone (their rounding error is below 2^-9 * tau *
// |grad / T| each).
constexpr float kLoTau = 1.0f / 256.0f;

// Pieces of the flag grid of the automatic split.
constexpr int kLoRows = 32;
constexpr int kLoCols = 64;

struct GemmShape {
    int64_t m_blocks;        // M / 128, rounded up
    int64_t n_tiles;         // N / 256, rounded up
    int64_t tiles_per_unit;  // N tiles per work unit (forward segments), else 1
    int64_t n_segs;          // ceil(n_tiles / tiles_per_unit)
    int64_t k_blocks;        // K / BK, rounded up
    int unit_order;          // 0: segment-major, 1: m-major, 2: segment-major within
                             //    groups of group_m row blocks (L2 rasterisation)
    int64_t group_m;         // row blocks per group of order 2 (set by launch_gemm)
    int64_t k_splits;        // FP32 grad_hidden: K cut into this many parts, one unit
                             //   each, written as FP32 partial sums (0 or 1 = whole K)
};

// Row blocks per group of the grouped unit order: the units in flight then
// share a group of row blocks of A and a few segments of B, which fit in L2.
// A group holds at most kGroupM row blocks and kGroupBytes of A (16 row
// blocks of 256 x 4096 bf16): at 32768 x 4096 x 151936 the forward read 17.7
// GB of DRAM per 13312 rows with 32 MB groups, 19.9 with 64 MB and 28.8 with 16.
constexpr int64_t kGroupM = 32;
constexpr int64_t kGroupBytes = int64_t(32) << 20;

// Operands of one GEMM kind:
//   A: [M, K] (a_mn = 0, row stride lda) or [K, M] (a_mn = 1)
//   B: [N, K] (b_mn = 0) or [K, N] (b_mn = 1)
struct GemmOperands {
    const void* A;
    int64_t lda;
    int a_mn;
    const void* B;
    int64_t ldb;
    int b_mn;
    int64_t M, N, K;
    const void* A_lo;  // 16-bit only: a second A of A's layout; the contraction then
                       // runs over K twice, A then A_lo, against the same B (nullptr: no)
    // planned second pass (automatic split): only the K blocks of each m block
    // listed by launch_lo_plan run over A_lo, with the pieces of A_lo not
    // written read as zeros (lo_cnt == nullptr: the whole second pass)
    const int* lo_cnt;
    const int64_t* lo_idx;
    int64_t lo_ld;
};

// Whether launch_gemm runs these kinds (M of each) on CTA pairs: 16-bit
// operands and every kind with at least 256 rows.
bool gemm_uses_pairs(int dtype, const int64_t* Ms, int nkinds);

// Tile output written by the epilogue ([rows, cols], row stride ld).
struct OutDesc {
    void* ptr;  // nullptr: the kind stores nothing (plain forward)
    int dtype;
    int64_t rows, cols, ld;
};

// One launch of the tensor-core GEMM kernel: one or two tile kinds (the
// first kind's units are handed out first).  FP32 operands run each kind on
// the CUDA-core path instead.
struct GemmLaunch {
    int dtype;  // LL_BF16 / LL_F16 / LL_F32
    int nkinds;
    EpiKind kind[2];
    GemmOperands op[2];
    GemmShape shape[2];
    EpiArgs ea[2];
    OutDesc out[2];
    int* counter;       // dynamic scheduling counter (must be 0), or nullptr
    int* zero_counter;  // counter of a later launch to zero, or nullptr
    int max_ctas;       // grid cap (0 = one CTA per SM), leaves SMs to a side stream
};
cudaError_t launch_gemm(const GemmLaunch& L, const DevInfo& dev, cudaStream_t s);

// --- small kernels (aux_kernels.cu) ------------------------------------------
// Shard-local targets: y - v0 for y in [v0, v0 + Vs), kTargetInOtherShard
// for other valid y in [0, V), -1 for invalid ones; zy (if given) = -inf.
cudaError_t launch_localize_targets(const int64_t* targets, int64_t N, int64_t v0, int64_t Vs,
                                    int64_t V, int64_t* local, float* zy, cudaStream_t s);
// The forward's per-(segment, row) partials from stored FP32 logits Z
// [rows, ldZ] (bias and temperature applied): the forward epilogue's fold,
// 32 columns at a time in ascending order, with the same arithmetic, so the
// partials are bitwise those of the fused epilogue; also the target logit
// zy[n] of rows whose target lies in [0, V).
cudaError_t launch_fwd_fold(const float* Z, int64_t ldZ, int64_t rows, int64_t V,
                            const int64_t* targets, float* part_m, float* part_s, float* zy,
                            int64_t part_ld, cudaStream_t s);
// The fold and then the merge of each row (logp, lse) in one launch, a warp
// per row: for rows of few segments (kFoldMergeSegs or fewer).
constexpr int64_t kFoldMergeSegs = 8;
cudaError_t launch_fwd_fold_merge(const float* Z, int64_t ldZ, int64_t rows, int64_t V,
                                  const int64_t* targets, float* part_m, float* part_s,
                                  float* zy, int64_t part_ld, float* logp, float* lse,
                                  cudaStream_t s);
cudaError_t launch_lse_merge(const float* part_m, const float* part_s, const float* zy,
                             int64_t part_ld, int64_t n_segs, const int64_t* targets, int64_t N,
                             int64_t V, float* logp, float* lse, cudaStream_t s);
// keys[i] = (y << 32 | i) for valid targets, all-ones otherwise; sorted
// ascending; offs[v] = first index whose target is >= v (v in [0, V]).
size_t token_sort_bytes(int64_t N);
cudaError_t launch_token_sort(const int64_t* targets, int64_t N, int64_t V, int64_t* keys,
                              int* offs, cudaStream_t s);
// grad_bias of a chunk from its partial rows [groups, V] (one per 32 rows
// of S, written by the recompute epilogue or the softmax-part kernel):
// db_acc (+)= their sum in a fixed order (the first chunk starts from +0);
// with `last`, adds the target entries tc[n] of the tokens of each vocab row
// (ascending token order) and writes grad_bias in out_dtype.
cudaError_t launch_db_finish(const float* partial, int64_t groups, int64_t V, float* db_acc,
                             int first, int last, const int* offs, const int64_t* keys,
                             const float* tc_all, void* grad_bias, int out_dtype, cudaStream_t s);
cudaError_t launch_fill_zero(void* p, int64_t n_elems, int dtype, cudaStream_t s);
constexpr int kMaxDhParts = 16;  // FP32 grad_hidden K split: most parts
// grad_hidden of a K-split contraction: dh[n, :] = the parts P[k][n, :]
// (k = 0 .. ks - 1, row pitch D, part pitch part_rows rows) added in
// ascending k, then the Dh epilogue's target column and zero rules (exact +0
// for dead rows, + c[n] * W[y_n] where the target lies in the vocab).
cudaError_t launch_dh_finish(const float* parts, int ks, int64_t part_rows, int64_t rows,
                             int64_t D, const int64_t* targets, const float* grad,
                             const float* tc, int64_t V, int shard, const float* W,
                             float* dh, int num_sms, cudaStream_t s);
// dst [C, ldd] = src^T for FP32 src [R, C] with row stride lds (both strides
// multiples of 4 floats, lds >= round_up(C, 4), ldd >= round_up(R, 4)).
cudaError_t launch_transpose32(const float* src, int64_t R, int64_t C, int64_t lds, float* dst,
                               int64_t ldd, cudaStream_t s);
// hT [D, ldT] = h^T for 16-bit h [N, D] (D % 8 == 0; ldT >= N, a multiple of 8).
cudaError_t launch_transpose16(const void* h, int64_t N, int64_t D, void* hT, int64_t ldT,
                               cudaStream_t s);
// out[i] = parts[0 * ld + i] + parts[1 * ld + i] + ... (ascending part
// order, FP32 accumulation, one rounding to dtype), i < n.
cudaError_t launch_sum_ordered(const void* parts, int64_t nparts, int64_t n, int64_t ld,
                               int dtype, void* out, int num_sms, cudaStream_t s);
// Plan of the second (S_lo) pass of the automatic hi / lo split, from the
// recompute's piece flags F [ceil(rows / 32), ceil(V / 64)], row pitch
// lo_flags_pitch(V) (1 = that piece of 32 rows x 64 columns of S_lo was
// written):
//  grad_hidden, per block of R rows (R = 128, or 256 on CTA pairs): the
//   64-column K blocks kb with a written piece in the block, ascending, as
//   (kb << 8 | bits) where bit i is row group i of the block (32 rows);
//   dh_cnt[mb] entries at dh_idx[mb * ceil(V / 64)].
//  grad_weight, per block of C vocab rows (C = 128 or 256): the 64-token K
//   blocks kb with a written piece in the block, ascending, as (kb << 8 |
//   bits), bit 2c + i being 64-column group c of the block and row group
//   2 kb + i; dw_cnt[vb] entries at dw_idx[vb * ceil(rows / 64)].
// A block with no entry runs no second pass.
cudaError_t launch_lo_plan(const uint8_t* F, int64_t rows, int64_t V, int R, int C,
                           int* dh_cnt, int64_t* dh_idx, int* dw_cnt, int64_t* dw_idx,
                           cudaStream_t s);
// Softmax part from stored FP32 logits Z [rows, ldZ] (bias included):
// S = -grad * exp(z - lse) off target (S dtype s_dtype), S = 0 and
// tc = grad * (1 - p) at the target, +0 rows when the target is invalid or
// the gradient zero.  Same arithmetic as the recompute epilogue.
// With db_part (not null) it also writes the grad_bias partials per 32 rows,
// as the recompute epilogue does.  S_lo (16-bit): the rests S - S_hi, all of
// them, or with lo_flags the automatic split's pieces and flags, as the
// recompute epilogue writes them.
cudaError_t launch_softmax_part(const float* Z, int64_t ldZ, int64_t rows, int64_t V,
                                const int64_t* targets, const float* grad, const float* lse,
                                void* S, int64_t ldS, int s_dtype, float* tc, float* db_part,
                                float inv_temp, void* S_lo, uint8_t* lo_flags,
                                cudaStream_t s);
cudaError_t launch_unsatisfied_wait(int* flag, int* status, uint64_t wait_ns, cudaStream_t s);

}  // namespace ll
