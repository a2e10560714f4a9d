// Small kernels around the GEMMs of the linear logp path:
//   * the ordered merge of per-segment (max, sum-exp) partials into lse and
//     logp (fixed ascending segment order -> batch-invariant);
//   * a deterministic sort of the tokens by target (bitonic network over
//     64-bit keys target << 32 | token), giving for every vocab row the list
//     of tokens that target it in ascending token order (used by the exact
//     one-hot part of grad_weight and grad_bias);
//   * fixed-order column sums of the softmax part for grad_bias;
//   * shard-local targets of a vocab shard;
//   * a +0 fill and the bounded-wait self test.
#include <math.h>

#include "ll_device.cuh"

namespace ll {
namespace {

// lse and logp of row r from its per-segment partials, in ascending segment
// order (one thread; shared by every kernel that merges, so that they give the
// same bits).
__device__ __forceinline__ void merge_row(const float* __restrict__ pm,
                                          const float* __restrict__ ps,
                                          const float* __restrict__ zy, int64_t ld,
                                          int64_t n_segs, const int64_t* __restrict__ targets,
                                          int64_t r, int64_t V, float* __restrict__ logp,
                                          float* __restrict__ lse_out) {
    float M = -INFINITY;
    for (int64_t j = 0; j < n_segs; ++j) M = fmaxf(M, pm[j * ld + r]);
    float lse = -INFINITY;
    if (M != -INFINITY) {
        float S = 0.f;
        for (int64_t j = 0; j < n_segs; ++j)
            S = fmaf(ps[j * ld + r], ex2(pm[j * ld + r] - M), S);
        lse = fmaf(M, kLn2, logf(S));
    }
    const int64_t y = targets[r];
    logp[r] = (y >= 0 && y < V) ? zy[r] - lse : 0.f;
    lse_out[r] = lse;
}

__global__ void lse_merge_kernel(const float* __restrict__ pm, const float* __restrict__ ps,
                                 const float* __restrict__ zy, int64_t ld, int64_t n_segs,
                                 const int64_t* __restrict__ targets, int64_t N, int64_t V,
                                 float* __restrict__ logp, float* __restrict__ lse_out) {
    const int64_t r = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    if (r >= N) return;
    merge_row(pm, ps, zy, ld, n_segs, targets, r, V, logp, lse_out);
}

// The forward epilogue's fold from stored logits (small problems, whose
// forward GEMM runs one vocab tile per unit and stores Z instead): one warp
// per (row, 1024-column segment), lane c holding the segment's 32-column
// chunk c.  The epilogue thread that owns the row folds the chunks in
// ascending order: columns past V read as -inf; mu = chunk max * log2(e);
// when mu exceeds the running max m2 the running sum s is rescaled by
// 2^(m2 - mu) and m2 = mu; then, unless m2 is still -inf, the chunk's 32
// terms 2^(z * log2(e) - m2) are added one after another in column order and
// their sum is added to s.  Here m2 after chunk c is the prefix max of mu
// (exact in any order), so every lane forms its chunk's sum with the same
// steps at once, and one pass over the lanes replays the rescales and adds
// of s in chunk order: the same bits as the epilogue.  Chunks wholly past V
// change nothing there (their terms are +0) and are not visited here.
// The fold of one (row, segment) by one warp; writes part_m / part_s (lane 0)
// and zy[row] (the lane whose chunk holds the target).
__device__ __forceinline__ void fold_segment(const float* __restrict__ Z, int64_t ldZ,
                                             int64_t V, int64_t seg, int64_t row, int64_t y,
                                             float* __restrict__ part_m,
                                             float* __restrict__ part_s,
                                             float* __restrict__ zy, int64_t part_ld, int lane) {
    const int64_t seg0 = seg * kSegCols;
    const int n_chunks = static_cast<int>(min(int64_t(32), (V - seg0 + 31) / 32));
    const int64_t col0 = seg0 + 32 * lane;
    const bool mine = lane < n_chunks;
    float v[32];
    const float* z = Z + row * ldZ + col0;
    if (mine && col0 + 32 <= V) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 f = *reinterpret_cast<const float4*>(z + 4 * q);
            v[4 * q] = f.x, v[4 * q + 1] = f.y, v[4 * q + 2] = f.z, v[4 * q + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = (mine && col0 + j < V) ? z[j] : -INFINITY;
    }
    const int64_t off = y - col0;
    if (mine && off >= 0 && off < 32) {
        float t = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j == off) t = v[j];
        zy[row] = t;
    }
    float cmax = v[0];
#pragma unroll
    for (int j = 1; j < 32; ++j) cmax = fmaxf(cmax, v[j]);
    const float mu = mine ? cmax * kLog2e : -INFINITY;
    float m2 = mu;  // prefix max over the lanes: the running max after chunk `lane`
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, m2, o);
        if (lane >= o) m2 = fmaxf(m2, t);
    }
    float acc = 0.f;
    if (mine && m2 != -INFINITY) {
#pragma unroll
        for (int j = 0; j < 32; ++j) acc += ex2(fmaf(v[j], kLog2e, -m2));
    }
    // the running sum, chunk by chunk as the epilogue forms it
    float rm = -INFINITY, s = 0.f;
    for (int c = 0; c < n_chunks; ++c) {
        const float mc = __shfl_sync(0xffffffffu, mu, c);
        const float ac = __shfl_sync(0xffffffffu, acc, c);
        if (mc > rm) {
            s = s * ex2(rm - mc);
            rm = mc;
        }
        if (rm != -INFINITY) s += ac;
    }
    if (lane == 0) {
        part_m[seg * part_ld + row] = rm;
        part_s[seg * part_ld + row] = s;
    }
}

__global__ void __launch_bounds__(256) fwd_fold_kernel(
    const float* __restrict__ Z, int64_t ldZ, int64_t rows, int64_t V,
    const int64_t* __restrict__ targets, float* __restrict__ part_m,
    float* __restrict__ part_s, float* __restrict__ zy, int64_t part_ld) {
    const int lane = threadIdx.x & 31;
    const int64_t n_segs = (V + kSegCols - 1) / kSegCols;
    const int64_t w = blockIdx.x * int64_t(blockDim.x / 32) + (threadIdx.x >> 5);
    if (w >= rows * n_segs) return;
    const int64_t seg = w / rows, row = w - seg * rows;
    fold_segment(Z, ldZ, V, seg, row, targets[row], part_m, part_s, zy, part_ld, lane);
}

// Rows with few segments: a block per row, warp w folding segment w, then
// thread 0 merges them (lse, logp) with merge_row: one launch instead of two,
// the same bits.
__global__ void __launch_bounds__(256) fwd_fold_merge_kernel(
    const float* __restrict__ Z, int64_t ldZ, int64_t rows, int64_t V,
    const int64_t* __restrict__ targets, float* __restrict__ part_m,
    float* __restrict__ part_s, float* __restrict__ zy, int64_t part_ld,
    float* __restrict__ logp, float* __restrict__ lse) {
    const int lane = threadIdx.x & 31;
    const int64_t n_segs = (V + kSegCols - 1) / kSegCols;  // the block's warp count
    const int64_t row = blockIdx.x;
    fold_segment(Z, ldZ, V, threadIdx.x >> 5, row, targets[row], part_m, part_s, zy, part_ld,
                 lane);
    __syncthreads();  // the row's partials and zy, written by the block's warps
    if (threadIdx.x == 0)
        merge_row(part_m, part_s, zy, part_ld, n_segs, targets, row, V, logp, lse);
}

// Targets of one vocab shard [v0, v0 + Vs) of a vocab of V entries.
__global__ void localize_targets_kernel(const int64_t* __restrict__ targets, int64_t N,
                                        int64_t v0, int64_t Vs, int64_t V,
                                        int64_t* __restrict__ local, float* __restrict__ zy) {
    const int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    if (i >= N) return;
    const int64_t y = targets[i];
    int64_t l = -1;
    if (y >= 0 && y < V) l = (y >= v0 && y < v0 + Vs) ? y - v0 : kTargetInOtherShard;
    local[i] = l;
    if (zy) zy[i] = -INFINITY;
}

constexpr int kSortSeg = 4096;  // keys sorted per CTA in shared memory
constexpr int kSortThreads = 1024;

__global__ void make_keys_kernel(const int64_t* __restrict__ targets, int64_t N, int64_t V,
                                 int64_t n_pad, unsigned long long* __restrict__ keys) {
    const int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    if (i >= n_pad) return;
    unsigned long long k = ~0ull;
    if (i < N) {
        const int64_t y = targets[i];
        if (y >= 0 && y < V)
            k = (static_cast<unsigned long long>(y) << 32) | static_cast<unsigned long long>(i);
    }
    keys[i] = k;
}

__device__ __forceinline__ void cmp_swap(unsigned long long& a, unsigned long long& b, bool up) {
    if ((a > b) == up) {
        const unsigned long long t = a;
        a = b;
        b = t;
    }
}

// Bitonic steps with stride j < kSortSeg inside each CTA's segment.
// full = 1: every merge size k = 2 .. kSortSeg (sorts each segment);
// full = 0: only the strides j = kSortSeg/2 .. 1 of the merge size k.
__global__ void __launch_bounds__(kSortThreads) bitonic_local_kernel(unsigned long long* keys,
                                                                     int64_t k_fixed, int full) {
    __shared__ unsigned long long s[kSortSeg];
    const int64_t base = blockIdx.x * int64_t(kSortSeg);
    for (int t = threadIdx.x; t < kSortSeg; t += kSortThreads) s[t] = keys[base + t];
    __syncthreads();
    const int64_t k_lo = full ? 2 : k_fixed;
    const int64_t k_hi = full ? kSortSeg : k_fixed;
    for (int64_t k = k_lo; k <= k_hi; k <<= 1) {
        const int j0 = full ? static_cast<int>(k >> 1) : (kSortSeg >> 1);
        for (int j = j0; j > 0; j >>= 1) {
            for (int p = threadIdx.x; p < kSortSeg / 2; p += kSortThreads) {
                // pair index p -> lower element i of the pair (j is a power of two)
                const int i = ((p & ~(j - 1)) << 1) | (p & (j - 1));
                const bool up = ((base + i) & k) == 0;
                cmp_swap(s[i], s[i + j], up);
            }
            __syncthreads();
        }
    }
    for (int t = threadIdx.x; t < kSortSeg; t += kSortThreads) keys[base + t] = s[t];
}

// The whole sort of n <= kSortSeg keys (n a power of two) in one block:
// keys made from the targets (as make_keys_kernel), bitonic network in
// shared memory, written back.  Same sorted keys as the multi-launch path.
__global__ void __launch_bounds__(kSortThreads) sort_small_kernel(
    const int64_t* __restrict__ targets, int64_t N, int64_t V, int n,
    unsigned long long* __restrict__ keys) {
    __shared__ unsigned long long s[kSortSeg];
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        unsigned long long k = ~0ull;
        if (i < N) {
            const int64_t y = targets[i];
            if (y >= 0 && y < V)
                k = (static_cast<unsigned long long>(y) << 32) | static_cast<unsigned long long>(i);
        }
        s[i] = k;
    }
    __syncthreads();
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int p = threadIdx.x; p < n / 2; p += blockDim.x) {
                const int i = ((p & ~(j - 1)) << 1) | (p & (j - 1));
                cmp_swap(s[i], s[i + j], (i & k) == 0);
            }
            __syncthreads();
        }
    }
    for (int i = threadIdx.x; i < n; i += blockDim.x) keys[i] = s[i];
}

__global__ void bitonic_global_kernel(unsigned long long* keys, int64_t n, int64_t k, int64_t j) {
    const int64_t p = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    if (p >= n / 2) return;
    const int64_t i = ((p & ~(j - 1)) << 1) | (p & (j - 1));  // j is a power of two
    const bool up = (i & k) == 0;
    unsigned long long a = keys[i], b = keys[i + j];
    cmp_swap(a, b, up);
    keys[i] = a;
    keys[i + j] = b;
}

// offs[v] = first index of a key >= v << 32 (v = 0..V).
__global__ void offsets_kernel(const unsigned long long* __restrict__ keys, int64_t n, int64_t V,
                               int* __restrict__ offs) {
    const int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    if (v > V) return;
    const unsigned long long key = static_cast<unsigned long long>(v) << 32;
    int64_t lo = 0, hi = n;
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (keys[mid] < key)
            lo = mid + 1;
        else
            hi = mid;
    }
    offs[v] = static_cast<int>(lo);
}

// grad_bias from the chunk's partial rows (one per 32 rows of S): a block
// takes 32 columns; warp w sums rows w, w + 8, w + 16, ... in ascending
// order, and the block adds the running sum of the earlier chunks and then
// warps 0..7 in that order -- a fixed order for given rows per chunk.  On the
// last chunk the exact one-hot part (tc of the tokens whose target is v, in
// ascending token order) is added and the result stored.
template <typename TO>
__global__ void __launch_bounds__(256) db_finish_kernel(
    const float* __restrict__ partial, int64_t groups, int64_t V, float* __restrict__ db_acc,
    int first, int last, const int* __restrict__ offs,
    const unsigned long long* __restrict__ keys, const float* __restrict__ tc_all,
    TO* __restrict__ out) {
    __shared__ float part[8][32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t v = blockIdx.x * int64_t(32) + lane;
    float acc = 0.f;
    if (v < V) {
#pragma unroll 4
        for (int64_t g = warp; g < groups; g += 8) acc = acc + partial[g * V + v];
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (warp != 0 || v >= V) return;
    float t = first ? 0.f : db_acc[v];
#pragma unroll
    for (int w = 0; w < 8; ++w) t = t + part[w][lane];
    if (last) {
        for (int i = offs[v]; i < offs[v + 1]; ++i) t = t + tc_all[keys[i] & 0xffffffffull];
        out[v] = Elem<TO>::from_f(t + 0.f);
    } else {
        db_acc[v] = t;
    }
}

// 5-bit bit reversal: the order in which a 32-row group's rows enter the
// column sums below.
__host__ __device__ constexpr int brev5(int i) {
    return ((i & 1) << 4) | ((i & 2) << 2) | (i & 4) | ((i & 8) >> 2) | ((i & 16) >> 4);
}

// Softmax part from the stored FP32 logits of a chunk, with the values the
// recompute epilogue forms: p = 2^(z * log2e - lse * log2e), S = -grad * p off
// target, S = 0 and tc = grad * (1 - p) at the target.
//
// A block takes one group of 32 rows; each warp a 128-column slice of it
// (4 columns a lane, so every row's slice is one coalesced 512-byte read and a
// 256-byte 16-bit store), column slices strided over grid.y and the warps.
// The rows are visited in bit-reversed order, and (with db_part) each lane
// folds them into its columns' sums like a binary counter: entries 2k and
// 2k + 1 of that order are rows r and r + 16, then pairs of pairs are rows
// r, r + 8, and so on.  The sum of a column is thus the same binary tree
// (rows paired across bit 4 of the row, then bit 3, ..., bit 0) that the
// recompute epilogue's lane butterfly builds, and so bitwise its value.
// Loads in flight per warp and blocks per SM, from a sweep on GB300 (rows of
// FP32 logits, 16-bit S): without the column sums 4 rows a batch at 6
// blocks per SM (~6 TB/s), with them 8 rows at 3 (~5.5 TB/s).
template <typename T, bool DB, bool LO_ALL>
__global__ void __launch_bounds__(256, DB ? 3 : 6) softmax_part_kernel(
    const float* __restrict__ Z, int64_t ldZ, int64_t rows, int64_t V,
    const int64_t* __restrict__ targets, const float* __restrict__ grad,
    const float* __restrict__ lse, T* __restrict__ S, int64_t ldS, float* __restrict__ tc,
    float* __restrict__ db_part, float inv_temp, T* __restrict__ S_lo,
    uint8_t* __restrict__ lo_flags) {
    constexpr int kAhead = DB ? 8 : 4;  // rows whose loads are in flight together
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t r0 = blockIdx.x * int64_t(32);
    // lane r holds the parameters of row r0 + r
    const int64_t my_row = r0 + lane;
    const bool rvalid = my_row < rows;
    const int64_t my_y = rvalid ? targets[my_row] : -1;
    const float my_g = rvalid ? grad[my_row] : 0.f;
    const bool live = rvalid && my_y >= 0 && my_y < V && my_g != 0.f;
    const float my_coef = live ? -my_g * inv_temp : 0.f;
    const float my_lse2 = rvalid ? lse[my_row] * kLog2e : 0.f;
    if (rvalid && !(my_y >= 0 && my_y < V) && blockIdx.y == 0 && warp == 0) tc[my_row] = 0.f;
    const int nr = static_cast<int>(rows - r0 < 32 ? rows - r0 : 32);
    const int64_t step = int64_t(gridDim.y) * 8 * 128;
    for (int64_t c = (int64_t(blockIdx.y) * 8 + warp) * 128 + 4 * lane; c - 4 * lane < V;
         c += step) {
        float acc[5][4];  // pending subtree sums, one per binary-counter level
        bool kept = false;  // automatic split: an entry of this lane's columns keeps its rest
#pragma unroll
        for (int i0 = 0; i0 < 32; i0 += kAhead) {
            float z[kAhead][4];
#pragma unroll
            for (int u = 0; u < kAhead; ++u) {
                const int r = brev5(i0 + u);
                z[u][0] = z[u][1] = z[u][2] = z[u][3] = 0.f;
                if (r < nr && c < V) {
                    // c + 3 < round_up(V, 4) <= ldZ: the vector stays in the row
                    const float4 f = *reinterpret_cast<const float4*>(Z + (r0 + r) * ldZ + c);
                    z[u][0] = f.x;
                    z[u][1] = f.y;
                    z[u][2] = f.z;
                    z[u][3] = f.w;
                }
            }
#pragma unroll
            for (int u = 0; u < kAhead; ++u) {
                const int k = i0 + u;
                const int r = brev5(k);
                const float coef = __shfl_sync(0xffffffffu, my_coef, r);
                const float lse2 = __shfl_sync(0xffffffffu, my_lse2, r);
                const int64_t y = __shfl_sync(0xffffffffu, my_y, r);
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                if (r < nr && c < V) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[j] = ex2(fmaf(z[u][j], kLog2e, -lse2));
                    const int64_t off = y - c;
                    if (off >= 0 && off < 4) {
                        float py = 0.f;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (j == off) py = v[j];
                        tc[r0 + r] = coef != 0.f ? -coef * (1.f - py) : 0.f;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (j == off) v[j] = 0.f;
                    }
                    if (!LO_ALL && lo_flags && coef != 0.f) {  // p >= kLoTau: flag below
                        float pm = v[0];
#pragma unroll
                        for (int j = 1; j < 4; ++j)
                            if (c + j < V) pm = fmaxf(pm, v[j]);
                        kept |= pm >= kLoTau;
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[j] = coef * v[j];
                    T* srow = S + (r0 + r) * ldS;
                    if constexpr (sizeof(T) == 4) {  // FP32 S, no split
                        if (c + 4 <= V) {
                            *reinterpret_cast<float4*>(srow + c) =
                                make_float4(v[0], v[1], v[2], v[3]);
                        } else {
                            for (int j = 0; j < 4 && c + j < V; ++j) srow[c + j] = v[j];
                        }
                    } else if constexpr (!LO_ALL) {
                        uint2 hu;  // S rounded to T
                        T* hi = reinterpret_cast<T*>(&hu);
#pragma unroll
                        for (int j = 0; j < 4; ++j) hi[j] = Elem<T>::from_f(v[j]);
                        if (c + 4 <= V) {
                            *reinterpret_cast<uint2*>(srow + c) = hu;
                        } else {
                            for (int j = 0; j < 4 && c + j < V; ++j) srow[c + j] = hi[j];
                        }
                    } else {
                        uint2 hu, lu;  // S rounded to T; the rest S - S_hi rounded to T
                        T* hi = reinterpret_cast<T*>(&hu);
                        T* lo = reinterpret_cast<T*>(&lu);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            hi[j] = Elem<T>::from_f(v[j]);
                            lo[j] = Elem<T>::from_f(v[j] - Elem<T>::to_f(hi[j]));
                        }
                        T* lrow = S_lo + (r0 + r) * ldS;
                        if (c + 4 <= V) {
                            *reinterpret_cast<uint2*>(srow + c) = hu;
                            *reinterpret_cast<uint2*>(lrow + c) = lu;
                        } else {
                            for (int j = 0; j < 4 && c + j < V; ++j) {
                                srow[c + j] = hi[j];
                                lrow[c + j] = lo[j];
                            }
                        }
                    }
                }
                if constexpr (DB) {  // binary counter over the visiting order
                    bool carry = true;
#pragma unroll
                    for (int lvl = 0; lvl < 5; ++lvl) {
                        if (!carry) break;
                        if ((k >> lvl) & 1) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) v[j] = acc[lvl][j] + v[j];
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j) acc[lvl][j] = v[j];
                            carry = false;
                        }
                    }
                    if (k == 31) {  // v is the sum of all 32 rows
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (c + j < V) db_part[blockIdx.x * V + c + j] = v[j];
                    }
                }
            }
        }
        if constexpr (sizeof(T) == 2 && !LO_ALL) {
            // Automatic split: flag each 64-column piece of these 32 rows (a
            // half warp's columns) holding an entry with p >= kLoTau; the
            // pieces are written by lo_pieces_kernel.
            if (lo_flags) {  // every piece gets its flag: 1 = to be written
                const unsigned m = __ballot_sync(0xffffffffu, kept);
                if ((lane & 15) == 0 && c < V)
                    lo_flags[blockIdx.x * lo_flags_pitch(V) + c / kLoCols] =
                        ((lane < 16 ? m : m >> 16) & 0xffffu) != 0;
            }
        }
    }
}

__global__ void fill_zero_kernel(uint32_t* p, int64_t n_words) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_words;
         i += int64_t(gridDim.x) * blockDim.x)
        p[i] = 0u;
}
__global__ void fill_zero_u16_kernel(uint16_t* p, int64_t n) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x)
        p[i] = 0u;
}

// Waits on an mbarrier that nothing arrives on; the bounded wait must give
// up, record the timeout and return.
__global__ void unsatisfied_wait_kernel(int* flag, int* status, uint64_t wait_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool ok = mbar_wait(&bar, 0, wait_ns, nullptr);
        if (!ok) set_status(status, LL_ERR_DEVICE_TIMEOUT);
        *flag = ok ? 2 : 1;
    }
}

// out[i] = sum over k = 0, 1, ..., nparts - 1 (in that order) of
// parts[k * ld + i], accumulated in FP32 and rounded once to T.  A thread
// takes 4 consecutive elements (one 16-byte load per part for FP32 when the
// rows are 16-byte aligned), grid-stride over the row.
template <typename T, bool VEC>
__global__ void __launch_bounds__(256) sum_ordered_kernel(const T* __restrict__ parts,
                                                          int64_t nparts, int64_t n, int64_t ld,
                                                          T* __restrict__ out) {
    for (int64_t i = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) * 4; i < n;
         i += int64_t(gridDim.x) * blockDim.x * 4) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (VEC && i + 4 <= n) {
            for (int64_t k = 0; k < nparts; ++k) {
                const float4 f = *reinterpret_cast<const float4*>(
                    reinterpret_cast<const float*>(parts) + k * ld + i);
                if (k == 0) {
                    acc[0] = f.x, acc[1] = f.y, acc[2] = f.z, acc[3] = f.w;
                } else {
                    acc[0] += f.x, acc[1] += f.y, acc[2] += f.z, acc[3] += f.w;
                }
            }
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + i) =
                make_float4(acc[0], acc[1], acc[2], acc[3]);
        } else {
            const int m = static_cast<int>(n - i < 4 ? n - i : 4);
            for (int64_t k = 0; k < nparts; ++k)
                for (int j = 0; j < m; ++j) {
                    const float x = Elem<T>::to_f(parts[k * ld + i + j]);
                    acc[j] = k == 0 ? x : acc[j] + x;
                }
            for (int j = 0; j < m; ++j) out[i + j] = Elem<T>::from_f(acc[j]);
        }
    }
}

int64_t pow2_at_least(int64_t n) {
    int64_t p = 64;
    while (p < n) p <<= 1;
    return p;
}

}  // namespace

cudaError_t launch_fwd_fold(const float* Z, int64_t ldZ, int64_t rows, int64_t V,
                            const int64_t* targets, float* part_m, float* part_s, float* zy,
                            int64_t part_ld, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    note_launches(1);
    const int64_t warps = rows * ((V + kSegCols - 1) / kSegCols);
    fwd_fold_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, s>>>(
        Z, ldZ, rows, V, targets, part_m, part_s, zy, part_ld);
    return cudaGetLastError();
}

cudaError_t launch_fwd_fold_merge(const float* Z, int64_t ldZ, int64_t rows, int64_t V,
                                  const int64_t* targets, float* part_m, float* part_s,
                                  float* zy, int64_t part_ld, float* logp, float* lse,
                                  cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    const int64_t n_segs = (V + kSegCols - 1) / kSegCols;
    if (n_segs > kFoldMergeSegs || rows > int64_t(1) << 31) return cudaErrorInvalidValue;
    note_launches(1);
    fwd_fold_merge_kernel<<<static_cast<unsigned>(rows), static_cast<unsigned>(32 * n_segs), 0,
                            s>>>(Z, ldZ, rows, V, targets, part_m, part_s, zy, part_ld, logp,
                                 lse);
    return cudaGetLastError();
}

cudaError_t launch_lse_merge(const float* part_m, const float* part_s, const float* zy,
                             int64_t part_ld, int64_t n_segs, const int64_t* targets, int64_t N,
                             int64_t V, float* logp, float* lse, cudaStream_t s) {
    const int threads = 256;
    const int64_t blocks = (N + threads - 1) / threads;
    note_launches(1);
    lse_merge_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(
        part_m, part_s, zy, part_ld, n_segs, targets, N, V, logp, lse);
    return cudaGetLastError();
}

cudaError_t launch_localize_targets(const int64_t* targets, int64_t N, int64_t v0, int64_t Vs,
                                    int64_t V, int64_t* local, float* zy, cudaStream_t s) {
    if (N <= 0) return cudaSuccess;
    const int threads = 256;
    note_launches(1);
    localize_targets_kernel<<<static_cast<unsigned>((N + threads - 1) / threads), threads, 0, s>>>(
        targets, N, v0, Vs, V, local, zy);
    return cudaGetLastError();
}

size_t token_sort_bytes(int64_t N) { return static_cast<size_t>(pow2_at_least(N)) * 8; }

cudaError_t launch_token_sort(const int64_t* targets, int64_t N, int64_t V, int64_t* keys_,
                              int* offs, cudaStream_t s) {
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(keys_);
    const int64_t n = pow2_at_least(N);
    if (n <= kSortSeg) {  // one block sorts all keys
        note_launches(2);
        const int threads = static_cast<int>(n / 2 < kSortThreads ? n / 2 : kSortThreads);
        sort_small_kernel<<<1, threads, 0, s>>>(targets, N, V, static_cast<int>(n), keys);
        offsets_kernel<<<static_cast<unsigned>((V + 1 + 255) / 256), 256, 0, s>>>(keys, n, V,
                                                                                  offs);
        return cudaGetLastError();
    }
    note_launches(3);
    make_keys_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(targets, N, V, n,
                                                                            keys);
    const unsigned segs = static_cast<unsigned>(n / kSortSeg);
    bitonic_local_kernel<<<segs, kSortThreads, 0, s>>>(keys, 0, 1);
    for (int64_t k = 2 * kSortSeg; k <= n; k <<= 1) {
        for (int64_t j = k >> 1; j >= kSortSeg; j >>= 1, note_launches(1))
            bitonic_global_kernel<<<static_cast<unsigned>((n / 2 + 255) / 256), 256, 0, s>>>(
                keys, n, k, j);
        note_launches(1);
        bitonic_local_kernel<<<segs, kSortThreads, 0, s>>>(keys, k, 0);
    }
    offsets_kernel<<<static_cast<unsigned>((V + 1 + 255) / 256), 256, 0, s>>>(keys, n, V, offs);
    return cudaGetLastError();
}

// Automatic split of the single call: the pieces of S_lo that the softmax
// part flagged, each written whole (32 rows x 64 columns: the rest
// S - S_hi of every entry with p >= kLoTau, zero elsewhere) from the stored
// FP32 logits with the softmax part's arithmetic, so they are bitwise the
// recompute epilogue's pieces.  One warp per 32-row group; a lane takes two
// columns of a piece.
template <typename T>
__global__ void __launch_bounds__(256) lo_pieces_kernel(
    const float* __restrict__ Z, int64_t ldZ, int64_t rows, int64_t V,
    const int64_t* __restrict__ targets, const float* __restrict__ grad,
    const float* __restrict__ lse, T* __restrict__ S_lo, int64_t ldS,
    const uint8_t* __restrict__ lo_flags, float inv_temp) {
    const int lane = threadIdx.x & 31;
    const int64_t g = blockIdx.x * int64_t(8) + (threadIdx.x >> 5);
    const int64_t r0 = g * 32;
    if (r0 >= rows) return;
    const int64_t my_row = r0 + lane;
    const bool rvalid = my_row < rows;
    const int64_t my_y = rvalid ? targets[my_row] : -1;
    const float my_g = rvalid ? grad[my_row] : 0.f;
    const bool live = rvalid && my_y >= 0 && my_y < V && my_g != 0.f;
    const float my_coef = live ? -my_g * inv_temp : 0.f;
    const float my_lse2 = rvalid ? lse[my_row] * kLog2e : 0.f;
    const int nr = static_cast<int>(rows - r0 < 32 ? rows - r0 : 32);
    const int64_t fld = (V + kLoCols - 1) / kLoCols;
    const int64_t pitch = lo_flags_pitch(V);
    for (int64_t kb0 = 0; kb0 < fld; kb0 += 32) {
        const int64_t kb = kb0 + lane;
        unsigned m = __ballot_sync(0xffffffffu, kb < fld && lo_flags[g * pitch + kb] != 0);
        while (m) {
            const int64_t c = (kb0 + __ffs(m) - 1) * kLoCols + 2 * lane;
            m &= m - 1;
#pragma unroll 1
            for (int r = 0; r < nr; ++r) {
                const float coef = __shfl_sync(0xffffffffu, my_coef, r);
                const float lse2 = __shfl_sync(0xffffffffu, my_lse2, r);
                const int64_t y = __shfl_sync(0xffffffffu, my_y, r);
                if (c >= V) continue;
                // c is even and ldZ a multiple of 8: an aligned pair in the row
                const float2 f = *reinterpret_cast<const float2*>(Z + (r0 + r) * ldZ + c);
                float v[2] = {ex2(fmaf(f.x, kLog2e, -lse2)), ex2(fmaf(f.y, kLog2e, -lse2))};
                const int64_t off = y - c;
                if (off == 0) v[0] = 0.f;
                if (off == 1) v[1] = 0.f;
                T lo[2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const bool keep = coef != 0.f && c + j < V && v[j] >= kLoTau;
                    const float s = coef * v[j];
                    lo[j] = Elem<T>::from_f(keep ? s - Elem<T>::to_f(Elem<T>::from_f(s)) : 0.f);
                }
                T* lrow = S_lo + (r0 + r) * ldS;
                if (c + 2 <= V) {
                    *reinterpret_cast<uint32_t*>(lrow + c) = *reinterpret_cast<uint32_t*>(lo);
                } else {
                    lrow[c] = lo[0];
                }
            }
        }
    }
}

// One warp per block of the plan: first the grad_hidden row blocks, then
// the grad_weight vocab blocks.  The flags are read 16 bytes at a time; a
// lane's listed K blocks go to its place in the warp's ascending list (a
// prefix count over the lanes).
__device__ __forceinline__ int warp_excl_prefix(int x, int lane, int* total) {
    int v = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    *total = __shfl_sync(0xffffffffu, v, 31);
    return v - x;
}

__global__ void lo_plan_kernel(const uint8_t* __restrict__ F, int64_t rows, int64_t V, int R,
                               int C, int* __restrict__ dh_cnt, int64_t* __restrict__ dh_idx,
                               int* __restrict__ dw_cnt, int64_t* __restrict__ dw_idx) {
    const int lane = threadIdx.x & 31;
    const int64_t item = blockIdx.x * int64_t(blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t fld = (V + kLoCols - 1) / kLoCols;
    const int64_t pitch = lo_flags_pitch(V);
    const int64_t groups = (rows + kLoRows - 1) / kLoRows;
    const int64_t n_dh = (rows + R - 1) / R;
    const int64_t n_dw = (V + C - 1) / C;
    if (item < n_dh) {
        // K blocks kb of the row block: lane takes 16 consecutive kb per step
        const int64_t mb = item;
        const int64_t g0 = mb * (R / kLoRows);
        const int ng = static_cast<int>(min(int64_t(R / kLoRows), groups - g0));
        int cnt = 0;
        for (int64_t kb0 = 0; kb0 < fld; kb0 += 32 * 16) {
            const int64_t kb = kb0 + 16 * lane;
            uint32_t bits[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) bits[j] = 0;
            if (kb < fld) {
                for (int i = 0; i < ng; ++i) {
                    const uint4 w = *reinterpret_cast<const uint4*>(F + (g0 + i) * pitch + kb);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if ((ws[j >> 2] >> (8 * (j & 3))) & 0xffu) bits[j] |= 1u << i;
                }
            }
            int n = 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) n += (bits[j] != 0 && kb + j < fld);
            int total;
            int at = cnt + warp_excl_prefix(n, lane, &total);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (bits[j] != 0 && kb + j < fld) dh_idx[mb * fld + at++] = ((kb + j) << 8) | bits[j];
            cnt += total;
        }
        if (lane == 0) dh_cnt[mb] = cnt;
    } else if (item < n_dh + n_dw) {
        // K blocks kb (64 tokens = row groups 2 kb, 2 kb + 1) of the vocab block
        const int64_t vb = item - n_dh;
        const int64_t c0 = vb * (C / kLoCols);
        const int nc = static_cast<int>(min(int64_t(C / kLoCols), fld - c0));
        const int64_t kbs = (rows + 63) / 64;
        int cnt = 0;
        for (int64_t kb0 = 0; kb0 < kbs; kb0 += 32) {
            const int64_t kb = kb0 + lane;
            uint32_t bits = 0;
            if (kb < kbs)
                for (int i = 0; i < 2; ++i) {
                    const int64_t g = 2 * kb + i;
                    if (g >= groups) break;
                    for (int c = 0; c < nc; ++c)
                        if (F[g * pitch + c0 + c]) bits |= 1u << (2 * c + i);
                }
            const unsigned m = __ballot_sync(0xffffffffu, bits != 0);
            if (bits) dw_idx[vb * kbs + cnt + __popc(m & ((1u << lane) - 1))] = (kb << 8) | bits;
            cnt += __popc(m);
        }
        if (lane == 0) dw_cnt[vb] = cnt;
    }
}

cudaError_t launch_lo_plan(const uint8_t* F, int64_t rows, int64_t V, int R, int C,
                           int* dh_cnt, int64_t* dh_idx, int* dw_cnt, int64_t* dw_idx,
                           cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    const int64_t items = (rows + R - 1) / R + (V + C - 1) / C;
    note_launches(1);
    lo_plan_kernel<<<static_cast<unsigned>((items + 7) / 8), 256, 0, s>>>(F, rows, V, R, C,
                                                                          dh_cnt, dh_idx,
                                                                          dw_cnt, dw_idx);
    return cudaGetLastError();
}

cudaError_t launch_softmax_part(const float* Z, int64_t ldZ, int64_t rows, int64_t V,
                                const int64_t* targets, const float* grad, const float* lse,
                                void* S, int64_t ldS, int s_dtype, float* tc, float* db_part,
                                float inv_temp, void* S_lo, uint8_t* lo_flags, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    note_launches(1);
    // a block: 32 rows x (8 warps x 128 columns) per step of its column loop
    int64_t gy = (V + 1023) / 1024;
    if (gy > 65535) gy = 65535;
    const dim3 grid(static_cast<unsigned>((rows + 31) / 32), static_cast<unsigned>(gy));
    const bool db = db_part != nullptr;
    // S_lo without flags: every entry's rest, written by the softmax part
    const bool all = S_lo != nullptr && lo_flags == nullptr;
    if (s_dtype == LL_BF16) {
        auto* Sp = static_cast<__nv_bfloat16*>(S);
        auto* Lp = static_cast<__nv_bfloat16*>(S_lo);
        if (db && all)
            softmax_part_kernel<__nv_bfloat16, true, true><<<grid, 256, 0, s>>>(
                Z, ldZ, rows, V, targets, grad, lse, Sp, ldS, tc, db_part, inv_temp, Lp, nullptr);
        else if (db)
            softmax_part_kernel<__nv_bfloat16, true, false><<<grid, 256, 0, s>>>(
                Z, ldZ, rows, V, targets, grad, lse, Sp, ldS, tc, db_part, inv_temp, Lp, lo_flags);
        else if (all)
            softmax_part_kernel<__nv_bfloat16, false, true><<<grid, 256, 0, s>>>(
                Z, ldZ, rows, V, targets, grad, lse, Sp, ldS, tc, nullptr, inv_temp, Lp, nullptr);
        else
            softmax_part_kernel<__nv_bfloat16, false, false><<<grid, 256, 0, s>>>(
                Z, ldZ, rows, V, targets, grad, lse, Sp, ldS, tc, nullptr, inv_temp, Lp, lo_flags);
    } else if (s_dtype == LL_F16) {
        auto* Sp = static_cast<__half*>(S);
        auto* Lp = static_cast<__half*>(S_lo);
        if (db && all)
            softmax_part_kernel<__half, true, true><<<grid, 256, 0, s>>>(
                Z, ldZ, rows, V, targets, grad, lse, Sp, ldS, tc, db_part, inv_temp, Lp, nullptr);
        else if (db)
            softmax_part_kernel<__half, true, false><<<grid, 256, 0, s>>>(
                Z, ldZ, rows, V, targets, grad, lse, Sp, ldS, tc, db_part, inv_temp, Lp, lo_flags);
        else if (all)
            softmax_part_kernel<__half, false, true><<<grid, 256, 0, s>>>(
                Z, ldZ, rows, V, targets, grad, lse, Sp, ldS, tc, nullptr, inv_temp, Lp, nullptr);
        else
            softmax_part_kernel<__half, false, false><<<grid, 256, 0, s>>>(
                Z, ldZ, rows, V, targets, grad, lse, Sp, ldS, tc, nullptr, inv_temp, Lp, lo_flags);
    } else {
        auto* Sp = static_cast<float*>(S);
        lo_flags = nullptr;  // FP32 S: no split
        if (db)
            softmax_part_kernel<float, true, false><<<grid, 256, 0, s>>>(
                Z, ldZ, rows, V, targets, grad, lse, Sp, ldS, tc, db_part, inv_temp, nullptr,
                nullptr);
        else
            softmax_part_kernel<float, false, false><<<grid, 256, 0, s>>>(
                Z, ldZ, rows, V, targets, grad, lse, Sp, ldS, tc, nullptr, inv_temp, nullptr,
                nullptr);
    }
    if (lo_flags && S_lo) {  // the flagged pieces of S_lo
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        note_launches(1);
        const unsigned gb = static_cast<unsigned>(((rows + 31) / 32 + 7) / 8);
        if (s_dtype == LL_BF16)
            lo_pieces_kernel<__nv_bfloat16><<<gb, 256, 0, s>>>(
                Z, ldZ, rows, V, targets, grad, lse, static_cast<__nv_bfloat16*>(S_lo), ldS,
                lo_flags, inv_temp);
        else
            lo_pieces_kernel<__half><<<gb, 256, 0, s>>>(Z, ldZ, rows, V, targets, grad, lse,
                                                        static_cast<__half*>(S_lo), ldS,
                                                        lo_flags, inv_temp);
    }
    return cudaGetLastError();
}

cudaError_t launch_db_finish(const float* partial, int64_t groups, int64_t V, float* db_acc,
                             int first, int last, const int* offs, const int64_t* keys,
                             const float* tc_all, void* grad_bias, int out_dtype, cudaStream_t s) {
    note_launches(1);
    const unsigned fb = static_cast<unsigned>((V + 31) / 32);
    const unsigned long long* k = reinterpret_cast<const unsigned long long*>(keys);
    if (out_dtype == LL_F32)
        db_finish_kernel<float><<<fb, 256, 0, s>>>(partial, groups, V, db_acc, first, last, offs,
                                                   k, tc_all, static_cast<float*>(grad_bias));
    else if (out_dtype == LL_F16)
        db_finish_kernel<__half><<<fb, 256, 0, s>>>(partial, groups, V, db_acc, first, last, offs,
                                                    k, tc_all, static_cast<__half*>(grad_bias));
    else
        db_finish_kernel<__nv_bfloat16><<<fb, 256, 0, s>>>(
            partial, groups, V, db_acc, first, last, offs, k, tc_all,
            static_cast<__nv_bfloat16*>(grad_bias));
    return cudaGetLastError();
}

cudaError_t launch_sum_ordered(const void* parts, int64_t nparts, int64_t n, int64_t ld,
                               int dtype, void* out, int num_sms, cudaStream_t s) {
    if (n <= 0 || nparts <= 0) return cudaSuccess;
    note_launches(1);
    const int64_t threads = (n + 3) / 4;
    int64_t blocks = (threads + 255) / 256;
    const int64_t cap = int64_t(num_sms) * 8;  // 8 resident blocks of 256 per SM
    if (blocks > cap) blocks = cap;
    const unsigned gb = static_cast<unsigned>(blocks < 1 ? 1 : blocks);
    if (dtype == LL_F32) {
        const bool vec = ld % 4 == 0 && reinterpret_cast<uintptr_t>(parts) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(out) % 16 == 0;
        if (vec)
            sum_ordered_kernel<float, true><<<gb, 256, 0, s>>>(
                static_cast<const float*>(parts), nparts, n, ld, static_cast<float*>(out));
        else
            sum_ordered_kernel<float, false><<<gb, 256, 0, s>>>(
                static_cast<const float*>(parts), nparts, n, ld, static_cast<float*>(out));
    } else if (dtype == LL_BF16) {
        sum_ordered_kernel<__nv_bfloat16, false><<<gb, 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(parts), nparts, n, ld,
            static_cast<__nv_bfloat16*>(out));
    } else {
        sum_ordered_kernel<__half, false><<<gb, 256, 0, s>>>(
            static_cast<const __half*>(parts), nparts, n, ld, static_cast<__half*>(out));
    }
    return cudaGetLastError();
}

// grad_hidden of an FP32 K-split contraction: the parts' partial sums of
// S . W added in ascending part order, then the rules of the grad_hidden
// epilogue: + c_n * W[y_n] where the target lies in this vocab, the softmax
// part alone (+ 0) for a target in another vocab shard, exact +0 for a dead
// row (invalid target or zero upstream gradient).  Four values per thread
// (D % 8 == 0 and every row 16-byte aligned), grid-stride over the rows.
__global__ void __launch_bounds__(256) dh_finish_kernel(
    const float* __restrict__ parts, int ks, int64_t part_rows, int64_t rows, int64_t D,
    const int64_t* __restrict__ targets, const float* __restrict__ grad,
    const float* __restrict__ tc, int64_t V, int shard, const float* __restrict__ W,
    float* __restrict__ dh) {
    const int64_t n4 = rows * (D / 4);
    const int64_t part_pitch = part_rows * D;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t r = i / (D / 4);
        const int64_t d = (i - r * (D / 4)) * 4;
        const int64_t y = targets[r];
        const bool here = y >= 0 && y < V;
        const bool live = (here || (shard && y == kTargetInOtherShard)) && grad[r] != 0.f;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live) {
            // all parts' loads in flight first, then the ascending sum
            const float* p = parts + r * D + d;
            float4 b[kMaxDhParts];
#pragma unroll
            for (int k = 0; k < kMaxDhParts; ++k)
                if (k < ks) b[k] = *reinterpret_cast<const float4*>(p + k * part_pitch);
            a = b[0];
#pragma unroll
            for (int k = 1; k < kMaxDhParts; ++k)
                if (k < ks) a.x += b[k].x, a.y += b[k].y, a.z += b[k].z, a.w += b[k].w;
            if (here) {
                const float c = tc[r];
                const float4 w = *reinterpret_cast<const float4*>(W + y * D + d);
                a.x = fmaf(c, w.x, a.x) + 0.f;
                a.y = fmaf(c, w.y, a.y) + 0.f;
                a.z = fmaf(c, w.z, a.z) + 0.f;
                a.w = fmaf(c, w.w, a.w) + 0.f;
            } else {
                a.x += 0.f, a.y += 0.f, a.z += 0.f, a.w += 0.f;
            }
        }
        *reinterpret_cast<float4*>(dh + r * D + d) = a;
    }
}

cudaError_t launch_dh_finish(const float* parts, int ks, int64_t part_rows, int64_t rows,
                             int64_t D, const int64_t* targets, const float* grad,
                             const float* tc, int64_t V, int shard, const float* W,
                             float* dh, int num_sms, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    if (ks < 1 || ks > kMaxDhParts || D % 4 != 0 || reinterpret_cast<uintptr_t>(parts) % 16 ||
        reinterpret_cast<uintptr_t>(W) % 16 || reinterpret_cast<uintptr_t>(dh) % 16)
        return cudaErrorInvalidValue;
    note_launches(1);
    int64_t blocks = (rows * (D / 4) + 255) / 256;
    const int64_t cap = int64_t(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    dh_finish_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        parts, ks, part_rows, rows, D, targets, grad, tc, V, shard, W, dh);
    return cudaGetLastError();
}

// hT[d, n] = h[n, d] for 16-bit h [N, D] (row stride D, D % 8 == 0) into
// hT [D, ldT] (ldT >= N, a multiple of 8): 64 x 64 tiles through shared
// memory, 16-byte loads and stores.
__global__ void __launch_bounds__(256) transpose16_kernel(const uint16_t* __restrict__ h,
                                                          int64_t N, int64_t D,
                                                          uint16_t* __restrict__ hT, int64_t ldT) {
    __shared__ uint16_t tile[64][64 + 8];
    const int64_t n0 = blockIdx.x * int64_t(64), d0 = blockIdx.y * int64_t(64);
    const int c = (threadIdx.x & 7) * 8;
    for (int r = threadIdx.x >> 3; r < 64; r += 32) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (n0 + r < N && d0 + c < D) v = *reinterpret_cast<const uint4*>(h + (n0 + r) * D + d0 + c);
        const uint16_t* e = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
        for (int j = 0; j < 8; ++j) tile[r][c + j] = e[j];
    }
    __syncthreads();
    for (int r = threadIdx.x >> 3; r < 64; r += 32) {
        if (d0 + r >= D || n0 + c >= N) continue;
        uint4 v;
        uint16_t* e = reinterpret_cast<uint16_t*>(&v);
#pragma unroll
        for (int j = 0; j < 8; ++j) e[j] = tile[c + j][r];
        *reinterpret_cast<uint4*>(hT + (d0 + r) * ldT + n0 + c) = v;
    }
}

cudaError_t launch_transpose16(const void* h, int64_t N, int64_t D, void* hT, int64_t ldT,
                               cudaStream_t s) {
    if (N <= 0 || D <= 0) return cudaSuccess;
    note_launches(1);
    const dim3 grid(static_cast<unsigned>((N + 63) / 64), static_cast<unsigned>((D + 63) / 64));
    transpose16_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(h), N, D,
                                            static_cast<uint16_t*>(hT), ldT);
    return cudaGetLastError();
}

// dst[c, r] = src[r, c] for FP32 src [R, C] (row stride lds, a multiple of 4
// with lds >= round_up(C, 4)) into dst [C, ldd] (ldd a multiple of 4, >=
// round_up(R, 4)): 32 x 32 tiles through shared memory, 16-byte loads and
// stores.  A row's last vector may read src padding past C and write dst
// padding past R; neither is read as data.
__global__ void __launch_bounds__(256) transpose32_kernel(const float* __restrict__ src,
                                                          int64_t R, int64_t C, int64_t lds,
                                                          float* __restrict__ dst, int64_t ldd) {
    __shared__ float tile[32][32 + 1];
    const int q = (threadIdx.x & 7) * 4, t = threadIdx.x >> 3;  // t: 0..31
    const int64_t tr = (R + 31) / 32, n_tiles = tr * ((C + 31) / 32);
    for (int64_t i = blockIdx.x; i < n_tiles; i += gridDim.x) {  // any R, C
        const int64_t r0 = (i % tr) * 32, c0 = (i / tr) * 32;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r0 + t < R && c0 + q < C)
            v = *reinterpret_cast<const float4*>(src + (r0 + t) * lds + c0 + q);
        __syncthreads();  // the previous tile's reads of `tile` are done
        tile[t][q] = v.x, tile[t][q + 1] = v.y, tile[t][q + 2] = v.z, tile[t][q + 3] = v.w;
        __syncthreads();
        if (c0 + t < C && r0 + q < R) {
            const float4 w =
                make_float4(tile[q][t], tile[q + 1][t], tile[q + 2][t], tile[q + 3][t]);
            *reinterpret_cast<float4*>(dst + (c0 + t) * ldd + r0 + q) = w;
        }
    }
}

cudaError_t launch_transpose32(const float* src, int64_t R, int64_t C, int64_t lds, float* dst,
                               int64_t ldd, cudaStream_t s) {
    if (R <= 0 || C <= 0) return cudaSuccess;
    if (lds % 4 || ldd % 4 || lds < ((C + 3) / 4) * 4 || ldd < ((R + 3) / 4) * 4 ||
        reinterpret_cast<uintptr_t>(src) % 16 || reinterpret_cast<uintptr_t>(dst) % 16)
        return cudaErrorInvalidValue;
    note_launches(1);
    const int64_t n_tiles = ((R + 31) / 32) * ((C + 31) / 32);
    const int64_t cap = int64_t(1) << 20;  // blocks; more tiles are visited grid-stride
    transpose32_kernel<<<static_cast<unsigned>(n_tiles < cap ? n_tiles : cap), 256, 0, s>>>(
        src, R, C, lds, dst, ldd);
    return cudaGetLastError();
}

cudaError_t launch_fill_zero(void* p, int64_t n_elems, int dtype, cudaStream_t s) {
    if (n_elems <= 0) return cudaSuccess;
    note_launches(1);
    if (dtype == LL_F32) {
        fill_zero_kernel<<<1024, 256, 0, s>>>(static_cast<uint32_t*>(p), n_elems);
    } else {
        fill_zero_u16_kernel<<<1024, 256, 0, s>>>(static_cast<uint16_t*>(p), n_elems);
    }
    return cudaGetLastError();
}

cudaError_t launch_unsatisfied_wait(int* flag, int* status, uint64_t wait_ns, cudaStream_t s) {
    note_launches(1);
    unsatisfied_wait_kernel<<<1, 32, 0, s>>>(flag, status, wait_ns);
    return cudaGetLastError();
}

}  // namespace ll
