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

__global__ void lse_merge_kernel(const float* __restrict__ pm, const float* __restrict__ ps,
                                 const float* __restrict__ zy, int64_t ld, int64_t n_segs,
                                 const int64_t* __restrict__ targets, int64_t N, int64_t V,
                                 float* __restrict__ logp, float* __restrict__ lse_out) {
    const int64_t r = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    if (r >= N) return;
    float M = -INFINITY;
    for (int64_t j = 0; j < n_segs; ++j) M = fmaxf(M, pm[j * ld + r]);
    float lse = -INFINITY;
    if (M != -INFINITY) {
        float S = 0.f;
        for (int64_t j = 0; j < n_segs; ++j) S += ps[j * ld + r] * ex2(pm[j * ld + r] - M);
        lse = M * kLn2 + logf(S);
    }
    const int64_t y = targets[r];
    logp[r] = (y >= 0 && y < V) ? zy[r] - lse : 0.f;
    lse_out[r] = lse;
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

template <typename T>
__global__ void db_partial_kernel(const T* __restrict__ S, int64_t ldS, int64_t rows, int64_t V,
                                  int64_t rows_per_group, float* __restrict__ partial) {
    const int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    const int64_t g = blockIdx.y;
    if (v >= V) return;
    const int64_t r0 = g * rows_per_group;
    const int64_t r1 = min(rows, r0 + rows_per_group);
    float acc = 0.f;
    for (int64_t r = r0; r < r1; ++r) acc += Elem<T>::to_f(S[r * ldS + v]);
    partial[g * V + v] = acc;
}

template <typename TO>
__global__ void db_finish_kernel(const float* __restrict__ partial, int64_t groups, int64_t V,
                                 float* __restrict__ db_acc, int first, int last,
                                 const int* __restrict__ offs,
                                 const unsigned long long* __restrict__ keys,
                                 const float* __restrict__ tc_all, TO* __restrict__ out) {
    const int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    if (v >= V) return;
    float acc = first ? 0.f : db_acc[v];
    for (int64_t g = 0; g < groups; ++g) acc = acc + partial[g * V + v];
    if (last) {
        for (int i = offs[v]; i < offs[v + 1]; ++i) {
            acc = acc + tc_all[keys[i] & 0xffffffffull];
        }
        out[v] = Elem<TO>::from_f(acc + 0.f);
    } else {
        db_acc[v] = acc;
    }
}

// Softmax part from stored FP32 logits, tile by tile exactly as the
// recompute epilogue forms it: a warp takes 32 rows x 32 columns with lane =
// row, p = 2^(z * log2e - lse * log2e), S = -grad * p off target, S = 0 and
// tc = grad * (1 - p) at the target, and (with db_part) the same butterfly
// column sums over the 32 rows.  Grid: x = row groups of 32, y = column
// blocks of 4 warps x 32 columns (strided).
template <typename T>
__global__ void __launch_bounds__(128) softmax_part_kernel(
    const float* __restrict__ Z, int64_t ldZ, int64_t rows, int64_t V,
    const int64_t* __restrict__ targets, const float* __restrict__ grad,
    const float* __restrict__ lse, T* __restrict__ S, int64_t ldS, float* __restrict__ tc,
    float* __restrict__ db_part, float inv_temp, T* __restrict__ S_lo) {
    const int lane = threadIdx.x & 31;
    const int64_t row = blockIdx.x * int64_t(32) + lane;
    const bool rvalid = row < rows;
    const int64_t y = rvalid ? targets[row] : -1;
    const float g = rvalid ? grad[row] : 0.f;
    const bool live = rvalid && y >= 0 && y < V && g != 0.f;
    const float coef = live ? -g * inv_temp : 0.f;
    const float lse2 = rvalid ? lse[row] * kLog2e : 0.f;
    const int64_t nchunks = (V + 31) / 32;
    for (int64_t ch = blockIdx.y * 4 + (threadIdx.x >> 5); ch < nchunks; ch += gridDim.y * 4) {
        const int64_t col0 = ch * 32;
        float v[32];
        if (rvalid) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (col0 + 8 * q + 8 <= V) {
                    load8(Z + row * ldZ + col0 + 8 * q, f);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (col0 + 8 * q + j < V) f[j] = Z[row * ldZ + col0 + 8 * q + j];
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) v[8 * q + j] = f[j];
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = ex2(fmaf(v[j], kLog2e, -lse2));
            const int64_t off = y - col0;
            if (off >= 0 && off < 32) {
                float py = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j == off) py = v[j];
                tc[row] = coef != 0.f ? -coef * (1.f - py) : 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j == off) v[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = coef * v[j];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (col0 + 8 * q >= V) break;
                float f[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) f[j] = v[8 * q + j];
                if (col0 + 8 * q + 8 <= V) {
                    store8(S + row * ldS + col0 + 8 * q, f);
                } else {
                    for (int j = 0; j < 8 && col0 + 8 * q + j < V; ++j)
                        S[row * ldS + col0 + 8 * q + j] = Elem<T>::from_f(f[j]);
                }
                if (S_lo) {  // hi / lo split: the rounding rest S - S_hi
#pragma unroll
                    for (int j = 0; j < 8; ++j) f[j] -= Elem<T>::to_f(Elem<T>::from_f(f[j]));
                    if (col0 + 8 * q + 8 <= V) {
                        store8(S_lo + row * ldS + col0 + 8 * q, f);
                    } else {
                        for (int j = 0; j < 8 && col0 + 8 * q + j < V; ++j)
                            S_lo[row * ldS + col0 + 8 * q + j] = Elem<T>::from_f(f[j]);
                    }
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        if (db_part) {  // column sums over the 32 rows, the recompute's butterfly
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const bool up = (lane & o) != 0;
#pragma unroll
                for (int j = 0; j < o; ++j) {
                    const float keep = up ? v[j + o] : v[j];
                    const float send = up ? v[j] : v[j + o];
                    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            const int64_t col = col0 + lane;
            if (col < V && blockIdx.x * int64_t(32) < rows) db_part[blockIdx.x * V + col] = v[0];
        }
    }
    if (rvalid && !(y >= 0 && y < V) && blockIdx.y == 0 && threadIdx.x < 32) tc[row] = 0.f;
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

int64_t pow2_at_least(int64_t n) {
    int64_t p = kSortSeg;
    while (p < n) p <<= 1;
    return p;
}

}  // namespace

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

size_t db_partial_bytes(int64_t Nc, int64_t V) {
    const int64_t groups = Nc < 64 ? (Nc > 0 ? Nc : 1) : 64;
    return static_cast<size_t>(groups + 1) * static_cast<size_t>(V) * 4;
}

cudaError_t launch_db_chunk(const void* S, int64_t ldS, int s_dtype, int64_t rows, int64_t V,
                            float* partial, float* db_acc, int first, int last, const int* offs,
                            const int64_t* keys, const float* tc_all, void* grad_bias,
                            int out_dtype, cudaStream_t s) {
    const int64_t groups = rows < 64 ? (rows > 0 ? rows : 1) : 64;
    const int64_t rpg = (rows + groups - 1) / groups;
    const dim3 grid(static_cast<unsigned>((V + 255) / 256), static_cast<unsigned>(groups));
    note_launches(2);
    if (s_dtype == LL_F32)
        db_partial_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(S), ldS, rows, V,
                                                      rpg, partial);
    else if (s_dtype == LL_F16)
        db_partial_kernel<__half><<<grid, 256, 0, s>>>(static_cast<const __half*>(S), ldS, rows,
                                                       V, rpg, partial);
    else
        db_partial_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(S), ldS, rows, V, rpg, partial);
    const unsigned fb = static_cast<unsigned>((V + 255) / 256);
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

cudaError_t launch_softmax_part(const float* Z, int64_t ldZ, int64_t rows, int64_t V,
                                const int64_t* targets, const float* grad, const float* lse,
                                void* S, int64_t ldS, int s_dtype, float* tc, float* db_part,
                                float inv_temp, void* S_lo, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    note_launches(1);
    const int64_t nchunks = (V + 31) / 32;
    int64_t gy = (nchunks + 3) / 4;
    if (gy > 64) gy = 64;
    const dim3 grid(static_cast<unsigned>((rows + 31) / 32), static_cast<unsigned>(gy));
    if (s_dtype == LL_BF16)
        softmax_part_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(
            Z, ldZ, rows, V, targets, grad, lse, static_cast<__nv_bfloat16*>(S), ldS, tc, db_part,
            inv_temp, static_cast<__nv_bfloat16*>(S_lo));
    else if (s_dtype == LL_F16)
        softmax_part_kernel<__half><<<grid, 128, 0, s>>>(Z, ldZ, rows, V, targets, grad, lse,
                                                         static_cast<__half*>(S), ldS, tc, db_part,
                                                         inv_temp, static_cast<__half*>(S_lo));
    else
        softmax_part_kernel<float><<<grid, 128, 0, s>>>(Z, ldZ, rows, V, targets, grad, lse,
                                                        static_cast<float*>(S), ldS, tc, db_part,
                                                        inv_temp, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_db_finish(const float* partial, int64_t groups, int64_t V, float* db_acc,
                             int first, int last, const int* offs, const int64_t* keys,
                             const float* tc_all, void* grad_bias, int out_dtype, cudaStream_t s) {
    note_launches(1);
    const unsigned fb = static_cast<unsigned>((V + 255) / 256);
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
