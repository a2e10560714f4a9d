// Logits-input logp forward and backward (HBM-streaming).
//
// RL-Kernel PR #495, "Summary": logp of the target token from [N, V]
// logits, one block per row, fixed reduction tree (deterministic and
// batch-invariant), 0 / zero gradient for targets outside [0, V).  Unlike
// the kernel on that page (a max pass and a sum-exp pass, and the backward
// re-reading the row three times), the forward here keeps an online running
// max and rescaled sum in one pass, and the backward uses the saved lse, so
// each row is read once (forward) or read once and written once (backward).
//
// Element-to-thread assignment depends only on the column index and the
// block size, never on the row index or N, which gives batch invariance.
//
// With a known upstream gradient, logits_fwd_bwd_kernel runs both per row,
// back to back, so the row's second read is served by L2: one HBM read and
// one write per row (4 V bytes instead of the two kernels' 6 V).
#include <math.h>

#include "ll_device.cuh"

namespace ll {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;  // 16-byte loads in flight per thread

struct MS {
    float m;  // running max, log2 units
    float s;  // sum of 2^(u - m)
};

__device__ __forceinline__ MS ms_combine(MS a, MS b) {
    const float M = fmaxf(a.m, b.m);
    if (M == -INFINITY) return {-INFINITY, 0.f};
    return {M, a.s * ex2(a.m - M) + b.s * ex2(b.m - M)};
}

// Fold 8 values (natural units) into the running (m, s).
__device__ __forceinline__ void ms_fold8(MS& st, const float (&f)[8]) {
    const float vmax =
        max3f(max3f(f[0], f[1], f[2]), max3f(f[3], f[4], f[5]), fmaxf(f[6], f[7]));
    const float mu = vmax * kLog2e;
    if (mu > st.m) {
        st.s = st.s * ex2(st.m - mu);
        st.m = mu;
    }
    if (st.m != -INFINITY) {
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) acc += ex2(fmaf(f[j], kLog2e, -st.m));
        st.s += acc;
    }
}

__device__ __forceinline__ void ms_fold1(MS& st, float z) {
    const float mu = z * kLog2e;
    if (mu > st.m) {
        st.s = st.s * ex2(st.m - mu);
        st.m = mu;
    }
    if (st.m != -INFINITY) st.s += ex2(fmaf(z, kLog2e, -st.m));
}

// Block-wide combine in a fixed order: butterfly within each warp (lane 0's
// value is used), then warp results in ascending warp order by thread 0.
template <int NT = kThreads>
__device__ __forceinline__ MS block_reduce(MS st, MS* sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MS other;
        other.m = __shfl_xor_sync(0xffffffffu, st.m, o);
        other.s = __shfl_xor_sync(0xffffffffu, st.s, o);
        st = ms_combine(st, other);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sh[warp] = st;
    __syncthreads();
    MS r = {-INFINITY, 0.f};
    if (threadIdx.x == 0) {
        for (int w = 0; w < NT / 32; ++w) r = ms_combine(r, sh[w]);
    }
    return r;
}

// 8 elements as loaded (16-bit types: one 16-byte vector, kept packed until
// used, so a deep unroll costs 4 registers per vector; float: two vectors).
template <typename T>
struct Raw8 {
    uint4 a, b;  // b unused for 16-bit types
};
template <typename T, bool HINT>
__device__ __forceinline__ Raw8<T> ld_raw(const T* p, uint64_t pol) {
    Raw8<T> r;
    if constexpr (HINT) {
        r.a = ld16_hint(p, pol);
        if constexpr (sizeof(T) == 4) r.b = ld16_hint(p + 4, pol);
    } else {
        r.a = *reinterpret_cast<const uint4*>(p);
        if constexpr (sizeof(T) == 4) r.b = *reinterpret_cast<const uint4*>(p + 4);
    }
    return r;
}
template <typename T>
__device__ __forceinline__ void unpack(const Raw8<T>& r, float (&f)[8]) {
    if constexpr (sizeof(T) == 4) {
        f[0] = __uint_as_float(r.a.x); f[1] = __uint_as_float(r.a.y);
        f[2] = __uint_as_float(r.a.z); f[3] = __uint_as_float(r.a.w);
        f[4] = __uint_as_float(r.b.x); f[5] = __uint_as_float(r.b.y);
        f[6] = __uint_as_float(r.b.z); f[7] = __uint_as_float(r.b.w);
    } else {
        const T* e = reinterpret_cast<const T*>(&r.a);
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = Elem<T>::to_f(e[j]);
    }
}
template <typename T, bool HINT>
__device__ __forceinline__ void st8(T* p, const float (&f)[8], uint64_t pol) {
    if constexpr (HINT)
        store8_hint(p, f, pol);
    else
        store8(p, f);
}

// The tempered logits x / T (it = 1 / T); T = 1 skips the exact multiply.
__device__ __forceinline__ void scale8(float (&f)[8], float it) {
    if (it == 1.f) return;
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] *= it;
}

// Gradient of 8 tempered logits z (columns c0 .. c0 + 7) of a live row:
// g * (onehot - p), p = 2^(z log2e - lse2).  Off target onehot - p = -p
// exactly (0 - p and -p differ only for p = +0, where either gives +0 after
// the + 0), so only the target column takes the 1 - p form.
__device__ __forceinline__ void grad8(float (&f)[8], int64_t c0, int64_t y, float g,
                                      float lse2) {
    float p[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        p[j] = ex2(fmaf(f[j], kLog2e, -lse2));
        f[j] = fmaf(g, -p[j], 0.f);  // + 0 keeps empty results at +0
    }
    const int64_t off = y - c0;
    if (off >= 0 && off < 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j == off) f[j] = fmaf(g, 1.f - p[j], 0.f);
    }
}

// This thread's (max, sum-exp) of row x: 8-element vectors tid, tid + T,
// tid + 2T, ... (T = block size) in that order, U of them loaded at a time
// (the order, hence the result, does not depend on U), then the scalar tail.
// it = 1 / temperature: the fold sees the tempered logits x * it (exact for it = 1).
template <typename T, int U, bool HINT, int NT = kThreads>
__device__ __forceinline__ MS row_partial(const T* x, int64_t V, int vec_ok, uint64_t pol,
                                          float it) {
    MS st = {-INFINITY, 0.f};
    int64_t done = 0;
    if (vec_ok) {
        const int64_t nvec = V / 8;
        int64_t i = threadIdx.x;
        for (; i + (U - 1) * NT < nvec; i += U * NT) {
            Raw8<T> r[U];
#pragma unroll
            for (int u = 0; u < U; ++u) r[u] = ld_raw<T, HINT>(x + (i + u * NT) * 8, pol);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float f[8];
                unpack(r[u], f);
                scale8(f, it);
                ms_fold8(st, f);
            }
        }
        for (; i < nvec; i += NT) {
            float f[8];
            unpack(ld_raw<T, HINT>(x + i * 8, pol), f);
            scale8(f, it);
            ms_fold8(st, f);
        }
        done = nvec * 8;
    }
    for (int64_t j = done + threadIdx.x; j < V; j += NT)
        ms_fold1(st, Elem<T>::to_f(x[j]) * it);
    return st;
}

// lse of a row from thread 0's block result.
__device__ __forceinline__ float lse_of(const MS& r) {
    return (r.m == -INFINITY) ? -INFINITY : r.m * kLn2 + logf(r.s);
}

__device__ __forceinline__ float grad_elem(float z, int64_t c, int64_t y, float g, float lse2) {
    const float p = ex2(fmaf(z, kLog2e, -lse2));
    const float oh = (c == y) ? 1.f : 0.f;
    return fmaf(g, oh - p, 0.f);  // + 0 keeps empty results at +0
}

// Gradient row o = g * (onehot(y) - exp(x - lse)) (all +0 when !live); each
// thread reads a vector of x and writes the same vector of o, so o may be x.
// With a temperature (it = 1 / T) the caller passes g * it and the tempered
// lse; the logits are scaled by it here.
template <typename T, int U, bool HINT, int NT = kThreads>
__device__ __forceinline__ void row_grad(const T* x, T* o, int64_t V, int vec_ok, int64_t y,
                                         float g, bool live, float lse2, uint64_t pol_ld,
                                         uint64_t pol_st, float it) {
    int64_t done = 0;
    if (vec_ok) {
        const int64_t nvec = V / 8;
        if (!live) {
            const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int64_t i = threadIdx.x; i < nvec; i += NT) st8<T, HINT>(o + i * 8, z, pol_st);
        } else {
            int64_t i = threadIdx.x;
            for (; i + (U - 1) * NT < nvec; i += U * NT) {
                Raw8<T> r[U];
#pragma unroll
                for (int u = 0; u < U; ++u)
                    r[u] = ld_raw<T, HINT>(x + (i + u * NT) * 8, pol_ld);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t c0 = (i + u * NT) * 8;
                    float f[8];
                    unpack(r[u], f);
#pragma unroll
                    scale8(f, it);
                    grad8(f, c0, y, g, lse2);
                    st8<T, HINT>(o + c0, f, pol_st);
                }
            }
            for (; i < nvec; i += NT) {
                float f[8];
                const int64_t c0 = i * 8;
                unpack(ld_raw<T, HINT>(x + c0, pol_ld), f);
                scale8(f, it);
                grad8(f, c0, y, g, lse2);
                st8<T, HINT>(o + c0, f, pol_st);
            }
        }
        done = nvec * 8;
    }
    for (int64_t j = done + threadIdx.x; j < V; j += NT) {
        const float v = live ? grad_elem(Elem<T>::to_f(x[j]) * it, j, y, g, lse2) : 0.f;
        o[j] = Elem<T>::from_f(v);
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) logits_fwd_kernel(const T* __restrict__ logits,
                                                              int64_t ld,
                                                              const int64_t* __restrict__ targets,
                                                              int64_t V, float* __restrict__ logp,
                                                              float* __restrict__ lse_out,
                                                              int vec_ok, float it) {
    __shared__ MS sh[kWarps];
    const int64_t row = blockIdx.x;
    const T* x = logits + row * ld;
    const MS r = block_reduce(row_partial<T, kUnroll, false>(x, V, vec_ok, 0, it), sh);
    if (threadIdx.x == 0) {
        const float lse = lse_of(r);
        const int64_t y = targets[row];
        const bool valid = (y >= 0) && (y < V);
        logp[row] = valid ? Elem<T>::to_f(x[y]) * it - lse : 0.f;
        lse_out[row] = lse;
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) logits_bwd_kernel(
    const float* __restrict__ grad, const T* __restrict__ logits, int64_t ld,
    const int64_t* __restrict__ targets, const float* __restrict__ lse, int64_t V,
    T* __restrict__ out, int vec_ok, float it) {
    const int64_t row = blockIdx.x;
    const int64_t y = targets[row];
    const float g = grad[row];
    const bool live = (y >= 0) && (y < V) && (g != 0.f);
    row_grad<T, kUnroll, false>(logits + row * ld, out + row * ld, V, vec_ok, y, g * it, live,
                                lse[row] * kLog2e, 0, 0, it);
}

// Forward and backward of each row in turn (a known upstream gradient): the
// row's second read, right after its first, finds it in L2, so HBM sees one
// read and one write per row.  The blocks are persistent (rows blockIdx.x,
// blockIdx.x + gridDim.x, ...), which bounds the rows in flight, hence the
// L2 footprint; the first read keeps its lines (evict_last), the second read
// and the gradient stores release theirs (evict_first).  The row code is the
// one of logits_fwd_kernel and logits_bwd_kernel, so every result is bitwise
// theirs.  grad_logits may be the logits buffer itself.
template <typename T, int U, int NT = kThreads>
__global__ void __launch_bounds__(NT) logits_fwd_bwd_kernel(
    const float* __restrict__ grad, const T* logits, int64_t ld,
    const int64_t* __restrict__ targets, int64_t N, int64_t V, float* __restrict__ logp,
    float* __restrict__ lse_out, T* out, int vec_ok, float it) {
    __shared__ MS sh[NT / 32];
    __shared__ float lse_sh;
    const uint64_t keep = l2_evict_last(), drop = l2_evict_first();
    for (int64_t row = blockIdx.x; row < N; row += gridDim.x) {
        const T* x = logits + row * ld;
        const MS r = block_reduce<NT>(row_partial<T, U, true, NT>(x, V, vec_ok, keep, it), sh);
        const int64_t y = targets[row];
        const float g = grad[row];
        const bool valid = (y >= 0) && (y < V);
        if (threadIdx.x == 0) {
            const float lse = lse_of(r);
            logp[row] = valid ? Elem<T>::to_f(x[y]) * it - lse : 0.f;
            lse_out[row] = lse;
            lse_sh = lse;
        }
        __syncthreads();  // lse_sh; also thread 0 is done with sh and x[y]
        row_grad<T, U, true, NT>(x, out + row * ld, V, vec_ok, y, g * it, valid && g != 0.f,
                             lse_sh * kLog2e, drop, drop, it);
    }
}

// 16-byte copy from global to shared memory that does not pass through
// registers (cp.async); completed by cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Rows held on chip (16-bit logits): each row is read from HBM once and
// kept in the block's registers and shared memory between its forward and
// backward, so nothing of it has to survive in L2.  One block of kThreads
// per SM; thread t owns the 16-byte vectors t, t + kThreads, t + 2 kThreads,
// ... of the row (the assignment of row_partial / row_grad): the first
// kOnchipRegVecs in registers, the next `ks` in shared memory (filled by
// cp.async).  The forward folds them in ascending order and reduces with
// block_reduce, the backward writes the gradient from the same copies, so
// every result is bitwise that of logits_fwd_kernel and logits_bwd_kernel.
// While the backward consumes a register or a shared-memory vector, the same
// vector of the block's next row is loaded into its place, so the next
// row's HBM reads overlap this row's gradient stores.  (Holding the first
// vectors in shared memory and the last in registers, so that the next
// row's shared-memory part is requested first, measured slower: 4.39 against
// 3.94 ms at 32768 x 151936.)  A thread reads its whole row before writing
// any of it: grad_logits may be the logits.
constexpr int kOnchipRegVecs = 16;
constexpr int kOnchipMaxSmemVecs = 27;  // 27 x 512 x 16 B = 216 KB of shared memory

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) logits_fwd_bwd_onchip_kernel(
    const float* __restrict__ grad, const T* logits, int64_t ld,
    const int64_t* __restrict__ targets, int64_t N, int64_t V, float* __restrict__ logp,
    float* __restrict__ lse_out, T* out, float it, int ks) {
    extern __shared__ uint4 sm[];  // [ks][kThreads]
    __shared__ MS sh[kWarps];
    __shared__ float lse_sh;
    const int t = threadIdx.x;
    const int64_t nvec = V / 8;
    const uint64_t drop = l2_evict_first();
    uint4 rr[kOnchipRegVecs];
    int64_t row = blockIdx.x;
    if (row >= N) return;
    {  // the first row's loads
        const T* x = logits + row * ld;
        for (int k = 0; k < ks; ++k) {
            const int64_t i = t + int64_t(kThreads) * (kOnchipRegVecs + k);
            if (i < nvec) cp_async16(&sm[k * kThreads + t], x + i * 8);
        }
#pragma unroll
        for (int k = 0; k < kOnchipRegVecs; ++k) {
            const int64_t i = t + int64_t(kThreads) * k;
            if (i < nvec) rr[k] = *reinterpret_cast<const uint4*>(x + i * 8);
        }
    }
    for (; row < N; row += gridDim.x) {
        const T* x = logits + row * ld;
        // forward: this thread's vectors in ascending order, then the tail
        MS st = {-INFINITY, 0.f};
#pragma unroll
        for (int k = 0; k < kOnchipRegVecs; ++k) {
            if (t + int64_t(kThreads) * k < nvec) {
                Raw8<T> r;
                r.a = rr[k];
                float f[8];
                unpack(r, f);
                scale8(f, it);
                ms_fold8(st, f);
            }
        }
        cp_async_wait_all();
        for (int k = 0; k < ks; ++k) {
            if (t + int64_t(kThreads) * (kOnchipRegVecs + k) < nvec) {
                Raw8<T> r;
                r.a = sm[k * kThreads + t];
                float f[8];
                unpack(r, f);
                scale8(f, it);
                ms_fold8(st, f);
            }
        }
        for (int64_t j = nvec * 8 + t; j < V; j += kThreads)
            ms_fold1(st, Elem<T>::to_f(x[j]) * it);
        const MS red = block_reduce(st, sh);
        const int64_t y = targets[row];
        const float g = grad[row];
        const bool valid = (y >= 0) && (y < V);
        if (t == 0) {
            const float lse = lse_of(red);
            logp[row] = valid ? Elem<T>::to_f(x[y]) * it - lse : 0.f;
            lse_out[row] = lse;
            lse_sh = lse;
        }
        __syncthreads();  // lse_sh; also thread 0 is done with sh and x[y]
        const bool live = valid && g != 0.f;
        const float gi = g * it;
        const float lse2 = lse_sh * kLog2e;
        // backward from the on-chip copies; each consumed vector is refilled
        // with the same vector of the next row
        const int64_t next = row + gridDim.x;
        const T* xn = logits + next * ld;
        T* o = out + row * ld;
#pragma unroll
        for (int k = 0; k < kOnchipRegVecs; ++k) {
            const int64_t i = t + int64_t(kThreads) * k;
            if (i < nvec) {
                float f[8];
                if (live) {
                    Raw8<T> r;
                    r.a = rr[k];
                    unpack(r, f);
                    scale8(f, it);
                    grad8(f, i * 8, y, gi, lse2);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) f[j] = 0.f;
                }
                st8<T, true>(o + i * 8, f, drop);
                if (next < N) rr[k] = *reinterpret_cast<const uint4*>(xn + i * 8);
            }
        }
        for (int k = 0; k < ks; ++k) {
            const int64_t i = t + int64_t(kThreads) * (kOnchipRegVecs + k);
            if (i < nvec) {
                float f[8];
                if (live) {
                    Raw8<T> r;
                    r.a = sm[k * kThreads + t];
                    unpack(r, f);
                    scale8(f, it);
                    grad8(f, i * 8, y, gi, lse2);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) f[j] = 0.f;
                }
                st8<T, true>(o + i * 8, f, drop);
                if (next < N) cp_async16(&sm[k * kThreads + t], xn + i * 8);
            }
        }
        for (int64_t j = nvec * 8 + t; j < V; j += kThreads) {
            const float v = live ? grad_elem(Elem<T>::to_f(x[j]) * it, j, y, gi, lse2) : 0.f;
            o[j] = Elem<T>::from_f(v);
        }
    }
    cp_async_wait_all();
}

template <typename T>
bool vec_ok(const void* p, int64_t ld) {
    return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((ld * int64_t(sizeof(T))) % 16 == 0);
}

}  // namespace

cudaError_t launch_logits_fwd(const void* logits, int64_t ld, int dtype, const int64_t* targets,
                              int64_t N, int64_t V, float* logp, float* lse, float it,
                              cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(N));
    note_launches(1);
    switch (dtype) {
        case LL_BF16:
            logits_fwd_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(
                static_cast<const __nv_bfloat16*>(logits), ld, targets, V, logp, lse,
                vec_ok<__nv_bfloat16>(logits, ld), it);
            break;
        case LL_F16:
            logits_fwd_kernel<__half><<<grid, kThreads, 0, s>>>(
                static_cast<const __half*>(logits), ld, targets, V, logp, lse,
                vec_ok<__half>(logits, ld), it);
            break;
        default:
            logits_fwd_kernel<float><<<grid, kThreads, 0, s>>>(
                static_cast<const float*>(logits), ld, targets, V, logp, lse,
                vec_ok<float>(logits, ld), it);
    }
    return cudaGetLastError();
}

cudaError_t launch_logits_bwd(const float* grad, const void* logits, int64_t ld, int dtype,
                              const int64_t* targets, const float* lse, int64_t N, int64_t V,
                              void* grad_logits, float it, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(N));
    note_launches(1);
    switch (dtype) {
        case LL_BF16: {
            const int ok = vec_ok<__nv_bfloat16>(logits, ld) && vec_ok<__nv_bfloat16>(grad_logits, ld);
            logits_bwd_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(
                grad, static_cast<const __nv_bfloat16*>(logits), ld, targets, lse, V,
                static_cast<__nv_bfloat16*>(grad_logits), ok, it);
            break;
        }
        case LL_F16: {
            const int ok = vec_ok<__half>(logits, ld) && vec_ok<__half>(grad_logits, ld);
            logits_bwd_kernel<__half><<<grid, kThreads, 0, s>>>(
                grad, static_cast<const __half*>(logits), ld, targets, lse, V,
                static_cast<__half*>(grad_logits), ok, it);
            break;
        }
        default: {
            const int ok = vec_ok<float>(logits, ld) && vec_ok<float>(grad_logits, ld);
            logits_bwd_kernel<float><<<grid, kThreads, 0, s>>>(
                grad, static_cast<const float*>(logits), ld, targets, lse, V,
                static_cast<float*>(grad_logits), ok, it);
        }
    }
    return cudaGetLastError();
}

// Resident blocks of the fused kernel per SM (rows in flight per SM).
constexpr int kFusedBlocksPerSm = 2;
constexpr int kFusedUnroll = 8;

// The on-chip kernel for 16-bit rows that fit: vectors per thread beyond the
// registers' share, or -1 when the row does not fit (or is not vectorised).
int onchip_smem_vecs(int64_t V, int ok) {
    if (!ok) return -1;
    const int64_t per_thread = (V / 8 + kThreads - 1) / kThreads;
    const int64_t ks = per_thread > kOnchipRegVecs ? per_thread - kOnchipRegVecs : 0;
    return ks <= kOnchipMaxSmemVecs ? static_cast<int>(ks) : -1;
}

template <typename T>
cudaError_t launch_onchip(const float* grad, const T* logits, int64_t ld, const int64_t* targets,
                          int64_t N, int64_t V, float* logp, float* lse, T* out, float it,
                          int ks, const DevInfo& dev, cudaStream_t s) {
    auto kern = logits_fwd_bwd_onchip_kernel<T>;
    const int smem = ks * kThreads * 16;
    static int configured[64] = {0};
    if (dev.device < 64 && !configured[dev.device]) {
        const cudaError_t e = cudaFuncSetAttribute(
            kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kOnchipMaxSmemVecs * kThreads * 16);
        if (e != cudaSuccess) return e;
        configured[dev.device] = 1;
    }
    const int64_t blocks = N < dev.num_sms ? N : dev.num_sms;
    kern<<<static_cast<unsigned>(blocks), kThreads, smem, s>>>(grad, logits, ld, targets, N, V,
                                                               logp, lse, out, it, ks);
    return cudaGetLastError();
}

cudaError_t launch_logits_fused(const float* grad, const void* logits, int64_t ld, int dtype,
                                const int64_t* targets, int64_t N, int64_t V, float* logp,
                                float* lse, void* grad_logits, float it, const DevInfo& dev,
                                cudaStream_t s) {
    if (N <= 0) return cudaSuccess;
    if (dtype == LL_BF16 || dtype == LL_F16) {
        const int ok = dtype == LL_BF16
                           ? vec_ok<__nv_bfloat16>(logits, ld) && vec_ok<__nv_bfloat16>(grad_logits, ld)
                           : vec_ok<__half>(logits, ld) && vec_ok<__half>(grad_logits, ld);
        const int ks = onchip_smem_vecs(V, ok);
        if (ks >= 0) {
            note_launches(1);
            if (dtype == LL_BF16)
                return launch_onchip<__nv_bfloat16>(
                    grad, static_cast<const __nv_bfloat16*>(logits), ld, targets, N, V, logp, lse,
                    static_cast<__nv_bfloat16*>(grad_logits), it, ks, dev, s);
            return launch_onchip<__half>(grad, static_cast<const __half*>(logits), ld, targets, N,
                                         V, logp, lse, static_cast<__half*>(grad_logits), it, ks,
                                         dev, s);
        }
    }
    int64_t blocks = int64_t(dev.num_sms) * kFusedBlocksPerSm;
    if (blocks > N) blocks = N;
    const dim3 grid(static_cast<unsigned>(blocks));
    note_launches(1);
    switch (dtype) {
        case LL_BF16: {
            const int ok = vec_ok<__nv_bfloat16>(logits, ld) && vec_ok<__nv_bfloat16>(grad_logits, ld);
            logits_fwd_bwd_kernel<__nv_bfloat16, kFusedUnroll><<<grid, kThreads, 0, s>>>(
                grad, static_cast<const __nv_bfloat16*>(logits), ld, targets, N, V, logp, lse,
                static_cast<__nv_bfloat16*>(grad_logits), ok, it);
            break;
        }
        case LL_F16: {
            const int ok = vec_ok<__half>(logits, ld) && vec_ok<__half>(grad_logits, ld);
            logits_fwd_bwd_kernel<__half, kFusedUnroll><<<grid, kThreads, 0, s>>>(
                grad, static_cast<const __half*>(logits), ld, targets, N, V, logp, lse,
                static_cast<__half*>(grad_logits), ok, it);
            break;
        }
        default: {
            const int ok = vec_ok<float>(logits, ld) && vec_ok<float>(grad_logits, ld);
            logits_fwd_bwd_kernel<float, kFusedUnroll><<<grid, kThreads, 0, s>>>(
                grad, static_cast<const float*>(logits), ld, targets, N, V, logp, lse,
                static_cast<float*>(grad_logits), ok, it);
        }
    }
    return cudaGetLastError();
}

}  // namespace ll
