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
    float vmax = f[0];
#pragma unroll
    for (int j = 1; j < 8; ++j) vmax = fmaxf(vmax, f[j]);
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
        for (int w = 0; w < kWarps; ++w) r = ms_combine(r, sh[w]);
    }
    return r;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) logits_fwd_kernel(const T* __restrict__ logits,
                                                              int64_t ld,
                                                              const int64_t* __restrict__ targets,
                                                              int64_t V, float* __restrict__ logp,
                                                              float* __restrict__ lse_out,
                                                              int vec_ok) {
    __shared__ MS sh[kWarps];
    const int64_t row = blockIdx.x;
    const T* x = logits + row * ld;
    MS st = {-INFINITY, 0.f};
    int64_t done = 0;
    if (vec_ok) {
        const int64_t nvec = V / 8;
        int64_t i = threadIdx.x;
        for (; i + (kUnroll - 1) * kThreads < nvec; i += kUnroll * kThreads) {
            float f[kUnroll][8];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) load8(x + (i + u * kThreads) * 8, f[u]);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) ms_fold8(st, f[u]);
        }
        for (; i < nvec; i += kThreads) {
            float f[8];
            load8(x + i * 8, f);
            ms_fold8(st, f);
        }
        done = nvec * 8;
    }
    for (int64_t j = done + threadIdx.x; j < V; j += kThreads) ms_fold1(st, Elem<T>::to_f(x[j]));
    const MS r = block_reduce(st, sh);
    if (threadIdx.x == 0) {
        const float lse = (r.m == -INFINITY) ? -INFINITY : r.m * kLn2 + logf(r.s);
        const int64_t y = targets[row];
        const bool valid = (y >= 0) && (y < V);
        logp[row] = valid ? Elem<T>::to_f(x[y]) - lse : 0.f;
        lse_out[row] = lse;
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) logits_bwd_kernel(
    const float* __restrict__ grad, const T* __restrict__ logits, int64_t ld,
    const int64_t* __restrict__ targets, const float* __restrict__ lse, int64_t V,
    T* __restrict__ out, int vec_ok) {
    const int64_t row = blockIdx.x;
    const T* x = logits + row * ld;
    T* o = out + row * ld;
    const int64_t y = targets[row];
    const float g = grad[row];
    const bool live = (y >= 0) && (y < V) && (g != 0.f);
    const float lse2 = lse[row] * kLog2e;
    int64_t done = 0;
    if (vec_ok) {
        const int64_t nvec = V / 8;
        if (!live) {
            const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int64_t i = threadIdx.x; i < nvec; i += kThreads) store8(o + i * 8, z);
        } else {
            int64_t i = threadIdx.x;
            for (; i + (kUnroll - 1) * kThreads < nvec; i += kUnroll * kThreads) {
                float f[kUnroll][8];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) load8(x + (i + u * kThreads) * 8, f[u]);
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int64_t c0 = (i + u * kThreads) * 8;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float p = ex2(fmaf(f[u][j], kLog2e, -lse2));
                        const float oh = (c0 + j == y) ? 1.f : 0.f;
                        f[u][j] = fmaf(g, oh - p, 0.f);  // + 0 keeps empty results at +0
                    }
                    store8(o + c0, f[u]);
                }
            }
            for (; i < nvec; i += kThreads) {
                float f[8];
                const int64_t c0 = i * 8;
                load8(x + c0, f);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float p = ex2(fmaf(f[j], kLog2e, -lse2));
                    const float oh = (c0 + j == y) ? 1.f : 0.f;
                    f[j] = fmaf(g, oh - p, 0.f);
                }
                store8(o + c0, f);
            }
        }
        done = nvec * 8;
    }
    for (int64_t j = done + threadIdx.x; j < V; j += kThreads) {
        float v = 0.f;
        if (live) {
            const float p = ex2(fmaf(Elem<T>::to_f(x[j]), kLog2e, -lse2));
            v = fmaf(g, (j == y ? 1.f : 0.f) - p, 0.f);
        }
        o[j] = Elem<T>::from_f(v);
    }
}

template <typename T>
bool vec_ok(const void* p, int64_t ld) {
    return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((ld * int64_t(sizeof(T))) % 16 == 0);
}

}  // namespace

cudaError_t launch_logits_fwd(const void* logits, int64_t ld, int dtype, const int64_t* targets,
                              int64_t N, int64_t V, float* logp, float* lse, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(N));
    note_launches(1);
    switch (dtype) {
        case LL_BF16:
            logits_fwd_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(
                static_cast<const __nv_bfloat16*>(logits), ld, targets, V, logp, lse,
                vec_ok<__nv_bfloat16>(logits, ld));
            break;
        case LL_F16:
            logits_fwd_kernel<__half><<<grid, kThreads, 0, s>>>(
                static_cast<const __half*>(logits), ld, targets, V, logp, lse,
                vec_ok<__half>(logits, ld));
            break;
        default:
            logits_fwd_kernel<float><<<grid, kThreads, 0, s>>>(
                static_cast<const float*>(logits), ld, targets, V, logp, lse,
                vec_ok<float>(logits, ld));
    }
    return cudaGetLastError();
}

cudaError_t launch_logits_bwd(const float* grad, const void* logits, int64_t ld, int dtype,
                              const int64_t* targets, const float* lse, int64_t N, int64_t V,
                              void* grad_logits, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(N));
    note_launches(1);
    switch (dtype) {
        case LL_BF16: {
            const int ok = vec_ok<__nv_bfloat16>(logits, ld) && vec_ok<__nv_bfloat16>(grad_logits, ld);
            logits_bwd_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(
                grad, static_cast<const __nv_bfloat16*>(logits), ld, targets, lse, V,
                static_cast<__nv_bfloat16*>(grad_logits), ok);
            break;
        }
        case LL_F16: {
            const int ok = vec_ok<__half>(logits, ld) && vec_ok<__half>(grad_logits, ld);
            logits_bwd_kernel<__half><<<grid, kThreads, 0, s>>>(
                grad, static_cast<const __half*>(logits), ld, targets, lse, V,
                static_cast<__half*>(grad_logits), ok);
            break;
        }
        default: {
            const int ok = vec_ok<float>(logits, ld) && vec_ok<float>(grad_logits, ld);
            logits_bwd_kernel<float><<<grid, kThreads, 0, s>>>(
                grad, static_cast<const float*>(logits), ld, targets, lse, V,
                static_cast<float*>(grad_logits), ok);
        }
    }
    return cudaGetLastError();
}

}  // namespace ll
