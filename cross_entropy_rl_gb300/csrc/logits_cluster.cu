// Logits-input logp forward and backward in one pass, rows held on chip
// (a known upstream gradient: the forward of RL-Kernel PR #495, "Summary",
// and its backward, fused).  Each row of logits is read from HBM once and its
// gradient written once, 4 V bytes per row, whatever L2 holds.
//
// A row does not fit in one SM (151936 bf16 = 297 KB), so a thread-block
// cluster of C CTAs takes one row at a time: CTA j copies the contiguous
// slice j of the row (slice boundaries depend only on V and C) into one of
// two shared-memory buffers with cp.async from all its threads, the next
// row's slice loading into the other buffer meanwhile.  The CTA folds its
// slice into a (max, sum-exp) pair with a fixed reduction tree and pushes
// the pair into a slot of every CTA of the cluster (st.async into
// distributed shared memory, counted by a transaction mbarrier per slot);
// each CTA combines the C pairs in ascending rank order (all compute the
// same lse) and writes its slice's gradient grad * (onehot - exp(z - lse))
// straight from registers.  The result of a row depends only on the row, V
// and the dtype: deterministic and batch-invariant.
#include <math.h>

#include "ll_device.cuh"

namespace ll {
namespace {

constexpr int kCT = 512;                    // threads per CTA
constexpr int kCW = kCT / 32;
constexpr int kCSlots = 4;                  // exchange slots (rows in flight)
constexpr int kCMaxCluster = 8;
constexpr size_t kCBudget = 208 * 1024;     // two slice buffers + the tail

struct MSc {
    float m, s;  // max (log2 domain) and the sum of 2^(x - m)
};

struct CTail {
    uint64_t xch[kCSlots];                // all C pairs of a row arrived
    float2 slot[kCSlots][kCMaxCluster];   // pair of row k from CTA j: slot[k % kCSlots][j]
    MSc wred[kCW];
    float lse;
};

struct ClusterArgs {
    const void* logits;
    void* grad_out;
    int64_t ld, N, V, L;  // L: slice length in elements (multiple of 8)
    const int64_t* targets;
    const float* grad;
    float* logp;
    float* lse;
    float it;  // 1 / temperature
    int* status;
    uint64_t wait_ns;
};

__device__ __forceinline__ uint32_t cl_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// 8-byte store into a CTA's shared memory, counted on that CTA's mbarrier
__device__ __forceinline__ void st_async_f2(uint32_t remote, float x, float y,
                                            uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
            remote),
        "f"(x), "f"(y), "r"(remote_bar)
        : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// every group but the latest one has landed (this thread's copies)
__device__ __forceinline__ void cp_async_wait_but_one() {
    asm volatile("cp.async.wait_group 1;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ MSc combine(MSc a, MSc b) {
    const float M = fmaxf(a.m, b.m);
    if (M == -INFINITY) return {-INFINITY, 0.f};
    return {M, a.s * ex2(a.m - M) + b.s * ex2(b.m - M)};
}
__device__ __forceinline__ MSc shfl_xor(MSc v, int o) {
    return {__shfl_xor_sync(0xffffffffu, v.m, o), __shfl_xor_sync(0xffffffffu, v.s, o)};
}

template <typename T>
__global__ void __launch_bounds__(kCT, 1) logits_cluster_kernel(const ClusterArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const uint32_t C = cl_size();
    const uint32_t rank = cl_rank();
    const size_t slice_bytes = size_t(a.L) * sizeof(T);
    T* buf[2] = {reinterpret_cast<T*>(smem_raw), reinterpret_cast<T*>(smem_raw + slice_bytes)};
    CTail* t = reinterpret_cast<CTail*>(smem_raw + 2 * slice_bytes);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float it = a.it;

    const int64_t c0 = int64_t(rank) * a.L;  // this CTA's slice [c0, c1)
    const int64_t c1 = min(a.V, c0 + a.L);
    const int64_t len = c1 > c0 ? c1 - c0 : 0;
    const int64_t nvec = len / 8;                                   // 8-element vectors
    const int64_t nchunk = len * int64_t(sizeof(T)) / 16;           // 16-byte copies

    if (tid == 0) {
        for (int i = 0; i < kCSlots; ++i) mbar_init(&t->xch[i], 1);
        fence_mbar_init();
    }
    cluster_barrier();  // every CTA's barriers exist before a peer stores to them

    const char* X = static_cast<const char*>(a.logits);
    T* G = static_cast<T*>(a.grad_out);
    const int64_t first = cl_id(), step = cl_count();
    const int64_t K = first < a.N ? (a.N - 1 - first) / step + 1 : 0;  // rows of this cluster
    const int64_t row_bytes = a.ld * int64_t(sizeof(T));
    const uint64_t drop = l2_evict_first();

    auto load = [&](int64_t k) {  // slice of this cluster's row k into buf[k & 1]
        if (k < K) {
            const char* src = X + (first + k * step) * row_bytes + c0 * int64_t(sizeof(T));
            char* dst = reinterpret_cast<char*>(buf[k & 1]);
            for (int64_t i = tid; i < nchunk; i += kCT) cp_async16(dst + i * 16, src + i * 16);
        }
        cp_async_commit();  // one group per row, empty past the last
    };

    bool ok = true;
    load(0);
    for (int64_t k = 0; k < K; ++k) {
        const int64_t row = first + k * step;
        load(k + 1);
        cp_async_wait_but_one();  // row k's copies (this thread's)
        __syncthreads();          // everyone's
        const T* z = buf[k & 1];
        const int64_t y = a.targets[row];
        const float g = a.grad[row];
        const bool valid = y >= 0 && y < a.V;
        const bool live = valid && g != 0.f;
        const bool mine = valid && y >= c0 && y < c1;

        // ---- this slice's (max, sum-exp): thread tid folds vectors tid, tid + kCT, ...
        MSc st = {-INFINITY, 0.f};
        for (int64_t i = tid; i < nvec; i += kCT) {
            float f[8];
            load8(z + i * 8, f);
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] *= it;
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
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) st = combine(st, shfl_xor(st, o));
        if (lane == 0) t->wred[warp] = st;
        __syncthreads();

        // ---- warp 0: push the slice's pair to every CTA, then the row's lse
        if (warp == 0) {
            MSc p = lane < kCW ? t->wred[lane] : MSc{-INFINITY, 0.f};
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) p = combine(p, shfl_xor(p, o));
            const int si = static_cast<int>(k % kCSlots);
            if (lane < static_cast<int>(C))
                st_async_f2(cluster_addr(&t->slot[si][rank], lane), p.m, p.s,
                            cluster_addr(&t->xch[si], lane));
            if (lane == 0) mbar_arrive_expect_tx(&t->xch[si], C * 8u);
            bool got = mbar_wait(&t->xch[si], static_cast<uint32_t>((k / kCSlots) & 1),
                                 a.wait_ns, nullptr);
            got = __all_sync(0xffffffffu, got);
            float2 q = make_float2(-INFINITY, 0.f);
            if (lane < static_cast<int>(C)) q = t->slot[si][lane];
            MSc tot = {-INFINITY, 0.f};
            for (uint32_t j = 0; j < C; ++j)
                tot = combine(tot, {__shfl_sync(0xffffffffu, q.x, j),
                                    __shfl_sync(0xffffffffu, q.y, j)});
            if (lane == 0) {
                const float l = tot.m == -INFINITY ? -INFINITY : tot.m * kLn2 + logf(tot.s);
                t->lse = l;
                if (rank == 0) {
                    a.lse[row] = l;
                    if (!valid) a.logp[row] = 0.f;
                }
                if (mine) a.logp[row] = Elem<T>::to_f(z[y - c0]) * it - l;
            }
            ok = got;
        }
        ok = __syncthreads_and(ok);
        if (!ok) break;

        // ---- the gradient of the slice, from the buffer to global memory
        const float lse2 = t->lse * kLog2e;
        const float gi = g * it;
        T* o = G + row * a.ld + c0;
        for (int64_t i = tid; i < nvec; i += kCT) {
            float f[8];
            load8(z + i * 8, f);
            const int64_t cb = c0 + i * 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (live) {
                    const float pj = ex2(fmaf(f[j] * it, kLog2e, -lse2));
                    f[j] = fmaf(gi, (cb + j == y ? 1.f : 0.f) - pj, 0.f);
                } else {
                    f[j] = 0.f;
                }
            }
            store8_hint(o + i * 8, f, drop);
        }
        __syncthreads();  // buf[k & 1] is refilled by the next iteration's load
    }
    cp_async_wait_all();
    if (!ok && tid == 0) set_status(a.status, LL_ERR_DEVICE_TIMEOUT);
    cluster_barrier();  // no CTA leaves while a peer may still store to its slots
}

// Cluster size for V: the smallest C in {1, 2, 4, 8} whose two slice buffers
// fit the shared-memory budget; L = the slice length.  0 if none.
int cluster_for(int64_t V, size_t es, int64_t* L_out) {
    for (int C = 1; C <= kCMaxCluster; C <<= 1) {
        const int64_t L = (((V + C - 1) / C) + 7) / 8 * 8;
        if (2 * size_t(L) * es + sizeof(CTail) + 128 <= kCBudget) {
            *L_out = L;
            return C;
        }
    }
    return 0;
}

}  // namespace

cudaError_t launch_logits_cluster(const float* grad, const void* logits, int64_t ld, int dtype,
                                  const int64_t* targets, int64_t N, int64_t V, float* logp,
                                  float* lse, void* grad_logits, float it, const DevInfo& dev,
                                  cudaStream_t s, bool* used) {
    *used = false;
    const size_t es = dtype == LL_F32 ? 4 : 2;
    // whole 16-byte vectors in every slice and row
    const bool aligned = reinterpret_cast<uintptr_t>(logits) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(grad_logits) % 16 == 0 &&
                         (ld * int64_t(es)) % 16 == 0 && V % 8 == 0;
    int64_t L = 0;
    const int C = aligned ? cluster_for(V, es, &L) : 0;
    if (C == 0) return cudaSuccess;
    ClusterArgs a;
    a.logits = logits;
    a.grad_out = grad_logits;
    a.ld = ld;
    a.N = N;
    a.V = V;
    a.L = L;
    a.targets = targets;
    a.grad = grad;
    a.logp = logp;
    a.lse = lse;
    a.it = it;
    a.status = dev.status;
    a.wait_ns = wait_limit_ns();
    const size_t smem = 2 * size_t(L) * es + sizeof(CTail) + 128;
    void (*kern)(const ClusterArgs) = dtype == LL_BF16  ? logits_cluster_kernel<__nv_bfloat16>
                                      : dtype == LL_F16 ? logits_cluster_kernel<__half>
                                                        : logits_cluster_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kCT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(C * (dev.num_sms / C));
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess || clusters < 1) {
        cudaGetLastError();
        return cudaSuccess;  // no resident cluster of this size
    }
    if (int64_t(clusters) > N) clusters = static_cast<int>(N);
    cfg.gridDim = dim3(static_cast<unsigned>(C * clusters));
    note_launches(1);
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e == cudaSuccess) *used = true;
    return e;
}

}  // namespace ll
