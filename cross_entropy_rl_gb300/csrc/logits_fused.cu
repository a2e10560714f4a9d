// Logits-input logp forward and backward in one pass, for an upstream
// gradient known before the forward (the forward of RL-Kernel PR #495,
// "Summary", and its backward, fused): each row of logits is read from HBM
// once and its gradient written once, 4 V bytes per row instead of the
// 2 V (forward) + 4 V (backward) of the two kernels.
//
// A row does not fit in one SM's shared memory (151936 bf16 = 297 KB), so a
// thread-block cluster of C CTAs takes one row at a time: CTA j holds the
// contiguous slice j of the row (slice boundaries depend only on V and C),
// loaded by one bulk copy into a ring of shared-memory slice buffers (the
// next rows are prefetched while the current one is processed).  Each CTA
// folds its slice into a running (max, sum-exp) pair with a fixed reduction
// tree, the C pairs are combined in ascending rank order through distributed
// shared memory (every CTA computes the same lse), the gradient
// grad * (onehot - exp(z - lse)) overwrites the slice in place and one bulk
// copy writes it out.  The result of a row depends only on the row and V:
// deterministic and batch-invariant.
#include <math.h>

#include "ll_device.cuh"

namespace ll {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int kMaxBufs = 6;                   // slice buffers per CTA (ring)
constexpr size_t kSliceBudget = 200 * 1024;   // shared memory for the ring

struct FusedArgs {
    const void* logits;
    void* grad_out;
    int64_t ld, N, V, L;  // L: slice length in elements (multiple of 8)
    int nbuf;             // ring depth: rows in flight = nbuf - 2 loads + 2 stores
    const int64_t* targets;
    const float* grad;
    float* logp;
    float* lse;
    int* status;
    uint64_t wait_ns;
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}
// (m, s) pair stored at the same shared-memory offset in CTA `rank`
__device__ __forceinline__ float2 ld_peer_f2(const float2* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote)
                 : "r"(smem_u32(local)), "r"(rank));
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(remote)
                 : "memory");
    return v;
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// at most one bulk store (the latest) may still be reading shared memory
__device__ __forceinline__ void bulk_wait_read_but_one() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

struct MS {
    float m, s;
};
__device__ __forceinline__ MS combine(MS a, MS b) {
    const float M = fmaxf(a.m, b.m);
    if (M == -INFINITY) return {-INFINITY, 0.f};
    return {M, a.s * ex2(a.m - M) + b.s * ex2(b.m - M)};
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) logits_fused_kernel(const FusedArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int nbuf = a.nbuf;
    const size_t slice_bytes = size_t(a.L) * sizeof(T);
    uint8_t* tail = smem_raw + nbuf * slice_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(tail);                 // [kMaxBufs]
    float2* slot = reinterpret_cast<float2*>(tail + 8 * kMaxBufs);      // [2] (m, s) per parity
    MS* wred = reinterpret_cast<MS*>(tail + 8 * kMaxBufs + 16);         // [kWarps]
    float* lse_sh = reinterpret_cast<float*>(tail + 8 * kMaxBufs + 16 + kWarps * sizeof(MS));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const int64_t c0 = int64_t(rank) * a.L;  // this CTA's slice [c0, c1)
    const int64_t c1 = min(a.V, c0 + a.L);
    const int64_t len = c1 > c0 ? c1 - c0 : 0;
    const uint32_t bytes = static_cast<uint32_t>(len * sizeof(T));
    const int64_t nvec = len / 8;

    if (tid == 0) {
        for (int i = 0; i < nbuf; ++i) mbar_init(&full[i], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const T* X = static_cast<const T*>(a.logits);
    T* G = static_cast<T*>(a.grad_out);
    const int64_t first = cluster_id(), step = cluster_count();
    // rows of this cluster: first, first + step, ...; the ring keeps the
    // loads of the next nbuf - 2 rows in flight; a buffer is refilled two
    // rows after its store was issued, so only the latest store may still
    // be reading shared memory then
    const int ahead = nbuf - 2;
    auto buf_of = [&](int64_t kk) {
        return reinterpret_cast<T*>(smem_raw + (kk % nbuf) * slice_bytes);
    };
    bool ok = true;
    if (tid == 0 && len > 0) {
        for (int kk = 0; kk < ahead; ++kk) {
            const int64_t r = first + kk * step;
            if (r >= a.N) break;
            mbar_arrive_expect_tx(&full[kk], bytes);
            bulk_load(buf_of(kk), X + r * a.ld + c0, bytes, &full[kk]);
        }
    }
    int64_t k = 0;
    for (int64_t row = first; row < a.N; row += step, ++k) {
        const int bi = static_cast<int>(k % nbuf);
        const int b = static_cast<int>(k & 1);  // partial-slot parity
        const int64_t pre = row + ahead * step;
        if (tid == 0 && len > 0 && pre < a.N) {
            bulk_wait_read_but_one();  // the store of row k - 2 has read its buffer
            const int pb = static_cast<int>((k + ahead) % nbuf);
            mbar_arrive_expect_tx(&full[pb], bytes);
            bulk_load(buf_of(k + ahead), X + pre * a.ld + c0, bytes, &full[pb]);
        }
        if (len > 0 && !mbar_wait(&full[bi], static_cast<uint32_t>((k / nbuf) & 1), a.wait_ns,
                                  nullptr))
            ok = false;
        ok = __syncthreads_and(ok);
        const T* z = buf_of(k);
        // ---- this slice's (max, sum-exp), fixed assignment and tree
        MS st = {-INFINITY, 0.f};
        if (ok) {
            for (int64_t i = tid; i < nvec; i += kThreads) {
                float f[8];
                load8(z + i * 8, f);
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
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            MS other;
            other.m = __shfl_xor_sync(0xffffffffu, st.m, o);
            other.s = __shfl_xor_sync(0xffffffffu, st.s, o);
            st = combine(st, other);
        }
        const int64_t y = a.targets[row];
        const float g = a.grad[row];
        const bool valid = y >= 0 && y < a.V;
        const bool live = valid && g != 0.f;
        const bool mine = valid && y >= c0 && y < c1;
        float zy = 0.f;
        if (lane == 0) wred[warp] = st;
        if (tid == 0 && mine) zy = Elem<T>::to_f(z[y - c0]);  // before the slice is overwritten
        __syncthreads();
        if (tid == 0) {
            MS r = {-INFINITY, 0.f};
            for (int w = 0; w < kWarps; ++w) r = combine(r, wred[w]);
            slot[b] = make_float2(r.m, r.s);
        }
        cluster_sync();
        // ---- the row's lse from the C slices, in ascending rank order
        if (tid == 0) {
            MS tot = {-INFINITY, 0.f};
            for (uint32_t j = 0; j < C; ++j) {
                const float2 p = ld_peer_f2(&slot[b], j);
                tot = combine(tot, {p.x, p.y});
            }
            const float l = tot.m == -INFINITY ? -INFINITY : tot.m * kLn2 + logf(tot.s);
            *lse_sh = l;
            if (rank == 0) {
                a.lse[row] = l;
                if (!valid) a.logp[row] = 0.f;
            }
            if (mine) a.logp[row] = zy - l;
        }
        __syncthreads();
        const float lse = *lse_sh;
        // ---- gradient in place, then one bulk store of the slice
        const float lse2 = lse * kLog2e;
        T* zw = buf_of(k);
        if (ok) {
            for (int64_t i = tid; i < nvec; i += kThreads) {
                float f[8];
                load8(zw + i * 8, f);
                const int64_t cb = c0 + i * 8;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (live) {
                        const float p = ex2(fmaf(f[j], kLog2e, -lse2));
                        f[j] = fmaf(g, (cb + j == y ? 1.f : 0.f) - p, 0.f);
                    } else {
                        f[j] = 0.f;
                    }
                }
                store8(zw + i * 8, f);
            }
        }
        fence_proxy_async_shared_cta();
        __syncthreads();
        if (tid == 0 && len > 0 && ok) bulk_store(G + row * a.ld + c0, zw, bytes);
    }
    if (tid == 0) bulk_wait_all();
    if (!ok && tid == 0) set_status(a.status, LL_ERR_DEVICE_TIMEOUT);
    cluster_sync();  // no CTA leaves while a peer may still read its slots
}

}  // namespace

// Cluster size and ring depth for V: the smallest C in {2, 4, 8} whose
// slices fit at least 4 buffers in the shared-memory budget (else the
// deepest ring C = 8 allows, at least 2), or 0 when the kernel does not apply.
static int fused_cluster(int64_t V, size_t es, int64_t* L_out, int* nbuf_out) {
    int bestC = 0, bestN = 0;
    int64_t bestL = 0;
    for (int C = 2; C <= kMaxCluster; C <<= 1) {
        const int64_t L = (((V + C - 1) / C) + 7) / 8 * 8;
        int64_t n = static_cast<int64_t>((kSliceBudget - 1024) / (size_t(L) * es));
        if (n > kMaxBufs) n = kMaxBufs;
        if (n >= 4 || (C == kMaxCluster && n >= 2)) {
            bestC = C;
            bestN = static_cast<int>(n);
            bestL = L;
            break;
        }
    }
    *L_out = bestL;
    *nbuf_out = bestN;
    return bestC;
}

cudaError_t launch_logits_fused(const float* grad, const void* logits, int64_t ld, int dtype,
                                const int64_t* targets, int64_t N, int64_t V, float* logp,
                                float* lse, void* grad_logits, const DevInfo& dev,
                                cudaStream_t s, bool* used) {
    *used = false;
    const size_t es = dtype == LL_F32 ? 4 : 2;
    int64_t L = 0;
    int nbuf = 0;
    const int C = fused_cluster(V, es, &L, &nbuf);
    // bulk copies: 16-byte aligned rows; slices of whole 8-element vectors
    const bool aligned = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(grad_logits) % 16 == 0) &&
                         (ld * int64_t(es)) % 16 == 0 && V % 8 == 0;
    if (C == 0 || !aligned) return cudaSuccess;
    FusedArgs a;
    a.logits = logits;
    a.grad_out = grad_logits;
    a.ld = ld;
    a.N = N;
    a.V = V;
    a.L = L;
    a.nbuf = nbuf;
    a.targets = targets;
    a.grad = grad;
    a.logp = logp;
    a.lse = lse;
    a.status = dev.status;
    a.wait_ns = wait_limit_ns();
    const size_t smem = size_t(nbuf) * size_t(L) * es + 1024;
    void (*kern)(const FusedArgs) = dtype == LL_BF16  ? logits_fused_kernel<__nv_bfloat16>
                                    : dtype == LL_F16 ? logits_fused_kernel<__half>
                                                      : logits_fused_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(C * (dev.num_sms / C));
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess || clusters < 1) {
        cudaGetLastError();
        return cudaSuccess;  // no resident cluster of this size: two-kernel path
    }
    if (int64_t(clusters) > N) clusters = static_cast<int>(N);
    cfg.gridDim = dim3(static_cast<unsigned>(C * clusters));
    note_launches(1);
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e == cudaSuccess) *used = true;
    return e;
}

}  // namespace ll
