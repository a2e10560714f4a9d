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
// folds its slice into a (max, sum-exp) pair with a fixed reduction tree and
// pushes the pair into a slot of every CTA of the cluster (st.async into
// distributed shared memory, counted by a transaction mbarrier per slot);
// each CTA then combines the C pairs in ascending rank order (all compute the
// same lse), overwrites its slice with grad * (onehot - exp(z - lse)) and
// bulk-copies it out.  The CTAs never meet at a cluster barrier inside the
// loop: a CTA pushes the pair of row k + 1 before it needs the pairs of
// row k, so the exchange is off the critical path.  The result of a row
// depends only on the row and V: deterministic and batch-invariant.
#include <math.h>

#include "ll_device.cuh"

namespace ll {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 16;
constexpr int kMaxBufs = 8;                   // slice buffers per CTA (ring)
constexpr int kSlots = 4;                     // exchange slots (rows in flight)
constexpr size_t kSliceBudget = 208 * 1024;   // shared memory for the ring

struct FusedArgs {
    const void* logits;
    void* grad_out;
    int64_t ld, N, V, L;  // L: slice length in elements (multiple of 8)
    int nbuf;             // ring depth: nbuf - 3 rows loaded ahead
    const int64_t* targets;
    const float* grad;
    float* logp;
    float* lse;
    int* status;
    uint64_t wait_ns;
};

struct MS {
    float m, s;  // running max (log2 domain) and the sum of 2^(x - m)
};

// Shared memory after the slice ring.
struct Tail {
    uint64_t full[kMaxBufs];             // slice loaded (transaction bytes)
    uint64_t xch[kSlots];                // all C pairs of a row arrived
    float2 slot[kSlots][kMaxCluster];    // pair of row k from CTA j: slot[k % kSlots][j]
    MS wred[kWarps];                     // per-warp partials of the slice
    float lse;                           // lse of the row being finished
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
// shared::cluster address of `local`'s counterpart in CTA `rank`
__device__ __forceinline__ uint32_t peer_addr(const void* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote)
                 : "r"(smem_u32(local)), "r"(rank));
    return remote;
}
// 8-byte store into a peer's shared memory, counted on the peer's mbarrier
__device__ __forceinline__ void st_async_f2(uint32_t remote, float x, float y,
                                            uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
            remote),
        "f"(x), "f"(y), "r"(remote_bar)
        : "memory");
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

__device__ __forceinline__ MS combine(MS a, MS b) {
    const float M = fmaxf(a.m, b.m);
    if (M == -INFINITY) return {-INFINITY, 0.f};
    return {M, a.s * ex2(a.m - M) + b.s * ex2(b.m - M)};
}
__device__ __forceinline__ MS shfl_xor(MS v, int o) {
    return {__shfl_xor_sync(0xffffffffu, v.m, o), __shfl_xor_sync(0xffffffffu, v.s, o)};
}

// (max, sum-exp) of this thread's share of a slice, folded across the warp
// (the butterfly leaves the same pair in every lane: combine is symmetric).
template <typename T>
__device__ __forceinline__ MS slice_partial(const T* z, int64_t nvec, int tid) {
    MS st = {-INFINITY, 0.f};
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
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) st = combine(st, shfl_xor(st, o));
    return st;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) logits_fused_kernel(const FusedArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int nbuf = a.nbuf;
    const int ahead = nbuf - 3;  // rows loaded beyond the two being worked on
    const size_t slice_bytes = size_t(a.L) * sizeof(T);
    Tail* t = reinterpret_cast<Tail*>(smem_raw + nbuf * slice_bytes);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const int64_t c0 = int64_t(rank) * a.L;  // this CTA's slice [c0, c1)
    const int64_t c1 = min(a.V, c0 + a.L);
    const int64_t len = c1 > c0 ? c1 - c0 : 0;
    const uint32_t bytes = static_cast<uint32_t>(len * sizeof(T));
    const int64_t nvec = len / 8;

    if (tid == 0) {
        for (int i = 0; i < nbuf; ++i) mbar_init(&t->full[i], 1);
        for (int i = 0; i < kSlots; ++i) mbar_init(&t->xch[i], 1);
        fence_mbar_init();
    }
    cluster_sync();  // every CTA's barriers exist before a peer stores to them

    const T* X = static_cast<const T*>(a.logits);
    T* G = static_cast<T*>(a.grad_out);
    const int64_t first = cluster_id(), step = cluster_count();
    const int64_t K = first < a.N ? (a.N - 1 - first) / step + 1 : 0;  // rows of this cluster
    int64_t issued = 0;    // tid 0: loads issued for rows [0, issued)
    int64_t consumed = 0;  // loads of rows [0, consumed) seen complete by this thread
    auto buf_of = [&](int64_t k) {
        return reinterpret_cast<T*>(smem_raw + (k % nbuf) * slice_bytes);
    };
    auto issue_load = [&](int64_t k) {  // tid 0 only
        if (k >= K || len == 0) return;
        issued = k + 1;
        uint64_t* bar = &t->full[k % nbuf];
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load(buf_of(k), X + (first + k * step) * a.ld + c0, bytes, bar);
    };
    auto wait_load = [&](int64_t k) {
        return len == 0 ||
               mbar_wait(&t->full[k % nbuf], static_cast<uint32_t>((k / nbuf) & 1), a.wait_ns,
                         nullptr);
    };
    // warp 0 after the block's per-warp partials are in t->wred: fold them
    // and push the slice's pair of row k to every CTA (lane j -> CTA j)
    auto push_pair = [&](int64_t k) {
        MS p = lane < kWarps ? t->wred[lane] : MS{-INFINITY, 0.f};
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) p = combine(p, shfl_xor(p, o));
        if (lane < static_cast<int>(C)) {
            const int si = static_cast<int>(k % kSlots);
            st_async_f2(peer_addr(&t->slot[si][rank], lane), p.m, p.s,
                        peer_addr(&t->xch[si], lane));
        }
    };

    bool ok = true;
    if (tid == 0)
        for (int64_t k = 0; k <= ahead; ++k) issue_load(k);
    if (K > 0) {
        ok = wait_load(0);
        consumed = ok ? 1 : 0;
        const MS st = slice_partial(buf_of(0), ok ? nvec : 0, tid);
        if (lane == 0) t->wred[warp] = st;
        ok = __syncthreads_and(ok);
        if (warp == 0 && ok) push_pair(0);
        __syncthreads();  // t->wred is rewritten by the first iteration
    }
    for (int64_t k = 0; k < K && ok; ++k) {
        const int64_t row = first + k * step;
        const int64_t y = a.targets[row];
        const float g = a.grad[row];
        const bool valid = y >= 0 && y < a.V;
        const bool live = valid && g != 0.f;
        const bool mine = valid && y >= c0 && y < c1;
        if (tid == 0) {
            // the buffer of row k + 1 + ahead last held row k - 2, whose
            // store is not the latest one issued
            bulk_wait_read_but_one();
            issue_load(k + 1 + ahead);
        }
        // ---- warp 0: the row's lse from the C pairs, in ascending rank order
        if (warp == 0) {
            const int si = static_cast<int>(k % kSlots);
            if (lane == 0) mbar_arrive_expect_tx(&t->xch[si], C * 8u);
            bool got = mbar_wait(&t->xch[si], static_cast<uint32_t>((k / kSlots) & 1),
                                 a.wait_ns, nullptr);
            got = __all_sync(0xffffffffu, got);
            float2 q = make_float2(-INFINITY, 0.f);
            if (lane < static_cast<int>(C)) q = t->slot[si][lane];
            MS tot = {-INFINITY, 0.f};
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
                if (mine) a.logp[row] = Elem<T>::to_f(buf_of(k)[y - c0]) - l;
            }
            ok = got;
        }
        // ---- the next row's partial while the pairs of this one settle
        if (k + 1 < K) {
            const bool loaded = wait_load(k + 1);
            if (loaded) consumed = k + 2;
            const MS st = slice_partial(buf_of(k + 1), loaded ? nvec : 0, tid);
            if (lane == 0) t->wred[warp] = st;
            ok = ok && loaded;
        }
        ok = __syncthreads_and(ok);
        if (!ok) break;
        if (warp == 0 && k + 1 < K) push_pair(k + 1);
        // ---- gradient in place, then one bulk store of the slice
        const float lse2 = t->lse * kLog2e;
        T* zw = buf_of(k);
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
        fence_proxy_async_shared_cta();
        __syncthreads();
        if (tid == 0 && len > 0) bulk_store(G + row * a.ld + c0, zw, bytes);
    }
    if (tid == 0) {
        bulk_wait_all();
        if (!ok) {
            set_status(a.status, LL_ERR_DEVICE_TIMEOUT);
            // loads still in flight into this CTA's ring: wait for them (bounded)
            for (int64_t r = consumed; r < issued; ++r)
                mbar_wait(&t->full[r % nbuf], static_cast<uint32_t>((r / nbuf) & 1), a.wait_ns,
                          nullptr);
        }
    }
    cluster_sync();  // no CTA leaves while a peer may still store to its slots
}

}  // namespace

// Cluster size and ring depth for V: the smallest C in {2, 4, 8, 16} whose
// slices fit at least 5 buffers (2 rows being worked on, 2 loaded ahead, one
// store draining) in the shared-memory budget, else the first C that fits 4;
// 0 when the kernel does not apply.
static int fused_cluster(int64_t V, size_t es, int64_t* L_out, int* nbuf_out) {
    int bestC = 0, bestN = 0;
    int64_t bestL = 0;
    for (int want = 5; want >= 4 && bestC == 0; --want) {
        for (int C = 2; C <= kMaxCluster; C <<= 1) {
            const int64_t L = (((V + C - 1) / C) + 7) / 8 * 8;
            int64_t n = static_cast<int64_t>((kSliceBudget - 1024) / (size_t(L) * es));
            if (n > kMaxBufs) n = kMaxBufs;
            if (n >= want) {
                bestC = C;
                bestN = static_cast<int>(n);
                bestL = L;
                break;
            }
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
    static_assert(sizeof(Tail) <= 1024, "tail of the shared-memory ring");
    const size_t smem = size_t(nbuf) * size_t(L) * es + 1024;
    void (*kern)(const FusedArgs) = dtype == LL_BF16  ? logits_fused_kernel<__nv_bfloat16>
                                    : dtype == LL_F16 ? logits_fused_kernel<__half>
                                                      : logits_fused_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (C > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return cudaSuccess;  // two-kernel path
        }
    }
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
