// FP32-operand GEMMs of the linear logp path on the CUDA cores (FFMA), with
// the same fused epilogues as the tensor-core path.
//
// Used when hidden / weight are FP32 (the small FP32 problem and the FP32
// row of the dtype sweep).  A 128 x 256 output tile is accumulated by 256
// threads (8 x 16 values each, sequential K, so every logit is the same
// FP32 dot product whatever the batch), staged in shared memory, and handed
// row by row to the epilogue in 32-column chunks.
#include "epilogue.cuh"

namespace ll {
namespace {

constexpr int kThreads = 256;
constexpr int kBKs = 16;
constexpr int kAld = kBM + 4;
constexpr int kBld = kBN + 4;
constexpr int kCld = kBN + 1;
constexpr int kSmemBytes = (kBKs * kAld + kBKs * kBld + kBM * kCld) * 4;

template <EpiKind E, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kThreads, 1)
    simt_gemm_kernel(const float* __restrict__ A, int64_t lda, const float* __restrict__ B,
                     int64_t ldb, int64_t M, int64_t N, int64_t K, const GemmShape sh,
                     const EpiArgs ea) {
    extern __shared__ float sm[];
    float* As = sm;
    float* Bs = As + kBKs * kAld;
    float* Cs = Bs + kBKs * kBld;
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int64_t n_units = sh.m_blocks * sh.n_segs;
    RowEpilogue<E, float> epi;
    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
        int64_t mb, seg;
        if (sh.unit_order == 0) {
            seg = u / sh.m_blocks;
            mb = u % sh.m_blocks;
        } else if (sh.unit_order == 1) {
            mb = u / sh.n_segs;
            seg = u % sh.n_segs;
        } else {
            const int64_t per_group = kGroupM * sh.n_segs;
            const int64_t g = u / per_group;
            const int64_t in_g = u % per_group;
            const int64_t gm = min(kGroupM, sh.m_blocks - g * kGroupM);
            seg = in_g / gm;
            mb = g * kGroupM + in_g % gm;
        }
        const int64_t t0 = seg * sh.tiles_per_unit;
        const int64_t t1 = min(t0 + sh.tiles_per_unit, sh.n_tiles);
        if (tid < kBM) epi.begin_unit(ea, mb * kBM + tid);
        for (int64_t t = t0; t < t1; ++t) {
            float acc[8][16];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[i][j] = 0.f;
            for (int64_t k0 = 0; k0 < K; k0 += kBKs) {
                __syncthreads();
                for (int e = tid; e < kBM * kBKs; e += kThreads) {
                    const int m = A_MN ? e % kBM : e / kBKs;
                    const int k = A_MN ? e / kBM : e % kBKs;
                    const int64_t gm = mb * kBM + m, gk = k0 + k;
                    float v = 0.f;
                    if (gm < M && gk < K) v = A_MN ? A[gk * lda + gm] : A[gm * lda + gk];
                    As[k * kAld + m] = v;
                }
                for (int e = tid; e < kBN * kBKs; e += kThreads) {
                    const int n = B_MN ? e % kBN : e / kBKs;
                    const int k = B_MN ? e / kBN : e % kBKs;
                    const int64_t gn = t * kBN + n, gk = k0 + k;
                    float v = 0.f;
                    if (gn < N && gk < K) v = B_MN ? B[gk * ldb + gn] : B[gn * ldb + gk];
                    Bs[k * kBld + n] = v;
                }
                __syncthreads();
#pragma unroll 4
                for (int k = 0; k < kBKs; ++k) {
                    float a[8], b[16];
#pragma unroll
                    for (int i = 0; i < 8; ++i) a[i] = As[k * kAld + ty + 16 * i];
#pragma unroll
                    for (int j = 0; j < 16; ++j) b[j] = Bs[k * kBld + tx + 16 * j];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                }
            }
            __syncthreads();
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 16; ++j) Cs[(ty + 16 * i) * kCld + tx + 16 * j] = acc[i][j];
            __syncthreads();
            if (tid < kBM) {
#pragma unroll 1
                for (int c = 0; c < kBN / 32; ++c) {
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = Cs[tid * kCld + c * 32 + j];
                    epi.chunk(ea, v, t * kBN + c * 32);
                    epi.store_direct(ea, v, t * kBN + c * 32);
                    epi.db_partials(ea, v, t * kBN + c * 32);
                }
            }
        }
        if (tid < kBM) epi.end_unit(ea, seg);
    }
}

template <EpiKind E, bool A_MN, bool B_MN>
cudaError_t launch_simt(const float* A, int64_t lda, const float* B, int64_t ldb, int64_t M,
                        int64_t N, int64_t K, const GemmShape& sh, const EpiArgs& ea,
                        const DevInfo& dev, int max_ctas, cudaStream_t s) {
    auto kern = simt_gemm_kernel<E, A_MN, B_MN>;
    static int configured[64] = {0};
    if (dev.device < 64 && !configured[dev.device]) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        configured[dev.device] = 1;
    }
    const int64_t units = sh.m_blocks * sh.n_segs;
    const int cap = (max_ctas > 0 && max_ctas < dev.num_sms) ? max_ctas : dev.num_sms;
    const int grid = static_cast<int>(units < cap ? units : cap);
    note_launches(1);
    kern<<<grid, kThreads, kSmemBytes, s>>>(A, lda, B, ldb, M, N, K, sh, ea);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_f32(EpiKind kind, const void* A, int64_t lda, int a_mn, const void* B,
                            int64_t ldb, int b_mn, int64_t M, int64_t N, int64_t K,
                            const GemmShape& sh, const EpiArgs& ea, const DevInfo& dev,
                            int max_ctas, cudaStream_t s) {
    const float* a = static_cast<const float*>(A);
    const float* b = static_cast<const float*>(B);
    switch (kind) {
        case EpiKind::Fwd:
            return launch_simt<EpiKind::Fwd, false, false>(a, lda, b, ldb, M, N, K, sh, ea, dev, max_ctas, s);
        case EpiKind::Recomp:
            return launch_simt<EpiKind::Recomp, false, false>(a, lda, b, ldb, M, N, K, sh, ea, dev,
                                                              max_ctas, s);
        case EpiKind::Dh:
            return launch_simt<EpiKind::Dh, false, true>(a, lda, b, ldb, M, N, K, sh, ea, dev, max_ctas, s);
        case EpiKind::Dw:
            return launch_simt<EpiKind::Dw, true, true>(a, lda, b, ldb, M, N, K, sh, ea, dev, max_ctas, s);
    }
    (void)a_mn;
    (void)b_mn;
    return cudaErrorInvalidValue;
}

}  // namespace ll
