// Tensor-core GEMM with fused epilogues for the 16-bit operand paths
// (bf16 / fp16 operands, FP32 accumulation in TMEM).
//
// The three contractions of the fused linear logp (RL-Kernel issue #261,
// "Current accumulation": the chunked matmul and its accumulation into an
// FP32 gradient table; Liger-Kernel PR #1324, "Details": no [V, H]
// temporary) run here:
//   forward / recompute   z  = h . W^T        A = h [rows, D]  (K-major)
//                                              B = W [V, D]     (K-major)
//   grad_hidden           dh = S . W          A = S [rows, V]  (K-major)
//                                              B = W [V, D]     (MN-major)
//   grad_weight           dW += S^T . h       A = S [rows, V]  (MN-major)
//                                              B = h [rows, D]  (MN-major)
//
// Design (sm_103a): one persistent CTA per SM, 6 warps.
//   warp 0      TMA producer: 128-byte-swizzled tiles into a 4-stage ring
//   warp 1      allocates 512 TMEM columns, issues tcgen05.mma (128x256x16)
//   warps 2..5  epilogue: tcgen05.ld of its 32 TMEM lanes, fused epilogue
// Two 256-column accumulators in TMEM let the epilogue of one tile overlap
// the MMAs of the next.  Work units are walked in a static round-robin order
// so that the result never depends on scheduling.
#include <mutex>
#include <type_traits>

#include "epilogue.cuh"

namespace ll {
namespace {

constexpr int kBK = 64;  // K elements per stage (128 bytes of 16-bit values)
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kBN * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kMnBoxBytes = 64 * kBK * 2;  // one 64(MN) x 64(K) box, 8 KB
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;

struct Bars {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void decode_unit(const GemmShape& sh, int64_t u, int64_t& mb,
                                            int64_t& seg) {
    if (sh.unit_order == 0) {
        seg = u / sh.m_blocks;
        mb = u % sh.m_blocks;
    } else {
        mb = u / sh.n_segs;
        seg = u % sh.n_segs;
    }
}

template <EpiKind E, typename T, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const GemmShape sh,
                   const EpiArgs ea) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars* bars = reinterpret_cast<Bars*>(smem + kStages * kStageBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t n_units = sh.m_blocks * sh.n_segs;
    volatile int* abort = &bars->abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->tfull[b], 1);
            mbar_init(&bars->tempty[b], 4);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_phase[kStages];
        bool issued[kStages];
        for (int s = 0; s < kStages; ++s) issued[s] = false;
        bool ok = true;
        for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            int64_t mb, seg;
            decode_unit(sh, u, mb, seg);
            const int64_t t0 = seg * sh.tiles_per_unit;
            const int64_t t1 = min(t0 + sh.tiles_per_unit, sh.n_tiles);
            for (int64_t t = t0; t < t1 && ok; ++t) {
                for (int64_t kb = 0; kb < sh.k_blocks; ++kb) {
                    if (!__all_sync(0xffffffffu, mbar_wait(&bars->empty[stage], phase ^ 1, ea.wait_ns, abort))) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        uint64_t* fb = &bars->full[stage];
                        uint8_t* sa = smem + stage * kStageBytes;
                        uint8_t* sb = sa + kABytes;
                        mbar_arrive_expect_tx(fb, kStageBytes);
                        const int32_t k0 = static_cast<int32_t>(kb * kBK);
                        const int32_t m0 = static_cast<int32_t>(mb * kBM);
                        const int32_t n0 = static_cast<int32_t>(t * kBN);
                        if constexpr (!A_MN) {
                            tma_load_2d(sa, &tmA, fb, k0, m0);
                        } else {
#pragma unroll
                            for (int j = 0; j < kBM / 64; ++j)
                                tma_load_2d(sa + j * kMnBoxBytes, &tmA, fb, m0 + 64 * j, k0);
                        }
                        if constexpr (!B_MN) {
                            tma_load_2d(sb, &tmB, fb, k0, n0);
                        } else {
#pragma unroll
                            for (int j = 0; j < kBN / 64; ++j)
                                tma_load_2d(sb + j * kMnBoxBytes, &tmB, fb, n0 + 64 * j, k0);
                        }
                    }
                    __syncwarp();
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
        if (!ok) {
            if (lane == 0) set_status(ea.status, LL_ERR_DEVICE_TIMEOUT);
            bars->abort = 1;
            // let every issued copy land before the CTA may exit
            for (int s = 0; s < kStages; ++s)
                if (issued[s]) mbar_wait(&bars->full[s], issued_phase[s], ea.wait_ns, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        constexpr int fmt = std::is_same<T, __half>::value ? 0 : 1;
        constexpr uint32_t idesc = instr_desc(fmt, A_MN, B_MN, kBM, kBN);
        int stage = 0;
        uint32_t phase = 0;
        int buf = 0;
        uint32_t bphase = 0;
        bool ok = true;
        const uint32_t sbase = smem_u32(smem);
        for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            int64_t mb, seg;
            decode_unit(sh, u, mb, seg);
            const int64_t t0 = seg * sh.tiles_per_unit;
            const int64_t t1 = min(t0 + sh.tiles_per_unit, sh.n_tiles);
            for (int64_t t = t0; t < t1 && ok; ++t) {
                if (!__all_sync(0xffffffffu, mbar_wait(&bars->tempty[buf], bphase ^ 1, ea.wait_ns, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + buf * kBN;
                for (int64_t kb = 0; kb < sh.k_blocks; ++kb) {
                    if (!__all_sync(0xffffffffu, mbar_wait(&bars->full[stage], phase, ea.wait_ns, abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t sa = sbase + stage * kStageBytes;
                        const uint32_t sb = sa + kABytes;
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            const uint64_t ad =
                                A_MN ? smem_desc_sw128(sa + kk * 2048, kMnBoxBytes, 1024)
                                     : smem_desc_sw128(sa + kk * 32, 16, 1024);
                            const uint64_t bd =
                                B_MN ? smem_desc_sw128(sb + kk * 2048, kMnBoxBytes, 1024)
                                     : smem_desc_sw128(sb + kk * 32, 16, 1024);
                            tc_mma<0>(d_tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc_commit(&bars->empty[stage]);
                    }
                    __syncwarp();
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if (lane == 0) tc_commit(&bars->tfull[buf]);
                __syncwarp();
                if (++buf == 2) {
                    buf = 0;
                    bphase ^= 1;
                }
            }
        }
        if (!ok) {
            if (lane == 0) set_status(ea.status, LL_ERR_DEVICE_TIMEOUT);
            bars->abort = 1;
        }
        // every MMA issued by this warp completes before TMEM is released
        if (lane == 0) tc_commit(&bars->drain);
        __syncwarp();
        mbar_wait(&bars->drain, 0, ea.wait_ns, nullptr);
    } else {
        // ------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lanes [32q, 32q + 32)
        const int r_in_tile = q * 32 + lane;
        int buf = 0;
        uint32_t bphase = 0;
        bool ok = true;
        RowEpilogue<E, T> epi;
        for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            int64_t mb, seg;
            decode_unit(sh, u, mb, seg);
            const int64_t t0 = seg * sh.tiles_per_unit;
            const int64_t t1 = min(t0 + sh.tiles_per_unit, sh.n_tiles);
            epi.begin_unit(ea, mb * kBM + r_in_tile);
            for (int64_t t = t0; t < t1; ++t) {
                if (!__all_sync(0xffffffffu, mbar_wait(&bars->tfull[buf], bphase, ea.wait_ns, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem + buf * kBN + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
                for (int c = 0; c < kBN / 32; ++c) {
                    uint32_t r[32];
                    __syncwarp();  // tcgen05.ld is warp-collective (.sync.aligned)
                    tmem_ld32(taddr + c * 32, r);
                    tmem_ld_wait(r);
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    epi.chunk(ea, v, t * kBN + c * 32);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->tempty[buf]);
                if (++buf == 2) {
                    buf = 0;
                    bphase ^= 1;
                }
            }
            if (!ok) break;
            epi.end_unit(ea, seg);
        }
        if (!ok) {
            if (lane == 0) set_status(ea.status, LL_ERR_DEVICE_TIMEOUT);
            bars->abort = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D map over a row-major [rows, cols] matrix with row stride `ld`
// elements; box = box_cols x box_rows, 128-byte swizzle, zero fill.
bool make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int esize,
              int64_t cols, int64_t rows, int64_t ld, int box_cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols),
                               static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <EpiKind E, typename T, bool A_MN, bool B_MN>
cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b, const GemmShape& sh,
                       const EpiArgs& ea, const DevInfo& dev, cudaStream_t s) {
    auto kern = gemm_tc_kernel<E, T, A_MN, B_MN>;
    static int configured[64] = {0};
    if (dev.device < 64 && !configured[dev.device]) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        configured[dev.device] = 1;
    }
    const int64_t units = sh.m_blocks * sh.n_segs;
    const int grid = static_cast<int>(units < dev.num_sms ? units : dev.num_sms);
    note_launches(1);
    kern<<<grid, kThreads, kSmemBytes, s>>>(a, b, sh, ea);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch(EpiKind kind, const CUtensorMap& a, const CUtensorMap& b,
                     const GemmShape& sh, const EpiArgs& ea, const DevInfo& dev,
                     cudaStream_t s) {
    switch (kind) {
        case EpiKind::Fwd: return launch_one<EpiKind::Fwd, T, false, false>(a, b, sh, ea, dev, s);
        case EpiKind::Recomp:
            return launch_one<EpiKind::Recomp, T, false, false>(a, b, sh, ea, dev, s);
        case EpiKind::Dh: return launch_one<EpiKind::Dh, T, false, true>(a, b, sh, ea, dev, s);
        case EpiKind::Dw: return launch_one<EpiKind::Dw, T, true, true>(a, b, sh, ea, dev, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

// FP32 operands run on the CUDA-core kernel (simt_f32.cu).
cudaError_t launch_gemm_f32(EpiKind kind, const void* A, int64_t lda, int a_mn, const void* B,
                            int64_t ldb, int b_mn, int64_t M, int64_t N, int64_t K,
                            const GemmShape& shape, const EpiArgs& ea, const DevInfo& dev,
                            cudaStream_t s);

cudaError_t launch_gemm(EpiKind kind, int dtype, const void* A, int64_t lda, int a_mn,
                        const void* B, int64_t ldb, int b_mn, int64_t M, int64_t N, int64_t K,
                        const GemmShape& shape, const EpiArgs& ea, const DevInfo& dev,
                        cudaStream_t s) {
    if (dtype == LL_F32)
        return launch_gemm_f32(kind, A, lda, a_mn, B, ldb, b_mn, M, N, K, shape, ea, dev, s);
    const CUtensorMapDataType dt =
        dtype == LL_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap ma, mb;
    // K-major operand: [rows, K] box K=64 x rows; MN-major: [K, MN] box 64 x 64.
    const bool oka = a_mn ? make_map(&ma, A, dt, 2, M, K, lda, 64, kBK)
                          : make_map(&ma, A, dt, 2, K, M, lda, kBK, kBM);
    const bool okb = b_mn ? make_map(&mb, B, dt, 2, N, K, ldb, 64, kBK)
                          : make_map(&mb, B, dt, 2, K, N, ldb, kBK, kBN);
    if (!oka || !okb) return cudaErrorInvalidValue;
    if (dtype == LL_BF16) return dispatch<__nv_bfloat16>(kind, ma, mb, shape, ea, dev, s);
    return dispatch<__half>(kind, ma, mb, shape, ea, dev, s);
}

}  // namespace ll
