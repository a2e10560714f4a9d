#include "gemm_common.cuh"

namespace ll {
namespace {

// ------------------------------------------------------ FP32 (3 x TF32)
// FP32 operands on the tensor cores: each operand x is split exactly into
// hi = x with its 13 low mantissa bits cleared (a TF32 value) and
// lo = x - hi, and every K step runs three kind::tf32 MMAs,
// hi*hi + hi*lo + lo*hi (the lo*lo term, ~2^-22 of the product, is
// dropped).  TMA lands 16 K-values of A [128 x 16] and B [256 x 16] in a
// raw stage as they lie in memory: K-major operands in 64-byte rows
// (64-byte swizzle), MN-major operands in 32-wide 128-byte boxes.  Eight
// converter warps write the hi and lo parts of both into a converted stage,
// always K-major with 64-byte rows: kind::tf32 takes no MN-major operand, so
// the converters transpose MN-major tiles on the way.  When every operand of
// a launch is K-major (forward, recompute) the raw stage is already in that
// layout and serves as hi itself, so the converters write lo alone.  This
// relies on kind::tf32 ignoring the 13 low mantissa bits of its FP32 inputs:
// measured on GB300, the unmasked values give bitwise the same results.
constexpr int kAfBytes = kBM * kBKf * 4;       // 8 KB
constexpr int kBfBytes = kBN * kBKf * 4;       // 16 KB
constexpr int kRawBytes = kAfBytes + kBfBytes; // 24 KB (one raw stage)
constexpr int kConvBytes = 2 * kRawBytes;      // hi A, hi B, lo A, lo B
constexpr int kRawStages = 4;
constexpr int kConvStages = 2;
// Launches whose operands are all K-major (forward, recompute): the raw
// stage itself serves as hi and the converters write lo alone, so a
// converted stage is half as large and the memory goes to a deeper raw ring
// (TMA lookahead): 6 x 24 KB raw + 2 x 24 KB lo (measured best of 4 + 4,
// 5 + 3 and 6 + 2).  A raw stage is freed by the MMA commit.
constexpr int kRawStagesKK = 6;
constexpr int kLoStagesKK = 2;
constexpr int kMaxRaw = kRawStagesKK > kRawStages ? kRawStagesKK : kRawStages;
constexpr int kMaxConv = kLoStagesKK > kConvStages ? kLoStagesKK : kConvStages;
static_assert(kRawStagesKK * kRawBytes + kLoStagesKK * kRawBytes == kStages * kStageBytes,
              "tf32 rings (all K-major) fill the 16-bit kernel's stage memory");
constexpr int kMnBoxF = 32 * kBKf * 4;         // one 32(MN) x 16(K) box, 2 KB
constexpr int kConvWarps = 8;                  // hi / lo converter warps
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kThreadsF = 192 + kConvThreads;  // producer, MMA, 4 epilogue, converters
static_assert(kConvThreads % 128 == 0, "converters split whole 128-thread groups");
static_assert(kRawStages * kRawBytes + kConvStages * kConvBytes == kStages * kStageBytes,
              "tf32 rings fill the 16-bit kernel's stage memory");

struct BarsF {
    uint64_t full[kMaxRaw];        // TMA landed in the raw stage
    uint64_t rempty[kMaxRaw];      // raw stage free (converters done; all K-major: MMAs done)
    uint64_t conv[kMaxConv];       // hi / lo (all K-major: lo) written
    uint64_t empty[kMaxConv];      // MMAs done with the converted stage
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t sfull[kSchedDepth];
    uint64_t sempty[kSchedDepth];
    uint64_t drain;
    int sched[kSchedDepth];
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(BarsF) <= 512, "barrier block");

template <bool A_MN, bool B_MN>
__device__ __forceinline__ void load_stage_f(uint8_t* st, const CUtensorMap* tmA,
                                             const CUtensorMap* tmB, uint64_t* fb, int32_t k0,
                                             int32_t m0, int32_t n0) {
    uint8_t* sa = st;
    uint8_t* sb = st + kAfBytes;
    mbar_arrive_expect_tx(fb, kRawBytes);
    if constexpr (!A_MN) {
        tma_load_2d(sa, tmA, fb, k0, m0);
    } else {
#pragma unroll
        for (int j = 0; j < kBM / 32; ++j) tma_load_2d(sa + j * kMnBoxF, tmA, fb, m0 + 32 * j, k0);
    }
    if constexpr (!B_MN) {
        tma_load_2d(sb, tmB, fb, k0, n0);
    } else {
#pragma unroll
        for (int j = 0; j < kBN / 32; ++j) tma_load_2d(sb + j * kMnBoxF, tmB, fb, n0 + 32 * j, k0);
    }
}

// K-major operand with 64-byte rows: 8-row groups of 512 B, a K step of
// 8 values is 32 B along the row.
__device__ __forceinline__ uint64_t desc_f(uint32_t base, int kk) {
    return smem_desc_sw64(base + kk * 32, 16, 512);
}

constexpr uint32_t kIdescF = instr_desc(2 /*tf32*/, 0, 0, kBM, kBN);

// hi: A at hi, B at hi + 8 KB; lo likewise (a converted stage holds hi then
// lo; all K-major: hi is the raw stage, lo a stage of its own).
__device__ __forceinline__ void mma_stage_f(uint32_t d_tmem, uint32_t hi, uint32_t lo,
                                            bool first) {
    const uint32_t a_hi = hi, b_hi = hi + kAfBytes;
    const uint32_t a_lo = lo, b_lo = lo + kAfBytes;
#pragma unroll
    for (int kk = 0; kk < kBKf / 8; ++kk) {
        tc_mma<1>(d_tmem, desc_f(a_hi, kk), desc_f(b_hi, kk), kIdescF,
                  (!first || kk > 0) ? 1u : 0u);
        tc_mma<1>(d_tmem, desc_f(a_hi, kk), desc_f(b_lo, kk), kIdescF, 1u);
        tc_mma<1>(d_tmem, desc_f(a_lo, kk), desc_f(b_hi, kk), kIdescF, 1u);
    }
}

__device__ __forceinline__ void split_tf32(const uint4& x, uint4& hi, uint4& lo) {
    hi.x = x.x & 0xFFFFE000u;
    hi.y = x.y & 0xFFFFE000u;
    hi.z = x.z & 0xFFFFE000u;
    hi.w = x.w & 0xFFFFE000u;
    lo.x = __float_as_uint(__uint_as_float(x.x) - __uint_as_float(hi.x));
    lo.y = __float_as_uint(__uint_as_float(x.y) - __uint_as_float(hi.y));
    lo.z = __float_as_uint(__uint_as_float(x.z) - __uint_as_float(hi.z));
    lo.w = __float_as_uint(__uint_as_float(x.w) - __uint_as_float(hi.w));
}

// One operand of ROWS rows x 16 K-values from its raw stage into hi / lo in
// K-major 64-byte rows (row r at r * 64, 16-byte chunk c at c ^ ((r >> 1) & 3),
// the 64-byte swizzle).  ct = converter thread 0..kConvThreads - 1.
template <bool MN, int ROWS>
__device__ __forceinline__ void convert_operand(const uint8_t* raw, uint8_t* hi, uint8_t* lo,
                                                int ct) {
    if constexpr (!MN) {
        // already in that layout: split 16-byte vectors in place
#pragma unroll
        for (int e = ct; e < ROWS * 4; e += kConvThreads) {
            const uint4 x = *reinterpret_cast<const uint4*>(raw + e * 16);
            uint4 h, l;
            split_tf32(x, h, l);
            *reinterpret_cast<uint4*>(hi + e * 16) = h;
            *reinterpret_cast<uint4*>(lo + e * 16) = l;
        }
    } else {
        // box j: K-row k (128 B) holds MN values 32j..32j+31, 16-byte chunk c
        // (MN values 4c..4c+3) at c ^ (k & 7).  Thread (mn = ct & 31,
        // q = ct >> 5) gathers K values 4q..4q+3 of one MN index.
        // (the converter threads split the boxes: thread ct takes boxes
        // ct / 128, ct / 128 + kConvThreads / 128, ...)
        const int m = ct & 31, q = (ct >> 5) & 3;
        const uint32_t src = static_cast<uint32_t>((m & 3) * 4);
#pragma unroll
        for (int j = ct >> 7; j < ROWS / 32; j += kConvThreads / 128) {
            const uint8_t* box = raw + j * kMnBoxF;
            uint4 x;
            uint32_t* xv = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int k = 4 * q + i;
                xv[i] = *reinterpret_cast<const uint32_t*>(box + k * 128 +
                                                           (((m >> 2) ^ (k & 7)) * 16) + src);
            }
            uint4 h, l;
            split_tf32(x, h, l);
            const int r = j * 32 + m;
            const int off = r * 64 + ((q ^ ((r >> 1) & 3)) * 16);
            *reinterpret_cast<uint4*>(hi + off) = h;
            *reinterpret_cast<uint4*>(lo + off) = l;
        }
    }
}

// All K-major: lo = x - (x with its 13 low mantissa bits cleared) of both
// operands, at the raw stage's offsets.
__device__ __forceinline__ void convert_stage_lo(const uint8_t* raw, uint8_t* lo, int ct) {
#pragma unroll
    for (int e = ct; e < (kBM + kBN) * 4; e += kConvThreads) {
        const uint4 x = *reinterpret_cast<const uint4*>(raw + e * 16);
        uint4 h, l;
        split_tf32(x, h, l);
        *reinterpret_cast<uint4*>(lo + e * 16) = l;
    }
}

template <bool A_MN, bool B_MN>
__device__ __forceinline__ void convert_stage(const uint8_t* raw, uint8_t* cv, int ct) {
    convert_operand<A_MN, kBM>(raw, cv, cv + kRawBytes, ct);
    convert_operand<B_MN, kBN>(raw + kAfBytes, cv + kAfBytes, cv + kRawBytes + kAfBytes, ct);
}

template <class K0, class K1, int NK>
__global__ void __launch_bounds__(kThreadsF, 1)
    gemm_tf32_kernel(const __grid_constant__ CUtensorMap tmA0,
                     const __grid_constant__ CUtensorMap tmB0,
                     const __grid_constant__ CUtensorMap tmO0,
                     const __grid_constant__ CUtensorMap tmA1,
                     const __grid_constant__ CUtensorMap tmB1,
                     const __grid_constant__ CUtensorMap tmO1, const KParams P,
                     const EpiArgs ea0, const EpiArgs ea1) {
    using T = float;
    // all operands K-major: the raw stage is the hi operand (see kRawStagesKK)
    constexpr bool KK = !K0::kAmn && !K0::kBmn && (NK == 1 || (!K1::kAmn && !K1::kBmn));
    constexpr int kR = KK ? kRawStagesKK : kRawStages;  // raw ring
    constexpr int kC = KK ? kLoStagesKK : kConvStages;  // converted ring
    constexpr int kCB = KK ? kRawBytes : kConvBytes;    // converted stage bytes
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* outbuf = smem + kStages * kStageBytes;
    BarsF* bars = reinterpret_cast<BarsF*>(outbuf + kOutBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t total = P.n_units[0] + (NK > 1 ? P.n_units[1] : 0);
    const uint64_t wait_ns = ea0.wait_ns;
    int* status = ea0.status;
    volatile int* abort = &bars->abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kR; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->rempty[s], KK ? 1 : kConvWarps);  // MMA commit, or converters
        }
        for (int s = 0; s < kC; ++s) {
            mbar_init(&bars->conv[s], kConvWarps);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->tfull[b], 1);
            mbar_init(&bars->tempty[b], 4);
        }
        for (int s = 0; s < kSchedDepth; ++s) {
            mbar_init(&bars->sfull[s], 1);
            mbar_init(&bars->sempty[s], 5 + kConvWarps);  // MMA + 4 epilogue + converters
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA0);
        tma_prefetch_desc(&tmB0);
        if (NK > 1) {
            tma_prefetch_desc(&tmA1);
            tma_prefetch_desc(&tmB1);
        }
        if (P.zero_counter && blockIdx.x == 0) *P.zero_counter = 0;
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    // every role but the producer takes the unit sequence from the ring
    auto next_unit = [&](int& sslot, uint32_t& sphase, bool& ok) -> int {
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->sfull[sslot], sphase, wait_ns, abort))) {
            ok = false;
            return -1;
        }
        const int u = *reinterpret_cast<volatile int*>(&bars->sched[sslot]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->sempty[sslot]);
        if (++sslot == kSchedDepth) {
            sslot = 0;
            sphase ^= 1;
        }
        return u;
    };

    if (warp == 0) {
        // ------------------------------------------- scheduler + TMA producer
        int stage = 0, sslot = 0;
        uint32_t phase = 0, sphase = 0;
        // stages with a load issued, and the phase it completes (bit per stage)
        uint32_t issued = 0, issued_phase = 0;
        bool ok = true;
        int64_t next_static = blockIdx.x;
        while (ok) {
            int64_t u;
            if (P.dynamic) {
                int got = 0;
                if (lane == 0) got = atomicAdd(P.counter, 1);
                u = __shfl_sync(0xffffffffu, got, 0);
            } else {
                u = next_static;
                next_static += gridDim.x;
            }
            if (u >= total) u = -1;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&bars->sempty[sslot], sphase ^ 1, wait_ns, abort))) {
                ok = false;
                break;
            }
            if (lane == 0) {
                bars->sched[sslot] = static_cast<int>(u);
                mbar_arrive(&bars->sfull[sslot]);
            }
            __syncwarp();
            if (++sslot == kSchedDepth) {
                sslot = 0;
                sphase ^= 1;
            }
            if (u < 0) break;
            const Unit un = decode_unit(P, u);
            for (int64_t t = un.t0; t < un.t1 && ok; ++t) {
                for (int64_t kb = 0; kb < un.k_blocks; ++kb) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(&bars->rempty[stage], phase ^ 1, wait_ns, abort))) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        uint8_t* st = smem + stage * kRawBytes;
                        const int32_t k0 = static_cast<int32_t>((un.k_begin + kb) * kBKf);
                        const int32_t m0 = static_cast<int32_t>(un.mb * kBM);
                        const int32_t n0 = static_cast<int32_t>(t * kBN);
                        if (NK == 1 || un.kind == 0)
                            load_stage_f<K0::kAmn, K0::kBmn>(st, &tmA0, &tmB0,
                                                             &bars->full[stage], k0, m0, n0);
                        else
                            load_stage_f<K1::kAmn, K1::kBmn>(st, &tmA1, &tmB1,
                                                             &bars->full[stage], k0, m0, n0);
                    }
                    __syncwarp();
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == kR) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
        if (!ok) {
            if (lane == 0) set_status(status, LL_ERR_DEVICE_TIMEOUT);
            bars->abort = 1;
            for (int s = 0; s < kR; ++s)
                if ((issued >> s) & 1u)
                    mbar_wait(&bars->full[s], (issued_phase >> s) & 1u, wait_ns, nullptr);
        }
    } else if (warp >= 6) {
        // ------------------------------------------------ hi / lo converters
        const int ct = threadIdx.x - 6 * 32;  // 0..kConvThreads - 1
        int rs = 0, cs = 0, sslot = 0;
        uint32_t rphase = 0, cphase = 0, sphase = 0;
        bool ok = true;
        uint8_t* conv_base = smem + kR * kRawBytes;
        while (ok) {
            const int u = next_unit(sslot, sphase, ok);
            if (!ok || u < 0) break;
            const Unit un = decode_unit(P, u);
            const int64_t steps = (un.t1 - un.t0) * un.k_blocks;
            for (int64_t i = 0; i < steps; ++i) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&bars->full[rs], rphase, wait_ns, abort) &&
                                    mbar_wait(&bars->empty[cs], cphase ^ 1, wait_ns, abort))) {
                    ok = false;
                    break;
                }
                const uint8_t* raw = smem + rs * kRawBytes;
                uint8_t* cv = conv_base + cs * kCB;
                if constexpr (KK)
                    convert_stage_lo(raw, cv, ct);
                else if (NK == 1 || un.kind == 0)
                    convert_stage<K0::kAmn, K0::kBmn>(raw, cv, ct);
                else
                    convert_stage<K1::kAmn, K1::kBmn>(raw, cv, ct);
                fence_proxy_async_shared_cta();
                __syncwarp();
                if (lane == 0) {
                    if (!KK) mbar_arrive(&bars->rempty[rs]);  // all K-major: the MMAs free it
                    mbar_arrive(&bars->conv[cs]);
                }
                if (++rs == kR) {
                    rs = 0;
                    rphase ^= 1;
                }
                if (++cs == kC) {
                    cs = 0;
                    cphase ^= 1;
                }
            }
        }
        if (!ok) {
            if (lane == 0) set_status(status, LL_ERR_DEVICE_TIMEOUT);
            bars->abort = 1;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        int stage = 0, sslot = 0, buf = 0, rs = 0;
        uint32_t phase = 0, sphase = 0, bphase = 0, rphase = 0;
        bool ok = true;
        const uint32_t rbase = smem_u32(smem);
        const uint32_t sbase = rbase + kR * kRawBytes;
        while (ok) {
            const int u = next_unit(sslot, sphase, ok);
            if (!ok || u < 0) break;
            const Unit un = decode_unit(P, u);
            for (int64_t t = un.t0; t < un.t1 && ok; ++t) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&bars->tempty[buf], bphase ^ 1, wait_ns, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + buf * kBN;
                for (int64_t kb = 0; kb < un.k_blocks; ++kb) {
                    // all K-major: the raw stage (hi) too, which its converters
                    // have seen land already
                    if (!__all_sync(0xffffffffu,
                                    (!KK || mbar_wait(&bars->full[rs], rphase, wait_ns, abort)) &&
                                        mbar_wait(&bars->conv[stage], phase, wait_ns, abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t cvs = sbase + stage * kCB;
                        if constexpr (KK) {
                            mma_stage_f(d_tmem, rbase + rs * kRawBytes, cvs, kb == 0);
                            tc_commit(&bars->rempty[rs]);
                        } else {
                            mma_stage_f(d_tmem, cvs, cvs + kRawBytes, kb == 0);
                        }
                        tc_commit(&bars->empty[stage]);
                    }
                    __syncwarp();
                    if (++stage == kC) {
                        stage = 0;
                        phase ^= 1;
                    }
                    if (++rs == kR) {
                        rs = 0;
                        rphase ^= 1;
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
            if (lane == 0) set_status(status, LL_ERR_DEVICE_TIMEOUT);
            bars->abort = 1;
        }
        if (lane == 0) tc_commit(&bars->drain);
        __syncwarp();
        mbar_wait(&bars->drain, 0, wait_ns, nullptr);
    } else {
        // ------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int r_in_tile = q * 32 + lane;
        uint8_t* wbuf = outbuf + q * 2 * kOutBufBytes;
        int sslot = 0, buf = 0, sidx = 0;
        uint32_t sphase = 0, bphase = 0;
        bool ok = true;
        typename K0::Epi epi0;
        typename K1::Epi epi1;
        while (ok) {
            const int u = next_unit(sslot, sphase, ok);
            if (!ok || u < 0) break;
            const Unit un = decode_unit(P, u);
            const int kind = (NK == 1) ? 0 : un.kind;
            const EpiArgs& ea = kind == 0 ? ea0 : ea1;
            const CUtensorMap* tmO = kind == 0 ? &tmO0 : &tmO1;
            const bool reduce = P.reduce[kind] != 0;
            const bool stores = P.out_rows[kind] > 0;
            // a K part of grad_hidden stores its partial sum at rows part * M
            const int64_t row0 = un.mb * kBM + q * 32 + un.kpart * P.part_rows[kind];
            if (kind == 0)
                epi0.begin_unit(ea, un.mb * kBM + r_in_tile);
            else
                epi1.begin_unit(ea, un.mb * kBM + r_in_tile);
            for (int64_t t = un.t0; t < un.t1; ++t) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&bars->tfull[buf], bphase, wait_ns, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem + buf * kBN + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
                for (int c = 0; c < kBN / 32; ++c) {
                    uint32_t r[32];
                    __syncwarp();
                    tmem_ld32(taddr + c * 32, r);
                    tmem_ld_wait(r);
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    const int64_t col0 = t * kBN + c * 32;
                    if (kind == 0)
                        epi0.chunk(ea, v, col0);
                    else
                        epi1.chunk(ea, v, col0);
                    if (!stores) continue;
                    // a box past the output is neither staged nor stored (each
                    // staging buffer holds exactly one store in flight)
                    const bool put = row0 < P.out_rows[kind] && col0 < P.out_cols[kind];
                    uint8_t* sb = wbuf + (sidx & 1) * kOutBufBytes;
                    if (put) {
                        if (lane == 0) bulk_wait_read_1();
                        __syncwarp();
                        stage_row<T>(sb, lane, v, false, 0);
                    }
                    if (kind == 0) epi0.db_partials(ea, v, col0);
                    if (!put) continue;
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (reduce)
                            tma_reduce_add_2d(tmO, sb, static_cast<int32_t>(col0),
                                              static_cast<int32_t>(row0));
                        else
                            tma_store_2d(tmO, sb, static_cast<int32_t>(col0),
                                         static_cast<int32_t>(row0));
                        bulk_commit();
                    }
                    ++sidx;
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
            if (kind == 0)
                epi0.end_unit(ea, un.seg);
            else
                epi1.end_unit(ea, un.seg);
        }
        if (lane == 0) bulk_wait_all();
        if (!ok) {
            if (lane == 0) set_status(status, LL_ERR_DEVICE_TIMEOUT);
            bars->abort = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <class K0, class K1, int NK>
cudaError_t launch_f(const CUtensorMap* m, const KParams& P, const EpiArgs& ea0,
                     const EpiArgs& ea1, const DevInfo& dev, int max_ctas, cudaStream_t s) {
    auto kern = gemm_tf32_kernel<K0, K1, NK>;
    static int configured[64] = {0};
    if (dev.device < 64 && !configured[dev.device]) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        configured[dev.device] = 1;
    }
    const int64_t units = P.n_units[0] + (NK > 1 ? P.n_units[1] : 0);
    const int cap = (max_ctas > 0 && max_ctas < dev.num_sms) ? max_ctas : dev.num_sms;
    int grid = static_cast<int>(units < cap ? units : cap);
    if (grid < 1) grid = 1;
    note_launches(1);
    kern<<<grid, kThreadsF, kSmemBytes, s>>>(m[0], m[1], m[2], m[3], m[4], m[5], P, ea0, ea1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t dispatch_f32(const GemmLaunch& L, const CUtensorMap* m, const KParams& P,
                         const DevInfo& dev, cudaStream_t s) {
    using Fwd = Kind<float, EpiKind::Fwd, false, false>;
    using Rec = Kind<float, EpiKind::Recomp, false, false>;
    // gradient operands as the backward passes them: K-major copies (W^T,
    // S^T, h^T: the converters only split), or W, S and h themselves (the
    // converters transpose)
    using DhT = Kind<float, EpiKind::Dh, false, false>;
    using DwT = Kind<float, EpiKind::Dw, false, false>;
    using DhM = Kind<float, EpiKind::Dh, false, true>;
    using DwM = Kind<float, EpiKind::Dw, true, true>;
    const int mc = L.max_ctas;
    auto is = [&](int k, int a_mn, int b_mn) {
        return L.op[k].a_mn == a_mn && L.op[k].b_mn == b_mn;
    };
    if (L.nkinds == 1) {
        switch (L.kind[0]) {
            case EpiKind::Fwd:
                if (!is(0, 0, 0)) break;
                return launch_f<Fwd, Fwd, 1>(m, P, L.ea[0], L.ea[0], dev, mc, s);
            case EpiKind::Recomp:
                if (!is(0, 0, 0)) break;
                return launch_f<Rec, Rec, 1>(m, P, L.ea[0], L.ea[0], dev, mc, s);
            case EpiKind::Dh:
                if (is(0, 0, 0)) return launch_f<DhT, DhT, 1>(m, P, L.ea[0], L.ea[0], dev, mc, s);
                if (is(0, 0, 1)) return launch_f<DhM, DhM, 1>(m, P, L.ea[0], L.ea[0], dev, mc, s);
                break;
            case EpiKind::Dw:
                if (is(0, 0, 0)) return launch_f<DwT, DwT, 1>(m, P, L.ea[0], L.ea[0], dev, mc, s);
                if (is(0, 1, 1)) return launch_f<DwM, DwM, 1>(m, P, L.ea[0], L.ea[0], dev, mc, s);
                break;
        }
    } else if (L.kind[0] == EpiKind::Dh && L.kind[1] == EpiKind::Dw) {
        if (is(0, 0, 0) && is(1, 0, 0))
            return launch_f<DhT, DwT, 2>(m, P, L.ea[0], L.ea[1], dev, mc, s);
        if (is(0, 0, 1) && is(1, 1, 1))
            return launch_f<DhM, DwM, 2>(m, P, L.ea[0], L.ea[1], dev, mc, s);
    }
    return cudaErrorInvalidValue;
}


}  // namespace ll
