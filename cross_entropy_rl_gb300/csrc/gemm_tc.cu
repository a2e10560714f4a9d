// Tensor-core GEMMs with fused epilogues for the 16-bit operand paths
// (bf16 / fp16 operands, FP32 accumulation in TMEM).
//
// The three contractions of the fused linear logp (RL-Kernel issue #261,
// "Current accumulation": the chunked matmul accumulated into an FP32
// gradient table; Liger-Kernel PR #1324, "Details": no [V, H] temporary):
//   forward / recompute   z  = h . W^T        A = h [rows, D]  (K-major)
//                                              B = W [V, D]     (K-major)
//   grad_hidden           dh = S . W          A = S [rows, V]  (K-major)
//                                              B = W [V, D]     (MN-major)
//   grad_weight           dW += S^T . h       A = S [rows, V]  (MN-major)
//                                              B = h [rows, D]  (MN-major)
//
// Design (sm_103a): one persistent CTA per SM, 6 warps.
//   warp 0      scheduler + TMA producer: picks work units (static
//               round-robin, or an atomic counter), publishes them in a
//               shared-memory ring, loads 128-byte-swizzled tiles into a
//               4-stage ring
//   warp 1      allocates 512 TMEM columns, issues tcgen05.mma (128x256x16)
//   warps 2..5  epilogue: tcgen05.ld of its 32 TMEM lanes, fused epilogue,
//               output rows staged in swizzled shared memory and written by
//               TMA bulk-tensor stores (or reduce-adds); the forward may also
//               store its FP32 logits tile (single fwd+bwd call)
// One launch may carry two tile kinds (grad_hidden and grad_weight tiles of
// the same chunk), the long kind first, so that the dynamic scheduler evens
// out the SMs' work.  Two 256-column accumulators in TMEM let the epilogue
// of one tile overlap the MMAs of the next.  Which SM computes a tile never
// changes any result: every output element is one MMA accumulation over K
// in a fixed order.
#include "gemm_common.cuh"

namespace ll {
namespace {

template <typename T, class K0, class K1, int NK>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmO1,
                   const __grid_constant__ CUtensorMap tmL0, const __grid_constant__ CUtensorMap tmL1,
                   const KParams P, const EpiArgs ea0, const EpiArgs ea1) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* outbuf = smem + kStages * kStageBytes;
    Bars* bars = reinterpret_cast<Bars*>(outbuf + kOutBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t total = P.n_units[0] + (NK > 1 ? P.n_units[1] : 0);
    const uint64_t wait_ns = ea0.wait_ns;
    int* status = ea0.status;
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
        for (int s = 0; s < kSchedDepth; ++s) {
            mbar_init(&bars->sfull[s], 1);
            mbar_init(&bars->sempty[s], 5);  // MMA warp + 4 epilogue warps
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
            const int n_lo = unit_lo_count(P, u);
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&bars->sempty[sslot], sphase ^ 1, wait_ns, abort))) {
                ok = false;
                break;
            }
            if (lane == 0) {
                bars->sched[sslot] = static_cast<int>(u);
                bars->sched_lo[sslot] = n_lo;
                mbar_arrive(&bars->sfull[sslot]);
            }
            __syncwarp();
            if (++sslot == kSchedDepth) {
                sslot = 0;
                sphase ^= 1;
            }
            if (u < 0) break;
            const Unit un = decode_unit(P, u, n_lo);
            for (int64_t t = un.t0; t < un.t1 && ok; ++t) {
                for (int64_t kb = 0; kb < un.k_blocks; ++kb) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(&bars->empty[stage], phase ^ 1, wait_ns, abort))) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        uint8_t* sa = smem + stage * kStageBytes;
                        // a hi / lo split runs K twice: A, then A_lo, against the same B
                        const int64_t ks = P.k_split[un.kind];
                        const bool lo = ks > 0 && kb >= ks;
                        const int32_t m0 = static_cast<int32_t>(un.mb * kBM);
                        const int32_t n0 = static_cast<int32_t>(t * kBN);
                        if (lo && P.lo_cnt[un.kind]) {  // planned second pass
                            int32_t k0;
                            uint32_t bits;
                            lo_block(P, un, kb - ks, &k0, &bits);
                            if (NK == 1 || un.kind == 0)
                                load_stage_lo<K0::kAmn, K0::kBmn>(sa, &tmL0, &tmB0,
                                                                  &bars->full[stage], k0, m0, n0,
                                                                  bits);
                            else
                                load_stage_lo<K1::kAmn, K1::kBmn>(sa, &tmL1, &tmB1,
                                                                  &bars->full[stage], k0, m0, n0,
                                                                  bits);
                        } else {
                            const int32_t k0 = static_cast<int32_t>((lo ? kb - ks : kb) * kBK);
                            if (NK == 1 || un.kind == 0)
                                load_stage<K0::kAmn, K0::kBmn>(sa, lo ? &tmL0 : &tmA0, &tmB0,
                                                               &bars->full[stage], k0, m0, n0);
                            else
                                load_stage<K1::kAmn, K1::kBmn>(sa, lo ? &tmL1 : &tmA1, &tmB1,
                                                               &bars->full[stage], k0, m0, n0);
                        }
                    }
                    __syncwarp();
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
        if (!ok) {
            if (lane == 0) set_status(status, LL_ERR_DEVICE_TIMEOUT);
            bars->abort = 1;
            for (int s = 0; s < kStages; ++s)
                if ((issued >> s) & 1u)
                    mbar_wait(&bars->full[s], (issued_phase >> s) & 1u, wait_ns, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        int stage = 0, sslot = 0, buf = 0;
        uint32_t phase = 0, sphase = 0, bphase = 0;
        bool ok = true;
        const uint32_t sbase = smem_u32(smem);
        while (ok) {
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->sfull[sslot], sphase, wait_ns, abort))) {
                ok = false;
                break;
            }
            const int u = *reinterpret_cast<volatile int*>(&bars->sched[sslot]);
            const int n_lo = *reinterpret_cast<volatile int*>(&bars->sched_lo[sslot]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->sempty[sslot]);
            if (++sslot == kSchedDepth) {
                sslot = 0;
                sphase ^= 1;
            }
            if (u < 0) break;
            const Unit un = decode_unit(P, u, n_lo);
            for (int64_t t = un.t0; t < un.t1 && ok; ++t) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&bars->tempty[buf], bphase ^ 1, wait_ns, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + buf * kBN;
                for (int64_t kb = 0; kb < un.k_blocks; ++kb) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(&bars->full[stage], phase, wait_ns, abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t sa = sbase + stage * kStageBytes;
                        if (NK == 1 || un.kind == 0)
                            mma_stage<K0::kAmn, K0::kBmn, K0::kIdesc>(d_tmem, sa, kb == 0);
                        else
                            mma_stage<K1::kAmn, K1::kBmn, K1::kIdesc>(d_tmem, sa, kb == 0);
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
            if (lane == 0) set_status(status, LL_ERR_DEVICE_TIMEOUT);
            bars->abort = 1;
        }
        if (lane == 0) tc_commit(&bars->drain);
        __syncwarp();
        mbar_wait(&bars->drain, 0, wait_ns, nullptr);
    } else {
        // ------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lanes [32q, 32q + 32)
        const int r_in_tile = q * 32 + lane;
        uint8_t* wbuf = outbuf + q * 2 * kOutBufBytes;
        int sslot = 0, buf = 0, sidx = 0;
        uint32_t sphase = 0, bphase = 0;
        bool ok = true;
        typename K0::Epi epi0;
        typename K1::Epi epi1;
        while (ok) {
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->sfull[sslot], sphase, wait_ns, abort))) {
                ok = false;
                break;
            }
            const int u = *reinterpret_cast<volatile int*>(&bars->sched[sslot]);
            const int n_lo = *reinterpret_cast<volatile int*>(&bars->sched_lo[sslot]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->sempty[sslot]);
            if (++sslot == kSchedDepth) {
                sslot = 0;
                sphase ^= 1;
            }
            if (u < 0) break;
            const Unit un = decode_unit(P, u, n_lo);
            const int kind = (NK == 1) ? 0 : un.kind;
            const EpiArgs& ea = kind == 0 ? ea0 : ea1;
            const CUtensorMap* tmO = kind == 0 ? &tmO0 : &tmO1;
            const bool out16 = P.out16[kind] != 0;
            const bool reduce = P.reduce[kind] != 0;
            // every kind but the plain forward stores its tile; the forward
            // stores its logits tile too when given an output (one fwd+bwd call)
            const bool stores = P.out_rows[kind] > 0;
            const int64_t row0 = un.mb * kBM + q * 32;  // first output row of this warp
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
                    __syncwarp();  // tcgen05.ld is warp-collective (.sync.aligned)
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
                    const int h = out16 ? (c & 1) : 0;
                    // first column of the staged box (two chunks for 16-bit
                    // outputs); a box past the output is neither staged nor
                    // stored, so each staging buffer holds exactly one store
                    const int64_t x0 = out16 ? col0 - 32 * h : col0;
                    const bool put = row0 < P.out_rows[kind] && x0 < P.out_cols[kind];
                    uint8_t* sb = wbuf + (sidx & 1) * kOutBufBytes;
                    if (put) {
                        if (h == 0) {  // the store that last used this buffer has read it
                            if (lane == 0) bulk_wait_read_1();
                            __syncwarp();
                        }
                        stage_row<T>(sb, lane, v, out16, h);
                    }
                    if (kind == 0) {
                        epi0.store_lo(ea, v, col0);  // hi / lo split of S (recompute only)
                        epi0.db_partials(ea, v, col0);  // grad_bias partials, consumes v
                    }
                    if (put && (!out16 || h == 1)) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (reduce)
                                tma_reduce_add_2d(tmO, sb, static_cast<int32_t>(x0),
                                                  static_cast<int32_t>(row0));
                            else
                                tma_store_2d(tmO, sb, static_cast<int32_t>(x0),
                                             static_cast<int32_t>(row0));
                            bulk_commit();
                        }
                        ++sidx;
                    }
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

// ------------------------------------------- CTA pairs (cta_group::2)
// The same GEMM on a pair of CTAs (a cluster of two SMs): one 256 x 256
// output tile per pair, each CTA holding 128 rows of A and 128 of the 256
// columns of B in its shared memory and 128 rows x 256 columns of the
// accumulator in its TMEM.  The even CTA (the leader) runs the scheduler and
// issues the M = 256 MMAs (tcgen05.mma.cta_group::2), which read both CTAs'
// operand tiles; every CTA loads its own tiles, their transaction bytes
// counted on the leader's stage barrier.  MMA completion is multicast to both
// CTAs (stage free, accumulator ready); each CTA's epilogue then works on its
// own 128 rows exactly like the single-CTA kernel.  Per SM, a k-step moves
// A 16 KB + B 16 KB instead of 16 + 32 KB: a third less operand traffic for
// the same tensor work.
constexpr int kPairStages = 6;
constexpr int kBHalf = kBN / 2;
constexpr int kPairStageBytes = kABytes + kBHalf * kBK * 2;  // 32 KB
static_assert(kPairStages * kPairStageBytes == kStages * kStageBytes, "same stage memory");

struct BarsPair {
    uint64_t full[kPairStages];   // leader: both CTAs' tiles landed
    uint64_t empty[kPairStages];  // both: the pair MMAs are done with the stage
    uint64_t tfull[2];            // both: accumulator ready
    uint64_t tempty[2];           // leader: both CTAs' epilogues drained it
    uint64_t sfull[kSchedDepth];  // both: unit id written
    uint64_t sempty[kSchedDepth]; // leader: every consumer of the pair read it
    uint64_t drain;
    int sched[kSchedDepth];
    int sched_lo[kSchedDepth];  // second-pass K blocks of the unit in sched
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(BarsPair) <= 512, "barrier block");

template <bool A_MN, bool B_MN>
__device__ __forceinline__ void load_stage_pair(uint8_t* sa, const CUtensorMap* tmA,
                                                const CUtensorMap* tmB, uint32_t bar_cl,
                                                int32_t k0, int32_t m0, int32_t n0) {
    uint8_t* sb = sa + kABytes;
    if constexpr (!A_MN) {
        tma_load_2d_pair(sa, tmA, bar_cl, k0, m0);
    } else {
#pragma unroll
        for (int j = 0; j < kBM / 64; ++j)
            tma_load_2d_pair(sa + j * kMnBoxBytes, tmA, bar_cl, m0 + 64 * j, k0);
    }
    if constexpr (!B_MN) {
        tma_load_2d_pair(sb, tmB, bar_cl, k0, n0);
    } else {
#pragma unroll
        for (int j = 0; j < kBHalf / 64; ++j)
            tma_load_2d_pair(sb + j * kMnBoxBytes, tmB, bar_cl, n0 + 64 * j, k0);
    }
}

template <bool A_MN, bool B_MN>
__device__ __forceinline__ void load_stage_pair_lo(uint8_t* sa, const CUtensorMap* tmL,
                                                   const CUtensorMap* tmB, uint32_t bar_cl,
                                                   int32_t k0, int32_t m0, int32_t n0,
                                                   uint32_t bits) {
    uint8_t* sb = sa + kABytes;
    load_a_pieces<A_MN>(sa, k0, m0, bits, [&](uint8_t* d, int32_t x, int32_t y) {
        tma_load_2d_pair(d, tmL, bar_cl, x, y);
    });
    if constexpr (!B_MN) {
        tma_load_2d_pair(sb, tmB, bar_cl, k0, n0);
    } else {
#pragma unroll
        for (int j = 0; j < kBHalf / 64; ++j)
            tma_load_2d_pair(sb + j * kMnBoxBytes, tmB, bar_cl, n0 + 64 * j, k0);
    }
}

template <bool A_MN, bool B_MN, uint32_t IDESC>
__device__ __forceinline__ void mma_stage_pair(uint32_t d_tmem, uint32_t sa, bool first) {
    const uint32_t sb = sa + kABytes;
#pragma unroll
    for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint64_t ad = A_MN ? smem_desc_sw128(sa + kk * 2048, kMnBoxBytes, 1024)
                                 : smem_desc_sw128(sa + kk * 32, 16, 1024);
        const uint64_t bd = B_MN ? smem_desc_sw128(sb + kk * 2048, kMnBoxBytes, 1024)
                                 : smem_desc_sw128(sb + kk * 32, 16, 1024);
        tc_mma_pair(d_tmem, ad, bd, IDESC, (!first || kk > 0) ? 1u : 0u);
    }
}

template <typename T, class K0, class K1, int NK>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA0,
                     const __grid_constant__ CUtensorMap tmB0,
                     const __grid_constant__ CUtensorMap tmO0,
                     const __grid_constant__ CUtensorMap tmA1,
                     const __grid_constant__ CUtensorMap tmB1,
                     const __grid_constant__ CUtensorMap tmO1,
                     const __grid_constant__ CUtensorMap tmL0,
                     const __grid_constant__ CUtensorMap tmL1, const KParams P,
                     const EpiArgs ea0, const EpiArgs ea1) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* outbuf = smem + kPairStages * kPairStageBytes;
    BarsPair* bars = reinterpret_cast<BarsPair*>(outbuf + kOutBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int64_t pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    const int64_t total = P.n_units[0] + (NK > 1 ? P.n_units[1] : 0);
    const uint64_t wait_ns = ea0.wait_ns;
    int* status = ea0.status;
    volatile int* abort = &bars->abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->tfull[b], 1);
            mbar_init(&bars->tempty[b], 8);  // 4 epilogue warps in each CTA
        }
        for (int s = 0; s < kSchedDepth; ++s) {
            mbar_init(&bars->sfull[s], 1);
            // leader: its MMA warp and 4 epilogue warps, the peer's producer
            // and 4 epilogue warps
            mbar_init(&bars->sempty[s], 10);
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
        tmem_alloc_pair(&bars->tmem_base, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_barrier();  // both CTAs' barriers exist before either signals the other's
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    // every consumer of the unit ring arrives on the leader's slot barrier
    auto next_unit = [&](int& sslot, uint32_t& sphase, bool& ok, int& n_lo) -> int {
        if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->sfull[sslot], sphase, wait_ns, abort))) {
            ok = false;
            return -1;
        }
        const int u = *reinterpret_cast<volatile int*>(&bars->sched[sslot]);
        n_lo = *reinterpret_cast<volatile int*>(&bars->sched_lo[sslot]);
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(cluster_addr(&bars->sempty[sslot], 0));
        if (++sslot == kSchedDepth) {
            sslot = 0;
            sphase ^= 1;
        }
        return u;
    };

    if (warp == 0) {
        // ------------------- scheduler (leader) + TMA producer (both CTAs)
        int stage = 0, sslot = 0;
        uint32_t phase = 0, sphase = 0;
        bool ok = true;
        int64_t next_static = pair;
        while (ok) {
            int64_t u;
            int n_lo = 0;
            if (leader) {
                if (P.dynamic) {
                    int got = 0;
                    if (lane == 0) got = atomicAdd(P.counter, 1);
                    u = __shfl_sync(0xffffffffu, got, 0);
                } else {
                    u = next_static;
                    next_static += n_pairs;
                }
                if (u >= total) u = -1;
                n_lo = unit_lo_count(P, u);
                if (!__all_sync(0xffffffffu,
                                mbar_wait_cl(&bars->sempty[sslot], sphase ^ 1, wait_ns, abort))) {
                    ok = false;
                    break;
                }
                if (lane == 0) {  // the slot in both CTAs, then its barrier in both
                    bars->sched[sslot] = static_cast<int>(u);
                    bars->sched_lo[sslot] = n_lo;
                    st_cluster_u32(cluster_addr(&bars->sched[sslot], 1), static_cast<uint32_t>(u));
                    st_cluster_u32(cluster_addr(&bars->sched_lo[sslot], 1),
                                   static_cast<uint32_t>(n_lo));
                    mbar_arrive(&bars->sfull[sslot]);
                    mbar_arrive_cluster(cluster_addr(&bars->sfull[sslot], 1));
                }
                __syncwarp();
                if (++sslot == kSchedDepth) {
                    sslot = 0;
                    sphase ^= 1;
                }
            } else {
                u = next_unit(sslot, sphase, ok, n_lo);
                if (!ok) break;
            }
            if (u < 0) break;
            const Unit un = decode_unit(P, u, n_lo);
            const uint32_t full_cl0 = cluster_addr(&bars->full[0], 0);
            for (int64_t t = un.t0; t < un.t1 && ok; ++t) {
                for (int64_t kb = 0; kb < un.k_blocks; ++kb) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait_cl(&bars->empty[stage], phase ^ 1, wait_ns, abort))) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        uint8_t* sa = smem + stage * kPairStageBytes;
                        const uint32_t bar_cl = full_cl0 + stage * 8u;
                        // the leader expects both CTAs' bytes on its stage barrier
                        if (leader) mbar_arrive_expect_tx(&bars->full[stage], 2 * kPairStageBytes);
                        const int64_t ks = P.k_split[un.kind];
                        const bool lo = ks > 0 && kb >= ks;
                        const int32_t m0 = static_cast<int32_t>(un.mb * 2 * kBM + rank * kBM);
                        const int32_t n0 = static_cast<int32_t>(t * kBN + rank * kBHalf);
                        if (lo && P.lo_cnt[un.kind]) {  // planned second pass
                            int32_t k0;
                            uint32_t bits;
                            lo_block(P, un, kb - ks, &k0, &bits);
                            bits >>= 4 * rank;  // this CTA's half of the pair's pieces
                            if (NK == 1 || un.kind == 0)
                                load_stage_pair_lo<K0::kAmn, K0::kBmn>(sa, &tmL0, &tmB0, bar_cl,
                                                                       k0, m0, n0, bits);
                            else
                                load_stage_pair_lo<K1::kAmn, K1::kBmn>(sa, &tmL1, &tmB1, bar_cl,
                                                                       k0, m0, n0, bits);
                        } else {
                            const int32_t k0 = static_cast<int32_t>((lo ? kb - ks : kb) * kBK);
                            if (NK == 1 || un.kind == 0)
                                load_stage_pair<K0::kAmn, K0::kBmn>(sa, lo ? &tmL0 : &tmA0,
                                                                    &tmB0, bar_cl, k0, m0, n0);
                            else
                                load_stage_pair<K1::kAmn, K1::kBmn>(sa, lo ? &tmL1 : &tmA1,
                                                                    &tmB1, bar_cl, k0, m0, n0);
                        }
                    }
                    __syncwarp();
                    if (++stage == kPairStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
        if (!ok) {
            if (lane == 0) set_status(status, LL_ERR_DEVICE_TIMEOUT);
            bars->abort = 1;
        }
    } else if (warp == 1) {
        // ------------------------------------------- MMA issuer (leader only)
        if (leader) {
            int stage = 0, sslot = 0, buf = 0;
            uint32_t phase = 0, sphase = 0, bphase = 0;
            bool ok = true;
            const uint32_t sbase = smem_u32(smem);
            while (ok) {
                int n_lo = 0;
                const int u = next_unit(sslot, sphase, ok, n_lo);
                if (!ok || u < 0) break;
                const Unit un = decode_unit(P, u, n_lo);
                for (int64_t t = un.t0; t < un.t1 && ok; ++t) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait_cl(&bars->tempty[buf], bphase ^ 1, wait_ns, abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + buf * kBN;
                    for (int64_t kb = 0; kb < un.k_blocks; ++kb) {
                        if (!__all_sync(0xffffffffu,
                                        mbar_wait_cl(&bars->full[stage], phase, wait_ns, abort))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (lane == 0) {
                            const uint32_t sa = sbase + stage * kPairStageBytes;
                            if (NK == 1 || un.kind == 0)
                                mma_stage_pair<K0::kAmn, K0::kBmn, K0::kIdescPair>(d_tmem, sa,
                                                                                   kb == 0);
                            else
                                mma_stage_pair<K1::kAmn, K1::kBmn, K1::kIdescPair>(d_tmem, sa,
                                                                                   kb == 0);
                            tc_commit_pair_both(&bars->empty[stage]);
                        }
                        __syncwarp();
                        if (++stage == kPairStages) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                    if (!ok) break;
                    if (lane == 0) tc_commit_pair_both(&bars->tfull[buf]);
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
            if (lane == 0) tc_commit_pair_local(&bars->drain);
            __syncwarp();
            mbar_wait(&bars->drain, 0, wait_ns, nullptr);
        }
    } else {
        // ------------------------------------------- epilogue (both CTAs)
        const int q = warp & 3;
        const int r_in_tile = q * 32 + lane;
        uint8_t* wbuf = outbuf + q * 2 * kOutBufBytes;
        int sslot = 0, buf = 0, sidx = 0;
        uint32_t sphase = 0, bphase = 0;
        bool ok = true;
        typename K0::Epi epi0;
        typename K1::Epi epi1;
        while (ok) {
            int n_lo = 0;
            const int u = next_unit(sslot, sphase, ok, n_lo);
            if (!ok || u < 0) break;
            const Unit un = decode_unit(P, u, n_lo);
            const int kind = (NK == 1) ? 0 : un.kind;
            const EpiArgs& ea = kind == 0 ? ea0 : ea1;
            const CUtensorMap* tmO = kind == 0 ? &tmO0 : &tmO1;
            const bool out16 = P.out16[kind] != 0;
            const bool reduce = P.reduce[kind] != 0;
            const bool stores = P.out_rows[kind] > 0;
            const int64_t base_row = un.mb * 2 * kBM + rank * kBM;  // this CTA's 128 rows
            const int64_t row0 = base_row + q * 32;
            if (kind == 0)
                epi0.begin_unit(ea, base_row + r_in_tile);
            else
                epi1.begin_unit(ea, base_row + r_in_tile);
            for (int64_t t = un.t0; t < un.t1; ++t) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait_cl(&bars->tfull[buf], bphase, wait_ns, abort))) {
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
                    const int h = out16 ? (c & 1) : 0;
                    const int64_t x0 = out16 ? col0 - 32 * h : col0;  // as in gemm_tc_kernel
                    const bool put = row0 < P.out_rows[kind] && x0 < P.out_cols[kind];
                    uint8_t* sb = wbuf + (sidx & 1) * kOutBufBytes;
                    if (put) {
                        if (h == 0) {
                            if (lane == 0) bulk_wait_read_1();
                            __syncwarp();
                        }
                        stage_row<T>(sb, lane, v, out16, h);
                    }
                    if (kind == 0) {
                        epi0.store_lo(ea, v, col0);
                        epi0.db_partials(ea, v, col0);
                    }
                    if (put && (!out16 || h == 1)) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (reduce)
                                tma_reduce_add_2d(tmO, sb, static_cast<int32_t>(x0),
                                                  static_cast<int32_t>(row0));
                            else
                                tma_store_2d(tmO, sb, static_cast<int32_t>(x0),
                                             static_cast<int32_t>(row0));
                            bulk_commit();
                        }
                        ++sidx;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(cluster_addr(&bars->tempty[buf], 0));
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
    cluster_barrier();  // the leader's MMAs are done with both CTAs' memory
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
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

CUtensorMapDataType map_type(int dtype) {
    return dtype == LL_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                            : dtype == LL_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
}

// 2-D map over a row-major [rows, cols] matrix with row stride `ld`
// elements; box = box_cols x box_rows, 128-byte swizzle, zero fill.
bool make_map(CUtensorMap* map, const void* base, int dtype, int64_t cols, int64_t rows,
              int64_t ld, int box_cols, int box_rows,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int es = dtype == LL_F32 ? 4 : 2;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * es};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols),
                               static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, map_type(dtype), 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// pair = 1: B tiles of a CTA pair's half (128 columns) for a K-major B.
bool operand_maps(const GemmOperands& g, int dtype, CUtensorMap* ma, CUtensorMap* mb,
                  int pair = 0) {
    // K-major operand: [rows, K], box 64(K) x rows; MN-major: [K, MN], box 64 x 64.
    const bool oka = g.a_mn ? make_map(ma, g.A, dtype, g.M, g.K, g.lda, 64, kBK)
                            : make_map(ma, g.A, dtype, g.K, g.M, g.lda, kBK, kBM);
    const bool okb = g.b_mn ? make_map(mb, g.B, dtype, g.N, g.K, g.ldb, 64, kBK)
                            : make_map(mb, g.B, dtype, g.K, g.N, g.ldb, kBK,
                                       pair ? kBHalf : kBN);
    return oka && okb;
}

// Store map of an epilogue output ([rows, cols], row stride ld): boxes of
// 32 rows x 128 bytes.  TMA clips the parts of a box outside [rows, cols].
bool out_map(CUtensorMap* m, const OutDesc& o) {
    if (!o.ptr) {
        memset(m, 0, sizeof(*m));
        return true;
    }
    const int box_cols = o.dtype == LL_F32 ? 32 : 64;
    return make_map(m, o.ptr, o.dtype, o.cols, o.rows, o.ld, box_cols, 32);
}

template <typename T, class K0, class K1, int NK>
cudaError_t launch_k(const CUtensorMap* m, const KParams& P, const EpiArgs& ea0,
                     const EpiArgs& ea1, const DevInfo& dev, int max_ctas, cudaStream_t s) {
    auto kern = gemm_tc_kernel<T, K0, K1, NK>;
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
    kern<<<grid, kThreads, kSmemBytes, s>>>(m[0], m[1], m[2], m[3], m[4], m[5], m[6], m[7], P,
                                            ea0, ea1);
    return cudaGetLastError();
}

// CTA pairs: 2 x pairs CTAs (clusters of two), one pair per two SMs.
template <typename T, class K0, class K1, int NK>
cudaError_t launch_p(const CUtensorMap* m, const KParams& P, const EpiArgs& ea0,
                     const EpiArgs& ea1, const DevInfo& dev, int max_ctas, cudaStream_t s) {
    auto kern = gemm_pair_kernel<T, K0, K1, NK>;
    static int configured[64] = {0};
    if (dev.device < 64 && !configured[dev.device]) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        configured[dev.device] = 1;
    }
    const int64_t units = P.n_units[0] + (NK > 1 ? P.n_units[1] : 0);
    const int cap = ((max_ctas > 0 && max_ctas < dev.num_sms) ? max_ctas : dev.num_sms) / 2;
    int pairs = static_cast<int>(units < cap ? units : cap);
    if (pairs < 1) pairs = 1;
    note_launches(1);
    kern<<<2 * pairs, kThreads, kSmemBytes, s>>>(m[0], m[1], m[2], m[3], m[4], m[5], m[6], m[7],
                                                 P, ea0, ea1);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch(const GemmLaunch& L, const CUtensorMap* m, const KParams& P,
                     const DevInfo& dev, cudaStream_t s, bool pair) {
    using Fwd = Kind<T, EpiKind::Fwd, false, false>;
    using Rec = Kind<T, EpiKind::Recomp, false, false>;
    using Dh = Kind<T, EpiKind::Dh, false, true>;
    using Dw = Kind<T, EpiKind::Dw, true, false>;  // B = h^T, K-major
    const int mc = L.max_ctas;
    if (L.nkinds == 1) {
        switch (L.kind[0]) {
            case EpiKind::Fwd:
                return pair ? launch_p<T, Fwd, Fwd, 1>(m, P, L.ea[0], L.ea[0], dev, mc, s)
                            : launch_k<T, Fwd, Fwd, 1>(m, P, L.ea[0], L.ea[0], dev, mc, s);
            case EpiKind::Recomp:
                return pair ? launch_p<T, Rec, Rec, 1>(m, P, L.ea[0], L.ea[0], dev, mc, s)
                            : launch_k<T, Rec, Rec, 1>(m, P, L.ea[0], L.ea[0], dev, mc, s);
            case EpiKind::Dh:
                return pair ? launch_p<T, Dh, Dh, 1>(m, P, L.ea[0], L.ea[0], dev, mc, s)
                            : launch_k<T, Dh, Dh, 1>(m, P, L.ea[0], L.ea[0], dev, mc, s);
            case EpiKind::Dw:
                return pair ? launch_p<T, Dw, Dw, 1>(m, P, L.ea[0], L.ea[0], dev, mc, s)
                            : launch_k<T, Dw, Dw, 1>(m, P, L.ea[0], L.ea[0], dev, mc, s);
        }
    } else if (L.kind[0] == EpiKind::Dh && L.kind[1] == EpiKind::Dw) {
        return pair ? launch_p<T, Dh, Dw, 2>(m, P, L.ea[0], L.ea[1], dev, mc, s)
                    : launch_k<T, Dh, Dw, 2>(m, P, L.ea[0], L.ea[1], dev, mc, s);
    }
    return cudaErrorInvalidValue;
}

// 16-bit operands on CTA pairs (gemm_pair_kernel) for problems of >= 256 rows.
constexpr bool kUsePairs = true;

// FP32 operand maps: K-major [rows, K] box 16(K) x rows, 64-byte swizzle;
// MN-major [K, MN] box 32 x 16, 128-byte swizzle.
bool operand_maps_f32(const GemmOperands& g, CUtensorMap* ma, CUtensorMap* mb) {
    const bool oka = g.a_mn ? make_map(ma, g.A, LL_F32, g.M, g.K, g.lda, 32, kBKf)
                            : make_map(ma, g.A, LL_F32, g.K, g.M, g.lda, kBKf, kBM,
                                       CU_TENSOR_MAP_SWIZZLE_64B);
    const bool okb = g.b_mn ? make_map(mb, g.B, LL_F32, g.N, g.K, g.ldb, 32, kBKf)
                            : make_map(mb, g.B, LL_F32, g.K, g.N, g.ldb, kBKf, kBN,
                                       CU_TENSOR_MAP_SWIZZLE_64B);
    return oka && okb;
}

}  // namespace

bool gemm_uses_pairs(int dtype, const int64_t* Ms, int nkinds) {
    bool pair = dtype != LL_F32 && kUsePairs;
    for (int k = 0; k < nkinds; ++k) pair = pair && Ms[k] >= 2 * kBM;
    return pair;
}

cudaError_t launch_gemm(const GemmLaunch& L, const DevInfo& dev, cudaStream_t s) {
    CUtensorMap m[8];  // A, B, out of kind 0; of kind 1; A_lo of kind 0, 1
    memset(m, 0, sizeof(m));
    KParams P;
    memset(&P, 0, sizeof(P));
    GemmLaunch G = L;
    // 16-bit operands run on CTA pairs (256 x 256 tiles) when every kind has
    // at least 256 rows; smaller problems keep the single-CTA kernel
    int64_t Ms[2] = {G.op[0].M, G.nkinds > 1 ? G.op[1].M : 0};
    const bool pair = gemm_uses_pairs(G.dtype, Ms, G.nkinds);
    for (int k = 0; k < G.nkinds; ++k) {
        const bool okm = G.dtype == LL_F32
                             ? operand_maps_f32(G.op[k], &m[3 * k], &m[3 * k + 1])
                             : operand_maps(G.op[k], G.dtype, &m[3 * k], &m[3 * k + 1], pair);
        if (!okm) return cudaErrorInvalidValue;
        if (!out_map(&m[3 * k + 2], G.out[k])) return cudaErrorInvalidValue;
        P.sh[k] = G.shape[k];
        if (pair) P.sh[k].m_blocks = (G.op[k].M + 2 * kBM - 1) / (2 * kBM);
        {   // grouped order: as many row blocks of A per group as fit kGroupBytes
            const int64_t blk = (pair ? 2 * kBM : kBM) * G.op[k].K * (G.dtype == LL_F32 ? 4 : 2);
            const int64_t gm = kGroupBytes / (blk > 0 ? blk : 1);
            P.sh[k].group_m = gm < 4 ? 4 : (gm > kGroupM ? kGroupM : gm);
        }
        // the host sizes K blocks for the 16-bit kernel (64 values); the
        // tf32 kernel takes 16 per stage
        if (G.dtype == LL_F32) P.sh[k].k_blocks = (G.op[k].K + kBKf - 1) / kBKf;
        if (G.op[k].A_lo) {  // hi / lo split: A_lo after A along K
            if (G.dtype == LL_F32) return cudaErrorInvalidValue;
            const GemmOperands& g = G.op[k];
            P.k_split[k] = P.sh[k].k_blocks;
            if (g.lo_cnt) {
                // planned second pass: A_lo read in 32-row pieces
                const bool ok = g.a_mn ? make_map(&m[6 + k], g.A_lo, G.dtype, g.M, g.K, g.lda,
                                                  64, 32)
                                       : make_map(&m[6 + k], g.A_lo, G.dtype, g.K, g.M, g.lda,
                                                  kBK, 32);
                if (!ok) return cudaErrorInvalidValue;
                P.lo_cnt[k] = g.lo_cnt;
                P.lo_idx[k] = g.lo_idx;
                P.lo_ld[k] = g.lo_ld;
            } else {
                GemmOperands lo = g;
                lo.A = lo.A_lo;
                CUtensorMap unused;
                if (!operand_maps(lo, G.dtype, &m[6 + k], &unused, pair))
                    return cudaErrorInvalidValue;
                P.sh[k].k_blocks *= 2;
            }
        }
        if (P.sh[k].k_splits > 1) {  // FP32 grad_hidden only: units per K part
            if (G.dtype != LL_F32 || G.kind[k] != EpiKind::Dh || P.sh[k].tiles_per_unit != 1 ||
                !G.ea[k].dh_part || G.out[k].rows != P.sh[k].k_splits * P.sh[k].m_blocks * kBM)
                return cudaErrorInvalidValue;
            P.sh[k].n_segs = P.sh[k].n_tiles * P.sh[k].k_splits;
            P.part_rows[k] = P.sh[k].m_blocks * kBM;
        }
        P.n_units[k] = P.sh[k].m_blocks * P.sh[k].n_segs;
        P.out16[k] = G.out[k].dtype != LL_F32;
        P.out_rows[k] = G.out[k].rows;
        P.out_cols[k] = G.out[k].cols;
        if (G.kind[k] == EpiKind::Dw && !G.ea[k].first_chunk) {
            // later token chunks: an FP32 table is updated by the store's
            // reduce-add; a 16-bit table is read, added in FP32 and rounded
            P.reduce[k] = !P.out16[k];
            G.ea[k].dw_add_prev = P.out16[k];
        }
    }
    if (G.nkinds == 1) {
        m[3] = m[0];
        m[4] = m[1];
        m[5] = m[2];
        m[7] = m[6];
        P.k_split[1] = P.k_split[0];
        P.lo_cnt[1] = P.lo_cnt[0];
        P.lo_idx[1] = P.lo_idx[0];
        P.lo_ld[1] = P.lo_ld[0];
        P.part_rows[1] = P.part_rows[0];
    }
    P.dynamic = G.counter != nullptr;
    P.counter = G.counter;
    P.zero_counter = G.zero_counter;
    if (G.dtype == LL_F32) return dispatch_f32(G, m, P, dev, s);
    if (G.dtype == LL_BF16) return dispatch<__nv_bfloat16>(G, m, P, dev, s, pair);
    return dispatch<__half>(G, m, P, dev, s, pair);
}

}  // namespace ll
