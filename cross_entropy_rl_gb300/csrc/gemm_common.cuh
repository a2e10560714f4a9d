// Shared pieces of the tensor-core GEMM kernels: tile and stage geometry,
// the launch parameters, the unit decoding of the persistent schedulers, the
// operand kinds, TMA bulk stores and the epilogue's row staging.  Included by
// gemm_tc.cu (16-bit operands: single CTAs and CTA pairs, and the host side
// of every launch) and gemm_tf32.cu (FP32 operands).
#pragma once
#include <string.h>

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
constexpr int kSchedDepth = 4;
constexpr int kOutBufBytes = 32 * 128;  // one warp's 32 rows x 128 bytes
constexpr int kOutBytes = 4 * 2 * kOutBufBytes;
constexpr int kSmemBytes = kStages * kStageBytes + kOutBytes + 1024 /*align*/ + 512 /*bars*/;

constexpr int kBKf = 16;                       // K values per stage

struct Bars {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t sfull[kSchedDepth];
    uint64_t sempty[kSchedDepth];
    uint64_t drain;
    int sched[kSchedDepth];
    int sched_lo[kSchedDepth];  // second-pass K blocks of the unit in sched
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

}  // namespace

// Launch-wide parameters (by value).
struct KParams {
    GemmShape sh[2];
    int64_t n_units[2];  // units of kind 0, then kind 1
    int dynamic;         // 1: units handed out by an atomic counter
    int* counter;        // zero before the launch when dynamic
    int* zero_counter;   // if set, CTA 0 zeroes it (for the next launch)
    int out16[2];        // output element of the kind is 16-bit
    int reduce[2];       // TMA reduce-add instead of store
    int64_t out_rows[2], out_cols[2];
    int64_t k_split[2];  // 16-bit: K blocks from the first A map; later blocks read the
                         // second A map (A_lo) at K block kb - k_split (0 = one A)
    // planned second pass (automatic split): lo_cnt[kind][mb] K blocks of A_lo
    // after the first pass, the j-th being lo_idx[kind][mb * lo_ld + j] =
    // (K block << 8 | bits of the written pieces); nullptr = whole second pass
    const int* lo_cnt[2];
    const int64_t* lo_idx[2];
    int64_t lo_ld[2];
    int64_t part_rows[2];  // K split: rows between two parts' partial sums
};

namespace {

// ----------------------------------------------------------- bulk stores
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x,
                                             int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, const void* src,
                                                  int32_t x, int32_t y) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group"
        " [%0, {%2, %3}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

struct Unit {
    int kind;
    int64_t mb, seg, t0, t1, k_blocks;
    int64_t k_begin, kpart;  // K split: first K block and part index of the unit
};

// n_lo: K blocks of the unit's planned second pass (0 without a plan); the
// scheduler reads it once from the plan and publishes it with the unit id.
__device__ __forceinline__ Unit decode_unit(const KParams& P, int64_t u, int n_lo = 0) {
    Unit r;
    r.kind = u < P.n_units[0] ? 0 : 1;
    const GemmShape& sh = P.sh[r.kind];
    const int64_t v = r.kind ? u - P.n_units[0] : u;
    if (sh.unit_order == 0) {
        r.seg = v / sh.m_blocks;
        r.mb = v % sh.m_blocks;
    } else if (sh.unit_order == 1) {
        r.mb = v / sh.n_segs;
        r.seg = v % sh.n_segs;
    } else {
        const int64_t G = sh.group_m;
        const int64_t per_group = G * sh.n_segs;
        const int64_t g = v / per_group;
        const int64_t in_g = v % per_group;
        const int64_t gm = min(G, sh.m_blocks - g * G);
        r.seg = in_g / gm;
        r.mb = g * G + in_g % gm;
    }
    r.k_begin = 0;
    r.kpart = 0;
    int64_t kb_total = sh.k_blocks;
    if (sh.k_splits > 1) {  // seg = tile * k_splits + part
        r.kpart = r.seg % sh.k_splits;
        r.seg /= sh.k_splits;
        const int64_t per = (kb_total + sh.k_splits - 1) / sh.k_splits;
        r.k_begin = r.kpart * per;
        kb_total = min(per, kb_total - r.k_begin);
    }
    r.t0 = r.seg * sh.tiles_per_unit;
    r.t1 = min(r.t0 + sh.tiles_per_unit, sh.n_tiles);
    r.k_blocks = kb_total + n_lo;
    return r;
}

// The planned second pass's K-block count of unit u (scheduler side).
__device__ __forceinline__ int unit_lo_count(const KParams& P, int64_t u) {
    if (u < 0) return 0;
    const Unit r = decode_unit(P, u);
    return P.lo_cnt[r.kind] ? P.lo_cnt[r.kind][r.mb] : 0;
}

// The planned second pass's K block (scaled to elements) and piece bits.
__device__ __forceinline__ void lo_block(const KParams& P, const Unit& un, int64_t j,
                                         int32_t* k0, uint32_t* bits) {
    const int64_t e = P.lo_idx[un.kind][un.mb * P.lo_ld[un.kind] + j];
    *k0 = static_cast<int32_t>((e >> 8) * kBK);
    *bits = static_cast<uint32_t>(e & 0xff);
}

// A_lo of the planned second pass in pieces of 32 rows (K-major A: 4 per
// 128-row tile) or of 32 K rows (MN-major A: 2 in each 64-wide box): a piece
// whose bit is set is read from A_lo, any other from rows [-32, 0), outside
// the tensor, which the copy fills with zeros.  Same bytes and shared-memory
// layout as the whole-tile load (a 32-row piece is 4 KB, a multiple of the
// 1 KB swizzle pattern).  `load(dst, x, y)` issues one piece.
template <bool A_MN, class Load>
__device__ __forceinline__ void load_a_pieces(uint8_t* sa, int32_t k0, int32_t m0,
                                              uint32_t bits, Load load) {
    if constexpr (!A_MN) {
#pragma unroll
        for (int i = 0; i < kBM / 32; ++i)
            load(sa + i * 32 * 128, k0, ((bits >> i) & 1) ? m0 + 32 * i : -32);
    } else {
#pragma unroll
        for (int j = 0; j < kBM / 64; ++j)
#pragma unroll
            for (int i = 0; i < 2; ++i)
                load(sa + j * kMnBoxBytes + i * 32 * 128, m0 + 64 * j,
                     ((bits >> (2 * j + i)) & 1) ? k0 + 32 * i : -32);
    }
}

template <typename T, EpiKind E, bool A_MN, bool B_MN>
struct Kind {
    using Epi = RowEpilogue<E, T>;
    static constexpr bool kAmn = A_MN, kBmn = B_MN;
    static constexpr int kFmt = std::is_same<T, __half>::value   ? 0
                                : std::is_same<T, float>::value ? 2  // tf32
                                                                : 1;
    static constexpr uint32_t kIdesc = instr_desc(kFmt, A_MN, B_MN, kBM, kBN);
    static constexpr uint32_t kIdescPair = instr_desc(kFmt, A_MN, B_MN, 2 * kBM, kBN);
};

template <bool A_MN, bool B_MN>
__device__ __forceinline__ void load_stage(uint8_t* sa, const CUtensorMap* tmA,
                                           const CUtensorMap* tmB, uint64_t* fb, int32_t k0,
                                           int32_t m0, int32_t n0) {
    uint8_t* sb = sa + kABytes;
    mbar_arrive_expect_tx(fb, kStageBytes);
    if constexpr (!A_MN) {
        tma_load_2d(sa, tmA, fb, k0, m0);
    } else {
#pragma unroll
        for (int j = 0; j < kBM / 64; ++j) tma_load_2d(sa + j * kMnBoxBytes, tmA, fb, m0 + 64 * j, k0);
    }
    if constexpr (!B_MN) {
        tma_load_2d(sb, tmB, fb, k0, n0);
    } else {
#pragma unroll
        for (int j = 0; j < kBN / 64; ++j) tma_load_2d(sb + j * kMnBoxBytes, tmB, fb, n0 + 64 * j, k0);
    }
}

template <bool A_MN, bool B_MN>
__device__ __forceinline__ void load_stage_lo(uint8_t* sa, const CUtensorMap* tmL,
                                              const CUtensorMap* tmB, uint64_t* fb, int32_t k0,
                                              int32_t m0, int32_t n0, uint32_t bits) {
    uint8_t* sb = sa + kABytes;
    mbar_arrive_expect_tx(fb, kStageBytes);
    load_a_pieces<A_MN>(sa, k0, m0, bits, [&](uint8_t* d, int32_t x, int32_t y) {
        tma_load_2d(d, tmL, fb, x, y);
    });
    if constexpr (!B_MN) {
        tma_load_2d(sb, tmB, fb, k0, n0);
    } else {
#pragma unroll
        for (int j = 0; j < kBN / 64; ++j) tma_load_2d(sb + j * kMnBoxBytes, tmB, fb, n0 + 64 * j, k0);
    }
}

template <bool A_MN, bool B_MN, uint32_t IDESC>
__device__ __forceinline__ void mma_stage(uint32_t d_tmem, uint32_t sa, bool first) {
    const uint32_t sb = sa + kABytes;
#pragma unroll
    for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint64_t ad = A_MN ? smem_desc_sw128(sa + kk * 2048, kMnBoxBytes, 1024)
                                 : smem_desc_sw128(sa + kk * 32, 16, 1024);
        const uint64_t bd = B_MN ? smem_desc_sw128(sb + kk * 2048, kMnBoxBytes, 1024)
                                 : smem_desc_sw128(sb + kk * 32, 16, 1024);
        tc_mma<0>(d_tmem, ad, bd, IDESC, (!first || kk > 0) ? 1u : 0u);
    }
}

// Stage 32 values of this thread's row into the warp's swizzled buffer
// (32 rows x 128 bytes, 16-byte chunk c of row r at chunk c ^ (r & 7), the
// layout of a 128-byte-swizzled TMA box): fp32 fills the whole row; 16-bit
// fills half `h` of it.
template <typename T>
__device__ __forceinline__ void stage_row(uint8_t* buf, int lane, const float (&v)[32], bool out16,
                                          int h) {
    uint8_t* rowp = buf + lane * 128;
    const int sw = lane & 7;
    if (!out16) {
#pragma unroll
        for (int sl = 0; sl < 8; ++sl)
            *reinterpret_cast<float4*>(rowp + ((sl ^ sw) << 4)) =
                make_float4(v[4 * sl], v[4 * sl + 1], v[4 * sl + 2], v[4 * sl + 3]);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint4 u;
            T* e = reinterpret_cast<T*>(&u);
#pragma unroll
            for (int j = 0; j < 8; ++j) e[j] = Elem<T>::from_f(v[8 * k + j]);
            *reinterpret_cast<uint4*>(rowp + (((4 * h + k) ^ sw) << 4)) = u;
        }
    }
}

}  // namespace

// FP32 operands (gemm_tf32.cu): launches the tf32 kernel for a built launch.
cudaError_t dispatch_f32(const GemmLaunch& L, const CUtensorMap* m, const KParams& P,
                         const DevInfo& dev, cudaStream_t s);

}  // namespace ll
