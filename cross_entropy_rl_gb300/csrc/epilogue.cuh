// Fused GEMM epilogues of the linear log-probability path.
//
// Each epilogue thread owns one row of the output tile (one TMEM lane on the
// tensor-core path) and sees that row in chunks of 32 consecutive columns.
// The four kinds:
//
//   Fwd     z = h W^T (+b) tile -> running max / rescaled sum-exp of the row
//           over the vocab tiles of one segment (online softmax), target
//           logit picked up when it falls in the tile.  Per-segment partials
//           are merged afterwards in ascending segment order.
//   Recomp  the same z tile recomputed -> p = exp(z - lse); stores the
//           off-target part of g, S[n, v] = -grad_logp * p (S = 0 at the
//           target), to the chunk workspace, and the FP32 target entry
//           c[n] = grad_logp * (1 - p[n, y]) to a per-token array.
//   Dh      acc = S . W tile -> adds c[n] * W[y] in FP32, stores grad_hidden.
//   Dw      acc = S^T . h tile -> on the first token chunk 0 + acc (a +0
//           start), on later chunks the running grad_weight is added (here,
//           or by the TMA reduce-add of the store); on the last chunk the
//           target part sum over tokens with target v of c[n] * h[n] is
//           added in ascending token order.
//
// g = grad_logp * (onehot - p) is split into its target column, kept exact
// in FP32 (c), and the off-target entries S, stored in 16 bits.  The 16-bit
// rounding then only touches the entries -grad * p[n, v], v != y, whose sum
// over v is grad * (1 - p[n, y]); a sharp distribution (p[n, y] -> 1) makes
// that error vanish instead of leaving a 2^-9 * |grad| error at the target.
// Zero rules (issue #261, "Correctness boundary"): rows with an invalid
// target or a zero upstream gradient store exact +0; sums start from +0.
// In a vocab shard (ea.shard) a row whose target lies in another shard keeps
// its softmax part and has no target column here.
#pragma once
#include "ll_device.cuh"

namespace ll {

// Storage tag that selects T in the run-time-typed loads and stores below.
template <typename T>
constexpr int own_tag() { return sizeof(T) == 4 ? LL_F32 : LL_BF16; }

template <typename T>
__device__ __forceinline__ float ld_elem(const void* p, int64_t i) {
    return Elem<T>::to_f(static_cast<const T*>(p)[i]);
}

// Store 32 values to p[0..31] (16-byte aligned), dtype chosen at run time
// (LL_F32 or the 16-bit type T); only 8-element groups below `limit`.
template <typename T>
__device__ __forceinline__ void store_row32(void* base, int64_t idx, const float (&v)[32],
                                            int64_t col0, int64_t limit, int out_dtype) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (col0 + 8 * g >= limit) break;
        float f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = v[8 * g + j];
        if (out_dtype == LL_F32)
            store8(static_cast<float*>(base) + idx + 8 * g, f);
        else
            store8(static_cast<T*>(base) + idx + 8 * g, f);
    }
}

template <typename T>
__device__ __forceinline__ void load_row32(const void* base, int64_t idx, float (&v)[32],
                                           int64_t col0, int64_t limit, int in_dtype) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (col0 + 8 * g < limit) {
            if (in_dtype == LL_F32)
                load8(static_cast<const float*>(base) + idx + 8 * g, f);
            else
                load8(static_cast<const T*>(base) + idx + 8 * g, f);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) v[8 * g + j] = f[j];
    }
}

template <EpiKind E, typename T>
struct RowEpilogue {
    int64_t row;   // row in the M dimension of the launch
    bool rvalid;
    int64_t y;
    float coef;    // Recomp: -grad / T (0 for dead rows); Dh: c[row] (0 for dead rows)
    bool live;     // Recomp / Dh: valid target and non-zero upstream gradient
    bool onehot;   // Dh: the target column lies in this launch's vocab
    float lse2;    // Recomp: lse * log2(e)
    float m2, s;   // Fwd: running max (log2 units) and sum
    float zyv;
    bool found;
    int oh_beg, oh_end;  // Dw: one-hot token range in the sorted key list
    float lo_prev[32];   // Recomp, automatic split: the rest of the even chunk of a piece
    bool lo_any_prev;
    uint32_t lo_keep;    // Recomp, automatic split: entries of the chunk with p >= kLoTau

    __device__ __forceinline__ void begin_unit(const EpiArgs& ea, int64_t row_) {
        row = row_;
        rvalid = row < ea.M;
        if constexpr (E == EpiKind::Fwd) {
            m2 = -INFINITY;
            s = 0.f;
            found = false;
            zyv = 0.f;
            y = rvalid ? ea.targets[row] : -1;
        } else if constexpr (E == EpiKind::Recomp || E == EpiKind::Dh) {
            y = rvalid ? ea.targets[row] : -1;
            const float g = rvalid ? ea.grad[row] : 0.f;
            const bool here = y >= 0 && y < ea.V;
            live = rvalid && (here || (ea.shard && y == kTargetInOtherShard)) && g != 0.f;
            onehot = live && here;
            if constexpr (E == EpiKind::Recomp)
                coef = live ? -g * ea.inv_temp : 0.f;  // d(z / T)/dz = 1 / T
            else
                coef = onehot ? ea.tc[row] : 0.f;
            if constexpr (E == EpiKind::Recomp) lse2 = rvalid ? ea.lse[row] * kLog2e : 0.f;
        } else {  // Dw: row is a vocab index
            oh_beg = oh_end = 0;
            if (ea.last_chunk && rvalid) {
                oh_beg = ea.offs[row];
                oh_end = ea.offs[row + 1];
            }
        }
    }

    __device__ __forceinline__ void chunk(const EpiArgs& ea, float (&v)[32], int64_t col0) {
        if constexpr (E == EpiKind::Fwd || E == EpiKind::Recomp) {
            const int64_t V = ea.Ncols;
            if (ea.bias) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (col0 + j < V) v[j] += ld_elem<T>(ea.bias, col0 + j);
            }
            if (ea.inv_temp != 1.f) {  // the tempered logits z / T
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] *= ea.inv_temp;
            }
            if constexpr (E == EpiKind::Fwd) {
                if (ea.z_only) return;  // logits stored; the fold runs as its own kernel
                if (col0 + 32 > V) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + j >= V) v[j] = -INFINITY;
                }
                const int64_t off = y - col0;
                if (off >= 0 && off < 32) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j == off) zyv = v[j];
                    found = true;
                }
                float cmax = v[0];
#pragma unroll
                for (int j = 1; j < 32; ++j) cmax = fmaxf(cmax, v[j]);
                const float mu = cmax * kLog2e;
                if (mu > m2) {
                    s = s * ex2(m2 - mu);
                    m2 = mu;
                }
                if (m2 != -INFINITY) {
                    float acc = 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) acc += ex2(fmaf(v[j], kLog2e, -m2));
                    s += acc;
                }
            } else {  // Recomp: S = -grad * exp(z - lse), target entry apart
                lo_keep = 0;
                if (!rvalid) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.f;
                    return;
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = ex2(fmaf(v[j], kLog2e, -lse2));
                const int64_t off = y - col0;
                if (off >= 0 && off < 32) {
                    float py = 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j == off) py = v[j];
                    // -coef = grad for live rows, 0 otherwise
                    ea.tc[row] = coef != 0.f ? -coef * (1.f - py) : 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j == off) v[j] = 0.f;
                }
                if (ea.lo_flags && coef != 0.f) {  // automatic split: which rests to keep
                    if (max32(v) >= kLoTau) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + j < V && v[j] >= kLoTau) lo_keep |= 1u << j;
                    }
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = coef * v[j];
            }
        } else if constexpr (E == EpiKind::Dh) {
            if (!rvalid || ea.dh_part) return;  // a K part: stored as summed
            const int64_t D = ea.Ncols;
            if (onehot) {
                float w[32];
                load_row32<T>(ea.W, y * ea.ldW + col0, w, col0, D, own_tag<T>());
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = fmaf(coef, w[j], v[j]) + 0.f;
            } else if (live) {  // target in another vocab shard: softmax part only
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = v[j] + 0.f;
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
        } else {  // Dw
            if (!rvalid) return;
            const int64_t D = ea.Ncols;
            if (ea.first_chunk) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f + v[j];
            } else if (ea.dw_add_prev) {
                float prev[32];
                load_row32<T>(ea.out, row * ea.ld_out + col0, prev, col0, D, ea.out_dtype);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = prev[j] + v[j];
            }
            for (int i = oh_beg; i < oh_end; ++i) {
                const int64_t n = static_cast<int64_t>(ea.keys[i] & 0xffffffffll);
                const float g = ea.tc_all[n];
                if (g == 0.f) continue;
                float hv[32];
                load_row32<T>(ea.h_all, n * ea.ld_h + col0, hv, col0, D, own_tag<T>());
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = fmaf(g, hv[j], v[j]);
            }
        }
    }

    // grad_bias partials of the recompute: the sums over this warp's 32 rows
    // of each of the chunk's 32 columns of S (off-target entries, FP32, rows
    // outside the problem count 0), by a fixed butterfly over the lanes: at
    // each step a lane keeps the half of its columns selected by its lane
    // bit and adds the partner's copy of that half; lane l ends with the sum
    // of column l.  Written to db_part[row / 32][col].  All 32 lanes of the
    // warp must call it (consecutive rows); v is consumed.
    __device__ __forceinline__ void db_partials(const EpiArgs& ea, float (&v)[32],
                                                int64_t col0) {
        if constexpr (E == EpiKind::Recomp) {
            if (!ea.db_part) return;
            const int lane = threadIdx.x & 31;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const bool up = (lane & off) != 0;
#pragma unroll
                for (int j = 0; j < off; ++j) {
                    const float keep = up ? v[j + off] : v[j];
                    const float send = up ? v[j] : v[j + off];
                    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            const int64_t col = col0 + lane;
            // warps whose 32 rows all lie past the problem write nothing, so
            // partial rows stay within ceil(M / 32)
            if (col < ea.Ncols && (row & ~int64_t(31)) < ea.M)
                ea.db_part[(row >> 5) * ea.Ncols + col] = v[0];
        }
    }

    // Recomp with a hi / lo split of S: S_lo = S - S_hi, S_hi being S rounded
    // to T (what the tile store writes), in direct row stores.  The two 16-bit
    // parts carry S to ~2^-17 relative instead of 2^-9.
    // Automatic split (ea.lo_flags): only entries with p >= kLoTau (marked by
    // chunk()) keep their rest, the others count 0, so a row's S_lo depends
    // on that row alone.  The rests are written in pieces of 32 rows (this
    // warp) x 64 columns (an even and the following odd chunk): a piece
    // holding any kept entry is written whole (zeros included), and every
    // piece's flag is set to whether it was written (no clearing needed).
    // All 32 lanes of the warp call it for every chunk of the tile in order.
    __device__ __forceinline__ void store_lo(const EpiArgs& ea, const float (&v)[32],
                                             int64_t col0) {
        if constexpr (E == EpiKind::Recomp && sizeof(T) == 2) {
            if (!ea.S_lo) return;
            if (!ea.lo_flags) {
                if (!rvalid) return;
                float lo[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) lo[j] = v[j] - Elem<T>::to_f(Elem<T>::from_f(v[j]));
                store_row32<T>(ea.S_lo, row * ea.ldS + col0, lo, col0, ea.Ncols, own_tag<T>());
                return;
            }
            const bool any = __any_sync(0xffffffffu, lo_keep != 0);
            const bool even = ((col0 / 32) & 1) == 0;
            if (any) {  // the kept entries' rests, zeros elsewhere
                float* dst = even ? lo_prev : nullptr;
                float lo[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    lo[j] = ((lo_keep >> j) & 1) ? v[j] - Elem<T>::to_f(Elem<T>::from_f(v[j]))
                                                 : 0.f;
                if (dst) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) lo_prev[j] = lo[j];
                } else if (rvalid) {
                    store_row32<T>(ea.S_lo, row * ea.ldS + col0, lo, col0, ea.Ncols,
                                   own_tag<T>());
                }
            }
            if (even) {
                lo_any_prev = any;
                return;
            }
            // odd chunk: the piece [col0 - 32, col0 + 32) is complete
            const bool written = any || lo_any_prev;
            if (written && rvalid) {
                float z[32];
                if (!lo_any_prev) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) z[j] = 0.f;
                }
                store_row32<T>(ea.S_lo, row * ea.ldS + col0 - 32, lo_any_prev ? lo_prev : z,
                               col0 - 32, ea.Ncols, own_tag<T>());
                if (!any) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) z[j] = 0.f;
                    store_row32<T>(ea.S_lo, row * ea.ldS + col0, z, col0, ea.Ncols,
                                   own_tag<T>());
                }
            }
            const int64_t piece = (col0 - 32) / kLoCols;
            if ((threadIdx.x & 31) == 0 && rvalid && piece < ea.lo_flags_cols)
                ea.lo_flags[(row / kLoRows) * ea.lo_flags_ld + piece] = written ? 1 : 0;
        }
    }

    __device__ __forceinline__ void end_unit(const EpiArgs& ea, int64_t seg) {
        if constexpr (E == EpiKind::Fwd) {
            if (!rvalid || ea.z_only) return;
            ea.part_m[seg * ea.part_ld + row] = m2;
            ea.part_s[seg * ea.part_ld + row] = s;
            if (found) ea.zy[row] = zyv;
        }
    }
};

}  // namespace ll
