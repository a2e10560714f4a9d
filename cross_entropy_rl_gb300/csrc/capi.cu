// C ABI of the fused linear log-probability library: argument validation,
// device guard, workspace layout and the launch sequence of each call.
// Declarations and the contract of every entry point: ll_linear_logp.h.
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "ll_internal.h"

namespace ll {

__device__ int g_ll_status;  // first device-side error since the last check

static uint64_t g_wait_limit_ns = 2000000000ull;
uint64_t wait_limit_ns() { return g_wait_limit_ns; }

static std::atomic<long long> g_launches{0};
void note_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// ------------------------------------------------------------------ tracing
// When enabled, every phase of a call is bracketed by CUDA events recorded
// on the call's stream; ll_profile_summary() aggregates them per phase.
namespace {
struct ProfRec {
    const char* label;
    cudaEvent_t a, b;
};
std::atomic<int> g_prof_on{0};
std::mutex g_prof_mu;
std::vector<ProfRec> g_prof;

struct Phase {
    const char* label;
    cudaStream_t s;
    cudaEvent_t a = nullptr, b = nullptr;
    Phase(const char* l, cudaStream_t st) : label(l), s(st) {
        if (!g_prof_on.load()) return;
        if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) {
            a = b = nullptr;
            return;
        }
        cudaEventRecord(a, s);
    }
    ~Phase() {
        if (!a) return;
        cudaEventRecord(b, s);
        std::lock_guard<std::mutex> lk(g_prof_mu);
        g_prof.push_back({label, a, b});
    }
};
}  // namespace

namespace {

constexpr size_t kAlign = 256;
constexpr int kSideSms = 2;  // SMs left to the side stream during an overlapped GEMM

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }
size_t esize(int dtype) { return dtype == LL_F32 ? 4 : 2; }
bool dtype_ok(int dt) { return dt == LL_F32 || dt == LL_F16 || dt == LL_BF16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

struct DevCache {
    bool ready = false;
    int num_sms = 0;
    int* status = nullptr;
    int cc_major = 0, cc_minor = 0;
    cudaStream_t side = nullptr;  // side stream for work that overlaps a GEMM
};
DevCache g_dev[64];
std::mutex g_dev_mu;

// Switches to the device owning `ptr` for the lifetime of the guard.
struct DeviceGuard {
    int prev = -1;
    int dev = -1;
    int err = LL_OK;
    explicit DeviceGuard(const void* ptr) {
        cudaPointerAttributes attr;
        if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
            cudaGetLastError();
            err = LL_ERR_INVALID_ARG;
            return;
        }
        if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) {
            err = LL_ERR_INVALID_ARG;
            return;
        }
        dev = attr.device;
        if (dev < 0 || dev >= 64) {
            err = LL_ERR_INVALID_ARG;
            return;
        }
        if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) {
            err = LL_ERR_CUDA;
            return;
        }
    }
    ~DeviceGuard() {
        if (prev >= 0 && prev != dev) cudaSetDevice(prev);
    }
};

int device_info(int dev, DevInfo* out) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevCache& c = g_dev[dev];
    if (!c.ready) {
        if (cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return LL_ERR_CUDA;
        cudaDeviceGetAttribute(&c.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&c.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ll_status) != cudaSuccess) {
            cudaGetLastError();
            return LL_ERR_UNSUPPORTED;
        }
        c.status = static_cast<int*>(p);
        if (cudaStreamCreateWithFlags(&c.side, cudaStreamNonBlocking) != cudaSuccess) {
            cudaGetLastError();
            c.side = nullptr;
        }
        c.ready = true;
    }
    if (!(c.cc_major == 10 && c.cc_minor == 3)) return LL_ERR_UNSUPPORTED;
    out->device = dev;
    out->num_sms = c.num_sms;
    out->status = c.status;
    out->side = c.side;
    return LL_OK;
}

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return LL_OK;
    fprintf(stderr, "ll: CUDA error %s\n", cudaGetErrorString(e));
    return LL_ERR_CUDA;
}

// ---------------------------------------------------------------- layouts
// A small forward (fewer than 128 units of 128 rows x one 1024-column
// segment, its FP32 logits within 4 MiB) runs its GEMM one vocab tile per
// unit, so that its few segments spread over 4x as many SMs, and stores the
// logits; fwd_fold_kernel then forms the partials with the epilogue's own
// arithmetic (bitwise the fused epilogue's).  Depends on (N, V) only.
bool fwd_z_only(int64_t N, int64_t V) {
    const int64_t units = cdiv(N, kBM) * cdiv(cdiv(V, kBN), kVocabTilesPerSeg);
    return N > 0 && units < 128 && size_t(N) * size_t(round_up(V, 8)) * 4 <= (size_t(4) << 20);
}

struct FwdLayout {
    int64_t n_segs, ldZ;
    bool z_only;
    size_t part_m, part_s, zy, Z, total;
};
FwdLayout fwd_layout(int64_t N, int64_t V) {
    FwdLayout L;
    L.n_segs = cdiv(cdiv(V, kBN), kVocabTilesPerSeg);
    L.ldZ = round_up(V, 8);
    L.z_only = fwd_z_only(N, V);
    size_t off = 0;
    L.part_m = off;
    off = align_up(off + size_t(L.n_segs) * size_t(N) * 4);
    L.part_s = off;
    off = align_up(off + size_t(L.n_segs) * size_t(N) * 4);
    L.zy = off;
    off = align_up(off + size_t(N) * 4);
    L.Z = off;
    if (L.z_only) off = align_up(off + size_t(N) * size_t(L.ldZ) * 4);
    L.total = N == 0 ? 0 : off;
    return L;
}

constexpr size_t kAutoChunkBytes = size_t(2) << 30;  // softmax workspace budget

// Rows of grad_bias partials a chunk of Nc tokens writes: one per 32 rows.
int64_t db_groups(int64_t Nc) { return Nc > 32 ? cdiv(Nc, 32) : 1; }

// Hi / lo split of the softmax part S (ll_options.split_s; 16-bit operands).
enum SplitMode { kSplitAuto = 0, kSplitAll = 1, kSplitNone = 2 };

// FP32 grad_hidden over a narrow hidden size (D <= 512: one or two column
// tiles per row block): the K = V contraction is cut into ks parts of at least
// 16 K blocks, one unit each, whose FP32 partial sums a finishing pass adds in
// ascending part order.  A few row blocks then spread over many SMs.  ks
// depends on (D, V) alone, so a row's grad_hidden stays independent of the
// batch and of the token chunks.
int64_t dh_k_splits(int dtype, int64_t D, int64_t V) {
    if (dtype != LL_F32 || D > 512) return 1;
    const int64_t ks = cdiv(V, 16) / 16;  // 16 K values per TF32 K block
    return ks < 2 ? 1 : (ks > kMaxDhParts ? kMaxDhParts : ks);
}

// FP32 gradient operands transposed to K-major (W^T once per call, the
// chunk's S^T and h^T), so that the tf32 kernel's converters only split and
// never transpose: the same bits as the MN-major operands, faster from a few
// GFLOP of gradient work on; below that the transposes cost more than they
// save (128 x 256 x 4096: 2 launches, +16 us against -2 us).
bool f32_kmajor_grads(int dtype, int64_t N, int64_t D, int64_t V) {
    return dtype == LL_F32 && double(N) * double(D) * double(V) >= 4294967296.0;
}

struct BwdLayout {
    int64_t chunks, Nc, ldS, ldZ, n_segs, lo_fld, dh_ks;
    size_t dh_parts;  // FP32 K-split grad_hidden: ks x round_up(Nc, 128) x D partial sums
    size_t S, S_lo, Z, part_m, part_s, zy, tc, keys, offs, ctr, db, total;
    size_t lo_flags, dh_cnt, dh_idx, dw_cnt, dw_idx;  // automatic split
    size_t hT;      // h^T [D, ldT] in the operand dtype (grad_weight's K-major B operand)
    int64_t ldT;
    // FP32: the other operands transposed to K-major for the tf32 kernel,
    // whose converters then only split (no transposes): W^T [D, ldWT] (once
    // per call) for grad_hidden, the chunk's S^T [V, ldST] for grad_weight
    size_t WT, ST;
    int64_t ldWT, ldST;
};
// fused = 1: the single fwd+bwd call, which also keeps the chunk's FP32
// logits Z and the forward partials.
// split_mode (SplitMode): all / automatic keep an S_lo buffer (16-bit
// dtypes); automatic also the piece flags and the second pass's plan.
BwdLayout bwd_layout(int64_t N, int64_t D, int64_t V, int dtype, int token_chunks, int need_db,
                     int fused = 0, int split_mode = kSplitNone) {
    BwdLayout L;
    L.ldS = round_up(V, 8);
    L.ldZ = round_up(V, 8);
    L.n_segs = cdiv(cdiv(V, kBN), kVocabTilesPerSeg);
    L.lo_fld = cdiv(V, kLoCols);
    const bool split = dtype != LL_F32 && split_mode != kSplitNone;
    const bool lo_auto = split && split_mode == kSplitAuto;
    // The automatic chunk count depends on the softmax part S alone, so the
    // two calls, the single call and the hi / lo split choose the same chunks
    // (and so give the same grad_weight bits); the single call's FP32 logits
    // and the split's S_lo come on top of the budget.
    const size_t row_bytes = size_t(L.ldS) * esize(dtype);
    const int64_t n1 = N > 0 ? N : 1;
    int64_t k = token_chunks;
    if (k <= 0) {
        k = 1;
        while (size_t(round_up(cdiv(n1, k), kBM)) * row_bytes > kAutoChunkBytes && k < n1) ++k;
    }
    if (k > n1) k = n1;
    L.Nc = token_chunks > 0 ? cdiv(n1, k) : round_up(cdiv(n1, k), kBM);
    if (L.Nc > n1) L.Nc = n1;
    L.chunks = cdiv(n1, L.Nc);
    size_t off = 0;
    L.S = off;
    off = align_up(off + size_t(L.Nc) * size_t(L.ldS) * esize(dtype));
    L.S_lo = off;
    if (split) off = align_up(off + size_t(L.Nc) * size_t(L.ldS) * esize(dtype));
    L.lo_flags = L.dh_cnt = L.dh_idx = L.dw_cnt = L.dw_idx = off;
    if (lo_auto) {  // plan sized for single-CTA blocks (128 rows / vocab rows)
        off = align_up(off + size_t(cdiv(L.Nc, kLoRows)) * size_t(lo_flags_pitch(V)));
        L.dh_cnt = off;
        off = align_up(off + size_t(cdiv(L.Nc, kBM)) * 4);
        L.dh_idx = off;
        off = align_up(off + size_t(cdiv(L.Nc, kBM)) * size_t(L.lo_fld) * 8);
        L.dw_cnt = off;
        off = align_up(off + size_t(cdiv(V, kBM)) * 4);
        L.dw_idx = off;
        off = align_up(off + size_t(cdiv(V, kBM)) * size_t(cdiv(L.Nc, 64)) * 8);
    }
    L.Z = L.part_m = L.part_s = L.zy = off;
    if (fused) {
        L.Z = off;
        off = align_up(off + size_t(L.Nc) * size_t(L.ldZ) * 4);
        L.part_m = off;
        off = align_up(off + size_t(L.n_segs) * size_t(L.Nc) * 4);
        L.part_s = off;
        off = align_up(off + size_t(L.n_segs) * size_t(L.Nc) * 4);
        L.zy = off;
        off = align_up(off + size_t(L.Nc) * 4);
    }
    L.tc = off;
    off = align_up(off + size_t(n1) * 4);
    L.keys = off;
    off = align_up(off + token_sort_bytes(n1));
    L.offs = off;
    off = align_up(off + size_t(V + 1) * 4);
    L.ctr = off;
    off = align_up(off + 64);
    L.db = off;
    if (need_db) off = align_up(off + size_t(db_groups(L.Nc) + 1) * size_t(V) * 4);
    L.hT = off;
    L.ldT = round_up(L.Nc, 8);
    off = align_up(off + size_t(D) * size_t(L.ldT) * esize(dtype));
    L.WT = L.ST = off;
    L.ldWT = round_up(V, 4);
    L.ldST = round_up(L.Nc, 4);
    if (f32_kmajor_grads(dtype, N, D, V)) {
        off = align_up(off + size_t(D) * size_t(L.ldWT) * 4);
        L.ST = off;
        off = align_up(off + size_t(V) * size_t(L.ldST) * 4);
    }
    L.dh_ks = dh_k_splits(dtype, D, V);
    L.dh_parts = off;
    if (L.dh_ks > 1) off = align_up(off + size_t(L.dh_ks) * size_t(round_up(L.Nc, kBM)) *
                                              size_t(D) * 4);
    L.total = off;
    return L;
}

int check_sizes(int64_t N, int64_t D, int64_t V) {
    if (N < 0 || D < 1 || V < 1) return LL_ERR_SHAPE;
    if (V > kMaxV || N > (int64_t(1) << 31) - 256 || D > (int64_t(1) << 31) - 256)
        return LL_ERR_SHAPE;
    return LL_OK;
}

// A vocab shard [v0, v0 + Vs) of V: starts on a segment boundary and ends on
// one unless it is the last shard.
int check_shard(int64_t Vs, int64_t v0, int64_t V) {
    if (V < 1 || V > kMaxV || Vs < 1 || v0 < 0 || v0 > V - Vs) return LL_ERR_SHAPE;
    if (v0 % kSegCols != 0) return LL_ERR_SHAPE;
    if (v0 + Vs != V && Vs % kSegCols != 0) return LL_ERR_SHAPE;
    return LL_OK;
}

// Options of a call: *inv_temp = 1 / temperature, *split = SplitMode of S.
// NULL = defaults.
int read_options(const ll_options* o, float* inv_temp, int* split = nullptr) {
    *inv_temp = 1.f;
    if (split) *split = kSplitAuto;
    if (!o) return LL_OK;
    for (int r : o->reserved)
        if (r != 0) return LL_ERR_INVALID_ARG;
    if (o->split_s < kSplitAuto || o->split_s > kSplitNone) return LL_ERR_INVALID_ARG;
    if (split) *split = o->split_s;
    const float T = o->temperature;
    if (!(T > 0.f) || !(T < INFINITY)) return LL_ERR_INVALID_ARG;
    const float it = 1.f / T;
    if (!(it > 0.f) || !(it < INFINITY)) return LL_ERR_INVALID_ARG;
    *inv_temp = it;
    return LL_OK;
}

// Shard-local targets after the backward's (or at the forward's) workspace.
size_t local_targets_bytes(int64_t N) { return align_up(size_t(N > 0 ? N : 1) * 8); }

}  // namespace
}  // namespace ll

using namespace ll;

extern "C" {

const char* ll_status_string(int status) {
    switch (status) {
        case LL_OK: return "ok";
        case LL_ERR_INVALID_ARG: return "invalid argument";
        case LL_ERR_DTYPE: return "unsupported dtype";
        case LL_ERR_SHAPE: return "invalid shape";
        case LL_ERR_ALIGN: return "misaligned pointer or stride";
        case LL_ERR_WORKSPACE: return "workspace missing or too small";
        case LL_ERR_CUDA: return "CUDA error";
        case LL_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case LL_ERR_UNSUPPORTED: return "unsupported device";
        default: return "unknown status";
    }
}

int ll_version(void) { return 100; }

size_t ll_workspace_size(int64_t N, int64_t D, int64_t V, int dtype, int token_chunks,
                         int is_backward, int flags) {
    (void)D;
    if (N < 0 || V < 1 || !dtype_ok(dtype)) return 0;
    if (!is_backward) return fwd_layout(N, V).total;
    const int mode = (flags >> 1) & 3;
    if (mode > kSplitNone) return 0;
    return bwd_layout(N, D, V, dtype, token_chunks, flags & 1, is_backward == 2, mode).total;
}

void ll_set_wait_limit_ns(int64_t ns) { g_wait_limit_ns = ns > 0 ? uint64_t(ns) : 2000000000ull; }

}  // extern "C"

namespace ll {
namespace {
// The forward GEMM: per (row, vocab segment) partials [n_segs, N] and the
// target logit of rows whose target lies in [0, V).
cudaError_t forward_gemm(const void* hidden, const void* weight, const void* bias,
                         const int64_t* targets, int64_t N, int64_t D, int64_t V, int dtype,
                         float* part_m, float* part_s, float* zy, int shard, float inv_temp,
                         const DevInfo& dev, cudaStream_t s, float* Z = nullptr,
                         int64_t ldZ = 0) {
    // Z: store the logits there, one vocab tile per unit, and leave the
    // partials to fwd_fold_kernel
    GemmShape sh;
    memset(&sh, 0, sizeof(sh));
    sh.m_blocks = cdiv(N, kBM);
    sh.n_tiles = cdiv(V, kBN);
    sh.tiles_per_unit = Z ? 1 : kVocabTilesPerSeg;
    sh.n_segs = cdiv(sh.n_tiles, sh.tiles_per_unit);
    sh.k_blocks = cdiv(D, 64);
    sh.unit_order = 2;
    EpiArgs ea;
    memset(&ea, 0, sizeof(ea));
    ea.M = N;
    ea.Ncols = V;
    ea.V = V;
    ea.targets = targets;
    ea.bias = bias;
    ea.part_m = part_m;
    ea.part_s = part_s;
    ea.zy = zy;
    ea.part_ld = N;
    ea.status = dev.status;
    ea.wait_ns = wait_limit_ns();
    ea.shard = shard;
    ea.inv_temp = inv_temp;
    ea.z_only = Z != nullptr;
    GemmLaunch G;
    memset(&G, 0, sizeof(G));
    G.dtype = dtype;
    G.nkinds = 1;
    G.kind[0] = EpiKind::Fwd;
    G.op[0] = GemmOperands{hidden, D, 0, weight, D, 0, N, V, D, nullptr, nullptr, nullptr, 0};
    G.shape[0] = sh;
    G.ea[0] = ea;
    if (Z) G.out[0] = OutDesc{Z, LL_F32, N, V, ldZ};
    Phase ph(dtype == LL_F32 ? "fwd_gemm_f32" : "fwd_gemm", s);
    return launch_gemm(G, dev, s);
}

// Validation shared by the forward entry points.
int forward_checks(const void* hidden, const void* weight, const int64_t* targets, int64_t N,
                   int64_t D, int64_t V, int dtype) {
    int st = check_sizes(N, D, V);
    if (st) return st;
    if (!dtype_ok(dtype)) return LL_ERR_DTYPE;
    if (!weight) return LL_ERR_INVALID_ARG;
    if (N == 0) return LL_OK;
    if (!hidden || !targets) return LL_ERR_INVALID_ARG;
    if (D % 8 != 0 || !aligned16(hidden) || !aligned16(weight)) return LL_ERR_ALIGN;
    return LL_OK;
}
}  // namespace
}  // namespace ll

extern "C" {

int ll_forward(const void* hidden, const void* weight, const void* bias, const int64_t* targets,
               int64_t N, int64_t D, int64_t V, int dtype, float* logp, float* lse,
               void* workspace, size_t ws_bytes, void* stream) {
    return ll_forward_ex(hidden, weight, bias, targets, N, D, V, dtype, logp, lse, workspace,
                         ws_bytes, nullptr, stream);
}

int ll_forward_ex(const void* hidden, const void* weight, const void* bias,
                  const int64_t* targets, int64_t N, int64_t D, int64_t V, int dtype,
                  float* logp, float* lse, void* workspace, size_t ws_bytes,
                  const ll_options* opt, void* stream) {
    float it;
    int st = read_options(opt, &it);
    if (st) return st;
    st = forward_checks(hidden, weight, targets, N, D, V, dtype);
    if (st || N == 0) return st;
    if (!logp || !lse) return LL_ERR_INVALID_ARG;
    const FwdLayout L = fwd_layout(N, V);
    if (!workspace || ws_bytes < L.total) return LL_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return LL_ERR_WORKSPACE;
    DeviceGuard guard(hidden);
    if (guard.err) return guard.err;
    DevInfo dev;
    if ((st = device_info(guard.dev, &dev))) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    float* part_m = reinterpret_cast<float*>(ws + L.part_m);
    float* part_s = reinterpret_cast<float*>(ws + L.part_s);
    float* zy = reinterpret_cast<float*>(ws + L.zy);
    float* Z = L.z_only ? reinterpret_cast<float*>(ws + L.Z) : nullptr;
    cudaError_t e = forward_gemm(hidden, weight, bias, targets, N, D, V, dtype, part_m, part_s,
                                 zy, 0, it, dev, s, Z, L.ldZ);
    if (e != cudaSuccess) return cuda_status(e);
    if (Z && L.n_segs <= kFoldMergeSegs) {  // fold and merge in one launch
        Phase ph("fwd_fold", s);
        return cuda_status(
            launch_fwd_fold_merge(Z, L.ldZ, N, V, targets, part_m, part_s, zy, N, logp, lse, s));
    }
    if (Z) {
        Phase ph("fwd_fold", s);
        e = launch_fwd_fold(Z, L.ldZ, N, V, targets, part_m, part_s, zy, N, s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    {
        Phase ph("lse_merge", s);
        e = launch_lse_merge(part_m, part_s, zy, N, L.n_segs, targets, N, V, logp, lse, s);
    }
    return cuda_status(e);
}

}  // extern "C"

namespace ll {
namespace {
// The backward, or (fused = 1) the forward and backward in one call when
// grad_logp is known up front: the chunk's forward GEMM then keeps its FP32
// logits and the softmax part is formed from them, instead of recomputing z.
int backward_impl(const float* grad_logp, const void* hidden, const void* weight,
                  const void* bias, const int64_t* targets, const float* lse, int64_t N,
                  int64_t D, int64_t V, int dtype, int need_dh, int need_dw, int need_db,
                  void* grad_hidden, int dh_dtype, void* grad_weight, int dw_dtype,
                  void* grad_bias, int token_chunks, void* workspace, size_t ws_bytes,
                  void* stream, int fused, float* logp_out, float* lse_out, int shard = 0,
                  float inv_temp = 1.f, int split = kSplitAuto) {
    int st = check_sizes(N, D, V);
    if (st) return st;
    if (!dtype_ok(dtype)) return LL_ERR_DTYPE;
    if ((need_dh | need_dw | need_db) & ~1) return LL_ERR_INVALID_ARG;
    if (token_chunks < 0) return LL_ERR_INVALID_ARG;
    if (need_dh && !(dh_dtype == dtype || dh_dtype == LL_F32)) return LL_ERR_DTYPE;
    if ((need_dw || need_db) && !(dw_dtype == dtype || dw_dtype == LL_F32)) return LL_ERR_DTYPE;
    if (!weight) return LL_ERR_INVALID_ARG;
    if (need_dw && !grad_weight) return LL_ERR_INVALID_ARG;
    if (need_db && !grad_bias) return LL_ERR_INVALID_ARG;
    if (need_dh && N > 0 && !grad_hidden) return LL_ERR_INVALID_ARG;
    if (D % 8 != 0 || !aligned16(weight)) return LL_ERR_ALIGN;
    if (need_dw && !aligned16(grad_weight)) return LL_ERR_ALIGN;
    if (fused && N > 0 && (!logp_out || !lse_out)) return LL_ERR_INVALID_ARG;
    if (!fused && !need_dh && !need_dw && !need_db) return LL_OK;

    DeviceGuard guard(weight);
    if (guard.err) return guard.err;
    DevInfo dev;
    if ((st = device_info(guard.dev, &dev))) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;

    if (N == 0) {  // empty batch: requested table gradients are +0
        if (need_dw) e = launch_fill_zero(grad_weight, V * D, dw_dtype, s);
        if (e == cudaSuccess && need_db) e = launch_fill_zero(grad_bias, V, dw_dtype, s);
        return cuda_status(e);
    }
    if (!grad_logp || !hidden || !targets || (!fused && !lse)) return LL_ERR_INVALID_ARG;
    if (!aligned16(hidden) || (need_dh && !aligned16(grad_hidden))) return LL_ERR_ALIGN;
    const BwdLayout L = bwd_layout(N, D, V, dtype, token_chunks, need_db, fused, split);
    if (!workspace || ws_bytes < L.total) return LL_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return LL_ERR_WORKSPACE;

    char* ws = static_cast<char*>(workspace);
    void* S = ws + L.S;
    // FP32 keeps S in FP32: nothing to split
    const bool has_lo = dtype != LL_F32 && split != kSplitNone;
    const bool lo_auto = has_lo && split == kSplitAuto;
    void* S_lo = has_lo ? static_cast<void*>(ws + L.S_lo) : nullptr;
    uint8_t* lo_flags = lo_auto ? reinterpret_cast<uint8_t*>(ws + L.lo_flags) : nullptr;
    int* dh_cnt = reinterpret_cast<int*>(ws + L.dh_cnt);
    int64_t* dh_idx = reinterpret_cast<int64_t*>(ws + L.dh_idx);
    int* dw_cnt = reinterpret_cast<int*>(ws + L.dw_cnt);
    int64_t* dw_idx = reinterpret_cast<int64_t*>(ws + L.dw_idx);
    float* tc = reinterpret_cast<float*>(ws + L.tc);
    int64_t* keys = reinterpret_cast<int64_t*>(ws + L.keys);
    int* offs = reinterpret_cast<int*>(ws + L.offs);
    int* counter = reinterpret_cast<int*>(ws + L.ctr);
    float* db_part = reinterpret_cast<float*>(ws + L.db);
    float* db_acc = db_part + db_groups(L.Nc) * V;  // after the partial rows
    const size_t es = esize(dtype);
    float* Z = reinterpret_cast<float*>(ws + L.Z);
    float* part_m = reinterpret_cast<float*>(ws + L.part_m);
    float* part_s = reinterpret_cast<float*>(ws + L.part_s);
    float* zy = reinterpret_cast<float*>(ws + L.zy);
    if (fused) lse = lse_out;

    // The token sort (only the last chunk's grad_weight / grad_bias epilogue
    // reads it) runs on a side stream, overlapping the first recompute (or
    // forward) GEMM, which leaves kSideSms SMs free for it.
    cudaEvent_t sort_done = nullptr;
    const bool need_sort = need_dw || need_db;
    bool overlap = false;
    if (need_sort) {
        cudaEvent_t fork = nullptr;
        overlap = dev.side != nullptr &&
                  cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) == cudaSuccess &&
                  cudaEventCreateWithFlags(&sort_done, cudaEventDisableTiming) == cudaSuccess;
        cudaStream_t ss = s;
        if (overlap) {
            cudaEventRecord(fork, s);
            cudaStreamWaitEvent(dev.side, fork, 0);
            ss = dev.side;
        }
        {
            Phase ph("token_sort", ss);
            e = launch_token_sort(targets, N, V, keys, offs, ss);
        }
        if (overlap) {
            cudaEventRecord(sort_done, ss);
            cudaEventDestroy(fork);
        }
        if (e != cudaSuccess) return cuda_status(e);
    }

    // grad_weight's B operand, the chunk's h^T: K-major (tokens contiguous)
    // for the tensor cores, so that only its A operand (S) is read MN-major
    void* hT = ws + L.hT;
    float* WT = reinterpret_cast<float*>(ws + L.WT);
    float* ST = reinterpret_cast<float*>(ws + L.ST);
    const bool f32_t = f32_kmajor_grads(dtype, N, D, V);
    if (f32_t && need_dh) {  // W^T: grad_hidden's B operand, K-major
        Phase ph("transpose_w", s);
        e = launch_transpose32(static_cast<const float*>(weight), V, D, D, WT, L.ldWT, s);
        if (e != cudaSuccess) return cuda_status(e);
    }

    EpiArgs base;
    memset(&base, 0, sizeof(base));
    base.V = V;
    base.bias = bias;
    base.status = dev.status;
    base.wait_ns = wait_limit_ns();
    base.shard = shard;
    base.inv_temp = inv_temp;

    // grad_bias is finished on the side stream, beside the gradient launch: it
    // needs the chunk's partials (step 1) and, at the last chunk, the token
    // sort, which runs earlier on that stream.  The next chunk's step 1
    // rewrites the partials, so it first waits for this chunk's finishing.
    cudaEvent_t db_fork = nullptr, db_done = nullptr;
    bool db_side = need_db && dev.side != nullptr &&
                   cudaEventCreateWithFlags(&db_fork, cudaEventDisableTiming) == cudaSuccess &&
                   cudaEventCreateWithFlags(&db_done, cudaEventDisableTiming) == cudaSuccess;
    if (!db_side) {
        if (db_fork) cudaEventDestroy(db_fork);
        if (db_done) cudaEventDestroy(db_done);
    }

    for (int64_t c = 0; c < L.chunks; ++c) {
        const int64_t r0 = c * L.Nc;
        const int64_t rows = (N - r0) < L.Nc ? (N - r0) : L.Nc;
        const char* h_c = static_cast<const char*>(hidden) + size_t(r0) * size_t(D) * es;
        if (db_side && c > 0) cudaStreamWaitEvent(s, db_done, 0);

        // (1) recompute z for the chunk, store S = -grad * p off target and c
        if (!fused) {
            GemmLaunch G;
            memset(&G, 0, sizeof(G));
            G.dtype = dtype;
            G.nkinds = 1;
            G.kind[0] = EpiKind::Recomp;
            G.op[0] = GemmOperands{h_c, D, 0, weight, D, 0, rows, V, D, nullptr, nullptr, nullptr, 0};
            GemmShape& sh = G.shape[0];
            sh.m_blocks = cdiv(rows, kBM);
            sh.n_tiles = cdiv(V, kBN);
            // the recompute's tiles are independent (no running state across a
            // segment): a small problem takes one tile per unit, so that its few
            // tiles spread over the SMs
            const bool few = sh.m_blocks * cdiv(sh.n_tiles, kVocabTilesPerSeg) <
                             int64_t(2) * dev.num_sms;
            sh.tiles_per_unit = few ? 1 : kVocabTilesPerSeg;
            sh.n_segs = cdiv(sh.n_tiles, sh.tiles_per_unit);
            sh.k_blocks = cdiv(D, 64);
            sh.unit_order = 2;
            EpiArgs& ea = G.ea[0];
            ea = base;
            ea.M = rows;
            ea.Ncols = V;
            ea.targets = targets + r0;
            ea.lse = lse + r0;
            ea.grad = grad_logp + r0;
            ea.S = S;
            ea.S_lo = S_lo;
            ea.lo_flags = lo_flags;
            ea.lo_flags_ld = lo_flags_pitch(V);
            ea.lo_flags_cols = L.lo_fld;
            ea.ldS = L.ldS;
            ea.tc = tc + r0;
            ea.db_part = need_db ? db_part : nullptr;
            G.out[0] = OutDesc{S, dtype, rows, V, L.ldS};
            G.zero_counter = counter;  // for the gradient launch that follows
            if (overlap && c == 0) G.max_ctas = dev.num_sms - kSideSms;
            Phase ph(dtype == LL_F32 ? "recompute_gemm_f32" : "recompute_gemm", s);
            e = launch_gemm(G, dev, s);
            if (e != cudaSuccess) return cuda_status(e);
        } else {
            // (1') forward GEMM of the chunk keeping its FP32 logits, the
            // ordered LSE merge (logp, lse), then S and c from the logits
            GemmLaunch G;
            memset(&G, 0, sizeof(G));
            G.dtype = dtype;
            G.nkinds = 1;
            G.kind[0] = EpiKind::Fwd;
            G.op[0] = GemmOperands{h_c, D, 0, weight, D, 0, rows, V, D, nullptr, nullptr, nullptr, 0};
            GemmShape& sh = G.shape[0];
            sh.m_blocks = cdiv(rows, kBM);
            sh.n_tiles = cdiv(V, kBN);
            // few units: one vocab tile per unit and the fold as its own
            // kernel (the same bits; the logits are stored either way)
            const bool fold = sh.m_blocks * L.n_segs < int64_t(2) * dev.num_sms;
            sh.tiles_per_unit = fold ? 1 : kVocabTilesPerSeg;
            sh.n_segs = fold ? sh.n_tiles : L.n_segs;
            sh.k_blocks = cdiv(D, 64);
            sh.unit_order = 2;
            EpiArgs& ea = G.ea[0];
            ea = base;
            ea.M = rows;
            ea.Ncols = V;
            ea.targets = targets + r0;
            ea.part_m = part_m;
            ea.part_s = part_s;
            ea.zy = zy;
            ea.part_ld = L.Nc;
            ea.Z = Z;
            ea.ldZ = L.ldZ;
            ea.z_only = fold;
            G.out[0] = OutDesc{Z, LL_F32, rows, V, L.ldZ};
            G.zero_counter = counter;
            if (overlap && c == 0) G.max_ctas = dev.num_sms - kSideSms;
            {
                Phase ph(dtype == LL_F32 ? "fwd_gemm_f32" : "fwd_gemm", s);
                e = launch_gemm(G, dev, s);
            }
            if (e != cudaSuccess) return cuda_status(e);
            if (ea.z_only && L.n_segs <= kFoldMergeSegs) {  // fold and merge in one launch
                Phase ph("fwd_fold", s);
                e = launch_fwd_fold_merge(Z, L.ldZ, rows, V, targets + r0, part_m, part_s, zy,
                                          L.Nc, logp_out + r0, lse_out + r0, s);
            } else {
                if (ea.z_only) {
                    Phase ph("fwd_fold", s);
                    e = launch_fwd_fold(Z, L.ldZ, rows, V, targets + r0, part_m, part_s, zy,
                                        L.Nc, s);
                    if (e != cudaSuccess) return cuda_status(e);
                }
                Phase ph("lse_merge", s);
                e = launch_lse_merge(part_m, part_s, zy, L.Nc, L.n_segs, targets + r0, rows, V,
                                     logp_out + r0, lse_out + r0, s);
            }
            if (e != cudaSuccess) return cuda_status(e);
            {
                Phase ph("softmax_part", s);
                e = launch_softmax_part(Z, L.ldZ, rows, V, targets + r0, grad_logp + r0,
                                        lse_out + r0, S, L.ldS, dtype, tc + r0,
                                        need_db ? db_part : nullptr, inv_temp, S_lo, lo_flags,
                                        s);
            }
            if (e != cudaSuccess) return cuda_status(e);
        }
        if (db_side) {  // (4) grad_bias, beside what follows
            cudaEventRecord(db_fork, s);
            cudaStreamWaitEvent(dev.side, db_fork, 0);
            {
                Phase ph("db_sums", dev.side);
                e = launch_db_finish(db_part, cdiv(rows, 32), V, db_acc, c == 0,
                                     c == L.chunks - 1, offs, keys, tc, grad_bias, dw_dtype,
                                     dev.side);
            }
            if (e != cudaSuccess) return cuda_status(e);
            cudaEventRecord(db_done, dev.side);
        }
        if (overlap && c == L.chunks - 1) {  // the last chunk's epilogues read the sort
            cudaStreamWaitEvent(s, sort_done, 0);
            cudaEventDestroy(sort_done);
            overlap = false;
        }
        // (2)+(3) grad_hidden rows of the chunk (S . W + c * W[y]) and
        // grad_weight += S^T . h (+ the target part on the last chunk), in
        // one launch: grad_hidden tiles (K = V) first, grad_weight tiles after
        if ((need_dh || need_dw) && lo_auto) {
            // the automatic split's second pass: which K blocks of which
            // blocks have written pieces of S_lo, at the launch's block size
            int64_t Ms[2];
            int nk = 0;
            if (need_dh) Ms[nk++] = rows;
            if (need_dw) Ms[nk++] = V;
            const int blk = gemm_uses_pairs(dtype, Ms, nk) ? 2 * kBM : kBM;
            Phase ph("lo_plan", s);
            e = launch_lo_plan(lo_flags, rows, V, blk, blk, dh_cnt, dh_idx, dw_cnt, dw_idx, s);
            if (e != cudaSuccess) return cuda_status(e);
        }
        if (need_dw && (f32_t || dtype != LL_F32)) {
            Phase ph("transpose_h", s);
            if (f32_t) {  // h^T and S^T: grad_weight's operands, K-major
                e = launch_transpose32(reinterpret_cast<const float*>(h_c), rows, D, D,
                                       static_cast<float*>(hT), L.ldT, s);
                if (e == cudaSuccess)
                    e = launch_transpose32(static_cast<const float*>(S), rows, V, L.ldS, ST,
                                           L.ldST, s);
            } else {
                e = launch_transpose16(h_c, rows, D, hT, L.ldT, s);
            }
            if (e != cudaSuccess) return cuda_status(e);
        }
        if (need_dh || need_dw) {
            GemmLaunch G;
            memset(&G, 0, sizeof(G));
            G.dtype = dtype;
            int k = 0;
            if (need_dh) {
                G.kind[k] = EpiKind::Dh;
                if (f32_t)  // K-major B: W^T [D, V]
                    G.op[k] = GemmOperands{S, L.ldS, 0, WT, L.ldWT, 0, rows, D, V, nullptr,
                                           nullptr, nullptr, 0};
                else if (dtype == LL_F32)  // MN-major B: W itself
                    G.op[k] = GemmOperands{S, L.ldS, 0, weight, D, 1, rows, D, V, nullptr,
                                           nullptr, nullptr, 0};
                else
                    G.op[k] = GemmOperands{S, L.ldS, 0, weight, D, 1, rows, D, V, S_lo,
                                           lo_auto ? dh_cnt : nullptr, dh_idx, L.lo_fld};
                GemmShape& sh = G.shape[k];
                sh.m_blocks = cdiv(rows, kBM);
                sh.n_tiles = cdiv(D, kBN);
                sh.tiles_per_unit = 1;
                sh.n_segs = sh.n_tiles;
                sh.k_blocks = cdiv(V, 64);
                sh.unit_order = 1;  // a row block's D tiles run together and share its S rows in L2
                EpiArgs& ea = G.ea[k];
                ea = base;
                ea.M = rows;
                ea.Ncols = D;
                ea.targets = targets + r0;
                ea.grad = grad_logp + r0;
                ea.tc = tc + r0;
                ea.W = weight;
                ea.ldW = D;
                ea.out = static_cast<char*>(grad_hidden) + size_t(r0) * size_t(D) * esize(dh_dtype);
                ea.ld_out = D;
                ea.out_dtype = dh_dtype;
                G.out[k] = OutDesc{ea.out, dh_dtype, rows, D, D};
                if (L.dh_ks > 1) {  // K parts: raw partial sums, finished below
                    sh.k_splits = L.dh_ks;
                    ea.dh_part = 1;
                    G.out[k] = OutDesc{ws + L.dh_parts, LL_F32, L.dh_ks * round_up(rows, kBM), D,
                                       D};
                }
                ++k;
            }
            if (need_dw) {
                G.kind[k] = EpiKind::Dw;
                if (f32_t)  // K-major A and B: S^T [V, rows], h^T [D, rows]
                    G.op[k] = GemmOperands{ST, L.ldST, 0, hT, L.ldT, 0, V, D, rows, nullptr,
                                           nullptr, nullptr, 0};
                else if (dtype == LL_F32)  // MN-major A and B: S and the chunk's h
                    G.op[k] = GemmOperands{S, L.ldS, 1, h_c, D, 1, V, D, rows, nullptr,
                                           nullptr, nullptr, 0};
                else  // K-major B: the chunk's h^T [D, rows]; A = S read MN-major
                    G.op[k] = GemmOperands{S, L.ldS, 1, hT, L.ldT, 0, V, D, rows, S_lo,
                                           lo_auto ? dw_cnt : nullptr, dw_idx, cdiv(rows, 64)};
                GemmShape& sh = G.shape[k];
                sh.m_blocks = cdiv(V, kBM);
                sh.n_tiles = cdiv(D, kBN);
                sh.tiles_per_unit = 1;
                sh.n_segs = sh.n_tiles;
                sh.k_blocks = cdiv(rows, 64);
                sh.unit_order = 1;
                EpiArgs& ea = G.ea[k];
                ea = base;
                ea.M = V;
                ea.Ncols = D;
                ea.out = grad_weight;
                ea.ld_out = D;
                ea.out_dtype = dw_dtype;
                ea.first_chunk = c == 0;
                ea.last_chunk = c == L.chunks - 1;
                ea.offs = offs;
                ea.keys = keys;
                ea.tc_all = tc;
                ea.h_all = hidden;
                ea.ld_h = D;
                G.out[k] = OutDesc{grad_weight, dw_dtype, V, D, D};
                ++k;
            }
            G.nkinds = k;
            G.counter = k == 2 ? counter : nullptr;
            const char* label = dtype == LL_F32 ? "grad_gemm_f32" : "grad_gemm";
            {
                Phase ph(label, s);
                e = launch_gemm(G, dev, s);
            }
            if (e != cudaSuccess) return cuda_status(e);
            if (need_dh && L.dh_ks > 1) {
                Phase ph("dh_finish", s);
                e = launch_dh_finish(reinterpret_cast<const float*>(ws + L.dh_parts),
                                     static_cast<int>(L.dh_ks), round_up(rows, kBM), rows, D,
                                     targets + r0, grad_logp + r0, tc + r0, V, shard,
                                     static_cast<const float*>(weight),
                                     static_cast<float*>(grad_hidden) + r0 * D, dev.num_sms, s);
                if (e != cudaSuccess) return cuda_status(e);
            }
        }
        // (4) grad_bias: fixed-order column sums of S (+ one-hot part at the end)
        if (need_db && !db_side) {
            Phase ph("db_sums", s);
            // partials per 32 rows from the recompute epilogue (or, in the
            // single call, from the softmax-part kernel with the same sums)
            e = launch_db_finish(db_part, cdiv(rows, 32), V, db_acc, c == 0, c == L.chunks - 1,
                                 offs, keys, tc, grad_bias, dw_dtype, s);
            if (e != cudaSuccess) return cuda_status(e);
        }
    }
    if (overlap) {  // nothing read the sort (no chunk needed it): still join it
        cudaStreamWaitEvent(s, sort_done, 0);
        cudaEventDestroy(sort_done);
    }
    if (db_side) {  // the call ends when grad_bias is done
        cudaStreamWaitEvent(s, db_done, 0);
        cudaEventDestroy(db_fork);
        cudaEventDestroy(db_done);
    }
    return LL_OK;
}
}  // namespace
}  // namespace ll

extern "C" {

int ll_backward_ex(const float* grad_logp, const void* hidden, const void* weight,
                   const void* bias, const int64_t* targets, const float* lse, int64_t N,
                   int64_t D, int64_t V, int dtype, int need_dh, int need_dw, int need_db,
                   void* grad_hidden, int dh_dtype, void* grad_weight, int dw_dtype,
                   void* grad_bias, int token_chunks, void* workspace, size_t ws_bytes,
                   const ll_options* opt, void* stream) {
    float it;
    int split;
    int st = read_options(opt, &it, &split);
    if (st) return st;
    return backward_impl(grad_logp, hidden, weight, bias, targets, lse, N, D, V, dtype, need_dh,
                         need_dw, need_db, grad_hidden, dh_dtype, grad_weight, dw_dtype,
                         grad_bias, token_chunks, workspace, ws_bytes, stream, 0, nullptr,
                         nullptr, 0, it, split);
}

int ll_backward(const float* grad_logp, const void* hidden, const void* weight, const void* bias,
                const int64_t* targets, const float* lse, int64_t N, int64_t D, int64_t V,
                int dtype, int need_dh, int need_dw, int need_db, void* grad_hidden,
                int dh_dtype, void* grad_weight, int dw_dtype, void* grad_bias,
                int token_chunks, void* workspace, size_t ws_bytes, void* stream) {
    return ll_backward_ex(grad_logp, hidden, weight, bias, targets, lse, N, D, V, dtype, need_dh,
                          need_dw, need_db, grad_hidden, dh_dtype, grad_weight, dw_dtype,
                          grad_bias, token_chunks, workspace, ws_bytes, nullptr, stream);
}

int ll_forward_backward_ex(const float* grad_logp, const void* hidden, const void* weight,
                           const void* bias, const int64_t* targets, int64_t N, int64_t D,
                           int64_t V, int dtype, float* logp, float* lse, int need_dh,
                           int need_dw, int need_db, void* grad_hidden, int dh_dtype,
                           void* grad_weight, int dw_dtype, void* grad_bias,
                           int token_chunks, void* workspace, size_t ws_bytes,
                           const ll_options* opt, void* stream) {
    float it;
    int split;
    int st = read_options(opt, &it, &split);
    if (st) return st;
    return backward_impl(grad_logp, hidden, weight, bias, targets, nullptr, N, D, V, dtype,
                         need_dh, need_dw, need_db, grad_hidden, dh_dtype, grad_weight, dw_dtype,
                         grad_bias, token_chunks, workspace, ws_bytes, stream, 1, logp, lse, 0,
                         it, split);
}

int ll_forward_backward(const float* grad_logp, const void* hidden, const void* weight,
                        const void* bias, const int64_t* targets, int64_t N, int64_t D,
                        int64_t V, int dtype, float* logp, float* lse, int need_dh,
                        int need_dw, int need_db, void* grad_hidden, int dh_dtype,
                        void* grad_weight, int dw_dtype, void* grad_bias, int token_chunks,
                        void* workspace, size_t ws_bytes, void* stream) {
    return ll_forward_backward_ex(grad_logp, hidden, weight, bias, targets, N, D, V, dtype, logp,
                                  lse, need_dh, need_dw, need_db, grad_hidden, dh_dtype,
                                  grad_weight, dw_dtype, grad_bias, token_chunks, workspace,
                                  ws_bytes, nullptr, stream);
}

int64_t ll_shard_segments(int64_t Vs) { return Vs > 0 ? cdiv(Vs, kSegCols) : 0; }

size_t ll_workspace_size_shard(int64_t N, int64_t D, int64_t Vs, int dtype, int token_chunks,
                               int is_backward, int flags) {
    (void)D;
    if (N < 0 || Vs < 1 || !dtype_ok(dtype)) return 0;
    if (N == 0) return 0;
    if (!is_backward) return local_targets_bytes(N);
    const int mode = (flags >> 1) & 3;
    if (mode > kSplitNone) return 0;
    return bwd_layout(N, D, Vs, dtype, token_chunks, flags & 1, 0, mode).total +
           local_targets_bytes(N);
}

int ll_forward_shard(const void* hidden, const void* weight, const void* bias,
                     const int64_t* targets, int64_t N, int64_t D, int64_t Vs, int64_t v0,
                     int64_t V, int dtype, float* part_m, float* part_s, float* zy,
                     void* workspace, size_t ws_bytes, const ll_options* opt, void* stream) {
    float it;
    int st = read_options(opt, &it);
    if (st) return st;
    if ((st = check_shard(Vs, v0, V))) return st;
    st = forward_checks(hidden, weight, targets, N, D, Vs, dtype);
    if (st || N == 0) return st;
    if (!part_m || !part_s || !zy) return LL_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < local_targets_bytes(N)) return LL_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return LL_ERR_WORKSPACE;
    DeviceGuard guard(hidden);
    if (guard.err) return guard.err;
    DevInfo dev;
    if ((st = device_info(guard.dev, &dev))) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int64_t* local = static_cast<int64_t*>(workspace);
    cudaError_t e = launch_localize_targets(targets, N, v0, Vs, V, local, zy, s);
    if (e != cudaSuccess) return cuda_status(e);
    return cuda_status(forward_gemm(hidden, weight, bias, local, N, D, Vs, dtype, part_m, part_s,
                                    zy, 1, it, dev, s));
}

int ll_lse_merge(const float* part_m, const float* part_s, int64_t n_segs, int64_t part_ld,
                 const float* zy, const int64_t* targets, int64_t N, int64_t V, float* logp,
                 float* lse, void* stream) {
    if (N < 0 || V < 1 || V > kMaxV || n_segs < 1 || part_ld < N) return LL_ERR_SHAPE;
    if (N == 0) return LL_OK;
    if (!part_m || !part_s || !zy || !targets || !logp || !lse) return LL_ERR_INVALID_ARG;
    DeviceGuard guard(part_m);
    if (guard.err) return guard.err;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Phase ph("lse_merge", s);
    return cuda_status(launch_lse_merge(part_m, part_s, zy, part_ld, n_segs, targets, N, V, logp,
                                        lse, s));
}

int ll_backward_shard(const float* grad_logp, const void* hidden, const void* weight,
                      const void* bias, const int64_t* targets, const float* lse, int64_t N,
                      int64_t D, int64_t Vs, int64_t v0, int64_t V, int dtype, int need_dh,
                      int need_dw, int need_db, void* grad_hidden, int dh_dtype,
                      void* grad_weight, int dw_dtype, void* grad_bias, int token_chunks,
                      void* workspace, size_t ws_bytes, const ll_options* opt, void* stream) {
    float it;
    int split;
    int st = read_options(opt, &it, &split);
    if (st) return st;
    if ((st = check_shard(Vs, v0, V))) return st;
    if ((st = check_sizes(N, D, Vs))) return st;
    if (!dtype_ok(dtype)) return LL_ERR_DTYPE;
    if (N == 0 || !(need_dh | need_dw | need_db))
        return backward_impl(grad_logp, hidden, weight, bias, targets, lse, N, D, Vs, dtype,
                             need_dh, need_dw, need_db, grad_hidden, dh_dtype, grad_weight,
                             dw_dtype, grad_bias, token_chunks, workspace, ws_bytes, stream, 0,
                             nullptr, nullptr, 1, it, split);
    if (!targets || !weight) return LL_ERR_INVALID_ARG;
    const size_t tail = local_targets_bytes(N);
    if (!workspace || ws_bytes < tail) return LL_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return LL_ERR_WORKSPACE;
    const size_t body = ws_bytes - tail;
    const BwdLayout L = bwd_layout(N, D, Vs, dtype, token_chunks, need_db, 0, split);
    if (body < L.total) return LL_ERR_WORKSPACE;
    // checks of backward_impl that must pass before anything is launched
    if ((need_dh | need_dw | need_db) & ~1 || token_chunks < 0) return LL_ERR_INVALID_ARG;
    if (need_dh && !(dh_dtype == dtype || dh_dtype == LL_F32)) return LL_ERR_DTYPE;
    if ((need_dw || need_db) && !(dw_dtype == dtype || dw_dtype == LL_F32)) return LL_ERR_DTYPE;
    if ((need_dw && !grad_weight) || (need_db && !grad_bias) || (need_dh && !grad_hidden))
        return LL_ERR_INVALID_ARG;
    if (!grad_logp || !hidden || !lse) return LL_ERR_INVALID_ARG;
    if (D % 8 != 0 || !aligned16(weight) || !aligned16(hidden) ||
        (need_dw && !aligned16(grad_weight)) || (need_dh && !aligned16(grad_hidden)))
        return LL_ERR_ALIGN;
    DeviceGuard guard(weight);
    if (guard.err) return guard.err;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int64_t* local = reinterpret_cast<int64_t*>(static_cast<char*>(workspace) + body);
    cudaError_t e = launch_localize_targets(targets, N, v0, Vs, V, local, nullptr, s);
    if (e != cudaSuccess) return cuda_status(e);
    return backward_impl(grad_logp, hidden, weight, bias, local, lse, N, D, Vs, dtype, need_dh,
                         need_dw, need_db, grad_hidden, dh_dtype, grad_weight, dw_dtype,
                         grad_bias, token_chunks, workspace, body, stream, 0, nullptr, nullptr,
                         1, it, split);
}

int logits_logp_fwd(const void* logits, int64_t ld, int dtype, const int64_t* targets, int64_t N,
                    int64_t V, float* logp, float* lse, void* stream) {
    return logits_logp_fwd_ex(logits, ld, dtype, targets, N, V, logp, lse, nullptr, stream);
}

int logits_logp_fwd_ex(const void* logits, int64_t ld, int dtype, const int64_t* targets,
                       int64_t N, int64_t V, float* logp, float* lse, const ll_options* opt,
                       void* stream) {
    float it;
    if (read_options(opt, &it)) return LL_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return LL_ERR_DTYPE;
    if (N < 0 || V < 1 || V > kMaxV || ld < V || N > (int64_t(1) << 31) - 1) return LL_ERR_SHAPE;
    if (N == 0) return LL_OK;
    if (!logits || !targets || !logp || !lse) return LL_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(logits) % esize(dtype)) return LL_ERR_ALIGN;
    DeviceGuard guard(logits);
    if (guard.err) return guard.err;
    DevInfo dev;
    int st = device_info(guard.dev, &dev);
    if (st) return st;
    Phase ph("logits_fwd", static_cast<cudaStream_t>(stream));
    return cuda_status(launch_logits_fwd(logits, ld, dtype, targets, N, V, logp, lse, it,
                                         static_cast<cudaStream_t>(stream)));
}

int logits_logp_bwd(const float* grad_logp, const void* logits, int64_t ld, int dtype,
                    const int64_t* targets, const float* lse, int64_t N, int64_t V,
                    void* grad_logits, void* stream) {
    return logits_logp_bwd_ex(grad_logp, logits, ld, dtype, targets, lse, N, V, grad_logits,
                              nullptr, stream);
}

int logits_logp_bwd_ex(const float* grad_logp, const void* logits, int64_t ld, int dtype,
                       const int64_t* targets, const float* lse, int64_t N, int64_t V,
                       void* grad_logits, const ll_options* opt, void* stream) {
    float it;
    if (read_options(opt, &it)) return LL_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return LL_ERR_DTYPE;
    if (N < 0 || V < 1 || V > kMaxV || ld < V || N > (int64_t(1) << 31) - 1) return LL_ERR_SHAPE;
    if (N == 0) return LL_OK;
    if (!grad_logp || !logits || !targets || !lse || !grad_logits) return LL_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(logits) % esize(dtype) ||
        reinterpret_cast<uintptr_t>(grad_logits) % esize(dtype))
        return LL_ERR_ALIGN;
    const char* a = static_cast<const char*>(logits);
    const char* b = static_cast<const char*>(grad_logits);
    const size_t span = size_t(N) * size_t(ld) * esize(dtype);
    if (a < b + span && b < a + span) return LL_ERR_INVALID_ARG;  // no aliasing
    DeviceGuard guard(logits);
    if (guard.err) return guard.err;
    DevInfo dev;
    int st = device_info(guard.dev, &dev);
    if (st) return st;
    Phase ph("logits_bwd", static_cast<cudaStream_t>(stream));
    return cuda_status(launch_logits_bwd(grad_logp, logits, ld, dtype, targets, lse, N, V,
                                         grad_logits, it, static_cast<cudaStream_t>(stream)));
}

int logits_logp_fwd_bwd(const float* grad_logp, const void* logits, int64_t ld, int dtype,
                        const int64_t* targets, int64_t N, int64_t V, float* logp, float* lse,
                        void* grad_logits, void* stream) {
    return logits_logp_fwd_bwd_ex(grad_logp, logits, ld, dtype, targets, N, V, logp, lse,
                                  grad_logits, nullptr, stream);
}

int logits_logp_fwd_bwd_ex(const float* grad_logp, const void* logits, int64_t ld, int dtype,
                           const int64_t* targets, int64_t N, int64_t V, float* logp,
                           float* lse, void* grad_logits, const ll_options* opt,
                           void* stream) {
    float it;
    if (read_options(opt, &it)) return LL_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return LL_ERR_DTYPE;
    if (N < 0 || V < 1 || V > kMaxV || ld < V || N > (int64_t(1) << 31) - 1) return LL_ERR_SHAPE;
    if (N == 0) return LL_OK;
    if (!grad_logp || !logits || !targets || !logp || !lse || !grad_logits)
        return LL_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(logits) % esize(dtype) ||
        reinterpret_cast<uintptr_t>(grad_logits) % esize(dtype))
        return LL_ERR_ALIGN;
    const char* a = static_cast<const char*>(logits);
    const char* b = static_cast<const char*>(grad_logits);
    const size_t span = size_t(N) * size_t(ld) * esize(dtype);
    // in place (the same buffer) or apart; a partial overlap is refused
    if (a != b && a < b + span && b < a + span) return LL_ERR_INVALID_ARG;
    DeviceGuard guard(logits);
    if (guard.err) return guard.err;
    DevInfo dev;
    int st = device_info(guard.dev, &dev);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Phase ph("logits_fused", s);
    return cuda_status(launch_logits_fused(grad_logp, logits, ld, dtype, targets, N, V, logp, lse,
                                           grad_logits, it, dev, s));
}

int ll_sum_ordered(const void* parts, int64_t nparts, int64_t n, int64_t ld, int dtype,
                   void* out, void* stream) {
    if (!dtype_ok(dtype)) return LL_ERR_DTYPE;
    if (nparts < 0 || n < 0 || ld < n) return LL_ERR_SHAPE;
    if (n == 0) return LL_OK;
    if (nparts == 0 || !parts || !out) return LL_ERR_INVALID_ARG;
    const char* p0 = static_cast<const char*>(parts);
    const char* p1 = p0 + size_t(nparts) * size_t(ld) * esize(dtype);
    const char* o0 = static_cast<const char*>(out);
    const char* o1 = o0 + size_t(n) * esize(dtype);
    if (o0 < p1 && p0 < o1) return LL_ERR_INVALID_ARG;  // out may not overlap the parts
    DeviceGuard guard(parts);
    if (guard.err) return guard.err;
    DevInfo dev;
    int st = device_info(guard.dev, &dev);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Phase ph("sum_ordered", s);
    return cuda_status(launch_sum_ordered(parts, nparts, n, ld, dtype, out, dev.num_sms, s));
}

int ll_check_status(void* stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LL_ERR_CUDA;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return cuda_status(cudaGetLastError());
    DevInfo info;
    int st = device_info(dev, &info);
    if (st) return st;
    int v = 0;
    if (cudaMemcpy(&v, info.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return LL_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        cudaMemcpy(info.status, &zero, sizeof(int), cudaMemcpyHostToDevice);
    }
    return v;
}

long long ll_launch_count(void) { return g_launches.load(); }

void ll_profile_enable(int on) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (auto& r : g_prof) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    g_prof.clear();
    g_prof_on.store(on ? 1 : 0);
}

int ll_profile_summary(char* buf, size_t len) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    std::vector<std::string> labels;
    std::vector<double> total;
    std::vector<long> count;
    for (auto& r : g_prof) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) return -LL_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return -LL_ERR_CUDA;
        size_t i = 0;
        while (i < labels.size() && labels[i] != r.label) ++i;
        if (i == labels.size()) {
            labels.push_back(r.label);
            total.push_back(0.0);
            count.push_back(0);
        }
        total[i] += ms;
        count[i] += 1;
    }
    std::string out;
    char line[160];
    for (size_t i = 0; i < labels.size(); ++i) {
        snprintf(line, sizeof(line), "%s %ld %.6f\n", labels[i].c_str(), count[i], total[i]);
        out += line;
    }
    if (buf && len) {
        strncpy(buf, out.c_str(), len - 1);
        buf[len - 1] = 0;
    }
    return static_cast<int>(labels.size());
}

int ll_debug_unsatisfied_wait(int* device_flag, void* stream) {
    if (!device_flag) return LL_ERR_INVALID_ARG;
    DeviceGuard guard(device_flag);
    if (guard.err) return guard.err;
    DevInfo dev;
    int st = device_info(guard.dev, &dev);
    if (st) return st;
    return cuda_status(launch_unsatisfied_wait(device_flag, dev.status, wait_limit_ns(),
                                               static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
