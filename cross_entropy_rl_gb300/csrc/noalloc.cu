// ll_forward_noalloc: the forward for callers that cannot allocate device
// memory.
//
// Some callers have no way to call cudaMalloc: a host framework that hands a
// step only the buffers it planned ahead of time and forbids allocation
// while the step runs (an allocation can synchronise the device or break a
// fixed memory pool), or plugin code that has no access to the
// application's allocator.  They still own the inputs and outputs, but they
// cannot provide the forward's scratch workspace.  This entry point keeps
// that scratch in a fixed-size array inside the library image instead: every
// GPU that loads the library holds the array (kNoAllocScratchBytes) until the
// process exits.
//
// The array's name is only a host-side stand-in in host code, so its device
// address is looked up with cudaGetSymbolAddress, once per device, with that
// device current; the first call on a device does this set-up, so that first
// call should come before any stream capture.  The address is kept for the
// life of the process: do not call this entry point on a device after
// cudaDeviceReset of that device (the library's module, and the array with it,
// is reloaded at a new address).  All calls on a device share the one array
// and it keeps the last call's contents: the forward writes every scratch
// entry it reads before reading it, so nothing needs clearing, and calls that
// may overlap on the GPU (different streams, or host threads) race on it.
#include <stdio.h>

#include <mutex>

#include "ll_internal.h"

namespace ll {

// Scratch of the forward's per-(segment, row) partials and target logits.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64];

// Device address of the scratch on the current device `dev`.
int noalloc_scratch(int dev, void** out) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            fprintf(stderr, "ll_forward_noalloc: cudaGetSymbolAddress failed: %s\n",
                    cudaGetErrorString(e));
            return LL_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return LL_OK;
}

}  // namespace
}  // namespace ll

extern "C" int ll_forward_noalloc(const void* hidden, const void* weight, const void* bias,
                                  const int64_t* targets, int64_t N, int64_t D, int64_t V,
                                  int dtype, float* logp, float* lse, void* stream) {
    using namespace ll;
    // ll_forward's own argument checks, with no workspace: an invalid argument
    // gives ll_forward's error, N == 0 gives LL_OK with nothing launched, and
    // a valid problem that needs scratch gives LL_ERR_WORKSPACE.  Nothing
    // runs on the device in any of these cases.
    const int pre = ll_forward(hidden, weight, bias, targets, N, D, V, dtype, logp, lse,
                               nullptr, 0, stream);
    if (pre != LL_ERR_WORKSPACE) return pre;
    const size_t need = ll_workspace_size(N, D, V, dtype, 0, 0, 0);
    if (need > kNoAllocScratchBytes) {
        fprintf(stderr,
                "ll_forward_noalloc: N=%lld, V=%lld needs %zu bytes of scratch; the static "
                "scratch holds %zu (use ll_forward with a workspace)\n",
                static_cast<long long>(N), static_cast<long long>(V), need,
                kNoAllocScratchBytes);
        return LL_ERR_WORKSPACE;
    }
    // the device that owns the hidden states (ll_forward runs there), current
    // while the address is looked up
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, hidden) != cudaSuccess) {
        cudaGetLastError();
        return LL_ERR_INVALID_ARG;
    }
    if ((attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) ||
        attr.device < 0 || attr.device >= 64)
        return LL_ERR_INVALID_ARG;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(attr.device) != cudaSuccess)
        return LL_ERR_CUDA;
    void* scratch = nullptr;
    int st = noalloc_scratch(attr.device, &scratch);
    if (st == LL_OK)
        st = ll_forward(hidden, weight, bias, targets, N, D, V, dtype, logp, lse, scratch,
                        kNoAllocScratchBytes, stream);
    if (prev != attr.device) cudaSetDevice(prev);
    return st;
}
