// nha_forward_noalloc: the forward with its scratch in a fixed device array
// compiled into the library, for callers that must not allocate device memory
// (code under an allocator that is owned by someone else, or plugins that
// receive only input and output buffers from their host).  The operation itself is nha_forward's.
#include <cudaTypedefs.h>

#include <mutex>

#include "nha.h"
#include "nha_kernels.h"

namespace {

constexpr size_t kScratchBytes = (size_t)NHA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch.  Every GPU that loads the library holds it until the process
// exits.  In host code this name is only a stand-in; the device address comes
// from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char nha_noalloc_scratch[NHA_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
// Per device: the context the address was looked up in, and the address.  A
// new primary context (after cudaDeviceReset) reloads the module, so the
// lookup is repeated whenever the current context differs.
void* g_ctx[kMaxDevices] = {nullptr};
void* g_addr[kMaxDevices] = {nullptr};
PFN_cuCtxGetCurrent_v4000 g_get_ctx = nullptr;
std::once_flag g_get_ctx_once;

void resolve_get_ctx() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_get_ctx = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
}

}  // namespace

extern "C" nha_status_t nha_forward_noalloc(const void* q, const void* k, const void* v,
                                            const float* log_alpha, void* o, float* lse, int B, int H, int T,
                                            int d, int m, int w, int C, nha_dtype_t dtype, float rope_base,
                                            void* stream) {
    // Validation only: with no workspace nha_forward returns before enqueuing
    // anything -- NHA_OK for an empty problem, NHA_ERR_WORKSPACE for a valid
    // one, or the argument's own error.
    const nha_status_t st = nha_forward(q, k, v, log_alpha, o, lse, B, H, T, d, m, w, C, dtype, rope_base,
                                        nullptr, 0, nullptr);
    if (st != NHA_ERR_WORKSPACE) return st;
    const size_t need = nha_workspace_bytes(B, H, T, d, m, w, C, dtype, 0);
    if (need > kScratchBytes)
        return nha::set_error(NHA_ERR_WORKSPACE,
                              "nha_forward_noalloc: this shape needs %zu bytes of scratch, the built-in "
                              "scratch holds %zu; call nha_forward with a workspace instead",
                              need, kScratchBytes);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nha::set_error(NHA_ERR_CUDA, "nha_forward_noalloc: no usable current device");
    std::call_once(g_get_ctx_once, resolve_get_ctx);
    if (g_get_ctx == nullptr)
        return nha::set_error(NHA_ERR_CUDA, "nha_forward_noalloc: cuCtxGetCurrent is not available");
    CUcontext ctx = nullptr;  // null until the runtime has set up the device's context
    if (g_get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    void* ptr = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (ctx == nullptr || g_addr[dev] == nullptr || g_ctx[dev] != (void*)ctx) {
            void* p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, nha_noalloc_scratch);
            if (e != cudaSuccess || p == nullptr)
                return nha::set_error(NHA_ERR_CUDA, "nha_forward_noalloc: cudaGetSymbolAddress failed: %s",
                                      cudaGetErrorString(e));
            // the lookup has made the device's primary context current
            if (g_get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr)
                return nha::set_error(NHA_ERR_CUDA, "nha_forward_noalloc: no current CUDA context");
            g_addr[dev] = p;
            g_ctx[dev] = (void*)ctx;
        }
        ptr = g_addr[dev];
    }
    return nha_forward(q, k, v, log_alpha, o, lse, B, H, T, d, m, w, C, dtype, rope_base, ptr, kScratchBytes,
                       stream);
}
