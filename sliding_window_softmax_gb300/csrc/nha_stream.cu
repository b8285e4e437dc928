// A second stream for kernels that do not depend on one another, joined to
// the caller's stream with events (stream capture records the fork and the
// join as graph edges).  One side stream and four events per host thread and
// device, created on first use and kept until the process exits.
#include "nha_kernels.h"

namespace nha {

namespace {
constexpr int kMaxDevices = 64;
thread_local Fork g_fork[kMaxDevices];
}  // namespace

cudaError_t get_fork(Fork** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    Fork& f = g_fork[dev];
    if (f.side == nullptr) {
        cudaStream_t s = nullptr;
        if ((e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking)) != cudaSuccess) return e;
        for (int k = 0; k < Fork::kEvents; k++)
            if ((e = cudaEventCreateWithFlags(&f.ev[k], cudaEventDisableTiming)) != cudaSuccess) return e;
        f.side = s;
    }
    *out = &f;
    return cudaSuccess;
}

cudaError_t fork_side(cudaStream_t main, Fork& f, int k) {
    cudaError_t e = cudaEventRecord(f.ev[k], main);
    if (e != cudaSuccess) return e;
    return cudaStreamWaitEvent(f.side, f.ev[k], 0);
}

cudaError_t join_side(cudaStream_t main, Fork& f, int k) {
    cudaError_t e = cudaEventRecord(f.ev[k], f.side);
    if (e != cudaSuccess) return e;
    return cudaStreamWaitEvent(main, f.ev[k], 0);
}

}  // namespace nha
