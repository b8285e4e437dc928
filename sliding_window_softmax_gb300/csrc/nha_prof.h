// Launch accounting and optional per-kernel CUDA-event timing.
#pragma once

#include <cuda_runtime.h>

namespace nha {

// Brackets one kernel launch: counts it and, while a profiling session is
// open, records CUDA events around it on the launch stream.
class LaunchScope {
  public:
    LaunchScope(const char* name, cudaStream_t s);
    ~LaunchScope();

  private:
    const char* name_;
    cudaStream_t s_;
    int slot_;
};

}  // namespace nha

#define NHA_LAUNCH(name, stream, ...)          \
    do {                                       \
        ::nha::LaunchScope scope_((name), (stream)); \
        __VA_ARGS__;                           \
    } while (0)
