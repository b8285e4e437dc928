// Internal interface of the decode-state prefill (nha_prefill.cu).
#pragma once

#include <cuda_runtime.h>

namespace nha {

// Decode state after a prompt of T tokens.  k, v [BH, T, D] in the element
// type, la [BH, T, M]; out: SK, SV [BH, M, D] fp32 = the long memory after
// token T - w - 1 (zero when T <= w), ring_k, ring_v [BH, max(w, 1), D] and
// ring_la [BH, max(w, 1), M] with token s in entry s mod w for
// s in [max(0, T - w), T - 1] (other entries untouched; no ring when w = 0).
// With wvec, head h uses window wvec[h] and ring entries s mod wvec[h] of its
// w-entry ring; a window outside [0, w] gives NaN states and no ring writes.
struct PrefillArgs {
    const void* k;
    const void* v;
    const float* la;
    float* SK;
    float* SV;
    void* ring_k;
    void* ring_v;
    float* ring_la;
    int BH, T, w;
    const int* wvec;  // if set: device array [H] of per-head windows in [0, w] (w = the ring's length)
    int H;
};

template <typename Tin, int D, int M>
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t st);

}  // namespace nha
