// Internal interface of the recurrent decode step (nha_decode.cu).
#pragma once

#include <cuda_runtime.h>

#include "nha_common.cuh"

namespace nha {

// Decode step for token t.  q, k, v, o [BH, D] in the element type; la
// [BH, M]; SK, SV [BH, M, D] fp32, updated in place; ring_k, ring_v
// [BH, max(w, 1), D] in the element type and ring_la [BH, max(w, 1), M] fp32,
// token s in entry s mod w (not used when w = 0).  With tpos, sequence b's
// heads decode their own position tpos[b]; a head whose position lies outside
// [0, 2^18) gets o = NaN and its state and ring are left untouched.  With
// wvec, head h keeps a window of wvec[h] tokens in the first wvec[h] entries
// of its w-entry ring (same NaN rule for a window outside [0, w]).
struct DecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* la;
    void* o;
    float* SK;
    float* SV;
    void* ring_k;
    void* ring_v;
    float* ring_la;
    int BH, t, w;
    const int* tpos;  // if set: device array [B] of per-sequence positions (t unused)
    const int* wvec;  // if set: device array [H] of per-head windows in [0, w] (w = the ring's length)
    int H;            // heads per sequence (b = bh / H indexes tpos)
    int sms;          // multiprocessors of the device (sizes the clusters)
    int overlap;      // the kernel before this launch writes none of its states and ring: stream them in early
    RopeTab rope;
};

template <typename Tin, int D, int M>
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);

}  // namespace nha
