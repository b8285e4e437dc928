// Decode state after a prompt ("Native Hybrid Attention for Efficient Sequence
// Modeling", Paper-Notes page, 关键设计/层内混合: the K^long recurrence with
// the token shift).  After T tokens the long memory holds tokens 0 .. T-w-1,
// each absorbed with its own gate, and the window holds the last w tokens:
// exactly what the decode step of token T reads.
//
// One CTA per (head, K or V), 8 d threads: thread (column c, slot group)
// carries m/8 slot entries of column c in registers through the absorbed
// tokens in order; the tokens' rows and gates are staged in shared memory a
// chunk at a time (alpha and 1 - alpha formed once per token and slot).  The
// same CTA copies the last w tokens into the ring.
#include "nha_common.cuh"
#include "nha_prefill.h"
#include "nha_prof.h"

namespace nha {

namespace {
constexpr int kPrefillChunk = 32;  // tokens staged at once

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
}  // namespace

template <typename Tin, int D, int M>
__global__ void __launch_bounds__(8 * D) prefill_state_kernel(const PrefillArgs a) {
    constexpr int NT = 8 * D, SPT = M / 8;
    __shared__ float s_al[kPrefillChunk][M], s_u[kPrefillChunk][M], s_x[kPrefillChunk][D];
    const int bh = blockIdx.x >> 1, which = blockIdx.x & 1;  // which: 0 = K, 1 = V
    const int tid = threadIdx.x, c = tid % D, ig = tid / D;  // slots ig * SPT .. ig * SPT + SPT - 1
    const int T = a.T, w = a.wvec ? a.wvec[bh % a.H] : a.w;  // this head's window
    const size_t wst = a.w > 0 ? a.w : 1;                       // ring entries per head in memory
    const Tin* X = (const Tin*)(which ? a.v : a.k) + (size_t)bh * T * D;
    const float* la = a.la + (size_t)bh * T * M;
    if (w < 0 || w > a.w) {  // a window outside the ring: NaN states, ring untouched
        float* out = (which ? a.SV : a.SK) + (size_t)bh * M * D;
        for (int x = tid; x < M * D; x += NT) out[x] = __int_as_float(0x7fc00000);
        return;
    }
    const int J = T - w;  // tokens 0 .. J - 1 have left the window
    float S[SPT];
#pragma unroll
    for (int q = 0; q < SPT; q++) S[q] = 0.0f;
    for (int c0 = 0; c0 < J; c0 += kPrefillChunk) {
        const int n = min(kPrefillChunk, J - c0);
        __syncthreads();  // the previous chunk is consumed
        for (int x = tid; x < n * M; x += NT) {
            const int r = x / M, i = x % M;
            const float l = la[(size_t)(c0 + r) * M + i];
            s_al[r][i] = expf(l);
            s_u[r][i] = -expm1f(l);
        }
        for (int x = tid; x < n * D; x += NT) {
            const int r = x / D, e = x % D;
            s_x[r][e] = to_f(X[(size_t)(c0 + r) * D + e]);
        }
        __syncthreads();
        for (int r = 0; r < n; r++) {
            const float xv = s_x[r][c];
#pragma unroll
            for (int q = 0; q < SPT; q++) {
                const int i = ig * SPT + q;
                S[q] = s_al[r][i] * S[q] + s_u[r][i] * xv;
            }
        }
    }
    float* out = (which ? a.SV : a.SK) + (size_t)bh * M * D;
#pragma unroll
    for (int q = 0; q < SPT; q++) out[(size_t)(ig * SPT + q) * D + c] = S[q];
    // the window: the last min(w, T) tokens, token s in ring entry s mod w
    if (w > 0) {
        const int s0 = max(0, T - w), n = T - s0;
        Tin* ring = (Tin*)(which ? a.ring_v : a.ring_k) + (size_t)bh * wst * D;
        for (int x = tid; x < n * D; x += NT) {
            const int s = s0 + x / D, e = x % D;
            ring[(size_t)(s % w) * D + e] = X[(size_t)s * D + e];
        }
        if (which == 0) {
            float* rl = a.ring_la + (size_t)bh * wst * M;
            for (int x = tid; x < n * M; x += NT) {
                const int s = s0 + x / M, i = x % M;
                rl[(size_t)(s % w) * M + i] = la[(size_t)s * M + i];
            }
        }
    }
}

template <typename Tin, int D, int M>
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t st) {
    if (a.BH == 0) return cudaSuccess;
    NHA_LAUNCH("decode_prefill", st,
               prefill_state_kernel<Tin, D, M><<<2 * a.BH, 8 * D, 0, st>>>(a));
    return cudaGetLastError();
}

#define NHA_PREFILL_INST(Tin, D, M) template cudaError_t launch_prefill<Tin, D, M>(const PrefillArgs&, cudaStream_t);
NHA_PREFILL_INST(float, 64, 16)
NHA_PREFILL_INST(float, 64, 32)
NHA_PREFILL_INST(float, 64, 64)
NHA_PREFILL_INST(float, 128, 16)
NHA_PREFILL_INST(float, 128, 32)
NHA_PREFILL_INST(float, 128, 64)
NHA_PREFILL_INST(__nv_bfloat16, 64, 16)
NHA_PREFILL_INST(__nv_bfloat16, 64, 32)
NHA_PREFILL_INST(__nv_bfloat16, 64, 64)
NHA_PREFILL_INST(__nv_bfloat16, 128, 16)
NHA_PREFILL_INST(__nv_bfloat16, 128, 32)
NHA_PREFILL_INST(__nv_bfloat16, 128, 64)

}  // namespace nha
