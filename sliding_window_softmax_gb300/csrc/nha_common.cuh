// Shared device-side definitions of the NHA CUDA library (sm_103a).
//
// Notation (per (b,h) head; "Native Hybrid Attention for Efficient Sequence
// Modeling", Paper-Notes page, sections 关键设计/层内混合 and
// Chunkwise 并行计算):
//   T tokens, window w (clamped to T), R = T - w = number of tokens whose
//   long memory some query reads (query t reads the state after token
//   j = t - w).  State index space j is cut into chunks of C = 64; chunk c
//   covers j in [cC, cC + C) and its queries are t = j + w.  Queries t < w
//   (W0 = min(w, T) of them) see only the window: NL = ceil(W0 / C) leading
//   tiles.  Within a chunk, b is the chunk-local inclusive cumsum of
//   log_alpha per slot and G = b at the chunk's last row.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nha {

constexpr int kChunk = 64;

// theta_i / pi split into a 6-significant-bit head and an fp32 tail, so that
// pos * head is exact in fp32 for |pos| < 2^18 and the angle can be reduced
// modulo 2*pi exactly before sincospif.
struct RopeTab {
    float f_hi[64];
    float f_lo[64];
};

struct Shape {
    int BH;      // B * H
    int T;       // tokens
    int w;       // window, already clamped to [0, T]
    int R;       // T - w
    int NC;      // ceil(R / C): chunks of state index space
    int NL;      // ceil(min(w, T) / C): leading window-only query tiles
    int NKT;     // ceil(T / C): key tiles
    float sigma; // 1 / sqrt(d)
    // Layout of the per-head workspace arrays, the same for every head:
    int NCS;     // chunks per head in the [BH, NCS, ...] arrays (NC, or ceil(T / C) with per-head windows)
    int W0S;     // rows per head of the [BH, W0S, m] arrays of the queries t < w (the largest min(w, T))
    // Per-head windows (device [H], or [B * H] when wbh is set; or null):
    // head h = bh % H (or the pair bh) has window min(max(windows[.], 0), w);
    // w above is then the largest window.
    const int* windows;
    int H;
    int wbh;
    // Sequence lengths (device [B + 1] offsets, or null): sequence b = bh / H
    // holds T_b = seq[b + 1] - seq[b] tokens (clamped to [0, TS]) in the first
    // rows of its [TS] rows; the head's shape is that of a T_b-token call.
    const int* seq;
    int TS;      // rows per head in the [BH, TS, ...] token arrays: the call's T

    // The call's status word (device int): kernels OR in kStatus* bits for
    // conditions only the device sees; the call sets it to zero first.
    int* status;
};

// Status bits (include/nha.h: NHA_STATUS_*).
constexpr int kStatusTimeoutBit = 1;    // a bounded wait gave up; the results are void
constexpr int kStatusGateRangeBit = 2;  // a chunk's per-slot log_alpha sum fell below kGateRange
constexpr float kGateRange = -160.0f;   // the intra-chunk gate factorisation is exact in fp32 above it

// True when heads differ in shape (per-head windows or per-sequence lengths):
// grids are then sized for the largest head and CTAs past a head's own tiles
// return at once.
__host__ __device__ __forceinline__ bool varied(const Shape& sh) { return sh.windows != nullptr || sh.seq != nullptr; }

// The shape seen by head bh: its own tokens and window and the counts that
// follow from them (the layout fields NCS, W0S, TS are the call's).
__device__ __forceinline__ Shape head_shape(const Shape& call, int bh) {
    Shape s = call;
    if (varied(call)) {
        int Tb = call.T;
        if (call.seq != nullptr) {
            const int b = bh / call.H;
            Tb = min(max(__ldg(call.seq + b + 1) - __ldg(call.seq + b), 0), call.TS);
        }
        int wh = call.w;
        if (call.windows != nullptr) wh = min(max(__ldg(call.windows + (call.wbh ? bh : bh % call.H)), 0), call.w);
        s.T = Tb;
        s.w = min(wh, Tb);
        s.R = Tb - s.w;
        s.NC = (s.R + kChunk - 1) / kChunk;
        s.NL = (s.w + kChunk - 1) / kChunk;
        s.NKT = (Tb + kChunk - 1) / kChunk;
    }
    return s;
}

__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float v) { *p = v; }
__device__ __forceinline__ void st(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// cos / sin of pos * theta_i.
__device__ __forceinline__ void rope_cs(const RopeTab& rt, int pos, int i, float& c, float& s) {
    float xh = (float)pos * rt.f_hi[i];       // exact (|pos| < 2^18, 6-bit head)
    xh = xh - 2.0f * rintf(0.5f * xh);        // exact reduction modulo 2 (i.e. 2*pi)
    float x = fmaf((float)pos, rt.f_lo[i], xh);
    sincospif(x, &s, &c);
}

__device__ __forceinline__ float warp_max4(float v) {
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
    return v;
}
__device__ __forceinline__ float warp_sum4(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    return v;
}

// exp(a - b) that returns 0 when a is -inf (covers an empty row so far, where
// b is -inf as well).
__device__ __forceinline__ float exp_diff(float a, float b) {
    return (a == -INFINITY) ? 0.0f : expf(a - b);
}

// Gate coefficients of one chunk (rows j0 .. j0 + nc - 1 of log_alpha).
// With b the chunk-local inclusive cumsum of log_alpha, G = b[nc-1] and the
// per-slot reference rho = G / 2:
//   Eq[r][i] = exp(b[r][i] - rho[i])              (query / row side)
//   Ek[r][i] = exp(rho[i] - b[r][i]) * u[r][i]     (key / column side)
//   Fk[r][i] = exp(rho[i] - b[r][i])               (optional)
// so that exp(b[r] - b[s]) u[s] = Eq[r] Ek[s] for every pair s <= r, with both
// factors bounded by exp(|G| / 2).  Rows r >= nc are zero.  Also writes
// sG[i] = G and sExpRho[i] = exp(rho).  Uses threads 0..M-1; the caller
// synchronises afterwards.
template <int M>
__device__ void chunk_gates(const float* __restrict__ la_rows, int nc, float* sEq, float* sEk,
                            float* sFk, int pitch, float* sG, float* sExpRho) {
    const int i = threadIdx.x;
    if (i < M) {
        float b = 0.0f;
        for (int r = 0; r < nc; r++) {
            float l = la_rows[(size_t)r * M + i];
            b += l;
            sEq[r * pitch + i] = b;
            sEk[r * pitch + i] = -expm1f(l);
        }
        const float G = nc > 0 ? b : 0.0f;
        const float rho = 0.5f * G;
        for (int r = 0; r < kChunk; r++) {
            if (r < nc) {
                float br = sEq[r * pitch + i];
                float f = expf(rho - br);
                sEq[r * pitch + i] = expf(br - rho);
                sEk[r * pitch + i] = f * sEk[r * pitch + i];
                if (sFk) sFk[r * pitch + i] = f;
            } else {
                sEq[r * pitch + i] = 0.0f;
                sEk[r * pitch + i] = 0.0f;
                if (sFk) sFk[r * pitch + i] = 0.0f;
            }
        }
        sG[i] = G;
        sExpRho[i] = expf(rho);
    }
}

// Rows [row0, row0 + n) of a [T, D] tensor into shared memory (fp32, row
// pitch `pitch`), zero-filling rows n .. kChunk-1.  With rope != nullptr the rows
// are rotated by RoPE at absolute positions row0 + r.
template <typename Tin, int D>
__device__ void load_rows(const Tin* __restrict__ src, int row0, int n, float* dst, int pitch,
                          const RopeTab* rope) {
    constexpr int H = D / 2;
    if (rope == nullptr) {
        for (int e = threadIdx.x; e < kChunk * D; e += blockDim.x) {
            int r = e / D, c = e % D;
            dst[r * pitch + c] = (r < n) ? ld(src + (size_t)(row0 + r) * D + c) : 0.0f;
        }
    } else {
        for (int e = threadIdx.x; e < kChunk * H; e += blockDim.x) {
            int r = e / H, i = e % H;
            float a = 0.0f, b = 0.0f;
            if (r < n) {
                const Tin* row = src + (size_t)(row0 + r) * D;
                float x = ld(row + i), y = ld(row + i + H), cs, sn;
                rope_cs(*rope, row0 + r, i, cs, sn);
                a = x * cs - y * sn;
                b = y * cs + x * sn;
            }
            dst[r * pitch + i] = a;
            dst[r * pitch + i + H] = b;
        }
    }
}

}  // namespace nha
