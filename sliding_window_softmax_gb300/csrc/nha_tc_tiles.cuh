// Shared-memory tile movers and synchronisation helpers of the tcgen05
// kernels (bf16 operands in the 128B-swizzled layout of nha_tc.cuh).
#pragma once

#include "nha_common.cuh"
#include "nha_tc.cuh"

namespace nha {
using namespace tc;

constexpr int kTcThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr long long kWaitCycles = 1LL << 32;  // about 2 s at 2 GHz

// u = 1 - exp(l) for l <= 0 without the cancellation of 1 - exp(l) near 0:
// for |l| < 1/16 the Taylor series of exp(l) - 1 to the cubic term (relative
// error below l^3 / 24, under 1e-5), else 1 - 2^(l log2 e) on the MUFU
// (relative error of the difference below 1e-6 there).
__device__ __forceinline__ float one_minus_exp(float l) {
    if (l > -0.0625f) return -l * fmaf(l, fmaf(l, 1.0f / 6.0f, 0.5f), 1.0f);
    return 1.0f - fexp(l);
}

__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
    uint4 u;
    u.x = pack_bf16(f[0], f[1]);
    u.y = pack_bf16(f[2], f[3]);
    u.z = pack_bf16(f[4], f[5]);
    u.w = pack_bf16(f[6], f[7]);
    return u;
}

// Rotate 8 (x, y) pairs; c[q] holds (cos, sin) of pairs 2q and 2q + 1.
__device__ __forceinline__ void rotate8v(float* x, float* y, const float4 (&c)[4]) {
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const float4 t = c[q];
        float a = x[2 * q], b = y[2 * q];
        x[2 * q] = a * t.x - b * t.y;
        y[2 * q] = b * t.x + a * t.y;
        a = x[2 * q + 1];
        b = y[2 * q + 1];
        x[2 * q + 1] = a * t.z - b * t.w;
        y[2 * q + 1] = b * t.z + a * t.w;
    }
}

// Rotate 8 (x, y) pairs by the angles whose (cos, sin) are at cs[0..7].
__device__ __forceinline__ void rotate8(float* x, float* y, const float2* __restrict__ cs) {
    const float4* c4 = reinterpret_cast<const float4*>(cs);
    float4 c[4];
#pragma unroll
    for (int q = 0; q < 4; q++) c[q] = __ldg(c4 + q);
    rotate8v(x, y, c);
}

// Store n (multiple of 8) fp32 values as bf16 into row `row` of a 128-row tile
// starting at column col0 (multiple of 8).
__device__ __forceinline__ void store_row(unsigned char* tile, int row, int col0, const float* v, int n) {
    for (int c = 0; c < n; c += 8)
        *reinterpret_cast<uint4*>(tile + sw_chunk(row, (col0 + c) >> 3, 128)) = pack8(v + c);
}

// Barrier over the tile threads: the whole CTA, or (kProd) the 256 tile
// threads alone, on hardware barrier 1, in kernels that add a producer warp.
template <bool kProd>
__device__ __forceinline__ void tile_sync() {
    if constexpr (kProd)
        named_sync(1, kTcThreads);
    else
        __syncthreads();
}

struct TcCtl {
    uint64_t* bar;
    uint32_t phase;
    int* s_abort;
    int* status;
    bool named = false;  // the 256 tile threads only (barrier 1), not the whole CTA
    // Wait for the MMAs committed last; uniform across the tile threads; false on timeout.
    __device__ bool wait() {
        const bool ok = mbar_wait(bar, phase, kWaitCycles);
        phase ^= 1u;
        fence_after_sync();
        if (named ? named_sync_or(1, kTcThreads, !ok) : __syncthreads_or(!ok)) {
            if (threadIdx.x == 0) atomicOr(status, kStatusTimeoutBit);
            return false;
        }
        return true;
    }
};

template <bool kProd = false>
__device__ __forceinline__ void sync_for_mma() {
    fence_async_smem();
    fence_before_sync();
    tile_sync<kProd>();
    fence_after_sync();
}


// Inclusive cumsum of x over the 64 rows of this thread's chunk (tile rows
// 0-63 or 64-127), for the HM slots i = h HM + jj.  s_tot: [4][M] scratch.
template <int M, bool kProd = false>
__device__ __forceinline__ void chunk_prefix(float (&x)[M / 2], float* s_tot, int warp, int lane, int h) {
    constexpr int HM = M / 2;
    const int wq = warp & 3;
#pragma unroll
    for (int jj = 0; jj < HM; jj++) {
        float v = x[jj];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += y;
        }
        x[jj] = v;
        if (lane == 31) s_tot[wq * M + h * HM + jj] = v;
    }
    tile_sync<kProd>();
    if (wq & 1)
#pragma unroll
        for (int jj = 0; jj < HM; jj++) x[jj] += s_tot[(wq - 1) * M + h * HM + jj];
    tile_sync<kProd>();
}

// Inclusive suffix sum of x over the 64 rows of this thread's chunk.
template <int M>
__device__ __forceinline__ void chunk_suffix(float (&x)[M / 2], float* s_tot, int warp, int lane, int h) {
    constexpr int HM = M / 2;
    const int wq = warp & 3;
#pragma unroll
    for (int jj = 0; jj < HM; jj++) {
        float v = x[jj];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_down_sync(0xffffffffu, v, off);
            if (lane + off < 32) v += y;
        }
        x[jj] = v;
        if (lane == 0) s_tot[wq * M + h * HM + jj] = v;
    }
    __syncthreads();
    if (!(wq & 1))
#pragma unroll
        for (int jj = 0; jj < HM; jj++) x[jj] += s_tot[(wq + 1) * M + h * HM + jj];
    __syncthreads();
}

// Gates of this thread's row: loads log_alpha (0 past the valid rows), the
// chunk-local cumsum b and the chunk totals sG[2][M] (zero for an empty chunk).
template <int M, bool kProd = false>
__device__ __forceinline__ void gates_from_l(const float (&l)[M / 2], float (&b)[M / 2], float* s_tot, float* sG,
                                             int warp, int lane, int h, int r, int nrows);

template <int M, bool kProd = false>
__device__ __forceinline__ void row_gates(const float* __restrict__ la_row, bool valid, float (&l)[M / 2],
                                          float (&b)[M / 2], float* s_tot, float* sG, int warp, int lane,
                                          int h, int r, int nrows) {
    constexpr int HM = M / 2;
#pragma unroll
    for (int jj = 0; jj < HM; jj += 4) {
        const float4 v = valid ? __ldg(reinterpret_cast<const float4*>(la_row + h * HM + jj))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        l[jj] = v.x; l[jj + 1] = v.y; l[jj + 2] = v.z; l[jj + 3] = v.w;
    }
    gates_from_l<M, kProd>(l, b, s_tot, sG, warp, lane, h, r, nrows);
}

// Same, with log_alpha of the tile's 128 rows already in shared memory: the
// fp32 [128][M] tile as TMA writes it in 32-column boxes of 16 KB with
// 128-byte swizzle (columns past M read as zero).
template <int M, bool kProd = false>
__device__ __forceinline__ void row_gates_tile(const unsigned char* tile, bool valid, float (&l)[M / 2],
                                               float (&b)[M / 2], float* s_tot, float* sG, int warp, int lane,
                                               int h, int r, int nrows) {
    constexpr int HM = M / 2;
#pragma unroll
    for (int jj = 0; jj < HM; jj += 4) {
        const int col = h * HM + jj, c = (col & 31) >> 2;
        const float4 v = valid ? *reinterpret_cast<const float4*>(tile + (col >> 5) * 16384 + r * 128 + ((c ^ (r & 7)) << 4))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        l[jj] = v.x; l[jj + 1] = v.y; l[jj + 2] = v.z; l[jj + 3] = v.w;
    }
    gates_from_l<M, kProd>(l, b, s_tot, sG, warp, lane, h, r, nrows);
}

template <int M, bool kProd>
__device__ __forceinline__ void gates_from_l(const float (&l)[M / 2], float (&b)[M / 2], float* s_tot, float* sG,
                                             int warp, int lane, int h, int r, int nrows) {
    constexpr int HM = M / 2;
#pragma unroll
    for (int jj = 0; jj < HM; jj++) b[jj] = l[jj];
    chunk_prefix<M, kProd>(b, s_tot, warp, lane, h);
    const int cc = r >> 6, last = min(nrows, 64 * (cc + 1)) - 1;
    if (r == last)
#pragma unroll
        for (int jj = 0; jj < HM; jj++) sG[cc * M + h * HM + jj] = b[jj];
    tile_sync<kProd>();
}

__device__ __forceinline__ void zero_cols(unsigned char* tile, int row, int c0, int c1) {
    for (int c = c0; c < c1; c += 8)
        *reinterpret_cast<uint4*>(tile + sw_chunk(row, c >> 3, 128)) = make_uint4(0, 0, 0, 0);
}

// Masked copy of 64 TMEM columns (this half's) into a bf16 tile row:
// keep (row, col) iff h == own chunk and (upper ? col >= row : col <= row).
__device__ __forceinline__ void mask_to_tile(uint32_t taddr, unsigned char* tile, int r, int h, int cr,
                                             bool row_ok, bool upper) {
    float vv[64];
    tmem_ld(taddr + 64 * h, vv, 64);
#pragma unroll
    for (int jj = 0; jj < 64; jj++) {
        const int col = 64 * h + jj;
        const bool keep = row_ok && h == cr && (upper ? col >= r : col <= r);
        if (!keep) vv[jj] = 0.0f;
    }
    store_row(tile, r, 64 * h, vv, 64);
}

}  // namespace nha
