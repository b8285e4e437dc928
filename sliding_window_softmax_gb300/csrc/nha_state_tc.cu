// Slot states at chunk boundaries for the bf16 path.
//
// Per chunk c (C = 64 state indices) the contribution to the state at the
// chunk's end is dS_c = U_c^T X_c with U_c[s][i] = exp(G_i - b_{s,i}) u_{s,i}
// ("Native Hybrid Attention for Efficient Sequence Modeling", Paper-Notes page,
// 关键设计/层内混合: K^long_t = Diag(alpha_t) K^long_{t-1} + (1 - alpha_t) (x) k_t,
// unrolled over one chunk), for X = K and X = V.  A 128-row tile holds two
// chunks; the tensor core forms dS^T = X^T [U_c1 | U_c2] (d rows, 2m columns)
// in one MMA per tensor.  A second kernel scans the chunks:
// S_prev(c + 1) = exp(G_c) S_prev(c) + dS_c.
#include "nha_common.cuh"
#include "nha_kernels.h"
#include "nha_prof.h"
#include "nha_tc.cuh"
#include "nha_tc_tiles.cuh"

namespace nha {

template <int D, int M>
__global__ void __launch_bounds__(kTcThreads, 1)
state_tc_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                const float* __restrict__ la, float* __restrict__ SK, float* __restrict__ SV,
                float* __restrict__ G, Shape sh, int* __restrict__ status) {
    constexpr int HM = M / 2;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* XK = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* XV = XK + 32768;  // [128 s][128 d] (d >= D zero)
    unsigned char* XU = XV + 32768;  // [128 s][2M] chunk-blocked coefficients
    float* s_tot = reinterpret_cast<float*>(XU + 32768);  // [4][M]
    float* sG = s_tot + 4 * M;                             // [2][M]
    __shared__ uint64_t bar;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = ((warp & 3) << 5) | lane, h = warp >> 2, cr = r >> 6;
    const int bh = blockIdx.y, j0 = blockIdx.x * 128, n = min(128, sh.R - j0);
    const int c1 = j0 / kChunk;
    const bool has2 = n > kChunk, row_ok = r < n;
    const size_t hoff = (size_t)bh * sh.T;

    if (tid < 2 * M) sG[tid] = 0.0f;
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
        s_abort = 0;
    }
    if (warp == 0) tmem_alloc(&s_tmem, 256);
    load_tile<D>(k + hoff * D, j0, n, XK, nullptr);
    load_tile<D>(v + hoff * D, j0, n, XV, nullptr);
    if (D < 128) {  // the MMA reads 128 columns of d: zero the unused block
        for (int e = tid; e < 128 * 8; e += kTcThreads) {
            const int rr = e >> 3, ch = 8 + (e & 7);
            *reinterpret_cast<uint4*>(XK + sw_chunk(rr, ch, 128)) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(XV + sw_chunk(rr, ch, 128)) = make_uint4(0, 0, 0, 0);
        }
    }
    // gates of this row: b = chunk-local inclusive cumsum, G = chunk total
    float l[HM], b[HM];
#pragma unroll
    for (int jj = 0; jj < HM; jj += 4) {
        const float4 q = row_ok ? __ldg(reinterpret_cast<const float4*>(la + (hoff + j0 + r) * M + h * HM + jj))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        l[jj] = q.x; l[jj + 1] = q.y; l[jj + 2] = q.z; l[jj + 3] = q.w;
    }
#pragma unroll
    for (int jj = 0; jj < HM; jj++) b[jj] = l[jj];
    chunk_prefix<M>(b, s_tot, warp, lane, h);
    {
        const int last = min(n, 64 * (cr + 1)) - 1;
        if (r == last)
#pragma unroll
            for (int jj = 0; jj < HM; jj++) sG[cr * M + h * HM + jj] = b[jj];
    }
    __syncthreads();
    {
        float u[HM], z[HM];
#pragma unroll
        for (int jj = 0; jj < HM; jj++) {
            u[jj] = row_ok ? fexp(sG[cr * M + h * HM + jj] - b[jj]) * (-expm1f(l[jj])) : 0.0f;
            z[jj] = 0.0f;
        }
        store_row(XU, r, cr * M + h * HM, u, HM);
        store_row(XU, r, (1 - cr) * M + h * HM, z, HM);
    }
    if (tid < 2 * M) {
        const int cc = tid / M;
        if (cc == 0 || has2) G[((size_t)bh * sh.NC + c1 + cc) * M + (tid % M)] = sG[tid];
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = s_tmem;
    if (tid == 0) {
        const uint32_t sk = smem_u32(XK), sv = smem_u32(XV), su = smem_u32(XU);
        for (int kk = 0; kk < 8; kk++)
            mma_bf16(tm, desc_mn(sk, 128, kk), desc_mn(su, 128, kk), idesc_bf16(128, 2 * M, true) | (1u << 15), kk > 0);
        for (int kk = 0; kk < 8; kk++)
            mma_bf16(tm + 128, desc_mn(sv, 128, kk), desc_mn(su, 128, kk), idesc_bf16(128, 2 * M, true) | (1u << 15), kk > 0);
        mma_commit(&bar);
    }
    const bool ok = mbar_wait(&bar, 0, kWaitCycles);
    fence_after_sync();
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            atomicExch(status, kStatusTimeout);
            mbar_wait(&bar, 0, kWaitCycles);
        }
    } else {
        // TMEM row = d; thread half h holds chunk h's M slots
        const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);
        const int d = r;
        const bool keep = d < D && (h == 0 || has2);
        float* dk = SK + ((size_t)bh * sh.NC + c1 + h) * M * D + d;
        float* dv = SV + ((size_t)bh * sh.NC + c1 + h) * M * D + d;
        for (int c0 = 0; c0 < M; c0 += (M < 32 ? M : 32)) {
            float vk[32], vv[32];
            tmem_ld(tl + h * M + c0, vk, M < 32 ? M : 32);
            tmem_ld(tl + 128 + h * M + c0, vv, M < 32 ? M : 32);
            if (keep)
                for (int i = 0; i < (M < 32 ? M : 32); i++) {
                    dk[(size_t)(c0 + i) * D] = vk[i];
                    dv[(size_t)(c0 + i) * D] = vv[i];
                }
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 256);
}

// Exclusive scan over chunks, in place (forward dir > 0 or reverse dir < 0),
// eight chunks of loads in flight per thread.  Same contract as the scan of
// the fp32 path; also writes a bf16 copy of every result (the operand the
// tensor-core kernels load).
__global__ void __launch_bounds__(256)
state_scan8_kernel(float* __restrict__ X0, float* __restrict__ X1, __nv_bfloat16* __restrict__ B0,
                   __nv_bfloat16* __restrict__ B1, const float* __restrict__ G, int NC, int M, int D, int dir) {
    const int e = 2 * (blockIdx.x * 256 + threadIdx.x);  // two adjacent elements of one slot row
    if (e >= M * D) return;
    const int bh = blockIdx.y, i = e / D;
    float* X = (blockIdx.z == 0) ? X0 : X1;
    __nv_bfloat16* Xb = (blockIdx.z == 0) ? B0 : B1;
    float2 S = make_float2(0.0f, 0.0f);
    for (int n0 = 0; n0 < NC; n0 += 8) {
        float2 x[8];
        float g[8];
#pragma unroll
        for (int q = 0; q < 8; q++) {
            const int n = n0 + q;
            const int c = dir > 0 ? n : NC - 1 - n;
            if (n < NC) {
                x[q] = *reinterpret_cast<const float2*>(X + ((size_t)bh * NC + c) * M * D + e);
                g[q] = G[((size_t)bh * NC + c) * M + i];
            }
        }
#pragma unroll
        for (int q = 0; q < 8; q++) {
            const int n = n0 + q;
            if (n < NC) {
                const int c = dir > 0 ? n : NC - 1 - n;
                const size_t o = ((size_t)bh * NC + c) * M * D + e;
                *reinterpret_cast<float2*>(X + o) = S;
                *reinterpret_cast<__nv_bfloat162*>(Xb + o) = __floats2bfloat162_rn(S.x, S.y);
                const float f = expf(g[q]);
                S.x = f * S.x + x[q].x;
                S.y = f * S.y + x[q].y;
            }
        }
    }
}

cudaError_t launch_scan8(float* X0, float* X1, __nv_bfloat16* B0, __nv_bfloat16* B1, const float* G,
                         const Shape& sh, int M, int D, int dir, cudaStream_t st) {
    NHA_LAUNCH(dir > 0 ? "state_scan" : "state_scan_rev", st,
               state_scan8_kernel<<<dim3((M * D / 2 + 255) / 256, sh.BH, 2), 256, 0, st>>>(X0, X1, B0, B1, G,
                                                                                           sh.NC, M, D, dir));
    return cudaGetLastError();
}

template <int D, int M>
cudaError_t tc_states(const __nv_bfloat16* k, const __nv_bfloat16* v, const float* la, float* SK, float* SV,
                      __nv_bfloat16* SKb, __nv_bfloat16* SVb, float* G, const Shape& sh, int* status,
                      cudaStream_t st) {
    if (sh.NC == 0) return cudaSuccess;
    const size_t sm = 1024 + 3 * 32768 + 6 * M * sizeof(float);
    auto kern = state_tc_kernel<D, M>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    NHA_LAUNCH("state_chunk", st,
               kern<<<dim3((sh.R + 127) / 128, sh.BH), kTcThreads, sm, st>>>(k, v, la, SK, SV, G, sh, status));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_scan8(SK, SV, SKb, SVb, G, sh, M, D, +1, st);
}

#define NHA_ST_INST(D, M)                                                                              \
    template cudaError_t tc_states<D, M>(const __nv_bfloat16*, const __nv_bfloat16*, const float*, float*, \
                                         float*, __nv_bfloat16*, __nv_bfloat16*, float*, const Shape&, int*,  \
                                         cudaStream_t);
NHA_ST_INST(64, 16)
NHA_ST_INST(64, 32)
NHA_ST_INST(64, 64)
NHA_ST_INST(128, 16)
NHA_ST_INST(128, 32)
NHA_ST_INST(128, 64)

}  // namespace nha
