// Tensor-core (tcgen05) backward of the NHA window branch for bf16 inputs.
//
// With P = exp(S - lse) the window probabilities (S = RoPE(q) RoPE(k)^T / sqrt(d)
// over the band, lse from the forward), D_t = dout_t . o_t and
// dS = P o (dout V^T - D):
//   dq~ = sigma dS K~,   dk~ = sigma dS^T Q~,   dv = P^T dout
// in rotated coordinates, then dq = R_t^T dq~ and dk = R_s^T dk~.
// Two kernels, no atomics: a query-major one (dq) and a key-major one
// (dk, dv), each recomputing S and dP on the tensor core.
// D_t is needed exactly: the dlog_alpha reverse cumsum sums terms whose total
// is zero (the loss sees the cumulative gates only through differences), so
// an error in D from the bf16-rounded o accumulates along the sequence.  The
// query-major kernel therefore forms dS with D^ = dout . o_bf16, and also
// accumulates sum_s P dP (the window part of the exact D) and sum_s P k~; the
// slot-branch query kernel adds the slot part of D and corrects
// dq += sigma (D^ - D) R^T sum_s P k~.  The key-major kernel runs afterwards
// with the exact D.  Results are the window branch's fp32 partial gradients;
// the slot branch adds its own parts and writes the final outputs.
#include "nha_common.cuh"
#include "nha_kernels.h"
#include "nha_prof.h"
#include "nha_tc.cuh"
#include "nha_tc_tiles.cuh"

namespace nha {

// dot of two bf16 half rows (columns [h D/2, (h + 1) D/2))
template <int D>
__device__ __forceinline__ float half_row_dot(const __nv_bfloat16* __restrict__ x,
                                              const __nv_bfloat16* __restrict__ y, int h) {
    constexpr int HD = D / 2;
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < HD; c += 8) {
        float fx[8], fy[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(x + h * HD + c)), fx);
        unpack8(__ldg(reinterpret_cast<const uint4*>(y + h * HD + c)), fy);
#pragma unroll
        for (int i = 0; i < 8; i++) s += fx[i] * fy[i];
    }
    return s;
}

// Epilogue shared by both kernels: read the rotated-space gradient of this
// row from TMEM columns [col0, col0 + D), scale, rotate back by R_pos^T and
// write fp32.  Thread half h owns frequency pairs [h D/4, (h + 1) D/4).
template <int D>
__device__ __forceinline__ void store_unrotated(uint32_t taddr, bool valid_acc, float scale, int pos,
                                                bool row_ok, int h, const float2* __restrict__ tab,
                                                float* __restrict__ out) {
    constexpr int Q4 = D / 4, H = D / 2;
    float g0[Q4], g1[Q4];
    if (valid_acc) {
        tmem_ld(taddr + h * Q4, g0, Q4);
        tmem_ld(taddr + H + h * Q4, g1, Q4);
    } else {
#pragma unroll
        for (int i = 0; i < Q4; i++) g0[i] = g1[i] = 0.0f;
    }
    if (!row_ok) return;
    const float2* cs = tab + (size_t)pos * H + h * Q4;
#pragma unroll
    for (int i = 0; i < Q4; i += 4) {
        float4 lo, hi;
        float r0[4], r1[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const float2 c = __ldg(cs + i + j);
            const float a = g0[i + j] * scale, b = g1[i + j] * scale;
            r0[j] = a * c.x + b * c.y;
            r1[j] = b * c.x - a * c.y;
        }
        lo = make_float4(r0[0], r0[1], r0[2], r0[3]);
        hi = make_float4(r1[0], r1[1], r1[2], r1[3]);
        *reinterpret_cast<float4*>(out + h * Q4 + i) = lo;
        *reinterpret_cast<float4*>(out + H + h * Q4 + i) = hi;
    }
}

// ---------------------------------------------------------------------------------------
// Query-major: one CTA per (128 queries, head), all T queries.
template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
bwd_wdq_tc_kernel(const BwdArgs a, const float2* __restrict__ tab, int* __restrict__ status) {
    extern __shared__ unsigned char smem_raw[];
    constexpr int TB = 128 * D * 2;
    unsigned char* X0 = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* X1 = X0 + TB;  // K~ block
    unsigned char* X2 = X1 + TB;  // V block
    unsigned char* X3 = X2 + TB;  // dout tile
    unsigned char* X4 = X3 + TB;      // dS [128 q][128 keys]
    unsigned char* X5 = X4 + 32768;   // P  [128 q][128 keys]
    float* red = reinterpret_cast<float*>(X5 + 32768);  // [2][128]
    __shared__ uint64_t bar;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const Shape sh = a.sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = ((warp & 3) << 5) | lane, h = warp >> 2;
    const int tbase = blockIdx.x * 128, nq = min(128, sh.T - tbase), bh = blockIdx.y;
    const size_t hoff = (size_t)bh * sh.T;
    const __nv_bfloat16* k = (const __nv_bfloat16*)a.k + hoff * D;
    const __nv_bfloat16* v = (const __nv_bfloat16*)a.v + hoff * D;
    const __nv_bfloat16* dout = (const __nv_bfloat16*)a.dout + hoff * D;
    const float sig2 = sh.sigma * kLog2e;
    const int t = tbase + r;
    const bool row_ok = r < nq;

    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
        s_abort = 0;
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    load_tile<D>((const __nv_bfloat16*)a.q + hoff * D, tbase, nq, X0, tab);
    load_tile<D>(dout, tbase, nq, X3, nullptr);
    const float dpart = row_ok ? half_row_dot<D>(dout + (size_t)t * D, (const __nv_bfloat16*)a.o + (hoff + t) * D, h) : 0.0f;
    red[h * 128 + r] = dpart;
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t tS = 0, tP = 128, tQ = 256, tV = 384;
    const float Dr = red[r] + red[128 + r];  // from the bf16 o
    if (h == 0 && row_ok) a.Dhat[hoff + t] = Dr;
    float dwin = 0.0f;
    const float lse2 = row_ok ? a.lse[hoff + t] * kLog2e : 0.0f;
    TcCtl ctl{&bar, 0u, &s_abort, status};
    bool ok = true, acc = false;

    if (sh.w > 0) {
        const int klo = max(0, tbase - sh.w + 1), khi = tbase + nq - 1;
        for (int kb = klo; kb <= khi && ok; kb += 128) {
            const int nk = min(128, khi - kb + 1);
            load_tile<D>(k, kb, nk, X1, tab);
            load_tile<D>(v, kb, nk, X2, nullptr);
            sync_for_mma();
            if (tid == 0) {
                const uint32_t s0 = smem_u32(X0), s1 = smem_u32(X1), s2 = smem_u32(X2), s3 = smem_u32(X3);
                for (int kk = 0; kk < D / 16; kk++)
                    mma_bf16(tm + tS, desc_k(s0, 128, kk), desc_k(s1, 128, kk), idesc_bf16(128, 128, false), kk > 0);
                for (int kk = 0; kk < D / 16; kk++)
                    mma_bf16(tm + tP, desc_k(s3, 128, kk), desc_k(s2, 128, kk), idesc_bf16(128, 128, false), kk > 0);
                mma_commit(&bar);
            }
            ok = ctl.wait();
            if (!ok) break;
            float sv[64], dp[64];
            tmem_ld(tl + tS + 64 * h, sv, 64);
            tmem_ld(tl + tP + 64 * h, dp, 64);
#pragma unroll
            for (int jj = 0; jj < 64; jj++) {
                const int c = 64 * h + jj, key = kb + c;
                const bool valid = row_ok && c < nk && key <= t && key > t - sh.w;
                const float p = valid ? ex2(sv[jj] * sig2 - lse2) : 0.0f;
                dwin += p * dp[jj];
                sv[jj] = p * (dp[jj] - Dr);
                dp[jj] = p;
            }
            store_row(X4, r, 64 * h, sv, 64);
            store_row(X5, r, 64 * h, dp, 64);
            sync_for_mma();
            if (tid == 0) {
                const uint32_t s1 = smem_u32(X1), s4 = smem_u32(X4), s5 = smem_u32(X5);
                for (int kk = 0; kk < 8; kk++)
                    mma_bf16(tm + tQ, desc_k(s4, 128, kk), desc_mn(s1, 128, kk), idesc_bf16(128, D, true),
                             (acc || kk > 0) ? 1u : 0u);
                for (int kk = 0; kk < 8; kk++)
                    mma_bf16(tm + tV, desc_k(s5, 128, kk), desc_mn(s1, 128, kk), idesc_bf16(128, D, true),
                             (acc || kk > 0) ? 1u : 0u);
                mma_commit(&bar);
            }
            acc = true;
            ok = ctl.wait();
        }
    }
    red[h * 128 + r] = dwin;
    __syncthreads();
    if (h == 0 && row_ok) a.Dwin[hoff + t] = red[r] + red[128 + r];
    if (ok) {
        store_unrotated<D>(tl + tQ, acc, sh.sigma, t, row_ok, h, tab, a.dqw + (hoff + t) * D);
        store_unrotated<D>(tl + tV, acc, sh.sigma, t, row_ok, h, tab, a.dqwV + (hoff + t) * D);
    } else if (row_ok) {
        a.dqw[(hoff + t) * D + h] = __int_as_float(0x7fc00000);
    }
    if (!ok && tid == 0) mbar_wait(&bar, ctl.phase ^ 1u, kWaitCycles);
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

// ---------------------------------------------------------------------------------------
// Key-major: one CTA per (128 keys, head).  Row of the tile = key.
template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
bwd_wkv_tc_kernel(const BwdArgs a, const float2* __restrict__ tab, int* __restrict__ status) {
    extern __shared__ unsigned char smem_raw[];
    constexpr int TB = 128 * D * 2;
    unsigned char* X0 = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* X1 = X0 + TB;      // V tile (keys)
    unsigned char* X2 = X1 + TB;      // Q~ block
    unsigned char* X3 = X2 + TB;      // dout block
    unsigned char* X4 = X3 + TB;      // P^T [128 keys][128 q]
    unsigned char* X5 = X4 + 32768;   // dS^T
    float* sL2 = reinterpret_cast<float*>(X5 + 32768);  // [128] lse (log2 domain)
    float* sD = sL2 + 128;                                // [128]
    __shared__ uint64_t bar;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const Shape sh = a.sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rk = ((warp & 3) << 5) | lane, h = warp >> 2;
    const int sbase = blockIdx.x * 128, nk = min(128, sh.T - sbase), bh = blockIdx.y;
    const size_t hoff = (size_t)bh * sh.T;
    const __nv_bfloat16* q = (const __nv_bfloat16*)a.q + hoff * D;
    const __nv_bfloat16* dout = (const __nv_bfloat16*)a.dout + hoff * D;
    const float sig2 = sh.sigma * kLog2e;
    const int key = sbase + rk;
    const bool row_ok = rk < nk;

    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
        s_abort = 0;
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    load_tile<D>((const __nv_bfloat16*)a.k + hoff * D, sbase, nk, X0, tab);
    load_tile<D>((const __nv_bfloat16*)a.v + hoff * D, sbase, nk, X1, nullptr);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t tS = 0, tP = 128, tV = 256, tK = 256 + D;
    TcCtl ctl{&bar, 0u, &s_abort, status};
    bool ok = true, acc = false;

    if (sh.w > 0) {
        const int thi = min(sh.T - 1, sbase + nk - 1 + sh.w - 1);
        for (int qb = sbase; qb <= thi && ok; qb += 128) {
            const int nq = min(128, thi - qb + 1);
            load_tile<D>(q, qb, nq, X2, tab);
            load_tile<D>(dout, qb, nq, X3, nullptr);
            if (tid < 128) {
                sL2[tid] = tid < nq ? a.lse[hoff + qb + tid] * kLog2e : 0.0f;
                sD[tid] = tid < nq ? a.Dv[hoff + qb + tid] : 0.0f;
            }
            sync_for_mma();
            if (tid == 0) {
                const uint32_t s0 = smem_u32(X0), s1 = smem_u32(X1), s2 = smem_u32(X2), s3 = smem_u32(X3);
                for (int kk = 0; kk < D / 16; kk++)
                    mma_bf16(tm + tS, desc_k(s0, 128, kk), desc_k(s2, 128, kk), idesc_bf16(128, 128, false), kk > 0);
                for (int kk = 0; kk < D / 16; kk++)
                    mma_bf16(tm + tP, desc_k(s1, 128, kk), desc_k(s3, 128, kk), idesc_bf16(128, 128, false), kk > 0);
                mma_commit(&bar);
            }
            ok = ctl.wait();
            if (!ok) break;
            float sv[64], dp[64];
            tmem_ld(tl + tS + 64 * h, sv, 64);
            tmem_ld(tl + tP + 64 * h, dp, 64);
#pragma unroll
            for (int jj = 0; jj < 64; jj++) {
                const int c = 64 * h + jj, t = qb + c;
                const bool valid = row_ok && c < nq && key <= t && key > t - sh.w;
                const float p = valid ? ex2(sv[jj] * sig2 - sL2[c]) : 0.0f;
                sv[jj] = p;
                dp[jj] = p * (dp[jj] - sD[c]);
            }
            store_row(X4, rk, 64 * h, sv, 64);
            store_row(X5, rk, 64 * h, dp, 64);
            sync_for_mma();
            if (tid == 0) {
                const uint32_t s2 = smem_u32(X2), s3 = smem_u32(X3), s4 = smem_u32(X4), s5 = smem_u32(X5);
                for (int kk = 0; kk < 8; kk++)
                    mma_bf16(tm + tV, desc_k(s4, 128, kk), desc_mn(s3, 128, kk), idesc_bf16(128, D, true),
                             (acc || kk > 0) ? 1u : 0u);
                for (int kk = 0; kk < 8; kk++)
                    mma_bf16(tm + tK, desc_k(s5, 128, kk), desc_mn(s2, 128, kk), idesc_bf16(128, D, true),
                             (acc || kk > 0) ? 1u : 0u);
                mma_commit(&bar);
            }
            acc = true;
            ok = ctl.wait();
        }
    }
    if (ok) {
        // dv: plain copy of this half row
        constexpr int HD = D / 2;
        float* ov = a.dvw + (hoff + key) * D + h * HD;
        for (int c0 = 0; c0 < HD; c0 += 32) {
            float vv[32];
            if (acc) {
                tmem_ld32(tl + tV + h * HD + c0, vv);
            } else {
#pragma unroll
                for (int i = 0; i < 32; i++) vv[i] = 0.0f;
            }
            if (row_ok)
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<float4*>(ov + c0 + i) = make_float4(vv[i], vv[i + 1], vv[i + 2], vv[i + 3]);
        }
        store_unrotated<D>(tl + tK, acc, sh.sigma, key, row_ok, h, tab, a.dkw + (hoff + key) * D);
    } else if (row_ok) {
        a.dkw[(hoff + key) * D + h] = __int_as_float(0x7fc00000);
    }
    if (!ok && tid == 0) mbar_wait(&bar, ctl.phase ^ 1u, kWaitCycles);
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

template <int D>
size_t wdq_smem() { return 1024 + 4 * 128 * D * 2 + 2 * 32768 + 256 * sizeof(float); }
template <int D>
size_t wkv_smem() { return 1024 + 4 * 128 * D * 2 + 2 * 32768 + 256 * sizeof(float); }

template <int D, int M>
cudaError_t tc_backward(const BwdArgs& a, float2* tab, int* status, cudaStream_t st) {
    const Shape& sh = a.sh;
    cudaError_t e = tc_states<D, M>((const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v, a.la, a.SK, a.SV, a.G,
                                    sh, status, st);
    if (e != cudaSuccess) return e;
    if ((e = launch_rope_table(tab, sh.T, D / 2, a.rope, st)) != cudaSuccess) return e;
    const dim3 grid((sh.T + 127) / 128, sh.BH);
    {
        auto kern = bwd_wdq_tc_kernel<D>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wdq_smem<D>())) != cudaSuccess)
            return e;
        NHA_LAUNCH("bwd_wdq_tc", st, kern<<<grid, kTcThreads, wdq_smem<D>(), st>>>(a, tab, status));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return tc_bwd_slot<D, M>(a, tab, status, st);
}

template <int D>
cudaError_t launch_wkv(const BwdArgs& a, const float2* tab, int* status, cudaStream_t st) {
    const dim3 grid((a.sh.T + 127) / 128, a.sh.BH);
    auto kern = bwd_wkv_tc_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wkv_smem<D>());
    if (e != cudaSuccess) return e;
    NHA_LAUNCH("bwd_wkv_tc", st, kern<<<grid, kTcThreads, wkv_smem<D>(), st>>>(a, tab, status));
    return cudaGetLastError();
}
template cudaError_t launch_wkv<64>(const BwdArgs&, const float2*, int*, cudaStream_t);
template cudaError_t launch_wkv<128>(const BwdArgs&, const float2*, int*, cudaStream_t);

#define NHA_TCB_INST(D, M) template cudaError_t tc_backward<D, M>(const BwdArgs&, float2*, int*, cudaStream_t);
NHA_TCB_INST(64, 16)
NHA_TCB_INST(64, 32)
NHA_TCB_INST(64, 64)
NHA_TCB_INST(128, 16)
NHA_TCB_INST(128, 32)
NHA_TCB_INST(128, 64)

}  // namespace nha
