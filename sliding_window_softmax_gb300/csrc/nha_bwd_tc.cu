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
// write bf16.  Thread half h owns frequency pairs [h D/4, (h + 1) D/4).
template <int D>
__device__ __forceinline__ void store_unrotated(uint32_t taddr, bool valid_acc, float scale, int pos,
                                                bool row_ok, int h, const float2* __restrict__ tab,
                                                __nv_bfloat16* __restrict__ out) {
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
    for (int i = 0; i < Q4; i += 8) {
        float r0[8], r1[8];
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const float2 c = __ldg(cs + i + j);
            const float a = g0[i + j] * scale, b = g1[i + j] * scale;
            r0[j] = a * c.x + b * c.y;
            r1[j] = b * c.x - a * c.y;
        }
        *reinterpret_cast<uint4*>(out + h * Q4 + i) = pack8(r0);
        *reinterpret_cast<uint4*>(out + H + h * Q4 + i) = pack8(r1);
    }
}

// ---------------------------------------------------------------------------------------
// Query-major: one CTA per (128 queries, head), all T queries.  Key/value
// blocks are double-buffered cp.async copies of RoPE(k) and v; dS reuses the
// block's V buffer once dP = dout V^T has been formed.
template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
bwd_wdq_tc_kernel(const BwdArgs a, const __nv_bfloat16* __restrict__ qr, const __nv_bfloat16* __restrict__ kr,
                  const float2* __restrict__ tab, int* __restrict__ status) {
    extern __shared__ unsigned char smem_raw[];
    constexpr int TB = 128 * D * 2;
    unsigned char* X0 = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* X3 = X0 + TB;  // dout tile
    unsigned char* KB[2];
    unsigned char* VB[2];         // V block, then dS [128 q][128 keys]
    KB[0] = X3 + TB;
    VB[0] = KB[0] + 32768;
    KB[1] = VB[0] + 32768;
    VB[1] = KB[1] + 32768;
    unsigned char* XP = VB[1] + 32768;  // P [128 q][128 keys]
    float* red = reinterpret_cast<float*>(XP + 32768);  // [2][128]
    __shared__ uint64_t bar;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const Shape sh = a.sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = ((warp & 3) << 5) | lane, h = warp >> 2;
    const int tbase = blockIdx.x * 128, nq = min(128, sh.T - tbase), bh = blockIdx.y;
    const size_t hoff = (size_t)bh * sh.T;
    const __nv_bfloat16* v = (const __nv_bfloat16*)a.v + hoff * D;
    const __nv_bfloat16* dout = (const __nv_bfloat16*)a.dout + hoff * D;
    qr += hoff * D;
    kr += hoff * D;
    const float sig2 = sh.sigma * kLog2e;
    const int t = tbase + r;
    const bool row_ok = r < nq;
    const int klo = max(0, tbase - sh.w + 1), khi = tbase + nq - 1;
    const int nb = sh.w > 0 ? (khi - klo) / 128 + 1 : 0;

    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
        s_abort = 0;
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    load_tile_async<D>(qr, tbase, nq, X0);
    load_tile_async<D>(dout, tbase, nq, X3);
    if (nb > 0) {
        load_tile_async<D>(kr, klo, min(128, khi - klo + 1), KB[0]);
        load_tile_async<D>(v, klo, min(128, khi - klo + 1), VB[0]);
    }
    cp_async_commit();
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
    const float lse2 = row_ok ? a.lse[hoff + t] * kLog2e : 0.0f;
    float dwin = 0.0f;
    TcCtl ctl{&bar, 0u, &s_abort, status};
    bool ok = true, acc = false;

    // S = Q~ K~_b^T and dP = dout V_b^T of block i (stage i & 1)
    auto issue_a = [&](int i) {
        const uint32_t s0 = smem_u32(X0), s1 = smem_u32(KB[i & 1]), s2 = smem_u32(VB[i & 1]), s3 = smem_u32(X3);
        for (int kk = 0; kk < D / 16; kk++)
            mma_bf16(tm + tS, desc_k(s0, 128, kk), desc_k(s1, 128, kk), idesc_bf16(128, 128, false), kk > 0);
        for (int kk = 0; kk < D / 16; kk++)
            mma_bf16(tm + tP, desc_k(s3, 128, kk), desc_k(s2, 128, kk), idesc_bf16(128, 128, false), kk > 0);
    };
    if (nb > 0) {
        cp_async_wait<0>();
        sync_for_mma();
        if (tid == 0) {
            issue_a(0);
            mma_commit(&bar);
        }
    }
    // One wait per block: the commit after block i's S / dP also covers block
    // i - 1's dq MMAs, issued just before them.
    for (int i = 0; i < nb && ok; i++) {
        const int kb = klo + i * 128, nk = min(128, khi - kb + 1), cur = i & 1;
        ok = ctl.wait();
        if (!ok) break;
        if (i + 1 < nb) {  // stage of block i - 1, whose MMAs are complete
            const int kn = kb + 128, nn = min(128, khi - kn + 1);
            load_tile_async<D>(kr, kn, nn, KB[cur ^ 1]);
            load_tile_async<D>(v, kn, nn, VB[cur ^ 1]);
            cp_async_commit();
        }
        float sv[64], dp[64];
        tmem_ld(tl + tS + 64 * h, sv, 64);
        tmem_ld(tl + tP + 64 * h, dp, 64);
        const int clo = max(0, t - sh.w + 1 - kb) - 64 * h;
        const int chi = (row_ok ? min(nk - 1, t - kb) : -1) - 64 * h;
#pragma unroll
        for (int jj = 0; jj < 64; jj++) {
            const bool valid = jj >= clo && jj <= chi;
            const float p = valid ? ex2(sv[jj] * sig2 - lse2) : 0.0f;
            dwin += p * dp[jj];
            sv[jj] = p * (dp[jj] - Dr);
            dp[jj] = p;
        }
        store_row(VB[cur], r, 64 * h, sv, 64);  // dS over the consumed V block
        store_row(XP, r, 64 * h, dp, 64);
        if (i + 1 < nb) cp_async_wait<0>();
        sync_for_mma();
        if (tid == 0) {
            const uint32_t s1 = smem_u32(KB[cur]), s4 = smem_u32(VB[cur]), s5 = smem_u32(XP);
            for (int kk = 0; kk < 8; kk++)
                mma_bf16(tm + tQ, desc_k(s4, 128, kk), desc_mn(s1, 128, kk), idesc_bf16(128, D, true),
                         (acc || kk > 0) ? 1u : 0u);
            for (int kk = 0; kk < 8; kk++)
                mma_bf16(tm + tV, desc_k(s5, 128, kk), desc_mn(s1, 128, kk), idesc_bf16(128, D, true),
                         (acc || kk > 0) ? 1u : 0u);
            if (i + 1 < nb) issue_a(i + 1);
            mma_commit(&bar);
        }
        acc = true;
    }
    if (ok && nb > 0) ok = ctl.wait();  // the last block's dq MMAs
    cp_async_wait<0>();
    red[h * 128 + r] = dwin;
    __syncthreads();
    if (h == 0 && row_ok) a.Dwin[hoff + t] = red[r] + red[128 + r];
    if (ok) {
        store_unrotated<D>(tl + tQ, acc, sh.sigma, t, row_ok, h, tab, a.hdqw + (hoff + t) * D);
        store_unrotated<D>(tl + tV, acc, sh.sigma, t, row_ok, h, tab, a.hdqwV + (hoff + t) * D);
    } else if (row_ok) {
        a.hdqw[(hoff + t) * D + h] = __float2bfloat16_rn(__int_as_float(0x7fc00000));
    }
    if (!ok && tid == 0) mbar_wait(&bar, ctl.phase ^ 1u, kWaitCycles);
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

// ---------------------------------------------------------------------------------------
// Key-major: one CTA per (128 keys, head).  Row of the tile = key.  Query
// blocks of 64 are streamed through two cp.async stages.
template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
bwd_wkv_tc_kernel(const BwdArgs a, const __nv_bfloat16* __restrict__ qr, const __nv_bfloat16* __restrict__ kr,
                  const float2* __restrict__ tab, int* __restrict__ status) {
    extern __shared__ unsigned char smem_raw[];
    constexpr int TB = 128 * D * 2, QBB = 64 * D * 2;
    unsigned char* XK = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* XV = XK + TB;
    unsigned char* QB[2];
    unsigned char* OB[2];
    QB[0] = XV + TB;
    OB[0] = QB[0] + QBB;
    QB[1] = OB[0] + QBB;
    OB[1] = QB[1] + QBB;
    unsigned char* PT = OB[1] + QBB;   // P^T  [128 keys][64 q]
    unsigned char* ST = PT + 16384;    // dS^T [128 keys][64 q]
    float* sL2 = reinterpret_cast<float*>(ST + 16384);  // [2][64] lse (log2 domain)
    float* sD = sL2 + 128;                                // [2][64]
    __shared__ uint64_t bar;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const Shape sh = a.sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rk = ((warp & 3) << 5) | lane, h = warp >> 2;
    const int sbase = blockIdx.x * 128, nk = min(128, sh.T - sbase), bh = blockIdx.y;
    const size_t hoff = (size_t)bh * sh.T;
    const __nv_bfloat16* dout = (const __nv_bfloat16*)a.dout + hoff * D;
    qr += hoff * D;
    kr += hoff * D;
    const float sig2 = sh.sigma * kLog2e;
    const int key = sbase + rk;
    const bool row_ok = rk < nk;
    const int thi = sh.w > 0 ? min(sh.T - 1, sbase + nk - 1 + sh.w - 1) : sbase - 1;
    const int nb = thi >= sbase ? (thi - sbase) / 64 + 1 : 0;

    auto prefetch = [&](int i, int stage) {
        const int qb = sbase + i * 64, nq = min(64, thi - qb + 1);
        load_tile_async<D>(qr, qb, nq, QB[stage], 64);
        load_tile_async<D>(dout, qb, nq, OB[stage], 64);
        if (tid < 64) {
            const int tt = tid < nq ? tid : 0;
            cp_async4(sL2 + stage * 64 + tid, a.lse + hoff + qb + tt, tid < nq);
            cp_async4(sD + stage * 64 + tid, a.Dv + hoff + qb + tt, tid < nq);
        }
        cp_async_commit();
    };

    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
        s_abort = 0;
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    load_tile_async<D>(kr, sbase, nk, XK);
    load_tile_async<D>((const __nv_bfloat16*)a.v + hoff * D, sbase, nk, XV);
    cp_async_commit();
    if (nb > 0) prefetch(0, 0);
    cp_async_wait<0>();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t tS = 0, tP = 64, tV = 128, tK = 256;
    TcCtl ctl{&bar, 0u, &s_abort, status};
    bool ok = true, acc = false;

    // S^T = K~ Q~_b^T and dP^T = V dout_b^T of block i (stage i & 1)
    auto issue_a = [&](int i) {
        const uint32_t sk = smem_u32(XK), sv = smem_u32(XV), sq = smem_u32(QB[i & 1]), so = smem_u32(OB[i & 1]);
        for (int kk = 0; kk < D / 16; kk++)
            mma_bf16(tm + tS, desc_k(sk, 128, kk), desc_k(sq, 64, kk), idesc_bf16(128, 64, false), kk > 0);
        for (int kk = 0; kk < D / 16; kk++)
            mma_bf16(tm + tP, desc_k(sv, 128, kk), desc_k(so, 64, kk), idesc_bf16(128, 64, false), kk > 0);
    };
    if (nb > 0) {
        fence_async_smem();
        __syncthreads();
        fence_after_sync();
        if (tid == 0) {
            issue_a(0);
            mma_commit(&bar);
        }
    }
    // One wait per block: the commit after block i's S / dP also covers block
    // i - 1's dV / dK, which were issued just before them.
    for (int i = 0; i < nb && ok; i++) {
        const int qb = sbase + i * 64, nq = min(64, thi - qb + 1), cur = i & 1;
        ok = ctl.wait();
        if (!ok) break;
        if (i + 1 < nb) prefetch(i + 1, cur ^ 1);  // stage of block i - 1, whose MMAs are complete
        float sv[32], dp[32];
        tmem_ld(tl + tS + 32 * h, sv, 32);
        tmem_ld(tl + tP + 32 * h, dp, 32);
        // queries t = qb + c seeing this key: c in [key - qb, key + w - 1 - qb]
        const int clo = key - qb - 32 * h;
        const int chi = (row_ok ? min(nq - 1, key + sh.w - 1 - qb) : -1) - 32 * h;
#pragma unroll
        for (int jj = 0; jj < 32; jj++) {
            const int c = 32 * h + jj;
            const bool valid = jj >= clo && jj <= chi;
            const float p = valid ? ex2(sv[jj] * sig2 - sL2[cur * 64 + c] * kLog2e) : 0.0f;
            sv[jj] = p;
            dp[jj] = p * (dp[jj] - sD[cur * 64 + c]);
        }
        store_row(PT, rk, 32 * h, sv, 32);
        store_row(ST, rk, 32 * h, dp, 32);
        if (i + 1 < nb) cp_async_wait<0>();
        sync_for_mma();
        if (tid == 0) {
            const uint32_t sq = smem_u32(QB[cur]), so = smem_u32(OB[cur]), sp = smem_u32(PT), ss = smem_u32(ST);
            for (int kk = 0; kk < 4; kk++)
                mma_bf16(tm + tV, desc_k(sp, 128, kk), desc_mn(so, 64, kk), idesc_bf16(128, D, true),
                         (acc || kk > 0) ? 1u : 0u);
            for (int kk = 0; kk < 4; kk++)
                mma_bf16(tm + tK, desc_k(ss, 128, kk), desc_mn(sq, 64, kk), idesc_bf16(128, D, true),
                         (acc || kk > 0) ? 1u : 0u);
            if (i + 1 < nb) issue_a(i + 1);
            mma_commit(&bar);
        }
        acc = true;
    }
    if (ok && nb > 0) ok = ctl.wait();  // the last block's dV / dK
    cp_async_wait<0>();
    if (ok) {
        constexpr int HD = D / 2;
        __nv_bfloat16* ov = a.hdvw + (hoff + key) * D + h * HD;
        for (int c0 = 0; c0 < HD; c0 += 32) {
            float vv[32];
            if (acc) {
                tmem_ld32(tl + tV + h * HD + c0, vv);
            } else {
#pragma unroll
                for (int q = 0; q < 32; q++) vv[q] = 0.0f;
            }
            if (row_ok)
#pragma unroll
                for (int q = 0; q < 32; q += 8) *reinterpret_cast<uint4*>(ov + c0 + q) = pack8(vv + q);
        }
        store_unrotated<D>(tl + tK, acc, sh.sigma, key, row_ok, h, tab, a.hdkw + (hoff + key) * D);
    } else if (row_ok) {
        a.hdkw[(hoff + key) * D + h] = __float2bfloat16_rn(__int_as_float(0x7fc00000));
    }
    if (!ok && tid == 0) mbar_wait(&bar, ctl.phase ^ 1u, kWaitCycles);
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

template <int D>
size_t wdq_smem() { return 1024 + 2 * 128 * D * 2 + 5 * 32768 + 256 * sizeof(float); }
template <int D>
size_t wkv_smem() { return 1024 + 2 * 128 * D * 2 + 4 * 64 * D * 2 + 2 * 16384 + 256 * sizeof(float); }

template <int D, int M>
cudaError_t tc_backward(const BwdArgs& a, float2* tab, __nv_bfloat16* qr, __nv_bfloat16* kr, int* status,
                        cudaStream_t st) {
    const Shape& sh = a.sh;
    cudaError_t e = tc_states<D, M>((const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v, a.la, a.SK, a.SV,
                                    a.SKb, a.SVb, a.G, sh, status, st);
    if (e != cudaSuccess) return e;
    if ((e = launch_rope_table(tab, sh.T, D / 2, a.rope, st)) != cudaSuccess) return e;
    if (sh.w > 0 && (e = launch_rope_qk<D>(a.q, a.k, qr, kr, tab, sh, st)) != cudaSuccess) return e;
    const dim3 grid((sh.T + 127) / 128, sh.BH);
    {
        auto kern = bwd_wdq_tc_kernel<D>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wdq_smem<D>())) != cudaSuccess)
            return e;
        NHA_LAUNCH("bwd_wdq_tc", st, kern<<<grid, kTcThreads, wdq_smem<D>(), st>>>(a, qr, kr, tab, status));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return tc_bwd_slot<D, M>(a, qr, kr, tab, status, st);
}

template <int D>
cudaError_t launch_wkv(const BwdArgs& a, const __nv_bfloat16* qr, const __nv_bfloat16* kr, const float2* tab,
                       int* status, cudaStream_t st) {
    const dim3 grid((a.sh.T + 127) / 128, a.sh.BH);
    auto kern = bwd_wkv_tc_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wkv_smem<D>());
    if (e != cudaSuccess) return e;
    NHA_LAUNCH("bwd_wkv_tc", st, kern<<<grid, kTcThreads, wkv_smem<D>(), st>>>(a, qr, kr, tab, status));
    return cudaGetLastError();
}
template cudaError_t launch_wkv<64>(const BwdArgs&, const __nv_bfloat16*, const __nv_bfloat16*, const float2*,
                                    int*, cudaStream_t);
template cudaError_t launch_wkv<128>(const BwdArgs&, const __nv_bfloat16*, const __nv_bfloat16*, const float2*,
                                     int*, cudaStream_t);

#define NHA_TCB_INST(D, M) \
    template cudaError_t tc_backward<D, M>(const BwdArgs&, float2*, __nv_bfloat16*, __nv_bfloat16*, int*, cudaStream_t);
NHA_TCB_INST(64, 16)
NHA_TCB_INST(64, 32)
NHA_TCB_INST(64, 64)
NHA_TCB_INST(128, 16)
NHA_TCB_INST(128, 32)
NHA_TCB_INST(128, 64)

}  // namespace nha
