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
#include "nha_tma.h"

namespace nha {

// ---------------------------------------------------------------------------------------
// Query-major: one CTA per (128 queries, head).  Warp 8 is the producer: TMA
// copies of the RoPE(q), dout and o tiles and of 128-key blocks of RoPE(k), v
// through two stages; lane 0 issues every MMA.  Warps 0-7 turn S, dP into P,
// dS.  The softmax warps hand the S / dP columns of TMEM back as soon as they
// have read them, so block i + 1's S, dP run on the tensor core during block
// i's softmax.  D^ = dout . o comes from the two tiles in shared memory.
//
// Barriers per block i: full[i & 1] (K, V block landed), sfull (S, dP in
// TMEM), sfree (S, dP read out; 8 warp arrivals), pready (dS over the V block
// and P stored; 8 warp arrivals), bdone[i & 1] (dq += dS K~, dqV += P K~ done).
constexpr int kWdqThreads = 288;

struct WdqMaps {
    CUtensorMap q, dout, o, k, v, tab;
};

template <int D>
__global__ void __launch_bounds__(kWdqThreads, 1)
bwd_wdq_tc_kernel(const BwdArgs a, const __grid_constant__ WdqMaps maps, int* __restrict__ status) {
    extern __shared__ unsigned char smem_raw[];
    constexpr int TB = 128 * D * 2, HD = D / 2, Q4 = D / 4, CH = D / 8;
    unsigned char* X0 = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* X3 = X0 + TB;  // dout tile
    unsigned char* KB[2];
    unsigned char* VB[2];  // V block, then dS [128 q][128 keys]
    KB[0] = X3 + TB;
    VB[0] = KB[0] + 32768;
    KB[1] = VB[0] + 32768;
    VB[1] = KB[1] + 32768;
    unsigned char* XP = VB[1] + 32768;                  // o tile, then P [128 q][128 keys]
    float* red = reinterpret_cast<float*>(XP + 32768);  // [2][128]
    __shared__ uint64_t qbar, full[2], sfull, sfree, pready, bdone[2], tbar, drain;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.y;
    const Shape sh = head_shape(a.sh, bh);
    const int tbase = blockIdx.x * 128, nq = min(128, sh.T - tbase);
    if (nq <= 0) return;  // past this head's queries (per-sequence lengths)
    const size_t hoff = (size_t)bh * sh.TS;
    const int klo = max(0, tbase - sh.w + 1), khi = tbase + nq - 1;
    const int nb = sh.w > 0 ? (khi - klo) / 128 + 1 : 0;
    volatile int* abort = &s_abort;

    if (tid == 0) {
        mbar_init(&qbar, 1);
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&sfull, 1);
        mbar_init(&sfree, 8);
        mbar_init(&pready, 8);
        mbar_init(&bdone[0], 1);
        mbar_init(&bdone[1], 1);
        mbar_init(&tbar, 1);
        mbar_init(&drain, 1);
        s_abort = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t tS = 0, tP = 128, tQ = 256, tV = 384;

    int last_ph[2] = {-1, -1};  // producer: phase of the last block load into each stage
    bool tab_issued = false;
    if (warp == 8) {
        // ---------------- producer (lane 0) ----------------
        if (lane == 0) {
            auto load_block = [&](int j) {
                const int b = j & 1, kb = klo + j * 128;
                mbar_arrive_expect_tx(&full[b], 2 * TB);
#pragma unroll
                for (int x = 0; x < D; x += 64) {
                    tma_load_3d(KB[b] + x * 256, &maps.k, x, kb, bh, &full[b]);
                    tma_load_3d(VB[b] + x * 256, &maps.v, x, kb, bh, &full[b]);
                }
                last_ph[b] = (j >> 1) & 1;
            };
            auto issue_a = [&](int j) {  // S = Q~ K~_j^T, dP = dout V_j^T
                const uint32_t s0 = smem_u32(X0), s3 = smem_u32(X3), sk = smem_u32(KB[j & 1]),
                               sv = smem_u32(VB[j & 1]);
                for (int kk = 0; kk < D / 16; kk++)
                    mma_bf16(tm + tS, desc_k(s0, 128, kk), desc_k(sk, 128, kk), idesc_bf16(128, 128, false), kk > 0);
                for (int kk = 0; kk < D / 16; kk++)
                    mma_bf16(tm + tP, desc_k(s3, 128, kk), desc_k(sv, 128, kk), idesc_bf16(128, 128, false), kk > 0);
                mma_commit(&sfull);
            };
            mbar_arrive_expect_tx(&qbar, (nb > 0 ? 3 : 2) * TB);
#pragma unroll
            for (int x = 0; x < D; x += 64) {
                if (nb > 0) tma_load_3d(X0 + x * 256, &maps.q, x, tbase, bh, &qbar);
                tma_load_3d(X3 + x * 256, &maps.dout, x, tbase, bh, &qbar);
                tma_load_3d(XP + x * 256, &maps.o, x, tbase, bh, &qbar);
            }
            bool ok = true;
            if (nb > 0) {
                load_block(0);
                if (nb > 1) load_block(1);
                ok = mbar_wait_ab(&qbar, 0, kWaitCycles, abort) && mbar_wait_ab(&full[0], 0, kWaitCycles, abort);
                if (ok) issue_a(0);
                for (int i = 0; i < nb && ok; i++) {
                    if (i + 1 < nb) {  // S, dP of block i read out; block i + 1 landed
                        if (!(ok = mbar_wait_ab(&sfree, i & 1, kWaitCycles, abort))) break;
                        if (!(ok = mbar_wait_ab(&full[(i + 1) & 1], ((i + 1) >> 1) & 1, kWaitCycles, abort))) break;
                        fence_after_sync();
                        issue_a(i + 1);
                    }
                    if (!(ok = mbar_wait_ab(&pready, i & 1, kWaitCycles, abort))) break;
                    fence_after_sync();
                    {
                        const uint32_t sk = smem_u32(KB[i & 1]), sd = smem_u32(VB[i & 1]), sp = smem_u32(XP);
                        for (int kk = 0; kk < 8; kk++)
                            mma_bf16(tm + tQ, desc_k(sd, 128, kk), desc_mn(sk, 128, kk), idesc_bf16(128, D, true),
                                     (i > 0 || kk > 0) ? 1u : 0u);
                        for (int kk = 0; kk < 8; kk++)
                            mma_bf16(tm + tV, desc_k(sp, 128, kk), desc_mn(sk, 128, kk), idesc_bf16(128, D, true),
                                     (i > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(&bdone[i & 1]);
                    }
                    if (i + 2 < nb) {  // block i's stage is free once its dq MMAs are done
                        if (!(ok = mbar_wait_ab(&bdone[i & 1], (i >> 1) & 1, kWaitCycles, abort))) break;
                        load_block(i + 2);
                    }
                    if (i == nb - 1) {
                        // RoPE table tile for the epilogue, into the stage of block
                        // nb - 2 (its MMAs finished before pready of block nb - 1)
                        unsigned char* dst = KB[(i + 1) & 1];
                        mbar_arrive_expect_tx(&tbar, 128 * D * 4);
#pragma unroll
                        for (int x = 0; x < D; x += 32) tma_load_2d(dst + x * 512, &maps.tab, x, tbase, &tbar);
                        tab_issued = true;
                    }
                }
            }
        }
    } else {
        // ---------------- softmax warps ----------------
        const int r = ((warp & 3) << 5) | lane, h = warp >> 2;
        const int t = tbase + r;
        const bool row_ok = r < nq;
        const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);
        const float sig2 = sh.sigma * kLog2e;
        const float lse2 = row_ok ? a.lse[hoff + t] * kLog2e : 0.0f;
        bool ok = mbar_wait_ab(&qbar, 0, kWaitCycles, abort);
        {  // D^ = dout_t . o_t (bf16 tiles), half a row per thread
            float part = 0.0f;
            if (ok)
#pragma unroll
                for (int c = 0; c < CH / 2; c++) {
                    float x[8], y[8];
                    unpack8(*reinterpret_cast<const uint4*>(X3 + sw_chunk(r, h * (CH / 2) + c, 128)), x);
                    unpack8(*reinterpret_cast<const uint4*>(XP + sw_chunk(r, h * (CH / 2) + c, 128)), y);
#pragma unroll
                    for (int e = 0; e < 8; e++) part += x[e] * y[e];
                }
            red[h * 128 + r] = part;
        }
        named_sync(1, 256);  // also: every o read done before P overwrites the tile
        const float Dr = red[r] + red[128 + r];
        if (h == 0 && row_ok) a.Dhat[hoff + t] = Dr;
        float2 dwin2 = make_float2(0.0f, 0.0f), dwin2b = make_float2(0.0f, 0.0f);
        const float2 sg2 = make_float2(sig2, sig2), nl2 = make_float2(-lse2, -lse2), nD2 = make_float2(-Dr, -Dr);
        for (int i = 0; i < nb && ok; i++) {
            const int kb = klo + i * 128, nk = min(128, khi - kb + 1), b = i & 1;
            if (!(ok = mbar_wait_ab(&sfull, i & 1, kWaitCycles, abort))) break;
            fence_after_sync();
            float sv[64], dp[64];
            tmem_ld64x2(tl + tS + 64 * h, tl + tP + 64 * h, sv, dp);
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sfree);
            const int clo = max(0, t - sh.w + 1 - kb) - 64 * h;
            const int chi = (row_ok ? min(nk - 1, t - kb) : -1) - 64 * h;
            if (clo <= 0 && chi >= 63) {
                // every key of this half-row is in the band: packed pairs, no masks
#pragma unroll
                for (int jj = 0; jj < 64; jj += 4) {
                    const float2 s0 = __ffma2_rn(make_float2(sv[jj], sv[jj + 1]), sg2, nl2);
                    const float2 s1 = __ffma2_rn(make_float2(sv[jj + 2], sv[jj + 3]), sg2, nl2);
                    const float2 p0 = make_float2(ex2(s0.x), ex2(s0.y)), p1 = make_float2(ex2(s1.x), ex2(s1.y));
                    const float2 d0 = make_float2(dp[jj], dp[jj + 1]), d1 = make_float2(dp[jj + 2], dp[jj + 3]);
                    dwin2 = __ffma2_rn(p0, d0, dwin2);
                    dwin2b = __ffma2_rn(p1, d1, dwin2b);
                    const float2 g0 = __fmul2_rn(p0, __fadd2_rn(d0, nD2)), g1 = __fmul2_rn(p1, __fadd2_rn(d1, nD2));
                    sv[jj] = g0.x; sv[jj + 1] = g0.y; sv[jj + 2] = g1.x; sv[jj + 3] = g1.y;
                    dp[jj] = p0.x; dp[jj + 1] = p0.y; dp[jj + 2] = p1.x; dp[jj + 3] = p1.y;
                }
            } else {
#pragma unroll
                for (int jj = 0; jj < 64; jj++) {
                    const bool valid = jj >= clo && jj <= chi;
                    const float p = valid ? ex2(sv[jj] * sig2 - lse2) : 0.0f;
                    dwin2.x += p * dp[jj];
                    sv[jj] = p * (dp[jj] - Dr);
                    dp[jj] = p;
                }
            }
            // P of block i - 1 no longer read by the tensor core
            if (i >= 1 && !(ok = mbar_wait_ab(&bdone[(i - 1) & 1], ((i - 1) >> 1) & 1, kWaitCycles, abort))) break;
            store_row(VB[b], r, 64 * h, sv, 64);  // dS over the consumed V block
            store_row(XP, r, 64 * h, dp, 64);
            fence_async_smem();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&pready);
        }
        const float dwin = (dwin2.x + dwin2.y) + (dwin2b.x + dwin2b.y);
        named_sync(1, 256);
        red[h * 128 + r] = dwin;
        named_sync(1, 256);
        if (h == 0 && row_ok) a.Dwin[hoff + t] = red[r] + red[128 + r];
        // epilogue: sigma R^T(t) of the dq and dqV accumulators, in bf16, staged
        // in the stage of the last block and written by TMA
        if (ok && nb > 0)
            ok = mbar_wait_ab(&bdone[(nb - 1) & 1], ((nb - 1) >> 1) & 1, kWaitCycles, abort) &&
                 mbar_wait_ab(&tbar, 0, kWaitCycles, abort);
        unsigned char* stQ = KB[(nb + 1) & 1];
        unsigned char* stV = VB[(nb + 1) & 1];
        if (ok) {
            fence_after_sync();
            const unsigned char* tabs = KB[nb & 1];
#pragma unroll
            for (int pass = 0; pass < 2; pass++) {
                float g0[Q4], g1[Q4];
                if (nb > 0) {
                    const uint32_t ta = tl + (pass == 0 ? tQ : tV) + h * Q4;
                    if constexpr (Q4 == 32) {
                        tmem_ld32x2(ta, ta + HD, g0, g1);
                    } else {
                        tmem_ld(ta, g0, Q4);
                        tmem_ld(ta + HD, g1, Q4);
                    }
#pragma unroll
                    for (int q = 0; q < Q4; q += 2) {
                        // (cos, sin) pairs h Q4 + q, + 1: one 16-byte chunk of the swizzled tile
                        const int pi = h * Q4 + q, bx = pi >> 4, c = (pi & 15) >> 1;
                        const float4 cs = *reinterpret_cast<const float4*>(tabs + bx * 16384 + r * 128 +
                                                                           ((c ^ (r & 7)) << 4));
                        const float a0 = g0[q] * sh.sigma, b0 = g1[q] * sh.sigma;
                        const float a1 = g0[q + 1] * sh.sigma, b1 = g1[q + 1] * sh.sigma;
                        g0[q] = a0 * cs.x + b0 * cs.y;
                        g1[q] = b0 * cs.x - a0 * cs.y;
                        g0[q + 1] = a1 * cs.z + b1 * cs.w;
                        g1[q + 1] = b1 * cs.z - a1 * cs.w;
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < Q4; q++) g0[q] = g1[q] = 0.0f;
                }
                unsigned char* stg = pass == 0 ? stQ : stV;
                store_row(stg, r, h * Q4, g0, Q4);
                store_row(stg, r, HD + h * Q4, g1, Q4);
            }
            fence_async_smem();
        }
        const int bad = named_sync_or(1, 256, !ok);
        if (!bad) {  // rows [0, nq) of both staged tiles, 16-byte chunks, coalesced
            constexpr int CHR = D / 8;
            __nv_bfloat16* o1 = a.hdqw + (hoff + tbase) * D;
            __nv_bfloat16* o2 = a.hdqwV + (hoff + tbase) * D;
            for (int e = tid; e < nq * CHR; e += 256) {
                const int rr = e / CHR, ch = e % CHR;
                const uint32_t off = sw_chunk(rr, ch, 128);
                *reinterpret_cast<uint4*>(o1 + (size_t)rr * D + ch * 8) = *reinterpret_cast<const uint4*>(stQ + off);
                *reinterpret_cast<uint4*>(o2 + (size_t)rr * D + ch * 8) = *reinterpret_cast<const uint4*>(stV + off);
            }
        }
        if (bad && row_ok) a.hdqw[(hoff + t) * D + h] = __float2bfloat16_rn(__int_as_float(0x7fc00000));
    }
    fence_before_sync();
    __syncthreads();
    if (s_abort) {  // let the copies and MMAs in flight land before the TMEM and the CTA go
        if (warp == 8 && lane == 0) {
            mma_commit(&drain);
            mbar_wait(&drain, 0, kWaitCycles);
            mbar_wait(&qbar, 0, kWaitCycles);
            for (int q = 0; q < 2; q++)
                if (last_ph[q] >= 0) mbar_wait(&full[q], (uint32_t)last_ph[q], kWaitCycles);
            if (tab_issued) mbar_wait(&tbar, 0, kWaitCycles);
        }
        __syncthreads();
        if (tid == 0) atomicOr(status, kStatusTimeoutBit);
    }
    if (warp == 0) tmem_dealloc(tm, 512);
}

// ---------------------------------------------------------------------------------------
// Key-major: one CTA per (128 keys, head).  Row of the tile = key.  Warp 8 is
// the producer: it streams 64-query blocks of RoPE(q) and dout through three
// TMA stages (lse and D beside them by cp.async) and issues every MMA.  Warps
// 0-7 turn S^T, dP^T into P^T, dS^T.  S^T / dP^T live in two TMEM buffers, so
// block i + 1's run on the tensor core while block i's softmax runs.
//
// Per block i, barriers: full[i % 3] (stage landed), sfull[i & 1] (S^T, dP^T
// of block i in TMEM), pready (P^T, dS^T of block i stored; 8 warp arrivals),
// bdone[i & 1] (dV += P^T dout, dK += dS^T q of block i done).  Every wait is
// bounded and gives up once any thread flags an abort.
constexpr int kWkvThreads = 288, kWkvStages = 3;

struct WkvMaps {
    CUtensorMap q, dout, k, v, tab;
};

template <int D>
__global__ void __launch_bounds__(kWkvThreads, 1)
bwd_wkv_tc_kernel(const BwdArgs a, const __grid_constant__ WkvMaps maps, int* __restrict__ status) {
    extern __shared__ unsigned char smem_raw[];
    constexpr int TB = 128 * D * 2, QBB = 64 * D * 2, NS = kWkvStages, HD = D / 2, Q4 = D / 4;
    unsigned char* XK = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* XV = XK + TB;
    unsigned char* QB0 = XV + TB;                 // stage s: RoPE(q) at QB0 + 2 s QBB, dout after it
    unsigned char* PT = QB0 + NS * 2 * QBB;       // P^T  [128 keys][64 q]
    unsigned char* ST = PT + 16384;               // dS^T [128 keys][64 q]
    float* sL = reinterpret_cast<float*>(ST + 16384);  // [NS][64] lse
    float* sD = sL + NS * 64;                          // [NS][64] D
    __shared__ uint64_t kvbar, full[NS], sfull[2], pready, bdone[2], tbar, drain;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sbase = blockIdx.x * 128, bh = blockIdx.y;
    const Shape sh = head_shape(a.sh, bh);
    if (sbase >= sh.T) return;  // past this head's keys (per-sequence lengths)
    const size_t hoff = (size_t)bh * sh.TS;
    const int thi = sh.w > 0 ? min(sh.T - 1, sbase + min(128, sh.T - sbase) - 1 + sh.w - 1) : sbase - 1;
    const int nb = thi >= sbase ? (thi - sbase) / 64 + 1 : 0;
    volatile int* abort = &s_abort;

    if (tid == 0) {
        mbar_init(&kvbar, 1);
        for (int q = 0; q < NS; q++) mbar_init(&full[q], 33);  // expect_tx arrival + 32 cp.async arrivals
        for (int q = 0; q < 2; q++) {
            mbar_init(&sfull[q], 1);
            mbar_init(&bdone[q], 1);
        }
        mbar_init(&pready, 8);
        mbar_init(&tbar, 1);
        mbar_init(&drain, 1);
        s_abort = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t tV = 256, tK = 256 + D;  // S^T / dP^T of buffer b at columns 128 b and 128 b + 64

    int last_ph[NS];  // producer: phase of the last load issued into each stage
#pragma unroll
    for (int q = 0; q < NS; q++) last_ph[q] = -1;
    bool tab_issued = false;
    if (warp == 8) {
        // ---------------- producer ----------------
        auto load_stage = [&](int j) {
            const int stg = j % NS, qb = sbase + j * 64;
            unsigned char* qd = QB0 + stg * 2 * QBB;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[stg], 2 * QBB);
#pragma unroll
                for (int x = 0; x < D; x += 64) {
                    tma_load_3d(qd + x * 128, &maps.q, x, qb, bh, &full[stg]);
                    tma_load_3d(qd + QBB + x * 128, &maps.dout, x, qb, bh, &full[stg]);
                }
            }
#pragma unroll
            for (int c = lane; c < 64; c += 32) {
                const bool in = qb + c < sh.T;
                const size_t o = hoff + (in ? qb + c : 0);
                cp_async4(sL + stg * 64 + c, a.lse + o, in);
                cp_async4(sD + stg * 64 + c, a.Dv + o, in);
            }
            cp_async_mbar_arrive(&full[stg]);
            last_ph[stg] = (j / NS) & 1;
        };
        auto issue_a = [&](int j) {  // S^T = K~ Q~_j^T, dP^T = V dout_j^T into buffer j & 1
            const uint32_t tS = tm + 128 * (j & 1), tP = tS + 64;
            const uint32_t qd = smem_u32(QB0 + (j % NS) * 2 * QBB), sk = smem_u32(XK), sv = smem_u32(XV);
            for (int kk = 0; kk < D / 16; kk++)
                mma_bf16(tS, desc_k(sk, 128, kk), desc_k(qd, 64, kk), idesc_bf16(128, 64, false), kk > 0);
            for (int kk = 0; kk < D / 16; kk++)
                mma_bf16(tP, desc_k(sv, 128, kk), desc_k(qd + QBB, 64, kk), idesc_bf16(128, 64, false), kk > 0);
            mma_commit(&sfull[j & 1]);
        };
        bool ok = true;
        if (nb > 0) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&kvbar, 2 * TB);
#pragma unroll
                for (int x = 0; x < D; x += 64) {
                    tma_load_3d(XK + x * 256, &maps.k, x, sbase, bh, &kvbar);
                    tma_load_3d(XV + x * 256, &maps.v, x, sbase, bh, &kvbar);
                }
            }
            for (int j = 0; j < min(NS, nb); j++) load_stage(j);
            ok = mbar_wait_ab(&kvbar, 0, kWaitCycles, abort) && mbar_wait_ab(&full[0], 0, kWaitCycles, abort);
            if (ok && lane == 0) issue_a(0);
            __syncwarp();
            for (int i = 0; i < nb && ok; i++) {
                if (i + 1 < nb) {  // buffer (i + 1) & 1 was read by block i - 1, released through pready
                    if (!(ok = mbar_wait_ab(&full[(i + 1) % NS], ((i + 1) / NS) & 1, kWaitCycles, abort))) break;
                    if (lane == 0) issue_a(i + 1);
                    __syncwarp();
                }
                if (!(ok = mbar_wait_ab(&pready, i & 1, kWaitCycles, abort))) break;
                fence_after_sync();
                if (lane == 0) {
                    const uint32_t qd = smem_u32(QB0 + (i % NS) * 2 * QBB), sp = smem_u32(PT), ss = smem_u32(ST);
                    for (int kk = 0; kk < 4; kk++)
                        mma_bf16(tm + tV, desc_k(sp, 128, kk), desc_mn(qd + QBB, 64, kk), idesc_bf16(128, D, true),
                                 (i > 0 || kk > 0) ? 1u : 0u);
                    for (int kk = 0; kk < 4; kk++)
                        mma_bf16(tm + tK, desc_k(ss, 128, kk), desc_mn(qd, 64, kk), idesc_bf16(128, D, true),
                                 (i > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&bdone[i & 1]);
                }
                __syncwarp();
                if (i >= 1 && i - 1 + NS < nb) {  // block i - 1 done with its stage: refill it
                    if (!(ok = mbar_wait_ab(&bdone[(i - 1) & 1], ((i - 1) >> 1) & 1, kWaitCycles, abort))) break;
                    load_stage(i - 1 + NS);
                }
            }
            // RoPE table tile for the epilogue, over the last stage and P^T / dS^T
            // once the last MMAs are done
            if (ok && (ok = mbar_wait_ab(&bdone[(nb - 1) & 1], ((nb - 1) >> 1) & 1, kWaitCycles, abort)) &&
                lane == 0) {
                mbar_arrive_expect_tx(&tbar, 128 * D * 4);
#pragma unroll
                for (int x = 0; x < D; x += 32) tma_load_2d(QB0 + 2 * TB + x * 512, &maps.tab, x, sbase, &tbar);
                tab_issued = true;
            }
        }
    } else {
        // ---------------- softmax warps ----------------
        const int rk = ((warp & 3) << 5) | lane, h = warp >> 2;
        const int key = sbase + rk;
        const bool row_ok = key < sh.T;
        const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);
        const float sig2 = sh.sigma * kLog2e;
        bool ok = true;
        for (int i = 0; i < nb; i++) {
            const int qb = sbase + i * 64, nq = min(64, thi - qb + 1), stg = i % NS, b = i & 1;
            if (!(ok = mbar_wait_ab(&sfull[b], (i >> 1) & 1, kWaitCycles, abort) &&
                       mbar_wait_ab(&full[stg], (i / NS) & 1, kWaitCycles, abort)))
                break;
            fence_after_sync();
            float sv[32], dp[32];
            tmem_ld32x2(tl + 128 * b + 32 * h, tl + 128 * b + 64 + 32 * h, sv, dp);
            // queries t = qb + c seeing this key: c in [key - qb, key + w - 1 - qb]
            const int clo = key - qb - 32 * h;
            const int chi = (row_ok ? min(nq - 1, key + sh.w - 1 - qb) : -1) - 32 * h;
            const float* l2 = sL + stg * 64 + 32 * h;
            const float* dd = sD + stg * 64 + 32 * h;
            if (clo <= 0 && chi >= 31) {
                // every query of this half-row sees the key: packed pairs, no masks
                const float2 sg2 = make_float2(sig2, sig2), nlg = make_float2(-kLog2e, -kLog2e);
#pragma unroll
                for (int jj = 0; jj < 32; jj += 4) {
                    const float4 L4 = *reinterpret_cast<const float4*>(l2 + jj);
                    const float4 D4 = *reinterpret_cast<const float4*>(dd + jj);
                    const float2 s0 = __ffma2_rn(make_float2(sv[jj], sv[jj + 1]), sg2,
                                                 __fmul2_rn(make_float2(L4.x, L4.y), nlg));
                    const float2 s1 = __ffma2_rn(make_float2(sv[jj + 2], sv[jj + 3]), sg2,
                                                 __fmul2_rn(make_float2(L4.z, L4.w), nlg));
                    const float2 p0 = make_float2(ex2(s0.x), ex2(s0.y)), p1 = make_float2(ex2(s1.x), ex2(s1.y));
                    const float2 g0 = __fmul2_rn(p0, __fadd2_rn(make_float2(dp[jj], dp[jj + 1]),
                                                                make_float2(-D4.x, -D4.y)));
                    const float2 g1 = __fmul2_rn(p1, __fadd2_rn(make_float2(dp[jj + 2], dp[jj + 3]),
                                                                make_float2(-D4.z, -D4.w)));
                    sv[jj] = p0.x; sv[jj + 1] = p0.y; sv[jj + 2] = p1.x; sv[jj + 3] = p1.y;
                    dp[jj] = g0.x; dp[jj + 1] = g0.y; dp[jj + 2] = g1.x; dp[jj + 3] = g1.y;
                }
            } else {
#pragma unroll
                for (int jj = 0; jj < 32; jj++) {
                    const bool valid = jj >= clo && jj <= chi;
                    const float p = valid ? ex2(sv[jj] * sig2 - l2[jj] * kLog2e) : 0.0f;
                    sv[jj] = p;
                    dp[jj] = valid ? p * (dp[jj] - dd[jj]) : 0.0f;
                }
            }
            // P^T, dS^T of block i - 1 no longer read by the tensor core
            if (i >= 1 && !(ok = mbar_wait_ab(&bdone[(i - 1) & 1], ((i - 1) >> 1) & 1, kWaitCycles, abort))) break;
            store_row(PT, rk, 32 * h, sv, 32);
            store_row(ST, rk, 32 * h, dp, 32);
            fence_async_smem();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&pready);
        }
        // epilogue: dV = sum P^T dout, dK = sigma R^T(key) sum dS^T q~ in bf16,
        // staged through the (now idle) stage buffers and written by TMA
        if (ok && nb > 0) ok = mbar_wait_ab(&bdone[(nb - 1) & 1], ((nb - 1) >> 1) & 1, kWaitCycles, abort);
        if (ok) {
            fence_after_sync();
            unsigned char* oV = QB0;       // [128 keys][D] tile
            unsigned char* oK = QB0 + TB;  // [128 keys][D] tile
            for (int c0 = 0; c0 < HD; c0 += 32) {
                float vv[32];
                if (nb > 0) {
                    tmem_ld(tl + tV + h * HD + c0, vv, HD < 32 ? HD : 32);
                } else {
#pragma unroll
                    for (int q = 0; q < 32; q++) vv[q] = 0.0f;
                }
                store_row(oV, rk, h * HD + c0, vv, HD < 32 ? HD : 32);
            }
            float g0[Q4], g1[Q4];
            if (nb > 0) {
                if constexpr (Q4 == 32) {
                    tmem_ld32x2(tl + tK + h * Q4, tl + tK + HD + h * Q4, g0, g1);
                } else {
                    tmem_ld(tl + tK + h * Q4, g0, Q4);
                    tmem_ld(tl + tK + HD + h * Q4, g1, Q4);
                }
                ok = mbar_wait_ab(&tbar, 0, kWaitCycles, abort);
                const unsigned char* tabs = QB0 + 2 * TB;
#pragma unroll
                for (int q = 0; q < Q4; q += 2) {
                    // (cos, sin) pairs h Q4 + q, + 1: one 16-byte chunk of the swizzled tile
                    const int pi = h * Q4 + q, bx = pi >> 4, c = (pi & 15) >> 1;
                    const float4 cs =
                        *reinterpret_cast<const float4*>(tabs + bx * 16384 + rk * 128 + ((c ^ (rk & 7)) << 4));
                    const float a0 = g0[q] * sh.sigma, b0 = g1[q] * sh.sigma;
                    const float a1 = g0[q + 1] * sh.sigma, b1 = g1[q + 1] * sh.sigma;
                    g0[q] = a0 * cs.x + b0 * cs.y;
                    g1[q] = b0 * cs.x - a0 * cs.y;
                    g0[q + 1] = a1 * cs.z + b1 * cs.w;
                    g1[q + 1] = b1 * cs.z - a1 * cs.w;
                }
            } else {
#pragma unroll
                for (int q = 0; q < Q4; q++) g0[q] = g1[q] = 0.0f;
            }
            store_row(oK, rk, h * Q4, g0, Q4);
            store_row(oK, rk, HD + h * Q4, g1, Q4);
            fence_async_smem();
        }
        // all 256 softmax threads agree before one of them issues the stores
        const int bad = named_sync_or(1, 256, !ok);
        if (!bad) {  // rows [0, nk) of both staged tiles, 16-byte chunks, coalesced
            constexpr int CHR = D / 8;
            const int nk = min(128, sh.T - sbase);
            __nv_bfloat16* o1 = a.hdvw + (hoff + sbase) * D;
            __nv_bfloat16* o2 = a.hdkw + (hoff + sbase) * D;
            for (int e = tid; e < nk * CHR; e += 256) {
                const int rr = e / CHR, ch = e % CHR;
                const uint32_t off = sw_chunk(rr, ch, 128);
                *reinterpret_cast<uint4*>(o1 + (size_t)rr * D + ch * 8) = *reinterpret_cast<const uint4*>(QB0 + off);
                *reinterpret_cast<uint4*>(o2 + (size_t)rr * D + ch * 8) =
                    *reinterpret_cast<const uint4*>(QB0 + TB + off);
            }
        }
        if (bad && row_ok) a.hdkw[(hoff + key) * D + h] = __float2bfloat16_rn(__int_as_float(0x7fc00000));
    }
    fence_before_sync();
    __syncthreads();
    if (s_abort) {  // let the copies and MMAs in flight land before the TMEM and the CTA go
        if (warp == 8) {
            if (lane == 0) {
                mma_commit(&drain);
                mbar_wait(&drain, 0, kWaitCycles);
                if (nb > 0) mbar_wait(&kvbar, 0, kWaitCycles);
                for (int q = 0; q < NS; q++)
                    if (last_ph[q] >= 0) mbar_wait(&full[q], (uint32_t)last_ph[q], kWaitCycles);
                if (tab_issued) mbar_wait(&tbar, 0, kWaitCycles);
            }
            cp_async_wait_all();
        }
        __syncthreads();
        if (tid == 0) atomicOr(status, kStatusTimeoutBit);
    }
    if (warp == 0) tmem_dealloc(tm, 512);
}

template <int D>
size_t wdq_smem() { return 1024 + 2 * 128 * D * 2 + 5 * 32768 + 256 * sizeof(float); }
template <int D>
size_t wkv_smem() {
    return 1024 + 2 * 128 * D * 2 + 2 * kWkvStages * 64 * D * 2 + 2 * 16384 + 2 * kWkvStages * 64 * sizeof(float);
}

template <int D, int M>
cudaError_t tc_backward(const BwdArgs& a, float2* tab, __nv_bfloat16* qr, __nv_bfloat16* kr, int* status,
                        cudaStream_t st) {
    const Shape& sh = a.sh;
    Fork* f = nullptr;
    cudaError_t e = get_fork(&f);
    if (e != cudaSuccess) return e;
    // RoPE(q), RoPE(k) and the (cos, sin) table of the window kernels'
    // epilogues on the side stream while the chunk states are formed (unless
    // the forward's are reused)
    if (!a.reuse) {
        if (sh.w > 0) {
            if ((e = fork_side(st, *f, 0)) != cudaSuccess) return e;
            if ((e = launch_rope_qk<D>(a.q, a.k, qr, kr, tab, a.rope, sh, f->side)) != cudaSuccess) return e;
        }
        e = tc_states<D, M>((const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v, a.la, a.SK, a.SV, a.SKb, a.SVb,
                            a.G, false, a.io, sh, status, st);
        if (e != cudaSuccess) return e;
        if (sh.w > 0 && (e = join_side(st, *f, 1)) != cudaSuccess) return e;
    }
    const dim3 grid((sh.T + 127) / 128, sh.BH);
    {
        WdqMaps maps;
        if ((e = tmap_rows_bf16(&maps.q, qr, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.dout, a.dout, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.o, a.o, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.k, kr, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.v, a.v, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_tab(&maps.tab, tab, D / 2, sh.T)) != cudaSuccess)
            return e;
        auto kern = bwd_wdq_tc_kernel<D>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wdq_smem<D>())) != cudaSuccess)
            return e;
        NHA_LAUNCH("bwd_wdq_tc", st, kern<<<grid, kWdqThreads, wdq_smem<D>(), st>>>(a, maps, status));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return tc_bwd_slot<D, M>(a, qr, kr, tab, status, st);
}

template <int D>
cudaError_t launch_wkv(const BwdArgs& a, const __nv_bfloat16* qr, const __nv_bfloat16* kr, const float2* tab,
                       int* status, cudaStream_t st) {
    const Shape& sh = a.sh;
    WkvMaps maps;
    cudaError_t e;
    if ((e = tmap_rows_bf16(&maps.q, qr, D, sh.T, sh.BH, 64)) != cudaSuccess ||
        (e = tmap_rows_bf16(&maps.dout, a.dout, D, sh.T, sh.BH, 64)) != cudaSuccess ||
        (e = tmap_rows_bf16(&maps.k, kr, D, sh.T, sh.BH, 128)) != cudaSuccess ||
        (e = tmap_rows_bf16(&maps.v, a.v, D, sh.T, sh.BH, 128)) != cudaSuccess ||
        (e = tmap_tab(&maps.tab, tab, D / 2, sh.T)) != cudaSuccess)
        return e;
    const dim3 grid((sh.T + 127) / 128, sh.BH);
    auto kern = bwd_wkv_tc_kernel<D>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wkv_smem<D>());
    if (e != cudaSuccess) return e;
    NHA_LAUNCH("bwd_wkv_tc", st, kern<<<grid, kWkvThreads, wkv_smem<D>(), st>>>(a, maps, status));
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
