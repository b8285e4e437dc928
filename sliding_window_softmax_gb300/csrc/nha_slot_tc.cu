// Tensor-core (tcgen05) backward of the NHA slot branch for bf16 inputs.
//
// Per tile of 128 rows = two C = 64 gate chunks.  With b the chunk-local
// cumsum of log_alpha, rho = G / 2 (G = b at the chunk's end), Eq = exp(b - rho),
// Ek = exp(rho - b) u, Fk = exp(rho - b), Eb = exp(b), eG = exp(G - rho), M the
// within-chunk causal mask, and S_prev the slot states carried into the chunk:
//
// query side (rows = queries t = j + w of state indices j):
//   L    = sigma [Eb o (Q S^K_prev^T) + Eq o ((Q K_c^T o M) Ek)]       P_L = exp(L - lse)
//   dP_L = Eb o (dout S^V_prev^T) + Eq o ((dout V_c^T o M) Ek)        dL = P_L o (dP_L - D)
//   dq  += (sigma dL o Eb) S^K_prev + (((sigma dL o Eq) Ek^T) o M) K_c
//   dR^K_c = (Eb o sigma dL)^T Q,  dR^V_c = (Eb o P_L)^T dout          (adjoint contributions)
//   db1  = dL o L + P_L o dP_L
// key side (rows = tokens s; Rc = adjoint carried in from later chunks):
//   dk  += ((Ek (sigma dL o Eq)^T) o M^T) Q_t + (Ek o eG) Rc^K
//   dv  += ((Ek (P_L o Eq)^T) o M^T) dout_t + (Ek o eG) Rc^V
//   du   = Fk o [((K_c Q_t^T o M^T)(sigma dL o Eq)) + eG o (K_c Rc^K^T)] + (same with V, dout, P_L, Rc^V)
//   db   = db1 - u o du;  dlog_alpha = suffix-sum of db in the chunk - alpha o du
//          (+ the totals of all later chunks: the adjoint scan adds them to db1
//          of each chunk's last state row, so the suffix sum carries them)
// ("Native Hybrid Attention for Efficient Sequence Modeling", Paper-Notes page,
// 关键设计/层内混合 recurrence and Chunkwise 并行计算; the backward is the
// derivative of that chunked form.)
#include "nha_common.cuh"
#include "nha_kernels.h"
#include "nha_prof.h"
#include "nha_tc.cuh"
#include "nha_tc_tiles.cuh"
#include "nha_tma.h"

namespace nha {

__host__ __device__ constexpr uint32_t idesc_am(int M, int N, bool a_mn, bool b_mn) {
    return idesc_bf16(M, N, b_mn) | ((a_mn ? 1u : 0u) << 15);
}

// ---------------------------------------------------------------------------------------
struct SqMaps {
    CUtensorMap q, dout, k, v, sk, sv, dqw, dqwv, la;
};

template <int D, int M>
__global__ void __launch_bounds__(kTcThreads, 1)
bwd_sq_tc_kernel(const BwdArgs a, const __grid_constant__ SqMaps maps, int* __restrict__ status) {
    constexpr int HM = M / 2, HD = D / 2, TB = 128 * D * 2;
    constexpr int SSZ = ((2 * M * D * 2) + 1023) / 1024 * 1024;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* XE = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* XdO = XE + 16384;  // dout rows of the tile's queries
    unsigned char* XKV = XdO + TB;    // V_c, then K_c
    unsigned char* XS = XKV + TB;     // [S^V pair], then [S^K pair]   (2M rows)
    unsigned char* XM = XS + SSZ;     // masked products / G2
    unsigned char* XQ = XM + 32768;   // Q, then sigma dL o Eq
    unsigned char* XG = XQ + TB;      // G1 = sigma dL o Eb, chunk-blocked [128][2M]
    float* s_tot = reinterpret_cast<float*>(XG + 32768);  // [4][M]
    float* sG = s_tot + 4 * M;                             // [2][M]
    float* red = sG + 2 * M;                               // [2][128]
    // d = 64 leaves room for both window partials of dq, fetched once the
    // tile's first operand tiles have landed; d = 128 brings each into a tile
    // its products have consumed
    constexpr bool kPreP = D == 64;
    unsigned char* XP = reinterpret_cast<unsigned char*>(((uintptr_t)(red + 256) + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bar, lbar, ebar[2], gbar;  // MMAs; operand tiles; the two window partials; log_alpha
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = ((warp & 3) << 5) | lane, h = warp >> 2, cr = r >> 6;
    // heads fastest, tiles in decreasing order: the window-only leading tiles
    // (a copy each) start last
    const int bh = blockIdx.x, x = gridDim.y - 1 - blockIdx.y;
    const Shape sh = head_shape(a.sh, bh);
    const int W0 = sh.T - sh.R, NLT = (W0 + 127) / 128;
    if (x >= NLT + (sh.R + 127) / 128) return;  // past this head's tiles (per-head windows)
    const size_t hoff = (size_t)bh * sh.TS;
    if (x < NLT) {  // window-only queries: D = its window part; dq = window branch only
        const int tb = x * 128, n = min(128, W0 - tb);
        for (int e = tid; e < n * D / 8; e += kTcThreads) {
            const int row = e / (D / 8);
            const size_t tt = hoff + tb + row;
            const float corr = a.Dhat[tt] - a.Dwin[tt];
            float f[8], cv[8];
            unpack8(*reinterpret_cast<const uint4*>(a.hdqw + (hoff + tb) * D + e * 8), f);
            unpack8(*reinterpret_cast<const uint4*>(a.hdqwV + (hoff + tb) * D + e * 8), cv);
#pragma unroll
            for (int q = 0; q < 8; q++) f[q] += corr * cv[q];
            *reinterpret_cast<uint4*>((__nv_bfloat16*)a.dq + (hoff + tb) * D + e * 8) = pack8(f);
        }
        for (int e = tid; e < n; e += kTcThreads) a.Dv[hoff + tb + e] = a.Dwin[hoff + tb + e];
        return;
    }
    const int j0 = (x - NLT) * 128, nq = min(128, sh.R - j0), tbase = j0 + sh.w;
    const int c1 = j0 / kChunk;
    const bool has2 = nq > kChunk, row_ok = r < nq;
    const int t = tbase + r, j = j0 + r;
    const size_t jrow = (size_t)bh * sh.NCS * kChunk + j;
    const float sig = sh.sigma;

    if (tid < 2 * M) sG[tid] = 0.0f;
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_init(&lbar, 1);
        mbar_init(&ebar[0], 1);
        mbar_init(&ebar[1], 1);
        mbar_init(&gbar, 1);
        mbar_fence_init();
        s_abort = 0;
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t R0 = 0, R1 = 128, R2 = 256, R3 = 384;
    TcCtl ctl{&bar, 0u, &s_abort, status};
    bool ok = true;
    // TMA copies, issued by thread 0.  Rows past the tile's queries hold other
    // rows or zeros; every product they enter is masked or has a zero factor.
    int l_issued = 0, l_waited = 0, e_issued = 0, e_waited = 0;  // thread 0's bookkeeping
    bool g_issued = false, g_waited = false;
    auto wait_copies = [&](uint64_t* b, int& waited) {  // thread 0
        if (mbar_wait(b, (uint32_t)(waited & 1), kWaitCycles))
            waited++;
        else
            atomicExch(&s_abort, 1);
    };
    auto wait_partial = [&](int i) {  // thread 0: partial i landed (its barrier's only phase)
        if (mbar_wait(&ebar[i], 0, kWaitCycles))
            e_waited++;
        else
            atomicExch(&s_abort, 1);
    };

    // ---- value side: dP_L (tile loads in flight while the gates are computed);
    // log_alpha rows into XG, free until G1 is formed
    if (tid == 0) {
        g_issued = true;
        mbar_arrive_expect_tx(&gbar, (uint32_t)(((M + 31) / 32) * 16384));
#pragma unroll
        for (int xx = 0; xx < M; xx += 32) tma_load_3d(XG + xx * 512, &maps.la, xx, j0, bh, &gbar);
        l_issued++;
        mbar_arrive_expect_tx(&lbar, 3 * TB + 2 * M * D * 2);
#pragma unroll
        for (int xx = 0; xx < D; xx += 64) {
            tma_load_3d(XdO + xx * 256, &maps.dout, xx, tbase, bh, &lbar);
            tma_load_3d(XKV + xx * 256, &maps.v, xx, j0, bh, &lbar);
            tma_load_3d(XS + xx * 4 * M, &maps.sv, xx, c1 * M, bh, &lbar);
            tma_load_3d(XQ + xx * 256, &maps.q, xx, tbase, bh, &lbar);
        }
    }
    if (mbar_wait(&gbar, 0, kWaitCycles)) {
        g_waited = true;
    } else {
        atomicExch(&s_abort, 1);
    }
    float l[HM], b[HM];
    row_gates_tile<M>(XG, row_ok, l, b, s_tot, sG, warp, lane, h, r, nq);
    float rho[HM];
#pragma unroll
    for (int jj = 0; jj < HM; jj++) rho[jj] = 0.5f * sG[cr * M + h * HM + jj];
    {  // Ek tile
        float ek[HM];
#pragma unroll
        for (int jj = 0; jj < HM; jj++) ek[jj] = row_ok ? fexp(rho[jj] - b[jj]) * one_minus_exp(l[jj]) : 0.0f;
        store_row(XE, r, h * HM, ek, HM);
    }
    const float lse_r = row_ok ? a.lse[hoff + t] : 0.0f;
    const float Dwin_r = row_ok ? a.Dwin[hoff + t] : 0.0f;
    const float Dhat_r = row_ok ? a.Dhat[hoff + t] : 0.0f;
    float D_r = 0.0f;  // exact D = window part + slot part, set below

    sync_for_mma();
    if (tid == 0) {
        wait_copies(&lbar, l_waited);
        fence_after_sync();
        const uint32_t sd = smem_u32(XdO), sk = smem_u32(XKV), ss = smem_u32(XS);
        for (int kk = 0; kk < D / 16; kk++)
            mma_bf16(tm + R0, desc_k(sd, 128, kk), desc_k(sk, 128, kk), idesc_bf16(128, 128, false), kk > 0);
        for (int kk = 0; kk < D / 16; kk++)
            mma_bf16(tm + R1, desc_k(sd, 128, kk), desc_k(ss, 2 * M, kk), idesc_bf16(128, 2 * M, false), kk > 0);
        mma_commit(&bar);
    }
    float dpl[HM];
    if ((ok = ctl.wait() && !s_abort)) {
        if (tid == 0) {  // V_c and [S^V] consumed: the key side's tiles go in flight
            l_issued++;
            mbar_arrive_expect_tx(&lbar, TB + 2 * M * D * 2);
#pragma unroll
            for (int xx = 0; xx < D; xx += 64) {
                tma_load_3d(XKV + xx * 256, &maps.k, xx, j0, bh, &lbar);
                tma_load_3d(XS + xx * 4 * M, &maps.sk, xx, c1 * M, bh, &lbar);
            }
        }
        mask_to_tile(tl + R0, XM, r, h, cr, row_ok, false);
        sync_for_mma();
        if (tid == 0) {
            const uint32_t sm = smem_u32(XM), se = smem_u32(XE);
            for (int kk = 0; kk < 8; kk++)
                mma_bf16(tm + R0, desc_k(sm, 128, kk), desc_mn(se, 128, kk), idesc_bf16(128, M, true), kk > 0);
            mma_commit(&bar);
        }
        ok = ctl.wait();
    }
    if (ok) {
        float so[HM], pin[HM];
        tmem_ld(tl + R1 + cr * M + h * HM, so, HM);
        tmem_ld(tl + R0 + h * HM, pin, HM);
#pragma unroll
        for (int jj = 0; jj < HM; jj++) dpl[jj] = fexp(b[jj]) * so[jj] + fexp(b[jj] - rho[jj]) * pin[jj];
        // ---- key side: slot logits
        sync_for_mma();
        if (tid == 0) {
            wait_copies(&lbar, l_waited);
            if (kPreP) {  // both dq partials at once, into XP (one phase of ebar[0])
                e_issued++;
                mbar_arrive_expect_tx(&ebar[0], 2 * TB);
#pragma unroll
                for (int xx = 0; xx < D; xx += 64) {
                    tma_load_3d(XP + xx * 256, &maps.dqw, xx, tbase, bh, &ebar[0]);
                    tma_load_3d(XP + TB + xx * 256, &maps.dqwv, xx, tbase, bh, &ebar[0]);
                }
            }
            fence_after_sync();
            const uint32_t sq = smem_u32(XQ), sk = smem_u32(XKV), ss = smem_u32(XS);
            for (int kk = 0; kk < D / 16; kk++)
                mma_bf16(tm + R0, desc_k(sq, 128, kk), desc_k(sk, 128, kk), idesc_bf16(128, 128, false), kk > 0);
            for (int kk = 0; kk < D / 16; kk++)
                mma_bf16(tm + R1, desc_k(sq, 128, kk), desc_k(ss, 2 * M, kk), idesc_bf16(128, 2 * M, false), kk > 0);
            mma_commit(&bar);
        }
        ok = ctl.wait();
    }
    if (ok) {
        mask_to_tile(tl + R0, XM, r, h, cr, row_ok, false);
        sync_for_mma();
        if (tid == 0) {
            const uint32_t sm = smem_u32(XM), se = smem_u32(XE);
            for (int kk = 0; kk < 8; kk++)
                mma_bf16(tm + R0, desc_k(sm, 128, kk), desc_mn(se, 128, kk), idesc_bf16(128, M, true), kk > 0);
            mma_commit(&bar);
        }
        ok = ctl.wait();
    }
    float weq[HM];
    if (ok) {
        float si[HM], lin[HM], g1[HM], g2[HM], z[HM];
        tmem_ld(tl + R1 + cr * M + h * HM, si, HM);
        tmem_ld(tl + R0 + h * HM, lin, HM);
        __nv_bfloat16* wsDL = a.hDL + jrow * M + h * HM;
        __nv_bfloat16* wsPL = a.hPL + jrow * M + h * HM;
        float* wsDB = a.wsDB1 + jrow * M + h * HM;
        float Lv[HM], pl[HM];
        float sp = 0.0f;
#pragma unroll
        for (int jj = 0; jj < HM; jj++) {
            const float eb = fexp(b[jj]), eq = fexp(b[jj] - rho[jj]);
            Lv[jj] = sig * (eb * si[jj] + eq * lin[jj]);
            pl[jj] = row_ok ? fexp(Lv[jj] - lse_r) : 0.0f;
            sp += pl[jj] * dpl[jj];
        }
        red[h * 128 + r] = sp;
        __syncthreads();
        D_r = Dwin_r + red[r] + red[128 + r];
        if (h == 0 && row_ok) a.Dv[hoff + t] = D_r;
        float sdl[HM], db1[HM];
#pragma unroll
        for (int jj = 0; jj < HM; jj++) {
            const float eb = fexp(b[jj]), eq = fexp(b[jj] - rho[jj]);
            const float dl = pl[jj] * (dpl[jj] - D_r);
            db1[jj] = dl * Lv[jj] + pl[jj] * dpl[jj];
            sdl[jj] = sig * dl;
            g1[jj] = sig * dl * eb;
            g2[jj] = pl[jj] * eb;
            weq[jj] = sig * dl * eq;
            z[jj] = 0.0f;
        }
        if (row_ok) {
#pragma unroll
            for (int jj = 0; jj < HM; jj += 8) {
                *reinterpret_cast<uint4*>(wsDL + jj) = pack8(sdl + jj);
                *reinterpret_cast<uint4*>(wsPL + jj) = pack8(pl + jj);
            }
#pragma unroll
            for (int jj = 0; jj < HM; jj += 4)
                *reinterpret_cast<float4*>(wsDB + jj) = make_float4(db1[jj], db1[jj + 1], db1[jj + 2], db1[jj + 3]);
        }
        // chunk-blocked [128][2M] tiles; columns >= 2M are zero
        store_row(XG, r, cr * M + h * HM, g1, HM);
        store_row(XG, r, (1 - cr) * M + h * HM, z, HM);
        store_row(XM, r, cr * M + h * HM, g2, HM);
        store_row(XM, r, (1 - cr) * M + h * HM, z, HM);
        if (2 * M < 128) {
            const int span = (128 - 2 * M) / 2;
            zero_cols(XG, r, 2 * M + h * span, 2 * M + (h + 1) * span);
            zero_cols(XM, r, 2 * M + h * span, 2 * M + (h + 1) * span);
        }
        sync_for_mma();
        if (tid == 0) {  // dR^K = G1^T Q, dR^V = G2^T dout (A read MN-major: rows = slots)
            const uint32_t sg = smem_u32(XG), sq = smem_u32(XQ), sm = smem_u32(XM), sd = smem_u32(XdO);
            for (int kk = 0; kk < 8; kk++)
                mma_bf16(tm + R1, desc_mn(sg, 128, kk), desc_mn(sq, 128, kk), idesc_am(128, D, true, true), kk > 0);
            for (int kk = 0; kk < 8; kk++)
                mma_bf16(tm + R2, desc_mn(sm, 128, kk), desc_mn(sd, 128, kk), idesc_am(128, D, true, true), kk > 0);
            mma_commit(&bar);
        }
        ok = ctl.wait() && !s_abort;
    }
    if (ok) {
        if (!kPreP && tid == 0) {  // dout consumed: the window partial dq goes in flight into its tile
            e_issued++;
            mbar_arrive_expect_tx(&ebar[0], TB);
#pragma unroll
            for (int xx = 0; xx < D; xx += 64) tma_load_3d(XdO + xx * 256, &maps.dqw, xx, tbase, bh, &ebar[0]);
        }
        // Row n of the result = slot n % M of chunk n / M.  Each 32-column slab of
        // both results goes through shared memory so every global store is a
        // run of whole rows.
        float* slab = reinterpret_cast<float*>(XM);  // [2][128 rows][32] fp32 = 32 KB
        for (int c0 = 0; c0 < D; c0 += 32) {
            if (h == (c0 < HD ? 0 : 1)) {
                float vk[32], vv[32];
                tmem_ld32(tl + R1 + c0, vk);
                tmem_ld32(tl + R2 + c0, vv);
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const int sw = (e + 4 * (r & 7)) & 31;  // rotate 16-byte chunks across rows
                    *reinterpret_cast<float4*>(slab + r * 32 + sw) = make_float4(vk[e], vk[e + 1], vk[e + 2], vk[e + 3]);
                    *reinterpret_cast<float4*>(slab + 4096 + r * 32 + sw) = make_float4(vv[e], vv[e + 1], vv[e + 2], vv[e + 3]);
                }
            }
            __syncthreads();
            for (int e = tid; e < 2 * 2 * M * 4; e += kTcThreads) {  // (array, row n < 2M, 8 columns)
                const int arr = e / (2 * M * 4), n = (e / 4) % (2 * M), ch = e % 4;
                const int cc = n / M, i = n % M;
                if (cc == 0 || has2) {
                    const float* src = slab + arr * 4096 + n * 32;
                    const float4 lo = *reinterpret_cast<const float4*>(src + ((8 * ch + 4 * (n & 7)) & 31));
                    const float4 hi = *reinterpret_cast<const float4*>(src + ((8 * ch + 4 + 4 * (n & 7)) & 31));
                    __nv_bfloat16* dst =
                        (arr == 0 ? a.hRK : a.hRV) + (((size_t)bh * sh.NCS + c1 + cc) * M + i) * D + c0 + 8 * ch;
                    *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16(lo.x, lo.y), pack_bf16(lo.z, lo.w),
                                                                pack_bf16(hi.x, hi.y), pack_bf16(hi.z, hi.w));
                }
            }
            __syncthreads();
        }
        // ---- dq_slot = G1 [S^K pair] + ((sigma dL o Eq) Ek^T o M) K_c
        store_row(XQ, r, h * HM, weq, HM);
        sync_for_mma();
        if (tid == 0) {
            const uint32_t sg = smem_u32(XG), ss = smem_u32(XS), sq = smem_u32(XQ), se = smem_u32(XE);
            for (int kk = 0; kk < 2 * M / 16; kk++)
                mma_bf16(tm + R3, desc_k(sg, 128, kk), desc_mn(ss, 2 * M, kk), idesc_bf16(128, D, true), kk > 0);
            for (int kk = 0; kk < M / 16; kk++)
                mma_bf16(tm + R0, desc_k(sq, 128, kk), desc_k(se, 128, kk), idesc_bf16(128, 128, false), kk > 0);
            mma_commit(&bar);
        }
        ok = ctl.wait();
    }
    if (ok) {
        if (!kPreP && tid == 0) {  // G1 consumed: the dq correction partial goes in flight into its tile
            e_issued++;
            mbar_arrive_expect_tx(&ebar[1], TB);
#pragma unroll
            for (int xx = 0; xx < D; xx += 64) tma_load_3d(XG + xx * 256, &maps.dqwv, xx, tbase, bh, &ebar[1]);
        }
        mask_to_tile(tl + R0, XM, r, h, cr, row_ok, false);
        sync_for_mma();
        if (tid == 0) {
            const uint32_t sm = smem_u32(XM), sk = smem_u32(XKV);
            for (int kk = 0; kk < 8; kk++)
                mma_bf16(tm + R3, desc_k(sm, 128, kk), desc_mn(sk, 128, kk), idesc_bf16(128, D, true), 1u);
            mma_commit(&bar);
        }
        ok = ctl.wait();
    }
    if (ok) {
        // dq = window partial + (D^ - D) correction + slot part, staged in XM
        // (its mask is consumed), copied out coalesced
        const float corr = Dhat_r - D_r;
        if (tid == 0) {
            wait_partial(0);
            if (!kPreP) wait_partial(1);
        }
        const unsigned char* pq = kPreP ? XP : XdO;      // window partial dq
        const unsigned char* pc = kPreP ? XP + TB : XG;  // its D correction partial
        ok = !__syncthreads_or(s_abort);
        if (ok) {
#pragma unroll
            for (int c0 = 0; c0 < HD; c0 += 32) {
                float g[32];
                tmem_ld32(tl + R3 + h * HD + c0, g);
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    const uint32_t off = sw_chunk(r, (h * HD + c0 + e) >> 3, 128);
                    float f[8], c8[8];
                    unpack8(*reinterpret_cast<const uint4*>(pq + off), f);
                    unpack8(*reinterpret_cast<const uint4*>(pc + off), c8);
#pragma unroll
                    for (int q = 0; q < 8; q++) f[q] += g[e + q] + corr * c8[q];
                    *reinterpret_cast<uint4*>(XM + off) = pack8(f);
                }
            }
            __syncthreads();
            constexpr int CH = D / 8;
            __nv_bfloat16* ob = (__nv_bfloat16*)a.dq + (hoff + tbase) * D;
            for (int e = tid; e < nq * CH; e += kTcThreads) {
                const int rr = e / CH, ch = e % CH;
                *reinterpret_cast<uint4*>(ob + (size_t)rr * D + ch * 8) =
                    *reinterpret_cast<const uint4*>(XM + sw_chunk(rr, ch, 128));
            }
        }
    }
    if (!ok && row_ok && h == 0) ((__nv_bfloat16*)a.dq)[(hoff + t) * D] = __float2bfloat16_rn(__int_as_float(0x7fc00000));
    if (!ok && tid == 0) {  // let in-flight MMAs and copies drain
        mbar_wait(&bar, ctl.phase ^ 1u, kWaitCycles);
        for (int q = l_waited; q < l_issued; q++) mbar_wait(&lbar, (uint32_t)(q & 1), kWaitCycles);
        for (int q = e_waited; q < e_issued; q++) mbar_wait(&ebar[q], 0, kWaitCycles);
        if (g_issued && !g_waited) mbar_wait(&gbar, 0, kWaitCycles);
        atomicOr(status, kStatusTimeoutBit);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

// ---------------------------------------------------------------------------------------
struct SkMaps {
    CUtensorMap q, dout, k, v, rk, rv, dkw, dvw, la, dl, pl, db1;
};

template <int D, int M>
__global__ void __launch_bounds__(kTcThreads, 1)
bwd_sk_tc_kernel(const BwdArgs a, const __grid_constant__ SkMaps maps, int* __restrict__ status) {
    constexpr int HM = M / 2, HD = D / 2, TB = 128 * D * 2;
    constexpr int SSZ = ((2 * M * D * 2) + 1023) / 1024 * 1024;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* XE = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* XW = XE + 16384;   // W o Eq  [128 j][M]
    unsigned char* XEG = XW + 16384;  // Ek o eG chunk-blocked [128][2M]
    unsigned char* XA = XEG + 32768;  // q_t or dout_t rows
    unsigned char* XB = XA + TB;      // k_c or v_c rows
    unsigned char* XR = XB + TB;      // [Rc pair]  (2M rows)
    unsigned char* XM1 = XR + SSZ;
    unsigned char* XM2 = XM1 + 32768;
    float* s_tot = reinterpret_cast<float*>(XM2 + 32768);  // [4][M]; exp(G / 2) [2][M] during the passes
    float* sG = s_tot + 4 * M;                              // [2][M]
    // d = 64 leaves room for both window partials (dk, dv rows of the tile)
    // from the start; d = 128 brings each into XB as soon as the pass's first
    // products have consumed its k (v) rows, and the second pass's v rows
    // follow the first pass's dk
    constexpr bool kPreP = D == 64;
    unsigned char* XP = reinterpret_cast<unsigned char*>(((uintptr_t)(sG + 2 * M) + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bar, lbar, ebar, dbar, gbar, vbar;  // MMAs; pass operands; window partials; db1;
                                                            // log_alpha + dL; the second pass's v rows (d = 128)
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = ((warp & 3) << 5) | lane, h = warp >> 2, cr = r >> 6;
    // heads fastest, key tiles in increasing order: the tiles past the last
    // state row (a copy each) start last
    const int bh = blockIdx.x, x = blockIdx.y;
    const Shape sh = head_shape(a.sh, bh);
    const size_t hoff = (size_t)bh * sh.TS;
    const int sbase = x * 128, nk = min(128, sh.T - sbase);
    if (nk <= 0) return;  // past this head's keys (per-sequence lengths)
    const int nc = max(0, min(128, sh.R - sbase));
    const int s = sbase + r;
    const bool row_ok = r < nk, slot_ok = r < nc;
    if (nc == 0) {  // tokens that never enter a state read by a query
        if (row_ok) {
            const uint4* gk = reinterpret_cast<const uint4*>(a.hdkw + (hoff + s) * D + h * HD);
            const uint4* gv = reinterpret_cast<const uint4*>(a.hdvw + (hoff + s) * D + h * HD);
            uint4* ok_ = reinterpret_cast<uint4*>((__nv_bfloat16*)a.dk + (hoff + s) * D + h * HD);
            uint4* ov_ = reinterpret_cast<uint4*>((__nv_bfloat16*)a.dv + (hoff + s) * D + h * HD);
            for (int c = 0; c < HD / 8; c++) {
                ok_[c] = gk[c];
                ov_[c] = gv[c];
            }
            float* dla = a.dla + (hoff + s) * M + h * HM;
#pragma unroll
            for (int jj = 0; jj < HM; jj++) dla[jj] = 0.0f;
        }
        return;
    }
    const int c1 = sbase / kChunk;

    if (tid < 2 * M) sG[tid] = 0.0f;
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_init(&lbar, 1);
        mbar_init(&ebar, 1);
        mbar_init(&dbar, 1);
        mbar_init(&gbar, 1);
        mbar_init(&vbar, 1);
        mbar_fence_init();
        s_abort = 0;
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t R0 = 0, R1 = 128, R2 = 256, R3 = 384;
    TcCtl ctl{&bar, 0u, &s_abort, status};
    bool ok = true;

    // TMA (thread 0): q_t / dout_t rows, k / v rows and the [Rc pair] of a
    // pass.  Rows past the tile's states hold other tokens or zeros; every
    // product they enter is multiplied by a zero gate or masked away.
    int l_issued = 0, l_waited = 0, e_issued = 0, e_waited = 0;  // thread 0's copy bookkeeping
    bool d_issued = false, g_issued = false, g_waited = false, v_issued = false, v_waited = false;
    // the second pass also brings P_L into XW (W o Eq is formed in place)
    auto issue_loads = [&](int pass) {
        if (tid != 0) return;
        const bool with_b = kPreP || pass == 0;  // XB holds the first pass's dk at d = 128
        l_issued++;
        mbar_arrive_expect_tx(&lbar, (with_b ? 2 : 1) * TB + 2 * M * D * 2 + (pass == 1 ? 16384 : 0));
#pragma unroll
        for (int xx = 0; xx < D; xx += 64) {
            tma_load_3d(XA + xx * 256, pass == 0 ? &maps.q : &maps.dout, xx, sbase + sh.w, bh, &lbar);
            if (with_b) tma_load_3d(XB + xx * 256, pass == 0 ? &maps.k : &maps.v, xx, sbase, bh, &lbar);
            tma_load_3d(XR + xx * 4 * M, pass == 0 ? &maps.rk : &maps.rv, xx, c1 * M, bh, &lbar);
        }
        if (pass == 1) tma_load_3d(XW, &maps.pl, 0, sbase, bh, &lbar);
    };
    auto issue_v = [&]() {  // d = 128: the second pass's v rows into XB, once dk is out
        if (tid != 0) return;
        fence_async_smem();
        v_issued = true;
        mbar_arrive_expect_tx(&vbar, TB);
#pragma unroll
        for (int xx = 0; xx < D; xx += 64) tma_load_3d(XB + xx * 256, &maps.v, xx, sbase, bh, &vbar);
    };
    // d = 128: window partial dk or dv of the tile's rows into XB (its k or v
    // rows are consumed by the pass's first products)
    auto issue_partial = [&](int pass) {
        if (tid != 0) return;
        e_issued++;
        mbar_arrive_expect_tx(&ebar, TB);
#pragma unroll
        for (int xx = 0; xx < D; xx += 64)
            tma_load_3d(XB + xx * 256, pass == 0 ? &maps.dkw : &maps.dvw, xx, sbase, bh, &ebar);
    };
    if (kPreP && tid == 0) {  // both partials at once, into XP (one phase of ebar)
        e_issued++;
        mbar_arrive_expect_tx(&ebar, 2 * TB);
#pragma unroll
        for (int xx = 0; xx < D; xx += 64) {
            tma_load_3d(XP + xx * 256, &maps.dkw, xx, sbase, bh, &ebar);
            tma_load_3d(XP + TB + xx * 256, &maps.dvw, xx, sbase, bh, &ebar);
        }
    }
    if (tid == 0) {  // log_alpha rows into XM1 (free until the first masks), sigma dL into XW
        g_issued = true;
        mbar_arrive_expect_tx(&gbar, (uint32_t)(((M + 31) / 32) * 16384 + 16384));
#pragma unroll
        for (int xx = 0; xx < M; xx += 32) tma_load_3d(XM1 + xx * 512, &maps.la, xx, sbase, bh, &gbar);
        tma_load_3d(XW, &maps.dl, 0, sbase, bh, &gbar);
    }
    issue_loads(0);  // in flight while the gates are computed
    if (mbar_wait(&gbar, 0, kWaitCycles)) {
        g_waited = true;
    } else {
        atomicExch(&s_abort, 1);
    }
    float l[HM], b[HM];
    row_gates_tile<M>(XM1, slot_ok, l, b, s_tot, sG, warp, lane, h, r, nc);
    // bq = b - rho (rho = G / 2) is all the passes need of b; exp(G - rho) =
    // exp(rho), one value per chunk and slot, is formed once into s_tot (free
    // until the closing suffix sum)
    if (tid < 2 * M) s_tot[tid] = fexp(0.5f * sG[tid]);
    const float* Grow = sG + cr * M + h * HM;
    const float* EGrow = s_tot + cr * M + h * HM;
#pragma unroll
    for (int jj = 0; jj < HM; jj++) b[jj] -= 0.5f * Grow[jj];
    __syncthreads();
    {
        float ek[HM], eke[HM], z[HM];
#pragma unroll
        for (int jj = 0; jj < HM; jj++) {
            ek[jj] = slot_ok ? fexp(-b[jj]) * one_minus_exp(l[jj]) : 0.0f;
            eke[jj] = ek[jj] * EGrow[jj];
            z[jj] = 0.0f;
        }
        store_row(XE, r, h * HM, ek, HM);
        store_row(XEG, r, cr * M + h * HM, eke, HM);
        store_row(XEG, r, (1 - cr) * M + h * HM, z, HM);
    }
    float du[HM];
#pragma unroll
    for (int jj = 0; jj < HM; jj++) du[jj] = 0.0f;

    for (int pass = 0; pass < 2 && ok; pass++) {
        if (pass == 1) {  // the second pass's tiles, P_L among them
            if (mbar_wait(&lbar, 1, kWaitCycles)) {
                if (tid == 0) l_waited++;
            } else {
                atomicExch(&s_abort, 1);
            }
            if (!kPreP) {
                if (mbar_wait(&vbar, 0, kWaitCycles)) {
                    if (tid == 0) v_waited = true;
                } else {
                    atomicExch(&s_abort, 1);
                }
            }
        }
        {
            float weq[HM];
#pragma unroll
            for (int jj = 0; jj < HM; jj += 8) {
                float w8[8];
                if (slot_ok) {
                    unpack8(*reinterpret_cast<const uint4*>(XW + sw_chunk(r, (h * HM + jj) >> 3, 128)), w8);
                } else {
#pragma unroll
                    for (int q = 0; q < 8; q++) w8[q] = 0.0f;
                }
#pragma unroll
                for (int q = 0; q < 8; q++) weq[jj + q] = w8[q] * fexp(b[jj + q]);
            }
            store_row(XW, r, h * HM, weq, HM);
        }
        sync_for_mma();
        if (tid == 0) {
            // the first pass's tiles landed (the second pass's were waited above)
            if (pass == 0) {
                if (mbar_wait(&lbar, 0, kWaitCycles))
                    l_waited++;
                else
                    atomicExch(&s_abort, 1);
            }
            fence_after_sync();
            const uint32_t se = smem_u32(XE), sw = smem_u32(XW), sa = smem_u32(XA), sb = smem_u32(XB),
                           sr = smem_u32(XR);
            for (int kk = 0; kk < M / 16; kk++)
                mma_bf16(tm + R0, desc_k(se, 128, kk), desc_k(sw, 128, kk), idesc_bf16(128, 128, false), kk > 0);
            for (int kk = 0; kk < D / 16; kk++)
                mma_bf16(tm + R1, desc_k(sb, 128, kk), desc_k(sa, 128, kk), idesc_bf16(128, 128, false), kk > 0);
            for (int kk = 0; kk < D / 16; kk++)
                mma_bf16(tm + R2, desc_k(sb, 128, kk), desc_k(sr, 2 * M, kk), idesc_bf16(128, 2 * M, false), kk > 0);
            mma_commit(&bar);
        }
        if (!(ok = ctl.wait())) break;
        if (!kPreP) issue_partial(pass);  // k (v) rows consumed
        mask_to_tile(tl + R0, XM1, r, h, cr, slot_ok, true);
        mask_to_tile(tl + R1, XM2, r, h, cr, slot_ok, true);
        float inter[HM];
        tmem_ld(tl + R2 + cr * M + h * HM, inter, HM);
        sync_for_mma();
        if (tid == 0) {
            const uint32_t s1 = smem_u32(XM1), s2 = smem_u32(XM2), sa = smem_u32(XA), sg = smem_u32(XEG),
                           sr = smem_u32(XR), sw = smem_u32(XW);
            for (int kk = 0; kk < 8; kk++)
                mma_bf16(tm + R3, desc_k(s1, 128, kk), desc_mn(sa, 128, kk), idesc_bf16(128, D, true), kk > 0);
            for (int kk = 0; kk < 2 * M / 16; kk++)
                mma_bf16(tm + R3, desc_k(sg, 128, kk), desc_mn(sr, 2 * M, kk), idesc_bf16(128, D, true), 1u);
            for (int kk = 0; kk < 8; kk++)
                mma_bf16(tm + R0, desc_k(s2, 128, kk), desc_mn(sw, 128, kk), idesc_bf16(128, M, true), kk > 0);
            mma_commit(&bar);
        }
        if (!(ok = ctl.wait()) || s_abort) {
            ok = false;
            break;
        }
        if (pass == 0) issue_loads(1);  // the operand tiles are free: next pass in flight
        if (pass == 1 && tid == 0) {    // db1 rows of the tile for the gate gradient, into XA
            d_issued = true;             // (32-column boxes, 128-byte swizzle, like log_alpha)
            mbar_arrive_expect_tx(&dbar, (uint32_t)(((M + 31) / 32) * 16384));
#pragma unroll
            for (int xx = 0; xx < M; xx += 32) tma_load_3d(XA + xx * 512, &maps.db1, xx, sbase, bh, &dbar);
        }
        {
            float intra[HM];
            tmem_ld(tl + R0 + h * HM, intra, HM);
#pragma unroll
            for (int jj = 0; jj < HM; jj++)
                du[jj] += fexp(-b[jj]) * (intra[jj] + EGrow[jj] * inter[jj]);
        }
        // dk (dv) = window partial + slot part, staged in XM2 and copied out
        if (!kPreP || pass == 0) {
            if (mbar_wait(&ebar, kPreP ? 0u : (uint32_t)pass, kWaitCycles)) {
                if (tid == 0) e_waited++;
            } else {
                atomicExch(&s_abort, 1);
            }
        }
        const unsigned char* part = kPreP ? XP + pass * TB : XB;
#pragma unroll
        for (int c0 = 0; c0 < HD; c0 += 32) {
            float g[32];
            tmem_ld32(tl + R3 + h * HD + c0, g);
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
                const uint32_t off = sw_chunk(r, (h * HD + c0 + e) >> 3, 128);
                float f[8];
                unpack8(*reinterpret_cast<const uint4*>(part + off), f);
#pragma unroll
                for (int q = 0; q < 8; q++) f[q] += g[e + q];
                *reinterpret_cast<uint4*>(XM2 + off) = pack8(f);
            }
        }
        fence_before_sync();
        if (__syncthreads_or(s_abort)) {
            ok = false;
            break;
        }
        if (!kPreP && pass == 0) issue_v();  // dk read out of XB
        {  // rows [0, nk) of the staged tile, 16-byte chunks, coalesced
            constexpr int CH = D / 8;
            __nv_bfloat16* ob = (__nv_bfloat16*)(pass == 0 ? a.dk : a.dv) + (hoff + sbase) * D;
            for (int e = tid; e < nk * CH; e += kTcThreads) {
                const int rr = e / CH, ch = e % CH;
                *reinterpret_cast<uint4*>(ob + (size_t)rr * D + ch * 8) =
                    *reinterpret_cast<const uint4*>(XM2 + sw_chunk(rr, ch, 128));
            }
        }
    }
    if (ok) {
        // db = db1 - u du;  dlog_alpha = (suffix sum of db in the chunk) - alpha du.
        // The carry of all later chunks sits in db1 of the chunk's last state row
        // (added by the adjoint scan), so the suffix sum hands it to every row.
        if (!mbar_wait(&dbar, 0, kWaitCycles)) atomicExch(&s_abort, 1);
        float db[HM];
#pragma unroll
        for (int jj = 0; jj < HM; jj += 4) {
            const int col = h * HM + jj, c = (col & 31) >> 2;
            const float4 d4 = slot_ok ? *reinterpret_cast<const float4*>(XA + (col >> 5) * 16384 + r * 128 +
                                                                          ((c ^ (r & 7)) << 4))
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
            const float dd[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
            for (int q = 0; q < 4; q++) db[jj + q] = slot_ok ? dd[q] - one_minus_exp(l[jj + q]) * du[jj + q] : 0.0f;
        }
        chunk_suffix<M>(db, s_tot, warp, lane, h);
        // staged in XB (16-byte chunk q of the half row at q ^ (r & 7)), copied out coalesced
        constexpr int QM = HM / 4 - 1;
        float* st = reinterpret_cast<float*>(XB) + r * M + h * HM;
#pragma unroll
        for (int jj = 0; jj < HM; jj += 4) {
            float o4[4];
#pragma unroll
            for (int q = 0; q < 4; q++) o4[q] = slot_ok ? db[jj + q] - fexp(l[jj + q]) * du[jj + q] : 0.0f;
            *reinterpret_cast<float4*>(st + 4 * ((jj / 4) ^ (r & QM))) = make_float4(o4[0], o4[1], o4[2], o4[3]);
        }
        if (__syncthreads_or(s_abort)) {
            ok = false;
        } else {
            constexpr int C4 = M / 4;  // 16-byte chunks per row
            float* ob = a.dla + (hoff + sbase) * M;
            for (int e = tid; e < nk * C4; e += kTcThreads) {
                const int rr = e / C4, c = e % C4, hh = c / (HM / 4), q = c % (HM / 4);
                *reinterpret_cast<float4*>(ob + (size_t)rr * M + 4 * c) = *reinterpret_cast<const float4*>(
                    reinterpret_cast<const float*>(XB) + rr * M + hh * HM + 4 * (q ^ (rr & QM)));
            }
        }
    }
    if (!ok && row_ok && h == 0) {
        a.dla[(hoff + s) * M] = __int_as_float(0x7fc00000);
    }
    if (!ok && tid == 0) {  // let in-flight MMAs and copies drain
        mbar_wait(&bar, ctl.phase ^ 1u, kWaitCycles);
        for (int q = l_waited; q < l_issued; q++) mbar_wait(&lbar, (uint32_t)(q & 1), kWaitCycles);
        for (int q = e_waited; q < e_issued; q++) mbar_wait(&ebar, (uint32_t)(q & 1), kWaitCycles);
        if (d_issued) mbar_wait(&dbar, 0, kWaitCycles);
        if (v_issued && !v_waited) mbar_wait(&vbar, 0, kWaitCycles);
        if (g_issued && !g_waited) mbar_wait(&gbar, 0, kWaitCycles);
        atomicOr(status, kStatusTimeoutBit);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

template <int D, int M>
size_t sq_smem() {
    const size_t base = 1024 + 16384 + 3 * 128 * D * 2 + ((2 * M * D * 2) + 1023) / 1024 * 1024 + 2 * 32768 +
                        6 * M * 4 + 256 * 4;
    return D == 64 ? (base + 1023) / 1024 * 1024 + 2 * 128 * D * 2 : base;  // + the two dq partials
}
template <int D, int M>
size_t sk_smem() {
    const size_t base = 1024 + 2 * 16384 + 32768 + 2 * 128 * D * 2 + ((2 * M * D * 2) + 1023) / 1024 * 1024 +
                        2 * 32768 + 6 * M * 4;
    return D == 64 ? (base + 1023) / 1024 * 1024 + 2 * 128 * D * 2 : base;  // + the two window partials
}

template <int D, int M>
cudaError_t tc_bwd_slot(const BwdArgs& a, const __nv_bfloat16* qr, const __nv_bfloat16* kr, const float2* tab,
                        int* status, cudaStream_t st) {
    const Shape& sh = a.sh;
    cudaError_t e;
    const int W0 = sh.T - sh.R;
    // with per-head windows a head has at most ceil(T / 128) + 1 query tiles
    const int qtiles = varied(sh) ? (sh.T + 127) / 128 + 1 : (W0 + 127) / 128 + (sh.R + 127) / 128;
    {
        SqMaps maps;
        const int ncm = (sh.NCS > 0 ? sh.NCS : 1) * M;
        if ((e = tmap_rows_bf16(&maps.q, a.q, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.dout, a.dout, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.k, a.k, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.v, a.v, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.sk, a.SKb, D, ncm, sh.BH, 2 * M)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.sv, a.SVb, D, ncm, sh.BH, 2 * M)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.dqw, a.hdqw, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.dqwv, a.hdqwV, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_f32(&maps.la, a.la, M, sh.T, sh.BH)) != cudaSuccess)
            return e;
        auto kern = bwd_sq_tc_kernel<D, M>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sq_smem<D, M>())) != cudaSuccess)
            return e;
        if (qtiles > 0)
            NHA_LAUNCH("bwd_sq_tc", st, kern<<<dim3(sh.BH, qtiles), kTcThreads, sq_smem<D, M>(), st>>>(a, maps, status));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        // queries t < w reading initial states: their slot part of D and dq
        if ((e = launch_h0_bwd_lead<__nv_bfloat16, D, M>(a, true, st)) != cudaSuccess) return e;
    }
    // the bandwidth-bound adjoint scan shares the SMs with the key-major kernel
    Fork* f = nullptr;
    if ((e = get_fork(&f)) != cudaSuccess) return e;
    if ((e = fork_side(st, *f, 2)) != cudaSuccess) return e;
    if ((e = launch_adj_scan(a, M, D, f->side)) != cudaSuccess) return e;
    if ((e = launch_wkv<D>(a, qr, kr, tab, status, st)) != cudaSuccess) return e;
    if ((e = join_side(st, *f, 3)) != cudaSuccess) return e;
    {
        SkMaps maps;
        const int ncm = (sh.NCS > 0 ? sh.NCS : 1) * M;
        if ((e = tmap_rows_bf16(&maps.q, a.q, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.dout, a.dout, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.k, a.k, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.v, a.v, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.rk, a.RKb, D, ncm, sh.BH, 2 * M)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.rv, a.RVb, D, ncm, sh.BH, 2 * M)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.dkw, a.hdkw, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.dvw, a.hdvw, D, sh.T, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_f32(&maps.la, a.la, M, sh.T, sh.BH)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.dl, a.hDL, M, ncm / M * kChunk, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_bf16(&maps.pl, a.hPL, M, ncm / M * kChunk, sh.BH, 128)) != cudaSuccess ||
            (e = tmap_rows_f32(&maps.db1, a.wsDB1, M, ncm / M * kChunk, sh.BH)) != cudaSuccess)
            return e;
        auto kern = bwd_sk_tc_kernel<D, M>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sk_smem<D, M>())) != cudaSuccess)
            return e;
        NHA_LAUNCH("bwd_sk_tc", st,
                   kern<<<dim3(sh.BH, (sh.T + 127) / 128), kTcThreads, sk_smem<D, M>(), st>>>(a, maps, status));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return launch_dh0<__nv_bfloat16, D, M>(a, st);
}

#define NHA_TCS_INST(D, M)                                                                              \
    template cudaError_t tc_bwd_slot<D, M>(const BwdArgs&, const __nv_bfloat16*, const __nv_bfloat16*, \
                                           const float2*, int*, cudaStream_t);
NHA_TCS_INST(64, 16)
NHA_TCS_INST(64, 32)
NHA_TCS_INST(64, 64)
NHA_TCS_INST(128, 16)
NHA_TCS_INST(128, 32)
NHA_TCS_INST(128, 64)

}  // namespace nha
