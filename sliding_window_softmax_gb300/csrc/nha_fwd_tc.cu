// Tensor-core (tcgen05) forward of the NHA operator for bf16 inputs.
//
// One CTA (256 threads) per (tile of 128 queries, head).  Query tile x < NLT
// holds queries t < w (window only); tile NLT + ct holds the queries
// t = j + w of state indices j in [128 ct, 128 ct + 128), i.e. two C = 64 gate
// chunks.  Rows of the tile live in TMEM lanes; warps w and w + 4 share the
// 32 lanes of warp w % 4 and split the columns in halves.
//
// Slot branch ("Native Hybrid Attention for Efficient Sequence Modeling",
// Paper-Notes page, Chunkwise 并行计算: linear-channel logits from the carried
// state plus cumulative / reverse gate products inside the chunk):
//   L   = sigma [ Eb o (Q S^K_prev^T) + Eq o ((Q K_c^T o M) Ek) ]
//   O_s = (p o Eb) S^V_prev + ([(p o Eq) Ek^T] o M) V_c
// with M the within-chunk causal mask, Eq = exp(b - rho), Ek = exp(rho - b) u,
// Eb = exp(b) (b: chunk-local cumsum of log_alpha).  Every product is a
// tcgen05.mma with operands in 128B-swizzled shared memory.
// Window branch: S = RoPE(Q) RoPE(K)^T over the band of 128-key blocks,
// online softmax in the log2 domain with a lazy rescale of the TMEM
// accumulator (only when the running max grows by more than 2^8), P V.
#include "nha_common.cuh"
#include "nha_kernels.h"
#include "nha_prof.h"
#include "nha_tc.cuh"
#include "nha_tc_tiles.cuh"
#include "nha_tma.h"

namespace nha {
using namespace tc;

// Forward CTA: 8 tile warps and a producer warp; three K~ / V stages.
constexpr int kFwdThreads = 288, kFwdStages = 3;

struct FwdMaps {
    CUtensorMap q, k, v, la;  // RoPE(q), RoPE(k) and v rows (window); log_alpha rows
    CUtensorMap qs, ks, sk, sv;  // q, k rows and [S^K], [S^V] pairs (slot branch)
};

template <int D, int M>
__global__ void __launch_bounds__(kFwdThreads, 1)
fwd_tc_kernel(const FwdArgs a, const __grid_constant__ FwdMaps maps, int* __restrict__ status) {
    constexpr int HM = M / 2, HD = D / 2, TB = 128 * D * 2, NS = kFwdStages;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* X0 = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* KB[NS];
    unsigned char* VB[NS];
#pragma unroll
    for (int q = 0; q < NS; q++) {
        KB[q] = X0 + TB + q * 65536;  // K~ block, then P  (slot phase: K_c, masks, A_inter / [S^K], [S^V] pair)
        VB[q] = KB[q] + 32768;        // V block           (slot phase: V_c / Ek, then pEq at +16 KB)
    }
    // slot-phase scratch and the epilogue's (m, l) exchange, in the last stage's
    // V buffer (free during both)
    float* s_tot = reinterpret_cast<float*>(VB[NS - 1]);  // [4][M]
    float* sG = s_tot + 4 * M;                             // [2][M]
    float* redm = sG + 2 * M;                              // [2][128]
    float* reds = redm + 256;                              // [2][128]
    __shared__ uint64_t bar, gbar, sbar, qbar, full[NS], sfull[2], pready, bdone[2], drain[2], s1done, s2free;
    __shared__ int s_sv_issued;  // the producer issued the [S^V] pair copy (sbar phase 1)
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int x = blockIdx.x, bh = blockIdx.y;
    const Shape sh = head_shape(a.sh, bh);
    const int W0 = sh.T - sh.R;
    const int NLT = (W0 + 127) / 128;
    if (x >= NLT + (sh.R + 127) / 128) return;  // past this head's tiles (per-head windows)
    const bool slot = x >= NLT;
    int tbase, nq, j0 = 0;
    if (!slot) {
        tbase = x * 128;
        nq = min(128, W0 - tbase);
    } else {
        j0 = (x - NLT) * 128;
        nq = min(128, sh.R - j0);
        tbase = j0 + sh.w;
    }
    const size_t hoff = (size_t)bh * sh.TS;
    const int klo = max(0, tbase - sh.w + 1), khi = tbase + nq - 1;
    const int nb = sh.w > 0 ? (khi - klo) / 128 + 1 : 0;
    volatile int* abort = &s_abort;

    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_init(&gbar, 1);
        mbar_init(&sbar, 1);
        mbar_init(&s1done, 1);
        mbar_init(&s2free, 8);
        s_sv_issued = 0;
        mbar_init(&qbar, 1);
        for (int q = 0; q < NS; q++) mbar_init(&full[q], 1);
        for (int q = 0; q < 2; q++) {
            mbar_init(&sfull[q], 1);
            mbar_init(&bdone[q], 1);
        }
        mbar_init(&pready, 8);
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        s_abort = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = s_tmem;
    // TMEM columns: S buffers at 0 and 128; O_0 (slot branch and the first 64
    // keys of every window block) at 256, O_1 (the other 64 keys) at 256 + D
    const uint32_t tA = 0, tO = 256, tO1 = 256 + D;

    int last_ph[NS];  // producer: phase of the last load issued into each stage
#pragma unroll
    for (int q = 0; q < NS; q++) last_ph[q] = -1;

    // Window block j goes through stage (j + 2) % NS: block 0 through the last
    // stage, whose K~ buffer held the slot phase's log_alpha rows and whose V
    // buffer its scratch, so it can be loaded before the slot phase ends.
    auto stage_of = [](int j) { return (j + 2) % NS; };
    if (warp == 8) {
        // ---------------- producer ----------------
        auto load_block = [&](int j) {
            const int stg = stage_of(j), kb = klo + j * 128;
            mbar_arrive_expect_tx(&full[stg], 2 * TB);
#pragma unroll
            for (int xx = 0; xx < D; xx += 64) {
                tma_load_3d(KB[stg] + xx * 256, &maps.k, xx, kb, bh, &full[stg]);
                tma_load_3d(VB[stg] + xx * 256, &maps.v, xx, kb, bh, &full[stg]);
            }
            last_ph[stg] = (j / NS) & 1;
        };
        bool q_early = false, b0_early = false;
        if (slot && lane == 0) {
            // The slot phase's first products (Q K_c^T and Q [S^K]^T) as soon as
            // their operands land, while the tile warps form the gates; then the
            // [S^V] pair into the [S^K] buffer they consumed, so its copy runs
            // during the gates and the slot logits.
            if (mbar_wait_ab(&sbar, 0, kWaitCycles, abort)) {
                fence_after_sync();
                const uint32_t s0 = smem_u32(X0), s1 = smem_u32(KB[0]), s3 = smem_u32(KB[1]);
                for (int kk = 0; kk < D / 16; kk++)
                    mma_bf16(tm + tA, desc_k(s0, 128, kk), desc_k(s1, 128, kk), idesc_bf16(128, 128, false), kk > 0);
                for (int kk = 0; kk < D / 16; kk++)
                    mma_bf16(tm + tO, desc_k(s0, 128, kk), desc_k(s3, 2 * M, kk), idesc_bf16(128, 2 * M, false), kk > 0);
                mma_commit(&bar);
                mma_commit(&s1done);
                if (mbar_wait_ab(&s1done, 0, kWaitCycles, abort)) {
                    s_sv_issued = 1;
                    mbar_arrive_expect_tx(&sbar, 2 * M * D * 2);
#pragma unroll
                    for (int xx = 0; xx < D; xx += 64)
                        tma_load_3d(KB[1] + xx * 4 * M, &maps.sv, xx, (j0 / kChunk) * M, bh, &sbar);
                    // q is read by the first products only: RoPE(q) for the window may replace it
                    if (nb > 0) {
                        q_early = true;
                        mbar_arrive_expect_tx(&qbar, TB);
#pragma unroll
                        for (int xx = 0; xx < D; xx += 64) tma_load_3d(X0 + xx * 256, &maps.q, xx, tbase, bh, &qbar);
                    }
                }
            }
            // the window's first block once the tile warps are done with the last stage
            if (nb > 0 && !s_abort && mbar_wait_ab(&s2free, 0, kWaitCycles, abort)) {
                b0_early = true;
                load_block(0);
            }
        }
        __syncwarp();
        named_sync(2, kFwdThreads);  // the slot phase is done with the stage buffers
        if (lane == 0 && nb > 0 && !s_abort) {
            const bool o0 = slot;  // O_0 already holds the slot branch
            auto issue_s = [&](int j) {
                const uint32_t s0 = smem_u32(X0), s1 = smem_u32(KB[stage_of(j)]);
                for (int kk = 0; kk < D / 16; kk++)
                    mma_bf16(tm + 128 * (j & 1), desc_k(s0, 128, kk), desc_k(s1, 128, kk),
                             idesc_bf16(128, 128, false), kk > 0);
                mma_commit(&sfull[j & 1]);
            };
            if (!q_early) {
                mbar_arrive_expect_tx(&qbar, TB);
#pragma unroll
                for (int xx = 0; xx < D; xx += 64) tma_load_3d(X0 + xx * 256, &maps.q, xx, tbase, bh, &qbar);
            }
            for (int j = b0_early ? 1 : 0; j < min(NS, nb); j++) load_block(j);
            bool ok = mbar_wait_ab(&qbar, 0, kWaitCycles, abort) &&
                      mbar_wait_ab(&full[stage_of(0)], 0, kWaitCycles, abort);
            if (ok) issue_s(0);
            for (int i = 0; i < nb && ok; i++) {
                if (i + 1 < nb) {  // S buffer (i + 1) & 1 was read by block i - 1 (before its pready)
                    if (!(ok = mbar_wait_ab(&full[stage_of(i + 1)], ((i + 1) / NS) & 1, kWaitCycles, abort))) break;
                    issue_s(i + 1);
                }
                if (!(ok = mbar_wait_ab(&pready, i & 1, kWaitCycles, abort))) break;
                fence_after_sync();
                {
                    const uint32_t sp = smem_u32(KB[stage_of(i)]), sv = smem_u32(VB[stage_of(i)]);
                    for (int kk = 0; kk < 4; kk++)
                        mma_bf16(tm + tO, desc_k(sp, 128, kk), desc_mn(sv, 128, kk), idesc_bf16(128, D, true),
                                 (o0 || i > 0 || kk > 0) ? 1u : 0u);
                    for (int kk = 4; kk < 8; kk++)
                        mma_bf16(tm + tO1, desc_k(sp, 128, kk), desc_mn(sv, 128, kk), idesc_bf16(128, D, true),
                                 (i > 0 || kk > 4) ? 1u : 0u);
                    mma_commit(&bdone[i & 1]);
                }
                if (i >= 1 && i - 1 + NS < nb) {  // block i - 1 done with its stage: refill it
                    if (!(ok = mbar_wait_ab(&bdone[(i - 1) & 1], ((i - 1) >> 1) & 1, kWaitCycles, abort))) break;
                    load_block(i - 1 + NS);
                }
            }
        }
    } else {
        // ---------------- tile threads (warps 0-7) ----------------
        const int r = ((warp & 3) << 5) | lane, h = warp >> 2, cr = r >> 6;
        const bool row_ok = r < nq;
        const float sig2 = sh.sigma * kLog2e;
        const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);  // this warp's lanes
        if (tid < 2 * M) sG[tid] = 0.0f;
        named_sync(1, kTcThreads);
        TcCtl ctl{&bar, 0u, &s_abort, status, true};
        bool ok = true;
        // online-softmax state of this thread's half of the keys (log2 domain);
        // half 0 also carries the slot branch
        float m = -INFINITY, l = 0.0f;
        bool o_valid = false;

        if (slot) {
            const int c1 = j0 / kChunk;
            // operand tiles by TMA (thread 0): q, k_c, v_c rows and the [S^K] pair.
            // Rows past the tile's states are other rows or zeros; the masks and
            // zero gates keep them out of every product.
            if (tid == 0) {  // log_alpha rows first (the gates wait for them), into the last stage's K~ buffer
                mbar_arrive_expect_tx(&gbar, (uint32_t)(((M + 31) / 32) * 16384));
#pragma unroll
                for (int xx = 0; xx < M; xx += 32) tma_load_3d(KB[NS - 1] + xx * 512, &maps.la, xx, j0, bh, &gbar);
            }
            if (tid == 0) {
                mbar_arrive_expect_tx(&sbar, 3 * TB + 2 * M * D * 2);
#pragma unroll
                for (int xx = 0; xx < D; xx += 64) {
                    tma_load_3d(X0 + xx * 256, &maps.qs, xx, tbase, bh, &sbar);
                    tma_load_3d(KB[0] + xx * 256, &maps.ks, xx, j0, bh, &sbar);
                    tma_load_3d(VB[0] + xx * 256, &maps.v, xx, j0, bh, &sbar);
                    tma_load_3d(KB[1] + xx * 4 * M, &maps.sk, xx, c1 * M, bh, &sbar);
                }
            }
            if (!mbar_wait(&gbar, 0, kWaitCycles)) *abort = 1;
            float lg[HM], b[HM], rho[HM];
            row_gates_tile<M, true>(KB[NS - 1], row_ok, lg, b, s_tot, sG, warp, lane, h, r, nq);
            {
                float ek[HM];
#pragma unroll
                for (int jj = 0; jj < HM; jj++) {
                    rho[jj] = 0.5f * sG[cr * M + h * HM + jj];
                    ek[jj] = row_ok ? fexp(rho[jj] - b[jj]) * one_minus_exp(lg[jj]) : 0.0f;
                }
                store_row(VB[1], r, h * HM, ek, HM);
            }
            sync_for_mma<true>();
            ok = ctl.wait();  // Q K_c^T and Q [S^K]^T, issued by the producer warp
            if (ok) {
                // A = Q K_c^T masked to the row's own chunk and s <= r ([S^V] is on its way)
                mask_to_tile(tl + tA, KB[0], r, h, cr, row_ok, false);
                sync_for_mma<true>();
                if (tid == 0) {
                    const uint32_t s1 = smem_u32(KB[0]), s2 = smem_u32(VB[1]);
                    for (int kk = 0; kk < 8; kk++)
                        mma_bf16(tm + tA, desc_k(s1, 128, kk), desc_mn(s2, 128, kk), idesc_bf16(128, M, true), kk > 0);
                    mma_commit(&bar);
                }
                ok = ctl.wait();
            }
            if (ok) {
                float sint[HM], lin[HM], L[HM];
                tmem_ld(tl + tO + cr * M + h * HM, sint, HM);
                tmem_ld(tl + tA + h * HM, lin, HM);
                float mx = -INFINITY;
#pragma unroll
                for (int jj = 0; jj < HM; jj++) {
                    L[jj] = row_ok ? sig2 * (fexp(b[jj]) * sint[jj] + fexp(b[jj] - rho[jj]) * lin[jj]) : -INFINITY;
                    mx = fmaxf(mx, L[jj]);
                }
                redm[h * 128 + r] = mx;
                named_sync(1, kTcThreads);
                m = fmaxf(redm[r], redm[128 + r]);
                float ps = 0.0f, pe[HM], pq[HM], z[HM];
#pragma unroll
                for (int jj = 0; jj < HM; jj++) {
                    const float p = (m == -INFINITY) ? 0.0f : ex2(L[jj] - m);
                    ps += p;
                    pe[jj] = p * fexp(b[jj]);
                    pq[jj] = p * fexp(b[jj] - rho[jj]);
                    z[jj] = 0.0f;
                }
                reds[h * 128 + r] = ps;
                // A_inter [128][2M]: this row's chunk block holds p o Eb, the other block zero
                store_row(KB[0], r, cr * M + h * HM, pe, HM);
                store_row(KB[0], r, (1 - cr) * M + h * HM, z, HM);
                store_row(VB[1] + 16384, r, h * HM, pq, HM);  // pEq, after Ek
                named_sync(1, kTcThreads);
                l = reds[r] + reds[128 + r];
                // the last stage (log_alpha rows, scratch) is free: the producer loads window block 0
                __syncwarp();
                if (lane == 0) mbar_arrive(&s2free);
                sync_for_mma<true>();
                if (tid == 0) {
                    if (!mbar_wait(&sbar, 1, kWaitCycles)) *abort = 1;  // the [S^V] pair
                    fence_after_sync();
                    const uint32_t s1 = smem_u32(KB[0]), s2 = smem_u32(VB[1]), s3 = smem_u32(KB[1]);
                    for (int kk = 0; kk < 2 * M / 16; kk++)
                        mma_bf16(tm + tO, desc_k(s1, 128, kk), desc_mn(s3, 2 * M, kk), idesc_bf16(128, D, true), kk > 0);
                    for (int kk = 0; kk < M / 16; kk++)
                        mma_bf16(tm + tA, desc_k(s2 + 16384, 128, kk), desc_k(s2, 128, kk), idesc_bf16(128, 128, false),
                                 kk > 0);
                    mma_commit(&bar);
                }
                ok = ctl.wait();
            }
            if (ok) {
                mask_to_tile(tl + tA, KB[0], r, h, cr, row_ok, false);
                sync_for_mma<true>();
                if (tid == 0) {
                    const uint32_t s1 = smem_u32(KB[0]), s2 = smem_u32(VB[0]);
                    for (int kk = 0; kk < 8; kk++)
                        mma_bf16(tm + tO, desc_k(s1, 128, kk), desc_mn(s2, 128, kk), idesc_bf16(128, D, true), 1);
                    mma_commit(&bar);
                }
                ok = ctl.wait();
                o_valid = true;
            }
        }

        if (h == 1) {  // the slot branch belongs to half 0's softmax state
            m = -INFINITY;
            l = 0.0f;
        }
        if (!ok && tid == 0) *abort = 1;  // slot phase gave up: the producer stands down
        fence_before_sync();
        asm volatile("bar.arrive 2, %0;\n" ::"n"(kFwdThreads) : "memory");  // stages free for the producer

        // ---- window branch: 128-key blocks of the band [tbase - w + 1, tbase + nq - 1]
        const int t = tbase + r;
        for (int i = 0; i < nb && ok; i++) {
            const int kb = klo + i * 128, nk = min(128, khi - kb + 1), b = i & 1, stg = stage_of(i);
            if (!(ok = mbar_wait_ab(&sfull[b], (i >> 1) & 1, kWaitCycles, abort))) break;
            fence_after_sync();
            float sv[64];
            tmem_ld(tl + 128 * b + 64 * h, sv, 64);
            float bm = -INFINITY;
            // valid keys of this row: columns [clo, chi] of the block
            const int clo = max(0, t - sh.w + 1 - kb) - 64 * h;
            const int chi = (row_ok ? min(nk - 1, t - kb) : -1) - 64 * h;
            const bool full = clo <= 0 && chi >= 63;  // the whole half-row is in the band
            if (full) {
                // raw scores: max first (sig2 > 0 keeps the order), scaled in the exponent below
                float m0 = sv[0], m1 = sv[1], m2 = sv[2], m3 = sv[3];
#pragma unroll
                for (int jj = 4; jj < 64; jj += 4) {
                    m0 = fmaxf(m0, sv[jj]);
                    m1 = fmaxf(m1, sv[jj + 1]);
                    m2 = fmaxf(m2, sv[jj + 2]);
                    m3 = fmaxf(m3, sv[jj + 3]);
                }
                bm = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)) * sig2;
            } else {
#pragma unroll
                for (int jj = 0; jj < 64; jj++) {
                    sv[jj] = (jj >= clo && jj <= chi) ? sv[jj] * sig2 : -INFINITY;
                    bm = fmaxf(bm, sv[jj]);
                }
            }
            // P V of block i - 1 done: its accumulator may be rescaled below
            if (i >= 1 && !(ok = mbar_wait_ab(&bdone[(i - 1) & 1], ((i - 1) >> 1) & 1, kWaitCycles, abort))) break;
            const bool acc_live = h == 0 ? (o_valid || i > 0) : i > 0;  // this half's O holds data
            const float mnew = fmaxf(m, bm);
            bool resc = false;
            float scale = 1.0f;
            if (!acc_live || m == -INFINITY) {
                m = mnew;
            } else if (mnew > m + 8.0f) {
                resc = true;
                scale = ex2(m - mnew);
                m = mnew;
                l *= scale;
            }
            if (__any_sync(0xffffffffu, resc)) {
                const uint32_t to = tl + (h == 0 ? tO : tO1);
                for (int c0 = 0; c0 < D; c0 += 32) {
                    float ov[32];
                    tmem_ld32(to + c0, ov);
#pragma unroll
                    for (int jj = 0; jj < 32; jj++) ov[jj] *= scale;
                    tmem_st32(to + c0, ov);
                }
            }
            float ps = 0.0f;
            if (full) {  // m is finite here: the half-row has at least one key
                const float2 sg2 = make_float2(sig2, sig2), nm2 = make_float2(-m, -m);
                float2 a0 = make_float2(0.0f, 0.0f), a1 = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int jj = 0; jj < 64; jj += 4) {
                    const float2 s0 = __ffma2_rn(make_float2(sv[jj], sv[jj + 1]), sg2, nm2);
                    const float2 s1 = __ffma2_rn(make_float2(sv[jj + 2], sv[jj + 3]), sg2, nm2);
                    const float2 p0 = make_float2(ex2(s0.x), ex2(s0.y)), p1 = make_float2(ex2(s1.x), ex2(s1.y));
                    a0 = __fadd2_rn(a0, p0);
                    a1 = __fadd2_rn(a1, p1);
                    sv[jj] = p0.x; sv[jj + 1] = p0.y; sv[jj + 2] = p1.x; sv[jj + 3] = p1.y;
                }
                ps = (a0.x + a0.y) + (a1.x + a1.y);
            } else {
#pragma unroll
                for (int jj = 0; jj < 64; jj++) {
                    const float p = (m == -INFINITY) ? 0.0f : ex2(sv[jj] - m);
                    sv[jj] = p;
                    ps += p;
                }
            }
            l += ps;
            store_row(KB[stg], r, 64 * h, sv, 64);  // P over the consumed K~ block
            fence_async_smem();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&pready);
        }
        if (ok && nb > 0) ok = mbar_wait_ab(&bdone[(nb - 1) & 1], ((nb - 1) >> 1) & 1, kWaitCycles, abort);

        // ---- epilogue: merge the halves, o = (f0 O_0 + f1 O_1) / l, lse = m ln2 + log l
        redm[h * 128 + r] = m;
        reds[h * 128 + r] = l;
        if (named_sync_or(1, kTcThreads, !ok)) ok = false;
        const float m0 = redm[r], m1 = redm[128 + r];
        const float mm = fmaxf(m0, m1);
        const float f0 = m0 == -INFINITY ? 0.0f : ex2(m0 - mm), f1 = m1 == -INFINITY ? 0.0f : ex2(m1 - mm);
        const float lt = reds[r] * f0 + reds[128 + r] * f1;
        const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
        const bool o0 = o_valid || nb > 0, o1 = nb > 0;
        unsigned char* stg = KB[0];
        if (ok) {
            fence_after_sync();
            for (int c0 = 0; c0 < HD; c0 += 32) {
                float u0[32], u1[32];
                if (o0 && o1) {
                    tmem_ld32x2(tl + tO + h * HD + c0, tl + tO1 + h * HD + c0, u0, u1);
                } else {
                    if (o0) tmem_ld32(tl + tO + h * HD + c0, u0);
#pragma unroll
                    for (int jj = 0; jj < 32; jj++) {
                        if (!o0) u0[jj] = 0.0f;
                        u1[jj] = 0.0f;
                    }
                }
#pragma unroll
                for (int jj = 0; jj < 32; jj++) u0[jj] = (u0[jj] * f0 + u1[jj] * f1) * inv;
                store_row(stg, r, h * HD + c0, u0, 32);
            }
        }
        const int bad = named_sync_or(1, kTcThreads, !ok);
        if (!bad) {  // rows [0, nq) of the tile, 16-byte chunks, coalesced
            constexpr int CH = D / 8;
            __nv_bfloat16* ob = (__nv_bfloat16*)a.o + (hoff + tbase) * D;
            for (int e = tid; e < nq * CH; e += kTcThreads) {
                const int rr = e / CH, ch = e % CH;
                *reinterpret_cast<uint4*>(ob + (size_t)rr * D + ch * 8) =
                    *reinterpret_cast<const uint4*>(stg + sw_chunk(rr, ch, 128));
            }
            if (h == 0 && row_ok) a.lse[hoff + t] = mm * kLn2 + logf(lt);
        } else if (h == 0 && row_ok) {
            a.lse[hoff + t] = __int_as_float(0x7fc00000);  // NaN marks the failed tile
        }
    }
    fence_before_sync();
    __syncthreads();
    if (s_abort) {  // let the copies and MMAs in flight land before the TMEM and the CTA go
        if (tid == 0) {  // slot-branch MMAs and log_alpha copy (issued by this thread)
            mma_commit(&drain[0]);
            mbar_wait(&drain[0], 0, kWaitCycles);
            if (slot) mbar_wait(&gbar, 0, kWaitCycles);
        }
        if (warp == 8 && lane == 0) {  // its MMAs, the slot operand copies (sbar phases 0, 1), window copies
            mma_commit(&drain[1]);
            mbar_wait(&drain[1], 0, kWaitCycles);
            if (slot) mbar_wait(&sbar, s_sv_issued ? 1u : 0u, kWaitCycles);  // phase 1 completes after phase 0
            if (nb > 0) mbar_wait(&qbar, 0, kWaitCycles);
            for (int q = 0; q < NS; q++)
                if (last_ph[q] >= 0) mbar_wait(&full[q], (uint32_t)last_ph[q], kWaitCycles);
        }
        __syncthreads();
        if (tid == 0) atomicOr(status, kStatusTimeoutBit);
    }
    if (warp == 0) tmem_dealloc(tm, 512);
}

// RoPE applied once per call: qr = RoPE(q), kr = RoPE(k) at absolute positions.
// RoPE(q), RoPE(k) in bf16.  Thread = (position t, 8 frequency pairs, 4
// heads): the (cos, sin) pairs are formed once, with the exact reduction of
// rope_cs, and serve the four heads; with tab != nullptr the threads of the
// first head group also write them to the (cos, sin) table [T][D/2].
template <int D>
__global__ void __launch_bounds__(256)
rope_qk_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
               __nv_bfloat16* __restrict__ qr, __nv_bfloat16* __restrict__ kr, float2* __restrict__ tab,
               const RopeTab rt, int BH, int T) {
    constexpr int H = D / 2, CHH = D / 16;
    const long e = (long)blockIdx.x * 256 + threadIdx.x;
    const int HG = (BH + 3) / 4;
    if (e >= (long)T * CHH * HG) return;
    const int ch = (int)(e % CHH);
    const long rest = e / CHH;
    const int t = (int)(rest % T), hg = (int)(rest / T);
    float4 c[4];
#pragma unroll
    for (int p = 0; p < 4; p++) {
        float c0, s0, c1, s1;
        rope_cs(rt, t, ch * 8 + 2 * p, c0, s0);
        rope_cs(rt, t, ch * 8 + 2 * p + 1, c1, s1);
        c[p] = make_float4(c0, s0, c1, s1);
    }
    if (tab != nullptr && hg == 0) {
        float4* tp = reinterpret_cast<float4*>(tab + (size_t)t * H + ch * 8);
#pragma unroll
        for (int p = 0; p < 4; p++) tp[p] = c[p];
    }
    uint4 in[4][2][2];  // [head][q / k][half]: every load issued before any store
#pragma unroll
    for (int hh = 0; hh < 4; hh++) {
        const int bh = hg * 4 + hh;
        const size_t row = (size_t)(bh < BH ? bh : 0) * T + t;
#pragma unroll
        for (int which = 0; which < 2; which++) {
            const __nv_bfloat16* src = (which == 0 ? q : k) + row * D + ch * 8;
            in[hh][which][0] = __ldg(reinterpret_cast<const uint4*>(src));
            in[hh][which][1] = __ldg(reinterpret_cast<const uint4*>(src + H));
        }
    }
#pragma unroll
    for (int hh = 0; hh < 4; hh++) {
        const int bh = hg * 4 + hh;
        if (bh >= BH) break;
        const size_t row = (size_t)bh * T + t;
#pragma unroll
        for (int which = 0; which < 2; which++) {
            float x[8], y[8];
            unpack8(in[hh][which][0], x);
            unpack8(in[hh][which][1], y);
            rotate8v(x, y, c);
            __nv_bfloat16* dst = (which == 0 ? qr : kr) + row * D + ch * 8;
            *reinterpret_cast<uint4*>(dst) = pack8(x);
            *reinterpret_cast<uint4*>(dst + H) = pack8(y);
        }
    }
}

template <int D>
cudaError_t launch_rope_qk(const void* q, const void* k, __nv_bfloat16* qr, __nv_bfloat16* kr, float2* tab,
                           const RopeTab& rt, const Shape& sh, cudaStream_t st) {
    const long n = (long)sh.T * (D / 16) * ((sh.BH + 3) / 4);
    if (n == 0) return cudaSuccess;
    NHA_LAUNCH("rope_qk", st,
               rope_qk_kernel<D><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(
                   (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, qr, kr, tab, rt, sh.BH, sh.T));
    return cudaGetLastError();
}
template cudaError_t launch_rope_qk<64>(const void*, const void*, __nv_bfloat16*, __nv_bfloat16*, float2*,
                                        const RopeTab&, const Shape&, cudaStream_t);
template cudaError_t launch_rope_qk<128>(const void*, const void*, __nv_bfloat16*, __nv_bfloat16*, float2*,
                                         const RopeTab&, const Shape&, cudaStream_t);

template <int D, int M>
size_t tc_fwd_smem() {
    return 1024 + 128 * D * 2 + kFwdStages * 65536;
}

template <int D, int M>
cudaError_t tc_forward(const FwdArgs& a, float2* tab, __nv_bfloat16* qr, __nv_bfloat16* kr, int* status,
                       cudaStream_t st) {
    const Shape& sh = a.sh;
    Fork* f = nullptr;
    cudaError_t e = get_fork(&f);
    if (e != cudaSuccess) return e;
    // RoPE(q), RoPE(k) on the side stream while the chunk states are formed;
    // the (cos, sin) table too, for a backward that reuses this workspace
    if (sh.w > 0) {
        if ((e = fork_side(st, *f, 0)) != cudaSuccess) return e;
        if ((e = launch_rope_qk<D>(a.q, a.k, qr, kr, tab, a.rope, sh, f->side)) != cudaSuccess) return e;
    }
    e = tc_states<D, M>((const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v, a.la, a.SK, a.SV, a.SKb, a.SVb, a.G,
                        false, a.io, sh, status, st);
    if (e != cudaSuccess) return e;
    if (sh.w > 0 && (e = join_side(st, *f, 1)) != cudaSuccess) return e;
    const int W0 = sh.T - sh.R;
    // with per-head windows a head has at most ceil(T / 128) + 1 tiles
    const int tiles = varied(sh) ? (sh.T + 127) / 128 + 1 : (W0 + 127) / 128 + (sh.R + 127) / 128;
    if (tiles == 0) return cudaSuccess;
    FwdMaps maps;
    if ((e = tmap_rows_bf16(&maps.q, qr, D, sh.T, sh.BH, 128)) != cudaSuccess ||
        (e = tmap_rows_bf16(&maps.k, kr, D, sh.T, sh.BH, 128)) != cudaSuccess ||
        (e = tmap_rows_bf16(&maps.v, a.v, D, sh.T, sh.BH, 128)) != cudaSuccess ||
        (e = tmap_rows_f32(&maps.la, a.la, M, sh.T, sh.BH)) != cudaSuccess ||
        (e = tmap_rows_bf16(&maps.qs, a.q, D, sh.T, sh.BH, 128)) != cudaSuccess ||
        (e = tmap_rows_bf16(&maps.ks, a.k, D, sh.T, sh.BH, 128)) != cudaSuccess ||
        (e = tmap_rows_bf16(&maps.sk, a.SKb, D, (sh.NCS > 0 ? sh.NCS : 1) * M, sh.BH, 2 * M)) != cudaSuccess ||
        (e = tmap_rows_bf16(&maps.sv, a.SVb, D, (sh.NCS > 0 ? sh.NCS : 1) * M, sh.BH, 2 * M)) != cudaSuccess)
        return e;
    const size_t sm = tc_fwd_smem<D, M>();
    auto kern = fwd_tc_kernel<D, M>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    NHA_LAUNCH("fwd_tc", st, kern<<<dim3(tiles, sh.BH), kFwdThreads, sm, st>>>(a, maps, status));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_h0_fwd_lead<__nv_bfloat16, D, M>(a, st);  // queries t < w reading initial states
}

#define NHA_TC_INST(D, M) \
    template cudaError_t tc_forward<D, M>(const FwdArgs&, float2*, __nv_bfloat16*, __nv_bfloat16*, int*, cudaStream_t);
NHA_TC_INST(64, 16)
NHA_TC_INST(64, 32)
NHA_TC_INST(64, 64)
NHA_TC_INST(128, 16)
NHA_TC_INST(128, 32)
NHA_TC_INST(128, 64)

}  // namespace nha
