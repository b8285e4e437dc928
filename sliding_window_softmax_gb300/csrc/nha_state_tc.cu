// Slot states at chunk boundaries for the bf16 path.
//
// Per chunk c (C = 64 state indices) the contribution to the state at the
// chunk's end is dS_c = U_c^T X_c with U_c[s][i] = exp(G_i - b_{s,i}) u_{s,i}
// ("Native Hybrid Attention for Efficient Sequence Modeling", Paper-Notes page,
// 关键设计/层内混合: K^long_t = Diag(alpha_t) K^long_{t-1} + (1 - alpha_t) (x) k_t,
// unrolled over one chunk), for X = K and X = V, and the states entering the
// chunks follow S_prev(c + 1) = exp(G_c) S_prev(c) + dS_c.
//
// One kernel, state_scan: one CTA per (head, K or V) walks the chunks in
// order.  A copy warp streams X_c and the chunk's log_alpha rows through
// shared-memory stages; eight gate warps form U_c (bf16, 64 columns, slots
// past m zero) and exp(G_c) from the log_alpha rows (the array named G holds
// exp(G_c) on this path: the scans use nothing else of it); one warp forms
// dS_c^T = X_c^T U_c on the tensor core into one of two TMEM buffers; four
// warps (thread = one column d of the state) carry the state in fp32
// registers and write S_prev(c).
#include "nha_common.cuh"
#include "nha_kernels.h"
#include "nha_prof.h"
#include "nha_tc.cuh"
#include "nha_tc_tiles.cuh"
#include "nha_tma.h"

namespace nha {

constexpr int kScanThreads = 448, kScanStages = 4;  // 4 state warps (0-3), 8 gate warps (4-11), MMA warp, copy warp

struct StateMaps {
    CUtensorMap x[2];  // K, V rows, box {64, 64}
};

// One CTA per (head, K or V) walks the chunks in order.  The copy warp
// streams chunk c's rows X_c (TMA) and its log_alpha rows (bulk copy) into a
// stage; the gate warps form the chunk coefficients from log_alpha (per slot:
// the chunk-local cumsum b, the total G, U[s][i] = exp(G_i - b_{s,i}) u_{s,i}
// with u = -expm1(log_alpha), written as the bf16 MMA operand) and exp(G);
// the MMA warp forms dS_c^T = X_c^T U_c on the tensor core into one of two
// TMEM buffers; the state warps (thread = one column d) carry the state in
// fp32 registers, S_prev(c + 1) = exp(G_c) S_prev(c) + dS_c, and write the
// bf16 state entering every chunk.
template <int D, int M>
__global__ void __launch_bounds__(kScanThreads, 1)
state_scan_tc_kernel(const __grid_constant__ StateMaps maps, const float* __restrict__ la, float* __restrict__ G,
                     float* __restrict__ SK, float* __restrict__ SV, __nv_bfloat16* __restrict__ SKb,
                     __nv_bfloat16* __restrict__ SVb, const StateIO io, Shape call, int want_f32,
                     int* __restrict__ status) {
    constexpr int NS = kScanStages;
    constexpr int NSL = M;
    constexpr int NPART = 256 / M, RPT = kChunk / NPART;  // gate threads per slot, rows per gate thread
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    // stage s: X_c [64 tokens][128 d] (d >= D zero), U_c [64 tokens][64], log_alpha [64][M], exp(G_c) [M]
    auto XT = [&](int st) { return base + st * 16384; };
    auto UT = [&](int st) { return base + NS * 16384 + st * 8192; };
    auto LA = [&](int st) { return reinterpret_cast<float*>(base + NS * 24576 + st * 16384); };
    auto GS = [&](int st) { return reinterpret_cast<float*>(base + NS * 40960 + st * 256); };
    __shared__ uint64_t full[NS], ufull[NS], empty[NS], sfull[2], tfree[2], pbar[2], drain;
    __shared__ float PT[2][NPART][M];  // the gate threads' row-part totals, by chunk parity
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, tz = blockIdx.y, i0 = 0;  // tz 0: K, 1: V
    const Shape sh = head_shape(call, bh);
    const int NC = sh.NC, NCS = sh.NCS;  // this head's chunks; chunks per head in the arrays
    volatile int* abort = &s_abort;
    if (tid == 0) {
        for (int q = 0; q < NS; q++) {
            mbar_init(&full[q], 1);
            mbar_init(&ufull[q], 8);
            mbar_init(&empty[q], 4);
        }
        for (int q = 0; q < 2; q++) {
            mbar_init(&sfull[q], 1);
            mbar_init(&tfree[q], 4);
            mbar_init(&pbar[q], 8);
        }
        mbar_init(&drain, 1);
        s_abort = 0;
        mbar_fence_init();
    }
    if (D < 128)  // the MMA spans 128 columns of d: the upper block stays zero
        for (int e = tid; e < NS * 512; e += kScanThreads)
            reinterpret_cast<uint4*>(XT(e / 512) + 8192)[e % 512] = make_uint4(0, 0, 0, 0);
    if (warp == 0) tmem_alloc(&s_tmem, 128);
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = s_tmem;

    int last_ph[NS];
#pragma unroll
    for (int q = 0; q < NS; q++) last_ph[q] = -1;
    auto rows_of = [&](int c) { return min(kChunk, sh.R - c * kChunk); };  // tokens of chunk c
    if (warp == 12) {
        // ---------------- MMA issuer (lane 0): once a chunk's coefficients are
        // formed and its TMEM buffer is read out ----------------
        if (lane == 0) {
            for (int c = 0; c < NC; c++) {
                const int st = c % NS;
                if (!mbar_wait_ab(&full[st], (c / NS) & 1, kWaitCycles, abort)) break;
                if (!mbar_wait_ab(&ufull[st], (c / NS) & 1, kWaitCycles, abort)) break;
                if (c >= 2 && !mbar_wait_ab(&tfree[c & 1], ((c - 2) >> 1) & 1, kWaitCycles, abort)) break;
                fence_after_sync();
                const uint32_t sx = smem_u32(XT(st)), su = smem_u32(UT(st));
                for (int kk = 0; kk < 4; kk++)
                    mma_bf16(tm + 64 * (c & 1), desc_mn(sx, 64, kk), desc_mn(su, 64, kk),
                             idesc_bf16(128, NSL, true) | (1u << 15), kk > 0);
                mma_commit(&sfull[c & 1]);
            }
        }
    } else if (warp == 13) {
        // ---------------- loader (lane 0): refills a stage once its chunk is consumed ----------------
        if (lane == 0) {
            auto load = [&](int c) {
                const int st = c % NS, nr = rows_of(c);
                mbar_arrive_expect_tx(&full[st], (D / 64) * 8192 + (uint32_t)(nr * M * 4));
#pragma unroll
                for (int x = 0; x < D; x += 64) tma_load_3d(XT(st) + x * 128, &maps.x[tz], x, c * kChunk, bh, &full[st]);
                bulk_load(LA(st), la + ((size_t)bh * sh.TS + (size_t)c * kChunk) * M, (uint32_t)(nr * M * 4), &full[st]);
                last_ph[st] = (c / NS) & 1;
            };
            for (int c = 0; c < min(NS, NC); c++) load(c);
            for (int c = NS; c < NC; c++) {
                if (!mbar_wait_ab(&empty[(c - NS) % NS], ((c - NS) / NS) & 1, kWaitCycles, abort)) break;
                load(c);
            }
        }
    } else if (warp >= 4) {
        // ---------------- gate warps: thread = (slot, RPT consecutive rows) ----------------
        // A warp reads consecutive slots of a row (no shared-memory bank
        // conflicts).  Each thread sums its rows; the NPART parts of a slot lie
        // in different warps and exchange their totals through shared memory
        // and the pbar barrier (bounded wait, double-buffered by chunk parity).
        // With E_s = exp(G - b_s) (E_{-1} = exp(G)), U[s] = E_s u_s = E_s - E_{s-1}:
        // one exp per element, and rows past the chunk's tokens (log_alpha 0)
        // give U = 0 by themselves.
        const int g = tid - 128, slot = g % M, part = g / M, r0 = part * RPT;
        for (int c = 0; c < NC; c++) {
            const int st = c % NS, nr = rows_of(c), pb = c & 1;
            if (!mbar_wait_ab(&full[st], (c / NS) & 1, kWaitCycles, abort)) break;
            const float* lr = LA(st);
            float b[RPT], acc = 0.0f;
#pragma unroll
            for (int r = 0; r < RPT; r++) {
                acc += (r0 + r < nr) ? lr[(r0 + r) * M + slot] : 0.0f;
                b[r] = acc;
            }
            PT[pb][part][slot] = acc;
            __syncwarp();
            if (lane == 0) mbar_arrive(&pbar[pb]);
            if (!mbar_wait_ab(&pbar[pb], (c >> 1) & 1, kWaitCycles, abort)) break;
            float off = 0.0f, Gt = 0.0f;  // parts before this one; the chunk total
#pragma unroll
            for (int p2 = 0; p2 < NPART; p2++) {
                const float t = PT[pb][p2][slot];
                if (p2 < part) off += t;
                Gt += t;
            }
            float ep = fexp(Gt - off);  // E of the row before this part's first row
            unsigned char* ut = UT(st);
#pragma unroll
            for (int r = 0; r < RPT; r++) {
                const float e = fexp(Gt - (b[r] + off));
                *reinterpret_cast<__nv_bfloat16*>(ut + sw_off(r0 + r, slot, 64)) = __float2bfloat16_rn(e - ep);
                ep = e;
            }
            if (part == 0) {  // E_{-1} = exp(G): the chunk's decay
                const float eg = fexp(Gt);
                GS(st)[slot] = eg;
                if (tz == 0) G[((size_t)bh * NCS + c) * M + slot] = eg;  // for the backward's adjoint scan
                if (Gt < kGateRange) atomicOr(status, kStatusGateRangeBit);
            }
            fence_async_smem();  // U is an MMA operand: generic writes -> async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(&ufull[st]);
        }
    } else {
        // ---------------- state warps: thread = column d ----------------
        const int d = tid;
        const uint32_t tl = tm + ((uint32_t)(warp * 32) << 16);
        __nv_bfloat16* Sb = (tz == 0 ? SKb : SVb) + (size_t)bh * NCS * M * D + (size_t)i0 * D + d;
        float* Sf = (tz == 0 ? SK : SV) + (size_t)bh * NCS * M * D + (size_t)i0 * D + d;
        float S[NSL];  // the state entering chunk c: h0 (or zero) before chunk 0
        {
            const float* h0 = tz == 0 ? io.h0k : io.h0v;
#pragma unroll
            for (int i = 0; i < NSL; i++) S[i] = (h0 != nullptr && d < D) ? h0[((size_t)bh * M + i) * D + d] : 0.0f;
        }
        bool done = true;
        for (int c = 0; c < NC; c++) {
            const int st = c % NS, b = c & 1;
            if (!mbar_wait_ab(&sfull[b], (c >> 1) & 1, kWaitCycles, abort) ||
                !mbar_wait_ab(&ufull[st], (c / NS) & 1, kWaitCycles, abort)) {
                done = false;
                break;
            }
            fence_after_sync();
            {
                // bf16 copies: lanes d, d ^ 1 swap one value so that each stores a
                // packed pair (columns d & ~1, d | 1) of slot i (even lane) or i + 1 (odd)
                const size_t o = (size_t)c * M * D;
                const bool odd = lane & 1;
#pragma unroll
                for (int i = 0; i < NSL; i += 2) {
                    const float recv = __shfl_xor_sync(0xffffffffu, odd ? S[i] : S[i + 1], 1);
                    const uint32_t pk = odd ? pack_bf16(recv, S[i + 1]) : pack_bf16(S[i], recv);
                    if (d < D)
                        *reinterpret_cast<uint32_t*>(Sb + o + (size_t)(i + (odd ? 1 : 0)) * D - (odd ? 1 : 0)) = pk;
                }
                if (want_f32 && d < D)
#pragma unroll
                    for (int i = 0; i < NSL; i++) Sf[o + (size_t)i * D] = S[i];
            }
            // S_prev(c + 1) = exp(G_c) S_prev(c) + dS_c, dS_c read from TMEM in
            // groups of at most 32 columns (fewer registers live at once)
            const float4* g4 = reinterpret_cast<const float4*>(GS(st) + i0);  // exp(G_c)
            constexpr int GRP = NSL < 32 ? NSL : 32;
#pragma unroll
            for (int h = 0; h < NSL; h += GRP) {
                float dS[GRP];
                tmem_ld(tl + 64 * b + h, dS, GRP);
#pragma unroll
                for (int i = 0; i < GRP; i += 4) {
                    const float4 gv = g4[(h + i) / 4];
                    S[h + i] = gv.x * S[h + i] + dS[i];
                    S[h + i + 1] = gv.y * S[h + i + 1] + dS[i + 1];
                    S[h + i + 2] = gv.z * S[h + i + 2] + dS[i + 2];
                    S[h + i + 3] = gv.w * S[h + i + 3] + dS[i + 3];
                }
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&tfree[b]);
                mbar_arrive(&empty[st]);
            }
        }
        // the final state (after the last chunk): fp32 for the caller, bf16 for
        // the backward's carry of the last chunk; NaN if the scan gave up
        if (d < D) {
            float* hT = tz == 0 ? io.hTk : io.hTv;
#pragma unroll
            for (int i = 0; i < NSL; i++) {
                const float val = done ? S[i] : __int_as_float(0x7fc00000);
                if (hT != nullptr) hT[((size_t)bh * M + i) * D + d] = val;
                if (io.htb != nullptr) io.htb[(((size_t)bh * 2 + tz) * M + i) * D + d] = __float2bfloat16_rn(val);
            }
            // with per-head windows the arrays hold more chunks than this head
            // has: the consumers read states in pairs (c, c + 1), so the chunk
            // after the last one must hold zeros, not stale memory
            if (NC < NCS)
#pragma unroll
                for (int i = 0; i < NSL; i++) Sb[(size_t)NC * M * D + (size_t)i * D] = __float2bfloat16_rn(0.0f);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (s_abort) {  // let the copies and MMAs in flight land before the TMEM and the CTA go
        if (warp == 12 && lane == 0) {
            mma_commit(&drain);
            mbar_wait(&drain, 0, kWaitCycles);
        }
        if (warp == 13 && lane == 0)
            for (int q = 0; q < NS; q++)
                if (last_ph[q] >= 0) mbar_wait(&full[q], (uint32_t)last_ph[q], kWaitCycles);
        __syncthreads();
        if (tid == 0) atomicOr(status, kStatusTimeoutBit);
    }
    if (warp == 0) tmem_dealloc(tm, 128);
}

constexpr int kAdjDepth = 7, kAdjWarps = 2;

// Reverse chunk scan of the slot adjoints, fused with the dlog_alpha carry.
// R_c, the adjoint carried into chunk c from the later chunks, follows
// R_{c - 1} = exp(G_c) R_c + dR_c (dR_c: the chunk's own contribution, from the
// query-side kernel in bf16; the sum is carried in fp32); it is written in
// bf16 for the key-side kernel.  The carry
// of chunk c, sum_d R_c[i][d] S_prev(c + 1)[i][d] over K and V (the bf16
// states; for the last chunk the final state, present only with its
// gradient), is the total over all later rows of the gate gradient that every
// row of chunk c receives; it is added to db1 of the chunk's last state row,
// whose in-chunk suffix sum in the key-side kernel hands it to every row.
//
// One warp per (head, slot): lane l holds elements d in [PL l, PL l + PL) of
// the K and the V adjoint, so the carry is a warp sum and no barrier is
// needed.  Each lane streams its own pieces of the next kAdjDepth chunks
// (contributions, states, the decay and the db1 entry) into its own shared
// memory stages with cp.async; a CTA of two warps needs about 15 KB and 64
// threads, so two fit beside a key-major window CTA (d = 128) on one SM and
// the scan runs in that kernel's shadow on the side stream.
template <int D>
struct AdjStage {
    static constexpr int PL = D / 32;
    __nv_bfloat16 xk[32 * PL], xv[32 * PL];    // dR_c, K and V
    __nv_bfloat16 sk[32 * PL], sv[32 * PL];    // S_prev(c + 1), K and V
    float g, db;                               // exp(G_c) of the slot, db1 entry of the chunk's last row
    float pad[2];
};

template <int D>
__global__ void __launch_bounds__(32 * kAdjWarps)
adj_scan_kernel(const __nv_bfloat16* __restrict__ RK, const __nv_bfloat16* __restrict__ RV,
                const __nv_bfloat16* __restrict__ SK,
                const __nv_bfloat16* __restrict__ SV, const float* __restrict__ G, __nv_bfloat16* __restrict__ RKb,
                __nv_bfloat16* __restrict__ RVb, float* __restrict__ db1, const float* __restrict__ dhTk,
                const float* __restrict__ dhTv, const __nv_bfloat16* __restrict__ htb, float* __restrict__ rend,
                Shape call, int M) {
    constexpr int PL = D / 32, NP = kAdjDepth;
    using Stage = AdjStage<D>;
    extern __shared__ __align__(16) unsigned char adj_smem[];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const long wid = (long)blockIdx.x * kAdjWarps + wib;
    if (wid >= (long)call.BH * M) return;  // whole warp
    const int bh = (int)(wid / M), i = (int)(wid % M);
    Stage* stages = reinterpret_cast<Stage*>(adj_smem) + (size_t)wib * NP;
    const Shape sh = head_shape(call, bh);
    const int NC = sh.NC, NCS = sh.NCS;  // this head's chunks; chunks per head in the arrays
    const bool has_dhT = dhTk != nullptr;
    const int e0 = lane * PL;
    auto row = [&](int c) { return (((size_t)bh * NCS + c) * M + i) * D + e0; };  // [BH][NCS][M][D]
    auto db_at = [&](int c) {
        const int last = min(c * kChunk + kChunk, sh.R) - 1;
        return ((size_t)bh * NCS * kChunk + last) * M + i;
    };
    // one commit group per chunk and lane (empty past the first chunk)
    auto issue = [&](int c) {
        if (c >= 0) {
            Stage& st = stages[c % NP];
            const size_t o = row(c);
            const __nv_bfloat16 *sk, *sv;
            bool sval = true;
            if (c + 1 < NC) {
                sk = SK + row(c + 1);
                sv = SV + row(c + 1);
            } else {  // the final state (bf16 copy), with its gradient only
                sk = htb + (((size_t)bh * 2 + 0) * M + i) * D + e0;
                sv = htb + (((size_t)bh * 2 + 1) * M + i) * D + e0;
                sval = has_dhT;
            }
            if constexpr (PL == 4) {
                cp_async8(st.xk + e0, RK + o, true);
                cp_async8(st.xv + e0, RV + o, true);
                cp_async8(st.sk + e0, sk, sval);
                cp_async8(st.sv + e0, sv, sval);
            } else {
                cp_async4(st.xk + e0, RK + o, true);
                cp_async4(st.xv + e0, RV + o, true);
                cp_async4(st.sk + e0, sk, sval);
                cp_async4(st.sv + e0, sv, sval);
            }
            if (lane == 0) {
                cp_async4(&st.g, G + ((size_t)bh * NCS + c) * M + i, true);
                cp_async4(&st.db, db1 + db_at(c), true);
            }
        }
        cp_async_commit();
    };
    // R enters the last chunk as the gradient of the final state (zero without one)
    float rk[PL], rv[PL];
#pragma unroll
    for (int e = 0; e < PL; e++) {
        rk[e] = has_dhT ? dhTk[((size_t)bh * M + i) * D + e0 + e] : 0.0f;
        rv[e] = has_dhT ? dhTv[((size_t)bh * M + i) * D + e0 + e] : 0.0f;
    }
#pragma unroll
    for (int p = 0; p < NP; p++) issue(NC - 1 - p);
    for (int c = NC - 1; c >= 0; c--) {
        cp_async_wait<NP - 1>();  // this lane's pieces of chunk c
        const Stage& st = stages[c % NP];
        const size_t o = row(c);
        uint32_t pk[PL / 2], pv[PL / 2];
#pragma unroll
        for (int e = 0; e < PL; e += 2) {
            pk[e / 2] = pack_bf16(rk[e], rk[e + 1]);
            pv[e / 2] = pack_bf16(rv[e], rv[e + 1]);
        }
        if constexpr (PL == 4) {
            *reinterpret_cast<uint2*>(RKb + o) = make_uint2(pk[0], pk[1]);
            *reinterpret_cast<uint2*>(RVb + o) = make_uint2(pv[0], pv[1]);
        } else {
            *reinterpret_cast<uint32_t*>(RKb + o) = pk[0];
            *reinterpret_cast<uint32_t*>(RVb + o) = pv[0];
        }
        float t = 0.0f;
#pragma unroll
        for (int e = 0; e < PL; e++)
            t += rk[e] * __bfloat162float(st.sk[e0 + e]) + rv[e] * __bfloat162float(st.sv[e0 + e]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        const float g = __shfl_sync(0xffffffffu, lane == 0 ? st.g : 0.0f, 0);  // exp(G_c), landed in lane 0's stage
        if (lane == 0 && (c + 1 < NC || has_dhT)) db1[db_at(c)] = st.db + t;
#pragma unroll
        for (int e = 0; e < PL; e++) {
            rk[e] = g * rk[e] + __bfloat162float(st.xk[e0 + e]);
            rv[e] = g * rv[e] + __bfloat162float(st.xv[e0 + e]);
        }
        issue(c - NP);  // into the stage just read (this lane's own pieces)
    }
    cp_async_wait<0>();
    if (rend != nullptr)  // the adjoint of the state before chunk 0 (part of dh0)
#pragma unroll
        for (int e = 0; e < PL; e++) {
            rend[(((size_t)bh * 2 + 0) * M + i) * D + e0 + e] = rk[e];
            rend[(((size_t)bh * 2 + 1) * M + i) * D + e0 + e] = rv[e];
        }
    // per-head windows and sequence lengths: zeros after this head's last
    // chunk (read as the pair's second half by the key-side kernel)
    if (NC < NCS)
#pragma unroll
        for (int e = 0; e < PL; e++) {
            RKb[row(NC) + e] = __float2bfloat16_rn(0.0f);
            RVb[row(NC) + e] = __float2bfloat16_rn(0.0f);
        }
}

cudaError_t launch_adj_scan(const BwdArgs& a, int M, int D, cudaStream_t st) {
    const Shape& sh = a.sh;
    if (sh.NCS == 0) return cudaSuccess;
    const long warps = (long)sh.BH * M;
    const unsigned grid = (unsigned)((warps + kAdjWarps - 1) / kAdjWarps);
    if (D == 128) {
        const size_t sm = sizeof(AdjStage<128>) * kAdjDepth * kAdjWarps;
        // all of the SM's memory as shared memory, the configuration of the
        // key-major kernel its CTAs run beside
        cudaError_t e = cudaFuncSetAttribute(adj_scan_kernel<128>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        NHA_LAUNCH("adj_scan", st,
                   adj_scan_kernel<128><<<grid, 32 * kAdjWarps, sm, st>>>(a.hRK, a.hRV, a.SKb, a.SVb, a.G, a.RKb, a.RVb,
                                                                          a.wsDB1, a.dhTk, a.dhTv, a.io.htb, a.rend,
                                                                          sh, M));
    } else {
        const size_t sm = sizeof(AdjStage<64>) * kAdjDepth * kAdjWarps;
        NHA_LAUNCH("adj_scan", st,
                   adj_scan_kernel<64><<<grid, 32 * kAdjWarps, sm, st>>>(a.hRK, a.hRV, a.SKb, a.SVb, a.G, a.RKb, a.RVb,
                                                                         a.wsDB1, a.dhTk, a.dhTv, a.io.htb, a.rend,
                                                                         sh, M));
    }
    return cudaGetLastError();
}

template <int D, int M>
cudaError_t tc_states(const __nv_bfloat16* k, const __nv_bfloat16* v, const float* la, float* SK, float* SV,
                      __nv_bfloat16* SKb, __nv_bfloat16* SVb, float* G, bool want_f32,
                      const StateIO& io, const Shape& sh, int* status, cudaStream_t st) {
    if (sh.NCS == 0) return launch_final_states_copy(io, sh.BH, M, D, st);
    StateMaps maps;
    cudaError_t e;
    if ((e = tmap_rows_bf16(&maps.x[0], k, D, sh.T, sh.BH, 64)) != cudaSuccess ||
        (e = tmap_rows_bf16(&maps.x[1], v, D, sh.T, sh.BH, 64)) != cudaSuccess)
        return e;
    const size_t sm = 1024 + kScanStages * (16384 + 8192 + 16384 + 256);
    auto kern = state_scan_tc_kernel<D, M>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) != cudaSuccess)
        return e;
    NHA_LAUNCH("state_scan", st,
               kern<<<dim3(sh.BH, 2), kScanThreads, sm, st>>>(maps, la, G, SK, SV, SKb, SVb, io, sh,
                                                              want_f32 ? 1 : 0, status));
    return cudaGetLastError();
}

#define NHA_ST_INST(D, M)                                                                              \
    template cudaError_t tc_states<D, M>(const __nv_bfloat16*, const __nv_bfloat16*, const float*, float*, \
                                         float*, __nv_bfloat16*, __nv_bfloat16*, float*, bool,                 \
                                         const StateIO&, const Shape&, int*, cudaStream_t);
NHA_ST_INST(64, 16)
NHA_ST_INST(64, 32)
NHA_ST_INST(64, 64)
NHA_ST_INST(128, 16)
NHA_ST_INST(128, 32)
NHA_ST_INST(128, 64)

}  // namespace nha
