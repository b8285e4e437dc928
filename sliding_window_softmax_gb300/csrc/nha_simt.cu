// SIMT (CUDA-core, fp32) kernels of the chunkwise NHA operator.
//
// These serve the fp32 element type and are the straightforward form of the
// algorithm that the tensor-core kernels follow.  The chunkwise form
// ("Native Hybrid Attention for Efficient Sequence Modeling", Paper-Notes
// page, section Chunkwise 并行计算): the state index space j = t - w is cut
// into chunks of C tokens; per chunk, linear-channel (slot) logits come from
// the state carried in from earlier chunks plus the intra-chunk term built
// from cumulative / reverse gate products, window logits come from the
// shifted band of keys, one softmax covers both, and the value readout sums a
// slot branch and a window branch.
//
// Forward launches: state_chunk -> state_scan -> fwd_main.
// Backward launches: state_chunk -> state_scan -> bwd_rowdot -> bwd_window_dq
//   -> bwd_window_dkdv -> bwd_slot_query -> state_scan (reverse) ->
//   bwd_slot_key -> bwd_dla_carry.
#include "nha_common.cuh"
#include "nha_kernels.h"
#include "nha_prof.h"

namespace nha {

constexpr int kThreads = 256;

// ---------------------------------------------------------------------------------------
// Per-chunk contributions to the slot states at the chunk's end:
//   dS^K_c[i] = sum_{s in chunk} exp(G_i - b_{s,i}) u_{s,i} k_s   (m x d), likewise V,
// and G_c = the chunk's total log gate.  Grid (NC, BH).
template <typename Tin, int D, int M>
__global__ void __launch_bounds__(kThreads)
state_chunk_kernel(const Tin* __restrict__ k, const Tin* __restrict__ v,
                   const float* __restrict__ la, float* __restrict__ SK, float* __restrict__ SV,
                   float* __restrict__ G, Shape call) {
    extern __shared__ float smem[];
    constexpr int LX = D + 1, LG = M + 1;
    float* sX = smem;                  // [C][LX]
    float* sCoef = sX + kChunk * LX;   // [C][LG]
    float* sU = sCoef + kChunk * LG;   // [C][LG]
    const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const Shape sh = head_shape(call, bh);
    if (c >= sh.NC) return;  // past this head's chunks (per-head windows)
    const int j0 = c * kChunk, nc = min(kChunk, sh.R - j0);
    const size_t row0 = (size_t)bh * sh.TS;
    if (tid < M) {
        const float* lr = la + (row0 + j0) * M;
        float b = 0.0f;
        for (int r = 0; r < nc; r++) {
            float l = lr[(size_t)r * M + tid];
            b += l;
            sCoef[r * LG + tid] = b;
            sU[r * LG + tid] = -expm1f(l);
        }
        for (int r = 0; r < kChunk; r++)
            sCoef[r * LG + tid] = (r < nc) ? expf(b - sCoef[r * LG + tid]) * sU[r * LG + tid] : 0.0f;
        G[((size_t)bh * sh.NCS + c) * M + tid] = b;
        if (b < kGateRange && sh.status != nullptr) atomicOr(sh.status, kStatusGateRangeBit);
    }
    for (int pass = 0; pass < 2; pass++) {
        const Tin* src = (pass == 0 ? k : v) + row0 * D;
        float* dst = (pass == 0 ? SK : SV) + ((size_t)bh * sh.NCS + c) * M * D;
        __syncthreads();
        load_rows<Tin, D>(src, j0, nc, sX, LX, nullptr);
        __syncthreads();
        for (int e = tid; e < M * D; e += kThreads) {
            const int i = e / D, col = e % D;
            float acc = 0.0f;
            for (int s = 0; s < nc; s++) acc += sCoef[s * LG + i] * sX[s * LX + col];
            dst[e] = acc;
        }
    }
}

// ---------------------------------------------------------------------------------------
// Exclusive scan over chunks, in place:
//   forward (dir > 0):  X[c] <- S_c,  S_{c+1} = exp(G_c) S_c + X[c],  S_0 = init (h0 or 0)
//   reverse (dir < 0):  X[c] <- S_c,  S_{c-1} = exp(G_c) S_c + X[c],  S_{NC-1} = init (dhT or 0)
// Forward gives the slot state before each chunk; reverse gives, per chunk,
// the adjoint carried in from all later chunks.  init0 / init1 ([BH, M, D] or
// NULL) seed the K / V scans; out0 / out1 ([BH, M, D] or NULL) and outw
// ([BH][2][M][D] or NULL) receive the value after the last step (the final
// state; the adjoint carried past chunk 0).  Grid (ceil(M*D/256), BH, 2).
__global__ void __launch_bounds__(kThreads)
state_scan_kernel(float* __restrict__ X0, float* __restrict__ X1, const float* __restrict__ G,
                  Shape call, int M, int D, int dir, const float* __restrict__ init0, const float* __restrict__ init1,
                  float* __restrict__ out0, float* __restrict__ out1, float* __restrict__ outw) {
    const int e = blockIdx.x * kThreads + threadIdx.x;
    if (e >= M * D) return;
    const int bh = blockIdx.y, i = e / D, z = blockIdx.z;
    const int NC = head_shape(call, bh).NC, NCS = call.NCS;  // this head's chunks; chunks per head in the arrays
    float* X = (z == 0) ? X0 : X1;
    const float* init = z == 0 ? init0 : init1;
    float S = init != nullptr ? init[(size_t)bh * M * D + e] : 0.0f;
    for (int n = 0; n < NC; n++) {
        const int c = dir > 0 ? n : NC - 1 - n;
        const size_t idx = ((size_t)bh * NCS + c) * M * D + e;
        float x = X[idx];
        X[idx] = S;
        S = expf(G[((size_t)bh * NCS + c) * M + i]) * S + x;
    }
    float* out = z == 0 ? out0 : out1;
    if (out != nullptr) out[(size_t)bh * M * D + e] = S;
    if (outw != nullptr) outw[((size_t)bh * 2 + z) * M * D + e] = S;
}

// ---------------------------------------------------------------------------------------
// Forward.  One CTA per (query tile, head).  Tiles 0..NL-1 hold queries
// t < w (window only); tile NL + c holds the queries t = j + w of state chunk
// c.  Thread (r, tq): query row r = tid / 4, columns tq + 4 * n.
template <typename Tin, int D, int M>
__global__ void __launch_bounds__(kThreads) fwd_main_kernel(const FwdArgs a) {
    extern __shared__ float smem[];
    constexpr int LX = D + 1, LP = kChunk + 1, LG = M + 1;
    constexpr int NCOL = D / 4, NSL = M / 4;
    float* sQ = smem;
    float* sX1 = sQ + kChunk * LX;
    float* sX2 = sX1 + kChunk * LX;
    float* sP = sX2 + kChunk * LX;
    float* sEq = sP + kChunk * LP;
    float* sEk = sEq + kChunk * LG;
    float* sL = sEk + kChunk * LG;
    float* sG = sL + kChunk * LG;
    float* sER = sG + M;
    const int tid = threadIdx.x, r = tid >> 2, tq = tid & 3;
    const int x = blockIdx.x, bh = blockIdx.y;
    const Shape sh = head_shape(a.sh, bh);
    if (x >= sh.NL + sh.NC) return;  // past this head's tiles (per-head windows)
    const bool slot = x >= sh.NL;
    int tbase, nq, c = 0, j0 = 0;
    if (!slot) {
        tbase = x * kChunk;
        nq = min(kChunk, min(sh.w, sh.T) - tbase);
    } else {
        c = x - sh.NL;
        j0 = c * kChunk;
        nq = min(kChunk, sh.R - j0);
        tbase = j0 + sh.w;
    }
    const size_t hoff = (size_t)bh * sh.TS;
    const Tin* q = (const Tin*)a.q + hoff * D;
    const Tin* k = (const Tin*)a.k + hoff * D;
    const Tin* v = (const Tin*)a.v + hoff * D;
    const float sig = sh.sigma;

    float acc[NCOL];
#pragma unroll
    for (int n = 0; n < NCOL; n++) acc[n] = 0.0f;
    float mrow = -INFINITY, lrow = 0.0f;

    load_rows<Tin, D>(q, tbase, nq, sQ, LX, nullptr);
    if (slot) {
        chunk_gates<M>(a.la + (hoff + j0) * M, nq, sEq, sEk, nullptr, LG, sG, sER);
        load_rows<Tin, D>(k, j0, nq, sX1, LX, nullptr);
        const float* SKp = a.SK + ((size_t)bh * sh.NCS + c) * M * D;
        for (int e = tid; e < M * D; e += kThreads) sX2[(e / D) * LX + e % D] = SKp[e];
        __syncthreads();
        // A[r][s] = q_{t(r)} . k_{j0+s}, causal s <= r (un-rotated)
#pragma unroll 1
        for (int n = 0; n < kChunk / 4; n++) {
            const int s = tq + 4 * n;
            float t = 0.0f;
            if (s <= r)
                for (int cc = 0; cc < D; cc++) t += sQ[r * LX + cc] * sX1[s * LX + cc];
            sP[r * LP + s] = t;
        }
        __syncthreads();
        // slot logits L = sigma (Eb o (Q S^K_prev^T) + Eq o (A Ek))
        float lv[NSL];
        float mx = -INFINITY;
        for (int n = 0; n < NSL; n++) {
            const int i = tq + 4 * n;
            float inter = 0.0f, intra = 0.0f;
            for (int cc = 0; cc < D; cc++) inter += sQ[r * LX + cc] * sX2[i * LX + cc];
            for (int s = 0; s <= r; s++) intra += sP[r * LP + s] * sEk[s * LG + i];
            const float eq = sEq[r * LG + i];
            lv[n] = (r < nq) ? sig * (eq * sER[i] * inter + eq * intra) : -INFINITY;
            mx = fmaxf(mx, lv[n]);
        }
        mx = warp_max4(mx);
        float sum = 0.0f;
        for (int n = 0; n < NSL; n++) {
            const int i = tq + 4 * n;
            const float p = exp_diff(lv[n], mx);
            sL[r * LG + i] = p;
            sum += p;
        }
        sum = warp_sum4(sum);
        mrow = mx;
        lrow = sum;
        __syncthreads();
        // Bm[r][s] = sum_i p[r][i] Eq[r][i] Ek[s][i], s <= r
        for (int n = 0; n < kChunk / 4; n++) {
            const int s = tq + 4 * n;
            float t = 0.0f;
            if (s <= r)
                for (int i = 0; i < M; i++) t += sL[r * LG + i] * sEq[r * LG + i] * sEk[s * LG + i];
            sP[r * LP + s] = t;
        }
        load_rows<Tin, D>(v, j0, nq, sX1, LX, nullptr);
        const float* SVp = a.SV + ((size_t)bh * sh.NCS + c) * M * D;
        for (int e = tid; e < M * D; e += kThreads) sX2[(e / D) * LX + e % D] = SVp[e];
        __syncthreads();
        for (int n = 0; n < NCOL; n++) {
            const int col = tq + 4 * n;
            float t = 0.0f;
            for (int i = 0; i < M; i++) t += sL[r * LG + i] * sEq[r * LG + i] * sER[i] * sX2[i * LX + col];
            for (int s = 0; s <= r; s++) t += sP[r * LP + s] * sX1[s * LX + col];
            acc[n] = t;
        }
        __syncthreads();
    }
    // rotate Q in place for the window branch
    __syncthreads();
    for (int e = tid; e < kChunk * (D / 2); e += kThreads) {
        const int rr = e / (D / 2), i = e % (D / 2);
        if (rr < nq) {
            float cs, sn;
            rope_cs(a.rope, tbase + rr, i, cs, sn);
            const float x0 = sQ[rr * LX + i], x1 = sQ[rr * LX + i + D / 2];
            sQ[rr * LX + i] = x0 * cs - x1 * sn;
            sQ[rr * LX + i + D / 2] = x1 * cs + x0 * sn;
        }
    }
    __syncthreads();
    if (sh.w > 0 && nq > 0) {
        const int klo = max(0, tbase - sh.w + 1), khi = tbase + nq - 1;
        const int t = tbase + r;
        for (int kb = klo; kb <= khi; kb += kChunk) {
            const int nk = min(kChunk, khi - kb + 1);
            load_rows<Tin, D>(k, kb, nk, sX1, LX, &a.rope);
            load_rows<Tin, D>(v, kb, nk, sX2, LX, nullptr);
            __syncthreads();
            float sv[kChunk / 4];
            float mx = -INFINITY;
            for (int n = 0; n < kChunk / 4; n++) {
                const int s = tq + 4 * n, key = kb + s;
                float val = -INFINITY;
                if (r < nq && s < nk && key <= t && key > t - sh.w) {
                    float dt = 0.0f;
                    for (int cc = 0; cc < D; cc++) dt += sQ[r * LX + cc] * sX1[s * LX + cc];
                    val = sig * dt;
                }
                sv[n] = val;
                mx = fmaxf(mx, val);
            }
            mx = warp_max4(mx);
            const float mnew = fmaxf(mrow, mx);
            const float scale = exp_diff(mrow, mnew);
            float sum = 0.0f;
            for (int n = 0; n < kChunk / 4; n++) {
                const float p = exp_diff(sv[n], mnew);
                sP[r * LP + tq + 4 * n] = p;
                sum += p;
            }
            sum = warp_sum4(sum);
            lrow = lrow * scale + sum;
            mrow = mnew;
            __syncthreads();
            for (int n = 0; n < NCOL; n++) {
                const int col = tq + 4 * n;
                float tt = 0.0f;
                for (int s = 0; s < nk; s++) tt += sP[r * LP + s] * sX2[s * LX + col];
                acc[n] = acc[n] * scale + tt;
            }
            __syncthreads();
        }
    }
    if (r < nq) {
        const float inv = 1.0f / lrow;
        Tin* o = (Tin*)a.o + (hoff + tbase + r) * D;
        for (int n = 0; n < NCOL; n++) st(o + tq + 4 * n, acc[n] * inv);
        if (tq == 0) a.lse[hoff + tbase + r] = mrow + logf(lrow);
    }
}

// ---------------------------------------------------------------------------------------
// Backward, step 1: D_t = dout_t . o_t.  One warp per row.
template <typename Tin, int D>
__global__ void __launch_bounds__(kThreads)
bwd_rowdot_kernel(const Tin* __restrict__ o, const Tin* __restrict__ dout, float* __restrict__ Dv,
                  long rows) {
    const long row = (long)blockIdx.x * (kThreads / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float s = 0.0f;
    for (int c = lane; c < D; c += 32) s += ld(o + row * D + c) * ld(dout + row * D + c);
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) Dv[row] = s;
}

// Backward, window dq (rotated space, then R_t^T), fp32 into the workspace.
// One CTA per (query tile of C tokens, head), all T queries.
template <typename Tin, int D, int M>
__global__ void __launch_bounds__(kThreads) bwd_window_dq_kernel(const BwdArgs a) {
    extern __shared__ float smem[];
    constexpr int LX = D + 1, LP = kChunk + 1, NCOL = D / 4;
    float* sQ = smem;
    float* sdO = sQ + kChunk * LX;
    float* sK = sdO + kChunk * LX;
    float* sV = sK + kChunk * LX;
    float* sP = sV + kChunk * LX;
    const int tid = threadIdx.x, r = tid >> 2, tq = tid & 3, bh = blockIdx.y;
    const Shape sh = head_shape(a.sh, bh);
    const int tbase = blockIdx.x * kChunk, nq = min(kChunk, sh.T - tbase);
    if (nq <= 0) return;  // past this head's queries (per-sequence lengths)
    const size_t hoff = (size_t)bh * sh.TS;
    const Tin* k = (const Tin*)a.k + hoff * D;
    const Tin* v = (const Tin*)a.v + hoff * D;
    load_rows<Tin, D>((const Tin*)a.q + hoff * D, tbase, nq, sQ, LX, &a.rope);
    load_rows<Tin, D>((const Tin*)a.dout + hoff * D, tbase, nq, sdO, LX, nullptr);
    const float lse_r = (r < nq) ? a.lse[hoff + tbase + r] : 0.0f;
    const float D_r = (r < nq) ? a.Dv[hoff + tbase + r] : 0.0f;
    float g[NCOL];
    for (int n = 0; n < NCOL; n++) g[n] = 0.0f;
    const float sig = sh.sigma;
    const int t = tbase + r;
    if (sh.w > 0) {
        const int klo = max(0, tbase - sh.w + 1), khi = tbase + nq - 1;
        for (int kb = klo; kb <= khi; kb += kChunk) {
            const int nk = min(kChunk, khi - kb + 1);
            __syncthreads();
            load_rows<Tin, D>(k, kb, nk, sK, LX, &a.rope);
            load_rows<Tin, D>(v, kb, nk, sV, LX, nullptr);
            __syncthreads();
            for (int n = 0; n < kChunk / 4; n++) {
                const int s = tq + 4 * n, key = kb + s;
                float ds = 0.0f;
                if (r < nq && s < nk && key <= t && key > t - sh.w) {
                    float qk = 0.0f, dp = 0.0f;
                    for (int cc = 0; cc < D; cc++) {
                        qk += sQ[r * LX + cc] * sK[s * LX + cc];
                        dp += sdO[r * LX + cc] * sV[s * LX + cc];
                    }
                    const float p = expf(sig * qk - lse_r);
                    ds = p * (dp - D_r);
                }
                sP[r * LP + s] = ds;
            }
            __syncthreads();
            for (int n = 0; n < NCOL; n++) {
                const int col = tq + 4 * n;
                float tt = 0.0f;
                for (int s = 0; s < nk; s++) tt += sP[r * LP + s] * sK[s * LX + col];
                g[n] += sig * tt;
            }
        }
    }
    if (r < nq) {
        float* out = a.dqw + (hoff + t) * D;
        for (int n = 0; n < NCOL / 2; n++) {
            const int col = tq + 4 * n;
            float cs, sn;
            rope_cs(a.rope, t, col, cs, sn);
            const float g0 = g[n], g1 = g[n + NCOL / 2];
            out[col] = g0 * cs + g1 * sn;
            out[col + D / 2] = g1 * cs - g0 * sn;
        }
    }
}

// Backward, window dk / dv, fp32 into the workspace.  One CTA per (key tile,
// head); thread (s, tq): key row s = tid / 4.
template <typename Tin, int D, int M>
__global__ void __launch_bounds__(kThreads) bwd_window_dkdv_kernel(const BwdArgs a) {
    extern __shared__ float smem[];
    constexpr int LX = D + 1, LP = kChunk + 1, NCOL = D / 4;
    float* sK = smem;
    float* sV = sK + kChunk * LX;
    float* sQ = sV + kChunk * LX;
    float* sdO = sQ + kChunk * LX;
    float* sPt = sdO + kChunk * LX;
    float* sDt = sPt + kChunk * LP;
    float* sLse = sDt + kChunk * LP;
    float* sD = sLse + kChunk;
    const int tid = threadIdx.x, s = tid >> 2, tq = tid & 3, bh = blockIdx.y;
    const Shape sh = head_shape(a.sh, bh);
    const int sbase = blockIdx.x * kChunk, nk = min(kChunk, sh.T - sbase);
    if (nk <= 0) return;  // past this head's keys (per-sequence lengths)
    const size_t hoff = (size_t)bh * sh.TS;
    const Tin* q = (const Tin*)a.q + hoff * D;
    const Tin* dout = (const Tin*)a.dout + hoff * D;
    load_rows<Tin, D>((const Tin*)a.k + hoff * D, sbase, nk, sK, LX, &a.rope);
    load_rows<Tin, D>((const Tin*)a.v + hoff * D, sbase, nk, sV, LX, nullptr);
    float gk[NCOL], gv[NCOL];
    for (int n = 0; n < NCOL; n++) gk[n] = gv[n] = 0.0f;
    const float sig = sh.sigma;
    const int key = sbase + s;
    if (sh.w > 0) {
        const int tlo = sbase, thi = min(sh.T - 1, sbase + nk - 1 + sh.w - 1);
        for (int qb = tlo; qb <= thi; qb += kChunk) {
            const int nq = min(kChunk, thi - qb + 1);
            __syncthreads();
            load_rows<Tin, D>(q, qb, nq, sQ, LX, &a.rope);
            load_rows<Tin, D>(dout, qb, nq, sdO, LX, nullptr);
            if (tid < kChunk) {
                sLse[tid] = tid < nq ? a.lse[hoff + qb + tid] : 0.0f;
                sD[tid] = tid < nq ? a.Dv[hoff + qb + tid] : 0.0f;
            }
            __syncthreads();
            for (int n = 0; n < kChunk / 4; n++) {
                const int rr = tq + 4 * n, t = qb + rr;
                float p = 0.0f, ds = 0.0f;
                if (s < nk && rr < nq && key <= t && key > t - sh.w) {
                    float qk = 0.0f, dp = 0.0f;
                    for (int cc = 0; cc < D; cc++) {
                        qk += sQ[rr * LX + cc] * sK[s * LX + cc];
                        dp += sdO[rr * LX + cc] * sV[s * LX + cc];
                    }
                    p = expf(sig * qk - sLse[rr]);
                    ds = p * (dp - sD[rr]);
                }
                sPt[s * LP + rr] = p;
                sDt[s * LP + rr] = ds;
            }
            __syncthreads();
            for (int n = 0; n < NCOL; n++) {
                const int col = tq + 4 * n;
                float tk = 0.0f, tv = 0.0f;
                for (int rr = 0; rr < nq; rr++) {
                    tk += sDt[s * LP + rr] * sQ[rr * LX + col];
                    tv += sPt[s * LP + rr] * sdO[rr * LX + col];
                }
                gk[n] += sig * tk;
                gv[n] += tv;
            }
        }
    }
    if (s < nk) {
        float* ok = a.dkw + (hoff + key) * D;
        float* ov = a.dvw + (hoff + key) * D;
        for (int n = 0; n < NCOL / 2; n++) {
            const int col = tq + 4 * n;
            float cs, sn;
            rope_cs(a.rope, key, col, cs, sn);
            const float g0 = gk[n], g1 = gk[n + NCOL / 2];
            ok[col] = g0 * cs + g1 * sn;
            ok[col + D / 2] = g1 * cs - g0 * sn;
        }
        for (int n = 0; n < NCOL; n++) ov[tq + 4 * n] = gv[n];
    }
}

// ---------------------------------------------------------------------------------------
// Backward, slot branch on the query side.  Tiles like the forward.  Leading
// tiles only finalise dq = dq_window.  Chunk tiles recompute the slot logits,
//   dP_L = dout . V^long,  dL = P_L (dP_L - D),
// add dq_slot = sigma (dL o Eb) S^K_prev + sigma [(dL o Eq) Ek^T o causal] K_c,
// and store sigma dL, P_L, db1 = dL L + P_L dP_L (per slot and row) and the
// per-chunk adjoint contributions
//   dR^K_c = (Eb o sigma dL)^T Q,   dR^V_c = (Eb o P_L)^T dout.
template <typename Tin, int D, int M>
__global__ void __launch_bounds__(kThreads) bwd_slot_query_kernel(const BwdArgs a) {
    extern __shared__ float smem[];
    constexpr int LX = D + 1, LP = kChunk + 1, LG = M + 1, NCOL = D / 4, NSL = M / 4;
    float* sQ = smem;
    float* sdO = sQ + kChunk * LX;
    float* sX1 = sdO + kChunk * LX;
    float* sX2 = sX1 + kChunk * LX;
    float* sP = sX2 + kChunk * LX;
    float* sEq = sP + kChunk * LP;
    float* sEk = sEq + kChunk * LG;
    float* sDL = sEk + kChunk * LG;
    float* sPL = sDL + kChunk * LG;
    float* sG = sPL + kChunk * LG;
    float* sER = sG + M;
    const int tid = threadIdx.x, r = tid >> 2, tq = tid & 3, bh = blockIdx.y, x = blockIdx.x;
    const Shape sh = head_shape(a.sh, bh);
    if (x >= sh.NL + sh.NC) return;  // past this head's tiles (per-head windows)
    const size_t hoff = (size_t)bh * sh.TS;
    if (x < sh.NL) {
        const int tbase = x * kChunk, nq = min(kChunk, min(sh.w, sh.T) - tbase);
        for (int e = tid; e < nq * D; e += kThreads)
            st((Tin*)a.dq + (hoff + tbase) * D + e, a.dqw[(hoff + tbase) * D + e]);
        return;
    }
    const int c = x - sh.NL, j0 = c * kChunk, nq = min(kChunk, sh.R - j0), tbase = j0 + sh.w;
    const Tin* q = (const Tin*)a.q + hoff * D;
    const Tin* k = (const Tin*)a.k + hoff * D;
    const Tin* v = (const Tin*)a.v + hoff * D;
    const Tin* dout = (const Tin*)a.dout + hoff * D;
    const float sig = sh.sigma;
    const float lse_r = (r < nq) ? a.lse[hoff + tbase + r] : 0.0f;
    const float D_r = (r < nq) ? a.Dv[hoff + tbase + r] : 0.0f;
    chunk_gates<M>(a.la + (hoff + j0) * M, nq, sEq, sEk, nullptr, LG, sG, sER);
    load_rows<Tin, D>(q, tbase, nq, sQ, LX, nullptr);
    load_rows<Tin, D>(dout, tbase, nq, sdO, LX, nullptr);
    // --- value side: dP_L = Eb o (dO S^V_prev^T) + Eq o ((dO V_c^T o causal) Ek)
    load_rows<Tin, D>(v, j0, nq, sX1, LX, nullptr);
    {
        const float* SVp = a.SV + ((size_t)bh * sh.NCS + c) * M * D;
        for (int e = tid; e < M * D; e += kThreads) sX2[(e / D) * LX + e % D] = SVp[e];
    }
    __syncthreads();
    for (int n = 0; n < kChunk / 4; n++) {
        const int s = tq + 4 * n;
        float t = 0.0f;
        if (s <= r)
            for (int cc = 0; cc < D; cc++) t += sdO[r * LX + cc] * sX1[s * LX + cc];
        sP[r * LP + s] = t;
    }
    __syncthreads();
    float dpl[NSL];
    for (int n = 0; n < NSL; n++) {
        const int i = tq + 4 * n;
        float inter = 0.0f, intra = 0.0f;
        for (int cc = 0; cc < D; cc++) inter += sdO[r * LX + cc] * sX2[i * LX + cc];
        for (int s = 0; s <= r; s++) intra += sP[r * LP + s] * sEk[s * LG + i];
        const float eq = sEq[r * LG + i];
        dpl[n] = eq * sER[i] * inter + eq * intra;
    }
    __syncthreads();
    // --- key side: slot logits L, P_L, dL
    load_rows<Tin, D>(k, j0, nq, sX1, LX, nullptr);
    {
        const float* SKp = a.SK + ((size_t)bh * sh.NCS + c) * M * D;
        for (int e = tid; e < M * D; e += kThreads) sX2[(e / D) * LX + e % D] = SKp[e];
    }
    __syncthreads();
    for (int n = 0; n < kChunk / 4; n++) {
        const int s = tq + 4 * n;
        float t = 0.0f;
        if (s <= r)
            for (int cc = 0; cc < D; cc++) t += sQ[r * LX + cc] * sX1[s * LX + cc];
        sP[r * LP + s] = t;
    }
    __syncthreads();
    const size_t jrow = (size_t)bh * sh.NCS * kChunk + j0 + r;  // row in [BH][NCS*C][M] arrays
    for (int n = 0; n < NSL; n++) {
        const int i = tq + 4 * n;
        float inter = 0.0f, intra = 0.0f;
        for (int cc = 0; cc < D; cc++) inter += sQ[r * LX + cc] * sX2[i * LX + cc];
        for (int s = 0; s <= r; s++) intra += sP[r * LP + s] * sEk[s * LG + i];
        const float eq = sEq[r * LG + i];
        const float L = sig * (eq * sER[i] * inter + eq * intra);
        float pl = 0.0f, dl = 0.0f, db1 = 0.0f;
        if (r < nq) {
            pl = expf(L - lse_r);
            dl = pl * (dpl[n] - D_r);
            db1 = dl * L + pl * dpl[n];
            a.wsDL[jrow * M + i] = sig * dl;
            a.wsPL[jrow * M + i] = pl;
            a.wsDB1[jrow * M + i] = db1;
        }
        sDL[r * LG + i] = sig * dl;
        sPL[r * LG + i] = pl;
    }
    __syncthreads();
    // Bk[r][s] = sum_i sigma dL[r][i] Eq[r][i] Ek[s][i], s <= r
    for (int n = 0; n < kChunk / 4; n++) {
        const int s = tq + 4 * n;
        float t = 0.0f;
        if (s <= r)
            for (int i = 0; i < M; i++) t += sDL[r * LG + i] * sEq[r * LG + i] * sEk[s * LG + i];
        sP[r * LP + s] = t;
    }
    __syncthreads();
    if (r < nq) {
        const size_t orow = (hoff + tbase + r) * D;
        for (int n = 0; n < NCOL; n++) {
            const int col = tq + 4 * n;
            float t = 0.0f;
            for (int i = 0; i < M; i++) t += sDL[r * LG + i] * sEq[r * LG + i] * sER[i] * sX2[i * LX + col];
            for (int s = 0; s <= r; s++) t += sP[r * LP + s] * sX1[s * LX + col];
            st((Tin*)a.dq + orow + col, a.dqw[orow + col] + t);
        }
    }
    // dR^K_c[i][col] = sum_r Eb[r][i] sigma dL[r][i] q_r[col];  dR^V_c likewise with P_L, dout
    float* RK = a.RK + ((size_t)bh * sh.NCS + c) * M * D;
    float* RV = a.RV + ((size_t)bh * sh.NCS + c) * M * D;
    for (int e = tid; e < M * D; e += kThreads) {
        const int i = e / D, col = e % D;
        float rk = 0.0f, rv = 0.0f;
        for (int rr = 0; rr < nq; rr++) {
            const float eb = sEq[rr * LG + i] * sER[i];
            rk += eb * sDL[rr * LG + i] * sQ[rr * LX + col];
            rv += eb * sPL[rr * LG + i] * sdO[rr * LX + col];
        }
        RK[e] = rk;
        RV[e] = rv;
    }
}

// ---------------------------------------------------------------------------------------
// Backward, slot branch on the key side.  One CTA per (key tile = state chunk,
// head); thread (s, tq).  With R^K_s = sum_{j >= s} exp(b_j - b_s) o A^K_j the
// reverse state (A^K_j = sigma dL_j (x) q_{j+w}) and Rc^K the adjoint carried
// in from later chunks:
//   dk_s += u_s^T R^K_s = sum_{j>=s in chunk} [sum_i Ek[s][i] sigma dL[j][i] Eq[j][i]] q_{t(j)}
//           + sum_i exp(G_i - b_{s,i}) u_{s,i} Rc^K[i]
//   du_{s,i} = k_s . R^K_s[i] + v_s . R^V_s[i]
// and likewise dv from P_L, dout and Rc^V.  Then db = db1 - u o du, a
// suffix sum of db inside the chunk, and dlog_alpha = suffix - alpha o du
// (the later chunks' totals are added by bwd_dla_carry).
template <typename Tin, int D, int M>
__device__ void slot_key_phase(const float* sA, const float* sB, const float* sW,
                               const float* sRc, const float* sEq, const float* sEk,
                               const float* sFk, const float* sEG, float* sM1, float* sM2,
                               float* grad, float* du, int s, int tq) {
    constexpr int LX = D + 1, LP = kChunk + 1, LG = M + 1, NCOL = D / 4, NSL = M / 4;
    // sM1[s][j] = sum_i Ek[s][i] W[j][i] Eq[j][i];  sM2[s][j] = b_s . a_{t(j)}   (j >= s)
    for (int n = 0; n < kChunk / 4; n++) {
        const int j = tq + 4 * n;
        float m1 = 0.0f, m2 = 0.0f;
        if (j >= s) {
            for (int i = 0; i < M; i++) m1 += sEk[s * LG + i] * sW[j * LG + i] * sEq[j * LG + i];
            for (int cc = 0; cc < D; cc++) m2 += sB[s * LX + cc] * sA[j * LX + cc];
        }
        sM1[s * LP + j] = m1;
        sM2[s * LP + j] = m2;
    }
    __syncthreads();
    for (int n = 0; n < NCOL; n++) {
        const int col = tq + 4 * n;
        float t = 0.0f;
        for (int j = s; j < kChunk; j++) t += sM1[s * LP + j] * sA[j * LX + col];
        for (int i = 0; i < M; i++) t += sEG[i] * sEk[s * LG + i] * sRc[i * LX + col];
        grad[n] += t;
    }
    for (int n = 0; n < NSL; n++) {
        const int i = tq + 4 * n;
        float intra = 0.0f, inter = 0.0f;
        for (int j = s; j < kChunk; j++) intra += sM2[s * LP + j] * sW[j * LG + i] * sEq[j * LG + i];
        for (int cc = 0; cc < D; cc++) inter += sB[s * LX + cc] * sRc[i * LX + cc];
        du[n] += sFk[s * LG + i] * (intra + sEG[i] * inter);
    }
    __syncthreads();
}

template <typename Tin, int D, int M>
__global__ void __launch_bounds__(kThreads) bwd_slot_key_kernel(const BwdArgs a) {
    extern __shared__ float smem[];
    constexpr int LX = D + 1, LP = kChunk + 1, LG = M + 1, NCOL = D / 4, NSL = M / 4;
    float* sA = smem;                 // q_{t(j)} or dout_{t(j)}
    float* sB = sA + kChunk * LX;     // k_s or v_s
    float* sRc = sB + kChunk * LX;    // Rc^K or Rc^V
    float* sW = sRc + kChunk * LX;    // sigma dL or P_L
    float* sEq = sW + kChunk * LG;
    float* sEk = sEq + kChunk * LG;
    float* sFk = sEk + kChunk * LG;
    float* sM1 = sFk + kChunk * LG;
    float* sM2 = sM1 + kChunk * LP;
    float* sG = sM2 + kChunk * LP;
    float* sER = sG + M;
    float* sEG = sER + M;  // exp(G / 2) = exp(G - rho)
    const int tid = threadIdx.x, s = tid >> 2, tq = tid & 3, bh = blockIdx.y, x = blockIdx.x;
    const Shape sh = head_shape(a.sh, bh);
    const size_t hoff = (size_t)bh * sh.TS;
    const int sbase = x * kChunk, nk = min(kChunk, sh.T - sbase);
    if (nk <= 0) return;  // past this head's keys (per-sequence lengths)
    const int nc = (x < sh.NC) ? min(kChunk, sh.R - sbase) : 0;
    float gk[NCOL], gv[NCOL], du[NSL];
    for (int n = 0; n < NCOL; n++) gk[n] = gv[n] = 0.0f;
    for (int n = 0; n < NSL; n++) du[n] = 0.0f;
    if (nc > 0) {
        const Tin* q = (const Tin*)a.q + hoff * D;
        const Tin* k = (const Tin*)a.k + hoff * D;
        const Tin* v = (const Tin*)a.v + hoff * D;
        const Tin* dout = (const Tin*)a.dout + hoff * D;
        const size_t jrow0 = (size_t)bh * sh.NCS * kChunk + sbase;
        chunk_gates<M>(a.la + (hoff + sbase) * M, nc, sEq, sEk, sFk, LG, sG, sER);
        __syncthreads();
        if (tid < M) sEG[tid] = expf(0.5f * sG[tid]);
        for (int pass = 0; pass < 2; pass++) {
            const float* W = pass == 0 ? a.wsDL : a.wsPL;
            const float* Rc = (pass == 0 ? a.RK : a.RV) + ((size_t)bh * sh.NCS + x) * M * D;
            load_rows<Tin, D>(pass == 0 ? q : dout, sbase + sh.w, nc, sA, LX, nullptr);
            load_rows<Tin, D>(pass == 0 ? k : v, sbase, nc, sB, LX, nullptr);
            for (int e = tid; e < M * D; e += kThreads) sRc[(e / D) * LX + e % D] = Rc[e];
            for (int e = tid; e < kChunk * M; e += kThreads) {
                const int j = e / M, i = e % M;
                sW[j * LG + i] = j < nc ? W[(jrow0 + j) * M + i] : 0.0f;
            }
            __syncthreads();
            slot_key_phase<Tin, D, M>(sA, sB, sW, sRc, sEq, sEk, sFk, sEG, sM1, sM2,
                                      pass == 0 ? gk : gv, du, s, tq);
        }
        // db = db1 - u du; suffix sum over the chunk; dlog_alpha = suffix - alpha du
        float* sDB = sM1;  // [C][LG] fits in [C][LP] since M <= C
        for (int n = 0; n < NSL; n++) {
            const int i = tq + 4 * n;
            float db = 0.0f;
            if (s < nc) {
                const float l = a.la[(hoff + sbase + s) * M + i];
                db = a.wsDB1[(jrow0 + s) * M + i] - (-expm1f(l)) * du[n];
            }
            sDB[s * LG + i] = db;
        }
        __syncthreads();
        if (tid < M) {
            float acc = 0.0f;
            for (int rr = nc - 1; rr >= 0; rr--) {
                acc += sDB[rr * LG + tid];
                sDB[rr * LG + tid] = acc;
            }
        }
        __syncthreads();
    }
    if (s < nk) {
        const size_t orow = (hoff + sbase + s) * D;
        for (int n = 0; n < NCOL; n++) {
            const int col = tq + 4 * n;
            st((Tin*)a.dk + orow + col, a.dkw[orow + col] + gk[n]);
            st((Tin*)a.dv + orow + col, a.dvw[orow + col] + gv[n]);
        }
        for (int n = 0; n < NSL; n++) {
            const int i = tq + 4 * n;
            float val = 0.0f;
            if (s < nc) {
                const float l = a.la[(hoff + sbase + s) * M + i];
                val = sM1[s * LG + i] - expf(l) * du[n];
            }
            a.dla[(hoff + sbase + s) * M + i] = val;
        }
    }
}

// dlog_alpha rows of chunk c += sum of db over all later chunks.  That sum
// telescopes: with F_r = sum_{j >= r} db_j = d loss / d log_alpha_r through
// alpha_r alone = alpha_r (R_r . S_{r-1}) (R_r the adjoint of the state after
// token r), and j' the first token of chunk c + 1,
//   sum_{c' > c} (db summed over chunk c') = F_{j'} = Rc(c) . S_prev(c + 1)
// per slot, where Rc(c) = alpha_{j'} R_{j'} is the adjoint carried into the end
// of chunk c (reverse scan) and S_prev(c + 1) = S_{j'-1} the state before
// chunk c + 1 (forward scan).  Computing it at the boundary avoids summing
// thousands of terms whose total is zero.  Grid (NC, BH); one warp per slot.
template <int M>
__global__ void __launch_bounds__(kThreads) bwd_dla_carry_kernel(const BwdArgs a, int D) {
    const int c = blockIdx.x, bh = blockIdx.y;
    const Shape sh = head_shape(a.sh, bh);
    if (c >= sh.NC) return;  // past this head's chunks (per-head windows)
    const int j0 = c * kChunk, nc = min(kChunk, sh.R - j0);
    __shared__ float carry[64];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (c + 1 < sh.NC || a.dhTk != nullptr) {
        // the state after chunk c: the next chunk's entering state, or the final state
        const size_t cur = ((size_t)bh * sh.NCS + c) * M * D;
        const float* SKn = c + 1 < sh.NC ? a.SK + cur + (size_t)M * D : a.io.htf + (size_t)bh * 2 * M * D;
        const float* SVn = c + 1 < sh.NC ? a.SV + cur + (size_t)M * D : a.io.htf + ((size_t)bh * 2 + 1) * M * D;
        for (int i = warp; i < M; i += kThreads / 32) {
            float acc = 0.0f;
            for (int d = lane; d < D; d += 32) {
                const size_t o = (size_t)i * D + d;
                acc += a.RK[cur + o] * SKn[o] + a.RV[cur + o] * SVn[o];
            }
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) carry[i] = acc;
        }
    } else if (threadIdx.x < M) {
        carry[threadIdx.x] = 0.0f;
    }
    __syncthreads();
    const size_t hoff = (size_t)bh * sh.TS;
    for (int e = threadIdx.x; e < nc * M; e += kThreads) a.dla[(hoff + j0) * M + e] += carry[e % M];
}

// ---------------------------------------------------------------------------------------
// Host-side launchers.
template <typename K>
static cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

#define NHA_CHECK(...)                                \
    do {                                              \
        cudaError_t e_ = (__VA_ARGS__);                       \
        if (e_ != cudaSuccess) return e_;             \
    } while (0)

template <typename Tin, int D, int M>
cudaError_t simt_states(const Tin* k, const Tin* v, const float* la, float* SK, float* SV,
                               float* G, const StateIO& io, const Shape& sh, cudaStream_t st) {
    if (sh.NCS == 0) return launch_final_states_copy(io, sh.BH, M, D, st);
    constexpr int LX = D + 1, LG = M + 1;
    size_t sm = sizeof(float) * (size_t)(kChunk * LX + 2 * kChunk * LG);
    auto kern = state_chunk_kernel<Tin, D, M>;
    NHA_CHECK(set_smem(kern, sm));
    NHA_LAUNCH("state_chunk", st, kern<<<dim3(sh.NCS, sh.BH), kThreads, sm, st>>>(k, v, la, SK, SV, G, sh));
    NHA_CHECK(cudaGetLastError());
    NHA_LAUNCH("state_scan", st,
               state_scan_kernel<<<dim3((M * D + kThreads - 1) / kThreads, sh.BH, 2), kThreads, 0, st>>>(
                   SK, SV, G, sh, M, D, +1, io.h0k, io.h0v, io.hTk, io.hTv, io.htf));
    return cudaGetLastError();
}

template <typename Tin, int D, int M>
cudaError_t simt_forward(const FwdArgs& a, cudaStream_t st) {
    const Shape& sh = a.sh;
    NHA_CHECK(simt_states<Tin, D, M>((const Tin*)a.k, (const Tin*)a.v, a.la, a.SK, a.SV, a.G, a.io, sh, st));
    constexpr int LX = D + 1, LP = kChunk + 1, LG = M + 1;
    size_t sm = sizeof(float) * (size_t)(3 * kChunk * LX + kChunk * LP + 3 * kChunk * LG + 2 * M);
    auto kern = fwd_main_kernel<Tin, D, M>;
    NHA_CHECK(set_smem(kern, sm));
    // with per-head windows a head has at most ceil(T / C) + 1 tiles
    const int tiles = varied(sh) ? sh.NKT + 1 : sh.NL + sh.NC;
    if (tiles > 0) NHA_LAUNCH("fwd_main", st, kern<<<dim3(tiles, sh.BH), kThreads, sm, st>>>(a));
    NHA_CHECK(cudaGetLastError());
    return launch_h0_fwd_lead<Tin, D, M>(a, st);  // queries t < w reading initial states
}

template <typename Tin, int D, int M>
cudaError_t simt_bwd_slot(const BwdArgs& a, cudaStream_t st) {
    const Shape& sh = a.sh;
    constexpr int LX = D + 1, LP = kChunk + 1, LG = M + 1;
    {
        size_t sm = sizeof(float) * (size_t)(4 * kChunk * LX + kChunk * LP + 4 * kChunk * LG + 2 * M);
        auto kern = bwd_slot_query_kernel<Tin, D, M>;
        NHA_CHECK(set_smem(kern, sm));
        const int tiles = varied(sh) ? sh.NKT + 1 : sh.NL + sh.NC;
        if (tiles > 0) NHA_LAUNCH("bwd_slot_query", st, kern<<<dim3(tiles, sh.BH), kThreads, sm, st>>>(a));
        NHA_CHECK(cudaGetLastError());
        NHA_CHECK(launch_h0_bwd_lead<Tin, D, M>(a, false, st));  // queries t < w reading initial states
    }
    if (sh.NCS > 0) {
        NHA_LAUNCH("state_scan_rev", st,
                   state_scan_kernel<<<dim3((M * D + kThreads - 1) / kThreads, sh.BH, 2), kThreads, 0, st>>>(
                       a.RK, a.RV, a.G, sh, M, D, -1, a.dhTk, a.dhTv, nullptr, nullptr, a.rend));
        NHA_CHECK(cudaGetLastError());
    }
    {
        size_t sm = sizeof(float) * (size_t)(3 * kChunk * LX + 4 * kChunk * LG + 2 * kChunk * LP + 3 * M);
        auto kern = bwd_slot_key_kernel<Tin, D, M>;
        NHA_CHECK(set_smem(kern, sm));
        NHA_LAUNCH("bwd_slot_key", st, kern<<<dim3(sh.NKT, sh.BH), kThreads, sm, st>>>(a));
        NHA_CHECK(cudaGetLastError());
    }
    if (sh.NCS > 1 || (sh.NCS > 0 && a.dhTk != nullptr)) {
        NHA_LAUNCH("bwd_dla_carry", st, bwd_dla_carry_kernel<M><<<dim3(sh.NCS, sh.BH), kThreads, 0, st>>>(a, D));
        NHA_CHECK(cudaGetLastError());
    }
    return launch_dh0<Tin, D, M>(a, st);
}

template <typename Tin, int D, int M>
cudaError_t simt_backward(const BwdArgs& a, cudaStream_t st) {
    const Shape& sh = a.sh;
    constexpr int LX = D + 1, LP = kChunk + 1;
    if (!a.reuse)
        NHA_CHECK(simt_states<Tin, D, M>((const Tin*)a.k, (const Tin*)a.v, a.la, a.SK, a.SV, a.G, a.io, sh, st));
    const long rows = (long)sh.BH * sh.T;
    NHA_LAUNCH("bwd_rowdot", st,
               bwd_rowdot_kernel<Tin, D><<<(unsigned)((rows + 7) / 8), kThreads, 0, st>>>(
                   (const Tin*)a.o, (const Tin*)a.dout, a.Dv, rows));
    NHA_CHECK(cudaGetLastError());
    {
        size_t sm = sizeof(float) * (size_t)(4 * kChunk * LX + kChunk * LP);
        auto kern = bwd_window_dq_kernel<Tin, D, M>;
        NHA_CHECK(set_smem(kern, sm));
        NHA_LAUNCH("bwd_window_dq", st, kern<<<dim3(sh.NKT, sh.BH), kThreads, sm, st>>>(a));
        NHA_CHECK(cudaGetLastError());
    }
    {
        size_t sm = sizeof(float) * (size_t)(4 * kChunk * LX + 2 * kChunk * LP + 2 * kChunk);
        auto kern = bwd_window_dkdv_kernel<Tin, D, M>;
        NHA_CHECK(set_smem(kern, sm));
        NHA_LAUNCH("bwd_window_dkdv", st, kern<<<dim3(sh.NKT, sh.BH), kThreads, sm, st>>>(a));
        NHA_CHECK(cudaGetLastError());
    }
    return simt_bwd_slot<Tin, D, M>(a, st);
}

#define NHA_INST(Tin, D, M)                                                          \
    template cudaError_t simt_states<Tin, D, M>(const Tin*, const Tin*, const float*, float*, \
                                                float*, float*, const StateIO&, const Shape&, cudaStream_t); \
    template cudaError_t simt_forward<Tin, D, M>(const FwdArgs&, cudaStream_t);      \
    template cudaError_t simt_backward<Tin, D, M>(const BwdArgs&, cudaStream_t);    \
    template cudaError_t simt_bwd_slot<Tin, D, M>(const BwdArgs&, cudaStream_t);

#define NHA_INST_D(Tin, D) NHA_INST(Tin, D, 16) NHA_INST(Tin, D, 32) NHA_INST(Tin, D, 64)
NHA_INST_D(float, 64)
NHA_INST_D(float, 128)
NHA_INST_D(__nv_bfloat16, 64)
NHA_INST_D(__nv_bfloat16, 128)

}  // namespace nha
