// Initial and final slot states of the chunkwise operator.
//
// The initial states h0 = (h0k, h0v) are the long memory before token 0 (the
// ai.info page, Future Directions, names learned initial slot states; the
// Paper-Notes page's chunkwise form, Chunkwise 并行计算, carries a state from
// chunk to chunk).  The chunk scans start from h0 instead of zero, so every
// query t >= w sees it through the states they read.  The queries t < w,
// which see no token of the long memory yet, read h0 itself: their slot
// logits are q_t . h0k[i] / sqrt(d) with no gate, and their slot readout is
// sum_i p_i h0v[i].  The chunk kernels treat those queries as window-only;
// the kernels here add the slot branch of h0 to them (forward), and its
// gradients (backward), in fp32 on the CUDA cores: m * d multiply-adds per
// query and branch.  dh0 = the state adjoint the reverse chunk scan carries
// past chunk 0 plus these queries' terms.  The final states hT are the long
// memory after the last token that left the window.
#include "nha_common.cuh"
#include "nha_kernels.h"
#include "nha_prof.h"
#include "nha_tc.cuh"

namespace nha {

namespace {

constexpr int kH0Threads = 256, kH0Rows = 64;  // 8 warps, 8 rows per warp

// hT = h0 (or zero) and the scans' workspace copies, when no chunk is scanned.
__global__ void __launch_bounds__(256)
final_states_copy_kernel(const StateIO io, int BH, int MD) {
    const long e = (long)blockIdx.x * 256 + threadIdx.x;
    if (e >= (long)BH * MD) return;
    const long bh = e / MD, r = e % MD;
    const float k = io.h0k != nullptr ? io.h0k[e] : 0.0f;
    const float v = io.h0v != nullptr ? io.h0v[e] : 0.0f;
    if (io.hTk != nullptr) io.hTk[e] = k;
    if (io.hTv != nullptr) io.hTv[e] = v;
    if (io.htb != nullptr) {
        io.htb[(bh * 2) * MD + r] = __float2bfloat16_rn(k);
        io.htb[(bh * 2 + 1) * MD + r] = __float2bfloat16_rn(v);
    }
    if (io.htf != nullptr) {
        io.htf[(bh * 2) * MD + r] = k;
        io.htf[(bh * 2 + 1) * MD + r] = v;
    }
}

// h0k, h0v of head bh into shared memory, rows padded to D + 1 floats.
template <int D, int M>
__device__ void load_h0(const StateIO& io, int bh, float* sK, float* sV) {
    for (int e = threadIdx.x; e < M * D; e += kH0Threads) {
        const int i = e / D, c = e % D;
        sK[i * (D + 1) + c] = io.h0k[((size_t)bh * M + i) * D + c];
        sV[i * (D + 1) + c] = io.h0v[((size_t)bh * M + i) * D + c];
    }
}

// Slot logits of one query row against h0k, lane = slot (lane, lane + 32):
// L[s] for the lane's slots, -inf past m.
template <int D, int M>
__device__ __forceinline__ void h0_logits(const float* sK, const float* qrow, float sigma, float (&L)[2], int lane) {
#pragma unroll
    for (int s = 0; s < 2; s++) {
        const int i = lane + 32 * s;
        float acc = 0.0f;
        if (i < M) {
            const float* kr = sK + i * (D + 1);
#pragma unroll 8
            for (int c = 0; c < D; c++) acc = fmaf(qrow[c], kr[c], acc);
        }
        L[s] = i < M ? sigma * acc : -INFINITY;
    }
}

// Forward of the queries t < W0 = min(w, T): one warp per row.
template <typename Tin, int D, int M>
__global__ void __launch_bounds__(kH0Threads)
h0_fwd_lead_kernel(const FwdArgs a) {
    extern __shared__ float smem[];
    float* sK = smem;                    // [M][D + 1]
    float* sV = sK + M * (D + 1);        // [M][D + 1]
    float* sRow = sV + M * (D + 1);      // [8 warps][D]  q row
    float* sP = sRow + 8 * D;            // [8 warps][M]  slot weights
    const int bh = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Shape sh = head_shape(a.sh, bh);
    const int W0 = sh.T - sh.R;
    if (blockIdx.x * kH0Rows >= W0) return;  // past this head's rows (per-head windows)
    load_h0<D, M>(a.io, bh, sK, sV);
    __syncthreads();
    const size_t hoff = (size_t)bh * sh.TS;
    float* qrow = sRow + warp * D;
    float* prow = sP + warp * M;
    for (int rr = warp; rr < kH0Rows; rr += 8) {
        const int t = blockIdx.x * kH0Rows + rr;
        if (t >= W0) break;
        const Tin* q = (const Tin*)a.q + (hoff + t) * D;
        for (int c = lane; c < D; c += 32) qrow[c] = ld(q + c);
        __syncwarp();
        float L[2];
        h0_logits<D, M>(sK, qrow, sh.sigma, L, lane);
        float ms = fmaxf(L[0], L[1]);
        for (int off = 16; off > 0; off >>= 1) ms = fmaxf(ms, __shfl_xor_sync(0xffffffffu, ms, off));
        float zs = expf(L[0] - ms) + expf(L[1] - ms);
        for (int off = 16; off > 0; off >>= 1) zs += __shfl_xor_sync(0xffffffffu, zs, off);
        // merge with the window branch the chunk kernels left in (o, lse)
        const float lw = a.lse[hoff + t];
        const float ls = ms + logf(zs);
        const float mx = fmaxf(lw, ls);
        const float lse = mx + logf(expf(lw - mx) + expf(ls - mx));
        const float fw = expf(lw - lse);
#pragma unroll
        for (int s = 0; s < 2; s++)
            if (lane + 32 * s < M) prow[lane + 32 * s] = expf(L[s] - lse);
        __syncwarp();
        Tin* o = (Tin*)a.o + (hoff + t) * D;
        for (int c = lane; c < D; c += 32) {
            float acc = fw * ld(o + c);
#pragma unroll 8
            for (int i = 0; i < M; i++) acc = fmaf(prow[i], sV[i * (D + 1) + c], acc);
            st(o + c, acc);
        }
        if (lane == 0) a.lse[hoff + t] = lse;
        __syncwarp();
    }
}

// Backward of the same rows (lse: the forward's final lse).  tc: the bf16
// path, whose query-side kernel left dq = window part + (D^ - D_win) correction
// and D = D_win for these rows: the exact D gains the slot part, dq is
// rebuilt from the window partials.  Otherwise dq holds the window part and D
// is exact already (D = dout . o, fp32).
template <typename Tin, int D, int M, bool kTc>
__global__ void __launch_bounds__(kH0Threads)
h0_bwd_lead_kernel(const BwdArgs a) {
    extern __shared__ float smem[];
    float* sK = smem;
    float* sV = sK + M * (D + 1);
    float* sRow = sV + M * (D + 1);  // [8 warps][2][D]  q row, dout row
    float* sP = sRow + 16 * D;       // [8 warps][M]     sigma dL
    const int bh = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Shape sh = head_shape(a.sh, bh);
    const int W0 = sh.T - sh.R, W0S = a.sh.W0S;
    if (blockIdx.x * kH0Rows >= W0) return;  // past this head's rows (per-head windows)
    load_h0<D, M>(a.io, bh, sK, sV);
    __syncthreads();
    const size_t hoff = (size_t)bh * sh.TS;
    float* qrow = sRow + warp * 2 * D;
    float* grow = qrow + D;
    float* prow = sP + warp * M;
    for (int rr = warp; rr < kH0Rows; rr += 8) {
        const int t = blockIdx.x * kH0Rows + rr;
        if (t >= W0) break;
        const Tin* q = (const Tin*)a.q + (hoff + t) * D;
        const Tin* g = (const Tin*)a.dout + (hoff + t) * D;
        for (int c = lane; c < D; c += 32) {
            qrow[c] = ld(q + c);
            grow[c] = ld(g + c);
        }
        __syncwarp();
        float L[2], dP[2];
        h0_logits<D, M>(sK, qrow, sh.sigma, L, lane);
#pragma unroll
        for (int s = 0; s < 2; s++) {
            const int i = lane + 32 * s;
            float acc = 0.0f;
            if (i < M)
#pragma unroll 8
                for (int c = 0; c < D; c++) acc = fmaf(grow[c], sV[i * (D + 1) + c], acc);
            dP[s] = acc;
        }
        const float lse = a.lse[hoff + t];
        float P[2], slot = 0.0f;
#pragma unroll
        for (int s = 0; s < 2; s++) {
            P[s] = (lane + 32 * s < M) ? expf(L[s] - lse) : 0.0f;
            slot += P[s] * dP[s];
        }
        for (int off = 16; off > 0; off >>= 1) slot += __shfl_xor_sync(0xffffffffu, slot, off);
        const float Dt = kTc ? a.Dwin[hoff + t] + slot : a.Dv[hoff + t];
#pragma unroll
        for (int s = 0; s < 2; s++) {
            const int i = lane + 32 * s;
            if (i < M) {
                const float sdl = sh.sigma * P[s] * (dP[s] - Dt);
                prow[i] = sdl;
                a.ldl[((size_t)bh * W0S + t) * M + i] = sdl;
                a.lpl[((size_t)bh * W0S + t) * M + i] = P[s];
            }
        }
        __syncwarp();
        if (kTc) {
            if (lane == 0) a.Dv[hoff + t] = Dt;
            const float corr = a.Dhat[hoff + t] - Dt;
            const __nv_bfloat16* gw = a.hdqw + (hoff + t) * D;
            const __nv_bfloat16* gc = a.hdqwV + (hoff + t) * D;
            __nv_bfloat16* dq = (__nv_bfloat16*)a.dq + (hoff + t) * D;
            for (int c = lane; c < D; c += 32) {
                float acc = __bfloat162float(gw[c]) + corr * __bfloat162float(gc[c]);
#pragma unroll 8
                for (int i = 0; i < M; i++) acc = fmaf(prow[i], sK[i * (D + 1) + c], acc);
                dq[c] = __float2bfloat16_rn(acc);
            }
        } else {
            Tin* dq = (Tin*)a.dq + (hoff + t) * D;
            for (int c = lane; c < D; c += 32) {
                float acc = ld(dq + c);
#pragma unroll 8
                for (int i = 0; i < M; i++) acc = fmaf(prow[i], sK[i * (D + 1) + c], acc);
                st(dq + c, acc);
            }
        }
        __syncwarp();
    }
}

// dh0[z][i][d] = base + sum_{t < W0} X_t[i] Y_t[d] with (X, Y) = (sigma dL, q)
// for z = 0 (K) and (P_L, dout) for z = 1 (V); base = the adjoint the reverse
// chunk scan carries past chunk 0, or dhT (zero without it) when no chunk.
// Thread = (4 slots, column d); grid (M / 4 * D / 256, BH, 2).
template <typename Tin, int D, int M>
__global__ void __launch_bounds__(256)
dh0_kernel(const BwdArgs a) {
    const int bh = blockIdx.y, z = blockIdx.z;
    const Shape sh = head_shape(a.sh, bh);
    const int W0 = sh.T - sh.R;
    const int e = blockIdx.x * 256 + threadIdx.x;  // over (M / 4) * D
    if (e >= (M / 4) * D) return;
    const int i0 = 4 * (e / D), d = e % D;
    float acc[4];
#pragma unroll
    for (int s = 0; s < 4; s++) {
        const size_t o = ((size_t)bh * M + i0 + s) * D + d;
        if (sh.NC > 0)
            acc[s] = a.rend[(((size_t)bh * 2 + z) * M + i0 + s) * D + d];
        else {
            const float* dh = z == 0 ? a.dhTk : a.dhTv;
            acc[s] = dh != nullptr ? dh[o] : 0.0f;
        }
    }
    if (W0 > 0) {
        const float* X = (z == 0 ? a.ldl : a.lpl) + (size_t)bh * a.sh.W0S * M + i0;
        const Tin* Y = (const Tin*)(z == 0 ? a.q : a.dout) + (size_t)bh * sh.TS * D + d;
        for (int t = 0; t < W0; t++) {
            const float4 x = *reinterpret_cast<const float4*>(X + (size_t)t * M);
            const float y = ld(Y + (size_t)t * D);
            acc[0] = fmaf(x.x, y, acc[0]);
            acc[1] = fmaf(x.y, y, acc[1]);
            acc[2] = fmaf(x.z, y, acc[2]);
            acc[3] = fmaf(x.w, y, acc[3]);
        }
    }
    float* out = z == 0 ? a.dh0k : a.dh0v;
#pragma unroll
    for (int s = 0; s < 4; s++) out[((size_t)bh * M + i0 + s) * D + d] = acc[s];
}

// decay[bh][i] = exp(sum of log_alpha[bh][j][i] over j < T - w): the factor the
// tokens that leave the window apply to the state a segment starts from.
// Thread = (head, slot), a sequential sum in fp32.
__global__ void __launch_bounds__(256)
gate_total_kernel(const float* __restrict__ la, float* __restrict__ decay, int BH, int T, int M, int R) {
    const long e = (long)blockIdx.x * 256 + threadIdx.x;
    if (e >= (long)BH * M) return;
    const long bh = e / M, i = e % M;
    const float* p = la + (size_t)bh * T * M + i;
    float s = 0.0f;
    for (int j = 0; j < R; j++) s += p[(size_t)j * M];
    decay[e] = expf(s);
}

// out = decay o prev + cur for K and V (decay [BH][M] broadcast over d); out
// may be cur.
__global__ void __launch_bounds__(256)
state_combine_kernel(const float* __restrict__ decay, const float* __restrict__ pk, const float* __restrict__ pv,
                     const float* ck, const float* cv, float* ok, float* ov, int BH, int M, int D) {
    const long e = (long)blockIdx.x * 256 + threadIdx.x;
    if (e >= (long)BH * M * D) return;
    const float a = decay[e / D];
    ok[e] = fmaf(a, pk[e], ck[e]);
    ov[e] = fmaf(a, pv[e], cv[e]);
}

// A bounded wait on an mbarrier that nothing arrives at: it gives up after
// `cycles` SM clock cycles and reports it in the status word, the way every
// tensor-core kernel reports a wait that ran out.  One thread, no copies or
// tensor-core work in flight.
__global__ void selftest_wait_kernel(int* status, long long cycles) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    tc::mbar_init(&bar, 1);
    tc::mbar_fence_init();
    if (!tc::mbar_wait(&bar, 0, cycles)) atomicOr(status, kStatusTimeoutBit);
}

template <int D, int M>
size_t h0_smem(int rowfloats) {
    return sizeof(float) * (size_t)(2 * M * (D + 1) + 8 * rowfloats * D + 8 * M);
}

}  // namespace

cudaError_t launch_selftest_wait(int* status, long long cycles, cudaStream_t st) {
    NHA_LAUNCH("selftest_wait", st, selftest_wait_kernel<<<1, 32, 0, st>>>(status, cycles));
    return cudaGetLastError();
}

cudaError_t launch_gate_total(const float* la, float* decay, int BH, int T, int M, int R, cudaStream_t st) {
    const long n = (long)BH * M;
    if (n == 0) return cudaSuccess;
    NHA_LAUNCH("gate_total", st,
               gate_total_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(la, decay, BH, T, M, R));
    return cudaGetLastError();
}

cudaError_t launch_state_combine(const float* decay, const float* pk, const float* pv, const float* ck,
                                 const float* cv, float* ok, float* ov, int BH, int M, int D, cudaStream_t st) {
    const long n = (long)BH * M * D;
    if (n == 0) return cudaSuccess;
    NHA_LAUNCH("state_combine", st,
               state_combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(decay, pk, pv, ck, cv, ok, ov, BH,
                                                                                 M, D));
    return cudaGetLastError();
}

cudaError_t launch_final_states_copy(const StateIO& io, int BH, int M, int D, cudaStream_t st) {
    if (io.hTk == nullptr && io.hTv == nullptr && io.htb == nullptr && io.htf == nullptr) return cudaSuccess;
    const long n = (long)BH * M * D;
    if (n == 0) return cudaSuccess;
    NHA_LAUNCH("final_states", st,
               final_states_copy_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(io, BH, M * D));
    return cudaGetLastError();
}

template <typename Tin, int D, int M>
cudaError_t launch_h0_fwd_lead(const FwdArgs& a, cudaStream_t st) {
    const int W0 = a.sh.T - a.sh.R;
    if (a.io.h0k == nullptr || W0 == 0 || a.sh.BH == 0) return cudaSuccess;
    const size_t sm = h0_smem<D, M>(1);
    auto kern = h0_fwd_lead_kernel<Tin, D, M>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    NHA_LAUNCH("h0_fwd_lead", st,
               kern<<<dim3((W0 + kH0Rows - 1) / kH0Rows, a.sh.BH), kH0Threads, sm, st>>>(a));
    return cudaGetLastError();
}

template <typename Tin, int D, int M>
cudaError_t launch_h0_bwd_lead(const BwdArgs& a, bool tc, cudaStream_t st) {
    const int W0 = a.sh.T - a.sh.R;
    if (a.io.h0k == nullptr || W0 == 0 || a.sh.BH == 0) return cudaSuccess;
    const size_t sm = h0_smem<D, M>(2);
    const dim3 grid((W0 + kH0Rows - 1) / kH0Rows, a.sh.BH);
    cudaError_t e;
    if (tc) {
        auto kern = h0_bwd_lead_kernel<Tin, D, M, true>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) != cudaSuccess)
            return e;
        NHA_LAUNCH("h0_bwd_lead", st, kern<<<grid, kH0Threads, sm, st>>>(a));
    } else {
        auto kern = h0_bwd_lead_kernel<Tin, D, M, false>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) != cudaSuccess)
            return e;
        NHA_LAUNCH("h0_bwd_lead", st, kern<<<grid, kH0Threads, sm, st>>>(a));
    }
    return cudaGetLastError();
}

template <typename Tin, int D, int M>
cudaError_t launch_dh0(const BwdArgs& a, cudaStream_t st) {
    if (a.dh0k == nullptr || a.sh.BH == 0) return cudaSuccess;
    const int n = (M / 4) * D;
    NHA_LAUNCH("dh0", st, dh0_kernel<Tin, D, M><<<dim3((n + 255) / 256, a.sh.BH, 2), 256, 0, st>>>(a));
    return cudaGetLastError();
}

#define NHA_H0_INST(Tin, D, M)                                                               \
    template cudaError_t launch_h0_fwd_lead<Tin, D, M>(const FwdArgs&, cudaStream_t);        \
    template cudaError_t launch_h0_bwd_lead<Tin, D, M>(const BwdArgs&, bool, cudaStream_t); \
    template cudaError_t launch_dh0<Tin, D, M>(const BwdArgs&, cudaStream_t);
#define NHA_H0_INST_D(Tin, D) NHA_H0_INST(Tin, D, 16) NHA_H0_INST(Tin, D, 32) NHA_H0_INST(Tin, D, 64)
NHA_H0_INST_D(float, 64)
NHA_H0_INST_D(float, 128)
NHA_H0_INST_D(__nv_bfloat16, 64)
NHA_H0_INST_D(__nv_bfloat16, 128)

}  // namespace nha
