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

namespace nha {
using namespace tc;

__global__ void rope_table_kernel(float2* __restrict__ tab, int T, int H2, RopeTab rt) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= T * H2) return;
    float c, s;
    rope_cs(rt, e / H2, e % H2, c, s);
    tab[e] = make_float2(c, s);
}

template <int D, int M>
__global__ void __launch_bounds__(kTcThreads, 1)
fwd_tc_kernel(const FwdArgs a, const __nv_bfloat16* __restrict__ qr, const __nv_bfloat16* __restrict__ kr,
              int* __restrict__ status) {
    constexpr int HM = M / 2, HD = D / 2, TB = 128 * D * 2;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* X0 = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* KB[2];
    unsigned char* VB[2];
    KB[0] = X0 + TB;        // K~ block / P      (slot phase: K_c, masks, A_inter)
    VB[0] = KB[0] + 32768;  // V block           (slot phase: V_c)
    KB[1] = VB[0] + 32768;  //                   (slot phase: [S^K] then [S^V] pair)
    VB[1] = KB[1] + 32768;  //                   (slot phase: Ek, then pEq at +16 KB)
    float* s_tot = reinterpret_cast<float*>(VB[1] + 32768);  // [4][M]
    float* sG = s_tot + 4 * M;                                // [2][M]
    float* redm = sG + 2 * M;                                 // [2][128]
    float* reds = redm + 256;                                 // [2][128]
    __shared__ uint64_t bar;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const Shape sh = a.sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = ((warp & 3) << 5) | lane, h = warp >> 2, cr = r >> 6;
    const int W0 = sh.T - sh.R;
    const int NLT = (W0 + 127) / 128;
    const int x = blockIdx.x, bh = blockIdx.y;
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
    const bool row_ok = r < nq;
    const size_t hoff = (size_t)bh * sh.T;
    const __nv_bfloat16* q = (const __nv_bfloat16*)a.q + hoff * D;
    const __nv_bfloat16* k = (const __nv_bfloat16*)a.k + hoff * D;
    const __nv_bfloat16* v = (const __nv_bfloat16*)a.v + hoff * D;
    qr += hoff * D;
    kr += hoff * D;
    const float sig2 = sh.sigma * kLog2e;

    if (tid < 2 * M) sG[tid] = 0.0f;
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
        s_abort = 0;
    }
    if (warp == 0) tmem_alloc(&s_tmem, 256);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = s_tmem;
    const uint32_t tl = tm + ((uint32_t)((warp & 3) * 32) << 16);  // this warp's lanes
    const uint32_t tA = 0, tO = 128;                                 // column offsets
    TcCtl ctl{&bar, 0u, &s_abort, status};
    bool ok = true;

    float m = -INFINITY, l = 0.0f;  // running max (log2 domain) and sum of the row
    bool o_valid = false;

    if (slot) {
        const int c1 = j0 / kChunk;
        const bool has2 = nq > kChunk;
        const __nv_bfloat16* SK1 = a.SKb + ((size_t)bh * sh.NC + c1) * M * D;
        const __nv_bfloat16* SV1 = a.SVb + ((size_t)bh * sh.NC + c1) * M * D;
        load_tile_async<D>(q, tbase, nq, X0);
        load_tile_async<D>(k, j0, nq, KB[0]);
        load_tile_async<D>(v, j0, nq, VB[0]);
        load_state_pair_async<D, M>(SK1, has2 ? SK1 + M * D : nullptr, KB[1]);
        cp_async_commit();
        float lg[HM], b[HM], rho[HM];
        row_gates<M>(a.la + (hoff + j0 + r) * M, row_ok, lg, b, s_tot, sG, warp, lane, h, r, nq);
        {
            float ek[HM];
#pragma unroll
            for (int jj = 0; jj < HM; jj++) {
                rho[jj] = 0.5f * sG[cr * M + h * HM + jj];
                ek[jj] = row_ok ? fexp(rho[jj] - b[jj]) * (-expm1f(lg[jj])) : 0.0f;
            }
            store_row(VB[1], r, h * HM, ek, HM);
        }
        cp_async_wait<0>();
        sync_for_mma();
        if (tid == 0) {
            const uint32_t s0 = smem_u32(X0), s1 = smem_u32(KB[0]), s3 = smem_u32(KB[1]);
            for (int kk = 0; kk < D / 16; kk++)
                mma_bf16(tm + tA, desc_k(s0, 128, kk), desc_k(s1, 128, kk), idesc_bf16(128, 128, false), kk > 0);
            for (int kk = 0; kk < D / 16; kk++)
                mma_bf16(tm + tO, desc_k(s0, 128, kk), desc_k(s3, 2 * M, kk), idesc_bf16(128, 2 * M, false), kk > 0);
            mma_commit(&bar);
        }
        ok = ctl.wait();
        if (ok) {
            // A = Q K_c^T masked to the row's own chunk and s <= r; [S^V] replaces [S^K]
            mask_to_tile(tl + tA, KB[0], r, h, cr, row_ok, false);
            load_state_pair_async<D, M>(SV1, has2 ? SV1 + M * D : nullptr, KB[1]);
            cp_async_commit();
            sync_for_mma();
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
            __syncthreads();
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
            __syncthreads();
            l = reds[r] + reds[128 + r];
            cp_async_wait<0>();  // [S^V] pair
            sync_for_mma();
            if (tid == 0) {
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
            sync_for_mma();
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

    // ---- window branch over the band of keys [tbase - w + 1, tbase + nq - 1],
    // key/value blocks double-buffered: block i + 1 loads while block i computes
    if (ok && sh.w > 0) {
        const int klo = max(0, tbase - sh.w + 1), khi = tbase + nq - 1;
        const int nb = (khi - klo) / 128 + 1;
        const int t = tbase + r;
        load_tile_async<D>(qr, tbase, nq, X0);
        load_tile_async<D>(kr, klo, min(128, khi - klo + 1), KB[0]);
        load_tile_async<D>(v, klo, min(128, khi - klo + 1), VB[0]);
        cp_async_commit();
        auto issue_s = [&](int i) {
            const uint32_t s0 = smem_u32(X0), s1 = smem_u32(KB[i & 1]);
            for (int kk = 0; kk < D / 16; kk++)
                mma_bf16(tm + tA, desc_k(s0, 128, kk), desc_k(s1, 128, kk), idesc_bf16(128, 128, false), kk > 0);
        };
        cp_async_wait<0>();
        sync_for_mma();
        if (tid == 0) {
            issue_s(0);
            mma_commit(&bar);
        }
        // One wait per block: the commit after block i's S also covers block
        // i - 1's P V, issued just before it.
        for (int i = 0; i < nb && ok; i++) {
            const int kb = klo + i * 128, nk = min(128, khi - kb + 1), cur = i & 1;
            ok = ctl.wait();
            if (!ok) break;
            if (i + 1 < nb) {  // stage of block i - 1, whose P V is complete
                const int kn = kb + 128, nn = min(128, khi - kn + 1);
                load_tile_async<D>(kr, kn, nn, KB[cur ^ 1]);
                load_tile_async<D>(v, kn, nn, VB[cur ^ 1]);
                cp_async_commit();
            }
            float sv[64];
            tmem_ld(tl + tA + 64 * h, sv, 64);
            float bm = -INFINITY;
            // valid keys of this row: columns [clo, chi] of the block
            const int clo = max(0, t - sh.w + 1 - kb) - 64 * h;
            const int chi = (row_ok ? min(nk - 1, t - kb) : -1) - 64 * h;
#pragma unroll
            for (int jj = 0; jj < 64; jj++) {
                sv[jj] = (jj >= clo && jj <= chi) ? sv[jj] * sig2 : -INFINITY;
                bm = fmaxf(bm, sv[jj]);
            }
            redm[h * 128 + r] = bm;
            __syncthreads();
            bm = fmaxf(redm[r], redm[128 + r]);
            const float mnew = fmaxf(m, bm);
            bool resc = false;
            float scale = 1.0f;
            if (!o_valid || m == -INFINITY) {
                m = mnew;
            } else if (mnew > m + 8.0f) {
                resc = true;
                scale = ex2(m - mnew);
                m = mnew;
                l *= scale;
            }
            if (o_valid && __any_sync(0xffffffffu, resc)) {
                for (int c0 = 0; c0 < HD; c0 += 32) {
                    float ov[32];
                    tmem_ld32(tl + tO + h * HD + c0, ov);
#pragma unroll
                    for (int jj = 0; jj < 32; jj++) ov[jj] *= scale;
                    tmem_st32(tl + tO + h * HD + c0, ov);
                }
            }
            float ps = 0.0f;
#pragma unroll
            for (int jj = 0; jj < 64; jj++) {
                const float p = (m == -INFINITY) ? 0.0f : ex2(sv[jj] - m);
                sv[jj] = p;
                ps += p;
            }
            reds[h * 128 + r] = ps;
            store_row(KB[cur], r, 64 * h, sv, 64);
            if (i + 1 < nb) cp_async_wait<0>();
            sync_for_mma();
            l += reds[r] + reds[128 + r];
            if (tid == 0) {
                const uint32_t s1 = smem_u32(KB[cur]), s2 = smem_u32(VB[cur]);
                for (int kk = 0; kk < 8; kk++)
                    mma_bf16(tm + tO, desc_k(s1, 128, kk), desc_mn(s2, 128, kk), idesc_bf16(128, D, true),
                             (o_valid || kk > 0) ? 1u : 0u);
                if (i + 1 < nb) issue_s(i + 1);
                mma_commit(&bar);
            }
            o_valid = true;
        }
        if (ok) ok = ctl.wait();  // the last block's P V
        cp_async_wait<0>();
    }

    // ---- epilogue: o = O / l, lse = m ln2 + log l
    if (ok) {
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
        const int t = tbase + r;
        __nv_bfloat16* orow = (__nv_bfloat16*)a.o + (hoff + t) * D;
        for (int c0 = 0; c0 < HD; c0 += 32) {
            float ov[32];
            tmem_ld32(tl + tO + h * HD + c0, ov);
            if (row_ok) {
#pragma unroll
                for (int jj = 0; jj < 32; jj++) ov[jj] *= inv;
#pragma unroll
                for (int qq = 0; qq < 4; qq++)
                    *reinterpret_cast<uint4*>(orow + h * HD + c0 + qq * 8) = pack8(ov + qq * 8);
            }
        }
        if (h == 0 && row_ok) a.lse[hoff + t] = m * kLn2 + logf(l);
    } else if (h == 0 && row_ok) {
        a.lse[hoff + tbase + r] = __int_as_float(0x7fc00000);  // NaN marks the failed tile
    }
    if (!ok && tid == 0) mbar_wait(&bar, ctl.phase ^ 1u, kWaitCycles);  // let in-flight MMAs drain
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 256);
}

// RoPE applied once per call: qr = RoPE(q), kr = RoPE(k) at absolute positions.
template <int D>
__global__ void __launch_bounds__(256)
rope_qk_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
               __nv_bfloat16* __restrict__ qr, __nv_bfloat16* __restrict__ kr, const float2* __restrict__ tab,
               long rows, int T) {
    constexpr int H = D / 2, CHH = D / 16;
    const long e = (long)blockIdx.x * 256 + threadIdx.x;
    if (e >= rows * CHH) return;
    const long row = e / CHH;
    const int ch = (int)(e % CHH), pos = (int)(row % T);
    const float2* cs = tab + (size_t)pos * H + ch * 8;
#pragma unroll
    for (int which = 0; which < 2; which++) {
        const __nv_bfloat16* src = (which == 0 ? q : k) + row * D;
        __nv_bfloat16* dst = (which == 0 ? qr : kr) + row * D;
        float x[8], y[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(src + ch * 8)), x);
        unpack8(__ldg(reinterpret_cast<const uint4*>(src + H + ch * 8)), y);
        rotate8(x, y, cs);
        *reinterpret_cast<uint4*>(dst + ch * 8) = pack8(x);
        *reinterpret_cast<uint4*>(dst + H + ch * 8) = pack8(y);
    }
}

template <int D>
cudaError_t launch_rope_qk(const void* q, const void* k, __nv_bfloat16* qr, __nv_bfloat16* kr, const float2* tab,
                           const Shape& sh, cudaStream_t st) {
    const long rows = (long)sh.BH * sh.T, n = rows * (D / 16);
    NHA_LAUNCH("rope_qk", st,
               rope_qk_kernel<D><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(
                   (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, qr, kr, tab, rows, sh.T));
    return cudaGetLastError();
}
template cudaError_t launch_rope_qk<64>(const void*, const void*, __nv_bfloat16*, __nv_bfloat16*, const float2*,
                                        const Shape&, cudaStream_t);
template cudaError_t launch_rope_qk<128>(const void*, const void*, __nv_bfloat16*, __nv_bfloat16*, const float2*,
                                         const Shape&, cudaStream_t);

cudaError_t launch_rope_table(float2* tab, int T, int H2, const RopeTab& rt, cudaStream_t st) {
    const int n = T * H2;
    NHA_LAUNCH("rope_table", st, rope_table_kernel<<<(n + 255) / 256, 256, 0, st>>>(tab, T, H2, rt));
    return cudaGetLastError();
}

template <int D, int M>
size_t tc_fwd_smem() {
    return 1024 + 128 * D * 2 + 4 * 32768 + sizeof(float) * (6 * M + 512);
}

template <int D, int M>
cudaError_t tc_forward(const FwdArgs& a, float2* tab, __nv_bfloat16* qr, __nv_bfloat16* kr, int* status,
                       cudaStream_t st) {
    const Shape& sh = a.sh;
    cudaError_t e = tc_states<D, M>((const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v, a.la, a.SK, a.SV,
                                    a.SKb, a.SVb, a.G, sh, status, st);
    if (e != cudaSuccess) return e;
    e = launch_rope_table(tab, sh.T, D / 2, a.rope, st);
    if (e != cudaSuccess) return e;
    if (sh.w > 0 && (e = launch_rope_qk<D>(a.q, a.k, qr, kr, tab, sh, st)) != cudaSuccess) return e;
    const int W0 = sh.T - sh.R;
    const int tiles = (W0 + 127) / 128 + (sh.R + 127) / 128;
    const size_t sm = tc_fwd_smem<D, M>();
    auto kern = fwd_tc_kernel<D, M>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    if (tiles > 0)
        NHA_LAUNCH("fwd_tc", st, kern<<<dim3(tiles, sh.BH), kTcThreads, sm, st>>>(a, qr, kr, status));
    return cudaGetLastError();
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
