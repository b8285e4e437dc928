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
fwd_tc_kernel(const FwdArgs a, const float2* __restrict__ tab, int* __restrict__ status) {
    constexpr int HM = M / 2, HD = D / 2;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* X0 = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* X1 = X0 + 128 * D * 2;  // 32 KB
    unsigned char* X2 = X1 + 32768;        // 32 KB
    unsigned char* X3 = X2 + 32768;        // [2M][D]
    float* sB = reinterpret_cast<float*>(X3 + 2 * M * D * 2);  // [128][M]
    float* sU = sB + 128 * M;                                   // [128][M]
    float* sRho = sU + 128 * M;                                 // [2][M]
    float* redm = sRho + 2 * M;                                 // [2][128]
    float* reds = redm + 256;                                   // [2][128]
    __shared__ uint64_t bar;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const Shape sh = a.sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = ((warp & 3) << 5) | lane, h = warp >> 2;
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
    const size_t hoff = (size_t)bh * sh.T;
    const __nv_bfloat16* q = (const __nv_bfloat16*)a.q + hoff * D;
    const __nv_bfloat16* k = (const __nv_bfloat16*)a.k + hoff * D;
    const __nv_bfloat16* v = (const __nv_bfloat16*)a.v + hoff * D;
    const float sig2 = sh.sigma * kLog2e;

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
    const int cr = r >> 6;  // chunk of this row inside a slot tile (uniform per warp)

    if (slot) {
        const int c1 = j0 / kChunk;
        const bool has2 = nq > kChunk;
        load_tile<D>(q, tbase, nq, X0, nullptr);
        load_tile<D>(k, j0, nq, X1, nullptr);
        load_state_pair<D, M>(a.SK + ((size_t)bh * sh.NC + c1) * M * D,
                              has2 ? a.SK + ((size_t)bh * sh.NC + c1 + 1) * M * D : nullptr, X3);
        for (int e = tid; e < 128 * M; e += kTcThreads) {
            const int rr = e / M;
            const float lg = rr < nq ? a.la[(hoff + j0 + rr) * M + (e % M)] : 0.0f;
            sB[e] = lg;
            sU[e] = -expm1f(lg);
        }
        sync_for_mma();
        if (tid == 0) {
            const uint32_t s0 = smem_u32(X0), s1 = smem_u32(X1), s3 = smem_u32(X3);
            for (int kk = 0; kk < D / 16; kk++)
                mma_bf16(tm + tA, desc_k(s0, 128, kk), desc_k(s1, 128, kk), idesc_bf16(128, 128, false), kk > 0);
            for (int kk = 0; kk < D / 16; kk++)
                mma_bf16(tm + tO, desc_k(s0, 128, kk), desc_k(s3, 2 * M, kk), idesc_bf16(128, 2 * M, false), kk > 0);
            mma_commit(&bar);
        }
        // chunk-local inclusive cumsum of log_alpha, per slot (overlaps the MMAs)
        if (tid < 2 * M) {
            const int i = tid % M, cc = tid / M;
            const int r0 = cc * kChunk, r1 = min(nq, r0 + kChunk);
            float b = 0.0f;
            for (int rr = r0; rr < r1; rr++) {
                b += sB[rr * M + i];
                sB[rr * M + i] = b;
            }
            sRho[cc * M + i] = 0.5f * b;
        }
        __syncthreads();
        // Ek tile [128 s][M] in X2
        for (int e = tid; e < 128 * (M / 8); e += kTcThreads) {
            const int s = e / (M / 8), ch = e % (M / 8);
            float f[8];
#pragma unroll
            for (int jj = 0; jj < 8; jj++) {
                const int i = ch * 8 + jj;
                f[jj] = s < nq ? expf(sRho[(s >> 6) * M + i] - sB[s * M + i]) * sU[s * M + i] : 0.0f;
            }
            *reinterpret_cast<uint4*>(X2 + sw_chunk(s, ch, 128)) = pack8(f);
        }
        ok = ctl.wait();
        if (ok) {
            // A = Q K_c^T, masked to the row's own chunk and s <= r
            float vv[64];
            tmem_ld(tl + tA + 64 * h, vv, 64);
#pragma unroll
            for (int jj = 0; jj < 64; jj++) {
                const int col = 64 * h + jj;
                if (!(h == cr && col <= r && r < nq)) vv[jj] = 0.0f;
            }
            store_row(X1, r, 64 * h, vv, 64);
            // Sint (this row's chunk half) is kept in TMEM until the logits
            load_state_pair<D, M>(a.SV + ((size_t)bh * sh.NC + c1) * M * D,
                                  has2 ? a.SV + ((size_t)bh * sh.NC + c1 + 1) * M * D : nullptr, X3);
        }
        if (ok) {
            sync_for_mma();
            if (tid == 0) {
                const uint32_t s1 = smem_u32(X1), s2 = smem_u32(X2);
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
                const int i = h * HM + jj;
                const float bb = sB[r * M + i];
                const float eq = expf(bb - sRho[cr * M + i]);
                const float eb = expf(bb);
                L[jj] = (r < nq) ? sig2 * (eb * sint[jj] + eq * lin[jj]) : -INFINITY;
                mx = fmaxf(mx, L[jj]);
            }
            redm[h * 128 + r] = mx;
            __syncthreads();
            m = fmaxf(redm[r], redm[128 + r]);
            float ps = 0.0f, pe[HM], pq[HM];
#pragma unroll
            for (int jj = 0; jj < HM; jj++) {
                const int i = h * HM + jj;
                const float p = (m == -INFINITY) ? 0.0f : ex2(L[jj] - m);
                ps += p;
                const float bb = sB[r * M + i];
                pe[jj] = p * expf(bb);
                pq[jj] = p * expf(bb - sRho[cr * M + i]);
            }
            reds[h * 128 + r] = ps;
            // A_inter [128][2M] in X1: this row's chunk block holds p o Eb, the other block zero
            float z[HM];
#pragma unroll
            for (int jj = 0; jj < HM; jj++) z[jj] = 0.0f;
            store_row(X1, r, cr * M + h * HM, pe, HM);
            store_row(X1, r, (1 - cr) * M + h * HM, z, HM);
            // pEq [128][M] in the second half of X2 (after Ek; a 128-row swizzled
            // tile spans 16 KB whatever its width)
            store_row(X2 + 16384, r, h * HM, pq, HM);
            __syncthreads();
            l = reds[r] + reds[128 + r];
            sync_for_mma();
            if (tid == 0) {
                const uint32_t s1 = smem_u32(X1), s2 = smem_u32(X2), s3 = smem_u32(X3);
                for (int kk = 0; kk < 2 * M / 16; kk++)
                    mma_bf16(tm + tO, desc_k(s1, 128, kk), desc_mn(s3, 2 * M, kk), idesc_bf16(128, D, true), kk > 0);
                for (int kk = 0; kk < M / 16; kk++)
                    mma_bf16(tm + tA, desc_k(s2 + 16384, 128, kk), desc_k(s2, 128, kk),
                             idesc_bf16(128, 128, false), kk > 0);
                mma_commit(&bar);
            }
            ok = ctl.wait();
        }
        if (ok) {
            float vv[64];
            tmem_ld(tl + tA + 64 * h, vv, 64);
#pragma unroll
            for (int jj = 0; jj < 64; jj++) {
                const int col = 64 * h + jj;
                if (!(h == cr && col <= r && r < nq)) vv[jj] = 0.0f;
            }
            store_row(X1, r, 64 * h, vv, 64);
            load_tile<D>(v, j0, nq, X2, nullptr);
            sync_for_mma();
            if (tid == 0) {
                const uint32_t s1 = smem_u32(X1), s2 = smem_u32(X2);
                for (int kk = 0; kk < 8; kk++)
                    mma_bf16(tm + tO, desc_k(s1, 128, kk), desc_mn(s2, 128, kk), idesc_bf16(128, D, true), 1);
                mma_commit(&bar);
            }
            ok = ctl.wait();
            o_valid = true;
        }
        if (ok) rotate_tile<D>(X0, tbase, nq, tab);
    } else {
        load_tile<D>(q, tbase, nq, X0, tab);
    }

    // ---- window branch over the band of keys [tbase - w + 1, tbase + nq - 1]
    if (ok && sh.w > 0) {
        const int klo = max(0, tbase - sh.w + 1), khi = tbase + nq - 1;
        const int t = tbase + r;
        for (int kb = klo; kb <= khi && ok; kb += 128) {
            const int nk = min(128, khi - kb + 1);
            load_tile<D>(k, kb, nk, X1, tab);
            load_tile<D>(v, kb, nk, X2, nullptr);
            sync_for_mma();
            if (tid == 0) {
                const uint32_t s0 = smem_u32(X0), s1 = smem_u32(X1);
                for (int kk = 0; kk < D / 16; kk++)
                    mma_bf16(tm + tA, desc_k(s0, 128, kk), desc_k(s1, 128, kk), idesc_bf16(128, 128, false), kk > 0);
                mma_commit(&bar);
            }
            ok = ctl.wait();
            if (!ok) break;
            float sv[64];
            tmem_ld(tl + tA + 64 * h, sv, 64);
            float bm = -INFINITY;
#pragma unroll
            for (int jj = 0; jj < 64; jj++) {
                const int c = 64 * h + jj, key = kb + c;
                const bool valid = r < nq && c < nk && key <= t && key > t - sh.w;
                sv[jj] = valid ? sv[jj] * sig2 : -INFINITY;
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
            store_row(X1, r, 64 * h, sv, 64);
            sync_for_mma();
            l += reds[r] + reds[128 + r];
            if (tid == 0) {
                const uint32_t s1 = smem_u32(X1), s2 = smem_u32(X2);
                for (int kk = 0; kk < 8; kk++)
                    mma_bf16(tm + tO, desc_k(s1, 128, kk), desc_mn(s2, 128, kk), idesc_bf16(128, D, true),
                             (o_valid || kk > 0) ? 1u : 0u);
                mma_commit(&bar);
            }
            o_valid = true;
            ok = ctl.wait();
        }
    }

    // ---- epilogue: o = O / l, lse = m ln2 + log l
    if (ok) {
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
        const int t = tbase + r;
        __nv_bfloat16* orow = (__nv_bfloat16*)a.o + (hoff + t) * D;
        for (int c0 = 0; c0 < HD; c0 += 32) {
            float ov[32];
            tmem_ld32(tl + tO + h * HD + c0, ov);
            if (r < nq) {
#pragma unroll
                for (int jj = 0; jj < 32; jj++) ov[jj] *= inv;
#pragma unroll
                for (int qq = 0; qq < 4; qq++)
                    *reinterpret_cast<uint4*>(orow + h * HD + c0 + qq * 8) = pack8(ov + qq * 8);
            }
        }
        if (h == 0 && r < nq) a.lse[hoff + t] = m * kLn2 + logf(l);
    } else if (h == 0 && r < nq) {
        a.lse[hoff + tbase + r] = __int_as_float(0x7fc00000);  // NaN marks the failed tile
    }
    if (!ok && tid == 0) mbar_wait(&bar, ctl.phase ^ 1u, kWaitCycles);  // let in-flight MMAs drain
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 256);
}

cudaError_t launch_rope_table(float2* tab, int T, int H2, const RopeTab& rt, cudaStream_t st) {
    const int n = T * H2;
    NHA_LAUNCH("rope_table", st, rope_table_kernel<<<(n + 255) / 256, 256, 0, st>>>(tab, T, H2, rt));
    return cudaGetLastError();
}

template <int D, int M>
size_t tc_fwd_smem() {
    return 1024 + 128 * D * 2 + 32768 + 32768 + 2 * M * D * 2 + sizeof(float) * (2 * 128 * M + 2 * M + 512);
}

template <int D, int M>
cudaError_t tc_forward(const FwdArgs& a, float2* tab, int* status, cudaStream_t st) {
    const Shape& sh = a.sh;
    cudaError_t e = simt_states<__nv_bfloat16, D, M>((const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v,
                                                     a.la, a.SK, a.SV, a.G, sh, st);
    if (e != cudaSuccess) return e;
    e = launch_rope_table(tab, sh.T, D / 2, a.rope, st);
    if (e != cudaSuccess) return e;
    const int W0 = sh.T - sh.R;
    const int tiles = (W0 + 127) / 128 + (sh.R + 127) / 128;
    const size_t sm = tc_fwd_smem<D, M>();
    auto kern = fwd_tc_kernel<D, M>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    if (tiles > 0)
        NHA_LAUNCH("fwd_tc", st, kern<<<dim3(tiles, sh.BH), kTcThreads, sm, st>>>(a, tab, status));
    return cudaGetLastError();
}

#define NHA_TC_INST(D, M) template cudaError_t tc_forward<D, M>(const FwdArgs&, float2*, int*, cudaStream_t);
NHA_TC_INST(64, 16)
NHA_TC_INST(64, 32)
NHA_TC_INST(64, 64)
NHA_TC_INST(128, 16)
NHA_TC_INST(128, 32)
NHA_TC_INST(128, 64)

}  // namespace nha
