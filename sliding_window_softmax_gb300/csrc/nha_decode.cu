// Recurrent decode step: one new token t per head ("Native Hybrid Attention for
// Efficient Sequence Modeling", Paper-Notes page, 关键设计/层内混合: the K^long
// recurrence, the token shift into the long memory and o_t, for a single
// query; section 局限 names this recurrent mode as the part left unoptimised).
// Matrix-vector work bound by the reads of the slot states and the ring, so
// SIMT, organised around keeping enough of those reads in flight.
//
// One thread-block cluster of ks CTAs (1..8) per head.  A CTA's 256 threads
// form groups of D/8 lanes; a lane owns 8 elements of every d-vector: i and
// i + d/2 for i in [4j, 4j + 4), j its index in the group, so each rotate-half
// pair of RoPE sits in one lane.  The head's items, slot rows (when a token
// leaves the window) and window tokens s in [max(0, t-w+1), t-1], are dealt
// round-robin over the cluster's groups.  Every lane streams its own pieces of
// its group's next items from global memory into its own shared-memory stages
// with cp.async, kDecStages items deep, so no lane waits on another's copy and
// the SM keeps tens of KB of reads in flight.  A slot item absorbs the
// leaving token into the row (written back in place) and scores it.  A window
// item scores the raw key: with pairs taken as complex numbers, the rotary
// logit RoPE(q, t) . RoPE(k_s, s) = Re(k_s conj(W_s)), W_s = RoPE(q, t) e^{-i theta s},
// and W advances from one of the group's tokens to the next (positions step
// by a constant) by one complex product, re-seeded exactly every kReseed
// items.  Each group runs an online softmax in base 2 with its lanes' share of
// the output; the groups of a CTA merge in shared memory, the CTAs of the
// cluster through distributed shared memory.
#include <cooperative_groups.h>
#include <stdlib.h>

#include "nha_common.cuh"
#include "nha_decode.h"
#include "nha_prof.h"

namespace cg = cooperative_groups;

namespace nha {

namespace {
constexpr int kDecThreads = 256;
constexpr int kDecStages = 6;  // pipeline entries a lane has in flight or ready
constexpr int kReseed = 16;    // window items between exact cos/sin evaluations
constexpr int kPieces = 2;     // 16-byte shared-memory pieces per lane and stage

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
template <int BYTES>
__device__ __forceinline__ void cp_async(void* smem, const void* gmem) {
    if constexpr (BYTES == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2;\n" ::"r"(smem_u32(smem)), "l"(gmem), "n"(BYTES)
                     : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// 4 consecutive elements as fp32
__device__ __forceinline__ void load4(const float4* p, float (&x)[4]) {
    const float4 v = *p;
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void load4(const uint2* p, float (&x)[4]) {
    const uint2 v = *p;
    x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xffff0000u);
    x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xffff0000u);
}
template <typename Tin>
struct Vec4;  // 4 elements of Tin
template <>
struct Vec4<float> { using T = float4; };
template <>
struct Vec4<__nv_bfloat16> { using T = uint2; };

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// 2^x (the MUFU approximation, relative error below 2^-22; ex2(-inf) = 0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// Programmatic dependent launch: wait until the grids this one depends on
// have finished and their writes are visible; let the next launch start.
__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

template <int GL>
__device__ __forceinline__ float group_sum(float x, unsigned mask) {
#pragma unroll
    for (int off = GL / 2; off > 0; off >>= 1) x += __shfl_xor_sync(mask, x, off);
    return x;
}
}  // namespace

template <typename Tin, int D, int M>
__global__ void __launch_bounds__(kDecThreads, 4) decode_step_kernel(const DecodeArgs a) {
    constexpr int H2 = D / 2, GL = D / 8, NG = kDecThreads / GL;
    using V4 = typename Vec4<Tin>::T;
    extern __shared__ float4 stage[];  // [kDecStages][kPieces][kDecThreads]; later the groups' partials
    __shared__ float sq[D], sqr[D], skj[D], svj[D], slj[M];
    __shared__ Tin tk[D], tv[D];  // token t's k, v (raw), its log_alpha
    __shared__ float tla[M];
    __shared__ float2 cst[H2];  // cos, sin at position t
    __shared__ float2 gst[H2];  // e^{-i theta G}: the rotation between a group's consecutive tokens
    __shared__ float gmx[NG], gsum[NG];
    __shared__ float bm, bs, bacc[D];  // this CTA's merged partial, read by the cluster
    cg::cluster_group cl = cg::this_cluster();
    const int ks = (int)cl.num_blocks(), rank = (int)cl.block_rank();
    const int tid = threadIdx.x, grp = tid / GL, j = tid % GL, lane = tid & 31;
    const unsigned gmask = (GL == 32 ? 0xffffffffu : ((1u << GL) - 1u) << (lane / GL * GL));
    const int bh = blockIdx.x / ks;
    const int g = rank * NG + grp, G = ks * NG;
    // Launched as a programmatic dependent of the kernel before it on the
    // stream: nothing that kernel may write is read before grid_wait().  With
    // `overlap` (positions and windows from the host, and the caller's word
    // that the earlier kernel writes none of this call's states and ring) the
    // first stages of states and ring are requested before the wait.
    const bool early = a.overlap && a.tpos == nullptr && a.wvec == nullptr;
    if (!early) grid_wait();
    const int t = a.tpos ? a.tpos[bh / a.H] : a.t;
    const int w = a.wvec ? a.wvec[bh % a.H] : a.w;  // this head's window
    const int wr = w > 0 ? w : 1;                    // ring entries the head cycles through
    const size_t wst = a.w > 0 ? a.w : 1;            // ring entries per head in memory
    // a position or window outside the supported range: NaN out, state untouched
    if (t < 0 || t >= (1 << 18) || w < 0 || w > a.w) {
        if (early) grid_wait();
        grid_launch_dependents();
        for (int e = rank * (D / ks) + tid; e < (rank + 1) * (D / ks); e += kDecThreads)
            ((Tin*)a.o)[(size_t)bh * D + e] = from_f<Tin>(__int_as_float(0x7fc00000));
        return;  // every CTA of the cluster serves this head and returns here, before any cluster barrier
    }
    const float scale = rsqrtf((float)D);
    const bool absorb = t - w >= 0;
    const int eo = absorb && w > 0 ? (t - w) % w : 0;  // ring entry of the token that leaves
    const int s_lo = max(0, t - w + 1);                 // first window token
    const int nwin = max(0, t - s_lo);                  // window tokens before t

    const Tin* q = (const Tin*)a.q + (size_t)bh * D;
    const Tin* k = (const Tin*)a.k + (size_t)bh * D;
    const Tin* v = (const Tin*)a.v + (size_t)bh * D;
    const float* la = a.la + (size_t)bh * M;
    const Tin* rk = (const Tin*)a.ring_k + (size_t)bh * wst * D;
    const Tin* rv = (const Tin*)a.ring_v + (size_t)bh * wst * D;
    float* SK = a.SK + (size_t)bh * M * D;
    float* SV = a.SV + (size_t)bh * M * D;

    // ---- this group's items: slot rows g, g + G, ... then window tokens s_lo + g, s_lo + g + G, ...
    // Each item streams through the lane's stages as pipeline entries of two
    // 16-byte pieces: a slot row as two entries (its S^K pieces, then its S^V
    // pieces), a bf16 window token as one entry (k lo|hi, then v lo|hi, 8 bytes
    // each), an fp32 window token as two (k lo, k hi; then v lo, v hi).
    constexpr int EW = sizeof(Tin) == 2 ? 1 : 2;  // entries of a window token
    const int ns = absorb && g < M ? (M - g + G - 1) / G : 0;
    const int nw = g < nwin ? (nwin - g + G - 1) / G : 0;
    const int n_entries = 2 * ns + EW * nw;
    // issue cursor: the next entry, its stage and (window part) ring entry
    int i_en = 0, i_stage = 0, i_ring = (s_lo + g) % wr;
    const int ring_step = G % wr;
    // issue the next entry (if any) as its own commit group: every call commits
    // one group, so "entry n complete" is "all but the last (issued - n - 1) groups"
    auto issue_commit = [&]() {
        if (i_en < n_entries) {
            float4* st = stage + (size_t)i_stage * kPieces * kDecThreads + tid;
            if (i_en < 2 * ns) {
                const int i = g + G * (i_en >> 1);
                const float* src = ((i_en & 1) ? SV : SK) + (size_t)i * D + 4 * j;
                cp_async<16>(st, src);
                cp_async<16>(st + kDecThreads, src + H2);
            } else {
                const size_t e = (size_t)i_ring * D + 4 * j;
                const int x = i_en - 2 * ns;
                if constexpr (EW == 1) {
                    char* b = reinterpret_cast<char*>(st);
                    cp_async<8>(b, rk + e);
                    cp_async<8>(b + 8, rk + e + H2);
                    cp_async<8>(b + 16 * kDecThreads, rv + e);
                    cp_async<8>(b + 16 * kDecThreads + 8, rv + e + H2);
                } else {
                    const Tin* src = (x & 1) ? rv : rk;
                    cp_async<16>(st, src + e);
                    cp_async<16>(st + kDecThreads, src + e + H2);
                }
                if (EW == 1 || (x & 1)) {  // the token's last entry: on to the group's next token
                    i_ring += ring_step;
                    if (i_ring >= wr) i_ring -= wr;
                }
            }
            i_en++;
            i_stage = i_stage + 1 == kDecStages ? 0 : i_stage + 1;
        }
        cp_async_commit();
    };
#pragma unroll
    for (int x = 0; x < kDecStages - 1; x++) issue_commit();

    // ---- cos/sin at t and G, and the token that leaves the window when it
    // comes from the ring (none of it from the earlier kernel, so before the
    // wait when the launch overlaps)
    for (int i = tid; i < H2; i += kDecThreads) {
        float c, sn;
        rope_cs(a.rope, t, i, c, sn);
        cst[i] = make_float2(c, sn);
        rope_cs(a.rope, G, i, c, sn);
        gst[i] = make_float2(c, -sn);
    }
    if (absorb && w > 0) {
        for (int e = tid; e < D; e += kDecThreads) {
            skj[e] = to_f(rk[(size_t)eo * D + e]);
            svj[e] = to_f(rv[(size_t)eo * D + e]);
        }
        for (int i = tid; i < M; i += kDecThreads) slj[i] = a.ring_la[((size_t)bh * wst + eo) * M + i];
    }
    if (early) grid_wait();
    grid_launch_dependents();  // the next launch may start; it waits for this grid to finish

    // ---- q, RoPE(q, t), token t's k, v, log_alpha (the leaving token too when w = 0)
    for (int e = tid; e < D; e += kDecThreads) {
        const Tin ke = k[e], ve = v[e];
        tk[e] = ke;
        tv[e] = ve;
        if (absorb && w == 0) {
            skj[e] = to_f(ke);
            svj[e] = to_f(ve);
        }
    }
    for (int i = tid; i < M; i += kDecThreads) {
        const float l = la[i];
        tla[i] = l;
        if (absorb && w == 0) slj[i] = l;
    }
    for (int i = tid; i < H2; i += kDecThreads) {
        const float x = to_f(q[i]), y = to_f(q[i + H2]);
        const float2 cs = cst[i];  // written by this thread above
        sq[i] = x;
        sq[i + H2] = y;
        sqr[i] = x * cs.x - y * cs.y;
        sqr[i + H2] = y * cs.x + x * cs.y;
    }
    __syncthreads();

    // the lane's elements: lo = 4j .. 4j+3, hi = d/2 + 4j .. d/2 + 4j+3
    constexpr float kLog2e = 1.4426950408889634f;
    const float l2scale = scale * kLog2e;  // logits in base-2 units
    float mx = -INFINITY, sum = 0.0f, acc[8];
#pragma unroll
    for (int f = 0; f < 8; f++) acc[f] = 0.0f;
    auto push = [&](float l, const float (&vl)[4], const float (&vh)[4]) {
        if (l > mx) {  // uniform in the group (every lane holds the group's sum)
            const float sc = ex2(mx - l);
            sum *= sc;
#pragma unroll
            for (int f = 0; f < 8; f++) acc[f] *= sc;
            mx = l;
        }
        const float p = ex2(l - mx);
        sum += p;
#pragma unroll
        for (int f = 0; f < 4; f++) {
            acc[f] = fmaf(p, vl[f], acc[f]);
            acc[4 + f] = fmaf(p, vh[f], acc[4 + f]);
        }
    };
    // W = RoPE(q, t) e^{-i theta s} of the group's current token
    float wre[4], wim[4];

    int c_stage = 0;  // stage of the next entry to consume
    auto stage_at = [&](int ahead) {
        const int x = c_stage + ahead;
        return stage + (size_t)(x >= kDecStages ? x - kDecStages : x) * kPieces * kDecThreads + tid;
    };
    auto advance = [&](int n) {
        c_stage += n;
        if (c_stage >= kDecStages) c_stage -= kDecStages;
    };
    // ---- slot rows: absorb token t - w with its own gate, then L_i = q . S^K[i] / sqrt(d)
    for (int r = 0; r < ns; r++) {
        cp_async_wait<kDecStages - 3>();  // the row's S^K and S^V entries
        const int i = g + G * r;
        const float al = expf(slj[i]), u = -expm1f(slj[i]);
        float kl[4], kh[4], vl[4], vh[4];
        load4(stage_at(0), kl);
        load4(stage_at(0) + kDecThreads, kh);
        load4(stage_at(1), vl);
        load4(stage_at(1) + kDecThreads, vh);
        advance(2);
        float dot = 0.0f;
#pragma unroll
        for (int f = 0; f < 4; f++) {
            kl[f] = al * kl[f] + u * skj[4 * j + f];
            kh[f] = al * kh[f] + u * skj[H2 + 4 * j + f];
            vl[f] = al * vl[f] + u * svj[4 * j + f];
            vh[f] = al * vh[f] + u * svj[H2 + 4 * j + f];
            dot += sq[4 * j + f] * kl[f] + sq[H2 + 4 * j + f] * kh[f];
        }
        float* dk = SK + (size_t)i * D + 4 * j;
        float* dv = SV + (size_t)i * D + 4 * j;
        *(float4*)dk = make_float4(kl[0], kl[1], kl[2], kl[3]);
        *(float4*)(dk + H2) = make_float4(kh[0], kh[1], kh[2], kh[3]);
        *(float4*)dv = make_float4(vl[0], vl[1], vl[2], vl[3]);
        *(float4*)(dv + H2) = make_float4(vh[0], vh[1], vh[2], vh[3]);
        push(group_sum<GL>(dot, gmask) * l2scale, vl, vh);
        issue_commit();
        issue_commit();
    }
    // ---- window tokens, two per iteration: Re(k_s conj(W_s)) / sqrt(d)
    int reseed = 0;  // items until the next exact evaluation of W
    for (int r = 0; r < nw; r += 2) {
        const bool two = r + 1 < nw;
        cp_async_wait<kDecStages - 1 - 2 * EW>();  // both tokens' entries (a missing one's groups are empty)
        if (reseed == 0) {
            const int s = s_lo + g + G * r;
#pragma unroll
            for (int f = 0; f < 4; f++) {
                float c, sn;
                rope_cs(a.rope, s, 4 * j + f, c, sn);
                const float ql = sqr[4 * j + f], qh = sqr[H2 + 4 * j + f];
                wre[f] = ql * c + qh * sn;
                wim[f] = qh * c - ql * sn;
            }
            reseed = kReseed;
        }
        reseed -= 2;
        float k1l[4], k1h[4], k2l[4], k2h[4], v1l[4], v1h[4], v2l[4], v2h[4];
        if constexpr (EW == 1) {
            const char* b1 = reinterpret_cast<const char*>(stage_at(0));
            const char* b2 = reinterpret_cast<const char*>(stage_at(1));
            load4((const V4*)b1, k1l);
            load4((const V4*)(b1 + 8), k1h);
            load4((const V4*)b2, k2l);
            load4((const V4*)(b2 + 8), k2h);
        } else {
            load4((const V4*)stage_at(0), k1l);
            load4((const V4*)(stage_at(0) + kDecThreads), k1h);
            load4((const V4*)stage_at(2), k2l);
            load4((const V4*)(stage_at(2) + kDecThreads), k2h);
        }
        float d1 = 0.0f, d2 = 0.0f;
#pragma unroll
        for (int f = 0; f < 4; f++) {
            const float2 gs = gst[4 * j + f];
            d1 = fmaf(k1l[f], wre[f], fmaf(k1h[f], wim[f], d1));
            float re = wre[f] * gs.x - wim[f] * gs.y;
            float im = wre[f] * gs.y + wim[f] * gs.x;
            d2 = fmaf(k2l[f], re, fmaf(k2h[f], im, d2));
            wre[f] = re * gs.x - im * gs.y;
            wim[f] = re * gs.y + im * gs.x;
        }
#pragma unroll
        for (int off = GL / 2; off > 0; off >>= 1) {
            d1 += __shfl_xor_sync(gmask, d1, off);
            d2 += __shfl_xor_sync(gmask, d2, off);
        }
        if constexpr (EW == 1) {
            const char* b1 = reinterpret_cast<const char*>(stage_at(0) + kDecThreads);
            const char* b2 = reinterpret_cast<const char*>(stage_at(1) + kDecThreads);
            load4((const V4*)b1, v1l);
            load4((const V4*)(b1 + 8), v1h);
            load4((const V4*)b2, v2l);
            load4((const V4*)(b2 + 8), v2h);
        } else {
            load4((const V4*)stage_at(1), v1l);
            load4((const V4*)(stage_at(1) + kDecThreads), v1h);
            load4((const V4*)stage_at(3), v2l);
            load4((const V4*)(stage_at(3) + kDecThreads), v2h);
        }
        advance(2 * EW);
        // one online-softmax update for both (a missing second token weighs 0)
        const float l1 = d1 * l2scale, l2 = two ? d2 * l2scale : -INFINITY;
        const float mn = fmaxf(mx, fmaxf(l1, l2));
        const float sc = ex2(mx - mn), p1 = ex2(l1 - mn), p2 = ex2(l2 - mn);
        sum = fmaf(sum, sc, p1 + p2);
#pragma unroll
        for (int f = 0; f < 4; f++) {
            const float b2l = two ? v2l[f] : 0.0f, b2h = two ? v2h[f] : 0.0f;
            acc[f] = fmaf(acc[f], sc, fmaf(p1, v1l[f], p2 * b2l));
            acc[4 + f] = fmaf(acc[4 + f], sc, fmaf(p1, v1h[f], p2 * b2h));
        }
        mx = mn;
#pragma unroll
        for (int x = 0; x < 2 * EW; x++) issue_commit();
    }
    cp_async_wait<0>();
    // ---- token t itself (window, relative position 0), by group 0 of the cluster
    if (g == 0 && w > 0) {
        float vl[4], vh[4], d0 = 0.0f;
#pragma unroll
        for (int f = 0; f < 4; f++) {
            const float x = to_f(tk[4 * j + f]), y = to_f(tk[H2 + 4 * j + f]);
            vl[f] = to_f(tv[4 * j + f]);
            vh[f] = to_f(tv[H2 + 4 * j + f]);
            const float2 cs = cst[4 * j + f];
            d0 += sqr[4 * j + f] * (x * cs.x - y * cs.y) + sqr[H2 + 4 * j + f] * (y * cs.x + x * cs.y);
        }
        push(group_sum<GL>(d0, gmask) * l2scale, vl, vh);
    }
    // ---- merge the groups of this CTA (their accumulators reuse the stages)
    __syncthreads();
    float* gacc = reinterpret_cast<float*>(stage);  // [NG][D]
    if (j == 0) {
        gmx[grp] = mx;
        gsum[grp] = sum;
    }
#pragma unroll
    for (int f = 0; f < 4; f++) {
        gacc[grp * D + 4 * j + f] = acc[f];
        gacc[grp * D + H2 + 4 * j + f] = acc[4 + f];
    }
    __syncthreads();
    {
        float m = -INFINITY;
        for (int x = 0; x < NG; x++) m = fmaxf(m, gmx[x]);
        for (int e = tid; e < D; e += kDecThreads) {
            float r = 0.0f;
            for (int x = 0; x < NG; x++)
                if (gmx[x] != -INFINITY) r += gacc[x * D + e] * ex2(gmx[x] - m);
            bacc[e] = r;
        }
        if (tid == 0) {
            float tot = 0.0f;
            for (int x = 0; x < NG; x++)
                if (gmx[x] != -INFINITY) tot += gsum[x] * ex2(gmx[x] - m);
            bm = m;
            bs = tot;
        }
    }
    // every CTA of the cluster has read the leaving token and published its partial
    cl.sync();
    // token t takes the ring entry of the token that left; the window keys
    // s < t read other entries
    if (w > 0 && rank == 0) {
        const int en = t % w;
        Tin* wk = (Tin*)a.ring_k + ((size_t)bh * wst + en) * D;
        Tin* wv = (Tin*)a.ring_v + ((size_t)bh * wst + en) * D;
        for (int e = tid; e < D; e += kDecThreads) {
            wk[e] = tk[e];
            wv[e] = tv[e];
        }
        for (int i = tid; i < M; i += kDecThreads) a.ring_la[((size_t)bh * wst + en) * M + i] = tla[i];
    }
    // ---- merge the cluster: CTA `rank` writes o[e] for e in its share of d.
    // Every remote read is issued at once: threads 0..ks-1 fetch the ranks'
    // (max, sum); thread (e, r) of the first D threads fetches rank r's
    // accumulator entry e, and the ks lanes of an e sum by shuffles.
    {
        __shared__ float rm[16], rs[16];
        if (tid < ks) {
            rm[tid] = *cl.map_shared_rank(&bm, tid);
            rs[tid] = *cl.map_shared_rank(&bs, tid);
        }
        __syncthreads();
        float mx = -INFINITY;
        for (int r = 0; r < ks; r++) mx = fmaxf(mx, rm[r]);
        float tot = 0.0f;
        for (int r = 0; r < ks; r++) tot += rm[r] == -INFINITY ? 0.0f : rs[r] * ex2(rm[r] - mx);
        const float inv = 1.0f / tot;  // tot >= 1: the largest logit contributes exp(0)
        const int per = D / ks;
        if (tid < D) {  // whole warps: D is a multiple of 32
            const int e = rank * per + tid / ks, r = tid % ks;
            float o = rm[r] == -INFINITY ? 0.0f : cl.map_shared_rank(bacc, r)[e] * ex2(rm[r] - mx);
            for (int off = ks / 2; off > 0; off >>= 1) o += __shfl_xor_sync(0xffffffffu, o, off);
            if (r == 0) ((Tin*)a.o)[(size_t)bh * D + e] = from_f<Tin>(o * inv);
        }
    }
    // keep this CTA's shared memory alive until the cluster has read it
    cl.sync();
}

constexpr size_t kDecSmem = (size_t)kDecStages * kPieces * kDecThreads * sizeof(float4);

// Cluster size: doubled, up to 8 (the portable limit), while the grid stays
// within one wave of resident CTAs and every group keeps at least four items.
// (With per-sequence positions the host does not know them: sized as if every
// window were full and a token leaving it.)
static int decode_cluster(const DecodeArgs& a, int m, int d, int resident) {
    const int t = a.tpos ? a.w + 1 : a.t;
    const int s_lo = t - a.w + 1 > 0 ? t - a.w + 1 : 0;
    const int items = (t - a.w >= 0 ? m : 0) + (t - s_lo > 0 ? t - s_lo : 0);
    const int groups = kDecThreads / (d / 8);
    int ks = 1;
    while (ks < 8 && (long long)a.BH * ks * 2 <= (long long)resident * a.sms && ks * 2 * groups * 4 <= items)
        ks *= 2;
    return ks;
}

template <typename Tin, int D, int M>
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
    if (a.BH == 0) return cudaSuccess;
    static_assert(kDecStages * kPieces * kDecThreads * sizeof(float4) >= (kDecThreads / (D / 8)) * D * sizeof(float),
                  "the group partials reuse the stages");
    auto kern = decode_step_kernel<Tin, D, M>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecSmem);
    if (e != cudaSuccess) return e;
    static const int resident = [&] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kDecThreads, kDecSmem) != cudaSuccess || n < 1)
            n = 1;
        return n;
    }();
    int ks = decode_cluster(a, M, D, resident);
    // tuning override of the cluster size (1, 2, 4, 8 or 16 CTAs per head; 16 is a non-portable cluster size)
    if (const char* env = getenv("NHA_DECODE_CLUSTER")) {
        const int v = atoi(env);
        if (v == 1 || v == 2 || v == 4 || v == 8 || v == 16) ks = v;
    }
    if (ks > 8 && (e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.BH * ks));
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = kDecSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // may start before the previous kernel on the stream has finished (the
    // kernel waits for it before touching anything it may write)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    NHA_LAUNCH("decode_step", st, e = cudaLaunchKernelEx(&cfg, kern, a));
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

#define NHA_DEC_INST(Tin, D, M) template cudaError_t launch_decode<Tin, D, M>(const DecodeArgs&, cudaStream_t);
NHA_DEC_INST(float, 64, 16)
NHA_DEC_INST(float, 64, 32)
NHA_DEC_INST(float, 64, 64)
NHA_DEC_INST(float, 128, 16)
NHA_DEC_INST(float, 128, 32)
NHA_DEC_INST(float, 128, 64)
NHA_DEC_INST(__nv_bfloat16, 64, 16)
NHA_DEC_INST(__nv_bfloat16, 64, 32)
NHA_DEC_INST(__nv_bfloat16, 64, 64)
NHA_DEC_INST(__nv_bfloat16, 128, 16)
NHA_DEC_INST(__nv_bfloat16, 128, 32)
NHA_DEC_INST(__nv_bfloat16, 128, 64)

}  // namespace nha
