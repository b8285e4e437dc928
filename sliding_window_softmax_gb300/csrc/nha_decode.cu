// Recurrent decode step: one new token t per head ("Native Hybrid Attention for
// Efficient Sequence Modeling", Paper-Notes page, 关键设计/层内混合: the K^long
// recurrence, the token shift into the long memory and o_t, for a single
// query; section 局限 names this recurrent mode as the part left unoptimised).
// Matrix-vector work bound by the state and ring reads, so SIMT.
//
// One thread-block cluster of ks CTAs (1..8) per head, 8 warps each.  The
// cluster's 8 ks warps share the head's work: warp g absorbs the leaving token
// into slot rows i = g, g + 8 ks, ... (fp32 read-modify-write, coalesced over
// the lanes) and scores them, and scores the window keys s0 + g, s0 + g + 8 ks,
// ..., each with an online softmax and an output accumulator in its lanes.
// Lane l holds the elements {l, l + 32, ...} of a d-vector, so a rotate-half
// pair (i, i + d/2) sits in one lane.  The warps of a CTA merge in shared
// memory, the CTAs of the cluster through distributed shared memory.
#include <cooperative_groups.h>

#include "nha_common.cuh"
#include "nha_decode.h"
#include "nha_prof.h"

namespace cg = cooperative_groups;

namespace nha {

namespace {
constexpr int kDecThreads = 256, kDecWarps = kDecThreads / 32;
constexpr int kDecBatch = 4;  // window keys a warp loads before it scores them

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Online softmax of one warp: running max and sum (same in every lane) and
// the lane's share of the output accumulator.
template <int E>
struct WarpSoftmax {
    float mx = -INFINITY, sum = 0.0f, acc[E];
    __device__ WarpSoftmax() {
#pragma unroll
        for (int e = 0; e < E; e++) acc[e] = 0.0f;
    }
    __device__ void push(float logit, const float (&val)[E]) {
        const float mn = fmaxf(mx, logit);
        const float sc = expf(mx - mn);  // 0 while mx = -inf
        const float p = expf(logit - mn);
        sum = sum * sc + p;
#pragma unroll
        for (int e = 0; e < E; e++) acc[e] = acc[e] * sc + p * val[e];
        mx = mn;
    }
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}
}  // namespace

template <typename Tin, int D, int M>
__global__ void __launch_bounds__(kDecThreads) decode_step_kernel(const DecodeArgs a) {
    constexpr int E = D / 32, H2 = D / 2;
    __shared__ float sq[D], sqr[D], skj[D], svj[D], slj[M];
    __shared__ float wm[kDecWarps], ws[kDecWarps], wacc[kDecWarps][D];
    __shared__ float bm, bs, bacc[D];  // this CTA's merged partial, read by the cluster
    cg::cluster_group cl = cg::this_cluster();
    const int ks = (int)cl.num_blocks(), rank = (int)cl.block_rank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x / ks;
    const int g = rank * kDecWarps + warp, G = ks * kDecWarps;
    const int t = a.t, w = a.w, wr = w > 0 ? w : 1;
    const float scale = rsqrtf((float)D);
    const bool absorb = t - w >= 0;
    const int eo = absorb && w > 0 ? (t - w) % w : 0;  // ring entry of the token that leaves

    const Tin* q = (const Tin*)a.q + (size_t)bh * D;
    const Tin* k = (const Tin*)a.k + (size_t)bh * D;
    const Tin* v = (const Tin*)a.v + (size_t)bh * D;
    const float* la = a.la + (size_t)bh * M;
    const Tin* rk = (const Tin*)a.ring_k + (size_t)bh * wr * D;
    const Tin* rv = (const Tin*)a.ring_v + (size_t)bh * wr * D;

    // ---- q, RoPE(q, t), and the token that leaves the window
    for (int e = tid; e < D; e += kDecThreads) {
        sq[e] = to_f(q[e]);
        if (absorb) {
            skj[e] = to_f(w > 0 ? rk[(size_t)eo * D + e] : k[e]);
            svj[e] = to_f(w > 0 ? rv[(size_t)eo * D + e] : v[e]);
        }
    }
    if (absorb)
        for (int i = tid; i < M; i += kDecThreads) slj[i] = w > 0 ? a.ring_la[((size_t)bh * wr + eo) * M + i] : la[i];
    for (int i = tid; i < H2; i += kDecThreads) {
        float c, s;
        rope_cs(a.rope, t, i, c, s);
        const float x = to_f(q[i]), y = to_f(q[i + H2]);
        sqr[i] = x * c - y * s;
        sqr[i + H2] = y * c + x * s;
    }
    __syncthreads();

    WarpSoftmax<E> sm;
    // ---- slots: absorb token t - w with its own gate, then L_i = q . S^K[i] / sqrt(d)
    if (absorb) {
        for (int i = g; i < M; i += G) {
            const float al = expf(slj[i]), u = -expm1f(slj[i]);
            float* sk = a.SK + ((size_t)bh * M + i) * D;
            float* sv = a.SV + ((size_t)bh * M + i) * D;
            float dot = 0.0f, val[E];
#pragma unroll
            for (int e = 0; e < E; e++) {
                const int c = lane + 32 * e;
                const float nk = al * sk[c] + u * skj[c];
                const float nv = al * sv[c] + u * svj[c];
                sk[c] = nk;
                sv[c] = nv;
                dot += sq[c] * nk;
                val[e] = nv;
            }
            sm.push(warp_sum(dot) * scale, val);
        }
    }
    // ---- window keys s in [max(0, t - w + 1), t]: RoPE(q, t) . RoPE(k_s, s) / sqrt(d)
    // (token t is read from the inputs, older ones from ring entry s mod w)
    const int s0 = max(0, t - w + 1);
    for (int base = s0 + g; base <= t; base += G * kDecBatch) {
        float kv[kDecBatch][E], vv[kDecBatch][E];
#pragma unroll
        for (int b = 0; b < kDecBatch; b++) {
            const int s = base + b * G;
            if (s <= t) {
                const Tin* ks_ = s == t ? k : rk + (size_t)(s % wr) * D;
                const Tin* vs_ = s == t ? v : rv + (size_t)(s % wr) * D;
#pragma unroll
                for (int e = 0; e < E; e++) {
                    kv[b][e] = to_f(ks_[lane + 32 * e]);
                    vv[b][e] = to_f(vs_[lane + 32 * e]);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < kDecBatch; b++) {
            const int s = base + b * G;
            if (s > t) break;
            float dot = 0.0f;
#pragma unroll
            for (int e = 0; e < E / 2; e++) {  // the pair (lane + 32 e, lane + 32 e + d/2)
                const int i = lane + 32 * e;
                float c, sn;
                rope_cs(a.rope, s, i, c, sn);
                const float x = kv[b][e], y = kv[b][e + E / 2];
                dot += sqr[i] * (x * c - y * sn) + sqr[i + H2] * (y * c + x * sn);
            }
            sm.push(warp_sum(dot) * scale, vv[b]);
        }
    }
    // ---- merge the warps of this CTA
    if (lane == 0) {
        wm[warp] = sm.mx;
        ws[warp] = sm.sum;
    }
#pragma unroll
    for (int e = 0; e < E; e++) wacc[warp][lane + 32 * e] = sm.acc[e];
    __syncthreads();
    {
        float mx = -INFINITY;
#pragma unroll
        for (int x = 0; x < kDecWarps; x++) mx = fmaxf(mx, wm[x]);
        float f[kDecWarps], tot = 0.0f;
#pragma unroll
        for (int x = 0; x < kDecWarps; x++) {
            f[x] = wm[x] == -INFINITY ? 0.0f : expf(wm[x] - mx);
            tot += ws[x] * f[x];
        }
        for (int e = tid; e < D; e += kDecThreads) {
            float r = 0.0f;
#pragma unroll
            for (int x = 0; x < kDecWarps; x++) r += wacc[x][e] * f[x];
            bacc[e] = r;
        }
        if (tid == 0) {
            bm = mx;
            bs = tot;
        }
    }
    // every CTA of the cluster has read the leaving token and published its partial
    cl.sync();
    // token t takes the ring entry of the token that left; the window keys
    // s < t read other entries
    if (w > 0 && rank == 0) {
        const int en = t % w;
        Tin* wk = (Tin*)a.ring_k + ((size_t)bh * wr + en) * D;
        Tin* wv = (Tin*)a.ring_v + ((size_t)bh * wr + en) * D;
        for (int e = tid; e < D; e += kDecThreads) {
            wk[e] = k[e];
            wv[e] = v[e];
        }
        for (int i = tid; i < M; i += kDecThreads) a.ring_la[((size_t)bh * wr + en) * M + i] = la[i];
    }
    // ---- merge the cluster: CTA `rank` writes o[e] for e in its share of d
    {
        float mx = -INFINITY;
        for (int r = 0; r < ks; r++) mx = fmaxf(mx, *cl.map_shared_rank(&bm, r));
        float tot = 0.0f;
        for (int r = 0; r < ks; r++) {
            const float mr = *cl.map_shared_rank(&bm, r);
            tot += mr == -INFINITY ? 0.0f : *cl.map_shared_rank(&bs, r) * expf(mr - mx);
        }
        const float inv = 1.0f / tot;  // tot >= 1: the largest logit contributes exp(0)
        const int per = D / ks;
        for (int e = rank * per + tid; e < (rank + 1) * per; e += kDecThreads) {
            float o = 0.0f;
            for (int r = 0; r < ks; r++) {
                const float mr = *cl.map_shared_rank(&bm, r);
                if (mr != -INFINITY) o += cl.map_shared_rank(bacc, r)[e] * expf(mr - mx);
            }
            ((Tin*)a.o)[(size_t)bh * D + e] = from_f<Tin>(o * inv);
        }
    }
    // keep this CTA's shared memory alive until the cluster has read it
    cl.sync();
}

// Cluster size: doubled, up to 8 (the portable limit), while the grid fits
// in one wave of four CTAs per SM (the register file holds four 256-thread
// CTAs at 64 registers) and every warp keeps at least one slot or key.
static int decode_cluster(const DecodeArgs& a, int m) {
    const int s0 = a.t - a.w + 1 > 0 ? a.t - a.w + 1 : 0;
    const int items = (a.t - a.w >= 0 ? m : 0) + (a.t - s0 + 1);
    int ks = 1;
    while (ks < 8 && (long long)a.BH * ks * 2 <= 4LL * a.sms && ks * 2 * kDecWarps <= items) ks *= 2;
    return ks;
}

template <typename Tin, int D, int M>
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
    if (a.BH == 0) return cudaSuccess;
    const int ks = decode_cluster(a, M);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.BH * ks));
    cfg.blockDim = dim3(kDecThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaSuccess;
    NHA_LAUNCH("decode_step", st, e = cudaLaunchKernelEx(&cfg, decode_step_kernel<Tin, D, M>, a));
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
