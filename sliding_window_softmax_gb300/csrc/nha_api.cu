// C-ABI layer of libnha: argument validation, workspace planning, RoPE
// frequency tables and the launch sequence on the caller's stream.
// Declarations and the full contract are in include/nha.h.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "nha.h"
#include "nha_decode.h"
#include "nha_kernels.h"
#include "nha_prefill.h"

namespace {

thread_local char g_err[512] = "";

nha_status_t fail(nha_status_t s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

nha_status_t ok() {
    g_err[0] = '\0';
    return NHA_OK;
}

// Host-side fault injection for tests: NHA_FAULT_INJECT=<site> makes the call
// fail with NHA_ERR_INTERNAL at that step, before anything is enqueued there.
bool inject(const char* site) {
    const char* e = getenv("NHA_FAULT_INJECT");
    return e != nullptr && strcmp(e, site) == 0;
}

constexpr int kMaxT = 1 << 18;

struct Plan {
    nha::Shape sh;
    int d, m;
    // workspace offsets, in floats
    size_t SK, SV, SKb, SVb, G, TAB, STATUS, QR, KR, HTB, HTF, Dv, Dhat, Dwin, dqwV, dqw, dkw, dvw, DL, PL, DB1, RK,
        RV, RKb, RVb, REND, LDL, LPL, total;
};

nha_status_t check_shape(int B, int H, int T, int d, int m, int w, int C, nha_dtype_t dt) {
    if (B < 0 || H < 0 || T < 0 || w < 0 || d <= 0 || m <= 0 || C <= 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "negative or zero size (B=%d H=%d T=%d d=%d m=%d w=%d C=%d)",
                    B, H, T, d, m, w, C);
    if (dt != NHA_DTYPE_F32 && dt != NHA_DTYPE_BF16)
        return fail(NHA_ERR_INVALID_ARGUMENT, "unknown dtype %d", (int)dt);
    if (d != 64 && d != 128) return fail(NHA_ERR_UNSUPPORTED, "head dim d=%d not in {64, 128}", d);
    if (m != 16 && m != 32 && m != 64) return fail(NHA_ERR_UNSUPPORTED, "slots m=%d not in {16, 32, 64}", m);
    if (C != nha::kChunk) return fail(NHA_ERR_UNSUPPORTED, "chunk C=%d unsupported (only %d)", C, nha::kChunk);
    if (T > kMaxT) return fail(NHA_ERR_UNSUPPORTED, "T=%d above the supported %d", T, kMaxT);
    long long elems = (long long)B * H * T * (d > m ? d : m);
    if (elems >= (1LL << 31)) return fail(NHA_ERR_UNSUPPORTED, "B*H*T*max(d,m)=%lld >= 2^31", elems);
    return NHA_OK;
}

// backward && reuse: the chunk states, gate totals, RoPE table and rotated q, k
// come from the forward's workspace, so this plan holds only the backward's own
// buffers.
// per_head: the heads have their own windows in [0, w] or sequences their own
// lengths in [0, T]; the per-head arrays are then laid out for the largest
// number of chunks (w = 0, T tokens).
Plan make_plan(int B, int H, int T, int d, int m, int w, bool backward, bool reuse = false, bool per_head = false) {
    Plan p;
    memset(&p, 0, sizeof(p));
    p.d = d;
    p.m = m;
    nha::Shape& sh = p.sh;
    sh.BH = B * H;
    sh.T = T;
    sh.w = w < T ? w : T;
    sh.R = T - sh.w;
    sh.NC = (sh.R + nha::kChunk - 1) / nha::kChunk;
    sh.NL = (sh.w + nha::kChunk - 1) / nha::kChunk;
    sh.NKT = (T + nha::kChunk - 1) / nha::kChunk;
    sh.sigma = (float)(1.0 / sqrt((double)d));
    sh.NCS = per_head ? sh.NKT : sh.NC;
    sh.W0S = T - sh.R;
    sh.windows = nullptr;
    sh.H = H;
    sh.wbh = 0;
    sh.seq = nullptr;
    sh.TS = T;
    sh.status = nullptr;
    size_t off = 0;
    auto take = [&](size_t n) {
        size_t o = off;
        off += (n + 63) & ~(size_t)63;  // keep every sub-buffer 256-byte aligned
        return o;
    };
    const size_t BH = (size_t)sh.BH, NC = (size_t)sh.NCS, Tz = (size_t)T;
    p.STATUS = take(16);
    if (!(backward && reuse)) {
        p.SK = take(BH * NC * m * d);
        p.SV = take(BH * NC * m * d);
        p.SKb = take(BH * NC * m * d / 2);
        p.SVb = take(BH * NC * m * d / 2);
        p.G = take(BH * NC * m);
        p.TAB = take(Tz * (size_t)d);  // RoPE (cos, sin) per position and frequency
        p.QR = take(BH * Tz * d / 2);  // RoPE(q), bf16
        p.KR = take(BH * Tz * d / 2);  // RoPE(k), bf16
        p.HTB = take(BH * 2 * m * d / 2);  // final states, bf16 [BH][2][m][d] (last chunk's carry)
        p.HTF = take(BH * 2 * m * d);      // final states, fp32 (same, fp32 path)
    }
    if (backward) {
        p.Dv = take(BH * Tz);
        p.Dhat = take(BH * Tz);
        p.Dwin = take(BH * Tz);
        p.dqwV = take(BH * Tz * d);
        p.dqw = take(BH * Tz * d);
        p.dkw = take(BH * Tz * d);
        p.dvw = take(BH * Tz * d);
        p.DL = take(BH * NC * nha::kChunk * m);
        p.PL = take(BH * NC * nha::kChunk * m);
        p.DB1 = take(BH * NC * nha::kChunk * m);
        p.RK = take(BH * NC * m * d);
        p.RV = take(BH * NC * m * d);
        p.RKb = take(BH * NC * m * d / 2);
        p.RVb = take(BH * NC * m * d / 2);
        p.REND = take(BH * 2 * m * d);  // the state adjoint carried past chunk 0
        const size_t W0 = (size_t)sh.W0S;
        p.LDL = take(BH * W0 * m);  // sigma dL of the queries t < w (initial states)
        p.LPL = take(BH * W0 * m);  // their P_L
    }
    p.total = off;
    return p;
}

void make_rope(nha::RopeTab& rt, int d, float base) {
    memset(&rt, 0, sizeof(rt));
    for (int i = 0; i < d / 2; i++) {
        double f = pow((double)base, -2.0 * i / d) / M_PI;  // theta_i / pi
        int e;
        double mant = frexp(f, &e);                            // f = mant * 2^e, mant in [0.5, 1)
        double hi = ldexp(nearbyint(mant * 64.0) / 64.0, e);   // 6 significant bits
        rt.f_hi[i] = (float)hi;
        rt.f_lo[i] = (float)(f - hi);
    }
}

bool misaligned(const void* p) { return ((uintptr_t)p & 15u) != 0; }

// Optional arguments of the _ex entry points: which are set, and that each
// is valid for the call (forward or backward) it is given to.
nha_status_t check_extras(const nha_extras_t* ex, bool backward) {
    if (ex == nullptr) return NHA_OK;
    if (!backward && ex->fwd_workspace != nullptr)
        return fail(NHA_ERR_INVALID_ARGUMENT, "fwd_workspace is an input of the backward only");
    const struct {
        const void* k;
        const void* v;
        const char* name;
        bool fwd, bwd;  // the call that takes it
    } pairs[] = {{ex->h0_k, ex->h0_v, "h0", true, true},
                 {ex->hT_k, ex->hT_v, "hT", true, false},
                 {ex->dhT_k, ex->dhT_v, "dhT", false, true},
                 {ex->dh0_k, ex->dh0_v, "dh0", false, true}};
    for (const auto& pr : pairs) {
        if ((pr.k == nullptr) != (pr.v == nullptr))
            return fail(NHA_ERR_INVALID_ARGUMENT, "%s_k and %s_v must be given together", pr.name, pr.name);
        if (pr.k == nullptr) continue;
        if (backward ? !pr.bwd : !pr.fwd)
            return fail(NHA_ERR_INVALID_ARGUMENT, "%s is not an argument of the %s", pr.name,
                        backward ? "backward" : "forward");
        if (misaligned(pr.k) || misaligned(pr.v))
            return fail(NHA_ERR_INVALID_ARGUMENT, "%s is not 16-byte aligned", pr.name);
    }
    if (ex->dh0_k != nullptr && ex->h0_k == nullptr)
        return fail(NHA_ERR_INVALID_ARGUMENT, "dh0 needs h0 (the gradient of an input that is not given)");
    if (ex->windows != nullptr && ((uintptr_t)ex->windows & 3u) != 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "windows array is not 4-byte aligned");
    if (ex->windows_per_sequence != 0 && ex->windows_per_sequence != 1)
        return fail(NHA_ERR_INVALID_ARGUMENT, "windows_per_sequence=%d is neither 0 nor 1", ex->windows_per_sequence);
    if (ex->windows_per_sequence && ex->windows == nullptr)
        return fail(NHA_ERR_INVALID_ARGUMENT, "windows_per_sequence without a windows array");
    if (ex->cu_seqlens != nullptr && ((uintptr_t)ex->cu_seqlens & 3u) != 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "cu_seqlens array is not 4-byte aligned");
    if (ex->status != nullptr && ((uintptr_t)ex->status & 3u) != 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "status is not 4-byte aligned");
    return NHA_OK;
}

bool per_head(const nha_extras_t* ex) { return ex != nullptr && (ex->windows != nullptr || ex->cu_seqlens != nullptr); }

// The per-head and per-sequence fields of a call's shape.
void set_varied(nha::Shape& sh, const nha_extras_t* ex) {
    if (ex == nullptr) return;
    sh.windows = ex->windows;
    sh.wbh = ex->windows_per_sequence;
    sh.seq = ex->cu_seqlens;
}

nha::StateIO state_io(const nha_extras_t* ex, bool forward) {
    nha::StateIO io{};
    if (ex != nullptr) {
        io.h0k = ex->h0_k;
        io.h0v = ex->h0_v;
        if (forward) {
            io.hTk = ex->hT_k;
            io.hTv = ex->hT_v;
        }
    }
    return io;
}

cudaError_t run_forward_tc(const Plan& p, const nha::FwdArgs& a, float* ws, cudaStream_t s) {
    float2* tab = (float2*)(ws + p.TAB);
    int* status = a.sh.status;
    __nv_bfloat16* qr = (__nv_bfloat16*)(ws + p.QR);
    __nv_bfloat16* kr = (__nv_bfloat16*)(ws + p.KR);
    switch (p.d * 1000 + p.m) {
        case 64016: return nha::tc_forward<64, 16>(a, tab, qr, kr, status, s);
        case 64032: return nha::tc_forward<64, 32>(a, tab, qr, kr, status, s);
        case 64064: return nha::tc_forward<64, 64>(a, tab, qr, kr, status, s);
        case 128016: return nha::tc_forward<128, 16>(a, tab, qr, kr, status, s);
        case 128032: return nha::tc_forward<128, 32>(a, tab, qr, kr, status, s);
        case 128064: return nha::tc_forward<128, 64>(a, tab, qr, kr, status, s);
    }
    return cudaErrorInvalidValue;
}

template <typename Tin>
cudaError_t run_forward(const Plan& p, const nha::FwdArgs& a, cudaStream_t s) {
    switch (p.d * 1000 + p.m) {
        case 64016: return nha::simt_forward<Tin, 64, 16>(a, s);
        case 64032: return nha::simt_forward<Tin, 64, 32>(a, s);
        case 64064: return nha::simt_forward<Tin, 64, 64>(a, s);
        case 128016: return nha::simt_forward<Tin, 128, 16>(a, s);
        case 128032: return nha::simt_forward<Tin, 128, 32>(a, s);
        case 128064: return nha::simt_forward<Tin, 128, 64>(a, s);
    }
    return cudaErrorInvalidValue;
}

// fws, fp: the workspace and plan holding the forward's buffers (the
// backward's own, or the forward's when they are reused)
cudaError_t run_backward_tc(const Plan& p, const nha::BwdArgs& a, float* ws, const Plan& fp, float* fws,
                            cudaStream_t s) {
    float2* tab = (float2*)(fws + fp.TAB);
    int* status = a.sh.status;
    __nv_bfloat16* qr = (__nv_bfloat16*)(fws + fp.QR);
    __nv_bfloat16* kr = (__nv_bfloat16*)(fws + fp.KR);
    switch (p.d * 1000 + p.m) {
        case 64016: return nha::tc_backward<64, 16>(a, tab, qr, kr, status, s);
        case 64032: return nha::tc_backward<64, 32>(a, tab, qr, kr, status, s);
        case 64064: return nha::tc_backward<64, 64>(a, tab, qr, kr, status, s);
        case 128016: return nha::tc_backward<128, 16>(a, tab, qr, kr, status, s);
        case 128032: return nha::tc_backward<128, 32>(a, tab, qr, kr, status, s);
        case 128064: return nha::tc_backward<128, 64>(a, tab, qr, kr, status, s);
    }
    return cudaErrorInvalidValue;
}

template <typename Tin>
cudaError_t run_backward(const Plan& p, const nha::BwdArgs& a, cudaStream_t s) {
    switch (p.d * 1000 + p.m) {
        case 64016: return nha::simt_backward<Tin, 64, 16>(a, s);
        case 64032: return nha::simt_backward<Tin, 64, 32>(a, s);
        case 64064: return nha::simt_backward<Tin, 64, 64>(a, s);
        case 128016: return nha::simt_backward<Tin, 128, 16>(a, s);
        case 128032: return nha::simt_backward<Tin, 128, 32>(a, s);
        case 128064: return nha::simt_backward<Tin, 128, 64>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

namespace nha {
nha_status_t set_error(nha_status_t s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}
}  // namespace nha

extern "C" {

size_t nha_workspace_bytes(int B, int H, int T, int d, int m, int w, int C, nha_dtype_t dtype,
                           int backward) {
    if (check_shape(B, H, T, d, m, w, C, dtype) != NHA_OK) return 0;
    Plan p = make_plan(B, H, T, d, m, w, backward != 0);
    return p.total * sizeof(float);
}

nha_status_t nha_forward(const void* q, const void* k, const void* v, const float* log_alpha,
                         void* o, float* lse, int B, int H, int T, int d, int m, int w, int C,
                         nha_dtype_t dtype, float rope_base, void* workspace, size_t ws_bytes,
                         void* stream) {
    return nha_forward_ex(q, k, v, log_alpha, o, lse, B, H, T, d, m, w, C, dtype, rope_base, nullptr, workspace,
                          ws_bytes, stream);
}

nha_status_t nha_backward(const void* q, const void* k, const void* v, const float* log_alpha,
                          const void* o, const float* lse, const void* dout, void* dq, void* dk,
                          void* dv, float* dlog_alpha, int B, int H, int T, int d, int m, int w,
                          int C, nha_dtype_t dtype, float rope_base, void* workspace,
                          size_t ws_bytes, void* stream) {
    return nha_backward_ex(q, k, v, log_alpha, o, lse, dout, dq, dk, dv, dlog_alpha, B, H, T, d, m, w, C, dtype,
                           rope_base, nullptr, workspace, ws_bytes, stream);
}

size_t nha_workspace_bytes_ex(int B, int H, int T, int d, int m, int w, int C, nha_dtype_t dtype, int backward,
                              const nha_extras_t* ex) {
    if (check_shape(B, H, T, d, m, w, C, dtype) != NHA_OK) return 0;
    const bool reuse = backward && ex != nullptr && ex->fwd_workspace != nullptr;
    Plan p = make_plan(B, H, T, d, m, w, backward != 0, reuse, per_head(ex));
    return p.total * sizeof(float);
}

nha_status_t nha_forward_ex(const void* q, const void* k, const void* v, const float* log_alpha, void* o,
                            float* lse, int B, int H, int T, int d, int m, int w, int C, nha_dtype_t dtype,
                            float rope_base, const nha_extras_t* ex, void* workspace, size_t ws_bytes,
                            void* stream) {
    if (inject("validate")) return fail(NHA_ERR_INTERNAL, "fault injected at validate");
    nha_status_t st = check_shape(B, H, T, d, m, w, C, dtype);
    if (st != NHA_OK) return st;
    if (!(rope_base > 1.0f) || !isfinite(rope_base))
        return fail(NHA_ERR_INVALID_ARGUMENT, "rope_base must be a finite value > 1");
    if ((st = check_extras(ex, false)) != NHA_OK) return st;
    if ((long long)B * H * T == 0) return ok();
    const void* ptrs[] = {q, k, v, log_alpha, o, lse};
    const char* names[] = {"q", "k", "v", "log_alpha", "o", "lse"};
    for (int i = 0; i < 6; i++) {
        if (ptrs[i] == nullptr) return fail(NHA_ERR_INVALID_ARGUMENT, "%s is NULL", names[i]);
        if (misaligned(ptrs[i])) return fail(NHA_ERR_INVALID_ARGUMENT, "%s is not 16-byte aligned", names[i]);
    }
    Plan p = make_plan(B, H, T, d, m, w, false, false, per_head(ex));
    const size_t need = p.total * sizeof(float);
    if (need > 0 && (workspace == nullptr || ws_bytes < need))
        return fail(NHA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? ws_bytes : (size_t)0);
    if (need > 0 && misaligned(workspace))
        return fail(NHA_ERR_INVALID_ARGUMENT, "workspace is not 16-byte aligned");
    if (inject("forward_launch")) return fail(NHA_ERR_INTERNAL, "fault injected at forward_launch");
    float* ws = (float*)workspace;
    nha::FwdArgs a;
    a.q = q; a.k = k; a.v = v; a.la = log_alpha; a.o = o; a.lse = lse;
    a.SK = ws + p.SK; a.SV = ws + p.SV; a.G = ws + p.G;
    a.SKb = (__nv_bfloat16*)(ws + p.SKb); a.SVb = (__nv_bfloat16*)(ws + p.SVb);
    a.io = state_io(ex, true);
    a.io.htb = (__nv_bfloat16*)(ws + p.HTB);
    a.io.htf = ws + p.HTF;
    a.sh = p.sh;
    set_varied(a.sh, ex);
    a.sh.status = (ex != nullptr && ex->status != nullptr) ? ex->status : (int*)(ws + p.STATUS);
    make_rope(a.rope, d, rope_base);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(a.sh.status, 0, sizeof(int), s);
    if (e == cudaSuccess)
        e = dtype == NHA_DTYPE_F32 ? run_forward<float>(p, a, s) : run_forward_tc(p, a, ws, s);
    if (e != cudaSuccess) return fail(NHA_ERR_CUDA, "forward launch failed: %s", cudaGetErrorString(e));
    return ok();
}

nha_status_t nha_backward_ex(const void* q, const void* k, const void* v, const float* log_alpha, const void* o,
                             const float* lse, const void* dout, void* dq, void* dk, void* dv, float* dlog_alpha,
                             int B, int H, int T, int d, int m, int w, int C, nha_dtype_t dtype, float rope_base,
                             const nha_extras_t* ex, void* workspace, size_t ws_bytes, void* stream) {
    if (inject("validate")) return fail(NHA_ERR_INTERNAL, "fault injected at validate");
    nha_status_t st = check_shape(B, H, T, d, m, w, C, dtype);
    if (st != NHA_OK) return st;
    if (!(rope_base > 1.0f) || !isfinite(rope_base))
        return fail(NHA_ERR_INVALID_ARGUMENT, "rope_base must be a finite value > 1");
    if ((st = check_extras(ex, true)) != NHA_OK) return st;
    if ((long long)B * H * T == 0) return ok();
    const void* ptrs[] = {q, k, v, log_alpha, o, lse, dout, dq, dk, dv, dlog_alpha};
    const char* names[] = {"q", "k", "v", "log_alpha", "o", "lse", "dout", "dq", "dk", "dv", "dlog_alpha"};
    for (int i = 0; i < 11; i++) {
        if (ptrs[i] == nullptr) return fail(NHA_ERR_INVALID_ARGUMENT, "%s is NULL", names[i]);
        if (misaligned(ptrs[i])) return fail(NHA_ERR_INVALID_ARGUMENT, "%s is not 16-byte aligned", names[i]);
    }
    const bool reuse = ex != nullptr && ex->fwd_workspace != nullptr;
    Plan p = make_plan(B, H, T, d, m, w, true, reuse, per_head(ex));
    const size_t need = p.total * sizeof(float);
    if (workspace == nullptr || ws_bytes < need)
        return fail(NHA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? ws_bytes : (size_t)0);
    if (misaligned(workspace)) return fail(NHA_ERR_INVALID_ARGUMENT, "workspace is not 16-byte aligned");
    Plan fp = p;
    float* ws = (float*)workspace;
    float* fws = ws;
    if (reuse) {
        fp = make_plan(B, H, T, d, m, w, false, false, per_head(ex));
        const size_t fneed = fp.total * sizeof(float);
        if (ex->fwd_ws_bytes < fneed)
            return fail(NHA_ERR_WORKSPACE, "forward workspace of %zu bytes expected, %zu given", fneed,
                        ex->fwd_ws_bytes);
        if (misaligned(ex->fwd_workspace))
            return fail(NHA_ERR_INVALID_ARGUMENT, "forward workspace is not 16-byte aligned");
        fws = (float*)const_cast<void*>(ex->fwd_workspace);
    }
    if (inject("backward_launch")) return fail(NHA_ERR_INTERNAL, "fault injected at backward_launch");
    nha::BwdArgs a;
    a.q = q; a.k = k; a.v = v; a.la = log_alpha; a.o = o; a.lse = lse; a.dout = dout;
    a.dq = dq; a.dk = dk; a.dv = dv; a.dla = dlog_alpha;
    a.SK = fws + fp.SK; a.SV = fws + fp.SV; a.G = fws + fp.G; a.Dv = ws + p.Dv;
    a.Dhat = ws + p.Dhat; a.Dwin = ws + p.Dwin; a.dqwV = ws + p.dqwV;
    a.dqw = ws + p.dqw; a.dkw = ws + p.dkw; a.dvw = ws + p.dvw;
    a.wsDL = ws + p.DL; a.wsPL = ws + p.PL; a.wsDB1 = ws + p.DB1;
    a.RK = ws + p.RK; a.RV = ws + p.RV;
    a.SKb = (__nv_bfloat16*)(fws + fp.SKb); a.SVb = (__nv_bfloat16*)(fws + fp.SVb);
    a.RKb = (__nv_bfloat16*)(ws + p.RKb); a.RVb = (__nv_bfloat16*)(ws + p.RVb);
    a.hdqw = (__nv_bfloat16*)a.dqw; a.hdqwV = (__nv_bfloat16*)a.dqwV;
    a.hdkw = (__nv_bfloat16*)a.dkw; a.hdvw = (__nv_bfloat16*)a.dvw;
    a.hDL = (__nv_bfloat16*)a.wsDL; a.hPL = (__nv_bfloat16*)a.wsPL;
    a.hRK = (__nv_bfloat16*)a.RK; a.hRV = (__nv_bfloat16*)a.RV;
    a.reuse = reuse;
    a.io = state_io(ex, false);
    a.io.htb = (__nv_bfloat16*)(fws + fp.HTB);
    a.io.htf = fws + fp.HTF;
    a.dhTk = ex ? ex->dhT_k : nullptr;
    a.dhTv = ex ? ex->dhT_v : nullptr;
    a.dh0k = ex ? ex->dh0_k : nullptr;
    a.dh0v = ex ? ex->dh0_v : nullptr;
    a.rend = ws + p.REND;
    a.ldl = ws + p.LDL;
    a.lpl = ws + p.LPL;
    a.sh = p.sh;
    set_varied(a.sh, ex);
    a.sh.status = (ex != nullptr && ex->status != nullptr) ? ex->status : (int*)(ws + p.STATUS);
    make_rope(a.rope, d, rope_base);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(a.sh.status, 0, sizeof(int), s);
    if (e == cudaSuccess)
        e = dtype == NHA_DTYPE_F32 ? run_backward<float>(p, a, s) : run_backward_tc(p, a, ws, fp, fws, s);
    if (e != cudaSuccess) return fail(NHA_ERR_CUDA, "backward launch failed: %s", cudaGetErrorString(e));
    return ok();
}

}  // extern "C"

namespace {
// Shared by nha_decode_step (host position t) and nha_decode_step_varlen
// (device positions tpos[B], t unused).
nha_status_t decode_call(const void* q, const void* k, const void* v, const float* log_alpha, void* o,
                         float* state_k, float* state_v, void* ring_k, void* ring_v, float* ring_la, int t,
                         const int* tpos, const int* wvec, int B, int H, int d, int m, int w, nha_dtype_t dtype,
                         float rope_base, void* stream, unsigned flags = 0) {
    if (inject("validate")) return fail(NHA_ERR_INTERNAL, "fault injected at validate");
    if (B < 0 || H < 0 || t < 0 || w < 0 || d <= 0 || m <= 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "negative or zero size (B=%d H=%d t=%d d=%d m=%d w=%d)", B, H, t,
                    d, m, w);
    if (dtype != NHA_DTYPE_F32 && dtype != NHA_DTYPE_BF16)
        return fail(NHA_ERR_INVALID_ARGUMENT, "unknown dtype %d", (int)dtype);
    if (d != 64 && d != 128) return fail(NHA_ERR_UNSUPPORTED, "head dim d=%d not in {64, 128}", d);
    if (m != 16 && m != 32 && m != 64) return fail(NHA_ERR_UNSUPPORTED, "slots m=%d not in {16, 32, 64}", m);
    if (t >= kMaxT) return fail(NHA_ERR_UNSUPPORTED, "position t=%d not below %d", t, kMaxT);
    if (w > kMaxT) return fail(NHA_ERR_UNSUPPORTED, "window w=%d above %d", w, kMaxT);
    const long long BH = (long long)B * H, wr = w > 0 ? w : 1;
    if (BH * wr * (d > m ? d : m) >= (1LL << 31) || BH * 8 >= (1LL << 31))
        return fail(NHA_ERR_UNSUPPORTED, "B*H*max(w,1)*max(d,m) >= 2^31");
    if (!(rope_base > 1.0f) || !isfinite(rope_base))
        return fail(NHA_ERR_INVALID_ARGUMENT, "rope_base must be a finite value > 1");
    if (BH == 0) return ok();
    const void* ptrs[] = {q, k, v, log_alpha, o, state_k, state_v, ring_k, ring_v, ring_la};
    const char* names[] = {"q", "k", "v", "log_alpha", "o", "state_k", "state_v", "ring_k", "ring_v", "ring_la"};
    const int nptr = w > 0 ? 10 : 7;  // the ring is not used when w = 0
    for (int i = 0; i < nptr; i++) {
        if (ptrs[i] == nullptr) return fail(NHA_ERR_INVALID_ARGUMENT, "%s is NULL", names[i]);
        if (misaligned(ptrs[i])) return fail(NHA_ERR_INVALID_ARGUMENT, "%s is not 16-byte aligned", names[i]);
    }
    if (tpos != nullptr && ((uintptr_t)tpos & 3u) != 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "positions array is not 4-byte aligned");
    if (wvec != nullptr && ((uintptr_t)wvec & 3u) != 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "windows array is not 4-byte aligned");
    if (inject("decode_launch")) return fail(NHA_ERR_INTERNAL, "fault injected at decode_launch");
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(NHA_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
    nha::DecodeArgs a;
    a.q = q; a.k = k; a.v = v; a.la = log_alpha; a.o = o;
    a.SK = state_k; a.SV = state_v;
    a.ring_k = w > 0 ? ring_k : nullptr;
    a.ring_v = w > 0 ? ring_v : nullptr;
    a.ring_la = w > 0 ? ring_la : nullptr;
    a.BH = (int)BH; a.t = t; a.w = w; a.tpos = tpos; a.wvec = wvec; a.H = H; a.sms = sms;
    a.overlap = (flags & NHA_DECODE_OVERLAP) ? 1 : 0;
    make_rope(a.rope, d, rope_base);
    cudaStream_t s = (cudaStream_t)stream;
    const bool f32 = dtype == NHA_DTYPE_F32;
    switch (d * 1000 + m) {
        case 64016: e = f32 ? nha::launch_decode<float, 64, 16>(a, s) : nha::launch_decode<__nv_bfloat16, 64, 16>(a, s); break;
        case 64032: e = f32 ? nha::launch_decode<float, 64, 32>(a, s) : nha::launch_decode<__nv_bfloat16, 64, 32>(a, s); break;
        case 64064: e = f32 ? nha::launch_decode<float, 64, 64>(a, s) : nha::launch_decode<__nv_bfloat16, 64, 64>(a, s); break;
        case 128016: e = f32 ? nha::launch_decode<float, 128, 16>(a, s) : nha::launch_decode<__nv_bfloat16, 128, 16>(a, s); break;
        case 128032: e = f32 ? nha::launch_decode<float, 128, 32>(a, s) : nha::launch_decode<__nv_bfloat16, 128, 32>(a, s); break;
        case 128064: e = f32 ? nha::launch_decode<float, 128, 64>(a, s) : nha::launch_decode<__nv_bfloat16, 128, 64>(a, s); break;
        default: e = cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return fail(NHA_ERR_CUDA, "decode launch failed: %s", cudaGetErrorString(e));
    return ok();
}
}  // namespace

extern "C" {

nha_status_t nha_decode_step(const void* q, const void* k, const void* v, const float* log_alpha, void* o,
                             float* state_k, float* state_v, void* ring_k, void* ring_v, float* ring_la, int t,
                             int B, int H, int d, int m, int w, nha_dtype_t dtype, float rope_base, void* stream) {
    return decode_call(q, k, v, log_alpha, o, state_k, state_v, ring_k, ring_v, ring_la, t, nullptr, nullptr, B, H,
                       d, m, w, dtype, rope_base, stream);
}

nha_status_t nha_decode_step_ex(const void* q, const void* k, const void* v, const float* log_alpha, void* o,
                                float* state_k, float* state_v, void* ring_k, void* ring_v, float* ring_la, int t,
                                int B, int H, int d, int m, int w, nha_dtype_t dtype, float rope_base, unsigned flags,
                                void* stream) {
    if ((flags & ~(unsigned)NHA_DECODE_OVERLAP) != 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "unknown decode flags 0x%x", flags);
    return decode_call(q, k, v, log_alpha, o, state_k, state_v, ring_k, ring_v, ring_la, t, nullptr, nullptr, B, H,
                       d, m, w, dtype, rope_base, stream, flags);
}

nha_status_t nha_decode_step_varlen(const void* q, const void* k, const void* v, const float* log_alpha, void* o,
                                    float* state_k, float* state_v, void* ring_k, void* ring_v, float* ring_la,
                                    const int* positions, const int* windows, int B, int H, int d, int m, int w,
                                    nha_dtype_t dtype, float rope_base, void* stream) {
    if (positions == nullptr && (long long)B * H > 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "positions is NULL");
    return decode_call(q, k, v, log_alpha, o, state_k, state_v, ring_k, ring_v, ring_la, 0, positions, windows, B, H,
                       d, m, w, dtype, rope_base, stream);
}

nha_status_t nha_decode_prefill(const void* k, const void* v, const float* log_alpha, float* state_k,
                                float* state_v, void* ring_k, void* ring_v, float* ring_la, const int* windows,
                                int B, int H, int T, int d, int m, int w, nha_dtype_t dtype, void* stream) {
    if (inject("validate")) return fail(NHA_ERR_INTERNAL, "fault injected at validate");
    if (B < 0 || H < 0 || T < 0 || w < 0 || d <= 0 || m <= 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "negative or zero size (B=%d H=%d T=%d d=%d m=%d w=%d)", B, H, T,
                    d, m, w);
    if (dtype != NHA_DTYPE_F32 && dtype != NHA_DTYPE_BF16)
        return fail(NHA_ERR_INVALID_ARGUMENT, "unknown dtype %d", (int)dtype);
    if (d != 64 && d != 128) return fail(NHA_ERR_UNSUPPORTED, "head dim d=%d not in {64, 128}", d);
    if (m != 16 && m != 32 && m != 64) return fail(NHA_ERR_UNSUPPORTED, "slots m=%d not in {16, 32, 64}", m);
    if (T > kMaxT) return fail(NHA_ERR_UNSUPPORTED, "T=%d above the supported %d", T, kMaxT);
    if (w > kMaxT) return fail(NHA_ERR_UNSUPPORTED, "window w=%d above %d", w, kMaxT);
    const long long BH = (long long)B * H, wr = w > 0 ? w : 1;
    const long long rows = T > wr ? T : wr;
    if (BH * rows * (d > m ? d : m) >= (1LL << 31) || 2 * BH >= (1LL << 31))
        return fail(NHA_ERR_UNSUPPORTED, "B*H*max(T,w,1)*max(d,m) >= 2^31");
    if (BH == 0) return ok();
    const void* ptrs[] = {k, v, log_alpha, state_k, state_v, ring_k, ring_v, ring_la};
    const char* names[] = {"k", "v", "log_alpha", "state_k", "state_v", "ring_k", "ring_v", "ring_la"};
    const int first = T > 0 ? 0 : 3;       // no prompt: k, v, log_alpha are not read
    const int nptr = w > 0 ? 8 : 5;       // the ring is not used when w = 0
    for (int i = first; i < nptr; i++) {
        if (ptrs[i] == nullptr) return fail(NHA_ERR_INVALID_ARGUMENT, "%s is NULL", names[i]);
        if (misaligned(ptrs[i])) return fail(NHA_ERR_INVALID_ARGUMENT, "%s is not 16-byte aligned", names[i]);
    }
    if (windows != nullptr && ((uintptr_t)windows & 3u) != 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "windows array is not 4-byte aligned");
    if (inject("prefill_launch")) return fail(NHA_ERR_INTERNAL, "fault injected at prefill_launch");
    nha::PrefillArgs a;
    a.k = k; a.v = v; a.la = log_alpha;
    a.SK = state_k; a.SV = state_v;
    a.ring_k = w > 0 ? ring_k : nullptr;
    a.ring_v = w > 0 ? ring_v : nullptr;
    a.ring_la = w > 0 ? ring_la : nullptr;
    a.BH = (int)BH; a.T = T; a.w = w; a.wvec = windows; a.H = H;
    cudaStream_t s = (cudaStream_t)stream;
    const bool f32 = dtype == NHA_DTYPE_F32;
    cudaError_t e;
    switch (d * 1000 + m) {
        case 64016: e = f32 ? nha::launch_prefill<float, 64, 16>(a, s) : nha::launch_prefill<__nv_bfloat16, 64, 16>(a, s); break;
        case 64032: e = f32 ? nha::launch_prefill<float, 64, 32>(a, s) : nha::launch_prefill<__nv_bfloat16, 64, 32>(a, s); break;
        case 64064: e = f32 ? nha::launch_prefill<float, 64, 64>(a, s) : nha::launch_prefill<__nv_bfloat16, 64, 64>(a, s); break;
        case 128016: e = f32 ? nha::launch_prefill<float, 128, 16>(a, s) : nha::launch_prefill<__nv_bfloat16, 128, 16>(a, s); break;
        case 128032: e = f32 ? nha::launch_prefill<float, 128, 32>(a, s) : nha::launch_prefill<__nv_bfloat16, 128, 32>(a, s); break;
        case 128064: e = f32 ? nha::launch_prefill<float, 128, 64>(a, s) : nha::launch_prefill<__nv_bfloat16, 128, 64>(a, s); break;
        default: e = cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return fail(NHA_ERR_CUDA, "prefill launch failed: %s", cudaGetErrorString(e));
    return ok();
}

nha_status_t nha_gate_total(const float* log_alpha, float* decay, int B, int H, int T, int m, int w, void* stream) {
    if (inject("validate")) return fail(NHA_ERR_INTERNAL, "fault injected at validate");
    if (B < 0 || H < 0 || T < 0 || w < 0 || m <= 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "negative or zero size (B=%d H=%d T=%d m=%d w=%d)", B, H, T, m, w);
    if (m != 16 && m != 32 && m != 64) return fail(NHA_ERR_UNSUPPORTED, "slots m=%d not in {16, 32, 64}", m);
    if (T > kMaxT) return fail(NHA_ERR_UNSUPPORTED, "T=%d above the supported %d", T, kMaxT);
    if ((long long)B * H * T * m >= (1LL << 31)) return fail(NHA_ERR_UNSUPPORTED, "B*H*T*m >= 2^31");
    if ((long long)B * H == 0) return ok();
    if (decay == nullptr || misaligned(decay)) return fail(NHA_ERR_INVALID_ARGUMENT, "decay is NULL or misaligned");
    const int R = T > w ? T - w : 0;
    if (R > 0 && (log_alpha == nullptr || misaligned(log_alpha)))
        return fail(NHA_ERR_INVALID_ARGUMENT, "log_alpha is NULL or misaligned");
    cudaError_t e = nha::launch_gate_total(log_alpha, decay, B * H, T, m, R, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail(NHA_ERR_CUDA, "gate_total launch failed: %s", cudaGetErrorString(e));
    return ok();
}

static nha_status_t varlen_call(const void* src, void* dst, const int* cu, int B, int H, int T, int Ttot, int width,
                                int elem_bytes, bool pad, void* stream) {
    if (inject("validate")) return fail(NHA_ERR_INTERNAL, "fault injected at validate");
    if (B < 0 || H < 0 || T < 0 || Ttot < 0 || width <= 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "negative or zero size (B=%d H=%d T=%d Ttot=%d width=%d)", B, H, T, Ttot,
                    width);
    if (elem_bytes != 2 && elem_bytes != 4)
        return fail(NHA_ERR_INVALID_ARGUMENT, "elem_bytes=%d is neither 2 nor 4", elem_bytes);
    const long long row_bytes = (long long)width * elem_bytes;
    if (row_bytes % 4 != 0) return fail(NHA_ERR_INVALID_ARGUMENT, "row of %lld bytes is not a multiple of 4", row_bytes);
    if ((long long)B * H * T * row_bytes / 4 >= (1LL << 31) || (long long)H * Ttot * row_bytes / 4 >= (1LL << 31))
        return fail(NHA_ERR_UNSUPPORTED, "arrays of 2^31 or more 4-byte words");
    if ((long long)B * H * T == 0) return ok();
    const void* ptrs[] = {src, dst, cu};
    const char* names[] = {pad ? "packed" : "padded", pad ? "padded" : "packed", "cu_seqlens"};
    for (int i = 0; i < 3; i++) {
        if (ptrs[i] == nullptr) return fail(NHA_ERR_INVALID_ARGUMENT, "%s is NULL", names[i]);
        if (((uintptr_t)ptrs[i] & 3u) != 0) return fail(NHA_ERR_INVALID_ARGUMENT, "%s is not 4-byte aligned", names[i]);
    }
    cudaError_t e = nha::launch_varlen_copy(src, dst, cu, B, H, T, Ttot, (int)row_bytes, pad, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail(NHA_ERR_CUDA, "varlen copy launch failed: %s", cudaGetErrorString(e));
    return ok();
}

nha_status_t nha_varlen_pad(const void* packed, void* padded, const int* cu_seqlens, int B, int H, int T, int Ttot,
                            int width, int elem_bytes, void* stream) {
    return varlen_call(packed, padded, cu_seqlens, B, H, T, Ttot, width, elem_bytes, true, stream);
}

nha_status_t nha_varlen_unpad(const void* padded, void* packed, const int* cu_seqlens, int B, int H, int T, int Ttot,
                              int width, int elem_bytes, void* stream) {
    return varlen_call(padded, packed, cu_seqlens, B, H, T, Ttot, width, elem_bytes, false, stream);
}

nha_status_t nha_state_combine(const float* decay, const float* prev_k, const float* prev_v, const float* cur_k,
                               const float* cur_v, float* out_k, float* out_v, int B, int H, int m, int d,
                               void* stream) {
    if (inject("validate")) return fail(NHA_ERR_INTERNAL, "fault injected at validate");
    if (B < 0 || H < 0 || m <= 0 || d <= 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "negative or zero size (B=%d H=%d m=%d d=%d)", B, H, m, d);
    if ((long long)B * H * m * d >= (1LL << 31)) return fail(NHA_ERR_UNSUPPORTED, "B*H*m*d >= 2^31");
    if ((long long)B * H == 0) return ok();
    const void* ptrs[] = {decay, prev_k, prev_v, cur_k, cur_v, out_k, out_v};
    const char* names[] = {"decay", "prev_k", "prev_v", "cur_k", "cur_v", "out_k", "out_v"};
    for (int i = 0; i < 7; i++) {
        if (ptrs[i] == nullptr) return fail(NHA_ERR_INVALID_ARGUMENT, "%s is NULL", names[i]);
        if (misaligned(ptrs[i])) return fail(NHA_ERR_INVALID_ARGUMENT, "%s is not 16-byte aligned", names[i]);
    }
    cudaError_t e = nha::launch_state_combine(decay, prev_k, prev_v, cur_k, cur_v, out_k, out_v, B * H, m, d,
                                              (cudaStream_t)stream);
    if (e != cudaSuccess) return fail(NHA_ERR_CUDA, "state_combine launch failed: %s", cudaGetErrorString(e));
    return ok();
}

nha_status_t nha_selftest_wait(int* status, long long cycles, void* stream) {
    if (status == nullptr || ((uintptr_t)status & 3u) != 0)
        return fail(NHA_ERR_INVALID_ARGUMENT, "status is NULL or not 4-byte aligned");
    if (cycles <= 0 || cycles > (1LL << 32))
        return fail(NHA_ERR_INVALID_ARGUMENT, "cycles=%lld outside (0, 2^32]", cycles);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), s);
    if (e == cudaSuccess) e = nha::launch_selftest_wait(status, cycles, s);
    if (e != cudaSuccess) return fail(NHA_ERR_CUDA, "selftest launch failed: %s", cudaGetErrorString(e));
    return ok();
}

const char* nha_status_string(nha_status_t status) {
    switch (status) {
        case NHA_OK: return "NHA_OK";
        case NHA_ERR_INVALID_ARGUMENT: return "NHA_ERR_INVALID_ARGUMENT";
        case NHA_ERR_UNSUPPORTED: return "NHA_ERR_UNSUPPORTED";
        case NHA_ERR_WORKSPACE: return "NHA_ERR_WORKSPACE";
        case NHA_ERR_CUDA: return "NHA_ERR_CUDA";
        case NHA_ERR_INTERNAL: return "NHA_ERR_INTERNAL";
    }
    return "NHA_ERR_UNKNOWN";
}

const char* nha_last_error(void) { return g_err; }

}  // extern "C"
