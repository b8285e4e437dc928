// Internal interface between the C-ABI layer (nha_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "nha_common.cuh"

#include "nha.h"

namespace nha {

// Records the thread-local message returned by nha_last_error and returns s.
nha_status_t set_error(nha_status_t s, const char* fmt, ...);

// Side stream of this host thread on the current device, for work that runs
// beside the caller's stream: fork_side makes the side stream wait for what
// `main` has enqueued so far, join_side makes `main` wait for what the side
// stream has; event k is used once per call (k < kEvents).
struct Fork {
    static constexpr int kEvents = 4;
    cudaStream_t side = nullptr;
    cudaEvent_t ev[kEvents] = {};
};
cudaError_t get_fork(Fork** out);
cudaError_t fork_side(cudaStream_t main, Fork& f, int k);
cudaError_t join_side(cudaStream_t main, Fork& f, int k);

// Optional initial / final slot states of a call (fp32 [BH, M, D] each, NULL
// when absent) and the workspace copies the chunk scans keep of the final
// states: htb bf16 [BH][2 (K, V)][M][D] (bf16 path), htf fp32 [BH][2][M][D]
// (fp32 path).
struct StateIO {
    const float* h0k;
    const float* h0v;
    float* hTk;
    float* hTv;
    __nv_bfloat16* htb;
    float* htf;
};

// Forward arguments.  q, k, v, o are [BH, T, D] in the element type; la is
// [BH, T, M]; lse [BH, T].  Workspace: SK, SV [BH, NC, M, D] and G [BH, NC, M].
struct FwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* la;
    void* o;
    float* lse;
    float* SK;
    float* SV;
    float* G;
    __nv_bfloat16* SKb;  // bf16 copies of SK, SV (bf16 path)
    __nv_bfloat16* SVb;
    StateIO io;
    Shape sh;
    RopeTab rope;
};

// Backward arguments.  Workspace beyond the forward's: Dv [BH, T];
// dqw, dkw, dvw [BH, T, D] (window-branch partial gradients, fp32);
// wsDL, wsPL, wsDB1 [BH, NC * C, M]; RK, RV [BH, NC, M, D] (the chunks' adjoint
// contributions; the bf16 path keeps them in bf16 through hRK, hRV).
struct BwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* la;
    const void* o;
    const float* lse;
    const void* dout;
    void* dq;
    void* dk;
    void* dv;
    float* dla;
    float* SK;
    float* SV;
    float* G;
    float* Dv;     // D_t = dout_t . o_t
    float* Dhat;   // D from the rounded o (bf16 path)
    float* Dwin;   // window part of sum_s P dP (bf16 path)
    float* dqwV;   // sigma R^T sum_s P k~ (bf16 path: dq correction for D - Dhat)
    float* dqw;
    float* dkw;
    float* dvw;
    float* wsDL;
    float* wsPL;
    float* wsDB1;
    float* RK;
    float* RV;
    __nv_bfloat16* SKb;  // bf16 chunk states (SKb, SVb) and carried adjoints (RKb, RVb), bf16 path
    __nv_bfloat16* SVb;
    __nv_bfloat16* RKb;
    __nv_bfloat16* RVb;
    // bf16 path: the window partials and sigma dL, P_L are kept in bf16 (they
    // alias the storage of the fp32 arrays above)
    __nv_bfloat16* hdqw;
    __nv_bfloat16* hdqwV;
    __nv_bfloat16* hdkw;
    __nv_bfloat16* hdvw;
    __nv_bfloat16* hDL;
    __nv_bfloat16* hPL;
    // bf16 path: the chunks' adjoint contributions dR_c in bf16 (aliasing RK,
    // RV); the reverse scan carries their sum in fp32
    __nv_bfloat16* hRK;
    __nv_bfloat16* hRV;
    // the chunk states, gate totals, RoPE table and RoPE(q), RoPE(k) above are
    // the forward's, left in its workspace: the backward does not recompute them
    bool reuse;
    // initial states h0 (io.h0k, io.h0v) and the final states' workspace copies;
    // the gradient with respect to the final states (dhTk, dhTv [BH, M, D] or
    // NULL) and the initial states' gradient (dh0k, dh0v, written when h0 is
    // given); rend [BH][2][M][D]: the state adjoint the reverse scan carries past
    // chunk 0; ldl, lpl [BH][W0][M]: sigma dL and P_L of the queries t < w that
    // read h0
    StateIO io;
    const float* dhTk;
    const float* dhTv;
    float* dh0k;
    float* dh0v;
    float* rend;
    float* ldl;
    float* lpl;
    Shape sh;
    RopeTab rope;
};

// A wait that runs out on purpose (status word check).
cudaError_t launch_selftest_wait(int* status, long long cycles, cudaStream_t st);

// Segment summaries for cutting a sequence into segments: the gate product of
// the tokens that leave the window (decay [BH][M]) and out = decay o prev + cur.
cudaError_t launch_gate_total(const float* la, float* decay, int BH, int T, int M, int R, cudaStream_t st);
// Packed [H, Ttot, row] <-> padded [B, H, T, row] token rows by sequence
// offsets cu [B + 1] (pad: rows past a sequence zero; unpad: its rows only).
cudaError_t launch_varlen_copy(const void* src, void* dst, const int* cu, int B, int H, int T, int Ttot,
                               int row_bytes, bool pad, cudaStream_t st);
cudaError_t launch_state_combine(const float* decay, const float* pk, const float* pv, const float* ck,
                                 const float* cv, float* ok, float* ov, int BH, int M, int D, cudaStream_t st);

// Initial / final slot states outside the chunk kernels.
// hT = h0 (or zero) when no token leaves the window (no chunk to scan).
cudaError_t launch_final_states_copy(const StateIO& io, int BH, int M, int D, cudaStream_t st);
// Queries t < w reading h0, forward: merges the slot branch of h0 into the
// window-only o, lse the chunk kernels wrote for those rows.
template <typename Tin, int D, int M>
cudaError_t launch_h0_fwd_lead(const FwdArgs& a, cudaStream_t st);
// Same queries, backward: their slot-branch gradients (dq; the exact D for the
// bf16 path), and sigma dL, P_L for dh0.  tc: the bf16 path's partials (window
// dq and its D correction); otherwise dq already holds the window part.
template <typename Tin, int D, int M>
cudaError_t launch_h0_bwd_lead(const BwdArgs& a, bool tc, cudaStream_t st);
// dh0 = the adjoint carried past chunk 0 (dhT when no chunk) + the t < w queries' terms.
template <typename Tin, int D, int M>
cudaError_t launch_dh0(const BwdArgs& a, cudaStream_t st);

template <typename Tin, int D, int M>
cudaError_t simt_states(const Tin* k, const Tin* v, const float* la, float* SK, float* SV, float* G,
                        const StateIO& io, const Shape& sh, cudaStream_t st);
template <typename Tin, int D, int M>
cudaError_t simt_forward(const FwdArgs& a, cudaStream_t st);
// bf16 tensor-core forward; tab: RoPE (cos, sin) table [T][D/2] in the workspace,
// status: device word set non-zero if a kernel gave up waiting on its tensor core.
// qr, kr: workspace [BH][T][D] bf16 for RoPE(q), RoPE(k).
template <int D, int M>
cudaError_t tc_forward(const FwdArgs& a, float2* tab, __nv_bfloat16* qr, __nv_bfloat16* kr, int* status,
                       cudaStream_t st);
// RoPE(q), RoPE(k) into qr, kr; with tab != nullptr also the (cos, sin) table [T][D/2].
template <int D>
cudaError_t launch_rope_qk(const void* q, const void* k, __nv_bfloat16* qr, __nv_bfloat16* kr, float2* tab,
                           const RopeTab& rt, const Shape& sh, cudaStream_t st);
template <typename Tin, int D, int M>
cudaError_t simt_backward(const BwdArgs& a, cudaStream_t st);
// Slot-branch backward (query side, reverse adjoint scan, key side, dlog_alpha
// carry); expects the window-branch partials dqw, dkw, dvw and Dv in place.
template <typename Tin, int D, int M>
cudaError_t simt_bwd_slot(const BwdArgs& a, cudaStream_t st);
// bf16 backward: window branch on the tensor core, then the slot branch.
template <int D, int M>
cudaError_t tc_backward(const BwdArgs& a, float2* tab, __nv_bfloat16* qr, __nv_bfloat16* kr, int* status,
                        cudaStream_t st);
// bf16 slot-branch backward on the tensor core (same contract as simt_bwd_slot).
template <int D, int M>
cudaError_t tc_bwd_slot(const BwdArgs& a, const __nv_bfloat16* qr, const __nv_bfloat16* kr, const float2* tab,
                        int* status, cudaStream_t st);
// Key-major window dk / dv (needs the exact D_t in a.Dv).
template <int D>
cudaError_t launch_wkv(const BwdArgs& a, const __nv_bfloat16* qr, const __nv_bfloat16* kr, const float2* tab,
                       int* status, cudaStream_t st);
// bf16 path: reverse adjoint scan (hRK, hRV contributions in; RKb, RVb out) and
// the per-chunk dlog_alpha carry, added to wsDB1 of each chunk's last state row.
cudaError_t launch_adj_scan(const BwdArgs& a, int M, int D, cudaStream_t st);
// bf16 path: the chunk decays exp(G) (into G) and the states entering every
// chunk in bf16 (and fp32 if want_f32), the chunk coefficients formed on chip.
template <int D, int M>
cudaError_t tc_states(const __nv_bfloat16* k, const __nv_bfloat16* v, const float* la, float* SK, float* SV,
                      __nv_bfloat16* SKb, __nv_bfloat16* SVb, float* G, bool want_f32,
                      const StateIO& io, const Shape& sh, int* status, cudaStream_t st);

}  // namespace nha
