// Packed <-> padded token rows for calls over sequences of different lengths.
//
// packed [H, Ttot, width]: the B sequences concatenated along the token axis
// (sequence b in rows cu[b] .. cu[b + 1] - 1); padded [B, H, T, width]:
// sequence b in rows t < T_b = clamp(cu[b + 1] - cu[b], 0, T) of batch entry
// b, the layout the chunkwise kernels read with per-sequence lengths.  One
// warp per padded row moves the row as 16-byte pieces when the row and both
// bases allow it, else as 4-byte words; the pad direction writes zeros in
// the rows past T_b so that the tiles overlapping them read finite padding.
#include "nha_common.cuh"
#include "nha_kernels.h"
#include "nha_prof.h"

namespace nha {

namespace {
constexpr int kVarlenThreads = 256;  // 8 warps, one padded row each

template <typename Word, bool kPad>
__global__ void __launch_bounds__(kVarlenThreads)
varlen_copy_kernel(const void* __restrict__ src, void* __restrict__ dst, const int* __restrict__ cu, int B, int H,
                   int T, int Ttot, int words) {
    const long row = (long)blockIdx.x * (kVarlenThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= (long)B * H * T) return;
    const int t = (int)(row % T), h = (int)((row / T) % H), b = (int)(row / ((long)T * H));
    const int start = __ldg(cu + b), Tb = min(max(__ldg(cu + b + 1) - start, 0), T);
    const long prow = (long)start + t;  // the row's index in the packed array
    const bool live = t < Tb && prow >= 0 && prow < Ttot;
    const size_t pad_off = (size_t)row * words, pk_off = ((size_t)h * Ttot + (size_t)(live ? prow : 0)) * words;
    if (kPad) {
        Word* out = reinterpret_cast<Word*>(dst) + pad_off;
        const Word* in = reinterpret_cast<const Word*>(src) + pk_off;
        for (int e = lane; e < words; e += 32) {
            Word x;
            if (live)
                x = in[e];
            else
                memset(&x, 0, sizeof(Word));
            out[e] = x;
        }
    } else if (live) {
        const Word* in = reinterpret_cast<const Word*>(src) + pad_off;
        Word* out = reinterpret_cast<Word*>(dst) + pk_off;
        for (int e = lane; e < words; e += 32) out[e] = in[e];
    }
}
}  // namespace

cudaError_t launch_varlen_copy(const void* src, void* dst, const int* cu, int B, int H, int T, int Ttot,
                               int row_bytes, bool pad, cudaStream_t st) {
    const long rows = (long)B * H * T;
    if (rows == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((rows + kVarlenThreads / 32 - 1) / (kVarlenThreads / 32));
    const bool wide = row_bytes % 16 == 0 && ((uintptr_t)src & 15u) == 0 && ((uintptr_t)dst & 15u) == 0;
    if (wide) {
        const int words = row_bytes / 16;
        if (pad)
            NHA_LAUNCH("varlen_pad", st, (varlen_copy_kernel<uint4, true><<<grid, kVarlenThreads, 0, st>>>(
                                             src, dst, cu, B, H, T, Ttot, words)));
        else
            NHA_LAUNCH("varlen_unpad", st, (varlen_copy_kernel<uint4, false><<<grid, kVarlenThreads, 0, st>>>(
                                               src, dst, cu, B, H, T, Ttot, words)));
    } else {
        const int words = row_bytes / 4;
        if (pad)
            NHA_LAUNCH("varlen_pad", st, (varlen_copy_kernel<uint32_t, true><<<grid, kVarlenThreads, 0, st>>>(
                                             src, dst, cu, B, H, T, Ttot, words)));
        else
            NHA_LAUNCH("varlen_unpad", st, (varlen_copy_kernel<uint32_t, false><<<grid, kVarlenThreads, 0, st>>>(
                                               src, dst, cu, B, H, T, Ttot, words)));
    }
    return cudaGetLastError();
}

}  // namespace nha
