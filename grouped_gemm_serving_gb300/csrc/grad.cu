// Gradients of the bf16 grouped GEMM C[p, n] = sum_c A[p, c] B[e, n, c] over
// each expert's rows (training of the MoE layer, "Mixture of Experts in
// transformers"; section 3 of "Hugging Face Transformers: MoE and FP8 kernel
// optimisation": the gradients of sentinel rows must be written, as zeros).
//
//   dgrad  dA[p, c] = sum_n dC[p, n] B[e, n, c]: the grouped GEMM kernel with
//          B read in place as an MN-major operand (the c features contiguous);
//          it writes zeros for the sentinel rows and never reads them.
//   wgrad  dB[e, n, c] = sum over expert e's rows of dC[p, n] A[p, c]: the
//          grouped GEMM's weight-gradient kernel reads dC and A in place as
//          MN-major operands (tcgen05 cta_group::2, A's features as the MMA's
//          256 rows and dC's as its columns, TMEM accumulators, TMA), 64 rows
//          of the expert per k-block; the expert's last, partial k-block comes
//          from a zero-padded copy of its cnt mod 64 last rows (the tails), so
//          no k-block reaches into the next expert's rows.
// Both run on the device from offsets: no host synchronisation.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kMaxE = 256;
constexpr int kTailCols = 512;   // columns per CTA of the tail copy

// The tails of the weight gradient: for expert e with r = cnt_e mod 64 > 0,
// rows [offsets[e + 1] - r, offsets[e + 1]) of X [M_cap, C] go to rows
// [64e, 64e + r) of tail [64E, C] and rows [64e + r, 64e + 64) are zeroed.
// blockIdx.z picks the operand (0: dC, 1: A); a CTA copies kTailCols columns
// of one expert with 16-byte loads and stores.  Offsets that are not a
// monotone prefix within M_cap are reported and no row is read.
__global__ void __launch_bounds__(256)
wgrad_tail_kernel(const uint16_t* __restrict__ dC, int N, const uint16_t* __restrict__ A, int K,
                  const int32_t* __restrict__ offsets, int E, int M_cap, uint16_t* __restrict__ tails, int* err) {
    const int e = blockIdx.x;
    const uint16_t* X = blockIdx.z == 0 ? dC : A;
    const int C = blockIdx.z == 0 ? N : K;
    uint16_t* tail = tails + (blockIdx.z == 0 ? 0 : static_cast<int64_t>(64) * E * N);
    const int c0 = blockIdx.y * kTailCols;
    if (c0 >= C) return;
    int bad = 0;
    for (int i = threadIdx.x; i < E; i += blockDim.x) bad |= offsets[i + 1] < offsets[i];
    if (threadIdx.x == 0) bad |= offsets[0] != 0 || offsets[E] > M_cap;
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) moe::raise_device_error(err, MOE_DEVERR_OFFSETS);
        return;
    }
    const int lo = offsets[e], hi = offsets[e + 1];
    const int r = (hi - lo) % 64;
    if (r == 0) return;   // every k-block of this expert is read in place
    constexpr int kVecs = kTailCols / 8;   // 16-byte vectors per row
    for (int i = threadIdx.x; i < 64 * kVecs; i += blockDim.x) {
        const int j = i / kVecs, c = c0 + 8 * (i % kVecs);
        if (c >= C) continue;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (j < r) v = *reinterpret_cast<const uint4*>(X + static_cast<int64_t>(hi - r + j) * C + c);
        *reinterpret_cast<uint4*>(tail + (static_cast<int64_t>(e) * 64 + j) * C + c) = v;
    }
}

}  // namespace

extern "C" size_t moe_grouped_gemm_dgrad_workspace_size(int E, int N, int K) {
    (void)E; (void)N; (void)K;
    return 0;   // the weights are read in place
}

extern "C" moe_status_t moe_grouped_gemm_dgrad(const void* dC, const void* B, const int32_t* offsets, int E,
                                               int M_cap, int N, int K, void* dA, void* ws, size_t ws_bytes,
                                               moe_stream_t stream) {
    (void)ws; (void)ws_bytes;
    MOE_CHECK_ARG(dC && B && offsets && dA && E >= 1 && E <= kMaxE && M_cap >= 1);
    MOE_CHECK_ARG(N >= 8 && N % 8 == 0 && K >= 8 && K % 8 == 0);
    MOE_CHECK_ARG(moe::aligned16(dC) && moe::aligned16(B) && moe::aligned16(dA));
    return moe::dgrad_gemm(dC, B, offsets, E, M_cap, N, K, dA, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t moe_grouped_gemm_wgrad_workspace_size(int E, int M_cap, int N, int K) {
    if (E < 1 || E > kMaxE || M_cap < 1 || N < 8 || K < 8) return 0;
    return static_cast<size_t>(N + K) * 64 * static_cast<size_t>(E) * 2;   // the tails
}

extern "C" moe_status_t moe_grouped_gemm_wgrad(const void* A, const void* dC, const int32_t* offsets, int E,
                                               int M_cap, int N, int K, void* dB, void* ws, size_t ws_bytes,
                                               moe_stream_t stream) {
    MOE_CHECK_ARG(A && dC && offsets && dB && E >= 1 && E <= kMaxE && M_cap >= 1);
    MOE_CHECK_ARG(N >= 8 && N % 8 == 0 && K >= 8 && K % 8 == 0);
    MOE_CHECK_ARG(moe::aligned16(A) && moe::aligned16(dC) && moe::aligned16(dB));
    const size_t need = moe_grouped_gemm_wgrad_workspace_size(E, M_cap, N, K);
    if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
    MOE_CHECK_ARG(moe::aligned16(ws));
    int* err = moe::device_error_word();
    if (!err) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int span = (N > K ? N : K);
    wgrad_tail_kernel<<<dim3(static_cast<unsigned>(E), (span + kTailCols - 1) / kTailCols, 2), 256, 0, s>>>(
        static_cast<const uint16_t*>(dC), N, static_cast<const uint16_t*>(A), K, offsets, E, M_cap,
        static_cast<uint16_t*>(ws), err);
    MOE_CHECK_LAUNCH();
    return moe::wgrad_gemm(dC, A, ws, offsets, E, M_cap, N, K, dB, s);
}
