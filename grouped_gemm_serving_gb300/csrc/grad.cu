// Gradients of the bf16 grouped GEMM C[p, n] = sum_c A[p, c] B[e, n, c] over
// each expert's rows (training of the MoE layer, "Mixture of Experts in
// transformers"; section 3 of "Hugging Face Transformers: MoE and FP8 kernel
// optimisation": the gradients of sentinel rows must be written, as zeros).
//
//   dgrad  dA[p, c] = sum_n dC[p, n] B[e, n, c]: the forward grouped GEMM
//          (moe_grouped_gemm) on B transposed to [E, K, N]; it writes zeros for
//          the sentinel rows and never reads them.
//   wgrad  dB[e, n, c] = sum over expert e's rows of dC[p, n] A[p, c]: dC and A
//          are transposed so that each expert's rows run along the contraction
//          dimension from a 64-aligned start, zero-padded to whole 64-element
//          k-blocks; then the grouped GEMM's weight-gradient mode walks each
//          expert's own k-blocks (tcgen05, TMEM accumulators, TMA).
// The padded layout is computed on the device from offsets: no host
// synchronisation.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kTile = 32;
constexpr int kMaxE = 256;

// Wt[e, k, n] = W[e, n, k]; 32x32 tiles through shared memory.
__global__ void __launch_bounds__(256)
transpose_weights_kernel(const uint16_t* __restrict__ W, int N, int K, uint16_t* __restrict__ Wt) {
    __shared__ uint16_t tile[kTile][kTile + 1];
    const int e = blockIdx.z, n0 = blockIdx.y * kTile, k0 = blockIdx.x * kTile;
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int64_t base = static_cast<int64_t>(e) * N * K;
    for (int i = ty; i < kTile; i += 8) {
        const int n = n0 + i, k = k0 + tx;
        tile[i][tx] = n < N && k < K ? W[base + static_cast<int64_t>(n) * K + k] : 0;
    }
    __syncthreads();
    for (int i = ty; i < kTile; i += 8) {
        const int k = k0 + i, n = n0 + tx;
        if (k < K && n < N) Wt[base + static_cast<int64_t>(k) * N + n] = tile[tx][i];
    }
}

// Xt[c, q] for q in [0, P): the row of X that expert e's padded run puts at q,
// or zero.  Expert e's run starts at poff[e] = 64 * sum_{e' < e} ceil(cnt_e'/64)
// and holds its cnt_e rows (offsets[e] ..) followed by zeros.
__global__ void __launch_bounds__(256)
pad_transpose_kernel(const uint16_t* __restrict__ X, int C, const int32_t* __restrict__ offsets, int E,
                     int M_cap, int64_t P, uint16_t* __restrict__ Xt, int* err) {
    __shared__ int poff[kMaxE + 1];
    __shared__ int bad;
    __shared__ uint16_t tile[kTile][kTile + 1];
    const int tx = threadIdx.x, ty = threadIdx.y;
    if (ty == 0) {   // one warp: check offsets; prefix of the padded counts, 8 experts per lane
        int v[8], sum = 0, b = tx == 0 && (offsets[0] != 0 || offsets[E] > M_cap);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = tx * 8 + i;
            v[i] = 0;
            if (e < E) {
                const int cnt = offsets[e + 1] - offsets[e];
                if (cnt < 0) b = 1;
                v[i] = cnt > 0 ? (cnt + 63) / 64 * 64 : 0;
            }
            sum += v[i];
        }
        b = __any_sync(0xffffffffu, b);
        if (tx == 0) bad = b;
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (tx >= off) incl += o;
        }
        int run = incl - sum;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = tx * 8 + i;
            if (e < E) { poff[e] = run; run += v[i]; }
        }
        if (tx == 31) poff[E] = incl;
    }
    __syncthreads();
    if (bad || poff[E] > P) {   // offsets that are not a monotone prefix within M_cap: nothing is read
        if (blockIdx.x == 0 && blockIdx.y == 0 && tx == 0 && ty == 0) moe::raise_device_error(err, MOE_DEVERR_OFFSETS);
        return;
    }
    const int64_t q0 = static_cast<int64_t>(blockIdx.x) * kTile;
    const int c0 = blockIdx.y * kTile;
    for (int i = ty; i < kTile; i += 8) {
        const int64_t q = q0 + i;
        const int c = c0 + tx;
        uint16_t v = 0;
        if (q < poff[E] && c < C) {
            int lo = 0, hi = E;   // largest e with poff[e] <= q
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (poff[mid] <= q) lo = mid; else hi = mid;
            }
            const int64_t j = q - poff[lo];
            if (j < offsets[lo + 1] - offsets[lo]) v = X[(offsets[lo] + j) * C + c];
        }
        tile[i][tx] = v;
    }
    __syncthreads();
    for (int i = ty; i < kTile; i += 8) {
        const int c = c0 + i;
        const int64_t q = q0 + tx;
        if (c < C && q < P) Xt[static_cast<int64_t>(c) * P + q] = tile[tx][i];
    }
}

// Columns of the padded layout: enough for any offsets with offsets[E] <= M_cap.
int64_t padded_cols(int E, int M_cap) {
    return (static_cast<int64_t>(M_cap) + 63) / 64 * 64 + static_cast<int64_t>(E) * 64;
}

}  // namespace

extern "C" size_t moe_grouped_gemm_dgrad_workspace_size(int E, int N, int K) {
    if (E < 1 || E > kMaxE || N < 8 || K < 8) return 0;
    return static_cast<size_t>(E) * N * K * 2;
}

extern "C" moe_status_t moe_grouped_gemm_dgrad(const void* dC, const void* B, const int32_t* offsets, int E,
                                               int M_cap, int N, int K, void* dA, void* ws, size_t ws_bytes,
                                               moe_stream_t stream) {
    MOE_CHECK_ARG(dC && B && offsets && dA && E >= 1 && E <= kMaxE && M_cap >= 1);
    MOE_CHECK_ARG(N >= 8 && N % 8 == 0 && K >= 8 && K % 8 == 0);
    MOE_CHECK_ARG(moe::aligned16(dC) && moe::aligned16(B) && moe::aligned16(dA));
    const size_t need = moe_grouped_gemm_dgrad_workspace_size(E, N, K);
    if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
    MOE_CHECK_ARG(moe::aligned16(ws));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint16_t* Bt = static_cast<uint16_t*>(ws);
    const dim3 grid((K + kTile - 1) / kTile, (N + kTile - 1) / kTile, E);
    transpose_weights_kernel<<<grid, dim3(kTile, 8), 0, s>>>(static_cast<const uint16_t*>(B), N, K, Bt);
    MOE_CHECK_LAUNCH();
    // dA = dC Bt[e]^T with Bt [E, K, N]: the forward GEMM, N and K exchanged
    return moe_grouped_gemm(MOE_BF16, dC, nullptr, Bt, nullptr, offsets, E, M_cap, K, N, MOE_EPI_STORE, dA,
                            nullptr, stream);
}

extern "C" size_t moe_grouped_gemm_wgrad_workspace_size(int E, int M_cap, int N, int K) {
    if (E < 1 || E > kMaxE || M_cap < 1 || N < 8 || K < 8) return 0;
    return static_cast<size_t>(N + K) * static_cast<size_t>(padded_cols(E, M_cap)) * 2;
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
    const int64_t P = padded_cols(E, M_cap);
    MOE_CHECK_ARG(P < INT_MAX);
    uint16_t* dCt = static_cast<uint16_t*>(ws);             // [N, P]
    uint16_t* At = dCt + static_cast<int64_t>(N) * P;       // [K, P]
    const int64_t qb = (P + kTile - 1) / kTile;
    pad_transpose_kernel<<<dim3(static_cast<unsigned>(qb), (N + kTile - 1) / kTile), dim3(kTile, 8), 0, s>>>(
        static_cast<const uint16_t*>(dC), N, offsets, E, M_cap, P, dCt, err);
    MOE_CHECK_LAUNCH();
    pad_transpose_kernel<<<dim3(static_cast<unsigned>(qb), (K + kTile - 1) / kTile), dim3(kTile, 8), 0, s>>>(
        static_cast<const uint16_t*>(A), K, offsets, E, M_cap, P, At, err);
    MOE_CHECK_LAUNCH();
    return moe::wgrad_gemm(dCt, At, P, offsets, E, M_cap, N, K, dB, s);
}
