// Gradients of the bf16 grouped GEMM C[p, n] = sum_c A[p, c] B[e, n, c] over
// each expert's rows (training of the MoE layer, "Mixture of Experts in
// transformers"; section 3 of "Hugging Face Transformers: MoE and FP8 kernel
// optimisation": the gradients of sentinel rows must be written, as zeros).
//
//   dgrad  dA[p, c] = sum_n dC[p, n] B[e, n, c]: the grouped GEMM kernel with
//          B read in place as an MN-major operand (the c features contiguous);
//          it writes zeros for the sentinel rows and never reads them.
//   wgrad  dB[e, n, c] = sum over expert e's rows of dC[p, n] A[p, c]: dC and A
//          are transposed so that each expert's rows run along the contraction
//          dimension from a 64-aligned start, zero-padded to whole 64-element
//          k-blocks; then the grouped GEMM's weight-gradient kernel walks each
//          expert's own k-blocks on CTA pairs (tcgen05 cta_group::2, the
//          transposed A as the MMA's 256 rows and the transposed dC's rows as
//          its columns, TMEM accumulators, TMA).
// The padded layout is computed on the device from offsets: no host
// synchronisation.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kTile = 64;      // elements per side of a transposed tile
constexpr int kPitch = 66;     // shared-memory row pitch in elements (33 words: fewer bank conflicts)
constexpr int kColTiles = 8;   // column tiles per CTA of the padded transpose
constexpr int kMaxE = 256;

// One 64 x 64 bf16 tile: rows src_row(r) of src (or zeros), columns
// [c0, c0 + 64) (C a multiple of 8), into dst[c0 + i][q0 + r].  16-byte global
// loads and stores; the tile passes through shared memory as 4-byte words.
template <class SrcRow>
__device__ __forceinline__ void transpose_tile(const uint16_t* __restrict__ src, int64_t src_pitch, int C,
                                               SrcRow src_row, uint16_t* __restrict__ dst, int64_t dst_pitch,
                                               int64_t q0, int64_t q_end, int c0, uint16_t (*tile)[kPitch]) {
    const int t = threadIdx.x;
#pragma unroll
    for (int i = 0; i < 2; ++i) {            // 64 rows x 8 vectors
        const int idx = t + 256 * i, r = idx >> 3, v = idx & 7;
        const int c = c0 + 8 * v;
        const int64_t row = src_row(r);
        uint4 x = make_uint4(0, 0, 0, 0);
        if (row >= 0 && c < C) x = *reinterpret_cast<const uint4*>(src + row * src_pitch + c);
        uint32_t* w = reinterpret_cast<uint32_t*>(&tile[r][8 * v]);
        w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {            // 64 output rows x 8 vectors
        const int idx = t + 256 * i, cc = idx >> 3, v = idx & 7;
        const int c = c0 + cc;
        const int64_t q = q0 + 8 * v;
        if (c < C && q < q_end) {
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                o[j] = static_cast<uint32_t>(tile[8 * v + 2 * j][cc]) |
                       (static_cast<uint32_t>(tile[8 * v + 2 * j + 1][cc]) << 16);
            *reinterpret_cast<uint4*>(dst + static_cast<int64_t>(c) * dst_pitch + q) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    __syncthreads();
}

// Xt[c, q] for q in [0, P): the row of X that expert e's padded run puts at q,
// or zero.  Expert e's run starts at poff[e] = 64 * sum_{e' < e} ceil(cnt_e'/64)
// and holds its cnt_e rows (offsets[e] ..) followed by zeros.  A CTA resolves
// its 64 columns q to source rows once, then transposes kColTiles tiles.
__global__ void __launch_bounds__(256)
pad_transpose_kernel(const uint16_t* __restrict__ X, int C, const int32_t* __restrict__ offsets, int E,
                     int M_cap, int64_t P, uint16_t* __restrict__ Xt, int* err) {
    __shared__ int poff[kMaxE + 1];
    __shared__ int bad;
    __shared__ int64_t srow[kTile];
    __shared__ __align__(16) uint16_t tile[kTile][kPitch];
    const int tx = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (warp == 0) {   // check offsets; prefix of the padded counts, 8 experts per lane
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
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) moe::raise_device_error(err, MOE_DEVERR_OFFSETS);
        return;
    }
    const int64_t q0 = static_cast<int64_t>(blockIdx.x) * kTile;
    if (threadIdx.x < kTile) {
        const int64_t q = q0 + threadIdx.x;
        int64_t row = -1;
        if (q < poff[E]) {
            int lo = 0, hi = E;   // largest e with poff[e] <= q
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (poff[mid] <= q) lo = mid; else hi = mid;
            }
            const int64_t j = q - poff[lo];
            if (j < offsets[lo + 1] - offsets[lo]) row = offsets[lo] + j;
        }
        srow[threadIdx.x] = row;
    }
    __syncthreads();
    for (int ct = 0; ct < kColTiles; ++ct) {
        const int c0 = (blockIdx.y * kColTiles + ct) * kTile;
        if (c0 >= C) break;
        transpose_tile(X, C, C, [&](int r) { return srow[r]; }, Xt, P, q0, P, c0, tile);
    }
}

// Columns of the padded layout: enough for any offsets with offsets[E] <= M_cap.
int64_t padded_cols(int E, int M_cap) {
    return (static_cast<int64_t>(M_cap) + 63) / 64 * 64 + static_cast<int64_t>(E) * 64;
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
    const int64_t qb = P / kTile;   // P is a multiple of 64
    const int span = kTile * kColTiles;
    pad_transpose_kernel<<<dim3(static_cast<unsigned>(qb), (N + span - 1) / span), 256, 0, s>>>(
        static_cast<const uint16_t*>(dC), N, offsets, E, M_cap, P, dCt, err);
    MOE_CHECK_LAUNCH();
    pad_transpose_kernel<<<dim3(static_cast<unsigned>(qb), (K + span - 1) / span), 256, 0, s>>>(
        static_cast<const uint16_t*>(A), K, offsets, E, M_cap, P, At, err);
    MOE_CHECK_LAUNCH();
    return moe::wgrad_gemm(dCt, At, P, offsets, E, M_cap, N, K, dB, s);
}
