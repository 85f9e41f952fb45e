// moe_batched_matmul: the batched expert backend ("Mixture of Experts in
// transformers", pluggable expert backends: batched_mm computes every routed
// (token, expert) product on its own; batched_fp8_matmul of section 1 of
// "Hugging Face Transformers: MoE and FP8 kernel optimisation" is its FP8
// form): out[t*k + j] = W[topk_ids[t, j]] x[t], no weighting, no sum over j.
//
// The products are computed GB300-style rather than one small GEMM per slot:
// the slots are sorted by expert (moe_route_sort on the given ids), the token
// rows permuted into expert order (moe_permute), one grouped GEMM runs over
// them (moe_grouped_gemm, store epilogue; sentinel rows come out as zeros),
// and gather_rows_kernel puts each slot's product row back in slot order.
// Each expert's weights are read once per call, however many slots pick it.
#include <climits>

#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerBlock = kThreads / 32;
constexpr size_t kAlign = 256;

// out[f] = C[row_pos[f]] for every slot f < R: one warp per row, 16-byte
// vectors.  A row_pos outside [0, R) is reported and its row left untouched.
__global__ void __launch_bounds__(kThreads)
gather_rows_kernel(const uint4* __restrict__ C, const int32_t* __restrict__ row_pos, int64_t R, int row_vecs,
                   uint4* __restrict__ out, int* err) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
    for (int64_t f = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5); f < R; f += nwarps) {
        const int p = row_pos[f];
        if (p < 0 || p >= R) {
            if (lane == 0) moe::raise_device_error(err, MOE_DEVERR_ROUTE);
            continue;
        }
        const uint4* src = C + static_cast<int64_t>(p) * row_vecs;
        uint4* dst = out + f * row_vecs;
        for (int v = lane; v < row_vecs; v += 32) dst[v] = __ldg(src + v);
    }
}

struct Carver {
    size_t off = 0;
    size_t take(size_t bytes) {
        const size_t o = off;
        off += (bytes + kAlign - 1) & ~(kAlign - 1);
        return o;
    }
};

struct Layout {
    size_t ids, route, sorted_rows, row_pos, offsets, xp, xps, c, total;
};

bool valid(moe_dtype_t dtype, int T, int K, int k, int E, int N) {
    if (T < 1 || k < 1 || E < 1 || E > 256 || k > E || k > 32 || N < 8 || K < 8) return false;
    if (static_cast<int64_t>(T) * k >= INT_MAX) return false;
    if (dtype == MOE_FP8_E4M3_B128) return K % 128 == 0 && N % 128 == 0;
    return dtype == MOE_BF16 && K % 8 == 0 && N % 8 == 0;
}

Layout layout(moe_dtype_t dtype, int T, int K, int k, int E, int N) {
    const size_t R = static_cast<size_t>(T) * k;
    const bool fp8 = dtype == MOE_FP8_E4M3_B128;
    Carver c;
    Layout l{};
    l.ids = c.take(R * 4);
    l.route = c.take(moe_route_sort_workspace_size(T, E, k));
    l.sorted_rows = c.take(R * 4);
    l.row_pos = c.take(R * 4);
    l.offsets = c.take(static_cast<size_t>(E + 1) * 4);
    l.xp = c.take(R * K * (fp8 ? 1 : 2));
    l.xps = fp8 ? c.take(static_cast<size_t>(K / 128) * R * 4) : 0;
    l.c = c.take(R * N * 2);
    l.total = c.off;
    return l;
}

#define MOE_TRY(call)                          \
    do {                                       \
        const moe_status_t st_ = (call);       \
        if (st_ != MOE_OK) return st_;         \
    } while (0)

}  // namespace

extern "C" size_t moe_batched_matmul_workspace_size(moe_dtype_t dtype, int T, int K, int k, int E, int N) {
    if (!valid(dtype, T, K, k, E, N)) return 0;
    return layout(dtype, T, K, k, E, N).total;
}

extern "C" moe_status_t moe_batched_matmul(moe_dtype_t dtype, const void* x, const float* x_scales, int T, int K,
                                           const int32_t* topk_ids, int k, const void* W, const float* W_scales,
                                           int E, int N, void* out, void* ws, size_t ws_bytes,
                                           moe_stream_t stream) {
    MOE_CHECK_ARG(valid(dtype, T, K, k, E, N));
    MOE_CHECK_ARG(x && topk_ids && W && out);
    MOE_CHECK_ARG(moe::aligned16(x) && moe::aligned16(topk_ids) && moe::aligned16(W) && moe::aligned16(out));
    const bool fp8 = dtype == MOE_FP8_E4M3_B128;
    if (fp8) MOE_CHECK_ARG(x_scales && W_scales && moe::aligned16(x_scales));
    const Layout l = layout(dtype, T, K, k, E, N);
    if (!ws || ws_bytes < l.total) return MOE_ERR_WORKSPACE;
    MOE_CHECK_ARG(moe::aligned16(ws));
    int* err = moe::device_error_word();
    if (!err) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(ws);
    const int R = T * k;
    int32_t* ids = reinterpret_cast<int32_t*>(base + l.ids);
    int32_t* sorted_rows = reinterpret_cast<int32_t*>(base + l.sorted_rows);
    int32_t* row_pos = reinterpret_cast<int32_t*>(base + l.row_pos);
    int32_t* offsets = reinterpret_cast<int32_t*>(base + l.offsets);
    void* xp = base + l.xp;
    float* xps = fp8 ? reinterpret_cast<float*>(base + l.xps) : nullptr;
    void* C = base + l.c;

    // the caller's ids stay untouched (the sort rewrites a bad id as the sentinel)
    MOE_CHECK_CUDA(cudaMemcpyAsync(ids, topk_ids, static_cast<size_t>(R) * 4, cudaMemcpyDeviceToDevice, s));
    MOE_TRY(moe_route_sort(nullptr, nullptr, nullptr, ids, nullptr, T, E, k, 1, sorted_rows, row_pos, offsets,
                           base + l.route, moe_route_sort_workspace_size(T, E, k), stream));
    MOE_TRY(moe_permute(dtype, x, x_scales, T, K, k, sorted_rows, offsets, E, R, xp, xps, stream));
    MOE_TRY(moe_grouped_gemm(dtype, xp, xps, W, W_scales, offsets, E, R, N, K, MOE_EPI_STORE, C, nullptr, stream));
    const int row_vecs = N * 2 / 16;
    const int64_t want = (static_cast<int64_t>(R) + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int cap = 16 * (moe::sm_count() > 0 ? moe::sm_count() : 1);
    const int grid = static_cast<int>(want < cap ? want : cap);
    gather_rows_kernel<<<grid, kThreads, 0, s>>>(static_cast<const uint4*>(C), row_pos, R, row_vecs,
                                                 static_cast<uint4*>(out), err);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}
