// Data movement around the grouped GEMMs (section 1 of "LlamaFactory Triton
// fused MoE kernel": moe_scatter before the first grouped GEMM, silu(gate) *
// up between them, moe_gather after the second), all HBM-bound: every
// kernel moves 16-byte vectors with coalesced loads and stores.
#include <climits>

#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerBlock = kThreads / 32;

// Reads L = offsets[E] and checks 0 <= L <= M_cap; a bad value is reported
// and the caller skips all work.
__device__ __forceinline__ int live_rows(const int32_t* offsets, int E, int M_cap, int* err) {
    const int L = offsets[E];
    if (L < 0 || L > M_cap) {
        moe::raise_device_error(err, MOE_DEVERR_OFFSETS);
        return -1;
    }
    return L;
}

// xp[p] = x[sorted_rows[p] / k] for p < L; one warp per (row, segment)
// (the loop also covers a smaller grid).  row_vecs = bytes per row / 16; a
// row is split into segs segments of seg_vecs vectors (segs = 1 unless there
// are too few rows to fill the GPU).  FP8 rows also move their group scales
// into the group-major layout xp_scales[g * M_cap + p]: the warp of every
// eighth row (segment 0) moves the scales of rows p .. p+7, so that a group's
// eight values fill one 32-byte sector instead of eight rows each scattering
// a value over every group's line.
__global__ void __launch_bounds__(kThreads, 8)   // 32 registers: 64 warps per SM
permute_kernel(const uint4* __restrict__ x, const float* __restrict__ x_scales, int T, int k,
               int row_vecs, int segs, int seg_vecs, int G, const int32_t* __restrict__ sorted_rows,
               const int32_t* __restrict__ offsets, int E, int M_cap, uint4* __restrict__ xp,
               float* __restrict__ xp_scales, int* err) {
    const int L = live_rows(offsets, E, M_cap, err);
    if (L < 0) return;
    const int lane = threadIdx.x & 31;
    const int warp0 = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int nwarps = gridDim.x * kWarpsPerBlock;
    const int64_t n = static_cast<int64_t>(L) * segs;
    for (int64_t w = warp0; w < n; w += nwarps) {
        const int p = static_cast<int>(w / segs);
        const int seg = static_cast<int>(w - static_cast<int64_t>(p) * segs);
        if (x_scales && seg == 0 && (p & 7) == 0) {
            // lane l: row p + l % 8, groups l / 8, l / 8 + 4, ...; a row
            // with a bad slot is skipped here and reported by its own warp
            const int pr = p + (lane & 7);
            int tr = -1;
            if (pr < L) {
                const int sr = sorted_rows[pr];
                if (sr >= 0 && sr / k < T) tr = sr / k;
            }
            if (tr >= 0)
                for (int g = lane >> 3; g < G; g += 4)
                    xp_scales[static_cast<int64_t>(g) * M_cap + pr] = __ldg(x_scales + static_cast<int64_t>(tr) * G + g);
        }
        const int slot = sorted_rows[p];
        const int t = slot / k;
        if (slot < 0 || t >= T) {
            if (seg == 0) moe::raise_device_error(err, MOE_DEVERR_ROUTE);
            continue;
        }
        const uint4* src = x + static_cast<int64_t>(t) * row_vecs;
        uint4* dst = xp + static_cast<int64_t>(p) * row_vecs;
        const int v_end = min(row_vecs, (seg + 1) * seg_vecs);
#pragma unroll 4
        for (int i = seg * seg_vecs + lane; i < v_end; i += 32) dst[i] = __ldg(src + i);
    }
}

// h = silu(g) * u over 8 columns per thread; rows >= L are zero.
__global__ void __launch_bounds__(kThreads)
swiglu_kernel(const uint4* __restrict__ Y1, const int32_t* __restrict__ offsets, int E, int M_cap,
              int I, uint4* __restrict__ h, int* err) {
    const int L = live_rows(offsets, E, M_cap, err);
    if (L < 0) return;
    const int cv = I / 8;                       // 16-byte vectors per h row
    const int64_t n = static_cast<int64_t>(M_cap) * cv;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int64_t p = i / cv;
        const int c = static_cast<int>(i - p * cv);
        uint4 o = make_uint4(0, 0, 0, 0);
        if (p < L) {
            const uint4 g = __ldg(Y1 + p * 2 * cv + c);
            const uint4 u = __ldg(Y1 + p * 2 * cv + cv + c);
            const uint32_t gs[4] = {g.x, g.y, g.z, g.w}, us[4] = {u.x, u.y, u.z, u.w};
            uint32_t os[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float g0 = moe::bf16_lo(gs[j]), g1 = moe::bf16_hi(gs[j]);
                const float h0 = g0 / (1.0f + expf(-g0)) * moe::bf16_lo(us[j]);
                const float h1 = g1 / (1.0f + expf(-g1)) * moe::bf16_hi(us[j]);
                os[j] = moe::pack_bf16x2(h0, h1);
            }
            o = make_uint4(os[0], os[1], os[2], os[3]);
        }
        h[i] = o;
    }
}

// out[t] = sum_j w[t,j] * Y2[row_pos[t*k+j]] over non-sentinel slots, fp32 in
// j order; one warp per token, 8 columns (one 16-byte vector) per lane step.
// KG slots are loaded at a time.  With KG = 4 (top-k up to 4) the kernel
// fits 64 registers, so four blocks share an SM: a 4096-token grid then runs
// in one wave with 32 warps per SM, where KG = 8 (118 registers) allows two
// blocks and left the second wave two-thirds full.
template <int KG, int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
combine_kernel(const uint4* __restrict__ Y2, const int32_t* __restrict__ ids,
               const float* __restrict__ w, const int32_t* __restrict__ row_pos, int T, int k,
               int row_vecs, int E, int64_t M_cap, uint4* __restrict__ out, int* err) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (t >= T) return;
    // lane j < k holds slot j's row (or -1) and weight
    int my_row = -1;
    float my_w = 0.0f;
    if (lane < k) {
        const int64_t f = static_cast<int64_t>(t) * k + lane;
        const int id = ids[f];
        if (id != E) {
            const int pos = row_pos[f];
            if (pos < 0 || pos >= M_cap) {
                moe::raise_device_error(err, MOE_DEVERR_ROUTE);
            } else {
                my_row = pos;
                my_w = w[f];
            }
        }
    }
    uint4* dst = out + static_cast<int64_t>(t) * row_vecs;
    // Two 32-vector chunks per pass.  The trip counts are the same for every
    // lane, so the shuffles see a full warp.  Up to KG slots' vectors of both
    // chunks are loaded before any is used, so they are in flight together;
    // they are then accumulated in slot order.
    for (int c0 = 0; c0 < row_vecs; c0 += 64) {
        const int ca = c0 + lane, cb = c0 + 32 + lane;
        const bool ina = ca < row_vecs, inb = cb < row_vecs;
        float acc[2][8];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[h][i] = 0.0f;
        for (int j0 = 0; j0 < k; j0 += KG) {
            uint4 va[KG], vb[KG];
            float wj[KG];
            bool use[KG];
#pragma unroll
            for (int g = 0; g < KG; ++g) {
                const int j = j0 + g;
                const int row = __shfl_sync(0xffffffffu, my_row, j & 31);
                wj[g] = __shfl_sync(0xffffffffu, my_w, j & 31);
                use[g] = j < k && row >= 0;   // sentinel slots are skipped
                const uint4* src = Y2 + static_cast<int64_t>(row) * row_vecs;
                va[g] = use[g] && ina ? __ldg(src + ca) : make_uint4(0, 0, 0, 0);
                vb[g] = use[g] && inb ? __ldg(src + cb) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int g = 0; g < KG; ++g) {
                if (!use[g]) continue;
                const uint32_t a4[4] = {va[g].x, va[g].y, va[g].z, va[g].w};
                const uint32_t b4[4] = {vb[g].x, vb[g].y, vb[g].z, vb[g].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[0][2 * i] = fmaf(wj[g], moe::bf16_lo(a4[i]), acc[0][2 * i]);
                    acc[0][2 * i + 1] = fmaf(wj[g], moe::bf16_hi(a4[i]), acc[0][2 * i + 1]);
                    acc[1][2 * i] = fmaf(wj[g], moe::bf16_lo(b4[i]), acc[1][2 * i]);
                    acc[1][2 * i + 1] = fmaf(wj[g], moe::bf16_hi(b4[i]), acc[1][2 * i + 1]);
                }
            }
        }
        if (ina)
            dst[ca] = make_uint4(moe::pack_bf16x2(acc[0][0], acc[0][1]), moe::pack_bf16x2(acc[0][2], acc[0][3]),
                                 moe::pack_bf16x2(acc[0][4], acc[0][5]), moe::pack_bf16x2(acc[0][6], acc[0][7]));
        if (inb)
            dst[cb] = make_uint4(moe::pack_bf16x2(acc[1][0], acc[1][1]), moe::pack_bf16x2(acc[1][2], acc[1][3]),
                                 moe::pack_bf16x2(acc[1][4], acc[1][5]), moe::pack_bf16x2(acc[1][6], acc[1][7]));
    }
}

// The same sum for small T, with several warps per token so that the grid
// still fills the GPU: warp w handles token w / segs, vectors
// [seg * seg_vecs, ...) of its row.  Same arithmetic and order per element.
constexpr int kCombineChunks = 1;   // 32-vector chunks a warp loads per pass

__global__ void __launch_bounds__(kThreads)
combine_split_kernel(const uint4* __restrict__ Y2, const int32_t* __restrict__ ids,
               const float* __restrict__ w, const int32_t* __restrict__ row_pos, int T, int k,
               int row_vecs, int segs, int seg_vecs, int E, int64_t M_cap, uint4* __restrict__ out,
               int* err) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    const int t = static_cast<int>(gw / segs);
    const int seg = static_cast<int>(gw - static_cast<int64_t>(t) * segs);
    if (t >= T) return;
    // lane j < k holds slot j's row (or -1) and weight
    int my_row = -1;
    float my_w = 0.0f;
    if (lane < k) {
        const int64_t f = static_cast<int64_t>(t) * k + lane;
        const int id = ids[f];
        if (id != E) {
            const int pos = row_pos[f];
            if (pos < 0 || pos >= M_cap) {
                if (seg == 0) moe::raise_device_error(err, MOE_DEVERR_ROUTE);
            } else {
                my_row = pos;
                my_w = w[f];
            }
        }
    }
    uint4* dst = out + static_cast<int64_t>(t) * row_vecs;
    const int v_end = min(row_vecs, (seg + 1) * seg_vecs);
    // The trip counts are the same for every lane, so the shuffles see a full
    // warp.  Up to KG slots' vectors of every chunk are loaded before any is
    // used; they are then accumulated in slot order.
    constexpr int KG = 8, CH = kCombineChunks;
    for (int c0 = seg * seg_vecs; c0 < v_end; c0 += 32 * CH) {
        float acc[CH][8];
#pragma unroll
        for (int h = 0; h < CH; ++h)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[h][i] = 0.0f;
        for (int j0 = 0; j0 < k; j0 += KG) {
            uint4 v[KG][CH];
            float wj[KG];
            bool use[KG];
#pragma unroll
            for (int g = 0; g < KG; ++g) {
                const int j = j0 + g;
                const int row = __shfl_sync(0xffffffffu, my_row, j & 31);
                wj[g] = __shfl_sync(0xffffffffu, my_w, j & 31);
                use[g] = j < k && row >= 0;   // sentinel slots are skipped
#pragma unroll
                for (int h = 0; h < CH; ++h) {
                    const int c = c0 + 32 * h + lane;
                    v[g][h] = use[g] && c < v_end ? __ldg(Y2 + static_cast<int64_t>(row) * row_vecs + c)
                                                  : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int g = 0; g < KG; ++g) {
                if (!use[g]) continue;
#pragma unroll
                for (int h = 0; h < CH; ++h) {
                    const uint32_t vs[4] = {v[g][h].x, v[g][h].y, v[g][h].z, v[g][h].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[h][2 * i] = fmaf(wj[g], moe::bf16_lo(vs[i]), acc[h][2 * i]);
                        acc[h][2 * i + 1] = fmaf(wj[g], moe::bf16_hi(vs[i]), acc[h][2 * i + 1]);
                    }
                }
            }
        }
#pragma unroll
        for (int h = 0; h < CH; ++h) {
            const int c = c0 + 32 * h + lane;
            if (c < v_end)
                dst[c] = make_uint4(moe::pack_bf16x2(acc[h][0], acc[h][1]), moe::pack_bf16x2(acc[h][2], acc[h][3]),
                                    moe::pack_bf16x2(acc[h][4], acc[h][5]), moe::pack_bf16x2(acc[h][6], acc[h][7]));
        }
    }
}

int persistent_blocks(int64_t work_warps) {
    const int64_t want = (work_warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int64_t cap = static_cast<int64_t>(moe::sm_count() > 0 ? moe::sm_count() : 148) * 8;
    return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

extern "C" moe_status_t moe_permute(moe_dtype_t dtype, const void* x, const float* x_scales, int T,
                                    int H, int k, const int32_t* sorted_rows,
                                    const int32_t* offsets, int E, int M_cap, void* xp,
                                    float* xp_scales, moe_stream_t stream) {
    MOE_CHECK_ARG(x && sorted_rows && offsets && xp && T >= 1 && H >= 1 && k >= 1 && E >= 1);
    MOE_CHECK_ARG(static_cast<int64_t>(T) * k <= M_cap && M_cap < INT_MAX);
    MOE_CHECK_ARG(moe::aligned16(x) && moe::aligned16(xp));
    const bool fp8 = dtype == MOE_FP8_E4M3_B128;
    if (!fp8 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    int row_vecs, G = 0;
    if (fp8) {
        MOE_CHECK_ARG(H % 128 == 0 && x_scales && xp_scales);
        row_vecs = H / 16;
        G = H / 128;
    } else {
        MOE_CHECK_ARG(H % 8 == 0);
        row_vecs = H / 8;
    }
    int* err = moe::device_error_word();
    if (!err) return MOE_ERR_CUDA;
    // fewer rows than 8 warps per SM: split rows into segments of whole
    // 32-vector chunks until there are ~32 warps per SM
    const int sm = moe::sm_count() > 0 ? moe::sm_count() : 148;
    const int max_segs = (row_vecs + 31) / 32;
    const int64_t want = M_cap < sm * kWarpsPerBlock ? (static_cast<int64_t>(sm) * 32 + M_cap - 1) / M_cap : 1;
    const int segs = static_cast<int>(want < max_segs ? (want > 1 ? want : 1) : max_segs);
    const int seg_vecs = ((row_vecs + segs - 1) / segs + 31) / 32 * 32;
    // one warp per (row, segment): the block scheduler balances the rows,
    // where a grid capped at a few blocks per SM dealt them out unevenly
    const int64_t units = static_cast<int64_t>(M_cap) * segs;
    MOE_CHECK_ARG((units + kWarpsPerBlock - 1) / kWarpsPerBlock < INT_MAX);
    permute_kernel<<<static_cast<int>((units + kWarpsPerBlock - 1) / kWarpsPerBlock), kThreads, 0,
                     reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(x), fp8 ? x_scales : nullptr, T, k, row_vecs, segs, seg_vecs, G, sorted_rows,
        offsets, E, M_cap, static_cast<uint4*>(xp), fp8 ? xp_scales : nullptr, err);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

extern "C" moe_status_t moe_swiglu(const void* Y1, const int32_t* offsets, int E, int M_cap, int I,
                                   void* h, moe_stream_t stream) {
    MOE_CHECK_ARG(Y1 && offsets && h && E >= 1 && M_cap >= 1 && I >= 8 && I % 8 == 0);
    MOE_CHECK_ARG(moe::aligned16(Y1) && moe::aligned16(h));
    int* err = moe::device_error_word();
    if (!err) return MOE_ERR_CUDA;
    const int64_t vecs = static_cast<int64_t>(M_cap) * (I / 8);
    const int blocks = persistent_blocks((vecs + 31) / 32);
    swiglu_kernel<<<blocks, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(Y1), offsets, E, M_cap, I, static_cast<uint4*>(h), err);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

extern "C" moe_status_t moe_combine(const void* Y2, const int32_t* topk_ids, const float* topk_w,
                                    const int32_t* row_pos, int T, int k, int H, int E, void* out,
                                    moe_stream_t stream) {
    MOE_CHECK_ARG(Y2 && topk_ids && topk_w && row_pos && out);
    MOE_CHECK_ARG(T >= 1 && k >= 1 && k <= 32 && E >= 1 && H >= 8 && H % 8 == 0);
    MOE_CHECK_ARG(moe::aligned16(Y2) && moe::aligned16(out));
    int* err = moe::device_error_word();
    if (!err) return MOE_ERR_CUDA;
    const int sm = moe::sm_count() > 0 ? moe::sm_count() : 148;
    if (T >= sm * kWarpsPerBlock) {   // at least a block of tokens per SM: one warp per token
        const int blocks = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
        auto kern = k <= 4 ? combine_kernel<4, 4> : combine_kernel<8, 1>;
        kern<<<blocks, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
            static_cast<const uint4*>(Y2), topk_ids, topk_w, row_pos, T, k, H / 8, E,
            static_cast<int64_t>(T) * k, static_cast<uint4*>(out), err);
        MOE_CHECK_LAUNCH();
        return MOE_OK;
    }
    // few tokens: split each row over warps until the grid has ~32 warps per SM
    const int row_vecs = H / 8, step = 32 * kCombineChunks;
    const int max_segs = (row_vecs + step - 1) / step;
    const int64_t want = (static_cast<int64_t>(sm) * 32 + T - 1) / T;
    const int segs = static_cast<int>(want < max_segs ? (want > 1 ? want : 1) : max_segs);
    const int seg_vecs = ((row_vecs + segs - 1) / segs + step - 1) / step * step;
    const int64_t blocks = (static_cast<int64_t>(T) * segs + kWarpsPerBlock - 1) / kWarpsPerBlock;
    combine_split_kernel<<<static_cast<int>(blocks), kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(Y2), topk_ids, topk_w, row_pos, T, k, row_vecs, segs, seg_vecs, E,
        static_cast<int64_t>(T) * k, static_cast<uint4*>(out), err);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}
