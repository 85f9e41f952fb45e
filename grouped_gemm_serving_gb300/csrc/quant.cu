// Fine-grained FP8 quantisation (section 1 of "Hugging Face Transformers:
// MoE and FP8 kernel optimisation": fp8_act_quant / per_token_cast_to_fp8 for
// activations, 128x128-block scaled e4m3 weights for grouped_fp8_matmul).
//
// Scale rule for a group or block: s = amax / 448 in fp32 (IEEE division),
// s = 1 when amax = 0; each element becomes e4m3_rn_satfinite(v / s), the
// division again IEEE fp32 and the conversion the hardware's
// round-to-nearest-even, saturating cvt.
#include <cuda_fp8.h>

#include "common.cuh"

namespace {

__device__ __forceinline__ float fp8_scale(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, float s) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(a, s), __fdiv_rn(b, s)), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(c, s), __fdiv_rn(d, s)), __NV_SATFINITE, __NV_E4M3);
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// A half-warp per (row, 128-column group): lane l of the half holds columns
// 8l .. 8l+7 (one 16-byte load), so a warp covers two groups at a time.  Each
// warp walks its pairs of groups a grid-stride apart, kUnroll at a time with
// all their loads issued first, so that enough bytes are in flight.  The
// per-element IEEE divisions dominate the instruction count.
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(256)
act_quant_kernel(const uint4* __restrict__ x, int64_t groups, uint2* __restrict__ q,
                 float* __restrict__ scales) {
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
    for (int64_t base = warp; base * 2 < groups; base += nwarps * kUnroll) {
        uint4 v[kUnroll];
        int64_t grp[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {       // group = 2 * pair + half, 256 bytes each
            grp[u] = 2 * (base + u * nwarps) + half;
            v[u] = grp[u] < groups ? __ldg(x + grp[u] * 16 + hl) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            float f[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                f[2 * i] = moe::bf16_lo(w[i]);
                f[2 * i + 1] = moe::bf16_hi(w[i]);
            }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            const float sc = fp8_scale(amax);
            if (grp[u] < groups) {
                q[grp[u] * 16 + hl] = make_uint2(quant4(f[0], f[1], f[2], f[3], sc), quant4(f[4], f[5], f[6], f[7], sc));
                if (hl == 0) scales[grp[u]] = sc;
            }
        }
    }
}

// One CTA per (expert, 128-row block, 128-column block); thread t covers row
// t/2 of the block, columns (t%2)*64 .. +63.
__global__ void __launch_bounds__(256)
weight_quant_kernel(const uint16_t* __restrict__ w, int N, int K, uint8_t* __restrict__ q,
                    float* __restrict__ scales) {
    __shared__ float warp_max[8];
    const int NB = (N + 127) / 128, KB = K / 128;
    const int kb = blockIdx.x % KB;
    const int nb = (blockIdx.x / KB) % NB;
    const int64_t e = blockIdx.x / (static_cast<int64_t>(KB) * NB);
    const int r = nb * 128 + (threadIdx.x >> 1);
    const int c0 = kb * 128 + (threadIdx.x & 1) * 64;
    const bool live = r < N;
    const uint4* src = reinterpret_cast<const uint4*>(w + (e * N + r) * static_cast<int64_t>(K) + c0);
    uint4 v[8];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = live ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
        const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            amax = fmaxf(amax, fmaxf(fabsf(moe::bf16_lo(u[j])), fabsf(moe::bf16_hi(u[j]))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, warp_max[i]);
    const float s = fp8_scale(amax);
    if (threadIdx.x == 0) scales[(e * NB + nb) * KB + kb] = s;
    if (!live) return;
    uint4* dst = reinterpret_cast<uint4*>(q + (e * N + r) * static_cast<int64_t>(K) + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 a = v[2 * i], b = v[2 * i + 1];
        uint4 o;
        o.x = quant4(moe::bf16_lo(a.x), moe::bf16_hi(a.x), moe::bf16_lo(a.y), moe::bf16_hi(a.y), s);
        o.y = quant4(moe::bf16_lo(a.z), moe::bf16_hi(a.z), moe::bf16_lo(a.w), moe::bf16_hi(a.w), s);
        o.z = quant4(moe::bf16_lo(b.x), moe::bf16_hi(b.x), moe::bf16_lo(b.y), moe::bf16_hi(b.y), s);
        o.w = quant4(moe::bf16_lo(b.z), moe::bf16_hi(b.z), moe::bf16_lo(b.w), moe::bf16_hi(b.w), s);
        dst[i] = o;
    }
}

}  // namespace

extern "C" moe_status_t moe_act_quant_fp8(const void* x, int M, int K, uint8_t* q, float* scales,
                                          moe_stream_t stream) {
    MOE_CHECK_ARG(x && q && scales && M >= 1 && K >= 128 && K % 128 == 0);
    MOE_CHECK_ARG(moe::aligned16(x) && moe::aligned16(q) && moe::aligned16(scales));
    const int64_t groups = static_cast<int64_t>(M) * (K / 128);
    const int64_t pairs = (groups + 1) / 2;                      // a warp handles a pair at a time
    // one pair per warp up to a full GPU of warps; beyond that each warp
    // takes several pairs, kUnroll of them in flight
    const int64_t cap = static_cast<int64_t>(moe::sm_count() > 0 ? moe::sm_count() : 148) * 64;
    const int64_t warps = pairs < cap ? pairs : cap;
    const int64_t blocks = (warps + 7) / 8;
    act_quant_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(x), groups, reinterpret_cast<uint2*>(q), scales);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

extern "C" moe_status_t moe_weight_quant_fp8(const void* w, int E, int N, int K, uint8_t* q,
                                             float* scales, moe_stream_t stream) {
    MOE_CHECK_ARG(w && q && scales && E >= 1 && N >= 1 && K >= 128 && K % 128 == 0);
    MOE_CHECK_ARG(moe::aligned16(w) && moe::aligned16(q) && moe::aligned16(scales));
    const int64_t blocks = static_cast<int64_t>(E) * ((N + 127) / 128) * (K / 128);
    MOE_CHECK_ARG(blocks < INT32_MAX);
    weight_quant_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(w), N, K, q, scales);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}
