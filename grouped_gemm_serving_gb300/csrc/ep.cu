// moe_ep_local_ids: the router-side step of expert parallelism as "Mixture of
// Experts in transformers" describes it (section on expert parallelism): the
// experts are sharded on their first dimension, and each rank remaps the
// router's global expert ids to its own local ids; picks of other ranks'
// experts become the local sentinel, so that the rank's sort leaves them out
// of its histogram and its combine skips them (section 2 of the transformers
// MoE/FP8 write-up).  The partial outputs of the ranks then sum to the layer.
//
// One pass over the ids, 16-byte vectors (four slots per thread), grid sized
// to the number of vectors; an id outside [0, E_global] is reported and
// treated as a sentinel.
#include <climits>

#include "common.cuh"

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ int32_t localize(int32_t id, int E_global, int first, int E_local, int* err) {
    if (id < 0 || id > E_global) {
        moe::raise_device_error(err, MOE_DEVERR_ROUTE);
        return E_local;
    }
    return (id >= first && id - first < E_local && id < E_global) ? id - first : E_local;
}

__global__ void __launch_bounds__(kThreads)
ep_local_ids_kernel(const int32_t* __restrict__ ids, int64_t R, int E_global, int first, int E_local,
                    int32_t* __restrict__ local_ids, int* err) {
    const int64_t nvec = R / 4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t v = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; v < nvec; v += stride) {
        const int4 a = reinterpret_cast<const int4*>(ids)[v];
        reinterpret_cast<int4*>(local_ids)[v] =
            make_int4(localize(a.x, E_global, first, E_local, err), localize(a.y, E_global, first, E_local, err),
                      localize(a.z, E_global, first, E_local, err), localize(a.w, E_global, first, E_local, err));
    }
    // the R % 4 slots of the tail
    const int64_t t = nvec * 4 + static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (t < R) local_ids[t] = localize(ids[t], E_global, first, E_local, err);
}

}  // namespace

extern "C" moe_status_t moe_ep_local_ids(const int32_t* topk_ids, int T, int k, int E_global, int first_expert,
                                         int E_local, int32_t* local_ids, moe_stream_t stream) {
    MOE_CHECK_ARG(topk_ids && local_ids && T >= 1 && k >= 1 && static_cast<int64_t>(T) * k < INT_MAX);
    MOE_CHECK_ARG(E_global >= 1 && E_global <= 256 && E_local >= 1 && first_expert >= 0 &&
                  first_expert + E_local <= E_global);
    MOE_CHECK_ARG(moe::aligned16(topk_ids) && moe::aligned16(local_ids));
    int* err = moe::device_error_word();
    if (!err) return MOE_ERR_CUDA;
    const int64_t R = static_cast<int64_t>(T) * k;
    const int64_t nvec = R / 4;
    const int64_t want = (nvec + kThreads - 1) / kThreads;
    const int cap = 8 * (moe::sm_count() > 0 ? moe::sm_count() : 1);   // grid-stride beyond 8 blocks per SM
    const int grid = static_cast<int>(want < 1 ? 1 : want < cap ? want : cap);
    ep_local_ids_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        topk_ids, R, E_global, first_expert, E_local, local_ids, err);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}
