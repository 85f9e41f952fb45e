// moe_route_sort: top-k routing, sentinel marking, per-expert histogram and
// the stable counting sort of the routed slots by expert id.
//
// Routing follows "Mixture of Experts in transformers" (MoE basics: the
// router picks k of the E experts per token); the sort follows section 2 of
// "Hugging Face Transformers: MoE and FP8 kernel optimisation": sentinel
// slots (id E) are left out of the histogram and sort after every live slot,
// so offsets[E] counts the live rows and no sentinel lands on the last expert.
//
// Kernels (one stream, no host synchronisation):
//   1. route_topk_hist  one warp per token: k rounds of warp arg-max over
//                       l' = logits + bias (ties to the lower id; two warp
//                       reductions per round on order-preserving keys), softmax
//                       weights, sentinel mask; then a warp-aggregated
//                       (__match_any_sync) atomic histogram per sort block.
//   2. route_scatter    one CTA per sort block of up to 1024 slots: global
//                       bin starts from the histograms (warp shuffle scan),
//                       then a stable in-order rank of every slot from
//                       per-warp match_any peer masks.  Writes sorted_rows,
//                       row_pos and (block 0) offsets.
// A small batch (one sort block, little routing work) instead runs
//   route_small         one CTA of 32 warps: the same per-token routing, then
//                       the sort of its <= 1024 slots in shared memory.
#include <atomic>
#include <climits>
#include <mutex>

#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxSlotsPerBlock = 1024;
constexpr int kMaxE = 256;
constexpr int kMaxK = 32;

struct SortGeometry {
    int tokens_per_block;  // tokens whose slots form one sort block
    int slots_per_block;
    int blocks;
};

SortGeometry geometry(int T, int k) {
    SortGeometry g;
    g.tokens_per_block = kMaxSlotsPerBlock / k > 0 ? kMaxSlotsPerBlock / k : 1;
    g.slots_per_block = g.tokens_per_block * k;
    g.blocks = (T + g.tokens_per_block - 1) / g.tokens_per_block;
    return g;
}

// Order-preserving map of a float to an unsigned key: a larger float gives a
// larger key and +0 and -0 the same key.  NaN maps to 0, below every number,
// so it is never picked; 0 also marks a logit already picked.
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(v + 0.0f);   // -0 + 0 = +0
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Ids outside [0, E] cannot be placed: they are sorted as sentinels and the
// error word records the bad input.
__device__ __forceinline__ int checked_id(int id, int E, int* err) {
    if (id < 0 || id > E) {
        moe::raise_device_error(err, MOE_DEVERR_ROUTE);
        return E;
    }
    return id;
}

// Routes token t on one warp: the k picks (or the given ids), the weights
// and the sentinel mask, written to ids/w.  Returns, in lane j < k, the
// checked id of slot j.  A bad id (a given id outside [0, E], or a pick that
// NaN logits left unfilled) is reported, returned as E and written back to
// ids as E, so that the sort, the combine and ids agree that the slot is a
// sentinel.
template <int NV>   // logits per lane: E <= 32 * NV
__device__ __forceinline__ int route_token(const float* __restrict__ logits, const float* __restrict__ bias,
                                           const uint8_t* __restrict__ mask, int32_t* ids,
                                           float* __restrict__ w, int t, int E, int k, int renormalize,
                                           int* err) {
    const int lane = threadIdx.x & 31;
    const int64_t slot0 = static_cast<int64_t>(t) * k;
    int my_id = E;  // lane j < k: the id of slot j

    if (logits) {
        const float* row = logits + static_cast<int64_t>(t) * E;
        float v[NV];
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int e = lane + 32 * j;
            if (e < E) {
                const float l = row[e];
                v[j] = bias ? l + bias[e] : l;
            } else {
                v[j] = -INFINITY;
            }
        }
        // each pick: the largest key over the warp (one warp reduction), then
        // the lowest expert id holding it (a second one); a lane's candidate
        // is its first slot with its largest key, the lowest id of the lane
        uint32_t key[NV];
#pragma unroll
        for (int j = 0; j < NV; ++j) key[j] = lane + 32 * j < E ? order_key(v[j]) : 0u;
        uint32_t taken = 0;   // bit j: this lane's slot j was picked
        float my_v = -INFINITY;
        for (int r = 0; r < k; ++r) {
            uint32_t bk = 0u;
            int bj = 0;
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const uint32_t kj = (taken >> j) & 1u ? 0u : key[j];
                if (kj > bk) { bk = kj; bj = j; }
            }
            const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
            const int bi = __reduce_min_sync(0xffffffffu, m != 0u && bk == m ? lane + 32 * bj : INT_MAX);
            if (m != 0u && (bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (lane == r) { my_v = m != 0u ? key_value(m) : -INFINITY; my_id = bi; }
        }
        const float mx = __shfl_sync(0xffffffffu, my_v, 0);  // pick 0 is the maximum
        float part = 0.0f;
        if (renormalize) {
            part = lane < k ? expf(my_v - mx) : 0.0f;
        } else {
#pragma unroll
            for (int j = 0; j < NV; ++j)
                if (lane + 32 * j < E) part += expf(v[j] - mx);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane < k) {
            w[slot0 + lane] = expf(my_v - mx) / part;
            if (mask && mask[slot0 + lane]) my_id = E;
            my_id = checked_id(my_id, E, err);
            ids[slot0 + lane] = my_id;
        }
    } else if (lane < k) {
        const int given = ids[slot0 + lane];
        my_id = mask && mask[slot0 + lane] ? E : checked_id(given, E, err);
        if (my_id != given) ids[slot0 + lane] = my_id;
    }
    return my_id;
}

template <int NV>
__global__ void __launch_bounds__(kThreads)
route_topk_hist(const float* __restrict__ logits, const float* __restrict__ bias,
                const uint8_t* __restrict__ mask, int32_t* ids, float* __restrict__ w, int T,
                int E, int k, int renormalize, int slots_per_block, int* counts, int* err) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const int64_t slot0 = static_cast<int64_t>(t) * k;
    const int my_id = route_token<NV>(logits, bias, mask, ids, w, t, E, k, renormalize, err);

    // histogram of this token's slots into its sort block, one atomic per
    // distinct id in the warp
    const unsigned active = __ballot_sync(0xffffffffu, lane < k);
    if (lane < k) {
        const unsigned peers = __match_any_sync(active, my_id);
        if (lane == __ffs(peers) - 1) {
            const int blk = static_cast<int>(slot0 / slots_per_block);
            atomicAdd(&counts[blk * (E + 1) + my_id], __popc(peers));
        }
    }
}

__global__ void __launch_bounds__(kThreads)
route_scatter(const int32_t* ids, int64_t R, int E, int slots_per_block, int nblocks,
              const int* __restrict__ counts, int32_t* __restrict__ sorted_rows,
              int32_t* __restrict__ row_pos, int32_t* __restrict__ offsets, int* err) {
    __shared__ int tot[kMaxE + 1];
    __shared__ int start[kMaxE + 1];
    __shared__ int whist[kWarps][kMaxE + 1];
    const int nb = E + 1;
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // warp w owns a contiguous run of at most 128 of the block's slots; its ids
    // are loaded once, up front, so the loads overlap the count summation
    const int64_t blk0 = static_cast<int64_t>(b) * slots_per_block;
    const int64_t blk1 = blk0 + slots_per_block < R ? blk0 + slots_per_block : R;
    const int per_warp = (slots_per_block + kWarps - 1) / kWarps;
    const int64_t w0 = blk0 + static_cast<int64_t>(warp) * per_warp;
    const int64_t w1 = w0 + per_warp < blk1 ? w0 + per_warp : blk1;
    constexpr int kChunks = kMaxSlotsPerBlock / kWarps / 32;
    int idr[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        const int64_t sl = w0 + c * 32 + lane;
        idr[c] = sl < w1 ? ids[sl] : 0;
    }

    // 1. per bin: total over all blocks and the count in blocks before this one
    for (int bin = threadIdx.x; bin < nb; bin += kThreads) {
        int all = 0, before = 0;
        int bb = 0;
        for (; bb + 16 <= nblocks; bb += 16) {   // sixteen independent loads in flight
            int c[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) c[i] = counts[(bb + i) * nb + bin];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                all += c[i];
                before += bb + i < b ? c[i] : 0;
            }
        }
        for (; bb < nblocks; ++bb) {
            const int c = counts[bb * nb + bin];
            all += c;
            before += bb < b ? c : 0;
        }
        tot[bin] = all;
        start[bin] = before;
    }
    for (int i = threadIdx.x; i < kWarps * nb; i += kThreads) whist[i / nb][i % nb] = 0;
    __syncthreads();

    // 2. exclusive scan of the totals over bins (warp 0: 9 bins per lane)
    if (warp == 0) {
        constexpr int PER = (kMaxE + 1 + 31) / 32;
        int local[PER];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int bin = lane * PER + i;
            local[i] = bin < nb ? tot[bin] : 0;
            sum += local[i];
        }
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        int run = incl - sum;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int bin = lane * PER + i;
            if (bin < nb) {
                const int bin_start = run;
                run += local[i];
                if (b == 0) offsets[bin] = bin_start;   // offsets[E] = live rows
                start[bin] += bin_start;                // global base of this block's slots
            }
        }
    }
    __syncthreads();

    // 3. stable ranks within the warp's run, in slot order
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int c = 0; c < kChunks; ++c)
        idr[c] = w0 + c * 32 + lane < w1 ? checked_id(idr[c], E, err) : -1;   // -1: no slot here

#pragma unroll
    for (int c = 0; c < kChunks; ++c) {                         // pass A: per-warp histogram
        if (w0 + c * 32 >= w1) break;
        const int id = idr[c];
        const unsigned peers = __match_any_sync(0xffffffffu, id);
        if (id >= 0 && lane == __ffs(peers) - 1) whist[warp][id] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    for (int bin = threadIdx.x; bin < nb; bin += kThreads) {   // exclusive prefix over warps
        int acc = 0;
        for (int wi = 0; wi < kWarps; ++wi) {
            const int c = whist[wi][bin];
            whist[wi][bin] = acc;
            acc += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {                         // pass B: positions
        if (w0 + c * 32 >= w1) break;
        const int64_t s = w0 + c * 32 + lane;
        const int id = idr[c];
        const unsigned peers = __match_any_sync(0xffffffffu, id);
        int pos = 0;
        if (id >= 0) pos = start[id] + whist[warp][id] + __popc(peers & lt);
        __syncwarp();
        if (id >= 0) {
            sorted_rows[pos] = static_cast<int32_t>(s);
            row_pos[s] = pos;
            if (lane == __ffs(peers) - 1) whist[warp][id] += __popc(peers);
        }
        __syncwarp();
    }
}

// A batch whose slots form a single sort block (T * k <= 1024) and whose
// tokens are few: one CTA of 32 warps routes the tokens (warp w takes tokens
// w, w + 32, ...), then sorts the slots in shared memory.  It replaces the
// histogram memset and the second launch of the two-kernel path, which cost
// more than the work itself at decode batch sizes (64 tokens, 32 experts:
// 10.2 against 13.3 us) -- as long as each warp routes few tokens of few
// logits: 128 tokens of 256 experts took 28.7 us against 17.4.
constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / 32;

template <int NV>
__global__ void __launch_bounds__(kSmallThreads)
route_small(const float* __restrict__ logits, const float* __restrict__ bias,
            const uint8_t* __restrict__ mask, int32_t* ids, float* __restrict__ w, int T, int E, int k,
            int renormalize, int32_t* __restrict__ sorted_rows, int32_t* __restrict__ row_pos,
            int32_t* __restrict__ offsets, int* err) {
    __shared__ int sid[kMaxSlotsPerBlock];
    __shared__ int whist[kSmallWarps][kMaxE + 1];
    __shared__ int bin_start[kMaxE + 1];
    __shared__ int bin_total[kMaxE + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = E + 1;
    const int R = T * k;
    for (int i = threadIdx.x; i < kSmallWarps * nb; i += kSmallThreads) whist[i / nb][i % nb] = 0;
    for (int t = warp; t < T; t += kSmallWarps) {
        const int id = route_token<NV>(logits, bias, mask, ids, w, t, E, k, renormalize, err);
        if (lane < k) sid[t * k + lane] = id;
    }
    __syncthreads();

    // slot s = threadIdx.x: per-warp histograms, then for every bin the
    // exclusive prefix over warps and the total
    const int s = threadIdx.x;
    const int id = s < R ? sid[s] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, id);
    if (id >= 0 && lane == __ffs(peers) - 1) whist[warp][id] = __popc(peers);
    __syncthreads();
    for (int bin = threadIdx.x; bin < nb; bin += kSmallThreads) {
        int acc = 0;
        for (int wi = 0; wi < kSmallWarps; ++wi) {
            const int c = whist[wi][bin];
            whist[wi][bin] = acc;
            acc += c;
        }
        bin_total[bin] = acc;
    }
    __syncthreads();
    if (warp == 0) {   // exclusive scan of the totals over bins
        constexpr int PER = (kMaxE + 1 + 31) / 32;
        int tot[PER];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int bin = lane * PER + i;
            tot[i] = bin < nb ? bin_total[bin] : 0;
            sum += tot[i];
        }
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        int run = incl - sum;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int bin = lane * PER + i;
            if (bin < nb) {
                bin_start[bin] = run;
                offsets[bin] = run;   // offsets[E] = live rows
                run += tot[i];
            }
        }
    }
    __syncthreads();
    if (id >= 0) {
        const int pos = bin_start[id] + whist[warp][id] + __popc(peers & ((1u << lane) - 1u));
        sorted_rows[pos] = s;
        row_pos[s] = pos;
    }
}

// Whether the single-CTA path takes this batch: one sort block, and at most
// four (tokens per warp) x (logits per lane) of routing work per warp.
bool use_small(int T, int E, int k) {
    const int nv = E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : 8;
    return static_cast<int64_t>(T) * k <= kMaxSlotsPerBlock && (T + kSmallWarps - 1) / kSmallWarps * nv <= 4;
}

void launch_small(cudaStream_t s, const float* logits, const float* bias, const uint8_t* mask, int32_t* ids,
                  float* w, int T, int E, int k, int renormalize, int32_t* sorted_rows, int32_t* row_pos,
                  int32_t* offsets, int* err) {
    if (E <= 32)
        route_small<1><<<1, kSmallThreads, 0, s>>>(logits, bias, mask, ids, w, T, E, k, renormalize, sorted_rows, row_pos, offsets, err);
    else if (E <= 64)
        route_small<2><<<1, kSmallThreads, 0, s>>>(logits, bias, mask, ids, w, T, E, k, renormalize, sorted_rows, row_pos, offsets, err);
    else if (E <= 128)
        route_small<4><<<1, kSmallThreads, 0, s>>>(logits, bias, mask, ids, w, T, E, k, renormalize, sorted_rows, row_pos, offsets, err);
    else
        route_small<8><<<1, kSmallThreads, 0, s>>>(logits, bias, mask, ids, w, T, E, k, renormalize, sorted_rows, row_pos, offsets, err);
}

void launch_topk_hist(cudaStream_t s, const float* logits, const float* bias, const uint8_t* mask,
                      int32_t* ids, float* w, int T, int E, int k, int renormalize,
                      int slots_per_block, int* counts, int* err) {
    const dim3 grid((T + kWarps - 1) / kWarps);
    if (E <= 32)
        route_topk_hist<1><<<grid, kThreads, 0, s>>>(logits, bias, mask, ids, w, T, E, k, renormalize, slots_per_block, counts, err);
    else if (E <= 64)
        route_topk_hist<2><<<grid, kThreads, 0, s>>>(logits, bias, mask, ids, w, T, E, k, renormalize, slots_per_block, counts, err);
    else if (E <= 128)
        route_topk_hist<4><<<grid, kThreads, 0, s>>>(logits, bias, mask, ids, w, T, E, k, renormalize, slots_per_block, counts, err);
    else
        route_topk_hist<8><<<grid, kThreads, 0, s>>>(logits, bias, mask, ids, w, T, E, k, renormalize, slots_per_block, counts, err);
}

}  // namespace

extern "C" size_t moe_route_sort_workspace_size(int T, int E, int k) {
    if (T < 1 || E < 1 || E > kMaxE || k < 1 || k > E || k > kMaxK) return 0;
    const SortGeometry g = geometry(T, k);
    const size_t bytes = static_cast<size_t>(g.blocks) * (E + 1) * sizeof(int);
    return (bytes + 255) & ~static_cast<size_t>(255);
}

extern "C" moe_status_t moe_route_sort(const float* logits, const float* expert_bias,
                                       const uint8_t* sentinel_mask, int32_t* topk_ids,
                                       float* topk_w, int T, int E, int k, int renormalize,
                                       int32_t* sorted_rows, int32_t* row_pos, int32_t* offsets,
                                       void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_CHECK_ARG(T >= 1 && E >= 1 && E <= kMaxE && k >= 1 && k <= E && k <= kMaxK);
    MOE_CHECK_ARG(static_cast<int64_t>(T) * k < INT_MAX);
    MOE_CHECK_ARG(topk_ids && sorted_rows && row_pos && offsets);
    MOE_CHECK_ARG(!logits || topk_w);
    MOE_CHECK_ARG(moe::aligned16(topk_ids) && moe::aligned16(sorted_rows) &&
                  moe::aligned16(row_pos) && moe::aligned16(offsets));
    MOE_CHECK_ARG(!logits || (moe::aligned16(logits) && moe::aligned16(topk_w)));
    MOE_CHECK_ARG(!expert_bias || moe::aligned16(expert_bias));
    const size_t need = moe_route_sort_workspace_size(T, E, k);
    if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
    int* err = moe::device_error_word();
    if (!err) return MOE_ERR_CUDA;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (use_small(T, E, k)) {
        launch_small(s, logits, logits ? expert_bias : nullptr, sentinel_mask, topk_ids, topk_w, T, E, k,
                     renormalize, sorted_rows, row_pos, offsets, err);
        MOE_CHECK_LAUNCH();
        return MOE_OK;
    }
    const SortGeometry g = geometry(T, k);
    int* counts = static_cast<int*>(ws);
    MOE_CHECK_CUDA(cudaMemsetAsync(counts, 0, static_cast<size_t>(g.blocks) * (E + 1) * sizeof(int), s));
    launch_topk_hist(s, logits, logits ? expert_bias : nullptr, sentinel_mask, topk_ids, topk_w, T, E,
                     k, renormalize, g.slots_per_block, counts, err);
    MOE_CHECK_LAUNCH();
    route_scatter<<<g.blocks, kThreads, 0, s>>>(topk_ids, static_cast<int64_t>(T) * k, E,
                                                g.slots_per_block, g.blocks, counts, sorted_rows,
                                                row_pos, offsets, err);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant.  The per-sort-block histogram lives in a static
// device array instead of caller workspace, for callers that may not allocate
// device memory themselves (see moe_route_sort_noalloc in moe.h).
namespace {

constexpr size_t kStaticScratchBytes = 256 * 1024;
constexpr size_t kStaticScratchInts = kStaticScratchBytes / sizeof(int);
static __device__ __align__(256) int g_route_scratch[kStaticScratchInts];

constexpr int kMaxDevices = 64;
std::atomic<int*> g_route_scratch_ptr[kMaxDevices];
std::mutex g_route_scratch_mu;

// Device address of g_route_scratch on the current device, looked up once
// per device (the host-side symbol is only a stand-in, not a device address).
int* static_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    int* p = g_route_scratch_ptr[dev].load(std::memory_order_acquire);
    if (p) return p;
    std::lock_guard<std::mutex> lk(g_route_scratch_mu);
    p = g_route_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_route_scratch) != cudaSuccess || !addr) return nullptr;
        p = static_cast<int*>(addr);
        g_route_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace

extern "C" moe_status_t moe_route_sort_noalloc(const float* logits, const float* expert_bias,
                                               const uint8_t* sentinel_mask, int32_t* topk_ids,
                                               float* topk_w, int T, int E, int k, int renormalize,
                                               int32_t* sorted_rows, int32_t* row_pos,
                                               int32_t* offsets, moe_stream_t stream) {
    MOE_CHECK_ARG(T >= 1 && E >= 1 && E <= kMaxE && k >= 1 && k <= E && k <= kMaxK);
    MOE_CHECK_ARG(static_cast<int64_t>(T) * k < INT_MAX);
    MOE_CHECK_ARG(topk_ids && sorted_rows && row_pos && offsets);
    MOE_CHECK_ARG(!logits || topk_w);
    MOE_CHECK_ARG(moe::aligned16(topk_ids) && moe::aligned16(sorted_rows) &&
                  moe::aligned16(row_pos) && moe::aligned16(offsets));
    MOE_CHECK_ARG(!logits || (moe::aligned16(logits) && moe::aligned16(topk_w)));
    MOE_CHECK_ARG(!expert_bias || moe::aligned16(expert_bias));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (use_small(T, E, k)) {   // one CTA, shared memory only: the static array is not used
        int* err = moe::device_error_word();
        if (!err) return MOE_ERR_CUDA;
        launch_small(s, logits, logits ? expert_bias : nullptr, sentinel_mask, topk_ids, topk_w, T, E, k,
                     renormalize, sorted_rows, row_pos, offsets, err);
        MOE_CHECK_LAUNCH();
        return MOE_OK;
    }
    const SortGeometry g = geometry(T, k);
    const size_t ints = static_cast<size_t>(g.blocks) * (E + 1);
    if (ints > kStaticScratchInts) return MOE_ERR_WORKSPACE;   // beyond the static scratch
    int* err = moe::device_error_word();
    if (!err) return MOE_ERR_CUDA;
    int* counts = static_scratch();
    if (!counts) return MOE_ERR_CUDA;

    MOE_CHECK_CUDA(cudaMemsetAsync(counts, 0, ints * sizeof(int), s));
    launch_topk_hist(s, logits, logits ? expert_bias : nullptr, sentinel_mask, topk_ids, topk_w, T, E,
                     k, renormalize, g.slots_per_block, counts, err);
    MOE_CHECK_LAUNCH();
    route_scatter<<<g.blocks, kThreads, 0, s>>>(topk_ids, static_cast<int64_t>(T) * k, E,
                                                g.slots_per_block, g.blocks, counts, sorted_rows,
                                                row_pos, offsets, err);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}
