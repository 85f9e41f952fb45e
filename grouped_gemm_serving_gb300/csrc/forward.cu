// moe_forward: the whole expert layer enqueued on one stream, in the order of
// the fused pipeline of "LlamaFactory Triton fused MoE kernel" (section 1):
// route + sort -> [quantise x] -> scatter -> grouped GEMM gate_up with fused
// silu(gate) * up [and fused FP8 quantisation of h] -> grouped GEMM down ->
// weighted gather.  With MOE_FWD_GATHER the scatter is folded into the
// gate_up GEMM, which then reads its rows from token order
// (moe_grouped_gemm_gather) and no permuted copy of x is held.  Offsets stay
// on the device; there is no host synchronisation.  With MOE_FWD_HOST_IO, x
// is copied in on a second stream while the batch is routed, and a pinned
// output buffer is written in place by the combine.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kAlign = 256;

struct Carver {
    size_t off = 0;
    size_t take(size_t bytes) {
        const size_t o = off;
        off += (bytes + kAlign - 1) & ~(kAlign - 1);
        return o;
    }
};

struct Layout {
    size_t route, ids, w, sorted_rows, row_pos, offsets;
    size_t xq, xs;          // FP8: quantised x and its scales
    size_t xp, xps;         // permuted activations (+ FP8 scales, group-major)
    size_t h, hs;           // gate_up output after SwiGLU (+ FP8 scales)
    size_t y2;              // down output, bf16
    size_t x_dev, logits_dev, out_dev;  // host-I/O staging
    size_t counters;        // fused combine (bf16)
    size_t total;
};

bool valid_args(const moe_forward_args* a) {
    if (!a) return false;
    if (a->T < 1 || a->E < 1 || a->E > 256 || a->k < 1 || a->k > a->E || a->k > 32) return false;
    if (a->H < 8 || a->H % 8 || a->I < 8 || a->I % 8) return false;
    if (static_cast<int64_t>(a->T) * a->k >= (1ll << 31) - 1) return false;
    if (a->dtype == MOE_FP8_E4M3_B128) {
        if (a->H % 128 || a->I % 128 || !a->W1_scales || !a->W2_scales) return false;
    } else if (a->dtype != MOE_BF16) {
        return false;
    }
    if (!a->x || !a->W1 || !a->W2 || !a->out) return false;
    if (!a->logits && (!a->topk_ids || !a->topk_w)) return false;
    return true;
}

// Whether the scatter runs as its own kernel: unless MOE_FWD_GATHER asks
// otherwise, and always when the gathering GEMM cannot take H (it fetches
// rows in whole 128-byte k-blocks).
bool separate_scatter(const moe_forward_args* a) {
    const int esz = a->dtype == MOE_FP8_E4M3_B128 ? 1 : 2;
    return !(a->flags & MOE_FWD_GATHER) || (a->H * esz) % 128 != 0;
}

Layout layout(const moe_forward_args* a) {
    const size_t T = a->T, E = a->E, k = a->k, H = a->H, I = a->I, R = T * k;
    const bool fp8 = a->dtype == MOE_FP8_E4M3_B128;
    const bool scatter = separate_scatter(a);
    Carver c;
    Layout l{};
    l.route = c.take(moe_route_sort_workspace_size(a->T, a->E, a->k));
    l.ids = a->topk_ids ? 0 : c.take(R * 4);
    l.w = a->topk_w ? 0 : c.take(R * 4);
    l.sorted_rows = c.take(R * 4);
    l.row_pos = c.take(R * 4);
    l.offsets = c.take((E + 1) * 4);
    if (fp8) {
        l.xq = c.take(T * H);
        l.xs = c.take(T * (H / 128) * 4);
        if (scatter) {
            l.xp = c.take(R * H);
            l.xps = c.take((H / 128) * R * 4);
        }
        l.h = c.take(R * I);
        l.hs = c.take((I / 128) * R * 4);
    } else {
        if (scatter) l.xp = c.take(R * H * 2);
        l.h = c.take(R * I * 2);
    }
    l.y2 = c.take(R * H * 2);
    if ((a->flags & MOE_FWD_FUSED_COMBINE) && !fp8) l.counters = c.take(moe_grouped_gemm_combine_workspace_size(a->T, a->H));
    if (a->flags & MOE_FWD_HOST_IO) {
        l.x_dev = c.take(T * H * 2);
        l.logits_dev = a->logits ? c.take(T * E * 4) : 0;
        l.out_dev = c.take(T * H * 2);
    }
    l.total = c.off;
    return l;
}

// The device address of pinned (page-locked, mapped) host memory, which a
// kernel may write in place; NULL for pageable host memory.
void* mapped_host_view(const void* p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

// A second stream per device for the host-to-device copy of x, with the two
// events that fork it from and join it to the caller's stream, and the event
// that chains the kernels of successive host-I/O calls.  Created on first use
// and kept for the life of the process; the mutex keeps the record/wait
// sequences of concurrent calls from interleaving.
struct CopyStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, ready = nullptr, chain = nullptr;
    bool chained = false;   // chain holds the last call's kernels
    std::mutex mu;
};
constexpr int kMaxDevices = 64;
CopyStream g_copy[kMaxDevices];
std::mutex g_copy_init;

CopyStream* copy_stream() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    CopyStream& c = g_copy[dev];
    std::lock_guard<std::mutex> lk(g_copy_init);
    if (!c.stream) {
        cudaStream_t st = nullptr;
        cudaEvent_t a = nullptr, b = nullptr, ch = nullptr;
        if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&a, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&b, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&ch, cudaEventDisableTiming) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        c.fork = a;
        c.ready = b;
        c.chain = ch;
        c.stream = st;
    }
    return &c;
}

#define MOE_TRY(call)                          \
    do {                                       \
        const moe_status_t st_ = (call);       \
        if (st_ != MOE_OK) return st_;         \
    } while (0)

}  // namespace

extern "C" size_t moe_forward_workspace_size(const moe_forward_args* args) {
    if (!valid_args(args)) return 0;
    return layout(args).total;
}

extern "C" moe_status_t moe_forward(const moe_forward_args* a, void* ws, size_t ws_bytes,
                                    moe_stream_t stream) {
    if (!valid_args(a)) return MOE_ERR_INVALID_ARG;
    const Layout l = layout(a);
    if (!ws || ws_bytes < l.total) return MOE_ERR_WORKSPACE;
    MOE_CHECK_ARG(moe::aligned16(ws));
    uint8_t* base = static_cast<uint8_t*>(ws);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int T = a->T, E = a->E, k = a->k, H = a->H, I = a->I, R = T * k;
    const bool fp8 = a->dtype == MOE_FP8_E4M3_B128;
    const bool host_io = (a->flags & MOE_FWD_HOST_IO) != 0;
    const bool scatter = separate_scatter(a);

    const void* x = a->x;
    const float* logits = a->logits;
    void* out = a->out;
    bool copy_out = false;
    CopyStream* cs = nullptr;
    std::unique_lock<std::mutex> cs_lock;
    bool capturing = false;
    if (host_io) {
        // x (the large input) is copied in on a second stream while the
        // logits are copied and the batch routed on `stream`; the caller's
        // stream waits for x before the first kernel that reads it.  The
        // output of a pinned `out` is written in place by the combine (unless
        // MOE_FWD_STAGED_OUT); pageable output memory gets a staged copy.
        // (Kernels reading pinned inputs over the host link in place were
        // slower than the copy engine; for one call at a time, writing the
        // output in place was faster than a copy.)
        cs = copy_stream();
        if (!cs) return MOE_ERR_CUDA;
        cs_lock = std::unique_lock<std::mutex>(cs->mu);
        void* xd = base + l.x_dev;
        MOE_CHECK_CUDA(cudaEventRecord(cs->fork, s));   // earlier users of the staging buffer are done
        MOE_CHECK_CUDA(cudaStreamWaitEvent(cs->stream, cs->fork, 0));
        MOE_CHECK_CUDA(cudaMemcpyAsync(xd, a->x, static_cast<size_t>(T) * H * 2, cudaMemcpyHostToDevice,
                                       cs->stream));
        MOE_CHECK_CUDA(cudaEventRecord(cs->ready, cs->stream));
        x = xd;
        if (logits) {
            float* ld = reinterpret_cast<float*>(base + l.logits_dev);
            MOE_CHECK_CUDA(cudaMemcpyAsync(ld, a->logits, static_cast<size_t>(T) * E * 4,
                                           cudaMemcpyHostToDevice, s));
            logits = ld;
        }
        // the kernels of host-I/O calls run in call order: this call's wait
        // for the previous call's (which may be on another stream), after the
        // copies above so that they do not wait for them
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        MOE_CHECK_CUDA(cudaStreamIsCapturing(s, &cap));
        capturing = cap != cudaStreamCaptureStatusNone;
        if (!capturing && cs->chained) MOE_CHECK_CUDA(cudaStreamWaitEvent(s, cs->chain, 0));
        void* ov = (a->flags & MOE_FWD_STAGED_OUT) ? nullptr : mapped_host_view(a->out);
        if (ov) {
            out = ov;
        } else {
            out = base + l.out_dev;
            copy_out = true;
        }
    }
    int32_t* ids = a->topk_ids ? a->topk_ids : reinterpret_cast<int32_t*>(base + l.ids);
    float* w = a->topk_w ? a->topk_w : reinterpret_cast<float*>(base + l.w);
    int32_t* sorted_rows = reinterpret_cast<int32_t*>(base + l.sorted_rows);
    int32_t* row_pos = reinterpret_cast<int32_t*>(base + l.row_pos);
    int32_t* offsets = reinterpret_cast<int32_t*>(base + l.offsets);

    MOE_TRY(moe_route_sort(logits, a->expert_bias, a->sentinel_mask, ids, w, T, E, k, a->renormalize,
                           sorted_rows, row_pos, offsets, base + l.route,
                           moe_route_sort_workspace_size(T, E, k), stream));
    if (cs) MOE_CHECK_CUDA(cudaStreamWaitEvent(s, cs->ready, 0));   // x has arrived before anything reads it
    void* y2 = base + l.y2;
    if (!fp8) {
        void* h = base + l.h;
        if (scatter) {
            void* xp = base + l.xp;
            MOE_TRY(moe_permute(MOE_BF16, x, nullptr, T, H, k, sorted_rows, offsets, E, R, xp, nullptr, stream));
            MOE_TRY(moe_grouped_gemm(MOE_BF16, xp, nullptr, a->W1, nullptr, offsets, E, R, 2 * I, H,
                                     MOE_EPI_SWIGLU, h, nullptr, stream));
        } else {
            MOE_TRY(moe_grouped_gemm_gather(MOE_BF16, x, nullptr, T, k, sorted_rows, a->W1, nullptr, offsets, E,
                                            R, 2 * I, H, MOE_EPI_SWIGLU, h, nullptr, stream));
        }
        if (a->flags & MOE_FWD_FUSED_COMBINE) {
            MOE_TRY(moe_grouped_gemm_combine(h, a->W2, offsets, E, R, H, I, ids, w, sorted_rows, row_pos, T, k, y2,
                                             out, base + l.counters, moe_grouped_gemm_combine_workspace_size(T, H),
                                             stream));
        } else {
            MOE_TRY(moe_grouped_gemm(MOE_BF16, h, nullptr, a->W2, nullptr, offsets, E, R, H, I,
                                     MOE_EPI_STORE, y2, nullptr, stream));
        }
    } else {
        uint8_t* xq = base + l.xq;
        float* xs = reinterpret_cast<float*>(base + l.xs);
        uint8_t* h = base + l.h;
        float* hs = reinterpret_cast<float*>(base + l.hs);
        MOE_TRY(moe_act_quant_fp8(x, T, H, xq, xs, stream));
        if (scatter) {
            uint8_t* xp = base + l.xp;
            float* xps = reinterpret_cast<float*>(base + l.xps);
            MOE_TRY(moe_permute(MOE_FP8_E4M3_B128, xq, xs, T, H, k, sorted_rows, offsets, E, R, xp, xps, stream));
            MOE_TRY(moe_grouped_gemm(MOE_FP8_E4M3_B128, xp, xps, a->W1, a->W1_scales, offsets, E, R, 2 * I, H,
                                     MOE_EPI_SWIGLU_QUANT_FP8, h, hs, stream));
        } else {
            MOE_TRY(moe_grouped_gemm_gather(MOE_FP8_E4M3_B128, xq, xs, T, k, sorted_rows, a->W1, a->W1_scales,
                                            offsets, E, R, 2 * I, H, MOE_EPI_SWIGLU_QUANT_FP8, h, hs, stream));
        }
        MOE_TRY(moe_grouped_gemm(MOE_FP8_E4M3_B128, h, hs, a->W2, a->W2_scales, offsets, E, R, H, I,
                                 MOE_EPI_STORE, y2, nullptr, stream));
    }
    if (fp8 || !(a->flags & MOE_FWD_FUSED_COMBINE)) MOE_TRY(moe_combine(y2, ids, w, row_pos, T, k, H, E, out, stream));
    if (cs) {
        if (!capturing) {
            MOE_CHECK_CUDA(cudaEventRecord(cs->chain, s));
            cs->chained = true;
        }
        cs_lock.unlock();
    }
    if (copy_out)
        MOE_CHECK_CUDA(cudaMemcpyAsync(a->out, out, static_cast<size_t>(T) * H * 2, cudaMemcpyDeviceToHost, s));
    return MOE_OK;
}
