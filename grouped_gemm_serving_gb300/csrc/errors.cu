// Status strings, the per-device error word and device queries.
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace {
constexpr int kMaxDevices = 64;
__device__ int g_device_error;             // one word per device context
std::atomic<int*> g_err_ptr[kMaxDevices];  // its device address, per device
std::atomic<int> g_sm_count[kMaxDevices];
std::mutex g_init_mu;
}  // namespace

namespace moe {

int* device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    int* p = g_err_ptr[dev].load(std::memory_order_acquire);
    if (p) return p;
    std::lock_guard<std::mutex> lk(g_init_mu);
    p = g_err_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess) return nullptr;
        p = static_cast<int*>(addr);
        g_err_ptr[dev].store(p, std::memory_order_release);
    }
    return p;
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace moe

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE_CHECK: return "a kernel rejected its device-side input";
        case MOE_ERR_TIMEOUT: return "a device pipeline wait timed out";
    }
    return "unknown status";
}

moe_status_t moe_get_device_error(int32_t* code, moe_stream_t stream) {
    if (!code) return MOE_ERR_INVALID_ARG;
    int* p = moe::device_error_word();
    if (!p) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    const int zero = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (v != 0 && cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
        return MOE_ERR_CUDA;
    *code = v;
    if (v == 0) return MOE_OK;
    return v == MOE_DEVERR_TIMEOUT ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE_CHECK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Self-test of the bounded-wait path: one thread waits on an mbarrier that
// nothing ever arrives on, with the given limit, and records a timeout.
namespace {
__global__ void wait_timeout_kernel(uint64_t limit_ns, int* err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    moe::mbar_init(moe::smem_u32(&bar), 1);
    moe::fence_barrier_init();
    if (!moe::mbar_wait(moe::smem_u32(&bar), 0, &abort_flag, limit_ns))
        moe::raise_device_error(err, MOE_DEVERR_TIMEOUT);
}
}  // namespace

extern "C" moe_status_t moe_selftest_wait_timeout(uint64_t limit_ns, moe_stream_t stream) {
    if (limit_ns == 0 || limit_ns > 2000000000ull) return MOE_ERR_INVALID_ARG;
    int* err = moe::device_error_word();
    if (!err) return MOE_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, err);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
}
