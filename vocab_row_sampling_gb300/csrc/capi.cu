// capi.cu -- status strings, the device error flag and launch bookkeeping of
// libdrs.
#include <atomic>
#include <mutex>

#include "drs_internal.h"

namespace drs {

__device__ int g_device_error = 0;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mutex;
int* g_flag_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::atomic<uint32_t> g_generation{0x5eed0000u};

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}
}  // namespace

int* device_error_flag() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_flag_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        g_flag_ptr[dev] = static_cast<int*>(p);
    }
    return g_flag_ptr[dev];
}

uint32_t next_generation() {
    uint32_t g = g_generation.fetch_add(1, std::memory_order_relaxed) + 1;
    return g == 0 ? next_generation() : g;
}

// A second stream per device and a pair of events for the row calls that
// split their rows between the cluster kernel and the two passes (the two
// parts run at the same time on different SMs): created on first use, kept
// until the process exits.
namespace {
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr;
    cudaEvent_t join = nullptr;
};
SideStream g_side[kMaxDevices];
}  // namespace

bool side_stream(cudaStream_t* stream, cudaEvent_t* fork, cudaEvent_t* join) {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_mutex);
    SideStream& s = g_side[dev];
    if (!s.stream) {
        if (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess) return false;
        if (cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess)
            return false;
    }
    *stream = s.stream;
    *fork = s.fork;
    *join = s.join;
    return true;
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

// ------------------------------------------------------- kernel timing

namespace {
// Events around the kernels of the last kTimedCalls row-statistics calls
// (ring), on the device that was current when timing was switched on.
struct KernelTimer {
    bool on = false;
    int device = -1;
    int calls = 0;
    cudaEvent_t ev[kTimedCalls][kTimedKernels + 1] = {};
};
KernelTimer g_timer;
std::mutex g_timer_mutex;
}  // namespace

int kernel_timer_slot() {
    std::lock_guard<std::mutex> lock(g_timer_mutex);
    if (!g_timer.on || current_device() != g_timer.device) return -1;
    return g_timer.calls++ % kTimedCalls;
}

cudaEvent_t kernel_timer_event(int slot, int i) { return g_timer.ev[slot][i]; }

}  // namespace drs

extern "C" drs_status drs_kernel_timing(int enable) {
    using namespace drs;
    std::lock_guard<std::mutex> lock(g_timer_mutex);
    if (!enable) {
        g_timer.on = false;
        return DRS_OK;
    }
    const int dev = current_device();
    if (dev < 0) return DRS_ERR_CUDA;
    if (g_timer.device != dev) {
        if (g_timer.device >= 0) {
            int prev = 0;
            if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(g_timer.device) != cudaSuccess)
                return DRS_ERR_CUDA;
            for (auto& call : g_timer.ev)
                for (cudaEvent_t& e : call)
                    if (e) cudaEventDestroy(e), e = nullptr;
            if (cudaSetDevice(prev) != cudaSuccess) return DRS_ERR_CUDA;
        }
        for (auto& call : g_timer.ev)
            for (cudaEvent_t& e : call)
                if (cudaEventCreate(&e) != cudaSuccess) return DRS_ERR_CUDA;
        g_timer.device = dev;
    }
    g_timer.calls = 0;
    g_timer.on = true;
    return DRS_OK;
}

extern "C" drs_status drs_kernel_times(float* avg_ms, int32_t n, int32_t* calls) {
    using namespace drs;
    if (!avg_ms || n < 0 || !calls) return DRS_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_timer_mutex);
    const int m = g_timer.calls < kTimedCalls ? g_timer.calls : kTimedCalls;
    *calls = m;
    for (int i = 0; i < n; ++i) avg_ms[i] = 0.0f;
    if (m == 0) return DRS_OK;
    for (int c = 0; c < m; ++c) {
        if (cudaEventSynchronize(g_timer.ev[c][kTimedKernels]) != cudaSuccess) return DRS_ERR_CUDA;
        for (int i = 0; i < n && i < kTimedKernels; ++i) {
            float ms = 0.0f;
            if (cudaEventElapsedTime(&ms, g_timer.ev[c][i], g_timer.ev[c][i + 1]) != cudaSuccess)
                return DRS_ERR_CUDA;
            avg_ms[i] += ms / static_cast<float>(m);
        }
    }
    return DRS_OK;
}

extern "C" const char* drs_status_string(drs_status s) {
    switch (s) {
        case DRS_OK: return "DRS_OK";
        case DRS_ERR_INVALID_ARG: return "DRS_ERR_INVALID_ARG";
        case DRS_ERR_UNSUPPORTED: return "DRS_ERR_UNSUPPORTED";
        case DRS_ERR_CUDA: return "DRS_ERR_CUDA";
        case DRS_ERR_DEVICE_TIMEOUT: return "DRS_ERR_DEVICE_TIMEOUT";
    }
    return "DRS_ERR_UNKNOWN";
}

extern "C" drs_status drs_get_device_error(void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return DRS_ERR_CUDA;
    int* flag = drs::device_error_flag();
    if (!flag) return DRS_ERR_CUDA;
    int value = 0;
    if (cudaMemcpy(&value, flag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return DRS_ERR_CUDA;
    if (value != 0) {
        const int zero = 0;
        if (cudaMemcpy(flag, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return DRS_ERR_CUDA;
        return DRS_ERR_DEVICE_TIMEOUT;
    }
    return DRS_OK;
}
