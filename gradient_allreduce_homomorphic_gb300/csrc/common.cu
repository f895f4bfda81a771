// common.cu -- error reporting, launch checks and device queries.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace gar {

namespace {
thread_local char g_last_error[512] = "";
std::atomic<unsigned long long> g_launches{0};
}

int fail(int status, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return status;
}

int check_launch(const char *what) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(GAR_ECUDA, "%s: %s", what, cudaGetErrorString(e));
    return GAR_OK;
}

int sm_count() {
    static std::atomic<int> cached[64];  // 0: not looked up yet (threads may race to fill it: same value)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

namespace {
__device__ unsigned int g_device_status;  // per device: GAR_STATUS_* bits, zero at load
std::mutex g_status_mutex;
unsigned int *g_status_addr[64] = {};
}  // namespace

unsigned int *device_status() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mutex);
    if (!g_status_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status_addr[dev] = static_cast<unsigned int *>(p);
    }
    return g_status_addr[dev];
}

}  // namespace gar

extern "C" int gar_sync_status(gar_stream_t stream, uint32_t *status, int32_t clear) {
    if (!status) return gar::fail(GAR_EINVAL, "status is NULL");
    unsigned int *d = gar::device_status();
    if (!d) return gar::fail(GAR_ECUDA, "the device status word is not available");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemcpy(status, d, sizeof(unsigned int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && clear) e = cudaMemset(d, 0, sizeof(unsigned int));
    if (e != cudaSuccess) return gar::fail(GAR_ECUDA, "gar_sync_status: %s", cudaGetErrorString(e));
    return GAR_OK;
}

extern "C" int gar_version(void) { return 100; }

extern "C" const char *gar_last_error(void) { return gar::g_last_error; }

extern "C" uint64_t gar_launch_count(void) { return gar::g_launches.load(std::memory_order_relaxed); }
