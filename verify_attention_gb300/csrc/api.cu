// api.cu -- status strings, device status word, dispatch record, device facts.
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "attention.cuh"
#include "common.cuh"

namespace fp8kv {

static thread_local char g_dispatch[256] = "";
static std::atomic<unsigned long long> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void set_dispatch(const char* text) {
    strncpy(g_dispatch, text, sizeof g_dispatch - 1);
    g_dispatch[sizeof g_dispatch - 1] = 0;
}

int launch_status() { return cudaGetLastError() == cudaSuccess ? FP8KV_OK : FP8KV_ERR_CUDA; }

int num_sms() {
    static std::mutex mu;
    static std::vector<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;      // no device: plan for a GB300
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace fp8kv

extern "C" const char* fp8kv_status_string(int status) {
    switch (status) {
        case FP8KV_OK: return "ok";
        case FP8KV_ERR_INVALID_ARG: return "invalid argument";
        case FP8KV_ERR_UNSUPPORTED: return "unsupported shape";
        case FP8KV_ERR_WORKSPACE: return "workspace missing or too small";
        case FP8KV_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

extern "C" int fp8kv_last_dispatch(char* buf, size_t n) {
    const size_t len = strlen(fp8kv::g_dispatch);
    if (buf && n) {
        const size_t k = len < n - 1 ? len : n - 1;
        memcpy(buf, fp8kv::g_dispatch, k);
        buf[k] = 0;
    }
    return (int)len;
}

extern "C" int fp8kv_device_status(unsigned int* status, int clear) {
    if (!status) return FP8KV_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return FP8KV_ERR_CUDA;
    unsigned int s = 0;
    if (fp8kv::status_insert(&s, clear) || fp8kv::status_attention(&s, clear) ||
        fp8kv::status_attention_tc(&s, clear) || fp8kv::status_attention_layers(&s, clear))
        return FP8KV_ERR_CUDA;
    *status = s;
    return FP8KV_OK;
}

extern "C" unsigned long long fp8kv_launch_count(void) { return fp8kv::g_launches.load(std::memory_order_relaxed); }
