// api.cu -- status strings, version, per-device property cache and the
// device-side error word.
#include <map>
#include <mutex>
#include <tuple>

#include "tb_common.cuh"

namespace tb {

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
bool g_have[kMaxDevices] = {};
DeviceInfo g_info[kMaxDevices];
int* g_err_ptr[kMaxDevices] = {};
}  // namespace

// Set by kernels whose bounded waits give up; read by tb_device_error.
__device__ int g_device_error = 0;

bool current_device_info(int* device, DeviceInfo* info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    *device = dev;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_have[dev]) {
        DeviceInfo d{};
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return false;
        if (cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                   dev) != cudaSuccess)
            return false;
        g_info[dev] = d;
        g_have[dev] = true;
    }
    *info = g_info[dev];
    return true;
}

int* device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<int*>(p);
    }
    return g_err_ptr[dev];
}

namespace {
std::mutex g_occ_mu;
std::map<std::tuple<int, const void*, int, size_t>, int> g_occ;   // -> CTAs per SM
std::map<std::pair<int, const void*>, size_t> g_smem_limit;        // -> limit set so far
}  // namespace

int resident_ctas_per_sm(const void* kernel, int threads, size_t dyn_smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lk(g_occ_mu);
    try {
        const auto key = std::make_tuple(dev, kernel, threads, dyn_smem);
        const auto it = g_occ.find(key);
        if (it != g_occ.end()) return it->second;
        if (dyn_smem > 48 * 1024) {
            size_t& lim = g_smem_limit[std::make_pair(dev, kernel)];
            if (lim < dyn_smem) {
                if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)dyn_smem) != cudaSuccess)
                    return 0;
                lim = dyn_smem;
            }
        }
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, dyn_smem) !=
            cudaSuccess)
            return 0;
        g_occ.emplace(key, per_sm);
        return per_sm;
    } catch (...) {
        return 0;
    }
}

}  // namespace tb

extern "C" const char* tb_status_string(tb_status s) {
    switch (s) {
        case TB_OK: return "TB_OK";
        case TB_ERR_INVALID_VALUE: return "TB_ERR_INVALID_VALUE";
        case TB_ERR_UNSUPPORTED_DTYPE: return "TB_ERR_UNSUPPORTED_DTYPE";
        case TB_ERR_MISALIGNED: return "TB_ERR_MISALIGNED";
        case TB_ERR_ALIAS: return "TB_ERR_ALIAS";
        case TB_ERR_WORKSPACE: return "TB_ERR_WORKSPACE";
        case TB_ERR_OOM: return "TB_ERR_OOM";
        case TB_ERR_CUDA: return "TB_ERR_CUDA";
        case TB_ERR_DEVICE: return "TB_ERR_DEVICE";
        case TB_ERR_TIMEOUT: return "TB_ERR_TIMEOUT";
    }
    return "TB_ERR_UNKNOWN";
}

extern "C" int tb_version(void) { return 100; }

extern "C" tb_status tb_device_error(int* code, int reset) {
    if (!code) return TB_ERR_INVALID_VALUE;
    if (cudaDeviceSynchronize() != cudaSuccess) return TB_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, tb::g_device_error, sizeof(int)) != cudaSuccess) return TB_ERR_CUDA;
    if (reset && v) {
        int zero = 0;
        if (cudaMemcpyToSymbol(tb::g_device_error, &zero, sizeof(int)) != cudaSuccess)
            return TB_ERR_CUDA;
    }
    *code = v;
    return TB_OK;
}
