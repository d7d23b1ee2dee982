// api.cu -- status strings, version, per-device property cache, the identity of
// the current CUDA context and the device-side error word.
#include <cuda.h>

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
CachedAddress g_err_addr[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
std::once_flag g_ctx_once;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
}  // namespace

unsigned long long current_context_id() {
    std::call_once(g_ctx_once, [] {
        auto resolve = [](const char* name) -> void* {
            void* f = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess) {
                cudaGetLastError();   // clear this call's own error only
                return nullptr;
            }
            return q == cudaDriverEntryPointSuccess ? f : nullptr;
        };
        g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(resolve("cuCtxGetCurrent"));
        g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(resolve("cuCtxGetId"));
    });
    if (!g_ctx_get_current || !g_ctx_get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

void* CachedAddress::get(const void* symbol) {
    const unsigned long long id = current_context_id();
    if (id != 0 && id == ctx_id) return ptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    // The lookup creates the context if there was none yet: key on the id it has now.
    ctx_id = current_context_id();
    ptr = ctx_id != 0 ? p : nullptr;
    return p;
}

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
    return static_cast<int*>(g_err_addr[dev].get(&g_device_error));
}

namespace {
std::mutex g_occ_mu;
// Keyed on the context id as well: a kernel's raised shared-memory limit belongs
// to the context it was set in.
std::map<std::tuple<int, unsigned long long, const void*, int, size_t>, int> g_occ;  // -> CTAs per SM
std::map<std::tuple<int, unsigned long long, const void*>, size_t> g_smem_limit;     // -> limit set
}  // namespace

int resident_ctas_per_sm(const void* kernel, int threads, size_t dyn_smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lk(g_occ_mu);
    try {
        const auto key = std::make_tuple(dev, ctx, kernel, threads, dyn_smem);
        const auto it = g_occ.find(key);
        if (it != g_occ.end() && ctx != 0) return it->second;
        if (dyn_smem > 48 * 1024) {
            // without a context id nothing is cached: the limit is set every time
            size_t unused = 0;
            size_t& lim = ctx != 0 ? g_smem_limit[std::make_tuple(dev, ctx, kernel)] : unused;
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
        if (ctx != 0) g_occ.emplace(key, per_sm);
        return per_sm;
    } catch (...) {
        return 0;
    }
}

int resident_clusters(const void* kernel, int threads, size_t dyn_smem, int cluster) {
    if (cluster < 1 || resident_ctas_per_sm(kernel, threads, dyn_smem) == 0) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const unsigned long long ctx = current_context_id();
    static std::mutex mu;
    static std::map<std::tuple<int, unsigned long long, const void*, int, size_t, int>, int> cache;
    std::lock_guard<std::mutex> lk(mu);
    try {
        const auto key = std::make_tuple(dev, ctx, kernel, threads, dyn_smem, cluster);
        const auto it = cache.find(key);
        if (it != cache.end() && ctx != 0) return it->second;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)cluster);
        cfg.blockDim = dim3((unsigned)threads);
        cfg.dynamicSmemBytes = dyn_smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        if (ctx != 0) cache.emplace(key, n);
        return n;
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
