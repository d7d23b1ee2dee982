// tb_common.cuh -- helpers shared by the library's translation units:
// argument checks, 128-bit streaming loads/stores, 16-bit float conversions,
// per-device properties and the device-side error word.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "tb.h"

namespace tb {

// ---------------------------------------------------------------- host helpers
inline bool aligned_to(const void* p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline size_t dtype_size(tb_dtype d) { return d == TB_F32 ? 4 : 2; }

inline bool dtype_valid(tb_dtype d) { return d == TB_F32 || d == TB_F16 || d == TB_BF16; }

// Byte range [lo, hi) of a buffer; empty ranges never overlap anything.
struct Range {
    uintptr_t lo, hi;
};

inline Range range_of(const void* p, int64_t count, size_t esize) {
    uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + static_cast<uintptr_t>(count) * esize};
}

inline bool overlap(Range a, Range b) {
    if (a.lo == a.hi || b.lo == b.hi) return false;
    return a.lo < b.hi && b.lo < a.hi;
}

// Properties of a device, queried once and cached (thread-safe).
struct DeviceInfo {
    int sm_count;
    int max_smem_optin;   // bytes of dynamic shared memory a block may opt into
};

// Fills `info` for the current device; returns false on a CUDA error.
bool current_device_info(int* device, DeviceInfo* info);

// Unique id of the CUDA context current on this thread (0 when there is none or it
// cannot be read).  Ids are never reused within a process.
unsigned long long current_context_id();

// Device address of a __device__ variable in the current context, looked up with
// cudaGetSymbolAddress and cached against the context's id: a device reset ends
// the context, and the next context may load the module at other addresses, so a
// new id means a new lookup.  Not thread-safe by itself (callers hold a lock).
struct CachedAddress {
    unsigned long long ctx_id = 0;
    void* ptr = nullptr;
    void* get(const void* symbol);   // nullptr on a CUDA error
};

// Address of the device-side error word on the current device (nullptr on error).
int* device_error_word();

// CTAs of `kernel` that fit on one SM of the current device with `threads`
// threads and `dyn_smem` bytes of dynamic shared memory (0 on a CUDA error).
// First raises the kernel's dynamic shared-memory limit to dyn_smem when that
// is above the default; results are cached per (device, kernel, threads, smem).
int resident_ctas_per_sm(const void* kernel, int threads, size_t dyn_smem);

// Clusters of `cluster` CTAs of `kernel` that fit on the current device at once
// with `threads` threads and `dyn_smem` bytes of dynamic shared memory per CTA
// (0 on a CUDA error, or when such a cluster cannot be placed).  Raises the
// kernel's dynamic shared-memory limit first, as resident_ctas_per_sm does.
int resident_clusters(const void* kernel, int threads, size_t dyn_smem, int cluster);

inline tb_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? TB_OK : TB_ERR_CUDA;
}

// ---------------------------------------------------------------- programmatic dependent launch
// Kernels of this library are launched as programmatic dependents of the work
// before them in the stream: their CTAs may be placed on the SMs while the
// previous kernel drains, do their set-up (shared memory, barriers), and then
// wait in pdl_wait() until every prerequisite grid has completed and its memory
// is visible.  No global memory is loaded or stored before that wait (an L2
// prefetch, which returns nothing to the kernel, may be issued).  Launched
// without the attribute (or after work that is not a kernel), the wait returns
// at once.  pdl_trigger() lets the next programmatic dependent be scheduled
// early; that kernel still waits for this one to complete before it touches
// memory, so the trigger may be placed anywhere.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches `kernel` on `st` with the programmatic-stream-serialization attribute.
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Launches `kernel` on `st` in thread-block clusters of `cluster` CTAs along x
// (grid.x a multiple of `cluster`), in plain stream order: it starts once the
// previous work in the stream has completed, so every cluster finds its SMs free
// (its pdl_wait() returns at once).
template <class... KArgs, class... Args>
inline cudaError_t launch_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t st, int cluster, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- device helpers
// 128-bit loads/stores with the streaming (evict-first) cache policy: each
// element is touched once, so nothing is worth keeping in L1 or L2.
__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
    return __ldcs(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_stream_f4(float* p, float4 v) {
    __stcs(reinterpret_cast<float4*>(p), v);
}
__device__ __forceinline__ void st_stream_u4(void* p, uint4 v) {
    __stcs(reinterpret_cast<uint4*>(p), v);
}

// 16-bit storage types.  Conversions to fp32 are exact; conversions from fp32
// round to nearest even.
struct BF16 {
    using T = __nv_bfloat16;
    __device__ __forceinline__ static float to_f32(T x) { return __bfloat162float(x); }
    __device__ __forceinline__ static T from_f32(float x) { return __float2bfloat16_rn(x); }
};
struct F16 {
    using T = __half;
    __device__ __forceinline__ static float to_f32(T x) { return __half2float(x); }
    __device__ __forceinline__ static T from_f32(float x) { return __float2half_rn(x); }
};
struct F32 {
    using T = float;
    __device__ __forceinline__ static float to_f32(T x) { return x; }
    __device__ __forceinline__ static T from_f32(float x) { return x; }
};

// Unpack / pack 8 16-bit values held in a uint4.
template <class Fmt>
__device__ __forceinline__ void unpack8(uint4 u, float (&f)[8]) {
    const typename Fmt::T* h = reinterpret_cast<const typename Fmt::T*>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = Fmt::to_f32(h[i]);
}
template <class Fmt>
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 u;
    typename Fmt::T* h = reinterpret_cast<typename Fmt::T*>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = Fmt::from_f32(f[i]);
    return u;
}

// Elements per 16-byte vector for a storage format.
template <class Fmt>
struct Vec {
    static constexpr int kElems = 16 / sizeof(typename Fmt::T);
};

// Load / store one 16-byte vector of Fmt as kElems fp32 values.
template <class Fmt>
__device__ __forceinline__ void load_vec(const void* p, float (&f)[Vec<Fmt>::kElems]);
template <>
__device__ __forceinline__ void load_vec<F32>(const void* p, float (&f)[4]) {
    float4 v = ld_stream_f4(static_cast<const float*>(p));
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
template <>
__device__ __forceinline__ void load_vec<BF16>(const void* p, float (&f)[8]) {
    unpack8<BF16>(ld_stream_u4(p), f);
}
template <>
__device__ __forceinline__ void load_vec<F16>(const void* p, float (&f)[8]) {
    unpack8<F16>(ld_stream_u4(p), f);
}

template <class Fmt>
__device__ __forceinline__ void store_vec(void* p, const float (&f)[Vec<Fmt>::kElems]);
template <>
__device__ __forceinline__ void store_vec<F32>(void* p, const float (&f)[4]) {
    st_stream_f4(static_cast<float*>(p), make_float4(f[0], f[1], f[2], f[3]));
}
template <>
__device__ __forceinline__ void store_vec<BF16>(void* p, const float (&f)[8]) {
    st_stream_u4(p, pack8<BF16>(f));
}
template <>
__device__ __forceinline__ void store_vec<F16>(void* p, const float (&f)[8]) {
    st_stream_u4(p, pack8<F16>(f));
}

}  // namespace tb
