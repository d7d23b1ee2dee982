// cast.cu -- stand-alone precision casts of the mixed-precision training loop.
//
// "GPU 优化实战 Part 2：用 CUDA/ROCm 实现 LLM 反向传播与训练循环", sections
// "混合精度训练（FP16 / BF16）" and "完整训练循环（整合一切）" (the unscale cast and the
// copy-back cast of the loop): the low-precision gradient is cast to fp32 and
// multiplied by 1/loss_scale before the optimizer, and the fp32 master weights
// are cast back to a 16-bit working copy after it.  The fused AdamW step does both inside its single pass; these
// kernels exist for callers that keep the steps apart (and to time that unfused
// pipeline against the fused one).
//
//   tb_cast_to_f32   : dst = float(src) * scale   (one fp32 rounding of the product)
//   tb_cast_from_f32 : dst = round-to-nearest-even(src) in a 16-bit format
//
// Vector paths grid-stride over 4-element chunks, one chunk per lane per access:
// the fp32 side moves 16 bytes per lane and the 16-bit side 8, so every warp
// access covers whole 32-byte sectors; four chunks are in flight per thread.
// Widening a 16-bit source into a 32-byte aligned destination uses 8-element
// units instead: one 16-byte load and one 32-byte store (sm_100's 256-bit
// st.global) per lane, which measured 20% faster than two 16-byte stores per
// unit.  A scalar loop covers misaligned buffers and the ragged tail.  The grid
// has one CTA per pass of the loop (not a persistent grid), so the block
// scheduler balances the SMs.
#include <algorithm>

#include "tb_common.cuh"

namespace tb {
namespace {

constexpr int kThreads = 256;

// Eight 16-bit source elements (one 16-byte vector) as fp32.
template <class S>
__device__ __forceinline__ void load8(const void* p, int64_t i0, float (&f)[8]) {
    unpack8<S>(ld_stream_u4(static_cast<const typename S::T*>(p) + i0), f);
}

// Four source elements as fp32 (16-bit formats: one 8-byte access; fp32: 16 bytes).
template <class S>
__device__ __forceinline__ void load4(const void* p, int64_t i0, float (&f)[4]) {
    const uint2 u = __ldcs(reinterpret_cast<const uint2*>(static_cast<const typename S::T*>(p) + i0));
    const typename S::T* h = reinterpret_cast<const typename S::T*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = S::to_f32(h[i]);
}
template <>
__device__ __forceinline__ void load4<F32>(const void* p, int64_t i0, float (&f)[4]) {
    const float4 a = ld_stream_f4(static_cast<const float*>(p) + i0);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
}

__device__ __forceinline__ void st_stream_v8(float* p, const float (&f)[8]) {
    asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(f[0]),
                 "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7])
                 : "memory");
}

template <class S>
__global__ void __launch_bounds__(kThreads)
cast_to_f32_kernel(const void* __restrict__ src, float* __restrict__ dst, int64_t n, float scale,
                   int vec) {
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    int64_t done = 0;
    bool wide = false;
    if constexpr (sizeof(typename S::T) == 2) {
        if (vec == 2) {
            // 32-byte aligned destination: one 16-byte load and one 32-byte store per
            // unit, four units in flight per thread
            wide = true;
            const int64_t units = n / 8;
            for (int64_t u = tid; u < units; u += 4 * stride) {
                float f[4][8];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (u + j * stride < units) load8<S>(src, (u + j * stride) * 8, f[j]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (u + j * stride < units) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) f[j][q] *= scale;
                        st_stream_v8(dst + (u + j * stride) * 8, f[j]);
                    }
                }
            }
            done = units * 8;
        }
    }
    if (!wide && vec) {
        const int64_t chunks = n / 4;
        for (int64_t c = tid; c < chunks; c += 4 * stride) {
            float f[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (c + j * stride < chunks) load4<S>(src, (c + j * stride) * 4, f[j]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (c + j * stride < chunks)
                    st_stream_f4(dst + (c + j * stride) * 4, make_float4(f[j][0] * scale, f[j][1] * scale,
                                                                         f[j][2] * scale, f[j][3] * scale));
            }
        }
        done = chunks * 4;
    }
    const typename S::T* s = static_cast<const typename S::T*>(src);
    for (int64_t i = done + tid; i < n; i += stride) dst[i] = S::to_f32(s[i]) * scale;
}

template <class D>
__global__ void __launch_bounds__(kThreads)
cast_from_f32_kernel(const float* __restrict__ src, void* __restrict__ dst, int64_t n, int vec) {
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    typename D::T* d = static_cast<typename D::T*>(dst);
    int64_t done = 0;
    if (vec) {
        const int64_t chunks = n / 4;
        for (int64_t c = tid; c < chunks; c += 4 * stride) {
            float4 f[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (c + j * stride < chunks) f[j] = ld_stream_f4(src + (c + j * stride) * 4);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (c + j * stride < chunks) {
                    uint2 u;
                    typename D::T* h = reinterpret_cast<typename D::T*>(&u);
                    h[0] = D::from_f32(f[j].x);
                    h[1] = D::from_f32(f[j].y);
                    h[2] = D::from_f32(f[j].z);
                    h[3] = D::from_f32(f[j].w);
                    __stcs(reinterpret_cast<uint2*>(d + (c + j * stride) * 4), u);
                }
            }
        }
        done = chunks * 4;
    }
    for (int64_t i = done + tid; i < n; i += stride) d[i] = D::from_f32(src[i]);
}

// One CTA per `per_cta` elements: each CTA makes one pass of its loop and exits, and
// the block scheduler hands the next block to whichever SM has room.  A persistent
// grid gives every thread a fixed share, and the SMs of a GB300 do not stream at one
// rate; on 2^30 elements one pass per CTA measured 924 against 1,025 us (widening,
// 32-byte stores), 1,004 against 1,252 us (widening, 16-byte stores) and 899 against
// 976 us (narrowing).  The loops grid-stride, so the cap at the launch limit still
// covers every element.  0 when the occupancy query failed.
unsigned grid_for(const void* kernel, int64_t n, int64_t per_cta) {
    if (resident_ctas_per_sm(kernel, kThreads, 0) == 0) return 0;
    return (unsigned)std::max<int64_t>(1, std::min<int64_t>((n + per_cta - 1) / per_cta, INT32_MAX));
}

}  // namespace
}  // namespace tb

extern "C" tb_status tb_cast_to_f32(const void* src, tb_dtype src_dtype, float scale, float* dst,
                                    int64_t n, void* stream) {
    using namespace tb;
    if (n < 0) return TB_ERR_INVALID_VALUE;
    if (!dtype_valid(src_dtype)) return TB_ERR_UNSUPPORTED_DTYPE;
    if (n == 0) return TB_OK;
    if (!src || !dst || n > INT64_MAX / 8) return TB_ERR_INVALID_VALUE;
    const size_t es = dtype_size(src_dtype);
    if (!aligned_to(src, es) || !aligned_to(dst, 4)) return TB_ERR_MISALIGNED;
    if (overlap(range_of(src, n, es), range_of(dst, n, 4))) return TB_ERR_ALIAS;
    int dev = 0;
    DeviceInfo info{};
    if (!current_device_info(&dev, &info)) return TB_ERR_CUDA;
    // 2: 8-element units with 32-byte stores (16-bit source); 1: 4-element chunks
    int vec = es == 2 && aligned_to(src, 16) && aligned_to(dst, 32) ? 2
                  : aligned_to(src, 4 * es) && aligned_to(dst, 16) ? 1 : 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const void* k = src_dtype == TB_BF16 ? reinterpret_cast<const void*>(&cast_to_f32_kernel<BF16>)
                  : src_dtype == TB_F16  ? reinterpret_cast<const void*>(&cast_to_f32_kernel<F16>)
                                         : reinterpret_cast<const void*>(&cast_to_f32_kernel<F32>);
    void* args[] = {&src, &dst, &n, &scale, &vec};
    const unsigned grid = grid_for(k, n, (int64_t)kThreads * 32);   // 8,192 elements per CTA
    if (grid == 0 || cudaLaunchKernel(k, dim3(grid), dim3(kThreads), args, 0, st) != cudaSuccess)
        return TB_ERR_CUDA;
    return TB_OK;
}

extern "C" tb_status tb_cast_from_f32(const float* src, void* dst, tb_dtype dst_dtype, int64_t n,
                                      void* stream) {
    using namespace tb;
    if (n < 0) return TB_ERR_INVALID_VALUE;
    if (dst_dtype != TB_BF16 && dst_dtype != TB_F16) return TB_ERR_UNSUPPORTED_DTYPE;
    if (n == 0) return TB_OK;
    if (!src || !dst || n > INT64_MAX / 8) return TB_ERR_INVALID_VALUE;
    if (!aligned_to(src, 4) || !aligned_to(dst, 2)) return TB_ERR_MISALIGNED;
    if (overlap(range_of(src, n, 4), range_of(dst, n, 2))) return TB_ERR_ALIAS;
    int dev = 0;
    DeviceInfo info{};
    if (!current_device_info(&dev, &info)) return TB_ERR_CUDA;
    int vec = aligned_to(src, 16) && aligned_to(dst, 8);   // 4-element chunks
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const void* k = dst_dtype == TB_BF16 ? reinterpret_cast<const void*>(&cast_from_f32_kernel<BF16>)
                                         : reinterpret_cast<const void*>(&cast_from_f32_kernel<F16>);
    void* args[] = {&src, &dst, &n, &vec};
    const unsigned grid = grid_for(k, n, (int64_t)kThreads * 16);   // 4,096 elements per CTA
    if (grid == 0 || cudaLaunchKernel(k, dim3(grid), dim3(kThreads), args, 0, st) != cudaSuccess)
        return TB_ERR_CUDA;
    return TB_OK;
}
