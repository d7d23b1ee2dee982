// layernorm_bwd.cu -- LayerNorm backward from the saved mean / inv_std.
//
//   xhat = (x - mean) * inv_std,  dxhat = dY * gamma
//   dX   = inv_std * (dxhat - mean_D(dxhat) - xhat * mean_D(dxhat * xhat))
//   dgamma_j = sum_rows dY*xhat,  dbeta_j = sum_rows dY
// ("GPU 优化实战 Part 2：用 CUDA/ROCm 实现 LLM 反向传播与训练循环", section 2.2
// "LayerNorm 反向": saved mean/inv_std, gamma/beta gradients by reduction, dX
// from the normalised values; the reduction runs over rows, per feature.)
//
// Design (GB300):
//  * Kernel 1 (rows): persistent CTAs, each owning a contiguous block of rows.
//    One elected thread streams groups of x and dY rows into a ring of
//    shared-memory stages with 1-D bulk async copies (cp.async.bulk, completion
//    counted on an mbarrier), several groups ahead, so HBM stays busy without
//    holding the rows in registers.  It is launched as a programmatic
//    dependent: its CTAs set up their barriers and prefetch their first stage
//    into L2 while the previous kernel drains, and copy nothing before that
//    kernel has completed.  Each thread owns a fixed set of 16-byte column
//    vectors: it keeps gamma and its dgamma/dbeta partial sums for those
//    columns in registers across all rows of the CTA.  Phase 1 reads the staged
//    rows and forms the two row sums (dxhat, dxhat*xhat) with a warp butterfly
//    plus one shared-memory exchange and one barrier per group; phase 2
//    re-reads the staged rows (shared memory, not HBM), writes dX and
//    accumulates the column partials.  A stage is refilled one group later,
//    once every thread is past it.  At the end each CTA stores its column
//    partials to the workspace.  CTAs have 1..8 warps (ring bytes in proportion
//    to the warps, so short rows fit several CTAs per SM), or up to 16 for
//    16-bit rows of 4097..8192 columns (16 columns a thread instead of 32).
//  * Kernel 1' (rows longer than 16 KB): the same ring, with each row
//    split by columns over the 2..8 CTAs of a thread-block cluster.  Every CTA
//    keeps the gamma and partials of its column slice in registers (so two CTAs
//    still fit per SM) and the CTAs exchange their shares of the two row sums
//    through distributed shared memory (st.async into the peers' exchange
//    slots, counted on an mbarrier there) -- one exchange per row group.
//  * Kernel 2 (columns): adds the per-CTA (per-cluster) partials in a fixed
//    order -> dgamma, dbeta, bitwise reproducible run to run.
//  * Rows the bulk copies cannot take (unaligned buffers, byte lengths not a
//    multiple of 16) run a register-row kernel of the same structure with
//    scalar coalesced loads and an L2 prefetch of the rows ahead, up to 8192
//    columns; beyond that a last-resort kernel makes two global passes per row
//    and keeps the partials in the workspace.
//
// RMSNorm backward (tb_rmsnorm_bwd) runs the same kernels with kRms set:
//   xhat = x * inv_rms, dX = inv_rms * (dxhat - xhat * mean_D(dxhat * xhat)),
//   dgamma_j = sum_rows dY*xhat -- the LayerNorm above without the mean and beta.
//
// Every mbarrier wait is bounded (about one second of %globaltimer); on expiry
// the CTA sets the device error word, waits (bounded) for the copies it issued
// and returns.
#include <algorithm>
#include <type_traits>
#include <mutex>

#include "tb_common.cuh"

namespace tb {
namespace {

constexpr int kRowThreads = 256;               // max threads of the row kernels
constexpr int kMaxWarps = kRowThreads / 32;
constexpr int kWideWarps = 16;                 // warps of the wide ring variant (512 threads)
constexpr int kWidePairThreads = 320;          // wide CTAs up to this size run two per SM
constexpr int kMaxStages = 4;
constexpr int kMaxElemsPerThread = 32;
constexpr int kRingBudget = 96 * 1024;         // bytes of ring per CTA we aim for
constexpr int kStageTargetBytes = 32 * 1024;   // x + dY bytes per ring stage we aim for
constexpr int kBarRegion = 128;                // bytes reserved for the mbarriers
constexpr unsigned long long kWaitLimitNs = 1000000000ull;
constexpr int kMaxCluster = 8;                 // CTAs a row may be split over (portable size)
constexpr int64_t kSplitFromRowBytes = 16 * 1024;   // longer rows are split over a cluster
constexpr int64_t kSplitSliceTarget = 4096;    // columns per CTA we aim for when splitting

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with this parity to complete; false after limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1; it < (1u << 30); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0 && global_ns() - t0 > limit_ns) return false;
    }
    return false;
}

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared; completion is counted on `bar` (tx bytes).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// Asynchronous prefetch of global memory into L2 (no data reaches the SM).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Thread-block cluster: this CTA's rank, the cluster's CTA count, the cluster's index.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Store 4 bytes into another CTA's shared memory (remote_addr), counted as 4
// transaction bytes on that CTA's mbarrier (remote_bar).
__device__ __forceinline__ void st_async_remote(uint32_t remote_addr, float v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(
                     remote_addr),
                 "r"(__float_as_uint(v)), "r"(remote_bar)
                 : "memory");
}

// Every thread of every CTA of the cluster arrives and waits (the non-.aligned
// form: the threads of a warp need not arrive converged).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// As mbar_try_wait, acquiring what other CTAs of the cluster released into the phase.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint32_t bar, uint32_t parity,
                                                          unsigned long long limit_ns) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1; it < (1u << 30); ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 63u) == 0 && global_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// Read one 16-byte vector from shared memory as fp32 values.
template <class Fmt>
__device__ __forceinline__ void lds_vec(const void* p, float (&f)[Vec<Fmt>::kElems]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const typename Fmt::T* h = reinterpret_cast<const typename Fmt::T*>(&u);
#pragma unroll
    for (int e = 0; e < Vec<Fmt>::kElems; ++e) f[e] = Fmt::to_f32(h[e]);
}

// Warp sum of V values per lane (V a power of two <= 16) with V-1+5-log2(V)
// shuffles instead of 5V: each of the first log2(V) butterfly levels halves the
// values a lane carries.  Afterwards lane l holds the full sum of value
// multi_index<V>(l); the lanes whose bits below the last split are zero hold
// all V sums between them.
template <int V>
struct Log2 { static constexpr int value = V <= 1 ? 0 : 1 + Log2<V / 2>::value; };
template <>
struct Log2<1> { static constexpr int value = 0; };

template <int V>
__device__ __forceinline__ float warp_sum_multi(float (&v)[V], int lane) {
    constexpr int L = Log2<V>::value;
#pragma unroll
    for (int lvl = 0; lvl < L; ++lvl) {
        const int o = 16 >> lvl;
        const int half = V >> (lvl + 1);
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float r = v[0];
#pragma unroll
    for (int o = 16 >> L; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

template <int V>
__device__ __forceinline__ int multi_index(int lane) {
    constexpr int L = Log2<V>::value;
    int idx = 0;
#pragma unroll
    for (int lvl = 0; lvl < L; ++lvl)
        if (lane & (16 >> lvl)) idx += V >> (lvl + 1);
    return idx;
}

template <int V>
__device__ __forceinline__ bool multi_writer(int lane) {
    constexpr int L = Log2<V>::value;
    return L == 0 ? lane == 0 : (lane & ((32 >> L) - 1)) == 0;
}

// One 16-byte shared-memory vector as E/2 fp32 pairs (packed f32x2 math below).
// bf16 widens exactly by moving its bits to the high half (a byte permute for the
// low element, a mask for the high one); fp16 with the half2 conversion.
template <class Fmt>
struct Pairs {
    static constexpr int kN = Vec<Fmt>::kElems / 2;
};

template <class Fmt>
__device__ __forceinline__ void lds_pairs(const void* p, float2 (&f)[Pairs<Fmt>::kN]);
template <>
__device__ __forceinline__ void lds_pairs<F32>(const void* p, float2 (&f)[2]) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    f[0] = make_float2(u.x, u.y);
    f[1] = make_float2(u.z, u.w);
}
template <>
__device__ __forceinline__ void lds_pairs<BF16>(const void* p, float2 (&f)[4]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        f[i] = make_float2(__uint_as_float(__byte_perm(w[i], 0u, 0x1044)),
                           __uint_as_float(w[i] & 0xffff0000u));
}
template <>
__device__ __forceinline__ void lds_pairs<F16>(const void* p, float2 (&f)[4]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
}

// Store E/2 fp32 pairs as one 16-byte global vector (round to nearest even).
template <class Fmt>
__device__ __forceinline__ void stg_pairs(void* p, const float2 (&f)[Pairs<Fmt>::kN]);
template <>
__device__ __forceinline__ void stg_pairs<F32>(void* p, const float2 (&f)[2]) {
    st_stream_f4(static_cast<float*>(p), make_float4(f[0].x, f[0].y, f[1].x, f[1].y));
}
template <>
__device__ __forceinline__ void stg_pairs<BF16>(void* p, const float2 (&f)[4]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(f[i].x, f[i].y);
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    st_stream_u4(p, make_uint4(w[0], w[1], w[2], w[3]));
}
template <>
__device__ __forceinline__ void stg_pairs<F16>(void* p, const float2 (&f)[4]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(f[i].x, f[i].y);
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    st_stream_u4(p, make_uint4(w[0], w[1], w[2], w[3]));
}

// (x - mu) for the two 16-bit values packed in w, each widened inside the
// subtraction (sub.f32.bf16 / sub.f32.f16, mixed-precision forms of sm_100-class
// targets): the same values as widening first, one instruction fewer per element.
template <class Fmt> __device__ __forceinline__ float2 sub_mu_pair(uint32_t w, float mu);
template <> __device__ __forceinline__ float2 sub_mu_pair<BF16>(uint32_t w, float mu) {
    float lo, hi;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "sub.rn.f32.bf16 %0, l, %3;\n\tsub.rn.f32.bf16 %1, h, %3;\n\t}"
        : "=f"(lo), "=f"(hi) : "r"(w), "f"(mu));
    return make_float2(lo, hi);
}
template <> __device__ __forceinline__ float2 sub_mu_pair<F16>(uint32_t w, float mu) {
    float lo, hi;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "sub.rn.f32.f16 %0, l, %3;\n\tsub.rn.f32.f16 %1, h, %3;\n\t}"
        : "=f"(lo), "=f"(hi) : "r"(w), "f"(mu));
    return make_float2(lo, hi);
}

// ------------------------------------------------------------------ per-row math (both ring kernels)
// A thread owns the 16-byte column vectors vi = tid + k*nthreads (k < NV, vi <
// nvec) of the columns a CTA covers; g holds gamma for them, acc_g / acc_b the
// CTA's dgamma / dbeta partial sums.  xr and dyr point at the staged row (the
// CTA's columns of it) in shared memory.

// kMix (16-bit LayerNorm rows): x - mean by sub_mu_pair, from the raw staged words.

// Phase 1: this thread's shares of sum(dxhat) (sa) and sum(dxhat*xhat) (sb).
template <class Fmt, int NV, bool kRms, bool kMix = false>
__device__ __forceinline__ void row_shares(const unsigned char* xr, const unsigned char* dyr,
                                           const float2 (&g)[NV][Pairs<Fmt>::kN], float mu,
                                           float rs, int tid, int nthreads, int nvec, float& sa,
                                           float& sb) {
    constexpr int NP = Pairs<Fmt>::kN;
    float2 sa2 = make_float2(0.f, 0.f), sb2 = make_float2(0.f, 0.f);
    const float2 nmu = make_float2(-mu, -mu), rs2 = make_float2(rs, rs);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int vi = tid + k * nthreads;
        if constexpr (kMix) {
            if (vi < nvec) {
                const uint4 u = *reinterpret_cast<const uint4*>(xr + (size_t)vi * 16);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                float2 dy[NP];
                lds_pairs<Fmt>(dyr + (size_t)vi * 16, dy);
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    const float2 xh = __fmul2_rn(sub_mu_pair<Fmt>(w[q], mu), rs2);
                    const float2 dxh = __fmul2_rn(dy[q], g[k][q]);
                    sa2 = __fadd2_rn(sa2, dxh);
                    sb2 = __ffma2_rn(dxh, xh, sb2);
                }
            }
        } else if (vi < nvec) {
            float2 xv[NP], dy[NP];
            lds_pairs<Fmt>(xr + (size_t)vi * 16, xv);
            lds_pairs<Fmt>(dyr + (size_t)vi * 16, dy);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const float2 xh = kRms ? __fmul2_rn(xv[q], rs2)
                                       : __fmul2_rn(__fadd2_rn(xv[q], nmu), rs2);
                const float2 dxh = __fmul2_rn(dy[q], g[k][q]);
                if (!kRms) sa2 = __fadd2_rn(sa2, dxh);
                sb2 = __ffma2_rn(dxh, xh, sb2);
            }
        }
    }
    sa = sa2.x + sa2.y;
    sb = sb2.x + sb2.y;
}

// Phase 2: dX of the row (dxr: the CTA's first column of it in global memory)
// and the column partials, from the row means mean_a = mean(dxhat) and
// mean_b = mean(dxhat*xhat):
//   dX = rs*dxhat - rs*mean_a - rs*mean_b*xhat  (two packed FMAs per pair)
template <class Fmt, int NV, bool kRms, bool kMix = false>
__device__ __forceinline__ void row_dx(const unsigned char* xr, const unsigned char* dyr,
                                       typename Fmt::T* dxr, const float2 (&g)[NV][Pairs<Fmt>::kN],
                                       float2 (&acc_g)[NV][Pairs<Fmt>::kN],
                                       float2 (&acc_b)[NV][Pairs<Fmt>::kN], float mu, float rs,
                                       float mean_a, float mean_b, int tid, int nthreads,
                                       int nvec) {
    constexpr int NP = Pairs<Fmt>::kN;
    constexpr int E = Vec<Fmt>::kElems;
    const float2 nmu = make_float2(-mu, -mu), rs2 = make_float2(rs, rs);
    const float c0 = -(rs * mean_a), c1 = -(rs * mean_b);
    const float2 nc0 = make_float2(c0, c0), nc1 = make_float2(c1, c1);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int vi = tid + k * nthreads;
        if constexpr (kMix) {
            if (vi < nvec) {
                const uint4 u = *reinterpret_cast<const uint4*>(xr + (size_t)vi * 16);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                float2 dy[NP], out[NP];
                lds_pairs<Fmt>(dyr + (size_t)vi * 16, dy);
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    const float2 xh = __fmul2_rn(sub_mu_pair<Fmt>(w[q], mu), rs2);
                    const float2 dxh = __fmul2_rn(dy[q], g[k][q]);
                    out[q] = __ffma2_rn(dxh, rs2, __ffma2_rn(xh, nc1, nc0));
                    acc_g[k][q] = __ffma2_rn(dy[q], xh, acc_g[k][q]);
                    acc_b[k][q] = __fadd2_rn(acc_b[k][q], dy[q]);
                }
                stg_pairs<Fmt>(dxr + (size_t)vi * E, out);
            }
        } else if (vi < nvec) {
            float2 xv[NP], dy[NP], out[NP];
            lds_pairs<Fmt>(xr + (size_t)vi * 16, xv);
            lds_pairs<Fmt>(dyr + (size_t)vi * 16, dy);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const float2 xh = kRms ? __fmul2_rn(xv[q], rs2)
                                       : __fmul2_rn(__fadd2_rn(xv[q], nmu), rs2);
                const float2 dxh = __fmul2_rn(dy[q], g[k][q]);
                out[q] = __ffma2_rn(dxh, rs2, __ffma2_rn(xh, nc1, nc0));
                acc_g[k][q] = __ffma2_rn(dy[q], xh, acc_g[k][q]);
                if (!kRms) acc_b[k][q] = __fadd2_rn(acc_b[k][q], dy[q]);
            }
            stg_pairs<Fmt>(dxr + (size_t)vi * E, out);
        }
    }
}

// Sum of the W (8 or 16) per-warp values at p, in a fixed order.
template <int W = kMaxWarps>
__device__ __forceinline__ float cta_total(const float* p) {
    static_assert(W == 8 || W == 16, "8 or 16 warps");
    const float4 a0 = *reinterpret_cast<const float4*>(p);
    const float4 a1 = *reinterpret_cast<const float4*>(p + 4);
    const float t = ((a0.x + a0.y) + (a0.z + a0.w)) + ((a1.x + a1.y) + (a1.z + a1.w));
    if constexpr (W == 8) return t;
    else return t + cta_total<8>(p + 8);
}

// gamma of the thread's columns (zero past nvec); the partial sums start at zero.
template <class Fmt, int NV>
__device__ __forceinline__ void load_gamma(const float* __restrict__ gamma, float2 (&g)[NV][Pairs<Fmt>::kN],
                                           float2 (&acc_g)[NV][Pairs<Fmt>::kN],
                                           float2 (&acc_b)[NV][Pairs<Fmt>::kN], int tid,
                                           int nthreads, int nvec) {
    constexpr int E = Vec<Fmt>::kElems;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int vi = tid + k * nthreads;
#pragma unroll
        for (int q = 0; q < Pairs<Fmt>::kN; ++q) {
            g[k][q] = vi < nvec ? make_float2(gamma[vi * E + 2 * q], gamma[vi * E + 2 * q + 1])
                                : make_float2(0.f, 0.f);
            acc_g[k][q] = make_float2(0.f, 0.f);
            acc_b[k][q] = make_float2(0.f, 0.f);
        }
    }
}

// Store the thread's column partials (pg: dgamma partials of the CTA's first
// column; pb: dbeta partials, LayerNorm only).
template <class Fmt, int NV, bool kRms>
__device__ __forceinline__ void store_partials(float* pg, float* pb,
                                               const float2 (&acc_g)[NV][Pairs<Fmt>::kN],
                                               const float2 (&acc_b)[NV][Pairs<Fmt>::kN], int tid,
                                               int nthreads, int nvec) {
    constexpr int E = Vec<Fmt>::kElems;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int vi = tid + k * nthreads;
        if (vi < nvec) {
#pragma unroll
            for (int q = 0; q < Pairs<Fmt>::kN; q += 2) {
                *reinterpret_cast<float4*>(pg + vi * E + 2 * q) =
                    make_float4(acc_g[k][q].x, acc_g[k][q].y, acc_g[k][q + 1].x, acc_g[k][q + 1].y);
                if (!kRms)
                    *reinterpret_cast<float4*>(pb + vi * E + 2 * q) =
                        make_float4(acc_b[k][q].x, acc_b[k][q].y, acc_b[k][q + 1].x, acc_b[k][q + 1].y);
            }
        }
    }
}

// ------------------------------------------------------------------ row kernel (bulk-copy ring)
// A ring stage holds a group of R consecutive rows: [R rows of x | R rows of dY].
// Columns per thread NV*E up to 16 fit two CTAs per SM; 32 need the full budget.
// kRms: RMSNorm backward -- no mean subtraction (mean is not read), no sum of
// dxhat, no beta: dX = rs*(dxhat - xhat*mean(dxhat*xhat)), partial rows of D.
// W: warps the CTA may have -- 8, or 16 for the wide variant (up to 512 threads,
// 16 columns a thread: rows of 4097..8192 16-bit columns, which would otherwise
// need 32 columns a thread and leave one 8-warp CTA per SM).  kBound < W*32: an
// instance for CTAs of at most kBound threads, two per SM (the register budget
// that leaves): the wide variant on rows of up to 640 vectors; otherwise a wide
// CTA has its SM to itself.
template <class Fmt, int NV, int R, bool kRms, int W = kMaxWarps, int kBound = W * 32>
__global__ void __launch_bounds__(kBound, (kBound < W * 32) ? 2
                                          : (W > kMaxWarps || NV * Vec<Fmt>::kElems >= 32) ? 1 : 2)
ln_bwd_rows_ring_kernel(const typename Fmt::T* __restrict__ dY, const typename Fmt::T* __restrict__ x,
                        const float* __restrict__ mean, const float* __restrict__ inv_std,
                        const float* __restrict__ gamma, typename Fmt::T* __restrict__ dX,
                        float* __restrict__ partials, int64_t rows, int D, int stages,
                        int64_t rows_per_cta, int* err, unsigned long long wait_limit_ns,
                        int withhold_copies) {
    using T = typename Fmt::T;
    constexpr int E = Vec<Fmt>::kElems;
    // x - mean by mixed-precision subtraction: fp16 rows, and bf16 rows on the
    // 16-warp instance that has its SM to itself (on the 8-warp bf16 instances it
    // measured up to 1% slower, on the two-per-SM wide instance 3% slower)
    constexpr bool kMix = !kRms && (std::is_same<Fmt, F16>::value ||
                                    (std::is_same<Fmt, BF16>::value && W > kMaxWarps &&
                                     kBound == W * 32));
    extern __shared__ __align__(128) unsigned char smem[];
    // Per-warp row sums: value 2i is sum(dxhat) of row i, 2i+1 is sum(dxhat*xhat).
    // Slots of warps the CTA does not have stay zero.
    __shared__ __align__(16) float red[2][2 * R][W];

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nthreads = blockDim.x;
    const int nvec = D / E;
    const uint32_t row_bytes = (uint32_t)D * (uint32_t)sizeof(T);
    const uint32_t grp_bytes = (uint32_t)R * row_bytes;
    for (int i = tid; i < 2 * 2 * R * W; i += nthreads) (&red[0][0][0])[i] = 0.f;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    unsigned char* ring = smem + kBarRegion;   // stage s at ring + s * 2 * grp_bytes

    const int64_t r0 = (int64_t)blockIdx.x * rows_per_cta;
    const int64_t r1 = r0 + rows_per_cta < rows ? r0 + rows_per_cta : rows;
    const int64_t nrows = r1 > r0 ? r1 - r0 : 0;
    const int64_t ngroups = (nrows + R - 1) / R;

    uint64_t pol = 0;
    int64_t issued = 0;   // groups issued so far (thread 0 only)
    auto issue = [&](int64_t grp, int s) {
        const int64_t first = r0 + grp * R;
        const int64_t nr = nrows - grp * R < R ? nrows - grp * R : R;
        const uint32_t bytes = (uint32_t)nr * row_bytes;
        const uint32_t bar = smem_addr(&bars[s]);
        unsigned char* st = ring + (size_t)s * 2 * grp_bytes;
        mbar_arrive_expect_tx(bar, 2 * bytes);
        if (withhold_copies) return;   // self-test: the stage's barrier never completes
        bulk_g2s(smem_addr(st), x + first * D, bytes, bar, pol);
        bulk_g2s(smem_addr(st + grp_bytes), dY + first * D, bytes, bar, pol);
    };
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(smem_addr(&bars[s]), 1);
        mbar_init_fence();
        pol = evict_first_policy();
        // Start pulling the first stage's rows from HBM into L2 while the previous
        // kernel may still be draining.  A prefetch returns nothing to the kernel and
        // L2 is coherent, so the copies issued after the wait still see every write of
        // the previous kernel; the prefetch only shortens their trip.
        if (ngroups > 0 && !withhold_copies) {
            const uint32_t b0 = (uint32_t)(nrows < R ? nrows : R) * row_bytes;
            bulk_prefetch_l2(x + r0 * D, b0);
            bulk_prefetch_l2(dY + r0 * D, b0);
        }
    }
    // Up to here the kernel has touched only shared memory (and issued the L2
    // prefetch): the previous kernel may still be running (programmatic launch).
    // Every load and store of global memory comes after this wait.
    pdl_wait();
    if (tid == 0)
        for (; issued < ngroups && issued < stages; ++issued) issue(issued, (int)issued);

    constexpr int NP = Pairs<Fmt>::kN;
    float2 g[NV][NP], acc_g[NV][NP], acc_b[NV][NP];
    load_gamma<Fmt, NV>(gamma, g, acc_g, acc_b, tid, nthreads, nvec);
    float mu[R], rs[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        mu[i] = (!kRms && i < nrows) ? mean[r0 + i] : 0.f;
        rs[i] = i < nrows ? inv_std[r0 + i] : 0.f;
    }
    __syncthreads();   // barriers initialised before anyone waits on them

    const float inv_D = 1.0f / (float)D;
    int64_t fail_at = -1;
    // Stage and phase parity of the current group.  The 16-warp instantiation
    // advances them by counting: a 64-bit division by the run-time stage count in
    // each of its one-row groups cost it 14% at D = 8192.  The 8-warp ones divide:
    // counting measured 2% slower on their LayerNorm instances.
    constexpr bool kCount = W > kMaxWarps;
    int s_next = 0, s_prev = stages - 1;
    uint32_t parity_next = 0;
    for (int64_t grp = 0; grp < ngroups; ++grp) {
        const int s = kCount ? s_next : (int)(grp % stages);
        const uint32_t parity = kCount ? parity_next : (uint32_t)((grp / stages) & 1);
        const int64_t first = r0 + grp * R;
        const int nr = (int)(nrows - grp * R < R ? nrows - grp * R : R);
        // Prefetch the next group's statistics while this one is processed.
        float mu_n[R], rs_n[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int64_t rn = first + R + i;
            const bool has = rn < r1;
            mu_n[i] = (!kRms && has) ? mean[rn] : 0.f;
            rs_n[i] = has ? inv_std[rn] : 0.f;
        }
        const bool ok = mbar_wait_bounded(smem_addr(&bars[s]), parity, wait_limit_ns);
        const unsigned char* st = ring + (size_t)s * 2 * grp_bytes;

        // Phase 1: the two sums of every row of the group, from the staged rows.
        float sa[R], sb[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            sa[i] = 0.f;
            sb[i] = 0.f;
            if (ok && i < nr)
                row_shares<Fmt, NV, kRms, kMix>(st + (size_t)i * row_bytes,
                                          st + grp_bytes + (size_t)i * row_bytes, g, mu[i], rs[i],
                                          tid, nthreads, nvec, sa[i], sb[i]);
        }
        float sums[2 * R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            sums[2 * i] = sa[i];
            sums[2 * i + 1] = sb[i];
        }
        const float wsum = warp_sum_multi<2 * R>(sums, lane);
        const int buf = (int)(grp & 1);
        if (multi_writer<2 * R>(lane)) red[buf][multi_index<2 * R>(lane)][wid] = wsum;
        // Past this barrier every thread has finished the previous group entirely,
        // so its stage can be refilled; this group's stage is still read below.
        if (__syncthreads_or(!ok)) {
            fail_at = grp;
            break;
        }
        if (tid == 0 && grp >= 1 && issued < ngroups) {
            fence_proxy_async_smem();
            issue(issued, kCount ? s_prev : (int)((grp - 1) % stages));
            ++issued;
        }

        // Phase 2: dX and the column partials, re-reading the staged rows.
#pragma unroll
        for (int i = 0; i < R; ++i) {
            if (i < nr) {
                const float a = cta_total<W>(&red[buf][2 * i][0]);
                const float b = cta_total<W>(&red[buf][2 * i + 1][0]);
                const float mean_a = kRms ? 0.f : a * inv_D, mean_b = b * inv_D;
                row_dx<Fmt, NV, kRms, kMix>(st + (size_t)i * row_bytes,
                                      st + grp_bytes + (size_t)i * row_bytes, dX + (first + i) * D,
                                      g, acc_g, acc_b, mu[i], rs[i], mean_a, mean_b, tid, nthreads,
                                      nvec);
            }
        }
#pragma unroll
        for (int i = 0; i < R; ++i) {
            mu[i] = mu_n[i];
            rs[i] = rs_n[i];
        }
        if constexpr (kCount) {
            s_prev = s_next;
            if (++s_next == stages) {
                s_next = 0;
                parity_next ^= 1u;
            }
        }
    }

    if (fail_at >= 0) {
        // Groups [fail_at, issued) still have copies in flight (at most one per
        // stage): wait for them, bounded, before the CTA's shared memory is freed.
        if (tid == 0) {
            atomicExch(err, (int)TB_ERR_TIMEOUT);
            for (int64_t q = fail_at; q < issued; ++q)
                mbar_wait_bounded(smem_addr(&bars[q % stages]), (uint32_t)((q / stages) & 1),
                                  wait_limit_ns);
        }
        __syncthreads();
        return;
    }
    // Let the column reduction launch; it waits for this grid to finish before reading.
    pdl_trigger();

    float* pg = partials + (size_t)blockIdx.x * (kRms ? 1 : 2) * D;
    store_partials<Fmt, NV, kRms>(pg, pg + D, acc_g, acc_b, tid, nthreads, nvec);
}

// ------------------------------------------------------------------ row kernel (split over a cluster)
// Rows wider than one CTA's register budget are split by columns over the C
// CTAs of a thread-block cluster (2 <= C <= 8).  CTA k of a cluster owns the
// column slice [k*D/C, (k+1)*D/C): for every row of the cluster's row block it
// streams that slice of x and dY into its own ring (one bulk copy per row and
// tensor), keeps gamma and the column partials of the slice in registers, and
// forms the slice's share of the two row sums.  The shares travel through
// distributed shared memory: each CTA stores its 2R sums and a failure flag
// into the exchange slot of every other CTA with st.async, counted as
// transaction bytes on that CTA's exchange mbarrier (two slots, alternating by
// group).  Every CTA adds the C shares in rank order, so all of them use
// bitwise the same row sums.  A cluster owns one partial row of the workspace;
// its CTAs fill disjoint column ranges of it.
//
// Only the 2R+1 exchanging threads wait for the peers; the rest of the CTA meets
// them at the barrier that publishes the row sums (through shared memory).
// Slot reuse is safe without further handshakes: a CTA sends group g+2 into a
// slot only after it has received every share of group g+1, and each CTA sends
// its share of g+1 only after its threads have read the slot's group-g shares
// and after it has armed the slot's barrier for g+2 (expected bytes), so a
// phase is always armed before any peer's bytes for it arrive.
//
// The kernel is launched without the programmatic-dependent attribute: launched
// early, while the previous kernel still held SMs, clusters of three or more CTAs
// were placed so that part of the grid ran as a second wave (twice the time).
// A CTA whose ring wait gives up still sends its shares (with the flag set), so
// the whole cluster leaves the loop at the same group; every CTA then waits
// (bounded) for its own copies in flight, and the cluster synchronises once more
// before any CTA exits, so no CTA's shared memory goes away while a peer may
// still store into it.
template <class Fmt, int NV, int R, bool kRms>
__global__ void __launch_bounds__(kRowThreads, (NV * Vec<Fmt>::kElems >= 32) ? 1 : 2)
ln_bwd_rows_split_kernel(const typename Fmt::T* __restrict__ dY, const typename Fmt::T* __restrict__ x,
                         const float* __restrict__ mean, const float* __restrict__ inv_std,
                         const float* __restrict__ gamma, typename Fmt::T* __restrict__ dX,
                         float* __restrict__ partials, int64_t rows, int D, int stages,
                         int64_t rows_per_cluster, int* err, unsigned long long wait_limit_ns,
                         int withhold_copies) {
    using T = typename Fmt::T;
    constexpr int E = Vec<Fmt>::kElems;
    constexpr int kWords = 2 * R + 1;   // shares: 2R row sums, then the failure flag
    constexpr bool kMix = !kRms && sizeof(T) == 2;   // x - mean by mixed-precision subtraction
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(16) float red[2][2 * R][kMaxWarps];
    __shared__ float xs[2][kMaxCluster][kWords];
    __shared__ float rsum[2 * R];   // the group's row sums, published for phase 2

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nthreads = blockDim.x;
    const uint32_t rank = cluster_ctarank(), csize = cluster_nctarank();
    // Launched with 2..kMaxCluster CTAs per cluster only (with one, a CTA could
    // complete an exchange phase on its own ahead of its slower threads).
    if (csize < 2 || csize > (uint32_t)kMaxCluster) {   // uniform over the grid
        if (tid == 0) atomicExch(err, (int)TB_ERR_INVALID_VALUE);
        return;
    }
    const int Dc = D / (int)csize;
    const int col0 = (int)rank * Dc;
    const int nvec = Dc / E;
    const uint32_t slice_bytes = (uint32_t)Dc * (uint32_t)sizeof(T);
    const uint32_t half_bytes = (uint32_t)R * slice_bytes;   // x part of a stage; dY follows
    for (int i = tid; i < 2 * 2 * R * kMaxWarps; i += nthreads) (&red[0][0][0])[i] = 0.f;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);   // ring stages
    uint64_t* xbar = bars + kMaxStages;                   // exchange slots 0 and 1
    unsigned char* ring = smem + kBarRegion;              // stage s at ring + s * 2 * half_bytes

    const int64_t r0 = (int64_t)cluster_index() * rows_per_cluster;
    const int64_t r1 = r0 + rows_per_cluster < rows ? r0 + rows_per_cluster : rows;
    const int64_t nrows = r1 > r0 ? r1 - r0 : 0;
    const int64_t ngroups = (nrows + R - 1) / R;

    uint64_t pol = 0;
    int64_t issued = 0;   // groups issued so far (thread 0 only)
    auto issue = [&](int64_t grp, int s) {
        const int64_t first = r0 + grp * R;
        const int nr = (int)(nrows - grp * R < R ? nrows - grp * R : R);
        const uint32_t bar = smem_addr(&bars[s]);
        unsigned char* st = ring + (size_t)s * 2 * half_bytes;
        mbar_arrive_expect_tx(bar, 2u * (uint32_t)nr * slice_bytes);
        if (withhold_copies) return;   // self-test: the stage's barrier never completes
        for (int i = 0; i < nr; ++i) {
            const int64_t off = (first + i) * D + col0;
            bulk_g2s(smem_addr(st + (size_t)i * slice_bytes), x + off, slice_bytes, bar, pol);
            bulk_g2s(smem_addr(st + half_bytes + (size_t)i * slice_bytes), dY + off, slice_bytes,
                     bar, pol);
        }
    };
    const uint32_t xs_bytes = (csize - 1) * (uint32_t)kWords * 4u;   // a slot phase's bytes
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(smem_addr(&bars[s]), 1);
        mbar_init(smem_addr(&xbar[0]), 1);
        mbar_init(smem_addr(&xbar[1]), 1);
        // groups 0 and 1 armed now; group g+2 once group g's phase has completed
        mbar_arrive_expect_tx(smem_addr(&xbar[0]), xs_bytes);
        mbar_arrive_expect_tx(smem_addr(&xbar[1]), xs_bytes);
        mbar_init_fence();
        pol = evict_first_policy();
        if (ngroups > 0 && !withhold_copies) {
            const int nr0 = (int)(nrows < R ? nrows : R);
            for (int i = 0; i < nr0; ++i) {
                bulk_prefetch_l2(x + (r0 + i) * D + col0, slice_bytes);
                bulk_prefetch_l2(dY + (r0 + i) * D + col0, slice_bytes);
            }
        }
    }
    // Every CTA's barriers are initialised (and `red` zeroed) before any peer
    // stores into them.  Only shared memory has been touched so far.
    cluster_sync_all();
    pdl_wait();
    if (tid == 0)
        for (; issued < ngroups && issued < stages; ++issued) issue(issued, (int)issued);

    constexpr int NP = Pairs<Fmt>::kN;
    float2 g[NV][NP], acc_g[NV][NP], acc_b[NV][NP];
    load_gamma<Fmt, NV>(gamma + col0, g, acc_g, acc_b, tid, nthreads, nvec);
    float mu[R], rs[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        mu[i] = (!kRms && i < nrows) ? mean[r0 + i] : 0.f;
        rs[i] = i < nrows ? inv_std[r0 + i] : 0.f;
    }

    const float inv_D = 1.0f / (float)D;
    int64_t fail_at = -1;
    // Stage of this group and of the previous one, and the phase parity: advanced
    // by counting (a 64-bit division by the run-time stage count costs dozens of
    // instructions per group).
    int s = 0, prev_s = stages - 1;
    uint32_t parity = 0;
    for (int64_t grp = 0; grp < ngroups; ++grp) {
        const int64_t first = r0 + grp * R;
        const int nr = (int)(nrows - grp * R < R ? nrows - grp * R : R);
        float mu_n[R], rs_n[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int64_t rn = first + R + i;
            const bool has = rn < r1;
            mu_n[i] = (!kRms && has) ? mean[rn] : 0.f;
            rs_n[i] = has ? inv_std[rn] : 0.f;
        }
        const bool ok = mbar_wait_bounded(smem_addr(&bars[s]), parity, wait_limit_ns);
        const unsigned char* st = ring + (size_t)s * 2 * half_bytes;

        // Phase 1: this CTA's shares of the row sums of the group.
        float sums[2 * R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            sums[2 * i] = 0.f;
            sums[2 * i + 1] = 0.f;
            if (ok && i < nr)
                row_shares<Fmt, NV, kRms, kMix>(st + (size_t)i * slice_bytes,
                                          st + half_bytes + (size_t)i * slice_bytes, g, mu[i],
                                          rs[i], tid, nthreads, nvec, sums[2 * i], sums[2 * i + 1]);
        }
        const float wsum = warp_sum_multi<2 * R>(sums, lane);
        const int buf = (int)(grp & 1);
        if (multi_writer<2 * R>(lane)) red[buf][multi_index<2 * R>(lane)][wid] = wsum;
        // Past this barrier every thread has finished the previous group entirely.
        const bool failed_here = __syncthreads_or(!ok);
        if (tid == 0 && !failed_here && grp >= 1 && issued < ngroups) {
            fence_proxy_async_smem();
            issue(issued, prev_s);
            ++issued;
        }
        // Thread j < 2R owns row sum j, thread 2R the failure flag: it sends this
        // CTA's share to every other CTA of the cluster, waits for theirs, and adds
        // the C shares in rank order (the flags add up to the number of failed CTAs).
        bool xok = true, flagged = false;
        if (tid < kWords) {
            const uint32_t xbar_local = smem_addr(&xbar[buf]);
            const float own = tid < 2 * R ? cta_total(&red[buf][tid][0]) : (failed_here ? 1.f : 0.f);
            const uint32_t slot = smem_addr(&xs[buf][rank][tid]);
            for (uint32_t p = 0; p < csize; ++p)
                if (p != rank) st_async_remote(map_to_rank(slot, p), own, map_to_rank(xbar_local, p));
            xok = mbar_wait_cluster_bounded(xbar_local, (uint32_t)((grp >> 1) & 1), wait_limit_ns);
            if (tid == 0 && xok && grp + 2 < ngroups) mbar_arrive_expect_tx(xbar_local, xs_bytes);
            float t = 0.f;
            for (uint32_t c = 0; c < csize; ++c) t += c == rank ? own : xs[buf][c][tid];
            if (tid < 2 * R) rsum[tid] = t;
            else flagged = t != 0.f;
        }
        // One decision for the whole CTA; past it the row sums are visible to all.
        if (__syncthreads_or(!xok || flagged)) {
            fail_at = grp;
            break;
        }

        // Phase 2: dX and the column partials of this CTA's slice.
#pragma unroll
        for (int i = 0; i < R; ++i) {
            if (i < nr) {
                const float mean_a = kRms ? 0.f : rsum[2 * i] * inv_D, mean_b = rsum[2 * i + 1] * inv_D;
                row_dx<Fmt, NV, kRms, kMix>(st + (size_t)i * slice_bytes,
                                      st + half_bytes + (size_t)i * slice_bytes,
                                      dX + (first + i) * D + col0, g, acc_g, acc_b, mu[i], rs[i],
                                      mean_a, mean_b, tid, nthreads, nvec);
            }
        }
#pragma unroll
        for (int i = 0; i < R; ++i) {
            mu[i] = mu_n[i];
            rs[i] = rs_n[i];
        }
        prev_s = s;
        if (++s == stages) {
            s = 0;
            parity ^= 1u;
        }
    }

    if (fail_at >= 0) {
        if (tid == 0) {
            atomicExch(err, (int)TB_ERR_TIMEOUT);
            for (int64_t q = fail_at; q < issued; ++q)
                mbar_wait_bounded(smem_addr(&bars[q % stages]), (uint32_t)((q / stages) & 1),
                                  wait_limit_ns);
        }
        __syncthreads();
        cluster_sync_all();
        return;
    }
    pdl_trigger();
    float* pg = partials + (size_t)cluster_index() * (kRms ? 1 : 2) * D + col0;
    store_partials<Fmt, NV, kRms>(pg, pg + D, acc_g, acc_b, tid, nthreads, nvec);
    cluster_sync_all();
}

// ------------------------------------------------------------------ row kernel (registers, plain loads)
// Rows the bulk-copy rings cannot take -- unaligned buffers, or rows whose byte
// length is not a multiple of 16 -- of up to K*256 columns.  Thread t of T owns
// the columns t, t+T, ..., t+(K-1)T: it keeps gamma and its dgamma/dbeta partial
// sums for them in registers across all rows of the CTA.  One thread prefetches
// the rows ahead into L2 in blocks of about 16 KB (bulk prefetches of the
// 16-byte-aligned span covering them: rounding an address inside a row down or
// up to 16 bytes stays in the same 16-byte block, so in mapped memory), so each
// row's loads find their lines in L2.  Up to 8 columns a
// thread it also holds a row's x and dY values in registers between the two
// phases; with more, phase 2 reads the row again (it was just read, so from L1),
// which keeps the registers of 16 and 32 columns a thread low enough for two or
// three CTAs per SM.  Element loads and stores are scalar but coalesced (a warp
// touches consecutive elements).  One block reduction (double-buffered by row
// parity) per row.
template <class Fmt, int K, bool kRms>
__global__ void __launch_bounds__(kRowThreads, K > 8 ? 2 : 1)
ln_bwd_rows_reg_kernel(const typename Fmt::T* __restrict__ dY, const typename Fmt::T* __restrict__ x,
                       const float* __restrict__ mean, const float* __restrict__ inv_std,
                       const float* __restrict__ gamma, typename Fmt::T* __restrict__ dX,
                       float* __restrict__ partials, int64_t rows, int D, int64_t rows_per_cta) {
    __shared__ float red[2][2][kMaxWarps];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nthreads = blockDim.x, nwarps = nthreads >> 5;
    pdl_wait();   // the previous kernel has completed (programmatic launch)
    float g[K], acc_g[K], acc_b[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int j = tid + k * nthreads;
        g[k] = j < D ? gamma[j] : 0.f;
        acc_g[k] = 0.f;
        acc_b[k] = 0.f;
    }
    const int64_t r0 = (int64_t)blockIdx.x * rows_per_cta;
    const int64_t r1 = r0 + rows_per_cta < rows ? r0 + rows_per_cta : rows;
    const float inv_D = 1.0f / (float)D;
    constexpr bool kHold = K <= 8;   // keep the row in registers between the phases
    // Rows per prefetch block: about 16 KB of each tensor.
    const int64_t row_bytes = (int64_t)D * (int64_t)sizeof(typename Fmt::T);
    const int64_t pf_rows = row_bytes >= 16384 ? 1 : 16384 / row_bytes;
    auto prefetch_rows = [&](int64_t a, int64_t b) {   // rows [a, b) of x and dY into L2
        if (b > r1) b = r1;
        if (a >= b) return;
        const uintptr_t lo_x = reinterpret_cast<uintptr_t>(x + a * D) & ~(uintptr_t)15;
        const uintptr_t hi_x = (reinterpret_cast<uintptr_t>(x + b * D) + 15) & ~(uintptr_t)15;
        const uintptr_t lo_d = reinterpret_cast<uintptr_t>(dY + a * D) & ~(uintptr_t)15;
        const uintptr_t hi_d = (reinterpret_cast<uintptr_t>(dY + b * D) + 15) & ~(uintptr_t)15;
        bulk_prefetch_l2(reinterpret_cast<const void*>(lo_x), (uint32_t)(hi_x - lo_x));
        bulk_prefetch_l2(reinterpret_cast<const void*>(lo_d), (uint32_t)(hi_d - lo_d));
    };
    if (tid == 0) {   // the first two blocks
        prefetch_rows(r0, r0 + pf_rows);
        prefetch_rows(r0 + pf_rows, r0 + 2 * pf_rows);
    }
    int buf = 0;
    for (int64_t r = r0; r < r1; ++r, buf ^= 1) {
        // entering a block: fetch the block after next
        if (tid == 0 && (r - r0) % pf_rows == 0) prefetch_rows(r + 2 * pf_rows, r + 3 * pf_rows);
        const float mu = kRms ? 0.f : mean[r], rs = inv_std[r];
        const typename Fmt::T* xr = x + r * D;
        const typename Fmt::T* dyr = dY + r * D;
        float xv[kHold ? K : 1], dv[kHold ? K : 1];
        float sa = 0.f, sb = 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int j = tid + k * nthreads;
            const float xk = j < D ? Fmt::to_f32(xr[j]) : 0.f;
            const float dk = j < D ? Fmt::to_f32(dyr[j]) : 0.f;
            if constexpr (kHold) {
                xv[k] = xk;
                dv[k] = dk;
            }
            const float xh = (xk - mu) * rs;
            const float dxh = __fmul_rn(dk, g[k]);
            sa += dxh;
            sb = fmaf(dxh, xh, sb);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sa += __shfl_xor_sync(0xffffffffu, sa, o);
            sb += __shfl_xor_sync(0xffffffffu, sb, o);
        }
        if (lane == 0) {
            red[buf][0][wid] = sa;
            red[buf][1][wid] = sb;
        }
        __syncthreads();
        float a = 0.f, b = 0.f;
        for (int w = 0; w < nwarps; ++w) {
            a += red[buf][0][w];
            b += red[buf][1][w];
        }
        const float mean_a = kRms ? 0.f : a * inv_D, mean_b = b * inv_D;
        const float c0 = -(rs * mean_a), c1 = -(rs * mean_b);
        typename Fmt::T* dxr = dX + r * D;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int j = tid + k * nthreads;
            if (j < D) {
                float xk, dk;
                if constexpr (kHold) {
                    xk = xv[k];
                    dk = dv[k];
                } else {
                    // a load of its own (last use), not merged with phase 1's
                    xk = Fmt::to_f32(__ldlu(xr + j));
                    dk = Fmt::to_f32(__ldlu(dyr + j));
                }
                const float xh = (xk - mu) * rs;
                const float dxh = __fmul_rn(dk, g[k]);
                dxr[j] = Fmt::from_f32(fmaf(dxh, rs, fmaf(xh, c1, c0)));
                acc_g[k] = fmaf(dk, xh, acc_g[k]);
                if (!kRms) acc_b[k] += dk;
            }
        }
    }
    pdl_trigger();
    float* pg = partials + (size_t)blockIdx.x * (kRms ? 1 : 2) * D;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int j = tid + k * nthreads;
        if (j < D) {
            pg[j] = acc_g[k];
            if (!kRms) pg[D + j] = acc_b[k];
        }
    }
}

// ------------------------------------------------------------------ row kernel (plain loads)
// The last resort: unaligned rows longer than 8192 columns.  Two global passes
// per row, partials kept in the workspace.
template <class Fmt, bool kRms>
__global__ void __launch_bounds__(kRowThreads)
ln_bwd_rows_plain_kernel(const typename Fmt::T* __restrict__ dY, const typename Fmt::T* __restrict__ x,
                         const float* __restrict__ mean, const float* __restrict__ inv_std,
                         const float* __restrict__ gamma, typename Fmt::T* __restrict__ dX,
                         float* __restrict__ partials, int64_t rows, int64_t D, int64_t rows_per_cta) {
    __shared__ float red[2][2][kMaxWarps];
    pdl_wait();   // the previous kernel has completed (programmatic launch)
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    float* pg = partials + (size_t)blockIdx.x * (kRms ? 1 : 2) * D;
    float* pb = pg + D;
    for (int64_t j = tid; j < D; j += blockDim.x) {
        pg[j] = 0.f;
        if (!kRms) pb[j] = 0.f;
    }
    const int64_t r0 = (int64_t)blockIdx.x * rows_per_cta;
    const int64_t r1 = r0 + rows_per_cta < rows ? r0 + rows_per_cta : rows;
    const float inv_D = 1.0f / (float)D;
    int buf = 0;
    for (int64_t r = r0; r < r1; ++r, buf ^= 1) {
        const float mu = kRms ? 0.f : mean[r], rs = inv_std[r];
        const int64_t off = r * D;
        float sa = 0.f, sb = 0.f;
        for (int64_t j = tid; j < D; j += blockDim.x) {
            const float xh = (Fmt::to_f32(x[off + j]) - mu) * rs;
            const float dxh = __fmul_rn(Fmt::to_f32(dY[off + j]), gamma[j]);
            sa += dxh;
            sb += dxh * xh;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sa += __shfl_xor_sync(0xffffffffu, sa, o);
            sb += __shfl_xor_sync(0xffffffffu, sb, o);
        }
        if (lane == 0) {
            red[buf][0][wid] = sa;
            red[buf][1][wid] = sb;
        }
        __syncthreads();
        float a = 0.f, b = 0.f;
        for (int w = 0; w < nwarps; ++w) {
            a += red[buf][0][w];
            b += red[buf][1][w];
        }
        const float mean_a = kRms ? 0.f : a * inv_D, mean_b = b * inv_D;
        for (int64_t j = tid; j < D; j += blockDim.x) {
            const float dyv = Fmt::to_f32(dY[off + j]);
            const float xh = (Fmt::to_f32(x[off + j]) - mu) * rs;
            const float dxh = __fmul_rn(dyv, gamma[j]);
            dX[off + j] = Fmt::from_f32(rs * (dxh - mean_a - xh * mean_b));
            pg[j] += dyv * xh;   // column j belongs to this thread only
            if (!kRms) pb[j] += dyv;
        }
    }
    pdl_trigger();
}

// ------------------------------------------------------------------ column reduction
// partials: [G][W] fp32 (W = 2D for LayerNorm: dgamma then dbeta partials; W = D
// for RMSNorm); out column c < D -> out_a (dgamma), else out_b (dbeta).
// A CTA covers 32 columns with 32 warps: warp w sums partial rows w, w+32, ... in
// ascending order, then the 32 warp sums are added in warp order.  Two CTAs fit
// per SM (32 registers), so the whole grid is resident at once.  The order never
// depends on timing, so the result is bitwise reproducible.
constexpr int kColThreads = 1024;
constexpr int kColGroups = kColThreads / 32;

__global__ void __launch_bounds__(kColThreads, 2)
ln_bwd_colsum_kernel(const float* __restrict__ partials, int G, int64_t W, int64_t D,
                     float* __restrict__ dgamma, float* __restrict__ dbeta) {
    __shared__ float sm[kColGroups][33];
    pdl_trigger();   // the next kernel may be placed now; it waits for this one to complete
    pdl_wait();      // the row kernel (if any) has completed and flushed its partials
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t c = (int64_t)blockIdx.x * 32 + lane;
    float acc = 0.f;
    if (c < W) {
        // ten loads in flight per round, added in ascending row order: one round
        // covers the 320 partial rows of two CTAs per SM on 160 SMs
        for (int b = w; b < G; b += 10 * kColGroups) {
            float v[10];
#pragma unroll
            for (int q = 0; q < 10; ++q) {
                const int bb = b + q * kColGroups;
                v[q] = bb < G ? partials[(int64_t)bb * W + c] : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 10; ++q) acc += v[q];
        }
    }
    sm[w][lane] = acc;
    __syncthreads();
    if (w == 0 && c < W) {
        float t = 0.f;
#pragma unroll
        for (int q = 0; q < kColGroups; ++q) t += sm[q][lane];
        if (c < D) dgamma[c] = t; else dbeta[c - D] = t;
    }
}

// Launch the column reduction so that it may be scheduled while the row kernel
// drains (programmatic dependent launch); it waits inside for the row kernel.
cudaError_t launch_colsum(const float* ws, int G, int64_t W, int64_t D, float* dgamma,
                          float* dbeta, cudaStream_t st) {
    return launch_pdl(ln_bwd_colsum_kernel, dim3((unsigned)((W + 31) / 32)), dim3(kColThreads), 0,
                      st, ws, G, W, D, dgamma, dbeta);
}

// ------------------------------------------------------------------ launch planning
enum class Path { kRing, kRingWide, kSplit, kPlain };

struct LnPlan {
    Path path;
    int threads;
    int nv;          // vectors per thread (ring and split paths)
    int r;           // rows per ring stage (ring and split paths)
    int stages;      // ring stages
    size_t smem;     // dynamic shared memory (ring and split paths)
    int cluster = 1; // CTAs a row is split over (split path), else 1
    bool pair = false;  // wide ring path: the two-CTAs-per-SM instance
    int grid;        // CTAs of the row kernel
    int parts;       // partial rows in the workspace: grid / cluster
    int64_t rows_per_cta;   // rows per CTA (per cluster on the split path)
    unsigned long long wait_limit_ns = kWaitLimitNs;   // bound of every wait (ring path)
    int withhold_copies = 0;   // self-test only: issue no copies, so every wait runs out
};

// Largest NV instantiated: kMaxElemsPerThread columns per thread.
template <class Fmt>
constexpr int max_nv() { return kMaxElemsPerThread / Vec<Fmt>::kElems; }

// Rows per stage allowed for NV (registers: 2R sums, NV*E columns per thread).
inline int max_r_for(int nv) { return nv == 1 ? 8 : nv == 2 ? 2 : 1; }

// Op<Fmt, NV, R>::run(args...) for the instantiated (nv, r) pair.
template <class Fmt, template <class, int, int> class Op, class... Args>
auto with_ring_variant(int nv, int r, Args&&... args) {
    if (nv == 1) {
        if (r >= 8) return Op<Fmt, 1, 8>::run(args...);
        if (r >= 4) return Op<Fmt, 1, 4>::run(args...);
        if (r >= 2) return Op<Fmt, 1, 2>::run(args...);
        return Op<Fmt, 1, 1>::run(args...);
    }
    if (nv == 2) {
        if (r >= 2) return Op<Fmt, 2, 2>::run(args...);
        return Op<Fmt, 2, 1>::run(args...);
    }
    if (nv == 4) return Op<Fmt, 4, 1>::run(args...);
    return Op<Fmt, max_nv<Fmt>(), 1>::run(args...);
}

template <bool kRms>
struct RingOps {
    template <class Fmt, int NV, int R>
    struct Ptr {
        static const void* run() {
            return reinterpret_cast<const void*>(&ln_bwd_rows_ring_kernel<Fmt, NV, R, kRms>);
        }
    };
};

// The wide variant: 16-bit rows of 513..1024 vectors, two vectors a thread, one row a stage;
// `pair`: the instance bounded to kWidePairThreads threads, two CTAs per SM.
template <class Fmt>
const void* wide_kernel_for(bool rms, bool pair) {
    if (pair)
        return rms ? reinterpret_cast<const void*>(
                         &ln_bwd_rows_ring_kernel<Fmt, 2, 1, true, kWideWarps, kWidePairThreads>)
                   : reinterpret_cast<const void*>(
                         &ln_bwd_rows_ring_kernel<Fmt, 2, 1, false, kWideWarps, kWidePairThreads>);
    return rms ? reinterpret_cast<const void*>(&ln_bwd_rows_ring_kernel<Fmt, 2, 1, true, kWideWarps>)
               : reinterpret_cast<const void*>(&ln_bwd_rows_ring_kernel<Fmt, 2, 1, false, kWideWarps>);
}

template <class Fmt>
const void* ring_kernel_for(int nv, int r, bool rms) {
    return rms ? with_ring_variant<Fmt, RingOps<true>::template Ptr>(nv, r)
               : with_ring_variant<Fmt, RingOps<false>::template Ptr>(nv, r);
}

const void* ring_kernel(tb_dtype dt, int nv, int r, bool rms) {
    switch (dt) {
        case TB_F32: return ring_kernel_for<F32>(nv, r, rms);
        case TB_BF16: return ring_kernel_for<BF16>(nv, r, rms);
        default: return ring_kernel_for<F16>(nv, r, rms);
    }
}

// Op<Fmt, NV, R>::run(args...) for the split kernel's instantiated (nv, r) pairs:
// 16 or 32 columns per thread.
template <class Fmt, template <class, int, int> class Op, class... Args>
auto with_split_variant(int nv, int r, Args&&... args) {
    constexpr int nv16 = 16 / Vec<Fmt>::kElems;
    if (nv <= nv16) {
        if (nv16 == 2 && r >= 2) return Op<Fmt, nv16, (nv16 == 2 ? 2 : 1)>::run(args...);
        return Op<Fmt, nv16, 1>::run(args...);
    }
    return Op<Fmt, 2 * nv16, 1>::run(args...);
}

template <bool kRms>
struct SplitOps {
    template <class Fmt, int NV, int R>
    struct Ptr {
        static const void* run() {
            return reinterpret_cast<const void*>(&ln_bwd_rows_split_kernel<Fmt, NV, R, kRms>);
        }
    };
};

template <class Fmt>
const void* split_kernel_for(int nv, int r, bool rms) {
    return rms ? with_split_variant<Fmt, SplitOps<true>::template Ptr>(nv, r)
               : with_split_variant<Fmt, SplitOps<false>::template Ptr>(nv, r);
}

const void* split_kernel(tb_dtype dt, int nv, int r, bool rms) {
    switch (dt) {
        case TB_F32: return split_kernel_for<F32>(nv, r, rms);
        case TB_BF16: return split_kernel_for<BF16>(nv, r, rms);
        default: return split_kernel_for<F16>(nv, r, rms);
    }
}

// Op<Fmt, K>::run(args...) for the register row kernel's instantiated K.
template <class Fmt, template <class, int> class Op, class... Args>
auto with_reg_variant(int k, Args&&... args) {
    switch (k) {
        case 1: return Op<Fmt, 1>::run(args...);
        case 2: return Op<Fmt, 2>::run(args...);
        case 4: return Op<Fmt, 4>::run(args...);
        case 8: return Op<Fmt, 8>::run(args...);
        case 16: return Op<Fmt, 16>::run(args...);
        default: return Op<Fmt, 32>::run(args...);
    }
}

template <bool kRms>
struct RegOps {
    template <class Fmt, int K>
    struct Ptr {
        static const void* run() {
            return reinterpret_cast<const void*>(&ln_bwd_rows_reg_kernel<Fmt, K, kRms>);
        }
    };
    template <class Fmt, int K>
    struct Launch {
        using T = typename Fmt::T;
        static int run(const LnPlan& p, const T* dy, const T* x, const float* mean,
                       const float* inv_std, const float* gamma, T* dx, float* ws, int64_t rows,
                       int D, cudaStream_t st) {
            launch_pdl(ln_bwd_rows_reg_kernel<Fmt, K, kRms>, dim3((unsigned)p.grid),
                       dim3((unsigned)p.threads), 0, st, dy, x, mean, inv_std, gamma, dx, ws, rows,
                       D, p.rows_per_cta);
            return 0;
        }
    };
};

template <class Fmt>
const void* reg_kernel_for(int k, bool rms) {
    return rms ? with_reg_variant<Fmt, RegOps<true>::template Ptr>(k)
               : with_reg_variant<Fmt, RegOps<false>::template Ptr>(k);
}

const void* reg_kernel(tb_dtype dt, int k, bool rms) {
    switch (dt) {
        case TB_F32: return reg_kernel_for<F32>(k, rms);
        case TB_BF16: return reg_kernel_for<BF16>(k, rms);
        default: return reg_kernel_for<F16>(k, rms);
    }
}

template <class Fmt>
const void* plain_kernel_for(bool rms) {
    return rms ? reinterpret_cast<const void*>(&ln_bwd_rows_plain_kernel<Fmt, true>)
               : reinterpret_cast<const void*>(&ln_bwd_rows_plain_kernel<Fmt, false>);
}

const void* plain_kernel(tb_dtype dt, bool rms) {
    switch (dt) {
        case TB_F32: return plain_kernel_for<F32>(rms);
        case TB_BF16: return plain_kernel_for<BF16>(rms);
        default: return plain_kernel_for<F16>(rms);
    }
}

// Cluster size for splitting rows of D columns: the smallest C in [2, 8] that
// cuts a row into slices of whole 16-byte vectors of at most `target` columns
// (0 if there is none).
int split_cluster_size(int64_t D, int64_t E, int64_t target) {
    for (int64_t c = std::max<int64_t>(2, (D + target - 1) / target); c <= kMaxCluster; ++c)
        if (D % (c * E) == 0) return (int)c;
    return 0;
}

// Split path (rows longer than kSplitFromRowBytes): C CTAs per row, each with
// 16 columns per thread when the slice allows it, else 32.  (Up to 16 KB rows --
// 8192 16-bit or 4096 fp32 columns -- the single-CTA ring measured faster.)
bool make_split_plan(int64_t rows, int64_t D, tb_dtype dt, LnPlan* p, bool rms) {
    const int64_t es = (int64_t)dtype_size(dt);
    const int64_t E = 16 / es;
    int c = split_cluster_size(D, E, kSplitSliceTarget);
    if (c == 0) c = split_cluster_size(D, E, (int64_t)kMaxElemsPerThread * kRowThreads);
    if (c == 0) return false;
    const int64_t Dc = D / c;
    const int64_t nvec = Dc / E;
    const int nv = (int)((Dc <= (int64_t)16 * kRowThreads ? 16 : 32) / E);
    const int64_t need_threads = (nvec + nv - 1) / nv;   // nv vectors each, before rounding to warps
    const int threads = (int)std::min<int64_t>(kRowThreads, (need_threads + 31) / 32 * 32);
    const int64_t slice_bytes = Dc * es;
    // ring bytes in proportion to the CTA's warps, as on the ring path
    const int64_t budget = (int64_t)kRingBudget * (threads / 32) / kMaxWarps;
    const int64_t stage_target = std::min<int64_t>(kStageTargetBytes, budget / 3);
    int r = 1;
    while (r < max_r_for(nv) && (int64_t)(2 * r) * slice_bytes <= stage_target / 2) r *= 2;
    const int64_t stage_bytes = 2 * (int64_t)r * slice_bytes;
    const int stages =
        (int)std::min<int64_t>(kMaxStages, std::max<int64_t>(2, budget / stage_bytes));
    const size_t smem = kBarRegion + (size_t)stages * (size_t)stage_bytes;
    const int clusters = resident_clusters(split_kernel(dt, nv, r, rms), threads, smem, c);
    if (clusters == 0) return false;
    p->path = Path::kSplit;
    p->threads = threads;
    p->nv = nv;
    p->r = r;
    p->stages = stages;
    p->smem = smem;
    p->cluster = c;
    p->parts = (int)std::min<int64_t>(clusters, rows);
    p->grid = p->parts * c;
    p->rows_per_cta = (rows + p->parts - 1) / p->parts;
    return true;
}

// `aligned`: every row buffer 16-byte aligned (the caller checks pointers).
bool make_plan(int64_t rows, int64_t D, tb_dtype dt, bool aligned, const DeviceInfo& info,
               LnPlan* p, bool rms = false) {
    const int64_t es = (int64_t)dtype_size(dt);
    const int64_t E = 16 / es;
    const int64_t row_bytes = D * es;
    const int64_t nvec = D / E;
    p->path = Path::kPlain;
    p->cluster = 1;
    if (aligned && row_bytes % 16 == 0 && row_bytes > kSplitFromRowBytes && rows > 0 &&
        make_split_plan(rows, D, dt, p, rms))
        return true;
    // Wide ring: 16-bit rows of 513..1024 vectors, two a thread on up to 512 threads.
    if (aligned && row_bytes % 16 == 0 && es == 2 && nvec > 2 * kRowThreads &&
        nvec <= 2 * 32 * kWideWarps && rows > 0) {
        const int threads = (int)((nvec + 1) / 2 + 31) / 32 * 32;
        const int64_t budget = (int64_t)kRingBudget * (threads / 32) / kMaxWarps;
        const int64_t stage_bytes = 2 * row_bytes;
        const int stages =
            (int)std::min<int64_t>(kMaxStages, std::max<int64_t>(2, budget / stage_bytes));
        const size_t smem = kBarRegion + (size_t)stages * (size_t)stage_bytes;
        auto kernel = [&](bool pair) {
            return dt == TB_BF16 ? wide_kernel_for<BF16>(rms, pair) : wide_kernel_for<F16>(rms, pair);
        };
        bool pair = false;
        int per_sm = 0;
        if ((int64_t)smem <= info.max_smem_optin) {
            if (threads <= kWidePairThreads) {
                per_sm = resident_ctas_per_sm(kernel(true), threads, smem);
                pair = per_sm >= 2;
            }
            if (!pair) per_sm = resident_ctas_per_sm(kernel(false), threads, smem);
        }
        if (per_sm > 0) {
            p->path = Path::kRingWide;
            p->pair = pair;
            p->threads = threads;
            p->nv = 2;
            p->r = 1;
            p->stages = stages;
            p->smem = smem;
            p->grid = (int)std::min<int64_t>((int64_t)info.sm_count * per_sm, rows);
            p->parts = p->grid;
            p->rows_per_cta = (rows + p->grid - 1) / p->grid;
            return true;
        }
    }
    // Ring path: at most kMaxElemsPerThread columns per thread (gamma and the two
    // partial sums live in registers), i.e. D <= 8192.
    if (aligned && row_bytes % 16 == 0 && D <= (int64_t)kMaxElemsPerThread * kRowThreads) {
        const int threads = (int)std::min<int64_t>(kRowThreads, (nvec + 31) / 32 * 32);
        int nv = (int)((nvec + threads - 1) / threads);
        nv = nv <= 1 ? 1 : nv <= 2 ? 2 : nv <= 4 ? 4 : 8;
        // Ring bytes in proportion to the CTA's warps, so that CTAs of short rows -- one
        // to seven warps -- fit more per SM: 12 KB a warp in three stages for 16-bit
        // LayerNorm rows, 24 KB for 16-bit RMSNorm rows (fewer, larger groups), 8 KB in
        // two stages for fp32 rows -- each the best measured of 8..24 KB a warp and 2..4
        // stages at D = 512..1024.  A stage holds at most 16 KB of x and as much dY; eight
        // warps get 96 KB in every case.
        const bool short_row = threads < kRowThreads;
        const int64_t per_warp = !short_row ? kRingBudget / kMaxWarps
                                 : es == 4 ? 8 * 1024 : rms ? 24 * 1024 : 12 * 1024;
        const int nst = short_row && es == 4 ? 2 : 3;
        const int64_t budget = std::min<int64_t>(kRingBudget, per_warp * (threads / 32));
        const int64_t stage_target = std::min<int64_t>(kStageTargetBytes, budget / nst);
        int r = 1;
        while (r < max_r_for(nv) && (int64_t)(2 * r) * row_bytes <= stage_target / 2) r *= 2;
        const int64_t stage_bytes = 2 * (int64_t)r * row_bytes;
        const int stages =
            (int)std::min<int64_t>(kMaxStages, std::max<int64_t>(2, budget / stage_bytes));
        const size_t smem = kBarRegion + (size_t)stages * (size_t)stage_bytes;
        if ((int64_t)smem <= info.max_smem_optin) {
            const int per_sm = resident_ctas_per_sm(ring_kernel(dt, nv, r, rms), threads, smem);
            if (per_sm == 0) return false;
            p->path = Path::kRing;
            p->threads = threads;
            p->nv = nv;
            p->r = r;
            p->stages = stages;
            p->smem = smem;
            p->grid = info.sm_count * per_sm;
        }
    }
    if (p->path == Path::kPlain) {
        // Register rows (nv = columns a thread) up to 32 columns a thread, else the
        // last-resort kernel (nv = 0).
        const int threads = (int)std::min<int64_t>(kRowThreads, (D + 31) / 32 * 32);
        const int64_t per_thread = (D + threads - 1) / threads;
        int k = 0;
        if (per_thread <= 32) k = per_thread <= 1 ? 1 : per_thread <= 2 ? 2 : per_thread <= 4 ? 4
                                 : per_thread <= 8 ? 8 : per_thread <= 16 ? 16 : 32;
        const int per_sm = resident_ctas_per_sm(k ? reg_kernel(dt, k, rms) : plain_kernel(dt, rms),
                                                k ? threads : kRowThreads, 0);
        if (per_sm == 0) return false;
        p->threads = k ? threads : kRowThreads;
        p->nv = k;
        p->r = 0;
        p->stages = 0;
        p->smem = 0;
        p->grid = info.sm_count * (k ? per_sm : std::min(per_sm, 2));
    }
    p->grid = (int)std::min<int64_t>(p->grid, rows);
    p->parts = p->grid;
    p->rows_per_cta = p->grid > 0 ? (rows + p->grid - 1) / p->grid : 0;
    return true;
}

size_t workspace_bytes_for(const LnPlan& p, int64_t D, bool rms = false) {
    return (size_t)p.parts * (rms ? 1 : 2) * (size_t)D * sizeof(float);
}

template <bool kRms>
struct RingLaunchOps {
    template <class Fmt, int NV, int R>
    struct Launch {
        using T = typename Fmt::T;
        static int run(const LnPlan& p, const T* dy, const T* x, const float* mean,
                       const float* inv_std, const float* gamma, T* dx, float* ws, int64_t rows,
                       int D, int* err, cudaStream_t st) {
            launch_pdl(ln_bwd_rows_ring_kernel<Fmt, NV, R, kRms>, dim3((unsigned)p.grid),
                       dim3((unsigned)p.threads), p.smem, st, dy, x, mean, inv_std, gamma, dx, ws,
                       rows, D, p.stages, p.rows_per_cta, err, p.wait_limit_ns, p.withhold_copies);
            return 0;
        }
    };
};

template <bool kRms>
struct SplitLaunchOps {
    template <class Fmt, int NV, int R>
    struct Launch {
        using T = typename Fmt::T;
        static int run(const LnPlan& p, const T* dy, const T* x, const float* mean,
                       const float* inv_std, const float* gamma, T* dx, float* ws, int64_t rows,
                       int D, int* err, cudaStream_t st) {
            launch_cluster(ln_bwd_rows_split_kernel<Fmt, NV, R, kRms>, dim3((unsigned)p.grid),
                           dim3((unsigned)p.threads), p.smem, st, p.cluster, dy, x, mean, inv_std,
                           gamma, dx, ws, rows, D, p.stages, p.rows_per_cta, err, p.wait_limit_ns,
                           p.withhold_copies);
            return 0;
        }
    };
};

template <class Fmt>
void launch_rows(const LnPlan& p, const void* dY, const void* x, const float* mean,
                 const float* inv_std, const float* gamma, void* dX, float* ws, int64_t rows,
                 int64_t D, int* err, cudaStream_t st, bool rms = false) {
    using T = typename Fmt::T;
    const T* dy = static_cast<const T*>(dY);
    const T* xx = static_cast<const T*>(x);
    T* dx = static_cast<T*>(dX);
    if (p.path == Path::kRingWide && p.pair) {
        if constexpr (sizeof(T) == 2) {
            if (rms)
                launch_pdl(ln_bwd_rows_ring_kernel<Fmt, 2, 1, true, kWideWarps, kWidePairThreads>,
                           dim3((unsigned)p.grid), dim3((unsigned)p.threads), p.smem, st, dy, xx,
                           mean, inv_std, gamma, dx, ws, rows, (int)D, p.stages, p.rows_per_cta, err,
                           p.wait_limit_ns, p.withhold_copies);
            else
                launch_pdl(ln_bwd_rows_ring_kernel<Fmt, 2, 1, false, kWideWarps, kWidePairThreads>,
                           dim3((unsigned)p.grid), dim3((unsigned)p.threads), p.smem, st, dy, xx,
                           mean, inv_std, gamma, dx, ws, rows, (int)D, p.stages, p.rows_per_cta, err,
                           p.wait_limit_ns, p.withhold_copies);
        }
    } else if (p.path == Path::kRingWide) {
        if constexpr (sizeof(T) == 2) {
            if (rms)
                launch_pdl(ln_bwd_rows_ring_kernel<Fmt, 2, 1, true, kWideWarps>, dim3((unsigned)p.grid),
                           dim3((unsigned)p.threads), p.smem, st, dy, xx, mean, inv_std, gamma, dx, ws,
                           rows, (int)D, p.stages, p.rows_per_cta, err, p.wait_limit_ns,
                           p.withhold_copies);
            else
                launch_pdl(ln_bwd_rows_ring_kernel<Fmt, 2, 1, false, kWideWarps>, dim3((unsigned)p.grid),
                           dim3((unsigned)p.threads), p.smem, st, dy, xx, mean, inv_std, gamma, dx, ws,
                           rows, (int)D, p.stages, p.rows_per_cta, err, p.wait_limit_ns,
                           p.withhold_copies);
        }
    } else if (p.path == Path::kSplit) {
        if (rms)
            with_split_variant<Fmt, SplitLaunchOps<true>::template Launch>(
                p.nv, p.r, p, dy, xx, mean, inv_std, gamma, dx, ws, rows, (int)D, err, st);
        else
            with_split_variant<Fmt, SplitLaunchOps<false>::template Launch>(
                p.nv, p.r, p, dy, xx, mean, inv_std, gamma, dx, ws, rows, (int)D, err, st);
    } else if (p.path == Path::kRing) {
        if (rms)
            with_ring_variant<Fmt, RingLaunchOps<true>::template Launch>(
                p.nv, p.r, p, dy, xx, mean, inv_std, gamma, dx, ws, rows, (int)D, err, st);
        else
            with_ring_variant<Fmt, RingLaunchOps<false>::template Launch>(
                p.nv, p.r, p, dy, xx, mean, inv_std, gamma, dx, ws, rows, (int)D, err, st);
    } else if (p.nv > 0) {
        if (rms)
            with_reg_variant<Fmt, RegOps<true>::template Launch>(p.nv, p, dy, xx, mean, inv_std,
                                                                 gamma, dx, ws, rows, (int)D, st);
        else
            with_reg_variant<Fmt, RegOps<false>::template Launch>(p.nv, p, dy, xx, mean, inv_std,
                                                                  gamma, dx, ws, rows, (int)D, st);
    } else if (rms) {
        launch_pdl(ln_bwd_rows_plain_kernel<Fmt, true>, dim3((unsigned)p.grid), dim3((unsigned)p.threads),
                   0, st, dy, xx, mean, inv_std, gamma, dx, ws, rows, D, p.rows_per_cta);
    } else {
        launch_pdl(ln_bwd_rows_plain_kernel<Fmt, false>, dim3((unsigned)p.grid), dim3((unsigned)p.threads),
                   0, st, dy, xx, mean, inv_std, gamma, dx, ws, rows, D, p.rows_per_cta);
    }
}

}  // namespace
}  // namespace tb

extern "C" tb_status tb_layernorm_bwd_workspace_size(int64_t rows, int64_t D, tb_dtype io_dtype,
                                                     size_t* bytes) {
    using namespace tb;
    if (!bytes || rows < 0 || D < 0) return TB_ERR_INVALID_VALUE;
    if (!dtype_valid(io_dtype)) return TB_ERR_UNSUPPORTED_DTYPE;
    *bytes = 0;
    if (rows == 0 || D == 0) return TB_OK;
    int dev = 0;
    DeviceInfo info{};
    if (!current_device_info(&dev, &info)) return TB_ERR_CUDA;
    LnPlan p;
    // Size for the aligned layout; the fallback path never uses more CTAs.
    if (!make_plan(rows, D, io_dtype, true, info, &p)) return TB_ERR_CUDA;
    LnPlan q;
    if (!make_plan(rows, D, io_dtype, false, info, &q)) return TB_ERR_CUDA;
    *bytes = std::max(workspace_bytes_for(p, D), workspace_bytes_for(q, D));
    return TB_OK;
}

extern "C" tb_status tb_layernorm_bwd(const void* dY, const void* x, const float* mean,
                                      const float* inv_std, const float* gamma, void* dX,
                                      float* dgamma, float* dbeta, int64_t rows, int64_t D,
                                      tb_dtype io_dtype, void* workspace, size_t workspace_bytes,
                                      void* stream) {
    using namespace tb;
    if (rows < 0 || D < 0) return TB_ERR_INVALID_VALUE;
    if (!dtype_valid(io_dtype)) return TB_ERR_UNSUPPORTED_DTYPE;
    if (D == 0) return TB_OK;
    if (D > (int64_t)1 << 30) return TB_ERR_INVALID_VALUE;
    if (!dgamma || !dbeta || !gamma) return TB_ERR_INVALID_VALUE;
    if (rows > 0 && (!dY || !x || !mean || !inv_std || !dX)) return TB_ERR_INVALID_VALUE;
    if (rows > 0 && D > INT64_MAX / rows / 4) return TB_ERR_INVALID_VALUE;
    const size_t es = dtype_size(io_dtype);
    if (!aligned_to(dgamma, 4) || !aligned_to(dbeta, 4) || !aligned_to(gamma, 4)) return TB_ERR_MISALIGNED;
    if (rows > 0 && (!aligned_to(dY, es) || !aligned_to(x, es) || !aligned_to(dX, es) ||
                     !aligned_to(mean, 4) || !aligned_to(inv_std, 4)))
        return TB_ERR_MISALIGNED;
    const int64_t n = rows * D;
    const Range r_dx = range_of(dX, n, es), r_dg = range_of(dgamma, D, 4), r_db = range_of(dbeta, D, 4);
    const Range r_ws = range_of(workspace, (int64_t)workspace_bytes, 1);
    const Range ins[5] = {range_of(dY, n, es), range_of(x, n, es), range_of(mean, rows, 4),
                          range_of(inv_std, rows, 4), range_of(gamma, D, 4)};
    const Range outs[4] = {r_dx, r_dg, r_db, r_ws};
    for (const Range& o : outs)
        for (const Range& in : ins)
            if (overlap(o, in)) return TB_ERR_ALIAS;
    for (int a = 0; a < 4; ++a)
        for (int b = a + 1; b < 4; ++b)
            if (overlap(outs[a], outs[b])) return TB_ERR_ALIAS;

    int dev = 0;
    DeviceInfo info{};
    if (!current_device_info(&dev, &info)) return TB_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (rows == 0)
        return launch_colsum(nullptr, 0, 2 * D, D, dgamma, dbeta, st) == cudaSuccess ? TB_OK : TB_ERR_CUDA;
    const bool aligned = aligned_to(dY, 16) && aligned_to(x, 16) && aligned_to(dX, 16) &&
                         aligned_to(gamma, 16) && aligned_to(workspace, 16);
    LnPlan p;
    if (!make_plan(rows, D, io_dtype, aligned, info, &p)) return TB_ERR_CUDA;
    if (!workspace || workspace_bytes < workspace_bytes_for(p, D)) return TB_ERR_WORKSPACE;
    if (!aligned_to(workspace, 4)) return TB_ERR_MISALIGNED;
    int* err = device_error_word();
    if (!err) return TB_ERR_CUDA;
    float* ws = static_cast<float*>(workspace);
    switch (io_dtype) {
        case TB_F32: launch_rows<F32>(p, dY, x, mean, inv_std, gamma, dX, ws, rows, D, err, st); break;
        case TB_BF16: launch_rows<BF16>(p, dY, x, mean, inv_std, gamma, dX, ws, rows, D, err, st); break;
        default: launch_rows<F16>(p, dY, x, mean, inv_std, gamma, dX, ws, rows, D, err, st); break;
    }
    if (cudaGetLastError() != cudaSuccess) return TB_ERR_CUDA;
    return launch_colsum(ws, p.parts, 2 * D, D, dgamma, dbeta, st) == cudaSuccess ? TB_OK : TB_ERR_CUDA;
}

// ------------------------------------------------------------------ entry point without allocation
// Scratch for tb_layernorm_bwd_noalloc: the per-CTA column partials live in this
// file-scope device array instead of a caller workspace.  Every device that loads
// the library holds it (16 MiB) until the process exits.  Host code must not pass
// the symbol itself to a kernel: its device address is looked up per device.
namespace tb {
namespace {
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;
constexpr int64_t kNoAllocScratchFloats = (int64_t)(kNoAllocScratchBytes / sizeof(float));
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) float g_ln_scratch[kNoAllocScratchFloats];

std::mutex g_scratch_mu;
CachedAddress g_scratch_addr[kNoAllocMaxDevices];

// Device address of g_ln_scratch on `dev` (which must be current); nullptr on error.
// Looked up once per device with cudaGetSymbolAddress, and again only if the
// device's context has changed since (after a device reset).
float* noalloc_scratch(int dev) {
    if (dev < 0 || dev >= kNoAllocMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    return static_cast<float*>(g_scratch_addr[dev].get(&g_ln_scratch));
}
}  // namespace
}  // namespace tb

extern "C" tb_status tb_layernorm_bwd_noalloc(const void* dY, const void* x, const float* mean,
                                              const float* inv_std, const float* gamma, void* dX,
                                              float* dgamma, float* dbeta, int64_t rows, int64_t D,
                                              tb_dtype io_dtype, void* stream) {
    using namespace tb;
    if (rows < 0 || D < 0) return TB_ERR_INVALID_VALUE;
    if (!dtype_valid(io_dtype)) return TB_ERR_UNSUPPORTED_DTYPE;
    if (D == 0) return TB_OK;
    // Even one CTA needs 2*D partial sums: D beyond the scratch capacity is rejected.
    if (2 * D > kNoAllocScratchFloats) return TB_ERR_WORKSPACE;
    if (!dgamma || !dbeta || !gamma) return TB_ERR_INVALID_VALUE;
    if (rows > 0 && (!dY || !x || !mean || !inv_std || !dX)) return TB_ERR_INVALID_VALUE;
    if (rows > 0 && D > INT64_MAX / rows / 4) return TB_ERR_INVALID_VALUE;
    const size_t es = dtype_size(io_dtype);
    if (!aligned_to(dgamma, 4) || !aligned_to(dbeta, 4) || !aligned_to(gamma, 4)) return TB_ERR_MISALIGNED;
    if (rows > 0 && (!aligned_to(dY, es) || !aligned_to(x, es) || !aligned_to(dX, es) ||
                     !aligned_to(mean, 4) || !aligned_to(inv_std, 4)))
        return TB_ERR_MISALIGNED;
    const int64_t n = rows * D;
    const Range ins[5] = {range_of(dY, n, es), range_of(x, n, es), range_of(mean, rows, 4),
                          range_of(inv_std, rows, 4), range_of(gamma, D, 4)};
    const Range outs[3] = {range_of(dX, n, es), range_of(dgamma, D, 4), range_of(dbeta, D, 4)};
    for (const Range& o : outs)
        for (const Range& in : ins)
            if (overlap(o, in)) return TB_ERR_ALIAS;
    for (int a = 0; a < 3; ++a)
        for (int b = a + 1; b < 3; ++b)
            if (overlap(outs[a], outs[b])) return TB_ERR_ALIAS;

    int dev = 0;
    DeviceInfo info{};
    if (!current_device_info(&dev, &info)) return TB_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (rows == 0)
        return launch_colsum(nullptr, 0, 2 * D, D, dgamma, dbeta, st) == cudaSuccess ? TB_OK : TB_ERR_CUDA;
    float* ws = noalloc_scratch(dev);
    int* err = device_error_word();
    if (!ws || !err) return TB_ERR_CUDA;
    const bool aligned = aligned_to(dY, 16) && aligned_to(x, 16) && aligned_to(dX, 16) &&
                         aligned_to(gamma, 16);
    LnPlan p;
    if (!make_plan(rows, D, io_dtype, aligned, info, &p)) return TB_ERR_CUDA;
    // Fewer CTAs (clusters) when their partial sums would not fit in the scratch array.
    const int64_t max_parts = kNoAllocScratchFloats / (2 * D);
    if (p.parts > max_parts) {
        p.parts = (int)max_parts;
        p.grid = p.parts * p.cluster;
        p.rows_per_cta = (rows + p.parts - 1) / p.parts;
    }
    // Every CTA overwrites its whole partial row, so nothing needs clearing first.
    switch (io_dtype) {
        case TB_F32: launch_rows<F32>(p, dY, x, mean, inv_std, gamma, dX, ws, rows, D, err, st); break;
        case TB_BF16: launch_rows<BF16>(p, dY, x, mean, inv_std, gamma, dX, ws, rows, D, err, st); break;
        default: launch_rows<F16>(p, dY, x, mean, inv_std, gamma, dX, ws, rows, D, err, st); break;
    }
    if (cudaGetLastError() != cudaSuccess) return TB_ERR_CUDA;
    return launch_colsum(ws, p.parts, 2 * D, D, dgamma, dbeta, st) == cudaSuccess ? TB_OK : TB_ERR_CUDA;
}

// ------------------------------------------------------------------ RMSNorm backward
extern "C" tb_status tb_rmsnorm_bwd_workspace_size(int64_t rows, int64_t D, tb_dtype io_dtype,
                                                   size_t* bytes) {
    using namespace tb;
    if (!bytes || rows < 0 || D < 0) return TB_ERR_INVALID_VALUE;
    if (!dtype_valid(io_dtype)) return TB_ERR_UNSUPPORTED_DTYPE;
    *bytes = 0;
    if (rows == 0 || D == 0) return TB_OK;
    int dev = 0;
    DeviceInfo info{};
    if (!current_device_info(&dev, &info)) return TB_ERR_CUDA;
    LnPlan p, q;
    if (!make_plan(rows, D, io_dtype, true, info, &p, true)) return TB_ERR_CUDA;
    if (!make_plan(rows, D, io_dtype, false, info, &q, true)) return TB_ERR_CUDA;
    *bytes = std::max(workspace_bytes_for(p, D, true), workspace_bytes_for(q, D, true));
    return TB_OK;
}

extern "C" tb_status tb_rmsnorm_bwd(const void* dY, const void* x, const float* inv_rms,
                                    const float* gamma, void* dX, float* dgamma, int64_t rows,
                                    int64_t D, tb_dtype io_dtype, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    using namespace tb;
    if (rows < 0 || D < 0) return TB_ERR_INVALID_VALUE;
    if (!dtype_valid(io_dtype)) return TB_ERR_UNSUPPORTED_DTYPE;
    if (D == 0) return TB_OK;
    if (D > (int64_t)1 << 30) return TB_ERR_INVALID_VALUE;
    if (!dgamma || !gamma) return TB_ERR_INVALID_VALUE;
    if (rows > 0 && (!dY || !x || !inv_rms || !dX)) return TB_ERR_INVALID_VALUE;
    if (rows > 0 && D > INT64_MAX / rows / 4) return TB_ERR_INVALID_VALUE;
    const size_t es = dtype_size(io_dtype);
    if (!aligned_to(dgamma, 4) || !aligned_to(gamma, 4)) return TB_ERR_MISALIGNED;
    if (rows > 0 && (!aligned_to(dY, es) || !aligned_to(x, es) || !aligned_to(dX, es) ||
                     !aligned_to(inv_rms, 4)))
        return TB_ERR_MISALIGNED;
    const int64_t n = rows * D;
    const Range ins[4] = {range_of(dY, n, es), range_of(x, n, es), range_of(inv_rms, rows, 4),
                          range_of(gamma, D, 4)};
    const Range outs[3] = {range_of(dX, n, es), range_of(dgamma, D, 4),
                           range_of(workspace, (int64_t)workspace_bytes, 1)};
    for (const Range& o : outs)
        for (const Range& in : ins)
            if (overlap(o, in)) return TB_ERR_ALIAS;
    for (int a = 0; a < 3; ++a)
        for (int b = a + 1; b < 3; ++b)
            if (overlap(outs[a], outs[b])) return TB_ERR_ALIAS;

    int dev = 0;
    DeviceInfo info{};
    if (!current_device_info(&dev, &info)) return TB_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (rows == 0)
        return launch_colsum(nullptr, 0, D, D, dgamma, nullptr, st) == cudaSuccess ? TB_OK : TB_ERR_CUDA;
    const bool aligned = aligned_to(dY, 16) && aligned_to(x, 16) && aligned_to(dX, 16) &&
                         aligned_to(gamma, 16) && aligned_to(workspace, 16);
    LnPlan p;
    if (!make_plan(rows, D, io_dtype, aligned, info, &p, true)) return TB_ERR_CUDA;
    if (!workspace || workspace_bytes < workspace_bytes_for(p, D, true)) return TB_ERR_WORKSPACE;
    if (!aligned_to(workspace, 4)) return TB_ERR_MISALIGNED;
    int* err = device_error_word();
    if (!err) return TB_ERR_CUDA;
    float* ws = static_cast<float*>(workspace);
    switch (io_dtype) {
        case TB_F32: launch_rows<F32>(p, dY, x, nullptr, inv_rms, gamma, dX, ws, rows, D, err, st, true); break;
        case TB_BF16: launch_rows<BF16>(p, dY, x, nullptr, inv_rms, gamma, dX, ws, rows, D, err, st, true); break;
        default: launch_rows<F16>(p, dY, x, nullptr, inv_rms, gamma, dX, ws, rows, D, err, st, true); break;
    }
    if (cudaGetLastError() != cudaSuccess) return TB_ERR_CUDA;
    return launch_colsum(ws, p.parts, D, D, dgamma, nullptr, st) == cudaSuccess ? TB_OK : TB_ERR_CUDA;
}

// ------------------------------------------------------------------ self-test of the bounded waits
namespace tb {
namespace {
// Runs the row kernel of a plan for rows x D bf16 with every copy withheld, so
// every ring wait gives up after wait_limit_ns.
tb_status run_withheld(int64_t rows, int64_t D, Path want, int64_t wait_limit_ns,
                       const DeviceInfo& info, int* err, cudaStream_t st) {
    LnPlan p;
    if (!make_plan(rows, D, TB_BF16, true, info, &p) || p.path != want) return TB_ERR_CUDA;
    p.wait_limit_ns = (unsigned long long)wait_limit_ns;
    p.withhold_copies = 1;
    // One zeroed allocation holds x, dY, dX, mean, inv_std, gamma and the workspace,
    // each part starting on a 256-byte boundary.
    const size_t mat = ((size_t)rows * D * sizeof(uint16_t) + 255) / 256 * 256;
    const size_t off_dy = mat, off_dx = 2 * mat, off_mu = 3 * mat;
    const size_t off_rs = off_mu + ((size_t)rows * 4 + 255) / 256 * 256;
    const size_t off_g = off_rs + ((size_t)rows * 4 + 255) / 256 * 256;
    const size_t off_ws = off_g + ((size_t)D * sizeof(float) + 255) / 256 * 256;
    const size_t total = off_ws + workspace_bytes_for(p, D);
    unsigned char* buf = nullptr;
    if (cudaMalloc(&buf, total) != cudaSuccess) {
        cudaGetLastError();
        return TB_ERR_OOM;
    }
    tb_status status = TB_OK;
    if (cudaMemsetAsync(buf, 0, total, st) != cudaSuccess) {
        status = TB_ERR_CUDA;
    } else {
        launch_rows<BF16>(p, buf + off_dy, buf, reinterpret_cast<float*>(buf + off_mu),
                          reinterpret_cast<float*>(buf + off_rs), reinterpret_cast<float*>(buf + off_g),
                          buf + off_dx, reinterpret_cast<float*>(buf + off_ws), rows, D, err, st);
        if (cudaGetLastError() != cudaSuccess) status = TB_ERR_CUDA;
    }
    if (cudaStreamSynchronize(st) != cudaSuccess) status = TB_ERR_CUDA;
    if (cudaFree(buf) != cudaSuccess) status = TB_ERR_CUDA;
    return status;
}
}  // namespace
}  // namespace tb

extern "C" tb_status tb_layernorm_bwd_selftest_timeout(int64_t wait_limit_ns, void* stream) {
    using namespace tb;
    if (wait_limit_ns < 1000 || wait_limit_ns > (int64_t)kWaitLimitNs) return TB_ERR_INVALID_VALUE;
    int dev = 0;
    DeviceInfo info{};
    if (!current_device_info(&dev, &info)) return TB_ERR_CUDA;
    int* err = device_error_word();
    if (!err) return TB_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The single-CTA ring (rows of 256 columns), then the cluster-split ring
    // (rows of 16384 columns over four CTAs): every CTA of the cluster gives up
    // at the same group and the cluster ends together.
    const tb_status a = run_withheld(4, 256, Path::kRing, wait_limit_ns, info, err, st);
    if (a != TB_OK) return a;
    return run_withheld(4, 16384, Path::kSplit, wait_limit_ns, info, err, st);
}
