// adamw.cu -- fused, multi-tensor, mixed-precision AdamW step.
//
// Per element ("Mastering LLM Training with CUDA and ROCm", section "AdamW
// Algorithm"; "GPU 优化实战 Part 2", sections "AdamW 优化器——融合内核" and
// "混合精度训练（FP16 / BF16）"):
//   g = float(grad) * inv_loss_scale
//   m = b1*m + (1-b1)*g ;  v = b2*v + (1-b2)*g^2
//   param = param - lr*( (m/bc1) / (sqrt(v/bc2) + eps) + wd*param )
//   copy = rne(param) ;  grad = 0
//
// Design (GB300): one launch covers every tensor of the model.  The host plan
// holds a device table of tensors and a prefix sum of their "units" (8
// elements = one 16-byte vector of the 16-bit gradient and two of each fp32
// stream).  The flat unit space is cut into tiles of 2048 units (16,384
// elements) for a persistent grid (SM count x resident CTAs).  CTA b starts on
// tile b; every further tile is claimed from a counter in the plan, in
// increasing order, so all CTAs stream through the same region of HBM at once
// and a CTA on a faster SM simply takes more tiles (on GB300 some SMs stream a
// few per cent slower than others; with a fixed share per CTA the step would
// end with them).  The update is elementwise, so which CTA takes which tile
// changes no result bit.  Each CTA follows its tensor with a forward scan of
// the table.  A warp walks blocks of 256 elements, each lane taking two 4-element
// chunks 128 elements apart, so every warp access covers whole 32-byte sectors:
// 16-byte evict-first accesses for fp32, 8-byte ones for the 16-bit arrays, two
// blocks in flight per warp.  14 B read and 16 B written per element, one HBM
// pass.
// Tensors whose five pointers are not all 16-byte aligned, and the last
// partial unit of a tensor, take a scalar path.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <type_traits>
#include <unordered_set>
#include <vector>

#include "tb_common.cuh"

namespace tb {
namespace {

constexpr int kUnit = 8;        // elements per unit
constexpr int kThreads = 256;   // threads per CTA
constexpr int kUnroll = 2;      // 256-element blocks in flight per warp (16 elements per thread)
constexpr int64_t kTileUnits = (int64_t)kThreads * kUnroll * 4;   // 16384 elements
// The gradient-norm pass reads 2 bytes per element instead of 30: it takes 4x
// longer tiles (65,536 elements) so a CTA spends less of its time between tiles.
constexpr int64_t kNormTileUnits = 4 * kTileUnits;
// Grid of the gradient-norm pass.  On a large table each CTA owns a fixed chunk of
// kNormChunkTiles consecutive tiles (262,144 elements) and writes the chunk's
// partial at the chunk's index: one CTA per chunk, so the block scheduler hands
// chunks to whichever SM has room (a fixed share per CTA of a persistent grid ends
// with the slowest SMs; 7B table: 1.80 against 1.88 ms), and the partials still do
// not depend on timing.  Below four chunks per resident CTA slot the CTAs would be
// too short-lived to pay for their own start, and a persistent grid dealing tiles
// round-robin is kept (GPT-2-small table: 49.7 against 53.2 us).  Returns the
// chunk length in tiles, 0 for the round-robin grid.
constexpr int64_t kNormChunkTiles = 4;

int64_t norm_chunk_tiles(int64_t n_tiles, int64_t slots) {
    return n_tiles >= 4 * kNormChunkTiles * std::max<int64_t>(slots, 1) ? kNormChunkTiles : 0;
}
constexpr uint64_t kPlanMagic = 0x7462616461707731ull;

struct alignas(16) TensorEntry {
    float* p;
    float* m;
    float* v;
    void* g;
    void* c;
    int64_t n;
    int64_t unit_begin;   // prefix sum of ceil(n/8) over the preceding tensors
    int32_t vec_ok;       // all five pointers 16-byte aligned
    int32_t pad;
};
static_assert(sizeof(TensorEntry) == 64, "table entry is one 64-byte line");

// Tile counter of a plan's step kernel, in device memory after the table.  The
// host clears it with a 16-byte memset enqueued on the launch's stream right
// before every launch, so it is zero when a launch starts whatever an earlier
// launch left in it.  Launches of one plan must be stream-ordered (they update
// the same tensors and share this counter).
struct alignas(16) TileQueue {
    unsigned long long next;   // tiles claimed so far beyond the first one of each CTA
    unsigned long long pad;
};

// Per-step scalars, hoisted on the host.
struct Scalars {
    float lr, beta1, beta2, eps, wd;
    float omb1, omb2;   // 1 - beta, formed in fp32
    float bc1, bc2;     // 1 - beta^t, formed in double and rounded
    float inv_s;        // 1 / loss_scale
    float clip;         // gradient-norm clip factor (exactly 1 when not clipping)
};

// Copy-format tag of plans whose tensors have no working copy: nothing is written.
struct NoCopy {
    using T = uint16_t;
};
template <class C>
constexpr bool kHasCopy = !std::is_same<C, NoCopy>::value;
template <class G>
constexpr bool kF32Grad = std::is_same<G, F32>::value;

__device__ __forceinline__ void adamw_update(float& th, float& m, float& v, float g_scaled,
                                             const Scalars& s) {
    const float g = (g_scaled * s.inv_s) * s.clip;
    m = s.beta1 * m + s.omb1 * g;
    v = s.beta2 * v + s.omb2 * (g * g);
    const float m_hat = m / s.bc1;
    const float v_hat = v / s.bc2;
    const float u = m_hat / (sqrtf(v_hat) + s.eps);
    th = th - s.lr * (u + s.wd * th);
}

template <class G, class C>
__device__ __forceinline__ void scalar_element(const TensorEntry& t, int64_t i, const Scalars& s) {
    using GT = typename G::T;
    using CT = typename C::T;
    float th = t.p[i], m = t.m[i], v = t.v[i];
    GT* gp = static_cast<GT*>(t.g);
    adamw_update(th, m, v, G::to_f32(gp[i]), s);
    t.p[i] = th;
    t.m[i] = m;
    t.v[i] = v;
    if constexpr (kHasCopy<C>) static_cast<CT*>(t.c)[i] = C::from_f32(th);
    gp[i] = G::from_f32(0.0f);
}

// Units [a, e) of one tensor when the step is skipped: only the gradient is reset.
template <class G>
__device__ __forceinline__ void zero_segment(const TensorEntry& t, int64_t a, int64_t e) {
    using GT = typename G::T;
    const int64_t n = t.n;
    const int64_t full = n / kUnit;
    GT* gp = static_cast<GT*>(t.g);
    if (t.vec_ok) {
        const int64_t fe = e < full ? e : full;
        for (int64_t u = a + threadIdx.x; u < fe; u += kThreads) {
            if constexpr (kF32Grad<G>) {
                st_stream_f4(reinterpret_cast<float*>(gp) + u * kUnit, make_float4(0.f, 0.f, 0.f, 0.f));
                st_stream_f4(reinterpret_cast<float*>(gp) + u * kUnit + 4, make_float4(0.f, 0.f, 0.f, 0.f));
            } else {
                st_stream_u4(gp + u * kUnit, make_uint4(0u, 0u, 0u, 0u));
            }
        }
        if (full >= a && full < e)
            for (int64_t i = full * kUnit + threadIdx.x; i < n; i += kThreads) gp[i] = G::from_f32(0.0f);
    } else {
        const int64_t hi = e * kUnit < n ? e * kUnit : n;
        for (int64_t i = a * kUnit + threadIdx.x; i < hi; i += kThreads) gp[i] = G::from_f32(0.0f);
    }
}

// 4 consecutive 16-bit values (8 bytes) as fp32, and back (round to nearest even),
// with the streaming cache policy.
template <class Fmt>
__device__ __forceinline__ void ld4_16(const void* p, float (&f)[4]) {
    const uint2 u = __ldcs(reinterpret_cast<const uint2*>(p));
    const typename Fmt::T* h = reinterpret_cast<const typename Fmt::T*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = Fmt::to_f32(h[i]);
}
template <class Fmt>
__device__ __forceinline__ void st4_16(void* p, const float (&f)[4]) {
    uint2 u;
    typename Fmt::T* h = reinterpret_cast<typename Fmt::T*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = Fmt::from_f32(f[i]);
    __stcs(reinterpret_cast<uint2*>(p), u);
}

// Units [a, e) of one tensor (local unit indices).  A warp walks blocks of 256
// elements (32 units); lane l takes the 4-element chunks [4l, 4l+4) and
// [128+4l, 128+4l+4) of a block.  So every fp32 access of a warp covers 512
// contiguous bytes and every 16-bit access 256: each 32-byte sector a warp
// instruction touches is used whole.  kUnroll blocks per warp are in flight.
template <class G, class C>
__device__ __forceinline__ void process_segment(const TensorEntry& t, int64_t a, int64_t e,
                                                const Scalars& s) {
    using GT = typename G::T;
    using CT = typename C::T;
    const int64_t n = t.n;
    const int64_t full = n / kUnit;   // units holding 8 valid elements
    if (t.vec_ok) {
        constexpr int kWarps = kThreads / 32;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        // elements [e0, e1): e0 and e1 are multiples of 8, every chunk start a multiple
        // of 4, so a chunk that starts below e1 ends at or below it
        const int64_t e0 = a * kUnit, e1 = (e < full ? e : full) * kUnit;
        for (int64_t blk = e0 + (int64_t)warp * 256 * kUnroll; blk < e1;
             blk += (int64_t)kWarps * 256 * kUnroll) {
            float th[kUnroll][2][4], mm[kUnroll][2][4], vv[kUnroll][2][4], gg[kUnroll][2][4];
            bool act[kUnroll][2];
#pragma unroll
            for (int j = 0; j < kUnroll; ++j) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int64_t i0 = blk + j * 256 + h * 128 + 4 * lane;
                    act[j][h] = i0 < e1;
                    if (act[j][h]) {
                        const float4 a0 = ld_stream_f4(t.p + i0), b0 = ld_stream_f4(t.m + i0),
                                     c0 = ld_stream_f4(t.v + i0);
                        th[j][h][0] = a0.x; th[j][h][1] = a0.y; th[j][h][2] = a0.z; th[j][h][3] = a0.w;
                        mm[j][h][0] = b0.x; mm[j][h][1] = b0.y; mm[j][h][2] = b0.z; mm[j][h][3] = b0.w;
                        vv[j][h][0] = c0.x; vv[j][h][1] = c0.y; vv[j][h][2] = c0.z; vv[j][h][3] = c0.w;
                        if constexpr (kF32Grad<G>) {
                            const float4 g0 = ld_stream_f4(static_cast<const float*>(t.g) + i0);
                            gg[j][h][0] = g0.x; gg[j][h][1] = g0.y; gg[j][h][2] = g0.z; gg[j][h][3] = g0.w;
                        } else {
                            ld4_16<G>(static_cast<const GT*>(t.g) + i0, gg[j][h]);
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kUnroll; ++j) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (!act[j][h]) continue;
                    const int64_t i0 = blk + j * 256 + h * 128 + 4 * lane;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        adamw_update(th[j][h][q], mm[j][h][q], vv[j][h][q], gg[j][h][q], s);
                    st_stream_f4(t.p + i0, make_float4(th[j][h][0], th[j][h][1], th[j][h][2], th[j][h][3]));
                    st_stream_f4(t.m + i0, make_float4(mm[j][h][0], mm[j][h][1], mm[j][h][2], mm[j][h][3]));
                    st_stream_f4(t.v + i0, make_float4(vv[j][h][0], vv[j][h][1], vv[j][h][2], vv[j][h][3]));
                    if constexpr (kHasCopy<C>) st4_16<C>(static_cast<CT*>(t.c) + i0, th[j][h]);
                    if constexpr (kF32Grad<G>)
                        st_stream_f4(static_cast<float*>(t.g) + i0, make_float4(0.f, 0.f, 0.f, 0.f));
                    else
                        __stcs(reinterpret_cast<uint2*>(static_cast<GT*>(t.g) + i0), make_uint2(0u, 0u));
                }
            }
        }
        // The tensor's last, partial unit (fewer than 8 elements).
        if (full >= a && full < e) {
            for (int64_t i = full * kUnit + threadIdx.x; i < n; i += kThreads)
                scalar_element<G, C>(t, i, s);
        }
    } else {
        const int64_t hi = e * kUnit < n ? e * kUnit : n;
        for (int64_t i = a * kUnit + threadIdx.x; i < hi; i += kThreads)
            scalar_element<G, C>(t, i, s);
    }
}

// Index of the tensor holding unit u, searching forward from k (tiles of a CTA
// visit the unit space in increasing order): a few linear steps, then binary search.
__device__ __forceinline__ int tensor_of(const TensorEntry* __restrict__ tab, int ntab, int k,
                                         int64_t u) {
#pragma unroll 1
    for (int step = 0; step < 4; ++step) {
        if (k + 1 >= ntab || tab[k + 1].unit_begin > u) return k;
        ++k;
    }
    int lo = k, hi = ntab - 1;   // last index with unit_begin <= u
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tab[mid].unit_begin <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Tiles of kTileUnits consecutive units: CTA b takes tile b first, then claims
// tiles from q->next in increasing order, so at any moment all CTAs stream
// through one window of about grid*kTileUnits units and faster SMs take more.
// clip (device memory, may be null): {norm, factor, nonfinite} as written by the
// gradient-norm kernels; the gradient is multiplied by factor, and when nonfinite
// is set the step is skipped (only the gradient is reset).
// step_dev (device memory, may be null): the step t, read when the kernel runs;
// the bias corrections are then formed here, as the host forms them otherwise
// (1 - beta^t in double, rounded to fp32).  A t below 1 sets the error word to
// TB_ERR_INVALID_VALUE and nothing is updated.
template <class G, class C>
__global__ void __launch_bounds__(kThreads, 2)
adamw_multi_tensor_kernel(const TensorEntry* __restrict__ tab, int ntab, int64_t total_units,
                          int64_t n_tiles, Scalars s, const float* __restrict__ clip,
                          const int64_t* __restrict__ step_dev, int* err, TileQueue* q) {
    bool skip = false;
    if (clip) {
        s.clip = clip[1];
        skip = clip[2] != 0.0f;
    }
    if (step_dev) {
        __shared__ float s_bc[2];
        __shared__ int s_bad;
        if (threadIdx.x == 0) {
            const int64_t t = *step_dev;
            s_bad = t < 1;
            if (t < 1 && blockIdx.x == 0) atomicExch(err, (int)TB_ERR_INVALID_VALUE);
            s_bc[0] = (float)(1.0 - pow((double)s.beta1, (double)t));
            s_bc[1] = (float)(1.0 - pow((double)s.beta2, (double)t));
        }
        __syncthreads();
        if (s_bad) return;
        s.bc1 = s_bc[0];
        s.bc2 = s_bc[1];
    }
    // The next tile is claimed while this one streams (the claim's round trip
    // stays off the critical path); two slots, so one barrier per tile suffices.
    __shared__ long long s_tile[2];
    int k = 0;
    int it = 0;
    for (int64_t tile = blockIdx.x; tile < n_tiles; ++it) {
        if (threadIdx.x == 0)
            s_tile[(it + 1) & 1] = (long long)gridDim.x + (long long)atomicAdd(&q->next, 1ull);
        const int64_t u_lo = tile * kTileUnits;
        const int64_t u_hi = u_lo + kTileUnits < total_units ? u_lo + kTileUnits : total_units;
        k = tensor_of(tab, ntab, k, u_lo);
        int kk = k;
        int64_t u = u_lo;
        while (u < u_hi && kk < ntab) {
            const TensorEntry t = tab[kk];
            const int64_t t_end = (kk + 1 < ntab) ? tab[kk + 1].unit_begin : total_units;
            const int64_t seg_hi = u_hi < t_end ? u_hi : t_end;
            if (seg_hi > u) {
                if (skip) zero_segment<G>(t, u - t.unit_begin, seg_hi - t.unit_begin);
                else process_segment<G, C>(t, u - t.unit_begin, seg_hi - t.unit_begin, s);
            }
            u = seg_hi > u ? seg_hi : u;
            ++kk;
        }
        __syncthreads();
        tile = s_tile[(it + 1) & 1];
    }
}

// ------------------------------------------------------------------ gradient norm
// Sum of squares of the unscaled gradient over every tensor (reading only the
// gradient), plus a non-finite flag.  Each thread adds its squares in fp32 in
// rounds of at most 32, the round sums of a tile in fp32 and the tile sums in
// fp64; CTA b covers the tiles of chunk b (or tiles b, b + grid, ...) and writes
// one fp64 partial and one flag at index b; the finalize kernel adds the partials
// in index order.
template <class G>
__global__ void __launch_bounds__(kThreads)
adamw_grad_sumsq_kernel(const TensorEntry* __restrict__ tab, int ntab, int64_t total_units,
                        int64_t n_tiles, int64_t chunk, float inv_s, double* __restrict__ part,
                        int* __restrict__ flags) {
    using GT = typename G::T;
    double acc = 0.0;
    int bad = 0;
    int k = 0;
    // chunk > 0: tiles [b*chunk, (b+1)*chunk); chunk == 0: tiles b, b + grid, ...
    const int64_t t0 = chunk ? (int64_t)blockIdx.x * chunk : (int64_t)blockIdx.x;
    const int64_t t1 = chunk ? (t0 + chunk < n_tiles ? t0 + chunk : n_tiles) : n_tiles;
    const int64_t tstep = chunk ? 1 : (int64_t)gridDim.x;
    for (int64_t tile = t0; tile < t1; tile += tstep) {
        const int64_t u_lo = tile * kNormTileUnits;
        const int64_t u_hi = u_lo + kNormTileUnits < total_units ? u_lo + kNormTileUnits : total_units;
        k = tensor_of(tab, ntab, k, u_lo);
        float fs = 0.f;
        int kk = k;
        int64_t u = u_lo;
        while (u < u_hi && kk < ntab) {
            const TensorEntry t = tab[kk];
            const int64_t t_end = (kk + 1 < ntab) ? tab[kk + 1].unit_begin : total_units;
            const int64_t seg_hi = u_hi < t_end ? u_hi : t_end;
            if (seg_hi > u) {
                const int64_t a = u - t.unit_begin, e = seg_hi - t.unit_begin;
                const int64_t n = t.n, full = n / kUnit;
                const GT* gp = static_cast<const GT*>(t.g);
                int64_t lo_elem = a * kUnit, hi_elem = (e * kUnit < n) ? e * kUnit : n;
                if (t.vec_ok) {
                    const int64_t fe = e < full ? e : full;
                    // four units in flight per thread; absent ones read as zeros
                    if constexpr (kF32Grad<G>) {
                        const float* gf = reinterpret_cast<const float*>(gp);
                        for (int64_t u0 = a + threadIdx.x; u0 < fe; u0 += 4 * kThreads) {
                            float4 r[4][2];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int64_t uu = u0 + (int64_t)j * kThreads;
                                const bool in = uu < fe;
                                r[j][0] = in ? ld_stream_f4(gf + uu * kUnit) : make_float4(0.f, 0.f, 0.f, 0.f);
                                r[j][1] = in ? ld_stream_f4(gf + uu * kUnit + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                            float f1 = 0.f;   // the 32 squares of this round
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float v[8] = {r[j][0].x, r[j][0].y, r[j][0].z, r[j][0].w,
                                                    r[j][1].x, r[j][1].y, r[j][1].z, r[j][1].w};
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    bad |= !isfinite(v[q]);
                                    const float x = v[q] * inv_s;
                                    f1 += x * x;
                                }
                            }
                            fs += f1;
                        }
                    } else
                    for (int64_t u0 = a + threadIdx.x; u0 < fe; u0 += 4 * kThreads) {
                        uint4 r[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int64_t uu = u0 + (int64_t)j * kThreads;
                            r[j] = uu < fe ? ld_stream_u4(gp + uu * kUnit) : make_uint4(0u, 0u, 0u, 0u);
                        }
                        float f1 = 0.f;   // the 32 squares of this round
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float v[8];
                            unpack8<G>(r[j], v);
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                bad |= !isfinite(v[q]);
                                const float x = v[q] * inv_s;
                                f1 += x * x;
                            }
                        }
                        fs += f1;
                    }
                    lo_elem = fe > a ? fe * kUnit : lo_elem;   // scalar tail only
                }
                float f1 = 0.f;
                for (int64_t i = lo_elem + threadIdx.x, c = 1; i < hi_elem; i += kThreads, ++c) {
                    const float g = G::to_f32(gp[i]);
                    bad |= !isfinite(g);
                    const float x = g * inv_s;
                    f1 += x * x;
                    if ((c & 31) == 0) {   // 32 squares per first-level sum here too
                        fs += f1;
                        f1 = 0.f;
                    }
                }
                fs += f1;
            }
            u = seg_hi > u ? seg_hi : u;
            ++kk;
        }
        acc += (double)fs;
    }
    // CTA sum in a fixed order: warp butterfly, then warp 0 over the warp sums.
    __shared__ double wsum[kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = acc;
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < kThreads / 32; ++w) t += wsum[w];
        part[blockIdx.x] = t;
        flags[blockIdx.x] = bad;
    }
}

// out = {norm, clip factor, nonfinite ? 1 : 0} from the per-CTA partials, added in
// index order by one CTA (thread j takes j, j+256, ...; then a fixed tree).
__global__ void __launch_bounds__(kThreads)
adamw_grad_norm_finalize_kernel(const double* __restrict__ part, const int* __restrict__ flags,
                                int nparts, float max_norm, float* __restrict__ out) {
    __shared__ double sh[kThreads];
    double acc = 0.0;
    int bad = 0;
#pragma unroll 8
    for (int i = threadIdx.x; i < nparts; i += kThreads) {
        acc += part[i];
        bad |= flags[i];
    }
    sh[threadIdx.x] = acc;
    bad = __syncthreads_or(bad);
    for (int w = kThreads / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) sh[threadIdx.x] += sh[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const double norm = sqrt(sh[0]);
        const double f = (max_norm > 0.0f && norm > (double)max_norm) ? (double)max_norm / norm : 1.0;
        out[0] = (float)norm;
        out[1] = (float)f;
        out[2] = bad ? 1.0f : 0.0f;
    }
}

template <class G>
const void* step_kernel_for(tb_dtype c, bool copy) {
    if (!copy) return reinterpret_cast<const void*>(&adamw_multi_tensor_kernel<G, NoCopy>);
    return c == TB_BF16 ? reinterpret_cast<const void*>(&adamw_multi_tensor_kernel<G, BF16>)
                        : reinterpret_cast<const void*>(&adamw_multi_tensor_kernel<G, F16>);
}

// The step kernel for a gradient format, copy format and presence of copies.
const void* step_kernel(tb_dtype g, tb_dtype c, bool copy) {
    switch (g) {
        case TB_BF16: return step_kernel_for<BF16>(c, copy);
        case TB_F16: return step_kernel_for<F16>(c, copy);
        default: return step_kernel_for<F32>(c, copy);
    }
}

const void* norm_kernel(tb_dtype g) {
    switch (g) {
        case TB_BF16: return reinterpret_cast<const void*>(&adamw_grad_sumsq_kernel<BF16>);
        case TB_F16: return reinterpret_cast<const void*>(&adamw_grad_sumsq_kernel<F16>);
        default: return reinterpret_cast<const void*>(&adamw_grad_sumsq_kernel<F32>);
    }
}

}  // namespace
}  // namespace tb

struct tb_adamw_plan {
    uint64_t magic;
    int device;
    int n_tensors;
    tb_dtype grad_dtype;
    tb_dtype copy_dtype;
    tb::TensorEntry* d_table;
    int64_t total_units;
    int grid;        // CTAs of the step kernel
    int64_t norm_chunk;   // tiles per chunk of the gradient-norm kernel (0: round-robin)
    int norm_parts;       // CTAs of the gradient-norm kernel = chunks
    bool has_copy;   // the tensors have working copies (all of them, or none)
};

namespace tb {
namespace {
// Plans handed out and not yet destroyed.  A handle is checked against this set
// before it is dereferenced, so a destroyed or foreign pointer is rejected.
std::mutex g_plans_mu;
std::unordered_set<const tb_adamw_plan*> g_plans;

bool plan_register(const tb_adamw_plan* p) {
    std::lock_guard<std::mutex> lk(g_plans_mu);
    try {
        g_plans.insert(p);
    } catch (...) {
        return false;
    }
    return true;
}
bool plan_unregister(const tb_adamw_plan* p) {
    std::lock_guard<std::mutex> lk(g_plans_mu);
    return g_plans.erase(p) == 1;
}
bool plan_live(const tb_adamw_plan* p) {
    if (!p) return false;
    std::lock_guard<std::mutex> lk(g_plans_mu);
    return g_plans.count(p) == 1 && p->magic == kPlanMagic;
}
}  // namespace
}  // namespace tb

static tb_status plan_create_impl(const tb_tensor_desc* tensors, int n_tensors,
                                  tb_dtype grad_dtype, tb_dtype copy_dtype, tb_adamw_plan** out) {
    using namespace tb;
    if (!out || !tensors || n_tensors < 1) return TB_ERR_INVALID_VALUE;
    *out = nullptr;
    if (!dtype_valid(grad_dtype)) return TB_ERR_UNSUPPORTED_DTYPE;
    if (copy_dtype != TB_BF16 && copy_dtype != TB_F16) return TB_ERR_UNSUPPORTED_DTYPE;
    const size_t gs = dtype_size(grad_dtype);
    // Working copies: every tensor with elements has one, or none has.
    int with_copy = 0, sized = 0;
    for (int i = 0; i < n_tensors; ++i) {
        if (tensors[i].n > 0) {
            ++sized;
            with_copy += tensors[i].copy != nullptr;
        }
    }
    if (with_copy != 0 && with_copy != sized) return TB_ERR_INVALID_VALUE;
    const bool has_copy = with_copy > 0 || sized == 0;

    std::vector<TensorEntry> tab(n_tensors);
    std::vector<Range> ranges;
    ranges.reserve(5 * (size_t)n_tensors);
    int64_t units = 0;
    for (int i = 0; i < n_tensors; ++i) {
        const tb_tensor_desc& d = tensors[i];
        if (d.n < 0) return TB_ERR_INVALID_VALUE;
        if (d.n > 0 && (!d.param || !d.m || !d.v || !d.grad)) return TB_ERR_INVALID_VALUE;
        if (d.n > 0 && (!aligned_to(d.param, 4) || !aligned_to(d.m, 4) || !aligned_to(d.v, 4) ||
                        !aligned_to(d.grad, gs) || !aligned_to(d.copy, 2)))
            return TB_ERR_MISALIGNED;
        if (d.n > INT64_MAX / 8 - units * 8) return TB_ERR_INVALID_VALUE;
        TensorEntry& t = tab[i];
        t.p = d.param;
        t.m = d.m;
        t.v = d.v;
        t.g = d.grad;
        t.c = d.copy;
        t.n = d.n;
        t.unit_begin = units;
        t.vec_ok = aligned_to(d.param, 16) && aligned_to(d.m, 16) && aligned_to(d.v, 16) &&
                   aligned_to(d.grad, 16) && aligned_to(d.copy, 16);
        t.pad = 0;
        units += (d.n + kUnit - 1) / kUnit;
        ranges.push_back(range_of(d.param, d.n, 4));
        ranges.push_back(range_of(d.m, d.n, 4));
        ranges.push_back(range_of(d.v, d.n, 4));
        ranges.push_back(range_of(d.grad, d.n, gs));
        if (d.copy) ranges.push_back(range_of(d.copy, d.n, 2));
    }
    // No two buffers may overlap: sort by start, compare with the furthest end so far.
    ranges.erase(std::remove_if(ranges.begin(), ranges.end(),
                                [](const Range& r) { return r.lo == r.hi; }),
                 ranges.end());
    std::sort(ranges.begin(), ranges.end(), [](const Range& a, const Range& b) { return a.lo < b.lo; });
    uintptr_t reach = 0;
    for (size_t i = 0; i < ranges.size(); ++i) {
        if (i > 0 && ranges[i].lo < reach) return TB_ERR_ALIAS;
        reach = std::max(reach, ranges[i].hi);
    }

    int dev = 0;
    DeviceInfo info{};
    if (!current_device_info(&dev, &info)) return TB_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, step_kernel(grad_dtype, copy_dtype, has_copy),
                                                      kThreads, 0) != cudaSuccess)
        return TB_ERR_CUDA;
    per_sm = std::max(per_sm, 1);
    int norm_per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&norm_per_sm, norm_kernel(grad_dtype), kThreads,
                                                      0) != cudaSuccess)
        return TB_ERR_CUDA;
    const int64_t norm_tiles = (units + kNormTileUnits - 1) / kNormTileUnits;
    const int64_t slots = (int64_t)info.sm_count * std::max(norm_per_sm, 1);
    const int64_t norm_chunk = norm_chunk_tiles(norm_tiles, slots);
    const int64_t norm_parts =
        std::max<int64_t>(1, norm_chunk ? (norm_tiles + norm_chunk - 1) / norm_chunk
                                        : std::min<int64_t>(slots, norm_tiles));
    if (norm_parts > INT32_MAX) return TB_ERR_INVALID_VALUE;   // beyond any device's memory

    tb_adamw_plan* plan = new (std::nothrow) tb_adamw_plan;
    if (!plan) return TB_ERR_OOM;
    plan->magic = kPlanMagic;
    plan->device = dev;
    plan->n_tensors = n_tensors;
    plan->grad_dtype = grad_dtype;
    plan->copy_dtype = copy_dtype;
    plan->total_units = units;
    plan->grid = info.sm_count * per_sm;
    plan->norm_chunk = norm_chunk;
    plan->norm_parts = (int)norm_parts;
    plan->has_copy = has_copy;
    plan->d_table = nullptr;
    // The table, then the step kernel's tile counter (zero), copied up together.
    const size_t bytes = sizeof(TensorEntry) * (size_t)n_tensors + sizeof(TileQueue);
    tab.resize((size_t)n_tensors + 1);
    std::memset(static_cast<void*>(&tab[(size_t)n_tensors]), 0, sizeof(TensorEntry));
    static_assert(sizeof(TileQueue) <= sizeof(TensorEntry), "the counter fits in one table slot");
    cudaError_t e = cudaMalloc(&plan->d_table, bytes);
    if (e != cudaSuccess) {
        delete plan;
        cudaGetLastError();
        return e == cudaErrorMemoryAllocation ? TB_ERR_OOM : TB_ERR_CUDA;
    }
    if (cudaMemcpy(plan->d_table, tab.data(), bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaFree(plan->d_table);
        delete plan;
        return TB_ERR_CUDA;
    }
    if (!plan_register(plan)) {
        cudaFree(plan->d_table);
        delete plan;
        return TB_ERR_OOM;
    }
    *out = plan;
    return TB_OK;
}

extern "C" tb_status tb_adamw_plan_create(const tb_tensor_desc* tensors, int n_tensors,
                                          tb_dtype grad_dtype, tb_dtype copy_dtype,
                                          tb_adamw_plan** out) {
    try {
        return plan_create_impl(tensors, n_tensors, grad_dtype, copy_dtype, out);
    } catch (...) {   // host allocation of the table failed
        return TB_ERR_OOM;
    }
}

namespace tb {
namespace {
// The step kernel's tile counter: the slot after the plan's device table.
TileQueue* tile_queue(const tb_adamw_plan* plan) {
    return reinterpret_cast<TileQueue*>(plan->d_table + plan->n_tensors);
}

// step_dev non-null: the step is read on the device when the kernel runs and
// `step` is ignored.
tb_status adamw_step_impl(const tb_adamw_plan* plan, int64_t step, const tb_adamw_hparams* hp,
                          float inv_loss_scale, const float* clip, const int64_t* step_dev,
                          void* stream) {
    if (!hp || !plan_live(plan)) return TB_ERR_INVALID_VALUE;
    if (step_dev) step = 1;   // placeholder for the host-side scalars below
    if (step < 1) return TB_ERR_INVALID_VALUE;
    const float lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, eps = hp->eps, wd = hp->weight_decay;
    if (!std::isfinite(lr) || lr < 0.f) return TB_ERR_INVALID_VALUE;
    if (!(b1 >= 0.f && b1 < 1.f) || !(b2 >= 0.f && b2 < 1.f)) return TB_ERR_INVALID_VALUE;
    if (!std::isfinite(eps) || eps < 0.f) return TB_ERR_INVALID_VALUE;
    if (!std::isfinite(wd) || wd < 0.f) return TB_ERR_INVALID_VALUE;
    if (!std::isfinite(inv_loss_scale) || !(inv_loss_scale > 0.f)) return TB_ERR_INVALID_VALUE;
    if (clip && !aligned_to(clip, 4)) return TB_ERR_MISALIGNED;
    if (step_dev && !aligned_to(step_dev, 8)) return TB_ERR_MISALIGNED;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return TB_ERR_CUDA;
    if (dev != plan->device) return TB_ERR_DEVICE;
    if (plan->total_units == 0) return TB_OK;
    int* err = device_error_word();
    if (!err) return TB_ERR_CUDA;

    Scalars s;
    s.lr = lr;
    s.beta1 = b1;
    s.beta2 = b2;
    s.eps = eps;
    s.wd = wd;
    s.omb1 = 1.0f - b1;
    s.omb2 = 1.0f - b2;
    s.bc1 = static_cast<float>(1.0 - std::pow(static_cast<double>(b1), static_cast<double>(step)));
    s.bc2 = static_cast<float>(1.0 - std::pow(static_cast<double>(b2), static_cast<double>(step)));
    s.inv_s = inv_loss_scale;
    s.clip = 1.0f;

    int64_t n_tiles = (plan->total_units + kTileUnits - 1) / kTileUnits;
    const unsigned grid = (unsigned)std::min<int64_t>(plan->grid, n_tiles);
    const TensorEntry* tab = plan->d_table;
    int nt = plan->n_tensors;
    int64_t tu = plan->total_units;
    TileQueue* q = tile_queue(plan);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The counter starts every launch at zero, even after a launch that did not run
    // to its end.
    if (cudaMemsetAsync(q, 0, sizeof(TileQueue), st) != cudaSuccess) return TB_ERR_CUDA;
    void* args[] = {&tab, &nt, &tu, &n_tiles, &s, &clip, &step_dev, &err, &q};
    if (cudaLaunchKernel(step_kernel(plan->grad_dtype, plan->copy_dtype, plan->has_copy), dim3(grid),
                         dim3(kThreads), args, 0, st) != cudaSuccess)
        return TB_ERR_CUDA;
    return TB_OK;
}

// Partials of the gradient-norm kernel: one fp64 sum and one int flag per chunk.
size_t grad_norm_workspace(const tb_adamw_plan* plan) {
    return (size_t)plan->norm_parts * (sizeof(double) + sizeof(int));
}
}  // namespace
}  // namespace tb

extern "C" tb_status tb_adamw_step(const tb_adamw_plan* plan, int64_t step,
                                   const tb_adamw_hparams* hp, float inv_loss_scale,
                                   void* stream) {
    return tb::adamw_step_impl(plan, step, hp, inv_loss_scale, nullptr, nullptr, stream);
}

extern "C" tb_status tb_adamw_step_clipped(const tb_adamw_plan* plan, int64_t step,
                                           const tb_adamw_hparams* hp, float inv_loss_scale,
                                           const float* clip, void* stream) {
    if (!clip) return TB_ERR_INVALID_VALUE;
    return tb::adamw_step_impl(plan, step, hp, inv_loss_scale, clip, nullptr, stream);
}

extern "C" tb_status tb_adamw_step_device(const tb_adamw_plan* plan, const int64_t* step,
                                          const tb_adamw_hparams* hp, float inv_loss_scale,
                                          const float* clip, void* stream) {
    if (!step) return TB_ERR_INVALID_VALUE;
    return tb::adamw_step_impl(plan, 1, hp, inv_loss_scale, clip, step, stream);
}

extern "C" tb_status tb_adamw_grad_norm_workspace_size(const tb_adamw_plan* plan, size_t* bytes) {
    if (!bytes || !tb::plan_live(plan)) return TB_ERR_INVALID_VALUE;
    *bytes = tb::grad_norm_workspace(plan);
    return TB_OK;
}

extern "C" tb_status tb_adamw_grad_norm(const tb_adamw_plan* plan, float inv_loss_scale,
                                        float max_norm, float* out, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    using namespace tb;
    if (!out || !plan_live(plan)) return TB_ERR_INVALID_VALUE;
    if (!std::isfinite(inv_loss_scale) || !(inv_loss_scale > 0.f)) return TB_ERR_INVALID_VALUE;
    if (std::isnan(max_norm)) return TB_ERR_INVALID_VALUE;
    if (!aligned_to(out, 4)) return TB_ERR_MISALIGNED;
    if (!workspace || workspace_bytes < grad_norm_workspace(plan)) return TB_ERR_WORKSPACE;
    if (!aligned_to(workspace, 8)) return TB_ERR_MISALIGNED;
    if (overlap(range_of(out, 3, 4), range_of(workspace, (int64_t)workspace_bytes, 1))) return TB_ERR_ALIAS;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return TB_ERR_CUDA;
    if (dev != plan->device) return TB_ERR_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    double* part = static_cast<double*>(workspace);
    int* flags = reinterpret_cast<int*>(part + plan->norm_parts);
    const int64_t n_tiles = (plan->total_units + kNormTileUnits - 1) / kNormTileUnits;
    const int grid = plan->norm_parts;   // one CTA per chunk, or the round-robin grid
    if (plan->total_units > 0) {
        const TensorEntry* tab = plan->d_table;
        int nt = plan->n_tensors;
        int64_t tu = plan->total_units;
        int64_t nti = n_tiles;
        int64_t chunk = plan->norm_chunk;
        float inv = inv_loss_scale;
        void* args[] = {&tab, &nt, &tu, &nti, &chunk, &inv, &part, &flags};
        if (cudaLaunchKernel(norm_kernel(plan->grad_dtype), dim3(grid), dim3(kThreads), args, 0, st) !=
            cudaSuccess)
            return TB_ERR_CUDA;
    }
    adamw_grad_norm_finalize_kernel<<<1, kThreads, 0, st>>>(part, flags,
                                                            plan->total_units > 0 ? grid : 0,
                                                            max_norm, out);
    return launch_status();
}

extern "C" tb_status tb_adamw_selftest_stale_counter(const tb_adamw_plan* plan,
                                                     uint64_t next, void* stream) {
    using namespace tb;
    if (!plan_live(plan)) return TB_ERR_INVALID_VALUE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return TB_ERR_CUDA;
    if (dev != plan->device) return TB_ERR_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return TB_ERR_CUDA;
    const TileQueue stale = {static_cast<unsigned long long>(next), ~0ull};
    if (cudaMemcpy(tile_queue(plan), &stale, sizeof(stale), cudaMemcpyHostToDevice) != cudaSuccess)
        return TB_ERR_CUDA;
    return TB_OK;
}

extern "C" tb_status tb_adamw_plan_destroy(tb_adamw_plan* plan) {
    if (!plan) return TB_OK;
    if (!tb::plan_unregister(plan)) return TB_ERR_INVALID_VALUE;
    plan->magic = 0;
    tb_status st = TB_OK;
    if (plan->d_table && cudaFree(plan->d_table) != cudaSuccess) st = TB_ERR_CUDA;
    delete plan;
    return st;
}
