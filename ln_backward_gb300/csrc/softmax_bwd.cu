// softmax_bwd.cu -- row-wise softmax backward.
//
//   dX[r,i] = P[r,i] * (dY[r,i] - sum_j P[r,j] dY[r,j])
// ("GPU 优化实战 Part 2：用 CUDA/ROCm 实现 LLM 反向传播与训练循环", section 2.1
// "Softmax 反向内核").  The page's kernel gives one thread a whole row and walks
// it twice with a stride of `cols` between neighbouring threads; here a row is
// spread over the lanes of a group (4..32 lanes) or over a whole CTA so that
// every access is a coalesced 16-byte vector, the row is staged once in
// registers, the dot product is a butterfly of __shfl_xor_sync (plus shared
// memory across warps in the CTA path), and dX is written from the registers:
// each input element crosses HBM exactly once.
//
// Paths, chosen on the host:
//   group : rows of <= 256 vectors (1024 fp32 / 2048 16-bit), G lanes per row
//   pairs : causal 16-bit rows of 65..256 vectors (520..2048 columns) whose causal
//           block fits in the rows: rows q and period-1-q of a block on one warp
//   cta   : rows of <= 2048 vectors (8192 fp32 / 16384 16-bit), one CTA of 128..512
//           threads per row; causal rows whose causal block fits in the rows: rows q
//           and period-1-q of a block on one CTA of 128..512 threads
//   twopass: anything longer or not 16-byte aligned; reads the row twice
// The group, warp-pair and one-row CTA paths launch one CTA per row group when a CTA
// carries enough traffic (the hardware scheduler then balances the SMs), else a
// persistent grid; the CTA pairs always launch one CTA per pair.
//
// Causal variant (tb_softmax_bwd_causal): row r of an attention block can only be
// nonzero on its first min(cols, r mod period + 1 + offset) columns (the forward
// masked the rest, so P is exactly 0 there).  The kernels then read only the
// vectors that hold an unmasked column and write +0 to the others, which cuts the
// HBM reads of a square causal block roughly in half.
#include <algorithm>
#include <type_traits>

#include "tb_common.cuh"

namespace tb {
namespace {

// Value e of a 16-byte vector held as raw bits.
template <class Fmt>
__device__ __forceinline__ float vec_elem(const uint4& u, int e) {
    const typename Fmt::T* h = reinterpret_cast<const typename Fmt::T*>(&u);
    return Fmt::to_f32(h[e]);
}

template <class Fmt>
__device__ __forceinline__ uint4 vec_from(const float (&f)[Vec<Fmt>::kElems]) {
    uint4 u;
    typename Fmt::T* h = reinterpret_cast<typename Fmt::T*>(&u);
#pragma unroll
    for (int e = 0; e < Vec<Fmt>::kElems; ++e) h[e] = Fmt::from_f32(f[e]);
    return u;
}

// Two 16-bit values packed in a word, widened to fp32 (element 2q is the low half).
// widen_a and widen_b give the same values through different instructions.
template <class Fmt> __device__ __forceinline__ float2 widen_a(uint32_t w);
template <class Fmt> __device__ __forceinline__ float2 widen_b(uint32_t w);
template <> __device__ __forceinline__ float2 widen_a<BF16>(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <> __device__ __forceinline__ float2 widen_b<BF16>(uint32_t w) {
    return make_float2(__uint_as_float(__byte_perm(w, 0u, 0x1044)),
                       __uint_as_float(__byte_perm(w, 0u, 0x3244)));
}
template <> __device__ __forceinline__ float2 widen_a<F16>(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
}
template <> __device__ __forceinline__ float2 widen_b<F16>(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
}
template <class Fmt> __device__ __forceinline__ uint32_t narrow2(float2 r);
template <> __device__ __forceinline__ uint32_t narrow2<BF16>(float2 r) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(r.x, r.y);
    return *reinterpret_cast<const uint32_t*>(&h);
}
template <> __device__ __forceinline__ uint32_t narrow2<F16>(float2 r) {
    const __half2 h = __floats2half2_rn(r.x, r.y);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Mixed-precision forms of sm_100-class targets: a 16-bit element of a packed word
// used directly as an operand, widened exactly inside the instruction, so the
// results equal those of widening first.  half: 0 the low element, 1 the high one.
#define TB_FMA_MIX(TY)                                                                          \
    if (half)                                                                                   \
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t" \
            "fma.rn.f32." TY " %0, a1, b1, %3;\n\t}" : "=f"(d) : "r"(a), "r"(b), "f"(c));         \
    else                                                                                        \
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t" \
            "fma.rn.f32." TY " %0, a0, b0, %3;\n\t}" : "=f"(d) : "r"(a), "r"(b), "f"(c));
#define TB_SUB_MIX(TY)                                                                          \
    if (half)                                                                                   \
        asm("{\n\t.reg .b16 a0, a1;\n\tmov.b32 {a0, a1}, %1;\n\tsub.rn.f32." TY " %0, a1, %2;\n\t}" \
            : "=f"(d) : "r"(a), "f"(c));                                                        \
    else                                                                                        \
        asm("{\n\t.reg .b16 a0, a1;\n\tmov.b32 {a0, a1}, %1;\n\tsub.rn.f32." TY " %0, a0, %2;\n\t}" \
            : "=f"(d) : "r"(a), "f"(c));

// a*b + c and a - c for 16-bit a, b taken from a packed word
template <class Fmt> __device__ __forceinline__ float fma_mix(uint32_t a, uint32_t b, int half, float c);
template <class Fmt> __device__ __forceinline__ float sub_mix(uint32_t a, int half, float c);
template <> __device__ __forceinline__ float fma_mix<BF16>(uint32_t a, uint32_t b, int half, float c) {
    float d;
    TB_FMA_MIX("bf16")
    return d;
}
template <> __device__ __forceinline__ float fma_mix<F16>(uint32_t a, uint32_t b, int half, float c) {
    float d;
    TB_FMA_MIX("f16")
    return d;
}
template <> __device__ __forceinline__ float sub_mix<BF16>(uint32_t a, int half, float c) {
    float d;
    TB_SUB_MIX("bf16")
    return d;
}
template <> __device__ __forceinline__ float sub_mix<F16>(uint32_t a, int half, float c) {
    float d;
    TB_SUB_MIX("f16")
    return d;
}
#undef TB_FMA_MIX
#undef TB_SUB_MIX

// ------------------------------------------------------------------ group path
// G lanes per row (G divides 32), VPL vectors per lane; 256 threads per CTA.
// Number of leading columns of row r that can be nonzero: all of them for a dense
// matrix (period == 0); min(cols, r mod period + 1 + offset) under a causal mask.
__device__ __forceinline__ int64_t valid_cols(int64_t r, int64_t cols, int64_t period,
                                              int64_t offset) {
    if (period <= 0) return cols;
    const int64_t v = r % period + 1 + offset;
    return v < cols ? v : cols;
}

// Up to 4 staged vectors per input per lane (8 for fp32) three CTAs fit per SM.
template <class Fmt, int G, int VPL>
__global__ void __launch_bounds__(256, (VPL <= 4 || sizeof(typename Fmt::T) == 4) ? 3 : 2)
softmax_bwd_group_kernel(const uint4* __restrict__ dY, const uint4* __restrict__ P,
                         uint4* __restrict__ dX, int64_t rows, int nv, int64_t period,
                         int64_t offset) {
    constexpr int E = Vec<Fmt>::kElems;
    constexpr int kRowsPerWarp = 32 / G;
    // Packed f32x2 math on 16-bit rows where it measured faster and kept the
    // staged row in registers without spilling (bf16 at 8 vectors per lane,
    // fp16 at up to 4); the scalar form elsewhere.
    // fp16 rows of up to two vectors a lane: the packed form's sums (even and odd
    // elements apart) by the mixed-precision forms instead, the same values
    constexpr bool kMixEO = std::is_same<Fmt, F16>::value && VPL <= 2;
    constexpr bool kPacked = std::is_same<Fmt, BF16>::value ? VPL >= 8
                           : std::is_same<Fmt, F16>::value ? VPL <= 4 && !kMixEO : false;
    // bf16 rows of up to two vectors a lane: the dot product and dY - dot by the
    // mixed-precision forms (causal 512-column rows 0.829 -> 0.891 of the copy peak,
    // 256-column rows 0.706 -> 0.798; at four vectors a lane they measured slower)
    constexpr bool kMix = std::is_same<Fmt, BF16>::value && VPL <= 2;
    pdl_wait();      // the previous kernel has completed (programmatic launch)
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int sub = lane / G;        // row slot inside the warp
    const int gl = lane % G;         // lane inside the group
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r0 = warp * kRowsPerWarp; r0 < rows; r0 += nwarps * kRowsPerWarp) {
        const int64_t row = r0 + sub;
        const bool live = row < rows;
        const int64_t off = row * (int64_t)nv;
        // vectors holding at least one unmasked column; the rest are never read
        const int nvv = (int)((valid_cols(row, (int64_t)nv * E, period, offset) + E - 1) / E);
        uint4 p[VPL], d[VPL];
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int vi = gl + k * G;
            if (live && vi < nvv) {
                p[k] = __ldcs(P + off + vi);
                d[k] = __ldcs(dY + off + vi);
            } else {
                p[k] = make_uint4(0u, 0u, 0u, 0u);
                d[k] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        float dot = 0.f;
        if constexpr (kPacked) {
            // packed pairs of fp32 math on the widened 16-bit values
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const uint32_t pw[4] = {p[k].x, p[k].y, p[k].z, p[k].w};
                const uint32_t dw[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) acc = __ffma2_rn(widen_a<Fmt>(pw[q]), widen_a<Fmt>(dw[q]), acc);
            }
            dot = acc.x + acc.y;
        } else if constexpr (kMix) {
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const uint32_t pw[4] = {p[k].x, p[k].y, p[k].z, p[k].w};
                const uint32_t dw[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
#pragma unroll
                for (int e = 0; e < E; ++e) dot = fma_mix<Fmt>(pw[e / 2], dw[e / 2], e & 1, dot);
            }
        } else if constexpr (kMixEO) {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const uint32_t pw[4] = {p[k].x, p[k].y, p[k].z, p[k].w};
                const uint32_t dw[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    s0 = fma_mix<Fmt>(pw[w], dw[w], 0, s0);
                    s1 = fma_mix<Fmt>(pw[w], dw[w], 1, s1);
                }
            }
            dot = s0 + s1;
        } else {
#pragma unroll
            for (int k = 0; k < VPL; ++k)
#pragma unroll
                for (int e = 0; e < E; ++e) dot += vec_elem<Fmt>(p[k], e) * vec_elem<Fmt>(d[k], e);
        }
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o, G);
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int vi = gl + k * G;
            if (live && vi < nvv) {
                if constexpr (kPacked) {
                    // widened again (bf16: with byte permutes, so the values of the first
                    // pass are not kept alive across the reduction)
                    const uint32_t pw[4] = {p[k].x, p[k].y, p[k].z, p[k].w};
                    const uint32_t dw[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
                    const float2 ndot = make_float2(-dot, -dot);
                    uint32_t o[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 r = __fmul2_rn(widen_b<Fmt>(pw[q]), __fadd2_rn(widen_b<Fmt>(dw[q]), ndot));
                        o[q] = narrow2<Fmt>(r);
                    }
                    __stcs(dX + off + vi, make_uint4(o[0], o[1], o[2], o[3]));
                } else {
                    float out[E];
                    if constexpr (kMix || kMixEO) {
                        const uint32_t dw[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            out[e] = vec_elem<Fmt>(p[k], e) * sub_mix<Fmt>(dw[e / 2], e & 1, dot);
                    } else {
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            out[e] = vec_elem<Fmt>(p[k], e) * (vec_elem<Fmt>(d[k], e) - dot);
                    }
                    __stcs(dX + off + vi, vec_from<Fmt>(out));
                }
            } else if (live && vi < nv) {
                __stcs(dX + off + vi, make_uint4(0u, 0u, 0u, 0u));   // masked: dX = +0
            }
        }
    }
}

// ------------------------------------------------------------------ folded causal pairs
// 16-bit causal rows of 65..256 vectors.  Inside one causal block of `period` rows,
// row q opens min(cols, q + 1 + offset) columns and row period-1-q opens
// min(cols, period - q + offset): the two together open about period + 1 + 2 offset
// columns wherever q lies.  A warp takes such a pair, so every warp keeps about the
// same number of loads in flight; with one row per warp, the warps on the short rows
// of a block issue a load or two each and wait.  Lane l holds vectors l, l + 32, ...
// of the first row in its first slots and the same vectors of the second row in the
// slots after them: each row is summed in the order of the one-row-per-warp kernel
// (and of the dense kernel, whose extra terms are exact zeros), so the results are
// the same bit for bit.  The masked vectors of both rows are written as +0 right after
// the loads are issued, while they are in flight (here that measured faster than
// writing them after the dot products; in the one-row kernel it measured slower).
// An odd period leaves the middle row without a partner; rows past `rows` in a last,
// partial block are skipped.  VPL >= ceil(na / 32) + ceil(nb / 32) for every pair
// (checked on the host); a larger pair would lose vectors, never touch other memory.
// kEvenOdd: a lane sums even and odd elements apart and adds the two at the end, the
// order of the one-row kernel's packed pairs (bf16 rows of more than 128 vectors, fp16
// rows of up to 128); otherwise one running sum.
template <class Fmt, int VPL, bool kEvenOdd>
__global__ void __launch_bounds__(256, VPL <= 6 ? 3 : 2)
softmax_bwd_causal_pair_kernel(const uint4* __restrict__ dY, const uint4* __restrict__ P,
                               uint4* __restrict__ dX, int64_t rows, int nv, int64_t period,
                               int64_t offset, int64_t npairs) {
    constexpr int E = Vec<Fmt>::kElems;
    static_assert(E == 8, "16-bit rows only");
    pdl_wait();      // the previous kernel has completed (programmatic launch)
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t per_block = (period + 1) / 2;
    const int64_t cols = (int64_t)nv * E;
    for (int64_t pi = warp; pi < npairs; pi += nwarps) {
        const int64_t blk = pi / per_block;
        const int64_t q = pi - blk * per_block;
        const int64_t ra = blk * period + q;
        const int64_t rb = blk * period + (period - 1 - q);
        const bool live_a = ra < rows;
        const bool live_b = rb != ra && rb < rows;
        const int64_t ca = q + 1 + offset, cb = period - q + offset;
        const int na = live_a ? (int)(((ca < cols ? ca : cols) + E - 1) / E) : 0;
        const int nb = live_b ? (int)(((cb < cols ? cb : cols) + E - 1) / E) : 0;
        const int ka = (na + 31) >> 5;                  // slots of row a (warp-uniform)
        const int64_t offa = ra * (int64_t)nv;
        const int64_t offb = rb * (int64_t)nv;
        uint4 p[VPL], d[VPL];
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const bool in_a = k < ka;
            const int v = lane + 32 * (in_a ? k : k - ka);
            if (v < (in_a ? na : nb)) {
                const int64_t o = (in_a ? offa : offb) + v;
                p[k] = __ldcs(P + o);
                d[k] = __ldcs(dY + o);
            } else {
                p[k] = make_uint4(0u, 0u, 0u, 0u);
                d[k] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        // masked vectors, row a's [na, nv) then row b's [nb, nv), written as +0 while
        // the loads are in flight (they depend on none of them)
        {
            const int ma = live_a ? nv - na : 0;
            const int mb = live_b ? nv - nb : 0;
            uint4* const za = live_a ? dX + offa + na : dX;
            uint4* const zb = live_b ? dX + offb + nb - ma : dX;   // index j >= ma: zb + j
#pragma unroll 2
            for (int j = lane; j < ma + mb; j += 32)
                __stcs((j < ma ? za : zb) + j, make_uint4(0u, 0u, 0u, 0u));
        }
        float da = 0.f, db = 0.f;
        // the mixed-precision forms: 16-bit operands, fp32 sums (the packed pairs'
        // order is two such sums, even and odd elements, with the same values as
        // packed fp32 math on the widened elements)
        if constexpr (kEvenOdd) {
            float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const bool in_a = k < ka;
                float s0 = in_a ? a0 : b0, s1 = in_a ? a1 : b1;
                const uint32_t pw[4] = {p[k].x, p[k].y, p[k].z, p[k].w};
                const uint32_t dw[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    s0 = fma_mix<Fmt>(pw[w], dw[w], 0, s0);
                    s1 = fma_mix<Fmt>(pw[w], dw[w], 1, s1);
                }
                if (in_a) { a0 = s0; a1 = s1; } else { b0 = s0; b1 = s1; }
            }
            da = a0 + a1;
            db = b0 + b1;
        } else {
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const bool in_a = k < ka;
                float acc = in_a ? da : db;
                const uint32_t pw[4] = {p[k].x, p[k].y, p[k].z, p[k].w};
                const uint32_t dw[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
#pragma unroll
                for (int e = 0; e < E; ++e) acc = fma_mix<Fmt>(pw[e / 2], dw[e / 2], e & 1, acc);
                if (in_a) da = acc; else db = acc;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            da += __shfl_xor_sync(0xffffffffu, da, o);
            db += __shfl_xor_sync(0xffffffffu, db, o);
        }
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const bool in_a = k < ka;
            const int v = lane + 32 * (in_a ? k : k - ka);
            if (v < (in_a ? na : nb)) {
                const float dot = in_a ? da : db;
                const uint32_t pw[4] = {p[k].x, p[k].y, p[k].z, p[k].w};
                const uint32_t dw[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
                uint32_t o4[4];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float2 pf = widen_a<Fmt>(pw[w]);
                    o4[w] = narrow2<Fmt>(make_float2(pf.x * sub_mix<Fmt>(dw[w], 0, dot),
                                                     pf.y * sub_mix<Fmt>(dw[w], 1, dot)));
                }
                __stcs(dX + (in_a ? offa : offb) + v, make_uint4(o4[0], o4[1], o4[2], o4[3]));
            }
        }
    }
}

// ------------------------------------------------------------------ CTA path
// One CTA of T threads per row, T the smallest of 128, 256 and 512 that holds the row
// in at most four vectors a thread: with 512 threads on every row, rows of 257..384
// vectors left a quarter or more of the threads idle and rows of 513..1024 vectors ran
// at one or two vectors a thread (bf16 2,056 columns 0.73 of the copy peak, 6,144 0.87;
// with CTAs sized to the row 0.99 and 1.00).  16-bit rows take the mixed-precision
// forms (fewer registers than widening first, the same values); launch bounds hold
// 64 registers a thread, so 2..8 CTAs fit per SM.
template <class Fmt, int T, int VPL>
__global__ void __launch_bounds__(T, 65536 / (T * 64))
softmax_bwd_cta_kernel(const uint4* __restrict__ dY, const uint4* __restrict__ P,
                       uint4* __restrict__ dX, int64_t rows, int nv, int64_t period,
                       int64_t offset) {
    constexpr int E = Vec<Fmt>::kElems;
    constexpr int kWarps = T / 32;
    __shared__ float red[2][kWarps];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    int parity = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, parity ^= 1) {
        const int64_t off = row * (int64_t)nv;
        const int nvv = (int)((valid_cols(row, (int64_t)nv * E, period, offset) + E - 1) / E);
        uint4 p[VPL], d[VPL];
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int vi = tid + k * T;
            if (vi < nvv) {
                p[k] = __ldcs(P + off + vi);
                d[k] = __ldcs(dY + off + vi);
            } else {
                p[k] = make_uint4(0u, 0u, 0u, 0u);
                d[k] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            if constexpr (E == 8) {
                const uint32_t pw[4] = {p[k].x, p[k].y, p[k].z, p[k].w};
                const uint32_t dw[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
#pragma unroll
                for (int e = 0; e < E; ++e) dot = fma_mix<Fmt>(pw[e / 2], dw[e / 2], e & 1, dot);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) dot += vec_elem<Fmt>(p[k], e) * vec_elem<Fmt>(d[k], e);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (lane == 0) red[parity][wid] = dot;
        __syncthreads();   // one barrier per row: the other buffer is reused two rows later
        dot = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) dot += red[parity][w];
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int vi = tid + k * T;
            if (vi < nvv) {
                float out[E];
                if constexpr (E == 8) {
                    const uint32_t dw[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
#pragma unroll
                    for (int e = 0; e < E; ++e) out[e] = vec_elem<Fmt>(p[k], e) * sub_mix<Fmt>(dw[e / 2], e & 1, dot);
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        out[e] = vec_elem<Fmt>(p[k], e) * (vec_elem<Fmt>(d[k], e) - dot);
                }
                __stcs(dX + off + vi, vec_from<Fmt>(out));
            } else if (vi < nv) {
                __stcs(dX + off + vi, make_uint4(0u, 0u, 0u, 0u));
            }
        }
    }
}

// Folded pairs on the CTA path: causal rows of 257..2048 vectors (16-bit rows of
// 2,056..16,384 columns, fp32 rows of 1,028..8,192) whose causal block fits in the
// rows.  One CTA of T threads (128 or 256 with up to six slots a thread, 256 with up
// to ten at two CTAs per SM, else 512 with six) takes rows q and period-1-q of a
// block, as the warp version above does, so every CTA streams about one row's worth
// per pair.  With one row per 512-thread CTA, most of a CTA's threads load nothing on
// a block's short rows and wait at the barrier; smaller CTAs let several pairs per SM
// overlap one another's barrier and loads.  Thread t holds vectors t, t + T, ... of
// the first row in its first slots and the same vectors of the second row after them,
// sums them in order, then each warp's butterfly and the warp sums in warp order: the
// one-row CTA kernel's order at the same T, so where both pick the same CTA size the
// results equal the dense kernel's bit for bit, and elsewhere the same terms are
// grouped differently.  Masked vectors are written as +0 while the loads are in
// flight; one barrier per pair.  Launch bounds hold 2, 4, 6 and 8..10 slots to 32,
// 64, 85 and 128 registers a thread.
constexpr int cta_pair_regs(int VPL) { return VPL <= 2 ? 32 : VPL <= 4 ? 64 : VPL <= 6 ? 85 : 128; }
constexpr int cta_pair_min_blocks(int T, int VPL) {
    return 65536 / (T * cta_pair_regs(VPL)) > 0 ? 65536 / (T * cta_pair_regs(VPL)) : 1;
}

template <class Fmt, int T, int VPL>
__global__ void __launch_bounds__(T, cta_pair_min_blocks(T, VPL))
softmax_bwd_causal_cta_pair_kernel(const uint4* __restrict__ dY, const uint4* __restrict__ P,
                                   uint4* __restrict__ dX, int64_t rows, int nv, int64_t period,
                                   int64_t offset, int64_t npairs) {
    constexpr int E = Vec<Fmt>::kElems;
    constexpr bool k16 = E == 8;     // 16-bit rows: the mixed-precision forms
    constexpr int kWarps = T / 32;
    __shared__ float red[2][2][kWarps];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int64_t per_block = (period + 1) / 2;
    const int64_t cols = (int64_t)nv * E;
    int parity = 0;
    for (int64_t pi = blockIdx.x; pi < npairs; pi += gridDim.x, parity ^= 1) {
        const int64_t blk = pi / per_block;
        const int64_t q = pi - blk * per_block;
        const int64_t ra = blk * period + q;
        const int64_t rb = blk * period + (period - 1 - q);
        const bool live_a = ra < rows;
        const bool live_b = rb != ra && rb < rows;
        const int64_t ca = q + 1 + offset, cb = period - q + offset;
        const int na = live_a ? (int)(((ca < cols ? ca : cols) + E - 1) / E) : 0;
        const int nb = live_b ? (int)(((cb < cols ? cb : cols) + E - 1) / E) : 0;
        const int ka = (na + T - 1) / T;   // slots of row a (CTA-uniform)
        const int64_t offa = ra * (int64_t)nv;
        const int64_t offb = rb * (int64_t)nv;
        uint4 p[VPL], d[VPL];
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const bool in_a = k < ka;
            const int v = tid + T * (in_a ? k : k - ka);
            if (v < (in_a ? na : nb)) {
                const int64_t o = (in_a ? offa : offb) + v;
                p[k] = __ldcs(P + o);
                d[k] = __ldcs(dY + o);
            } else {
                p[k] = make_uint4(0u, 0u, 0u, 0u);
                d[k] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        {   // masked vectors, row a's [na, nv) then row b's [nb, nv)
            const int ma = live_a ? nv - na : 0;
            const int mb = live_b ? nv - nb : 0;
            uint4* const za = live_a ? dX + offa + na : dX;
            uint4* const zb = live_b ? dX + offb + nb - ma : dX;   // index j >= ma: zb + j
            for (int j = tid; j < ma + mb; j += T)
                __stcs((j < ma ? za : zb) + j, make_uint4(0u, 0u, 0u, 0u));
        }
        float da = 0.f, db = 0.f;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const bool in_a = k < ka;
            float acc = in_a ? da : db;
            if constexpr (k16) {
                const uint32_t pw[4] = {p[k].x, p[k].y, p[k].z, p[k].w};
                const uint32_t dw[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
#pragma unroll
                for (int e = 0; e < E; ++e) acc = fma_mix<Fmt>(pw[e / 2], dw[e / 2], e & 1, acc);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) acc = fmaf(vec_elem<Fmt>(p[k], e), vec_elem<Fmt>(d[k], e), acc);
            }
            if (in_a) da = acc; else db = acc;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            da += __shfl_xor_sync(0xffffffffu, da, o);
            db += __shfl_xor_sync(0xffffffffu, db, o);
        }
        if (lane == 0) {
            red[parity][0][wid] = da;
            red[parity][1][wid] = db;
        }
        __syncthreads();   // one barrier per pair: the other buffer is reused two pairs later
        da = 0.f;
        db = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            da += red[parity][0][w];
            db += red[parity][1][w];
        }
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const bool in_a = k < ka;
            const int v = tid + T * (in_a ? k : k - ka);
            if (v < (in_a ? na : nb)) {
                const float dot = in_a ? da : db;
                float out[E];
                if constexpr (k16) {
                    const uint32_t dw[4] = {d[k].x, d[k].y, d[k].z, d[k].w};
#pragma unroll
                    for (int e = 0; e < E; ++e) out[e] = vec_elem<Fmt>(p[k], e) * sub_mix<Fmt>(dw[e / 2], e & 1, dot);
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) out[e] = vec_elem<Fmt>(p[k], e) * (vec_elem<Fmt>(d[k], e) - dot);
                }
                __stcs(dX + (in_a ? offa : offb) + v, vec_from<Fmt>(out));
            }
        }
    }
}

// ------------------------------------------------------------------ two-pass path
constexpr int kTwoPassThreads = 256;

template <class Fmt>
__global__ void __launch_bounds__(kTwoPassThreads)
softmax_bwd_twopass_kernel(const typename Fmt::T* __restrict__ dY,
                           const typename Fmt::T* __restrict__ P,
                           typename Fmt::T* __restrict__ dX, int64_t rows, int64_t cols,
                           int64_t period, int64_t offset) {
    constexpr int kWarps = kTwoPassThreads / 32;
    __shared__ float red[2][kWarps];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    int parity = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, parity ^= 1) {
        const int64_t off = row * cols;
        const int64_t nvalid = valid_cols(row, cols, period, offset);
        float dot = 0.f;
        for (int64_t j = tid; j < nvalid; j += kTwoPassThreads)
            dot += Fmt::to_f32(P[off + j]) * Fmt::to_f32(dY[off + j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (lane == 0) red[parity][wid] = dot;
        __syncthreads();
        dot = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) dot += red[parity][w];
        for (int64_t j = tid; j < cols; j += kTwoPassThreads) {
            if (j < nvalid) {
                const float p = Fmt::to_f32(P[off + j]);
                dX[off + j] = Fmt::from_f32(p * (Fmt::to_f32(dY[off + j]) - dot));
            } else {
                dX[off + j] = Fmt::from_f32(0.0f);
            }
        }
    }
}

// ------------------------------------------------------------------ dispatch
// Grid shape.  A persistent grid (SM count x resident CTAs, grid-striding over the
// rows) gives every warp a fixed share of the rows, and the SMs of a GB300 do not
// stream at one rate: the CTAs of a persistent fp32 softmax at 98,304 x 1,024 end
// over a window of 70 us of a 185 us launch.  One CTA per row group instead lets the
// hardware scheduler hand the next group to whichever SM has room, so a faster SM
// simply runs more of them (185 -> 170 us there; every row is independent, so the
// results are the same bit for bit).  That pays only while a CTA carries enough
// traffic to cover its own launch: below about 40 KB per CTA (bf16 causal rows of
// 1,024 columns, half of them masked) the persistent grid measured faster.
constexpr double kOneShotCtaBytes = 40.0 * 1024;

// Mean number of open (readable) columns per row: all of them for a dense matrix;
// under the causal mask the mean over one period of min(cols, q + 1 + offset).
double mean_open_cols(int64_t cols, int64_t period, int64_t offset) {
    if (period <= 0) return (double)cols;
    // q + 1 + offset reaches cols at q = cols - 1 - offset
    const int64_t ramp = std::max<int64_t>(0, std::min<int64_t>(period, cols - 1 - offset));
    // q in [0, ramp): q + 1 + offset; q in [ramp, period): cols
    const double sum_ramp = (double)ramp * (double)(1 + offset) + (double)ramp * (double)(ramp - 1) / 2.0;
    return (sum_ramp + (double)(period - ramp) * (double)cols) / (double)period;
}

// CTAs for `want` row groups of `rows_per_cta` rows each: one per group when a CTA's
// estimated traffic (reads of the open columns of P and dY, writes of all of dX)
// reaches kOneShotCtaBytes, else a persistent grid.
int64_t grid_for(int64_t want, int64_t rows_per_cta, int64_t cols, int64_t period, int64_t offset,
                 size_t es, int sms, int per_sm) {
    const double cta_bytes = (double)rows_per_cta * (double)es *
                             (2.0 * mean_open_cols(cols, period, offset) + (double)cols);
    // (the kernels grid-stride, so a grid capped at the launch limit still covers every row)
    if (cta_bytes >= kOneShotCtaBytes) return std::max<int64_t>(1, std::min<int64_t>(want, INT32_MAX));
    return std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sms * per_sm));
}

template <class Fmt, int G, int VPL>
tb_status launch_group(const void* dY, const void* P, void* dX, int64_t rows, int nv,
                       int64_t period, int64_t offset, int sms, cudaStream_t st) {
    constexpr int kRowsPerCta = 256 / G;
    const int per_sm = resident_ctas_per_sm(
        reinterpret_cast<const void*>(&softmax_bwd_group_kernel<Fmt, G, VPL>), 256, 0);
    if (per_sm == 0) return TB_ERR_CUDA;
    const int64_t want = (rows + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t grid = grid_for(want, kRowsPerCta, (int64_t)nv * Vec<Fmt>::kElems, period, offset,
                                  sizeof(typename Fmt::T), sms, per_sm);
    if (launch_pdl(softmax_bwd_group_kernel<Fmt, G, VPL>, dim3((unsigned)grid), dim3(256), 0, st,
                   static_cast<const uint4*>(dY), static_cast<const uint4*>(P),
                   static_cast<uint4*>(dX), rows, nv, period, offset) != cudaSuccess)
        return TB_ERR_CUDA;
    return launch_status();
}

// Slots a thread needs for one folded pair whose vectors are dealt over `lanes`
// threads, at most: with na + nb <= period + 1 + 2 offset open vectors
// (ceil(a/E) + ceil(b/E) <= ceil((a+b)/E) + 1), ceil(na/lanes) + ceil(nb/lanes) <=
// ceil((na+nb)/lanes) + 1; and never more than two whole rows' worth.  (Called with
// period <= rows and offset <= cols: nothing overflows.)
int64_t pair_slots(int64_t nv, int E, int64_t period, int64_t offset, int64_t lanes = 32) {
    const int64_t vec = (period + 1 + 2 * offset + E - 1) / E + 1;
    return std::min<int64_t>(2 * ((nv + lanes - 1) / lanes), (vec + lanes - 1) / lanes + 1);
}

template <class Fmt, int VPL, bool kEvenOdd>
tb_status launch_pair_vpl(const void* dY, const void* P, void* dX, int64_t rows, int nv,
                      int64_t period, int64_t offset, int sms, cudaStream_t st) {
    constexpr int kPairsPerCta = 8;                 // one pair per warp
    const int per_sm = resident_ctas_per_sm(
        reinterpret_cast<const void*>(&softmax_bwd_causal_pair_kernel<Fmt, VPL, kEvenOdd>), 256, 0);
    if (per_sm == 0) return TB_ERR_CUDA;
    const int64_t npairs = ((rows + period - 1) / period) * ((period + 1) / 2);
    const int64_t want = (npairs + kPairsPerCta - 1) / kPairsPerCta;
    const int64_t grid = grid_for(want, 2 * kPairsPerCta, (int64_t)nv * Vec<Fmt>::kElems, period,
                                  offset, sizeof(typename Fmt::T), sms, per_sm);
    if (launch_pdl(softmax_bwd_causal_pair_kernel<Fmt, VPL, kEvenOdd>, dim3((unsigned)grid), dim3(256), 0, st,
                   static_cast<const uint4*>(dY), static_cast<const uint4*>(P),
                   static_cast<uint4*>(dX), rows, nv, period, offset, npairs) != cudaSuccess)
        return TB_ERR_CUDA;
    return launch_status();
}

// The smallest instance with at least k slots a lane (k <= 10).
template <class Fmt, bool kEvenOdd>
tb_status launch_pair(int64_t k, const void* dY, const void* P, void* dX, int64_t rows, int nv,
                      int64_t period, int64_t offset, int sms, cudaStream_t st) {
    if (k <= 4) return launch_pair_vpl<Fmt, 4, kEvenOdd>(dY, P, dX, rows, nv, period, offset, sms, st);
    if (k <= 6) return launch_pair_vpl<Fmt, 6, kEvenOdd>(dY, P, dX, rows, nv, period, offset, sms, st);
    return launch_pair_vpl<Fmt, 10, kEvenOdd>(dY, P, dX, rows, nv, period, offset, sms, st);
}

template <class Fmt, int T, int VPL>
tb_status launch_cta_pair_vpl(const void* dY, const void* P, void* dX, int64_t rows, int nv,
                              int64_t period, int64_t offset, int sms, cudaStream_t st) {
    const int per_sm = resident_ctas_per_sm(
        reinterpret_cast<const void*>(&softmax_bwd_causal_cta_pair_kernel<Fmt, T, VPL>), T, 0);
    if (per_sm == 0) return TB_ERR_CUDA;
    const int64_t npairs = ((rows + period - 1) / period) * ((period + 1) / 2);
    // one CTA per pair, whatever its traffic: against the persistent grid the 40 KB rule
    // would pick, bf16 4,096-column causal rows went from 0.90 to 0.99 of the copy peak,
    // 2,560 columns from 0.91 to 0.98, fp32 2,048 from 0.91 to 0.99
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(npairs, INT32_MAX));
    (void)sms;
    if (launch_pdl(softmax_bwd_causal_cta_pair_kernel<Fmt, T, VPL>, dim3((unsigned)grid), dim3(T),
                   0, st, static_cast<const uint4*>(dY), static_cast<const uint4*>(P),
                   static_cast<uint4*>(dX), rows, nv, period, offset, npairs) != cudaSuccess)
        return TB_ERR_CUDA;
    return launch_status();
}

// The instance of T threads with the fewest slots a thread, at least k: 2..6 slots at
// T = 128, 4..10 at T = 256, 6 at T = 512 (a pair that fits fewer slots of a larger CTA
// fits a smaller CTA, which the host prefers).
template <class Fmt, int T>
tb_status launch_cta_pair_t(int64_t k, const void* dY, const void* P, void* dX, int64_t rows, int nv,
                            int64_t period, int64_t offset, int sms, cudaStream_t st) {
    if constexpr (T == 128) {
        if (k <= 2) return launch_cta_pair_vpl<Fmt, T, 2>(dY, P, dX, rows, nv, period, offset, sms, st);
        if (k <= 4) return launch_cta_pair_vpl<Fmt, T, 4>(dY, P, dX, rows, nv, period, offset, sms, st);
        return launch_cta_pair_vpl<Fmt, T, 6>(dY, P, dX, rows, nv, period, offset, sms, st);
    } else if constexpr (T == 256) {
        if (k <= 4) return launch_cta_pair_vpl<Fmt, T, 4>(dY, P, dX, rows, nv, period, offset, sms, st);
        if (k <= 6) return launch_cta_pair_vpl<Fmt, T, 6>(dY, P, dX, rows, nv, period, offset, sms, st);
        if (k <= 8) return launch_cta_pair_vpl<Fmt, T, 8>(dY, P, dX, rows, nv, period, offset, sms, st);
        return launch_cta_pair_vpl<Fmt, T, 10>(dY, P, dX, rows, nv, period, offset, sms, st);
    } else {
        return launch_cta_pair_vpl<Fmt, T, 6>(dY, P, dX, rows, nv, period, offset, sms, st);
    }
}

template <class Fmt, int T, int VPL>
tb_status launch_cta(const void* dY, const void* P, void* dX, int64_t rows, int nv,
                     int64_t period, int64_t offset, int sms, cudaStream_t st) {
    const int per_sm = resident_ctas_per_sm(
        reinterpret_cast<const void*>(&softmax_bwd_cta_kernel<Fmt, T, VPL>), T, 0);
    if (per_sm == 0) return TB_ERR_CUDA;
    const int64_t grid = grid_for(rows, 1, (int64_t)nv * Vec<Fmt>::kElems, period, offset,
                                  sizeof(typename Fmt::T), sms, per_sm);
    if (launch_pdl(softmax_bwd_cta_kernel<Fmt, T, VPL>, dim3((unsigned)grid), dim3(T), 0, st,
                   static_cast<const uint4*>(dY), static_cast<const uint4*>(P),
                   static_cast<uint4*>(dX), rows, nv, period, offset) != cudaSuccess)
        return TB_ERR_CUDA;
    return launch_status();
}

template <class Fmt>
tb_status dispatch(const void* dY, const void* P, void* dX, int64_t rows, int64_t cols,
                   int64_t period, int64_t offset, bool aligned, int sms, cudaStream_t st) {
    constexpr int E = Vec<Fmt>::kElems;
    if (aligned && cols % E == 0 && cols / E <= 2048) {
        const int nv = (int)(cols / E);
        if constexpr (sizeof(typename Fmt::T) == 2) {
            // causal blocks that fit in the rows, rows of 65..256 vectors: folded pairs,
            // one per warp, at the occupancy of the one-row kernel there (3 CTAs per SM
            // up to 6 slots a lane, 2 beyond).  Shorter rows run the one-row kernel at
            // up to five CTAs per SM, which measured faster than pairs.
            if (period > 0 && period <= rows && nv > 64 && nv <= 256) {
                const int64_t k = pair_slots(nv, E, period, offset);
                // the one-row kernel's sum order: even and odd elements apart where it
                // takes packed pairs (bf16 rows of more than 128 vectors, fp16 rows of
                // up to 128), else one running sum
                const bool eo = std::is_same<Fmt, BF16>::value ? nv > 128 : nv <= 128;
                if (k <= 6 || (nv > 128 && k <= 10))
                    return eo ? launch_pair<Fmt, true>(k, dY, P, dX, rows, nv, period, offset, sms, st)
                              : launch_pair<Fmt, false>(k, dY, P, dX, rows, nv, period, offset, sms, st);
            }
        }
        if (nv <= 4) return launch_group<Fmt, 4, 1>(dY, P, dX, rows, nv, period, offset, sms, st);
        if (nv <= 8) return launch_group<Fmt, 8, 1>(dY, P, dX, rows, nv, period, offset, sms, st);
        if (nv <= 16) return launch_group<Fmt, 16, 1>(dY, P, dX, rows, nv, period, offset, sms, st);
        if (nv <= 32) return launch_group<Fmt, 32, 1>(dY, P, dX, rows, nv, period, offset, sms, st);
        if (nv <= 64) return launch_group<Fmt, 32, 2>(dY, P, dX, rows, nv, period, offset, sms, st);
        if (nv <= 128) return launch_group<Fmt, 32, 4>(dY, P, dX, rows, nv, period, offset, sms, st);
        if (nv <= 256) return launch_group<Fmt, 32, 8>(dY, P, dX, rows, nv, period, offset, sms, st);
        // causal rows whose causal blocks fit in the rows: folded pairs, one per CTA of
        // the fewest threads that need at most six slots each (128) or ten (256)
        if (period > 0 && period <= rows) {
            int64_t k = pair_slots(nv, E, period, offset, 128);
            if (k <= 6) return launch_cta_pair_t<Fmt, 128>(k, dY, P, dX, rows, nv, period, offset, sms, st);
            k = pair_slots(nv, E, period, offset, 256);
            if (k <= 10) return launch_cta_pair_t<Fmt, 256>(k, dY, P, dX, rows, nv, period, offset, sms, st);
            k = pair_slots(nv, E, period, offset, 512);
            if (k <= 6) return launch_cta_pair_t<Fmt, 512>(k, dY, P, dX, rows, nv, period, offset, sms, st);
        }
        if (nv <= 384) return launch_cta<Fmt, 128, 3>(dY, P, dX, rows, nv, period, offset, sms, st);
        if (nv <= 512) return launch_cta<Fmt, 128, 4>(dY, P, dX, rows, nv, period, offset, sms, st);
        if (nv <= 768) return launch_cta<Fmt, 256, 3>(dY, P, dX, rows, nv, period, offset, sms, st);
        if (nv <= 1024) return launch_cta<Fmt, 256, 4>(dY, P, dX, rows, nv, period, offset, sms, st);
        if (nv <= 1536) return launch_cta<Fmt, 512, 3>(dY, P, dX, rows, nv, period, offset, sms, st);
        return launch_cta<Fmt, 512, 4>(dY, P, dX, rows, nv, period, offset, sms, st);
    }
    using T = typename Fmt::T;
    const int per_sm = resident_ctas_per_sm(
        reinterpret_cast<const void*>(&softmax_bwd_twopass_kernel<Fmt>), kTwoPassThreads, 0);
    if (per_sm == 0) return TB_ERR_CUDA;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(rows, (int64_t)sms * per_sm));
    if (launch_pdl(softmax_bwd_twopass_kernel<Fmt>, dim3((unsigned)grid), dim3(kTwoPassThreads), 0,
                   st, static_cast<const T*>(dY), static_cast<const T*>(P), static_cast<T*>(dX),
                   rows, cols, period, offset) != cudaSuccess)
        return TB_ERR_CUDA;
    return launch_status();
}

}  // namespace
}  // namespace tb

namespace tb {
namespace {
tb_status softmax_bwd_entry(const void* dY, const void* P, void* dX, int64_t rows, int64_t cols,
                            int64_t period, int64_t offset, tb_dtype dtype, void* stream) {
    if (rows < 0 || cols < 0 || period < 0 || offset < 0) return TB_ERR_INVALID_VALUE;
    if (!dtype_valid(dtype)) return TB_ERR_UNSUPPORTED_DTYPE;
    if (rows == 0 || cols == 0) return TB_OK;
    if (!dY || !P || !dX) return TB_ERR_INVALID_VALUE;
    if (cols > INT64_MAX / rows / 4) return TB_ERR_INVALID_VALUE;
    // An offset of cols or more opens every column: clamp it so that the kernels'
    // r mod period + 1 + offset cannot overflow.
    if (offset > cols) offset = cols;
    const size_t es = dtype_size(dtype);
    if (!aligned_to(dY, es) || !aligned_to(P, es) || !aligned_to(dX, es)) return TB_ERR_MISALIGNED;
    const int64_t n = rows * cols;
    const Range out = range_of(dX, n, es);
    if (overlap(out, range_of(dY, n, es)) || overlap(out, range_of(P, n, es))) return TB_ERR_ALIAS;
    int dev = 0;
    DeviceInfo info{};
    if (!current_device_info(&dev, &info)) return TB_ERR_CUDA;
    const bool aligned = aligned_to(dY, 16) && aligned_to(P, 16) && aligned_to(dX, 16) &&
                         (cols * (int64_t)es) % 16 == 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dtype) {
        case TB_F32: return dispatch<F32>(dY, P, dX, rows, cols, period, offset, aligned, info.sm_count, st);
        case TB_BF16: return dispatch<BF16>(dY, P, dX, rows, cols, period, offset, aligned, info.sm_count, st);
        default: return dispatch<F16>(dY, P, dX, rows, cols, period, offset, aligned, info.sm_count, st);
    }
}
}  // namespace
}  // namespace tb

extern "C" tb_status tb_softmax_bwd(const void* dY, const void* P, void* dX, int64_t rows,
                                    int64_t cols, tb_dtype dtype, void* stream) {
    return tb::softmax_bwd_entry(dY, P, dX, rows, cols, 0, 0, dtype, stream);
}

extern "C" tb_status tb_softmax_bwd_causal(const void* dY, const void* P, void* dX, int64_t rows,
                                           int64_t cols, int64_t period, int64_t offset,
                                           tb_dtype dtype, void* stream) {
    if (period < 1) return TB_ERR_INVALID_VALUE;
    return tb::softmax_bwd_entry(dY, P, dX, rows, cols, period, offset, dtype, stream);
}
