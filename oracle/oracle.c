/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for the memory-bound half
 * of an LLM training step: the fused mixed-precision AdamW update, the row-wise
 * softmax backward, the LayerNorm backward and the RMSNorm backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file.  Its users are the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark.  It shares no code, header, table or helper with the
 * CUDA library: it has its own 16-bit float codecs, its own loops, its own
 * constants.
 *
 * Sources (web pages on the subject; cited as page title + section):
 *   [GPU-Opt-P2]  "GPU 优化实战 Part 2：用 CUDA/ROCm 实现 LLM 反向传播与训练循环"
 *   [Mastering]   "Mastering LLM Training with CUDA and ROCm: The Backpropagation
 *                  and Optimization Workflow"
 *
 * Every function is the plain definition of what it computes, written out
 * element by element or row by row, with no blocking, fusion or reordering
 * beyond what that definition states.  Two precisions exist for each method:
 *   *_f64  -- the definition evaluated in double precision (the accuracy
 *             yardstick the GPU is compared against);
 *   *_f32  -- the same steps in IEEE single precision, one rounding per
 *             operation, in the order the pages' fp32 kernels use (compiled
 *             with -ffp-contract=off so no multiply-add is fused).
 *
 * Readings taken where the pages are silent or disagree:
 *   - Weight decay SUBTRACTS eta*lambda*theta_t, taken on the pre-update theta
 *     ([Mastering] §"AdamW Algorithm" update rule; its CPU listing adds it,
 *     which contradicts its own equation and [GPU-Opt-P2]).
 *   - epsilon is added outside the square root (both pages).
 *   - Bias corrections 1-beta^t use the global step t >= 1; they are formed in
 *     double from the fp32 beta and (for the fp32 variant) rounded to fp32.
 *   - Gradients are unscaled by multiplying with 1/loss_scale
 *     ([GPU-Opt-P2] §"混合精度训练（FP16 / BF16）").
 *   - LayerNorm gamma/beta gradients reduce over ROWS (tokens), per column
 *     ([GPU-Opt-P2] §2.2 says "hidden dimension", which is the wrong axis for a
 *     per-feature scale); variance is the biased one and eps sits inside the
 *     square root, so eps enters the backward only through the saved inv_std.
 *
 * Parity pins for every function live in tests/test_oracle_*.py: closed forms,
 * invariants, finite differences and library cross-checks in float64.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <fenv.h>

#define ORC_F32 0
#define ORC_F16 1
#define ORC_BF16 2

/* ------------------------------------------------------------------------- */
/* 16-bit float codecs, written from the IEEE-754 binary16 and bfloat16 bit   */
/* layouts (sign | exponent | fraction).                                      */
/* ------------------------------------------------------------------------- */

/* Layout parameters of the two 16-bit formats. */
typedef struct {
    int frac_bits;  /* stored fraction bits */
    int exp_bits;   /* exponent field width */
    int bias;       /* exponent bias */
} orc_fmt;

static orc_fmt orc_format(int kind)
{
    orc_fmt f;
    if (kind == ORC_F16) { f.frac_bits = 10; f.exp_bits = 5; f.bias = 15; }
    else                 { f.frac_bits = 7;  f.exp_bits = 8; f.bias = 127; }
    return f;
}

/* Exact value of a 16-bit pattern. */
double orc_decode16(uint16_t h, int kind)
{
    orc_fmt f = orc_format(kind);
    int sign = (h >> 15) & 1;
    int e = (h >> f.frac_bits) & ((1 << f.exp_bits) - 1);
    int frac = h & ((1 << f.frac_bits) - 1);
    int emax_field = (1 << f.exp_bits) - 1;
    double mag;
    if (e == emax_field) {
        mag = frac ? NAN : INFINITY;
    } else if (e == 0) {
        /* subnormal: frac * 2^(1 - bias - frac_bits) */
        mag = ldexp((double)frac, 1 - f.bias - f.frac_bits);
    } else {
        mag = ldexp((double)((1 << f.frac_bits) | frac), e - f.bias - f.frac_bits);
    }
    return sign ? -mag : mag;
}

/* Round a double to the nearest 16-bit value, ties to even; overflow gives
 * infinity, NaN gives the canonical quiet NaN of the format. */
uint16_t orc_encode16_rne(double x, int kind)
{
    orc_fmt f = orc_format(kind);
    int emax_field = (1 << f.exp_bits) - 1;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)((emax_field << f.frac_bits) | (1 << (f.frac_bits - 1)));
    double a = fabs(x);
    uint16_t inf = (uint16_t)(sign | (emax_field << f.frac_bits));
    if (isinf(a)) return inf;
    if (a == 0.0) return sign;

    int emin = 1 - f.bias;            /* exponent of the smallest normal */
    int emax = emax_field - 1 - f.bias;
    int k;
    frexp(a, &k);                     /* a = r * 2^k, r in [0.5, 1) */
    int E = k - 1;                    /* a = 1.xxx * 2^E */
    if (E < emin) E = emin;           /* subnormal range shares the emin quantum */
    /* Quantum (value of one unit in the last place) at exponent E. */
    double q = ldexp(1.0, E - f.frac_bits);
    double r = a / q;                 /* exact: division by a power of two */
    int old = fegetround();
    fesetround(FE_TONEAREST);
    double R = nearbyint(r);          /* ties to even */
    fesetround(old);
    double val = R * q;
    if (val >= ldexp(1.0, emax + 1)) return inf;
    if (val == 0.0) return sign;
    /* Re-derive the exponent after rounding (a carry may have bumped it). */
    frexp(val, &k);
    int E2 = k - 1;
    if (E2 < emin) {
        /* subnormal: exponent field 0, fraction = val / 2^(emin - frac_bits) */
        uint32_t frac = (uint32_t)ldexp(val, -(emin - f.frac_bits));
        return (uint16_t)(sign | frac);
    }
    uint32_t mant = (uint32_t)ldexp(val, -(E2 - f.frac_bits));   /* 1.fff as an integer */
    uint32_t frac = mant - (1u << f.frac_bits);
    uint32_t ef = (uint32_t)(E2 + f.bias);
    return (uint16_t)(sign | (ef << f.frac_bits) | frac);
}

void orc_decode16_array(int64_t n, const uint16_t* h, int kind, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_decode16(h[i], kind);
}

void orc_encode16_array(int64_t n, const double* x, int kind, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_encode16_rne(x[i], kind);
}

/* ------------------------------------------------------------------------- */
/* AdamW with mixed precision                                                 */
/*   [Mastering] §"AdamW Algorithm" (update rule: m_t, v_t, bias-corrected    */
/*   m_hat, v_hat, theta_{t+1}); [GPU-Opt-P2] §"AdamW 优化器——融合内核"        */
/*   (fused per-parameter update, gradient reset to zero) and                  */
/*   §"混合精度训练（FP16 / BF16）" (fp32 master copy, static loss scale,        */
/*   gradient cast-and-unscale, low-precision working copy of the weights).    */
/* ------------------------------------------------------------------------- */

/* 1 - beta^t for the global step t (t >= 1), from the fp32 hyperparameter. */
double orc_bias_correction(float beta, int64_t t)
{
    return 1.0 - pow((double)beta, (double)t);
}

/*
 * One AdamW step over n elements, evaluated in double.
 *   theta, m, v : state held in double by the caller (updated in place)
 *   grad        : the scaled 16-bit gradient as raw bit patterns (grad_kind)
 *   copy        : receives the 16-bit working copy of the new theta (copy_kind)
 *   grad_out    : receives the zeroed gradient (may alias grad)
 * Hyperparameters are the fp32 values the caller passes to the GPU, widened.
 */
void orc_adamw_step_f64(int64_t n, double* theta, double* m, double* v,
                        const uint16_t* grad, int grad_kind, double inv_loss_scale,
                        int64_t t, float lr_f, float beta1_f, float beta2_f,
                        float eps_f, float wd_f,
                        uint16_t* copy, int copy_kind, uint16_t* grad_out)
{
    const double lr = lr_f, b1 = beta1_f, b2 = beta2_f, eps = eps_f, wd = wd_f;
    const double bc1 = orc_bias_correction(beta1_f, t);
    const double bc2 = orc_bias_correction(beta2_f, t);
    for (int64_t i = 0; i < n; ++i) {
        /* gradient of the unscaled loss */
        double g = orc_decode16(grad[i], grad_kind) * inv_loss_scale;
        /* first and second moment estimates */
        m[i] = b1 * m[i] + (1.0 - b1) * g;
        v[i] = b2 * v[i] + (1.0 - b2) * (g * g);
        /* bias-corrected estimates */
        double m_hat = m[i] / bc1;
        double v_hat = v[i] / bc2;
        /* parameter update with decoupled decay on theta_t */
        double th = theta[i];
        theta[i] = th - lr * m_hat / (sqrt(v_hat) + eps) - lr * wd * th;
        /* low-precision working copy and gradient reset */
        copy[i] = orc_encode16_rne(theta[i], copy_kind);
        grad_out[i] = 0;
    }
}

/*
 * The same step in IEEE single precision, one rounding per operation, state in
 * fp32 as the GPU holds it.  The decay is grouped as theta - lr*(u + wd*theta),
 * which is how [GPU-Opt-P2]'s fused kernel groups it; it equals the [Mastering]
 * equation up to rounding.
 */
void orc_adamw_step_f32(int64_t n, float* theta, float* m, float* v,
                        const uint16_t* grad, int grad_kind, float inv_loss_scale,
                        int64_t t, float lr, float beta1, float beta2,
                        float eps, float wd,
                        uint16_t* copy, int copy_kind, uint16_t* grad_out)
{
    const float bc1 = (float)orc_bias_correction(beta1, t);
    const float bc2 = (float)orc_bias_correction(beta2, t);
    const float one_minus_b1 = 1.0f - beta1;
    const float one_minus_b2 = 1.0f - beta2;
    for (int64_t i = 0; i < n; ++i) {
        float g = (float)orc_decode16(grad[i], grad_kind) * inv_loss_scale;
        float gg = g * g;
        m[i] = beta1 * m[i] + one_minus_b1 * g;
        v[i] = beta2 * v[i] + one_minus_b2 * gg;
        float m_hat = m[i] / bc1;
        float v_hat = v[i] / bc2;
        float u = m_hat / (sqrtf(v_hat) + eps);
        float th = theta[i];
        theta[i] = th - lr * (u + wd * th);
        copy[i] = orc_encode16_rne((double)theta[i], copy_kind);
        grad_out[i] = 0;
    }
}

/* ------------------------------------------------------------------------- */
/* Softmax backward: dX_i = P_i * (dY_i - sum_j P_j dY_j), per row.           */
/*   [GPU-Opt-P2] §2.1 "Softmax 反向内核" (formula and two-pass row scheme).  */
/* ------------------------------------------------------------------------- */

void orc_softmax_bwd_f64(int64_t rows, int64_t cols,
                         const double* dY, const double* P, double* dX)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double* p = P + r * cols;
        const double* dy = dY + r * cols;
        double* dx = dX + r * cols;
        double dot = 0.0;
        for (int64_t j = 0; j < cols; ++j) dot += p[j] * dy[j];
        for (int64_t j = 0; j < cols; ++j) dx[j] = p[j] * (dy[j] - dot);
    }
}

void orc_softmax_bwd_f32(int64_t rows, int64_t cols,
                         const float* dY, const float* P, float* dX)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float* p = P + r * cols;
        const float* dy = dY + r * cols;
        float* dx = dX + r * cols;
        float dot = 0.0f;
        for (int64_t j = 0; j < cols; ++j) dot += p[j] * dy[j];
        for (int64_t j = 0; j < cols; ++j) dx[j] = p[j] * (dy[j] - dot);
    }
}

/* ------------------------------------------------------------------------- */
/* LayerNorm backward from the saved per-row mean and inv_std.                */
/*   Forward: y = gamma * xhat + beta, xhat = (x - mean) * inv_std,           */
/*   inv_std = 1/sqrt(var + eps), mean and (biased) var over the D features.  */
/*   [GPU-Opt-P2] §2.2 "LayerNorm 反向" (saved mean/inv_std; gamma, beta      */
/*   gradients by reduction; dX from the normalised values); [Mastering]      */
/*   §"Layer Normalization Backpropagation".                                   */
/*   Chain rule through mean and inv_std gives, per row:                       */
/*     dxhat = dY * gamma                                                      */
/*     dX    = inv_std * (dxhat - mean_D(dxhat) - xhat * mean_D(dxhat * xhat))  */
/*   and per column j: dgamma_j = sum_rows dY*xhat, dbeta_j = sum_rows dY.     */
/* ------------------------------------------------------------------------- */

void orc_layernorm_bwd_f64(int64_t rows, int64_t D,
                           const double* dY, const double* x,
                           const double* mean, const double* inv_std,
                           const double* gamma,
                           double* dX, double* dgamma, double* dbeta)
{
    for (int64_t j = 0; j < D; ++j) { dgamma[j] = 0.0; dbeta[j] = 0.0; }
    for (int64_t r = 0; r < rows; ++r) {
        const double* xr = x + r * D;
        const double* dyr = dY + r * D;
        double* dxr = dX + r * D;
        double mu = mean[r], rs = inv_std[r];
        double sum_dxhat = 0.0, sum_dxhat_xhat = 0.0;
        for (int64_t j = 0; j < D; ++j) {
            double xhat = (xr[j] - mu) * rs;
            double dxhat = dyr[j] * gamma[j];
            sum_dxhat += dxhat;
            sum_dxhat_xhat += dxhat * xhat;
        }
        double mean_dxhat = sum_dxhat / (double)D;
        double mean_dxhat_xhat = sum_dxhat_xhat / (double)D;
        for (int64_t j = 0; j < D; ++j) {
            double xhat = (xr[j] - mu) * rs;
            double dxhat = dyr[j] * gamma[j];
            dxr[j] = rs * (dxhat - mean_dxhat - xhat * mean_dxhat_xhat);
            dgamma[j] += dyr[j] * xhat;
            dbeta[j] += dyr[j];
        }
    }
}

void orc_layernorm_bwd_f32(int64_t rows, int64_t D,
                           const float* dY, const float* x,
                           const float* mean, const float* inv_std,
                           const float* gamma,
                           float* dX, float* dgamma, float* dbeta)
{
    for (int64_t j = 0; j < D; ++j) { dgamma[j] = 0.0f; dbeta[j] = 0.0f; }
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * D;
        const float* dyr = dY + r * D;
        float* dxr = dX + r * D;
        float mu = mean[r], rs = inv_std[r];
        float sum_dxhat = 0.0f, sum_dxhat_xhat = 0.0f;
        for (int64_t j = 0; j < D; ++j) {
            float xhat = (xr[j] - mu) * rs;
            float dxhat = dyr[j] * gamma[j];
            sum_dxhat += dxhat;
            sum_dxhat_xhat += dxhat * xhat;
        }
        float mean_dxhat = sum_dxhat / (float)D;
        float mean_dxhat_xhat = sum_dxhat_xhat / (float)D;
        for (int64_t j = 0; j < D; ++j) {
            float xhat = (xr[j] - mu) * rs;
            float dxhat = dyr[j] * gamma[j];
            dxr[j] = rs * (dxhat - mean_dxhat - xhat * mean_dxhat_xhat);
            dgamma[j] += dyr[j] * xhat;
            dbeta[j] += dyr[j];
        }
    }
}

/* ------------------------------------------------------------------------- */
/* RMSNorm backward from the saved per-row inv_rms.                           */
/*   Forward: y = gamma * xhat, xhat = x * inv_rms, inv_rms = 1/sqrt(mean_D(x^2) + eps): */
/*   the LayerNorm of [GPU-Opt-P2] §2.2 "LayerNorm 反向" without the mean      */
/*   subtraction and without beta (the norm layers of the Llama-7B table).     */
/*   Chain rule through inv_rms gives, per row:                                */
/*     dxhat = dY * gamma                                                      */
/*     dX    = inv_rms * (dxhat - xhat * mean_D(dxhat * xhat))                 */
/*   and per column j: dgamma_j = sum_rows dY*xhat.                             */
/* ------------------------------------------------------------------------- */

void orc_rmsnorm_bwd_f64(int64_t rows, int64_t D,
                         const double* dY, const double* x, const double* inv_rms,
                         const double* gamma, double* dX, double* dgamma)
{
    for (int64_t j = 0; j < D; ++j) dgamma[j] = 0.0;
    for (int64_t r = 0; r < rows; ++r) {
        const double* xr = x + r * D;
        const double* dyr = dY + r * D;
        double* dxr = dX + r * D;
        double rs = inv_rms[r];
        double sum_dxhat_xhat = 0.0;
        for (int64_t j = 0; j < D; ++j) sum_dxhat_xhat += (dyr[j] * gamma[j]) * (xr[j] * rs);
        double mean_dxhat_xhat = sum_dxhat_xhat / (double)D;
        for (int64_t j = 0; j < D; ++j) {
            double xhat = xr[j] * rs;
            double dxhat = dyr[j] * gamma[j];
            dxr[j] = rs * (dxhat - xhat * mean_dxhat_xhat);
            dgamma[j] += dyr[j] * xhat;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Global gradient-norm clipping with a non-finite flag                       */
/*   [GPU-Opt-P2] §"完整训练循环（整合一切）", gradient clipping: the L2 norm */
/*   of the unscaled gradient over all parameters, then the gradients are     */
/*   scaled by max_norm / norm when norm > max_norm, before the AdamW step.  */
/* ------------------------------------------------------------------------- */

/* Sum of squares of the unscaled gradient over n elements, in double; sets
 * *nonfinite to 1 when any element is NaN or infinite (it is left unchanged
 * otherwise, so several tensors can share one flag). */
double orc_grad_sumsq_f64(int64_t n, const uint16_t* grad, int kind, double inv_loss_scale,
                          int* nonfinite)
{
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double g = orc_decode16(grad[i], kind);
        if (!isfinite(g)) *nonfinite = 1;
        g *= inv_loss_scale;
        s += g * g;
    }
    return s;
}

/* The factor the gradients are multiplied by: max_norm / norm when the norm
 * exceeds max_norm, else 1 (max_norm <= 0 disables clipping). */
double orc_clip_factor(double norm, double max_norm)
{
    if (max_norm > 0.0 && norm > max_norm) return max_norm / norm;
    return 1.0;
}

/*
 * One AdamW step on the clipped gradient g = (float(grad) * inv_loss_scale) * clip,
 * in double; otherwise identical to orc_adamw_step_f64.  With skip != 0 (a
 * non-finite gradient was found) the step does not happen: theta, m, v and the
 * copy (an in/out array here) are left as they are and only the gradient is
 * zeroed.
 */
void orc_adamw_step_clipped_f64(int64_t n, double* theta, double* m, double* v,
                                const uint16_t* grad, int grad_kind, double inv_loss_scale,
                                double clip, int skip,
                                int64_t t, float lr_f, float beta1_f, float beta2_f,
                                float eps_f, float wd_f,
                                uint16_t* copy, int copy_kind, uint16_t* grad_out)
{
    const double lr = lr_f, b1 = beta1_f, b2 = beta2_f, eps = eps_f, wd = wd_f;
    const double bc1 = orc_bias_correction(beta1_f, t);
    const double bc2 = orc_bias_correction(beta2_f, t);
    for (int64_t i = 0; i < n; ++i) {
        if (!skip) {
            double g = orc_decode16(grad[i], grad_kind) * inv_loss_scale * clip;
            m[i] = b1 * m[i] + (1.0 - b1) * g;
            v[i] = b2 * v[i] + (1.0 - b2) * (g * g);
            double m_hat = m[i] / bc1;
            double v_hat = v[i] / bc2;
            double th = theta[i];
            theta[i] = th - lr * m_hat / (sqrt(v_hat) + eps) - lr * wd * th;
            copy[i] = orc_encode16_rne(theta[i], copy_kind);
        }
        grad_out[i] = 0;
    }
}

/* ------------------------------------------------------------------------- */
/* Stand-alone casts of the mixed-precision loop                              */
/*   [GPU-Opt-P2] §"混合精度训练（FP16 / BF16）" and §"完整训练循环（整合一切）"  */
/*   unscale and copy-back casts: low-precision gradient -> fp32 times        */
/*   1/loss_scale; fp32 master -> 16-bit working copy.                         */
/* ------------------------------------------------------------------------- */

/* out = float(src * scale) with one rounding of the exact product (the product
 * of a 16-bit or fp32 value and an fp32 scale is exact in double). */
void orc_cast_to_f32(int64_t n, const void* src, int kind, float scale, float* out)
{
    for (int64_t i = 0; i < n; ++i) {
        double x = (kind == ORC_F32) ? (double)((const float*)src)[i]
                                     : orc_decode16(((const uint16_t*)src)[i], kind);
        out[i] = (float)(x * (double)scale);
    }
}

/* out = the 16-bit value nearest to src (ties to even). */
void orc_cast_from_f32(int64_t n, const float* src, int kind, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_encode16_rne((double)src[i], kind);
}
