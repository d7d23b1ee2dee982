/*
 * tb.h -- C ABI of the GB300 (sm_103a) memory-bound training-step library.
 *
 * The library implements the memory-bound half of an LLM training step as
 * hand-written CUDA kernels:
 *   - a fused, multi-tensor, mixed-precision AdamW update;
 *   - the row-wise softmax backward;
 *   - the LayerNorm backward (dX, dgamma, dbeta).
 *
 * Sources (web pages on the subject; cited by page title and section):
 *   [GPU-Opt-P2]  "GPU 优化实战 Part 2：用 CUDA/ROCm 实现 LLM 反向传播与训练循环"
 *   [Mastering]   "Mastering LLM Training with CUDA and ROCm: The Backpropagation
 *                  and Optimization Workflow"
 *
 * Conventions for every entry point
 *   - Buffers are device-accessible memory owned by the caller, row-major and
 *     contiguous.  The library keeps no pointer after a call returns, except the
 *     AdamW plan's copy of the tensor table (see tb_adamw_plan_create).
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream.  Work is enqueued on it and the call returns without waiting: a
 *     fault inside a kernel surfaces at the caller's next synchronisation.
 *   - Argument errors are reported synchronously, before anything is enqueued,
 *     as a tb_status.  A failed launch reports TB_ERR_CUDA.
 *   - The softmax, LayerNorm and RMSNorm kernels are launched as programmatic
 *     dependents of the work before them on `stream`: their blocks may start
 *     while the previous kernel drains, set up shared memory and (LayerNorm,
 *     RMSNorm) prefetch their first rows into L2, but they load and store no
 *     global memory before every earlier kernel on the stream has completed and
 *     its writes are visible.  Stream order is kept exactly.
 *   - fp32 pointers must be 4-byte aligned and 16-bit pointers 2-byte aligned
 *     (TB_ERR_MISALIGNED otherwise).  Any larger alignment is optional: 16-byte
 *     aligned buffers take the vectorised path, others a scalar one.
 *   - The calls are not thread-safe against tb_adamw_plan_destroy of the plan
 *     they use; otherwise they may be called from several host threads.
 */
#ifndef TB_H_
#define TB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tb_status {
    TB_OK = 0,
    TB_ERR_INVALID_VALUE = 1,     /* null pointer, negative size, step < 1, ... */
    TB_ERR_UNSUPPORTED_DTYPE = 2, /* dtype not accepted by this entry point     */
    TB_ERR_MISALIGNED = 3,        /* pointer not aligned to its element size    */
    TB_ERR_ALIAS = 4,             /* an output overlaps an input or another output */
    TB_ERR_WORKSPACE = 5,         /* workspace missing or smaller than required */
    TB_ERR_OOM = 6,               /* the library's own small allocation failed  */
    TB_ERR_CUDA = 7,              /* a CUDA runtime call or launch failed        */
    TB_ERR_DEVICE = 8,            /* plan used with another device current       */
    TB_ERR_TIMEOUT = 9            /* a kernel's bounded wait gave up (see tb_device_error) */
} tb_status;

typedef enum tb_dtype {
    TB_F32 = 0,   /* IEEE binary32 */
    TB_F16 = 1,   /* IEEE binary16 */
    TB_BF16 = 2   /* bfloat16 */
} tb_dtype;

/* Human-readable name of a status code (static storage; never NULL). */
const char* tb_status_string(tb_status status);

/* Library version as 10000*major + 100*minor + patch. */
int tb_version(void);

/*
 * tb_device_error -- read (and optionally clear) the device-side error word of
 * the current device.  Kernels that wait on an mbarrier for their own bulk
 * copies give up after about one second; they then set this word to
 * TB_ERR_TIMEOUT, drain what they issued and return early (their outputs are
 * then undefined).  tb_adamw_step_device sets it to TB_ERR_INVALID_VALUE when
 * the step counter it reads is below 1.  This call synchronises the current
 * device.
 *   code   out: 0 when no kernel gave up since the last reset
 *   reset  nonzero: clear the word after reading it
 * Returns TB_OK, TB_ERR_INVALID_VALUE (code == NULL) or TB_ERR_CUDA.
 */
tb_status tb_device_error(int* code, int reset);

/*
 * tb_layernorm_bwd_selftest_timeout -- exercises that failure path without a
 * GPU fault.  It runs the LayerNorm backward's two bulk-copy ring kernels on
 * small internal problems (4 x 256 bf16 on one CTA per row block, then 4 x
 * 16,384 bf16 split over a four-CTA cluster; zeroed buffers the call allocates
 * and frees) with their copies withheld, so that every wait on them runs out after
 * wait_limit_ns nanoseconds; each kernel then sets the device error word to
 * TB_ERR_TIMEOUT, waits (bounded as well) for the copies it would have issued,
 * and returns -- the CTAs of a cluster together, after telling each other of the
 * failure.  Nothing is in flight when it returns, so the context stays usable.
 * The call synchronises `stream`; afterwards tb_device_error reports
 * TB_ERR_TIMEOUT.
 *   wait_limit_ns  1,000 .. 1,000,000,000
 * Returns TB_OK once the kernel has finished, TB_ERR_INVALID_VALUE (limit out of
 * range), TB_ERR_OOM or TB_ERR_CUDA.
 */
tb_status tb_layernorm_bwd_selftest_timeout(int64_t wait_limit_ns, void* stream);

/* ======================================================================== */
/* Fused mixed-precision AdamW (multi-tensor)                               */
/* ======================================================================== */
/*
 * One pass over every element of every tensor computes, per element
 * ([Mastering] §"AdamW Algorithm" update rule; [GPU-Opt-P2] §"AdamW 优化器——
 * 融合内核" and §"混合精度训练（FP16 / BF16）"):
 *     g      = float(grad) * inv_loss_scale            (unscale)
 *     m      = beta1*m + (1-beta1)*g
 *     v      = beta2*v + (1-beta2)*g*g
 *     m_hat  = m / (1 - beta1^t),  v_hat = v / (1 - beta2^t)
 *     param  = param - lr*(m_hat/(sqrt(v_hat)+eps) + weight_decay*param_t)
 *     copy   = round-to-nearest-even(param) in copy_dtype
 *     grad   = +0
 * with decoupled weight decay taken on the pre-update parameter param_t.
 * The bias corrections and (1-beta) are formed once per call on the host.
 */
typedef struct tb_tensor_desc {
    float* param;   /* fp32 master weights [n], read and written in place        */
    float* m;       /* fp32 first moment   [n], read and written in place        */
    float* v;       /* fp32 second moment  [n], read and written in place        */
    void* grad;     /* loss-scaled gradient [n] in grad_dtype, read then zeroed  */
    void* copy;     /* working copy [n] in copy_dtype, written; NULL: none       */
    int64_t n;      /* element count (>= 0; 0 skips the tensor)                  */
} tb_tensor_desc;

typedef struct tb_adamw_hparams {
    float lr;            /* learning rate eta                         */
    float beta1;         /* first-moment decay, in [0, 1)             */
    float beta2;         /* second-moment decay, in [0, 1)            */
    float eps;           /* added to sqrt(v_hat), >= 0                */
    float weight_decay;  /* decoupled decay lambda, >= 0              */
} tb_adamw_hparams;

typedef struct tb_adamw_plan tb_adamw_plan;   /* opaque */

/*
 * tb_adamw_plan_create -- validate a table of parameter tensors and copy it to
 * the current device once, so that every later step is a single launch.
 *   tensors     host array of n_tensors descriptors (read during the call only)
 *   n_tensors   >= 1
 *   grad_dtype  TB_F16, TB_BF16 or TB_F32
 *   copy_dtype  TB_BF16 or TB_F16 (unused when the tensors have no copy)
 *               Either every tensor with n > 0 has a working copy, or none has
 *               (copy == NULL: the step writes no copy).
 *   out         receives the plan; the caller owns it and frees it with
 *               tb_adamw_plan_destroy.  The plan owns a device copy of the table
 *               (64 bytes per tensor) followed by the step kernel's 16-byte tile
 *               counter, and remembers the current device.
 *               Every call that takes a plan first looks it up among the plans
 *               created and not yet destroyed; any other pointer (a destroyed
 *               plan included) is rejected with TB_ERR_INVALID_VALUE without
 *               being dereferenced.
 * Errors: TB_ERR_INVALID_VALUE (null param/m/v/grad with n > 0, copies given for
 * some tensors only, n < 0, n_tensors < 1,
 * out == NULL), TB_ERR_UNSUPPORTED_DTYPE, TB_ERR_MISALIGNED, TB_ERR_ALIAS (any
 * two of the 5*n_tensors buffers overlap), TB_ERR_OOM, TB_ERR_CUDA.
 */
tb_status tb_adamw_plan_create(const tb_tensor_desc* tensors, int n_tensors,
                               tb_dtype grad_dtype, tb_dtype copy_dtype,
                               tb_adamw_plan** out);

/*
 * tb_adamw_step -- enqueue one fused AdamW step over every tensor of the plan.
 *   step            global step t >= 1 (the first update is t = 1)
 *   hp              hyperparameters (read during the call only)
 *   inv_loss_scale  1/loss_scale (exact for a power-of-two scale); > 0
 *   stream          cudaStream_t or NULL
 * The kernel's CTAs claim tiles of the flat parameter space from a counter kept
 * in the plan's device memory (so CTAs on faster SMs take more tiles).  Each call
 * enqueues a 16-byte cudaMemsetAsync of that counter on `stream` before the
 * launch, so every launch starts from zero whatever an earlier launch left
 * there.  Steps of one plan (plain, clipped or device) must run one after
 * another: on one stream, or ordered by events.  They update the same tensors
 * and share the counter, so they must be ordered in any case.
 * Errors: TB_ERR_INVALID_VALUE (plan/hp NULL, step < 1, beta outside [0,1),
 * eps, lr or weight_decay negative or not finite, inv_loss_scale <= 0),
 * TB_ERR_DEVICE (another device is current), TB_ERR_CUDA.
 */
tb_status tb_adamw_step(const tb_adamw_plan* plan, int64_t step,
                        const tb_adamw_hparams* hp, float inv_loss_scale,
                        void* stream);

/*
 * Global gradient-norm clipping with a non-finite check, fused into the step
 * without a host synchronisation ([GPU-Opt-P2] §"完整训练循环（整合一切）", its
 * gradient-clipping step: the L2 norm of the unscaled gradient over all
 * parameters; when it exceeds max_norm the gradients are scaled by
 * max_norm / norm before the optimizer).
 *
 * tb_adamw_grad_norm reads every gradient of the plan once (2 bytes per
 * parameter) and writes three floats to device memory `out`:
 *     out[0] = norm   = sqrt(sum_i (float(grad_i) * inv_loss_scale)^2)
 *     out[1] = factor = max_norm / norm if max_norm > 0 and norm > max_norm, else 1
 *     out[2] = 1 if any gradient element is NaN or infinite, else 0
 * Each thread adds its squares in fp32 in rounds of at most 32, adds the round
 * sums of one tile (at most 256 squares) in fp32 and the tile sums in fp64; each
 * CTA adds a fixed set of tiles (consecutive chunks of 262,144 elements on large
 * tables, tiles dealt round-robin on small ones) into one partial, and the
 * partials are added in a fixed order, so the result is reproducible.
 *   workspace  device scratch of tb_adamw_grad_norm_workspace_size() bytes,
 *              8-byte aligned (one fp64 partial and one flag per CTA)
 * Errors: TB_ERR_INVALID_VALUE, TB_ERR_MISALIGNED, TB_ERR_WORKSPACE, TB_ERR_ALIAS,
 * TB_ERR_DEVICE, TB_ERR_CUDA.
 *
 * tb_adamw_step_clipped is tb_adamw_step with the unscaled gradient multiplied by
 * clip[1] (clip = the `out` of tb_adamw_grad_norm, read on the device).  When
 * clip[2] != 0 the step does not happen: parameters, moments and the working copy
 * are left as they are and only the gradient is reset to zero.  Whether the
 * caller then advances its step counter is its choice (clip[2] can be read back
 * later).  Errors as tb_adamw_step, plus TB_ERR_INVALID_VALUE for clip == NULL.
 */
tb_status tb_adamw_grad_norm_workspace_size(const tb_adamw_plan* plan, size_t* bytes);

tb_status tb_adamw_grad_norm(const tb_adamw_plan* plan, float inv_loss_scale, float max_norm,
                             float* out, void* workspace, size_t workspace_bytes, void* stream);

tb_status tb_adamw_step_clipped(const tb_adamw_plan* plan, int64_t step,
                                const tb_adamw_hparams* hp, float inv_loss_scale,
                                const float* clip, void* stream);

/*
 * tb_adamw_step_device -- tb_adamw_step (clip == NULL) or tb_adamw_step_clipped
 * (clip != NULL) with the step counter in device memory: the kernel reads t from
 * `step` when it runs and forms the bias corrections 1 - beta^t itself (in
 * double, rounded to fp32, as the host does for the other entry points).  With
 * every per-step input on the device, a whole optimizer step -- counter
 * increment, gradient norm, update -- can be captured once in a CUDA graph and
 * replayed every iteration.  The counter is only read: the caller advances it.
 *   step   device int64, 8-byte aligned; a value below 1 makes the kernel set the
 *          device error word to TB_ERR_INVALID_VALUE and update nothing
 *   clip   NULL, or the device output of tb_adamw_grad_norm
 * Errors: as tb_adamw_step, plus TB_ERR_INVALID_VALUE (step == NULL) and
 * TB_ERR_MISALIGNED.
 */
tb_status tb_adamw_step_device(const tb_adamw_plan* plan, const int64_t* step,
                               const tb_adamw_hparams* hp, float inv_loss_scale,
                               const float* clip, void* stream);

/*
 * tb_adamw_selftest_stale_counter -- test hook for the tile counter above.  It
 * waits for `stream`, then writes `next` into the plan's tile counter (and a
 * nonzero value into the counter's second word) with a synchronous cudaMemcpy,
 * as a launch that stopped part-way would leave them.  The next step of the
 * plan must still update and zero every element.  Not for use in training.
 * Errors: TB_ERR_INVALID_VALUE (not a live plan), TB_ERR_DEVICE, TB_ERR_CUDA.
 */
tb_status tb_adamw_selftest_stale_counter(const tb_adamw_plan* plan, uint64_t next,
                                          void* stream);

/* Free a plan (NULL is accepted; a pointer that is not a live plan, e.g. one
 * destroyed already, returns TB_ERR_INVALID_VALUE).  Synchronises nothing: the
 * caller must not destroy a plan while a step that uses it may still be running. */
tb_status tb_adamw_plan_destroy(tb_adamw_plan* plan);

/* ======================================================================== */
/* Stand-alone casts                                                         */
/* ======================================================================== */
/*
 * The two casts of the pages' mixed-precision loop that the fused step does
 * internally ([GPU-Opt-P2] §"混合精度训练（FP16 / BF16）", §"完整训练循环（整合一切）"
 * its unscale cast and its copy-back cast), for callers that keep the optimizer
 * steps apart:
 *   tb_cast_to_f32   : dst[i] = float(src[i]) * scale (one fp32 rounding),
 *                      src in src_dtype (TB_F16, TB_BF16 or TB_F32), dst fp32
 *   tb_cast_from_f32 : dst[i] = round-to-nearest-even(src[i]) in dst_dtype
 *                      (TB_F16 or TB_BF16)
 *   0 <= n <= INT64_MAX / 8 elements (0: nothing is enqueued); src and dst must not
 *   overlap.
 * Errors: TB_ERR_INVALID_VALUE, TB_ERR_UNSUPPORTED_DTYPE, TB_ERR_MISALIGNED,
 * TB_ERR_ALIAS, TB_ERR_CUDA.
 */
tb_status tb_cast_to_f32(const void* src, tb_dtype src_dtype, float scale, float* dst,
                         int64_t n, void* stream);

tb_status tb_cast_from_f32(const float* src, void* dst, tb_dtype dst_dtype, int64_t n,
                           void* stream);

/* ======================================================================== */
/* Softmax backward                                                          */
/* ======================================================================== */
/*
 * tb_softmax_bwd -- for every row r of a [rows, cols] matrix
 *     dX[r,i] = P[r,i] * (dY[r,i] - sum_j P[r,j]*dY[r,j])
 * ([GPU-Opt-P2] §2.1 "Softmax 反向内核"), P being the forward softmax output.
 * The dot product is accumulated in fp32 whatever the I/O dtype.
 *   dY, P   inputs [rows, cols] in dtype
 *   dX      output [rows, cols] in dtype; must not overlap dY or P
 *   rows, cols  >= 0 (either 0: nothing is enqueued)
 *   dtype   TB_F32, TB_BF16 or TB_F16
 * Each element of dY and P is read from HBM once when a row fits on chip
 * (cols <= 8192 fp32 / 16384 16-bit, 16-byte aligned rows); longer or
 * unaligned rows are read twice.
 * Errors: TB_ERR_INVALID_VALUE, TB_ERR_UNSUPPORTED_DTYPE, TB_ERR_MISALIGNED,
 * TB_ERR_ALIAS, TB_ERR_CUDA.
 */
tb_status tb_softmax_bwd(const void* dY, const void* P, void* dX,
                         int64_t rows, int64_t cols, tb_dtype dtype, void* stream);

/*
 * tb_softmax_bwd_causal -- tb_softmax_bwd for the rows of causally masked
 * attention, reading only the part of each row the mask left open.
 * Row r can be nonzero only on its first
 *     valid(r) = min(cols, (r mod period) + 1 + offset)
 * columns: `period` is the query length S_q of one (batch, head) block whose
 * rows are stacked, `offset` = S_k - S_q (0 for square self-attention).  P must
 * be exactly 0 on every other column, as a masked forward softmax leaves it; the
 * kernel never reads those columns of P or dY and writes +0 to dX there.  On
 * such inputs the result equals tb_softmax_bwd's (masked entries are +-0 there)
 * bit for bit for rows of up to 2,048 16-bit / 1,024 fp32 columns; longer rows
 * sum the same dot-product terms in another grouping and agree within its fp32
 * rounding.  Every call on the same inputs returns the same bits.  When a
 * causal block fits in `rows` (period <= rows), rows q and period-1-q of a block
 * are processed together, so the work per warp or CTA does not depend on q.
 * HBM traffic per row: reads of the valid columns (rounded up to 16-byte
 * vectors) plus the full row of dX written.
 *   period >= 1, offset >= 0; other arguments and errors as tb_softmax_bwd.
 */
tb_status tb_softmax_bwd_causal(const void* dY, const void* P, void* dX, int64_t rows,
                                int64_t cols, int64_t period, int64_t offset,
                                tb_dtype dtype, void* stream);

/* ======================================================================== */
/* LayerNorm backward                                                        */
/* ======================================================================== */
/*
 * Forward being y = gamma * xhat + beta with xhat = (x - mean) * inv_std over
 * the D features of each row, the backward computes ([GPU-Opt-P2] §2.2
 * "LayerNorm 反向"; [Mastering] §"Layer Normalization Backpropagation"):
 *     dxhat   = dY * gamma
 *     dX      = inv_std * (dxhat - mean_D(dxhat) - xhat * mean_D(dxhat*xhat))
 *     dgamma  = sum over rows of dY * xhat     (per column)
 *     dbeta   = sum over rows of dY            (per column)
 * dgamma and dbeta are OVERWRITTEN (not accumulated).  They are reduced in two
 * stages -- per-CTA partial sums into the workspace, then a second kernel that
 * adds them in a fixed order -- so results are bitwise reproducible run to run
 * on the same device model.  Rows longer than 16 KB (more than 8,192 16-bit or
 * 4,096 fp32 columns; 16-byte aligned buffers, D a multiple of 2..8 times the
 * 16-byte vector) are split by columns over the CTAs of a thread-block cluster,
 * which exchange their shares of the row sums through distributed shared memory
 * and write one partial row per cluster; all CTAs of a cluster use bitwise the
 * same row sums.
 */

/*
 * tb_layernorm_bwd_workspace_size -- bytes of workspace tb_layernorm_bwd needs
 * for this shape on the current device (it depends on the SM count).
 * Errors: TB_ERR_INVALID_VALUE (bytes NULL, rows or D negative),
 * TB_ERR_UNSUPPORTED_DTYPE, TB_ERR_CUDA.
 */
tb_status tb_layernorm_bwd_workspace_size(int64_t rows, int64_t D, tb_dtype io_dtype,
                                          size_t* bytes);

/*
 * tb_layernorm_bwd
 *   dY, x      inputs [rows, D] in io_dtype (TB_F32, TB_BF16 or TB_F16)
 *   mean       fp32 [rows], the forward's saved row means
 *   inv_std    fp32 [rows], the forward's saved 1/sqrt(var + eps)
 *   gamma      fp32 [D]
 *   dX         output [rows, D] in io_dtype
 *   dgamma     output fp32 [D]
 *   dbeta      output fp32 [D]
 *   workspace  device scratch of at least tb_layernorm_bwd_workspace_size()
 *              bytes, 16-byte aligned; contents on entry are ignored
 *   stream     cudaStream_t or NULL
 * rows == 0 writes zeros to dgamma and dbeta; D == 0 enqueues nothing.
 * Outputs must not overlap any input, each other or the workspace.
 * Errors: TB_ERR_INVALID_VALUE, TB_ERR_UNSUPPORTED_DTYPE, TB_ERR_MISALIGNED,
 * TB_ERR_ALIAS, TB_ERR_WORKSPACE, TB_ERR_CUDA.
 */
tb_status tb_layernorm_bwd(const void* dY, const void* x, const float* mean,
                           const float* inv_std, const float* gamma,
                           void* dX, float* dgamma, float* dbeta,
                           int64_t rows, int64_t D, tb_dtype io_dtype,
                           void* workspace, size_t workspace_bytes, void* stream);

/* ======================================================================== */
/* RMSNorm backward                                                          */
/* ======================================================================== */
/*
 * The LayerNorm above without the mean subtraction and without beta (the norm
 * layers of Llama-style models): forward y = gamma * x * inv_rms with
 * inv_rms = 1/sqrt(mean_D(x^2) + eps).  Backward, per row and per column:
 *     dxhat  = dY * gamma,  xhat = x * inv_rms
 *     dX     = inv_rms * (dxhat - xhat * mean_D(dxhat * xhat))
 *     dgamma = sum over rows of dY * xhat      (overwritten, two-stage, deterministic)
 * Same kernels, layouts, alignment rules and errors as tb_layernorm_bwd, with
 * inv_rms in place of mean/inv_std and no dbeta.  The workspace is half the
 * LayerNorm one (one partial row of D floats per CTA).
 */
tb_status tb_rmsnorm_bwd_workspace_size(int64_t rows, int64_t D, tb_dtype io_dtype,
                                        size_t* bytes);

tb_status tb_rmsnorm_bwd(const void* dY, const void* x, const float* inv_rms,
                         const float* gamma, void* dX, float* dgamma,
                         int64_t rows, int64_t D, tb_dtype io_dtype,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * tb_layernorm_bwd_noalloc -- the same LayerNorm backward as tb_layernorm_bwd,
 * for callers that cannot allocate device memory when they run it.  (The pages
 * have no counterpart: this is a convenience of this library.)
 *
 * Who needs it: code that runs where a cudaMalloc is not an option -- inside a
 * framework that hands out every byte of device memory from its own pool (a
 * stray allocation there fails or fragments the pool), or a step loop that must
 * not call cudaMalloc/cudaFree because they can synchronise with the device.
 * Such callers have no buffer to pass as `workspace`, so this entry point keeps
 * its scratch (the per-CTA dgamma/dbeta partial sums) in a fixed array inside
 * the library and allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library call.
 *
 * The array holds TB_LAYERNORM_NOALLOC_SCRATCH_BYTES (16 MiB).  Every GPU that
 * loads the library holds it until the process exits.  A shape whose partial
 * sums would not fit runs with fewer CTAs; D > 2,097,152 (more than the array
 * holds for a single CTA) is rejected with TB_ERR_WORKSPACE.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture.  All calls share the one array and it keeps the last
 * call's contents (each call overwrites every part it later reads, so nothing
 * has to start at zero): calls whose work overlaps on the GPU -- for example on
 * two streams at once -- race on it and must be serialised by the caller.
 *
 * Arguments, results and errors are those of tb_layernorm_bwd without
 * `workspace` and `workspace_bytes`; results equal tb_layernorm_bwd's bit for
 * bit whenever the partial sums fit with the usual number of CTAs (for example
 * 16,384 x 4,096 bf16), and agree within rounding otherwise.
 */
#define TB_LAYERNORM_NOALLOC_SCRATCH_BYTES (16u << 20)

tb_status tb_layernorm_bwd_noalloc(const void* dY, const void* x, const float* mean,
                                   const float* inv_std, const float* gamma,
                                   void* dX, float* dgamma, float* dbeta,
                                   int64_t rows, int64_t D, tb_dtype io_dtype, void* stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* TB_H_ */
