/*
 * nrm.h -- C ABI of the row-wise normalization library for GB300 (sm_103a).
 *
 * Operators, each one asynchronous launch sequence on the caller's CUDA
 * stream:
 *   ln_fwd        LayerNorm over the rows of a [rows, N] tensor
 *   rms_fwd       RMSNorm over the rows of a [rows, N] tensor
 *   add_rms_fwd   fused residual add + RMSNorm (pre-norm residual stream)
 *   bn_fwd_train  BatchNorm2d training forward over an NCHW tensor
 *   bn_fwd_infer  BatchNorm2d inference forward (running statistics)
 *   bn_bwd        BatchNorm2d training backward (dx, dgamma, dbeta)
 *   softmax_fwd   row softmax over a [rows, N] tensor
 *   bn_fwd_partial_stats / bn_fwd_apply_stats, bn_bwd_partial_sums /
 *   bn_bwd_apply_sums   the local halves of synchronized BatchNorm
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.  Every data pointer is CALLER-OWNED DEVICE memory of the current
 *   CUDA device (cudaGetDevice at call time).  The library allocates nothing
 *   and keeps no per-call state; it only caches device attributes.  A host
 *   pointer is not detected unless pointer checks are switched on
 *   (nrm_set_pointer_checks); without them it makes the kernel fault.
 * Layout.  Row operators: row-major [rows, N], contiguous (row stride N;
 *   the *_ld entry points take a row stride per tensor).
 *   BatchNorm: NCHW with H*W flattened to HW; element (n, c, k) at
 *   ((n*C + c)*HW + k).  Parameters (gamma, beta, w) are [N] (rows ops) or
 *   [C] (BatchNorm) in the I/O type; statistics are always binary32.
 * Types.  dtype is an nrm_dtype: binary32, binary16 or bfloat16 for the
 *   data and the parameters.  All arithmetic is binary32; every output is
 *   rounded once to its type, round-to-nearest-even.
 * Optional pointers.  gamma/w NULL means 1, beta NULL means 0; NULL mean,
 *   rstd, save_mean, save_rstd means "do not write"; NULL running_mean or
 *   running_var means "no running-statistic update".
 * Alignment.  Any alignment and any N are accepted.  The vectorised kernels
 *   (16-byte loads and stores) run when every row pointer is 16-byte aligned
 *   and N is a multiple of 16/sizeof(element); otherwise a scalar kernel runs.
 * Aliasing.  Outputs may not overlap inputs or each other, with one
 *   exception: add_rms_fwd accepts residual_out == residual (the residual
 *   stream updated in place).  Any other overlap returns NRM_ERR_ALIAS.
 * Errors.  Arguments are validated before anything is launched; an invalid
 *   call returns a non-zero nrm_status and launches nothing.  After the
 *   launch, cudaGetLastError is checked (NRM_ERR_LAUNCH).  Errors raised
 *   later by the kernels (for example a fault from a bad pointer) surface on
 *   the stream, as with any CUDA launch.
 * Streams.  Calls are asynchronous on `stream` (0 = legacy default stream)
 *   and never synchronize.  Calls are thread-safe.
 * Empty input.  rows == 0 is a no-op that returns NRM_OK (row operators),
 *   whatever the pointers (empty tensors may have NULL data).
 */
#ifndef NRM_H
#define NRM_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NRM_F32 = 0,   /* IEEE binary32 */
    NRM_F16 = 1,   /* IEEE binary16 */
    NRM_BF16 = 2   /* bfloat16 */
} nrm_dtype;

typedef enum {
    NRM_OK = 0,
    NRM_ERR_NULL = 1,          /* a required pointer is NULL */
    NRM_ERR_SHAPE = 2,         /* negative extent, N < 1, size overflow, BN count < 2 */
    NRM_ERR_DTYPE = 3,         /* dtype is not an nrm_dtype */
    NRM_ERR_ALIAS = 4,         /* an output overlaps an input or another output */
    NRM_ERR_VALUE = 5,         /* eps < 0 or not finite; momentum outside [0, 1];
                                  a pointer not aligned to its element size */
    NRM_ERR_UNSUPPORTED = 6,   /* valid but not provided (e.g. a forced plan that
                                  cannot run this shape) */
    NRM_ERR_WORKSPACE = 7,     /* BatchNorm workspace NULL, too small or misaligned */
    NRM_ERR_DEVICE = 8,        /* no current CUDA device or attribute query failed */
    NRM_ERR_LAUNCH = 9,        /* cudaGetLastError reported a launch failure */
    NRM_ERR_POINTER = 10,      /* pointer checks on, and a pointer is not device
                                  memory of the current device */
    NRM_ERR_TOO_LARGE = 11     /* bn_fwd_train_noalloc: batch * C above its fixed
                                  capacity (65536) */
} nrm_status;

/*
 * LayerNorm forward over each row of x[rows, N]:
 *   mean = (1/N) sum_i x_i,   var = (1/N) sum_i (x_i - mean)^2   (biased)
 *   y_i  = (x_i - mean) / sqrt(var + eps) * gamma_i + beta_i
 * Definition: CUDA handbook LayerNorm walkthrough (lpnh.cn/news/2756757), §1;
 * optional gamma/beta and the statistics outputs as in its §2 and §7.
 *   x      [rows, N] dtype, read only
 *   gamma  [N] dtype or NULL (= 1);  beta [N] dtype or NULL (= 0)
 *   y      [rows, N] dtype, written; must not overlap x
 *   mean   [rows] binary32 or NULL;  rstd [rows] binary32 = 1/sqrt(var+eps), or NULL
 *   eps    >= 0, finite
 * Returns an nrm_status.
 */
int ln_fwd(const void *x, const void *gamma, const void *beta, void *y,
           float *mean, float *rstd, int64_t rows, int64_t N, float eps,
           int dtype, cudaStream_t stream);

/*
 * RMSNorm forward over each row of x[rows, N]:
 *   y_i = x_i / sqrt((1/N) sum_j x_j^2 + eps) * w_i
 * Definition: CUDA fused RMSNorm kernel page (diycv.top), §0.3 and §1-§2.
 *   x [rows, N] dtype;  w [N] dtype or NULL (= 1);  y [rows, N] dtype
 *   rstd [rows] binary32 = 1/sqrt(mean(x^2)+eps), or NULL
 */
int rms_fwd(const void *x, const void *w, void *y, float *rstd,
            int64_t rows, int64_t N, float eps, int dtype, cudaStream_t stream);

/*
 * Fused pre-norm path over each row:
 *   residual_out = round_to_dtype(binary32(x) + binary32(residual))
 *   y            = RMSNorm(residual_out, w)
 * The statistics use the rounded residual_out, the value the residual stream
 * carries on.  Definition: CUDA fused RMSNorm kernel page (diycv.top), §2 and §3.2.
 *   x, residual   [rows, N] dtype, read only
 *   w             [N] dtype or NULL (= 1)
 *   residual_out  [rows, N] dtype, written; may be the same pointer as residual
 *   y             [rows, N] dtype, written
 *   rstd          [rows] binary32, or NULL
 */
int add_rms_fwd(const void *x, const void *residual, const void *w,
                void *residual_out, void *y, float *rstd,
                int64_t rows, int64_t N, float eps, int dtype, cudaStream_t stream);

/*
 * The row operators on strided rows: row r of x starts at element r * ldx
 * (likewise ldr for residual, ldro for residual_out, ldy for y), for views
 * such as a column slice or a padded buffer (row stride 1028 for N = 1024),
 * the case the LayerNorm walkthrough (lpnh.cn/news/2756757) lists in §7.
 * Every ld* >= N; the contiguous entry points above are these with all
 * strides equal to N.  Vectorised kernels run when every row start is
 * 16-byte aligned (base pointers aligned and ld * element size a multiple
 * of 16); otherwise the scalar kernel runs.  Two strided tensors with the
 * same row stride are tested for overlap exactly (so y may share a padded
 * buffer with x in other columns); with different strides their outer
 * bounds are compared.  residual_out == residual in place requires
 * ldro == ldr.  Other arguments, results and errors as the contiguous
 * versions; ld < N returns NRM_ERR_SHAPE.
 */
int ln_fwd_ld(const void *x, int64_t ldx, const void *gamma, const void *beta, void *y,
              int64_t ldy, float *mean, float *rstd, int64_t rows, int64_t N, float eps,
              int dtype, cudaStream_t stream);
int rms_fwd_ld(const void *x, int64_t ldx, const void *w, void *y, int64_t ldy, float *rstd,
               int64_t rows, int64_t N, float eps, int dtype, cudaStream_t stream);
int add_rms_fwd_ld(const void *x, int64_t ldx, const void *residual, int64_t ldr,
                   const void *w, void *residual_out, int64_t ldro, void *y, int64_t ldy,
                   float *rstd, int64_t rows, int64_t N, float eps, int dtype,
                   cudaStream_t stream);
int softmax_fwd_ld(const void *x, int64_t ldx, void *y, int64_t ldy, float *row_max,
                   float *row_sum, int64_t rows, int64_t N, int dtype, cudaStream_t stream);

/*
 * add_rms_fwd on tensors in HOST memory (x, residual, residual_out, y; page-
 * locked memory is fastest), streamed through the device in chunks of rows
 * (about 4 MB of each tensor per chunk): the host->device copy of chunk k+1,
 * the kernel of chunk k and the device->host copy of chunk k-1 run at once
 * (two copy streams of the library and `stream`), so a call costs about the
 * time of moving its bytes over the host link.  No page describes this
 * entry point; it is the library's own host-memory path.
 *   w        [N] dtype, DEVICE memory, or NULL
 *   rstd     [rows] binary32, DEVICE memory, or NULL
 *   workspace  device memory, 256-byte aligned, at least
 *              add_rms_fwd_host_workspace_size(N, dtype) bytes (staging for
 *              three chunks); calls sharing one workspace must be ordered on
 *              the GPU (same stream or events).
 * residual_out may be the same host buffer as residual.  Asynchronous: the
 * host outputs are complete when `stream` is (e.g. after
 * cudaStreamSynchronize); the host inputs must stay valid until then.
 * Returns an nrm_status; a failure after some chunks were enqueued leaves the
 * outputs undefined.
 */
size_t add_rms_fwd_host_workspace_size(int64_t N, int dtype);
int add_rms_fwd_host(const void *x, const void *residual, const void *w, void *residual_out,
                     void *y, float *rstd, int64_t rows, int64_t N, float eps, int dtype,
                     void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Row softmax over each row of x[rows, N]:
 *   m = max_j x_j,   d = sum_j exp(x_j - m),   y_i = exp(x_i - m) / d
 * Definition: LLM-ops page (smarter.xin), section 1 "Softmax", with its
 * online (max, sum) form and the rule that merges two partial pairs by
 * rescaling both sums to the larger max; one CTA-wide merge per row.
 *   x        [rows, N] dtype, read only; -inf entries (masked) give y = 0
 *   y        [rows, N] dtype, written; must not overlap x
 *   row_max  [rows] binary32 = m, or NULL
 *   row_sum  [rows] binary32 = d, or NULL
 * A row whose entries are all -inf has no defined result (NaN).
 * Exponentials are binary32 expf; the output is rounded once to its type.
 */
int softmax_fwd(const void *x, void *y, float *row_max, float *row_sum,
                int64_t rows, int64_t N, int dtype, cudaStream_t stream);

/*
 * Bytes of device workspace bn_fwd_train needs for this shape (0 on invalid
 * arguments): 8 bytes per chunk of at most 1024 16-byte packs of each (n, c)
 * plane, P = batch * C * ceil(ceil(HW / (16 / element size)) / 1024) chunks,
 * rounded up to 16 bytes, plus 24 bytes per channel:
 * roundup16(8 * P) + 24 * C.  The workspace holds partial statistics, folded
 * per-channel statistics and per-channel control words that each call resets
 * itself; its content on entry does not matter and it is scratch on exit.
 */
size_t bn_fwd_train_workspace_size(int64_t batch, int64_t C, int64_t HW, int dtype);

/*
 * BatchNorm2d training forward over x[batch, C, HW] (NCHW).  Per channel c,
 * over all n and k (cnt = batch*HW):
 *   mean_c = (1/cnt) sum x,   var_c = (1/cnt) sum (x - mean_c)^2   (biased)
 *   y = (x - mean_c) / sqrt(var_c + eps) * gamma_c + beta_c
 *   save_mean[c] = mean_c,   save_rstd[c] = 1/sqrt(var_c + eps)
 *   running_mean[c] = (1 - momentum)*running_mean[c] + momentum*mean_c
 *   running_var[c]  = (1 - momentum)*running_var[c]  + momentum*var_c*cnt/(cnt-1)
 * Definition: BatchNorm CUDA implementation walkthrough (jianying88.com/news/30214),
 * §2.1 (forward) and §2.4 (training statistics, running mean).  The page gives
 * no running-variance rule; the unbiased update above is the torch.nn.BatchNorm2d
 * convention that page sets out to replace.
 *   x            [batch, C, HW] dtype
 *   gamma, beta  [C] dtype or NULL
 *   y            [batch, C, HW] dtype, must not overlap x
 *   save_mean, save_rstd        [C] binary32 or NULL
 *   running_mean, running_var   [C] binary32, read and updated in place, or NULL
 *   batch >= 1, C >= 1, HW >= 1, batch*HW >= 2; eps >= 0; 0 <= momentum <= 1
 *   workspace    device memory, 16-byte aligned, at least
 *                bn_fwd_train_workspace_size(batch, C, HW, dtype) bytes, owned
 *                by the caller; calls that share one workspace must be ordered
 *                on the GPU (same stream or events), or they race.
 */
int bn_fwd_train(const void *x, const void *gamma, const void *beta, void *y,
                 float *save_mean, float *save_rstd, float *running_mean,
                 float *running_var, int64_t batch, int64_t C, int64_t HW,
                 float eps, float momentum, int dtype, void *workspace,
                 size_t workspace_bytes, cudaStream_t stream);

/*
 * bn_fwd_train without a workspace argument: it allocates nothing.  No page
 * describes this entry point; it exists for callers that cannot allocate
 * device memory at call time (a runtime that reserves its whole device memory
 * budget at start-up and allows no later allocation, or a component that only
 * receives device pointers from another part of the program).  Same
 * arguments, results and errors as bn_fwd_train, minus the workspace.
 *   The partial statistics live in a fixed array inside the library, sized
 *   for batch * C <= 65536 (512 KB, held on every device that loads the
 *   library until the process exits); larger shapes return
 *   NRM_ERR_TOO_LARGE before anything is launched.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any
 *   stream capture on the device.
 *   All calls on one device share the array: calls that may overlap on the
 *   GPU (unordered streams) race and must not be issued.
 */
int bn_fwd_train_noalloc(const void *x, const void *gamma, const void *beta, void *y,
                         float *save_mean, float *save_rstd, float *running_mean,
                         float *running_var, int64_t batch, int64_t C, int64_t HW,
                         float eps, float momentum, int dtype, cudaStream_t stream);

/*
 * BatchNorm2d inference forward over x[batch, C, HW] (NCHW): every element is
 * normalized with its channel's running statistics,
 *   y = (x - running_mean[c]) / sqrt(running_var[c] + eps) * gamma_c + beta_c
 * Definition: BatchNorm CUDA implementation walkthrough
 * (jianying88.com/news/30214), §2.4 (inference uses the running mean and
 * variance in place of the batch's).  Element-wise: one read of x, one write
 * of y; no workspace.
 *   x            [batch, C, HW] dtype, read only
 *   gamma, beta  [C] dtype or NULL (= 1, 0)
 *   y            [batch, C, HW] dtype, written; must not overlap an input
 *   running_mean, running_var   [C] binary32, read only, required
 *   batch >= 0 (0: no-op), C >= 1, HW >= 1; eps >= 0, finite
 */
int bn_fwd_infer(const void *x, const void *gamma, const void *beta, void *y,
                 const float *running_mean, const float *running_var,
                 int64_t batch, int64_t C, int64_t HW, float eps, int dtype,
                 cudaStream_t stream);

/* Bytes of device workspace bn_bwd needs for this shape (0 on invalid
 * arguments): partial sums, sized as for bn_fwd_train_workspace_size;
 * content on entry does not matter. */
size_t bn_bwd_workspace_size(int64_t batch, int64_t C, int64_t HW, int dtype);

/*
 * BatchNorm2d training backward over NCHW tensors.  With the statistics the
 * training forward saved (mean_c = save_mean[c], rstd_c = save_rstd[c]),
 * xhat = (x - mean_c) * rstd_c and cnt = batch*HW, per channel c:
 *   dbeta[c]  = sum dy,   dgamma[c] = sum dy * xhat
 *   dx = gamma_c * rstd_c * (dy - dbeta[c]/cnt - xhat * dgamma[c]/cnt)
 * Definition: BatchNorm CUDA implementation walkthrough
 * (jianying88.com/news/30214), §3.1; computed in the two stages of its §3.2
 * (channel reduction, then an element-wise broadcast), recomputing xhat from
 * x and the saved statistics instead of storing it.
 *   dy, x        [batch, C, HW] dtype, read only
 *   gamma        [C] dtype or NULL (= 1)
 *   save_mean, save_rstd   [C] binary32, required (as bn_fwd_train wrote them)
 *   dx           [batch, C, HW] dtype, written; must not overlap an input
 *   dgamma, dbeta          [C] binary32, written, or NULL
 *   batch >= 1, C >= 1, HW >= 1
 *   workspace    device memory, 16-byte aligned, at least
 *                bn_bwd_workspace_size(...) bytes; calls sharing one
 *                workspace must be ordered on the GPU.
 */
int bn_bwd(const void *dy, const void *x, const void *gamma, const float *save_mean,
           const float *save_rstd, void *dx, float *dgamma, float *dbeta,
           int64_t batch, int64_t C, int64_t HW, int dtype, void *workspace,
           size_t workspace_bytes, cudaStream_t stream);

/*
 * Synchronized BatchNorm over a batch split across processes (BatchNorm CUDA
 * implementation walkthrough, jianying88.com/news/30214, §7.1: every device
 * reduces its part, the partial statistics are combined across devices, and
 * each device normalizes -- and runs the backward -- with the global ones).
 * The library computes the local parts; the caller exchanges the small
 * binary64 arrays (an all-gather in rank order) and passes them all back.
 * With one part these reduce to bn_fwd_train / bn_bwd.
 *
 * bn_fwd_partial_stats: stats[3*c + {0,1,2}] = (count, mean, M2) of channel c
 *   over this process's x[batch, C, HW], binary64, written.  Where the
 *   planes are packed 16-byte aligned rows, one launch of the training
 *   forward's cluster plan without its normalize: the channel's statistics
 *   folded over the cluster in binary32 (shifted by x[0, c, 0], as in the
 *   forward) and written in binary64; otherwise (or with NRM_PLAN_CTA or
 *   NRM_PLAN_GENERIC forced) per-chunk or per-plane partials folded in
 *   binary64.  workspace: at least bn_fwd_train_workspace_size(...) bytes,
 *   16-byte aligned, scratch.
 * bn_fwd_apply_stats: parts = nparts arrays as above, concatenated in rank
 *   order ([nparts][C][3]); they are combined in that order (Chan's pairwise
 *   rule, binary64), so every process computes the same statistics.  Then as
 *   bn_fwd_train on the local x: y, save_mean/save_rstd (global mean and
 *   1/sqrt(var + eps)) and the running statistics (unbiased with the global
 *   count, which must be at least 2).
 * bn_bwd_partial_sums: sums[2*c + {0,1}] = (sum dy, sum dy * xhat) of channel
 *   c over this process's batch, xhat from save_mean/save_rstd (the global
 *   statistics the forward saved), binary64.  workspace as above.
 * bn_bwd_apply_sums: parts = [nparts][C][2] in rank order, summed in that
 *   order; count = the global batch * HW.  Writes dx of the local batch
 *   (the bn_bwd formula with the global sums and count) and dgamma/dbeta =
 *   the global sums (binary32), or NULL.
 */
int bn_fwd_partial_stats(const void *x, double *stats, int64_t batch, int64_t C, int64_t HW,
                         int dtype, void *workspace, size_t workspace_bytes, cudaStream_t stream);
int bn_fwd_apply_stats(const void *x, const void *gamma, const void *beta, void *y,
                       const double *parts, int64_t nparts, float *save_mean, float *save_rstd,
                       float *running_mean, float *running_var, int64_t batch, int64_t C,
                       int64_t HW, float eps, float momentum, int dtype, cudaStream_t stream);
int bn_bwd_partial_sums(const void *dy, const void *x, const float *save_mean,
                        const float *save_rstd, double *sums, int64_t batch, int64_t C,
                        int64_t HW, int dtype, void *workspace, size_t workspace_bytes,
                        cudaStream_t stream);
int bn_bwd_apply_sums(const void *dy, const void *x, const void *gamma, const float *save_mean,
                      const float *save_rstd, const double *parts, int64_t nparts,
                      int64_t count, void *dx, float *dgamma, float *dbeta, int64_t batch,
                      int64_t C, int64_t HW, int dtype, cudaStream_t stream);

/* Static English text for a status code (never NULL). */
const char *nrm_status_string(int status);

/*
 * Kernel plans of the row operators, for tests and measurements.  The
 * default, NRM_PLAN_AUTO, lets the library pick by N, dtype and alignment.
 */
typedef enum {
    NRM_PLAN_AUTO = 0,
    NRM_PLAN_GENERIC = 1,   /* one CTA per row, scalar, two reads of the row */
    NRM_PLAN_WARP = 2,      /* one warp per row, row held in registers */
    NRM_PLAN_CTA = 3,       /* one CTA per row, row held in registers */
    NRM_PLAN_TMA = 4,       /* persistent CTAs of row groups; each group streams
                               rows into its own ring of shared-memory stages
                               with bulk asynchronous copies */
    NRM_PLAN_PERSIST = 5,   /* persistent CTAs; the next row is loaded into
                               registers while the current one is reduced */
    NRM_PLAN_WRAW = 6,      /* warp per row, the whole row's packs in registers,
                               shuffle-only reductions */
    NRM_PLAN_CLUSTER = 7    /* one row split over the CTAs of a thread-block
                               cluster (`groups` = CTAs per cluster: 2, 4 or
                               8, dividing the row's 16-byte packs); each CTA
                               holds a contiguous slice in registers and the
                               row sums meet in distributed shared memory */
} nrm_plan;

/*
 * Force a plan (and, where non-zero, the CTA size -- for NRM_PLAN_TMA the
 * size of one row group --, the 16-byte packs per thread, and for
 * NRM_PLAN_TMA the shared-memory stages per group, at most 16, and the row
 * groups per CTA, at most 15; for NRM_PLAN_CTA and NRM_PLAN_PERSIST `stages`
 * sets the L2 prefetch of rows ahead: 0 = automatic (one wave of resident
 * CTAs ahead), 1 = off, s >= 2 = s - 1 waves ahead) for every later row-operator call in this
 * process; plan 0 restores automatic choice.  A forced plan that cannot run
 * a given call makes that call return NRM_ERR_UNSUPPORTED.  bn_fwd_train
 * follows the forced plan too: NRM_PLAN_CTA selects its streaming two-kernel
 * plan (per-plane statistics into the workspace, then a dependent launch that
 * normalizes), NRM_PLAN_TMA one cluster of CTAs per channel (shared memory and
 * distributed shared memory, no workspace; as measurement hooks, `stages`
 * of 2, 4, 8 or 16 sets the CTAs per cluster and a non-zero `threads` caps
 * the number of clusters, each then taking several channels in turn, through
 * two buffers per CTA where they fit, else one),
 * NRM_PLAN_PERSIST the one-pass
 * plan (a reset of the workspace's control words, then one kernel whose
 * CTAs take statistics items and normalize items in a fixed interleaved
 * order, x read once from HBM; `stages` sets its L2 prefetch of the chunks
 * a CTA takes next: 0 = automatic, two rounds of the grid ahead, 1 = off,
 * s >= 2 = s - 1 rounds ahead, at most 8), NRM_PLAN_GENERIC the scalar two-kernel plan
 * for any layout; a forced plan the layout does not allow falls back to the
 * next plan that runs; bn_bwd takes NRM_PLAN_GENERIC as its scalar plan,
 * NRM_PLAN_PERSIST as its one-pass plan (dy and x read once) and anything
 * else as its streaming plan where the layout allows it;
 * bn_fwd_infer takes NRM_PLAN_GENERIC as its scalar element-wise kernel.
 * Returns NRM_OK or NRM_ERR_UNSUPPORTED for
 * an unknown plan.  Process-wide; not meant to change while calls run.
 */
int nrm_force_plan(int plan, int threads, int packs, int stages, int groups);

/*
 * Plan, CTA (group) size, packs per thread, stages and groups chosen by this
 * thread's most recent successful call (written to the non-NULL pointers).
 * After a BatchNorm call only the plan is set, as an nrm_plan code: NRM_PLAN_TMA
 * for the cluster plan, NRM_PLAN_CTA for the streaming plans (two kernels,
 * or one element-wise kernel for inference), NRM_PLAN_PERSIST for the
 * one-pass plans (training forward and backward), NRM_PLAN_GENERIC for the
 * scalar plans; the other four values are 0.
 */
void nrm_last_plan(int *plan, int *threads, int *packs, int *stages, int *groups);

/*
 * Kernels that wait on asynchronous copies (NRM_PLAN_TMA) bound every wait:
 * after `tries` unsuccessful polls they give up, record a fault bit, drain
 * their copies in flight (again bounded) and return, leaving the outputs of
 * that call undefined.  Sets the number of polls (default 2^20; 0 makes every
 * such wait give up at once, which tests use to exercise the path) and
 * returns the previous value.  Process-wide.
 */
unsigned nrm_set_wait_limit(unsigned tries);

/*
 * Read the current device's fault word: bit 0 = a kernel gave up a wait,
 * bit 1 = it also gave up draining its copies.  Synchronizes the device
 * first.  Clears the word when `clear` is non-zero.  Returns NRM_OK or
 * NRM_ERR_DEVICE.
 */
int nrm_device_fault(unsigned *bits, int clear);

/*
 * Switch pointer checks on (1) or off (0, the default).  When on, every call
 * asks cudaPointerGetAttributes about each non-NULL pointer and returns
 * NRM_ERR_POINTER, before launching, if one is not device (or managed) memory
 * of the current device.  Costs a few microseconds per call.  Returns the
 * previous setting.
 */
int nrm_set_pointer_checks(int enable);

/*
 * The streaming BatchNorm plans (bn_fwd_train's NRM_PLAN_CTA plan, bn_bwd)
 * read each input twice: once for the channel statistics, once to normalize.
 * With a budget of `bytes` they process the channels in groups whose inputs
 * take at most that many bytes (a launch pair per group), so that the
 * second read of a group can come from L2; 0, the default, makes one group
 * of all channels (measured fastest on GB300).  Returns the previous budget.
 * Process-wide; a measurement hook.
 */
size_t nrm_set_bn_group_bytes(size_t bytes);

#ifdef __cplusplus
}
#endif

#endif /* NRM_H */
