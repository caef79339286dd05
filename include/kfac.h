/*
 * kfac.h -- C ABI of the GB300 (sm_103a) K-FAC curvature-step library
 * (libkfac_gb300.so).
 *
 * The library implements the per-layer Kronecker-factored curvature step of
 * Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
 * Kronecker-Factored Approximate Curvature for Deep Convolutional Neural
 * Networks" (section 3.2, Eq. 4-7, and the diagonal BatchNorm Fisher of
 * section 1):
 *   kfac_factor_update   builds A = E[a a^T] / G = E[g g^T] and folds it into a
 *                        running average                      (Eq. 5)
 *   kfac_damp_invert     damps both factors of a layer (pi-split Tikhonov) and
 *                        inverts them                           (Eq. 6)
 *   kfac_precondition    G^-1 grad A^-1                         (Eq. 7)
 *   kfac_bn_diag_fisher  diagonal Fisher of BatchNorm parameters and the
 *                        damped diagonal preconditioned gradient
 *
 * Conventions shared by every entry point:
 *   - Every buffer pointer inside a descriptor is a DEVICE pointer on the
 *     current CUDA device, owned by the caller; descriptor arrays themselves
 *     are HOST memory and may be freed when the call returns.
 *   - The library allocates no device memory.  Calls that need scratch take a
 *     caller-owned device `workspace` of at least the size the matching
 *     *_workspace_size query returns (256-byte aligned); its contents need no
 *     initialisation and are clobbered.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous: results are ready once the stream has
 *     reached that point.  The library keeps no global state beyond the
 *     per-device streams and events of kfac_damp_invert (below); concurrent
 *     calls on different streams with disjoint buffers and workspaces are
 *     allowed.
 *   - KFAC_ERR_INVALID / KFAC_ERR_UNSUPPORTED / KFAC_ERR_WORKSPACE are
 *     returned BEFORE anything is enqueued (outputs untouched).  Every
 *     operand must be memory of the current device (or managed memory):
 *     host memory or another GPU's memory gives KFAC_ERR_INVALID (checked
 *     last, right before the call enqueues its work).
 *     KFAC_ERR_CUDA reports a launch failure (cudaGetLastError after a
 *     launch); the stream may then hold part of the work.
 *   - Matrices are row-major with an explicit leading dimension (elements).
 *     bf16 values are passed as uint16_t bit patterns.
 *   - Device error word: the first int32 of the workspace of
 *     kfac_factor_update, kfac_damp_invert and kfac_precondition.  Each call
 *     sets it to 0 on its stream before its kernels; its kernels OR bits into
 *     it, which the caller reads after synchronising the stream (the call's
 *     return status cannot report them: the kernels run after it returns):
 *       KFAC_ERRW_NONFINITE (16): a value the call wrote to an output (a
 *         factor, an inverse or one of the inversion's intermediate blocks,
 *         a preconditioned gradient, an updated weight) is NaN or infinite --
 *         e.g. the input held NaN/Inf or the statistic overflowed fp32 --
 *         or an entry of the upper triangle of a factor that
 *         kfac_damp_invert reads is.  The values are written as computed
 *         (NaN stays NaN); nothing is clamped.  Layers of the same call whose
 *         inputs are finite are not affected, but the bit does not say which
 *         layer it was (kfac_damp_invert's info does, per factor).
 *       1, 2, 4 (KFAC_ERRW_TIMEOUT_*): a wait of the tensor-core engine on a
 *         shared-memory barrier (operand stage, free stage, accumulator) ran
 *         past its limit (about 2 s; never expected in a healthy run).  The
 *         CTA then stops issuing work, waits (bounded) for the copies and
 *         products it already issued, releases its tensor memory and exits
 *         without trapping; 8 is set when that drain wait ran out too.  The
 *         call's outputs are then undefined.
 *     A word of 0 means no kernel of the call saw either condition.
 */
#ifndef KFAC_GB300_H
#define KFAC_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KFAC_OK = 0,
    KFAC_ERR_INVALID = 1,      /* null pointer, non-positive size, ld < width, ... */
    KFAC_ERR_UNSUPPORTED = 2,  /* valid but not implemented (dtype, shape limit)  */
    KFAC_ERR_NOT_PD = 3,       /* reserved for host-side reporting of info[]      */
    KFAC_ERR_CUDA = 4,         /* a CUDA launch or runtime call failed             */
    KFAC_ERR_WORKSPACE = 5     /* workspace missing, misaligned or too small      */
} kfac_status;

typedef enum { KFAC_BF16 = 0, KFAC_F32 = 1, KFAC_F16 = 2 } kfac_dtype;

/* Storage of a symmetric fp32 factor (only its upper triangle is stored or
 * read):
 *   KFAC_LAYOUT_FULL          row-major [d][ld], entry (i, j) at F[i*ld + j];
 *   KFAC_LAYOUT_PACKED_UPPER  the upper triangle row after row, d(d+1)/2
 *                             floats: entry (i, j), i <= j, at
 *                             F[i*d - i*(i+1)/2 + j]  (row i holds j = i..d-1);
 *                             the ld argument is ignored.
 * The packed form halves a factor's footprint (Osawa et al. section 1: the
 * symmetry of the Kronecker factors is exploited to reduce overhead). */
typedef enum { KFAC_LAYOUT_FULL = 0, KFAC_LAYOUT_PACKED_UPPER = 1 } kfac_layout;

/* Bits of the device error word (see above). */
enum {
    KFAC_ERRW_TIMEOUT_OPERAND = 1,
    KFAC_ERRW_TIMEOUT_STAGE = 2,
    KFAC_ERRW_TIMEOUT_ACCUM = 4,
    KFAC_ERRW_TIMEOUT_DRAIN = 8,
    KFAC_ERRW_NONFINITE = 16
};

/* Human-readable name of a status code (static string, never NULL). */
const char *kfac_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int kfac_version(void);

/* Number of kernel launches this library has enqueued in this process so far
 * (a diagnostic counter; every entry point adds the launches it makes). */
long long kfac_launch_count(void);

/* Optional per-kernel timing (diagnostic, off by default).  While enabled,
 * every kernel launch the library makes is bracketed by CUDA events recorded
 * on its launch stream (up to 65536 launches).  kfac_timing_read waits for
 * those events, writes for each kernel kind k < n the total device time in
 * milliseconds (ms[k]) and the number of launches (launches[k]), and clears
 * the record; it returns KFAC_OK or KFAC_ERR_CUDA.  kfac_timing_enable
 * returns the previous setting.  Kind names: kfac_timing_kind_name(k) ("" past
 * the last kind).  Launches enqueued during stream capture are recorded as
 * external event nodes of the graph: read the record after the graph has run. */
int kfac_timing_enable(int on);
int kfac_timing_read(double *ms, long long *launches, int n);
const char *kfac_timing_kind_name(int k);
/* The same record launch by launch, in enqueue order: for the first n launches
 * the start (ms after the first recorded launch's start), the duration (ms),
 * the kernel kind and the launch stream's handle (a value that tells streams
 * apart, nothing more); any output may be NULL.  Clears the record and
 * returns the number of launches it held (-1 if an event query failed). */
int kfac_timing_read_launches(double *start_ms, double *dur_ms, int *kind, unsigned long long *stream, int n);

/* ======================================================================
 * kfac_factor_update -- Kronecker factor statistic + running average.
 *
 * Osawa et al. section 3.2, Eq. 5: A_{l-1} is built from the layer's input
 * activations, G_l from the gradients of the layer's output.  For each
 * descriptor the call forms the patch matrix P [M x d] of the source tensor
 * and updates the UPPER triangle (i <= j) of the fp32 factor F in place:
 *
 *     F[i][j] <- beta * F[i][j] + alpha * sum_m P[m][i] * P[m][j]
 *
 * The running average F <- xi F + (1 - xi) P^T P / M is alpha = (1 - xi)/M,
 * beta = xi; accumulating one statistic over several chunks of rows uses
 * beta = xi on the first chunk and beta = 1 afterwards with alpha = (1-xi)/M_total.
 * Entries strictly below the diagonal are neither read nor written.
 *
 * Patch matrix (im2col; row m = (img*Ho + ho)*Wo + wo):
 *   P[m][(r*kw + s)*c + ch] = x[img][ho*stride_h - pad_h + r][wo*stride_w - pad_w + s][ch]
 *   (zero outside the image), Ho = (h + 2*pad_h - kh)/stride_h + 1 (same for Wo),
 *   and when append_one != 0 a last column of ones (an FC bias), so
 *   d = kh*kw*c + (append_one ? 1 : 0).
 * A fully connected layer or an output-gradient source [M x C] is
 * h = w = kh = kw = stride = 1, pad = 0, n = M rows.
 *
 * Fields:
 *   dtype   KFAC_BF16 or KFAC_F16 (tensor cores, fp32 accumulation; the
 *           paper computes in half precision) or KFAC_F32 (fp32 CUDA cores)
 *   x       device, dense NHWC [n][h][w][c] of dtype (channel stride 1)
 *   F, ldf  device fp32 factor in `layout`: KFAC_LAYOUT_FULL [d][ldf] with
 *           ldf >= d, or KFAC_LAYOUT_PACKED_UPPER (d(d+1)/2 floats, ldf
 *           ignored); its upper triangle is updated
 *   layout  kfac_layout of F (a trailing field: zero-initialised = FULL)
 * Errors: INVALID for null x/F, n,h,w,c,kh,kw,stride < 1, pad < 0, Ho/Wo < 1,
 *   ldf < d (full layout), an unknown dtype or layout; UNSUPPORTED for
 *   d > 65536 or more than 2^31 rows.
 * Workspace: kfac_factor_update_workspace_size(descs, count) bytes.
 * ==================================================================== */
typedef struct {
    int32_t dtype;
    const void *x;
    int32_t n, h, w, c;
    int32_t kh, kw, stride_h, stride_w, pad_h, pad_w;
    int32_t append_one;
    float *F;
    int64_t ldf;
    float alpha, beta;
    int32_t layout;
} kfac_factor_desc;

size_t kfac_factor_update_workspace_size(const kfac_factor_desc *descs, int count);
kfac_status kfac_factor_update(const kfac_factor_desc *descs, int count,
                               void *workspace, size_t workspace_bytes, void *stream);

/* ======================================================================
 * kfac_damp_invert -- damped inverses of both factors of each layer.
 *
 * Osawa et al. section 3.2, Eq. 6: (G (x) A)^-1 = G^-1 (x) A^-1.  Damping
 * (the paper states none; Tikhonov split by pi as in the K-FAC paper it
 * cites):
 *     pi = sqrt((tr A / dA) / (tr G / dG)),
 *     damp_A = pi * sqrt(gamma),  damp_G = sqrt(gamma) / pi      (pi_split != 0)
 *     damp_A = damp_G = sqrt(gamma)                              (pi_split == 0)
 * and writes the FULL symmetric fp32 inverses (both triangles, exactly
 * symmetric)
 *     A_inv = (A + damp_A I)^-1,  G_inv = (G + damp_G I)^-1
 * computed in fp32 through a Cholesky factorisation X = L L^T (left-looking,
 * 128-wide block columns; each 128 x 128 diagonal block factored and
 * inverted by one CTA), the triangular inverse W = L^-1 (recursive 2 x 2
 * blocking) and X^-1 = W^T W.  The block products run on tensor cores as
 * three tf32 products per slice on (hi, lo) splits of the fp32 operands with
 * fp32 accumulation.  Only the upper triangles of A and G are read.
 *
 * Streams: the call is ordered on `stream` as a whole.  Its middle part forks
 * onto library-owned streams of the current device (the longest chains at
 * high priority, the rest at low priority; created with their events on the
 * first call on a device) and joins back into `stream`, so stream capture
 * records a graph with parallel branches.  Make the first call on a device
 * outside stream capture.  Optional 16-bit copies of the inverses (bf16, or
 * fp16 when copy_dtype is KFAC_F16) are written when the *_bf16 pointers are
 * non-NULL (their ld must be a multiple of 8 elements and their base 16-byte
 * aligned, for the tensor-core preconditioner).  A and G may be stored in
 * either kfac_layout (layout_A, layout_G; the lda/ldg of a packed factor are
 * ignored); the inverses are always full row-major.
 *
 * Device outputs besides the inverses:
 *   info   int32 [2*count] (may be NULL): info[2l] for A of layer l,
 *          info[2l+1] for its G; 0 = success, k+1 = the k-th pivot was not
 *          positive or not finite (matrix not positive definite); the
 *          corresponding inverse is then undefined.  The call itself still
 *          returns KFAC_OK: read info after synchronising the stream.
 *   damp   float [2*count] (may be NULL): the damp_A, damp_G applied.
 * Errors: INVALID for null A/G/A_inv/G_inv, dA/dG < 1, ld < d (full layouts
 *   and the outputs), gamma < 0, an unknown layout or copy_dtype;
 *   UNSUPPORTED for d > 16384 or a 16-bit copy's ld not a multiple of 8.
 * Workspace: kfac_damp_invert_workspace_size(descs, count) bytes.
 * ==================================================================== */
typedef struct {
    const float *A; int32_t dA; int64_t lda;
    const float *G; int32_t dG; int64_t ldg;
    float *A_inv; int64_t ld_ainv;
    float *G_inv; int64_t ld_ginv;
    uint16_t *A_inv_bf16; int64_t ld_ainv_bf16;   /* optional 16-bit copy */
    uint16_t *G_inv_bf16; int64_t ld_ginv_bf16;   /* optional 16-bit copy */
    int32_t layout_A, layout_G;                   /* kfac_layout of A and G */
    int32_t copy_dtype;                           /* KFAC_BF16 (0) or KFAC_F16 */
} kfac_invert_desc;

size_t kfac_damp_invert_workspace_size(const kfac_invert_desc *descs, int count);
kfac_status kfac_damp_invert(const kfac_invert_desc *descs, int count, float gamma,
                             int pi_split, int32_t *info, float *damp,
                             void *workspace, size_t workspace_bytes, void *stream);

/* ======================================================================
 * kfac_precondition -- preconditioned gradient of each layer.
 *
 * Osawa et al. section 3.2, Eq. 7 in row-major form: for grad [dG x dA],
 *     out = G_inv * grad * A_inv            (out fp32 [dG][ld_out])
 * i.e. (G (x) A)^-1 vec(grad) with symmetric inverses.  A_inv and G_inv are
 * read as FULL matrices (kfac_damp_invert writes both triangles).
 * dtype KFAC_BF16: G_inv, A_inv, grad are bf16 (tensor cores, fp32
 *   accumulation; the intermediate grad*A_inv is rounded to bf16); each ld
 *   must be a multiple of 8 and each base 16-byte aligned.  Rows that start
 *   on 128-byte boundaries (ld a multiple of 64) are read in whole 128-byte
 *   segments and run faster (FC 4096: 0.36 against 0.31 ms); fp32 outputs
 *   whose rows start on 16-byte boundaries are stored 16 bytes at a time.
 * dtype KFAC_F16: the same with fp16 operands (the intermediate is rounded
 *   to fp16).
 * dtype KFAC_F32: all operands fp32 (CUDA cores).
 * Fused step on the weights (Osawa et al. section 3.2, Eq. 8): when w is not
 *   NULL, the epilogue of the second product also applies
 *       w <- w - eta * out               (w fp32 [dG][ld_w], in place)
 *   with the fp32 value of out before it is stored; out may then be NULL
 *   (the preconditioned gradient is not kept).  w must not overlap any other
 *   operand.  Zero-initialised trailing fields (w = NULL) leave w alone.
 * Errors: INVALID for null G_inv/A_inv/grad, both out and w NULL, d < 1,
 *   ld < width; UNSUPPORTED for a bf16 ld/alignment violation or d > 65536.
 * Workspace: kfac_precondition_workspace_size(descs, count, dtype) bytes.
 * ==================================================================== */
typedef struct {
    int32_t dG, dA;
    const void *G_inv; int64_t ld_ginv;
    const void *A_inv; int64_t ld_ainv;
    const void *grad;  int64_t ld_grad;
    float *out;        int64_t ld_out;    /* may be NULL when w is set */
    float *w;          int64_t ld_w;      /* optional: the layer's weights */
    float eta;                            /* learning rate of the step on w */
} kfac_precond_desc;

size_t kfac_precondition_workspace_size(const kfac_precond_desc *descs, int count, int dtype);
kfac_status kfac_precondition(const kfac_precond_desc *descs, int count, int dtype,
                              void *workspace, size_t workspace_bytes, void *stream);

/* ======================================================================
 * kfac_precondition_noalloc -- kfac_precondition without a caller workspace.
 *
 * The paper has no counterpart: this is a service for callers that cannot
 * allocate device memory -- host frameworks that own all device memory
 * through their own pool and do not let a library call cudaMalloc, step
 * loops in which cudaMalloc's implicit device-wide synchronisation would
 * stall the pipeline, and embedded callers whose device-memory budget is
 * fixed at start-up.  Same arguments, results and errors as
 * kfac_precondition (bitwise the same outputs), but the scratch comes from a
 * fixed array in the library's own device memory, kfac_noalloc_scratch_bytes()
 * bytes (32 MiB), held by every GPU that loads the library until the process
 * exits.  The call allocates nothing (no cudaMalloc, cudaFree or allocating
 * library routine).
 *   - KFAC_ERR_WORKSPACE when kfac_precondition_workspace_size() of the
 *     arguments exceeds kfac_noalloc_scratch_bytes() (split the layers over
 *     several calls, or use kfac_precondition with a workspace).
 *   - Set-up: the first call on a device (and the first call after that
 *     device's context was re-created, e.g. by cudaDeviceReset) looks up the
 *     array's device address with that device current (a runtime query, no
 *     allocation).  Make that first call before any stream capture begins.
 *   - All calls on a device share the one array and its contents persist
 *     from call to call (each call clears the parts that must start at zero:
 *     the error word, which is the array's first int32, and the split-K
 *     counters).  Calls whose GPU work overlaps (e.g. on two streams without
 *     ordering between them) race on the array: order them on one stream.
 * ==================================================================== */
size_t kfac_noalloc_scratch_bytes(void);
kfac_status kfac_precondition_noalloc(const kfac_precond_desc *descs, int count, int dtype,
                                      void *stream);

/* ======================================================================
 * kfac_bn_diag_fisher -- diagonal Fisher of BatchNorm parameters.
 *
 * Osawa et al. section 1 (contributions): the Fisher of BatchNormalization
 * layers is approximated as diagonal.  For each descriptor, from per-sample
 * gradients x [n_samples][C] (fp32, row-major, dense):
 *     F_c       <- xi * F_c + (1 - xi) * (1/n) sum_i x_ic^2   (xi = 0: plain)
 *     grad_mean_c = (1/n) sum_i x_ic
 *     precond_c   = grad_mean_c / (F_c + gamma)
 * F is read only when xi != 0.  grad_mean may be NULL.  The reduction order
 * is fixed, so results are bitwise reproducible run to run.
 * Errors: INVALID for null x/F/precond, C < 1, n_samples < 1, gamma < 0.
 * No workspace.
 * ==================================================================== */
typedef struct {
    const float *x;
    int32_t C;
    float *F;
    float *grad_mean;
    float *precond;
} kfac_bn_desc;

kfac_status kfac_bn_diag_fisher(const kfac_bn_desc *descs, int count, int n_samples,
                                float gamma, float xi, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* KFAC_GB300_H */
