// internal.h -- host-side interfaces between the translation units of
// libkfac_gb300 (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <initializer_list>

#include "common.cuh"

namespace kfac {

// ----------------------------------------------------- tensor-core GEMM
// One problem of the tcgen05 engine: C[M x N] = alpha * op(A) op(B) (+ beta C),
// fp32 accumulation.  Operands are read through tensor maps (see tc_make_map)
// that the caller uploads into device memory with tc_upload_maps; a problem
// names its maps by index and its operand sub-blocks by (row0, col0).
//   TC_KIND_BF16:   a_mn = 1: A stored [K][M] (M contiguous); 0: A stored [M][K].
//                   b_mn = 1: B stored [K][N] (N contiguous); 0: B stored [N][K].
//                   syrk = 1: B is A (Gram matrix of a [K][M] source), only
//                   tiles touching the upper triangle run and only i <= j is written.
//   TC_KIND_TF32X3: K-major only (A [M][K], B [N][K]); an operand names a run
//                   of four maps: hi with 128-row boxes, the (hi, lo) pair map
//                   with 128-row boxes (tc_make_pair_map), hi and lo with 32-row
//                   boxes; 3 MMAs per K slice.
enum TcKind : int { TC_KIND_BF16 = 0, TC_KIND_TF32X3 = 1 };
enum TcEpilogue : int {
    TC_EPI_ACCUM = 0,  // fp32 C[i][j] = beta*C[i][j] + alpha*acc (C read only if beta != 0)
    TC_EPI_STORE = 1,  // C (fp32, optional) and/or Cb (bf16, optional) = alpha*acc
    TC_EPI_SPLIT = 2   // v = alpha*acc + beta*(C + C_lo); C = tf32(v), C_lo = v - C;
                       // optional transposed copy into Ct / Ct_lo (C may then be null)
};

struct TcJob {
    int map_a, map_b;
    int a_mn, b_mn;
    int a_row0, a_col0, b_row0, b_col0;
    int M, N, K;
    int syrk;
    int sym;       // M == N, symmetric result (TF32X3, SPLIT or STORE epilogue): only tiles
                   // on or above the diagonal run and off-diagonal ones also write their
                   // transpose
    int lower;     // TF32X3: only tiles touching the lower triangle (i >= j) run, each
                   // written in full (no mirror)
    int ktri;      // TF32X3: the K range of output tile (tm, tn) starts at the tile's first
                   // column (B upper triangular in its K index: B[j][t] = 0 for t < j)
    int ktril;     // TF32X3: the K range of output tile (tm, tn) ends after the tile's last
                   // row (A lower triangular in its K index: A[i][t] = 0 for t > i)
    int no_split;
    int fine_split; // a latency-critical job: split its K range into pieces of about 12 K tiles
                    // (up to 16 pieces) whatever the rest of the launch
    int dyn;        // the launch hands out its work items dynamically (any job asks for it)
    int epi;
    float alpha, beta;
    float *C;
    float *C_lo;
    long long ldc;
    float *Ct;
    float *Ct_lo;
    long long ldct;
    uint16_t *Cb;
    long long ldcb;
    int f16;       // BF16 kind: both operands fp16 instead of bf16
    int cb_f16;    // Cb receives fp16 bits instead of bf16
    int packed;    // ACCUM: C is a packed upper triangle of a packed_d x packed_d
                   // matrix (entry (i, j) at C[i*packed_d - i*(i+1)/2 + j]; ldc unused)
    int packed_d;
    // STORE epilogue, not symmetric: W[i][j] -= eta * result[i][j] in place
    // (fp32, row stride ldw); C may then be null
    float *W;
    long long ldw;
    float eta;
    // BF16 SYRK of a convolution read straight from its NHWC input through an
    // im2col tensor map (map_a): K runs over output pixels, the MN index over
    // d = (r * k + s) * c + channel.  c is a multiple of 64.
    int im2col;
    int im_c, im_k, im_stride, im_pad, im_wo, im_howo;
};

// Tensor map of a row-major [rows][cols] matrix (ld elements) for the engine:
// 128-byte swizzle, box 128 bytes wide and box_rows rows (default 128).  The
// same map serves a K-major and an MN-major operand (the kernel picks the box
// coordinates).  A tf32x3 operand is a run of four maps: hi and lo with
// 128-row boxes, then hi and lo with 32-row boxes (B of narrow tiles).
bool tc_make_map(CUtensorMap *m, int kind, const void *ptr, long long ld, int rows, int cols, int box_rows = 0,
                 bool f16 = false);
// Tensor map of an fp32 (hi, lo) pair of row-major [rows][cols] matrices
// (ld elements each; lo at a fixed byte offset after hi) as one 3-D tensor
// [2][rows][cols]: a box is 128-byte rows x box_rows for both planes, hi
// landing first and lo right after it (one copy instead of two).
bool tc_make_pair_map(CUtensorMap *m, const float *hi, const float *lo, long long ld, int rows, int cols,
                      int box_rows);
// Im2col tensor map of a bf16 NHWC tensor [n][h][w][c] for a square k x k
// convolution (stride, pad): 64 channels x 128 output pixels per load,
// 128-byte swizzle.  Requires c % 64 == 0 and a 16-byte aligned base.
bool tc_make_im2col_map(CUtensorMap *m, const void *x, int n, int h, int w, int c, int k, int stride, int pad,
                        bool f16 = false);
// Copies host-built maps into device memory (128-byte aligned) on the stream.
kfac_status tc_upload_maps(const CUtensorMap *maps, int n, CUtensorMap *dev, cudaStream_t st);
// Workspace needed by tc_run for these jobs (split-K partials, counters).
size_t tc_workspace_bytes(const TcJob *jobs, int njobs, int kind, int max_ctas = 0);
// Enqueue the jobs (one or more persistent launches).  `err` is a device int
// that collects timeout codes.
// `max_ctas` (0: the SM count) caps the persistent grid, e.g. to leave SMs to
// a concurrent stream.
kfac_status tc_run(const TcJob *jobs, int njobs, int kind, const CUtensorMap *dev_maps, Arena &ws,
                   int *err, cudaStream_t st, int max_ctas = 0);

// ----------------------------------------------------- CUDA-core GEMM (fp32)
// C[M x N] = alpha * op(A) op(B) + beta * C, fp32.
//   ta = 0: A stored [M][K];  ta = 1: A stored [K][M]
//   tb = 0: B stored [K][N];  tb = 1: B stored [N][K]
//   upper = 1: only entries i <= j are written (and only tiles touching them run)
//   Ct (optional): also writes the transposed result Ct[j][i]
struct SgJob {
    const float *A;
    long long lda;
    int ta;
    const float *B;
    long long ldb;
    int tb;
    float *C;
    long long ldc;
    float *Ct;
    long long ldct;
    int M, N, K;
    float alpha, beta;
    int upper;
    float *W;        // W[i][j] -= eta * result[i][j] in place (row stride ldw); C may then be null
    long long ldw;
    float eta;
    int packed_d;    // upper: C is a packed upper triangle of this order (0: row-major, ldc)
};
// err: the call's device error word (ERR_NONFINITE is ORed in when a stored
// value is NaN or infinite), or null
kfac_status sg_run(const SgJob *jobs, int njobs, int *err, cudaStream_t st);

// ----------------------------------------------------- patches / reductions
// bf16 or fp32 im2col into P[M][ldp] (columns d..ldp-1 untouched).
struct Im2colJob {
    const void *x;
    int n, h, w, c, kh, kw, sh, sw, ph, pw;
    int ho, wo;
    int append_one;
    void *P;
    long long ldp;
};
// dtype KFAC_BF16 / KFAC_F16 (16-bit elements) or KFAC_F32
kfac_status im2col_run(const Im2colJob *jobs, int njobs, int dtype, cudaStream_t st);

// Bias row/column of an FC factor with append_one: for a bf16 source x[M][c]
// (no patch matrix formed), updates F[i][c] (i < c) with alpha * colsum_i
// and F[c][c] with alpha * M, both scaled by beta first.
struct ColsumJob {
    const uint16_t *x;
    long long M;
    int c;
    float *F;
    long long ldf;
    float alpha, beta;
    int f16;       // x holds fp16 (else bf16)
    int packed;    // F is a packed upper triangle of order c + 1 (ldf unused)
};
// Column sums of each job in row slabs with partials in `partial` (device,
// colsum_partial_floats(jobs) floats), then a fixed-order finish: results
// are bitwise reproducible.
size_t colsum_partial_floats(const ColsumJob *jobs, int njobs);
kfac_status colsum_run(const ColsumJob *jobs, int njobs, float *partial, cudaStream_t st);

// True when p is device memory of the current device or managed memory (or
// null); the entry points reject every other operand before enqueueing.
bool on_this_device(const void *p);
bool all_on_this_device(std::initializer_list<const void *> ps);

// ----------------------------------------------------- inversion
struct InvMatrix {
    const float *F;   // factor, upper triangle read
    long long ldf;
    int d;
    float *out;       // full symmetric inverse
    long long ldo;
    uint16_t *out_bf16;
    long long ldo_bf16;
    int packed;       // F is a packed upper triangle (ldf unused)
    int copy_f16;     // out_bf16 receives fp16 bits
};
size_t inv_workspace_bytes(const InvMatrix *mats, int nmats);
// damp[k] (device) is added to the diagonal of matrix k; info[k] receives 0
// or the 1-based index of the first bad pivot.
kfac_status inv_run(const InvMatrix *mats, int nmats, const float *damp_dev, int *info_dev,
                    Arena &ws, cudaStream_t st);
// Traces -> pi-split damping for each layer (pairs A, G) into damp_dev[2l], [2l+1].
kfac_status damping_run(const InvMatrix *mats, int nlayers, float gamma, int pi_split,
                        float *damp_dev, cudaStream_t st);

}  // namespace kfac
