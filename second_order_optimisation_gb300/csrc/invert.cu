// invert.cu -- damped inversion of the Kronecker factors in fp32.
//
// Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
// Kronecker-Factored Approximate Curvature ...", section 3.2, Eq. 6: the
// inverse of G (x) A is G^-1 (x) A^-1, so each factor is inverted on its own.
// Damping (not stated by the paper; the pi-split Tikhonov form of the K-FAC
// method it builds on):
//     pi = sqrt((tr A/dA) / (tr G/dG)),  damp_A = pi sqrt(gamma),  damp_G = sqrt(gamma)/pi.
//
// Algorithm: Cholesky X = L L^T of X = sym(F) + damp I, the triangular
// inverse W = L^-1, and X^-1 = W^T W (the order of a Cholesky-based
// inversion: factor, triangular inverse, product of the inverse factors).  X
// is padded with an identity block to a multiple of 128 (the inverse of
// diag(X, I) is diag(X^-1, I)).  The Cholesky factor is formed left-looking
// in 128-wide block columns (gen_chain), so every Schur-complement column
// comes from Cholesky panels (no growth) and the inverse keeps fp32-level
// accuracy on damped factors with condition numbers around 1e4; the 128 x 128
// diagonal blocks are factored and inverted by one CTA each (diag_kernel).
// The triangular inverse is recursive 2 x 2 blocking, the final product one
// triangular-aware product that writes the caller's symmetric fp32 inverse
// (and its bf16 copy) directly.  The products run on tcgen05 with three tf32
// products per slice (hi*hi + hi*lo + lo*hi) and fp32 accumulation on (hi, lo)
// pairs (hi exactly representable in tf32, hi + lo the fp32 value).  The
// matrices advance in batched rounds, one launch per round (schedule_rounds);
// the longest chains and the rest run as two concurrent groups (InvGroup).
// A pivot that is not positive and finite records its 1-based index in
// info[matrix]; nothing traps, and every wait on a barrier has a time limit.
#include <algorithm>
#include <cfloat>
#include <functional>
#include <memory>
#include <mutex>
#include <vector>

#include "internal.h"

namespace kfac {

namespace {

constexpr int NB = 128;    // block width of the sweep
#ifndef KFAC_INV_FUSED_PANEL
#define KFAC_INV_FUSED_PANEL 0
#endif
// The Cholesky panel below each diagonal block: formed by the diag kernel's
// other CTAs (1), or by a separate engine launch (0).  A tuning constant that
// may be set at build time.  Measured on the ResNet-50 factor set: the fused
// form widens each diag launch to one CTA per panel block, and those CTAs
// (each redoing the 128 x 128 factorisation) wait for SMs held by the second
// group's engine launches: 9.1 ms against 8.5 ms for the engine panel.
constexpr bool FUSED_PANEL = KFAC_INV_FUSED_PANEL;
#ifndef KFAC_INV_LOOKAHEAD
#define KFAC_INV_LOOKAHEAD 1
#endif
// Lookahead (see gen_chain): the rest of each Cholesky block column on the
// side stream, off the chain of diagonal blocks.  A tuning constant that may
// be set at build time.
constexpr bool LOOKAHEAD = KFAC_INV_LOOKAHEAD && !KFAC_INV_FUSED_PANEL;
#ifndef KFAC_INV_SIDE_DIAG_BULK
#define KFAC_INV_SIDE_DIAG_BULK 1
#endif
// With the lookahead: the diagonal update of block k + 1 keeps only its last
// term L[k+1, k] L[k+1, k]^T on the chain, the earlier terms run with the
// side update of column k (1); or the whole sum on the chain, split finely
// over K (0).  A tuning constant that may be set at build time.
constexpr bool SIDE_DIAG_BULK = KFAC_INV_SIDE_DIAG_BULK;
#ifndef KFAC_INV_SIDE_BULK
#define KFAC_INV_SIDE_BULK 1
#endif
// With the lookahead and SIDE_DIAG_BULK: the side update of block column
// k + 1 keeps only its last term L[k+2:, k] L[k+1, k]^T, and the earlier
// terms (of the column and of its diagonal block) run on a third stream as
// soon as the panel of column k - 1 is done (1); or the whole update runs on
// the side stream after the first panel block of k (0).  A tuning constant
// that may be set at build time.
constexpr bool SIDE_BULK = KFAC_INV_SIDE_BULK && SIDE_DIAG_BULK && LOOKAHEAD;
#ifndef KFAC_INV_BULK_REST
#define KFAC_INV_BULK_REST 0
#endif
// The bulk stream for the second (low-priority) group's chains too (1), or
// for the critical group's only (0).  A tuning constant that may be set at
// build time.
constexpr bool BULK_REST = KFAC_INV_BULK_REST;
#ifndef KFAC_INV_EARLY_TRI
#define KFAC_INV_EARLY_TRI 0
#endif
#ifndef KFAC_INV_EARLY_TRI_MIN_NB
#define KFAC_INV_EARLY_TRI_MIN_NB 8
#endif
// Early triangular inverse (see gen_chain): for a matrix of at least
// EARLY_TRI_MIN_NB block columns and at least 3/4 as many as the call's
// widest, each node of W = L^-1 runs on a third stream as soon as the
// Cholesky columns it reads are done, instead of after the whole
// factorisation.  Tuning constants that may be set at build time.  Measured:
// three 4608-wide factors alone 5.50 -> 5.25 ms, but the ResNet-50 factor set
// 7.06 -> 7.35 ms (graph; 8.4 ms unless the process allows more than the
// default 8 hardware queues): there the second group's work already fills
// the critical group's tail, and the inverse's products moved into the
// factorisation slow its chain.  Off by default.
constexpr bool EARLY_TRI = KFAC_INV_EARLY_TRI && LOOKAHEAD;
constexpr int EARLY_TRI_MIN_NB = KFAC_INV_EARLY_TRI_MIN_NB;
constexpr int MAT_MAX = 224;
// tensor maps of one matrix: X, Wt, LT pairs, each as hi and the (hi, lo)
// pair with 128-row boxes, and hi / lo with 32-row boxes
constexpr int MAPS_PER_MATRIX = 12;

inline int padded(int d) { return (int)ceil_div(d, NB) * NB; }

__device__ __forceinline__ float tf32_hi(float v) {
    return __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
}

// ---------------------------------------------------------------- damping

struct DampParams {
    const float *A[MAT_MAX / 2];
    const float *G[MAT_MAX / 2];
    long long lda[MAT_MAX / 2], ldg[MAT_MAX / 2];  // -1: packed upper triangle
    int dA[MAT_MAX / 2], dG[MAT_MAX / 2];
    int n;
    float gamma;
    int pi_split;
    float *damp;
    int base;
};

__global__ void __launch_bounds__(256) damping_kernel(const __grid_constant__ DampParams P) {
    pdl_wait();
    pdl_trigger();
    __shared__ float ra[256], rg[256];
    const int l = blockIdx.x;
    float ta = 0.f, tg = 0.f;
    // entry (i, i): row-major i*ld + i, or packed i*d - i*(i+1)/2 + i
    auto diag = [](int i, long long ld, int d) {
        return ld < 0 ? (long long)i * d - (long long)i * (i + 1) / 2 + i : (long long)i * ld + i;
    };
    for (int i = threadIdx.x; i < P.dA[l]; i += 256) ta += P.A[l][diag(i, P.lda[l], P.dA[l])];
    for (int i = threadIdx.x; i < P.dG[l]; i += 256) tg += P.G[l][diag(i, P.ldg[l], P.dG[l])];
    ra[threadIdx.x] = ta;
    rg[threadIdx.x] = tg;
    __syncthreads();
    for (int s = 128; s > 0; s >>= 1) {
        if (threadIdx.x < s) {
            ra[threadIdx.x] += ra[threadIdx.x + s];
            rg[threadIdx.x] += rg[threadIdx.x + s];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const float sg = sqrtf(P.gamma);
        float da = sg, dg = sg;
        if (P.pi_split) {
            const float na = ra[0] / (float)P.dA[l], ng = rg[0] / (float)P.dG[l];
            const float pi = sqrtf(na / ng);
            // a zero or non-finite trace leaves pi undefined: fall back to 1
            if (na > 0.f && ng > 0.f && isfinite(pi) && pi > 0.f) {
                da = pi * sg;
                dg = sg / pi;
            }
        }
        P.damp[2 * (P.base + l)] = da;
        P.damp[2 * (P.base + l) + 1] = dg;
    }
}

// ------------------------------------------------------------- prepare

struct TileMat {
    const float *F;   // factor (upper triangle read)
    long long ldf;    // -1: packed upper triangle (entry (i, j) at i*d - i*(i+1)/2 + j)
    float *Xh, *Xl;   // working pair [dp][dp]
    float *Dh, *Dl;   // diagonal 128 x 128 blocks, stacked [dp][128]
    int d, dp;
    int damp_idx;
    int tiles;        // 64-wide tiles per side
    int vec_f;        // F rows take 16-byte accesses
};

struct TileParams {
    TileMat m[MAT_MAX];
    int begin[MAT_MAX + 1];
    int n;
    const float *damp;
    int *error;       // the call's error word: ERR_NONFINITE for a NaN / inf factor entry
};

constexpr int TT = 64;  // prep tile

// The upper tile pair (si <= sj) of this CTA: matrix index and tile coordinates.
__device__ __forceinline__ const TileMat &tile_of(const TileParams &P, int &si, int &sj) {
    int lo = 0, hi = P.n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.begin[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    const TileMat &q = P.m[lo];
    int t = blockIdx.x - P.begin[lo], i = 0;
    while (t >= q.tiles - i) { t -= q.tiles - i; ++i; }
    si = i;
    sj = i + t;
    return q;
}

// X = lower part of sym(F) + damp I as a (hi, lo) pair on [d, d], identity on
// the padding: the blocks below the diagonal 128-blocks go into X, the
// diagonal 128-blocks into D (lower part, zeros above; the diag kernel reads
// them from there and writes W_kk over X's block).  X's diagonal blocks and
// everything above them are not written: no product reads them.  One
// CTA per upper 64 x 64 tile pair: the upper tile of F is read once (16-byte
// pieces where the rows allow) and written transposed to its lower position.
__global__ void __launch_bounds__(256) prep_kernel(const __grid_constant__ TileParams P) {
    pdl_wait();
    pdl_trigger();
    __shared__ float t[TT][TT + 1];
    int si, sj;
    const TileMat &q = tile_of(P, si, sj);
    const int tid = threadIdx.x, rr = tid >> 4, c4 = (tid & 15) * 4;
    bool bad = false;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const int r = rr + 16 * p, i = si * TT + r, j = sj * TT + c4;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (i < q.d) {
            const bool packed = q.ldf < 0;
            const float *src =
                q.F + (packed ? (long long)i * q.d - (long long)i * (i + 1) / 2 : (long long)i * q.ldf) + j;
            if (!packed && q.vec_f && j + 3 < q.d) {
                const float4 x = *reinterpret_cast<const float4 *>(src);
                v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
            } else {
                // (a packed row holds only j >= i: the lower half of a
                // diagonal tile is not read)
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (j + u < q.d && (!packed || j + u >= i)) v[u] = src[u];
            }
        }
        // a NaN or infinite entry of the upper triangle (the part read) is
        // reported; the lower half of a diagonal tile is not part of F
#pragma unroll
        for (int u = 0; u < 4; ++u) bad |= (si != sj || j + u >= i) && !(fabsf(v[u]) <= FLT_MAX);
#pragma unroll
        for (int u = 0; u < 4; ++u) t[r][c4 + u] = v[u];
    }
    if (__any_sync(0xffffffffu, bad) && (tid & 31) == 0) atomicOr(P.error, ERR_NONFINITE);
    __syncthreads();
    const float dv = P.damp[q.damp_idx];
#pragma unroll
    for (int side = 0; side < 2; ++side) {
        if (side == 1 && si == sj) break;
        const int ti = side ? sj : si, tj = side ? si : sj;
        const bool in_diag = (ti * TT) / NB == (tj * TT) / NB;  // inside a diagonal 128-block: D only
        // above the diagonal 128-blocks nothing reads X; inside one, D gets
        // the whole block (the diagonal updates read it back in full)
        if (side == 0 && si != sj && !in_diag) continue;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int r = rr + 16 * p, i = ti * TT + r;
            float h[4], l[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c4 + u, j = tj * TT + c;
                float v;
                if (i >= q.d || j >= q.d) v = (i == j) ? 1.f : 0.f;
                else if (side == 0 && si != sj) v = 0.f;     // strictly upper tile
                else if (side == 0) v = r >= c ? t[c][r] + (i == j ? dv : 0.f) : 0.f;  // diagonal tile
                else v = t[c][r];                             // lower position: F transposed
                h[u] = tf32_hi(v);
                l[u] = v - h[u];
            }
            if (in_diag) {
                const long long od = (long long)i * NB + (tj * TT) % NB + c4;
                *reinterpret_cast<float4 *>(q.Dh + od) = make_float4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<float4 *>(q.Dl + od) = make_float4(l[0], l[1], l[2], l[3]);
            } else {
                const long long o = (long long)i * q.dp + tj * TT + c4;
                *reinterpret_cast<float4 *>(q.Xh + o) = make_float4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<float4 *>(q.Xl + o) = make_float4(l[0], l[1], l[2], l[3]);
            }
        }
    }
}

// ------------------------------------------------------------------ diag

struct DiagJob {
    const float *Sh, *Sl;  // the Schur-complement block S_kk (lower triangle read), row pitch NB;
                           // no CTA of the launch writes it
    float *Xh, *Xl;    // (owner) block (k, k) of the working pair: W_kk = L_kk^-1 written over
                       // the whole block (zeros above the diagonal)
    float *Th, *Tl;    // (owner) the same block of the transposed pair: W_kk^T (zeros below)
    const float *Ph, *Pl;  // (panel) block (i, k) of the working pair, i > k
    float *Lh, *Ll;        // (panel) where its Cholesky panel L_ik = X_ik W_kk^T goes
    long long ld;
    int o;             // global index of the block's first row (for info)
    int panel;         // 0: the owner of the diagonal block, 1: one panel block
    int *info;
};

constexpr int DIAG_MAX = 300;  // CTAs per diag launch (parameter block < 32 KB)
struct DiagParams {
    DiagJob j[DIAG_MAX];
    int n;
};

// Cholesky factor and its inverse of one SPD 128 x 128 block S = L L^T, by
// one CTA of 256 threads: W = L^-1.  The owner CTA of a diagonal block writes
// W over the block and, transposed, into the same block of the transposed
// pair; each other CTA of the block column recomputes W (no CTA waits for
// another) and turns one block X_ik below it into the Cholesky panel
// L_ik = X_ik W^T (fp32 on CUDA cores, 8 x 8 outputs per thread).  Both steps
// of W run in shared memory, blocked by DB = 16:
//   1. right-looking Cholesky, for each 16-wide block column c:
//        L_cc = chol(S_cc)            one warp, lane r holding row r of the
//                                     16 x 16 block in registers; column
//                                     values by shuffle
//        L_ic = S_ic L_cc^-T          i past c: a thread per row (forward
//                                     substitution with L_cc)
//        S_ij -= L_ic L_jc^T          i >= j past c: 4 x 4 register tiles
//   2. W = L^-1 by block rows i, each in the iteration of step 1 that
//      factors block i:
//        T_ij = sum_{t=j}^{i-1} L_it W_tj  (j < i)   warps 1..7, after their
//                                                    share of the update
//        W_ii = L_ii^-1,  W_ij = -W_ii T_ij          threads 128..255, while
//                                                    threads below solve the panel
// 1 / sqrt is the hardware approximation refined by one Newton-Raphson step,
// y <- y (3 - x y^2) / 2.  A pivot outside [FLT_MIN, inf) is recorded and
// eliminated with w = 0 (the result is then undefined; finite unless the
// block held NaN or inf).
constexpr int DLD = NB + 4;  // row pitch (floats; rows stay 16-byte aligned)
constexpr int DB = 16;       // blocking of both steps
constexpr int DIAG_THREADS = 256;
constexpr size_t DIAG_SMEM = (2 * (size_t)NB * DLD + NB + 4) * sizeof(float);

__device__ __forceinline__ float rsqrt_nr(float x) {
    const float y = rsqrtf(x);
    return y * fmaf(-0.5f * x * y, y, 1.5f);
}

__device__ __forceinline__ void ld16(const float *src, float (&x)[DB]) {
#pragma unroll
    for (int q = 0; q < DB; q += 4) {
        const float4 v = *reinterpret_cast<const float4 *>(src + q);
        x[q] = v.x; x[q + 1] = v.y; x[q + 2] = v.z; x[q + 3] = v.w;
    }
}

__device__ __forceinline__ void st16(float *dst, const float (&x)[DB]) {
#pragma unroll
    for (int q = 0; q < DB; q += 4) *reinterpret_cast<float4 *>(dst + q) = make_float4(x[q], x[q + 1], x[q + 2], x[q + 3]);
}

// ROWS x 128 floats of an fp32 (hi, lo) pair in global memory (row pitch ld),
// summed into shared memory (row pitch sld): each thread issues up to eight
// 16-byte loads of each plane before it stores, so a block costs a few L2
// round trips rather than one per row group.
template <int THREADS, int ROWS>
__device__ __forceinline__ void stage_pair(float *dst, int sld, const float *hi, const float *lo, long long ld,
                                           int tid) {
    constexpr int N = ROWS * (NB / 4), PER = N / THREADS, BATCH = PER < 8 ? PER : 8;
    static_assert(N % THREADS == 0 && PER % BATCH == 0, "whole batches");
#pragma unroll
    for (int b = 0; b < PER; b += BATCH) {
        float4 h[BATCH], l[BATCH];
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int e = (b + u) * THREADS + tid;
            const long long off = (long long)(e >> 5) * ld + (e & 31) * 4;
            h[u] = __ldcg(reinterpret_cast<const float4 *>(hi + off));
            l[u] = __ldcg(reinterpret_cast<const float4 *>(lo + off));
        }
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int e = (b + u) * THREADS + tid;
            *reinterpret_cast<float4 *>(dst + (e >> 5) * sld + (e & 31) * 4) =
                make_float4(h[u].x + l[u].x, h[u].y + l[u].y, h[u].z + l[u].z, h[u].w + l[u].w);
        }
    }
}

__global__ void __launch_bounds__(DIAG_THREADS, 1) diag_kernel(const __grid_constant__ DiagParams P) {
    extern __shared__ float4 diag_smem4[];
    float *M = reinterpret_cast<float *>(diag_smem4);  // S, then L (lower triangle)
    float *Wm = M + NB * DLD;                           // W (lower triangle)
    float *invd = Wm + NB * DLD;                        // 1 / L_ii
    int *bad_s = reinterpret_cast<int *>(invd + NB);    // first failing pivot (NB: none)
    const DiagJob &J = P.j[blockIdx.x];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) *bad_s = NB;
    pdl_wait();
    pdl_trigger();
    stage_pair<DIAG_THREADS, NB>(M, DLD, J.Sh, J.Sl, NB, tid);
    __syncthreads();

    // 1. Cholesky, for each 16-wide block column c, with the trailing update
    //    of the previous block column split: warp 0 applies it to block c's
    //    diagonal block and factors that block while warps 1..7 apply it to
    //    everything else past c; then the panel below block c
#pragma unroll 1
    for (int c = 0; c < NB; c += DB) {
        if (warp == 0) {
            const int r = lane & (DB - 1);  // lanes 16..31 repeat rows 0..15 (only 0..15 store)
            float a[DB];
            ld16(M + (c + r) * DLD + c, a);
            if (c > 0) {
                // S_rj -= L[c+r][c-16 ..] . L[c+j][c-16 ..]  (the previous panel)
                float lr[DB];
                ld16(M + (c + r) * DLD + c - DB, lr);
#pragma unroll
                for (int j = 0; j < DB; ++j) {
                    float lj[DB];
                    ld16(M + (c + j) * DLD + c - DB, lj);
                    float x = a[j];
#pragma unroll
                    for (int t = 0; t < DB; ++t) x = fmaf(-lr[t], lj[t], x);
                    a[j] = x;
                }
            }
            float wr = 0.f;
            int bad = -1;
#pragma unroll
            for (int q = 0; q < DB; ++q) {
                const float piv = __shfl_sync(0xffffffffu, a[q], q);
                const bool ok = piv >= FLT_MIN && piv < INFINITY;
                const float w = ok ? rsqrt_nr(piv) : 0.f;
                bad = (!ok && bad < 0) ? q : bad;
                if (r == q) {
                    a[q] = ok ? piv * w : 0.f;  // L_qq
                    wr = w;
                } else if (r > q) {
                    a[q] *= w;                  // L_rq
                }
#pragma unroll
                for (int j = 1; j < DB; ++j) {
                    if (j > q) {
                        const float lj = __shfl_sync(0xffffffffu, a[q], j);
                        if (r >= j) a[j] = fmaf(-a[q], lj, a[j]);
                    }
                }
            }
            if (lane < DB) {
                st16(M + (c + r) * DLD + c, a);
                invd[c + r] = wr;
            }
            if (lane == 0 && bad >= 0) atomicMin(bad_s, c + bad);
        } else if (c > 0) {
            // the previous panel's update of the lower triangle past c, 4 x 4
            // tiles (I, Jt), without the 10 tiles of block c's diagonal block
            const int p = c - DB;
            const int nT = (NB - c) / 4;
            const int ntiles = nT * (nT + 1) / 2;
            for (int t = tid - 32 + 10; t < ntiles; t += DIAG_THREADS - 32) {
                int I = (int)((sqrtf(8.f * (float)t + 1.f) - 1.f) * 0.5f);
                while (I * (I + 1) / 2 > t) --I;
                while ((I + 1) * (I + 2) / 2 <= t) ++I;
                const int Jt = t - I * (I + 1) / 2;
                const int i0 = c + 4 * I, j0 = c + 4 * Jt;
                float acc[4][4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 v = *reinterpret_cast<const float4 *>(M + (i0 + u) * DLD + j0);
                    acc[u][0] = v.x; acc[u][1] = v.y; acc[u][2] = v.z; acc[u][3] = v.w;
                }
#pragma unroll
                for (int q = 0; q < DB; q += 4) {
                    float4 li[4], lj[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        li[u] = *reinterpret_cast<const float4 *>(M + (i0 + u) * DLD + p + q);
                        lj[u] = *reinterpret_cast<const float4 *>(M + (j0 + u) * DLD + p + q);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            float x = acc[u][v];
                            x = fmaf(-li[u].x, lj[v].x, x);
                            x = fmaf(-li[u].y, lj[v].y, x);
                            x = fmaf(-li[u].z, lj[v].z, x);
                            acc[u][v] = fmaf(-li[u].w, lj[v].w, x);
                        }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (I != Jt) {
                        *reinterpret_cast<float4 *>(M + (i0 + u) * DLD + j0) =
                            make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
                    } else {
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            if (v <= u) M[(i0 + u) * DLD + j0 + v] = acc[u][v];
                    }
                }
            }
        }
        if (warp > 0) {
            // W's block row c / 16, first half: T_cj = sum_{t=j}^{c-1} L_ct W_tj
            // for the block columns j < c (rows c .. c + 15 of the panels and
            // block rows of W before c are final); item (j, r, half) -> 8
            // entries of row r of T_cj, written over W's block (c, j)
#pragma unroll 1
            for (int it = tid - 32; it < c * 2; it += DIAG_THREADS - 32) {
                const int j = (it >> 5) * DB, r = (it & 31) >> 1, h = (it & 1) * 8;
                float acc[8];
#pragma unroll
                for (int v = 0; v < 8; ++v) acc[v] = 0.f;
                const float *lrow = M + (c + r) * DLD;
#pragma unroll 4
                for (int k = j; k < c; ++k) {
                    const float l = lrow[k];
                    const float4 w0 = *reinterpret_cast<const float4 *>(Wm + k * DLD + j + h);
                    const float4 w1 = *reinterpret_cast<const float4 *>(Wm + k * DLD + j + h + 4);
                    acc[0] = fmaf(l, w0.x, acc[0]); acc[1] = fmaf(l, w0.y, acc[1]);
                    acc[2] = fmaf(l, w0.z, acc[2]); acc[3] = fmaf(l, w0.w, acc[3]);
                    acc[4] = fmaf(l, w1.x, acc[4]); acc[5] = fmaf(l, w1.y, acc[5]);
                    acc[6] = fmaf(l, w1.z, acc[6]); acc[7] = fmaf(l, w1.w, acc[7]);
                }
                *reinterpret_cast<float4 *>(Wm + (c + r) * DLD + j + h) =
                    make_float4(acc[0], acc[1], acc[2], acc[3]);
                *reinterpret_cast<float4 *>(Wm + (c + r) * DLD + j + h + 4) =
                    make_float4(acc[4], acc[5], acc[6], acc[7]);
            }
        }
        __syncthreads();
        const int nrest = NB - c - DB;
        if (tid >= NB) {
            // W's block row c / 16, second half, by threads 128..255 while the
            // panel below runs: W_cc = L_cc^-1 (a thread per column q, zeros
            // above the diagonal), then W_cj = -W_cc T_cj (thread (j, q) owns
            // column q of block (c, j))
            const int u = tid - NB;
            if (u < DB) {
                const int q = u;
                float x[DB];
#pragma unroll
                for (int r = 0; r < DB; ++r) {
                    float v = r == q ? 1.f : 0.f;
#pragma unroll
                    for (int t = 0; t < r; ++t) v = fmaf(-M[(c + r) * DLD + c + t], x[t], v);
                    x[r] = v * invd[c + r];
                }
#pragma unroll
                for (int r = 0; r < DB; ++r) Wm[(c + r) * DLD + c + q] = x[r];
            }
            asm volatile("bar.sync 1, %0;" ::"n"(DIAG_THREADS - NB) : "memory");
            if (u < c) {
                const int j = (u / DB) * DB, q = u % DB;
                float tcol[DB], y[DB];
#pragma unroll
                for (int v = 0; v < DB; ++v) tcol[v] = Wm[(c + v) * DLD + j + q];
#pragma unroll
                for (int r = 0; r < DB; ++r) {
                    float a = 0.f;
#pragma unroll
                    for (int v = 0; v <= r; ++v) a = fmaf(Wm[(c + r) * DLD + c + v], tcol[v], a);
                    y[r] = -a;
                }
#pragma unroll
                for (int r = 0; r < DB; ++r) Wm[(c + r) * DLD + j + q] = y[r];
            }
        } else if (tid < nrest) {  // the panel: row i solves L_cc y = S_ic^T
            const int i = c + DB + tid;
            float x[DB];
            ld16(M + i * DLD + c, x);
#pragma unroll
            for (int q = 0; q < DB; ++q) {
                x[q] *= invd[c + q];
#pragma unroll
                for (int j = q + 1; j < DB; ++j) x[j] = fmaf(-x[q], M[(c + j) * DLD + c + q], x[j]);
            }
            st16(M + i * DLD + c, x);
        }
        __syncthreads();
    }

    if (J.panel) {
        // L_ik = X_ik W^T: X_ik (hi + lo) into M, then thread (ti, tj) forms
        // rows ti + 16 a (a < 8) and columns 8 tj .. 8 tj + 7; W is lower
        // triangular, so K stops at the block's last column (W's upper
        // entries inside a 16-block are the zeros written above)
        stage_pair<DIAG_THREADS, NB>(M, DLD, J.Ph, J.Pl, J.ld, tid);
        __syncthreads();
        const int ti = tid & 15, tj = tid >> 4;
        float acc[8][8];
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
            for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
        const int kend = 8 * tj + 8;
#pragma unroll 1
        for (int t = 0; t < kend; t += 4) {
            float4 w4[8];
#pragma unroll
            for (int b = 0; b < 8; ++b) w4[b] = *reinterpret_cast<const float4 *>(Wm + (8 * tj + b) * DLD + t);
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                const float4 x4 = *reinterpret_cast<const float4 *>(M + (ti + 16 * a) * DLD + t);
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    float v = acc[a][b];
                    v = fmaf(x4.x, w4[b].x, v);
                    v = fmaf(x4.y, w4[b].y, v);
                    v = fmaf(x4.z, w4[b].z, v);
                    acc[a][b] = fmaf(x4.w, w4[b].w, v);
                }
            }
        }
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const long long off = (long long)(ti + 16 * a) * J.ld + 8 * tj;
            float h[8], l[8];
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                h[b] = tf32_hi(acc[a][b]);
                l[b] = acc[a][b] - h[b];
            }
            *reinterpret_cast<float4 *>(J.Lh + off) = make_float4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<float4 *>(J.Lh + off + 4) = make_float4(h[4], h[5], h[6], h[7]);
            *reinterpret_cast<float4 *>(J.Ll + off) = make_float4(l[0], l[1], l[2], l[3]);
            *reinterpret_cast<float4 *>(J.Ll + off + 4) = make_float4(l[4], l[5], l[6], l[7]);
        }
        return;
    }
    // W (lower, zeros above) into X and W^T (upper, zeros below) into the transposed pair
    for (int e = tid; e < NB * NB / 4; e += DIAG_THREADS) {
        const int i = e >> 5, j = (e & 31) * 4;
        float w4[4], t4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            w4[u] = j + u <= i ? Wm[i * DLD + j + u] : 0.f;
            t4[u] = i <= j + u ? Wm[(j + u) * DLD + i] : 0.f;
        }
        float hw[4], ht[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            hw[u] = tf32_hi(w4[u]);
            ht[u] = tf32_hi(t4[u]);
        }
        const long long off = (long long)i * J.ld + j;
        *reinterpret_cast<float4 *>(J.Xh + off) = make_float4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<float4 *>(J.Xl + off) =
            make_float4(w4[0] - hw[0], w4[1] - hw[1], w4[2] - hw[2], w4[3] - hw[3]);
        *reinterpret_cast<float4 *>(J.Th + off) = make_float4(ht[0], ht[1], ht[2], ht[3]);
        *reinterpret_cast<float4 *>(J.Tl + off) =
            make_float4(t4[0] - ht[0], t4[1] - ht[1], t4[2] - ht[2], t4[3] - ht[3]);
    }
    if (tid == 0 && *bad_s < NB && J.info) atomicCAS(J.info, 0, J.o + *bad_s + 1);
    __syncthreads();
}

// ------------------------------------------------------------- scheduler

// One launch unit of a matrix's chain: a diag leaf, or engine problems that
// go into the same launch.
struct Op {
    int leaf;                 // launch kind: 0 engine, 1 diag kernel
    std::vector<DiagJob> dj;  // leaf: the owner of the diagonal block, then its panel blocks
    std::vector<TcJob> g;
    std::vector<TcJob> side;  // engine problems that may start once this op is done (lookahead,
                              // launched on the group's side stream)
    std::vector<TcJob> bulk;  // engine problems that may start once this op's side problems are done
                              // (launched on the group's bulk stream)
    int needs_side = -1;      // chain index of the op whose side problems must be done first
    int needs_bulk = -1;      // chain index of the op whose bulk problems must be done first
    int side_needs_bulk = -1; // the same, for this op's side problems
    bool needs_tri = false;   // waits for the chain's early triangular inverse
};

// One launch of a chain's early triangular inverse (a node's T or W21
// product), on the group's third stream once chain op `after` is done.
struct TriOp {
    int after;
    TcJob job;
};

// Working buffers of one matrix (fp32 (hi, lo) pairs, [dp][dp] each):
//   X   blocks below the diagonal 128-blocks: the factor, its block columns
//       updated into Schur-complement columns, then W = L^-1 (diagonal blocks
//       from the diag leaves, zeros above their diagonal; the rest from the
//       triangular inverse); blocks above the diagonal are never written or read
//   Wt  upper part: W^T (diagonal blocks in full, zeros below)
//   LT  lower blocks: the Cholesky panels L_ik (i > k);  upper blocks:
//       (L21 W11)^T of the triangular inverse
struct MatWork {
    int d, dp;
    float *Xh, *Xl, *Wh, *Wl, *Lh, *Ll;
    float *Dh, *Dl;  // diagonal 128 x 128 blocks of the Schur complement, stacked [dp][128]
    int mx, mw, ml;  // map indices (hi; lo at +1; 32-row boxes at +2, +3)
};

TcJob split_job(int ma, int ar, int ac, int mb, int br, int bc, int M, int N, int K, float alpha, float beta,
                float *Ch, float *Cl, float *Cth, float *Ctl, long long ld) {
    TcJob j{};
    j.map_a = ma; j.a_row0 = ar; j.a_col0 = ac;
    j.map_b = mb; j.b_row0 = br; j.b_col0 = bc;
    j.M = M; j.N = N; j.K = K;
    j.epi = TC_EPI_SPLIT;
    j.alpha = alpha; j.beta = beta;
    j.C = Ch; j.C_lo = Cl; j.ldc = ld;
    j.Ct = Cth; j.Ct_lo = Ctl; j.ldct = ld;
    return j;
}

// Nodes of the triangular-inverse recursion over [o, o + n) with their
// heights (a 128-row block: height 0).
int tri_nodes(int o, int n, std::vector<std::vector<std::pair<int, int>>> &by_height) {
    if (n == NB) return 0;
    const int nb = n / NB, h = NB * (nb / 2);
    const int ht = 1 + std::max(tri_nodes(o, h, by_height), tri_nodes(o + h, n - h, by_height));
    if ((int)by_height.size() <= ht) by_height.resize(ht + 1);
    by_height[ht].push_back({o, n});
    return ht;
}

// The chain of one matrix.
//  1. left-looking blocked Cholesky, 128-wide block columns k:
//       D_k = X[k, k] - L[k, :k] L[k, :k]^T,
//       X[k+1:, k] -= L[k+1:, :k] L[k, :k]^T              (engine; k > 0)
//       W_kk = L_kk^-1 from D_k                           (diag kernel)
//       L[k+1:, k] = X[k+1:, k] W_kk^T                    (engine, the panel)
//     every Schur-complement column comes from Cholesky panels (no growth).
//     With the lookahead only the diagonal update, the diag kernel and the
//     panel's first block stay on the chain; the rest of each column runs on
//     the side stream (details in gen_chain);
//  2. W = L^-1 by recursive 2 x 2 blocking, bottom up by height (the two
//     halves of a node are independent):
//       T = L21 W11,   W21 = -W22 T   (W21 over X's lower part, W21^T into Wt);
//  3. X^-1 = W^T W = Wt Wt^T, written into the caller's output.
// W11, W22 are lower triangular with zeros above in X and their transposes
// upper triangular with zeros below in Wt, so the products run over whole
// blocks; T reads W11^T from Wt only from each output tile's first column on
// (ktri), where Wt holds its upper part and diagonal blocks.
void gen_chain(std::vector<Op> &ops, std::vector<TriOp> &tri, bool early_tri, bool side_bulk, const MatWork &w,
               const InvMatrix &mat, int *info) {
    const long long ld = w.dp;
    const int nb = w.dp / NB;
    auto diag_op = [&](int k) {
        // W_kk from D_k (every CTA reads S_kk from D, which no CTA of the launch
        // writes; the owner writes W_kk over X's block), and with the fused
        // panel one more CTA per block below forming L[i, k] = X[i, k] W_kk^T
        const int kb = k * NB;
        const float *Dh = w.Dh + (long long)kb * NB, *Dl = w.Dl + (long long)kb * NB;
        Op op{};
        op.leaf = 1;
        op.dj.push_back(DiagJob{Dh, Dl, w.Xh + kb * ld + kb, w.Xl + kb * ld + kb, w.Wh + kb * ld + kb,
                                w.Wl + kb * ld + kb, nullptr, nullptr, nullptr, nullptr, ld, kb, 0, info});
        for (int i = k + 1; FUSED_PANEL && i < nb; ++i) {
            const long long c = (long long)i * NB * ld + kb;
            op.dj.push_back(DiagJob{Dh, Dl, nullptr, nullptr, nullptr, nullptr, w.Xh + c, w.Xl + c, w.Lh + c, w.Ll + c,
                                    ld, kb, 1, nullptr});
        }
        return op;
    };
    // L[r0:r1, k] = X[r0:r1, k] W_kk^T
    auto panel = [&](int k, int r0, int r1) {
        const int kb = k * NB;
        const long long c = (long long)r0 * ld + kb;
        return split_job(w.mx, r0, kb, w.mx, kb, kb, r1 - r0, NB, NB, 1.f, 0.f, w.Lh + c, w.Ll + c, nullptr, nullptr,
                         ld);
    };
    // C[r0:r1, k] -= L[r0:r1, :k] L[k, :k]^T  (C = D_k for the diagonal block)
    auto update = [&](int k, int r0, int r1, bool diag) {
        const int kb = k * NB;
        float *ch = diag ? w.Dh + (long long)kb * NB : w.Xh + (long long)r0 * ld + kb;
        float *cl = diag ? w.Dl + (long long)kb * NB : w.Xl + (long long)r0 * ld + kb;
        return split_job(w.ml, r0, 0, w.ml, kb, 0, r1 - r0, NB, kb, -1.f, 1.f, ch, cl, nullptr, nullptr,
                         diag ? NB : ld);
    };
    // D_c -= L[c, j0:j1] L[c, j0:j1]^T (block columns j0 .. j1 - 1)
    auto dupd = [&](int c, int j0, int j1) {
        const int cb = c * NB;
        return split_job(w.ml, cb, j0 * NB, w.ml, cb, j0 * NB, NB, NB, (j1 - j0) * NB, -1.f, 1.f,
                         w.Dh + (long long)cb * NB, w.Dl + (long long)cb * NB, nullptr, nullptr, NB);
    };
    // X[r0:r1, c] -= L[r0:r1, j0:j1] L[c, j0:j1]^T (block columns j0 .. j1 - 1)
    auto xupd = [&](int c, int r0, int r1, int j0, int j1) {
        const int cb = c * NB;
        const long long o = (long long)r0 * ld + cb;
        return split_job(w.ml, r0, j0 * NB, w.ml, cb, j0 * NB, r1 - r0, NB, (j1 - j0) * NB, -1.f, 1.f, w.Xh + o,
                         w.Xl + o, nullptr, nullptr, ld);
    };
    int last_side = -1, last_bulk = -1;  // chain indices of the last ops with side / bulk problems
    std::vector<int> i_diag(nb, -1), i_first(nb, -1);
    if (!LOOKAHEAD) {
        for (int k = 0; k < nb; ++k) {
            const int kb = k * NB;
            if (k > 0) {  // the diagonal block into D, the blocks below it in X
                Op op{};
                op.g.push_back(update(k, kb, kb + NB, true));
                if (k + 1 < nb) op.g.push_back(update(k, kb + NB, w.dp, false));
                ops.push_back(op);
            }
            ops.push_back(diag_op(k));
            if (!FUSED_PANEL && k + 1 < nb) {
                Op pn{};
                pn.g.push_back(panel(k, kb + NB, w.dp));
                ops.push_back(pn);
            }
        }
    } else {
        // Lookahead: the chain carries only what the next diagonal block
        // needs -- the first panel block L[k+1, k], then the last term of the
        // diagonal update, D_{k+1} -= L[k+1, k] L[k+1, k]^T -- and the rest of
        // each block column runs as side problems on the group's side stream,
        // in order: after the diag op of k, the panel L[k+2:, k]; after the
        // first panel block of k, the update X[k+2:, k+1] -= L[k+2:, :k+1]
        // L[k+1, :k+1]^T and the earlier terms of the next diagonal block,
        // D_{k+2} -= L[k+2, :k+1] L[k+2, :k+1]^T.  The first panel block of k
        // waits for the side launch after the first panel block of k - 1 (the
        // update of column k and the earlier terms of D_{k+1}, which the
        // diagonal update after it then completes), and the triangular
        // inverse for the last side launch.  (Without SIDE_DIAG_BULK the
        // chain's diagonal update runs over all of L[k+1, :k+1], split finely
        // over K, after the side panel of k - 1, the last one holding a block
        // of row k + 1.)  With SIDE_BULK the side update after the first
        // panel block of k keeps only the last term, X[k+2:, k+1] -=
        // L[k+2:, k] L[k+1, k]^T; the terms j < k of column k + 1 and of
        // D_{k+1} were subtracted on the bulk stream after the side panel of
        // k - 1, and both that last term and the diagonal update on the chain
        // wait for them.
        for (int k = 0; k < nb; ++k) {
            const int kb = k * NB;
            Op d = diag_op(k);
            if (!FUSED_PANEL && k + 2 < nb) {
                d.side.push_back(panel(k, kb + 2 * NB, w.dp));
                if (side_bulk) {  // the terms j <= k of column k + 2 and of D_{k+2}
                    if (k + 3 < nb) d.bulk.push_back(xupd(k + 2, kb + 3 * NB, w.dp, 0, k + 1));
                    d.bulk.push_back(dupd(k + 2, 0, k + 1));
                }
            }
            i_diag[k] = (int)ops.size();
            if (!d.side.empty()) last_side = i_diag[k];
            if (!d.bulk.empty()) last_bulk = i_diag[k];
            ops.push_back(d);
            if (k + 1 == nb) break;
            if (!FUSED_PANEL) {
                Op pf{};
                pf.g.push_back(panel(k, kb + NB, kb + 2 * NB));
                if (k >= 1) pf.needs_side = i_first[k - 1];
                if (k + 2 < nb && side_bulk) {
                    pf.side.push_back(xupd(k + 1, kb + 2 * NB, w.dp, k, k + 1));
                    if (k >= 1) pf.side_needs_bulk = i_diag[k - 1];
                } else if (k + 2 < nb) {
                    pf.side.push_back(update(k + 1, kb + 2 * NB, w.dp, false));
                    // D_{k+2} -= L[k+2, :k+1] L[k+2, :k+1]^T (its last term stays on the chain)
                    if (SIDE_DIAG_BULK) pf.side.push_back(dupd(k + 2, 0, k + 1));
                }
                i_first[k] = (int)ops.size();
                if (!pf.side.empty()) last_side = i_first[k];
                ops.push_back(pf);
            }
            Op ud{};
            if (SIDE_DIAG_BULK) {
                // D_{k+1} -= L[k+1, k] L[k+1, k]^T: the terms before it were
                // subtracted by the side launch the first panel block waited for
                ud.g.push_back(dupd(k + 1, k, k + 1));
                if (side_bulk && k >= 1) ud.needs_bulk = i_diag[k - 1];
            } else {
                ud.g.push_back(update(k + 1, kb + NB, kb + 2 * NB, true));
                ud.g.back().fine_split = 1;
                if (k >= 1) ud.needs_side = i_diag[k - 1];
            }
            ops.push_back(ud);
        }
    }
    // the two products of the triangular-inverse node over [o, o + n)
    auto node_t = [&](int o, int n) {
        const int h = NB * (n / NB / 2), m = n - h;
        const long long t12 = (long long)o * ld + o + h;
        // T = L21 W11 (B rows: W11^T rows, in Wt), stored as T^T in LT's upper part
        TcJob j = split_job(w.ml, o + h, o, w.mw, o, o, m, h, h, 1.f, 0.f, nullptr, nullptr, w.Lh + t12,
                            w.Ll + t12, ld);
        j.ktri = 1;
        return j;
    };
    auto node_x = [&](int o, int n) {
        const int h = NB * (n / NB / 2), m = n - h;
        const long long x21 = (long long)(o + h) * ld + o, t12 = (long long)o * ld + o + h;
        // W21 = -W22 T (A: W22 rows, in X; B rows: T^T rows, in LT), W21^T into Wt
        TcJob j = split_job(w.mx, o + h, o + h, w.ml, o, o + h, m, h, m, -1.f, 0.f, w.Xh + x21, w.Xl + x21,
                            w.Wh + t12, w.Wl + t12, ld);
        j.ktril = 1;  // W22 is lower triangular
        return j;
    };
    const size_t first_tri = ops.size();
    Op fin{};
    if (early_tri) {
        // Early triangular inverse: the nodes in post-order with each T
        // before the right subtree, every product a launch of its own on the
        // third stream.  T of node [o, o + n) (split at h) reads L21 -- the
        // panels of block columns below (o + h) / 128 -- and W11 (the left
        // subtree, earlier on the stream); the first panel block of column
        // c + 1 is done only after the side panel of column c (the side
        // stream runs that panel before the update the first block waits
        // for), so T waits for the first panel block of column (o + h) / 128
        // (of the column before it when that is the last one).  W21 needs
        // W22, whose last diagonal block comes from the diag op of column
        // (o + n) / 128 - 1.  Both write only what the factorisation no
        // longer reads: T^T above L's diagonal, W21 over X's block row
        // (the Schur columns there were consumed by their panels) and W21^T
        // above Wt's diagonal.
        std::function<void(int, int)> visit = [&](int o, int n) {
            if (n == NB) return;
            const int h = NB * (n / NB / 2);
            visit(o, h);
            const int c = (o + h) / NB;  // first column of the right half
            tri.push_back(TriOp{i_first[std::min(c, nb - 2)], node_t(o, n)});
            visit(o + h, n - h);
            tri.push_back(TriOp{i_diag[(o + n) / NB - 1], node_x(o, n)});
        };
        visit(0, w.dp);
        fin.needs_tri = true;
    } else {
        std::vector<std::vector<std::pair<int, int>>> by_height;
        tri_nodes(0, w.dp, by_height);
        for (size_t ht = 1; ht < by_height.size(); ++ht) {
            Op t{}, x{};
            for (const auto &nd : by_height[ht]) {
                t.g.push_back(node_t(nd.first, nd.second));
                x.g.push_back(node_x(nd.first, nd.second));
            }
            if (ops.size() == first_tri) {
                t.needs_side = last_side;
                t.needs_bulk = last_bulk;
            }
            ops.push_back(t);
            ops.push_back(x);
        }
    }
    if (ops.size() == first_tri) {
        fin.needs_side = last_side;
        fin.needs_bulk = last_bulk;
    }
    TcJob j{};
    j.map_a = j.map_b = w.mw;
    j.M = j.N = w.d;
    j.K = w.dp;
    j.sym = 1;
    j.ktri = 1;
    j.epi = TC_EPI_STORE;
    j.alpha = 1.f;
    j.C = mat.out;
    j.ldc = mat.ldo;
    j.Cb = mat.out_bf16;
    j.cb_f16 = mat.copy_f16;
    j.ldcb = mat.ldo_bf16;
    fin.g.push_back(j);
    ops.push_back(fin);
}

// Round schedule of a group of chains: the group's longest chain sets the
// sequence of rounds (one launch each, leaf or engine); every other chain of
// the group is embedded as late as possible into rounds of the same op kind,
// in order.  The long chain's late rounds are small, latency-bound launches
// with most SMs idle, and the shorter chains' work fills them.  Falls back to
// left-aligned lock-step (a leaf and an engine launch per round) if a chain
// does not embed.  Rounds list (chain, op) pairs.
std::vector<std::vector<std::pair<int, int>>> schedule_rounds(const std::vector<std::vector<Op>> &chains,
                                                              const std::vector<int> &members,
                                                              std::vector<int> &round_kind) {
    int crit = -1;
    for (int k : members)
        if (crit < 0 || chains[k].size() > chains[crit].size()) crit = k;
    std::vector<std::vector<std::pair<int, int>>> rounds;
    round_kind.clear();
    if (crit < 0) return rounds;
    const int R = (int)chains[crit].size();
    rounds.assign(R, {});
    for (int r = 0; r < R; ++r) round_kind.push_back(chains[crit][r].leaf);
    bool ok = true;
    std::vector<std::vector<int>> slot(chains.size());
    for (int k : members) {
        const int n = (int)chains[k].size();
        slot[k].assign(n, -1);
        int r = R - 1;
        for (int i = n - 1; i >= 0; --i) {
            while (r >= 0 && round_kind[r] != chains[k][i].leaf) --r;
            if (r < 0) { ok = false; break; }
            slot[k][i] = r--;
        }
        if (!ok) break;
    }
    if (ok) {
        for (int k : members)
            for (int i = 0; i < (int)chains[k].size(); ++i) rounds[slot[k][i]].push_back({k, i});
        return rounds;
    }
    size_t longest = 0;
    for (int k : members) longest = std::max(longest, chains[k].size());
    rounds.clear();
    round_kind.clear();
    for (size_t r = 0; r < longest; ++r)
        for (int kind : {1, 0}) {
            std::vector<std::pair<int, int>> v;
            for (int k : members)
                if (r < chains[k].size() && chains[k][r].leaf == kind) v.push_back({k, (int)r});
            if (!v.empty()) {
                rounds.push_back(v);
                round_kind.push_back(kind);
            }
        }
    return rounds;
}

// The chains run as two concurrent groups: the longest ones (the critical
// path of the call) on a high-priority stream, all others on a low-priority
// stream whose engine launches leave SMs free for the first group.  Each
// group has its own rounds and engine scratch.
#ifndef KFAC_INV_RESERVED_SMS
#define KFAC_INV_RESERVED_SMS 32
#endif
constexpr int RESERVED_SMS = KFAC_INV_RESERVED_SMS;  // SMs the second group's engine launches leave free
                                                     // (a tuning constant that may be set at build time)
#ifndef KFAC_INV_SIDE_FREE_SMS
#define KFAC_INV_SIDE_FREE_SMS 48
#endif
constexpr int SIDE_FREE_SMS = KFAC_INV_SIDE_FREE_SMS;  // SMs a group's side launches leave to its own chain
#ifndef KFAC_INV_SIDE_GROUPS
#define KFAC_INV_SIDE_GROUPS 2
#endif
#ifndef KFAC_INV_TRI_FREE_SMS
#define KFAC_INV_TRI_FREE_SMS 48
#endif
constexpr int TRI_FREE_SMS = KFAC_INV_TRI_FREE_SMS;  // SMs a group's early-inverse launches leave to the rest
#ifndef KFAC_INV_TRI_HIGH_PRIO
#define KFAC_INV_TRI_HIGH_PRIO 0
#endif
constexpr bool TRI_HIGH_PRIO = KFAC_INV_TRI_HIGH_PRIO;  // early-inverse streams at their group's priority (else low)
#ifndef KFAC_INV_BULK_FREE_SMS
#define KFAC_INV_BULK_FREE_SMS 48
#endif
constexpr int BULK_FREE_SMS = KFAC_INV_BULK_FREE_SMS;  // SMs a group's bulk launches leave to the rest
#ifndef KFAC_INV_BULK_HIGH_PRIO
#define KFAC_INV_BULK_HIGH_PRIO 1
#endif
constexpr bool BULK_HIGH_PRIO = KFAC_INV_BULK_HIGH_PRIO;  // bulk streams at their group's priority (else low)
constexpr int SIDE_GROUPS = KFAC_INV_SIDE_GROUPS;  // groups whose lookahead updates run on a side stream (the others
                                   // run them in their own stream, right after the enabling round)

// One launch of a group's early triangular inverse: the same step of every
// chain of one width, after the rounds that hold the ops it waits for.
struct TriStep {
    std::vector<TcJob> g;
    std::vector<int> wait_rounds;  // main-stream rounds to wait for
    int key = 0;                   // enqueued after this round (non-decreasing)
};

struct InvGroup {
    std::vector<int> members;  // chain indices
    std::vector<std::vector<std::pair<int, int>>> rounds;
    std::vector<int> round_kind;
    std::vector<std::vector<TcJob>> side;   // per round: side problems launched once it is done
    std::vector<std::vector<int>> waits;    // per round: rounds whose side launch must finish first
    std::vector<std::vector<TcJob>> bulk;   // per round: bulk problems launched once its side launch is done
    std::vector<std::vector<int>> bulk_waits;       // per round: rounds whose bulk launch must finish first
    std::vector<std::vector<int>> side_bulk_waits;  // the same, for the round's side launch
    int bulk_ctas = 0;
    char *bulk_ws = nullptr;
    size_t bulk_bytes = 0;
    std::vector<TriStep> tri;               // early triangular inverse, in stream order
    std::vector<std::vector<int>> tri_waits;  // per round: tri steps that must finish first
    std::vector<char> record_main;          // per round: a tri step waits for it
    int tri_ctas = 0;
    char *tri_ws = nullptr;
    size_t tri_bytes = 0;
    int max_ctas = 0;          // engine grid cap (0: all SMs)
    int side_ctas = 0;         // grid cap of the side launches
    char *tc_ws = nullptr;
    size_t tc_bytes = 0;
    char *side_ws = nullptr;   // the side launches' own engine scratch (they overlap the rounds)
    size_t side_bytes = 0;
};

struct InvPlan {
    int *err = nullptr;
    CUtensorMap *dev_maps = nullptr;
    std::vector<CUtensorMap> maps;
    std::vector<MatWork> work;
    std::vector<std::vector<Op>> chains;
    std::vector<std::vector<TriOp>> tri;  // per chain: its early triangular inverse (or empty)
    std::vector<InvGroup> groups;  // groups[0]: the critical chains
    size_t longest = 0;
};

// Workspace layout shared by the size query and the run.
kfac_status plan_inv(const InvMatrix *mats, int nmats, int *info_dev, Arena &ws, InvPlan &p, bool encode) {
    p.err = ws.take<int>(64);
    p.dev_maps = ws.take<CUtensorMap>(MAPS_PER_MATRIX * (size_t)std::max(nmats, 1));
    p.work.resize(nmats);
    p.chains.assign(nmats, {});
    p.tri.assign(nmats, {});
    // the early triangular inverse serves the longest chains (the critical
    // group's); the others keep theirs at the end of the chain, which costs
    // the critical group less in contention
    int nb_max = 0;
    for (int k = 0; k < nmats; ++k) nb_max = std::max(nb_max, padded(mats[k].d) / NB);
    for (int k = 0; k < nmats; ++k) {
        MatWork &w = p.work[k];
        w.d = mats[k].d;
        w.dp = padded(w.d);
        const size_t sq = (size_t)w.dp * w.dp;
        w.Xh = ws.take<float>(sq);
        w.Xl = ws.take<float>(sq);
        w.Wh = ws.take<float>(sq);
        w.Wl = ws.take<float>(sq);
        w.Lh = w.Ll = nullptr;
        w.Dh = ws.take<float>((size_t)w.dp * NB);
        w.Dl = ws.take<float>((size_t)w.dp * NB);
        if (w.dp > NB) {
            w.Lh = ws.take<float>(sq);
            w.Ll = ws.take<float>(sq);
        }
        float *bufs[6] = {w.Xh, w.Xl, w.Wh, w.Wl, w.Lh, w.Ll};
        const int base = (int)p.maps.size();
        for (int q = 0; q < 6; q += 2)  // per pair: hi, the (hi, lo) pair (128-row boxes), hi, lo (32-row boxes)
            for (int v = 0; v < 4; ++v) {
                p.maps.emplace_back();
                if (!encode || !bufs[q]) continue;
                const bool ok = v == 1 ? tc_make_pair_map(&p.maps.back(), bufs[q], bufs[q + 1], w.dp, w.dp, w.dp, 128)
                                       : tc_make_map(&p.maps.back(), TC_KIND_TF32X3, bufs[q + (v & 1)], w.dp, w.dp,
                                                     w.dp, v < 2 ? 128 : 32);
                if (!ok) return KFAC_ERR_CUDA;
            }
        w.mx = base;
        w.mw = base + 4;
        w.ml = base + 8;
        const int nbk = w.dp / NB;
        const bool early = EARLY_TRI && nbk >= EARLY_TRI_MIN_NB && 4 * nbk >= 3 * nb_max;
        gen_chain(p.chains[k], p.tri[k], early, SIDE_BULK, w, mats[k], info_dev ? info_dev + k : nullptr);
        p.longest = std::max(p.longest, p.chains[k].size());
    }
    if (p.maps.size() != (size_t)MAPS_PER_MATRIX * nmats) return KFAC_ERR_WORKSPACE;  // device map area
    // groups: chains at least 3/4 as long as the longest form the critical
    // group; the others run concurrently as a second group
    p.groups.assign(1, InvGroup{});
    InvGroup rest;
    for (int k = 0; k < nmats; ++k) {
        if (4 * p.chains[k].size() >= 3 * p.longest) p.groups[0].members.push_back(k);
        else rest.members.push_back(k);
    }
    if (!rest.members.empty()) {
        rest.max_ctas = std::max(1, device_sm_count() - RESERVED_SMS);
        p.groups.push_back(rest);
        // the second group's chains without the bulk stream (the chain's
        // ops, and so the grouping, are the same either way)
        for (int k : rest.members)
            if (SIDE_BULK && !BULK_REST) {
                const MatWork &w = p.work[k];
                const bool early = !p.tri[k].empty();
                p.chains[k].clear();
                p.tri[k].clear();
                gen_chain(p.chains[k], p.tri[k], early, false, w, mats[k], info_dev ? info_dev + k : nullptr);
            }
    }
    // rounds, side launches and engine scratch of each group
    const int sms = device_sm_count();
    std::vector<TcJob> round;
    for (InvGroup &g : p.groups) {
        g.rounds = schedule_rounds(p.chains, g.members, g.round_kind);
        g.side_ctas = std::max(1, (g.max_ctas > 0 ? g.max_ctas : sms) - SIDE_FREE_SMS);
        const size_t R = g.rounds.size();
        g.side.assign(R, {});
        g.waits.assign(R, {});
        g.bulk.assign(R, {});
        g.bulk_waits.assign(R, {});
        g.side_bulk_waits.assign(R, {});
        g.bulk_ctas = std::max(1, (g.max_ctas > 0 ? g.max_ctas : sms) - BULK_FREE_SMS);
        std::vector<std::vector<int>> round_of(p.chains.size());
        for (int k : g.members) round_of[k].assign(p.chains[k].size(), -1);
        for (size_t r = 0; r < R; ++r)
            for (const auto &ki : g.rounds[r]) round_of[ki.first][ki.second] = (int)r;
        size_t tcb = 0, sideb = 0, bulkb = 0;
        auto add_wait = [&](std::vector<int> &v, int k, int op) {
            if (op < 0) return;
            const int src = round_of[k][op];
            if (std::find(v.begin(), v.end(), src) == v.end()) v.push_back(src);
        };
        for (size_t r = 0; r < R; ++r) {
            round.clear();
            for (const auto &ki : g.rounds[r]) {
                const Op &op = p.chains[ki.first][ki.second];
                if (op.leaf == 0) round.insert(round.end(), op.g.begin(), op.g.end());
                g.side[r].insert(g.side[r].end(), op.side.begin(), op.side.end());
                g.bulk[r].insert(g.bulk[r].end(), op.bulk.begin(), op.bulk.end());
                add_wait(g.waits[r], ki.first, op.needs_side);
                add_wait(g.bulk_waits[r], ki.first, op.needs_bulk);
                add_wait(g.side_bulk_waits[r], ki.first, op.side_needs_bulk);
            }
            if (!g.bulk[r].empty() && g.side[r].empty()) return KFAC_ERR_UNSUPPORTED;  // (cannot happen)
            if (!g.bulk[r].empty()) {  // on the bulk stream (bulk_ctas) or inline (max_ctas)
                bulkb = std::max(bulkb, tc_workspace_bytes(g.bulk[r].data(), (int)g.bulk[r].size(), TC_KIND_TF32X3,
                                                           g.bulk_ctas));
                bulkb = std::max(bulkb, tc_workspace_bytes(g.bulk[r].data(), (int)g.bulk[r].size(), TC_KIND_TF32X3,
                                                           g.max_ctas));
            }
            tcb = std::max(tcb, tc_workspace_bytes(round.data(), (int)round.size(), TC_KIND_TF32X3, g.max_ctas));
            if (!g.side[r].empty()) {  // launched on the side stream (side_ctas) or inline (max_ctas)
                sideb = std::max(sideb, tc_workspace_bytes(g.side[r].data(), (int)g.side[r].size(), TC_KIND_TF32X3,
                                                           g.side_ctas));
                sideb = std::max(sideb, tc_workspace_bytes(g.side[r].data(), (int)g.side[r].size(), TC_KIND_TF32X3,
                                                           g.max_ctas));
            }
        }
        g.tc_bytes = tcb;
        g.tc_ws = ws.take<char>(tcb);
        for (size_t r = 0; r < R; ++r) {  // every awaited launch exists (else the wait would be a no-op)
            for (int src : g.waits[r])
                if (g.side[src].empty()) return KFAC_ERR_UNSUPPORTED;
            for (const auto *v : {&g.bulk_waits[r], &g.side_bulk_waits[r]})
                for (int src : *v)
                    if (g.bulk[src].empty() || src >= (int)r) return KFAC_ERR_UNSUPPORTED;
        }
        g.side_bytes = sideb;
        g.side_ws = ws.take<char>(sideb);
        g.bulk_bytes = bulkb;
        g.bulk_ws = ws.take<char>(bulkb);

        // early triangular inverse: chains of one padded width have the same
        // steps, batched into one launch each; the widths' sequences are
        // merged by the round each step can be enqueued after
        g.tri.clear();
        g.tri_waits.assign(R, {});
        g.record_main.assign(R, 0);
        g.tri_ctas = std::max(1, (g.max_ctas > 0 ? g.max_ctas : sms) - TRI_FREE_SMS);
        std::vector<int> cls_dp;
        std::vector<std::vector<int>> cls;
        for (int k : g.members) {
            if (p.tri[k].empty()) continue;
            size_t c = 0;
            while (c < cls_dp.size() && cls_dp[c] != p.work[k].dp) ++c;
            if (c == cls_dp.size()) { cls_dp.push_back(p.work[k].dp); cls.emplace_back(); }
            cls[c].push_back(k);
        }
        std::vector<std::pair<int, int>> last_of;  // (class, index in g.tri of its last step)
        std::vector<std::vector<TriStep>> seqs(cls.size());
        for (size_t c = 0; c < cls.size(); ++c) {
            const size_t nsteps = p.tri[cls[c][0]].size();
            int run = 0;
            for (size_t s = 0; s < nsteps; ++s) {
                TriStep st;
                for (int k : cls[c]) {
                    const TriOp &t = p.tri[k][s];
                    st.g.push_back(t.job);
                    const int r = round_of[k][t.after];
                    if (std::find(st.wait_rounds.begin(), st.wait_rounds.end(), r) == st.wait_rounds.end())
                        st.wait_rounds.push_back(r);
                    run = std::max(run, r);
                }
                st.key = run;
                seqs[c].push_back(st);
            }
        }
        std::vector<size_t> pos(cls.size(), 0);
        std::vector<int> last_step(cls.size(), -1);
        for (;;) {  // merge by key, each width's order kept
            int best = -1;
            for (size_t c = 0; c < cls.size(); ++c)
                if (pos[c] < seqs[c].size() && (best < 0 || seqs[c][pos[c]].key < seqs[best][pos[best]].key))
                    best = (int)c;
            if (best < 0) break;
            last_step[best] = (int)g.tri.size();
            g.tri.push_back(seqs[best][pos[best]++]);
        }
        size_t trib = 0;
        for (const TriStep &st : g.tri) {
            for (int r : st.wait_rounds) g.record_main[r] = 1;
            trib = std::max(trib, tc_workspace_bytes(st.g.data(), (int)st.g.size(), TC_KIND_TF32X3, g.tri_ctas));
        }
        // a chain's last op (the final product) waits for its width's last step
        for (size_t c = 0; c < cls.size(); ++c)
            for (int k : cls[c]) {
                const int r = round_of[k][(int)p.chains[k].size() - 1];
                if (!p.chains[k].back().needs_tri || last_step[c] < 0) return KFAC_ERR_UNSUPPORTED;
                if (g.tri[last_step[c]].key >= r) return KFAC_ERR_UNSUPPORTED;  // (cannot happen)
                if (std::find(g.tri_waits[r].begin(), g.tri_waits[r].end(), last_step[c]) == g.tri_waits[r].end())
                    g.tri_waits[r].push_back(last_step[c]);
            }
        g.tri_bytes = trib;
        g.tri_ws = ws.take<char>(trib);
    }
    return KFAC_OK;
}

cudaError_t diag_smem_attr() {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(diag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DIAG_SMEM);
    });
    return err;
}

// One launch per round of leaves (one CTA per diagonal block).
kfac_status diag_launch(const std::vector<DiagJob> &jobs, cudaStream_t st) {
    for (const DiagJob &j : jobs)  // the kernel reads and writes rows in 16-byte pieces
        if (j.ld % 4 != 0 || !j.Sh || !j.Sl || (uintptr_t)j.Sh % 16 != 0 || (uintptr_t)j.Sl % 16 != 0 ||
            (uintptr_t)j.Xh % 16 != 0 || (uintptr_t)j.Xl % 16 != 0 || (uintptr_t)j.Th % 16 != 0 ||
            (uintptr_t)j.Tl % 16 != 0 || (uintptr_t)j.Ph % 16 != 0 || (uintptr_t)j.Pl % 16 != 0 ||
            (uintptr_t)j.Lh % 16 != 0 || (uintptr_t)j.Ll % 16 != 0 || (j.panel && !(j.Ph && j.Pl && j.Lh && j.Ll)) ||
            (!j.panel && !(j.Xh && j.Xl && j.Th && j.Tl)))
            return KFAC_ERR_WORKSPACE;
    if (diag_smem_attr() != cudaSuccess) return KFAC_ERR_CUDA;
    std::unique_ptr<DiagParams> P(new DiagParams);
    size_t pos = 0;
    while (pos < jobs.size()) {
        int n = 0;
        for (; pos < jobs.size() && n < DIAG_MAX; ++pos) P->j[n++] = jobs[pos];
        P->n = n;
        KFAC_LAUNCH(KK_DIAG, st, diag_kernel, n, DIAG_THREADS, DIAG_SMEM, *P);
    }
    return KFAC_OK;
}

kfac_status prep_launch(std::vector<TileMat> &mats, const float *damp, int *err, cudaStream_t st) {
    std::unique_ptr<TileParams> P(new TileParams);
    size_t pos = 0;
    while (pos < mats.size()) {
        int n = 0, tiles = 0;
        while (pos < mats.size() && n < MAT_MAX) {
            TileMat m = mats[pos++];
            m.tiles = (int)ceil_div(m.dp, TT);
            m.vec_f = m.F && m.ldf > 0 && m.ldf % 4 == 0 && (uintptr_t)m.F % 16 == 0;
            P->m[n] = m;
            P->begin[n] = tiles;
            tiles += m.tiles * (m.tiles + 1) / 2;  // upper tile pairs
            ++n;
        }
        P->begin[n] = tiles;
        P->n = n;
        P->damp = damp;
        P->error = err;
        KFAC_LAUNCH(KK_PREP, st, prep_kernel, tiles, 256, 0, *P);
    }
    return KFAC_OK;
}

}  // namespace

size_t inv_workspace_bytes(const InvMatrix *mats, int nmats) {
    Arena a;
    InvPlan p;
    if (plan_inv(mats, nmats, nullptr, a, p, false) != KFAC_OK) return 0;
    return a.used;
}

kfac_status damping_run(const InvMatrix *mats, int nlayers, float gamma, int pi_split,
                        float *damp_dev, cudaStream_t st) {
    std::unique_ptr<DampParams> P(new DampParams);
    int pos = 0;
    while (pos < nlayers) {
        int n = 0;
        const int base = pos;
        while (pos < nlayers && n < MAT_MAX / 2) {
            const InvMatrix &A = mats[2 * pos], &G = mats[2 * pos + 1];
            P->A[n] = A.F; P->lda[n] = A.packed ? -1 : A.ldf; P->dA[n] = A.d;
            P->G[n] = G.F; P->ldg[n] = G.packed ? -1 : G.ldf; P->dG[n] = G.d;
            ++n;
            ++pos;
        }
        P->n = n;
        P->gamma = gamma;
        P->pi_split = pi_split;
        P->damp = damp_dev;
        P->base = base;
        KFAC_LAUNCH(KK_DAMPING, st, damping_kernel, n, 256, 0, *P);
    }
    return KFAC_OK;
}

namespace {

// Enqueue one group's rounds on a stream, its side launches (the lookahead
// updates) on a second stream and its bulk launches on a third: a side
// launch starts once the round that enables it is done (an event), a bulk
// launch once the side launch of its round is done, and a round or side
// launch that needs a side or bulk launch waits for its event.  ev_main /
// ev_side / ev_bulk hold one event per round.
kfac_status run_group(const InvPlan &p, const InvGroup &g, cudaStream_t st, cudaStream_t side, cudaStream_t bulk,
                      cudaStream_t tri, bool use_side, cudaEvent_t *ev_main, cudaEvent_t *ev_side,
                      cudaEvent_t *ev_bulk, cudaEvent_t *ev_tri) {
    std::vector<DiagJob> leaves;
    std::vector<TcJob> gemms;
    kfac_status s = KFAC_OK;
    size_t next_tri = 0;
    for (size_t r = 0; r < g.rounds.size(); ++r) {
        if (use_side) {
            for (int src : g.waits[r]) KFAC_CUDA_TRY(cudaStreamWaitEvent(st, ev_side[src], 0));
            for (int src : g.bulk_waits[r]) KFAC_CUDA_TRY(cudaStreamWaitEvent(st, ev_bulk[src], 0));
        }
        for (int t : g.tri_waits[r]) KFAC_CUDA_TRY(cudaStreamWaitEvent(st, ev_tri[t], 0));
        leaves.clear();
        gemms.clear();
        for (const auto &ki : g.rounds[r]) {
            const Op &op = p.chains[ki.first][ki.second];
            if (op.leaf == 1) leaves.insert(leaves.end(), op.dj.begin(), op.dj.end());
            else gemms.insert(gemms.end(), op.g.begin(), op.g.end());
        }
        if (!leaves.empty() && (s = diag_launch(leaves, st)) != KFAC_OK) return s;
        if (!gemms.empty()) {
            Arena tail(g.tc_ws, g.tc_bytes);
            if ((s = tc_run(gemms.data(), (int)gemms.size(), TC_KIND_TF32X3, p.dev_maps, tail, p.err, st,
                            g.max_ctas)) != KFAC_OK)
                return s;
        }
        if (!g.side[r].empty() && !use_side) {  // side and bulk problems inline, in that order
            Arena tail(g.side_ws, g.side_bytes);
            if ((s = tc_run(g.side[r].data(), (int)g.side[r].size(), TC_KIND_TF32X3, p.dev_maps, tail, p.err, st,
                            g.max_ctas)) != KFAC_OK)
                return s;
            Arena btail(g.bulk_ws, g.bulk_bytes);
            if (!g.bulk[r].empty() && (s = tc_run(g.bulk[r].data(), (int)g.bulk[r].size(), TC_KIND_TF32X3,
                                                  p.dev_maps, btail, p.err, st, g.max_ctas)) != KFAC_OK)
                return s;
        } else if (!g.side[r].empty()) {
            KFAC_CUDA_TRY(cudaEventRecord(ev_main[r], st));
            KFAC_CUDA_TRY(cudaStreamWaitEvent(side, ev_main[r], 0));
            for (int src : g.side_bulk_waits[r]) KFAC_CUDA_TRY(cudaStreamWaitEvent(side, ev_bulk[src], 0));
            Arena tail(g.side_ws, g.side_bytes);
            if ((s = tc_run(g.side[r].data(), (int)g.side[r].size(), TC_KIND_TF32X3, p.dev_maps, tail, p.err, side,
                            g.side_ctas)) != KFAC_OK)
                return s;
            KFAC_CUDA_TRY(cudaEventRecord(ev_side[r], side));
            if (!g.bulk[r].empty()) {
                KFAC_CUDA_TRY(cudaStreamWaitEvent(bulk, ev_side[r], 0));
                Arena btail(g.bulk_ws, g.bulk_bytes);
                if ((s = tc_run(g.bulk[r].data(), (int)g.bulk[r].size(), TC_KIND_TF32X3, p.dev_maps, btail, p.err,
                                bulk, g.bulk_ctas)) != KFAC_OK)
                    return s;
                KFAC_CUDA_TRY(cudaEventRecord(ev_bulk[r], bulk));
            }
        }
        if (g.record_main[r] && !(use_side && !g.side[r].empty())) KFAC_CUDA_TRY(cudaEventRecord(ev_main[r], st));
        // early triangular inverse: every step whose rounds are now enqueued
        for (; next_tri < g.tri.size() && g.tri[next_tri].key <= (int)r; ++next_tri) {
            const TriStep &ts = g.tri[next_tri];
            for (int wr : ts.wait_rounds) KFAC_CUDA_TRY(cudaStreamWaitEvent(tri, ev_main[wr], 0));
            Arena tail(g.tri_ws, g.tri_bytes);
            if ((s = tc_run(ts.g.data(), (int)ts.g.size(), TC_KIND_TF32X3, p.dev_maps, tail, p.err, tri,
                            g.tri_ctas)) != KFAC_OK)
                return s;
            KFAC_CUDA_TRY(cudaEventRecord(ev_tri[next_tri], tri));
        }
    }
    return KFAC_OK;
}

// Library-owned streams and events of one device: a main, a side, a bulk and
// an early-inverse stream for each of the two groups (created on first use; the mutex also keeps
// concurrent callers from interleaving their fork / join records on the
// shared events).
constexpr int EVENT_POOL = 1024;

struct GroupStreams {
    std::mutex mu;
    bool ready = false;
    cudaStream_t main[2] = {nullptr, nullptr}, side[2] = {nullptr, nullptr}, bulk[2] = {nullptr, nullptr},
                 tri[2] = {nullptr, nullptr};
    cudaEvent_t fork = nullptr, done[8] = {};
    std::vector<cudaEvent_t> pool;  // per-round events of the two groups
};

GroupStreams &group_streams(int dev) {
    static GroupStreams gs[64];
    return gs[dev & 63];
}

kfac_status ensure_streams(GroupStreams &g) {
    if (g.ready) return KFAC_OK;
    int least = 0, greatest = 0;
    KFAC_CUDA_TRY(cudaDeviceGetStreamPriorityRange(&least, &greatest));
    for (int k = 0; k < 2; ++k) {
        const int prio = k == 0 ? greatest : least;
        KFAC_CUDA_TRY(cudaStreamCreateWithPriority(&g.main[k], cudaStreamNonBlocking, prio));
        KFAC_CUDA_TRY(cudaStreamCreateWithPriority(&g.side[k], cudaStreamNonBlocking, prio));
        KFAC_CUDA_TRY(cudaStreamCreateWithPriority(&g.bulk[k], cudaStreamNonBlocking, BULK_HIGH_PRIO ? prio : least));
        KFAC_CUDA_TRY(cudaStreamCreateWithPriority(&g.tri[k], cudaStreamNonBlocking, TRI_HIGH_PRIO ? prio : least));
    }
    KFAC_CUDA_TRY(cudaEventCreateWithFlags(&g.fork, cudaEventDisableTiming));
    for (int k = 0; k < 8; ++k) KFAC_CUDA_TRY(cudaEventCreateWithFlags(&g.done[k], cudaEventDisableTiming));
    g.pool.resize(EVENT_POOL);
    for (cudaEvent_t &e : g.pool) KFAC_CUDA_TRY(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    g.ready = true;
    return KFAC_OK;
}

}  // namespace

kfac_status inv_run(const InvMatrix *mats, int nmats, const float *damp_dev, int *info_dev,
                    Arena &ws, cudaStream_t st) {
    InvPlan p;
    kfac_status s = plan_inv(mats, nmats, info_dev, ws, p, true);
    if (s != KFAC_OK) return s;
    if (!ws.fits()) return KFAC_ERR_WORKSPACE;
    KFAC_CUDA_TRY(cudaMemsetAsync(p.err, 0, sizeof(int), st));
    if ((s = tc_upload_maps(p.maps.data(), (int)p.maps.size(), p.dev_maps, st)) != KFAC_OK) return s;

    // 1. X = lower part of sym(F) + damp I (zero above), identity padding
    std::vector<TileMat> tm(nmats);
    for (int k = 0; k < nmats; ++k)
        tm[k] = TileMat{mats[k].F, mats[k].packed ? -1 : mats[k].ldf, p.work[k].Xh, p.work[k].Xl, p.work[k].Dh,
                        p.work[k].Dl, mats[k].d, p.work[k].dp, k, 0, 0};
    if ((s = prep_launch(tm, damp_dev, p.err, st)) != KFAC_OK) return s;

    // 2. rounds (see schedule_rounds), the last op of each chain writing the
    //    caller's inverse: each group on a main stream with a side stream for
    //    its lookahead updates, the critical group at high priority and the
    //    other at low priority, all forked from and joined back into the
    //    caller's stream
    int dev = 0;
    KFAC_CUDA_TRY(cudaGetDevice(&dev));
    GroupStreams &g = group_streams(dev);
    std::lock_guard<std::mutex> lock(g.mu);
    if ((s = ensure_streams(g)) != KFAC_OK) return s;
    size_t events = 0;
    for (const InvGroup &gr : p.groups) events += 3 * gr.rounds.size() + gr.tri.size();
    if (events > g.pool.size()) return KFAC_ERR_UNSUPPORTED;
    const int ngroups = (int)p.groups.size();
    KFAC_CUDA_TRY(cudaEventRecord(g.fork, st));
    for (int k = 0; k < ngroups; ++k) {
        KFAC_CUDA_TRY(cudaStreamWaitEvent(g.main[k], g.fork, 0));
        KFAC_CUDA_TRY(cudaStreamWaitEvent(g.side[k], g.fork, 0));
        KFAC_CUDA_TRY(cudaStreamWaitEvent(g.bulk[k], g.fork, 0));
        KFAC_CUDA_TRY(cudaStreamWaitEvent(g.tri[k], g.fork, 0));
    }
    kfac_status res[2] = {KFAC_OK, KFAC_OK};
    size_t ev = 0;
    for (int k = 0; k < ngroups; ++k) {
        const InvGroup &gr = p.groups[k];
        cudaEvent_t *em = g.pool.data() + ev, *es = em + gr.rounds.size(), *eb = es + gr.rounds.size(),
                    *et = eb + gr.rounds.size();
        ev += 3 * gr.rounds.size() + gr.tri.size();
        const PdlScope pdl(k == 0);  // early-launched CTAs of the low-priority group would hold SMs
        res[k] = run_group(p, gr, g.main[k], g.side[k], g.bulk[k], g.tri[k], k < SIDE_GROUPS, em, es, eb, et);
    }
    // join in every case, so that a capture or later work stays ordered
    for (int k = 0; k < ngroups; ++k) {
        const cudaStream_t sts[4] = {g.main[k], g.side[k], g.bulk[k], g.tri[k]};
        for (int q = 0; q < 4; ++q) {
            KFAC_CUDA_TRY(cudaEventRecord(g.done[4 * k + q], sts[q]));
            KFAC_CUDA_TRY(cudaStreamWaitEvent(st, g.done[4 * k + q], 0));
        }
    }
    if (res[0] != KFAC_OK) return res[0];
    return res[1];
}

}  // namespace kfac
