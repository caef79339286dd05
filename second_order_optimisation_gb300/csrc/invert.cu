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
#include <memory>
#include <mutex>
#include <vector>

#include "internal.h"

namespace kfac {

namespace {

constexpr int NB = 128;    // block width of the sweep
// Lookahead: split each Cholesky update into the last panel's share (kept on
// the chain) and the rest (on a side stream, overlapping the diag leaf and the
// panel).  Measured on the ResNet-50 step it gained nothing (the side
// launches' persistent CTAs hold SMs the chain needs next), so it is off.
constexpr bool LOOKAHEAD = false;
constexpr int MAT_MAX = 224;
// tensor maps of one matrix: X, Wt, LT pairs, each as hi / lo with 128-row
// and with 32-row boxes
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

// X = (lower part of sym(F) + damp I, zero strictly above the diagonal) as a
// (hi, lo) pair on [d, d], identity on the padding.  One CTA per upper 64 x 64
// tile pair: the upper tile of F is read once (16-byte pieces where the rows
// allow) and written transposed to its lower position; the upper position
// gets zeros (the diagonal tile: its lower triangle and zeros).
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
            const long long o = (long long)i * q.dp + tj * TT + c4;
            *reinterpret_cast<float4 *>(q.Xh + o) = make_float4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<float4 *>(q.Xl + o) = make_float4(l[0], l[1], l[2], l[3]);
        }
    }
}

// ------------------------------------------------------------------ diag

struct DiagJob {
    float *Xh, *Xl;    // block (k, k) of the working pair: its lower triangle is read, then
                       // W_kk = L_kk^-1 written over the whole block (zeros above the diagonal)
    float *Th, *Tl;    // the same block of the transposed pair: W_kk^T (zeros below)
    long long ld;
    int o;             // global index of the block's first row (for info)
    int *info;
};

struct DiagParams {
    DiagJob j[MAT_MAX];
    int n;
};

// Cholesky factor and its inverse of one SPD 128 x 128 block S = L L^T, by
// one CTA of 512 threads: W = L^-1, written over the block and, transposed,
// into the same block of the transposed pair.
//
// The sweep works on one array M (the lower triangle, in shared memory) that
// holds the Schur complement still to be factored in its columns past the
// current pivots and the rows of W in progress in the columns before.  A
// single pivot c, with w = 1 / sqrt(M_cc) and p_i = w M_ic (= L_ic), does
//   i > c, j < c:      M_ij -= p_i (w M_cj)    (rows of W in progress)
//   i > c, j = c:      M_ic  = -p_i w
//   i > c, c < j <= i: M_ij -= p_i p_j         (Schur complement)
//   i = c, j < c:      M_cj *= w;   M_cc = w   (row c of W final)
// The kernel runs these rules 8 pivots K = {c .. c+7} at a time:
//   1. each of threads 0..127 applies them to the 8 x 8 pivot block alone
//      (straight-line code on registers), giving W_K, and forms row j = tid
//      of Z [128 x 8]:
//        Z_j = W_K M[K][j]      (j before K: the final rows K of W, as columns)
//        Z_j = W_K^T e_(j-c)    (j in K)
//        Z_j = W_K M[j][K]      (j past K: the panel L_jK);
//   2. rows K:         M[K][j] = Z_j (j before K),  M[K][K] = W_K;
//      rows i past K:  M_ij = (j in K ? 0 : M_ij) - Z_i . Z_j  (j <= i),
//      one row and 8 columns per item, consecutive threads on consecutive rows
//      (the Z_i reads are contiguous, the Z_j reads broadcasts).
// 1 / sqrt is the hardware approximation refined by one Newton-Raphson step,
// y <- y (3 - x y^2) / 2.  A pivot outside [FLT_MIN, inf) is recorded and
// eliminated with w = 0 (the result is then undefined but finite).
constexpr int DLD = NB + 4;  // M row pitch (floats; rows stay 16-byte aligned)
constexpr int DIAG_THREADS = 512;
constexpr size_t DIAG_SMEM = ((size_t)NB * DLD + (size_t)NB * 8 + 64 + 4) * sizeof(float);

__device__ __forceinline__ float rsqrt_nr(float x) {
    const float y = rsqrtf(x);
    return y * fmaf(-0.5f * x * y, y, 1.5f);
}

// The single-pivot rules on an 8 x 8 lower block alone, in registers (every
// loop has constant bounds so that the block stays in registers): W_K in
// place; returns the first pivot (0..7) outside [FLT_MIN, inf), or -1.
__device__ __forceinline__ int pivot8(float (&w)[8][8]) {
    int bad = -1;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float piv = w[q][q];
        const bool ok = piv >= FLT_MIN && piv < INFINITY;
        const float wq = ok ? rsqrt_nr(piv) : 0.f;
        bad = (!ok && bad < 0) ? q : bad;
        float p[8], rowq[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) p[r] = r > q ? w[r][q] * wq : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) rowq[j] = wq * w[q][j];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (r <= q || j > r) continue;
                if (j < q) w[r][j] = fmaf(-p[r], rowq[j], w[r][j]);
                else if (j == q) w[r][j] = -p[r] * wq;
                else w[r][j] = fmaf(-p[r], p[j], w[r][j]);
            }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < q) w[q][j] *= wq;
        w[q][q] = wq;
    }
    return bad;
}

__global__ void __launch_bounds__(DIAG_THREADS, 1) diag_kernel(const __grid_constant__ DiagParams P) {
    extern __shared__ float4 diag_smem4[];
    float *M = reinterpret_cast<float *>(diag_smem4);
    float *Z = M + NB * DLD;       // [NB][8]
    float *wk = Z + NB * 8;          // [8][8]
    int *bad_s = reinterpret_cast<int *>(wk + 64);
    const DiagJob &J = P.j[blockIdx.x];
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid == 0) *bad_s = -1;
    pdl_wait();
    pdl_trigger();
    for (int e = tid; e < NB * NB / 4; e += DIAG_THREADS) {
        const int i = e >> 5, j = (e & 31) * 4;
        const long long off = (long long)i * J.ld + j;
        const float4 h = *reinterpret_cast<const float4 *>(J.Xh + off);
        const float4 l = *reinterpret_cast<const float4 *>(J.Xl + off);
        *reinterpret_cast<float4 *>(M + i * DLD + j) = make_float4(h.x + l.x, h.y + l.y, h.z + l.z, h.w + l.w);
    }
    __syncthreads();
#pragma unroll 1
    for (int s = 0; s < NB / 8; ++s) {
        const int c = 8 * s, E = c + 8;
        // 1. + 2. Z rows, one per thread t < 128; each such thread first turns
        //    the 8 x 8 pivot block into W_K itself (the single-pivot rules on
        //    the block alone, in registers): j < c: W_K M[K][j];  j in K:
        //    W_K^T e;  j past K: W_K M[j][K]
        if (tid < NB) {
            float w[8][8];
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int q = 0; q < 8; ++q) w[r][q] = q <= r ? M[(c + r) * DLD + c + q] : 0.f;
            const int bad = pivot8(w);
            if (tid == 0) {
#pragma unroll
                for (int r = 0; r < 8; ++r)
#pragma unroll
                    for (int q = 0; q < 8; ++q) wk[r * 8 + q] = w[r][q];
                if (bad >= 0 && *bad_s < 0) *bad_s = c + bad;
            }
            // Z_j = W_K x with x = M[K][j] (j before K), e_(j-c) (j in K), M[j][K] (j past K)
            const int j = tid;
            float x[8];
            if (j < c) {
#pragma unroll
                for (int r = 0; r < 8; ++r) x[r] = M[(c + r) * DLD + j];
            } else if (j < E) {
#pragma unroll
                for (int r = 0; r < 8; ++r) x[r] = j - c == r ? 1.f : 0.f;
            } else {
                const float4 a = *reinterpret_cast<const float4 *>(M + j * DLD + c);
                const float4 b = *reinterpret_cast<const float4 *>(M + j * DLD + c + 4);
                x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
            }
            float z[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float acc = 0.f;
#pragma unroll
                for (int r = 0; r < 8; ++r) acc = r <= q ? fmaf(w[q][r], x[r], acc) : acc;
                z[q] = acc;
            }
            *reinterpret_cast<float4 *>(Z + j * 8) = make_float4(z[0], z[1], z[2], z[3]);
            *reinterpret_cast<float4 *>(Z + j * 8 + 4) = make_float4(z[4], z[5], z[6], z[7]);
        }
        __syncthreads();
        // 3. rows K: M[K][j] = Z_j (j < c), W_K on the pivot block
        for (int e = tid; e < 8 * E; e += DIAG_THREADS) {
            const int q = e / E, j = e - q * E;
            if (j < c) M[(c + q) * DLD + j] = Z[j * 8 + q];
            else if (j - c <= q) M[(c + q) * DLD + j] = wk[q * 8 + (j - c)];
        }
        //    rows past K, one row i and 8 columns 8J .. 8J+7 (8J <= i) per
        //    item, consecutive threads on consecutive rows:
        //    M_ij = (j in K ? 0 : M_ij) - Z_i . Z_j  for j <= i
        for (int J = tid >> 7; J < 16; J += DIAG_THREADS / NB) {
            const int i = tid & (NB - 1);
            if (i < E || 8 * J > i) continue;
            float acc[8];
            {
                const float4 a = *reinterpret_cast<const float4 *>(M + i * DLD + 8 * J);
                const float4 b = *reinterpret_cast<const float4 *>(M + i * DLD + 8 * J + 4);
                acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w; acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
            }
            if (8 * J == c) {  // the columns K take -Z_i . W_K
#pragma unroll
                for (int v = 0; v < 8; ++v) acc[v] = 0.f;
            }
            const float4 za = *reinterpret_cast<const float4 *>(Z + i * 8);
            const float4 zb = *reinterpret_cast<const float4 *>(Z + i * 8 + 4);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const float4 a = *reinterpret_cast<const float4 *>(Z + (8 * J + v) * 8);
                const float4 b = *reinterpret_cast<const float4 *>(Z + (8 * J + v) * 8 + 4);
                float x = acc[v];
                x = fmaf(-za.x, a.x, x); x = fmaf(-za.y, a.y, x); x = fmaf(-za.z, a.z, x); x = fmaf(-za.w, a.w, x);
                x = fmaf(-zb.x, b.x, x); x = fmaf(-zb.y, b.y, x); x = fmaf(-zb.z, b.z, x); acc[v] = fmaf(-zb.w, b.w, x);
            }
            if (8 * J + 7 <= i) {
                *reinterpret_cast<float4 *>(M + i * DLD + 8 * J) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                *reinterpret_cast<float4 *>(M + i * DLD + 8 * J + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
            } else {
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    if (8 * J + v <= i) M[i * DLD + 8 * J + v] = acc[v];
            }
        }
        __syncthreads();
    }
    // W (lower, zeros above) into X and W^T (upper, zeros below) into the transposed pair
    for (int e = tid; e < NB * NB / 4; e += DIAG_THREADS) {
        const int i = e >> 5, j = (e & 31) * 4;
        float w4[4], t4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            w4[u] = j + u <= i ? M[i * DLD + j + u] : 0.f;
            t4[u] = i <= j + u ? M[(j + u) * DLD + i] : 0.f;
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
    if (tid == 0 && *bad_s >= 0 && J.info) atomicCAS(J.info, 0, J.o + *bad_s + 1);
    __syncthreads();
}

// ------------------------------------------------------------- scheduler

// One launch unit of a matrix's chain: a diag leaf, or engine problems that
// go into the same launch.
struct Op {
    int leaf;
    DiagJob dj;
    std::vector<TcJob> g;
    std::vector<TcJob> side;  // engine problems that may start once this op is done (lookahead,
                              // launched on the group's side stream)
    int needs_side = -1;      // chain index of the op whose side problems must be done first
};

// Working buffers of one matrix (fp32 (hi, lo) pairs, [dp][dp] each):
//   X   lower part: the factor, its block columns updated into Schur-complement
//       columns, then W = L^-1 (diagonal blocks from the diag leaves, the
//       rest from the triangular inverse); strictly upper part zero
//   Wt  upper part: W^T (diagonal blocks in full, zeros below)
//   LT  lower blocks: the Cholesky panels L_ik (i > k);  upper blocks:
//       (L21 W11)^T of the triangular inverse
struct MatWork {
    int d, dp;
    float *Xh, *Xl, *Wh, *Wl, *Lh, *Ll;
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
//       X[k:, k] -= L[k:, :k] L[k, :k]^T                 (engine; k > 0)
//       W_kk = L_kk^-1 from X[k, k]                      (diag leaf)
//       L[k+1:, k] = X[k+1:, k] W_kk^T                   (engine; the panel)
//     every Schur-complement column comes from Cholesky panels (no growth).
//     The update of column k by panels 0 .. k-2 needs nothing later than
//     panel k-2: it runs as a side problem once that panel is done (on the
//     group's side stream, while the diag leaf and panel of k-1 run), and
//     only the update by panel k-1 (K = 128) stays on the chain;
//  2. W = L^-1 by recursive 2 x 2 blocking, bottom up by height (the two
//     halves of a node are independent):
//       T = L21 W11,   W21 = -W22 T   (W21 over X's lower part, W21^T into Wt);
//  3. X^-1 = W^T W = Wt Wt^T, written into the caller's output.
// W11, W22 are lower triangular with zeros above in X and their transposes
// upper triangular with zeros below in Wt, so the products run over whole
// blocks; T reads W11^T from Wt only from each output tile's first column on
// (ktri), where Wt holds its upper part and diagonal blocks.
void gen_chain(std::vector<Op> &ops, const MatWork &w, const InvMatrix &mat, int *info) {
    const long long ld = w.dp;
    const int nb = w.dp / NB;
    std::vector<int> panel_op(nb, -1);
    for (int k = 0; k < nb; ++k) {
        const int kb = k * NB;
        if (k > 0 && !LOOKAHEAD) {
            Op op{};
            op.g.push_back(split_job(w.ml, kb, 0, w.ml, kb, 0, w.dp - kb, NB, kb, -1.f, 1.f, w.Xh + kb * ld + kb,
                                     w.Xl + kb * ld + kb, nullptr, nullptr, ld));
            ops.push_back(op);
        } else if (k > 0) {
            // the update by the last panel (k - 1) stays on the chain; the
            // earlier panels' share ran as the lookahead of panel k - 2
            Op op{};
            op.g.push_back(split_job(w.ml, kb, kb - NB, w.ml, kb, kb - NB, w.dp - kb, NB, NB, -1.f, 1.f,
                                     w.Xh + kb * ld + kb, w.Xl + kb * ld + kb, nullptr, nullptr, ld));
            if (k >= 2) op.needs_side = panel_op[k - 2];
            ops.push_back(op);
        }
        {
            Op op{};
            op.leaf = 1;
            op.dj = DiagJob{w.Xh + kb * ld + kb, w.Xl + kb * ld + kb, w.Wh + kb * ld + kb, w.Wl + kb * ld + kb,
                            ld, kb, info};
            ops.push_back(op);
        }
        if (k + 1 < nb) {
            const long long c = (long long)(kb + NB) * ld + kb;
            Op op{};
            op.g.push_back(split_job(w.mx, kb + NB, kb, w.mx, kb, kb, w.dp - kb - NB, NB, NB, 1.f, 0.f, w.Lh + c,
                                     w.Ll + c, nullptr, nullptr, ld));
            if (k + 2 < nb && LOOKAHEAD) {
                // lookahead: X[k2:, k2] -= L[k2:, :k+1] L[k2, :k+1]^T for block column k2 = k + 2
                const int k2b = (k + 2) * NB;
                op.side.push_back(split_job(w.ml, k2b, 0, w.ml, k2b, 0, w.dp - k2b, NB, kb + NB, -1.f, 1.f,
                                            w.Xh + k2b * ld + k2b, w.Xl + k2b * ld + k2b, nullptr, nullptr, ld));
            }
            panel_op[k] = (int)ops.size();
            ops.push_back(op);
        }
    }
    std::vector<std::vector<std::pair<int, int>>> by_height;
    tri_nodes(0, w.dp, by_height);
    for (size_t ht = 1; ht < by_height.size(); ++ht) {
        Op t{}, x{};
        for (const auto &nd : by_height[ht]) {
            const int o = nd.first, n = nd.second, h = NB * (n / NB / 2), m = n - h;
            const long long x21 = (long long)(o + h) * ld + o, t12 = (long long)o * ld + o + h;
            // T = L21 W11 (B rows: W11^T rows, in Wt), stored as T^T in LT's upper part
            t.g.push_back(split_job(w.ml, o + h, o, w.mw, o, o, m, h, h, 1.f, 0.f, nullptr, nullptr, w.Lh + t12,
                                    w.Ll + t12, ld));
            t.g.back().ktri = 1;
            // W21 = -W22 T (A: W22 rows, in X; B rows: T^T rows, in LT), W21^T into Wt
            x.g.push_back(split_job(w.mx, o + h, o + h, w.ml, o, o + h, m, h, m, -1.f, 0.f, w.Xh + x21,
                                    w.Xl + x21, w.Wh + t12, w.Wl + t12, ld));
            x.g.back().ktril = 1;  // W22 is lower triangular
        }
        ops.push_back(t);
        ops.push_back(x);
    }
    Op fin{};
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
        for (int kind = 1; kind >= 0; --kind) {
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
constexpr int RESERVED_SMS = 32;   // SMs the second group's engine launches leave free
constexpr int SIDE_FREE_SMS = 48;  // SMs a group's side launches leave to its own chain
constexpr int SIDE_GROUPS = 1;     // groups whose lookahead updates run on a side stream (the others
                                   // run them in their own stream, right after the enabling round)

struct InvGroup {
    std::vector<int> members;  // chain indices
    std::vector<std::vector<std::pair<int, int>>> rounds;
    std::vector<int> round_kind;
    std::vector<std::vector<TcJob>> side;   // per round: side problems launched once it is done
    std::vector<std::vector<int>> waits;    // per round: rounds whose side launch must finish first
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
    std::vector<InvGroup> groups;  // groups[0]: the critical chains
    size_t longest = 0;
};

// Workspace layout shared by the size query and the run.
kfac_status plan_inv(const InvMatrix *mats, int nmats, int *info_dev, Arena &ws, InvPlan &p, bool encode) {
    p.err = ws.take<int>(64);
    p.dev_maps = ws.take<CUtensorMap>(MAPS_PER_MATRIX * (size_t)std::max(nmats, 1));
    p.work.resize(nmats);
    p.chains.assign(nmats, {});
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
        if (w.dp > NB) {
            w.Lh = ws.take<float>(sq);
            w.Ll = ws.take<float>(sq);
        }
        float *bufs[6] = {w.Xh, w.Xl, w.Wh, w.Wl, w.Lh, w.Ll};
        const int base = (int)p.maps.size();
        for (int q = 0; q < 6; q += 2)  // per pair: hi, lo (128-row boxes), hi, lo (32-row boxes)
            for (int v = 0; v < 4; ++v) {
                p.maps.emplace_back();
                if (encode && bufs[q] &&
                    !tc_make_map(&p.maps.back(), TC_KIND_TF32X3, bufs[q + (v & 1)], w.dp, w.dp, w.dp, v < 2 ? 128 : 32))
                    return KFAC_ERR_CUDA;
            }
        w.mx = base;
        w.mw = base + 4;
        w.ml = base + 8;
        gen_chain(p.chains[k], w, mats[k], info_dev ? info_dev + k : nullptr);
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
        std::vector<std::vector<int>> round_of(p.chains.size());
        for (int k : g.members) round_of[k].assign(p.chains[k].size(), -1);
        for (size_t r = 0; r < R; ++r)
            for (const auto &ki : g.rounds[r]) round_of[ki.first][ki.second] = (int)r;
        size_t tcb = 0, sideb = 0;
        for (size_t r = 0; r < R; ++r) {
            round.clear();
            for (const auto &ki : g.rounds[r]) {
                const Op &op = p.chains[ki.first][ki.second];
                if (!op.leaf) round.insert(round.end(), op.g.begin(), op.g.end());
                g.side[r].insert(g.side[r].end(), op.side.begin(), op.side.end());
                if (op.needs_side >= 0) {
                    const int src = round_of[ki.first][op.needs_side];
                    if (std::find(g.waits[r].begin(), g.waits[r].end(), src) == g.waits[r].end())
                        g.waits[r].push_back(src);
                }
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
        g.side_bytes = sideb;
        g.side_ws = ws.take<char>(sideb);
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
    for (const DiagJob &j : jobs)  // the kernel writes rows in 16-byte pieces
        if (j.ld % 4 != 0 || (uintptr_t)j.Xh % 16 != 0 || (uintptr_t)j.Xl % 16 != 0 || (uintptr_t)j.Th % 16 != 0 ||
            (uintptr_t)j.Tl % 16 != 0)
            return KFAC_ERR_WORKSPACE;
    if (diag_smem_attr() != cudaSuccess) return KFAC_ERR_CUDA;
    std::unique_ptr<DiagParams> P(new DiagParams);
    size_t pos = 0;
    while (pos < jobs.size()) {
        int n = 0;
        for (; pos < jobs.size() && n < MAT_MAX; ++pos) P->j[n++] = jobs[pos];
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

// Enqueue one group's rounds on a stream, and its side launches (the
// lookahead updates) on a second stream: a side launch starts once the round
// that enables it is done (an event), and a round that needs a side launch
// waits for its event.  ev_main / ev_side hold one event per round.
kfac_status run_group(const InvPlan &p, const InvGroup &g, cudaStream_t st, cudaStream_t side, bool use_side,
                      cudaEvent_t *ev_main, cudaEvent_t *ev_side) {
    std::vector<DiagJob> leaves;
    std::vector<TcJob> gemms;
    kfac_status s = KFAC_OK;
    for (size_t r = 0; r < g.rounds.size(); ++r) {
        if (use_side)
            for (int src : g.waits[r]) KFAC_CUDA_TRY(cudaStreamWaitEvent(st, ev_side[src], 0));
        leaves.clear();
        gemms.clear();
        for (const auto &ki : g.rounds[r]) {
            const Op &op = p.chains[ki.first][ki.second];
            if (op.leaf) leaves.push_back(op.dj);
            else gemms.insert(gemms.end(), op.g.begin(), op.g.end());
        }
        if (!leaves.empty() && (s = diag_launch(leaves, st)) != KFAC_OK) return s;
        if (!gemms.empty()) {
            Arena tail(g.tc_ws, g.tc_bytes);
            if ((s = tc_run(gemms.data(), (int)gemms.size(), TC_KIND_TF32X3, p.dev_maps, tail, p.err, st,
                            g.max_ctas)) != KFAC_OK)
                return s;
        }
        if (!g.side[r].empty() && !use_side) {
            Arena tail(g.side_ws, g.side_bytes);
            if ((s = tc_run(g.side[r].data(), (int)g.side[r].size(), TC_KIND_TF32X3, p.dev_maps, tail, p.err, st,
                            g.max_ctas)) != KFAC_OK)
                return s;
        } else if (!g.side[r].empty()) {
            KFAC_CUDA_TRY(cudaEventRecord(ev_main[r], st));
            KFAC_CUDA_TRY(cudaStreamWaitEvent(side, ev_main[r], 0));
            Arena tail(g.side_ws, g.side_bytes);
            if ((s = tc_run(g.side[r].data(), (int)g.side[r].size(), TC_KIND_TF32X3, p.dev_maps, tail, p.err, side,
                            g.side_ctas)) != KFAC_OK)
                return s;
            KFAC_CUDA_TRY(cudaEventRecord(ev_side[r], side));
        }
    }
    return KFAC_OK;
}

// Library-owned streams and events of one device: a main and a side stream
// for each of the two groups (created on first use; the mutex also keeps
// concurrent callers from interleaving their fork / join records on the
// shared events).
constexpr int EVENT_POOL = 1024;

struct GroupStreams {
    std::mutex mu;
    bool ready = false;
    cudaStream_t main[2] = {nullptr, nullptr}, side[2] = {nullptr, nullptr};
    cudaEvent_t fork = nullptr, done[4] = {nullptr, nullptr, nullptr, nullptr};
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
    }
    KFAC_CUDA_TRY(cudaEventCreateWithFlags(&g.fork, cudaEventDisableTiming));
    for (int k = 0; k < 4; ++k) KFAC_CUDA_TRY(cudaEventCreateWithFlags(&g.done[k], cudaEventDisableTiming));
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
        tm[k] = TileMat{mats[k].F, mats[k].packed ? -1 : mats[k].ldf, p.work[k].Xh, p.work[k].Xl, mats[k].d,
                        p.work[k].dp, k, 0, 0};
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
    for (const InvGroup &gr : p.groups) events += 2 * gr.rounds.size();
    if (events > g.pool.size()) return KFAC_ERR_UNSUPPORTED;
    const int ngroups = (int)p.groups.size();
    KFAC_CUDA_TRY(cudaEventRecord(g.fork, st));
    for (int k = 0; k < ngroups; ++k) {
        KFAC_CUDA_TRY(cudaStreamWaitEvent(g.main[k], g.fork, 0));
        KFAC_CUDA_TRY(cudaStreamWaitEvent(g.side[k], g.fork, 0));
    }
    kfac_status res[2] = {KFAC_OK, KFAC_OK};
    size_t ev = 0;
    for (int k = 0; k < ngroups; ++k) {
        const InvGroup &gr = p.groups[k];
        cudaEvent_t *em = g.pool.data() + ev, *es = em + gr.rounds.size();
        ev += 2 * gr.rounds.size();
        const PdlScope pdl(k == 0);  // early-launched CTAs of the low-priority group would hold SMs
        res[k] = run_group(p, gr, g.main[k], g.side[k], k < SIDE_GROUPS, em, es);
    }
    // join in every case, so that a capture or later work stays ordered
    for (int k = 0; k < ngroups; ++k) {
        KFAC_CUDA_TRY(cudaEventRecord(g.done[2 * k], g.main[k]));
        KFAC_CUDA_TRY(cudaEventRecord(g.done[2 * k + 1], g.side[k]));
        KFAC_CUDA_TRY(cudaStreamWaitEvent(st, g.done[2 * k], 0));
        KFAC_CUDA_TRY(cudaStreamWaitEvent(st, g.done[2 * k + 1], 0));
    }
    if (res[0] != KFAC_OK) return res[0];
    return res[1];
}

}  // namespace kfac
