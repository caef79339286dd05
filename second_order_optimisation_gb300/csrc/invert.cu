// invert.cu -- damped inversion of the Kronecker factors in fp32.
//
// Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
// Kronecker-Factored Approximate Curvature ...", section 3.2, Eq. 6: the
// inverse of G (x) A is G^-1 (x) A^-1, so each factor is inverted on its own.
// Damping (not stated by the paper; the pi-split Tikhonov form of the K-FAC
// method it builds on):
//     pi = sqrt((tr A/dA) / (tr G/dG)),  damp_A = pi sqrt(gamma),  damp_G = sqrt(gamma)/pi.
//
// Algorithm (the matrices advance in batched rounds, one launch per round, see
// schedule_rounds; the longest chains and the rest run as two concurrent
// groups, see InvGroup):
//   1. traces -> damping values (one CTA per layer, fixed reduction order);
//   2. X = sym(F) + damp I, padded with an identity block to a multiple of
//      128 (the inverse of diag(X, I) is diag(X^-1, I)), stored as a (hi, lo)
//      pair with hi exactly representable in tf32 and hi + lo = X;
//   3. inversion by recursive 2x2 blocking on 128-row
//      block boundaries; the Schur complement X22 - X21 X11^-1 X12 is the
//      trailing update of a block Cholesky step:
//        X11 <- X11^-1                               (recursion / leaf)
//        T   <- X11 X12,   U <- T^T                  (tensor cores)
//        X22 <- X22 - X21 T       (symmetric: upper tiles + mirror)
//        X22 <- X22^-1                               (recursion / leaf)
//        X12 <- -T X22,    X21 <- X12^T              (tensor cores)
//        X11 <- X11 - X12 T^T     (symmetric: upper tiles + mirror)
//      The GEMMs run on tcgen05 with three tf32 products per slice
//      (hi*hi + hi*lo + lo*hi) and fp32 accumulation.  Leaves are 128 x 128
//      blocks inverted by one CTA, a Gauss-Jordan sweep with the block in
//      registers (leaf_kernel);
//   4. out = hi + lo of the upper triangle mirrored to the lower one (exact
//      symmetry), plus the optional bf16 copy.
// A pivot that is not positive and finite records its 1-based index in
// info[matrix]; nothing traps or waits.
#include <algorithm>
#include <cfloat>
#include <memory>
#include <mutex>
#include <vector>

#include "internal.h"

namespace kfac {

namespace {

constexpr int LEAF = 128;
constexpr int LEAF_THREADS = 256;  // leaf: publisher warp + 7 warps owning the block
constexpr int MAT_MAX = 224;
// tensor maps of one matrix: X, T, U pairs, each as hi / lo with 128-row and
// with 32-row boxes
constexpr int MAPS_PER_MATRIX = 12;

inline int padded(int d) { return (int)ceil_div(d, LEAF) * LEAF; }

__device__ __forceinline__ float tf32_hi(float v) {
    return __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
}

// ---------------------------------------------------------------- damping

struct DampParams {
    const float *A[MAT_MAX / 2];
    const float *G[MAT_MAX / 2];
    long long lda[MAT_MAX / 2], ldg[MAT_MAX / 2];
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
    for (int i = threadIdx.x; i < P.dA[l]; i += 256) ta += P.A[l][(long long)i * P.lda[l] + i];
    for (int i = threadIdx.x; i < P.dG[l]; i += 256) tg += P.G[l][(long long)i * P.ldg[l] + i];
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

// ------------------------------------------------------ prepare / finish

struct TileMat {
    const float *F;   // prep: factor (upper read); finish: unused
    long long ldf;
    float *Xh, *Xl;   // working pair [dp][dp]
    int d, dp;
    float *out;       // finish: full symmetric fp32 output
    long long ldo;
    uint16_t *out16;  // finish: optional bf16 copy
    long long ld16;
    int damp_idx;
    int tiles;        // 64-wide tiles per side
    int vec_f, vec_o, vec_b;  // F / out rows take 16-byte, out16 rows 8-byte accesses
};

struct TileParams {
    TileMat m[MAT_MAX];
    int begin[MAT_MAX + 1];
    int n;
    const float *damp;
};

constexpr int TT = 64;  // prep / finish tile

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

// Value (r, c) of output tile (ti, tj) from the staged upper tile t of the pair
// (si, sj) = (min, max): the tile itself, its transpose, or (diagonal tile) its
// upper triangle mirrored.
__device__ __forceinline__ float tile_val(const float (*t)[TT + 1], int si, int sj, bool transposed, int r, int c) {
    if (si != sj) return transposed ? t[c][r] : t[r][c];
    return r <= c ? t[r][c] : t[c][r];
}

// X = split(sym(F) + damp I) on [d, d], identity on the padding.  One CTA per
// upper 64 x 64 tile pair: the upper tile of F is read once (16-byte pieces
// where the rows allow) and written to both its own and its mirrored position.
__global__ void __launch_bounds__(256) prep_kernel(const __grid_constant__ TileParams P) {
    pdl_wait();
    pdl_trigger();
    __shared__ float t[TT][TT + 1];
    int si, sj;
    const TileMat &q = tile_of(P, si, sj);
    const int tid = threadIdx.x, rr = tid >> 4, c4 = (tid & 15) * 4;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const int r = rr + 16 * p, i = si * TT + r, j = sj * TT + c4;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (i < q.d) {
            const float *src = q.F + (long long)i * q.ldf + j;
            if (q.vec_f && j + 3 < q.d) {
                const float4 x = *reinterpret_cast<const float4 *>(src);
                v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (j + u < q.d) v[u] = src[u];
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) t[r][c4 + u] = v[u];
    }
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
                if (i >= q.d || j >= q.d) {
                    v = (i == j) ? 1.f : 0.f;
                } else {
                    v = tile_val(t, si, sj, side == 1, r, c);
                    if (i == j) v += dv;
                }
                h[u] = tf32_hi(v);
                l[u] = v - h[u];
            }
            const long long o = (long long)i * q.dp + tj * TT + c4;
            *reinterpret_cast<float4 *>(q.Xh + o) = make_float4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<float4 *>(q.Xl + o) = make_float4(l[0], l[1], l[2], l[3]);
        }
    }
}

// out = hi + lo of the upper triangle, mirrored; optional bf16 copy.  One CTA
// per upper 64 x 64 tile pair of [d, d].
__global__ void __launch_bounds__(256) finish_kernel(const __grid_constant__ TileParams P) {
    pdl_wait();
    pdl_trigger();
    __shared__ float t[TT][TT + 1];
    int si, sj;
    const TileMat &q = tile_of(P, si, sj);
    const int tid = threadIdx.x, rr = tid >> 4, c4 = (tid & 15) * 4;
    {
        float4 h[4], l[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {  // inside [dp, dp]: always in bounds
            const long long o = (long long)(si * TT + rr + 16 * p) * q.dp + sj * TT + c4;
            h[p] = *reinterpret_cast<const float4 *>(q.Xh + o);
            l[p] = *reinterpret_cast<const float4 *>(q.Xl + o);
        }
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int r = rr + 16 * p;
            t[r][c4] = h[p].x + l[p].x;
            t[r][c4 + 1] = h[p].y + l[p].y;
            t[r][c4 + 2] = h[p].z + l[p].z;
            t[r][c4 + 3] = h[p].w + l[p].w;
        }
    }
    __syncthreads();
#pragma unroll
    for (int side = 0; side < 2; ++side) {
        if (side == 1 && si == sj) break;
        const int ti = side ? sj : si, tj = side ? si : sj;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int r = rr + 16 * p, i = ti * TT + r, j = tj * TT + c4;
            if (i >= q.d) continue;
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = tile_val(t, si, sj, side == 1, r, c4 + u);
            float *dst = q.out + (long long)i * q.ldo + j;
            if (q.vec_o && j + 3 < q.d) {
                *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (j + u < q.d) dst[u] = v[u];
            }
            if (q.out16) {
                uint16_t *d16 = q.out16 + (long long)i * q.ld16 + j;
                if (q.vec_b && j + 3 < q.d) {
                    const uint32_t lo2 = f32_to_bf16_bits(v[0]) | ((uint32_t)f32_to_bf16_bits(v[1]) << 16);
                    const uint32_t hi2 = f32_to_bf16_bits(v[2]) | ((uint32_t)f32_to_bf16_bits(v[3]) << 16);
                    *reinterpret_cast<uint2 *>(d16) = make_uint2(lo2, hi2);
                } else {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (j + u < q.d) d16[u] = f32_to_bf16_bits(v[u]);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ leaf

struct LeafJob {
    float *Xh, *Xl;  // block start (row o, column o) of the working pair
    long long ld;
    int o;           // global offset, for info
    int *info;
};

struct LeafParams {
    LeafJob j[MAT_MAX];
    int n;
};

// 1 / x for a positive finite pivot: the hardware approximate reciprocal
// refined by one Newton-Raphson step, r <- r + r (1 - x r) (a short
// dependent chain for the publisher's serial 4 x 4 inverse).
__device__ __forceinline__ float recip_nr(float x) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    const float e = fmaf(-x, r, 1.0f);
    return fmaf(r, e, r);
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;  // two fp32 fused multiply-adds in one instruction
    asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
        " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// In-place inverse of one SPD 128 x 128 block by one CTA: a Gauss-Jordan
// sweep with the block held in registers, four pivots at a time.  A single
// pivot k maps
//   a_ij <- a_ij - a_ik a_kj / a_kk   (i, j != k)
//   a_kj <- a_kj / a_kk,  a_ik <- -a_ik / a_kk,  a_kk <- 1 / a_kk
// and after the last pivot the block holds its inverse.  No pivoting is
// needed: every leading principal block of an SPD matrix is SPD.  Four
// consecutive pivots K = {k .. k+3} (row group s = k / 4) together are the
// block step: with R the rows K, P = R[:, K] and W = P^-1 R,
//   a_ij -= a_iK W_Kj,  a_Kj <- W_Kj,  a_iK <- -a_iK P^-1,  a_KK <- P^-1.
// The sweep keeps the block sign-symmetric -- a_ik = -a_ki when exactly one
// of i, k has been pivoted, a_ik = a_ki otherwise -- so the pivot columns are
// s_i R[:, i] (s_i = -1 for pivoted i) and the new ones -s_i W[:, i]: every
// update is formed from rows K alone.
// Roles (8 warps): warp 0 is the publisher; warps 1..7 own the 32 row groups
// (lane l holds columns 4l .. 4l+3 of its warp's rows).  During step s the
// publisher takes the rows of group s+1 (copied to shared memory by their
// owner one step earlier), applies step s to them, inverts their 4 x 4
// diagonal block and publishes W, s R, -s W and P^-1 of group s+1, while the
// owners apply step s to their rows.  Warp 4 shares the publisher's SM
// sub-partition and owns only 2 groups, the others 5 each, so that the
// publisher's serial chain gets most of its sub-partition's issue slots.  A
// pivot that is not positive and finite is recorded in info and eliminated
// as 1 / a_kk = 0.
__device__ __forceinline__ int leaf_group_start(int hw) {  // first row group of row warp hw (1..7)
    return hw <= 3 ? 5 * (hw - 1) : hw == 4 ? 15 : 17 + 5 * (hw - 5);
}
__device__ __forceinline__ int leaf_group_count(int hw) { return hw == 4 ? 2 : 5; }

__global__ void __launch_bounds__(LEAF_THREADS, 1) leaf_kernel(const __grid_constant__ LeafParams P) {
    pdl_wait();
    pdl_trigger();
    constexpr int N = LEAF, NB = N / 4, MAXG = 5;
    __shared__ __align__(16) float wbuf[2][4][N];   // W = P^-1 R
    __shared__ __align__(16) float cbuf[2][4][N];   // s_i R[p][i]: the pivot columns
    __shared__ __align__(16) float fbuf[2][4][N];   // -s_i W[p][i]: the new pivot columns
    __shared__ __align__(16) float pbuf[2][16];     // P^-1
    __shared__ __align__(16) float rbuf[2][4][N];   // raw rows of the group after next, for the publisher
    __shared__ int bad;
    const LeafJob &J = P.j[blockIdx.x];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool publisher = warp == 0;
    const int g0 = publisher ? 0 : leaf_group_start(warp), gn = publisher ? 0 : leaf_group_count(warp);
    const unsigned FULL = 0xffffffffu;

    float a[4 * MAXG][4];
#pragma unroll
    for (int lg = 0; lg < MAXG; ++lg) {  // 16-byte pieces, all loads issued before the first use
        if (lg >= gn) break;
        float4 h[4], l[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const long long o = (long long)(4 * (g0 + lg) + p) * J.ld + 4 * lane;
            h[p] = *reinterpret_cast<const float4 *>(J.Xh + o);
            l[p] = *reinterpret_cast<const float4 *>(J.Xl + o);
        }
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            a[4 * lg + p][0] = h[p].x + l[p].x;
            a[4 * lg + p][1] = h[p].y + l[p].y;
            a[4 * lg + p][2] = h[p].z + l[p].z;
            a[4 * lg + p][3] = h[p].w + l[p].w;
        }
    }
    if (warp == 1) {  // groups 0 and 1 for the publisher (both owned by warp 1)
#pragma unroll
        for (int p = 0; p < 8; ++p)
            *reinterpret_cast<float4 *>(&rbuf[p >> 2][p & 3][4 * lane]) =
                make_float4(a[p][0], a[p][1], a[p][2], a[p][3]);
    }
    if (tid == 0) bad = -1;
    __syncthreads();

    // ---- publisher helpers (warp 8; lane l holds columns 4l .. 4l+3 of the rows)
    // the 4 x 4 diagonal block of the rows (only lane kn/4 holds P; the other
    // lanes' results are discarded), inverted by four scalar pivots
    auto publish = [&](const float (&R)[4][4], int kn) {
        float b[4][4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int q = 0; q < 4; ++q) b[p][q] = R[p][q];
        int first_bad = -1;  // branch-free inside the serial chain; recorded once below
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const float x = b[v][v];
            const bool ok = x > 0.f && x <= FLT_MAX;  // positive and finite (NaN fails both)
            first_bad = (!ok && first_bad < 0) ? kn + v : first_bad;
            const float d = ok ? recip_nr(x) : 0.f;
            float t[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) t[i] = b[i][v] * d;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (i != v && j != v) b[i][j] = fmaf(-t[i], b[v][j], b[i][j]);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j != v) b[v][j] *= d;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (i != v) b[i][v] = -t[i];
            b[v][v] = d;
        }
        if (lane == (kn >> 2) && first_bad >= 0 && bad < 0) bad = first_bad;
        float pi[4][4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int q = 0; q < 4; ++q) pi[p][q] = __shfl_sync(FULL, b[p][q], kn >> 2);
        const int buf = (kn >> 2) & 1;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            float w[4], c[4], f[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                w[t] = pi[p][0] * R[0][t];
#pragma unroll
                for (int q = 1; q < 4; ++q) w[t] = fmaf(pi[p][q], R[q][t], w[t]);
                const float sg = 4 * lane + t < kn ? -1.f : 1.f;
                c[t] = sg * R[p][t];
                f[t] = -sg * w[t];
            }
            *reinterpret_cast<float4 *>(&wbuf[buf][p][4 * lane]) = make_float4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<float4 *>(&cbuf[buf][p][4 * lane]) = make_float4(c[0], c[1], c[2], c[3]);
            *reinterpret_cast<float4 *>(&fbuf[buf][p][4 * lane]) = make_float4(f[0], f[1], f[2], f[3]);
        }
        if (lane == 0) {
#pragma unroll
            for (int p = 0; p < 4; ++p)
                *reinterpret_cast<float4 *>(&pbuf[buf][4 * p]) = make_float4(pi[p][0], pi[p][1], pi[p][2], pi[p][3]);
        }
    };
    auto load_rows = [&](float (&R)[4][4], int blk) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float4 t = *reinterpret_cast<const float4 *>(&rbuf[blk & 1][p][4 * lane]);
            R[p][0] = t.x; R[p][1] = t.y; R[p][2] = t.z; R[p][3] = t.w;
        }
    };

    // rows r0 .. r0+3 (of a row warp: local rows; of the publisher: R with
    // global first row i0) updated by the block step held in buf
    auto step_rows = [&](float (&X)[4][4], int i0, int buf, const float (&w)[4][4], bool colfix) {
        float cb[4][4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float4 t = *reinterpret_cast<const float4 *>(&cbuf[buf][p][i0]);
            cb[p][0] = t.x; cb[p][1] = t.y; cb[p][2] = t.z; cb[p][3] = t.w;
        }
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float2 m = make_float2(-cb[p][r], -cb[p][r]);
                const float2 lo = ffma2(m, make_float2(w[p][0], w[p][1]), make_float2(X[r][0], X[r][1]));
                const float2 hi = ffma2(m, make_float2(w[p][2], w[p][3]), make_float2(X[r][2], X[r][3]));
                X[r][0] = lo.x; X[r][1] = lo.y; X[r][2] = hi.x; X[r][3] = hi.y;
            }
        if (colfix) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 t = *reinterpret_cast<const float4 *>(&fbuf[buf][q][i0]);
                X[0][q] = t.x; X[1][q] = t.y; X[2][q] = t.z; X[3][q] = t.w;
            }
        }
    };

    if (publisher) {
        float R[4][4];
        load_rows(R, 0);
        publish(R, 0);
    }
    __syncthreads();
#pragma unroll 1
    for (int s = 0; s < NB; ++s) {
        const int k = 4 * s, buf = s & 1;
        float w[4][4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float4 t = *reinterpret_cast<const float4 *>(&wbuf[buf][p][4 * lane]);
            w[p][0] = t.x; w[p][1] = t.y; w[p][2] = t.z; w[p][3] = t.w;
        }
        const bool colfix = lane == s;  // this lane holds the pivot columns k .. k+3
        if (publisher) {
            if (s + 1 < NB) {  // group s+1: its rows as of step s-1, then step s
                float R[4][4];
                load_rows(R, s + 1);
                step_rows(R, k + 4, buf, w, colfix);
                publish(R, k + 4);
            }
        } else {
#pragma unroll
            for (int lg = 0; lg < MAXG; ++lg) {
                if (lg >= gn) break;
                float (&X)[4][4] = *reinterpret_cast<float (*)[4][4]>(&a[4 * lg][0]);
                step_rows(X, 4 * (g0 + lg), buf, w, colfix);
                if (g0 + lg == s) {  // the pivot rows and the pivot block
#pragma unroll
                    for (int p = 0; p < 4; ++p)
#pragma unroll
                        for (int c = 0; c < 4; ++c) X[p][c] = w[p][c];
                    if (colfix) {
#pragma unroll
                        for (int p = 0; p < 4; ++p) {
                            const float4 t = *reinterpret_cast<const float4 *>(&pbuf[buf][4 * p]);
                            X[p][0] = t.x; X[p][1] = t.y; X[p][2] = t.z; X[p][3] = t.w;
                        }
                    }
                }
                if (g0 + lg == s + 2 && s + 2 < NB) {  // rows of group s+2 (after this step) for the publisher
#pragma unroll
                    for (int p = 0; p < 4; ++p)
                        *reinterpret_cast<float4 *>(&rbuf[(s + 2) & 1][p][4 * lane]) =
                            make_float4(X[p][0], X[p][1], X[p][2], X[p][3]);
                }
            }
        }
        __syncthreads();
    }

#pragma unroll
    for (int lg = 0; lg < MAXG; ++lg) {
        if (lg >= gn) break;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float *v = a[4 * lg + p];
            const long long o = (long long)(4 * (g0 + lg) + p) * J.ld + 4 * lane;
            const float4 h = make_float4(tf32_hi(v[0]), tf32_hi(v[1]), tf32_hi(v[2]), tf32_hi(v[3]));
            *reinterpret_cast<float4 *>(J.Xh + o) = h;
            *reinterpret_cast<float4 *>(J.Xl + o) = make_float4(v[0] - h.x, v[1] - h.y, v[2] - h.z, v[3] - h.w);
        }
    }
    if (tid == 0 && bad >= 0 && J.info) atomicCAS(J.info, 0, J.o + bad + 1);
}

// ------------------------------------------------------------- scheduler

struct Op {
    int leaf;
    LeafJob lj;
    TcJob g;
};

// Working buffers of one matrix with d > LEAF.
struct MatWork {
    int d, dp;
    float *Xh, *Xl, *Th, *Tl, *Uh, *Ul;
    int mx, mt, mu;  // map indices (hi; lo at +1)
};

void gen_ops(std::vector<Op> &ops, const MatWork &w, int o, int n, int *info) {
    const long long ld = w.dp;
    if (n == LEAF) {
        Op op{};
        op.leaf = 1;
        op.lj = LeafJob{w.Xh + o * ld + o, w.Xl + o * ld + o, ld, o, info};
        ops.push_back(op);
        return;
    }
    const int nb = n / LEAF, h = LEAF * (nb / 2), m = n - h;
    gen_ops(ops, w, o, h, info);
    auto gemm = [&](int ma, int ar, int ac, int mb, int br, int bc, int M, int N, int K, float alpha,
                    float beta, float *Ch, float *Cl, float *Cth, float *Ctl, int sym) {
        Op op{};
        op.leaf = 0;
        TcJob &j = op.g;
        j.map_a = ma; j.a_row0 = ar; j.a_col0 = ac;
        j.map_b = mb; j.b_row0 = br; j.b_col0 = bc;
        j.M = M; j.N = N; j.K = K;
        j.epi = TC_EPI_SPLIT;
        j.alpha = alpha; j.beta = beta;
        j.C = Ch; j.C_lo = Cl; j.ldc = ld;
        j.Ct = Cth; j.Ct_lo = Ctl; j.ldct = ld;
        j.sym = sym;
        ops.push_back(op);
    };
    const long long x11 = o * ld + o, x12 = o * ld + o + h, x21 = (o + h) * ld + o, x22 = (o + h) * ld + o + h;
    const long long tt = o * ld;  // T block: rows [o, o+h), columns [0, m)
    // T = X11 X12 (B rows = X21 rows), U = T^T
    gemm(w.mx, o, o, w.mx, o + h, o, h, m, h, 1.f, 0.f, w.Th + tt, w.Tl + tt, w.Uh, w.Ul, 0);
    // X22 -= X21 T  (B rows = U rows)
    gemm(w.mx, o + h, o, w.mu, 0, 0, m, m, h, -1.f, 1.f, w.Xh + x22, w.Xl + x22, nullptr, nullptr, 1);
    gen_ops(ops, w, o + h, m, info);
    // X12 = -T X22 (X22 symmetric: B rows = X22 rows), X21 = X12^T
    gemm(w.mt, o, 0, w.mx, o + h, o + h, h, m, m, -1.f, 0.f, w.Xh + x12, w.Xl + x12, w.Xh + x21, w.Xl + x21, 0);
    // X11 -= X12 T^T (B rows = T rows)
    gemm(w.mx, o, o + h, w.mt, o, 0, h, h, m, -1.f, 1.f, w.Xh + x11, w.Xl + x11, nullptr, nullptr, 1);
}

// Round schedule of a group of chains: the group's longest chain sets the
// sequence of rounds (one launch each, leaf or GEMM); every other chain of the
// group is embedded as late as possible into rounds of the same op kind, in
// order.  The long chain's late rounds are small, latency-bound launches with
// most SMs idle, and the shorter chains' work fills them.  Falls back to
// left-aligned lock-step (a leaf and a GEMM launch per round) if a chain does
// not embed.  Rounds list (chain, op) pairs.
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
    // fallback: left-aligned lock-step, leaves then GEMMs in each step
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

// Workspace layout shared by the size query and the run.
// The chains run as two concurrent groups: the longest ones (the critical
// path of the call) on a high-priority stream, all others on a low-priority
// stream whose GEMM launches leave SMs free for the first group.  Each group
// has its own rounds and engine scratch.
constexpr int RESERVED_SMS = 32;  // SMs the second group's GEMM launches leave free

struct InvGroup {
    std::vector<int> members;  // chain indices
    std::vector<std::vector<std::pair<int, int>>> rounds;
    std::vector<int> round_kind;
    int max_ctas = 0;          // GEMM grid cap (0: all SMs)
    char *tc_ws = nullptr;
    size_t tc_bytes = 0;
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

kfac_status plan_inv(const InvMatrix *mats, int nmats, int *info_dev, Arena &ws, InvPlan &p, bool encode) {
    p.err = ws.take<int>(64);
    int nbig = 0;
    for (int k = 0; k < nmats; ++k) nbig += mats[k].d > LEAF;
    p.dev_maps = ws.take<CUtensorMap>(MAPS_PER_MATRIX * (size_t)std::max(nbig, 1));
    p.work.resize(nmats);
    p.chains.assign(nmats, {});
    for (int k = 0; k < nmats; ++k) {
        MatWork &w = p.work[k];
        w.d = mats[k].d;
        w.dp = padded(w.d);
        const size_t sq = (size_t)w.dp * w.dp;
        w.Xh = ws.take<float>(sq);
        w.Xl = ws.take<float>(sq);
        w.Th = w.Tl = w.Uh = w.Ul = nullptr;
        w.mx = w.mt = w.mu = -1;
        if (w.d > LEAF) {
            w.Th = ws.take<float>(sq);
            w.Tl = ws.take<float>(sq);
            w.Uh = ws.take<float>(sq);
            w.Ul = ws.take<float>(sq);
            float *bufs[6] = {w.Xh, w.Xl, w.Th, w.Tl, w.Uh, w.Ul};
            const int base = (int)p.maps.size();
            for (int q = 0; q < 6; q += 2)  // per pair: hi, lo (128-row boxes), hi, lo (32-row boxes)
                for (int v = 0; v < 4; ++v) {
                    p.maps.emplace_back();
                    if (encode && !tc_make_map(&p.maps.back(), TC_KIND_TF32X3, bufs[q + (v & 1)], w.dp, w.dp,
                                               w.dp, 0, v < 2 ? 128 : 32))
                        return KFAC_ERR_CUDA;
                }
            w.mx = base;
            w.mt = base + 4;
            w.mu = base + 8;
        }
        gen_ops(p.chains[k], w, 0, w.dp, info_dev ? info_dev + k : nullptr);
        p.longest = std::max(p.longest, p.chains[k].size());
    }
    if (p.maps.size() != (size_t)MAPS_PER_MATRIX * nbig) return KFAC_ERR_WORKSPACE;  // device map area
    // groups: chains at least 3/4 as long as the longest form the critical
    // group; a second group exists only if it is worth a stream of its own
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
    // engine scratch of each group: its largest GEMM round
    std::vector<TcJob> round;
    for (InvGroup &g : p.groups) {
        g.rounds = schedule_rounds(p.chains, g.members, g.round_kind);
        size_t tcb = 0;
        for (size_t r = 0; r < g.rounds.size(); ++r) {
            round.clear();
            for (const auto &ki : g.rounds[r])
                if (!p.chains[ki.first][ki.second].leaf) round.push_back(p.chains[ki.first][ki.second].g);
            tcb = std::max(tcb, tc_workspace_bytes(round.data(), (int)round.size(), TC_KIND_TF32X3, g.max_ctas));
        }
        g.tc_bytes = tcb;
        g.tc_ws = ws.take<char>(tcb);
    }
    return KFAC_OK;
}

kfac_status leaf_launch(const std::vector<LeafJob> &jobs, cudaStream_t st) {
    for (const LeafJob &j : jobs)  // the kernel moves rows in 16-byte pieces
        if (j.ld % 4 != 0 || (uintptr_t)j.Xh % 16 != 0 || (uintptr_t)j.Xl % 16 != 0) return KFAC_ERR_WORKSPACE;
    std::unique_ptr<LeafParams> P(new LeafParams);
    size_t pos = 0;
    while (pos < jobs.size()) {
        int n = 0;
        while (pos < jobs.size() && n < MAT_MAX) P->j[n++] = jobs[pos++];
        P->n = n;
        KFAC_LAUNCH(KK_LEAF, st, leaf_kernel, n, LEAF_THREADS, 0, *P);
    }
    return KFAC_OK;
}

template <bool PREP>
kfac_status tile_launch(std::vector<TileMat> &mats, const float *damp, cudaStream_t st) {
    std::unique_ptr<TileParams> P(new TileParams);
    size_t pos = 0;
    while (pos < mats.size()) {
        int n = 0, tiles = 0;
        while (pos < mats.size() && n < MAT_MAX) {
            TileMat m = mats[pos++];
            m.tiles = (int)ceil_div(PREP ? m.dp : m.d, TT);
            m.vec_f = m.F && m.ldf % 4 == 0 && (uintptr_t)m.F % 16 == 0;
            m.vec_o = m.out && m.ldo % 4 == 0 && (uintptr_t)m.out % 16 == 0;
            m.vec_b = m.out16 && m.ld16 % 4 == 0 && (uintptr_t)m.out16 % 8 == 0;
            P->m[n] = m;
            P->begin[n] = tiles;
            tiles += m.tiles * (m.tiles + 1) / 2;  // upper tile pairs
            ++n;
        }
        P->begin[n] = tiles;
        P->n = n;
        P->damp = damp;
        if (PREP) KFAC_LAUNCH(KK_PREP, st, prep_kernel, tiles, 256, 0, *P);
        else KFAC_LAUNCH(KK_FINISH, st, finish_kernel, tiles, 256, 0, *P);
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
            P->A[n] = A.F; P->lda[n] = A.ldf; P->dA[n] = A.d;
            P->G[n] = G.F; P->ldg[n] = G.ldf; P->dG[n] = G.d;
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

// Enqueue one group's rounds on a stream.
kfac_status run_group(const InvPlan &p, const InvGroup &g, cudaStream_t st) {
    std::vector<LeafJob> leaves;
    std::vector<TcJob> gemms;
    kfac_status s = KFAC_OK;
    for (size_t r = 0; r < g.rounds.size(); ++r) {
        leaves.clear();
        gemms.clear();
        for (const auto &ki : g.rounds[r]) {
            const Op &op = p.chains[ki.first][ki.second];
            if (op.leaf) leaves.push_back(op.lj); else gemms.push_back(op.g);
        }
        if (!leaves.empty() && (s = leaf_launch(leaves, st)) != KFAC_OK) return s;
        if (!gemms.empty()) {
            Arena tail(g.tc_ws, g.tc_bytes);
            if ((s = tc_run(gemms.data(), (int)gemms.size(), TC_KIND_TF32X3, p.dev_maps, tail, p.err, st,
                            g.max_ctas)) != KFAC_OK)
                return s;
        }
    }
    return KFAC_OK;
}

// Library-owned streams and events of one device for the two groups (created
// on first use; the mutex also keeps concurrent callers from interleaving
// their fork / join records on the shared events).
struct GroupStreams {
    std::mutex mu;
    bool ready = false;
    cudaStream_t hi = nullptr, lo = nullptr;
    cudaEvent_t fork = nullptr, done_hi = nullptr, done_lo = nullptr;
};

GroupStreams &group_streams(int dev) {
    static GroupStreams gs[64];
    return gs[dev & 63];
}

kfac_status ensure_streams(GroupStreams &g) {
    if (g.ready) return KFAC_OK;
    int least = 0, greatest = 0;
    KFAC_CUDA_TRY(cudaDeviceGetStreamPriorityRange(&least, &greatest));
    KFAC_CUDA_TRY(cudaStreamCreateWithPriority(&g.hi, cudaStreamNonBlocking, greatest));
    KFAC_CUDA_TRY(cudaStreamCreateWithPriority(&g.lo, cudaStreamNonBlocking, least));
    KFAC_CUDA_TRY(cudaEventCreateWithFlags(&g.fork, cudaEventDisableTiming));
    KFAC_CUDA_TRY(cudaEventCreateWithFlags(&g.done_hi, cudaEventDisableTiming));
    KFAC_CUDA_TRY(cudaEventCreateWithFlags(&g.done_lo, cudaEventDisableTiming));
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
    if (!p.maps.empty() && (s = tc_upload_maps(p.maps.data(), (int)p.maps.size(), p.dev_maps, st)) != KFAC_OK)
        return s;

    // 1. X = split(sym(F) + damp I), identity padding
    std::vector<TileMat> tm(nmats);
    for (int k = 0; k < nmats; ++k)
        tm[k] = TileMat{mats[k].F, mats[k].ldf, p.work[k].Xh, p.work[k].Xl, mats[k].d, p.work[k].dp,
                        mats[k].out, mats[k].ldo, mats[k].out_bf16, mats[k].ldo_bf16, k, 0, 0, 0, 0};
    if ((s = tile_launch<true>(tm, damp_dev, st)) != KFAC_OK) return s;

    // 2. rounds (see schedule_rounds): each round is one leaf or one GEMM
    //    launch; with two groups, the critical one runs on a high-priority
    //    stream and the other on a low-priority one, forked from and joined
    //    back into the caller's stream
    if (p.groups.size() == 1) {
        if ((s = run_group(p, p.groups[0], st)) != KFAC_OK) return s;
    } else {
        int dev = 0;
        KFAC_CUDA_TRY(cudaGetDevice(&dev));
        GroupStreams &g = group_streams(dev);
        std::lock_guard<std::mutex> lock(g.mu);
        if ((s = ensure_streams(g)) != KFAC_OK) return s;
        KFAC_CUDA_TRY(cudaEventRecord(g.fork, st));
        KFAC_CUDA_TRY(cudaStreamWaitEvent(g.hi, g.fork, 0));
        KFAC_CUDA_TRY(cudaStreamWaitEvent(g.lo, g.fork, 0));
        const kfac_status s0 = run_group(p, p.groups[0], g.hi);
        kfac_status s1;
        {
            const PdlScope no_pdl(false);
            s1 = run_group(p, p.groups[1], g.lo);
        }
        // join in every case, so that a capture or later work stays ordered
        KFAC_CUDA_TRY(cudaEventRecord(g.done_hi, g.hi));
        KFAC_CUDA_TRY(cudaEventRecord(g.done_lo, g.lo));
        KFAC_CUDA_TRY(cudaStreamWaitEvent(st, g.done_hi, 0));
        KFAC_CUDA_TRY(cudaStreamWaitEvent(st, g.done_lo, 0));
        if (s0 != KFAC_OK) return s0;
        if (s1 != KFAC_OK) return s1;
    }

    // 3. out = hi + lo, mirrored; bf16 copies
    return tile_launch<false>(tm, damp_dev, st);
}

}  // namespace kfac
