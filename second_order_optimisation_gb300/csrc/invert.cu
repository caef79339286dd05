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
//   3. inversion by recursive 2x2 blocking on 128-row block boundaries down
//      to leaves of 128 or 256 rows; the Schur complement X22 - X21 X11^-1 X12
//      is the trailing update of a block Cholesky step:
//        X11 <- X11^-1                               (recursion / leaf)
//        T   <- X11 X12,   U <- T^T                  (tensor cores)
//        X22 <- X22 - X21 T       (symmetric: upper tiles + mirror)
//        X22 <- X22^-1                               (recursion / leaf)
//        X12 <- -T X22,    X21 <- X12^T              (tensor cores)
//        X11 <- X11 - X12 T^T     (symmetric: upper tiles + mirror)
//      The GEMMs run on tcgen05 with three tf32 products per slice
//      (hi*hi + hi*lo + lo*hi) and fp32 accumulation.  A leaf is inverted
//      by one CTA with the block resident in TMEM: a Gauss-Jordan sweep in
//      32-wide block steps, each one rank-32 tensor-core product (tleaf_kernel);
//   4. out = hi + lo of the upper triangle mirrored to the lower one (exact
//      symmetry), plus the optional bf16 copy.
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

constexpr int LEAF = 128;
constexpr int LEAF_MAX = 256;  // largest leaf block (one CTA, block resident in TMEM)
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

// ------------------------------------------------------------------ leaves

struct LeafJob {
    float *Xh, *Xl;  // block start (row o, column o) of the working pair
    long long ld;
    int o;           // global offset, for info
    int *info;
    int n;           // block size: LEAF or 2 LEAF
};

struct LeafParams {
    LeafJob j[MAT_MAX];
    int n;
    int *error;      // timeout bits (TMEM-resident leaf)
};

// In-place inverse of one SPD N x N block (N = 128 or 256) by one CTA of N
// threads, a blocked Gauss-Jordan sweep whose block steps run on the tensor
// cores.  The block lives in TMEM for the whole sweep (row i at lane i % 128,
// columns (i / 128) N .. +N-1); the CTA holds all of TMEM when N = 256.
// Block step s pivots on K = {32s .. 32s+31}.  With C = A[:, K] (the pivot
// column panel), P = A[K, K], W = P^-1 A[K, :] and E_K the rows of the
// identity on K, the complete Gauss-Jordan update
//   a_ij -= a_iK W_Kj,  a_Kj <- W_Kj,  a_iK <- -a_iK P^-1,  a_KK <- P^-1
// is the single rank-32 product  A += (-C~) W~^T  where C~ = C - E_K (rows K
// of the panel become P - I) and W~ = W with the columns K replaced by
// I + P^-1; it runs as tf32 products of (hi, lo) splits (hi*hi + hi*lo +
// lo*hi) with fp32 accumulation in TMEM.  The block stays sign-symmetric
// (a_ij = -a_ji when exactly one of i, j has been pivoted), so A[K, j] is
// +-C[j, :] and W never needs the pivot rows themselves: the product on the
// columns K runs first and gives -C P^-1, and its rows are the columns of W
// up to sign.  The next step's panel columns are updated (and signalled) ahead
// of the rest of the product, whose MMAs overlap the next pivot block's
// inverse (P^-1: a 32 x 32 Gauss-Jordan sweep by the warp holding rows K).
// A pivot outside [FLT_MIN, inf) (not positive, subnormal or not finite) is
// recorded in info and eliminated as 1 / a_kk = 0; the inverse is then
// undefined, but the sweep runs to its end.
template <int N>
struct TLeafSmem {
    static constexpr int NH = N / 128;                 // 128-row halves
    static constexpr uint32_t A_TILE = 128 * 128;      // 128 rows x 32 tf32 (128-byte swizzled rows)
    static constexpr uint32_t B_TILE = N * 128;        // N rows x 32 tf32
    static constexpr uint32_t OFF_A = 0;               // [2 buffers][NH][hi, lo]
    static constexpr uint32_t OFF_B = OFF_A + 2 * NH * 2 * A_TILE;  // [hi, lo]
    static constexpr uint32_t OFF_K = OFF_B + 2 * B_TILE;           // pivot block B operand [hi, lo]
    static constexpr uint32_t OFF_BAR = OFF_K + 2 * 4096;
    static constexpr uint32_t BYTES = OFF_BAR + 64 + 1024;          // + alignment slack
    static constexpr int STG = 36;                                  // row pitch of the I/O staging (floats)
};

// Row r (32 tf32 of K) of a 128-byte-swizzled K-major operand tile, split
// into hi / lo tiles.
__device__ __forceinline__ void stage_row_split(uint8_t *hi, uint8_t *lo, int r, const float *x) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float4 v = make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
        const float4 h = make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z), tf32_hi(v.w));
        const uint32_t off = (uint32_t)r * 128u + ((uint32_t)(c ^ (r & 7)) << 4);
        *reinterpret_cast<float4 *>(hi + off) = h;
        *reinterpret_cast<float4 *>(lo + off) = make_float4(v.x - h.x, v.y - h.y, v.z - h.z, v.w - h.w);
    }
}

// D[128 x ncols] += A[128 x 32] B[ncols x 32]^T with (hi, lo) operand tiles.
__device__ __forceinline__ void tleaf_mma(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo,
                                          int ncols) {
    const uint32_t idesc = idesc_tf32_f32(128, ncols);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ah = smem_desc_sw128(a_hi + kk * 32, 16, 1024), al = smem_desc_sw128(a_lo + kk * 32, 16, 1024);
        const uint64_t bh = smem_desc_sw128(b_hi + kk * 32, 16, 1024), bl = smem_desc_sw128(b_lo + kk * 32, 16, 1024);
        tc_mma_tf32(d, ah, bh, idesc, 1u);
        tc_mma_tf32(d, ah, bl, idesc, 1u);
        tc_mma_tf32(d, al, bh, idesc, 1u);
    }
}

// 1 / x for a pivot in [FLT_MIN, inf): the flush-to-zero approximate
// reciprocal refined by one Newton-Raphson step, r <- r + r (1 - x r).
__device__ __forceinline__ float recip_ftz_nr(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return fmaf(r, fmaf(-x, r, 1.0f), r);
}

// In-place inverse of the 32 x 32 pivot block held by one warp (lane r: row
// r), Gauss-Jordan without pivoting (every leading block of an SPD matrix is
// SPD).  The pivot row is broadcast with shuffles.  The row registers rotate
// by one column per pivot (position j holds column (k + j) mod 32 before
// pivot k), so that the pivot column is always p[0] and every index is
// static; after 32 pivots the columns are back in place.  Rows i != k take
// a_ij - f a_kj with f = a_ik / a_kk; the pivot row takes f = 1 - 1 / a_kk,
// which turns the same FMA into a_kj / a_kk.  Returns the first pivot that
// was not in [FLT_MIN, inf) (-1 if none); such a pivot is eliminated as
// 1 / a_kk = 0.
__device__ __forceinline__ int pivot_block_inverse(float (&p)[32], int lane) {
    int bad = -1;
#pragma unroll 2
    for (int k = 0; k < 32; ++k) {
        float pk[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) pk[j] = __shfl_sync(0xffffffffu, p[j], k);
        const float d = pk[0];
        const bool ok = d >= 1.17549435e-38f && d < INFINITY;
        const float inv = ok ? recip_ftz_nr(d) : 0.f;
        if (!ok && bad < 0) bad = k;
        const bool own = lane == k;
        const float f = own ? 1.f - inv : p[0] * inv;
#pragma unroll
        for (int j = 0; j < 31; ++j) p[j] = fmaf(-f, pk[j + 1], p[j + 1]);
        p[31] = own ? inv : -f;  // column k, now at the last position
    }
    return bad;
}

template <int N>
__global__ void __launch_bounds__(N, 1) tleaf_kernel(const __grid_constant__ LeafParams P) {
    using S = TLeafSmem<N>;
    constexpr int NH = S::NH, NS = N / 32;
    constexpr uint32_t NCOL = N == 128 ? 128 : 512;
    extern __shared__ uint8_t tl_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)tl_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bar_k = (uint64_t *)(smem + S::OFF_BAR);
    uint64_t *bar_next = bar_k + 1;
    uint64_t *bar_done = bar_k + 2;
    uint32_t *tmem_slot = (uint32_t *)(bar_k + 3);
    int *bad_s = (int *)(tmem_slot + 1);
    volatile int *abort_s = bad_s + 1;  // a wait ran out: every thread leaves the sweep

    const LeafJob &J = P.j[blockIdx.x];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = warp >> 2, q = warp & 3;
    const int row = 128 * h + 32 * q + lane;   // this thread's row of the block
    const int row0 = row - lane;               // first row of this warp
    const uint32_t lane_field = (uint32_t)(32 * q) << 16;

    if (warp == 0) tmem_alloc(tmem_slot, NCOL);
    if (tid == 0) {
        mbar_init(bar_k, 1);
        mbar_init(bar_next, 1);
        mbar_init(bar_done, 1);
        *bad_s = -1;
        *abort_s = 0;
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_row = tmem + lane_field + (uint32_t)(h * N);  // column 0 of this thread's row
    pdl_wait();
    pdl_trigger();

    // ---- load: X = hi + lo into TMEM (coalesced through a per-warp stage)
    float *stg = (float *)(smem + S::OFF_A) + warp * 32 * S::STG;
#pragma unroll 1
    for (int c = 0; c < N / 32; ++c) {
        float4 hv[8], lv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const long long off = (long long)(row0 + 4 * k + (lane >> 3)) * J.ld + 32 * c + 4 * (lane & 7);
            hv[k] = *reinterpret_cast<const float4 *>(J.Xh + off);
            lv[k] = *reinterpret_cast<const float4 *>(J.Xl + off);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4 *>(&stg[(4 * k + (lane >> 3)) * S::STG + 4 * (lane & 7)]) =
                make_float4(hv[k].x + lv[k].x, hv[k].y + lv[k].y, hv[k].z + lv[k].z, hv[k].w + lv[k].w);
        __syncwarp();
        float v[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 t = *reinterpret_cast<const float4 *>(&stg[lane * S::STG + 4 * j]);
            v[4 * j] = t.x; v[4 * j + 1] = t.y; v[4 * j + 2] = t.z; v[4 * j + 3] = t.w;
        }
        tmem_st_32x32b_x32(t_row + 32 * c, v);
        __syncwarp();
    }
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();

    uint8_t *const kb_hi = smem + S::OFF_K, *const kb_lo = kb_hi + 4096;
    uint8_t *const bu_hi = smem + S::OFF_B, *const bu_lo = bu_hi + S::B_TILE;
#pragma unroll 1
    for (int s = 0; s < NS; ++s) {
        const int ks = 32 * s;
        const int pw = 4 * (ks >> 7) + ((ks & 127) >> 5);  // warp holding rows K
        uint8_t *const au_hi = smem + S::OFF_A + (uint32_t)(((s & 1) * NH + h) * 2) * S::A_TILE;
        uint8_t *const au_lo = au_hi + S::A_TILE;
        // panel C = A[:, K] (updated by the previous step's first MMAs); the
        // thread issuing the previous step's remaining MMAs joins later
        if (s > 0 && !mbar_wait(bar_next, (uint32_t)((s - 1) & 1))) *abort_s = 1;
        __syncwarp();  // warp 0 reconverges after its MMA issue (tcgen05.ld is warp-collective)
        tc_fence_after();
        float c[32];
        tmem_ld_32x32b_x32(t_row + ks, c);
        const bool in_k = row >= ks && row < ks + 32;
        {
            const int dj = in_k ? row - ks : -1;  // this row's column inside K
            float a[32];  // -(C - E_K)
#pragma unroll
            for (int j = 0; j < 32; ++j) a[j] = __int_as_float(__float_as_int(1.f) & -(int)(dj == j)) - c[j];
            stage_row_split(au_hi, au_lo, 32 * q + lane, a);
        }
        if (warp == pw) {  // P^-1, then the pivot block's B rows I + P^-1
            const int bad = pivot_block_inverse(c, lane);
            if (lane == 0 && bad >= 0 && *bad_s < 0) *bad_s = ks + bad;
#pragma unroll
            for (int j = 0; j < 32; ++j) c[j] += j == lane ? 1.f : 0.f;
            stage_row_split(kb_hi, kb_lo, lane, c);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (*abort_s) break;
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                const uint32_t a0 = smem_u32(smem + S::OFF_A + (uint32_t)(((s & 1) * NH + hh) * 2) * S::A_TILE);
                tleaf_mma(tmem + (uint32_t)(hh * N + ks), a0, a0 + S::A_TILE, smem_u32(kb_hi), smem_u32(kb_lo), 32);
            }
            tc_commit(bar_k);
        }
        // columns K now hold -C P^-1 (rows outside K) and P^-1 (rows K);
        // W[:, i] = +v (i pivoted before this step) or -v (i after K)
        if (!mbar_wait(bar_k, (uint32_t)(s & 1))) *abort_s = 1;
        __syncwarp();
        tc_fence_after();
        {
            float v[32];
            tmem_ld_32x32b_x32(t_row + ks, v);
            if (!in_k) {
                if (row > ks) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = -v[j];
                }
                stage_row_split(bu_hi, bu_lo, row, v);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (*abort_s) break;
        if (tid == 0) {
            tc_fence_after();
            const uint32_t bh = smem_u32(bu_hi), bl = smem_u32(bu_lo);
            const bool more = s + 1 < NS;
            if (more) {  // the next panel first
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) {
                    const uint32_t a0 = smem_u32(smem + S::OFF_A + (uint32_t)(((s & 1) * NH + hh) * 2) * S::A_TILE);
                    tleaf_mma(tmem + (uint32_t)(hh * N + ks + 32), a0, a0 + S::A_TILE, bh + (ks + 32) * 128,
                              bl + (ks + 32) * 128, 32);
                }
                tc_commit(bar_next);
            }
            const int r1 = more ? ks + 64 : N;  // remaining columns: [0, ks) and [r1, N)
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                const uint32_t a0 = smem_u32(smem + S::OFF_A + (uint32_t)(((s & 1) * NH + hh) * 2) * S::A_TILE);
                if (ks > 0) tleaf_mma(tmem + (uint32_t)(hh * N), a0, a0 + S::A_TILE, bh, bl, ks);
                if (r1 < N)
                    tleaf_mma(tmem + (uint32_t)(hh * N + r1), a0, a0 + S::A_TILE, bh + r1 * 128, bl + r1 * 128, N - r1);
            }
            if (!more) tc_commit(bar_done);
        }
    }
    bool ok = !*abort_s && mbar_wait(bar_done, 0u);
    ok = __syncthreads_and(ok);
    if (!ok && tid == 0 && P.error) atomicOr(P.error, ERR_TIMEOUT_LEAF);
    tc_fence_after();

    // ---- store: A^-1 as (hi, lo) (coalesced through the per-warp stage)
    if (ok) {
#pragma unroll 1
        for (int c = 0; c < N / 32; ++c) {
            float v[32];
            tmem_ld_32x32b_x32(t_row + 32 * c, v);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<float4 *>(&stg[lane * S::STG + 4 * j]) =
                    make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 t = *reinterpret_cast<const float4 *>(&stg[(4 * k + (lane >> 3)) * S::STG + 4 * (lane & 7)]);
                const float4 hh = make_float4(tf32_hi(t.x), tf32_hi(t.y), tf32_hi(t.z), tf32_hi(t.w));
                const long long off = (long long)(row0 + 4 * k + (lane >> 3)) * J.ld + 32 * c + 4 * (lane & 7);
                *reinterpret_cast<float4 *>(J.Xh + off) = hh;
                *reinterpret_cast<float4 *>(J.Xl + off) = make_float4(t.x - hh.x, t.y - hh.y, t.z - hh.z, t.w - hh.w);
            }
            __syncwarp();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, NCOL);
    }
    if (tid == 0 && *bad_s >= 0 && J.info) atomicCAS(J.info, 0, J.o + *bad_s + 1);
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
    if (n == LEAF || n == LEAF_MAX) {  // one leaf launch (TMEM-resident block)
        Op op{};
        op.leaf = 1;
        op.lj = LeafJob{w.Xh + o * ld + o, w.Xl + o * ld + o, ld, o, info, n};
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
                                               w.dp, v < 2 ? 128 : 32))
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

template <int N>
cudaError_t tleaf_smem_attr() {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(tleaf_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)TLeafSmem<N>::BYTES);
    });
    return err;
}

// One launch per leaf size present in the round (N threads, one CTA per block).
kfac_status leaf_launch(const std::vector<LeafJob> &jobs, int *err, cudaStream_t st) {
    for (const LeafJob &j : jobs)  // the kernel moves rows in 16-byte pieces
        if (j.ld % 4 != 0 || (uintptr_t)j.Xh % 16 != 0 || (uintptr_t)j.Xl % 16 != 0 ||
            (j.n != LEAF && j.n != LEAF_MAX))
            return KFAC_ERR_WORKSPACE;
    std::unique_ptr<LeafParams> P(new LeafParams);
    for (int size : {LEAF, LEAF_MAX}) {
        size_t pos = 0;
        while (pos < jobs.size()) {
            int n = 0;
            for (; pos < jobs.size() && n < MAT_MAX; ++pos)
                if (jobs[pos].n == size) P->j[n++] = jobs[pos];
            if (n == 0) break;
            P->n = n;
            P->error = err;
            if (size == 128) {
                if (tleaf_smem_attr<128>() != cudaSuccess) return KFAC_ERR_CUDA;
                KFAC_LAUNCH(KK_LEAF, st, tleaf_kernel<128>, n, 128, TLeafSmem<128>::BYTES, *P);
            } else {
                if (tleaf_smem_attr<256>() != cudaSuccess) return KFAC_ERR_CUDA;
                KFAC_LAUNCH(KK_LEAF, st, tleaf_kernel<256>, n, 256, TLeafSmem<256>::BYTES, *P);
            }
        }
        if (LEAF_MAX == LEAF) break;
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
        if (!leaves.empty() && (s = leaf_launch(leaves, p.err, st)) != KFAC_OK) return s;
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
