// patches.cu -- patch-matrix (im2col) formation and the FC bias column of a
// Kronecker factor.
//
// Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
// Kronecker-Factored Approximate Curvature ...", section 3.2, Eq. 5: A_{l-1}
// is formed from the input activations of layer l.  For a convolution the
// rows of the statistic are the receptive-field patches of every output
// position: P[m][(r*kw + s)*c + ch] = x[img][ho*sh - ph + r][wo*sw - pw + s][ch]
// (zero outside the image).  An FC bias adds a column of ones; its row/column
// of A is the column sum of the input and the row count, computed here
// without forming P.
#include <algorithm>
#include <memory>

#include "internal.h"

namespace kfac {

namespace {

constexpr int IM_MAX = 64;

struct ImParams {
    Im2colJob j[IM_MAX];
    long long begin[IM_MAX + 1];  // prefix of work units (units of 8 columns or 1 element)
    int vec8[IM_MAX];
    int n;
};

// One work unit writes 8 consecutive patch columns of one row (16 bytes of
// bf16) when c % 8 == 0, otherwise one element.
template <typename T>
__global__ void im2col_kernel(const __grid_constant__ ImParams P) {
    pdl_wait();
    pdl_trigger();
    const long long total = P.begin[P.n];
    for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < total;
         u += (long long)gridDim.x * blockDim.x) {
        int lo = 0, hi = P.n - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (P.begin[mid] <= u) lo = mid; else hi = mid - 1;
        }
        const Im2colJob &q = P.j[lo];
        // 32-bit index math (a job has fewer than 2^31 units and rows)
        const unsigned local = (unsigned)(u - P.begin[lo]);
        const int dcore = q.kh * q.kw * q.c;
        const int d = dcore + q.append_one;
        const bool v8 = P.vec8[lo] != 0;
        const unsigned per_row = v8 ? dcore / 8 : d;
        const unsigned m = local / per_row;
        const int cu = (int)(local - m * per_row);
        const unsigned t = m / (unsigned)q.wo;
        const int wo = (int)(m - t * (unsigned)q.wo);
        const unsigned img = t / (unsigned)q.ho;
        const int ho = (int)(t - img * (unsigned)q.ho);
        T *prow = (T *)q.P + (long long)m * q.ldp;
        const T *x = (const T *)q.x;
        if (v8) {
            const int col = cu * 8;
            const int rs = col / q.c, ch = col - rs * q.c;
            const int r = rs / q.kw, s = rs - r * q.kw;
            const int hi_ = ho * q.sh - q.ph + r, wi = wo * q.sw - q.pw + s;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (hi_ >= 0 && hi_ < q.h && wi >= 0 && wi < q.w)
                v = *(const uint4 *)(x + (((long long)img * q.h + hi_) * q.w + wi) * q.c + ch);
            *(uint4 *)(prow + col) = v;
            if (q.append_one && cu == per_row - 1) prow[dcore] = (T)1.0f;
        } else {
            const int col = cu;
            T v = (T)0.0f;
            if (col == dcore) {
                v = (T)1.0f;
            } else {
                const int rs = col / q.c, ch = col - rs * q.c;
                const int r = rs / q.kw, s = rs - r * q.kw;
                const int hi_ = ho * q.sh - q.ph + r, wi = wo * q.sw - q.pw + s;
                if (hi_ >= 0 && hi_ < q.h && wi >= 0 && wi < q.w)
                    v = x[(((long long)img * q.h + hi_) * q.w + wi) * q.c + ch];
            }
            prow[col] = v;
        }
    }
}

// Column sums of a bf16 [M][c] matrix, one CTA per 64 columns, fixed
// reduction order; then the bias row/column update of F.
constexpr int CS_MAX = 64;
struct CsParams {
    ColsumJob j[CS_MAX];
    int begin[CS_MAX + 1];  // prefix of 64-column chunks
    long long ldx[CS_MAX];
    int n;
};

__global__ void __launch_bounds__(256) colsum_kernel(const __grid_constant__ CsParams P) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[32][65];
    int lo = 0, hi = P.n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.begin[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    const ColsumJob &q = P.j[lo];
    const long long ldx = P.ldx[lo];
    const int c0 = (blockIdx.x - P.begin[lo]) * 64;
    const int cg = threadIdx.x & 7;   // 8 groups of 8 columns
    const int rg = threadIdx.x >> 3;  // 32 row groups
    float s[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) s[k] = 0.f;
    const int col = c0 + cg * 8;
    const bool vec = (q.c % 8 == 0) && ((ldx % 8) == 0) && ((uintptr_t)q.x % 16 == 0);
    for (long long m = rg; m < q.M; m += 32) {
        const uint16_t *row = q.x + m * ldx;
        if (vec && col + 8 <= q.c) {
            uint4 v = *(const uint4 *)(row + col);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                s[2 * k] += __uint_as_float(w[k] << 16);
                s[2 * k + 1] += __uint_as_float(w[k] & 0xFFFF0000u);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (col + k < q.c) s[k] += bf16_bits_to_f32(row[col + k]);
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) red[rg][cg * 8 + k] = s[k];
    __syncthreads();
    if (threadIdx.x < 64) {
        float t = 0.f;
        for (int r = 0; r < 32; ++r) t += red[r][threadIdx.x];
        const int i = c0 + threadIdx.x;
        if (i < q.c) {
            float *f = q.F + (long long)i * q.ldf + q.c;
            float o = q.alpha * t;
            if (q.beta != 0.f) o = fmaf(q.beta, *f, o);
            *f = o;
        }
        if (blockIdx.x == P.begin[lo] && threadIdx.x == 0) {
            float *f = q.F + (long long)q.c * q.ldf + q.c;
            float o = q.alpha * (float)q.M;
            if (q.beta != 0.f) o = fmaf(q.beta, *f, o);
            *f = o;
        }
    }
}

}  // namespace

kfac_status im2col_run(const Im2colJob *jobs, int njobs, int dtype, cudaStream_t st) {
    std::unique_ptr<ImParams> P(new ImParams);
    int pos = 0;
    while (pos < njobs) {
        int n = 0;
        long long units = 0;
        while (pos < njobs && n < IM_MAX) {
            const Im2colJob &j = jobs[pos++];
            P->j[n] = j;
            const int dcore = j.kh * j.kw * j.c;
            const long long M = (long long)j.n * j.ho * j.wo;
            const bool v8 = dtype == KFAC_BF16 && j.c % 8 == 0 && j.ldp % 8 == 0 &&
                            ((uintptr_t)j.x % 16 == 0) && ((uintptr_t)j.P % 16 == 0);
            P->vec8[n] = v8 ? 1 : 0;
            P->begin[n] = units;
            units += M * (v8 ? dcore / 8 : dcore + j.append_one);
            ++n;
        }
        P->begin[n] = units;
        P->n = n;
        if (units == 0) continue;
        const int threads = 256;
        const long long blocks = std::min<long long>(ceil_div(units, threads), 152LL * 16);
        if (dtype == KFAC_BF16)
            KFAC_LAUNCH(KK_IM2COL, st, im2col_kernel<__nv_bfloat16>, (int)blocks, threads, 0, *P);
        else
            KFAC_LAUNCH(KK_IM2COL, st, im2col_kernel<float>, (int)blocks, threads, 0, *P);
    }
    return KFAC_OK;
}

kfac_status colsum_run(const ColsumJob *jobs, int njobs, cudaStream_t st) {
    std::unique_ptr<CsParams> P(new CsParams);
    int pos = 0;
    while (pos < njobs) {
        int n = 0, chunks = 0;
        while (pos < njobs && n < CS_MAX) {
            const ColsumJob &j = jobs[pos++];
            P->j[n] = j;
            P->ldx[n] = j.c;  // dense rows
            P->begin[n] = chunks;
            chunks += (int)ceil_div(j.c, 64);
            ++n;
        }
        P->begin[n] = chunks;
        P->n = n;
        KFAC_LAUNCH(KK_COLSUM, st, colsum_kernel, chunks, 256, 0, *P);
    }
    return KFAC_OK;
}

}  // namespace kfac
