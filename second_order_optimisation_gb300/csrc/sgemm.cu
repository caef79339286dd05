// sgemm.cu -- batched fp32 CUDA-core GEMM for the fp32-input path of the
// K-FAC step (Osawa et al., "Large-Scale Distributed Second-Order
// Optimization Using Kronecker-Factored Approximate Curvature ...",
// section 3.2): the factor statistic P^T P of fp32 sources (Eq. 5) and the
// preconditioned gradient G^-1 grad A^-1 of fp32 operands (Eq. 7).
//
// C[M x N] = alpha * op(A) op(B) + beta * C (and optionally W -= eta * C, the
// step on the weights of Eq. 8), one 128x128 tile per CTA, 256
// threads with 8x8 register tiles, K in steps of 16 staged through shared
// memory with register prefetch of the next step.  One launch covers a list
// of independent problems (heterogeneous sizes).
#include <algorithm>
#include <memory>
#include <vector>

#include "internal.h"

namespace kfac {

namespace {

constexpr int SB = 128, SK = 16, STHREADS = 256, SG_MAX = 96;

struct SgProb {
    const float *A;
    const float *B;
    float *C;
    float *Ct;
    float *W;
    long long lda, ldb, ldc, ldct, ldw;
    float eta;
    int ta, tb, M, N, K, upper, tiles_n, tile_begin;
    int packed_d;  // upper: C is a packed upper triangle of this order (0: row-major)
    float alpha, beta;
};

struct SgParams {
    SgProb p[SG_MAX];
    int n;
    int *error;  // device error word (ERR_NONFINITE), or null
};

__global__ void __launch_bounds__(STHREADS) sgemm_kernel(const __grid_constant__ SgParams P) {
    pdl_wait();
    pdl_trigger();
    __shared__ __align__(16) float As[SK][SB];
    __shared__ __align__(16) float Bs[SK][SB];

    int lo = 0, hi = P.n - 1;
    const int bid = blockIdx.x;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.p[mid].tile_begin <= bid) lo = mid; else hi = mid - 1;
    }
    const SgProb &q = P.p[lo];
    int t = bid - q.tile_begin, tm, tn;
    if (q.upper) {
        int T = q.tiles_n;
        tm = 0;
        while (t >= T - tm) { t -= T - tm; ++tm; }
        tn = tm + t;
    } else {
        tm = t / q.tiles_n;
        tn = t - tm * q.tiles_n;
    }
    const int m0 = tm * SB, n0 = tn * SB;
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    float ra[8], rb[8];
    auto load = [&](int k0) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            int e = tid + r * STHREADS;
            int m, k;
            if (q.ta) { k = e >> 7; m = e & 127; } else { m = e >> 4; k = e & 15; }
            int gm = m0 + m, gk = k0 + k;
            ra[r] = (gm < q.M && gk < q.K)
                        ? (q.ta ? q.A[(long long)gk * q.lda + gm] : q.A[(long long)gm * q.lda + gk])
                        : 0.f;
            int n;
            if (q.tb) { n = e >> 4; k = e & 15; } else { k = e >> 7; n = e & 127; }
            int gn = n0 + n;
            gk = k0 + k;
            rb[r] = (gn < q.N && gk < q.K)
                        ? (q.tb ? q.B[(long long)gn * q.ldb + gk] : q.B[(long long)gk * q.ldb + gn])
                        : 0.f;
        }
    };
    auto store = [&]() {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            int e = tid + r * STHREADS;
            int m, k, n;
            if (q.ta) { k = e >> 7; m = e & 127; } else { m = e >> 4; k = e & 15; }
            As[k][m] = ra[r];
            if (q.tb) { n = e >> 4; k = e & 15; } else { k = e >> 7; n = e & 127; }
            Bs[k][n] = rb[r];
        }
    };

    load(0);
    for (int k0 = 0; k0 < q.K; k0 += SK) {
        __syncthreads();
        store();
        __syncthreads();
        if (k0 + SK < q.K) load(k0 + SK);
#pragma unroll
        for (int kk = 0; kk < SK; ++kk) {
            float4 a0 = *(const float4 *)&As[kk][ty * 4];
            float4 a1 = *(const float4 *)&As[kk][64 + ty * 4];
            float4 b0 = *(const float4 *)&Bs[kk][tx * 4];
            float4 b1 = *(const float4 *)&Bs[kk][64 + tx * 4];
            float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }

    bool bad = false;  // a value this thread stored was NaN or infinite
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int gi = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (gi >= q.M) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int gj = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
            if (gj >= q.N || (q.upper && gj < gi)) continue;
            float o = q.alpha * acc[i][j];
            if (q.C) {
                float *c = q.C + (q.packed_d ? (long long)gi * q.packed_d - (long long)gi * (gi + 1) / 2
                                             : (long long)gi * q.ldc) + gj;
                if (q.beta != 0.f) o = fmaf(q.beta, *c, o);
                *c = o;
            }
            if (q.Ct) q.Ct[(long long)gj * q.ldct + gi] = o;
            bad |= !(fabsf(o) <= 3.402823466e38f);
            if (q.W) {
                float *w = q.W + (long long)gi * q.ldw + gj;
                const float nw = fmaf(-q.eta, o, *w);
                bad |= !(fabsf(nw) <= 3.402823466e38f);
                *w = nw;
            }
        }
    }
    if (__any_sync(0xffffffffu, bad) && (tid & 31) == 0 && P.error) atomicOr(P.error, ERR_NONFINITE);
}

}  // namespace

kfac_status sg_run(const SgJob *jobs, int njobs, int *err, cudaStream_t st) {
    std::unique_ptr<SgParams> P(new SgParams);
    P->error = err;
    int pos = 0;
    while (pos < njobs) {
        int n = 0, tiles = 0;
        while (pos < njobs && n < SG_MAX) {
            const SgJob &j = jobs[pos++];
            if (j.M <= 0 || j.N <= 0) continue;
            SgProb &q = P->p[n];
            q.A = j.A; q.B = j.B; q.C = j.C; q.Ct = j.Ct;
            q.lda = j.lda; q.ldb = j.ldb; q.ldc = j.ldc; q.ldct = j.ldct;
            q.ta = j.ta; q.tb = j.tb; q.M = j.M; q.N = j.N; q.K = j.K;
            q.upper = j.upper;
            q.W = j.W; q.ldw = j.ldw; q.eta = j.eta;
            q.packed_d = j.upper ? j.packed_d : 0;
            q.alpha = j.alpha; q.beta = j.beta;
            int tm = (int)ceil_div(j.M, SB), tn = (int)ceil_div(j.N, SB);
            q.tiles_n = tn;
            q.tile_begin = tiles;
            tiles += j.upper ? tn * (tn + 1) / 2 : tm * tn;
            ++n;
        }
        if (n == 0) break;
        P->n = n;
        KFAC_LAUNCH(KK_SGEMM, st, sgemm_kernel, tiles, STHREADS, 0, *P);
    }
    return KFAC_OK;
}

}  // namespace kfac
