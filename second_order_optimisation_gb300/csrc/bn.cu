// bn.cu -- diagonal Fisher of BatchNorm parameters.
//
// Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
// Kronecker-Factored Approximate Curvature ...", section 1 (contributions):
// the Fisher of BatchNormalization layers is approximated as a diagonal
// matrix.  From per-sample gradients x[n][C] of a BN scale or shift vector:
//   F_c <- xi F_c + (1 - xi) mean_i x_ic^2,  g_c = mean_i x_ic,
//   out_c = g_c / (F_c + gamma).
//
// Pure HBM streaming: one launch covers every tensor; each CTA owns 64
// columns of one tensor over all rows (16 column quads x 16 row groups,
// float4 loads, four rows in flight per thread), then reduces the 16 row
// groups in a fixed order, so no cross-CTA step and bitwise-stable results.
#include <algorithm>
#include <memory>

#include "internal.h"

namespace kfac {

namespace {

constexpr int BN_MAX = 224;

struct BnParams {
    kfac_bn_desc d[BN_MAX];
    int begin[BN_MAX + 1];  // prefix of 64-column chunks
    int n;
    int ns;
    float gamma, xi;
};

__global__ void __launch_bounds__(256) bn_fisher_kernel(const __grid_constant__ BnParams P) {
    pdl_wait();
    pdl_trigger();
    __shared__ float4 red_s[16][17];
    __shared__ float4 red_q[16][17];
    int lo = 0, hi = P.n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.begin[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    const kfac_bn_desc &q = P.d[lo];
    const int C = q.C;
    const int c0 = (blockIdx.x - P.begin[lo]) * 64;
    const int cq = threadIdx.x & 15;  // column quad
    const int rg = threadIdx.x >> 4;  // row group
    const int col = c0 + cq * 4;
    const int ns = P.ns;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f), s2 = s;
    const bool vec = (C % 4 == 0) && ((uintptr_t)q.x % 16 == 0);
    if (vec && col < C) {
        const float4 *x = (const float4 *)(q.x + col);
        const long long ld4 = C / 4;
        int r = rg;
        for (; r + 48 < ns; r += 64) {
            float4 v0 = __ldcs(x + (long long)r * ld4);
            float4 v1 = __ldcs(x + (long long)(r + 16) * ld4);
            float4 v2 = __ldcs(x + (long long)(r + 32) * ld4);
            float4 v3 = __ldcs(x + (long long)(r + 48) * ld4);
#define ACC(v)                                                             \
    s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;                        \
    s2.x = fmaf(v.x, v.x, s2.x); s2.y = fmaf(v.y, v.y, s2.y);              \
    s2.z = fmaf(v.z, v.z, s2.z); s2.w = fmaf(v.w, v.w, s2.w);
            ACC(v0) ACC(v1) ACC(v2) ACC(v3)
        }
        for (; r < ns; r += 16) {
            float4 v = __ldcs(x + (long long)r * ld4);
            ACC(v)
        }
#undef ACC
    } else {
        float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
        for (int r = rg; r < ns; r += 16)
            for (int k = 0; k < 4; ++k)
                if (col + k < C) {
                    float v = q.x[(long long)r * C + col + k];
                    a[k] += v;
                    b[k] = fmaf(v, v, b[k]);
                }
        s = make_float4(a[0], a[1], a[2], a[3]);
        s2 = make_float4(b[0], b[1], b[2], b[3]);
    }
    red_s[rg][cq] = s;
    red_q[rg][cq] = s2;
    __syncthreads();
    if (threadIdx.x < 64) {
        const int qd = threadIdx.x >> 2, lane = threadIdx.x & 3;
        float ts = 0.f, tq = 0.f;
        for (int r = 0; r < 16; ++r) {
            const float *ps = (const float *)&red_s[r][qd];
            const float *pq = (const float *)&red_q[r][qd];
            ts += ps[lane];
            tq += pq[lane];
        }
        const int c = c0 + threadIdx.x;
        if (c < C) {
            const float inv_n = 1.0f / (float)ns;
            float f = tq * inv_n;
            if (P.xi != 0.f) f = fmaf(P.xi, q.F[c], (1.0f - P.xi) * f);
            const float g = ts * inv_n;
            q.F[c] = f;
            if (q.grad_mean) q.grad_mean[c] = g;
            q.precond[c] = g / (f + P.gamma);
        }
    }
}

}  // namespace

}  // namespace kfac

extern "C" kfac_status kfac_bn_diag_fisher(const kfac_bn_desc *descs, int count, int n_samples,
                                           float gamma, float xi, void *stream) {
    using namespace kfac;
    if (count < 0 || (count > 0 && !descs) || n_samples < 1 || !(gamma >= 0.f) || !(xi >= 0.f) ||
        !(xi <= 1.f))
        return KFAC_ERR_INVALID;
    for (int i = 0; i < count; ++i) {
        const kfac_bn_desc &d = descs[i];
        if (!d.x || !d.F || !d.precond || d.C < 1) return KFAC_ERR_INVALID;
    }
    if (count == 0) return KFAC_OK;
    for (int i = 0; i < count; ++i) {
        const kfac_bn_desc &d = descs[i];
        if (!all_on_this_device({d.x, d.F, d.precond, d.grad_mean})) return KFAC_ERR_INVALID;
    }
    cudaStream_t st = (cudaStream_t)stream;
    std::unique_ptr<BnParams> P(new BnParams);
    int pos = 0;
    while (pos < count) {
        int n = 0, chunks = 0;
        while (pos < count && n < BN_MAX) {
            P->d[n] = descs[pos++];
            P->begin[n] = chunks;
            chunks += (P->d[n].C + 63) / 64;
            ++n;
        }
        P->begin[n] = chunks;
        P->n = n;
        P->ns = n_samples;
        P->gamma = gamma;
        P->xi = xi;
        KFAC_LAUNCH(KK_BN, st, bn_fisher_kernel, chunks, 256, 0, *P);
    }
    return KFAC_OK;
}
