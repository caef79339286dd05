// invert.cu -- damped inversion of the Kronecker factors in fp32.
//
// Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
// Kronecker-Factored Approximate Curvature ...", section 3.2, Eq. 6: the
// inverse of G (x) A is G^-1 (x) A^-1, so each factor is inverted on its own.
// Damping (not stated by the paper; the pi-split Tikhonov form of the K-FAC
// method it builds on):
//     pi = sqrt((tr A/dA) / (tr G/dG)),  damp_A = pi sqrt(gamma),  damp_G = sqrt(gamma)/pi.
//
// Algorithm (every matrix of the call advances in lock-step, one batched
// launch per step):
//   1. traces -> damping values (one CTA per layer, fixed reduction order);
//   2. X = sym(F) + damp I into the output buffer (F's upper triangle read);
//   3. blocked Cholesky-based inversion by recursive 2x2 blocking
//        X11 <- X11^-1                               (recursion / leaf)
//        T   <- X11 X12                              (GEMM)
//        X22 <- X22 - X12^T T     (Schur complement = trailing Cholesky update)
//        X22 <- X22^-1                               (recursion / leaf)
//        X12 <- -T X22,  X21 <- X12^T                (GEMM)
//        X11 <- X11 - X12 T^T                        (GEMM)
//      leaves (n <= 128) run in one CTA in shared memory: Cholesky
//      X = U^T U, triangular inverse V = U^-1, then V V^T;
//   4. mirror the upper triangle to the lower one (exact symmetry) and write
//      the optional bf16 copies.
// A pivot that is not positive and finite records its 1-based global index in
// info[matrix]; nothing traps or waits.
#include <algorithm>
#include <memory>
#include <vector>

#include "internal.h"

namespace kfac {

namespace {

constexpr int LEAF = 128;
constexpr int LEAF_THREADS = 512;
constexpr int MAT_MAX = 224;

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

// --------------------------------------------------- symmetrise / mirror

struct SymMat {
    const float *src;
    long long lds;
    float *dst;
    long long ldd;
    uint16_t *dst16;
    long long ld16;
    int n;
    int tiles;      // tiles per side (32x32)
    int damp_idx;   // -1: none
};

struct SymParams {
    SymMat m[MAT_MAX];
    int begin[MAT_MAX + 1];
    int n;
    int in_place;   // 1: src == dst, mirror upper -> lower
    const float *damp;
};

__global__ void __launch_bounds__(256) sym_kernel(const __grid_constant__ SymParams P) {
    __shared__ float t[32][33];
    int lo = 0, hi = P.n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.begin[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    const SymMat &q = P.m[lo];
    const int tt = blockIdx.x - P.begin[lo];
    const int ti = tt / q.tiles, tj = tt - ti * q.tiles;
    const int si = min(ti, tj), sj = max(ti, tj);
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    // load source tile (si, sj) of the upper triangle
    for (int r = ty; r < 32; r += 8) {
        const int i = si * 32 + r, j = sj * 32 + tx;
        t[r][tx] = (i < q.n && j < q.n) ? q.src[(long long)i * q.lds + j] : 0.f;
    }
    __syncthreads();
    if (P.in_place && ti < tj && !q.dst16) return;
    const float dv = (q.damp_idx >= 0) ? P.damp[q.damp_idx] : 0.f;
    for (int r = ty; r < 32; r += 8) {
        const int i = ti * 32 + r, j = tj * 32 + tx;
        if (i >= q.n || j >= q.n) continue;
        float v;
        if (ti < tj) v = t[r][tx];
        else if (ti > tj) v = t[tx][r];
        else v = (r <= tx) ? t[r][tx] : t[tx][r];
        if (i == j) v += dv;
        if (!(P.in_place && ti < tj)) q.dst[(long long)i * q.ldd + j] = v;
        if (q.dst16) q.dst16[(long long)i * q.ld16 + j] = f32_to_bf16_bits(v);
    }
}

// ------------------------------------------------------------------ leaf

struct LeafJob {
    float *X;       // block start (row o, column o)
    long long ld;
    int n;
    int o;          // global offset, for info
    int *info;
};

struct LeafParams {
    LeafJob j[MAT_MAX];
    int n;
};

__global__ void __launch_bounds__(LEAF_THREADS) leaf_kernel(const __grid_constant__ LeafParams P) {
    extern __shared__ float sm[];
    const LeafJob &J = P.j[blockIdx.x];
    const int n = J.n, ls = n + 1;
    float *S = sm;              // n x (n+1)
    float *u = S + n * ls;      // n
    float *vd = u + n;          // n
    __shared__ int bad;
    const int tid = threadIdx.x, nt = blockDim.x;
    if (tid == 0) bad = -1;
    for (int e = tid; e < n * n; e += nt) {
        const int i = e / n, j = e - i * n;
        S[i * ls + j] = J.X[(long long)i * J.ld + j];
    }
    __syncthreads();
    // Cholesky, upper: S[k][j>=k] <- U[k][j]
    for (int k = 0; k < n; ++k) {
        const float d = S[k * ls + k];
        const bool okp = d > 0.f && isfinite(d);
        if (tid == 0 && !okp && bad < 0) bad = k;
        const float piv = okp ? sqrtf(d) : 1.f;
        const float rp = 1.0f / piv;
        for (int j = k + tid; j < n; j += nt) u[j] = (j == k) ? piv : S[k * ls + j] * rp;
        __syncthreads();
        const int c = n - k - 1;
        for (int e = tid; e < c * c; e += nt) {
            const int i = k + 1 + e / c, j = k + 1 + e % c;
            if (j >= i) S[i * ls + j] -= u[i] * u[j];
        }
        for (int j = k + tid; j < n; j += nt) S[k * ls + j] = u[j];
        __syncthreads();
    }
    // triangular inverse V = U^-1; V[i][j] (i<j) kept at S[j][i], diag in vd
    for (int e = tid; e < n * n; e += nt) {
        const int i = e / n, j = e - i * n;
        if (j < i) S[i * ls + j] = 0.f;
    }
    for (int i = tid; i < n; i += nt) vd[i] = 1.0f / S[i * ls + i];
    __syncthreads();
    for (int k = n - 1; k >= 0; --k) {
        const float r = vd[k];
        for (int j = k + 1 + tid; j < n; j += nt) S[j * ls + k] *= r;
        __syncthreads();
        // R[i][j] -= U[i][k] V[k][j] for i < k <= j
        const int w = n - k;
        for (int e = tid; e < k * w; e += nt) {
            const int j = k + e / k, i = e - (e / k) * k;
            const float vkj = (j == k) ? r : S[j * ls + k];
            S[j * ls + i] -= S[i * ls + k] * vkj;
        }
        __syncthreads();
    }
    // X = V V^T, X[i][j] = sum_{l >= max(i,j)} V[i][l] V[j][l]
    for (int e = tid; e < n * n; e += nt) {
        const int i = e / n, j = e - i * n;
        if (j < i) continue;
        float acc = 0.f;
        for (int l = j; l < n; ++l) {
            const float vil = (l == i) ? vd[i] : S[l * ls + i];
            const float vjl = (l == j) ? vd[j] : S[l * ls + j];
            acc = fmaf(vil, vjl, acc);
        }
        J.X[(long long)i * J.ld + j] = acc;
        J.X[(long long)j * J.ld + i] = acc;
    }
    if (tid == 0 && bad >= 0 && J.info) atomicCAS(J.info, 0, J.o + bad + 1);
}

size_t leaf_smem(int n) { return (size_t)(n * (n + 1) + 2 * n) * sizeof(float); }

// ------------------------------------------------------------- scheduler

struct Op {
    int leaf;
    LeafJob lj;
    SgJob g;
};

int split_of(int n) {
    int h = (n / 2 + 31) / 32 * 32;
    return std::min(h, n - 1);
}

void gen_ops(std::vector<Op> &ops, float *X, long long ld, float *T, long long ldt, int o, int n,
             int *info) {
    if (n <= LEAF) {
        Op op{};
        op.leaf = 1;
        op.lj = LeafJob{X + (long long)o * ld + o, ld, n, o, info};
        ops.push_back(op);
        return;
    }
    const int h = split_of(n), m = n - h;
    gen_ops(ops, X, ld, T, ldt, o, h, info);
    float *X11 = X + (long long)o * ld + o;
    float *X12 = X11 + h;
    float *X21 = X11 + (long long)h * ld;
    float *X22 = X21 + h;
    float *Tn = T + (long long)o * ldt;
    auto gemm = [&](const float *A, long long lda, int ta, const float *B, long long ldb, int tb,
                    float *C, long long ldc, float *Ct, long long ldct, int M, int N, int K,
                    float alpha, float beta) {
        Op op{};
        op.leaf = 0;
        op.g = SgJob{A, lda, ta, B, ldb, tb, C, ldc, Ct, ldct, M, N, K, alpha, beta, 0};
        ops.push_back(op);
    };
    gemm(X11, ld, 0, X12, ld, 0, Tn, ldt, nullptr, 0, h, m, h, 1.f, 0.f);      // T = X11 X12
    gemm(X12, ld, 1, Tn, ldt, 0, X22, ld, nullptr, 0, m, m, h, -1.f, 1.f);     // X22 -= X12^T T
    gen_ops(ops, X, ld, T, ldt, o + h, m, info);                               // X22 <- X22^-1
    gemm(Tn, ldt, 0, X22, ld, 0, X12, ld, X21, ld, h, m, m, -1.f, 0.f);        // X12 = -T X22
    gemm(X12, ld, 0, Tn, ldt, 1, X11, ld, nullptr, 0, h, h, m, -1.f, 1.f);     // X11 -= X12 T^T
}

kfac_status leaf_launch(const std::vector<LeafJob> &jobs, cudaStream_t st) {
    static bool attr_done = false;
    if (!attr_done) {
        if (cudaFuncSetAttribute(leaf_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)leaf_smem(LEAF)) != cudaSuccess)
            return KFAC_ERR_CUDA;
        attr_done = true;
    }
    std::unique_ptr<LeafParams> P(new LeafParams);
    size_t pos = 0;
    while (pos < jobs.size()) {
        int n = 0, nmax = 0;
        while (pos < jobs.size() && n < MAT_MAX) {
            P->j[n] = jobs[pos++];
            nmax = std::max(nmax, P->j[n].n);
            ++n;
        }
        P->n = n;
        leaf_kernel<<<n, LEAF_THREADS, leaf_smem(nmax), st>>>(*P);
        KFAC_LAUNCH_CHECK();
    }
    return KFAC_OK;
}

kfac_status sym_launch(std::vector<SymMat> &mats, int in_place, const float *damp, cudaStream_t st) {
    std::unique_ptr<SymParams> P(new SymParams);
    size_t pos = 0;
    while (pos < mats.size()) {
        int n = 0, tiles = 0;
        while (pos < mats.size() && n < MAT_MAX) {
            SymMat m = mats[pos++];
            m.tiles = (int)ceil_div(m.n, 32);
            P->m[n] = m;
            P->begin[n] = tiles;
            tiles += m.tiles * m.tiles;
            ++n;
        }
        P->begin[n] = tiles;
        P->n = n;
        P->in_place = in_place;
        P->damp = damp;
        sym_kernel<<<tiles, 256, 0, st>>>(*P);
        KFAC_LAUNCH_CHECK();
    }
    return KFAC_OK;
}

}  // namespace

size_t inv_workspace_bytes(const InvMatrix *mats, int nmats) {
    Arena a;
    for (int k = 0; k < nmats; ++k)
        if (mats[k].d > LEAF) a.take<float>((size_t)mats[k].d * mats[k].d);
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
        damping_kernel<<<n, 256, 0, st>>>(*P);
        KFAC_LAUNCH_CHECK();
    }
    return KFAC_OK;
}

kfac_status inv_run(const InvMatrix *mats, int nmats, const float *damp_dev, int *info_dev,
                    Arena &ws, cudaStream_t st) {
    // 1. X = sym(F) + damp I
    std::vector<SymMat> sm(nmats);
    for (int k = 0; k < nmats; ++k)
        sm[k] = SymMat{mats[k].F, mats[k].ldf, mats[k].out, mats[k].ldo, nullptr, 0, mats[k].d, 0, k};
    kfac_status s = sym_launch(sm, 0, damp_dev, st);
    if (s != KFAC_OK) return s;

    // 2. per-matrix op chains
    std::vector<std::vector<Op>> chains(nmats);
    size_t longest = 0;
    for (int k = 0; k < nmats; ++k) {
        float *T = mats[k].d > LEAF ? ws.take<float>((size_t)mats[k].d * mats[k].d) : nullptr;
        gen_ops(chains[k], mats[k].out, mats[k].ldo, T, mats[k].d, 0, mats[k].d,
                info_dev ? info_dev + k : nullptr);
        longest = std::max(longest, chains[k].size());
    }
    if (!ws.fits()) return KFAC_ERR_WORKSPACE;

    // 3. lock-step rounds: all leaves of a round in one launch, all GEMMs in one
    std::vector<LeafJob> leaves;
    std::vector<SgJob> gemms;
    for (size_t r = 0; r < longest; ++r) {
        leaves.clear();
        gemms.clear();
        for (int k = 0; k < nmats; ++k) {
            if (r >= chains[k].size()) continue;
            const Op &op = chains[k][r];
            if (op.leaf) leaves.push_back(op.lj); else gemms.push_back(op.g);
        }
        if (!leaves.empty() && (s = leaf_launch(leaves, st)) != KFAC_OK) return s;
        if (!gemms.empty() && (s = sg_run(gemms.data(), (int)gemms.size(), st)) != KFAC_OK) return s;
    }

    // 4. exact symmetry + bf16 copies
    for (int k = 0; k < nmats; ++k)
        sm[k] = SymMat{mats[k].out, mats[k].ldo, mats[k].out, mats[k].ldo, mats[k].out_bf16,
                       mats[k].ldo_bf16, mats[k].d, 0, -1};
    return sym_launch(sm, 1, damp_dev, st);
}

}  // namespace kfac
