// invert.cu -- damped inversion of the Kronecker factors in fp32.
//
// Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
// Kronecker-Factored Approximate Curvature ...", section 3.2, Eq. 6: the
// inverse of G (x) A is G^-1 (x) A^-1, so each factor is inverted on its own.
// Damping (not stated by the paper; the pi-split Tikhonov form of the K-FAC
// method it builds on):
//     pi = sqrt((tr A/dA) / (tr G/dG)),  damp_A = pi sqrt(gamma),  damp_G = sqrt(gamma)/pi.
//
// Algorithm (every matrix of the call advances in batched rounds, one launch
// per round, see schedule_rounds):
//   1. traces -> damping values (one CTA per layer, fixed reduction order);
//   2. X = sym(F) + damp I, padded with an identity block to a multiple of
//      128 (the inverse of diag(X, I) is diag(X^-1, I)), stored as a (hi, lo)
//      pair with hi exactly representable in tf32 and hi + lo = X;
//   3. blocked Cholesky-based inversion by recursive 2x2 blocking on 128-row
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
#include <memory>
#include <mutex>
#include <vector>

#include "internal.h"

namespace kfac {

namespace {

constexpr int LEAF = 128;
constexpr int LEAF_THREADS = 256;
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
    int tiles;        // per side
};

struct TileParams {
    TileMat m[MAT_MAX];
    int begin[MAT_MAX + 1];
    int n;
    const float *damp;
};

// X = split(sym(F) + damp I) on [d, d], identity on the padding.
__global__ void __launch_bounds__(256) prep_kernel(const __grid_constant__ TileParams P) {
    pdl_wait();
    pdl_trigger();
    __shared__ float t[32][33];
    int lo = 0, hi = P.n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.begin[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    const TileMat &q = P.m[lo];
    const int tt = blockIdx.x - P.begin[lo];
    const int ti = tt / q.tiles, tj = tt - ti * q.tiles;
    const int si = min(ti, tj), sj = max(ti, tj);
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int r = ty; r < 32; r += 8) {
        const int i = si * 32 + r, j = sj * 32 + tx;
        t[r][tx] = (i < q.d && j < q.d) ? q.F[(long long)i * q.ldf + j] : 0.f;
    }
    __syncthreads();
    const float dv = P.damp[q.damp_idx];
    for (int r = ty; r < 32; r += 8) {
        const int i = ti * 32 + r, j = tj * 32 + tx;
        float v;
        if (i >= q.d || j >= q.d) {
            v = (i == j) ? 1.f : 0.f;
        } else {
            if (ti < tj) v = t[r][tx];
            else if (ti > tj) v = t[tx][r];
            else v = (r <= tx) ? t[r][tx] : t[tx][r];
            if (i == j) v += dv;
        }
        const float h = tf32_hi(v);
        q.Xh[(long long)i * q.dp + j] = h;
        q.Xl[(long long)i * q.dp + j] = v - h;
    }
}

// out = hi + lo of the upper triangle, mirrored; optional bf16 copy.
__global__ void __launch_bounds__(256) finish_kernel(const __grid_constant__ TileParams P) {
    pdl_wait();
    pdl_trigger();
    __shared__ float t[32][33];
    int lo = 0, hi = P.n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.begin[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    const TileMat &q = P.m[lo];
    const int tt = blockIdx.x - P.begin[lo];
    const int ti = tt / q.tiles, tj = tt - ti * q.tiles;
    const int si = min(ti, tj), sj = max(ti, tj);
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int r = ty; r < 32; r += 8) {
        const int i = si * 32 + r, j = sj * 32 + tx;
        const long long o = (long long)i * q.dp + j;
        t[r][tx] = (i < q.d && j < q.d) ? q.Xh[o] + q.Xl[o] : 0.f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int i = ti * 32 + r, j = tj * 32 + tx;
        if (i >= q.d || j >= q.d) continue;
        float v;
        if (ti < tj) v = t[r][tx];
        else if (ti > tj) v = t[tx][r];
        else v = (r <= tx) ? t[r][tx] : t[tx][r];
        q.out[(long long)i * q.ldo + j] = v;
        if (q.out16) q.out16[(long long)i * q.ld16 + j] = f32_to_bf16_bits(v);
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

// In-place inverse of one SPD 128 x 128 block by one CTA of 256 threads: a
// Gauss-Jordan sweep with the block held in registers (warp w owns rows
// 16w .. 16w+15, lane l columns 4l .. 4l+3).  Pivot k (in order) maps
//   a_ij <- a_ij - a_ik a_kj / a_kk   (i, j != k)
//   a_kj <- a_kj / a_kk,  a_ik <- -a_ik / a_kk,  a_kk <- 1 / a_kk
// and after the last pivot the block holds its inverse.  No pivoting is
// needed: every leading principal block of an SPD matrix is SPD.  The sweep
// keeps the block sign-symmetric -- a_ik = -a_ki when exactly one of i, k has
// been pivoted, a_ik = a_ki otherwise -- so every update of pivot k is formed
// from row k alone.  The row's owner publishes it in shared memory (rowbuf:
// a_kj; colbuf: s_j a_kj / a_kk with s_j = -1 for pivoted j, i.e. the pivot
// column scaled), which costs one barrier per pivot.  A pivot that is not
// positive and finite is recorded in info and eliminated as 1 / a_kk = 0.
__global__ void __launch_bounds__(LEAF_THREADS, 1) leaf_kernel(const __grid_constant__ LeafParams P) {
    pdl_wait();
    pdl_trigger();
    constexpr int N = LEAF, RW = N / (LEAF_THREADS / 32);  // 16 rows per warp
    __shared__ __align__(16) float rowbuf[2][N];
    __shared__ __align__(16) float colbuf[2][N];
    __shared__ float dbuf[2];
    __shared__ int bad;
    const LeafJob &J = P.j[blockIdx.x];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned FULL = 0xffffffffu;

    float a[RW][4];
    {   // 16-byte pieces, every load issued before the first use (the host
        // guarantees 16-byte aligned rows)
        float4 h[RW], l[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            const long long o = (long long)(RW * warp + r) * J.ld + 4 * lane;
            h[r] = *reinterpret_cast<const float4 *>(J.Xh + o);
            l[r] = *reinterpret_cast<const float4 *>(J.Xl + o);
        }
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            a[r][0] = h[r].x + l[r].x;
            a[r][1] = h[r].y + l[r].y;
            a[r][2] = h[r].z + l[r].z;
            a[r][3] = h[r].w + l[r].w;
        }
    }
    if (tid == 0) bad = -1;
    __syncthreads();

    // Row kn (its pivot is element kn % 4 of lane kn / 4) published for the
    // next pivot; called by the owner warp of the row.
    auto publish = [&](int kn, const float (&row)[4], int e) {
        const float pv = __shfl_sync(FULL, row[e], kn >> 2);
        const bool ok = pv > 0.f && isfinite(pv);
        const float d = ok ? __frcp_rn(pv) : 0.f;
        if (!ok && lane == 0 && bad < 0) bad = kn;
        const int buf = kn & 1;
        *reinterpret_cast<float4 *>(&rowbuf[buf][4 * lane]) = make_float4(row[0], row[1], row[2], row[3]);
        float cv[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) cv[t] = (4 * lane + t < kn ? -row[t] : row[t]) * d;
        *reinterpret_cast<float4 *>(&colbuf[buf][4 * lane]) = make_float4(cv[0], cv[1], cv[2], cv[3]);
        if (lane == 0) dbuf[buf] = d;
    };

    if (warp == 0) publish(0, a[0], 0);
    __syncthreads();
#pragma unroll 1
    for (int kb = 0; kb < N / RW; ++kb) {
#pragma unroll
        for (int kk = 0; kk < RW; ++kk) {
            const int k = RW * kb + kk, buf = kk & 1;
            const float4 rc4 = *reinterpret_cast<const float4 *>(&rowbuf[buf][4 * lane]);
            const float rc[4] = {rc4.x, rc4.y, rc4.z, rc4.w};
            float cb[RW];
#pragma unroll
            for (int q = 0; q < RW / 4; ++q) {
                const float4 t = *reinterpret_cast<const float4 *>(&colbuf[buf][RW * warp + 4 * q]);
                cb[4 * q] = t.x; cb[4 * q + 1] = t.y; cb[4 * q + 2] = t.z; cb[4 * q + 3] = t.w;
            }
            // the owner of row k + 1 finishes that row first and publishes it,
            // so that the next pivot's latency overlaps the bulk update
            const int rn = (kk + 1) % RW;
            const bool next_owner = k + 1 < N && warp == (k + 1) / RW;
            if (next_owner) {
#pragma unroll
                for (int c = 0; c < 4; ++c) a[rn][c] = fmaf(-cb[rn], rc[c], a[rn][c]);
                if (lane == (k >> 2)) a[rn][kk & 3] = -cb[rn];
                publish(k + 1, a[rn], (kk + 1) & 3);
            }
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                if (r == rn && next_owner) continue;
#pragma unroll
                for (int c = 0; c < 4; ++c) a[r][c] = fmaf(-cb[r], rc[c], a[r][c]);
                if (lane == (k >> 2)) a[r][kk & 3] = -cb[r];  // column k
            }
            if (warp == kb) {  // row k and the pivot
                const float d = dbuf[buf];
#pragma unroll
                for (int c = 0; c < 4; ++c) a[kk][c] = rc[c] * d;
                if (lane == (k >> 2)) a[kk][kk & 3] = d;
            }
            __syncthreads();
        }
    }

#pragma unroll
    for (int r = 0; r < RW; ++r) {
        const long long o = (long long)(RW * warp + r) * J.ld + 4 * lane;
        const float4 h = make_float4(tf32_hi(a[r][0]), tf32_hi(a[r][1]), tf32_hi(a[r][2]), tf32_hi(a[r][3]));
        *reinterpret_cast<float4 *>(J.Xh + o) = h;
        *reinterpret_cast<float4 *>(J.Xl + o) =
            make_float4(a[r][0] - h.x, a[r][1] - h.y, a[r][2] - h.z, a[r][3] - h.w);
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

// Round schedule: the longest chain sets the sequence of rounds (one launch
// each, leaf or GEMM); every other chain is embedded as late as possible into
// rounds of the same op kind, in order.  The long chain's late rounds are
// small, latency-bound launches with most SMs idle, and the shorter chains'
// work fills them; one launch per round.  Falls back to left-aligned
// lock-step (a leaf and a GEMM launch per round) if a chain does not embed.
std::vector<std::vector<std::pair<int, int>>> schedule_rounds(const std::vector<std::vector<Op>> &chains,
                                                              std::vector<int> &round_kind) {
    int crit = -1;
    for (int k = 0; k < (int)chains.size(); ++k)
        if (crit < 0 || chains[k].size() > chains[crit].size()) crit = k;
    std::vector<std::vector<std::pair<int, int>>> rounds;
    round_kind.clear();
    if (crit < 0) return rounds;
    const int R = (int)chains[crit].size();
    rounds.assign(R, {});
    for (int r = 0; r < R; ++r) round_kind.push_back(chains[crit][r].leaf);
    bool ok = true;
    std::vector<std::vector<int>> slot(chains.size());
    for (int k = 0; k < (int)chains.size() && ok; ++k) {
        const int n = (int)chains[k].size();
        slot[k].assign(n, -1);
        int r = R - 1;
        for (int i = n - 1; i >= 0; --i) {
            while (r >= 0 && round_kind[r] != chains[k][i].leaf) --r;
            if (r < 0) { ok = false; break; }
            slot[k][i] = r--;
        }
    }
    if (ok) {
        for (int k = 0; k < (int)chains.size(); ++k)
            for (int i = 0; i < (int)chains[k].size(); ++i) rounds[slot[k][i]].push_back({k, i});
        return rounds;
    }
    // fallback: left-aligned lock-step, leaves then GEMMs in each step
    size_t longest = 0;
    for (const auto &c : chains) longest = std::max(longest, c.size());
    rounds.clear();
    round_kind.clear();
    for (size_t r = 0; r < longest; ++r)
        for (int kind = 1; kind >= 0; --kind) {
            std::vector<std::pair<int, int>> v;
            for (int k = 0; k < (int)chains.size(); ++k)
                if (r < chains[k].size() && chains[k][r].leaf == kind) v.push_back({k, (int)r});
            if (!v.empty()) {
                rounds.push_back(v);
                round_kind.push_back(kind);
            }
        }
    return rounds;
}

// Workspace layout shared by the size query and the run.
struct InvPlan {
    int *err = nullptr;
    CUtensorMap *dev_maps = nullptr;
    std::vector<CUtensorMap> maps;
    std::vector<MatWork> work;
    std::vector<std::vector<Op>> chains;
    std::vector<std::vector<std::pair<int, int>>> rounds;
    std::vector<int> round_kind;
    size_t longest = 0;
    char *tc_ws = nullptr;
    size_t tc_bytes = 0;
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
    // engine scratch: the largest GEMM round
    p.rounds = schedule_rounds(p.chains, p.round_kind);
    size_t tcb = 0;
    std::vector<TcJob> round;
    for (size_t r = 0; r < p.rounds.size(); ++r) {
        round.clear();
        for (const auto &ki : p.rounds[r])
            if (!p.chains[ki.first][ki.second].leaf) round.push_back(p.chains[ki.first][ki.second].g);
        tcb = std::max(tcb, tc_workspace_bytes(round.data(), (int)round.size(), TC_KIND_TF32X3));
    }
    p.tc_bytes = tcb;
    p.tc_ws = ws.take<char>(tcb);
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
            m.tiles = (int)ceil_div(PREP ? m.dp : m.d, 32);
            P->m[n] = m;
            P->begin[n] = tiles;
            tiles += m.tiles * m.tiles;
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
                        mats[k].out, mats[k].ldo, mats[k].out_bf16, mats[k].ldo_bf16, k, 0};
    if ((s = tile_launch<true>(tm, damp_dev, st)) != KFAC_OK) return s;

    // 2. rounds (see schedule_rounds): each round is one leaf or one GEMM launch
    std::vector<LeafJob> leaves;
    std::vector<TcJob> gemms;
    for (size_t r = 0; r < p.rounds.size(); ++r) {
        leaves.clear();
        gemms.clear();
        for (const auto &ki : p.rounds[r]) {
            const Op &op = p.chains[ki.first][ki.second];
            if (op.leaf) leaves.push_back(op.lj); else gemms.push_back(op.g);
        }
        if (!leaves.empty() && (s = leaf_launch(leaves, st)) != KFAC_OK) return s;
        if (!gemms.empty()) {
            Arena tail(p.tc_ws, p.tc_bytes);
            if ((s = tc_run(gemms.data(), (int)gemms.size(), TC_KIND_TF32X3, p.dev_maps, tail, p.err, st)) !=
                KFAC_OK)
                return s;
        }
    }

    // 3. out = hi + lo, mirrored; bf16 copies
    return tile_launch<false>(tm, damp_dev, st);
}

}  // namespace kfac
