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
#include <cstring>
#include <vector>
#include <memory>

#include "internal.h"

namespace kfac {

namespace {

constexpr int IM_MAX = 64;
constexpr int IM_ROWS = 32;      // patch rows per CTA (4 per warp)
constexpr int IM_TABLE = 2048;   // column units per row held in the CTA's table

struct ImParams {
    Im2colJob j[IM_MAX];
    int begin[IM_MAX + 1];  // prefix of CTAs (IM_ROWS patch rows each)
    int vec[IM_MAX];        // 1: a column unit is 16 bytes of channels, 0: one element
    int n;
};

// One CTA writes IM_ROWS consecutive patch rows of one job.  The columns of a
// row are cut into units (16 bytes of one tap's channels when c allows it,
// else single elements); a shared table gives each unit its tap (r, s) and
// first channel, so that a warp decomposes the output pixel of a row once
// and each lane then copies units with two compares and one address.
template <typename T>
__global__ void __launch_bounds__(256) im2col_kernel(const __grid_constant__ ImParams P) {
    pdl_wait();
    pdl_trigger();
    __shared__ int table[IM_TABLE];  // r | s << 8 | ch << 16 (rows longer than the table: computed per unit)
    int lo = 0, hi = P.n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.begin[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    const Im2colJob &q = P.j[lo];
    const bool vec = P.vec[lo] != 0;
    constexpr int VW = 16 / sizeof(T);  // elements per 16-byte unit
    const int dcore = q.kh * q.kw * q.c;
    const int units = vec ? dcore / VW : dcore;
    const int step = vec ? VW : 1;
    const bool tabled = units <= IM_TABLE;
    auto entry = [&](int e) {
        const int col = e * step, rs = col / q.c, ch = col - rs * q.c;
        const int r = rs / q.kw, sx = rs - r * q.kw;
        return r | (sx << 8) | (ch << 16);
    };
    if (tabled)
        for (int e = threadIdx.x; e < units; e += blockDim.x) table[e] = entry(e);
    __syncthreads();
    const long long M = (long long)q.n * q.ho * q.wo;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const T *x = (const T *)q.x;
#pragma unroll 1
    for (int rr = warp; rr < IM_ROWS; rr += 8) {
        const long long m = (long long)(blockIdx.x - P.begin[lo]) * IM_ROWS + rr;
        if (m >= M) break;
        const long long t = m / q.wo;
        const int wo = (int)(m - t * q.wo);
        const int img = (int)(t / q.ho), ho = (int)(t - (long long)img * q.ho);
        const int hb = ho * q.sh - q.ph, wb = wo * q.sw - q.pw;
        const T *xi = x + (long long)img * q.h * q.w * q.c;
        T *prow = (T *)q.P + m * q.ldp;
        for (int e = lane; e < units; e += 32) {
            const int tv = tabled ? table[e] : entry(e);
            const int hh = hb + (tv & 255), ww = wb + ((tv >> 8) & 255), ch = tv >> 16;
            const bool in = hh >= 0 && hh < q.h && ww >= 0 && ww < q.w;
            const T *src = xi + ((long long)hh * q.w + ww) * q.c + ch;
            if (vec) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (in) v = *reinterpret_cast<const uint4 *>(src);
                *reinterpret_cast<uint4 *>(prow + e * VW) = v;
            } else {
                prow[e] = in ? *src : (T)0.0f;
            }
        }
        if (q.append_one && lane == 0) prow[dcore] = (T)1.0f;
    }
}

// Patch rows of one output row strip (image img, output row ho, every wo) by
// one CTA, for convolutions whose kh input rows of the strip fit in shared
// memory (few channels, e.g. a network's first 7 x 7 layer on RGB input):
// the kh x Wn x c input window (zeros outside the image) is read once,
// coalesced, into shared memory; then consecutive threads write consecutive
// 16-byte pieces of the strip's patch rows, which are contiguous in P, so
// the whole strip goes out as one coalesced block.  A shared table maps each
// column of a patch row to its offset in the window (for output column wo,
// add wo * stride * c).
constexpr int IMS_MAX = 64;
constexpr int IMS_SMEM = 48 * 1024;   // input window + table (bytes)
struct ImsParams {
    Im2colJob j[IMS_MAX];
    int begin[IMS_MAX + 1];   // prefix of CTAs (n * ho strips per job)
    int n;
};

template <typename T>
__global__ void __launch_bounds__(256) im2col_strip_kernel(const __grid_constant__ ImsParams P) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ float4 ims_smem4[];
    int lo = 0, hi = P.n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.begin[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    const Im2colJob &q = P.j[lo];
    constexpr int VW = 16 / sizeof(T);
    const int strip = blockIdx.x - P.begin[lo];
    const int img = strip / q.ho, ho = strip - img * q.ho;
    const int dcore = q.kh * q.kw * q.c;
    const int Wn = (q.wo - 1) * q.sw + q.kw;      // input columns of the window
    int *table = reinterpret_cast<int *>(ims_smem4);           // dcore entries: (r * Wn + s) * c + ch
    T *win = reinterpret_cast<T *>(table + ((dcore + 3) & ~3));  // [kh][Wn][c]
    for (int e = threadIdx.x; e < dcore; e += blockDim.x) {
        const int rs = e / q.c, ch = e - rs * q.c, r = rs / q.kw, sx = rs - r * q.kw;
        table[e] = (r * Wn + sx) * q.c + ch;
    }
    const int hb = ho * q.sh - q.ph, wb = -q.pw;
    const T *xi = (const T *)q.x + (long long)img * q.h * q.w * q.c;
    const int rowlen = Wn * q.c;
    for (int e = threadIdx.x; e < q.kh * rowlen; e += blockDim.x) {
        const int r = e / rowlen, rest = e - r * rowlen;
        const int wc = rest / q.c, ch = rest - wc * q.c;
        const int hh = hb + r, ww = wb + wc;
        win[e] = (hh >= 0 && hh < q.h && ww >= 0 && ww < q.w) ? xi[((long long)hh * q.w + ww) * q.c + ch] : (T)0.0f;
    }
    __syncthreads();
    const int nun = q.ldp / VW;                   // 16-byte pieces of a patch row (padding included)
    T *pstrip = (T *)q.P + (long long)strip * q.wo * q.ldp;
    for (int idx = threadIdx.x; idx < q.wo * nun; idx += blockDim.x) {
        const int wo = idx / nun, u = idx - wo * nun;
        const int wofs = wo * q.sw * q.c;
        T vals[VW];
#pragma unroll
        for (int t = 0; t < VW; ++t) {
            const int e = u * VW + t;
            T v = (T)0.0f;
            if (e < dcore) {
                v = win[table[e] + wofs];
            } else if (e == dcore && q.append_one) {
                v = (T)1.0f;
            }
            vals[t] = v;
        }
        uint4 pk;
        memcpy(&pk, vals, 16);
        *reinterpret_cast<uint4 *>(pstrip + (long long)wo * q.ldp + u * VW) = pk;
    }
}

// Column sums of a 16-bit [M][c] matrix: CTA (chunk, slab) sums 64 columns
// over CS_ROWS rows into partial[slab][column]; the finish kernel adds the
// slabs in order and updates the bias row/column of F.  Both reductions have
// a fixed order, so the results are bitwise reproducible.
constexpr int CS_MAX = 64;
constexpr int CS_ROWS = 256;
struct CsParams {
    ColsumJob j[CS_MAX];
    int begin[CS_MAX + 1];  // prefix of CTAs: chunks x slabs per job
    long long pbase[CS_MAX];  // offset of the job's partials
    int n;
    float *partial;
};

__device__ __forceinline__ float h16_to_f32(uint16_t b, bool f16) {
    return f16 ? __half2float(__ushort_as_half(b)) : bf16_bits_to_f32(b);
}

__device__ __forceinline__ int job_of(const CsParams &P, int b) {
    int lo = 0, hi = P.n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.begin[mid] <= b) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ int slabs_of(const ColsumJob &q) { return (int)((q.M + CS_ROWS - 1) / CS_ROWS); }

__global__ void __launch_bounds__(256) colsum_kernel(const __grid_constant__ CsParams P) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[32][65];
    const int jb = job_of(P, blockIdx.x);
    const ColsumJob &q = P.j[jb];
    const int slabs = slabs_of(q);
    const int t = blockIdx.x - P.begin[jb];
    const int chunk = t / slabs, slab = t - chunk * slabs;
    const int c0 = chunk * 64;
    const int cg = threadIdx.x & 7;   // 8 groups of 8 columns
    const int rg = threadIdx.x >> 3;  // 32 row groups
    float s[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) s[k] = 0.f;
    const int col = c0 + cg * 8;
    const bool f16 = q.f16 != 0;
    const bool vec = (q.c % 8 == 0) && ((uintptr_t)q.x % 16 == 0);
    const long long m1 = min(q.M, (long long)(slab + 1) * CS_ROWS);
    for (long long m = (long long)slab * CS_ROWS + rg; m < m1; m += 32) {
        const uint16_t *row = q.x + m * q.c;
        if (vec && col + 8 <= q.c) {
            uint4 v = *(const uint4 *)(row + col);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                s[2 * k] += h16_to_f32((uint16_t)(w[k] & 0xFFFFu), f16);
                s[2 * k + 1] += h16_to_f32((uint16_t)(w[k] >> 16), f16);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (col + k < q.c) s[k] += h16_to_f32(row[col + k], f16);
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) red[rg][cg * 8 + k] = s[k];
    __syncthreads();
    if (threadIdx.x < 64 && c0 + threadIdx.x < q.c) {
        float a = 0.f;
        for (int r = 0; r < 32; ++r) a += red[r][threadIdx.x];
        P.partial[P.pbase[jb] + (long long)slab * q.c + c0 + threadIdx.x] = a;
    }
}

// F entry (i, c) of the bias column (i <= c), in either layout.
__device__ __forceinline__ float *bias_entry(const ColsumJob &q, int i) {
    const int d = q.c + 1;
    return q.F + (q.packed ? (long long)i * d - (long long)i * (i + 1) / 2 : (long long)i * q.ldf) + q.c;
}

__global__ void __launch_bounds__(256) colsum_finish_kernel(const __grid_constant__ CsParams P) {
    pdl_wait();
    pdl_trigger();
    // one thread per column 0 .. c of the job (column c: the ones column); begin counts CTAs of 256
    const int jb = job_of(P, blockIdx.x);
    const ColsumJob &q = P.j[jb];
    const int i = (blockIdx.x - P.begin[jb]) * 256 + threadIdx.x;
    if (i > q.c) return;
    float *f = bias_entry(q, i);
    float o;
    if (i < q.c) {
        const int slabs = slabs_of(q);
        const float *pp = P.partial + P.pbase[jb] + i;
        float a = 0.f;
        for (int sl = 0; sl < slabs; ++sl) a += pp[(long long)sl * q.c];
        o = q.alpha * a;
    } else {
        o = q.alpha * (float)q.M;  // the ones column with itself: the row count
    }
    if (q.beta != 0.f) o = fmaf(q.beta, *f, o);
    *f = o;
}

}  // namespace

// Strip kernel eligibility: 16-byte aligned rows whose padding absorbs the
// last 16-byte piece, and an input window that fits the shared budget.
size_t strip_smem(const Im2colJob &j, size_t esz) {
    const long long dcore = (long long)j.kh * j.kw * j.c;
    const long long win = (long long)j.kh * ((long long)(j.wo - 1) * j.sw + j.kw) * j.c * (long long)esz;
    return (size_t)(((dcore + 3) & ~3LL) * 4 + win);
}

bool strip_ok(const Im2colJob &j, size_t esz) {
    const int vw = (int)(16 / esz);
    const long long dcore = (long long)j.kh * j.kw * j.c;
    return j.ldp % vw == 0 && (uintptr_t)j.P % 16 == 0 && dcore + (j.append_one ? 1 : 0) <= j.ldp &&
           strip_smem(j, esz) <= (size_t)IMS_SMEM && (long long)j.n * j.ho < (1LL << 30);
}

template <typename T>
kfac_status strip_run(const std::vector<Im2colJob> &jobs, cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(im2col_strip_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, IMS_SMEM) !=
            cudaSuccess)
            return KFAC_ERR_CUDA;
        attr = true;
    }
    std::unique_ptr<ImsParams> P(new ImsParams);
    size_t pos = 0;
    while (pos < jobs.size()) {
        int n = 0;
        long long ctas = 0;
        while (pos < jobs.size() && n < IMS_MAX && ctas + (long long)jobs[pos].n * jobs[pos].ho < (1LL << 30)) {
            P->j[n] = jobs[pos];
            P->begin[n] = (int)ctas;
            ctas += (long long)jobs[pos].n * jobs[pos].ho;
            ++n;
            ++pos;
        }
        if (n == 0) return KFAC_ERR_UNSUPPORTED;
        P->begin[n] = (int)ctas;
        P->n = n;
        size_t smem = 0;  // the launch's largest window + table: more CTAs per SM than the budget
        for (int k = 0; k < n; ++k) smem = std::max(smem, strip_smem(P->j[k], sizeof(T)));
        KFAC_LAUNCH(KK_IM2COL, st, im2col_strip_kernel<T>, (int)ctas, 256, (int)smem, *P);
    }
    return KFAC_OK;
}

kfac_status im2col_run(const Im2colJob *all, int nall, int dtype, cudaStream_t st) {
    const size_t esz0 = dtype == KFAC_F32 ? 4 : 2;
    std::vector<Im2colJob> strips, rows;
    for (int k = 0; k < nall; ++k) (strip_ok(all[k], esz0) ? strips : rows).push_back(all[k]);
    if (!strips.empty()) {
        kfac_status s = dtype == KFAC_BF16  ? strip_run<__nv_bfloat16>(strips, st)
                        : dtype == KFAC_F16 ? strip_run<__half>(strips, st)
                                            : strip_run<float>(strips, st);
        if (s != KFAC_OK) return s;
    }
    const Im2colJob *jobs = rows.data();
    const int njobs = (int)rows.size();
    std::unique_ptr<ImParams> P(new ImParams);
    const size_t esz = dtype == KFAC_F32 ? 4 : 2;
    const int vw = (int)(16 / esz);
    int pos = 0;
    while (pos < njobs) {
        int n = 0;
        long long ctas = 0;
        while (pos < njobs && n < IM_MAX) {
            const Im2colJob &j = jobs[pos];
            const long long M = (long long)j.n * j.ho * j.wo;
            const bool vec = j.c % vw == 0 && j.ldp % vw == 0 && ((uintptr_t)j.x % 16 == 0) &&
                             ((uintptr_t)j.P % 16 == 0);
            if (j.kh > 255 || j.kw > 255 || j.c >= (1 << 15)) return KFAC_ERR_UNSUPPORTED;
            const long long c = ceil_div(M, IM_ROWS);
            if (ctas + c > (1LL << 30)) break;
            P->j[n] = j;
            P->vec[n] = vec ? 1 : 0;
            P->begin[n] = (int)ctas;
            ctas += c;
            ++n;
            ++pos;
        }
        if (n == 0) return KFAC_ERR_UNSUPPORTED;  // one job alone needs more than 2^30 CTAs
        P->begin[n] = (int)ctas;
        P->n = n;
        if (ctas == 0) continue;
        if (dtype == KFAC_BF16)
            KFAC_LAUNCH(KK_IM2COL, st, im2col_kernel<__nv_bfloat16>, (int)ctas, 256, 0, *P);
        else if (dtype == KFAC_F16)
            KFAC_LAUNCH(KK_IM2COL, st, im2col_kernel<__half>, (int)ctas, 256, 0, *P);
        else
            KFAC_LAUNCH(KK_IM2COL, st, im2col_kernel<float>, (int)ctas, 256, 0, *P);
    }
    return KFAC_OK;
}

size_t colsum_partial_floats(const ColsumJob *jobs, int njobs) {
    size_t n = 0;
    for (int k = 0; k < njobs; ++k) n += (size_t)ceil_div(jobs[k].M, CS_ROWS) * jobs[k].c;
    return n;
}

kfac_status colsum_run(const ColsumJob *jobs, int njobs, float *partial, cudaStream_t st) {
    std::unique_ptr<CsParams> P(new CsParams), F(new CsParams);
    int pos = 0;
    long long pb = 0;
    while (pos < njobs) {
        int n = 0, ctas = 0, fin = 0;
        while (pos < njobs && n < CS_MAX) {
            const ColsumJob &j = jobs[pos++];
            if (j.M < 1 || j.M >= (1LL << 31) || j.c < 1) return KFAC_ERR_UNSUPPORTED;
            P->j[n] = F->j[n] = j;
            P->pbase[n] = F->pbase[n] = pb;
            P->begin[n] = ctas;
            F->begin[n] = fin;
            const long long slabs = ceil_div(j.M, CS_ROWS);
            ctas += (int)(ceil_div(j.c, 64) * slabs);
            fin += (int)ceil_div(j.c + 1, 256);
            pb += slabs * j.c;
            ++n;
        }
        P->begin[n] = ctas;
        F->begin[n] = fin;
        P->n = F->n = n;
        P->partial = F->partial = partial;
        KFAC_LAUNCH(KK_COLSUM, st, colsum_kernel, ctas, 256, 0, *P);
        KFAC_LAUNCH(KK_COLSUM, st, colsum_finish_kernel, fin, 256, 0, *F);
    }
    return KFAC_OK;
}

}  // namespace kfac
