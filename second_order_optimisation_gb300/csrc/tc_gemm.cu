// tc_gemm.cu -- persistent tcgen05 (5th-generation tensor core) GEMM / SYRK
// engine for sm_103a with fp32 accumulation in TMEM.  Two operand kinds:
//
//   KIND_BF16   bf16 operands, one kind::f16 MMA per K=16 slice.  Used for the
//               Kronecker-factor statistic A = P^T P, G = Gam^T Gam (Osawa et
//               al., "Large-Scale Distributed Second-Order Optimization Using
//               Kronecker-Factored Approximate Curvature ...", section 3.2,
//               Eq. 5; both operands the same [rows x d] matrix read MN-major)
//               and for the two GEMMs of G^-1 grad A^-1 (Eq. 7).
//   KIND_TF32X3 fp32 operands carried as (hi, lo) pairs with hi exactly
//               representable in tf32; three kind::tf32 MMAs per K=8 slice
//               (hi*hi + hi*lo + lo*hi) give close to fp32 accuracy.  Used for
//               the Schur-complement updates of the damped inversion (Eq. 6).
//
// One launch runs a list of heterogeneous problems.  Each CTA (one per SM)
// walks a static, strided list of work items (problem, 128x128 output tile,
// K split).  Warp roles:
//   warp 0      TMA producer: 128-byte-swizzled tiles into a shared ring
//   warp 1      TMEM owner + MMA issuer (one thread)
//   warps 2..5  epilogue: tcgen05.ld TMEM -> registers -> global, with a
//               double-buffered accumulator so it overlaps the next tile
// Tensor maps live in the caller's workspace (written by a copy kernel at the
// start of the call); problems refer to them by index and address operand
// sub-blocks by coordinate offsets.  Split-K partial tiles are reduced by the
// last-arriving CTA of the tile in split order (deterministic; no spin-waits).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <mutex>
#include <vector>

#include "internal.h"

namespace kfac {

namespace {

constexpr int BM = 128, BN = 128;
constexpr int TILE_BYTES = 128 * 128;  // one tf32 operand tile: 128 rows x 128 bytes
constexpr int NUM_THREADS = 192;
constexpr int TMEM_ACC = 2 * BN;  // bf16: two accumulators (columns 0 and BN), alternating
constexpr int MAX_PROBS = 152;
constexpr int GROUP = 8;              // row blocks per band of the grouped tile order
#ifndef KFAC_BF16_ITEMS_PER_SM
#define KFAC_BF16_ITEMS_PER_SM 4.0  // bf16 K splits aim at this many work items per SM (tuning constant)
#endif
#ifndef KFAC_ZIGZAG
#define KFAC_ZIGZAG 1  // reverse the CTA order of work items every other round (tuning constant)
#endif
#ifndef KFAC_TF32X3_CHUNK
#define KFAC_TF32X3_CHUNK 8
#endif
#ifndef KFAC_TF32X3_NACC
#define KFAC_TF32X3_NACC 3  // tf32x3 chunk accumulators in TMEM (2 or 3; the running sum follows them)
#endif
#ifndef KFAC_TF32X3_MAX_SPLIT
#define KFAC_TF32X3_MAX_SPLIT 6
#endif
#ifndef KFAC_TF32X3_MIN_KT
#define KFAC_TF32X3_MIN_KT 64.0
#endif
// (both tuning constants may be set at build time)
constexpr int TF32X3_MAX_SPLIT = KFAC_TF32X3_MAX_SPLIT;   // K splits of a tf32x3 tile (the last CTA sums the partials)
// Planning choices for tf32x3 launches, as measured on the ResNet-50 factor
// set: splitting long K ranges before narrowing tiles is faster (7.34 ->
// 7.08 ms; each split keeps 128-wide tiles, which read an A row panel once
// per tile), fewer K tiles per split is slower, the grouped tile order makes
// no difference.
#ifndef KFAC_TF32X3_PREFER_SPLIT
#define KFAC_TF32X3_PREFER_SPLIT true
#endif
constexpr bool TF32X3_PREFER_SPLIT = KFAC_TF32X3_PREFER_SPLIT;  // split long K ranges before narrowing tiles
constexpr double TF32X3_MIN_KT = KFAC_TF32X3_MIN_KT;       // K tiles a tf32x3 split keeps at least
constexpr bool TF32X3_GROUPED = false;       // grouped tile order for tf32x3 launches
#ifndef KFAC_TF32X3_EARLY_RELEASE
#define KFAC_TF32X3_EARLY_RELEASE 1
#endif
// tf32x3 epilogue: move an item's sum into the running-sum columns and
// release its accumulator before the global stores (else after them)
constexpr bool TF32X3_EARLY_RELEASE = KFAC_TF32X3_EARLY_RELEASE;
constexpr int MAPS_PER_COPY = 240;
constexpr int STAGE_LD = 36;                              // epilogue staging row pitch (floats)
constexpr size_t EPI_STAGE_BYTES = 4 * 32 * STAGE_LD * sizeof(float);
constexpr size_t SMEM_BYTES = 192 * 1024 + 1024 /*align*/ + 512 /*barriers*/ + EPI_STAGE_BYTES;
constexpr int RING = 8;  // work items handed from the producer to the other roles (dynamic distribution)
#ifndef KFAC_DYNAMIC_WORK
#define KFAC_DYNAMIC_WORK 1
#endif
// Launches whose jobs ask for it (TcJob::dyn) take their work items from a
// launch-wide counter (longest first) as CTAs become free, instead of a
// static round-robin over CTAs.  Measured: the ResNet-50 factor statistics
// (108 problems of very different sizes) 1.24 -> 1.15 ms; the
// preconditioner (even tiles) and the inversion were no faster (a tuning
// constant).
constexpr bool DYNAMIC_WORK = KFAC_DYNAMIC_WORK;

template <int KIND> struct Traits;
template <> struct Traits<TC_KIND_BF16> {
    // 128 K per stage: every operand box is 64 x 128 elements (16 KB); a
    // streaming SM sustains about twice the bytes with 16 KB TMA boxes as
    // with 8 KB ones (the per-SM rate of box loads is the limit).  One
    // accumulation per work item.
    static constexpr int BK = 128, STAGES = 3, TILES = 2, ESZ = 2, TILE = 128 * 128 * 2;
    static constexpr int CHUNK = 1 << 30, TMEM_COLS = TMEM_ACC, NACC = 2;
};
template <> struct Traits<TC_KIND_TF32X3> {
    // A work item accumulates its K range in chunks of CHUNK K tiles (256 K),
    // rotating over NACC TMEM accumulators (three: the MMA warp can run two
    // chunks ahead of the epilogue while it stores an item); the epilogue
    // warps add each chunk into a running sum held in TMEM (columns NACC BN ..)
    // with fp32 round-to-nearest additions.  Long sums accumulated within one tensor-core
    // accumulator lose accuracy faster than that (the Cholesky updates of the
    // inversion run over K up to the factor's width).
    static constexpr int BK = 32, STAGES = 3, TILES = 4, ESZ = 4, TILE = TILE_BYTES;
    static constexpr int CHUNK = KFAC_TF32X3_CHUNK, TMEM_COLS = 512, NACC = KFAC_TF32X3_NACC;
    static_assert((NACC + 1) * BN <= TMEM_COLS, "accumulators and the running sum fit in TMEM");
};

struct TcProb {
    int map_a, map_b;        // map indices; tf32x3: the (hi, lo) pair map at map + 1 (B of a
                             // narrow tile: hi and lo with 32-row boxes at map + 2, map + 3)
    int a_row0, a_col0;      // operand sub-block origin inside its map (rows, columns)
    int b_row0, b_col0;
    int M, N, k_tiles;
    int bn;                  // output tile width: 128, or 64 / 32 to spread small problems over SMs
    int tiles_n, ksplit, work_begin;
    uint8_t a_mn, b_mn;      // MN-major operand (bf16 only)
    uint8_t syrk, sym, lower, ktri, ktril, grouped, epi;
    uint8_t vec;             // C (and C_lo) rows take 16-byte accesses (ldc % 4 == 0, aligned)
    uint8_t vecb;            // Cb rows take 8-byte accesses
    uint8_t vecw;            // W rows take 16-byte accesses
    uint8_t vect;            // Ct (and Ct_lo) rows take 16-byte accesses
    uint8_t im2col, im_k, im_stride, im_pad;  // operands through an im2col map (see TcJob)
    uint8_t f16, cb_f16;     // fp16 operands / fp16 copy Cb (else bf16)
    uint8_t packed;          // ACCUM: C packed upper triangle of order packed_d
    int packed_d;
    int tiles_m;             // 128-row blocks of the output
    int im_c, im_wo, im_ho, im_howo;
    float alpha, beta;
    float eta;               // STORE: W -= eta * result, in place (fp32, ldw)
    float *C;
    float *C_lo;
    long long ldc;
    float *Ct;
    float *Ct_lo;
    long long ldct;
    uint16_t *Cb;
    long long ldcb;
    float *W;
    long long ldw;
    float *partial;  // [tiles][ksplit][BM*BN] when ksplit > 1
    int *counters;   // [tiles]
};

struct TcParams {
    const CUtensorMap *maps;  // device (workspace)
    TcProb prob[MAX_PROBS];
    int nprob;
    int total_work;
    int *counter;             // dynamic distribution: the next work item (zeroed before the launch)
    int *error;
};
static_assert(sizeof(TcParams) <= 32000, "kernel parameter block too large");

struct MapCopyParams {
    CUtensorMap m[MAPS_PER_COPY];
    CUtensorMap *dst;
    int n;
};

__global__ void map_copy_kernel(const __grid_constant__ MapCopyParams P) {
    pdl_wait();
    pdl_trigger();
    // 8 threads per 128-byte map, 16 bytes each
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const int m = t >> 3, part = t & 7;
    if (m < P.n) {
        const uint4 *src = reinterpret_cast<const uint4 *>(&P.m[m]) + part;
        uint4 *dst = reinterpret_cast<uint4 *>(P.dst + m) + part;
        *dst = *src;
    }
    // make the generic-proxy writes visible to later tensor-map (async proxy) reads
    asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
}

struct Work {
    int p, tile, tm, tn, split, kt0, kt1;
};

// Work item w of the launch: (problem, output tile, K split).
__device__ __forceinline__ Work decode_work(const TcParams &P, int w) {
    int lo = 0, hi = P.nprob - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.prob[mid].work_begin <= w) lo = mid; else hi = mid - 1;
    }
    const TcProb &q = P.prob[lo];
    Work k;
    k.p = lo;
    const int local = w - q.work_begin;
    const int unit = local / q.ksplit;  // output tile
    k.split = local - unit * q.ksplit;
    const int T = q.tiles_n;
    if ((q.syrk || q.sym) && q.grouped) {
        // upper tiles in bands of GROUP row blocks; inside a band column by
        // column, rows innermost, so that the CTAs running at the same time
        // share their A row panels and B column panels in L2.  first(tm) =
        // tm * r with r = 128 / bn; row block tm holds T - first(tm) tiles.
        const int r = BM / q.bn;
        int u = unit, b0 = 0;
        for (;;) {
            const int gb = min(GROUP, q.tiles_m - b0);
            const int size = gb * T - r * (gb * b0 + gb * (gb - 1) / 2);
            if (u < size) break;
            u -= size;
            b0 += gb;
        }
        const int gb = min(GROUP, q.tiles_m - b0);
        const int stair = r * gb * (gb + 1) / 2;  // columns r*b0 .. r*(b0+gb)-1 hold 1 .. gb rows
        if (u < stair) {
            int tn = r * b0;
            for (;;) {
                const int cnt = tn / r - b0 + 1;
                if (u < cnt) { k.tm = b0 + u; k.tn = tn; break; }
                u -= cnt;
                ++tn;
            }
        } else {
            u -= stair;
            k.tn = r * (b0 + gb) + u / gb;
            k.tm = b0 + u % gb;
        }
        k.tile = k.tm * T - r * (k.tm * (k.tm - 1) / 2) + (k.tn - k.tm * r);
    } else if (q.sym && q.ktri) {
        // upper tiles column by column (column block tn holds row blocks
        // 0 .. the one holding its last column): K starts at the tile's first
        // column, so this order is longest first and the static round-robin
        // over CTAs balances
        int u = unit, tn = 0, base = 0;
        for (;;) {
            const int cnt = min(q.tiles_m, ((tn + 1) * q.bn - 1) / BM + 1);
            if (u < cnt) {
                k.tm = u;
                k.tn = tn;
                k.tile = base + u;
                break;
            }
            u -= cnt;
            base += cnt;
            ++tn;
        }
    } else if (q.syrk || q.sym) {
        // upper tiles only: row block tm (128 rows) runs column blocks from the
        // one holding its diagonal, first(tm) = tm * 128 / bn
        int u = unit, tm = 0, base = 0;
        for (;;) {
            const int first = tm * BM / q.bn, cnt = T - first;
            if (u < cnt) {
                k.tm = tm;
                k.tn = first + u;
                k.tile = base + u;
                break;
            }
            u -= cnt;
            base += cnt;
            ++tm;
        }
    } else if (q.lower) {
        // tiles touching the lower triangle: row block tm runs column blocks
        // 0 .. (tm + 1) * 128 / bn - 1
        int u = unit, tm = 0, base = 0;
        for (;;) {
            const int cnt = min(T, (tm + 1) * BM / q.bn);
            if (u < cnt) {
                k.tm = tm;
                k.tn = u;
                k.tile = base + u;
                break;
            }
            u -= cnt;
            base += cnt;
            ++tm;
        }
    } else if (q.grouped) {
        // bands of GROUP row blocks, column by column, rows innermost
        const int band = unit / (GROUP * T);
        const int b0 = band * GROUP, gb = min(GROUP, q.tiles_m - b0);
        const int rem = unit - band * GROUP * T;
        k.tn = rem / gb;
        k.tm = b0 + rem % gb;
        k.tile = k.tm * T + k.tn;
    } else if (q.ktri) {
        // column by column: K starts at the tile's first column, longest first
        k.tn = unit / q.tiles_m;
        k.tm = unit - k.tn * q.tiles_m;
        k.tile = k.tm * T + k.tn;
    } else if (q.ktril) {
        // row blocks from the last: K ends after the tile's last row, longest first
        const int r = unit / T;
        k.tm = q.tiles_m - 1 - r;
        k.tn = unit - r * T;
        k.tile = k.tm * T + k.tn;
    } else {
        k.tm = unit / T;
        k.tn = unit - k.tm * T;
        k.tile = unit;
    }
    // ktri (tf32x3 only, K tiles of 32): K starts at the tile's first column
    // (an upper tile of the product of an upper-triangular matrix with its
    // transpose)
    // ktril (tf32x3): K ends after the tile's last row (A lower triangular
    // in its K index: A[i][t] = 0 for t > i)
    const int kb = q.ktri ? k.tn * q.bn / Traits<TC_KIND_TF32X3>::BK : 0;
    const int ke = q.ktril ? min(q.k_tiles, (k.tm + 1) * BM / Traits<TC_KIND_TF32X3>::BK) : q.k_tiles;
    k.kt0 = kb + (int)((long long)k.split * (ke - kb) / q.ksplit);
    k.kt1 = kb + (int)((long long)(k.split + 1) * (ke - kb) / q.ksplit);
    return k;
}

__device__ __forceinline__ int ceil_div_dev(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ void acquire_map(const CUtensorMap *m) {
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"((uint64_t)m) : "memory");
}

// tf32 operand rows [mn0, mn0 + rows) x K [k0, k0 + 32) as 32-row boxes
// (128-byte rows; 32 rows keep the 8-row swizzle atoms of one tall box).
__device__ __forceinline__ void load_rows_tf32(uint8_t *dst, const CUtensorMap *map, int row0, int col0, int mn0,
                                               int rows, int k0, uint64_t *bar) {
    for (int r = 0; r < rows; r += 32) tma_load_2d(dst + r * 128, map, col0 + k0, row0 + mn0 + r, bar);
}

__device__ __forceinline__ void tma_load_im2col_4d(void *dst, const CUtensorMap *map, int c, int w, int h, int n,
                                                   uint16_t off_w, uint16_t off_h, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.im2col.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], {%7, %8};" ::"r"(smem_u32(dst)),
        "l"((uint64_t)map), "r"(c), "r"(w), "r"(h), "r"(n), "r"(smem_u32(bar)), "h"(off_w), "h"(off_h)
        : "memory");
}

// Producer state for a convolution's patch-matrix operands read through the
// im2col map.  A 128-wide MN (= d) block is two 64-wide halves, each one
// filter tap (r, s) and 64 channels; a K tile is 128 consecutive output pixels
// (rows past the end of the batch fall outside the tensor and read 0).  The
// taps are decomposed once per work item and the pixel position advances by
// 128 per K tile without divisions, so the single producer thread keeps up
// with the MMAs.
struct Im2colCursor {
    int c0[4], sx[4], r[4];  // A halves 0, 1; B halves 0, 1
    int img, ho, wo;         // first output pixel of the next K tile
};

__device__ __forceinline__ void im2col_taps(const TcProb &q, int mn0, int *c0, int *sx, int *r) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        // a half past the last tap only feeds outputs that are never stored:
        // load a valid one instead
        const int d0 = min(mn0 + 64 * half, q.M - 64);
        const int rs = d0 / q.im_c;
        c0[half] = d0 - rs * q.im_c;
        r[half] = rs / q.im_k;
        sx[half] = rs - r[half] * q.im_k;
    }
}

__device__ __forceinline__ void im2col_start(const TcProb &q, const Work &k, Im2colCursor &cur) {
    im2col_taps(q, k.tm * BM, cur.c0, cur.sx, cur.r);
    im2col_taps(q, k.tn * BN, cur.c0 + 2, cur.sx + 2, cur.r + 2);
    const int m0 = k.kt0 * 128;
    cur.img = m0 / q.im_howo;
    const int rem = m0 - cur.img * q.im_howo;
    cur.ho = rem / q.im_wo;
    cur.wo = rem - cur.ho * q.im_wo;
}

__device__ __forceinline__ void im2col_load(uint8_t *dst, const CUtensorMap *map, const TcProb &q,
                                            const Im2colCursor &cur, int which, uint64_t *bar) {
    const int w = cur.wo * q.im_stride - q.im_pad, h = cur.ho * q.im_stride - q.im_pad;
#pragma unroll
    for (int half = 0; half < 2; ++half)
        tma_load_im2col_4d(dst + 16384 * half, map, cur.c0[2 * which + half], w, h, cur.img,
                           (uint16_t)cur.sx[2 * which + half], (uint16_t)cur.r[2 * which + half], bar);
}

__device__ __forceinline__ void im2col_advance(const TcProb &q, Im2colCursor &cur) {
    cur.wo += 128;
    while (cur.wo >= q.im_wo) {
        cur.wo -= q.im_wo;
        if (++cur.ho == q.im_ho) {
            cur.ho = 0;
            ++cur.img;
        }
    }
}

// One 128 (M or N) x BK (K) operand tile into shared memory.
//   tf32, K-major source [MN][K]: one 32 x 128 box (128-byte rows).
//   bf16, K-major source [MN][K]: two 64 x 128 boxes (K 0-63 | 64-127), 16 KB apart.
//   bf16, MN-major source [K][MN]: two 64 x 128 boxes (MN 0-63 | 64-127), 16 KB apart.
__device__ __forceinline__ void load_tile(uint8_t *dst, const CUtensorMap *map, int mn_major, int row0,
                                          int col0, int mn0, int k0, uint64_t *bar) {
    tma_load_2d(dst, map, col0 + k0, row0 + mn0, bar);
}
__device__ __forceinline__ void load_tile_bf16(uint8_t *dst, const CUtensorMap *map, int mn_major, int row0,
                                               int col0, int mn0, int k0, uint64_t *bar) {
    if (mn_major) {
        tma_load_2d(dst, map, col0 + mn0, row0 + k0, bar);
        tma_load_2d(dst + 16384, map, col0 + mn0 + 64, row0 + k0, bar);
    } else {
        tma_load_2d(dst, map, col0 + k0, row0 + mn0, bar);
        tma_load_2d(dst + 16384, map, col0 + k0 + 64, row0 + mn0, bar);
    }
}

// Descriptors of the kk-th 32-byte K slice of a staged operand tile.
// tf32 (K-major): 128-byte rows, 8-row groups 1024 B apart (SBO); a slice is
//   32 B (8 tf32) inside the swizzled row.
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int mn_major, int kk) {
    return smem_desc_sw128(base + kk * 32, 16, 1024);
}
// bf16 (16 elements per slice, 8 slices per 128-K stage):
//   MN-major: 8-row K groups 1024 B apart (SBO), the two 64-wide MN blocks
//     16 KB apart (LBO); a slice spans two K groups.
//   K-major: slices 0-3 in the first 64-K box, 4-7 in the second (16 KB on).
__device__ __forceinline__ uint64_t operand_desc_bf16(uint32_t base, int mn_major, int kk) {
    return mn_major ? smem_desc_sw128(base + kk * 2048, 16384, 1024)
                    : smem_desc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}

__device__ __forceinline__ float tf32_hi(float v) {
    return __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
}

// Epilogue data layout.  A warp owns 32 accumulator rows (its TMEM lane
// quarter) and handles them in 32 x 32 chunks.  tcgen05.ld gives lane l row
// i0 + l; the chunk is restaged through shared memory so that lane l then
// holds row i0 + 4k + l/8, columns j0 + 4(l%8) .. +3 for k = 0..7: every
// global access is 16 bytes and a warp instruction covers four 128-byte rows.
// Old values of C (beta != 0) use the same layout, so they can be fetched
// before the accumulator is ready.
__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ float4 tf32_hi4(float4 v) {
    return make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z), tf32_hi(v.w));
}
__device__ __forceinline__ float4 sub4(float4 a, float4 b) {
    return make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w);
}
__device__ __forceinline__ float comp(float4 v, int t) { return t == 0 ? v.x : t == 1 ? v.y : t == 2 ? v.z : v.w; }

// The ragged-edge fallbacks of the epilogue's stores, out of line: the
// epilogue's unrolled row-group loops stay small enough for the instruction
// cache (inlined, each row group carried a scalar copy of its stores, and the
// loop's code, not its stores, set the time of a 32 x 32 chunk: ~3 us).
__device__ __noinline__ void store_pair_edge(float *C, float *C_lo, long long off, int n, float4 h, float4 l) {
    for (int t = 0; t < 4 && t < n; ++t) {
        C[off + t] = comp(h, t);
        C_lo[off + t] = comp(l, t);
    }
}
// components t0 <= t < n (of 4) of o into dst[t]
__device__ __noinline__ void store4_edge(float *dst, int t0, int n, float4 o) {
    for (int t = max(t0, 0); t < 4 && t < n; ++t) dst[t] = comp(o, t);
}
__device__ __noinline__ void store4b_edge(uint16_t *dst, int t0, int n, float4 o, bool h16) {
    for (int t = max(t0, 0); t < 4 && t < n; ++t) dst[t] = f32_to_16_bits(comp(o, t), h16);
}
// dw[t] -= eta o[t] for t < n; true when a result is NaN or infinite
__device__ __noinline__ bool step4_edge(float *dw, int n, float ne, float4 o) {
    bool bad = false;
    for (int t = 0; t < 4 && t < n; ++t) {
        const float nw = fmaf(ne, comp(o, t), dw[t]);
        bad |= !(fabsf(nw) <= 3.402823466e38f);
        dw[t] = nw;
    }
    return bad;
}
// src[t] for t0 <= t < n (of 4), zeros elsewhere
__device__ __noinline__ float4 load4_edge(const float *src, int t0, int n) {
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    for (int t = max(t0, 0); t < 4 && t < n; ++t) v[t] = src[t];
    return make_float4(v[0], v[1], v[2], v[3]);
}

// Offset of C's entry (i, 0): row-major with ldc, or the packed upper
// triangle (row i's entries j >= i start at i*d - i*(i+1)/2 + i).
__device__ __forceinline__ long long c_row(const TcProb &q, int i) {
    return q.packed ? (long long)i * q.packed_d - (long long)i * (i + 1) / 2 : (long long)i * q.ldc;
}

// Old values of the chunk at (i0, j0) (zeros where beta == 0 or out of range).
__device__ __forceinline__ void load_old(const TcProb &q, int i0, int j0, int lane, float4 (&oh)[8],
                                         float4 (&ol)[8]) {
    const int j = j0 + 4 * (lane & 7);
    const bool need = q.beta != 0.f && q.epi != TC_EPI_STORE;
    const bool lo = q.epi == TC_EPI_SPLIT;
    const bool full = q.vec && j + 3 < q.N;
    if (need && q.vec && !q.packed && i0 + 32 <= q.M && j0 + 32 <= q.N) {
        // an interior chunk: a loop with no edge code
        const long long off = (long long)(i0 + (lane >> 3)) * q.ldc + j, step = 4 * q.ldc;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            oh[k] = ld4(q.C + off + k * step);
            ol[k] = lo ? ld4(q.C_lo + off + k * step) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int i = i0 + 4 * k + (lane >> 3);
        float4 h = make_float4(0.f, 0.f, 0.f, 0.f), l = h;
        if (need && i < q.M) {
            const long long off = c_row(q, i) + j;
            if (full && (!q.packed || (off & 3) == 0)) {
                h = ld4(q.C + off);
                if (lo) l = ld4(q.C_lo + off);
            } else {
                const int t0 = q.packed ? i - j : 0;
                h = load4_edge(q.C + off, t0, q.N - j);
                if (lo) l = load4_edge(q.C_lo + off, t0, q.N - j);
            }
        }
        oh[k] = h;
        ol[k] = l;
    }
}

// Epilogue of one 32 x 32 chunk by one warp: v is the TMEM layout (lane =
// row), oh / ol the old values from load_old.  The transposed copy Ct (if any)
// is written straight from v (consecutive lanes are consecutive addresses of
// Ct); the mirror of a symmetric off-diagonal tile goes back through the stage.
// Returns true when a value this lane wrote is NaN or infinite.
__device__ __forceinline__ bool chunk_store(const TcProb &q, int i0, int j0, const float *v, float *stage,
                                            int lane, bool mirror, bool diagblk, float4 (&oh)[8], float4 (&ol)[8]) {
    const float a = q.alpha, b = q.beta;
    bool bad = false;
    // transposed stores of a whole chunk: the chunk goes through the stage
    // column by column (stage row c = output row j0 + c), so that lane l then
    // holds 4 consecutive outputs of row j0 + 4k + l/8 and every store is
    // 16 bytes (8 B for 16-bit outputs) in rows of 128 consecutive bytes
    const bool whole = i0 + 32 <= q.M && j0 + 32 <= q.N;
    const int tr = lane >> 3, tc = 4 * (lane & 7);
    if (q.epi == TC_EPI_SPLIT && q.Ct && whole && q.vect) {  // host guarantees beta == 0 here
#pragma unroll
        for (int c = 0; c < 32; ++c) stage[c * STAGE_LD + lane] = a * v[c];
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int r = 4 * k + tr;
            const float4 o = *reinterpret_cast<const float4 *>(&stage[r * STAGE_LD + tc]);
            const float4 h = tf32_hi4(o);
            const long long off = (long long)(j0 + r) * q.ldct + i0 + tc;
            st4(q.Ct + off, h);
            st4(q.Ct_lo + off, sub4(o, h));
        }
        __syncwarp();
    } else if (q.epi == TC_EPI_SPLIT && q.Ct) {
        const int i = i0 + lane;
        if (i < q.M) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const int j = j0 + c;
                if (j < q.N) {
                    const float o = a * v[c], h = tf32_hi(o);
                    q.Ct[(long long)j * q.ldct + i] = h;
                    q.Ct_lo[(long long)j * q.ldct + i] = o - h;
                }
            }
        }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4 *>(&stage[lane * STAGE_LD + 4 * c]) =
            make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    __syncwarp();
    float4 acc[8];
    const int sl = (lane >> 3) * STAGE_LD + 4 * (lane & 7);
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = *reinterpret_cast<const float4 *>(&stage[4 * k * STAGE_LD + sl]);
    __syncwarp();
    const int j = j0 + 4 * (lane & 7);
    const bool full = q.vec && j + 3 < q.N;
    if (q.epi == TC_EPI_ACCUM && whole && q.vec && !q.packed && (!q.syrk || j0 >= i0 + 32)) {
        // an interior chunk (entirely above the diagonal of a SYRK): no edge code in the loop
        float *dst = q.C + (long long)(i0 + (lane >> 3)) * q.ldc + j;
        const long long step = 4 * q.ldc;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 o = make_float4(fmaf(b, oh[k].x, a * acc[k].x), fmaf(b, oh[k].y, a * acc[k].y),
                                         fmaf(b, oh[k].z, a * acc[k].z), fmaf(b, oh[k].w, a * acc[k].w));
            bad |= !finite4(o);
            st4(dst + k * step, o);
        }
    } else if (q.epi == TC_EPI_ACCUM) {
        const bool upper = q.syrk;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = i0 + 4 * k + (lane >> 3);
            if (i >= q.M) continue;
            const float4 o = make_float4(fmaf(b, oh[k].x, a * acc[k].x), fmaf(b, oh[k].y, a * acc[k].y),
                                         fmaf(b, oh[k].z, a * acc[k].z), fmaf(b, oh[k].w, a * acc[k].w));
            bad |= j < q.N && !finite4(o);  // (past the last column the values are zero padding)
            float *dst = q.C + c_row(q, i) + j;
            if (full && (!upper || j >= i) && (!q.packed || ((uintptr_t)dst & 15) == 0)) {
                st4(dst, o);
            } else {
                store4_edge(dst, upper ? i - j : 0, q.N - j, o);
            }
        }
    } else if (q.epi == TC_EPI_STORE) {
        // a tile in a diagonal 128-block of a symmetric output (diagblk)
        // stores its upper part only and mirrors that, so the result is
        // exactly symmetric
        const bool up = diagblk;
        const bool fullb = q.vecb && j + 3 < q.N;
        if (whole && !up && !q.W && q.C && q.vec && (!q.Cb || q.vecb)) {
            // an interior chunk off the diagonal blocks: no edge code in the loop
            float *dst = q.C + (long long)(i0 + (lane >> 3)) * q.ldc + j;
            uint16_t *dstb = q.Cb ? q.Cb + (long long)(i0 + (lane >> 3)) * q.ldcb + j : nullptr;
            const long long step = 4 * q.ldc, stepb = 4 * q.ldcb;
            const bool h16 = q.cb_f16;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 o = make_float4(a * acc[k].x, a * acc[k].y, a * acc[k].z, a * acc[k].w);
                bad |= !finite4(o);
                st4(dst + k * step, o);
                if (dstb) {
                    const uint32_t lo2 = f32_to_16_bits(o.x, h16) | ((uint32_t)f32_to_16_bits(o.y, h16) << 16);
                    const uint32_t hi2 = f32_to_16_bits(o.z, h16) | ((uint32_t)f32_to_16_bits(o.w, h16) << 16);
                    *reinterpret_cast<uint2 *>(dstb + k * stepb) = make_uint2(lo2, hi2);
                }
            }
        } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = i0 + 4 * k + (lane >> 3);
            if (i >= q.M) continue;
            const float4 o = make_float4(a * acc[k].x, a * acc[k].y, a * acc[k].z, a * acc[k].w);
            bad |= j < q.N && !finite4(o);
            if (q.C) {
                float *dst = q.C + (long long)i * q.ldc + j;
                if (full && (!up || j >= i)) {
                    st4(dst, o);
                } else {
                    store4_edge(dst, up ? i - j : 0, q.N - j, o);
                }
            }
            if (q.W) {  // the step on the weights (never a symmetric output)
                float *dw = q.W + (long long)i * q.ldw + j;
                const float ne = -q.eta;
                if (q.vecw && j + 3 < q.N) {
                    float4 w4 = ld4(dw);
                    w4.x = fmaf(ne, o.x, w4.x); w4.y = fmaf(ne, o.y, w4.y);
                    w4.z = fmaf(ne, o.z, w4.z); w4.w = fmaf(ne, o.w, w4.w);
                    bad |= !finite4(w4);
                    st4(dw, w4);
                } else {
                    bad |= step4_edge(dw, q.N - j, ne, o);
                }
            }
            if (q.Cb) {
                uint16_t *dst = q.Cb + (long long)i * q.ldcb + j;
                if (fullb && (!up || j >= i)) {
                    const bool h16 = q.cb_f16;
                    const uint32_t lo2 = f32_to_16_bits(o.x, h16) | ((uint32_t)f32_to_16_bits(o.y, h16) << 16);
                    const uint32_t hi2 = f32_to_16_bits(o.z, h16) | ((uint32_t)f32_to_16_bits(o.w, h16) << 16);
                    *reinterpret_cast<uint2 *>(dst) = make_uint2(lo2, hi2);
                } else {
                    store4b_edge(dst, up ? i - j : 0, q.N - j, o, q.cb_f16);
                }
            }
        }
        }
        // a chunk of a diagonal block entirely above its diagonal mirrors
        // whole, one entirely below mirrors nothing, one on it goes entry by
        // entry (only j > i)
        const bool above = mirror || (up && j0 >= i0 + 32);
        if (above && whole && (!q.C || q.vec) && (!q.Cb || q.vecb)) {
#pragma unroll
            for (int c = 0; c < 32; ++c) stage[c * STAGE_LD + lane] = a * v[c];
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int r = 4 * k + tr;
                const float4 o = *reinterpret_cast<const float4 *>(&stage[r * STAGE_LD + tc]);
                if (q.C) st4(q.C + (long long)(j0 + r) * q.ldc + i0 + tc, o);
                if (q.Cb) {
                    const bool h16 = q.cb_f16;
                    const uint32_t lo2 = f32_to_16_bits(o.x, h16) | ((uint32_t)f32_to_16_bits(o.y, h16) << 16);
                    const uint32_t hi2 = f32_to_16_bits(o.z, h16) | ((uint32_t)f32_to_16_bits(o.w, h16) << 16);
                    *reinterpret_cast<uint2 *>(q.Cb + (long long)(j0 + r) * q.ldcb + i0 + tc) = make_uint2(lo2, hi2);
                }
            }
            __syncwarp();
        } else if ((mirror || up) && !(up && j0 + 32 <= i0)) {
            // symmetric output: the transposed position C[j][i0 .. i0+31],
            // straight from the TMEM layout (lane = row i0 + lane), so every
            // store instruction covers one contiguous row segment
            const int i = i0 + lane;
            if (i < q.M) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {  // (fully unrolled: v stays in registers)
                    const int jj = j0 + c;
                    if (jj >= q.N || (up && jj <= i)) continue;
                    const float o = a * v[c];
                    if (q.C) q.C[(long long)jj * q.ldc + i] = o;
                    if (q.Cb) q.Cb[(long long)jj * q.ldcb + i] = f32_to_16_bits(o, q.cb_f16);
                }
            }
        }
    } else if (whole && q.vec && q.C && !mirror) {  // TC_EPI_SPLIT, an interior chunk: no edge code
        const float *C0 = q.C;
        float *Ch = q.C + (long long)(i0 + (lane >> 3)) * q.ldc + j, *Cl = q.C_lo + (Ch - C0);
        const long long step = 4 * q.ldc;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 o = make_float4(fmaf(b, oh[k].x + ol[k].x, a * acc[k].x),
                                         fmaf(b, oh[k].y + ol[k].y, a * acc[k].y),
                                         fmaf(b, oh[k].z + ol[k].z, a * acc[k].z),
                                         fmaf(b, oh[k].w + ol[k].w, a * acc[k].w));
            bad |= !finite4(o);
            const float4 h = tf32_hi4(o), l = sub4(o, h);
            oh[k] = h;
            ol[k] = l;
            st4(Ch + k * step, h);
            st4(Cl + k * step, l);
        }
    } else {  // TC_EPI_SPLIT
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = i0 + 4 * k + (lane >> 3);
            const float4 o = make_float4(fmaf(b, oh[k].x + ol[k].x, a * acc[k].x),
                                         fmaf(b, oh[k].y + ol[k].y, a * acc[k].y),
                                         fmaf(b, oh[k].z + ol[k].z, a * acc[k].z),
                                         fmaf(b, oh[k].w + ol[k].w, a * acc[k].w));
            bad |= i < q.M && j < q.N && !finite4(o);
            const float4 h = tf32_hi4(o), l = sub4(o, h);
            oh[k] = h;  // the final pair, kept for the mirror below
            ol[k] = l;
            if (i >= q.M || !q.C) continue;  // (no C: only the transposed copy Ct)
            const long long off = (long long)i * q.ldc + j;
            if (full) {
                st4(q.C + off, h);
                st4(q.C_lo + off, l);
            } else {
                store_pair_edge(q.C, q.C_lo, off, q.N - j, h, l);
            }
        }
        if (mirror) {
            // symmetric output: this upper tile also fills its transposed
            // position; lane = row i0 + lane again, so that every store covers
            // 32 consecutive columns of C[j][i0 .. i0+31]
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                float *dst = part ? q.C_lo : q.C;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    *reinterpret_cast<float4 *>(&stage[4 * k * STAGE_LD + sl]) = part ? ol[k] : oh[k];
                __syncwarp();
                const int i = i0 + lane;
#pragma unroll 8
                for (int c = 0; c < 32; ++c) {
                    const int jj = j0 + c;
                    if (i < q.M && jj < q.N) dst[(long long)jj * q.ldc + i] = stage[lane * STAGE_LD + c];
                }
                __syncwarp();
            }
        }
    }
    return bad;
}

template <int KIND>
__global__ void __launch_bounds__(NUM_THREADS, 1) tc_gemm_kernel(const __grid_constant__ TcParams P) {
    using Tr = Traits<KIND>;
    constexpr int STAGE_BYTES = Tr::TILES * Tr::TILE;
    constexpr int KSLICES = Tr::BK * Tr::ESZ / 32;  // 32-byte MMA K slices per stage (4)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *full = (uint64_t *)(smem + Tr::STAGES * STAGE_BYTES);
    uint64_t *empty = full + Tr::STAGES;
    uint64_t *accf = empty + Tr::STAGES;
    uint64_t *acce = accf + Tr::NACC;
    uint64_t *drain = acce + Tr::NACC;  // completion of this CTA's products after an abort
    uint64_t *item_full = drain + 1;        // [RING] an item index is in the ring slot
    uint64_t *item_empty = item_full + RING;  // [RING] the MMA thread and the epilogue have read it
    volatile int *ring = (volatile int *)(item_empty + RING);
    uint32_t *tmem_slot = (uint32_t *)(ring + RING);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    volatile int *last_flag = abort_flag + 1;
    float *epi_stage = (float *)(smem + Tr::STAGES * STAGE_BYTES + 512);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int w_first = blockIdx.x, w_step = gridDim.x;
    // work item of round r: items are sorted longest first, and the CTA order
    // reverses every other round (a CTA that took a long item takes a short
    // one next), which evens out the CTAs' totals
    auto widx = [&](int r) { return r * w_step + ((KFAC_ZIGZAG && (r & 1)) ? w_step - 1 - w_first : w_first); };
    // dynamic distribution: the producer publishes item r of this CTA in ring
    // slot r % RING (-1: none left); the other roles read it in the same order
    const bool dyn = DYNAMIC_WORK && P.counter != nullptr;
    auto publish = [&](int r) -> int {
        if (!dyn) {
            const int w = widx(r);
            return w < P.total_work ? w : -1;
        }
        const int sl = r % RING;
        if (r >= RING && !mbar_wait(&item_empty[sl], ((r / RING) - 1) & 1)) {
            atomicOr(P.error, ERR_TIMEOUT_EMPTY);
            *abort_flag = 1;
        }
        int w = *abort_flag ? P.total_work : atomicAdd(P.counter, 1);
        if (w >= P.total_work) w = -1;
        ring[sl] = w;
        mbar_arrive(&item_full[sl]);
        return w;
    };
    auto take = [&](int r) -> int {
        if (!dyn) {
            const int w = widx(r);
            return w < P.total_work ? w : -1;
        }
        const int sl = r % RING;
        if (!mbar_wait(&item_full[sl], (r / RING) & 1)) {
            atomicOr(P.error, ERR_TIMEOUT_FULL);
            *abort_flag = 1;
            return -1;
        }
        const int w = ring[sl];
        mbar_arrive(&item_empty[sl]);
        return w;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < Tr::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < Tr::NACC; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 128);
        }
        mbar_init(drain, 1);
        for (int i = 0; i < RING; ++i) {
            mbar_init(&item_full[i], 1);
            mbar_init(&item_empty[i], 1 + 128);  // the MMA thread and the 128 epilogue threads
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, Tr::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the prologue above may overlap the preceding kernel; operands, maps and
    // outputs are touched only after it has completed
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int last_p = -1;
            int issued = 0;  // stages armed so far
            for (int r = 0;; ++r) {
                const int w = publish(r);
                if (w < 0 || *abort_flag) break;
                Work k = decode_work(P, w);
                const TcProb &q = P.prob[k.p];
                const CUtensorMap *ma = P.maps + q.map_a;
                const CUtensorMap *mb = P.maps + q.map_b;
                if (k.p != last_p) {  // consecutive items of one problem share its maps
                    acquire_map(ma);
                    acquire_map(mb);
                    if (KIND == TC_KIND_TF32X3) {
                        acquire_map(ma + 1);
                        acquire_map(mb + 1);
                    }
                    last_p = k.p;
                }
                const bool diag = KIND == TC_KIND_BF16 && q.syrk && k.tm == k.tn;
                Im2colCursor cur;
                if (KIND == TC_KIND_BF16 && q.im2col) im2col_start(q, k, cur);
                const uint32_t bytes = KIND == TC_KIND_TF32X3 ? (uint32_t)(2 * (BM + q.bn) * 128)
                                       : diag                 ? (uint32_t)Tr::TILE
                                                              : (uint32_t)STAGE_BYTES;
                for (int kt = k.kt0; kt < k.kt1 && !*abort_flag; ++kt) {
                    if (!mbar_wait(&empty[stage], phase ^ 1)) {
                        atomicOr(P.error, ERR_TIMEOUT_EMPTY);
                        *abort_flag = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], bytes);
                    uint8_t *sa = smem + stage * STAGE_BYTES;
                    const int k0 = kt * Tr::BK;
                    if (KIND == TC_KIND_BF16 && q.im2col) {
                        im2col_load(sa, ma, q, cur, 0, &full[stage]);
                        if (!diag) im2col_load(sa + Tr::TILE, mb, q, cur, 1, &full[stage]);
                        im2col_advance(q, cur);
                    } else if (KIND == TC_KIND_BF16) {
                        load_tile_bf16(sa, ma, q.a_mn, q.a_row0, q.a_col0, k.tm * BM, k0, &full[stage]);
                        if (!diag)
                            load_tile_bf16(sa + Tr::TILE, mb, q.b_mn, q.b_row0, q.b_col0, k.tn * BN, k0,
                                           &full[stage]);
                    } else {
                        // (hi, lo) pairs in one copy each: hi at the tile, lo right after it
                        tma_load_3d(sa, ma + 1, q.a_col0 + k0, q.a_row0 + k.tm * BM, 0, &full[stage]);
                        if (q.bn == BN) {
                            tma_load_3d(sa + 2 * TILE_BYTES, mb + 1, q.b_col0 + k0, q.b_row0 + k.tn * BN, 0,
                                        &full[stage]);
                        } else {  // narrow tile: B from the 32-row-box maps
                            load_rows_tf32(sa + 2 * TILE_BYTES, mb, q.b_row0, q.b_col0, k.tn * q.bn, q.bn, k0,
                                           &full[stage]);
                            load_rows_tf32(sa + 3 * TILE_BYTES, mb + 1, q.b_row0, q.b_col0, k.tn * q.bn, q.bn,
                                           k0, &full[stage]);
                        }
                    }
                    if (++stage == Tr::STAGES) { stage = 0; phase ^= 1; }
                    ++issued;
                }
            }
            if (*abort_flag) {
                // the run was cut short: before the CTA exits, wait (bounded)
                // for the copies this thread issued into the last STAGES
                // stages (older stages were consumed, so their copies landed)
                for (int n = 0; n < min(issued, Tr::STAGES); ++n) {
                    if (stage == 0) { stage = Tr::STAGES - 1; phase ^= 1; } else { --stage; }
                    if (!mbar_wait(&full[stage], phase)) atomicOr(P.error, ERR_TIMEOUT_DRAIN);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int cc = 0;  // accumulation chunks so far (accumulator cc % NACC)
            bool ok = true;
            for (int r = 0;; ++r) {
                const int w = take(r);
                if (w < 0 || !ok || *abort_flag) break;
                Work k = decode_work(P, w);
                const TcProb &q = P.prob[k.p];
                const bool diag = KIND == TC_KIND_BF16 && q.syrk && k.tm == k.tn;
                const uint32_t idesc = KIND == TC_KIND_BF16 ? idesc_bf16_f32(BM, BN, q.a_mn, q.b_mn, q.f16)
                                                            : idesc_tf32_f32(BM, q.bn);
                const int nchunk = max(1, (int)ceil_div_dev(k.kt1 - k.kt0, Tr::CHUNK));
                for (int ch = 0; ch < nchunk && ok; ++ch, ++cc) {
                    const int b = cc % Tr::NACC;
                    const uint32_t use = (uint32_t)(cc / Tr::NACC);
                    if (!mbar_wait(&acce[b], (use & 1) ^ 1)) {
                        atomicOr(P.error, ERR_TIMEOUT_ACC);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + b * BN;
                    const int k_lo = k.kt0 + ch * Tr::CHUNK;
                    const int k_hi = ch + 1 == nchunk ? k.kt1 : k_lo + Tr::CHUNK;
                    for (int kt = k_lo; kt < k_hi; ++kt) {
                        if (!mbar_wait(&full[stage], phase)) {
                            atomicOr(P.error, ERR_TIMEOUT_FULL);
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t s0 = smem_u32(smem + stage * STAGE_BYTES);
                        if (KIND == TC_KIND_BF16) {
                            const uint32_t b_base = diag ? s0 : s0 + Tr::TILE;
    #pragma unroll
                            for (int kk = 0; kk < KSLICES; ++kk)
                                tc_mma_f16(d_tmem, operand_desc_bf16(s0, q.a_mn, kk), operand_desc_bf16(b_base, q.b_mn, kk),
                                           idesc, (kt > k_lo || kk > 0) ? 1u : 0u);
                        } else {
                            const uint32_t ah = s0, al = s0 + TILE_BYTES, bh = s0 + 2 * TILE_BYTES,
                                           bl = s0 + 3 * TILE_BYTES;
    #pragma unroll
                            for (int kk = 0; kk < KSLICES; ++kk) {
                                const uint64_t dah = operand_desc(ah, 0, kk), dbh = operand_desc(bh, 0, kk);
                                tc_mma_tf32(d_tmem, dah, dbh, idesc, (kt > k_lo || kk > 0) ? 1u : 0u);
                                tc_mma_tf32(d_tmem, dah, operand_desc(bl, 0, kk), idesc, 1u);
                                tc_mma_tf32(d_tmem, operand_desc(al, 0, kk), dbh, idesc, 1u);
                            }
                        }
                        tc_commit(&empty[stage]);
                        if (++stage == Tr::STAGES) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    tc_commit(&accf[b]);
                }
            }
            if (*abort_flag) {
                // the run was cut short: wait (bounded) for every product
                // this thread issued before the accumulators are released
                tc_commit(drain);
                if (!mbar_wait(drain, 0)) atomicOr(P.error, ERR_TIMEOUT_DRAIN);
            }
        }
    } else {
        // epilogue warps 2..5 -> TMEM lane quarters 2,3,0,1
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int etid = threadIdx.x - 64;  // 0..127
        float *stage = epi_stage + (warp - 2) * 32 * STAGE_LD;
        const uint32_t t_quarter = tmem_base + ((uint32_t)(quarter * 32) << 16);
        const uint32_t t_sum = t_quarter + Tr::NACC * BN;  // running sum of a chunked item (tf32x3)
        int cc = 0;
        bool nonfin = false;  // a value this lane stored was NaN or infinite
        for (int r = 0;; ++r) {
            const int w = take(r);
            if (w < 0 || *abort_flag) break;
            Work k = decode_work(P, w);
            const TcProb &q = P.prob[k.p];
            const int i0 = k.tm * BM + quarter * 32;
            const int nch = q.bn / 32;
            const bool mirror = q.sym && k.tn >= (k.tm + 1) * (BM / q.bn);
            const bool diagblk = q.sym && !mirror;
            const int nchunk = max(1, (int)ceil_div_dev(k.kt1 - k.kt0, Tr::CHUNK));
            // all chunks but the last: add into the running sum
            bool ok = true;
            for (int ch = 0; ch + 1 < nchunk; ++ch, ++cc) {
                const int b = cc % Tr::NACC;
                if (!mbar_wait(&accf[b], (uint32_t)(cc / Tr::NACC) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < nch; ++c) {
                    float v[32];
                    if (ch > 0) {
                        float s2[32];
                        tmem_ld_pair_32x32b_x32(t_quarter + b * BN + c * 32, v, t_sum + c * 32, s2);
#pragma unroll
                        for (int t = 0; t < 32; ++t) v[t] += s2[t];
                    } else {
                        tmem_ld_32x32b_x32(t_quarter + b * BN + c * 32, v);
                    }
                    tmem_st_32x32b_x32(t_sum + c * 32, v);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&acce[b]);
            }
            if (!ok) {
                atomicOr(P.error, ERR_TIMEOUT_ACC);
                *abort_flag = 1;
                break;
            }
            const int b = cc % Tr::NACC;
            const uint32_t use = (uint32_t)(cc / Tr::NACC);
            ++cc;
            float4 oh[8], ol[8];
            // the first column chunk's old values load while the MMAs run
            if (q.ksplit == 1) load_old(q, i0, k.tn * q.bn, lane, oh, ol);
            if (!mbar_wait(&accf[b], use & 1)) {
                atomicOr(P.error, ERR_TIMEOUT_ACC);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            uint32_t t_row = t_quarter + b * BN;
            // a split with an empty K range (ktri tiles near the end) issued
            // no MMA: its accumulator holds nothing of this tile and counts as 0
            const bool empty = k.kt0 >= k.kt1;
            bool summed = nchunk > 1;
            if (KIND == TC_KIND_TF32X3 && TF32X3_EARLY_RELEASE) {
                // release the accumulator before the stores: the item's sum
                // goes into the running-sum columns and is stored from there,
                // so the next item's second chunk need not wait for the stores
#pragma unroll 1
                for (int c = 0; c < nch; ++c) {
                    float v[32];
                    if (summed) {
                        float s2[32];
                        tmem_ld_pair_32x32b_x32(t_row + c * 32, v, t_sum + c * 32, s2);
#pragma unroll
                        for (int t = 0; t < 32; ++t) v[t] += s2[t];
                    } else {
                        tmem_ld_32x32b_x32(t_row + c * 32, v);
                    }
                    tmem_st_32x32b_x32(t_sum + c * 32, v);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&acce[b]);
                t_row = t_sum;
                summed = false;
            }
            if (q.ksplit == 1) {
#pragma unroll 1
                for (int c = 0; c < nch; ++c) {
                    if (c > 0) load_old(q, i0, k.tn * q.bn + c * 32, lane, oh, ol);
                    float v[32];
                    if (summed) {
                        float s2[32];
                        tmem_ld_pair_32x32b_x32(t_row + c * 32, v, t_sum + c * 32, s2);
#pragma unroll
                        for (int t = 0; t < 32; ++t) v[t] += s2[t];
                    } else {
                        tmem_ld_32x32b_x32(t_row + c * 32, v);
                    }
                    if (empty) {
#pragma unroll
                        for (int t = 0; t < 32; ++t) v[t] = 0.f;
                    }
                    nonfin |= chunk_store(q, i0, k.tn * q.bn + c * 32, v, stage, lane, mirror, diagblk, oh, ol);
                }
                if (!(KIND == TC_KIND_TF32X3 && TF32X3_EARLY_RELEASE)) {
                    tc_fence_before();
                    mbar_arrive(&acce[b]);
                }
            } else {
                float4 *part = (float4 *)(q.partial + ((long long)k.tile * q.ksplit + k.split) * (BM * BN));
#pragma unroll 1
                for (int c = 0; c < nch; ++c) {
                    float v[32];
                    if (summed) {
                        float s2[32];
                        tmem_ld_pair_32x32b_x32(t_row + c * 32, v, t_sum + c * 32, s2);
#pragma unroll
                        for (int t = 0; t < 32; ++t) v[t] += s2[t];
                    } else {
                        tmem_ld_32x32b_x32(t_row + c * 32, v);
                    }
                    if (empty) {
#pragma unroll
                        for (int t = 0; t < 32; ++t) v[t] = 0.f;
                    }
#pragma unroll
                    for (int f = 0; f < 8; ++f)
                        part[(c * 8 + f) * BM + row] = make_float4(v[4 * f], v[4 * f + 1], v[4 * f + 2], v[4 * f + 3]);
                }
                if (!(KIND == TC_KIND_TF32X3 && TF32X3_EARLY_RELEASE)) {
                    tc_fence_before();
                    mbar_arrive(&acce[b]);
                }
                __threadfence();
                named_barrier_sync(1, 128);
                if (etid == 0) {
                    int old = atomicAdd(&q.counters[k.tile], 1);
                    *last_flag = (old == q.ksplit - 1) ? 1 : 0;
                }
                named_barrier_sync(1, 128);
                const bool last = *last_flag != 0;
                named_barrier_sync(1, 128);  // everyone has read last_flag
                if (last) {
                    __threadfence();
                    const float4 *base = (const float4 *)(q.partial + (long long)k.tile * q.ksplit * (BM * BN));
#pragma unroll 1
                    for (int c = 0; c < nch; ++c) {
                        load_old(q, i0, k.tn * q.bn + c * 32, lane, oh, ol);
                        float v[32];
#pragma unroll
                        for (int t = 0; t < 32; ++t) v[t] = 0.f;
                        for (int sp = 0; sp < q.ksplit; ++sp) {
                            const float4 *src = base + (long long)sp * (BM * BN / 4) + (c * 8) * BM + row;
#pragma unroll
                            for (int f = 0; f < 8; ++f) {
                                const float4 t = __ldcg(src + f * BM);
                                v[4 * f] += t.x; v[4 * f + 1] += t.y; v[4 * f + 2] += t.z; v[4 * f + 3] += t.w;
                            }
                        }
                        nonfin |= chunk_store(q, i0, k.tn * q.bn + c * 32, v, stage, lane, mirror, diagblk, oh, ol);
                    }
                    if (etid == 0) q.counters[k.tile] = 0;
                }
            }
        }
        if (__any_sync(0xffffffffu, nonfin) && lane == 0) atomicOr(P.error, ERR_NONFINITE);
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Tr::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host

struct Plan {
    int bn = BN;               // output tile width of every job in the call
    std::vector<int> order;    // job indices in launch order
    std::vector<int> ksplit;   // per job
    std::vector<int> tiles;    // per job
    std::vector<int> k_tiles;  // per job
};

int bk_of(int kind) { return kind == TC_KIND_BF16 ? Traits<TC_KIND_BF16>::BK : Traits<TC_KIND_TF32X3>::BK; }

int tiles_of(const TcJob &j, int bn) {
    const int tm = (int)ceil_div(j.M, BM), tn = (int)ceil_div(j.N, bn);
    if (j.lower) {  // row block t runs column blocks 0 .. (t+1)*128/bn - 1
        int n = 0;
        for (int t = 0; t < tm; ++t) n += std::min(tn, (t + 1) * BM / bn);
        return n;
    }
    if (!(j.syrk || j.sym)) return tm * tn;
    const int r = BM / bn;  // upper tiles: row block t runs column blocks t*r .. tn-1
    int n = 0;
    for (int t = 0; t < tm; ++t) n += std::max(0, tn - t * r);
    return n;
}

Plan make_plan(const TcJob *jobs, int n, int kind, int sms) {
    Plan p;
    p.ksplit.resize(n);
    p.tiles.resize(n);
    p.k_tiles.resize(n);
    // A launch with few 128-wide tiles leaves most SMs idle and funnels each
    // tile's loads and stores through one SM: narrow the tiles (tf32x3 only)
    // until the launch covers at least half of the SMs.
    // Long K ranges are split instead (each split keeps at least 8 K tiles),
    // which keeps 128-wide tiles and so reads each A row panel once per tile.
    if (kind == TC_KIND_TF32X3) {
        long long splittable = 0;
        for (int i = 0; i < n; ++i)
            splittable += (long long)tiles_of(jobs[i], BN) *
                          std::max(1, std::min(TF32X3_MAX_SPLIT, (int)(ceil_div(jobs[i].K, 32) / 8)));
        if (!TF32X3_PREFER_SPLIT || splittable < sms) {
            for (;;) {
                long long t = 0;
                for (int i = 0; i < n; ++i) t += tiles_of(jobs[i], p.bn);
                if (p.bn == 32 || 2 * t >= sms) break;
                p.bn /= 2;
            }
        }
    }
    double total = 0.0;
    for (int i = 0; i < n; ++i) {
        p.tiles[i] = tiles_of(jobs[i], p.bn);
        p.k_tiles[i] = (int)ceil_div(jobs[i].K, bk_of(kind));
        total += (double)p.tiles[i] * p.k_tiles[i];
    }
    // Split K only where one problem's tiles would otherwise be the critical
    // path: the longest work item should not exceed about twice the average
    // share of one SM.  A split costs a partial-tile round trip through L2, so
    // items keep at least 8 K tiles; a tf32x3 tile takes at most
    // TF32X3_MAX_SPLIT splits (its last CTA reads all partials).
    const double min_kt = kind == TC_KIND_BF16 ? 8.0 : TF32X3_MIN_KT;
    const double target = std::max(min_kt, total / (sms * (kind == TC_KIND_BF16 ? KFAC_BF16_ITEMS_PER_SM : 2.0)));
    for (int i = 0; i < n; ++i) {
        int ks = (int)std::ceil(p.k_tiles[i] / target);
        if (kind == TC_KIND_TF32X3) ks = std::min(ks, TF32X3_MAX_SPLIT);
        ks = std::max(1, std::min(ks, std::min(p.k_tiles[i], 256)));
        if (jobs[i].fine_split) ks = std::max(1, std::min(16, (int)ceil_div(p.k_tiles[i], 12)));
        if (jobs[i].no_split || jobs[i].ktri) ks = 1;  // (a ktri split would leave late tiles empty)
        p.ksplit[i] = ks;
    }
    p.order.resize(n);
    for (int i = 0; i < n; ++i) p.order[i] = i;
    // longest work items first (static round-robin then balances better)
    std::stable_sort(p.order.begin(), p.order.end(), [&](int a, int b) {
        double ca = (double)p.k_tiles[a] / p.ksplit[a], cb = (double)p.k_tiles[b] / p.ksplit[b];
        return ca > cb;
    });
    return p;
}

struct Buffers {
    std::vector<float *> part;
    std::vector<int *> cnt;
    int *cnt_base = nullptr;
    size_t ncnt = 0;
};

void take_buffers(const Plan &p, int n, Arena &ws, Buffers &b) {
    b.part.assign(n, nullptr);
    b.cnt.assign(n, nullptr);
    b.ncnt = 0;
    for (int i = 0; i < n; ++i)
        if (p.ksplit[i] > 1) b.ncnt += p.tiles[i];
    b.cnt_base = ws.take<int>(std::max<size_t>(b.ncnt, 1));
    size_t off = 0;
    for (int i = 0; i < n; ++i) {
        if (p.ksplit[i] > 1) {
            b.part[i] = ws.take<float>((size_t)p.tiles[i] * p.ksplit[i] * BM * BN);
            b.cnt[i] = b.cnt_base ? b.cnt_base + off : nullptr;
            off += p.tiles[i];
        }
    }
}

template <int KIND>
cudaError_t set_smem_attr() {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(tc_gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)SMEM_BYTES);
    });
    return err;
}

}  // namespace

bool tc_make_map(CUtensorMap *m, int kind, const void *ptr, long long ld, int rows, int cols, int box_rows,
                 bool f16) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    const int esz = kind == TC_KIND_BF16 ? 2 : 4;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * esz};
    const cuuint32_t inner = 128u / esz;  // 128-byte rows
    cuuint32_t box[2] = {inner, box_rows > 0 ? (cuuint32_t)box_rows : 128u};
    cuuint32_t estr[2] = {1u, 1u};
    const CUtensorMapDataType dt = kind == TC_KIND_BF16
                                       ? (f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)
                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUresult r = enc(m, dt, 2, (void *)ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool tc_make_pair_map(CUtensorMap *m, const float *hi, const float *lo, long long ld, int rows, int cols,
                      int box_rows) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc || lo <= hi) return false;
    const long long plane = (long long)((const char *)lo - (const char *)hi);
    if (plane % 16 != 0) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, 2};
    cuuint64_t strides[2] = {(cuuint64_t)ld * 4, (cuuint64_t)plane};
    cuuint32_t box[3] = {32u, (cuuint32_t)box_rows, 2u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, (void *)hi, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool tc_make_im2col_map(CUtensorMap *m, const void *x, int n, int h, int w, int c, int k, int stride, int pad,
                        bool f16) {
    EncodeIm2colFn enc = encode_im2col_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)c, (cuuint64_t)w, (cuuint64_t)h, (cuuint64_t)n};
    cuuint64_t strides[3] = {(cuuint64_t)c * 2, (cuuint64_t)w * c * 2, (cuuint64_t)h * w * c * 2};
    // base pixels run from -pad to the last one whose k x k window still
    // starts inside the padded input (offsets from the two corners)
    int lower[2] = {-pad, -pad};
    int upper[2] = {pad - (k - 1), pad - (k - 1)};
    cuuint32_t estr[4] = {1u, (cuuint32_t)stride, (cuuint32_t)stride, 1u};
    CUresult r = enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, (void *)x, dims,
                     strides, lower, upper, 64u, 128u, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

kfac_status tc_upload_maps(const CUtensorMap *maps, int n, CUtensorMap *dev, cudaStream_t st) {
    std::unique_ptr<MapCopyParams> P(new MapCopyParams);
    for (int base = 0; base < n; base += MAPS_PER_COPY) {
        const int cnt = std::min(MAPS_PER_COPY, n - base);
        std::memcpy(P->m, maps + base, sizeof(CUtensorMap) * cnt);
        P->dst = dev + base;
        P->n = cnt;
        KFAC_LAUNCH(KK_MAPCOPY, st, map_copy_kernel, (int)ceil_div(cnt * 8, 256), 256, 0, *P);
    }
    return KFAC_OK;
}

int cta_cap(int max_ctas) {
    const int sms = device_sm_count();
    return max_ctas > 0 ? std::min(max_ctas, sms) : sms;
}

size_t tc_workspace_bytes(const TcJob *jobs, int njobs, int kind, int max_ctas) {
    if (njobs <= 0) return 0;
    Plan p = make_plan(jobs, njobs, kind, cta_cap(max_ctas));
    Arena a;
    Buffers b;
    take_buffers(p, njobs, a, b);
    if (DYNAMIC_WORK) a.take<int>(1);  // the work counter
    return a.used;
}

kfac_status tc_run(const TcJob *jobs, int njobs, int kind, const CUtensorMap *dev_maps, Arena &ws,
                   int *err, cudaStream_t st, int max_ctas) {
    if (njobs <= 0) return KFAC_OK;
    if ((kind == TC_KIND_BF16 ? set_smem_attr<TC_KIND_BF16>() : set_smem_attr<TC_KIND_TF32X3>()) != cudaSuccess)
        return KFAC_ERR_CUDA;
    for (int i = 0; i < njobs; ++i) {
        const TcJob &j = jobs[i];
        if (j.Ct && j.beta != 0.f) return KFAC_ERR_INVALID;                       // transposed copy needs beta == 0
        if (j.sym && (kind != TC_KIND_TF32X3 || j.M != j.N || (j.epi != TC_EPI_SPLIT && j.epi != TC_EPI_STORE)))
            return KFAC_ERR_INVALID;
        if (j.lower && (kind != TC_KIND_TF32X3 || j.sym || j.syrk || j.epi != TC_EPI_SPLIT)) return KFAC_ERR_INVALID;
        if ((j.ktri || j.ktril) && kind != TC_KIND_TF32X3) return KFAC_ERR_INVALID;
        if (j.W && (j.epi != TC_EPI_STORE || j.sym)) return KFAC_ERR_INVALID;
        if (j.f16 && kind != TC_KIND_BF16) return KFAC_ERR_INVALID;
        if (j.packed && (j.epi != TC_EPI_ACCUM || !j.syrk || j.packed_d < j.N)) return KFAC_ERR_INVALID;
        if (!j.C && !j.Ct && !j.Cb && !j.W) return KFAC_ERR_INVALID;
    }
    const int sms = cta_cap(max_ctas);
    Plan p = make_plan(jobs, njobs, kind, sms);
    Buffers bufs;
    take_buffers(p, njobs, ws, bufs);
    if (!ws.fits()) return KFAC_ERR_WORKSPACE;
    if (bufs.ncnt) KFAC_CUDA_TRY(cudaMemsetAsync(bufs.cnt_base, 0, bufs.ncnt * sizeof(int), st));

    int *counter = DYNAMIC_WORK ? ws.take<int>(1) : nullptr;
    if (!ws.fits()) return KFAC_ERR_WORKSPACE;
    std::unique_ptr<TcParams> P(new TcParams);
    size_t pos = 0;
    while (pos < p.order.size()) {
        int nprob = 0, work = 0;
        while (pos < p.order.size() && nprob < MAX_PROBS) {
            const int ji = p.order[pos];
            const TcJob &j = jobs[ji];
            TcProb &q = P->prob[nprob];
            std::memset(&q, 0, sizeof(q));
            q.map_a = j.map_a;
            q.map_b = j.syrk ? j.map_a : j.map_b;
            q.a_mn = j.a_mn;
            q.b_mn = j.syrk ? j.a_mn : j.b_mn;
            q.a_row0 = j.a_row0; q.a_col0 = j.a_col0;
            q.b_row0 = j.syrk ? j.a_row0 : j.b_row0;
            q.b_col0 = j.syrk ? j.a_col0 : j.b_col0;
            q.M = j.M;
            q.N = j.N;
            q.k_tiles = p.k_tiles[ji];
            q.bn = p.bn;
            if (kind == TC_KIND_TF32X3 && p.bn < BN) q.map_b += 2;
            q.tiles_n = (int)ceil_div(j.N, p.bn);
            q.syrk = j.syrk;
            q.sym = j.sym;
            q.lower = j.lower;
            q.ktri = j.ktri;
            q.ktril = j.ktril;
            q.grouped = TF32X3_GROUPED && kind == TC_KIND_TF32X3 && !j.lower;
            q.tiles_m = (int)ceil_div(j.M, BM);
            q.ksplit = p.ksplit[ji];
            q.work_begin = work;
            q.epi = j.epi;
            q.alpha = j.alpha;
            q.beta = j.beta;
            q.C = j.C; q.C_lo = j.C_lo; q.ldc = j.ldc;
            q.Ct = j.Ct; q.Ct_lo = j.Ct_lo; q.ldct = j.ldct;
            q.Cb = j.Cb; q.ldcb = j.ldcb;
            q.vec = (j.ldc % 4 == 0) && ((uintptr_t)j.C % 16 == 0) && ((uintptr_t)j.C_lo % 16 == 0);
            q.vecb = (j.ldcb % 4 == 0) && ((uintptr_t)j.Cb % 8 == 0);
            q.W = j.W; q.ldw = j.ldw; q.eta = j.eta;
            q.f16 = j.f16 ? 1 : 0;
            q.cb_f16 = j.cb_f16 ? 1 : 0;
            q.packed = j.packed ? 1 : 0;
            q.packed_d = j.packed_d;
            q.vecw = (j.ldw % 4 == 0) && ((uintptr_t)j.W % 16 == 0);
            q.vect = (j.ldct % 4 == 0) && ((uintptr_t)j.Ct % 16 == 0) && ((uintptr_t)j.Ct_lo % 16 == 0);
            q.im2col = j.im2col ? 1 : 0;
            q.im_k = (uint8_t)j.im_k; q.im_stride = (uint8_t)j.im_stride; q.im_pad = (uint8_t)j.im_pad;
            q.im_c = j.im_c; q.im_wo = j.im_wo; q.im_howo = j.im_howo;
            q.im_ho = j.im_wo > 0 ? j.im_howo / j.im_wo : 0;
            q.partial = bufs.part[ji];
            q.counters = bufs.cnt[ji];
            work += p.tiles[ji] * p.ksplit[ji];
            ++nprob;
            ++pos;
        }
        P->maps = dev_maps;
        P->nprob = nprob;
        P->total_work = work;
        P->error = err;
        const int grid = std::max(1, std::min(work, sms));
        // dynamic distribution where CTAs take several items (a launch of at
        // most one or two rounds keeps the static order, and with it the
        // early launch of its prologue behind the previous kernel)
        bool asks = false;
        for (int i = 0; i < njobs; ++i) asks |= jobs[i].dyn != 0;
        const bool dyn = counter && asks && work > 2 * grid;
        P->counter = dyn ? counter : nullptr;
        if (dyn) KFAC_CUDA_TRY(cudaMemsetAsync(counter, 0, sizeof(int), st));
        if (kind == TC_KIND_BF16)
            KFAC_LAUNCH(KK_TC_BF16, st, tc_gemm_kernel<TC_KIND_BF16>, grid, NUM_THREADS, SMEM_BYTES, *P);
        else
            KFAC_LAUNCH(KK_TC_TF32X3, st, tc_gemm_kernel<TC_KIND_TF32X3>, grid, NUM_THREADS, SMEM_BYTES, *P);
    }
    return KFAC_OK;
}

}  // namespace kfac
