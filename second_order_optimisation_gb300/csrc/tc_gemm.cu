// tc_gemm.cu -- persistent tcgen05 (5th-generation tensor core) GEMM / SYRK
// engine for sm_103a, bf16 operands, fp32 accumulation in TMEM.
//
// Used for the Kronecker-factor statistic A = P^T P / G = Gam^T Gam
// (Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
// Kronecker-Factored Approximate Curvature ...", section 3.2, Eq. 5), whose
// operands are the same [rows x d] matrix read MN-major, and for the two
// chained GEMMs of the preconditioned gradient G^-1 grad A^-1 (Eq. 7).
//
// One launch runs a list of heterogeneous problems.  Each CTA (one per SM)
// walks a static, strided list of work items (problem, 128x128 output tile,
// K split).  Warp roles:
//   warp 0      TMA producer: 128-byte-swizzled tiles into a 6-stage ring
//   warp 1      TMEM owner + MMA issuer (one thread): tcgen05.mma 128x128x16
//   warps 2..5  epilogue: tcgen05.ld TMEM -> registers -> global, with a
//               double-buffered accumulator so it overlaps the next tile
// Split-K partial tiles are reduced by the last-arriving CTA of the tile in
// split order (deterministic; no spin-waits).  The epilogue either
// accumulates into an fp32 matrix (F <- beta F + alpha acc, optionally upper
// triangle only) or stores fp32 and/or bf16.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <mutex>
#include <vector>

#include "internal.h"

namespace kfac {

constexpr int BM = 128, BN = 128, BK = 64, STAGES = 6;
constexpr int TILE_A_BYTES = BM * BK * 2;  // 16 KB
constexpr int TILE_B_BYTES = BN * BK * 2;  // 16 KB
constexpr int STAGE_BYTES = TILE_A_BYTES + TILE_B_BYTES;
constexpr int MAX_MAPS = 112, MAX_PROBS = 112;
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;  // two accumulators
constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;

struct TcProb {
    int map_a, map_b;
    int a_mn, b_mn;
    int M, N;
    int k_tiles;
    int tiles_n;
    int syrk;
    int ksplit;
    int work_begin;
    int epi;
    float alpha, beta;
    float *C;
    long long ldc;
    uint16_t *Cb;
    long long ldcb;
    float *partial;  // [tiles][ksplit][BM*BN] when ksplit > 1
    int *counters;   // [tiles]
};

struct TcParams {
    CUtensorMap maps[MAX_MAPS];
    TcProb prob[MAX_PROBS];
    int nprob;
    int total_work;
    int *error;
};
static_assert(sizeof(TcParams) <= 32000, "kernel parameter block too large");

struct Work {
    int p, tile, tm, tn, split, kt0, kt1;
};

__device__ __forceinline__ Work decode_work(const TcParams &P, int w) {
    int lo = 0, hi = P.nprob - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.prob[mid].work_begin <= w) lo = mid; else hi = mid - 1;
    }
    const TcProb &q = P.prob[lo];
    Work k;
    k.p = lo;
    int local = w - q.work_begin;
    k.tile = local / q.ksplit;
    k.split = local - k.tile * q.ksplit;
    if (q.syrk) {
        int T = q.tiles_n, t = k.tile, tm = 0;
        while (t >= T - tm) { t -= T - tm; ++tm; }
        k.tm = tm;
        k.tn = tm + t;
    } else {
        k.tm = k.tile / q.tiles_n;
        k.tn = k.tile - k.tm * q.tiles_n;
    }
    k.kt0 = (int)((long long)k.split * q.k_tiles / q.ksplit);
    k.kt1 = (int)((long long)(k.split + 1) * q.k_tiles / q.ksplit);
    return k;
}

// Operand tile of 128 (M or N) x 64 (K) bf16 into shared memory.
//   MN-major source [K][MN]: two 64x64 boxes (MN 0-63 | 64-127), 8 KB apart.
//   K-major source  [MN][K]: one 64(K) x 128(MN) box.
__device__ __forceinline__ void load_operand(uint8_t *dst, const CUtensorMap *map, int mn, int mn0,
                                             int k0, uint64_t *bar) {
    if (mn) {
        tma_load_2d(dst, map, mn0, k0, bar);
        tma_load_2d(dst + 8192, map, mn0 + 64, k0, bar);
    } else {
        tma_load_2d(dst, map, k0, mn0, bar);
    }
}

// Descriptor of the kk-th K=16 slice of a staged operand tile.
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int mn, int kk) {
    // MN-major: 8-row K groups are 1024 B apart (SBO), the two 64-wide MN
    //           blocks 8192 B apart (LBO); a K=16 slice is two K groups.
    // K-major : rows 128 B, 8-row groups 1024 B apart (SBO); a K=16 slice is
    //           32 B inside the swizzled row.
    return mn ? smem_desc_sw128(base + kk * 2048, 8192, 1024)
              : smem_desc_sw128(base + kk * 32, 16, 1024);
}

__device__ __forceinline__ void epi_store(const TcProb &q, int i, int j0, const float *v, int n) {
    if (i >= q.M) return;
    if (q.epi == TC_EPI_ACCUM) {
        float *row = q.C + (long long)i * q.ldc;
        const bool upper = q.syrk;
        const float a = q.alpha, b = q.beta;
        for (int t = 0; t < n; ++t) {
            int j = j0 + t;
            if (j < q.N && (!upper || j >= i)) {
                float o = a * v[t];
                if (b != 0.f) o = fmaf(b, row[j], o);
                row[j] = o;
            }
        }
    } else {
        for (int t = 0; t < n; ++t) {
            int j = j0 + t;
            if (j < q.N) {
                float o = q.alpha * v[t];
                if (q.C) q.C[(long long)i * q.ldc + j] = o;
                if (q.Cb) q.Cb[(long long)i * q.ldcb + j] = f32_to_bf16_bits(o);
            }
        }
    }
}

__global__ void __launch_bounds__(NUM_THREADS, 1) tc_gemm_kernel(const __grid_constant__ TcParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *full = (uint64_t *)(smem + STAGES * STAGE_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *accf = empty + STAGES;
    uint64_t *acce = accf + 2;
    uint32_t *tmem_slot = (uint32_t *)(acce + 2);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    volatile int *last_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 128);
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int w = blockIdx.x; w < P.total_work && !*abort_flag; w += gridDim.x) {
                Work k = decode_work(P, w);
                const TcProb &q = P.prob[k.p];
                const CUtensorMap *ma = &P.maps[q.map_a];
                const CUtensorMap *mb = &P.maps[q.map_b];
                const bool diag = q.syrk && k.tm == k.tn;
                const uint32_t bytes = diag ? TILE_A_BYTES : STAGE_BYTES;
                for (int kt = k.kt0; kt < k.kt1; ++kt) {
                    if (!mbar_wait(&empty[stage], phase ^ 1)) {
                        atomicOr(P.error, ERR_TIMEOUT_EMPTY);
                        *abort_flag = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], bytes);
                    uint8_t *sa = smem + stage * STAGE_BYTES;
                    load_operand(sa, ma, q.a_mn, k.tm * BM, kt * BK, &full[stage]);
                    if (!diag) load_operand(sa + TILE_A_BYTES, mb, q.b_mn, k.tn * BN, kt * BK, &full[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            for (int w = blockIdx.x; w < P.total_work && !*abort_flag; w += gridDim.x, ++it) {
                Work k = decode_work(P, w);
                const TcProb &q = P.prob[k.p];
                const bool diag = q.syrk && k.tm == k.tn;
                const int b = it & 1;
                const uint32_t use = (uint32_t)(it >> 1);
                if (!mbar_wait(&acce[b], (use & 1) ^ 1)) {
                    atomicOr(P.error, ERR_TIMEOUT_ACC);
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * BN;
                const uint32_t idesc = idesc_bf16_f32(BM, BN, q.a_mn, q.b_mn);
                bool ok = true;
                for (int kt = k.kt0; kt < k.kt1; ++kt) {
                    if (!mbar_wait(&full[stage], phase)) {
                        atomicOr(P.error, ERR_TIMEOUT_FULL);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t b_base = diag ? a_base : a_base + TILE_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        tc_mma_f16(d_tmem, operand_desc(a_base, q.a_mn, kk),
                                   operand_desc(b_base, q.b_mn, kk), idesc,
                                   (kt > k.kt0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit(&accf[b]);
            }
        }
    } else {
        // epilogue warps 2..5 -> TMEM lane quarters 2,3,0,1
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int etid = threadIdx.x - 64;  // 0..127
        int it = 0;
        for (int w = blockIdx.x; w < P.total_work && !*abort_flag; w += gridDim.x, ++it) {
            Work k = decode_work(P, w);
            const TcProb &q = P.prob[k.p];
            const int b = it & 1;
            const uint32_t use = (uint32_t)(it >> 1);
            if (!mbar_wait(&accf[b], use & 1)) {
                atomicOr(P.error, ERR_TIMEOUT_ACC);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + b * BN;
            const int i = k.tm * BM + row;
            if (q.ksplit == 1) {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tmem_ld_32x32b_x32(t_row + c * 32, v);
                    epi_store(q, i, k.tn * BN + c * 32, v, 32);
                }
                tc_fence_before();
                mbar_arrive(&acce[b]);
            } else {
                float4 *part = (float4 *)(q.partial + ((long long)k.tile * q.ksplit + k.split) * (BM * BN));
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tmem_ld_32x32b_x32(t_row + c * 32, v);
#pragma unroll
                    for (int f = 0; f < 8; ++f)
                        part[(c * 8 + f) * BM + row] = make_float4(v[4 * f], v[4 * f + 1], v[4 * f + 2], v[4 * f + 3]);
                }
                tc_fence_before();
                mbar_arrive(&acce[b]);
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
                    for (int c4 = 0; c4 < BN / 4; ++c4) {
                        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int sp = 0; sp < q.ksplit; ++sp) {
                            float4 t = __ldcg(base + (long long)sp * (BM * BN / 4) + c4 * BM + row);
                            s.x += t.x; s.y += t.y; s.z += t.z; s.w += t.w;
                        }
                        float v[4] = {s.x, s.y, s.z, s.w};
                        epi_store(q, i, k.tn * BN + c4 * 4, v, 4);
                    }
                    if (etid == 0) q.counters[k.tile] = 0;
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host

namespace {

struct Plan {
    std::vector<int> order;    // job indices in launch order
    std::vector<int> ksplit;   // per job
    std::vector<int> tiles;    // per job
    std::vector<int> k_tiles;  // per job
};

int tiles_of(const TcJob &j) {
    int tm = (int)ceil_div(j.M, BM), tn = (int)ceil_div(j.N, BN);
    return j.syrk ? tn * (tn + 1) / 2 : tm * tn;
}

Plan make_plan(const TcJob *jobs, int n) {
    Plan p;
    p.ksplit.resize(n);
    p.tiles.resize(n);
    p.k_tiles.resize(n);
    double total = 0.0;
    for (int i = 0; i < n; ++i) {
        p.tiles[i] = tiles_of(jobs[i]);
        p.k_tiles[i] = (int)ceil_div(jobs[i].K, BK);
        total += (double)p.tiles[i] * p.k_tiles[i];
    }
    const int sms = device_sm_count();
    // aim for ~4 work items per SM, at least 8 K tiles (512 rows) per item
    double target = std::max(8.0, total / (sms * 4.0));
    for (int i = 0; i < n; ++i) {
        int ks = (int)std::ceil(p.k_tiles[i] / target);
        ks = std::max(1, std::min(ks, std::min(p.k_tiles[i], 256)));
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

void take_buffers(const Plan &p, const TcJob *jobs, int n, Arena &ws, std::vector<float *> &part,
                  std::vector<int *> &cnt, int **cnt_base, size_t *cnt_count) {
    part.assign(n, nullptr);
    cnt.assign(n, nullptr);
    size_t ncnt = 0;
    for (int i = 0; i < n; ++i)
        if (p.ksplit[i] > 1) ncnt += p.tiles[i];
    int *cb = ws.take<int>(std::max<size_t>(ncnt, 1));
    size_t off = 0;
    for (int i = 0; i < n; ++i) {
        if (p.ksplit[i] > 1) {
            part[i] = ws.take<float>((size_t)p.tiles[i] * p.ksplit[i] * BM * BN);
            cnt[i] = cb ? cb + off : nullptr;
            off += p.tiles[i];
        }
    }
    *cnt_base = cb;
    *cnt_count = ncnt;
    (void)jobs;
}

bool make_map(CUtensorMap *m, const uint16_t *ptr, long long ld, int rows, int cols, int mn) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {64u, mn ? 64u : 128u};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void *)ptr, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

size_t tc_workspace_bytes(const TcJob *jobs, int njobs) {
    if (njobs <= 0) return 0;
    Plan p = make_plan(jobs, njobs);
    Arena a;
    std::vector<float *> part;
    std::vector<int *> cnt;
    int *cb;
    size_t nc;
    take_buffers(p, jobs, njobs, a, part, cnt, &cb, &nc);
    return a.used;
}

kfac_status tc_run(const TcJob *jobs, int njobs, Arena &ws, int *err, cudaStream_t st) {
    if (njobs <= 0) return KFAC_OK;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return KFAC_ERR_CUDA;

    Plan p = make_plan(jobs, njobs);
    std::vector<float *> part;
    std::vector<int *> cnt;
    int *cnt_base;
    size_t ncnt;
    take_buffers(p, jobs, njobs, ws, part, cnt, &cnt_base, &ncnt);
    if (!ws.fits()) return KFAC_ERR_WORKSPACE;
    if (ncnt) KFAC_CUDA_TRY(cudaMemsetAsync(cnt_base, 0, ncnt * sizeof(int), st));

    const int sms = device_sm_count();
    std::unique_ptr<TcParams> P(new TcParams);
    size_t pos = 0;
    while (pos < p.order.size()) {
        std::memset(P.get(), 0, sizeof(TcParams));
        int nmaps = 0, nprob = 0, work = 0;
        while (pos < p.order.size() && nprob < MAX_PROBS && nmaps + 2 <= MAX_MAPS) {
            const int ji = p.order[pos];
            const TcJob &j = jobs[ji];
            TcProb &q = P->prob[nprob];
            q.map_a = nmaps;
            if (!make_map(&P->maps[nmaps++], j.a, j.lda, j.a_rows, j.a_cols, j.a_mn)) return KFAC_ERR_CUDA;
            if (j.syrk) {
                q.map_b = q.map_a;
            } else {
                q.map_b = nmaps;
                if (!make_map(&P->maps[nmaps++], j.b, j.ldb, j.b_rows, j.b_cols, j.b_mn)) return KFAC_ERR_CUDA;
            }
            q.a_mn = j.a_mn;
            q.b_mn = j.syrk ? j.a_mn : j.b_mn;
            q.M = j.M;
            q.N = j.N;
            q.k_tiles = p.k_tiles[ji];
            q.tiles_n = (int)ceil_div(j.N, BN);
            q.syrk = j.syrk;
            q.ksplit = p.ksplit[ji];
            q.work_begin = work;
            q.epi = j.epi;
            q.alpha = j.alpha;
            q.beta = j.beta;
            q.C = j.C;
            q.ldc = j.ldc;
            q.Cb = j.Cb;
            q.ldcb = j.ldcb;
            q.partial = part[ji];
            q.counters = cnt[ji];
            work += p.tiles[ji] * p.ksplit[ji];
            ++nprob;
            ++pos;
        }
        P->nprob = nprob;
        P->total_work = work;
        P->error = err;
        int grid = std::min(work, sms);
        tc_gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(*P);
        KFAC_LAUNCH_CHECK();
    }
    return KFAC_OK;
}

}  // namespace kfac
