// api.cu -- the C ABI of libkfac_gb300 (declared in include/kfac.h):
// argument validation, workspace planning and dispatch to the kernels.
//
// Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
// Kronecker-Factored Approximate Curvature for Deep Convolutional Neural
// Networks", section 3.2 (Eq. 5-7) and section 1 (diagonal BatchNorm Fisher).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <vector>

#include "internal.h"

static_assert(kfac::ERR_TIMEOUT_FULL == KFAC_ERRW_TIMEOUT_OPERAND && kfac::ERR_TIMEOUT_EMPTY == KFAC_ERRW_TIMEOUT_STAGE &&
                  kfac::ERR_TIMEOUT_ACC == KFAC_ERRW_TIMEOUT_ACCUM && kfac::ERR_TIMEOUT_DRAIN == KFAC_ERRW_TIMEOUT_DRAIN &&
                  kfac::ERR_NONFINITE == KFAC_ERRW_NONFINITE,
              "device error word bits match the public header");

namespace kfac {

static std::atomic<long long> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// Optional per-kernel timing: a pool of event pairs, one pair per launch
// while enabled (diagnostic; off by default).
namespace {
constexpr int TIMING_MAX = 65536;
struct TimingRec {
    int kind;
    cudaEvent_t start, stop;
    unsigned long long stream;  // the launch stream's handle (identifies the stream, nothing more)
};
std::mutex g_tmu;
bool g_timing = false;
std::vector<TimingRec> g_recs;      // in use
std::vector<TimingRec> g_free;      // recycled event pairs
}  // namespace

namespace {
// An event record on `st`; during stream capture an external event node of
// the graph, which records the event each time the graph runs.
void timing_record(cudaEvent_t e, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
    else
        cudaEventRecord(e, st);
}
}  // namespace

int timing_begin(int kind, cudaStream_t st) {
    if (!g_timing) return -1;
    std::lock_guard<std::mutex> lock(g_tmu);
    if (!g_timing || (int)g_recs.size() >= TIMING_MAX) return -1;
    TimingRec r{kind, nullptr, nullptr, (unsigned long long)(uintptr_t)st};
    if (!g_free.empty()) {
        r.start = g_free.back().start;
        r.stop = g_free.back().stop;
        g_free.pop_back();
    } else if (cudaEventCreate(&r.start) != cudaSuccess || cudaEventCreate(&r.stop) != cudaSuccess) {
        return -1;
    }
    timing_record(r.start, st);
    g_recs.push_back(r);
    return (int)g_recs.size() - 1;
}

void timing_end(int slot, cudaStream_t st) {
    if (slot < 0) return;
    std::lock_guard<std::mutex> lock(g_tmu);
    if (slot < (int)g_recs.size()) timing_record(g_recs[slot].stop, st);
}

namespace {
thread_local bool t_pdl = true;
}  // namespace
bool pdl_enabled() { return t_pdl; }
PdlScope::PdlScope(bool on) : prev(t_pdl) { t_pdl = on; }
PdlScope::~PdlScope() { t_pdl = prev; }

int device_sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

EncodeTiledFn encode_tiled_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    });
    return fn;
}

EncodeIm2colFn encode_im2col_fn() {
    static std::once_flag once;
    static EncodeIm2colFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeIm2colFn)p;
    });
    return fn;
}

// Every operand must be memory of the current device (or managed memory):
// host memory or another GPU's memory is rejected before anything runs.
bool on_this_device(const void *p) {
    if (!p) return true;  // (null pointers are checked where they are not allowed)
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of an unknown pointer
        return false;
    }
    if (a.type == cudaMemoryTypeManaged) return true;
    int dev = -1;
    if (a.type != cudaMemoryTypeDevice || cudaGetDevice(&dev) != cudaSuccess) return false;
    return a.device == dev;
}

bool all_on_this_device(std::initializer_list<const void *> ps) {
    for (const void *p : ps)
        if (!on_this_device(p)) return false;
    return true;
}

namespace {

struct FactorGeom {
    int ho, wo;
    long long M;
    int dcore, d;
    bool direct;  // bf16 source usable as the patch matrix itself
};

bool geom_of(const kfac_factor_desc &d, FactorGeom &g) {
    g.ho = (d.h + 2 * d.pad_h - d.kh) / d.stride_h + 1;
    g.wo = (d.w + 2 * d.pad_w - d.kw) / d.stride_w + 1;
    if (d.h + 2 * d.pad_h < d.kh || d.w + 2 * d.pad_w < d.kw || g.ho < 1 || g.wo < 1) return false;
    g.M = (long long)d.n * g.ho * g.wo;
    g.dcore = d.kh * d.kw * d.c;
    g.d = g.dcore + (d.append_one ? 1 : 0);
    g.direct = d.dtype != KFAC_F32 && d.kh == 1 && d.kw == 1 && d.stride_h == 1 &&
               d.stride_w == 1 && d.pad_h == 0 && d.pad_w == 0 && d.c % 8 == 0 &&
               ((uintptr_t)d.x % 16) == 0;
    return true;
}

kfac_status validate_factor(const kfac_factor_desc *descs, int count, std::vector<FactorGeom> &geo) {
    if (count < 0 || (count > 0 && !descs)) return KFAC_ERR_INVALID;
    geo.resize(count);
    for (int i = 0; i < count; ++i) {
        const kfac_factor_desc &d = descs[i];
        if (!d.x || !d.F) return KFAC_ERR_INVALID;
        if (d.dtype != KFAC_BF16 && d.dtype != KFAC_F32 && d.dtype != KFAC_F16) return KFAC_ERR_INVALID;
        if (d.layout != KFAC_LAYOUT_FULL && d.layout != KFAC_LAYOUT_PACKED_UPPER) return KFAC_ERR_INVALID;
        if (d.n < 1 || d.h < 1 || d.w < 1 || d.c < 1 || d.kh < 1 || d.kw < 1 || d.stride_h < 1 ||
            d.stride_w < 1 || d.pad_h < 0 || d.pad_w < 0)
            return KFAC_ERR_INVALID;
        if (!std::isfinite(d.alpha) || !std::isfinite(d.beta)) return KFAC_ERR_INVALID;
        if (!geom_of(d, geo[i])) return KFAC_ERR_INVALID;
        if (d.layout == KFAC_LAYOUT_FULL && d.ldf < geo[i].d) return KFAC_ERR_INVALID;
        if (geo[i].d > 65536 || geo[i].M >= (1LL << 31)) return KFAC_ERR_UNSUPPORTED;
        // a materialised patch matrix is indexed with 32-bit element counts
        if (!geo[i].direct && geo[i].M * (long long)(geo[i].d + 8) >= (1LL << 31)) return KFAC_ERR_UNSUPPORTED;
    }
    return KFAC_OK;
}

// Everything the factor update enqueues, laid out in one arena.
struct FactorPlan {
    std::vector<Im2colJob> im16, imh, im32;  // bf16, fp16, fp32 patch matrices
    std::vector<TcJob> tc;
    std::vector<SgJob> sg;
    std::vector<ColsumJob> cs;
    float *cs_partial = nullptr;
    int *err = nullptr;
    char *tc_ws = nullptr;
    size_t tc_bytes = 0;
    std::vector<CUtensorMap> maps;
    CUtensorMap *dev_maps = nullptr;
};

// Lays out the workspace (error word, tensor maps, patch matrices, engine
// scratch) and the jobs; tensor maps are encoded only when `encode` is set
// (the size query runs without real pointers).
kfac_status plan_factor(const kfac_factor_desc *descs, int count, const std::vector<FactorGeom> &geo,
                        Arena &ws, FactorPlan &p, bool encode) {
    p.err = ws.take<int>(64);
    int n16 = 0;
    for (int i = 0; i < count; ++i) n16 += descs[i].dtype != KFAC_F32;
    p.dev_maps = ws.take<CUtensorMap>(std::max(n16, 1));
    for (int i = 0; i < count; ++i) {
        const kfac_factor_desc &d = descs[i];
        const FactorGeom &g = geo[i];
        const bool packed = d.layout == KFAC_LAYOUT_PACKED_UPPER;
        const bool f16 = d.dtype == KFAC_F16;
        if (d.dtype == KFAC_F32) {
            // fp32 path: explicit patches (with the ones column) + CUDA-core SYRK
            const long long ldp = g.d;
            float *P = ws.take<float>((size_t)g.M * ldp);
            p.im32.push_back(Im2colJob{d.x, d.n, d.h, d.w, d.c, d.kh, d.kw, d.stride_h, d.stride_w,
                                       d.pad_h, d.pad_w, g.ho, g.wo, d.append_one, P, ldp});
            p.sg.push_back(SgJob{P, ldp, 1, P, ldp, 0, d.F, d.ldf, nullptr, 0, g.d, g.d, (int)g.M,
                                 d.alpha, d.beta, 1, nullptr, 0, 0.f, packed ? g.d : 0});
            continue;
        }
        // a convolution whose channels fill 64-wide taps is read straight
        // from its input through an im2col tensor map (no patch matrix)
        const bool implicit = !g.direct && !d.append_one && d.c % 64 == 0 && d.kh == d.kw &&
                              d.stride_h == d.stride_w && d.pad_h == d.pad_w && d.stride_h <= 8 &&
                              d.pad_h <= 127 && d.pad_h - (d.kh - 1) >= -128 && d.kh <= 255 &&
                              ((uintptr_t)d.x % 16) == 0;
        if (implicit) {
            TcJob j{};
            j.map_a = j.map_b = (int)p.maps.size();
            p.maps.emplace_back();
            if (encode &&
                !tc_make_im2col_map(&p.maps.back(), d.x, d.n, d.h, d.w, d.c, d.kh, d.stride_h, d.pad_h, f16))
                return KFAC_ERR_CUDA;
            j.a_mn = j.b_mn = 1;
            j.M = g.dcore; j.N = g.dcore; j.K = (int)g.M;
            j.syrk = 1;
            j.epi = TC_EPI_ACCUM;
            j.alpha = d.alpha; j.beta = d.beta;
            j.C = d.F; j.ldc = d.ldf;
            j.im2col = 1;
            j.im_c = d.c; j.im_k = d.kh; j.im_stride = d.stride_h; j.im_pad = d.pad_h;
            j.im_wo = g.wo; j.im_howo = g.ho * g.wo;
            j.f16 = f16;
            j.packed = packed; j.packed_d = g.d;
            j.dyn = 1;  // problems of very different sizes: hand the work items out dynamically
            p.tc.push_back(j);
            continue;
        }
        const uint16_t *src;
        long long lds;
        if (g.direct) {
            src = (const uint16_t *)d.x;
            lds = d.c;
        } else {
            lds = (g.dcore + 7) / 8 * 8;
            uint16_t *P = ws.take<uint16_t>((size_t)g.M * lds);
            (f16 ? p.imh : p.im16).push_back(Im2colJob{d.x, d.n, d.h, d.w, d.c, d.kh, d.kw, d.stride_h,
                                                        d.stride_w, d.pad_h, d.pad_w, g.ho, g.wo, 0, P, lds});
            src = P;
        }
        TcJob j{};
        j.map_a = j.map_b = (int)p.maps.size();
        p.maps.emplace_back();
        if (encode && !tc_make_map(&p.maps.back(), TC_KIND_BF16, src, lds, (int)g.M, g.dcore, 0, f16))
            return KFAC_ERR_CUDA;
        j.a_mn = j.b_mn = 1;
        j.M = g.dcore; j.N = g.dcore; j.K = (int)g.M;
        j.syrk = 1;
        j.epi = TC_EPI_ACCUM;
        j.alpha = d.alpha; j.beta = d.beta;
        j.C = d.F; j.ldc = d.ldf;
        j.f16 = f16;
        j.packed = packed; j.packed_d = g.d;
        j.dyn = 1;  // problems of very different sizes: hand the work items out dynamically
        p.tc.push_back(j);
        if (d.append_one) {
            // bias row/column: needs the source rows [M][c]; an FC layer has
            // h = w = kh = kw = 1 so the source is x itself
            if (!(d.kh == 1 && d.kw == 1 && d.h == 1 && d.w == 1)) return KFAC_ERR_UNSUPPORTED;
            p.cs.push_back(ColsumJob{(const uint16_t *)d.x, g.M, d.c, d.F, d.ldf, d.alpha, d.beta, f16, packed});
        }
    }
    p.cs_partial = ws.take<float>(std::max<size_t>(colsum_partial_floats(p.cs.data(), (int)p.cs.size()), 1));
    p.tc_bytes = tc_workspace_bytes(p.tc.data(), (int)p.tc.size(), TC_KIND_BF16);
    p.tc_ws = ws.take<char>(p.tc_bytes);
    return KFAC_OK;
}

}  // namespace
}  // namespace kfac

using namespace kfac;

extern "C" const char *kfac_status_string(int status) {
    switch (status) {
        case KFAC_OK: return "KFAC_OK";
        case KFAC_ERR_INVALID: return "KFAC_ERR_INVALID: invalid argument";
        case KFAC_ERR_UNSUPPORTED: return "KFAC_ERR_UNSUPPORTED: valid but not supported";
        case KFAC_ERR_NOT_PD: return "KFAC_ERR_NOT_PD: matrix not positive definite";
        case KFAC_ERR_CUDA: return "KFAC_ERR_CUDA: CUDA launch or runtime error";
        case KFAC_ERR_WORKSPACE: return "KFAC_ERR_WORKSPACE: workspace missing or too small";
        default: return "unknown kfac_status";
    }
}

extern "C" int kfac_version(void) { return 100; }

extern "C" long long kfac_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int kfac_timing_enable(int on) {
    std::lock_guard<std::mutex> lock(g_tmu);
    const int was = g_timing ? 1 : 0;
    g_timing = on != 0;
    return was;
}

extern "C" const char *kfac_timing_kind_name(int k) {
    static const char *names[KK_COUNT] = {"tc_gemm_bf16", "tc_gemm_tf32x3", "inv_diag", "inv_prep",
                                          "damping", "im2col", "colsum", "sgemm_f32", "bn_fisher",
                                          "map_copy"};
    return (k >= 0 && k < KK_COUNT) ? names[k] : "";
}

extern "C" int kfac_timing_read(double *ms, long long *launches, int n) {
    std::lock_guard<std::mutex> lock(g_tmu);
    for (int k = 0; k < n; ++k) {
        if (ms) ms[k] = 0.0;
        if (launches) launches[k] = 0;
    }
    int status = KFAC_OK;
    for (TimingRec &r : g_recs) {
        float t = 0.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
            status = KFAC_ERR_CUDA;
        if (r.kind < n) {
            if (ms) ms[r.kind] += t;
            if (launches) launches[r.kind] += 1;
        }
        g_free.push_back(r);
    }
    g_recs.clear();
    return status;
}

extern "C" int kfac_timing_read_launches(double *start_ms, double *dur_ms, int *kind, unsigned long long *stream,
                                         int n) {
    std::lock_guard<std::mutex> lock(g_tmu);
    int count = 0;
    bool failed = false;
    for (TimingRec &r : g_recs) {
        float t = 0.f, t0 = 0.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess ||
            cudaEventElapsedTime(&t0, g_recs.front().start, r.start) != cudaSuccess)
            failed = true;
        if (count < n) {
            if (start_ms) start_ms[count] = t0;
            if (dur_ms) dur_ms[count] = t;
            if (kind) kind[count] = r.kind;
            if (stream) stream[count] = r.stream;
        }
        ++count;
        g_free.push_back(r);
    }
    g_recs.clear();
    return failed ? -1 : count;
}

// ------------------------------------------------------------ factor update

extern "C" size_t kfac_factor_update_workspace_size(const kfac_factor_desc *descs, int count) {
    std::vector<FactorGeom> geo;
    if (validate_factor(descs, count, geo) != KFAC_OK) return 0;
    Arena a;
    FactorPlan p;
    if (plan_factor(descs, count, geo, a, p, false) != KFAC_OK) return 0;
    return a.used;
}

extern "C" kfac_status kfac_factor_update(const kfac_factor_desc *descs, int count, void *workspace,
                                          size_t workspace_bytes, void *stream) {
    std::vector<FactorGeom> geo;
    kfac_status s = validate_factor(descs, count, geo);
    if (s != KFAC_OK) return s;
    if (count == 0) return KFAC_OK;
    if (!workspace || ((uintptr_t)workspace % 256) != 0) return KFAC_ERR_WORKSPACE;
    Arena ws(workspace, workspace_bytes);
    FactorPlan p;
    if ((s = plan_factor(descs, count, geo, ws, p, false)) != KFAC_OK) return s;
    if (!ws.fits()) return KFAC_ERR_WORKSPACE;
    for (int i = 0; i < count; ++i)
        if (!all_on_this_device({descs[i].x, descs[i].F})) return KFAC_ERR_INVALID;
    ws = Arena(workspace, workspace_bytes);
    p = FactorPlan();
    if ((s = plan_factor(descs, count, geo, ws, p, true)) != KFAC_OK) return s;
    if (!ws.fits()) return KFAC_ERR_WORKSPACE;
    Arena tail(p.tc_ws, p.tc_bytes);
    cudaStream_t st = (cudaStream_t)stream;
    KFAC_CUDA_TRY(cudaMemsetAsync(p.err, 0, sizeof(int), st));
    if (!p.im16.empty() && (s = im2col_run(p.im16.data(), (int)p.im16.size(), KFAC_BF16, st)) != KFAC_OK)
        return s;
    if (!p.imh.empty() && (s = im2col_run(p.imh.data(), (int)p.imh.size(), KFAC_F16, st)) != KFAC_OK)
        return s;
    if (!p.im32.empty() && (s = im2col_run(p.im32.data(), (int)p.im32.size(), KFAC_F32, st)) != KFAC_OK)
        return s;
    if (!p.tc.empty()) {
        if ((s = tc_upload_maps(p.maps.data(), (int)p.maps.size(), p.dev_maps, st)) != KFAC_OK) return s;
        if ((s = tc_run(p.tc.data(), (int)p.tc.size(), TC_KIND_BF16, p.dev_maps, tail, p.err, st)) != KFAC_OK)
            return s;
    }
    if (!p.sg.empty() && (s = sg_run(p.sg.data(), (int)p.sg.size(), p.err, st)) != KFAC_OK) return s;
    if (!p.cs.empty() && (s = colsum_run(p.cs.data(), (int)p.cs.size(), p.cs_partial, st)) != KFAC_OK) return s;
    return KFAC_OK;
}

// ------------------------------------------------------------ damp + invert

namespace {

kfac_status validate_invert(const kfac_invert_desc *descs, int count, float gamma) {
    if (count < 0 || (count > 0 && !descs) || !(gamma >= 0.f) || !std::isfinite(gamma))
        return KFAC_ERR_INVALID;
    for (int i = 0; i < count; ++i) {
        const kfac_invert_desc &d = descs[i];
        if (!d.A || !d.G || !d.A_inv || !d.G_inv) return KFAC_ERR_INVALID;
        const bool pa = d.layout_A == KFAC_LAYOUT_PACKED_UPPER, pg = d.layout_G == KFAC_LAYOUT_PACKED_UPPER;
        if ((!pa && d.layout_A != KFAC_LAYOUT_FULL) || (!pg && d.layout_G != KFAC_LAYOUT_FULL) ||
            (d.copy_dtype != KFAC_BF16 && d.copy_dtype != KFAC_F16))
            return KFAC_ERR_INVALID;
        if (d.dA < 1 || d.dG < 1 || (!pa && d.lda < d.dA) || (!pg && d.ldg < d.dG) || d.ld_ainv < d.dA ||
            d.ld_ginv < d.dG)
            return KFAC_ERR_INVALID;
        if ((d.A_inv_bf16 && d.ld_ainv_bf16 < d.dA) || (d.G_inv_bf16 && d.ld_ginv_bf16 < d.dG))
            return KFAC_ERR_INVALID;
        if (d.dA > 16384 || d.dG > 16384) return KFAC_ERR_UNSUPPORTED;
        if ((d.A_inv_bf16 && (d.ld_ainv_bf16 % 8 || (uintptr_t)d.A_inv_bf16 % 16)) ||
            (d.G_inv_bf16 && (d.ld_ginv_bf16 % 8 || (uintptr_t)d.G_inv_bf16 % 16)))
            return KFAC_ERR_UNSUPPORTED;
    }
    return KFAC_OK;
}

std::vector<InvMatrix> inv_mats(const kfac_invert_desc *descs, int count) {
    std::vector<InvMatrix> m(2 * count);
    for (int i = 0; i < count; ++i) {
        const kfac_invert_desc &d = descs[i];
        const int h = d.copy_dtype == KFAC_F16;
        m[2 * i] = InvMatrix{d.A, d.lda, d.dA, d.A_inv, d.ld_ainv, d.A_inv_bf16, d.ld_ainv_bf16,
                             d.layout_A == KFAC_LAYOUT_PACKED_UPPER, h};
        m[2 * i + 1] = InvMatrix{d.G, d.ldg, d.dG, d.G_inv, d.ld_ginv, d.G_inv_bf16, d.ld_ginv_bf16,
                                 d.layout_G == KFAC_LAYOUT_PACKED_UPPER, h};
    }
    return m;
}

}  // namespace

extern "C" size_t kfac_damp_invert_workspace_size(const kfac_invert_desc *descs, int count) {
    if (validate_invert(descs, count, 0.f) != KFAC_OK) return 0;
    std::vector<InvMatrix> m = inv_mats(descs, count);
    Arena a;
    a.take<char>(inv_workspace_bytes(m.data(), (int)m.size()));  // starts with the error word
    a.take<float>(2 * (size_t)count);   // damping values
    a.take<int>(2 * (size_t)count);     // info
    return a.used;
}

extern "C" kfac_status kfac_damp_invert(const kfac_invert_desc *descs, int count, float gamma,
                                        int pi_split, int32_t *info, float *damp, void *workspace,
                                        size_t workspace_bytes, void *stream) {
    kfac_status s = validate_invert(descs, count, gamma);
    if (s != KFAC_OK) return s;
    if (count == 0) return KFAC_OK;
    if (!workspace || ((uintptr_t)workspace % 256) != 0) return KFAC_ERR_WORKSPACE;
    std::vector<InvMatrix> m = inv_mats(descs, count);
    // layout (the same takes as kfac_damp_invert_workspace_size): the
    // inversion's own workspace first (its first int32 is the error word),
    // then the damping values and info used when the caller passes none
    const size_t inv_bytes = inv_workspace_bytes(m.data(), (int)m.size());
    Arena ws(workspace, workspace_bytes);
    char *inv_ws = ws.take<char>(inv_bytes);
    float *dmp = ws.take<float>(2 * (size_t)count);
    int *inf = ws.take<int>(2 * (size_t)count);
    if (!ws.fits()) return KFAC_ERR_WORKSPACE;
    if (damp) dmp = damp;
    if (info) inf = info;
    for (int i = 0; i < count; ++i) {
        const kfac_invert_desc &d = descs[i];
        if (!all_on_this_device({d.A, d.G, d.A_inv, d.G_inv, d.A_inv_bf16, d.G_inv_bf16, info, damp}))
            return KFAC_ERR_INVALID;
    }
    cudaStream_t st = (cudaStream_t)stream;
    KFAC_CUDA_TRY(cudaMemsetAsync(inf, 0, 2 * (size_t)count * sizeof(int), st));
    if ((s = damping_run(m.data(), count, gamma, pi_split, dmp, st)) != KFAC_OK) return s;
    Arena inv_arena(inv_ws, inv_bytes);
    return inv_run(m.data(), (int)m.size(), dmp, inf, inv_arena, st);
}

// ------------------------------------------------------------ precondition

namespace {

kfac_status validate_precond(const kfac_precond_desc *descs, int count, int dtype) {
    if (count < 0 || (count > 0 && !descs)) return KFAC_ERR_INVALID;
    if (dtype != KFAC_BF16 && dtype != KFAC_F32 && dtype != KFAC_F16) return KFAC_ERR_INVALID;
    for (int i = 0; i < count; ++i) {
        const kfac_precond_desc &d = descs[i];
        if (!d.G_inv || !d.A_inv || !d.grad || (!d.out && !d.w)) return KFAC_ERR_INVALID;
        if (d.dG < 1 || d.dA < 1 || d.ld_ginv < d.dG || d.ld_ainv < d.dA || d.ld_grad < d.dA ||
            (d.out && d.ld_out < d.dA) || (d.w && d.ld_w < d.dA))
            return KFAC_ERR_INVALID;
        if (d.dG > 65536 || d.dA > 65536) return KFAC_ERR_UNSUPPORTED;
        if (dtype != KFAC_F32 &&
            (d.ld_ginv % 8 || d.ld_ainv % 8 || d.ld_grad % 8 || (uintptr_t)d.G_inv % 16 ||
             (uintptr_t)d.A_inv % 16 || (uintptr_t)d.grad % 16))
            return KFAC_ERR_UNSUPPORTED;
    }
    return KFAC_OK;
}

struct PrecondPlan {
    std::vector<TcJob> g1, g2;
    std::vector<SgJob> s1, s2;
    int *err = nullptr;
    char *tc_ws = nullptr;
    size_t tc_bytes = 0;
    std::vector<CUtensorMap> maps;
    CUtensorMap *dev_maps = nullptr;
};

kfac_status plan_precond(const kfac_precond_desc *descs, int count, int dtype, Arena &ws, PrecondPlan &p,
                         bool encode) {
    p.err = ws.take<int>(64);
    const bool f16 = dtype == KFAC_F16;
    if (dtype != KFAC_F32) p.dev_maps = ws.take<CUtensorMap>(4 * (size_t)count);
    auto map = [&](const void *ptr, long long ld, int rows, int cols) {
        p.maps.emplace_back();
        if (encode && !tc_make_map(&p.maps.back(), TC_KIND_BF16, ptr, ld, rows, cols, 0, f16)) return -1;
        return (int)p.maps.size() - 1;
    };
    for (int i = 0; i < count; ++i) {
        const kfac_precond_desc &d = descs[i];
        if (dtype != KFAC_F32) {
            const long long ldt = (d.dA + 63) / 64 * 64;  // T's rows on 128-byte boundaries
            uint16_t *T = ws.take<uint16_t>((size_t)d.dG * ldt);
            TcJob a{};  // T = grad * A_inv   (A_inv symmetric: its rows are the columns of B)
            a.map_a = map(d.grad, d.ld_grad, d.dG, d.dA);
            a.map_b = map(d.A_inv, d.ld_ainv, d.dA, d.dA);
            a.M = d.dG; a.N = d.dA; a.K = d.dA;
            a.epi = TC_EPI_STORE; a.alpha = 1.f; a.beta = 0.f;
            a.Cb = T; a.ldcb = ldt;
            a.f16 = f16; a.cb_f16 = f16;
            TcJob b{};  // out = G_inv * T   (T read MN-major)
            b.map_a = map(d.G_inv, d.ld_ginv, d.dG, d.dG);
            b.map_b = map(T, ldt, d.dG, d.dA);  // read MN-major (b_mn)
            b.b_mn = 1;
            b.M = d.dG; b.N = d.dA; b.K = d.dG;
            b.epi = TC_EPI_STORE; b.alpha = 1.f; b.beta = 0.f;
            b.f16 = f16;
            b.C = d.out; b.ldc = d.ld_out;
            b.W = d.w; b.ldw = d.ld_w; b.eta = d.eta;  // Eq. 8, fused into the epilogue
            if (a.map_a < 0 || a.map_b < 0 || b.map_a < 0 || b.map_b < 0) return KFAC_ERR_CUDA;
            p.g1.push_back(a);
            p.g2.push_back(b);
        } else {
            float *T = ws.take<float>((size_t)d.dG * d.dA);
            p.s1.push_back(SgJob{(const float *)d.grad, d.ld_grad, 0, (const float *)d.A_inv, d.ld_ainv, 0,
                                 T, d.dA, nullptr, 0, d.dG, d.dA, d.dA, 1.f, 0.f, 0});
            p.s2.push_back(SgJob{(const float *)d.G_inv, d.ld_ginv, 0, T, d.dA, 0, d.out, d.ld_out,
                                 nullptr, 0, d.dG, d.dA, d.dG, 1.f, 0.f, 0, d.w, d.ld_w, d.eta});
        }
    }
    size_t t1 = tc_workspace_bytes(p.g1.data(), (int)p.g1.size(), TC_KIND_BF16);
    size_t t2 = tc_workspace_bytes(p.g2.data(), (int)p.g2.size(), TC_KIND_BF16);
    p.tc_bytes = std::max(t1, t2);
    p.tc_ws = ws.take<char>(p.tc_bytes);
    return KFAC_OK;
}

}  // namespace

extern "C" size_t kfac_precondition_workspace_size(const kfac_precond_desc *descs, int count, int dtype) {
    if (validate_precond(descs, count, dtype) != KFAC_OK) return 0;
    Arena a;
    PrecondPlan p;
    if (plan_precond(descs, count, dtype, a, p, false) != KFAC_OK) return 0;
    return a.used;
}

extern "C" kfac_status kfac_precondition(const kfac_precond_desc *descs, int count, int dtype,
                                         void *workspace, size_t workspace_bytes, void *stream) {
    kfac_status s = validate_precond(descs, count, dtype);
    if (s != KFAC_OK) return s;
    if (count == 0) return KFAC_OK;
    if (!workspace || ((uintptr_t)workspace % 256) != 0) return KFAC_ERR_WORKSPACE;
    Arena ws(workspace, workspace_bytes);
    PrecondPlan p;
    if ((s = plan_precond(descs, count, dtype, ws, p, false)) != KFAC_OK) return s;
    if (!ws.fits()) return KFAC_ERR_WORKSPACE;
    for (int i = 0; i < count; ++i) {
        const kfac_precond_desc &d = descs[i];
        if (!all_on_this_device({d.G_inv, d.A_inv, d.grad, d.out, d.w})) return KFAC_ERR_INVALID;
    }
    ws = Arena(workspace, workspace_bytes);
    p = PrecondPlan();
    if ((s = plan_precond(descs, count, dtype, ws, p, true)) != KFAC_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    KFAC_CUDA_TRY(cudaMemsetAsync(p.err, 0, sizeof(int), st));  // the error word, for every dtype
    if (dtype != KFAC_F32) {
        if ((s = tc_upload_maps(p.maps.data(), (int)p.maps.size(), p.dev_maps, st)) != KFAC_OK) return s;
        Arena t_a(p.tc_ws, p.tc_bytes);
        if ((s = tc_run(p.g1.data(), (int)p.g1.size(), TC_KIND_BF16, p.dev_maps, t_a, p.err, st)) != KFAC_OK)
            return s;
        Arena t_b(p.tc_ws, p.tc_bytes);
        return tc_run(p.g2.data(), (int)p.g2.size(), TC_KIND_BF16, p.dev_maps, t_b, p.err, st);
    }
    if ((s = sg_run(p.s1.data(), (int)p.s1.size(), p.err, st)) != KFAC_OK) return s;
    return sg_run(p.s2.data(), (int)p.s2.size(), p.err, st);
}
