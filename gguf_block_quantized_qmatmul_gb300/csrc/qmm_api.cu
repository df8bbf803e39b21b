// qmm_api.cu -- the C ABI (include/qmm.h): argument checks, planning, launches.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "../../include/qmm.h"
#include "qmm_internal.h"

using namespace qmm;

namespace {

// Device error word [0] (timeouts of bounded waits) and, in [1], the log2 of
// the bounded waits' spin limit (0: the default of 2^31 SM clocks; lowered
// only by qmm_test_set_wait_limit).
__device__ unsigned g_qmm_err[2] = {0u, 0u};

constexpr int kMaxDev = 64;
struct DeviceInfo {
    std::atomic<unsigned*> err{nullptr};  // published last (release) once the sizes below are stored
    std::atomic<int> sm_count{0};
    std::atomic<int> smem_optin{0};
};
DeviceInfo g_dev[kMaxDev];

// Per-device constants: error-word address, SM count, opt-in shared memory.
// Host threads may race on a device's first call: each computes the same
// values, and every field is atomic.
cudaError_t device_info(unsigned** err, int* sms, int* smem, int* device = nullptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    DeviceInfo& di = g_dev[dev];
    unsigned* ep = di.err.load(std::memory_order_acquire);
    int n = 0, s = 0;
    if (ep) {
        n = di.sm_count.load(std::memory_order_relaxed);
        s = di.smem_optin.load(std::memory_order_relaxed);
    } else {
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_qmm_err)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&s, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
        ep = static_cast<unsigned*>(p);
        di.sm_count.store(n, std::memory_order_relaxed);
        di.smem_optin.store(s, std::memory_order_relaxed);
        di.err.store(ep, std::memory_order_release);
    }
    if (err) *err = ep;
    if (sms) *sms = n;
    if (smem) *smem = s;
    if (device) *device = dev;
    return cudaSuccess;
}

// Failure-test injection (qmm_test_inject): counts of calls still to fail.
std::atomic<int> g_inject_launch_failures{0};
std::atomic<int> g_inject_stalls{0};
std::atomic<int> g_inject_stall_stage{0};

// Takes one pending injection of a kind, if any.
bool take_injection(std::atomic<int>& pending) {
    int v = pending.load(std::memory_order_relaxed);
    while (v > 0)
        if (pending.compare_exchange_weak(v, v - 1, std::memory_order_relaxed)) return true;
    return false;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool valid_type(qmm_type t) {
    return t == QMM_Q8_0 || t == QMM_Q4_K || t == QMM_Q8_K || t == QMM_Q4_0 || t == QMM_Q5_0 || t == QMM_Q6_K;
}
// weight types: Q8_0, Q4_0, Q5_0 (with Q8_0 activations); Q4_K, Q6_K (with Q8K)
bool weight_type(qmm_type t) {
    return t == QMM_Q8_0 || t == QMM_Q4_K || t == QMM_Q4_0 || t == QMM_Q5_0 || t == QMM_Q6_K;
}
int internal_type(qmm_type t) {
    switch (t) {
        case QMM_Q8_0: return T_Q8_0;
        case QMM_Q4_K: return T_Q4_K;
        case QMM_Q8_K: return T_Q8_K;
        case QMM_Q4_0: return T_Q4_0;
        case QMM_Q5_0: return T_Q5_0;
        case QMM_Q6_K: return T_Q6_K;
        default: return T_F32;
    }
}

qmm_status check_shape(qmm_type t, int64_t rows, int64_t K) {
    if (rows < 0 || K < 0) return QMM_ERR_SHAPE;
    if (rows > INT32_MAX || K > INT32_MAX) return QMM_ERR_SHAPE;
    const int64_t bv = qmm_block_values(t);
    if (bv <= 0 || K % bv != 0) return QMM_ERR_SHAPE;
    return QMM_OK;
}

size_t round_up_sz(size_t v, size_t a) { return (v + a - 1) / a * a; }

size_t workspace_for(const StreamPlan& pl) {
    if (pl.p.kslices <= 1) return 0;
    return round_up_sz((size_t)pl.p.kslices * pl.p.M * pl.p.N * 4, 256) + (size_t)pl.p.mchunks * pl.p.ntiles * 4;
}

// The kernel a matmul call dispatches to and its plan.  Planning searches
// chunk sizes and K splits, so decisions are cached per host thread by
// (device, type, form, epilogue, M, N, K).
enum Kind { KIND_NONE, KIND_GEMV, KIND_DMMA, KIND_TC, KIND_TCX, KIND_STREAM };
struct Dispatch {
    Kind kind = KIND_NONE;
    GemvPlan gp;
    DmmaPlan dp;
    TcPlan tp;
    TcxPlan xp;
    StreamPlan sp;
    size_t workspace = 0;
    int launches = 0;
};

void plan_dispatch(int wt, int am, int epi, long long M, long long N, long long K, int sms, int smem, Dispatch& d) {
    d = Dispatch();
    // Q4_0, Q5_0, Q6_K above 16 rows go to the GEMMs only (K % 256 = 0), else to the streaming kernel
    const bool gemm_rows = M > kDecodeMaxM || wt == T_Q8_0 || wt == T_Q4_K;
    const bool code_f32 = wt == T_Q8_0 || wt == T_Q4_K || wt == T_Q6_K;  // the code GEMM's f32_act types
    if (am == A_INT8 && wt == T_Q8_0 && M <= kGemvMaxM && plan_gemv(wt, M, N, K, sms, smem, d.gp)) {  // decode: whole-row weight stream
        d.kind = KIND_GEMV;
        d.launches = 1;
    } else if (M <= kDmmaMaxM && plan_dmma(wt, am, M, N, K, sms, smem, d.dp, epi == E_Y)) {  // decode and small prefill on 16-row warp-MMA tiles
        d.kind = KIND_DMMA;
        d.workspace = d.dp.workspace;
        d.launches = 1 + (d.dp.ext_bytes ? 1 : 0) + (epi == E_Y && d.dp.p.kslices > 1 ? 1 : 0);
    } else if (epi == E_Y && am == A_F32 && code_f32 && M <= 64 && plan_tcx(wt, A_F32, M, N, K, sms, smem, d.xp)) {
        // Metal-form prefill up to 64 rows: exact f16 weight codes times two activation pieces on
        // tcgen05 (Q4_K 1.3-1.6x the three-pass GEMM there, Q8_0 1.1x; the three passes are
        // faster from 256 rows on)
        d.kind = KIND_TCX;
        d.workspace = d.xp.workspace;
        d.launches = wt == T_Q6_K ? 3 : 2;  // activation pieces, (Q6_K) repacked weights, GEMM
    } else if (epi == E_Y && am == A_F32 && gemm_rows && plan_tc(wt, M, N, K, sms, smem, d.tp)) {  // Metal-form prefill: tcgen05 GEMM
        d.kind = KIND_TC;
        d.workspace = d.tp.workspace;
        d.launches = 2;  // operand preparation, GEMM
    } else if (epi == E_Y && am == A_INT8 && gemm_rows && plan_tcx(wt, A_INT8, M, N, K, sms, smem, d.xp)) {
        // CPU-form prefill: exact integer block sums on tcgen05
        d.kind = KIND_TCX;
        d.workspace = d.xp.workspace;
        d.launches = wt == T_Q6_K ? 3 : 2;  // activation codes, (Q6_K) repacked weights, GEMM
    } else if (plan_stream(wt, am, epi, M, N, K, sms, smem, d.sp)) {
        d.kind = KIND_STREAM;
        d.workspace = epi == E_Y ? workspace_for(d.sp) : 0;
        d.launches = 1;
    }
}

struct CachedDispatch {
    bool used = false;
    int dev = -1, wt = 0, am = 0, epi = 0;
    long long M = 0, N = 0, K = 0;
    Dispatch d;
};
constexpr int kPlanCache = 16;
thread_local CachedDispatch t_plans[kPlanCache];
thread_local int t_plan_next = 0;

const Dispatch& get_dispatch(int dev, int wt, int am, int epi, long long M, long long N, long long K, int sms, int smem) {
    for (const CachedDispatch& c : t_plans)
        if (c.used && c.dev == dev && c.wt == wt && c.am == am && c.epi == epi && c.M == M && c.N == N && c.K == K) return c.d;
    CachedDispatch& c = t_plans[t_plan_next];
    t_plan_next = (t_plan_next + 1) % kPlanCache;
    c.used = true;
    c.dev = dev;
    c.wt = wt;
    c.am = am;
    c.epi = epi;
    c.M = M;
    c.N = N;
    c.K = K;
    plan_dispatch(wt, am, epi, M, N, K, sms, smem, c.d);
    return c.d;
}

qmm_status stream_call(qmm_type wtype, int am, int epi, const void* wq, const float* x, float* y, int32_t* sums,
                       int64_t M, int64_t N, int64_t K, void* ws, size_t ws_bytes, qmm_stream_t stream) {
    if (take_injection(g_inject_launch_failures)) return QMM_ERR_CUDA;  // test hook: no CUDA call made
    unsigned* err = nullptr;
    int sms = 0, smem = 0, dev = 0;
    if (device_info(&err, &sms, &smem, &dev) != cudaSuccess) return QMM_ERR_CUDA;
    const int wt = internal_type(wtype);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const Dispatch& d = get_dispatch(dev, wt, am, epi, M, N, K, sms, smem);
    if (d.kind == KIND_GEMV) {
        GemvPlan gp = d.gp;
        gp.p.wq = static_cast<const uint8_t*>(wq);
        gp.p.x = x;
        gp.p.y = y;
        gp.p.sums = sums;
        gp.p.err = err;
        const cudaError_t e = wt == T_Q8_0 ? launch_gemv_q8_0(epi, gp, smem, s) : launch_gemv_q4_k(epi, gp, smem, s);
        return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
    }
    if (d.kind == KIND_DMMA) {
        DmmaPlan dp = d.dp;
        dp.p.wq = static_cast<const uint8_t*>(wq);
        dp.p.x = x;
        dp.p.y = y;
        dp.p.sums = sums;
        dp.p.err = err;
        dp.p.stall_stage = take_injection(g_inject_stalls) ? g_inject_stall_stage.load(std::memory_order_relaxed) + 1 : 0;
        const bool split = epi == E_Y && dp.p.kslices > 1;
        if (split || dp.ext_bytes) {
            if (!ws || ws_bytes < dp.workspace) return QMM_ERR_WORKSPACE;
            if (split) dp.p.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + dp.ext_bytes);
        }
        if (dp.ext_bytes) {  // activations prepared once, fetched by every CTA
            dp.p.ext = static_cast<const uint8_t*>(ws);
            if (launch_dmma_prep(wt, am, dp, ws, s) != cudaSuccess) return QMM_ERR_CUDA;
        }
        if (launch_dmma(wt, am, epi, dp, smem, s) != cudaSuccess) return QMM_ERR_CUDA;
        if (split && launch_splitk_reduce(dp.p.partial, M * N, dp.p.kslices, y, s) != cudaSuccess) return QMM_ERR_CUDA;
        return QMM_OK;
    }
    if (d.kind == KIND_TC) {
        if (!ws || ws_bytes < d.tp.workspace) return QMM_ERR_WORKSPACE;
        TcPlan tp = d.tp;
        tp.p.err = err;
        return launch_tc(wt, tp, wq, x, ws, y, smem, s) == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
    }
    if (d.kind == KIND_TCX) {
        if (!ws || ws_bytes < d.xp.workspace) return QMM_ERR_WORKSPACE;
        TcxPlan xp = d.xp;
        xp.p.err = err;
        return launch_tcx(wt, xp, wq, x, ws, y, smem, s) == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
    }
    if (d.kind != KIND_STREAM) return QMM_ERR_SHAPE;
    StreamPlan pl = d.sp;
    pl.p.wq = static_cast<const uint8_t*>(wq);
    pl.p.x = x;
    pl.p.y = y;
    pl.p.sums = sums;
    pl.p.err = err;
    if (epi == E_Y && pl.p.kslices > 1) {
        const size_t need = workspace_for(pl);
        if (!ws || ws_bytes < need) return QMM_ERR_WORKSPACE;
        pl.p.partial = static_cast<float*>(ws);
        const size_t coff = round_up_sz((size_t)pl.p.kslices * pl.p.M * pl.p.N * 4, 256);
        pl.p.counters = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(ws) + coff);
        if (cudaMemsetAsync(pl.p.counters, 0, (size_t)pl.p.mchunks * pl.p.ntiles * 4, s) != cudaSuccess)
            return QMM_ERR_CUDA;
    }
    const cudaError_t e = wt == T_Q8_0   ? launch_stream_q8_0(am, epi, pl, smem, s)
                          : wt == T_Q4_K ? launch_stream_q4_k(am, epi, pl, smem, s)
                          : wt == T_Q4_0 ? launch_stream_q4_0(am, epi, pl, smem, s)
                          : wt == T_Q5_0 ? launch_stream_q5_0(am, epi, pl, smem, s)
                                         : launch_stream_q6_k(am, epi, pl, smem, s);
    return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

}  // namespace

extern "C" {

int64_t qmm_block_values(qmm_type t) {
    switch (t) {
        case QMM_F32: return 1;
        case QMM_Q8_0: return 32;
        case QMM_Q4_K: return 256;
        case QMM_Q8_K: return 256;
        case QMM_Q4_0: return 32;
        case QMM_Q5_0: return 32;
        case QMM_Q6_K: return 256;
        default: return 0;
    }
}

size_t qmm_block_bytes(qmm_type t) {
    switch (t) {
        case QMM_F32: return 4;
        case QMM_Q8_0: return 34;
        case QMM_Q4_K: return 144;
        case QMM_Q8_K: return 292;
        case QMM_Q4_0: return 18;
        case QMM_Q5_0: return 22;
        case QMM_Q6_K: return 210;
        default: return 0;
    }
}

size_t qmm_row_bytes(qmm_type t, int64_t K) {
    const int64_t bv = qmm_block_values(t);
    if (bv <= 0 || K < 0 || K % bv != 0) return 0;
    return (size_t)(K / bv) * qmm_block_bytes(t);
}

qmm_status qmm_quantize_weights(qmm_type wtype, const float* w, int64_t N, int64_t K, void* wq, qmm_stream_t stream) {
    if (!weight_type(wtype)) return QMM_ERR_TYPE;
    qmm_status st = check_shape(wtype, N, K);
    if (st != QMM_OK) return st;
    if (N == 0 || K == 0) return QMM_OK;
    if (!w || !wq) return QMM_ERR_NULL;
    if (!aligned(w, 16) || !aligned(wq, 16)) return QMM_ERR_ALIGN;
    const int t = internal_type(wtype);
    return launch_quantize(t, w, N, K, wq, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

qmm_status qmm_quantize_act(qmm_type atype, const float* x, int64_t M, int64_t K, void* xq, qmm_stream_t stream) {
    if (atype != QMM_Q8_0 && atype != QMM_Q8_K) return QMM_ERR_TYPE;
    qmm_status st = check_shape(atype, M, K);
    if (st != QMM_OK) return st;
    if (M == 0 || K == 0) return QMM_OK;
    if (!x || !xq) return QMM_ERR_NULL;
    if (!aligned(x, 16) || !aligned(xq, 16)) return QMM_ERR_ALIGN;
    const int t = atype == QMM_Q8_0 ? T_Q8_0 : T_Q8_K;
    return launch_quantize(t, x, M, K, xq, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

qmm_status qmm_dequantize(qmm_type t, const void* q, int64_t rows, int64_t K, float* out, qmm_stream_t stream) {
    if (!valid_type(t)) return QMM_ERR_TYPE;
    qmm_status st = check_shape(t, rows, K);
    if (st != QMM_OK) return st;
    if (rows == 0 || K == 0) return QMM_OK;
    if (!q || !out) return QMM_ERR_NULL;
    if (!aligned(q, 16) || !aligned(out, 16)) return QMM_ERR_ALIGN;
    const int tt = internal_type(t);
    return launch_dequantize(tt, q, rows, K, out, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? QMM_OK
                                                                                                          : QMM_ERR_CUDA;
}

}  // extern "C"

namespace {
// The dispatch of qmm_matmul for a shape, without launching anything:
// workspace bytes and the number of kernel launches (0 launches: invalid).
void dispatch_info(qmm_type wtype, qmm_act_mode mode, int64_t M, int64_t N, int64_t K, size_t* ws, int* launches) {
    *ws = 0;
    *launches = 0;
    if (!weight_type(wtype)) return;
    if (mode != QMM_INT8_ACT && mode != QMM_F32_ACT) return;
    if (check_shape(wtype, N, K) != QMM_OK || M <= 0 || M > INT32_MAX || N == 0 || K == 0) return;
    int sms = 0, smem = 0, dev = 0;
    if (device_info(nullptr, &sms, &smem, &dev) != cudaSuccess) return;
    const Dispatch& d = get_dispatch(dev, internal_type(wtype), mode == QMM_INT8_ACT ? A_INT8 : A_F32, E_Y,
                                     M, N, K, sms, smem);
    *ws = d.workspace;
    *launches = d.launches;
}
}  // namespace

extern "C" {

size_t qmm_matmul_workspace(qmm_type wtype, qmm_act_mode mode, int64_t M, int64_t N, int64_t K) {
    size_t ws;
    int n;
    dispatch_info(wtype, mode, M, N, K, &ws, &n);
    return ws;
}

int qmm_matmul_launches(qmm_type wtype, qmm_act_mode mode, int64_t M, int64_t N, int64_t K) {
    size_t ws;
    int n;
    dispatch_info(wtype, mode, M, N, K, &ws, &n);
    return n;
}

qmm_status qmm_matmul(qmm_type wtype, qmm_act_mode mode, const void* wq, const float* x, float* y, int64_t M,
                      int64_t N, int64_t K, void* workspace, size_t workspace_bytes, qmm_stream_t stream) {
    if (!weight_type(wtype)) return QMM_ERR_TYPE;
    if (mode != QMM_INT8_ACT && mode != QMM_F32_ACT) return QMM_ERR_TYPE;
    qmm_status st = check_shape(wtype, N, K);
    if (st != QMM_OK) return st;
    if (M < 0 || M > INT32_MAX) return QMM_ERR_SHAPE;
    if (M == 0 || N == 0) return QMM_OK;
    if (K == 0) return QMM_ERR_SHAPE;
    if (!wq || !x || !y) return QMM_ERR_NULL;
    if (!aligned(wq, 16) || !aligned(x, 16) || !aligned(y, 4)) return QMM_ERR_ALIGN;
    if (workspace && !aligned(workspace, 16)) return QMM_ERR_ALIGN;
    return stream_call(wtype, mode == QMM_INT8_ACT ? A_INT8 : A_F32, E_Y, wq, x, y, nullptr, M, N, K, workspace,
                       workspace_bytes, stream);
}

extern "C++" {
namespace {

// Both batch entry points: item i is get(i), a qmm_matmul_typed_desc.  Every
// item is checked before anything is launched; then one launch per kBatchMax
// live items, with the kernel of their one weight type when they share a
// 32-value type, else the kernel whose items carry their own types.
template <typename Get>
qmm_status batch_run(qmm_act_mode mode, int64_t count, bool have_items, Get get, qmm_stream_t stream) {
    if (mode != QMM_INT8_ACT && mode != QMM_F32_ACT) return QMM_ERR_TYPE;
    if (count < 0) return QMM_ERR_SHAPE;
    if (count == 0) return QMM_OK;
    if (!have_items) return QMM_ERR_NULL;
    int64_t live = 0;
    for (int64_t i = 0; i < count; ++i) {
        const qmm_matmul_typed_desc d = get(i);
        if (!weight_type(d.wtype)) return QMM_ERR_TYPE;
        if (d.M < 0 || d.N < 0 || d.K < 0 || d.N > INT32_MAX) return QMM_ERR_SHAPE;
        if (d.M == 0 || d.N == 0) continue;
        ++live;
        if (d.K == 0 || d.K % qmm_block_values(d.wtype) != 0 || d.M > QMM_BATCH_MAX_M || d.M * d.K > QMM_BATCH_MAX_MK)
            return QMM_ERR_SHAPE;
        if (!d.wq || !d.x || !d.y) return QMM_ERR_NULL;
        if (!aligned(d.wq, 16) || !aligned(d.x, 16) || !aligned(d.y, 4)) return QMM_ERR_ALIGN;
    }
    if (live == 0) return QMM_OK;
    unsigned* err = nullptr;
    int sms = 0, smem = 0;
    if (device_info(&err, &sms, &smem) != cudaSuccess) return QMM_ERR_CUDA;
    const int am = mode == QMM_INT8_ACT ? A_INT8 : A_F32;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    BatchParams p;  // ~16 KB: the item table travels in the launch parameters
    int64_t i = 0;
    while (i < count) {
        p.count = 0;
        p.total = 0;
        p.act_bytes = 0;
        p.err = err;
        int max_m = 1, kind = -1;
        for (; i < count && p.count < kBatchMax; ++i) {
            const qmm_matmul_typed_desc d = get(i);
            if (d.M == 0 || d.N == 0) continue;
            const int wt = internal_type(d.wtype);
            BatchItem& it = p.it[p.count++];
            it.wq = static_cast<const uint8_t*>(d.wq);
            it.x = d.x;
            it.y = d.y;
            it.M = (int)d.M;
            it.N = (int)d.N;
            it.K = (int)d.K;
            it.wt = wt;
            it.lpr = it.bpl = it.tr = 0;
            it.cpr = batch_row_cost(wt, am, (int)d.K);
            it.c0 = p.total;
            p.total += d.N * (int64_t)it.cpr;
            const int64_t ab = d.M * (d.K / unit_vals(wt)) * batch_act_unit(wt, am);
            if (ab > p.act_bytes) p.act_bytes = (int)ab;
            if (d.M > max_m) max_m = (int)d.M;
            kind = kind == -1 || kind == wt ? wt : T_MIX;
        }
        if (p.count == 0) break;
        if (!is_b32(kind)) kind = T_MIX;
        if (launch_batch(kind, am, p, max_m, sms, smem, s) != cudaSuccess) return QMM_ERR_CUDA;
    }
    return QMM_OK;
}

}  // namespace
}  // extern "C++"

qmm_status qmm_matmul_batch(qmm_type wtype, qmm_act_mode mode, const qmm_matmul_desc* items, int64_t count,
                            qmm_stream_t stream) {
    if (!weight_type(wtype)) return QMM_ERR_TYPE;
    return batch_run(mode, count, items != nullptr, [&](int64_t i) {
        const qmm_matmul_desc& d = items[i];
        return qmm_matmul_typed_desc{wtype, d.wq, d.x, d.y, d.M, d.N, d.K};
    }, stream);
}

qmm_status qmm_matmul_batch_typed(qmm_act_mode mode, const qmm_matmul_typed_desc* items, int64_t count,
                                  qmm_stream_t stream) {
    return batch_run(mode, count, items != nullptr, [&](int64_t i) { return items[i]; }, stream);
}

qmm_status qmm_block_sums(qmm_type wtype, const void* wq, const float* x, int64_t M, int64_t N, int64_t K,
                          int32_t* out, qmm_stream_t stream) {
    if (!weight_type(wtype)) return QMM_ERR_TYPE;
    qmm_status st = check_shape(wtype, N, K);
    if (st != QMM_OK) return st;
    if (M < 0 || M > INT32_MAX) return QMM_ERR_SHAPE;
    if (M == 0 || N == 0) return QMM_OK;
    if (K == 0) return QMM_ERR_SHAPE;
    if (!wq || !x || !out) return QMM_ERR_NULL;
    if (!aligned(wq, 16) || !aligned(x, 16) || !aligned(out, 4)) return QMM_ERR_ALIGN;
    return stream_call(wtype, A_INT8, E_SUMS, wq, x, nullptr, out, M, N, K, nullptr, 0, stream);
}

qmm_status qmm_test_inject(qmm_inject_kind kind, int count, int arg) {
    if (count < 0 || arg < 0) return QMM_ERR_SHAPE;
    switch (kind) {
        case QMM_INJECT_OFF:
            g_inject_launch_failures.store(0);
            g_inject_stalls.store(0);
            return QMM_OK;
        case QMM_INJECT_LAUNCH_FAILURE:
            g_inject_launch_failures.store(count);
            return QMM_OK;
        case QMM_INJECT_STALL:
            g_inject_stall_stage.store(arg);
            g_inject_stalls.store(count);
            return QMM_OK;
        default:
            return QMM_ERR_TYPE;
    }
}

qmm_status qmm_test_set_wait_limit(int log2_clocks) {
    if (log2_clocks != 0 && (log2_clocks < 16 || log2_clocks > 31)) return QMM_ERR_SHAPE;
    const unsigned v = (unsigned)log2_clocks;
    if (cudaMemcpyToSymbol(g_qmm_err, &v, sizeof(v), sizeof(unsigned)) != cudaSuccess) return QMM_ERR_CUDA;
    return QMM_OK;
}

qmm_status qmm_last_device_error(void) {
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_qmm_err, sizeof(v)) != cudaSuccess) return QMM_ERR_CUDA;
    if (v) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_qmm_err, &zero, sizeof(zero)) != cudaSuccess) return QMM_ERR_CUDA;
        return QMM_ERR_TIMEOUT;
    }
    return QMM_OK;
}

const char* qmm_status_string(qmm_status s) {
    switch (s) {
        case QMM_OK: return "ok";
        case QMM_ERR_NULL: return "a required pointer is NULL";
        case QMM_ERR_SHAPE: return "invalid shape: negative size or K not a multiple of the block size";
        case QMM_ERR_TYPE: return "type not valid for this call";
        case QMM_ERR_ALIGN: return "pointer misaligned (16 bytes for blocks, x and workspace; 4 for floats)";
        case QMM_ERR_WORKSPACE: return "workspace smaller than qmm_matmul_workspace()";
        case QMM_ERR_CUDA: return "CUDA runtime or launch error";
        case QMM_ERR_TIMEOUT: return "a device-side wait timed out";
        default: return "unknown status";
    }
}

}  // extern "C"
