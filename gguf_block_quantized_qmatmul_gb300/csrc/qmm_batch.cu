// qmm_batch.cu -- planning and launching of the batched-matmul kernel
// (qmm_batch.cuh); the launches of one weight type (Q8_0, Q4_0, Q5_0) are
// instantiated here, those whose items carry their own types (any mix,
// including Q4_K and Q6_K) in qmm_batch_mix.cu.
#include "qmm_internal.h"

namespace qmm {
namespace {

template <int WT>
cudaError_t go(int am, BatchParams& p, int mt, int grid, int smem_max, cudaStream_t s) {
    return am == A_INT8 ? batch_go_mt<WT, A_INT8>(p, mt, grid, smem_max, s)
                        : batch_go_mt<WT, A_F32>(p, mt, grid, smem_max, s);
}

// issue cost of one unit relative to a 32-value block: a 64-value piece of a
// super-block holds two blocks' values, and its 6-bit scales, mins and codes
// (and, for int8_act, the quad's exchanges) cost a little more
int unit_work(int wt) { return is_sb(wt) ? 3 : 1; }

}  // namespace

int batch_row_cost(int wt, int am, int K) {
    // time of 32 values at saturation, in units of about 10 fs (batches of one
    // type, M = 1, K = 1536 and 4096): the 32-value types with Q8_0 activations
    // and Q8_0 weights are bound by bytes, Q5_0 and Q4_0 by unpacking, so their
    // rows cost alike per value although their bytes differ by 1.5-1.9x
    int w;
    switch (wt) {
        case T_Q8_0: w = am == A_INT8 ? 28 : 36; break;
        case T_Q5_0: w = am == A_INT8 ? 29 : 34; break;
        case T_Q4_0: w = am == A_INT8 ? 22 : 29; break;
        case T_Q4_K: w = am == A_INT8 ? 21 : 30; break;
        default: w = am == A_INT8 ? 30 : 37; break;  // Q6_K
    }
    return K / 32 * w;
}

void plan_batch_item(int wt, int nu, long long rb, int am, int mt, int& lpr, int& bpl, int& tr) {
    // Lanes per row (lpr) and units per lane (bpl = ceil(nu / lpr)) for a row of
    // nu units of type wt (rb bytes), and rows per stage (tr).  int8_act on
    // super-blocks wants lane groups of a multiple of 4 lanes (a super-block's
    // four pieces on one quad of lanes).  A warp holds 32 / lpr lane groups of R
    // rows each; a stage is one pass of the 16 consumer warps over its rows, at
    // most kBatchStageCap bytes.  The cost of a pass is about 30 issue slots per
    // 32 values and row a lane takes, 12 per 32 values for the shared
    // activation loads, and the groups' reductions and bookkeeping; the plan
    // with the least cost per row wins.
    const int R = batch_rows_per_group(wt, am, mt);
    const int work = unit_work(wt);
    const bool quads = is_sb(wt) && am == A_INT8;
    const long long cap = std::max<long long>(1, (kBatchStageCap - 32) / rb);
    double best = 1e300;
    lpr = 32, bpl = (nu + 31) / 32, tr = (int)std::min<long long>(kBatchWarps, cap);
    for (int l = 1; l <= 32; ++l) {
        if (quads && l % 4 != 0) continue;
        const int b = (nu + l - 1) / l;
        if (!quads && (nu + b - 1) / b != l) continue;  // the same bpl with fewer lanes
        const long long t = std::min<long long>((long long)kBatchWarps * (32 / l) * R, cap);
        int levels = 0;
        while ((1 << levels) < l) ++levels;
        const double cost = ((30.0 * R + 12.0) * work * b + R * (3.0 * levels + 15.0) + 15.0) / (double)t;
        if (cost < best) best = cost, lpr = l, bpl = b, tr = (int)t;
    }
}

cudaError_t launch_batch(int wt, int am, const BatchParams& p0, int max_m, int sm_count, int smem_max, cudaStream_t s) {
    const int mt = max_m <= 1 ? 1 : max_m <= 2 ? 2 : max_m <= 4 ? 4 : 8;
    BatchParams p = p0;
    long long stage = 0, rows = 0;
    int last_k = -1, last_wt = -1, lpr = 0, bpl = 0, tr = 0;  // consecutive items of one type and K share a plan
    for (int i = 0; i < p.count; ++i) {
        BatchItem& it = p.it[i];
        const long long rb = (long long)(it.K / unit_vals(it.wt)) * unit_bytes(it.wt);
        if (it.K != last_k || it.wt != last_wt) {
            plan_batch_item(it.wt, batch_units(it.wt, it.K), rb, am, mt, lpr, bpl, tr);
            last_k = it.K, last_wt = it.wt;
        }
        it.lpr = lpr, it.bpl = bpl, it.tr = tr;
        stage = std::max(stage, (long long)it.tr * rb);
        rows += it.N;
    }
    // a slot holds a stage's rows plus the 16-byte alignment slack and the
    // few bytes the unit loads read past the last unit
    p.slot_bytes = (int)((stage + 32 + 127) / 128 * 128);

    long long grid = sm_count;
    if (grid > rows) grid = rows < 1 ? 1 : rows;
    if (wt == T_MIX) return launch_batch_mix(am, p, mt, (int)grid, smem_max, s);
    if (wt == T_Q8_0) return go<T_Q8_0>(am, p, mt, (int)grid, smem_max, s);
    if (wt == T_Q4_0) return go<T_Q4_0>(am, p, mt, (int)grid, smem_max, s);
    return go<T_Q5_0>(am, p, mt, (int)grid, smem_max, s);
}

}  // namespace qmm
