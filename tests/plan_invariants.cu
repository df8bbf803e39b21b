// plan_invariants.cu -- host-only check of the launch planners.
//
// Built and run by tests/test_plans.py on the CPU (no GPU is touched: only the
// inline host planners of the kernel headers are called).  For a grid of
// shapes it checks that every plan the decode, GEMV, streaming and tcgen05 planners
// return fits the device limits it was planned for and keeps the layout rules
// its kernel relies on: shared-memory regions in order and inside the
// allocation, at least the ring depth the kernel assumes, one CTA per SM, K
// slices that cover K exactly once, bank-spreading pitches, and the
// documented choice of a separate activation-preparing launch.  Prints one
// line per violation and "ok <plans>" at the end; exits 1 on any violation.
#include <cstdio>

#include "qmm_internal.h"

using namespace qmm;

namespace {
constexpr int kSms = 152;          // GB300
constexpr int kSmem = 232448;      // opt-in shared memory per block (227 KB)
int g_bad = 0;

#define CHECK(cond, ...)                                  \
    do {                                                  \
        if (!(cond)) {                                    \
            ++g_bad;                                      \
            std::printf("FAIL %s: ", #cond);              \
            std::printf(__VA_ARGS__);                     \
            std::printf("\n");                            \
        }                                                 \
    } while (0)

const char* tname(int wt) {
    return wt == T_Q8_0 ? "q8_0" : wt == T_Q4_K ? "q4_k" : wt == T_Q4_0 ? "q4_0" : wt == T_Q5_0 ? "q5_0" : "q6_k";
}

int check_dmma(int wt, int am, long long M, long long N, long long K) {
    DmmaPlan pl;
    if (!plan_dmma(wt, am, M, N, K, kSms, kSmem, pl, true)) return 0;
    const DmmaParams& p = pl.p;
    const int ub = unit_bytes(wt);
#define CASE "%s am%d M%lld N%lld K%lld", tname(wt), am, M, N, K
    CHECK(pl.smem <= (size_t)kSmem, CASE);
    CHECK(p.stages >= 2 && p.stages <= 8, CASE);
    CHECK(p.off_flags >= 256 && p.off_flags < p.off_act && p.off_act <= p.off_scale && p.off_scale <= p.off_aux &&
              p.off_aux <= p.off_red && p.off_red < p.off_stage,
          CASE);
    CHECK(p.off_stage % 128 == 0 && p.stage_bytes % 128 == 0, CASE);
    CHECK((size_t)p.off_stage + (size_t)p.stages * p.stage_bytes <= pl.smem, CASE);
    // the reduction buffer: 16 warps x 16 weight rows x the tile's activation columns
    CHECK(p.off_red + kDmmaWarps * kDmmaRows * dmma_red_cols(am, pl.nb) * 4 <= p.off_stage, CASE);
    // K slices cover the units exactly once; chunks lie inside a slice
    CHECK(p.kslices >= 1 && (long long)(p.kslices - 1) * p.slice_units < p.units &&
              (long long)p.kslices * p.slice_units >= p.units,
          CASE);
    CHECK(p.ups >= 1 && p.ups <= p.slice_units, CASE);
    if (p.row_pitch == 0) {  // whole tile in one copy
        CHECK(p.kslices == 1 && p.ups == p.slice_units && 16 * p.rb + 64 <= p.stage_bytes, CASE);
    } else {                 // one copy per row into pitched rows (16 mod 128: 32 banks for 8 rows)
        CHECK(p.row_pitch >= p.ups * ub + 16 && p.row_pitch % 128 == 16, CASE);
        CHECK(16LL * p.row_pitch <= p.stage_bytes, CASE);
    }
    // activation columns: 8 int8 rows or 4 f32 rows (hi and lo) per column set
    CHECK(pl.nb == (am == A_INT8 ? (M > 8 ? 2 : 1) : (M > 8 ? 4 : M > 4 ? 2 : 1)), CASE);
    CHECK((am == A_INT8 ? 8 : 4) * pl.nb >= M, CASE);
    if (am == A_INT8) CHECK(p.act_pitch % 128 == 16, CASE);
    else CHECK((2 * p.act_pitch) % 128 == 64, CASE);
    // one CTA per SM, every tile of every slice owned
    CHECK(pl.grid == p.per_slice * p.kslices && pl.grid <= kSms && p.per_slice >= 1 && p.per_slice <= p.ntiles, CASE);
    CHECK(p.ntiles == (int)((N + kDmmaRows - 1) / kDmmaRows), CASE);
    // a separate preparing launch only for large weights with more than 2 rows (4 for 32-value blocks)
    const bool ext = p.total_bytes >= kDmmaExtMinBytes && M > (is_b32(wt) ? 4 : 2);
    CHECK((pl.ext_bytes > 0) == ext, CASE);
    CHECK(pl.workspace == pl.ext_bytes + (p.kslices > 1 ? (size_t)p.kslices * M * N * 4 : 0), CASE);
    if (ext) {
        CHECK(p.ext_codes == 0 && p.ext_scale >= (am == A_INT8 ? M * K : 4 * M * K) && p.ext_aux >= p.ext_scale &&
                  (size_t)p.ext_aux <= pl.ext_bytes,
              CASE);
    }
#undef CASE
    return 1;
}

int check_gemv(int wt, long long M, long long N, long long K) {
    GemvPlan pl;
    if (!plan_gemv(wt, M, N, K, kSms, kSmem, pl)) return 0;
    const GemvParams& p = pl.p;
#define CASE "gemv %s M%lld N%lld K%lld", tname(wt), M, N, K
    CHECK(pl.smem <= (size_t)kSmem, CASE);
    CHECK(p.stages >= 3 && p.stages <= 8, CASE);
    CHECK(p.off_flags >= 256 && p.off_flags < p.off_codes && p.off_codes <= p.off_scale && p.off_scale <= p.off_aux &&
              p.off_aux <= p.off_red && p.off_red < p.off_stage,
          CASE);
    CHECK((size_t)p.off_stage + (size_t)p.stages * p.stage_bytes <= pl.smem, CASE);
    // a stage holds tr whole rows plus the 16-byte rounding of the copy at both ends
    CHECK((long long)p.tr * p.rb + 32 <= p.stage_bytes, CASE);
    CHECK(p.tr >= 1 && p.tr <= 16 && (p.tr & (p.tr - 1)) == 0, CASE);
    CHECK(p.ngroups == (int)((N + p.tr - 1) / p.tr), CASE);
    CHECK(pl.mt >= M && pl.mt <= 8, CASE);
    CHECK(pl.grid >= 1 && pl.grid <= kSms, CASE);
#undef CASE
    return 1;
}

int check_tc(int wt, long long M, long long N, long long K) {
    TcPlan pl;
    if (!plan_tc(wt, M, N, K, kSms, kSmem, pl)) return 0;
    const TcParams& p = pl.p;
#define CASE "tc %s M%lld N%lld K%lld", tname(wt), M, N, K
    CHECK(pl.smem <= (size_t)kSmem, CASE);
    CHECK(p.nraw >= 2 && p.nraw <= kTcRSMax, CASE);
    CHECK(p.off_raw == kTcS * 2 * p.piece && p.off_bar == p.off_raw + p.nraw * p.raw_stage, CASE);
    CHECK(p.raw_stage % 1024 == 0 && p.raw_stage >= kTcBW * p.raw_row, CASE);
    // the MMA's N: a multiple of 16 up to 256 that covers M in mtiles tiles
    CHECK(p.bx % 16 == 0 && p.bx >= 16 && p.bx <= kTcBXMax && (long long)p.bx * p.mtiles >= M, CASE);
    // TMEM: the accumulators plus four stages of 32 weight-piece columns fit the 512 columns
    CHECK((p.nacc == 2 ? 2 * 128 : 256) + kTcS * 64 <= kTcTmemCols && p.nacc == (p.bx <= 128 ? 2 : 1), CASE);
    // accumulation chunks: 1024 K with two accumulators, 4096 K with one
    CHECK(p.kchunk == (p.nacc == 2 ? 4 : 16), CASE);
    CHECK(p.ntiles == (int)((N + kTcBW - 1) / kTcBW) && p.tiles == p.mtiles * p.ntiles, CASE);
    CHECK(p.ks >= 1 && p.ks <= p.nrs && p.units == p.tiles * p.ks, CASE);
    CHECK(pl.grid == (p.units < kSms ? p.units : kSms), CASE);
    CHECK(pl.ws_alo >= (size_t)M * K * 2 && pl.ws_ais >= pl.ws_alo + (size_t)M * K * 2 && pl.ws_wis >= pl.ws_ais + M * 4 &&
              pl.ws_part >= pl.ws_wis + N * 4 && pl.workspace >= pl.ws_cnt,
          CASE);
    if (p.ks > 1) CHECK(pl.ws_cnt >= pl.ws_part + (size_t)p.ks * M * N * 4 && pl.workspace >= pl.ws_cnt + p.tiles * 4, CASE);
    // Q6_K: the super-blocks repacked into 240-byte slots (16-byte aligned rows for the tensor map)
    if (wt == T_Q6_K)
        CHECK(p.raw_row == kTcQ6Slot && pl.ws_w6 >= pl.ws_cnt && pl.ws_w6 % 256 == 0 &&
                  pl.workspace >= pl.ws_w6 + (size_t)N * (K / 256) * kTcQ6Slot && (K / 256 * kTcQ6Slot) % 16 == 0,
              CASE);
#undef CASE
    return 1;
}

int check_tcx(int wt, int am, long long M, long long N, long long K) {
    TcxPlan pl;
    if (!plan_tcx(wt, am, M, N, K, kSms, kSmem, pl)) return 0;
    const TcxParams& p = pl.p;
#define CASE "tcx %s M%lld N%lld K%lld", tname(wt), M, N, K
    CHECK(pl.smem <= (size_t)kSmem && p.nraw >= 3 && p.nraw <= kTxRawMax, CASE);
    CHECK(p.off_raw == tcx_stages(wt, am, pl.nx) * tcx_stage_bytes(wt, am, pl.nx) && p.off_raw % 1024 == 0 && tcx_raw_slot(wt, am) % 1024 == 0 &&
              p.off_bar == p.off_raw + p.nraw * tcx_raw_slot(wt, am) && (size_t)p.off_bar + 512 + 1024 <= pl.smem,
          CASE);
    CHECK((pl.nx == 64 || pl.nx == kTxX) && (pl.nx == 64) == (M <= 64), CASE);
    CHECK(p.nrs * 256 == K && (long long)p.mtiles * pl.nx >= M && (long long)(p.mtiles - 1) * pl.nx < M &&
              (long long)p.ntiles * kTxW >= N && p.tiles == p.mtiles * p.ntiles,
          CASE);
    // every K slice holds at least one raw stage, and the slices tile K
    CHECK(p.ks >= 1 && p.ks <= kTxMaxSplit && p.ks <= p.nrs && p.units == p.tiles * p.ks, CASE);
    for (int sp = 0; sp < p.ks; ++sp) {
        const int r0 = sp * p.nrs / p.ks, r1 = (sp + 1) * p.nrs / p.ks;
        CHECK(r1 > r0 && (sp > 0 || r0 == 0) && (sp < p.ks - 1 || r1 == p.nrs), CASE);
    }
    CHECK(pl.grid >= 1 && pl.grid <= kSms && pl.grid <= p.units && pl.mp % 4 == 0 && pl.mp >= M, CASE);
    CHECK(pl.am == am, CASE);
    CHECK(pl.ws_scales >= (size_t)M * K * 2 && pl.ws_scales % 256 == 0 && pl.ws_bsums % 256 == 0 &&
              pl.ws_bsums >= pl.ws_scales + (am == A_F32 ? (size_t)M * K * 2 : (size_t)(K / (wt == T_Q8_0 ? 32 : 256)) * pl.mp * 4) &&
              pl.ws_ais % 256 == 0 &&
              pl.ws_ais >= pl.ws_bsums + (wt == T_Q4_K || (wt == T_Q6_K && am == A_INT8) ? (size_t)M * (K / 16) * 2 * (am == A_F32 ? 2 : 1) : 0) &&
              pl.ws_w6 % 256 == 0 && pl.ws_w6 >= pl.ws_ais + (am == A_F32 ? (size_t)M * 4 : 0) &&
              pl.ws_part % 256 == 0 && pl.ws_part >= pl.ws_w6 + (wt == T_Q6_K ? (size_t)N * (K / 256) * 240 : 0) &&
              pl.ws_cnt % 256 == 0 && pl.ws_cnt >= pl.ws_part + (p.ks > 1 ? (size_t)p.ks * M * N * 4 : 0) &&
              pl.workspace >= pl.ws_cnt + (p.ks > 1 ? (size_t)p.tiles * 4 : 0),
          CASE);
#undef CASE
    return 1;
}

int check_stream(int wt, int am, int epi, long long M, long long N, long long K) {
    StreamPlan pl;
    if (!plan_stream(wt, am, epi, M, N, K, kSms, kSmem, pl)) return 0;
    const StreamParams& p = pl.p;
    const int ub = unit_bytes(wt);
#define CASE "stream %s am%d epi%d M%lld N%lld K%lld", tname(wt), am, epi, M, N, K
    CHECK(pl.smem <= (size_t)kSmem, CASE);
    CHECK(p.stages >= 2 && p.stages <= 8, CASE);
    CHECK(p.off_flags >= 128 && p.off_flags < p.off_codes && p.off_codes <= p.off_scale && p.off_scale <= p.off_aux &&
              p.off_aux <= p.off_rs && p.off_rs <= p.off_red && p.off_red < p.off_stage,
          CASE);
    CHECK((size_t)p.off_stage + (size_t)p.stages * kTileRows * p.row_stride <= pl.smem, CASE);
    CHECK(p.row_stride >= p.ups * ub + 32 && p.row_stride % 128 == 16, CASE);
    CHECK(p.kslices >= 1 && (long long)(p.kslices - 1) * p.slice_units < p.units &&
              (long long)p.kslices * p.slice_units >= p.units,
          CASE);
    CHECK(p.ups >= 1 && p.ups <= p.slice_units, CASE);
    CHECK((long long)p.mr * p.mchunks >= M && p.pairs == p.kslices * p.mchunks, CASE);
    CHECK(pl.grid == p.pairs * p.per_pair && p.per_pair >= 1 && p.per_pair <= p.ntiles, CASE);
    CHECK(pl.workspace == ((epi == E_Y && p.kslices > 1)
                               ? (size_t)p.kslices * M * N * 4 + (size_t)p.mchunks * p.ntiles * 4 + 256
                               : 0),
          CASE);
#undef CASE
    return 1;
}
}  // namespace

int main() {
    int plans = 0;
    const int types[5] = {T_Q8_0, T_Q4_K, T_Q4_0, T_Q5_0, T_Q6_K};
    const long long Ns[8] = {1, 16, 33, 192, 576, 4100, 14336, 28672};
    const long long Ks[10] = {32, 96, 256, 576, 1024, 1536, 4096, 8192, 14336, 65536};
    for (int wt : types)
        for (int am : {A_INT8, A_F32})
            for (long long M = 1; M <= kDmmaMaxM; ++M)
                for (long long N : Ns)
                    for (long long K : Ks) {
                        if (K % (is_b32(wt) ? 32 : 256)) continue;
                        plans += check_dmma(wt, am, M, N, K);
                    }
    for (int wt : {T_Q8_0, T_Q4_K})
        for (long long M : {1, 2, 4, 8})
            for (long long N : Ns)
                for (long long K : Ks) {
                    if (K % (wt == T_Q8_0 ? 32 : 256)) continue;
                    plans += check_gemv(wt, M, N, K);
                }
    for (int wt : types) {
        for (long long M : {17, 37, 64, 255, 256, 300, 1024, 4097})
            for (long long N : {128, 300, 4096, 14336})
                for (long long K : {256, 1024, 4096, 14336}) {
                    plans += check_tc(wt, M, N, K);
                    plans += check_tcx(wt, A_INT8, M, N, K);
                    if (wt == T_Q8_0 || wt == T_Q4_K || wt == T_Q6_K) plans += check_tcx(wt, A_F32, M, N, K);
                }
    }
    for (int wt : types)
        for (int am : {A_INT8, A_F32})
            for (int epi : {E_Y, E_SUMS}) {
                if (epi == E_SUMS && am == A_F32) continue;  // block sums are an int8_act hook
                for (long long M : {1, 9, 17, 37, 64, 100, 300, 1024})
                    for (long long N : {1, 33, 576, 4096, 14336})
                        for (long long K : {32, 576, 1536, 4096, 14336}) {
                            if (K % (is_b32(wt) ? 32 : 256)) continue;
                            plans += check_stream(wt, am, epi, M, N, K);
                        }
            }
    // the shapes the benchmark and the tests depend on must have plans
    DmmaPlan dp;
    for (int wt : types)
        for (int am : {A_INT8, A_F32})
            for (long long M : {1, 2, 4, 8, 16})
                CHECK(plan_dmma(wt, am, M, 28672, 8192, kSms, kSmem, dp, true), "no decode plan for %s am%d M%lld", tname(wt), am, M);
    TcPlan tp;
    TcxPlan xp;
    for (long long M : {37, 64, 256, 1024})
        for (int wt : types) {
            CHECK(plan_tc(wt, M, 14336, 4096, kSms, kSmem, tp), "no tcgen05 plan for %s M%lld", tname(wt), M);
            CHECK(plan_tcx(wt, A_INT8, M, 14336, 4096, kSms, kSmem, xp), "no exact prefill plan for %s M%lld", tname(wt), M);
            if (wt == T_Q4_K)
                CHECK(plan_tcx(wt, A_F32, M, 14336, 4096, kSms, kSmem, xp), "no f32_act code-GEMM plan for M%lld", M);
        }
    std::printf("%s %d plans\n", g_bad ? "FAILED" : "ok", plans);
    return g_bad ? 1 : 0;
}
