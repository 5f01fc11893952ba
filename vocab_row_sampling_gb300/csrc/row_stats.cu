// row_stats.cu -- one-read row statistics of temperature-scaled logits:
// argmax, Gumbel-max sample, softmax entropy and (optionally) the softmax in
// bf16/fp16 (page "vllm.model_executor.models.diffusion_gemma_sampler",
// module docstring, sample_row_stats and sample_row_stats_reference).
//
// Layout of the work. A row of V fp32 logits is split into G contiguous
// chunks of `chunk` columns (a multiple of 4). G CTAs -- a team -- own the G
// chunks of every row of the team; teams take rows round robin. The kernel
// is persistent: one CTA per SM, cooperative launch (all CTAs resident, so
// their bounded waits on each other cannot deadlock). A CTA has 15 compute
// warps (480 threads, VEC4 float4 slots each: slot i of thread t covers
// chunk columns 4*(i*480+t)+0..3) and one exchange warp.
//
// A row is handled in two halves LAG iterations apart, so that the team's
// exchange of the first half's results (a round trip through L2 that takes
// about as long as one iteration's compute) overlaps LAG iterations of work.
// Iteration k, before its one CTA barrier:
//   compute warps, first half of row k: wait for the bulk copy (TMA) that
//     staged the chunk iterations ahead; the warp max M_w of the scaled
//     logits s = x / Te (Te = max(T, 1e-10)) and the lowest column reaching
//     it (the argmax), e = e^(s - M_w) written back into the stage,
//     S_w = sum e and W_w = sum e (s - M_w) (the "online max and sum" of the
//     page), and for T > 0 the Gumbel-max score of the warp's argmax
//     element (a lower bound B of the row's best score). Division by Te > 0
//     is monotone, so while |M_w| < 256 the warp works on the raw logits:
//     the max is found among them, only the few candidates for the argmax
//     are divided (exactly), and e = 2^((x - x_max) log2(e) / Te) is within
//     a relative 2^-15 of e^(s - M_w). Warps with larger scaled values
//     divide every logit exactly first.
//   exchange warp: merges the team's first records of row k-LAG (M, S, W,
//     argmax, B) and its second records of row k-2LAG-1 (the race best);
//     member 0 writes argmax and entropy of row k-LAG and the sample of row
//     k-2LAG-1.
// After the barrier:
//   exchange warp: combines the warp partials of row k into the CTA's first
//     record and those of row k-LAG-1's race into its second record,
//     publishes both, and issues the bulk copy of a later row into the stage
//     row k-LAG-1 left.
//   compute warps, second half of row k-LAG, its e read back from the
//     stage: the pruned race against the row's B (an element can only win if
//     1 - u <= -log u <= e^(s - B) = e * e^(M_w - B); the few survivors are
//     rescored exactly from their logits), then the probabilities
//     e * e^(M_w - M) / S, rounded to nearest even and written to HBM.
//
// HBM traffic: every logit is read once (by the bulk copy) and every
// probability written once. No fp64 arithmetic (its rate on GB300 is a
// small fraction of fp32's).
#include <atomic>
#include <cfloat>
#include <climits>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "drs_device.cuh"
#include "drs_internal.h"

namespace drs {

namespace {

constexpr int kComputeWarps = kWarps - 1;     // warps 0..14
constexpr int kCompute = kComputeWarps * 32;  // 480 compute threads
constexpr int kExchangeWarp = kWarps - 1;     // warp 15
constexpr int kInfoRing = 8;                  // merged rows kept, by row % 8
// Three forms: LAG 2 with 5 stages of up to 6 float4 per thread (rows up to
// 32 * 11520 columns), LAG 1 with 4 stages of up to 8, and LAG 1 with 3
// stages (up to 32 * 15360 columns; the bulk copy then has only part of an
// iteration to land).
constexpr int kVec4Lag2 = 6;
constexpr int kVec4Lag1 = 8;
constexpr int kMaxStages = 5;
// The ring of exchange records must outlast 2 * LAG + 2 iterations.
static_assert(kRing >= 2 * 2 + 2, "exchange ring too short for LAG 2");

// log2(1.0002): the race's bound e^(s - best) is widened by 2e-4 so that
// rounding in it (at most a relative 2^-15 for e taken from the raw
// logits) never prunes an element whose fp32 score could win.
constexpr float kRaceMarginLog2 = 2.8851e-4f;
// Warps whose largest scaled logit is below this in magnitude work on the
// raw logits (see above).
constexpr float kRawDomainLimit = 256.0f;

struct RowStatsParams {
    const float* logits;
    int64_t row_stride;
    int64_t rows;
    int64_t row0;       // global index of row 0 (noise key, temperature slot)
    const float* temps;
    int64_t canvas_len;
    int64_t* argmax;
    int64_t* sample;
    float* entropy;
    void* probs;
    int64_t probs_row_stride;
    void* xchg;         // records: per CTA, kRing A slots (M, S, W, argmax,
                        // B) and kRing B slots (race best)
    int* err;
    PhiloxRoundKeys rk;
    int32_t vocab;
    int32_t team;       // CTAs per row
    int32_t chunk;      // columns per CTA (multiple of 4)
    int32_t num_teams;
    int32_t stage_bytes;
    int32_t use_tma;    // stages filled by bulk copies (rows 16-byte aligned)
    int32_t probs_dtype;
    int32_t probs_vec;  // 8-byte probability stores are aligned
    int32_t index32;    // global rows and canvas_len fit 32 bits
    int32_t fault;      // test hook: CTA 0 withholds its first record
};

// Test hook state: the next launch withholds one record (see
// drs_test_inject_fault).
std::atomic<int> g_inject_fault{0};

struct WarpPartial {
    float m, s, w, best;
    int arg, best_col;
};

struct WarpBest {
    float best;
    int col;
};

// What the merge of a row's first records leaves for the rest of the CTA.
struct RowInfo {
    float row_max;
    float log2s;
    float near_best;  // B: the best score among the warps' argmax elements
    int near_col;
    int arg;
    int noisy;
};

struct Scratch {
    uint64_t full[kMaxStages];
    WarpPartial p1[2][kComputeWarps];      // row k's warp partials, by row parity
    WarpBest p2[2][kComputeWarps];         // row j's race bests, by row parity
    RowInfo info[kInfoRing];               // merged rows
    float wref[kInfoRing][kComputeWarps];  // each warp's M_w, by row % 8
    int status;                            // a merge ran out of time
    int abort_load;                        // a bulk copy ran out of time
};

__device__ __forceinline__ void set_comp(float4& v, int q, float x) {
    if (q == 0) v.x = x;
    else if (q == 1) v.y = x;
    else if (q == 2) v.z = x;
    else v.w = x;
}

// Two probabilities rounded to nearest even and packed (first in the low
// half): bf16 or fp16.
__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16) {
    if (bf16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Temperature of a global row: temps[row / canvas_len].
__device__ __forceinline__ float row_temperature(const RowStatsParams& p, uint64_t grow_id) {
    const uint64_t slot = p.index32 ? static_cast<uint64_t>(static_cast<uint32_t>(grow_id) /
                                                            static_cast<uint32_t>(p.canvas_len))
                                    : grow_id / static_cast<uint64_t>(p.canvas_len);
    return p.temps[slot];
}

// Tag of the records of a team's row sequence k (never 0: rings are zeroed
// before each launch).
__device__ __forceinline__ uint32_t record_tag(int k) { return static_cast<uint32_t>(k) + 1u; }

// Elements of one float4 group that could still beat the row's best score
// B: winning needs -log u <= e^(s - B), so 1 - u (a lower bound of -log u)
// must be at most e^(s - B) = e * r_w (widened by the margin), with e =
// e^(s - M_w) from the stage. The group is first tested as a whole with its
// largest e and largest word.
__device__ __forceinline__ uint32_t race_group(const float4& e, uint4 w, float r_w) {
    const uint32_t wmax = max(max(w.x, w.y), max(w.z, w.w));
    uint32_t bits = 0;
    if (one_minus_u_lower(wmax) <= max4(e) * r_w) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (one_minus_u_lower(word_of(w, q)) <= comp(e, q) * r_w) bits |= 1u << q;
    }
    return bits;
}

// Score the survivors of `mask` (bit 4i+q: slot i, component q) exactly:
// s = x / max(T, 1e-10) from the logit in global memory (the stage holds e
// only), g from the element's Philox word; keep the best (score, column).
// The column that set the best already was scored the same way.
__device__ __noinline__ WarpBest race_rescore(uint32_t mask, const float* row_logits, float temp,
                                              int col0, int tid, uint64_t grow_id,
                                              const PhiloxRoundKeys& rk, WarpBest best) {
    const ScaledQuotient sq = ScaledQuotient::of(fmaxf(temp, kTempFloor));
    while (mask) {
        const int b = __ffs(mask) - 1;
        mask &= mask - 1;
        const int f = (b >> 2) * kCompute + tid;
        const int c = col0 + 4 * f + (b & 3);
        if (c == best.col) continue;
        const float s = sq.exact(__ldg(row_logits + c));
        const uint4 w = noise_words_rk(rk, grow_id, static_cast<uint32_t>((col0 >> 2) + f));
        const float score = s + gumbel_of_bits(word_of(w, b & 3));
        if (beats(score, c, best.best, best.col)) best = WarpBest{score, c};
    }
    return best;
}

}  // namespace

template <int VEC4, int LAG, int NSTAGE>
__global__ void __launch_bounds__(kThreads, 1)
    row_stats_kernel(const __grid_constant__ RowStatsParams p) {
    constexpr int kStages = NSTAGE;  // LAG + 1 rows held, the rest loading
    static_assert(kStages <= kMaxStages && kStages >= LAG + 2, "stages");
    extern __shared__ __align__(128) unsigned char smem[];
    Scratch& sc = *reinterpret_cast<Scratch*>(smem + kStages * p.stage_bytes);
    const bool use_tma = p.use_tma != 0;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const bool exchange = warp == kExchangeWarp;
    const int team_id = blockIdx.x / p.team;
    const int member = blockIdx.x - team_id * p.team;
    const int col0 = member * p.chunk;
    const int ncols = min(p.vocab - col0, p.chunk);
    const int nfull4 = ncols >> 2;
    const int nslot4 = (ncols + 3) >> 2;  // float4 slots holding a column
    const uint32_t copy_bytes = static_cast<uint32_t>(nfull4) * 16u;
    const int nrows = team_id < p.rows
                          ? static_cast<int>((p.rows - 1 - team_id) / p.num_teams + 1)
                          : 0;
    auto row_of = [&](int k) { return team_id + static_cast<int64_t>(k) * p.num_teams; };
    auto grow_of = [&](int k) { return static_cast<uint64_t>(p.row0 + row_of(k)); };

    if (tid == 0) {
        if (use_tma) {
            for (int s = 0; s < kStages; ++s) mbar_init(&sc.full[s], 1);
            fence_barrier_init();
        }
        sc.abort_load = 0;
        sc.status = 0;
    }
    __syncthreads();

    // Producer state, exchange-warp lane 0: rows issued to the stages.
    int issued = 0;
    auto issue_copy = [&]() {
        const int s = issued % kStages;
        mbar_arrive_expect_tx(&sc.full[s], copy_bytes);
        if (copy_bytes)
            tma_load_1d(smem + s * p.stage_bytes, p.logits + row_of(issued) * p.row_stride + col0,
                        copy_bytes, &sc.full[s]);
        ++issued;
    };
    if (use_tma && exchange && lane == 0) {
        while (issued < nrows && issued < kStages) issue_copy();
    }

    // Compute warps: the temperature of the next row, loaded an iteration
    // ahead.
    float temp_next = 0.0f;
    if (nrows > 0 && !exchange) temp_next = row_temperature(p, grow_of(0));

    bool aborted = false;
    int consumed = 0;
    for (int k = 0; k <= nrows + 2 * LAG; ++k) {
        const int par = k & 1;
        // ===================== before the barrier ===============================
        if (!exchange) {
            if (k < nrows) {
                // ---- compute warps: first half of row k -------------------------
                const int64_t row = row_of(k);
                const uint64_t grow_id = grow_of(k);
                const float* grow = p.logits + row * p.row_stride + col0;
                const int s = k % kStages;
                float4* stage4 = reinterpret_cast<float4*>(smem + s * p.stage_bytes);
                const float temp = temp_next;
                if (k + 1 < nrows) temp_next = row_temperature(p, grow_of(k + 1));

                bool timed_out = false;
                if (use_tma)
                    timed_out =
                        !mbar_wait_bounded(&sc.full[s], static_cast<uint32_t>((k / kStages) & 1));
                if (timed_out) sc.abort_load = 1;
                float4 v[VEC4];
#pragma unroll
                for (int i = 0; i < VEC4; ++i) {
                    const int f = i * kCompute + tid;
                    float4 x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                    if (i * kCompute < nslot4) {  // CTA-uniform: slot i holds columns
                        if (f < nfull4) {
                            if (use_tma) {
                                if (!timed_out) x = stage4[f];
                            } else {
                                x.x = grow[4 * f + 0];
                                x.y = grow[4 * f + 1];
                                x.z = grow[4 * f + 2];
                                x.w = grow[4 * f + 3];
                            }
                        } else if (f == nfull4) {
                            for (int q = 0; q < (ncols & 3); ++q) set_comp(x, q, grow[4 * f + q]);
                        }
                    }
                    v[i] = x;
                }

                const float te = fmaxf(temp, kTempFloor);
                const ScaledQuotient sq = ScaledQuotient::of(te);
                const bool noisy = temp > 0.0f;

                // max of the raw logits (division by te > 0 keeps the order)
                float mt = -INFINITY;
#pragma unroll
                for (int i = 0; i < VEC4; ++i) mt = fmaxf(mt, max4(v[i]));
                const float mxw = warp_max(mt);
                const float mw = mxw == -INFINITY ? -INFINITY : sq.exact(mxw);  // M_w
                // warp-uniform: raw domain, or exact quotients first
                const bool raw = !(fabsf(mw) >= kRawDomainLimit);
                float ref, scale;  // d = (v - ref) * scale is s - M_w
                float cthr;        // argmax candidates: v >= cthr
                if (raw) {
                    ref = mxw;
                    scale = sq.y;
                    // exact(x) == M_w needs x >= mxw - te * ulp(M_w)
                    cthr = mxw - fmaxf(fabsf(mxw) * 0x1p-20f, te * 0x1p-140f);
                } else {
#pragma unroll
                    for (int i = 0; i < VEC4; ++i) {
                        v[i].x = sq.exact(v[i].x);
                        v[i].y = sq.exact(v[i].y);
                        v[i].z = sq.exact(v[i].z);
                        v[i].w = sq.exact(v[i].w);
                    }
                    mt = sq.exact(mt);
                    ref = mw;
                    scale = 1.0f;
                    cthr = mw;
                }

                // argmax: the lowest column whose exact quotient is M_w
                int arg_t = INT_MAX;
                if (mt >= cthr && mw != -INFINITY) {
                    uint32_t cand = 0;  // bit 4i+q: columns in increasing order
#pragma unroll
                    for (int i = 0; i < VEC4; ++i)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (comp(v[i], q) >= cthr) cand |= 1u << (4 * i + q);
#pragma unroll 1
                    while (cand) {
                        const int b = __ffs(cand) - 1;
                        cand &= cand - 1;
                        const float x = pick(v, b);
                        if ((raw ? sq.exact(x) : x) == mw) {
                            arg_t = col0 + 4 * ((b >> 2) * kCompute + tid) + (b & 3);
                            break;
                        }
                    }
                }
                const int aw = warp_min_i(arg_t);

                // sums, four accumulators each; e = e^(s - M_w) waits in the
                // stage for the race and the probabilities
                const float lscale = kLog2e * scale;
                float st[4] = {0.0f, 0.0f, 0.0f, 0.0f}, wt[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int i = 0; i < VEC4; ++i) {
                    if (i * kCompute < nslot4) {
                        float4 ev;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            // -inf -> a finite difference whose e is 0
                            const float d = fmaxf(comp(v[i], q) - ref, -FLT_MAX);
                            const float e = ex2_approx(d * lscale);
                            set_comp(ev, q, e);
                            st[q] += e;
                            wt[q] = fmaf(e, d, wt[q]);
                        }
                        const int f = i * kCompute + tid;
                        if (f < nslot4) stage4[f] = ev;
                    }
                }
                // B candidate: the Gumbel-max score of the warp's argmax element
                float bs = -INFINITY;
                int bc = INT_MAX;
                if (noisy && aw != INT_MAX && arg_t == aw) {
                    const uint4 w = noise_words_rk(p.rk, grow_id, static_cast<uint32_t>(aw >> 2));
                    bs = mw + gumbel_of_bits(word_of(w, aw & 3));
                    bc = aw;
                }
                const float sw = warp_sum_f((st[0] + st[1]) + (st[2] + st[3]));
                const float ww = warp_sum_f((wt[0] + wt[1]) + (wt[2] + wt[3])) * scale;
                warp_best(bs, bc);
                if (lane == 0) {
                    sc.p1[par][warp] = WarpPartial{mw, sw, ww, bs, aw, bc};
                    sc.wref[k & (kInfoRing - 1)][warp] = mw;
                }
            }
        } else {
            // ---- exchange warp: first records of row k-LAG, second of k-2LAG-1 ----
            const bool do_a = k >= LAG && k - LAG < nrows;
            const bool do_b = k >= 2 * LAG + 1 && k - (2 * LAG + 1) < nrows;
            const int ka = k - LAG, kb = k - (2 * LAG + 1);
            // the temperature load overlaps the polling
            const float temp_a = (do_a && lane == 0) ? row_temperature(p, grow_of(ka)) : 0.0f;
            bool ok = true;
            uint64_t ra[6] = {0, 0, 0, 0, 0, 0}, rb[2] = {0, 0};
            if (lane < p.team && (do_a || do_b)) {
                const int cta = team_id * p.team + lane;
                ok = read_records(do_a ? record_a(p.xchg, cta, ka & (kRing - 1)) : nullptr,
                                  record_tag(ka), ra,
                                  do_b ? record_b(p.xchg, cta, kb & (kRing - 1)) : nullptr,
                                  record_tag(kb), rb);
            }
            const bool have = lane < p.team && ok;
            if (do_a) {
                const int64_t frow = row_of(ka);
                const float m = have ? payload_f(ra[0]) : -INFINITY;
                const float s_m = have ? payload_f(ra[1]) : 0.0f;
                const float w_m = have ? payload_f(ra[2]) : 0.0f;
                const int a_m = have ? static_cast<int>(payload_u(ra[3])) : INT_MAX;
                float b_m = have ? payload_f(ra[4]) : -INFINITY;
                int bc_m = have ? static_cast<int>(payload_u(ra[5])) : INT_MAX;
                const float big_m = warp_max(m);
                float s_l = 0.0f, w_l = 0.0f;
                if (m != -INFINITY) {
                    const float dm = m - big_m;
                    const float f = ex2_approx(dm * kLog2e);
                    s_l = f * s_m;
                    w_l = f * fmaf(dm, s_m, w_m);
                }
                const float s_tot = warp_sum_f(s_l);
                const float w_tot = warp_sum_f(w_l);
                const int arg_row = warp_min_i(m == big_m ? a_m : INT_MAX);
                warp_best(b_m, bc_m);
                if (lane == 0) {
                    RowInfo& ri = sc.info[ka & (kInfoRing - 1)];
                    ri.row_max = big_m;
                    ri.log2s = s_tot > 0.0f ? log2f(s_tot) : 0.0f;
                    ri.near_best = b_m;
                    ri.near_col = bc_m;
                    ri.arg = arg_row;
                    ri.noisy = temp_a > 0.0f && big_m != -INFINITY;
                    if (member == 0) {
                        p.argmax[frow] = arg_row;
                        p.entropy[frow] = s_tot > 0.0f ? logf(s_tot) - w_tot / s_tot : 0.0f;
                        if (!ri.noisy) p.sample[frow] = arg_row;
                    }
                }
            }
            if (do_b) {
                float b = have ? payload_f(rb[0]) : -INFINITY;
                int bcol = have ? static_cast<int>(payload_u(rb[1])) : INT_MAX;
                warp_best(b, bcol);
                if (lane == 0) {
                    const RowInfo& ri = sc.info[kb & (kInfoRing - 1)];
                    if (ri.noisy && member == 0) {
                        float bb = ri.near_best;
                        int bbc = ri.near_col;
                        if (beats(b, bcol, bb, bbc)) {
                            bb = b;
                            bbc = bcol;
                        }
                        p.sample[row_of(kb)] = bb != -INFINITY ? bbc : ri.arg;
                    }
                }
            }
            ok = __all_sync(0xffffffffu, ok);
            if (lane == 0) sc.status = ok ? 0 : 1;
        }

        __syncthreads();  // ============== the barrier of iteration k ===========

        if (sc.abort_load || sc.status) {
            aborted = true;
            break;
        }
        if (k < nrows) consumed = k + 1;

        // ===================== after the barrier ================================
        if (exchange) {
            if (k < nrows) {
                // ---- first record of row k --------------------------------------
                const WarpPartial wp = lane < kComputeWarps
                                           ? sc.p1[par][lane]
                                           : WarpPartial{-INFINITY, 0.0f, 0.0f, -INFINITY, INT_MAX,
                                                         INT_MAX};
                const float mc = warp_max(wp.m);
                float s_l = 0.0f, w_l = 0.0f;
                if (wp.m != -INFINITY) {
                    const float dm = wp.m - mc;
                    const float f = ex2_approx(dm * kLog2e);
                    s_l = f * wp.s;
                    w_l = f * fmaf(dm, wp.s, wp.w);
                }
                const float s_c = warp_sum_f(s_l);
                const float w_c = warp_sum_f(w_l);
                const int a_c = mc == -INFINITY ? col0 : warp_min_i(wp.m == mc ? wp.arg : INT_MAX);
                float b_c = wp.best;
                int bcol_c = wp.best_col;
                warp_best(b_c, bcol_c);
                if (lane == 0 && !(p.fault && blockIdx.x == 0 && k == 0))
                    publish_a(record_a(p.xchg, blockIdx.x, k & (kRing - 1)), record_tag(k), mc, s_c,
                              w_c, a_c, b_c, bcol_c);
            }
            const int kf = k - LAG - 1;
            if (kf >= 0 && kf < nrows) {
                // ---- second record of row k-LAG-1 (its race ran after barrier k-1)
                const WarpBest wb = lane < kComputeWarps ? sc.p2[kf & 1][lane]
                                                         : WarpBest{-INFINITY, INT_MAX};
                float b = wb.best;
                int bcol = wb.col;
                warp_best(b, bcol);
                if (lane == 0)
                    publish_b(record_b(p.xchg, blockIdx.x, kf & (kRing - 1)), record_tag(kf), b, bcol);
            }
            // The stage of row k-LAG-1 was read for the last time before this
            // barrier: it takes the next row to load.
            if (use_tma && lane == 0 && kf >= 0 && issued < nrows) {
                fence_proxy_async_smem();
                issue_copy();
            }
        } else if (k >= LAG && k - LAG < nrows) {
            // ---- compute warps: second half of row j = k-LAG -----------------------
            const int j = k - LAG;
            const RowInfo ri = sc.info[j & (kInfoRing - 1)];
            const float mw = sc.wref[j & (kInfoRing - 1)][warp];  // M_w of row j
            const int64_t frow = row_of(j);
            const uint64_t fgrow_id = grow_of(j);
            const float4* fstage =
                reinterpret_cast<const float4*>(smem + (j % kStages) * p.stage_bytes);
            float4 e[VEC4];
#pragma unroll
            for (int i = 0; i < VEC4; ++i) {
                const int f = i * kCompute + tid;
                e[i] = (i * kCompute < nslot4 && f < nslot4) ? fstage[f]
                                                             : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
            if (ri.noisy) {
                const float best = ri.near_best;
                // e^(s - B), widened by the race margin, is e * r_w.
                const float r_w =
                    mw == -INFINITY ? 0.0f : ex2_approx(fmaf(mw - best, kLog2e, kRaceMarginLog2));
                WarpBest wb{best, ri.near_col};
                uint32_t survivors = 0;
                // Philox four groups at a time, so that their chains overlap.
#pragma unroll
                for (int i0 = 0; i0 < VEC4; i0 += 4) {
                    constexpr int kGroup = 4;
                    bool pass[kGroup];
                    bool any = false;
#pragma unroll
                    for (int jj = 0; jj < kGroup; ++jj) {
                        // 1 - u >= 2^-24 always: below that bound no element of
                        // the group can win
                        pass[jj] = i0 + jj < VEC4 && (i0 + jj) * kCompute < nslot4 &&
                                   max4(e[min(i0 + jj, VEC4 - 1)]) * r_w >= 0x1p-24f;
                        any |= pass[jj];
                    }
                    // warp-uniform: when any lane needs this quad, every lane
                    // draws its blocks (straight-line, no divergence)
                    if (__any_sync(0xffffffffu, any)) {
                        uint4 w[kGroup];
#pragma unroll
                        for (int jj = 0; jj < kGroup; ++jj)
                            if (i0 + jj < VEC4)
                                w[jj] = noise_words_rk(
                                    p.rk, fgrow_id,
                                    static_cast<uint32_t>((col0 >> 2) + (i0 + jj) * kCompute + tid));
#pragma unroll
                        for (int jj = 0; jj < kGroup; ++jj)
                            if (i0 + jj < VEC4 && pass[jj])
                                survivors |= race_group(e[i0 + jj], w[jj], r_w) << (4 * (i0 + jj));
                    }
                }
                if (survivors)
                    wb = race_rescore(survivors, p.logits + frow * p.row_stride,
                                      row_temperature(p, fgrow_id), col0, tid, fgrow_id, p.rk, wb);
                warp_best(wb.best, wb.col);
                if (lane == 0) sc.p2[j & 1][warp] = wb;
            } else if (lane == 0) {
                sc.p2[j & 1][warp] = WarpBest{-INFINITY, INT_MAX};
            }

            if (p.probs_dtype != 0) {
                const float big_m = ri.row_max;
                // e^(s - M) / S = e * e^(M_w - M) / S
                const float f_w =
                    mw == -INFINITY ? 0.0f : ex2_approx(fmaf(mw - big_m, kLog2e, -ri.log2s));
                const bool bf16 = p.probs_dtype == 1;
                uint16_t* prow = static_cast<uint16_t*>(p.probs) + frow * p.probs_row_stride + col0;
#pragma unroll
                for (int i = 0; i < VEC4; ++i) {
                    const int f = i * kCompute + tid;
                    if (i * kCompute >= nslot4 || f >= nslot4) continue;
                    float pr[4] = {e[i].x * f_w, e[i].y * f_w, e[i].z * f_w, e[i].w * f_w};
                    if (big_m == -INFINITY) pr[0] = pr[1] = pr[2] = pr[3] = NAN;
                    const uint32_t lo = pack2(pr[0], pr[1], bf16);
                    const uint32_t hi = pack2(pr[2], pr[3], bf16);
                    if (p.probs_vec && f < nfull4) {
                        __stcs(reinterpret_cast<uint2*>(prow + 4 * f), make_uint2(lo, hi));
                    } else {
                        const uint16_t code[4] = {static_cast<uint16_t>(lo), static_cast<uint16_t>(lo >> 16),
                                                  static_cast<uint16_t>(hi), static_cast<uint16_t>(hi >> 16)};
                        for (int q = 0; q < 4; ++q)
                            if (4 * f + q < ncols) prow[4 * f + q] = code[q];
                    }
                }
            }
        }
    }

    if (aborted && tid == 0) raise_device_error(p.err, 1);
    // Bulk copies still in flight must land before the CTA's shared memory
    // is released.
    if (use_tma && exchange && lane == 0) {
        for (int seq = consumed; seq < issued; ++seq) {
            mbar_wait_bounded(&sc.full[seq % kStages], static_cast<uint32_t>((seq / kStages) & 1));
        }
    }
}

namespace {

struct RowStatsPlan {
    RowPlan rows;
    int lag;     // 2 or 1
    int nstage;  // 5 (LAG 2), 4 or 3 (LAG 1)
    int vec4;    // float4 slots per compute thread
};

// Team size G for one CTA per SM with 480 compute threads. The chunk must
// fit the registers and the stages shared memory. An iteration costs about
// max(chunk, round trip / LAG) + 1500 columns of work, the round trip of the
// team exchange through L2 (about 2.6 us) being worth some 18000 columns;
// the plan minimises ceil(rows / teams) times that, with teams = min(rows,
// sms / G) and the three-stage form counted 25% dearer. Ties go to the
// earlier form, then the smaller G.
RowStatsPlan plan_row_stats(int64_t rows, int vocab, int sms, size_t scratch) {
    const size_t budget = kSmemPerCta - scratch;
    struct Form {
        int lag, nstage, vec4;
        double pen;
    };
    constexpr double kChainCols = 18000.0;
    const Form forms[] = {{2, 5, kVec4Lag2, 1.0}, {1, 4, kVec4Lag1, 1.0}, {1, 3, kVec4Lag1, 1.25}};
    RowStatsPlan plan{{0, 0, 0, 0, 1}, 0, 0, 0};
    double best_cost = 0.0;
    const int capacity = sms > 1024 ? 1024 : sms;
    for (const Form& fm : forms) {
        int cap = static_cast<int>(budget / (4 * fm.nstage)) & ~31;
        if (cap > kCompute * fm.vec4 * 4) cap = kCompute * fm.vec4 * 4;
        const int g_min = (vocab + cap - 1) / cap;
        for (int g = g_min; g <= kMaxTeam && g <= capacity; ++g) {
            int chunk = (vocab + g - 1) / g;
            chunk = (chunk + 3) & ~3;
            if ((vocab + chunk - 1) / chunk != g) continue;
            int64_t teams = capacity / g;
            if (teams > rows) teams = rows;
            if (teams < 1) continue;
            const double per_row = (chunk > kChainCols / fm.lag ? chunk : kChainCols / fm.lag) + 1500.0;
            const double cost = fm.pen * static_cast<double>((rows + teams - 1) / teams) * per_row;
            if (plan.rows.team == 0 || cost < best_cost) {
                plan = RowStatsPlan{{g, chunk, static_cast<int>(teams), fm.vec4, 1}, fm.lag,
                                    fm.nstage, fm.vec4};
                best_cost = cost;
            }
        }
    }
    return plan;
}

template <int VEC4, int LAG, int NSTAGE>
drs_status launch_row_stats(RowStatsParams& prm, int grid, size_t smem, cudaStream_t stream) {
    auto kernel = row_stats_kernel<VEC4, LAG, NSTAGE>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return DRS_ERR_CUDA;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
    if (e != cudaSuccess || per_sm < 1) return DRS_ERR_CUDA;
    if (grid > per_sm * sm_count()) return DRS_ERR_UNSUPPORTED;
    void* args[] = {&prm};
    e = cudaLaunchCooperativeKernel(reinterpret_cast<void*>(kernel), dim3(grid),
                                    dim3(kThreads), args, smem, stream);
    return cuda_status(e);
}

}  // namespace

}  // namespace drs

extern "C" void drs_test_inject_fault(int code) { drs::g_inject_fault.store(code); }

extern "C" size_t drs_row_stats_workspace_bytes(int64_t rows, int64_t vocab) {
    (void)rows;
    (void)vocab;
    // The exchange records of up to 1024 resident CTAs.
    return static_cast<size_t>(1024) * drs::kXchgPerCta;
}

extern "C" drs_status drs_row_stats(const float* logits, int64_t rows, int64_t vocab,
                                    int64_t row_stride, const float* temps,
                                    int64_t canvas_len, uint64_t seed, int64_t row0,
                                    int64_t* argmax, int64_t* sample, float* entropy,
                                    drs_probs_dtype probs_dtype, void* probs,
                                    int64_t probs_row_stride, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    using namespace drs;
    if (rows < 0 || row0 < 0 || canvas_len < 1) return DRS_ERR_INVALID_ARG;
    if (vocab < 1 || row_stride < vocab) return DRS_ERR_INVALID_ARG;
    if (vocab > DRS_MAX_VOCAB) return DRS_ERR_UNSUPPORTED;
    if (!logits || !temps || !argmax || !sample || !entropy) return DRS_ERR_INVALID_ARG;
    if (probs_dtype != DRS_PROBS_NONE && probs_dtype != DRS_PROBS_BF16 &&
        probs_dtype != DRS_PROBS_FP16)
        return DRS_ERR_INVALID_ARG;
    if ((probs_dtype == DRS_PROBS_NONE) != (probs == nullptr)) return DRS_ERR_INVALID_ARG;
    if (probs && probs_row_stride < vocab) return DRS_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || !aligned(probs, 2)) return DRS_ERR_INVALID_ARG;
    if (rows == 0) return DRS_OK;
    const size_t need = drs_row_stats_workspace_bytes(rows, vocab);
    if (!workspace || workspace_bytes < need || !aligned(workspace, kWorkspaceAlign))
        return DRS_ERR_INVALID_ARG;

    const int sms = sm_count();
    if (sms <= 0) return DRS_ERR_CUDA;
    const size_t scratch = (sizeof(Scratch) + 127) & ~static_cast<size_t>(127);
    const RowStatsPlan rsp = plan_row_stats(rows, static_cast<int>(vocab), sms, scratch);
    const RowPlan& plan = rsp.rows;
    if (!plan.team) return DRS_ERR_UNSUPPORTED;
    // per-team row counts are int
    if ((rows + plan.num_teams - 1) / plan.num_teams > INT_MAX / 2) return DRS_ERR_UNSUPPORTED;

    RowStatsParams prm{};
    prm.logits = logits;
    prm.row_stride = row_stride;
    prm.rows = rows;
    prm.row0 = row0;
    prm.temps = temps;
    prm.canvas_len = canvas_len;
    prm.argmax = argmax;
    prm.sample = sample;
    prm.entropy = entropy;
    prm.probs = probs;
    prm.probs_row_stride = probs_row_stride;
    prm.xchg = workspace;
    prm.err = device_error_flag();
    prm.rk = PhiloxRoundKeys::of(seed);
    prm.vocab = static_cast<int32_t>(vocab);
    prm.team = plan.team;
    prm.chunk = plan.chunk;
    prm.num_teams = plan.num_teams;
    prm.probs_dtype = static_cast<int32_t>(probs_dtype);
    prm.probs_vec = probs && aligned(probs, 8) && (probs_row_stride % 4 == 0);
    prm.index32 = (row0 + rows <= static_cast<int64_t>(UINT32_MAX)) &&
                  (canvas_len <= static_cast<int64_t>(UINT32_MAX));
    prm.fault = g_inject_fault.exchange(0);
    if (!prm.err) return DRS_ERR_CUDA;

    // Shared memory: the stages of one chunk each (filled by bulk copies when
    // rows start 16-byte aligned; in every case they keep a row's e until its
    // second half) plus the scratch.
    const bool tma = aligned(logits, 16) && (row_stride % 4 == 0);
    prm.stage_bytes = (plan.chunk * 4 + 127) & ~127;
    prm.use_tma = tma ? 1 : 0;
    const size_t smem = static_cast<size_t>(rsp.nstage) * prm.stage_bytes + scratch;
    if (smem > kSmemPerCta) return DRS_ERR_UNSUPPORTED;
    const int grid = plan.team * plan.num_teams;
    // Zero the records this launch uses: a zero tag matches no row.
    if (cudaMemsetAsync(workspace, 0, static_cast<size_t>(grid) * kXchgPerCta,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return DRS_ERR_CUDA;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (rsp.lag == 2) return launch_row_stats<kVec4Lag2, 2, 5>(prm, grid, smem, st);
    if (rsp.nstage == 4) return launch_row_stats<kVec4Lag1, 1, 4>(prm, grid, smem, st);
    return launch_row_stats<kVec4Lag1, 1, 3>(prm, grid, smem, st);
}

// ---------------------------------------------------------------------------
// drs_row_stats_noalloc: drs_row_stats with its workspace in a fixed device
// array of this library instead of a caller buffer.
//
// Some callers cannot hand the library a workspace: plugin interfaces of
// inference runtimes that pass only input and output buffers at enqueue
// time, or code that must not call cudaMalloc because it synchronises the
// device or draws on a memory budget fixed at start-up. For them the
// exchange records live in g_noalloc_workspace below: every GPU that loads
// the library holds these bytes until the process exits, and all calls on a
// device share them.

namespace {

constexpr size_t kNoallocWorkspaceBytes = static_cast<size_t>(1024) * drs::kXchgPerCta;
static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoallocWorkspaceBytes];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64] = {};

// Device address of g_noalloc_workspace on the current device. In host code
// the array's name is a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
void* noalloc_workspace(drs_status* status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *status = DRS_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_workspace);
        if (e != cudaSuccess || !ptr) {
            *status = DRS_ERR_CUDA;
            return nullptr;
        }
        g_noalloc_ptr[dev] = ptr;
    }
    *status = DRS_OK;
    return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" drs_status drs_row_stats_noalloc(const float* logits, int64_t rows, int64_t vocab,
                                            int64_t row_stride, const float* temps,
                                            int64_t canvas_len, uint64_t seed, int64_t row0,
                                            int64_t* argmax, int64_t* sample, float* entropy,
                                            drs_probs_dtype probs_dtype, void* probs,
                                            int64_t probs_row_stride, void* stream) {
    if (drs_row_stats_workspace_bytes(rows, vocab) > kNoallocWorkspaceBytes)
        return DRS_ERR_UNSUPPORTED;
    if (rows <= 0)  // validation and the empty call need no workspace
        return drs_row_stats(logits, rows, vocab, row_stride, temps, canvas_len, seed, row0,
                             argmax, sample, entropy, probs_dtype, probs, probs_row_stride,
                             nullptr, 0, stream);
    drs_status st = DRS_OK;
    void* ws = noalloc_workspace(&st);
    if (!ws) return st;
    return drs_row_stats(logits, rows, vocab, row_stride, temps, canvas_len, seed, row0, argmax,
                         sample, entropy, probs_dtype, probs, probs_row_stride, ws,
                         kNoallocWorkspaceBytes, stream);
}
