// row_stats.cu -- one-read row statistics of temperature-scaled logits:
// argmax, Gumbel-max sample, softmax entropy and (optionally) the softmax in
// bf16/fp16 (page "vllm.model_executor.models.diffusion_gemma_sampler",
// module docstring, sample_row_stats and sample_row_stats_reference).
//
// Layout of the work. A row of V fp32 logits is split into G contiguous
// chunks of `chunk` columns (a multiple of 4). G CTAs -- a team -- own the G
// chunks of every row of the team; teams take rows round robin. The kernel
// is persistent: one CTA per SM, cooperative launch (all CTAs resident, so
// their bounded waits on each other cannot deadlock). A CTA has 14 compute
// warps (448 threads, VEC4 float4 slots each: slot i of thread t covers
// chunk columns 4*(i*448+t)+0..3), a publisher warp and a poller warp. They
// synchronise through mbarriers only, so that every warp runs at its own
// pace and the latency of one warp's work hides behind the others'.
//
// Compute warps, in order, for k = 0, 1, ...:
//   first half of row k: wait for the stage (bulk copy); the warp max M_w
//     of the scaled logits s = x / Te (Te = max(T, 1e-10)) and the lowest
//     column reaching it (the argmax), e = e^(s - M_w) written back into the
//     stage, S_w = sum e and W_w = sum e (s - M_w) (the "online max and
//     sum" of the page), and for T > 0 the Gumbel-max score of the warp's
//     argmax element (a lower bound B of the row's best score); arrive on
//     the row's first-half barrier. Division by Te > 0 is monotone, so while
//     |M_w| < 256 the warp works on the raw logits: the max is found among
//     them, only the few candidates for the argmax are divided (exactly),
//     and e = 2^(x log2(e) / Te - c) with c the rounded reference is within
//     a relative 2^-15 of e^(s - M_w). Warps with larger scaled values
//     divide every logit exactly first.
//   second half of row k-LAG, once the poller has merged the row: the
//     probabilities e * e^(M_w - M) / S (rounded to nearest even, written to
//     HBM), then the pruned race against the row's B (an element can only
//     win if 1 - u <= -log u <= e^(s - B) = e * e^(M_w - B); the float4
//     groups that pass a bound on their largest e go on a per-warp list,
//     shared out one Philox call per lane; the few survivors are rescored
//     exactly from their logits); arrive on the row's second-half barrier,
//     which also frees the stage.
// Publisher warp: per row, combines the compute warps' first-half partials
//   into the CTA's first record and publishes it; two rows later combines
//   their race bests into the second record, publishes it, and refills the
//   freed stage with a later row (bulk copy), with that row's temperature
//   quotient computed once for the CTA.
// Poller warp: per row, reads the team's first records (M, S, W, argmax, B)
//   and merges them for the compute warps, and reads the second records of
//   an earlier row; member 0 writes argmax, entropy and sample.
// LAG rows between a row's halves cover the team exchange, a round trip
// through L2.
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

constexpr int kComputeWarps = kWarps - 2;     // warps 0..13
constexpr int kCompute = kComputeWarps * 32;  // 448 compute threads
constexpr int kPublisherWarp = kWarps - 2;    // warp 14
constexpr int kPollerWarp = kWarps - 1;       // warp 15
static_assert(kPublisherWarp == kComputeWarps && kPollerWarp == kComputeWarps + 1, "warp roles");
constexpr int kRowRing = 8;                   // per-row shared state, by row % 8
// Three forms: LAG 2 with 5 stages of up to 6 float4 per thread (rows up to
// 32 * 10752 columns), LAG 1 with 4 stages of up to 9, and LAG 1 with 3
// stages (up to 32 * 16128 columns; the bulk copy then has less time to
// land).
constexpr int kVec4Lag2 = 6;
constexpr int kVec4Lag1 = 9;
constexpr int kMaxStages = 5;
constexpr int kMaxVec4Slots = 9;
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
    float m, s, w;
    int arg;
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

// A row's temperature and its quotient, set once by the publisher.
struct RowQuotient {
    float temp;
    float t, y;
    int mode;
};

struct Scratch {
    uint64_t full[kMaxStages];          // the stage holds the row (bulk copy landed)
    uint64_t a_done[kRowRing];          // the compute warps' first-half partials are in p1
    uint64_t b_done[kRowRing];          // second half done: race bests in p2, stage free
    uint64_t info_ready[kRowRing];      // the row's merged first records are in info
    WarpPartial p1[kRowRing][kComputeWarps];
    WarpBest p2[kRowRing][kComputeWarps];
    RowInfo info[kRowRing];
    RowQuotient rq[kRowRing];
    float wref[kRowRing][kComputeWarps];                   // each warp's M_w
    uint16_t worklist[kComputeWarps][32 * kMaxVec4Slots];  // race groups of a warp
    int abort;                                             // a wait ran out of time
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

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
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

// Score the survivors `bits` of the float4 group starting at column c4
// exactly: s = x / Te from the logit in global memory (the stage holds e
// only), g from the group's Philox words; keep the best (score, column).
// The column that set the best already was scored the same way.
__device__ __noinline__ WarpBest race_rescore(uint32_t bits, const float* row_logits, int c4,
                                              uint4 w, const RowQuotient rq, int skip_col,
                                              WarpBest best) {
    ScaledQuotient sq;
    sq.t = rq.t;
    sq.y = rq.y;
    sq.mode = rq.mode;
    while (bits) {
        const int q = __ffs(bits) - 1;
        bits &= bits - 1;
        const int c = c4 + q;
        if (c == skip_col) continue;
        const float s = sq.exact(__ldg(row_logits + c));
        const float score = s + gumbel_of_bits(word_of(w, q));
        if (beats(score, c, best.best, best.col)) best = WarpBest{score, c};
    }
    return best;
}

}  // namespace

template <int VEC4, int LAG, int NSTAGE>
__global__ void __launch_bounds__(kThreads, 1)
    row_stats_kernel(const __grid_constant__ RowStatsParams p) {
    static_assert(NSTAGE <= kMaxStages && NSTAGE >= LAG + 2, "stages");
    static_assert(VEC4 <= kMaxVec4Slots, "slots");
    extern __shared__ __align__(128) unsigned char smem[];
    Scratch& sc = *reinterpret_cast<Scratch*>(smem + NSTAGE * p.stage_bytes);
    volatile int* abort_flag = &sc.abort;
    const bool use_tma = p.use_tma != 0;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
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
    auto fail = [&]() {
        *abort_flag = 1;
        raise_device_error(p.err, 1);
    };

    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) mbar_init(&sc.full[s], 1);
        for (int r = 0; r < kRowRing; ++r) {
            mbar_init(&sc.a_done[r], kComputeWarps);
            mbar_init(&sc.b_done[r], kComputeWarps);
            mbar_init(&sc.info_ready[r], 1);
        }
        fence_barrier_init();
        sc.abort = 0;
    }
    __syncthreads();  // the only CTA barrier: everything after is mbarriers

    if (warp < kComputeWarps) {
        // ======================= compute warps ==================================
        for (int k = 0; k < nrows + LAG; ++k) {
            if (*abort_flag) break;
            if (k < nrows) {
                // ---- first half of row k ---------------------------------------
                const int64_t row = row_of(k);
                const float* grow = p.logits + row * p.row_stride + col0;
                float4* stage4 = reinterpret_cast<float4*>(smem + (k % NSTAGE) * p.stage_bytes);
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&sc.full[k % NSTAGE],
                                                               static_cast<uint32_t>((k / NSTAGE) & 1)))) {
                    if (lane == 0) fail();
                    break;
                }
                const RowQuotient rq = sc.rq[k & (kRowRing - 1)];
                ScaledQuotient sq;
                sq.t = rq.t;
                sq.y = rq.y;
                sq.mode = rq.mode;
                float4 v[VEC4];
#pragma unroll
                for (int i = 0; i < VEC4; ++i) {
                    const int f = i * kCompute + tid;
                    float4 x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                    if (i * kCompute < nslot4) {  // CTA-uniform: slot i holds columns
                        if (f < nfull4) {
                            if (use_tma) {
                                x = stage4[f];
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

                // max of the raw logits (division by Te > 0 keeps the order)
                float m4[VEC4];
                float mt = -INFINITY;
#pragma unroll
                for (int i = 0; i < VEC4; ++i) {
                    m4[i] = max4(v[i]);
                    mt = fmaxf(mt, m4[i]);
                }
                const float mxw = warp_max(mt);
                const float mw = mxw == -INFINITY ? -INFINITY : sq.exact(mxw);  // M_w
                // warp-uniform: raw domain, or exact quotients first
                const bool raw = !(fabsf(mw) >= kRawDomainLimit);
                // argmax: the lowest column whose exact quotient is M_w.
                // exact(x) == M_w needs x >= mxw - Te * ulp(M_w), so only the
                // slots whose max reaches that are searched, their logits
                // read again (the stage still holds them).
                const float cthr = mxw - fmaxf(fabsf(mxw) * 0x1p-20f, rq.t * 0x1p-140f);
                int arg_t = INT_MAX;
                if (mt >= cthr && mw != -INFINITY) {
                    uint32_t smask = 0;
#pragma unroll
                    for (int i = 0; i < VEC4; ++i)
                        if (m4[i] >= cthr) smask |= 1u << i;
#pragma unroll 1
                    while (smask && arg_t == INT_MAX) {
                        const int i = __ffs(smask) - 1;
                        smask &= smask - 1;
                        const int f = i * kCompute + tid;
                        float4 x4;
                        if (use_tma && f < nfull4) {
                            x4 = stage4[f];
                        } else {
                            x4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                            for (int q = 0; q < 4 && 4 * f + q < ncols; ++q) set_comp(x4, q, grow[4 * f + q]);
                        }
#pragma unroll 1
                        for (int q = 0; q < 4; ++q) {
                            const float x = comp(x4, q);
                            if (x >= cthr && sq.exact(x) == mw) {
                                arg_t = col0 + 4 * f + q;
                                break;
                            }
                        }
                    }
                }
                const int aw = warp_min_i(arg_t);
                if (!raw) {
#pragma unroll
                    for (int i = 0; i < VEC4; ++i) {
                        v[i].x = sq.exact(v[i].x);
                        v[i].y = sq.exact(v[i].y);
                        v[i].z = sq.exact(v[i].z);
                        v[i].w = sq.exact(v[i].w);
                    }
                }

                // t = (s - M_w) log2(e): raw domain x * log2(e)/Te - c with
                // c = RN(mxw * log2(e)/Te), else (s - M_w) * log2(e); -inf
                // gives a finite t whose e is 0
                float lscale, cref;
                if (raw) {
                    lscale = kLog2e * sq.y;
                    cref = mxw * lscale;
                } else {
                    lscale = kLog2e;
                    cref = 0.0f;
#pragma unroll
                    for (int i = 0; i < VEC4; ++i) {
                        v[i].x -= mw;
                        v[i].y -= mw;
                        v[i].z -= mw;
                        v[i].w -= mw;
                    }
                }
                // sums, four accumulators each; e waits in the stage
                float st[4] = {0.0f, 0.0f, 0.0f, 0.0f}, wt[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int i = 0; i < VEC4; ++i) {
                    if (i * kCompute < nslot4) {
                        float4 ev;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float t = fmaxf(fmaf(comp(v[i], q), lscale, -cref), -FLT_MAX);
                            const float e = ex2_approx(t);
                            set_comp(ev, q, e);
                            st[q] += e;
                            wt[q] = fmaf(e, t, wt[q]);
                        }
                        const int f = i * kCompute + tid;
                        if (f < nslot4) stage4[f] = ev;
                    }
                }
                const float sw = warp_sum_f((st[0] + st[1]) + (st[2] + st[3]));
                const float ww = warp_sum_f((wt[0] + wt[1]) + (wt[2] + wt[3])) * kLn2;
                if (lane == 0) {
                    sc.p1[k & (kRowRing - 1)][warp] = WarpPartial{mw, sw, ww, aw};
                    sc.wref[k & (kRowRing - 1)][warp] = mw;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sc.a_done[k & (kRowRing - 1)]);
            }

            const int j = k - LAG;
            if (j >= 0) {
                // ---- second half of row j --------------------------------------
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&sc.info_ready[j & (kRowRing - 1)],
                                                               static_cast<uint32_t>((j / kRowRing) & 1)))) {
                    if (lane == 0) fail();
                    break;
                }
                const RowInfo ri = sc.info[j & (kRowRing - 1)];
                const float mw = sc.wref[j & (kRowRing - 1)][warp];
                const int64_t frow = row_of(j);
                const float4* fstage =
                    reinterpret_cast<const float4*>(smem + (j % NSTAGE) * p.stage_bytes);
                float4 e[VEC4];
#pragma unroll
                for (int i = 0; i < VEC4; ++i) {
                    const int f = i * kCompute + tid;
                    e[i] = (i * kCompute < nslot4 && f < nslot4)
                               ? fstage[f]
                               : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                }
                // e^(s - B), widened by the race margin, is e * r_w; a group
                // whose largest e * r_w is below 2^-24 (<= 1 - u always) has
                // no element that can win.
                const float r_w = ri.noisy && mw != -INFINITY
                                      ? ex2_approx(fmaf(mw - ri.near_best, kLog2e, kRaceMarginLog2))
                                      : 0.0f;
                uint32_t pmask = 0;
#pragma unroll
                for (int i = 0; i < VEC4; ++i)
                    if (max4(e[i]) * r_w >= 0x1p-24f) pmask |= 1u << i;

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

                WarpBest wb{-INFINITY, INT_MAX};
                if (ri.noisy) {
                    wb = WarpBest{ri.near_best, ri.near_col};
                    // the groups that pass, listed warp-wide, one per lane
                    uint16_t* list = sc.worklist[warp];
                    const uint32_t lt = lanemask_lt();
                    int total = 0;
#pragma unroll
                    for (int i = 0; i < VEC4; ++i) {
                        const bool pass = (pmask >> i) & 1u;
                        const uint32_t b = __ballot_sync(0xffffffffu, pass);
                        if (pass) list[total + __popc(b & lt)] = static_cast<uint16_t>(i * kCompute + tid);
                        total += __popc(b);
                    }
                    __syncwarp();
                    const uint64_t fgrow_id = grow_of(j);
                    for (int n = lane; n < total; n += 32) {
                        const int f = list[n];
                        const float4 e4 = fstage[f];
                        const uint4 w = noise_words_rk(p.rk, fgrow_id, static_cast<uint32_t>((col0 >> 2) + f));
                        const uint32_t bits = race_group(e4, w, r_w);
                        if (bits)
                            wb = race_rescore(bits, p.logits + frow * p.row_stride, col0 + 4 * f, w,
                                              sc.rq[j & (kRowRing - 1)], ri.near_col, wb);
                    }
                    __syncwarp();  // the list is rewritten for the next row
                    warp_best(wb.best, wb.col);
                }
                if (lane == 0) sc.p2[j & (kRowRing - 1)][warp] = wb;
                __syncwarp();
                if (lane == 0) mbar_arrive(&sc.b_done[j & (kRowRing - 1)]);
            }
        }
    } else if (warp == kPublisherWarp) {
        // ======================= publisher warp ==================================
        // Stage a row: its temperature quotient for the CTA, then the bulk
        // copy (or, for rows that are not 16-byte aligned, a plain arrival:
        // the compute warps read global memory).
        float temp_next = nrows > 0 && lane == 0 ? row_temperature(p, grow_of(0)) : 0.0f;
        auto issue_row = [&](int r) {
            if (lane == 0) {
                const float temp = temp_next;
                if (r + 1 < nrows) temp_next = row_temperature(p, grow_of(r + 1));
                const ScaledQuotient q = ScaledQuotient::of(fmaxf(temp, kTempFloor));
                sc.rq[r & (kRowRing - 1)] = RowQuotient{temp, q.t, q.y, q.mode};
                uint64_t* bar = &sc.full[r % NSTAGE];
                if (use_tma) {
                    mbar_arrive_expect_tx(bar, copy_bytes);
                    if (copy_bytes)
                        tma_load_1d(smem + (r % NSTAGE) * p.stage_bytes,
                                    p.logits + row_of(r) * p.row_stride + col0, copy_bytes, bar);
                } else {
                    mbar_arrive(bar);
                }
            }
        };
        int issued = 0;
        while (issued < nrows && issued < NSTAGE) issue_row(issued++);
        for (int k = 0; k < nrows + LAG; ++k) {
            if (*abort_flag) break;
            if (k < nrows) {
                // ---- first record of row k ---------------------------------------
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&sc.a_done[k & (kRowRing - 1)],
                                                               static_cast<uint32_t>((k / kRowRing) & 1)))) {
                    if (lane == 0) fail();
                    break;
                }
                const WarpPartial wp = lane < kComputeWarps
                                           ? sc.p1[k & (kRowRing - 1)][lane]
                                           : WarpPartial{-INFINITY, 0.0f, 0.0f, INT_MAX};
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
                // B candidates: the Gumbel-max score of each warp's argmax
                // element, one lane per warp
                float b_c = -INFINITY;
                int bcol_c = INT_MAX;
                if (sc.rq[k & (kRowRing - 1)].temp > 0.0f && wp.arg != INT_MAX) {
                    const uint4 w = noise_words_rk(p.rk, grow_of(k), static_cast<uint32_t>(wp.arg >> 2));
                    b_c = wp.m + gumbel_of_bits(word_of(w, wp.arg & 3));
                    bcol_c = wp.arg;
                }
                warp_best(b_c, bcol_c);
                if (lane == 0 && !(p.fault && blockIdx.x == 0 && k == 0))
                    publish_a(record_a(p.xchg, blockIdx.x, k & (kRing - 1)), record_tag(k), mc, s_c,
                              w_c, a_c, b_c, bcol_c);
            }
            const int j = k - LAG;
            if (j >= 0) {
                // ---- second record of row j; its stage takes a later row ----------
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&sc.b_done[j & (kRowRing - 1)],
                                                               static_cast<uint32_t>((j / kRowRing) & 1)))) {
                    if (lane == 0) fail();
                    break;
                }
                const WarpBest wb = lane < kComputeWarps ? sc.p2[j & (kRowRing - 1)][lane]
                                                         : WarpBest{-INFINITY, INT_MAX};
                float b = wb.best;
                int bcol = wb.col;
                warp_best(b, bcol);
                if (lane == 0)
                    publish_b(record_b(p.xchg, blockIdx.x, j & (kRing - 1)), record_tag(j), b, bcol);
                if (issued < nrows) {
                    if (lane == 0) fence_proxy_async_smem();
                    issue_row(issued++);
                }
            }
        }
        // Bulk copies still in flight must land before the CTA's shared
        // memory is released.
        if (use_tma && lane == 0) {
            for (int r = issued > NSTAGE ? issued - NSTAGE : 0; r < issued; ++r)
                mbar_wait_bounded(&sc.full[r % NSTAGE], static_cast<uint32_t>((r / NSTAGE) & 1));
        }
    } else {
        // ======================= poller warp =====================================
        // Row m's first records, and the second records of row m-LAG-1. The
        // temperature (for the noise flag) is loaded a row ahead.
        float temp_m = nrows > 0 ? row_temperature(p, grow_of(0)) : 0.0f;
        for (int m = 0; m < nrows + LAG + 1; ++m) {
            if (*abort_flag) break;
            const float temp = temp_m;
            if (m + 1 < nrows) temp_m = row_temperature(p, grow_of(m + 1));
            const bool do_a = m < nrows;
            const int kb = m - (LAG + 1);
            const bool do_b = kb >= 0 && kb < nrows;
            bool ok = true;
            uint64_t ra[6] = {0, 0, 0, 0, 0, 0}, rb[2] = {0, 0};
            if (lane < p.team && (do_a || do_b)) {
                const int cta = team_id * p.team + lane;
                ok = read_records(do_a ? record_a(p.xchg, cta, m & (kRing - 1)) : nullptr,
                                  record_tag(m), ra,
                                  do_b ? record_b(p.xchg, cta, kb & (kRing - 1)) : nullptr,
                                  record_tag(kb), rb);
            }
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) fail();
                break;
            }
            const bool have = lane < p.team;
            if (do_a) {
                const int64_t frow = row_of(m);
                const float m_ = have ? payload_f(ra[0]) : -INFINITY;
                const float s_m = have ? payload_f(ra[1]) : 0.0f;
                const float w_m = have ? payload_f(ra[2]) : 0.0f;
                const int a_m = have ? static_cast<int>(payload_u(ra[3])) : INT_MAX;
                float b_m = have ? payload_f(ra[4]) : -INFINITY;
                int bc_m = have ? static_cast<int>(payload_u(ra[5])) : INT_MAX;
                const float big_m = warp_max(m_);
                float s_l = 0.0f, w_l = 0.0f;
                if (m_ != -INFINITY) {
                    const float dm = m_ - big_m;
                    const float f = ex2_approx(dm * kLog2e);
                    s_l = f * s_m;
                    w_l = f * fmaf(dm, s_m, w_m);
                }
                const float s_tot = warp_sum_f(s_l);
                const float w_tot = warp_sum_f(w_l);
                const int arg_row = warp_min_i(m_ == big_m ? a_m : INT_MAX);
                warp_best(b_m, bc_m);
                if (lane == 0) {
                    RowInfo& ri = sc.info[m & (kRowRing - 1)];
                    ri.row_max = big_m;
                    ri.log2s = s_tot > 0.0f ? log2f(s_tot) : 0.0f;
                    ri.near_best = b_m;
                    ri.near_col = bc_m;
                    ri.arg = arg_row;
                    ri.noisy = temp > 0.0f && big_m != -INFINITY;
                    mbar_arrive(&sc.info_ready[m & (kRowRing - 1)]);
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
                    const RowInfo& ri = sc.info[kb & (kRowRing - 1)];
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

// Team size G for one CTA per SM with 448 compute threads. The chunk must
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
